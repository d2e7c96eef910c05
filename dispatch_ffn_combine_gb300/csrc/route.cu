// route.cu -- router kernels: fp32 gate logits in a fixed summation order
// (the block computation lives in route_impl.cuh, shared with the fused
// layer kernel), then top-k with the renormalised softmax weights.
#include <atomic>
#include <math.h>

#include "route_impl.cuh"

namespace mk {
namespace {

using route_detail::RouteTile;

// 1-D grid, expert groups fastest: the blocks that read the same token rows
// run together, so x comes from HBM once and from L2 for the other groups.
template <int WT, int WE, int HT, int MINB>
__global__ void __launch_bounds__(256, MINB) route_logits_kernel(const uint16_t* __restrict__ x,
                                                              const float* __restrict__ wg,
                                                              const float* __restrict__ bias, int T, int d, int E,
                                                              float* __restrict__ logits) {
    using RT = RouteTile<WT, WE, HT, MINB>;
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_wait();  // as a programmatic dependent: the kernel ahead has finished
    pdl_launch_dependents();
    const int n_eg = (E + RT::CE - 1) / RT::CE;
    route_detail::route_block<WT, WE, HT, MINB>(smem, x, wg, bias, T, d, E, logits,
                                                 static_cast<int>(blockIdx.x / n_eg),
                                                 static_cast<int>(blockIdx.x % n_eg));
}

template <int WT, int WE, int HT, int MINB>
cudaError_t launch_logits_shape(const uint16_t* xb, const float* wg, const float* bias, int64_t T, int d, int E,
                                float* logits, cudaStream_t s, bool pdl) {
    using RT = RouteTile<WT, WE, HT, MINB>;
    static std::atomic<int> configured[64];  // per device: attributes set (repeating them is harmless)
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
        err = cudaFuncSetAttribute(route_logits_kernel<WT, WE, HT, MINB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   RT::SMEM);
        if (err != cudaSuccess) return err;
        if (dev < 64) configured[dev].store(1, std::memory_order_release);
    }
    const unsigned grid = static_cast<unsigned>(((E + RT::CE - 1) / RT::CE) * ((T + RT::CT - 1) / RT::CT));
    LaunchCfg lc(dim3(grid), dim3(256), RT::SMEM, s, pdl);
    err = cudaLaunchKernelEx(&lc.cfg, route_logits_kernel<WT, WE, HT, MINB>, xb, wg, bias, static_cast<int>(T), d, E,
                             logits);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

// One warp per token: k rounds of a warp-wide arg-max (larger logit wins,
// equal logits go to the lower expert id), then the softmax over the chosen k.
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, int64_t T, int E, int k,
                                                   int32_t* __restrict__ ids, float* __restrict__ w,
                                                   int32_t* __restrict__ counts) {
    pdl_wait();  // as a programmatic dependent: the logits are complete
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    constexpr int kNone = 0x7fffffff;
    float v[kMaxExperts / 32];
#pragma unroll
    for (int q = 0; q < kMaxExperts / 32; ++q) {
        const int e = lane + 32 * q;
        v[q] = (e < E) ? __ldg(logits + t * E + e) : 0.0f;
    }
    uint32_t taken = 0;
    float sel_v[kMaxTopK];
    int sel_i[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
        if (j >= k) break;
        float bv = 0.0f;
        int bi = kNone;
#pragma unroll
        for (int q = 0; q < kMaxExperts / 32; ++q) {
            const int e = lane + 32 * q;
            if (e < E && !((taken >> q) & 1u) && (bi == kNone || v[q] > bv)) {
                bv = v[q];
                bi = e;
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (oi != kNone && (bi == kNone || ov > bv || (ov == bv && oi < bi))) {
                bv = ov;
                bi = oi;
            }
        }
        sel_v[j] = bv;
        sel_i[j] = bi;
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    }
    if (lane == 0) {
        float ex[kMaxTopK];
        float z = 0.0f;
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
            if (j >= k) break;
            ex[j] = expf(sel_v[j] - sel_v[0]);
            z += ex[j];
        }
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
            if (j >= k) break;
            ids[t * k + j] = sel_i[j];
            w[t * k + j] = ex[j] / z;
            if (counts != nullptr) atomicAdd(counts + sel_i[j], 1);
        }
    }
}

}  // namespace

cudaError_t launch_route_logits(const bf16* x, const float* wg, const float* bias, int64_t T, int d, int E,
                                float* logits, cudaStream_t s, bool pdl) {
    const uint16_t* xb = reinterpret_cast<const uint16_t*>(x);
    // 32 x 32 blocks when there are enough experts, else 64 tokens x 16 experts
    // (expert rows past E are clamped duplicates whose logits are not stored).
    if (E >= 32) return launch_logits_shape<2, 4, 8, 1>(xb, wg, bias, T, d, E, logits, s, pdl);
    return launch_logits_shape<4, 2, 8, 1>(xb, wg, bias, T, d, E, logits, s, pdl);
}

cudaError_t launch_topk(const float* logits, int64_t T, int E, int k, int32_t* ids, float* w,
                        int32_t* counts_or_null, cudaStream_t s, bool pdl) {
    const unsigned blocks = static_cast<unsigned>((T + 7) / 8);
    LaunchCfg lc(dim3(blocks), dim3(256), 0, s, pdl);
    const cudaError_t err = cudaLaunchKernelEx(&lc.cfg, topk_kernel, logits, T, E, k, ids, w, counts_or_null);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace mk
