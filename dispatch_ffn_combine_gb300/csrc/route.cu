// route.cu -- router: fp32 gate logits in a fixed summation order, then top-k
// with the renormalised softmax weights.
//
// The pages name routing as the first step of the layer (mKernel README,
// kernel table, row "MoE Dispatch + FFN + Combine": "routes tokens to their
// expert ranks") but leave its arithmetic open.  Because the logits decide
// integers (which experts, hence every dispatch index), they are computed in
// one fixed order that the CPU oracle reproduces bit for bit:
//   32 interleaved partial sums s_j over i = j, j+32, ... (fused multiply-add,
//   round to nearest), then s_j += s_{j+off} for off = 16, 8, 4, 2, 1, then
//   + bias[e].
// A warp owns a 16-token x 8-expert block; lane j carries partial sum s_j of
// all 128 logits of the block, so the chains need no cross-lane traffic until
// the end.  The final tree is done as a transpose-reduction: at each level a
// lane keeps half of its accumulators and adds the partner's matching half,
// which performs exactly the additions s_j + s_{j+off} of the tree (fp32
// addition is commutative) with 124 shuffles instead of 640.
#include <math.h>

#include "mk_internal.h"

namespace mk {
namespace {

constexpr int kTT = 16;  // tokens per warp tile
constexpr int kTE = 8;   // experts per warp tile
constexpr int kAcc = kTT * kTE;

// One level of the transpose-reduction: lanes L and L^off exchange halves;
// each adds the partner's copy of the half it keeps.
template <int HALF>
__device__ __forceinline__ void reduce_level(float (&acc)[kAcc], int lane, int off) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int q = 0; q < HALF; ++q) {
        const float send = upper ? acc[q] : acc[q + HALF];
        const float keep = upper ? acc[q + HALF] : acc[q];
        const float recv = __shfl_xor_sync(0xffffffffu, send, off);
        acc[q] = __fadd_rn(keep, recv);
    }
}

template <int WT, int WE>
__global__ void __launch_bounds__(256) route_logits_kernel(const uint16_t* __restrict__ x,
                                                           const float* __restrict__ wg,
                                                           const float* __restrict__ bias, int T, int d, int E,
                                                           float* __restrict__ logits) {
    static_assert(WT * WE == 8, "8 warps per block");
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int wt = warp / WE;
    const int we = warp % WE;
    // 1-D grid, expert groups fastest: the blocks that read the same token rows
    // run together, so x comes from HBM once and from L2 for the other groups.
    const int n_eg = (E + kTE * WE - 1) / (kTE * WE);
    const int eg = static_cast<int>(blockIdx.x % n_eg);
    const int tg = static_cast<int>(blockIdx.x / n_eg);
    const int t0 = tg * (kTT * WT) + wt * kTT;
    const int e0 = eg * (kTE * WE) + we * kTE;
    if (t0 >= T || e0 >= E) return;  // uniform per warp; no block-level barrier below

    // Element offsets of this lane's first element in each row (rows past the
    // end are clamped to the last row; their results are not stored).
    int xo[kTT];
    int wo[kTE];
#pragma unroll
    for (int a = 0; a < kTT; ++a) xo[a] = min(t0 + a, T - 1) * d + lane;
#pragma unroll
    for (int b = 0; b < kTE; ++b) wo[b] = min(e0 + b, E - 1) * d + lane;

    float acc[kAcc];
#pragma unroll
    for (int q = 0; q < kAcc; ++q) acc[q] = 0.0f;

#pragma unroll 2
    for (int i = 0; i < d; i += 32) {
        float xv[kTT];
        float wv[kTE];
#pragma unroll
        for (int a = 0; a < kTT; ++a) xv[a] = __uint_as_float(static_cast<uint32_t>(__ldg(x + xo[a] + i)) << 16);
#pragma unroll
        for (int b = 0; b < kTE; ++b) wv[b] = __ldg(wg + wo[b] + i);
#pragma unroll
        for (int a = 0; a < kTT; ++a)
#pragma unroll
            for (int b = 0; b < kTE; ++b) acc[a * kTE + b] = __fmaf_rn(xv[a], wv[b], acc[a * kTE + b]);
    }

    // Transpose-reduction over the 32 lanes (see file comment).  After level
    // `off`, lane L holds, in acc[0 .. n/2), the level-`off` sums of partial
    // sum (L mod off) for half of its previous accumulators; after the last
    // level lane L holds the finished logits of accumulators 4L .. 4L+3.
    reduce_level<kAcc / 2>(acc, lane, 16);
    reduce_level<kAcc / 4>(acc, lane, 8);
    reduce_level<kAcc / 8>(acc, lane, 4);
    reduce_level<kAcc / 16>(acc, lane, 2);
    reduce_level<kAcc / 32>(acc, lane, 1);
    const int t = t0 + (lane >> 1);
    if (t < T) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = e0 + 4 * (lane & 1) + q;
            if (e < E) {
                float l = acc[q];
                if (bias != nullptr) l = __fadd_rn(l, __ldg(bias + e));
                logits[static_cast<int64_t>(t) * E + e] = l;
            }
        }
    }
}

// One warp per token: k rounds of a warp-wide arg-max (larger logit wins,
// equal logits go to the lower expert id), then the softmax over the chosen k.
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, int64_t T, int E, int k,
                                                   int32_t* __restrict__ ids, float* __restrict__ w,
                                                   int32_t* __restrict__ counts) {
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
                                float* logits, cudaStream_t s) {
    const uint16_t* xb = reinterpret_cast<const uint16_t*>(x);
    const int Ti = static_cast<int>(T);
    dim3 block(256);
    if (E >= 32) {
        const unsigned grid = static_cast<unsigned>(((E + 31) / 32) * ((T + 31) / 32));
        route_logits_kernel<2, 4><<<grid, block, 0, s>>>(xb, wg, bias, Ti, d, E, logits);
    } else if (E >= 16) {
        const unsigned grid = static_cast<unsigned>(((E + 15) / 16) * ((T + 63) / 64));
        route_logits_kernel<4, 2><<<grid, block, 0, s>>>(xb, wg, bias, Ti, d, E, logits);
    } else {
        const unsigned grid = static_cast<unsigned>(((E + 7) / 8) * ((T + 127) / 128));
        route_logits_kernel<8, 1><<<grid, block, 0, s>>>(xb, wg, bias, Ti, d, E, logits);
    }
    return cudaGetLastError();
}

cudaError_t launch_topk(const float* logits, int64_t T, int E, int k, int32_t* ids, float* w,
                        int32_t* counts_or_null, cudaStream_t s) {
    const unsigned blocks = static_cast<unsigned>((T + 7) / 8);
    topk_kernel<<<blocks, 256, 0, s>>>(logits, T, E, k, ids, w, counts_or_null);
    return cudaGetLastError();
}

}  // namespace mk
