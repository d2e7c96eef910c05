// combine.cu -- the weighted combine back to token order (mKernel README,
// kernel table, row "MoE Dispatch + FFN + Combine": "combines the weighted
// expert outputs back to each token's source rank"; on one GPU, back to the
// token's own row).
//
// The routing weight is already applied by the second GEMM's epilogue, so the
// combine is a plain gather-sum: y[t] = bf16( sum_j P[slot_row[t, j]] ), the k
// rows added in ascending slot order in fp32.  The order is fixed, so the
// result is bitwise reproducible run to run.  HBM-bound: reads k rows of P and
// writes one row of y per token, 16 bytes per thread per access.
#include "mk_device.cuh"
#include "mk_internal.h"

namespace mk {
namespace {

__global__ void __launch_bounds__(128) combine_kernel(const bf16* __restrict__ P, const int32_t* __restrict__ slot_row,
                                                      int64_t S, int d, int k, bf16* __restrict__ y) {
    __shared__ int64_t rows[kMaxTopK];
    const int64_t t = blockIdx.x;
    if (threadIdx.x < k) {
        const int64_t r = slot_row[t * k + threadIdx.x];
        rows[threadIdx.x] = (r >= 0 && r < S) ? r : -1;
    }
    __syncthreads();
    const int n16 = d / 8;
    uint4* dst = reinterpret_cast<uint4*>(y + t * d);
    for (int c = threadIdx.x; c < n16; c += blockDim.x) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        for (int j = 0; j < k; ++j) {
            const int64_t r = rows[j];
            if (r < 0) continue;
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(P + r * d) + c);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] = __fadd_rn(acc[2 * i], __uint_as_float(wv[i] << 16));
                acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __uint_as_float(wv[i] & 0xffff0000u));
            }
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        dst[c] = o;
    }
}

// Copy of `n16` 16-byte words between device memory and page-locked host
// memory mapped for the device, by a few CTAs' plain loads and stores
// (grid-stride): the pipelined host-buffer entry point's upload of x and
// download of y, each run beside another call's kernels on a handful of SMs
// instead of the copy engine.
__global__ void __launch_bounds__(256) bulk_copy_kernel(const uint4* __restrict__ src, uint4* dst, int64_t n16) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {  // four loads in flight per thread
        const uint4 a = __ldg(src + i), b = __ldg(src + i + stride), c = __ldg(src + i + 2 * stride),
                    e = __ldg(src + i + 3 * stride);
        dst[i] = a;
        dst[i + stride] = b;
        dst[i + 2 * stride] = c;
        dst[i + 3 * stride] = e;
    }
    for (; i < n16; i += stride) dst[i] = __ldg(src + i);
}

// The tile-synchronised path's combine, launched while gemm2 may still run:
// thread 0 waits until the dispatch has written every token's slot rows
// (tok_done), then threads j < k find the M-tile of row slot_row[t, j] (its
// expert by a binary search over the offsets) and wait until gemm2 has
// published that M-tile for every N block (p_ready); P is then read from L2
// (ld.global.cg: P is written during this kernel's lifetime, so the
// non-coherent read-only path may not be used).  Same sum, same order as
// combine_kernel.  A wait that runs out records MK_ERR_TIMEOUT and the token is
// skipped.
__global__ void __launch_bounds__(128) combine_sem_kernel(const bf16* P, const int32_t* slot_row,
                                                          const int32_t* offsets, const int32_t* mtile_start,
                                                          int64_t T, int d, int E, int k, bf16* y,
                                                          const uint32_t* tok_done, const uint32_t* p_ready, int pairs,
                                                          int n_tiles, int swap_max, uint32_t* status,
                                                          uint64_t timeout_ns) {
    __shared__ int64_t rows[kMaxTopK];
    __shared__ int ok;
    const int64_t t = blockIdx.x;
    const int64_t S = T * k;
    if (threadIdx.x == 0) {
        ok = wait_count_bounded(tok_done, static_cast<uint32_t>(T), nullptr, timeout_ns) ? 1 : 0;
        if (!ok) report_error(status, MK_ERR_TIMEOUT, kSiteCombineWait);
    }
    __syncthreads();
    if (!ok) return;
    if (threadIdx.x < k) {
        int64_t r = slot_row[t * k + threadIdx.x];
        if (r >= 0 && r < S) {
            int lo = 0, hi = E - 1;  // the expert holding row r: largest e with offsets[e] <= r
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (offsets[mid] <= r)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            const int in_e = static_cast<int>(r - offsets[lo]);
            const int cnt = offsets[lo + 1] - offsets[lo];
            const int g = mtile_start[lo] + in_e / kTileM;
            uint32_t want = 4u * static_cast<uint32_t>(n_tiles);
            if (pairs) {
                const int block_rows = min(2 * kTileM, cnt - (in_e / (2 * kTileM)) * (2 * kTileM));
                if (block_rows <= swap_max) want = 8u * static_cast<uint32_t>(n_tiles);
            }
            if (!wait_count_bounded(p_ready + g, want, nullptr, timeout_ns)) {
                report_error(status, MK_ERR_TIMEOUT, kSiteCombineWait);
                r = -1;
            }
        } else {
            r = -1;
        }
        rows[threadIdx.x] = r;
    }
    __syncthreads();
    const int n16 = d / 8;
    uint4* dst = reinterpret_cast<uint4*>(y + t * d);
    for (int c = threadIdx.x; c < n16; c += blockDim.x) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        for (int j = 0; j < k; ++j) {
            const int64_t r = rows[j];
            if (r < 0) continue;
            const uint4 v = __ldcg(reinterpret_cast<const uint4*>(P + r * d) + c);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] = __fadd_rn(acc[2 * i], __uint_as_float(wv[i] << 16));
                acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __uint_as_float(wv[i] & 0xffff0000u));
            }
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        dst[c] = o;
    }
}

}  // namespace

cudaError_t launch_combine_sem(const bf16* P, const int32_t* slot_row, const int32_t* offsets,
                               const int32_t* mtile_start, int64_t T, int d, int E, int k, bf16* y,
                               const TileSems& sem, bool pairs, int n_tiles, int swap_max, uint32_t* status,
                               uint64_t timeout_ns, cudaStream_t s) {
    LaunchCfg lc(dim3(static_cast<unsigned>(T)), dim3(128), 0, s, sem.pdl);
    const cudaError_t err =
        cudaLaunchKernelEx(&lc.cfg, combine_sem_kernel, P, slot_row, offsets, mtile_start, T, d, E, k, y,
                           static_cast<const uint32_t*>(sem.tok_done), static_cast<const uint32_t*>(sem.p_ready),
                           pairs ? 1 : 0, n_tiles, swap_max, status, timeout_ns);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

cudaError_t launch_bulk_copy(const void* src, void* dst, size_t bytes, int blocks, cudaStream_t s) {
    if (bytes == 0) return cudaSuccess;
    bulk_copy_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                                           static_cast<int64_t>(bytes / 16));
    return cudaGetLastError();
}

cudaError_t launch_combine(const bf16* P, const int32_t* slot_row, int64_t T, int d, int k, bf16* y,
                           cudaStream_t s, int64_t p_rows) {
    // P has p_rows rows (T * k unless the tokens are a chunk of a larger batch)
    combine_kernel<<<static_cast<unsigned>(T), 128, 0, s>>>(P, slot_row, p_rows >= 0 ? p_rows : T * k, d, k, y);
    return cudaGetLastError();
}

}  // namespace mk
