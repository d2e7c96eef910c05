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

}  // namespace

cudaError_t launch_combine(const bf16* P, const int32_t* slot_row, int64_t T, int d, int k, bf16* y,
                           cudaStream_t s, int64_t p_rows) {
    // P has p_rows rows (T * k unless the tokens are a chunk of a larger batch)
    combine_kernel<<<static_cast<unsigned>(T), 128, 0, s>>>(P, slot_row, p_rows >= 0 ? p_rows : T * k, d, k, y);
    return cudaGetLastError();
}

}  // namespace mk
