// gemm_impl.cuh -- pieces of the grouped expert GEMMs shared by the
// stand-alone GEMM kernels and the fused persistent layer kernel: tile
// constants, the two fused epilogues (SwiGLU for gemm1, routing weight for
// gemm2) and the TMA tensor-map encoding.
#pragma once

#include <cudaTypedefs.h>

#include <mutex>

#include "mk_device.cuh"
#include "mk_internal.h"

namespace mk {
namespace gemm_detail {

constexpr int BM = 128;
constexpr int BK = 64;  // one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;
constexpr int STAGES = 4;
constexpr int MMA_N = 256;
constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr uint32_t B_BYTES = MMA_N * BK * 2;
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 2 * MMA_N;
constexpr int NUM_THREADS = 192;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, MMA_N);

__device__ __forceinline__ float silu_mul(float g, float u) { return (g / (1.0f + expf(-g))) * u; }

// Epilogues for the TMEM lane this thread reads (every lane of the warp must
// call: tcgen05.ld is warp-wide); only rows with row_ok store.
//   SwiGLU, G gate columns at tbase, the matching G up columns at tbase + G:
//     h[n0 + c] = bf16(silu(g_c) * u_c), c < G
//   weighted, C columns at tbase:  P[n0 + c] = bf16(wr * acc_c), c < C
// A 128 x 256 single-CTA or 256 x 256 pair accumulator gives each lane
// G = 128 (gate | up) or C = 256.
template <int G>
__device__ __forceinline__ void epilogue_swiglu_w(uint32_t tbase, bool row_ok, bf16* orow, int n0, int n_valid) {
#pragma unroll 1
    for (int c = 0; c < G; c += 32) {
        uint32_t g[32], u[32];
        tmem_ld_32x32b_x32(tbase + c, g);
        tmem_ld_32x32b_x32(tbase + G + c, u);
        tmem_ld_wait();
        if (row_ok) {
            uint32_t pk[16];
#pragma unroll
            for (int q = 0; q < 16; ++q)
                pk[q] = pack_bf16x2(silu_mul(__uint_as_float(g[2 * q]), __uint_as_float(u[2 * q])),
                                    silu_mul(__uint_as_float(g[2 * q + 1]), __uint_as_float(u[2 * q + 1])));
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int col = n0 + c + 8 * v;
                if (col < n_valid)
                    *reinterpret_cast<uint4*>(orow + col) =
                        make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
        }
    }
}

template <int C>
__device__ __forceinline__ void epilogue_weighted_w(uint32_t tbase, bool row_ok, bf16* orow, int n0, int n_valid,
                                                    float wr) {
#pragma unroll 1
    for (int c = 0; c < C; c += 32) {
        uint32_t a[32];
        tmem_ld_32x32b_x32(tbase + c, a);
        tmem_ld_wait();
        if (row_ok) {
            uint32_t pk[16];
#pragma unroll
            for (int q = 0; q < 16; ++q)
                pk[q] = pack_bf16x2(__uint_as_float(a[2 * q]) * wr, __uint_as_float(a[2 * q + 1]) * wr);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int col = n0 + c + 8 * v;
                if (col < n_valid)
                    *reinterpret_cast<uint4*>(orow + col) =
                        make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
        }
    }
}

__device__ __forceinline__ void epilogue_swiglu(uint32_t tbase, bool row_ok, bf16* orow, int n0, int n_valid) {
    epilogue_swiglu_w<128>(tbase, row_ok, orow, n0, n_valid);
}

__device__ __forceinline__ void epilogue_weighted(uint32_t tbase, bool row_ok, bf16* orow, int n0, int n_valid,
                                                  float wr) {
    epilogue_weighted_w<MMA_N>(tbase, row_ok, orow, n0, n_valid, wr);
}

constexpr int PAIR_M = 2 * BM;  // rows of a CTA-pair tile

// Swap-tile epilogues: this thread's TMEM lane is one weight row (output
// column), its columns the block's rows.  A warp stores one output row per
// step (32 or 16 consecutive columns).
//   gemm2:  out[j][n] = bf16(wr[j] * acc_j), j < rows; the block's row weights
//           are loaded once, lane i holding rows i, i + 32, ...
__device__ __forceinline__ void epilogue_weighted_swap(uint32_t tbase, int rows, bf16* ocol, int64_t ld, bool n_ok,
                                                       const float* wr) {
    const int lane = threadIdx.x & 31;
    float wv[PAIR_M / 32];
#pragma unroll
    for (int c = 0; c < PAIR_M / 32; ++c) {
        const int j = 32 * c + lane;
        wv[c] = (wr != nullptr && j < rows) ? wr[j] : 1.0f;
    }
#pragma unroll 1
    for (int c = 0; 32 * c < rows; ++c) {
        uint32_t a[32];
        tmem_ld_32x32b_x32(tbase + 32 * c, a);
        float w_lane = wv[0];
#pragma unroll
        for (int q = 1; q < PAIR_M / 32; ++q)
            if (q == c) w_lane = wv[q];
        tmem_ld_wait();
        const int nj = rows - 32 * c;
        bf16* o = ocol + static_cast<int64_t>(32 * c) * ld;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            const float wj = __shfl_sync(0xffffffffu, w_lane, jj);
            if (n_ok && jj < nj) *o = __float2bfloat16_rn(__uint_as_float(a[jj]) * wj);
            o += ld;
        }
    }
}

//   gemm1:  lanes l and l + 16 hold the gate and up rows of one column; one
//           exchange per pair of block rows gives lane l the up value of the
//           even row and lane l + 16 the gate value of the odd one:
//           h[j][col] = bf16(silu(g_j) * u_j), even j by lanes 0-15, odd j by 16-31
__device__ __forceinline__ void epilogue_swiglu_swap(uint32_t tbase, int rows, bf16* ocol, int64_t ld, bool c_ok) {
    const bool lo = (threadIdx.x & 16) == 0;
#pragma unroll 1
    for (int j0 = 0; j0 < rows; j0 += 32) {
        uint32_t a[32];
        tmem_ld_32x32b_x32(tbase + j0, a);
        tmem_ld_wait();
        const int nj = rows - j0;
        bf16* o = ocol + static_cast<int64_t>(j0 + (lo ? 0 : 1)) * ld;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const float x = __shfl_xor_sync(0xffffffffu, __uint_as_float(lo ? a[2 * m + 1] : a[2 * m]), 16);
            const float g = lo ? __uint_as_float(a[2 * m]) : x;
            const float u = lo ? x : __uint_as_float(a[2 * m + 1]);
            if (c_ok && 2 * m + (lo ? 0 : 1) < nj) *o = __float2bfloat16_rn(silu_mul(g, u));
            o += 2 * ld;
        }
    }
}

// Tile-synchronised path: index of the first 128-row M-tile of a block of
// expert e's rows that starts at row0 (a multiple of 128 rows into the
// expert), in the tile table's numbering.
__device__ __forceinline__ int sem_tile0(const int32_t* offsets, const int32_t* mtile_start, int e, int row0) {
    return __ldg(mtile_start + e) + (row0 - __ldg(offsets + e)) / BM;
}

// ------------------------------------------------------------------ host side

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D bf16 tensor [rows, inner] (row-major), box {64, box_rows}, 128-byte swizzle.
inline bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gemm_detail
}  // namespace mk
