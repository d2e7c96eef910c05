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
//
// Stores: a lane holds one output row, so a plain store of 16 bytes per lane
// touches 32 rows per warp instruction.  Each lane's 64 outputs (128 bytes, 8
// pieces of 16 bytes) are first exchanged within groups of 8 lanes (an 8 x 8
// transpose of pieces by three butterfly rounds of shuffles), after which a
// warp store writes 128 contiguous bytes of each of 4 rows: 8x fewer L2 write
// requests for the same bytes.

// pk[4q .. 4q+3] is piece q of this lane's row.  Afterwards it is piece gi of
// row (group base + q), gi = this lane's position in its group of 8.
__device__ __forceinline__ void transpose_pieces8(uint32_t (&pk)[32], int gi) {
#pragma unroll
    for (int b = 4; b >= 1; b >>= 1) {
        const bool hi = (gi & b) != 0;
#pragma unroll
        for (int q0 = 0; q0 < 8; ++q0) {
            if (q0 & b) continue;
            const int q1 = q0 | b;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const uint32_t send = hi ? pk[4 * q0 + w] : pk[4 * q1 + w];
                const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, b);
                if (hi)
                    pk[4 * q0 + w] = recv;
                else
                    pk[4 * q1 + w] = recv;
            }
        }
    }
}

// Stores 64 outputs per row for the warp's 32 rows after transpose_pieces8:
// lane (8 g + gi) writes piece gi of row 8 g + s with its s-th store.
// rows[s] is row 8 g + s's pointer, ok the rows that store (bit = lane), col
// this lane's first column (n0 + chunk + 8 gi).
__device__ __forceinline__ void store_pieces8(const uint32_t (&pk)[32], bf16* const (&rows)[8], uint32_t ok, int gbase,
                                              int col, int n_valid) {
#pragma unroll
    for (int s = 0; s < 8; ++s)
        if (((ok >> (gbase + s)) & 1u) && col < n_valid)
            *reinterpret_cast<uint4*>(rows[s] + col) =
                make_uint4(pk[4 * s], pk[4 * s + 1], pk[4 * s + 2], pk[4 * s + 3]);
}

__device__ __forceinline__ void group_rows8(bf16* orow, bf16* (&rows)[8], int gbase) {
    const uint64_t mine = reinterpret_cast<uint64_t>(orow);
#pragma unroll
    for (int s = 0; s < 8; ++s) rows[s] = reinterpret_cast<bf16*>(__shfl_sync(0xffffffffu, mine, gbase + s));
}

template <int G>
__device__ __forceinline__ void epilogue_swiglu_w(uint32_t tbase, bool row_ok, bf16* orow, int n0, int n_valid) {
    const int lane = threadIdx.x & 31;
    const int gi = lane & 7, gbase = lane & ~7;
    const uint32_t ok = __ballot_sync(0xffffffffu, row_ok);
    bf16* rows[8];
    group_rows8(orow, rows, gbase);
#pragma unroll 1
    for (int c = 0; c < G; c += 64) {
        uint32_t pk[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t g[32], u[32];
            tmem_ld_32x32b_x32(tbase + c + 32 * half, g);
            tmem_ld_32x32b_x32(tbase + G + c + 32 * half, u);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 16; ++q)
                pk[16 * half + q] = pack_bf16x2(silu_mul(__uint_as_float(g[2 * q]), __uint_as_float(u[2 * q])),
                                                silu_mul(__uint_as_float(g[2 * q + 1]), __uint_as_float(u[2 * q + 1])));
        }
        transpose_pieces8(pk, gi);
        store_pieces8(pk, rows, ok, gbase, n0 + c + 8 * gi, n_valid);
    }
}

// `pace` (SM cycles, 0: none) spaces the starts of the 64-column chunks at
// least that far apart, so that a tile's stores spread over the next tile's
// main loop instead of landing in a burst while its first operand loads are
// in flight (gemm2's output is 4x its operand bytes per tile).
template <int C>
__device__ __forceinline__ void epilogue_weighted_w(uint32_t tbase, bool row_ok, bf16* orow, int n0, int n_valid,
                                                    float wr, uint32_t pace = 0) {
    const int lane = threadIdx.x & 31;
    const int gi = lane & 7, gbase = lane & ~7;
    const uint32_t ok = __ballot_sync(0xffffffffu, row_ok);
    bf16* rows[8];
    group_rows8(orow, rows, gbase);
    const long long t0 = clock64();
#pragma unroll 1
    for (int c = 0; c < C; c += 64) {
        if (pace != 0u && c != 0)
            while (clock64() - t0 < static_cast<long long>(c / 64) * pace) __nanosleep(128);
        uint32_t a[32], b[32];
        tmem_ld_32x32b_x32(tbase + c, a);
        tmem_ld_32x32b_x32(tbase + c + 32, b);
        tmem_ld_wait();
        uint32_t pk[32];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            pk[q] = pack_bf16x2(__uint_as_float(a[2 * q]) * wr, __uint_as_float(a[2 * q + 1]) * wr);
            pk[16 + q] = pack_bf16x2(__uint_as_float(b[2 * q]) * wr, __uint_as_float(b[2 * q + 1]) * wr);
        }
        transpose_pieces8(pk, gi);
        store_pieces8(pk, rows, ok, gbase, n0 + c + 8 * gi, n_valid);
    }
}

__device__ __forceinline__ void epilogue_swiglu(uint32_t tbase, bool row_ok, bf16* orow, int n0, int n_valid) {
    epilogue_swiglu_w<128>(tbase, row_ok, orow, n0, n_valid);
}

__device__ __forceinline__ void epilogue_weighted(uint32_t tbase, bool row_ok, bf16* orow, int n0, int n_valid,
                                                  float wr, uint32_t pace = 0) {
    epilogue_weighted_w<MMA_N>(tbase, row_ok, orow, n0, n_valid, wr, pace);
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
