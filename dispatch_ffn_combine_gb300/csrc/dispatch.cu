// dispatch.cu -- deterministic dispatch of routed token rows into
// expert-contiguous order, the single-GPU form of the README's "All-to-All
// dispatch" (mKernel README, kernel table, row "MoE Dispatch + FFN +
// Combine"; the paper's Table 3 describes the expert-parallel version as a
// TMA pull of tokens from peers, 16 tokens per chunk).
//
// Row order inside an expert's block is ascending token id, so every index is
// a pure function of the routing (no atomics decide a position):
//   1. count:   per chunk of 128 tokens, a 128-bit mask per expert marks the
//               tokens that chose it; popcounts give the chunk's per-expert
//               count and each (token, slot)'s rank inside the chunk.
//   2. scan:    per expert, an exclusive scan over chunks (chunk bases), then
//               an exclusive scan over experts (offsets) and of the per-expert
//               128-row tile counts (the grouped GEMM's tile table).
//   3. scatter: row = offsets[e] + chunk_base[c][e] + rank; copy the token row
//               once from HBM and write it to its k rows with 16-byte stores.
#include "mk_device.cuh"
#include "mk_internal.h"

namespace mk {
namespace {

__global__ void __launch_bounds__(256) count_kernel(const int32_t* __restrict__ ids, int64_t T, int E, int k,
                                                    int32_t* __restrict__ chunk_counts, int32_t* __restrict__ rank,
                                                    uint32_t* status) {
    __shared__ uint32_t mask[kMaxExperts][kChunkTokens / 32];
    const int64_t c = blockIdx.x;
    const int64_t t_begin = c * kChunkTokens;
    const int nt = static_cast<int>((T - t_begin < kChunkTokens) ? (T - t_begin) : kChunkTokens);
    for (int i = threadIdx.x; i < E * (kChunkTokens / 32); i += blockDim.x) (&mask[0][0])[i] = 0u;
    __syncthreads();
    for (int q = threadIdx.x; q < nt * k; q += blockDim.x) {
        const int tl = q / k;
        const int e = ids[t_begin * k + q];
        if (e < 0 || e >= E) {
            report_error(status, MK_ERR_BOUNDS, kSiteCountIds);
            continue;
        }
        const uint32_t bit = 1u << (tl & 31);
        const uint32_t old = atomicOr(&mask[e][tl >> 5], bit);
        if (old & bit) report_error(status, MK_ERR_BOUNDS, kSiteCountRepeat);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int n = 0;
#pragma unroll
        for (int w = 0; w < kChunkTokens / 32; ++w) n += __popc(mask[e][w]);
        chunk_counts[c * E + e] = n;
    }
    for (int q = threadIdx.x; q < nt * k; q += blockDim.x) {
        const int tl = q / k;
        const int e = ids[t_begin * k + q];
        int r = 0;
        if (e >= 0 && e < E) {
            const int w = tl >> 5;
            for (int ww = 0; ww < w; ++ww) r += __popc(mask[e][ww]);
            r += __popc(mask[e][w] & ((1u << (tl & 31)) - 1u));
        }
        rank[t_begin * k + q] = r;
    }
}

__device__ __forceinline__ int warp_inclusive_scan(int v, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += u;
    }
    return v;
}

// Exclusive scans over experts, by one warp (E <= 256: 8 experts per lane).
// Writes offsets[0..E] and mtile_start[0..E] from per-expert counts in smem.
__device__ void expert_scan_warp(const int32_t* s_counts, int E, int lane, int32_t* offsets, int32_t* mtile_start) {
    int cnt[8];
    int til[8];
    int sum_c = 0, sum_t = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = lane * 8 + i;
        cnt[i] = (e < E) ? s_counts[e] : 0;
        til[i] = (cnt[i] + kTileM - 1) / kTileM;
        sum_c += cnt[i];
        sum_t += til[i];
    }
    const int inc_c = warp_inclusive_scan(sum_c, lane);
    const int inc_t = warp_inclusive_scan(sum_t, lane);
    int run_c = inc_c - sum_c, run_t = inc_t - sum_t;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = lane * 8 + i;
        if (e < E) {
            offsets[e] = run_c;
            mtile_start[e] = run_t;
        }
        run_c += cnt[i];
        run_t += til[i];
    }
    if (lane == 31) {
        offsets[E] = inc_c;
        mtile_start[E] = inc_t;
    }
}

__global__ void __launch_bounds__(1024) scan_kernel(const int32_t* __restrict__ chunk_counts, int64_t nchunks, int E,
                                                    int32_t* __restrict__ chunk_base, int32_t* __restrict__ counts,
                                                    int32_t* __restrict__ offsets,
                                                    int32_t* __restrict__ mtile_start) {
    __shared__ int32_t s_counts[kMaxExperts];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    for (int e = warp; e < E; e += nwarps) {
        int running = 0;
        for (int64_t c0 = 0; c0 < nchunks; c0 += 32) {
            const int64_t c = c0 + lane;
            const int v = (c < nchunks) ? chunk_counts[c * E + e] : 0;
            const int inc = warp_inclusive_scan(v, lane);
            if (c < nchunks) chunk_base[c * E + e] = running + inc - v;
            running += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) {
            s_counts[e] = running;
            counts[e] = running;
        }
    }
    __syncthreads();
    if (warp == 0) expert_scan_warp(s_counts, E, lane, offsets, mtile_start);
}

// Tile table for caller-supplied offsets (expert FFN entry point).  Offsets
// that are not a non-decreasing sequence from 0 to S are rejected: the error
// is recorded and the table is zeroed so the GEMMs run no tiles.
__global__ void __launch_bounds__(32) mtile_table_kernel(const int32_t* __restrict__ offsets, int E, int64_t S,
                                                         int32_t* __restrict__ mtile_start, uint32_t* status) {
    __shared__ int32_t s_counts[kMaxExperts];
    __shared__ int bad;
    const int lane = threadIdx.x;
    if (lane == 0) bad = (offsets[0] != 0 || offsets[E] != S) ? 1 : 0;
    __syncwarp();
    for (int e = lane; e < E; e += 32) {
        const int n = offsets[e + 1] - offsets[e];
        if (n < 0) atomicExch(&bad, 1);
        s_counts[e] = n;
    }
    __syncwarp();
    if (bad) {
        if (lane == 0) report_error(status, MK_ERR_BOUNDS, 0x700);
        for (int e = lane; e <= E; e += 32) mtile_start[e] = 0;
        return;
    }
    int cnt[8], til[8], sum_t = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = lane * 8 + i;
        cnt[i] = (e < E) ? s_counts[e] : 0;
        til[i] = (cnt[i] + kTileM - 1) / kTileM;
        sum_t += til[i];
    }
    const int inc_t = warp_inclusive_scan(sum_t, lane);
    int run_t = inc_t - sum_t;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = lane * 8 + i;
        if (e < E) mtile_start[e] = run_t;
        run_t += til[i];
    }
    if (lane == 31) mtile_start[E] = inc_t;
}

// One block per token: read the row once, write it to its k destination rows.
__global__ void __launch_bounds__(128) scatter_kernel(const bf16* __restrict__ x, const int32_t* __restrict__ ids,
                                                      const float* __restrict__ w, int64_t T, int d, int E, int k,
                                                      const int32_t* __restrict__ offsets,
                                                      const int32_t* __restrict__ chunk_base,
                                                      const int32_t* __restrict__ rank, bf16* __restrict__ x_perm,
                                                      int32_t* __restrict__ row_token, float* __restrict__ row_weight,
                                                      int32_t* __restrict__ slot_row) {
    __shared__ int64_t rows[kMaxTopK];
    const int64_t t = blockIdx.x;
    const int64_t S = T * k;
    if (threadIdx.x < k) {
        const int j = threadIdx.x;
        const int e = ids[t * k + j];
        int64_t r = -1;
        if (e >= 0 && e < E) {
            r = static_cast<int64_t>(offsets[e]) + chunk_base[(t / kChunkTokens) * E + e] + rank[t * k + j];
            if (r < 0 || r >= S) r = -1;
        }
        rows[j] = r;
        slot_row[t * k + j] = static_cast<int32_t>(r);
        if (r >= 0) {
            row_token[r] = static_cast<int32_t>(t);
            if (row_weight != nullptr) row_weight[r] = (w != nullptr) ? w[t * k + j] : 1.0f;
        }
    }
    __syncthreads();
    const int n16 = d / 8;  // 16-byte chunks per row
    const uint4* src = reinterpret_cast<const uint4*>(x + t * d);
    for (int c = threadIdx.x; c < n16; c += blockDim.x) {
        const uint4 v = __ldg(src + c);
        for (int j = 0; j < k; ++j) {
            const int64_t r = rows[j];
            if (r >= 0) reinterpret_cast<uint4*>(x_perm + r * d)[c] = v;
        }
    }
}

}  // namespace

cudaError_t launch_count(const int32_t* ids, int64_t T, int E, int k, int32_t* chunk_counts, int32_t* rank,
                         uint32_t* status, cudaStream_t s) {
    count_kernel<<<static_cast<unsigned>(num_chunks(T)), 256, 0, s>>>(ids, T, E, k, chunk_counts, rank, status);
    return cudaGetLastError();
}

cudaError_t launch_scan(const int32_t* chunk_counts, int64_t nchunks, int E, int32_t* chunk_base, int32_t* counts,
                        int32_t* offsets, int32_t* mtile_start, cudaStream_t s) {
    scan_kernel<<<1, 1024, 0, s>>>(chunk_counts, nchunks, E, chunk_base, counts, offsets, mtile_start);
    return cudaGetLastError();
}

cudaError_t launch_mtile_table(const int32_t* offsets, int E, int64_t S, int32_t* mtile_start, uint32_t* status,
                               cudaStream_t s) {
    mtile_table_kernel<<<1, 32, 0, s>>>(offsets, E, S, mtile_start, status);
    return cudaGetLastError();
}

cudaError_t launch_scatter(const bf16* x, const int32_t* ids, const float* w, int64_t T, int d, int E, int k,
                           const int32_t* offsets, const int32_t* chunk_base, const int32_t* rank, bf16* x_perm,
                           int32_t* row_token, float* row_weight, int32_t* slot_row, cudaStream_t s) {
    scatter_kernel<<<static_cast<unsigned>(T), 128, 0, s>>>(x, ids, w, T, d, E, k, offsets, chunk_base, rank, x_perm,
                                                             row_token, row_weight, slot_row);
    return cudaGetLastError();
}

}  // namespace mk
