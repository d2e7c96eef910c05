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
    pdl_wait();  // as a programmatic dependent: the routing is complete
    pdl_launch_dependents();
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

// Scans after counting.  Block g takes experts [32 g, 32 g + 32), one per lane
// (loads coalesced across experts); warp w takes a contiguous segment of the
// chunks.  Per expert: segment sums, an exclusive scan over the segments, then
// the chunk bases.  The last block to finish (ticket in `done`, reset by that
// block) scans over experts: offsets and the 128-row tile table.
__global__ void __launch_bounds__(1024) scan_kernel(const int32_t* __restrict__ chunk_counts, int64_t nchunks, int E,
                                                    int32_t* __restrict__ chunk_base, int32_t* __restrict__ counts,
                                                    int32_t* __restrict__ offsets, int32_t* __restrict__ mtile_start,
                                                    uint32_t* done) {
    __shared__ int32_t s_part[32][33];
    __shared__ int32_t s_counts[kMaxExperts];
    __shared__ int s_last;
    pdl_wait();  // as a programmatic dependent: the chunk counts are complete
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int e = blockIdx.x * 32 + lane;
    const bool valid = e < E;
    const int64_t seg = (nchunks + 31) / 32;
    const int64_t c0 = warp * seg;
    const int64_t c1 = (c0 + seg < nchunks) ? c0 + seg : nchunks;
    int sum = 0;
    for (int64_t c = c0; c < c1; ++c) sum += valid ? __ldg(chunk_counts + c * E + e) : 0;
    s_part[warp][lane] = sum;
    __syncthreads();
    if (warp == 0) {  // exclusive scan over the 32 segments of expert `lane`
        int run = 0;
        for (int w = 0; w < 32; ++w) {
            const int v = s_part[w][lane];
            s_part[w][lane] = run;
            run += v;
        }
        if (valid) counts[e] = run;
    }
    __syncthreads();
    int run = s_part[warp][lane];
    for (int64_t c = c0; c < c1; ++c) {
        if (valid) {
            const int v = __ldg(chunk_counts + c * E + e);
            chunk_base[c * E + e] = run;
            run += v;
        }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(done, 1u) == gridDim.x - 1) ? 1 : 0;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int i = threadIdx.x; i < E; i += blockDim.x) s_counts[i] = __ldcg(counts + i);
    __syncthreads();
    if (warp == 0) expert_scan_warp(s_counts, E, lane, offsets, mtile_start);
    if (threadIdx.x == 0) *done = 0u;  // ready for the next call
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
// With mt_rows (the tile-synchronised path) each written row is published on
// its M-tile's counter and the token on tok_done, with release semantics after
// a proxy fence by every writing thread (the rows are read next by TMA).
__global__ void __launch_bounds__(128) scatter_kernel(const bf16* __restrict__ x, const int32_t* __restrict__ ids,
                                                      const float* __restrict__ w, int64_t T, int d, int E, int k,
                                                      const int32_t* __restrict__ offsets,
                                                      const int32_t* __restrict__ chunk_base,
                                                      const int32_t* __restrict__ rank, bf16* __restrict__ x_perm,
                                                      int32_t* __restrict__ row_token, float* __restrict__ row_weight,
                                                      int32_t* __restrict__ slot_row, uint32_t* mt_rows,
                                                      uint32_t* tok_done, const int32_t* __restrict__ mtile_start,
                                                      int drop_token0, int copy_rows) {
    __shared__ int64_t rows[kMaxTopK];
    __shared__ int32_t tiles[kMaxTopK];
    pdl_wait();  // as a programmatic dependent: offsets, chunk bases and ranks are complete
    pdl_launch_dependents();
    const int64_t t = blockIdx.x;
    const int64_t S = T * k;
    if (threadIdx.x < k) {
        const int j = threadIdx.x;
        const int e = ids[t * k + j];
        int64_t r = -1;
        int32_t g = -1;
        if (e >= 0 && e < E) {
            const int64_t in_e = static_cast<int64_t>(chunk_base[(t / kChunkTokens) * E + e]) + rank[t * k + j];
            r = static_cast<int64_t>(offsets[e]) + in_e;
            if (r < 0 || r >= S) r = -1;
            if (r >= 0 && mt_rows != nullptr) g = mtile_start[e] + static_cast<int32_t>(in_e / kTileM);
        }
        rows[j] = r;
        tiles[j] = g;
        slot_row[t * k + j] = static_cast<int32_t>(r);
        if (r >= 0) {
            row_token[r] = static_cast<int32_t>(t);
            if (row_weight != nullptr) row_weight[r] = (w != nullptr) ? w[t * k + j] : 1.0f;
        }
    }
    __syncthreads();
    const int n16 = copy_rows ? d / 8 : 0;  // 16-byte chunks per row (none: only the index tables)
    const uint4* src = reinterpret_cast<const uint4*>(x + t * d);
    for (int c = threadIdx.x; c < n16; c += blockDim.x) {
        const uint4 v = __ldg(src + c);
        for (int j = 0; j < k; ++j) {
            const int64_t r = rows[j];
            if (r >= 0) reinterpret_cast<uint4*>(x_perm + r * d)[c] = v;
        }
    }
    if (mt_rows != nullptr) {
        // every writer's proxy fence (the rows are read next through TMA); the
        // block barrier orders all threads' stores before the release increments,
        // which are cumulative over them
        fence_proxy_async_global();
        __syncthreads();
        const bool drop = drop_token0 != 0 && t == 0;  // test hook: these rows never count as landed
        if (threadIdx.x < k && tiles[threadIdx.x] >= 0 && !drop) red_release_gpu_add(mt_rows + tiles[threadIdx.x], 1u);
        if (threadIdx.x == 0) red_release_gpu_add(tok_done, 1u);
    }
}

}  // namespace

cudaError_t launch_count(const int32_t* ids, int64_t T, int E, int k, int32_t* chunk_counts, int32_t* rank,
                         uint32_t* status, cudaStream_t s, bool pdl) {
    LaunchCfg lc(dim3(static_cast<unsigned>(num_chunks(T))), dim3(256), 0, s, pdl);
    const cudaError_t err = cudaLaunchKernelEx(&lc.cfg, count_kernel, ids, T, E, k, chunk_counts, rank, status);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

cudaError_t launch_scan(const int32_t* chunk_counts, int64_t nchunks, int E, int32_t* chunk_base, int32_t* counts,
                        int32_t* offsets, int32_t* mtile_start, uint32_t* done, cudaStream_t s, bool pdl) {
    LaunchCfg lc(dim3((E + 31) / 32), dim3(1024), 0, s, pdl);
    const cudaError_t err = cudaLaunchKernelEx(&lc.cfg, scan_kernel, chunk_counts, nchunks, E, chunk_base, counts,
                                               offsets, mtile_start, done);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

cudaError_t launch_mtile_table(const int32_t* offsets, int E, int64_t S, int32_t* mtile_start, uint32_t* status,
                               cudaStream_t s) {
    mtile_table_kernel<<<1, 32, 0, s>>>(offsets, E, S, mtile_start, status);
    return cudaGetLastError();
}

cudaError_t launch_scatter(const bf16* x, const int32_t* ids, const float* w, int64_t T, int d, int E, int k,
                           const int32_t* offsets, const int32_t* chunk_base, const int32_t* rank, bf16* x_perm,
                           int32_t* row_token, float* row_weight, int32_t* slot_row, cudaStream_t s,
                           const TileSems* sem, const int32_t* mtile_start, bool copy_rows) {
    uint32_t* mt_rows = sem != nullptr ? sem->mt_rows : nullptr;
    uint32_t* tok_done = sem != nullptr ? sem->tok_done : nullptr;
    LaunchCfg lc(dim3(static_cast<unsigned>(T)), dim3(128), 0, s, sem != nullptr && sem->pdl);
    const cudaError_t err = cudaLaunchKernelEx(&lc.cfg, scatter_kernel, x, ids, w, T, d, E, k, offsets, chunk_base,
                                               rank, x_perm, row_token, row_weight, slot_row, mt_rows, tok_done,
                                               mtile_start, (sem != nullptr && sem->drop_token0) ? 1 : 0,
                                               copy_rows ? 1 : 0);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace mk
