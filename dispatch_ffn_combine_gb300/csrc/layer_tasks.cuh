// layer_tasks.cuh -- per-task device bodies of the layer's data-movement
// steps, run by one block of 256 threads: top-k of a token, per-chunk expert
// histogram and ranks, the scans over chunks and experts, the dispatch of a
// token chunk (row maps and row copies), and the combine of a token range.  The
// fused persistent kernel strings them together with ready flags; the
// stand-alone kernels of the unfused path have their own bodies.
#pragma once

#include <math.h>

#include "mk_device.cuh"
#include "mk_internal.h"

namespace mk {
namespace tasks {

constexpr int kThreads = 256;

// Top-k of one token by one warp: k rounds of a warp-wide arg-max (larger
// logit wins, equal logits go to the lower expert id), then the softmax over
// the chosen k in fp32.
__device__ __forceinline__ void topk_token(const float* __restrict__ logits, int64_t t, int E, int k,
                                           int32_t* __restrict__ ids, float* __restrict__ w) {
    const int lane = threadIdx.x & 31;
    constexpr int kNone = 0x7fffffff;
    float v[kMaxExperts / 32];
#pragma unroll
    for (int q = 0; q < kMaxExperts / 32; ++q) {
        const int e = lane + 32 * q;
        v[q] = (e < E) ? logits[t * E + e] : 0.0f;
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
        }
    }
}

// Expert histogram of one 128-token chunk and each (token, slot)'s rank among
// the chunk's rows of its expert (ascending token order).  `mask` is
// kMaxExperts * 4 words of shared memory.  All threads of the block call.
__device__ __forceinline__ void count_chunk(uint32_t* mask, const int32_t* __restrict__ ids, int64_t T, int E,
                                            int k, int64_t c, int32_t* __restrict__ chunk_counts,
                                            int32_t* __restrict__ rank) {
    const int64_t t_begin = c * kChunkTokens;
    const int nt = static_cast<int>((T - t_begin < kChunkTokens) ? (T - t_begin) : kChunkTokens);
    for (int i = threadIdx.x; i < E * (kChunkTokens / 32); i += kThreads) mask[i] = 0u;
    __syncthreads();
    for (int q = threadIdx.x; q < nt * k; q += kThreads) {
        const int tl = q / k;
        const int e = ids[t_begin * k + q];
        atomicOr(&mask[e * 4 + (tl >> 5)], 1u << (tl & 31));
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kThreads)
        chunk_counts[c * E + e] =
            __popc(mask[e * 4]) + __popc(mask[e * 4 + 1]) + __popc(mask[e * 4 + 2]) + __popc(mask[e * 4 + 3]);
    for (int q = threadIdx.x; q < nt * k; q += kThreads) {
        const int tl = q / k;
        const int e = ids[t_begin * k + q];
        const int wd = tl >> 5;
        int r = 0;
        for (int ww = 0; ww < wd; ++ww) r += __popc(mask[e * 4 + ww]);
        r += __popc(mask[e * 4 + wd] & ((1u << (tl & 31)) - 1u));
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

// Scans after the last chunk is counted: per expert over chunks (chunk bases),
// then over experts (offsets) and over per-expert 128-row tile counts.
// `s_counts` is kMaxExperts words of shared memory.  All threads call.
__device__ __forceinline__ void scan_all(int32_t* s_counts, const int32_t* __restrict__ chunk_counts, int64_t nchunks,
                                         int E, int32_t* __restrict__ chunk_base, int32_t* __restrict__ counts,
                                         int32_t* __restrict__ offsets, int32_t* __restrict__ mtile_start) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    for (int e = warp; e < E; e += kThreads / 32) {
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
    if (warp == 0) {
        int cnt[8], til[8], sum_c = 0, sum_t = 0;
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
}

// Dispatch of tokens [t_begin, t_begin + nt), all inside counting chunk c:
// the row of every (token, slot), the row -> token / weight maps, and the
// token rows copied into their k expert rows.  A warp per token reads the row
// once (8 independent 16-byte loads in flight per lane) and writes it k times.
__device__ __forceinline__ void dispatch_tokens(const int32_t* __restrict__ ids, const float* __restrict__ w, int d,
                                                int E, int k, int64_t c, int64_t t_begin, int nt,
                                                const int32_t* __restrict__ offsets,
                                                const int32_t* __restrict__ chunk_base,
                                                const int32_t* __restrict__ rank, const bf16* __restrict__ x,
                                                bf16* __restrict__ x_perm, int32_t* __restrict__ row_token,
                                                float* __restrict__ row_weight, int32_t* __restrict__ slot_row) {
    constexpr int U = 8;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n16 = d / 8;
    for (int tt = warp; tt < nt; tt += kThreads / 32) {
        const int64_t t = t_begin + tt;
        int64_t r_lane = 0;
        if (lane < k) {
            const int64_t tq = t * k + lane;
            const int e = ids[tq];
            r_lane = static_cast<int64_t>(offsets[e]) + chunk_base[c * E + e] + rank[tq];
            slot_row[tq] = static_cast<int32_t>(r_lane);
            row_token[r_lane] = static_cast<int32_t>(t);
            row_weight[r_lane] = w[tq];
        }
        int64_t rows[kMaxTopK];
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) rows[j] = __shfl_sync(0xffffffffu, r_lane, j);
        const uint4* src = reinterpret_cast<const uint4*>(x + t * d);
        for (int c0 = lane; c0 < n16; c0 += 32 * U) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (c0 + 32 * u < n16) v[u] = __ldg(src + c0 + 32 * u);
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j) {
                if (j < k) {
                    uint4* dst = reinterpret_cast<uint4*>(x_perm + rows[j] * d);
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        if (c0 + 32 * u < n16) dst[c0 + 32 * u] = v[u];
                }
            }
        }
    }
}

// y[t] = bf16( sum_j P[slot_row[t, j]] ), j ascending, fp32 sum, for tokens
// [t0, t0 + nt).  A warp per token; each lane loads its 16-byte piece of all
// k rows before adding them in slot order.  P is written earlier in the same
// launch by other blocks, so it is read from L2 (ld.global.cg), never through
// the non-coherent read-only path.
__device__ __forceinline__ void combine_tokens(const bf16* __restrict__ P, const int32_t* __restrict__ slot_row,
                                               int64_t t0, int nt, int d, int k, bf16* __restrict__ y) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n16 = d / 8;
    for (int tt = warp; tt < nt; tt += kThreads / 32) {
        const int64_t t = t0 + tt;
        int64_t rows[kMaxTopK];
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) rows[j] = (j < k) ? static_cast<int64_t>(slot_row[t * k + j]) : 0;
        for (int cc = lane; cc < n16; cc += 32) {
            uint4 v[kMaxTopK];
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j)
                if (j < k) v[j] = __ldcg(reinterpret_cast<const uint4*>(P + rows[j] * d) + cc);
            float acc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j) {
                if (j < k) {
                    const uint32_t wv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc[2 * q] = __fadd_rn(acc[2 * q], __uint_as_float(wv[q] << 16));
                        acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], __uint_as_float(wv[q] & 0xffff0000u));
                    }
                }
            }
            uint4 o;
            o.x = pack_bf16x2(acc[0], acc[1]);
            o.y = pack_bf16x2(acc[2], acc[3]);
            o.z = pack_bf16x2(acc[4], acc[5]);
            o.w = pack_bf16x2(acc[6], acc[7]);
            reinterpret_cast<uint4*>(y + t * d)[cc] = o;
        }
    }
}

}  // namespace tasks
}  // namespace mk
