// route_tc.cu -- the router with a tensor-core candidate filter.
//
// Routing is decided by fp32 gate logits in one fixed order: 32 interleaved
// fused-multiply-add chains s_j over i = j, j + 32, ..., then s_j += s_{j+off}
// for off = 16, 8, 4, 2, 1, then + bias[e] (the same bits as the plain router
// of route.cu and the CPU oracle).  The pages name routing as the layer's first
// step (mKernel README, kernel table, row "MoE Dispatch + FFN + Combine":
// "routes tokens to their expert ranks") and leave its arithmetic open; the
// order is fixed because the logits decide integers.  Computing all T x E of
// them in that order is 2 T d E flops of FP32-ALU work.  Here only the few
// logits that can matter are computed that way:
//
//  1. prep     each gate row is split into two bf16 parts, hi = bf16(w) and
//              mid = bf16(w - hi) (|w - hi - mid| <= 2^-16 |w|), stored
//              interleaved by 64-column blocks [hi_0 mid_0 hi_1 mid_1 ...],
//              and ||w_e||_2 is rounded up.
//  2. approx   A = x [hi|mid]^T + bias on the tensor cores (tcgen05, fp32
//              accumulation in TMEM), in chunks of 16 MMA steps whose sums the
//              epilogue adds in fp32.
//  3. select   per token, a bound B_te >= |A_te - l_te| (below) gives every
//              expert an interval [A - B, A + B] around its fixed-order logit.
//              With L the k-th largest lower end, every expert whose upper end
//              reaches L is a candidate.  An expert outside has k experts whose
//              logits are surely larger, so the exact top-k is among the
//              candidates.  Their fixed-order logits are computed (one warp
//              per logit, lane j runs chain j), then top-k (larger wins, ties
//              to the lower id) and the softmax over the k, as in route.cu.
//              Should an exact logit fall outside its interval (the error
//              model below did not hold), all E logits of that token are
//              computed in the fixed order instead.
//
// The bound, relative to N_te = ||x_t||_2 ||w_e||_2 >= sum_i |x_ti w_ei|:
//   tensor cores: each MMA step (16 products added to the fp32 accumulator)
//     is taken to err by at most eta (|acc| + sum |products|), eta = 2^-18.
//     That covers an accumulation that aligns the 17 addends of a step and
//     truncates each to 24 bits (17 * 2^-23 < 2^-18), with room to spare
//     over round-to-nearest fp32 (about 2^-23 per add); the whole approximate
//     logit was measured within 2^-20.6 N_te (d = 256) to 2^-22.6 N_te
//     (d = 7168), and a GPU test keeps that observed error under 2^-19 N_te.
//     A chunk of n_s = 16 steps then errs by at most (n_s + 2) eta S_chunk;
//   chunk sums in fp32: n_c u S; the bf16 split: 2^-16 S; the fixed-order
//     logit itself: (d/32 + 6) u S; bias adds and rounding of the bound
//     arithmetic: 8 u |A|;  u = 2^-24.
#include <atomic>
#include <math.h>

#include <algorithm>
#include <cmath>

#include "gemm_impl.cuh"

namespace mk {
namespace {

using gemm_detail::make_map;

constexpr int kChunkKb = 4;          // k-blocks of 64 per TMEM chunk (16 MMA steps)
constexpr int kApproxThreads = 320;  // producer, MMA issuer, 8 epilogue warps
constexpr int kSelThreads = 128;     // one token per block, 4 warps
constexpr double kEta = 1.0 / 262144.0;  // 2^-18, see the bound above

template <int N>
struct ApproxCfg {
    static constexpr int STAGES = (N >= 256) ? 4 : 6;
    static constexpr uint32_t A_BYTES = 128 * 64 * 2;
    static constexpr uint32_t B_BYTES = N * 64 * 2;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;  // a multiple of 1024
    static constexpr uint32_t ACC_STRIDE = (N < 64) ? 64 : N;   // TMEM columns per accumulator
    static constexpr uint32_t TMEM_COLS = 2 * ACC_STRIDE;      // 128, 256 or 512
    static constexpr int HALF = N / 2;                          // columns per epilogue thread
    static constexpr uint32_t IDESC = idesc_bf16_f32(128, N);
};

struct ApproxCtl {
    uint64_t full[6];
    uint64_t empty[6];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    uint32_t abort_flag;
    uint32_t zero;
};

template <int N>
constexpr size_t approx_smem() {
    return static_cast<size_t>(ApproxCfg<N>::STAGES) * ApproxCfg<N>::STAGE_BYTES + sizeof(ApproxCtl) + 1024;
}

// ------------------------------------------------------------------ prep

__global__ void __launch_bounds__(256) route_prep_kernel(const float* __restrict__ wg, int d,
                                                         bf16* __restrict__ wsplit, float* __restrict__ wnorm) {
    const int e = blockIdx.x;
    const float* w = wg + static_cast<size_t>(e) * d;
    bf16* o = wsplit + static_cast<size_t>(e) * 2 * d;
    double ss = 0.0;
    for (int i = threadIdx.x; i < d; i += 256) {
        const float v = w[i];
        const bf16 hi = __float2bfloat16_rn(v);
        const bf16 mid = __float2bfloat16_rn(__fsub_rn(v, __bfloat162float(hi)));  // v - hi is exact
        const int b = i >> 6, c = i & 63;
        o[(2 * b) * 64 + c] = hi;
        o[(2 * b + 1) * 64 + c] = mid;
        ss += static_cast<double>(v) * static_cast<double>(v);
    }
    __shared__ double red[8];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        double tot = 0.0;
        for (int i = 0; i < 8; ++i) tot += red[i];
        wnorm[e] = __double2float_ru(sqrt(tot) * (1.0 + 1e-12));
    }
}

// ------------------------------------------------------------------ approx

template <int N>
__global__ void __launch_bounds__(kApproxThreads, 1)
    route_approx_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                        const float* __restrict__ bias, int T, int E, int kb_total, float* __restrict__ approx,
                        uint32_t* status, uint64_t timeout_ns) {
    using C = ApproxCfg<N>;
    extern __shared__ uint8_t smem_raw[];
    pdl_wait();  // as a programmatic dependent: the split gate rows are complete
    pdl_launch_dependents();
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    ApproxCtl* ctl = reinterpret_cast<ApproxCtl*>(smem + C::STAGES * C::STAGE_BYTES);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * 128;
    const int n_chunks = (kb_total + kChunkKb - 1) / kChunkKb;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&ctl->tmem_full[a]), 1);
            mbar_init(smem_u32(&ctl->tmem_empty[a]), 8);
        }
        mbar_init(smem_u32(&ctl->drain), 1);
        ctl->abort_flag = 0;
        ctl->zero = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmX);
        prefetch_tensormap(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    volatile uint32_t* abort_word = &ctl->abort_flag;
    const volatile uint32_t* never = &ctl->zero;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            uint32_t stage = 0, phase = 0, issued = 0, last_par = 0;
            bool ok = true;
            for (int kb = 0; kb < kb_total; ++kb) {
                if (!mbar_wait_bounded(smem_u32(&ctl->empty[stage]), phase ^ 1u, abort_word, timeout_ns)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_u32(&ctl->full[stage]);
                const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
                mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
                tma_load_2d(sa, &tmX, (kb >> 1) * 64, m0, fb);  // x block kb/2 serves its hi and mid blocks
                tma_load_2d(sa + C::A_BYTES, &tmW, kb * 64, 0, fb);
                issued |= 1u << stage;
                last_par = (last_par & ~(1u << stage)) | (phase << stage);
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) {
                *abort_word = 1u;
                report_error(status, MK_ERR_TIMEOUT, kSiteGemmProducer);
            }
            for (int s = 0; s < C::STAGES; ++s)
                if ((issued >> s) & 1u)
                    mbar_wait_bounded(smem_u32(&ctl->full[s]), (last_par >> s) & 1u, never, timeout_ns);
        }
        __syncwarp();
    } else if (warp == 1) {
        {
            // ------------------------------------------------ MMA issuer
            // whole warp, one elected lane issues (see the grouped GEMMs)
            const bool leader = elect_one();
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int c = 0; ok && c < n_chunks; ++c) {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&ctl->tmem_empty[acc]), acc_phase ^ 1u,
                                                              abort_word, timeout_ns))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * C::ACC_STRIDE;
                const int kb0 = c * kChunkKb;
                const int kb1 = min(kb0 + kChunkKb, kb_total);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait_bounded(smem_u32(&ctl->full[stage]), phase, abort_word, timeout_ns))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (leader) {
                        const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
                        const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = sw128_kmajor_desc(sa + kk * 32);
                            const uint64_t bd = sw128_kmajor_desc(sb + kk * 32);
                            mma_bf16_ss(d_tmem, ad, bd, C::IDESC, (kb != kb0 || kk != 0) ? 1u : 0u);
                        }
                        mma_commit(smem_u32(&ctl->empty[stage]));
                    }
                    __syncwarp();
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (leader) mma_commit(smem_u32(&ctl->tmem_full[acc]));
                __syncwarp();
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (leader) {
                if (!ok) {
                    *abort_word = 1u;
                    report_error(status, MK_ERR_TIMEOUT, kSiteGemmMma);
                }
                mma_commit(smem_u32(&ctl->drain));
                if (!mbar_wait_bounded(smem_u32(&ctl->drain), 0u, never, timeout_ns))
                    report_error(status, MK_ERR_TIMEOUT, kSiteGemmDrain);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- epilogue: 8 warps,
        // warp w reads TMEM lanes 32 (w % 4) ..., column half (w - 2) / 4
        const int sub = warp & 3;
        const int hcol = (warp - 2) >> 2;
        const int row = sub * 32 + lane;
        float tot[C::HALF];
#pragma unroll
        for (int j = 0; j < C::HALF; ++j) tot[j] = 0.0f;
        uint32_t acc = 0, acc_phase = 0;
        bool ok = true;
        for (int c = 0; c < n_chunks; ++c) {
            if (!mbar_wait_bounded(smem_u32(&ctl->tmem_full[acc]), acc_phase, abort_word, timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) + acc * C::ACC_STRIDE +
                                   static_cast<uint32_t>(hcol * C::HALF);
#pragma unroll
            for (int q = 0; q < (C::HALF + 31) / 32; ++q) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(taddr + 32 * q, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (32 * q + j < C::HALF) tot[32 * q + j] = __fadd_rn(tot[32 * q + j], __uint_as_float(v[j]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->tmem_empty[acc]));
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (!ok) {
            if (lane == 0) {
                *abort_word = 1u;
                report_error(status, MK_ERR_TIMEOUT, kSiteGemmEpilogue);
            }
        } else if (m0 + row < T) {
            float* orow = approx + static_cast<size_t>(m0 + row) * E;
#pragma unroll
            for (int j = 0; j < C::HALF; ++j) {
                const int e = hcol * C::HALF + j;
                if (e < E) orow[e] = bias != nullptr ? __fadd_rn(tot[j], __ldg(bias + e)) : tot[j];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ select

// Fixed-order logits of two expert rows (w1 may be null) for the token row
// staged in shared memory: lane j runs chain j of each (x[j + 32 m] * w[j + 32 m],
// fused multiply-add in increasing m), then the 5-level tree.  16 loads of
// each row are in flight per lane.  Every lane of the warp calls; lane 0 holds
// the results.
__device__ __forceinline__ float2 fixed_order_logits2(const uint16_t* xs, const float* __restrict__ w0,
                                                      const float* __restrict__ w1, int d, int lane) {
    constexpr int U = 16;
    const int nf = d >> 5;
    const bool two = w1 != nullptr;
    const float* w1s = two ? w1 : w0;
    float s0 = 0.0f, s1 = 0.0f;
    int m = 0;
    for (; m + U <= nf; m += U) {
        float a[U], b[U];
#pragma unroll
        for (int u = 0; u < U; ++u) a[u] = __ldg(w0 + lane + 32 * (m + u));
        if (two) {
#pragma unroll
            for (int u = 0; u < U; ++u) b[u] = __ldg(w1s + lane + 32 * (m + u));
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float xv = __uint_as_float(static_cast<uint32_t>(xs[lane + 32 * (m + u)]) << 16);
            s0 = __fmaf_rn(xv, a[u], s0);
            if (two) s1 = __fmaf_rn(xv, b[u], s1);
        }
    }
    for (; m < nf; ++m) {
        const float xv = __uint_as_float(static_cast<uint32_t>(xs[lane + 32 * m]) << 16);
        s0 = __fmaf_rn(xv, __ldg(w0 + lane + 32 * m), s0);
        if (two) s1 = __fmaf_rn(xv, __ldg(w1s + lane + 32 * m), s1);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const float o0 = __shfl_down_sync(0xffffffffu, s0, off);
        const float o1 = __shfl_down_sync(0xffffffffu, s1, off);
        if (lane < off) {
            s0 = __fadd_rn(s0, o0);
            s1 = __fadd_rn(s1, o1);
        }
    }
    return make_float2(s0, s1);
}

__global__ void __launch_bounds__(kSelThreads) route_select_kernel(
    const bf16* __restrict__ x, const float* __restrict__ wg, const float* __restrict__ bias,
    const float* __restrict__ approx, const float* __restrict__ wnorm, int d, int E, int k, float c_rel,
    float c_abs, int32_t* __restrict__ ids, float* __restrict__ wout, int32_t* __restrict__ counts,
    uint32_t* __restrict__ fallbacks) {
    extern __shared__ __align__(16) uint8_t sel_smem[];
    uint16_t* xs = reinterpret_cast<uint16_t*>(sel_smem);                // token row, bf16 bits [d]
    int32_t* cand = reinterpret_cast<int32_t*>(sel_smem + 2 * d);        // candidate ids [E]
    float* cval = reinterpret_cast<float*>(cand + E);                    // their fixed-order logits
    __shared__ float red[kSelThreads / 32];
    __shared__ float s_nx;
    __shared__ int s_ncand;
    __shared__ int s_violated;
    pdl_wait();  // as a programmatic dependent: the approximate logits are complete
    pdl_launch_dependents();
    const int64_t t = blockIdx.x;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr int kNone = 0x7fffffff;

    // token row -> shared memory, and its squared norm
    const uint4* src = reinterpret_cast<const uint4*>(x + t * d);
    float ss = 0.0f;
    for (int i = threadIdx.x; i < d / 8; i += kSelThreads) {
        const uint4 v = __ldg(src + i);
        reinterpret_cast<uint4*>(xs)[i] = v;
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float lo = __uint_as_float(wv[q] << 16);
            const float hi = __uint_as_float(wv[q] & 0xffff0000u);
            ss = __fmaf_rn(lo, lo, ss);
            ss = __fmaf_rn(hi, hi, ss);
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
    if (lane == 0) red[warp] = ss;
    if (threadIdx.x == 0) s_violated = 0;
    __syncthreads();

    const float* arow = approx + t * E;
    if (warp == 0) {
        float tot = 0.0f;
#pragma unroll
        for (int i = 0; i < kSelThreads / 32; ++i) tot = __fadd_rn(tot, red[i]);
        // a sum of d squares in fp32 is within (d + 1) u of the true sum
        const float nx = sqrtf(tot * (1.0f + static_cast<float>(d + 8) * 0x1p-23f)) * (1.0f + 0x1p-20f);
        float lo[kMaxExperts / 32], up[kMaxExperts / 32];
#pragma unroll
        for (int q = 0; q < kMaxExperts / 32; ++q) {
            const int e = lane + 32 * q;
            lo[q] = up[q] = 0.0f;
            if (e < E) {
                const float a = __ldg(arow + e);
                const float b = c_rel * nx * __ldg(wnorm + e) + c_abs * fabsf(a);
                lo[q] = a - b;
                up[q] = a + b;
            }
        }
        // L: the k-th largest lower end
        uint32_t taken = 0;
        float L = 0.0f;
        for (int j = 0; j < k; ++j) {
            float bv = 0.0f;
            int bi = kNone;
#pragma unroll
            for (int q = 0; q < kMaxExperts / 32; ++q) {
                const int e = lane + 32 * q;
                if (e < E && !((taken >> q) & 1u) && (bi == kNone || lo[q] > bv)) {
                    bv = lo[q];
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
            L = bv;
            if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        }
        // candidates: upper end >= L, compacted in expert order
        int base = 0;
#pragma unroll
        for (int q = 0; q < kMaxExperts / 32; ++q) {
            const int e = lane + 32 * q;
            const bool is_c = e < E && up[q] >= L;
            const uint32_t bal = __ballot_sync(0xffffffffu, is_c);
            if (is_c) cand[base + __popc(bal & ((1u << lane) - 1u))] = e;
            base += __popc(bal);
        }
        if (lane == 0) {
            s_ncand = base;
            s_nx = nx;
        }
    }
    __syncthreads();

    // fixed-order logits of the candidates, one warp per candidate
    const int ncand = s_ncand;
    const float nx = s_nx;
    constexpr int kW = kSelThreads / 32;
    for (int c = 2 * warp; c < ncand; c += 2 * kW) {  // two candidates per warp at a time
        const int e0 = cand[c];
        const int e1 = (c + 1 < ncand) ? cand[c + 1] : -1;
        const float2 l2 = fixed_order_logits2(xs, wg + static_cast<size_t>(e0) * d,
                                              e1 >= 0 ? wg + static_cast<size_t>(e1) * d : nullptr, d, lane);
        if (lane == 0) {
            for (int q = 0; q < 2; ++q) {
                const int e = q ? e1 : e0;
                if (e < 0) break;
                float l = q ? l2.y : l2.x;
                if (bias != nullptr) l = __fadd_rn(l, __ldg(bias + e));
                cval[c + q] = l;
                const float a = __ldg(arow + e);
                const float b = c_rel * nx * __ldg(wnorm + e) + c_abs * fabsf(a);
                if (!(fabsf(l - a) <= b)) s_violated = 1;
            }
        }
    }
    __syncthreads();
    int nlist = ncand;
    if (s_violated) {  // the error model did not hold for this token: all E logits exactly
        if (threadIdx.x == 0 && fallbacks != nullptr) atomicAdd(fallbacks, 1u);
        for (int e = 2 * warp; e < E; e += 2 * kW) {
            const bool has1 = e + 1 < E;
            const float2 l2 = fixed_order_logits2(xs, wg + static_cast<size_t>(e) * d,
                                                  has1 ? wg + static_cast<size_t>(e + 1) * d : nullptr, d, lane);
            if (lane == 0) {
                for (int q = 0; q < (has1 ? 2 : 1); ++q) {
                    float l = q ? l2.y : l2.x;
                    if (bias != nullptr) l = __fadd_rn(l, __ldg(bias + e + q));
                    cand[e + q] = e + q;
                    cval[e + q] = l;
                }
            }
        }
        nlist = E;
        __syncthreads();
    }

    // top-k of the list (larger logit wins, ties to the lower id), softmax over the k
    if (warp == 0) {
        float sel_v[kMaxTopK];
        int sel_i[kMaxTopK];
        for (int j = 0; j < k; ++j) {
            float bv = 0.0f;
            int bi = kNone;
            for (int c = lane; c < nlist; c += 32) {
                const int e = cand[c];
                const float v = cval[c];
                bool used = false;
                for (int jj = 0; jj < j; ++jj) used |= (sel_i[jj] == e);
                if (!used && (bi == kNone || v > bv || (v == bv && e < bi))) {
                    bv = v;
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
        }
        if (lane == 0) {
            float ex[kMaxTopK];
            float z = 0.0f;
            for (int j = 0; j < k; ++j) {
                ex[j] = expf(sel_v[j] - sel_v[0]);
                z += ex[j];
            }
            for (int j = 0; j < k; ++j) {
                ids[t * k + j] = sel_i[j];
                wout[t * k + j] = ex[j] / z;
                if (counts != nullptr) atomicAdd(counts + sel_i[j], 1);
            }
        }
    }
}

template <int N>
cudaError_t launch_approx_n(const CUtensorMap& mx, const CUtensorMap& mw, const float* bias, int64_t T, int E,
                            int kb_total, float* approx, uint32_t* status, uint64_t timeout_ns, cudaStream_t s,
                            bool pdl) {
    static std::atomic<int> configured[64];  // per device: attributes set (repeating them is harmless)
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    auto fn = route_approx_kernel<N>;
    if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
        err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(approx_smem<N>()));
        if (err != cudaSuccess) return err;
        if (dev < 64) configured[dev].store(1, std::memory_order_release);
    }
    const unsigned grid = static_cast<unsigned>((T + 127) / 128);
    LaunchCfg lc(dim3(grid), dim3(kApproxThreads), approx_smem<N>(), s, pdl);
    err = cudaLaunchKernelEx(&lc.cfg, fn, mx, mw, bias, static_cast<int>(T), E, kb_total, approx, status, timeout_ns);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace

size_t route_select_smem(int d, int E) { return static_cast<size_t>(2) * d + static_cast<size_t>(8) * E; }

bool route_tc_supported(int d, int E) { return route_select_smem(d, E) <= 160 * 1024 && E <= kMaxExperts; }

cudaError_t launch_route_approx(const bf16* x, const float* wg, const float* bias, int64_t T, int d, int E,
                                float* approx, bf16* wsplit, float* wnorm, uint32_t* status, uint64_t timeout_ns,
                                cudaStream_t s, bool pdl) {
    route_prep_kernel<<<E, 256, 0, s>>>(wg, d, wsplit, wnorm);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const int N = E <= 16 ? 16 : E <= 32 ? 32 : E <= 64 ? 64 : E <= 128 ? 128 : 256;
    CUtensorMap mx, mw;
    if (!make_map(&mx, x, d, static_cast<uint64_t>(T), 128) ||
        !make_map(&mw, wsplit, static_cast<uint64_t>(2) * d, static_cast<uint64_t>(E), static_cast<uint32_t>(N)))
        return cudaErrorInvalidValue;
    const int kb_total = d / 32;  // 2d / 64
    switch (N) {
        case 16: return launch_approx_n<16>(mx, mw, bias, T, E, kb_total, approx, status, timeout_ns, s, pdl);
        case 32: return launch_approx_n<32>(mx, mw, bias, T, E, kb_total, approx, status, timeout_ns, s, pdl);
        case 64: return launch_approx_n<64>(mx, mw, bias, T, E, kb_total, approx, status, timeout_ns, s, pdl);
        case 128: return launch_approx_n<128>(mx, mw, bias, T, E, kb_total, approx, status, timeout_ns, s, pdl);
        default: return launch_approx_n<256>(mx, mw, bias, T, E, kb_total, approx, status, timeout_ns, s, pdl);
    }
}

cudaError_t launch_route_select(const bf16* x, const float* wg, const float* bias, int64_t T, int d, int E, int k,
                                const float* approx, const float* wnorm, int32_t* ids, float* w, int32_t* counts,
                                uint32_t* fallbacks, bool zero_bound, cudaStream_t s, bool pdl) {
    // bound coefficients (see the top of this file), rounded up
    const double u = 1.0 / 16777216.0;
    const int kb_total = d / 32;
    const int n_chunks = (kb_total + kChunkKb - 1) / kChunkKb;
    const double c_rel =
        (kEta * (4 * kChunkKb + 2) + (n_chunks + d / 32 + 6) * u + 1.0 / 65536.0) * (1.0 + 1.0 / 1024);
    const double c_abs = 8 * u;
    const float c_rel_f = zero_bound ? 0.0f : std::nextafter(static_cast<float>(c_rel), INFINITY);
    const float c_abs_f = zero_bound ? 0.0f : std::nextafter(static_cast<float>(c_abs), INFINITY);
    const size_t smem = route_select_smem(d, E);
    static std::atomic<int> configured[64];  // per device: attributes set (repeating them is harmless)
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (smem > 48 * 1024 && (dev >= 64 || !configured[dev].load(std::memory_order_acquire))) {
        err = cudaFuncSetAttribute(route_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(160 * 1024));
        if (err != cudaSuccess) return err;
        if (dev < 64) configured[dev].store(1, std::memory_order_release);
    }
    LaunchCfg lc(dim3(static_cast<unsigned>(T)), dim3(kSelThreads), smem, s, pdl);
    err = cudaLaunchKernelEx(&lc.cfg, route_select_kernel, x, wg, bias, approx, wnorm, d, E, k, c_rel_f, c_abs_f, ids,
                             w, counts, fallbacks);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace mk
