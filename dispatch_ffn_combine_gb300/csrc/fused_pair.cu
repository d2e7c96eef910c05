// fused_pair.cu -- the whole MoE layer as one persistent kernel on CTA pairs,
// whose clusters take data-movement ("mover") or compute roles.
//
// The design follows the mKernel paper ("mKernel: Fast Multi-GPU, Multi-Node
// Fused Kernels"): a persistent kernel whose blocks are assigned roles (§3,
// Fig. 2), an on-GPU controller that sets the number of communication blocks
// to n* = B * Rs*Cs / (Rp*Cp + Rs*Cs) from the remaining tasks R and their
// measured per-task cycles C (§3.2, Eq. 2), blocks that re-check their role
// between tasks, compute blocks that help communication while their input is
// not ready (§3.2), per-chunk counters whose last finisher publishes readiness
// (§3.1), and readiness flags per tile (§4).  On one GPU the expert-parallel
// exchanges of the README's "MoE Dispatch + FFN + Combine" row become HBM
// copies, so the mover role runs the router, the dispatch and the combine.
//
// GB300 layout: the kernel is launched as clusters of two CTAs on two SMs, as
// many clusters as fit on the GPU at once (all co-resident).  A
// cluster takes one role at a time, decided by CTA 0's first thread and sent
// to CTA 1 through distributed shared memory:
//   mover    each CTA runs its own mover task (two tickets per decision):
//              route blocks (32 tokens x 32 experts of gate logits; the last
//              block of a token group runs its top-k, the last top-k of a
//              128-token chunk its expert histogram, the last chunk the scans)
//              -> dispatch tasks (128 tokens, or 32 in small layers)
//              -> the combine (each CTA claims tokens a few at a time and
//                 stages every token's k rows in shared memory with TMA bulk
//                 copies)
//   compute  a GEMM session of CTA-pair tiles, the grouped GEMM kernel's
//            (gemm_pair.cu) roles: warp 0 of each CTA loads its halves with
//            TMA (cta_group::2, both CTAs' copies completing on CTA 0's
//            barrier), warp 1 of CTA 0 issues tcgen05.mma.cta_group::2
//            (M = 256, N = 256) into both CTAs' TMEM, warps 2-5 of each CTA
//            run the fused epilogue, warp 6 of CTA 0 claims tiles and writes
//            them into both CTAs' slot rings (warp 6 of CTA 1 relays CTA 1's
//            slot releases); 256 x 256 tiles, an expert's partial last block as
//            a swap tile; gemm1 tiles (pair block x 128 h columns) then gemm2
//            tiles (pair block x 256 output columns), claimed one ticket at a
//            time in the stand-alone kernels' grouped order.
// Readiness (bounded waits, every one):
//   dispatch tasks need the scans;
//   gemm1 tiles are claimable once every dispatch task has been claimed (so
//     every row is being written by a running block), and each tile starts as
//     soon as the rows of its own pair block have landed: the dispatch tasks
//     publish every row they write on its 128-row M-tile's counter;
//   gemm2 tile (pair block b, N block n) needs every gemm1 tile of b: each of
//     the 8 epilogue warps of a gemm1 tile publishes once on b's counter;
//   combine tasks need every gemm2 tile.
// A cluster claims only tasks whose inputs are being produced by running
// blocks, so claiming in order never deadlocks; every wait is bounded by
// %globaltimer and an abort word.
#include <algorithm>
#include <atomic>

#include "gemm_impl.cuh"
#include "layer_tasks.cuh"
#include "route_impl.cuh"

namespace mk {
namespace {

using namespace gemm_detail;

constexpr int kThreads = 256;
constexpr int FSTAGES = 7;                              // 7 x 32 KB operand stages
constexpr uint32_t PA_BYTES = BM * BK * 2;              // this CTA's 128 A rows, one k-block
constexpr uint32_t PB_BYTES = (MMA_N / 2) * BK * 2;     // this CTA's 128 of the 256 B rows
constexpr uint32_t PSTAGE_BYTES = PA_BYTES + PB_BYTES;  // 32 KB
constexpr uint32_t PTX_BYTES = 2 * PSTAGE_BYTES;        // both CTAs' copies of one stage
constexpr uint32_t PIDESC = idesc_bf16_f32(PAIR_M, MMA_N);
constexpr int kPairNGroup = 4;
constexpr int kSlots = 3;
// Readers of a tile slot that release it on their own CTA's `slot_empty`: CTA 0
// its producer, MMA and 4 epilogue warps, plus CTA 1's relay (one arrive for
// CTA 1's producer and 4 epilogue warps).
constexpr uint32_t kSlotConsumers0 = 7;
constexpr uint32_t kSlotConsumers1 = 5;
constexpr int kSchedWarp = 6;  // GEMM sessions: tile scheduler (CTA 0) / slot-release relay (CTA 1)
constexpr uint32_t kEpiPacePerKb = 80;  // gemm2's epilogue chunk spacing per k-block, as in gemm_pair.cu
constexpr int kEpiPaceMaxKb = 64;       // ... for K below this many k-blocks only
constexpr int kCombineBufs = 8;   // tokens whose rows are in flight per CTA in the combine (at most)
constexpr int kCombineClaim = 8;  // tokens per claim of the combine counter
constexpr int kCombineUnit = 32;  // tokens counted as one combine task by the controller
constexpr int kDispatchTokensSmall = 32;
static_assert(kChunkTokens % kDispatchTokensSmall == 0, "a dispatch task stays inside one counting chunk");

enum : int { kRoleMover = 0, kRoleCompute = 1 };
enum : int { kActExit = 0, kActIdle = 1, kActRoute = 2, kActIndex = 3, kActCombine = 5, kActGemm = 6 };

// Pipeline positions that persist across GEMM sessions (each role keeps its
// own fields here, not in registers the mover tasks need).
struct PipeState {
    uint32_t pr_stage, pr_phase, pr_slot, pr_slot_phase, pr_issued, pr_last_par;
    uint32_t mm_stage, mm_phase, mm_acc, mm_acc_phase, mm_slot, mm_slot_phase;
    uint32_t ep_acc, ep_acc_phase, ep_slot, ep_slot_phase;
    uint32_t sc_slot, sc_slot_phase;
    int role;
    int pad;
    unsigned long long last_progress;
    long long t_start;
    unsigned long long g_start;
};

struct FCtl {
    uint64_t full[FSTAGES];   // CTA 0: both CTAs' copies of the stage landed
    uint64_t empty[FSTAGES];  // each CTA: the pair MMAs that read the stage are done
    uint64_t tmem_full[2];    // each CTA: accumulator complete
    uint64_t tmem_empty[2];   // CTA 0: all 8 epilogue warps have read the accumulator
    uint64_t drain;           // CTA 0: every MMA issued has completed
    uint64_t slot_full[kSlots];
    uint64_t slot_empty[kSlots];
    int4 slot[kSlots];   // {e | mode << 16 (-1: end of session), row0, rows, n0}
    int4 slot2[kSlots];  // {pair block index, first M-tile index, more tiles follow, 0}
    PipeState ps;
    int32_t pstart[kMaxExperts + 1];  // CTA 0, per session: prefix over experts of their pair blocks
    uint32_t tmem_base;
    uint32_t abort_local;
    uint32_t zero;
    int action, arg0, arg1, flag;  // the cluster's decision (written into both CTAs by CTA 0)
    int pair_blocks;               // CTA 0: pair blocks of the layer (-1 until the scans are known)
    uint64_t cbar[kCombineBufs];   // combine: the k rows of a token have landed in buffer i
    int ctoken[kCombineBufs];      // combine: the token in buffer i (-1: none)
    uint32_t cphase;               // combine: completed-phase parity of each buffer's barrier
};

constexpr size_t kUnionBytes = static_cast<size_t>(FSTAGES) * PSTAGE_BYTES;
constexpr size_t kFusedSmem = kUnionBytes + sizeof(FCtl) + 1024;
static_assert(kFusedSmem <= 227u * 1024u, "fused kernel shared memory exceeds the per-CTA limit");

struct FPParams {
    const bf16* x;
    const float* wg;
    const float* bias;
    int T, d, E, k, f;
    float* logits;
    int32_t* ids;
    float* w;
    int32_t* chunk_counts;
    int32_t* chunk_base;
    int32_t* rank;
    int32_t* counts;
    int32_t* offsets;
    int32_t* mtile_start;
    int32_t* row_token;
    float* row_weight;
    int32_t* slot_row;
    bf16* x_perm;
    bf16* h;
    bf16* P;
    bf16* y;
    uint32_t* status;
    FusedSync* sync;
    uint32_t* route_done;  // [n_tg]
    uint32_t* topk_done;   // [nchunks]
    uint32_t* mt_rows;     // [M-tiles] rows landed
    uint32_t* h_done;      // [pair blocks] gemm1 epilogue warps done
    int n_tg, n_eg, ct, nchunks;
    int NR, ND, NK;  // route, dispatch and combine tasks
    int dtok;        // tokens per dispatch task
    int routed;      // 1: ids, weights, chunk counts, ranks and scans were computed before the launch
    int NT1, NT2;    // N tiles per pair block: gemm1 (128 h columns), gemm2 (256 output columns)
    int kb1, kb2;    // k-blocks
    int swap1, swap2;  // pair blocks with at most this many rows run as swap tiles
    int mover_ctas;    // 0 adaptive; > 0 blocks [0, n) prefer mover tasks; < 0 no block prefers them
    uint64_t timeout_ns;
    uint32_t* trace;
    int trace_cap;
};

struct FMaps {
    CUtensorMap a1, a1_16, a1_32, a1_64;  // x_perm rows in boxes of 128 / 16 / 32 / 64
    CUtensorMap w1, w3, w1q, w3q;         // gate / up weights, 128- and 16-row boxes
    CUtensorMap a2, a2_16, a2_32, a2_64;  // h rows
    CUtensorMap w2;                       // down weights, 128-row boxes
};

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long ld_relaxed64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void nanosleep_ns(uint32_t ns) { asm volatile("nanosleep.u32 %0;" ::"r"(ns)); }

__device__ __forceinline__ bool scans_ready(const FPParams& p) {
    return p.routed != 0 || ld_acquire_gpu(&p.sync->scan_done) != 0u;
}

// Pair blocks of the layer once the scans are known (an expert with t 128-row
// tiles has ceil(t / 2)); CTA 0's thread 0 computes it once and keeps it.
__device__ int pair_blocks(const FPParams& p, FCtl* ctl) {
    if (ctl->pair_blocks >= 0) return ctl->pair_blocks;
    int n = 0;
    for (int e = 0; e < p.E; ++e) n += (p.mtile_start[e + 1] - p.mtile_start[e] + 1) / 2;
    ctl->pair_blocks = n;
    return n;
}

struct Claim {
    int kind;
    int a0;
    int a1;
};

// ------------------------------------------------------------------ claiming
// Run by CTA 0's thread 0 for the cluster.  The mover queue is three ranges,
// route -> dispatch -> combine, each with its own head; all tasks of a range
// become ready at once, so the cluster claims two tickets of a range (one per
// CTA) with one fetch-add only after seeing it ready.

__device__ Claim claim_two(uint32_t* head, int n, int kind) {
    if (ld_relaxed(head) >= static_cast<uint32_t>(n)) return {kActIdle, -1, -1};
    const uint32_t h = atomicAdd(head, 2u);
    if (h >= static_cast<uint32_t>(n)) return {kActIdle, -1, -1};
    __threadfence();
    return {kind, static_cast<int>(h), h + 1 < static_cast<uint32_t>(n) ? static_cast<int>(h + 1) : -1};
}

__device__ Claim try_claim_mover(const FPParams& p, FCtl* ctl) {
    FusedSync* s = p.sync;
    Claim c = claim_two(&s->route_head, p.NR, kActRoute);
    if (c.kind != kActIdle) return c;
    if (!scans_ready(p)) return {kActIdle, -1, -1};
    c = claim_two(&s->index_head, p.ND, kActIndex);
    if (c.kind != kActIdle) return c;
    // the combine: both CTAs run the combine loop, which claims tokens itself
    if (ld_relaxed(&s->comb_head) >= static_cast<uint32_t>(p.T)) return {kActExit, -1, -1};
    const uint32_t want = 8u * static_cast<uint32_t>(pair_blocks(p, ctl) * p.NT2);
    if (ld_acquire_gpu(&s->p_done) != want) return {kActIdle, -1, -1};
    return {kActCombine, 0, 0};
}

// gemm1 tiles become claimable once every dispatch task has been claimed: the
// rows of every tile are then being written by running blocks, and a tile
// waits (bounded) only for its own pair block's rows.  gemm2 tiles wait for
// their pair block's gemm1 tiles, all claimed before any gemm2 tile by running
// clusters.  Neither wait can deadlock.
__device__ Claim try_claim_compute(const FPParams& p, FCtl* ctl) {
    FusedSync* s = p.sync;
    if (!scans_ready(p)) return {kActIdle, -1, -1};
    if (ld_acquire_gpu(&s->index_head) < static_cast<uint32_t>(p.ND)) return {kActIdle, -1, -1};
    const uint32_t total = static_cast<uint32_t>(pair_blocks(p, ctl) * (p.NT1 + p.NT2));
    if (ld_relaxed(&s->compute_head) >= total) return {kActExit, -1, -1};
    const uint32_t h = atomicAdd(&s->compute_head, 1u);
    if (h >= total) return {kActExit, -1, -1};
    return {kActGemm, static_cast<int>(h), -1};
}

// Eq. 2 of the paper, in blocks: the mover-block target that equalises the
// predicted finishing times of the two roles.  Before the scans the compute
// queue is empty and its size unknown, so every block is a mover.
__device__ int controller_target(const FPParams& p, FCtl* ctl) {
    FusedSync* s = p.sync;
    const int B = static_cast<int>(gridDim.x);
    if (!scans_ready(p)) return B;
    const double mover_total = static_cast<double>(p.NR) + p.ND + p.NK;
    const double compute_total = static_cast<double>(pair_blocks(p, ctl)) * (p.NT1 + p.NT2);
    const uint32_t claimed = min(ld_relaxed(&s->route_head), static_cast<uint32_t>(p.NR)) +
                             min(ld_relaxed(&s->index_head), static_cast<uint32_t>(p.ND)) +
                             min(ld_relaxed(&s->comb_head) / kCombineUnit, static_cast<uint32_t>(p.NK));
    const double Rs = fmax(0.0, mover_total - static_cast<double>(claimed));
    const double Rp = fmax(0.0, compute_total - static_cast<double>(ld_relaxed(&s->compute_head)));
    const unsigned long long cs = ld_relaxed64(&s->cyc[0]), cp = ld_relaxed64(&s->cyc[1]);
    const uint32_t ns = ld_relaxed(&s->ntask[0]), np = ld_relaxed(&s->ntask[1]);
    const double Cs = ns ? static_cast<double>(cs) / ns : 1.0;
    const double Cp = np ? static_cast<double>(cp) / np : Cs;
    const double den = Rp * Cp + Rs * Cs;
    if (den <= 0.0) return 0;
    int n = static_cast<int>(B * (Rs * Cs) / den + 0.5);
    return n < 0 ? 0 : (n > B ? B : n);
}

// The cluster's next task.  Its role (adaptive mode) moves toward the
// controller's target, two blocks at a time; the preferred queue is tried
// first, the other one when nothing preferred is ready (a stalled cluster
// helps the other role); with nothing ready anywhere the thread backs off and
// retries, up to the timeout.
__device__ Claim decide(const FPParams& p, FCtl* ctl, int& role, unsigned long long& last_progress) {
    FusedSync* s = p.sync;
    uint32_t backoff = 64;
    for (;;) {
        if (ld_relaxed(&s->abort_flag) != 0u) return {kActExit, -1, -1};
        if (p.mover_ctas == 0) {
            const int target = static_cast<int>(ld_relaxed(&s->target_movers));
            const uint32_t cur = ld_relaxed(&s->movers_active);
            if (role == kRoleCompute && static_cast<int>(cur) + 1 < target) {
                if (atomicCAS(&s->movers_active, cur, cur + 2) == cur) role = kRoleMover;
            } else if (role == kRoleMover && static_cast<int>(cur) - 1 > target) {
                if (atomicCAS(&s->movers_active, cur, cur - 2) == cur) role = kRoleCompute;
            }
        }
        Claim c1 = (role == kRoleMover) ? try_claim_mover(p, ctl) : try_claim_compute(p, ctl);
        if (c1.kind != kActIdle && c1.kind != kActExit) {
            last_progress = globaltimer_ns();
            return c1;
        }
        Claim c2 = (role == kRoleMover) ? try_claim_compute(p, ctl) : try_claim_mover(p, ctl);
        if (c2.kind != kActIdle && c2.kind != kActExit) {
            last_progress = globaltimer_ns();
            return c2;
        }
        if (c1.kind == kActExit && c2.kind == kActExit) return {kActExit, -1, -1};
        if (globaltimer_ns() - last_progress > p.timeout_ns) {
            report_error(p.status, MK_ERR_TIMEOUT, kSiteFusedIdle);
            atomicExch(&s->abort_flag, 1u);
            return {kActExit, -1, -1};
        }
        nanosleep_ns(backoff);
        backoff = backoff < 2048 ? 2 * backoff : 2048;
    }
}

// ------------------------------------------------------------------ mover tasks

// The router's block computation needs nearly every register of a thread; as
// a separate (not inlined) function it gets its own allocation.
template <int WT, int WE>
__device__ __noinline__ void fused_route_block(uint8_t* smem, const FPParams& p, int tg, int eg) {
    route_detail::route_block<WT, WE, 8, 1>(smem, reinterpret_cast<const uint16_t*>(p.x), p.wg, p.bias, p.T, p.d,
                                             p.E, p.logits, tg, eg);
}

// Dispatch of one task's tokens, then every row it wrote published on its
// 128-row M-tile's counter (proxy fence by every writer: the rows are read
// next through TMA; the block barrier orders all threads' stores before the
// release increments, which are cumulative over them).
__device__ __noinline__ void fused_dispatch(const FPParams& p, int64_t task) {
    const int64_t t_begin = task * p.dtok;
    const int nt = static_cast<int>(p.T - t_begin < p.dtok ? p.T - t_begin : p.dtok);
    const int64_t c = t_begin / kChunkTokens;
    tasks::dispatch_tokens(p.ids, p.w, p.d, p.E, p.k, c, t_begin, nt, p.offsets, p.chunk_base, p.rank, p.x,
                           p.x_perm, p.row_token, p.row_weight, p.slot_row);
    fence_proxy_async_global();
    __syncthreads();
    for (int q = threadIdx.x; q < nt * p.k; q += kThreads) {
        const int64_t tq = t_begin * p.k + q;
        const int e = p.ids[tq];
        const int in_e = p.chunk_base[c * p.E + e] + p.rank[tq];
        red_release_gpu_add(p.mt_rows + p.mtile_start[e] + in_e / BM, 1u);
    }
}

// The combine, run by a CTA until every token is claimed: y[t] = bf16( sum_j
// P[slot_row[t, j]] ), j ascending, fp32 (the kernel-per-step combine's sum and
// order).  Warp 0 claims kCombineClaim tokens at a time from the combine
// counter and copies the k rows of each token into shared memory with TMA bulk
// copies (lane j reads slot j's row index and copies that row), into a ring of
// up to kCombineBufs token buffers that stays full across claims, while all
// threads add the rows of the oldest token (16 bytes per thread per access,
// conflict-free).  When two token buffers do not fit in
// the shared union, tokens are claimed the same way and their rows read
// directly (a warp per token).
__device__ __noinline__ void fused_combine_loop(const FPParams& p, FCtl* ctl, uint8_t* smem) {
    const int tid = threadIdx.x;
    const uint32_t row_bytes = static_cast<uint32_t>(p.d) * 2u;
    const uint32_t tok_bytes = row_bytes * static_cast<uint32_t>(p.k);
    const int nbuf = min(kCombineBufs, static_cast<int>(kUnionBytes / tok_bytes));
    uint32_t* ctr = &p.sync->comb_head;
    if (nbuf < 2) {
        for (;;) {
            if (tid == 0) ctl->flag = static_cast<int>(atomicAdd(ctr, kCombineClaim));
            __syncthreads();
            const int t0 = ctl->flag;
            __syncthreads();
            if (t0 >= p.T) return;
            tasks::combine_tokens(p.P, p.slot_row, t0, min(kCombineClaim, p.T - t0), p.d, p.k, p.y);
        }
    }
    volatile uint32_t* abort_word = &ctl->abort_local;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    int cur = 0, cend = 0;  // warp 0: tokens claimed and not yet issued (the same in every lane)
    auto issue = [&](int b) {  // warp 0: the next token's k rows into buffer b (-1: none left)
        if (cur >= cend) {
            int c0 = 0;
            if (lane == 0) c0 = static_cast<int>(atomicAdd(ctr, kCombineClaim));
            c0 = __shfl_sync(0xffffffffu, c0, 0);
            cur = c0;
            cend = c0 < p.T ? min(c0 + kCombineClaim, p.T) : c0;
        }
        if (cur >= cend) {
            if (lane == 0) ctl->ctoken[b] = -1;
            return;
        }
        const int t = cur++;
        const uint32_t bar = smem_u32(&ctl->cbar[b]);
        const uint32_t dst = smem_u32(smem) + static_cast<uint32_t>(b) * tok_bytes;
        if (lane == 0) {
            ctl->ctoken[b] = t;
            mbar_arrive_expect_tx(bar, tok_bytes);
        }
        __syncwarp();
        if (lane < p.k) {  // lane j copies row j of the token (the slot rows are read in parallel)
            const int64_t r = p.slot_row[static_cast<int64_t>(t) * p.k + lane];
            bulk_load(dst + lane * row_bytes, p.P + r * p.d, row_bytes, bar);
        }
    };
    if (warp == 0) {
        fence_proxy_async_global();  // P was acquired with the decision; it is read next through TMA
        for (int b = 0; b < nbuf - 1; ++b) issue(b);
    }
    const int n16 = p.d / 8;
    for (int i = 0;; ++i) {
        const int b = i % nbuf;
        if (warp == 0) issue((i + nbuf - 1) % nbuf);  // that buffer was freed by the previous token
        __syncthreads();
        const int t = ctl->ctoken[b];
        if (t < 0) break;  // no token in this buffer, nor in any later one
        const uint32_t par = (ctl->cphase >> b) & 1u;
        const bool ok = mbar_wait_bounded(smem_u32(&ctl->cbar[b]), par, abort_word, p.timeout_ns);
        if (!__syncthreads_and(ok)) {
            if (tid == 0) {
                ctl->abort_local = 1u;
                atomicExch(&p.sync->abort_flag, 1u);
                report_error(p.status, MK_ERR_TIMEOUT, kSiteCombineWait);
            }
            return;
        }
        const uint8_t* buf = smem + static_cast<size_t>(b) * tok_bytes;
        uint4* dst = reinterpret_cast<uint4*>(p.y + static_cast<int64_t>(t) * p.d);
        for (int c = tid; c < n16; c += kThreads) {
            float acc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
            for (int j = 0; j < p.k; ++j) {
                const uint4 v = reinterpret_cast<const uint4*>(buf + j * row_bytes)[c];
                const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[2 * q] = __fadd_rn(acc[2 * q], __uint_as_float(wv[q] << 16));
                    acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], __uint_as_float(wv[q] & 0xffff0000u));
                }
            }
            uint4 o;
            o.x = pack_bf16x2(acc[0], acc[1]);
            o.y = pack_bf16x2(acc[2], acc[3]);
            o.z = pack_bf16x2(acc[4], acc[5]);
            o.w = pack_bf16x2(acc[6], acc[7]);
            dst[c] = o;
        }
        __syncthreads();  // every thread is done with buffer b before it is refilled
        if (tid == 0) ctl->cphase ^= 1u << b;
    }
    __syncthreads();
}

// Route task of one CTA, with the last-arriver chain behind it.
template <int WT, int WE>
__device__ void run_route_task(uint8_t* smem, const FPParams& p, FCtl* ctl, int arg) {
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    FusedSync* sync = p.sync;
    const int tg = arg / p.n_eg, eg = arg % p.n_eg;
    fused_route_block<WT, WE>(smem, p, tg, eg);
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const uint32_t old = atomicAdd(&p.route_done[tg], 1u);
        ctl->flag = (old == static_cast<uint32_t>(p.n_eg - 1)) ? 1 : 0;
        __threadfence();
    }
    __syncthreads();
    if (!ctl->flag) return;
    // last expert group of this token group: top-k of its tokens
    const int t0 = tg * p.ct;
    for (int tl = warp; tl < p.ct; tl += kThreads / 32)
        if (t0 + tl < p.T) tasks::topk_token(p.logits, t0 + tl, p.E, p.k, p.ids, p.w);
    __syncthreads();
    const int c = t0 / kChunkTokens;
    if (tid == 0) {
        const int nt_c = min(kChunkTokens, p.T - c * kChunkTokens);
        const int groups = (nt_c + p.ct - 1) / p.ct;
        __threadfence();
        const uint32_t old = atomicAdd(&p.topk_done[c], 1u);
        ctl->flag = (old == static_cast<uint32_t>(groups - 1)) ? 1 : 0;
        __threadfence();
    }
    __syncthreads();
    if (!ctl->flag) return;
    // last token group of this chunk: histogram and ranks
    tasks::count_chunk(reinterpret_cast<uint32_t*>(smem), p.ids, p.T, p.E, p.k, c, p.chunk_counts, p.rank);
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const uint32_t old = atomicAdd(&sync->count_done, 1u);
        ctl->flag = (old == static_cast<uint32_t>(p.nchunks - 1)) ? 1 : 0;
        __threadfence();
    }
    __syncthreads();
    if (!ctl->flag) return;
    // last chunk counted: the scans, then open the later queues
    tasks::scan_all(reinterpret_cast<int32_t*>(smem), p.chunk_counts, p.nchunks, p.E, p.chunk_base, p.counts,
                    p.offsets, p.mtile_start);
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        atomicExch(&sync->scan_done, 1u);
    }
}

// ------------------------------------------------------------------ GEMM session roles

__device__ __forceinline__ bool is_swap(int rows, int mode, const FPParams& p) {
    return rows <= (mode == 0 ? p.swap1 : p.swap2);
}
__device__ __forceinline__ int swap_n(int rows) { return (rows + 15) & ~15; }
__device__ __forceinline__ int swap_box(int half_n) {
    return half_n <= 16 ? 16 : half_n <= 32 ? 32 : half_n <= 64 ? 64 : 128;
}

// Pair tile t (gemm1 tiles first, then gemm2) -> mode, expert, pair block, N
// block: an expert's tiles of one GEMM occupy [pstart[e] * nt, pstart[e+1] * nt),
// in groups of kPairNGroup N blocks, each group over all the expert's pair
// blocks, N fastest.
struct PTile {
    int mode, e, row0, rows, n0, pb, g0;
};

__device__ __forceinline__ PTile decode_ptile(int tile, const FCtl* ctl, const FPParams& p, int nblocks) {
    PTile t;
    t.mode = tile < nblocks * p.NT1 ? 0 : 1;
    const int nt = t.mode == 0 ? p.NT1 : p.NT2;
    const int local = t.mode == 0 ? tile : tile - nblocks * p.NT1;
    const int g = local / nt;
    int lo = 0, hi = p.E - 1;  // largest e with pstart[e] <= g
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ctl->pstart[mid] <= g)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int p_e = ctl->pstart[lo + 1] - ctl->pstart[lo];
    const int l = local - ctl->pstart[lo] * nt;
    const int q = l / (p_e * kPairNGroup);
    const int nb = min(kPairNGroup, nt - q * kPairNGroup);
    const int r = l - q * p_e * kPairNGroup;
    const int j = r / nb;
    const int nblk = q * kPairNGroup + (r - j * nb);
    const int off = p.offsets[lo];
    const int cnt = p.offsets[lo + 1] - off;
    t.e = lo;
    t.row0 = off + j * PAIR_M;
    t.rows = min(PAIR_M, cnt - j * PAIR_M);
    t.n0 = nblk * (t.mode == 0 ? MMA_N / 2 : MMA_N);
    t.pb = ctl->pstart[lo] + j;
    t.g0 = p.mtile_start[lo] + 2 * j;
    return t;
}

__device__ __forceinline__ void raise_abort(FCtl* ctl, uint32_t peer) {
    ctl->abort_local = 1u;
    st_shared_cluster_u32(mapa_shared(smem_u32(&ctl->abort_local), peer), 1u);
}

// The session's pair-block table: every lane gets the layer's pair-block count;
// with `write`, the prefix over experts of their pair blocks goes to pstart
// (an expert with t 128-row tiles has ceil(t / 2) pair blocks).  Whole warp.
__device__ __forceinline__ int session_table(const FPParams& p, FCtl* ctl, bool write) {
    const int lane = threadIdx.x & 31;
    int cnt[kMaxExperts / 32], sum = 0;
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) {
        const int e = lane * (kMaxExperts / 32) + i;
        cnt[i] = (e < p.E) ? (p.mtile_start[e + 1] - p.mtile_start[e] + 1) / 2 : 0;
        sum += cnt[i];
    }
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
    }
    if (write) {
        int run = inc - sum;
#pragma unroll
        for (int i = 0; i < kMaxExperts / 32; ++i) {
            const int e = lane * (kMaxExperts / 32) + i;
            if (e < p.E) ctl->pstart[e] = run;
            run += cnt[i];
        }
        if (lane == 31) ctl->pstart[p.E] = inc;
    }
    __syncwarp();
    return __shfl_sync(0xffffffffu, inc, 31);
}

// Warp 6 of both CTAs during a GEMM session.
//   CTA 0, tile scheduler: once a slot is free, writes the next tile into both
//   CTAs' slot rings (the peer's through distributed shared memory), then claims
//   the one after it (one atomic ticket) unless the cluster should turn mover;
//   the session's first tile is `first`, an end marker closes it.
//   CTA 1, slot-release relay: once this CTA's producer and epilogue warps have
//   read a slot, one arrive (release at cluster scope, cumulative over theirs)
//   frees it on CTA 0.
// Keeping both off the producers means that neither pays a ticket's round trip
// or a cluster-scope release between two tiles' loads.
__device__ __noinline__ void gemm_scheduler(const FPParams& p, FCtl* ctl, int first, uint32_t rank) {
    FusedSync* sync = p.sync;
    PipeState* ps = &ctl->ps;
    volatile uint32_t* abort_word = &ctl->abort_local;
    const bool leader = elect_one();
    const int lead = __ffs(__ballot_sync(0xffffffffu, leader)) - 1;
    const uint32_t peer = rank ^ 1u;
    uint32_t slot = ps->sc_slot, slot_phase = ps->sc_slot_phase;
    bool ok = true;
    if (rank == 0) {
        const int nblocks = session_table(p, ctl, true);
        const int total = nblocks * (p.NT1 + p.NT2);
        const uint32_t peer_slot0 = mapa_shared(smem_u32(&ctl->slot[0]), peer);
        const uint32_t peer_slot2_0 = mapa_shared(smem_u32(&ctl->slot2[0]), peer);
        const uint32_t peer_slot_full0 = mapa_shared(smem_u32(&ctl->slot_full[0]), peer);
        int tile = first;
        for (;;) {
            int4 info = make_int4(-1, 0, 0, 0);
            int4 info2 = make_int4(0, 0, 0, 0);
            if (tile >= 0) {
                const PTile t = decode_ptile(tile, ctl, p, nblocks);
                info = make_int4(t.e | (t.mode << 16), t.row0, t.rows, t.n0);
                // z: more tiles follow than the clusters can hold at once (gemm2's epilogue paces
                // its stores only then)
                info2 = make_int4(t.pb, t.g0, tile + static_cast<int>(gridDim.x / 2) < total ? 1 : 0, 0);
            }
            if (!__all_sync(0xffffffffu, mbar_wait_bounded_cluster(smem_u32(&ctl->slot_empty[slot]), slot_phase ^ 1u,
                                                                  abort_word, p.timeout_ns))) {
                ok = false;
                break;
            }
            int next = -1;
            if (leader) {
                ctl->slot[slot] = info;
                ctl->slot2[slot] = info2;
                st_shared_cluster_v4(peer_slot0 + slot * static_cast<uint32_t>(sizeof(int4)), info);
                st_shared_cluster_v4(peer_slot2_0 + slot * static_cast<uint32_t>(sizeof(int4)), info2);
                mbar_arrive(smem_u32(&ctl->slot_full[slot]));
                mbar_arrive_cluster(peer_slot_full0 + slot * 8u);
                if (tile >= 0) {
                    // the next tile, unless this cluster should turn mover
                    const bool stay = (p.mover_ctas != 0) || ps->role == kRoleCompute ||
                                      static_cast<int>(ld_relaxed(&sync->movers_active)) >=
                                          static_cast<int>(ld_relaxed(&sync->target_movers));
                    if (stay && ld_relaxed(&sync->abort_flag) == 0u) {
                        const uint32_t h = atomicAdd(&sync->compute_head, 1u);
                        next = h < static_cast<uint32_t>(total) ? static_cast<int>(h) : -1;
                    }
                }
            }
            tile = __shfl_sync(0xffffffffu, next, lead);
            if (++slot == kSlots) {
                slot = 0;
                slot_phase ^= 1u;
            }
            if (info.x < 0) break;
        }
    } else {
        const uint32_t slot_empty0 = mapa_shared(smem_u32(&ctl->slot_empty[0]), 0);
        for (;;) {
            if (!__all_sync(0xffffffffu, mbar_wait_bounded_cluster(smem_u32(&ctl->slot_empty[slot]), slot_phase,
                                                                  abort_word, p.timeout_ns))) {
                ok = false;
                break;
            }
            const int e = ctl->slot[slot].x;
            __syncwarp();
            if (leader) mbar_arrive_cluster(slot_empty0 + slot * 8u);
            if (++slot == kSlots) {
                slot = 0;
                slot_phase ^= 1u;
            }
            if (e < 0) break;
        }
    }
    if (leader) {
        if (!ok) {
            raise_abort(ctl, peer);
            atomicExch(&sync->abort_flag, 1u);
            report_error(p.status, MK_ERR_TIMEOUT, kSiteGemmProducer);
        }
        ps->sc_slot = slot;
        ps->sc_slot_phase = slot_phase;
    }
    __syncwarp();
}

// Producer warp of both CTAs: follows the slots the scheduler writes and issues
// each tile's copies.  Returns the number of tiles the session ran.
__device__ __noinline__ int gemm_producer(const FPParams& p, const FMaps& m, FCtl* ctl, uint8_t* smem,
                                          uint32_t rank) {
    FusedSync* sync = p.sync;
    PipeState* ps = &ctl->ps;
    volatile uint32_t* abort_word = &ctl->abort_local;
    const volatile uint32_t* never = &ctl->zero;
    const bool leader = elect_one();
    const int lead = __ffs(__ballot_sync(0xffffffffu, leader)) - 1;
    const uint32_t peer = rank ^ 1u;
    uint32_t stage = ps->pr_stage, phase = ps->pr_phase, slot = ps->pr_slot, slot_phase = ps->pr_slot_phase,
             issued = ps->pr_issued, last_par = ps->pr_last_par;
    const uint32_t full0 = mapa_shared(smem_u32(&ctl->full[0]), 0);
    const int nblocks = session_table(p, ctl, false);
    int tiles_run = 0;
    bool ok = true;
    bool rows_all = false, h_all = false;  // every row landed / every gemm1 tile done (seen once)
    const uint32_t h_total = 8u * static_cast<uint32_t>(nblocks * p.NT1);  // gemm1 epilogue warps in all
    for (;;) {
        if (!__all_sync(0xffffffffu, mbar_wait_bounded_cluster(smem_u32(&ctl->slot_full[slot]), slot_phase,
                                                              abort_word, p.timeout_ns))) {
            ok = false;
            break;
        }
        const int4 info = ctl->slot[slot];
        const int4 info2 = ctl->slot2[slot];
        __syncwarp();
        if (leader) mbar_arrive(smem_u32(&ctl->slot_empty[slot]));
        if (++slot == kSlots) {
            slot = 0;
            slot_phase ^= 1u;
        }
        if (info.x < 0) break;
        ++tiles_run;
        const int mode = info.x >> 16;
        const int e = info.x & 0xffff;
        // readiness: gemm1 -- every row of the pair block has landed; gemm2 -- every gemm1
        // tile of the pair block has stored its h rows; then a proxy fence before the TMA reads.
        // Once the whole input of a GEMM is known complete (every dispatch task done, every
        // gemm1 tile done: one acquire), the session's later tiles of that GEMM skip the wait.
        if (!(mode == 0 ? rows_all : h_all)) {
            uint32_t ready = 1u;
            if (leader) {
                if (mode == 0 && ld_acquire_gpu(&sync->index_done) >= static_cast<uint32_t>(p.ND)) {
                    rows_all = true;
                } else if (mode == 1 && ld_acquire_gpu(&sync->h_tiles) >= h_total) {
                    h_all = true;
                } else if (mode == 0) {
                    for (int q = 0; q < (info.z > BM ? 2 : 1) && ready; ++q)
                        ready = wait_count_bounded(p.mt_rows + info2.y + q, static_cast<uint32_t>(min(BM, info.z - q * BM)),
                                                   abort_word, p.timeout_ns)
                                    ? 1u
                                    : 0u;
                } else {
                    ready = wait_count_bounded(p.h_done + info2.x, 8u * static_cast<uint32_t>(p.NT1), abort_word,
                                               p.timeout_ns)
                                ? 1u
                                : 0u;
                }
                fence_proxy_async_global();
            }
            rows_all = __shfl_sync(0xffffffffu, rows_all ? 1u : 0u, lead) != 0u;
            h_all = __shfl_sync(0xffffffffu, h_all ? 1u : 0u, lead) != 0u;
            if (!__shfl_sync(0xffffffffu, ready, lead)) {
                ok = false;
                break;
            }
        }
        const bool swap = is_swap(info.z, mode, p);
        const int kblocks = mode == 0 ? p.kb1 : p.kb2;
        const CUtensorMap* am = mode == 0 ? &m.a1 : &m.a2;
        const CUtensorMap* mb = mode == 0 ? (rank == 1 ? &m.w3 : &m.w1) : &m.w2;
        const int b_rows_per_expert = mode == 0 ? p.f : p.d;
        const int b_half_rows = mode == 0 ? 0 : MMA_N / 2;
        int a_row = info.y + static_cast<int>(rank) * BM;
        int b_row = e * b_rows_per_expert + info.w + static_cast<int>(rank) * b_half_rows;
        uint32_t stage_tx = PTX_BYTES;
        if (swap) {
            // weights into the A region (gemm1: 64 output columns per CTA, gemm2: 128), this
            // CTA's N / 2 block rows into the B region
            const int half_n = swap_n(info.z) >> 1;
            const int bx = swap_box(half_n);
            if (mode == 0)
                am = bx == 16 ? &m.a1_16 : bx == 32 ? &m.a1_32 : bx == 64 ? &m.a1_64 : &m.a1;
            else
                am = bx == 16 ? &m.a2_16 : bx == 32 ? &m.a2_32 : bx == 64 ? &m.a2_64 : &m.a2;
            a_row = info.y + static_cast<int>(rank) * half_n;
            b_row = e * b_rows_per_expert + info.w + static_cast<int>(rank) * (mode == 0 ? BM / 2 : MMA_N / 2);
            stage_tx = 2u * (PA_BYTES + static_cast<uint32_t>(bx) * BK * 2u);
        }
        for (int kb = 0; kb < kblocks; ++kb) {
            if (!__all_sync(0xffffffffu, mbar_wait_bounded_cluster(smem_u32(&ctl->empty[stage]), phase ^ 1u,
                                                                  abort_word, p.timeout_ns))) {
                ok = false;
                break;
            }
            if (leader) {
                const uint32_t fb = full0 + static_cast<uint32_t>(stage) * 8u;
                const uint32_t sa = smem_u32(smem + stage * PSTAGE_BYTES);
                const uint32_t sb = sa + PA_BYTES;
                if (rank == 0) mbar_arrive_expect_tx(smem_u32(&ctl->full[stage]), stage_tx);
                if (swap) {
                    if (mode == 0) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            tma_load_2d_pair(sa + q * 32 * BK * 2, &m.w1q, kb * BK, b_row + 16 * q, fb);
                            tma_load_2d_pair(sa + (q * 32 + 16) * BK * 2, &m.w3q, kb * BK, b_row + 16 * q, fb);
                        }
                    } else {
                        tma_load_2d_pair(sa, &m.w2, kb * BK, b_row, fb);
                    }
                    tma_load_2d_pair(sb, am, kb * BK, a_row, fb);
                } else {
                    tma_load_2d_pair(sa, am, kb * BK, a_row, fb);
                    tma_load_2d_pair(sb, mb, kb * BK, b_row, fb);
                }
            }
            __syncwarp();
            if (rank == 0) {
                issued |= 1u << stage;
                last_par = (last_par & ~(1u << stage)) | (phase << stage);
            }
            if (++stage == FSTAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
    }
    if (leader) {
        if (!ok) {
            raise_abort(ctl, peer);
            atomicExch(&sync->abort_flag, 1u);
            report_error(p.status, MK_ERR_TIMEOUT, kSiteGemmProducer);
            // CTA 0: every stage it armed completes (or times out) before the CTA leaves
            for (int s = 0; s < FSTAGES; ++s)
                if ((issued >> s) & 1u)
                    mbar_wait_bounded_cluster(smem_u32(&ctl->full[s]), (last_par >> s) & 1u, never, p.timeout_ns);
        }
        ps->pr_stage = stage;
        ps->pr_phase = phase;
        ps->pr_slot = slot;
        ps->pr_slot_phase = slot_phase;
        ps->pr_issued = issued;
        ps->pr_last_par = last_par;
        ps->last_progress = globaltimer_ns();
    }
    __syncwarp();
    return tiles_run;
}

// MMA issuer: warp 1 of CTA 0, converged, one elected lane issues.
__device__ __noinline__ void gemm_mma(const FPParams& p, FCtl* ctl, uint8_t* smem, uint32_t tmem_base) {
    FusedSync* sync = p.sync;
    PipeState* ps = &ctl->ps;
    volatile uint32_t* abort_word = &ctl->abort_local;
    const bool leader = elect_one();
    uint32_t stage = ps->mm_stage, phase = ps->mm_phase, acc = ps->mm_acc, acc_phase = ps->mm_acc_phase,
             slot = ps->mm_slot, slot_phase = ps->mm_slot_phase;
    bool ok = true;
    for (;;) {
        if (!__all_sync(0xffffffffu, mbar_wait_bounded_cluster(smem_u32(&ctl->slot_full[slot]), slot_phase,
                                                              abort_word, p.timeout_ns))) {
            ok = false;
            break;
        }
        const int4 info = ctl->slot[slot];
        __syncwarp();
        if (leader) mbar_arrive(smem_u32(&ctl->slot_empty[slot]));
        if (++slot == kSlots) {
            slot = 0;
            slot_phase ^= 1u;
        }
        if (info.x < 0) break;
        const int mode = info.x >> 16;
        const uint32_t idesc = is_swap(info.z, mode, p) ? idesc_bf16_f32(PAIR_M, swap_n(info.z)) : PIDESC;
        const int kblocks = mode == 0 ? p.kb1 : p.kb2;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded_cluster(smem_u32(&ctl->tmem_empty[acc]), acc_phase ^ 1u,
                                                              abort_word, p.timeout_ns))) {
            ok = false;
            break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * MMA_N;
        for (int kb = 0; kb < kblocks; ++kb) {
            if (!__all_sync(0xffffffffu, mbar_wait_bounded_cluster(smem_u32(&ctl->full[stage]), phase, abort_word,
                                                                  p.timeout_ns))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (leader) {
                const uint32_t sa = smem_u32(smem + stage * PSTAGE_BYTES);
                const uint32_t sb = sa + PA_BYTES;
#pragma unroll
                for (int kk = 0; kk < BK / UMMA_K; ++kk)
                    mma_bf16_ss_pair(d_tmem, sw128_kmajor_desc(sa + kk * UMMA_K * 2),
                                     sw128_kmajor_desc(sb + kk * UMMA_K * 2), idesc, (kb | kk) != 0 ? 1u : 0u);
                mma_commit_pair_mc(smem_u32(&ctl->empty[stage]), 0x3);
            }
            __syncwarp();
            if (++stage == FSTAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
        if (leader) mma_commit_pair_mc(smem_u32(&ctl->tmem_full[acc]), 0x3);
        __syncwarp();
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
    }
    if (leader) {
        if (!ok) {
            raise_abort(ctl, 1u);
            atomicExch(&sync->abort_flag, 1u);
            report_error(p.status, MK_ERR_TIMEOUT, kSiteGemmMma);
        }
        ps->mm_stage = stage;
        ps->mm_phase = phase;
        ps->mm_acc = acc;
        ps->mm_acc_phase = acc_phase;
        ps->mm_slot = slot;
        ps->mm_slot_phase = slot_phase;
    }
    __syncwarp();
}

// Epilogue warps 2-5 of both CTAs.  gemm1 tiles publish each warp's stores on
// the pair block's counter (proxy fence: gemm2 reads h through TMA); gemm2
// tiles are counted and published once at the end of the session (the
// combine waits for all of them).
__device__ __noinline__ void gemm_epilogue(const FPParams& p, FCtl* ctl, uint32_t tmem_base, uint32_t rank) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    FusedSync* sync = p.sync;
    PipeState* ps = &ctl->ps;
    volatile uint32_t* abort_word = &ctl->abort_local;
    const int sub = warp & 3;  // TMEM lanes [32*sub, 32*sub+32) are this warp's
    const int lane_in_tile = sub * 32 + lane;
    const uint32_t tmem_empty0 = mapa_shared(smem_u32(&ctl->tmem_empty[0]), 0);
    uint32_t acc = ps->ep_acc, acc_phase = ps->ep_acc_phase, slot = ps->ep_slot, slot_phase = ps->ep_slot_phase;
    uint32_t p_tiles = 0;
    bool ok = true;
    for (;;) {
        if (!mbar_wait_bounded_cluster(smem_u32(&ctl->slot_full[slot]), slot_phase, abort_word, p.timeout_ns)) {
            ok = false;
            break;
        }
        const int4 info = ctl->slot[slot];
        const int4 info2 = ctl->slot2[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->slot_empty[slot]));
        if (++slot == kSlots) {
            slot = 0;
            slot_phase ^= 1u;
        }
        if (info.x < 0) break;
        const int mode = info.x >> 16;
        if (!mbar_wait_bounded_cluster(smem_u32(&ctl->tmem_full[acc]), acc_phase, abort_word, p.timeout_ns)) {
            ok = false;
            break;
        }
        tc_fence_after();
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) + acc * MMA_N;
        bf16* out = mode == 0 ? p.h : p.P;
        const int64_t ld = mode == 0 ? p.f : p.d;
        const int n_valid = mode == 0 ? p.f : p.d;
        if (is_swap(info.z, mode, p)) {
            bf16* oblock = out + static_cast<int64_t>(info.y) * ld;
            if (mode == 0) {
                const int col = info.w + static_cast<int>(rank) * (BM / 2) + sub * 16 + (lane & 15);
                const bool c_ok = col < n_valid;
                epilogue_swiglu_swap(tbase, info.z, oblock + (c_ok ? col : 0), ld, c_ok);
            } else {
                const int n = info.w + static_cast<int>(rank) * (MMA_N / 2) + lane_in_tile;
                const bool n_ok = n < n_valid;
                epilogue_weighted_swap(tbase, info.z, oblock + (n_ok ? n : 0), ld, n_ok, p.row_weight + info.y);
            }
        } else {
            // full tile: TMEM lane = row of this CTA's 128
            const bool row_ok = static_cast<int>(rank) * BM + lane_in_tile < info.z;
            const int64_t r = static_cast<int64_t>(info.y) + static_cast<int>(rank) * BM + lane_in_tile;
            bf16* orow = out + (row_ok ? r : 0) * ld;
            if (mode == 0) {
                epilogue_swiglu(tbase, row_ok, orow, info.w, n_valid);
            } else {
                const float wr = row_ok ? p.row_weight[r] : 1.0f;
                const bool pace = info2.z != 0 && p.kb2 < kEpiPaceMaxKb;
                epilogue_weighted(tbase, row_ok, orow, info.w, n_valid, wr,
                                  pace ? static_cast<uint32_t>(p.kb2) * kEpiPacePerKb : 0u);
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tmem_empty0 + acc * 8u);
        if (mode == 0) {
            // h is read next by gemm2's TMA loads (async proxy): every lane's proxy fence, the
            // warp barrier, then one release increment on the pair block's counter
            fence_proxy_async_global();
            __syncwarp();
            if (lane == 0) {
                red_release_gpu_add(p.h_done + info2.x, 1u);
                red_release_gpu_add(&sync->h_tiles, 1u);
            }
        } else {
            ++p_tiles;
        }
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok && lane == 0) {
        raise_abort(ctl, rank ^ 1u);
        atomicExch(&sync->abort_flag, 1u);
        report_error(p.status, MK_ERR_TIMEOUT, kSiteGemmEpilogue);
    }
    // P is read next by the combine's bulk copies (async proxy): every lane's proxy
    // fence, the warp barrier, then one release increment for the session's tiles
    fence_proxy_async_global();
    __syncwarp();
    if (lane == 0 && p_tiles != 0u) red_release_gpu_add(&sync->p_done, p_tiles);  // the combine waits for all
    if (warp == 2 && lane == 0) {  // the four epilogue warps hold the same positions
        ps->ep_acc = acc;
        ps->ep_acc_phase = acc_phase;
        ps->ep_slot = slot;
        ps->ep_slot_phase = slot_phase;
    }
}

// ------------------------------------------------------------------ kernel

template <int WT, int WE>
__global__ void __launch_bounds__(kThreads, 1) fused_pair_kernel(const __grid_constant__ FMaps maps, const FPParams p) {
    using RT = route_detail::RouteTile<WT, WE, 8, 1>;
    static_assert(RT::SMEM <= static_cast<int>(kUnionBytes), "router stages fit the shared union");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    FCtl* ctl = reinterpret_cast<FCtl*>(smem + kUnionBytes);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    FusedSync* sync = p.sync;

    if (tid == 0) {
        for (int i = 0; i < FSTAGES; ++i) {
            mbar_init(smem_u32(&ctl->full[i]), 1);
            mbar_init(smem_u32(&ctl->empty[i]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&ctl->tmem_full[a]), 1);
            mbar_init(smem_u32(&ctl->tmem_empty[a]), 8);
        }
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(smem_u32(&ctl->slot_full[i]), 1);
            mbar_init(smem_u32(&ctl->slot_empty[i]), rank == 0 ? kSlotConsumers0 : kSlotConsumers1);
        }
        mbar_init(smem_u32(&ctl->drain), 1);
        for (int i = 0; i < kCombineBufs; ++i) mbar_init(smem_u32(&ctl->cbar[i]), 1);
        ctl->cphase = 0;
        ctl->abort_local = 0;
        ctl->zero = 0;
        ctl->pair_blocks = -1;
        ctl->ps = PipeState{};
        fence_mbar_init();
        prefetch_tensormap(&maps.a1);
        prefetch_tensormap(&maps.w1);
        prefetch_tensormap(&maps.w3);
        prefetch_tensormap(&maps.a2);
        prefetch_tensormap(&maps.w2);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&ctl->tmem_base), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers exist before any copy, commit or arrive targets them
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    PipeState* ps = &ctl->ps;

    // The cluster's role (CTA 0's thread 0 keeps it).  Adaptive mode starts with
    // every block a mover: with the routing computed in this kernel only route
    // tasks exist before the scans (otherwise the controller rebalances at the
    // first decision).
    if (rank == 0 && tid == 0) {
        int role = kRoleMover;
        const int cluster = static_cast<int>(blockIdx.x) / 2;
        if (p.mover_ctas > 0) role = (2 * cluster < p.mover_ctas) ? kRoleMover : kRoleCompute;
        if (p.mover_ctas < 0) role = kRoleCompute;
        if (p.mover_ctas == 0) {
            atomicAdd(&sync->movers_active, 2u);
            if (blockIdx.x == 0) atomicExch(&sync->target_movers, gridDim.x);
        }
        ps->role = role;
        ps->last_progress = globaltimer_ns();
    }

    for (;;) {
        if (rank == 0 && tid == 0) {
            int role = ps->role;
            unsigned long long lp = ps->last_progress;
            const Claim c = decide(p, ctl, role, lp);
            ps->role = role;
            ps->last_progress = lp;
            ctl->action = c.kind;
            ctl->arg0 = c.a0;
            ctl->arg1 = c.a1;
            // the same decision in CTA 1's shared memory (made visible by the cluster barrier)
            const uint32_t pa = mapa_shared(smem_u32(&ctl->action), peer);
            st_shared_cluster_u32(pa, static_cast<uint32_t>(c.kind));
            st_shared_cluster_u32(pa + 4, static_cast<uint32_t>(c.a0));
            st_shared_cluster_u32(pa + 8, static_cast<uint32_t>(c.a1));
        }
        cluster_sync_all();
        const int action = ctl->action;
        const int my_arg = rank == 0 ? ctl->arg0 : ctl->arg1;
        const int first_tile = ctl->arg0;
        if (tid == 0) {
            ps->t_start = clock64();
            ps->g_start = globaltimer_ns();
        }
        if (action == kActExit) break;

        int gemm_tiles = 0;
        if (action == kActRoute) {
            if (my_arg >= 0) run_route_task<WT, WE>(smem, p, ctl, my_arg);
        } else if (action == kActIndex) {
            if (my_arg >= 0) {
                fused_dispatch(p, my_arg);
                __syncthreads();
                if (tid == 0) red_release_gpu_add(&sync->index_done, 1u);
            }
        } else if (action == kActCombine) {
            fused_combine_loop(p, ctl, smem);
        } else if (action == kActGemm) {
            if (warp == 0) {
                gemm_tiles = gemm_producer(p, maps, ctl, smem, rank);
            } else if (warp == 1) {
                if (rank == 0) gemm_mma(p, ctl, smem, tmem_base);
            } else if (warp >= 2 && warp <= 5) {
                gemm_epilogue(p, ctl, tmem_base, rank);
            } else if (warp == kSchedWarp) {
                gemm_scheduler(p, ctl, first_tile, rank);
            }
        }
        __syncthreads();
        if (tid == 0 && (action != kActGemm || rank == 0) && (action == kActGemm || my_arg >= 0)) {
            const int r = (action == kActGemm) ? 1 : 0;
            const uint32_t n = (action == kActGemm) ? static_cast<uint32_t>(max(gemm_tiles, 1)) : 1u;
            if (p.trace != nullptr) {
                const uint32_t idx = atomicAdd(&sync->trace_n, 1u);
                if (idx < static_cast<uint32_t>(p.trace_cap)) {
                    const unsigned long long g1 = globaltimer_ns();
                    uint32_t* rec = p.trace + 8ull * idx;
                    rec[0] = blockIdx.x;
                    rec[1] = static_cast<uint32_t>(action);
                    rec[2] = static_cast<uint32_t>(action == kActGemm ? first_tile : my_arg);
                    rec[3] = (action == kActGemm)
                                 ? (n | ((first_tile >= pair_blocks(p, ctl) * p.NT1) ? 0x80000000u : 0u))
                                 : 0u;
                    rec[4] = static_cast<uint32_t>(ps->g_start);
                    rec[5] = static_cast<uint32_t>(ps->g_start >> 32);
                    rec[6] = static_cast<uint32_t>(g1);
                    rec[7] = static_cast<uint32_t>(g1 >> 32);
                }
            }
            atomicAdd(&sync->cyc[r], static_cast<unsigned long long>(clock64() - ps->t_start));
            atomicAdd(&sync->ntask[r], n);
            if (p.mover_ctas == 0 && rank == 0) {  // Eq. 2 after every finished task
                const uint32_t target = static_cast<uint32_t>(controller_target(p, ctl));
                if (ld_relaxed(&sync->target_movers) != target) atomicExch(&sync->target_movers, target);
            }
        }
        cluster_sync_all();  // CTA 1 has read the decision and finished its task before the next one
    }

    // Every MMA issued completes before either CTA frees TMEM or shared memory.
    if (rank == 0 && warp == 1) {
        const bool leader = elect_one();
        if (leader) {
            mma_commit_pair_mc(smem_u32(&ctl->drain), 0x1);
            if (!mbar_wait_bounded_cluster(smem_u32(&ctl->drain), 0u, &ctl->zero, p.timeout_ns))
                report_error(p.status, MK_ERR_TIMEOUT, kSiteGemmDrain);
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // neither CTA leaves while the other may still use its shared memory
    if (ctl->abort_local != 0u && tid == 0) {
        // after a timeout, copies the peer started may still complete on CTA 0's
        // barriers: keep both CTAs resident a little longer (bounded) before exit
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

template <int WT, int WE>
cudaError_t launch_shape(const FMaps& maps, const FPParams& p, cudaStream_t s) {
    static std::atomic<int> configured[64];    // per device: attributes set, max_clusters valid
    static std::atomic<int> max_clusters[64];  // written before `configured` (release / acquire)
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const int slot = dev < 64 ? dev : 0;
    auto fn = fused_pair_kernel<WT, WE>;
    if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
        err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kFusedSmem));
        if (err != cudaSuccess) return err;
        LaunchCfg probe(dim3(2 * std::max(1, device_sm_count() / 2)), dim3(kThreads), kFusedSmem, s, false, 2);
        int n = 0;
        err = cudaOccupancyMaxActiveClusters(&n, fn, &probe.cfg);
        if (err != cudaSuccess) return err;
        if (n < 1) return cudaErrorInvalidConfiguration;
        max_clusters[slot].store(n, std::memory_order_relaxed);
        if (dev < 64) configured[dev].store(1, std::memory_order_release);
    }
    // every cluster co-resident (the blocks wait on one another's tasks): the grid
    // is the number of clusters that fit at once (the runtime takes no cooperative
    // launch with a cluster dimension; with other work on the GPU a cluster that
    // cannot start makes the others' bounded waits run out: MK_ERR_TIMEOUT)
    const int clusters = max_clusters[slot].load(std::memory_order_relaxed);
    LaunchCfg lc(dim3(2 * clusters), dim3(kThreads), kFusedSmem, s, false, 2);
    err = cudaLaunchKernelEx(&lc.cfg, fn, maps, p);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

bool make_fused_maps(FMaps* m, const FusedArgs& a) {
    const uint64_t S = static_cast<uint64_t>(a.T) * a.k;
    const uint64_t w13 = static_cast<uint64_t>(a.E) * a.f;
    const uint64_t w2r = static_cast<uint64_t>(a.E) * a.d;
    return make_map(&m->a1, a.x_perm, a.d, S, BM) && make_map(&m->a1_16, a.x_perm, a.d, S, 16) &&
           make_map(&m->a1_32, a.x_perm, a.d, S, 32) && make_map(&m->a1_64, a.x_perm, a.d, S, 64) &&
           make_map(&m->w1, a.w1, a.d, w13, MMA_N / 2) && make_map(&m->w3, a.w3, a.d, w13, MMA_N / 2) &&
           make_map(&m->w1q, a.w1, a.d, w13, 16) && make_map(&m->w3q, a.w3, a.d, w13, 16) &&
           make_map(&m->a2, a.h, a.f, S, BM) && make_map(&m->a2_16, a.h, a.f, S, 16) &&
           make_map(&m->a2_32, a.h, a.f, S, 32) && make_map(&m->a2_64, a.h, a.f, S, 64) &&
           make_map(&m->w2, a.w2, a.f, w2r, MMA_N / 2);
}

}  // namespace

size_t fused_sync_bytes(int64_t T, int E, int k) {
    const int64_t n_tg = (T + 31) / 32;  // upper bound over the router block shapes
    const int64_t nch = num_chunks(T);
    const int64_t g_max = (T * k + kTileM - 1) / kTileM + E;  // M-tiles; also bounds the pair blocks
    return sizeof(FusedSync) + 4 * static_cast<size_t>(n_tg + nch + 2 * g_max);
}

cudaError_t launch_fused_pair(const FusedArgs& a, cudaStream_t s) {
    const int64_t T = a.T;
    const int d = a.d, E = a.E, k = a.k, f = a.f;
    FMaps maps;
    if (!make_fused_maps(&maps, a)) return cudaErrorInvalidValue;
    const bool wide = E >= 32;
    const int ct = wide ? 32 : 64, ce = wide ? 32 : 16;
    FPParams p;
    p.x = a.x;
    p.wg = a.wg;
    p.bias = a.bias;
    p.T = static_cast<int>(T);
    p.d = d;
    p.E = E;
    p.k = k;
    p.f = f;
    p.logits = a.logits;
    p.ids = a.ids;
    p.w = a.w;
    p.chunk_counts = a.chunk_counts;
    p.chunk_base = a.chunk_base;
    p.rank = a.rank;
    p.counts = a.counts;
    p.offsets = a.offsets;
    p.mtile_start = a.mtile_start;
    p.row_token = a.row_token;
    p.row_weight = a.row_weight;
    p.slot_row = a.slot_row;
    p.x_perm = a.x_perm;
    p.h = a.h;
    p.P = a.P;
    p.y = a.y;
    p.status = a.status;
    uint8_t* sb = static_cast<uint8_t*>(a.sync);
    p.sync = reinterpret_cast<FusedSync*>(sb);
    const int64_t n_tg_max = (T + 31) / 32;
    const int64_t nch = num_chunks(T);
    const int64_t g_max = (T * k + kTileM - 1) / kTileM + E;
    uint32_t* arr = reinterpret_cast<uint32_t*>(sb + sizeof(FusedSync));
    p.route_done = arr;
    p.topk_done = arr + n_tg_max;
    p.mt_rows = p.topk_done + nch;
    p.h_done = p.mt_rows + g_max;
    p.n_tg = static_cast<int>((T + ct - 1) / ct);
    p.n_eg = (E + ce - 1) / ce;
    p.ct = ct;
    p.nchunks = static_cast<int>(nch);
    p.routed = a.routed ? 1 : 0;
    p.NR = a.routed ? 0 : p.n_tg * p.n_eg;  // no router tasks when the routing came in
    p.dtok = nch < device_sm_count() ? kDispatchTokensSmall : kChunkTokens;
    p.ND = static_cast<int>((T + p.dtok - 1) / p.dtok);
    p.NK = static_cast<int>((T + kCombineUnit - 1) / kCombineUnit);  // combine work in the controller's units
    p.NT1 = (f + MMA_N / 2 - 1) / (MMA_N / 2);
    p.NT2 = (d + MMA_N - 1) / MMA_N;
    p.kb1 = d / BK;
    p.kb2 = f / BK;
    p.swap1 = pair_swap_max_rows(1, p.kb1);
    p.swap2 = pair_swap_max_rows(2, p.kb2);
    p.mover_ctas = a.mover_ctas;
    p.timeout_ns = a.timeout_ns;
    p.trace = a.trace;
    p.trace_cap = a.trace_cap;
    cudaError_t err = cudaMemsetAsync(a.sync, 0, fused_sync_bytes(T, E, k), s);
    if (err != cudaSuccess) return err;
    return wide ? launch_shape<2, 4>(maps, p, s) : launch_shape<4, 2>(maps, p, s);
}

}  // namespace mk
