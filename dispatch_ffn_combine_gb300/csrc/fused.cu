// fused.cu -- the whole MoE layer as one persistent kernel whose thread blocks
// take data-movement ("mover") or compute roles.
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
// Two task queues claimed in order with atomic tickets: the mover queue in
// three ranges with a head each, the compute queue with one head (when the
// routing comes in precomputed -- ids, weights, chunk counts and scans, from
// the router and count/scan kernels launched just before -- the mover queue
// starts at the dispatch tasks):
//   mover queue:   route blocks (32 tokens x 32 experts of gate logits)
//                  -> dispatch tasks (128 tokens, or 32 in small layers: rows
//                     of their slots, and the token rows copied into those
//                     rows, each read once)
//                  -> combine tasks (32 tokens)
//   compute queue: gemm1 tiles (expert M-tile x 128 h columns)
//                  -> gemm2 tiles (expert M-tile x 256 output columns)
// Inline chains (last finisher of a counter does the next step):
//   last route block of a token group -> top-k of its tokens
//   last top-k of a 128-token chunk   -> expert histogram + ranks of the chunk
//   last chunk counted                -> scans (offsets, chunk bases, tiles)
// Readiness: dispatch tasks need the scans; gemm1 tiles need every dispatch
// task (an expert's 128-row tile draws its rows from tokens all over the
// batch); gemm2 tile (g, n) needs all gemm1 tiles of g; combine tasks need
// every gemm2 tile.  Each of the four epilogue warps
// of a GEMM tile publishes its own 32 rows, so a tile counts 4 when done.  A block claims only tasks whose
// inputs are ready, so claiming in order never deadlocks; every wait is
// bounded by %globaltimer and an abort word.
#include <atomic>
#include "gemm_impl.cuh"
#include "layer_tasks.cuh"
#include "route_impl.cuh"

namespace mk {
namespace {

using namespace gemm_detail;

constexpr int kThreads = 256;
constexpr int kInfoSlots = 4;
constexpr int kCombineTokens = 32;
// A dispatch task is a counting chunk, or a quarter of one when the layer has
// fewer chunks than blocks (mid: 32 chunks for 152 blocks ran 0.430 ms, its
// quarters 0.395; large: 256 chunks 20.19 ms, 1024 quarters 20.38).
constexpr int kDispatchTokensSmall = 32;
static_assert(kChunkTokens % kDispatchTokensSmall == 0, "a dispatch task stays inside one counting chunk");

enum : int { kRoleMover = 0, kRoleCompute = 1 };
enum : int { kActExit = 0, kActIdle = 1, kActRoute = 2, kActIndex = 3, kActCombine = 5, kActGemm = 6 };

struct TileSlot {
    int end;
    int mode;  // 0 gemm1, 1 gemm2
    int g;     // expert M-tile index
    int row0;
    int rows;
    int n0;
    int kblocks;
    int pad;
};

// Pipeline positions that persist across GEMM sessions; each role keeps its
// own fields here between sessions (not in registers, which the router's
// block computation needs in full).
struct PipeState {
    uint32_t pr_stage, pr_phase, pr_slot, pr_slot_phase, pr_issued, pr_last_par;
    uint32_t mm_stage, mm_phase, mm_acc, mm_acc_phase, mm_slot, mm_slot_phase;
    uint32_t ep_acc, ep_acc_phase, ep_slot, ep_slot_phase;
    int role;
    int pad;
    unsigned long long last_progress;
    long long t_start;
    unsigned long long g_start;
};

struct FusedCtl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t info_full[kInfoSlots];
    uint64_t info_empty[kInfoSlots];
    TileSlot info[kInfoSlots];
    PipeState ps;
    int32_t s_offsets[kMaxExperts + 1];      // GEMM sessions: tile decode from shared memory
    int32_t s_mtile_start[kMaxExperts + 1];
    uint32_t tmem_base;
    uint32_t abort_local;
    uint32_t zero;
    int action;
    int arg;
    int flag;
};

constexpr size_t kUnionBytes = static_cast<size_t>(STAGES) * STAGE_BYTES;  // >= router stages
constexpr size_t kFusedSmem = kUnionBytes + sizeof(FusedCtl) + 1024;

struct FusedParams {
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
    uint32_t* h_done;      // [G_max]
    int n_tg, n_eg, ct, nchunks;
    int NR, ND, NK;  // route, dispatch and combine tasks
    int dtok;        // tokens per dispatch task (kChunkTokens or kDispatchTokensSmall)
    int routed;  // 1: ids, weights, chunk counts, ranks and scans were computed before the launch
    int NT1, NT2, kb1, kb2;
    int mover_ctas;  // 0 adaptive; > 0 blocks [0, n) prefer mover tasks; < 0 no block prefers them
    uint64_t timeout_ns;
    uint32_t* trace;
    int trace_cap;
};

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// The offsets, chunk bases and tile table exist (computed in this launch by
// the last chunk counted, or before it when the routing came in precomputed).
__device__ __forceinline__ bool scans_ready(const FusedParams& p) {
    return p.routed != 0 || ld_acquire(&p.sync->scan_done) != 0u;
}

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

// GEMM tile `local` of one GEMM (nt N blocks per M-tile) -> its M-tile g, its
// N block and its expert (`mts` / `offs`: the tile table and the expert
// offsets, the shared-memory copies a GEMM session makes): an expert's tiles occupy [mts[e] * nt, mts[e+1] * nt)
// in groups of kNGroup N blocks, each group over all the expert's M-tiles, N
// fastest, so tiles claimed close together share a weight block and a row
// block in L2 (the stand-alone GEMMs' order).
constexpr int kNGroup = 4;
__device__ __forceinline__ void decode_tile(const int32_t* mts, const int32_t* offs, int E, int nt, int local, int& g,
                                            int& n, int& e, int& row0, int& rows) {
    const int gi = local / nt;
    int lo = 0, hi = E - 1;  // largest e with mts[e] <= gi
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (mts[mid] <= gi)
            lo = mid;
        else
            hi = mid - 1;
    }
    e = lo;
    const int p_e = mts[lo + 1] - mts[lo];
    const int l = local - mts[lo] * nt;
    const int q = l / (p_e * kNGroup);
    const int nb = min(kNGroup, nt - q * kNGroup);
    const int r = l - q * p_e * kNGroup;
    const int j = r / nb;
    n = q * kNGroup + (r - j * nb);
    g = mts[lo] + j;
    const int off = offs[lo];
    row0 = off + j * BM;
    rows = min(BM, offs[lo + 1] - off - j * BM);
}

struct Claim {
    int kind;
    int arg;
    int n;  // compute claims: number of consecutive tiles
};

// ------------------------------------------------------------------ claiming
// Run by thread 0 only.  The mover queue is three ranges, route -> dispatch
// -> combine, each with its own head.  All tasks of a range become ready at
// once (route tasks from the start, dispatch tasks with the scans, combine
// tasks when every gemm2 quarter is published), so a block claims from a range
// only after seeing it ready, with a fetch-add that never fails under
// contention, and never holds a ticket whose inputs may still be missing.  An
// acquire fence after a claim orders the task's reads after the flags.

__device__ Claim try_claim_mover(const FusedParams& p) {
    FusedSync* s = p.sync;
    if (ld_relaxed(&s->route_head) < static_cast<uint32_t>(p.NR)) {
        const uint32_t h = atomicAdd(&s->route_head, 1u);
        if (h < static_cast<uint32_t>(p.NR)) {
            __threadfence();
            return {kActRoute, static_cast<int>(h), 1};
        }
    }
    if (!scans_ready(p)) return {kActIdle, 0, 0};
    if (ld_relaxed(&s->index_head) < static_cast<uint32_t>(p.ND)) {
        const uint32_t h = atomicAdd(&s->index_head, 1u);
        if (h < static_cast<uint32_t>(p.ND)) {
            __threadfence();
            return {kActIndex, static_cast<int>(h), 1};
        }
    }
    if (ld_relaxed(&s->comb_head) >= static_cast<uint32_t>(p.NK)) return {kActExit, 0, 0};
    const int G = p.mtile_start[p.E];
    if (ld_relaxed(&s->p_done) != static_cast<uint32_t>(4 * G * p.NT2)) return {kActIdle, 0, 0};
    const uint32_t h = atomicAdd(&s->comb_head, 1u);
    if (h >= static_cast<uint32_t>(p.NK)) return {kActExit, 0, 0};
    __threadfence();
    return {kActCombine, static_cast<int>(h), 1};
}

// Compute tiles are claimed one at a time with a fetch-add on the queue head,
// which never fails under contention and keeps the tiles in flight across the
// grid consecutive (in the grouped order of decode_tile they share weight and
// row blocks in L2).
// gemm1 tiles are claimable once every dispatch task is done, so they never
// wait; a gemm2 tile's inputs (the four epilogue quarters of every gemm1 tile
// of its M-tile) may still be in flight when it is claimed, and its producer
// waits for them.  That wait cannot deadlock: every gemm1 tile was claimed
// before any gemm2 tile, by a block that is running it, and gemm1 tiles wait
// on nothing.
__device__ Claim try_claim_compute(const FusedParams& p) {
    FusedSync* s = p.sync;
    if (!scans_ready(p)) return {kActIdle, 0, 0};
    if (ld_acquire(&s->index_done) != static_cast<uint32_t>(p.ND)) return {kActIdle, 0, 0};
    const int G = p.mtile_start[p.E];
    const uint32_t total = static_cast<uint32_t>(G) * (p.NT1 + p.NT2);
    if (ld_relaxed(&s->compute_head) >= total) return {kActExit, 0, 0};
    const uint32_t h = atomicAdd(&s->compute_head, 1u);
    if (h >= total) return {kActExit, 0, 0};
    return {kActGemm, static_cast<int>(h), 1};
}

// Inside a GEMM session the queue is known to be open (the dispatch finished
// before the session's first claim) and its size is known: a claim is one
// fetch-add, with no acquire load that would flush the producer's L1.
__device__ __forceinline__ int claim_next_tile(const FusedParams& p, uint32_t total) {
    const uint32_t h = atomicAdd(&p.sync->compute_head, 1u);
    return h < total ? static_cast<int>(h) : -1;
}

// Eq. 2 of the paper: the mover-block target that equalises the predicted
// finishing times of the two roles.  Before the scans the compute queue is
// empty and its size unknown, so every block is a mover.
__device__ int controller_target(const FusedParams& p) {
    FusedSync* s = p.sync;
    const int B = static_cast<int>(gridDim.x);
    if (!scans_ready(p)) return B;
    const int G = p.mtile_start[p.E];
    const double mover_total = static_cast<double>(p.NR) + p.ND + p.NK;
    const double compute_total = static_cast<double>(G) * (p.NT1 + p.NT2);
    const uint32_t claimed = min(ld_relaxed(&s->route_head), static_cast<uint32_t>(p.NR)) +
                             min(ld_relaxed(&s->index_head), static_cast<uint32_t>(p.ND)) +
                             min(ld_relaxed(&s->comb_head), static_cast<uint32_t>(p.NK));
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

// Thread 0's choice of the next task.  The block's role (adaptive mode) moves
// toward the controller's published target; the preferred queue is tried
// first, the other one when nothing preferred is ready (a stalled block helps
// the other role); with nothing ready anywhere the thread backs off and
// retries, up to the timeout.
__device__ Claim decide(const FusedParams& p, int& role, unsigned long long& last_progress) {
    FusedSync* s = p.sync;
    uint32_t backoff = 64;
    for (;;) {
        if (ld_relaxed(&s->abort_flag) != 0u) return {kActExit, 0, 0};
        if (p.mover_ctas == 0) {
            const int target = static_cast<int>(ld_relaxed(&s->target_movers));
            const uint32_t cur = ld_relaxed(&s->movers_active);
            if (role == kRoleCompute && static_cast<int>(cur) < target) {
                if (atomicCAS(&s->movers_active, cur, cur + 1) == cur) role = kRoleMover;
            } else if (role == kRoleMover && static_cast<int>(cur) > target) {
                if (atomicCAS(&s->movers_active, cur, cur - 1) == cur) role = kRoleCompute;
            }
        }
        Claim c1 = (role == kRoleMover) ? try_claim_mover(p) : try_claim_compute(p);
        if (c1.kind != kActIdle && c1.kind != kActExit) {
            last_progress = globaltimer_ns();
            return c1;
        }
        Claim c2 = (role == kRoleMover) ? try_claim_compute(p) : try_claim_mover(p);
        if (c2.kind != kActIdle && c2.kind != kActExit) {
            last_progress = globaltimer_ns();
            return c2;
        }
        if (c1.kind == kActExit && c2.kind == kActExit) return {kActExit, 0, 0};
        if (globaltimer_ns() - last_progress > p.timeout_ns) {
            report_error(p.status, MK_ERR_TIMEOUT, kSiteFusedIdle);
            atomicExch(&s->abort_flag, 1u);
            return {kActExit, 0, 0};
        }
        nanosleep_ns(backoff);
        backoff = backoff < 2048 ? 2 * backoff : 2048;
    }
}

// Publish a finished task: a release increment (orders every write of this
// thread, and those ordered before it by a block or warp barrier, before it).
__device__ __forceinline__ void publish_add(uint32_t* word, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(word), "r"(v) : "memory");
}

// The router's block computation needs nearly every register of a thread; as
// a separate (not inlined) function it gets its own allocation, and the
// persistent kernel's live state is saved around the call instead of being
// spilled inside its FMA loop.
template <int WT, int WE>
__device__ __noinline__ void fused_route_block(uint8_t* smem, const FusedParams& p, int tg, int eg) {
    route_detail::route_block<WT, WE, 8, 1>(smem, reinterpret_cast<const uint16_t*>(p.x), p.wg, p.bias, p.T, p.d,
                                             p.E, p.logits, tg, eg);
}

// The dispatch and combine bodies keep many loads in flight; separate
// functions keep their registers out of the persistent kernel's allocation.
__device__ __noinline__ void fused_dispatch(const FusedParams& p, int64_t task) {
    const int64_t t_begin = task * p.dtok;
    const int nt = static_cast<int>(p.T - t_begin < p.dtok ? p.T - t_begin : p.dtok);
    tasks::dispatch_tokens(p.ids, p.w, p.d, p.E, p.k, t_begin / kChunkTokens, t_begin, nt, p.offsets, p.chunk_base,
                           p.rank, p.x, p.x_perm, p.row_token, p.row_weight, p.slot_row);
}

__device__ __noinline__ void fused_combine(const FusedParams& p, int64_t t0, int nt) {
    tasks::combine_tokens(p.P, p.slot_row, t0, nt, p.d, p.k, p.y);
}

// ------------------------------------------------------------------ GEMM roles
// The three roles of a GEMM session, each a separate function (own register
// allocation).  `tile` / `run` are the first claimed tile and the length of
// its claimed run; pipeline positions live in ctl->ps between sessions.

struct GemmMaps {
    const CUtensorMap* a1;  // dispatched rows (x_perm)
    const CUtensorMap* w1;
    const CUtensorMap* w3;
    const CUtensorMap* a2;
    const CUtensorMap* w2;
};

__device__ __noinline__ void gemm_producer(const FusedParams& p, const GemmMaps& m, FusedCtl* ctl, uint8_t* smem,
                                           int arg, int arg_n, int lane) {
    // Whole warp, lane 0 does the work: the claims, the tile-info ring and the
    // TMA loads; the other lanes follow its decisions.  The stage waits of the
    // k-loop are made by every lane, so lane 0 issues the copies converged.
    FusedSync* sync = p.sync;
    PipeState* ps = &ctl->ps;
    volatile uint32_t* abort_local = &ctl->abort_local;
    const volatile uint32_t* never = &ctl->zero;
    const int G = p.mtile_start[p.E];
    const int n1 = G * p.NT1;
    uint32_t pr_stage = ps->pr_stage, pr_phase = ps->pr_phase, pr_slot = ps->pr_slot,
             pr_slot_phase = ps->pr_slot_phase, pr_issued = ps->pr_issued, pr_last_par = ps->pr_last_par;
    const int role = ps->role;
    for (int i = lane; i <= p.E; i += 32) {  // tile decode from shared memory for the whole session
        ctl->s_offsets[i] = p.offsets[i];
        ctl->s_mtile_start[i] = p.mtile_start[i];
    }
    __syncwarp();
    if (lane == 0) fence_proxy_async_global();  // dispatched rows were acquired with the claim
    int tile = arg;
    int run_left = arg_n;  // tiles left in the claimed run, this one included
    bool ok = true;
    int session_tiles = 0;
    for (;;) {
        TileSlot ts;
        ts.end = (tile < 0) ? 1 : 0;
        if (tile >= 0) {
            ts.mode = tile < n1 ? 0 : 1;
            const int local = ts.mode == 0 ? tile : tile - n1;
            const int nt_cnt = ts.mode == 0 ? p.NT1 : p.NT2;
            int e, nblk;
            decode_tile(ctl->s_mtile_start, ctl->s_offsets, p.E, nt_cnt, local, ts.g, nblk, e, ts.row0, ts.rows);
            ts.n0 = nblk * (ts.mode == 0 ? MMA_N / 2 : MMA_N);
            ts.kblocks = ts.mode == 0 ? p.kb1 : p.kb2;
            ts.pad = e;
        }
        uint32_t got = 1u;
        if (lane == 0) {
            got = mbar_wait_bounded(smem_u32(&ctl->info_empty[pr_slot]), pr_slot_phase ^ 1u, abort_local,
                                    p.timeout_ns)
                      ? 1u
                      : 0u;
            if (got) {
                ctl->info[pr_slot] = ts;
                mbar_arrive(smem_u32(&ctl->info_full[pr_slot]));
            }
        }
        if (!__shfl_sync(0xffffffffu, got, 0)) {
            ok = false;
            break;
        }
        if (++pr_slot == kInfoSlots) {
            pr_slot = 0;
            pr_slot_phase ^= 1u;
        }
        if (ts.end) break;
        ++session_tiles;
        // Next tile: the rest of the claimed run, else one claimed now (unless
        // this block should turn mover).  The claim is issued before this
        // tile's loads and its result used after them, so the atomic's latency
        // overlaps the loads.
        int next = -1;
        if (lane == 0) {
            if (run_left > 1) {
                next = tile + 1;
                --run_left;
            } else {
                const bool stay = (p.mover_ctas != 0) || role == kRoleCompute ||
                                  static_cast<int>(ld_relaxed(&sync->movers_active)) >=
                                      static_cast<int>(ld_relaxed(&sync->target_movers));
                if (stay && ld_relaxed(&sync->abort_flag) == 0u) {
                    next = claim_next_tile(p, static_cast<uint32_t>(G) * (p.NT1 + p.NT2));
                    run_left = 1;
                }
            }
        }
        if (ts.mode == 1) {
            // gemm2: all gemm1 quarters of this M-tile must be published; then a
            // proxy fence orders the TMA reads of h after that acquire
            uint32_t ready = 1u;
            if (lane == 0) {
                const uint32_t want = static_cast<uint32_t>(4 * p.NT1);
                if (ld_acquire(&p.h_done[ts.g]) != want) {
                    const uint64_t t0 = globaltimer_ns();
                    uint32_t backoff = 32;
                    while (ld_acquire(&p.h_done[ts.g]) != want) {
                        if (*abort_local != 0u || ld_relaxed(&sync->abort_flag) != 0u ||
                            globaltimer_ns() - t0 > p.timeout_ns) {
                            ready = 0u;
                            break;
                        }
                        nanosleep_ns(backoff);
                        backoff = backoff < 1024 ? 2 * backoff : 1024;
                    }
                }
                fence_proxy_async_global();
            }
            if (!__shfl_sync(0xffffffffu, ready, 0)) {
                ok = false;
                break;
            }
        }
        const int e = ts.pad;
        const int b_row = ts.mode == 0 ? e * p.f + ts.n0 : e * p.d + ts.n0;
        for (int kb = 0; kb < ts.kblocks; ++kb) {
            // the whole warp waits for the stage (lane 0 then issues from a converged warp)
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&ctl->empty[pr_stage]), pr_phase ^ 1u,
                                                          abort_local, p.timeout_ns))) {
                ok = false;
                break;
            }
            const uint32_t fb = smem_u32(&ctl->full[pr_stage]);
            const uint32_t sa = smem_u32(smem + pr_stage * STAGE_BYTES);
            const uint32_t sb = sa + A_BYTES;
            if (lane == 0) mbar_arrive_expect_tx(fb, STAGE_BYTES);
            if (ts.mode == 0) {
                if (lane == 0) {
                    tma_load_2d(sa, m.a1, kb * BK, ts.row0, fb);
                    tma_load_2d(sb, m.w1, kb * BK, b_row, fb);
                    tma_load_2d(sb + B_BYTES / 2, m.w3, kb * BK, b_row, fb);
                }
            } else if (lane == 0) {
                tma_load_2d(sa, m.a2, kb * BK, ts.row0, fb);
                tma_load_2d(sb, m.w2, kb * BK, b_row, fb);
            }
            pr_issued |= 1u << pr_stage;
            pr_last_par = (pr_last_par & ~(1u << pr_stage)) | (pr_phase << pr_stage);
            if (++pr_stage == STAGES) {
                pr_stage = 0;
                pr_phase ^= 1u;
            }
        }
        if (!ok) break;
        tile = __shfl_sync(0xffffffffu, next, 0);
    }
    if (lane == 0) {
        if (!ok) {
            *abort_local = 1u;
            atomicExch(&sync->abort_flag, 1u);
            report_error(p.status, MK_ERR_TIMEOUT, kSiteGemmProducer);
            for (int i = 0; i < STAGES; ++i)
                if ((pr_issued >> i) & 1u)
                    mbar_wait_bounded(smem_u32(&ctl->full[i]), (pr_last_par >> i) & 1u, never, p.timeout_ns);
        }
        ps->last_progress = globaltimer_ns();
        ctl->arg = session_tiles;  // read back by thread 0 for the cost estimate
        ps->pr_stage = pr_stage;
        ps->pr_phase = pr_phase;
        ps->pr_slot = pr_slot;
        ps->pr_slot_phase = pr_slot_phase;
        ps->pr_issued = pr_issued;
        ps->pr_last_par = pr_last_par;
    }
    __syncwarp();
}

// The whole warp runs the MMA role; one elected lane issues the MMAs, the
// commits and the arrivals (a converged issuing warp keeps the tensor pipe's
// queue fuller than a lone lane); wait results are made warp-uniform.
__device__ __noinline__ void gemm_mma(const FusedParams& p, FusedCtl* ctl, uint8_t* smem, uint32_t tmem_base) {
    FusedSync* sync = p.sync;
    PipeState* ps = &ctl->ps;
    volatile uint32_t* abort_local = &ctl->abort_local;
    const bool leader = elect_one();
    uint32_t mm_stage = ps->mm_stage, mm_phase = ps->mm_phase, mm_acc = ps->mm_acc,
             mm_acc_phase = ps->mm_acc_phase, mm_slot = ps->mm_slot, mm_slot_phase = ps->mm_slot_phase;
    bool ok = true;
    for (;;) {
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&ctl->info_full[mm_slot]), mm_slot_phase,
                                                      abort_local, p.timeout_ns))) {
            ok = false;
            break;
        }
        const TileSlot ts = ctl->info[mm_slot];
        __syncwarp();
        if (leader) mbar_arrive(smem_u32(&ctl->info_empty[mm_slot]));
        if (++mm_slot == kInfoSlots) {
            mm_slot = 0;
            mm_slot_phase ^= 1u;
        }
        if (ts.end) break;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&ctl->tmem_empty[mm_acc]), mm_acc_phase ^ 1u,
                                                      abort_local, p.timeout_ns))) {
            ok = false;
            break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + mm_acc * MMA_N;
        for (int kb = 0; kb < ts.kblocks; ++kb) {
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&ctl->full[mm_stage]), mm_phase, abort_local,
                                                          p.timeout_ns))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (leader) {
                const uint32_t sa = smem_u32(smem + mm_stage * STAGE_BYTES);
                const uint32_t sb = sa + A_BYTES;
#pragma unroll
                for (int kk = 0; kk < BK / UMMA_K; ++kk)
                    mma_bf16_ss(d_tmem, sw128_kmajor_desc(sa + kk * UMMA_K * 2),
                                sw128_kmajor_desc(sb + kk * UMMA_K * 2), IDESC, (kb | kk) != 0 ? 1u : 0u);
                mma_commit(smem_u32(&ctl->empty[mm_stage]));
            }
            __syncwarp();
            if (++mm_stage == STAGES) {
                mm_stage = 0;
                mm_phase ^= 1u;
            }
        }
        if (!ok) break;
        if (leader) mma_commit(smem_u32(&ctl->tmem_full[mm_acc]));
        __syncwarp();
        mm_acc ^= 1u;
        if (mm_acc == 0) mm_acc_phase ^= 1u;
    }
    if (leader) {
        if (!ok) {
            *abort_local = 1u;
            atomicExch(&sync->abort_flag, 1u);
            report_error(p.status, MK_ERR_TIMEOUT, kSiteGemmMma);
        }
        ps->mm_stage = mm_stage;
        ps->mm_phase = mm_phase;
        ps->mm_acc = mm_acc;
        ps->mm_acc_phase = mm_acc_phase;
        ps->mm_slot = mm_slot;
        ps->mm_slot_phase = mm_slot_phase;
    }
    __syncwarp();
}

__device__ __noinline__ void gemm_epilogue(const FusedParams& p, FusedCtl* ctl, uint32_t tmem_base, int warp,
                                           int lane) {
    FusedSync* sync = p.sync;
    PipeState* ps = &ctl->ps;
    volatile uint32_t* abort_local = &ctl->abort_local;
    const int sub = warp & 3;  // TMEM lanes [32*sub, 32*sub+32) are this warp's
    const int row_in_tile = sub * 32 + lane;
    uint32_t ep_acc = ps->ep_acc, ep_acc_phase = ps->ep_acc_phase, ep_slot = ps->ep_slot,
             ep_slot_phase = ps->ep_slot_phase;
    uint32_t p_quarters = 0;  // gemm2 quarters stored by this warp, published once at the end
    bool ok = true;
    for (;;) {
        if (!mbar_wait_bounded(smem_u32(&ctl->info_full[ep_slot]), ep_slot_phase, abort_local, p.timeout_ns)) {
            ok = false;
            break;
        }
        const TileSlot ts = ctl->info[ep_slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->info_empty[ep_slot]));
        if (++ep_slot == kInfoSlots) {
            ep_slot = 0;
            ep_slot_phase ^= 1u;
        }
        if (ts.end) break;
        if (!mbar_wait_bounded(smem_u32(&ctl->tmem_full[ep_acc]), ep_acc_phase, abort_local, p.timeout_ns)) {
            ok = false;
            break;
        }
        tc_fence_after();
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) + ep_acc * MMA_N;
        const bool row_ok = row_in_tile < ts.rows;
        const int64_t r = static_cast<int64_t>(ts.row0) + row_in_tile;
        if (ts.mode == 0) {
            epilogue_swiglu(tbase, row_ok, p.h + r * p.f, ts.n0, p.f);
        } else {
            const float wr = row_ok ? p.row_weight[r] : 1.0f;
            epilogue_weighted(tbase, row_ok, p.P + r * p.d, ts.n0, p.d, wr);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->tmem_empty[ep_acc]));
        if (ts.mode == 0) {
            // h is read next by other blocks' TMA loads (async proxy): proxy
            // fence, then this warp publishes its quarter of the tile
            fence_proxy_async_global();
            __syncwarp();
            if (lane == 0) publish_add(&p.h_done[ts.g], 1u);
        } else {
            ++p_quarters;
        }
        ep_acc ^= 1u;
        if (ep_acc == 0) ep_acc_phase ^= 1u;
    }
    if (!ok && lane == 0) {
        *abort_local = 1u;
        atomicExch(&sync->abort_flag, 1u);
        report_error(p.status, MK_ERR_TIMEOUT, kSiteGemmEpilogue);
    }
    __syncwarp();
    if (lane == 0 && p_quarters != 0u) publish_add(&sync->p_done, p_quarters);  // combine waits for all of them
    if (warp == 2 && lane == 0) {  // the four epilogue warps hold the same positions
        ps->ep_acc = ep_acc;
        ps->ep_acc_phase = ep_acc_phase;
        ps->ep_slot = ep_slot;
        ps->ep_slot_phase = ep_slot_phase;
    }
}

// ------------------------------------------------------------------ kernel

template <int WT, int WE>
__global__ void __launch_bounds__(kThreads, 1)
    fused_layer_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmW1,
                       const __grid_constant__ CUtensorMap tmW3, const __grid_constant__ CUtensorMap tmA2,
                       const __grid_constant__ CUtensorMap tmW2, const FusedParams p) {
    using RT = route_detail::RouteTile<WT, WE, 8, 1>;
    static_assert(RT::SMEM <= static_cast<int>(kUnionBytes), "router stages fit the shared union");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    FusedCtl* ctl = reinterpret_cast<FusedCtl*>(smem + kUnionBytes);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    FusedSync* sync = p.sync;

    if (tid == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(smem_u32(&ctl->full[i]), 1);
            mbar_init(smem_u32(&ctl->empty[i]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&ctl->tmem_full[a]), 1);
            mbar_init(smem_u32(&ctl->tmem_empty[a]), 4);
        }
        for (int i = 0; i < kInfoSlots; ++i) {
            mbar_init(smem_u32(&ctl->info_full[i]), 1);
            mbar_init(smem_u32(&ctl->info_empty[i]), 5);  // MMA thread + 4 epilogue warps
        }
        ctl->abort_local = 0;
        ctl->zero = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmA1);
        prefetch_tensormap(&tmW1);
        prefetch_tensormap(&tmW3);
        prefetch_tensormap(&tmA2);
        prefetch_tensormap(&tmW2);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;

    // Role of this block (thread 0 keeps it).  Adaptive mode starts with every
    // block a mover: with the routing computed in this kernel, only route
    // tasks exist before the scans (otherwise the controller rebalances at
    // the first decision).
    PipeState* ps = &ctl->ps;
    if (tid == 0) {
        *ps = PipeState{};
        int role = kRoleMover;
        if (p.mover_ctas > 0) role = (static_cast<int>(blockIdx.x) < p.mover_ctas) ? kRoleMover : kRoleCompute;
        if (p.mover_ctas < 0) role = kRoleCompute;
        if (p.mover_ctas == 0) {
            atomicAdd(&sync->movers_active, 1u);
            if (blockIdx.x == 0) atomicExch(&sync->target_movers, gridDim.x);
        }
        ps->role = role;
        ps->last_progress = globaltimer_ns();
    }
    __syncthreads();

    for (;;) {
        if (tid == 0) {
            int role = ps->role;
            unsigned long long lp = ps->last_progress;
            const Claim c = decide(p, role, lp);
            ps->role = role;
            ps->last_progress = lp;
            ctl->action = c.kind;
            ctl->arg = c.arg;
            ctl->flag = c.n;
            ps->t_start = clock64();
            ps->g_start = globaltimer_ns();
        }
        __syncthreads();
        const int action = ctl->action;
        const int arg = ctl->arg;
        const int arg_n = ctl->flag;
        __syncthreads();  // everyone has read the action before thread 0 may reuse the slot
        if (action == kActExit) break;

        if (action == kActRoute) {
            // ---------------------------------------------- gate logits block
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
            if (ctl->flag) {
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
                if (ctl->flag) {
                    // last token group of this chunk: histogram and ranks
                    tasks::count_chunk(reinterpret_cast<uint32_t*>(smem), p.ids, p.T, p.E, p.k, c, p.chunk_counts,
                                       p.rank);
                    __syncthreads();
                    if (tid == 0) {
                        __threadfence();
                        const uint32_t old = atomicAdd(&sync->count_done, 1u);
                        ctl->flag = (old == static_cast<uint32_t>(p.nchunks - 1)) ? 1 : 0;
                        __threadfence();
                    }
                    __syncthreads();
                    if (ctl->flag) {
                        // last chunk counted: the scans, then open the later queues
                        tasks::scan_all(reinterpret_cast<int32_t*>(smem), p.chunk_counts, p.nchunks, p.E,
                                        p.chunk_base, p.counts, p.offsets, p.mtile_start);
                        __syncthreads();
                        if (tid == 0) {
                            __threadfence();
                            atomicExch(&sync->scan_done, 1u);
                        }
                    }
                }
            }
        } else if (action == kActIndex) {
            fused_dispatch(p, arg);
            fence_proxy_async_global();  // the rows are read next by TMA (async proxy)
            __syncthreads();
            if (tid == 0) {
                fence_proxy_async_global();
                publish_add(&sync->index_done, 1u);
            }
        } else if (action == kActCombine) {
            const int t0 = arg * kCombineTokens;
            fused_combine(p, t0, min(kCombineTokens, p.T - t0));
        } else if (action == kActGemm) {
            // ---------------------------------------------- GEMM session
            const GemmMaps maps{&tmA1, &tmW1, &tmW3, &tmA2, &tmW2};
            if (warp == 0) {
                gemm_producer(p, maps, ctl, smem, arg, arg_n, lane);
            } else if (warp == 1) {
                gemm_mma(p, ctl, smem, tmem_base);
            } else if (warp >= 2 && warp <= 5) {
                gemm_epilogue(p, ctl, tmem_base, warp, lane);
            }
        }
        __syncthreads();
        if (tid == 0 && action != kActIdle) {
            const int r = (action == kActGemm) ? 1 : 0;
            const uint32_t n = (action == kActGemm) ? static_cast<uint32_t>(max(ctl->arg, 1)) : 1u;
            if (p.trace != nullptr) {
                const uint32_t idx = atomicAdd(&sync->trace_n, 1u);
                if (idx < static_cast<uint32_t>(p.trace_cap)) {
                    const unsigned long long g1 = globaltimer_ns();
                    uint32_t* rec = p.trace + 8ull * idx;
                    rec[0] = blockIdx.x;
                    rec[1] = static_cast<uint32_t>(action);
                    rec[2] = static_cast<uint32_t>(arg);
                    rec[3] = (action == kActGemm) ? (n | ((arg >= p.mtile_start[p.E] * p.NT1) ? 0x80000000u : 0u)) : 0u;
                    rec[4] = static_cast<uint32_t>(ps->g_start);
                    rec[5] = static_cast<uint32_t>(ps->g_start >> 32);
                    rec[6] = static_cast<uint32_t>(g1);
                    rec[7] = static_cast<uint32_t>(g1 >> 32);
                }
            }
            atomicAdd(&sync->cyc[r], static_cast<unsigned long long>(clock64() - ps->t_start));
            atomicAdd(&sync->ntask[r], n);
            if (p.mover_ctas == 0) {  // Eq. 2 after every finished task
                const uint32_t target = static_cast<uint32_t>(controller_target(p));
                if (ld_relaxed(&sync->target_movers) != target) atomicExch(&sync->target_movers, target);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int WT, int WE>
cudaError_t launch_fused_shape(const FusedArgs& a, const FusedParams& p, const CUtensorMap* maps, cudaStream_t s) {
    static std::atomic<int> configured[64];  // per device: attributes set (repeating them is harmless)
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    auto fn = fused_layer_kernel<WT, WE>;
    if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
        err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kFusedSmem));
        if (err != cudaSuccess) return err;
        if (dev < 64) configured[dev].store(1, std::memory_order_release);
    }
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, kFusedSmem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    const int grid = device_sm_count();  // one block per SM, all co-resident
    (void)a;
    void* args[] = {const_cast<CUtensorMap*>(&maps[0]), const_cast<CUtensorMap*>(&maps[1]),
                    const_cast<CUtensorMap*>(&maps[2]), const_cast<CUtensorMap*>(&maps[3]),
                    const_cast<CUtensorMap*>(&maps[4]), const_cast<FusedParams*>(&p)};
    err = cudaLaunchCooperativeKernel(reinterpret_cast<void*>(fn), dim3(grid), dim3(kThreads), args, kFusedSmem, s);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace

size_t fused_sync_bytes(int64_t T, int E, int k) {
    const int64_t n_tg = (T + 31) / 32;  // upper bound over the router block shapes
    const int64_t nch = num_chunks(T);
    const int64_t g_max = (T * k + kTileM - 1) / kTileM + E;
    return sizeof(FusedSync) + 4 * static_cast<size_t>(n_tg + nch + 2 * g_max);
}

cudaError_t launch_fused(const FusedArgs& a, cudaStream_t s) {
    const int64_t T = a.T;
    const int d = a.d, E = a.E, k = a.k, f = a.f;
    const int64_t S = T * k;
    CUtensorMap maps[5];
    if (!make_map(&maps[0], a.x_perm, d, S, BM) ||
        !make_map(&maps[1], a.w1, d, static_cast<uint64_t>(E) * f, MMA_N / 2) ||
        !make_map(&maps[2], a.w3, d, static_cast<uint64_t>(E) * f, MMA_N / 2) || !make_map(&maps[3], a.h, f, S, BM) ||
        !make_map(&maps[4], a.w2, f, static_cast<uint64_t>(E) * d, MMA_N))
        return cudaErrorInvalidValue;
    const bool wide = E >= 32;
    const int ct = wide ? 32 : 64, ce = wide ? 32 : 16;
    FusedParams p;
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
    uint32_t* arr = reinterpret_cast<uint32_t*>(sb + sizeof(FusedSync));
    p.route_done = arr;
    p.topk_done = arr + n_tg_max;
    p.h_done = p.topk_done + nch;
    p.n_tg = static_cast<int>((T + ct - 1) / ct);
    p.n_eg = (E + ce - 1) / ce;
    p.ct = ct;
    p.nchunks = static_cast<int>(nch);
    p.routed = a.routed ? 1 : 0;
    p.NR = a.routed ? 0 : p.n_tg * p.n_eg;  // no router tasks when the routing came in
    p.dtok = nch < device_sm_count() ? kDispatchTokensSmall : kChunkTokens;
    p.ND = static_cast<int>((T + p.dtok - 1) / p.dtok);
    p.NK = static_cast<int>((T + kCombineTokens - 1) / kCombineTokens);
    p.NT1 = (f + MMA_N / 2 - 1) / (MMA_N / 2);
    p.NT2 = (d + MMA_N - 1) / MMA_N;
    p.kb1 = d / BK;
    p.kb2 = f / BK;
    p.mover_ctas = a.mover_ctas;
    p.timeout_ns = a.timeout_ns;
    p.trace = a.trace;
    p.trace_cap = a.trace_cap;
    cudaError_t err = cudaMemsetAsync(a.sync, 0, fused_sync_bytes(T, E, k), s);
    if (err != cudaSuccess) return err;
    return wide ? launch_fused_shape<2, 4>(a, p, maps, s) : launch_fused_shape<4, 2>(a, p, maps, s);
}

}  // namespace mk
