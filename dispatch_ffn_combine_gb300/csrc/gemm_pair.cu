// gemm_pair.cu -- the grouped expert GEMMs on CTA pairs (tcgen05 cta_group::2).
//
// The same two GEMMs as the single-CTA kernel of gemm.cu (the expert FFN of
// the mKernel README's "MoE Dispatch + FFN + Combine" row: gemm1 -> SwiGLU ->
// gemm2), each output tile computed by a cluster of two CTAs on two SMs:
//
//   pair tile   256 rows of one expert x 256 accumulator columns.  CTA r holds
//               A rows [128 r, 128 r + 128) and half of the 256 B rows
//               (gemm1: CTA 0 the 128 gate rows of W1, CTA 1 the matching up
//               rows of W3; gemm2: W2 rows n0 + 128 r ...) and receives its
//               128 rows x 256 columns of the accumulator in its own TMEM.
//               One thread of CTA 0 issues the MMAs (M = 256, N = 256, K = 16).
//   swap tile   an expert's last pair block with fewer than 256 rows runs with
//               the operands exchanged: the 256 weight rows are the M side
//               (128 per CTA) and the block's rows the N side, N = rows rounded
//               up to 16 (CTA r holds rows [N/2 r, N/2 r + N/2), loaded with the
//               smallest 16/32/64/128-row box that covers them), so the MMAs
//               cost N/256 of a full tile's instead of a full tile's.  TMEM lane
//               l of CTA r then holds weight row 128 r + l for every block row.
//               gemm1 orders each CTA's 128 weight rows as four groups of 16
//               gate rows (W1) followed by the same 16 up rows (W3), so lanes
//               l and l + 16 of one warp hold the gate and up values of one
//               output column.  Each output element is the same dot product,
//               accumulated over K in the same order (the tests check that the
//               bits agree).  gemm1 keeps its blocks of 129-255 rows as full
//               tiles when K < 4096 (kSwapMaxRowsShortK).
//   why         per SM and k-block, 32 KB of operands cross L2 and shared
//               memory instead of 48 KB (B is split, not duplicated), so seven
//               stages (3584 cycles of MMA work) fit instead of four.
//   copies      each CTA loads its own A and B halves with TMA; all four
//               copies of a stage complete on CTA 0's `full` barrier, which
//               CTA 0 arms with both CTAs' bytes.
//   schedule    a scheduler warp of CTA 0 claims tiles in list order (one
//               atomic ticket each; the list keeps an expert's tiles in groups
//               of 4 N blocks over its pair blocks, so tiles claimed together
//               share weight and row blocks in L2) and writes each tile into
//               both CTAs' tile-slot rings (the peer's through distributed
//               shared memory).  Each CTA's slot readers release a slot on their
//               own CTA's barrier, and a relay warp of CTA 1 passes CTA 1's
//               release on to CTA 0, so no producer makes a cluster-scope
//               release or waits for a ticket between two tiles' loads (each
//               did, and the ~2 us gap drained the stage ring at every tile
//               start: gemm2 on the large layer 4.88 -> 4.64 ms).
//   release     the MMA commits arrive on both CTAs' `empty` and `tmem_full`
//               barriers (multicast); the 8 epilogue warps release an
//               accumulator on CTA 0's `tmem_empty` barrier.
//
// Every wait is bounded.  A CTA whose wait runs out records MK_ERR_TIMEOUT and
// raises the abort word of both CTAs; both leave through one cluster barrier,
// so neither exits while the other may still touch its shared memory.
#include <algorithm>
#include <atomic>

#include "gemm_impl.cuh"

namespace mk {
namespace {

using namespace gemm_detail;

constexpr int PSTAGES = 7;  // 224 KB: the most 32 KB stages that fit beside the control block
constexpr uint32_t PA_BYTES = BM * BK * 2;              // this CTA's 128 A rows, one k-block
constexpr uint32_t PB_BYTES = (MMA_N / 2) * BK * 2;     // this CTA's 128 of the 256 B rows
constexpr uint32_t PSTAGE_BYTES = PA_BYTES + PB_BYTES;  // 32 KB
constexpr uint32_t PTX_BYTES = 2 * PSTAGE_BYTES;        // both CTAs' copies of one stage
constexpr uint32_t PIDESC = idesc_bf16_f32(PAIR_M, MMA_N);
constexpr int kPairNGroup = 4;
constexpr int kPairSlots = 3;
constexpr int PNUM_THREADS = NUM_THREADS + 32;  // + warp 6: tile scheduler (CTA 0) / slot-release relay (CTA 1)
constexpr int kSchedWarp = PNUM_THREADS / 32 - 1;
// Readers of a tile slot that release it on their own CTA's `slot_empty`:
// CTA 0 its producer, MMA and 4 epilogue warps, plus CTA 1's relay (one
// arrive for CTA 1's producer and 4 epilogue warps).
constexpr uint32_t kSlotConsumers0 = 7;
constexpr uint32_t kSlotConsumers1 = 5;
// Which partial pair blocks run as swap tiles.  Measured (same GPU, every
// expert 256 + t rows): a swap tile costs 0.24-0.34 of a full tile for t <= 64
// and less than the full tile it replaces up to t ~ 240 with K = 7168; with
// K = 2048 gemm1's swap tiles of more than 128 rows cost up to 7 % more than
// full tiles (the SwiGLU epilogue and the eight 16-row weight copies per
// k-block against a short main loop), gemm2's none.
constexpr int kSwapMaxRows = PAIR_M - 1;
constexpr int kSwapMaxRowsShortK = BM;  // gemm1 with K < 64 k-blocks
// gemm2's full-tile epilogue spaces its four 64-column chunks by this many SM
// cycles per k-block of the tile (a k-block is 512 cycles of MMA work, so the
// chunks spread over ~60 % of the next tile's main loop).  Measured on the
// large layer: the MMA issuer's long operand waits at k-blocks 8-15 of a tile,
// where the previous tile's stores used to land in one burst, fell from 5.6 %
// to 1.9 % of its cycles (spacing 100), and gemm2 took 4.48-4.50 ms instead of
// 4.57-4.61 (spacing 80; 100: 4.53-4.56, 120: 4.56-4.61).  Only for short K
// (fewer than kEpiPaceMaxKb k-blocks), where a tile's output is a large share
// of its traffic: the Dispatch + GEMM kernel's K = 7168 tiles ran 2-4 % slower
// paced (their stores are a quarter as dense, and pacing holds the accumulator
// longer ahead of short swap tiles).
constexpr uint32_t kEpiPacePerKb = 80;
constexpr int kEpiPaceMaxKb = 64;

struct PairCtl {
    uint64_t full[PSTAGES];   // CTA 0: both CTAs' copies of the stage landed
    uint64_t empty[PSTAGES];  // each CTA: the pair MMAs that read the stage are done
    uint64_t tmem_full[2];    // each CTA: accumulator complete
    uint64_t tmem_empty[2];   // CTA 0: all 8 epilogue warps have read the accumulator
    uint64_t drain;           // CTA 0: every MMA issued has completed
    uint64_t slot_full[kPairSlots];   // each CTA: the scheduler wrote the tile slot
    uint64_t slot_empty[kPairSlots];  // each CTA: the slot's readers in this CTA have read it (CTA 0: and CTA 1's)
    int4 slot[kPairSlots];            // {e, row0, rows, n0}; e < 0 ends the list
    int slot_tile[kPairSlots];        // the tile's index in the list
    uint32_t tmem_base;
    uint32_t abort_flag;
    uint32_t zero;
    int32_t pstart[kMaxExperts + 1];  // prefix over experts of their pair blocks
};

// + 1024: the stages start at the first 1024-byte boundary (128-byte swizzle atoms)
constexpr size_t PSMEM_BYTES = static_cast<size_t>(PSTAGES) * PSTAGE_BYTES + sizeof(PairCtl) + 1024;
static_assert(PSMEM_BYTES <= 227u * 1024u, "pair GEMM shared memory exceeds the per-CTA limit");

struct PairParams {
    const int32_t* offsets;      // [E+1]
    const int32_t* mtile_start;  // [E+1] prefix of ceil(rows / 128); all zero when offsets were rejected
    const float* row_weight;     // gemm2 only, may be null
    bf16* out;
    int64_t out_ld;
    int E;
    int n_tiles;        // N blocks per pair block
    int tile_n;         // output columns per tile (128 gemm1, 256 gemm2)
    int n_valid;        // output columns of the whole GEMM
    int k_blocks;       // K / 64
    int b_rows_per_expert;
    int b_half_rows;    // row offset of CTA 1's half of B in a full tile (gemm1 0: own map; gemm2 128)
    int swap_max_rows;  // pair blocks with at most this many rows run as swap tiles (0: none)
    uint32_t* status;
    uint64_t timeout_ns;
    int stall_first_stage;  // test hook: CTA 0 of the pair that claims tile 0 never loads its first stage
    uint32_t* ticket;       // a zeroed word: tiles claimed so far
    // Tile-synchronised path (all null / 0 otherwise): per-M-tile semaphores.
    const uint32_t* wait_rows;    // gemm1: rows the dispatch has landed per M-tile
    const uint32_t* wait_h;       // gemm2: gemm1 epilogue completions per M-tile
    int wait_ntiles;              // gemm2: gemm1's N blocks per pair block
    int wait_swap_max;            // gemm2: gemm1's swap-tile threshold
    const uint32_t* weight_rows;  // gemm2: the dispatch's row counters, acquired before row weights
    uint32_t* post;               // this GEMM's epilogue completions per M-tile
    int pdl;                      // 1: let the next kernel launch after the prologue; 2: once the tiles run out
};

struct PairTile {
    int e;
    int row0;  // first row of the pair block
    int rows;  // valid rows of the pair block (1..256)
    int n0;
};

// A pair block with at most swap_max_rows rows (>= 128) runs as a swap tile.
__device__ __forceinline__ bool is_swap(int rows, const PairParams& p) { return rows <= p.swap_max_rows; }

// Swap tile: the MMA's N (block rows rounded up to 16) and the row count of
// the activation box each CTA loads (covers its N / 2 rows).
__device__ __forceinline__ int swap_n(int rows) { return (rows + 15) & ~15; }
__device__ __forceinline__ int swap_box(int half_n) {
    return half_n <= 16 ? 16 : half_n <= 32 ? 32 : half_n <= 64 ? 64 : 128;
}

// Tile t -> (expert, pair block, N block): an expert's tiles occupy
// [pstart[e] * n_tiles, pstart[e + 1] * n_tiles), in groups of kPairNGroup N
// blocks, each group over all the expert's pair blocks, N fastest.
__device__ __forceinline__ PairTile decode_pair_tile(int tile, const PairCtl* ctl, const PairParams& p) {
    const int g = tile / p.n_tiles;
    int lo = 0, hi = p.E - 1;  // largest e with pstart[e] <= g
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ctl->pstart[mid] <= g)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int p_e = ctl->pstart[lo + 1] - ctl->pstart[lo];
    const int l = tile - ctl->pstart[lo] * p.n_tiles;
    const int q = l / (p_e * kPairNGroup);
    const int nb = min(kPairNGroup, p.n_tiles - q * kPairNGroup);
    const int r = l - q * p_e * kPairNGroup;
    const int j = r / nb;
    const int nt = q * kPairNGroup + (r - j * nb);
    const int off = __ldg(p.offsets + lo);
    const int cnt = __ldg(p.offsets + lo + 1) - off;
    PairTile t;
    t.e = lo;
    t.row0 = off + j * PAIR_M;
    t.rows = min(PAIR_M, cnt - j * PAIR_M);
    t.n0 = nt * p.tile_n;
    return t;
}

__device__ __forceinline__ void raise_abort(PairCtl* ctl, uint32_t peer) {
    ctl->abort_flag = 1u;
    st_shared_cluster_u32(mapa_shared(smem_u32(&ctl->abort_flag), peer), 1u);
}

template <int MODE>  // 0: gemm1 + SwiGLU, 1: gemm2 + row weight
__global__ void __launch_bounds__(PNUM_THREADS, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                             const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmA16,
                             const __grid_constant__ CUtensorMap tmA32, const __grid_constant__ CUtensorMap tmA64,
                             const __grid_constant__ CUtensorMap tmB0q, const __grid_constant__ CUtensorMap tmB1q,
                             const PairParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    PairCtl* ctl = reinterpret_cast<PairCtl*>(smem + PSTAGES * PSTAGE_BYTES);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;

    // Tile table in shared memory: the pair-block prefix (an expert with t
    // 128-row blocks has ceil(t / 2) pair blocks).
    if (warp == 0) {
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
        int run = inc - sum;
#pragma unroll
        for (int i = 0; i < kMaxExperts / 32; ++i) {
            const int e = lane * (kMaxExperts / 32) + i;
            if (e < p.E) ctl->pstart[e] = run;
            run += cnt[i];
        }
        if (lane == 31) ctl->pstart[p.E] = inc;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < PSTAGES; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&ctl->tmem_full[a]), 1);
            mbar_init(smem_u32(&ctl->tmem_empty[a]), 8);
        }
        for (int i = 0; i < kPairSlots; ++i) {
            mbar_init(smem_u32(&ctl->slot_full[i]), 1);
            mbar_init(smem_u32(&ctl->slot_empty[i]), rank == 0 ? kSlotConsumers0 : kSlotConsumers1);
        }
        mbar_init(smem_u32(&ctl->drain), 1);
        ctl->abort_flag = 0;
        ctl->zero = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB0);
        if (MODE == 0) {
            prefetch_tensormap(&tmB1);
            prefetch_tensormap(&tmB0q);
            prefetch_tensormap(&tmB1q);
        }
        prefetch_tensormap(&tmA16);
        prefetch_tensormap(&tmA32);
        prefetch_tensormap(&tmA64);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&ctl->tmem_base), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers exist before any copy, commit or arrive targets them
    tc_fence_after();
    if (p.pdl == 1) pdl_launch_dependents();
    const uint32_t tmem_base = ctl->tmem_base;
    volatile uint32_t* abort_word = &ctl->abort_flag;
    const volatile uint32_t* never = &ctl->zero;
    const int total_tiles = ctl->pstart[p.E] * p.n_tiles;

    if (warp == 0) {
        {
            // ------------------------------------------------ TMA producer (both CTAs)
            // whole warp, one elected lane arrives and issues the copies.  The slot is
            // released on this CTA's own barrier: a local arrive, which does not wait for
            // the copies in flight the way a release at cluster scope would.
            const bool leader = elect_one();
            const int lead = __ffs(__ballot_sync(0xffffffffu, leader)) - 1;
            const uint32_t full0 = mapa_shared(smem_u32(&ctl->full[0]), 0);
            const CUtensorMap* mb = (MODE == 0 && rank == 1) ? &tmB1 : &tmB0;
            uint32_t stage = 0, phase = 0, issued = 0, last_par = 0, slot = 0, slot_phase = 0;
            bool ok = true;
            while (ok) {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded_cluster(smem_u32(&ctl->slot_full[slot]), slot_phase,
                                                                      abort_word, p.timeout_ns))) {
                    ok = false;
                    break;
                }
                const int4 info = ctl->slot[slot];
                const int cur_tile = ctl->slot_tile[slot];
                __syncwarp();
                if (leader) mbar_arrive(smem_u32(&ctl->slot_empty[slot]));
                if (++slot == kPairSlots) {
                    slot = 0;
                    slot_phase ^= 1u;
                }
                if (info.x < 0) break;
                if (p.wait_rows != nullptr || p.wait_h != nullptr) {
                    // tile-synchronised path: every row of the pair block has landed (gemm1) or
                    // every gemm1 tile of the block has stored its h rows (gemm2)
                    uint32_t ready = 1u;
                    if (leader) {
                        const int g0 = sem_tile0(p.offsets, p.mtile_start, info.x, info.y);
                        for (int q = 0; q < (info.z > BM ? 2 : 1) && ready; ++q) {
                            const uint32_t want =
                                p.wait_rows != nullptr
                                    ? static_cast<uint32_t>(min(BM, info.z - q * BM))
                                    : static_cast<uint32_t>(p.wait_ntiles * (info.z <= p.wait_swap_max ? 8 : 4));
                            const uint32_t* ctr = (p.wait_rows != nullptr ? p.wait_rows : p.wait_h) + g0 + q;
                            ready = wait_count_bounded(ctr, want, abort_word, p.timeout_ns) ? 1u : 0u;
                        }
                        fence_proxy_async_global();  // the rows are read next through TMA
                    }
                    if (!__shfl_sync(0xffffffffu, ready, lead)) {
                        ok = false;
                        break;
                    }
                }
                const bool swap = is_swap(info.z, p);
                int a_row = info.y + static_cast<int>(rank) * BM;
                int b_row = info.x * p.b_rows_per_expert + info.w + static_cast<int>(rank) * p.b_half_rows;
                uint32_t stage_tx = PTX_BYTES;
                const CUtensorMap* am = &tmA;
                if (swap) {
                    // weights into the A region (gemm1: 64 output columns per CTA,
                    // gemm2: 128), this CTA's N / 2 block rows into the B region
                    const int half_n = swap_n(info.z) >> 1;
                    const int bx = swap_box(half_n);
                    am = bx == 16 ? &tmA16 : bx == 32 ? &tmA32 : bx == 64 ? &tmA64 : &tmA;
                    a_row = info.y + static_cast<int>(rank) * half_n;
                    b_row = info.x * p.b_rows_per_expert + info.w +
                            static_cast<int>(rank) * (MODE == 0 ? BM / 2 : p.b_half_rows);
                    stage_tx = 2u * (PA_BYTES + static_cast<uint32_t>(bx) * BK * 2u);
                }
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!__all_sync(0xffffffffu, mbar_wait_bounded_cluster(smem_u32(&ctl->empty[stage]),
                                                                          phase ^ 1u, abort_word, p.timeout_ns))) {
                        ok = false;
                        break;
                    }
                    if (leader) {
                        const uint32_t fb = full0 + static_cast<uint32_t>(stage) * 8u;
                        const uint32_t sa = smem_u32(smem + stage * PSTAGE_BYTES);
                        const uint32_t sb = sa + PA_BYTES;
                        if (rank == 0) mbar_arrive_expect_tx(smem_u32(&ctl->full[stage]), stage_tx);
                        const bool stall = p.stall_first_stage && rank == 0 && cur_tile == 0 && kb == 0;
                        if (stall) {
                            // injected stall: the stage is armed but this CTA's half never comes
                        } else if (swap) {
                            if (MODE == 0) {
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    tma_load_2d_pair(sa + q * 32 * BK * 2, &tmB0q, kb * BK, b_row + 16 * q, fb);
                                    tma_load_2d_pair(sa + (q * 32 + 16) * BK * 2, &tmB1q, kb * BK, b_row + 16 * q, fb);
                                }
                            } else {
                                tma_load_2d_pair(sa, &tmB0, kb * BK, b_row, fb);
                            }
                            tma_load_2d_pair(sb, am, kb * BK, a_row, fb);
                        } else {
                            tma_load_2d_pair(sa, &tmA, kb * BK, a_row, fb);
                            tma_load_2d_pair(sb, mb, kb * BK, b_row, fb);
                        }
                    }
                    __syncwarp();
                    if (rank == 0) {
                        issued |= 1u << stage;
                        last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == PSTAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
            }
            if (p.pdl == 2) pdl_launch_dependents();  // no tile left to claim: the next kernel may launch
            if (leader) {
                if (!ok) {
                    raise_abort(ctl, peer);
                    report_error(p.status, MK_ERR_TIMEOUT, kSiteGemmProducer);
                }
                // CTA 0: every stage it armed completes (or times out) before the CTA exits.
                for (int s = 0; s < PSTAGES; ++s)
                    if ((issued >> s) & 1u)
                        mbar_wait_bounded_cluster(smem_u32(&ctl->full[s]), (last_par >> s) & 1u, never,
                                                  p.timeout_ns);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (rank == 0) {
            // ------------------------------------------------ MMA issuer (CTA 0 only)
            // The whole warp runs the loop and one elected lane issues the MMAs and
            // commits: a converged issuing warp keeps more MMAs queued ahead of
            // the tensor pipe than a lone diverged lane does.  Every wait result
            // is made warp-uniform before it is acted on.
            const bool leader = elect_one();
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0, slot = 0, slot_phase = 0;
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
                if (++slot == kPairSlots) {
                    slot = 0;
                    slot_phase ^= 1u;
                }
                if (info.x < 0) break;
                const uint32_t idesc = is_swap(info.z, p) ? idesc_bf16_f32(PAIR_M, swap_n(info.z)) : PIDESC;
                if (!__all_sync(0xffffffffu, mbar_wait_bounded_cluster(smem_u32(&ctl->tmem_empty[acc]),
                                                                      acc_phase ^ 1u, abort_word, p.timeout_ns))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * MMA_N;
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!__all_sync(0xffffffffu, mbar_wait_bounded_cluster(smem_u32(&ctl->full[stage]), phase,
                                                                          abort_word, p.timeout_ns))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (leader) {
                        const uint32_t sa = smem_u32(smem + stage * PSTAGE_BYTES);
                        const uint32_t sb = sa + PA_BYTES;
#pragma unroll
                        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                            const uint64_t ad = sw128_kmajor_desc(sa + kk * UMMA_K * 2);
                            const uint64_t bd = sw128_kmajor_desc(sb + kk * UMMA_K * 2);
                            mma_bf16_ss_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
                        }
                        mma_commit_pair_mc(smem_u32(&ctl->empty[stage]), 0x3);
                    }
                    __syncwarp();
                    if (++stage == PSTAGES) {
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
                    raise_abort(ctl, peer);
                    report_error(p.status, MK_ERR_TIMEOUT, kSiteGemmMma);
                }
                // All MMAs issued complete before either CTA frees TMEM or shared memory.
                mma_commit_pair_mc(smem_u32(&ctl->drain), 0x1);
                if (!mbar_wait_bounded_cluster(smem_u32(&ctl->drain), 0u, never, p.timeout_ns))
                    report_error(p.status, MK_ERR_TIMEOUT, kSiteGemmDrain);
            }
        }
        __syncwarp();
    } else if (warp == kSchedWarp) {
        const bool leader = elect_one();
        const int lead = __ffs(__ballot_sync(0xffffffffu, leader)) - 1;
        uint32_t slot = 0, slot_phase = 0;
        bool ok = true;
        if (rank == 0) {
            // ------------------------------------------------ tile scheduler (CTA 0)
            // Once a slot is free: claim the next tile (one atomic ticket), decode it and
            // write it into both CTAs' slot rings (the peer's through distributed shared
            // memory).  Kept off the producers so that neither pays the ticket's round trip
            // or a cluster-scope release between two tiles' loads.
            const uint32_t peer_slot0 = mapa_shared(smem_u32(&ctl->slot[0]), peer);
            const uint32_t peer_tile0 = mapa_shared(smem_u32(&ctl->slot_tile[0]), peer);
            const uint32_t peer_slot_full0 = mapa_shared(smem_u32(&ctl->slot_full[0]), peer);
            for (;;) {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded_cluster(smem_u32(&ctl->slot_empty[slot]),
                                                                      slot_phase ^ 1u, abort_word, p.timeout_ns))) {
                    ok = false;
                    break;
                }
                uint32_t tk = 0;
                if (leader) tk = atomicAdd(p.ticket, 1u);
                tk = __shfl_sync(0xffffffffu, tk, lead);
                const int tile = tk < static_cast<uint32_t>(total_tiles) ? static_cast<int>(tk) : -1;
                int4 nfo = make_int4(-1, 0, 0, 0);
                if (tile >= 0) {
                    const PairTile ti = decode_pair_tile(tile, ctl, p);
                    nfo = make_int4(ti.e, ti.row0, ti.rows, ti.n0);
                }
                if (leader) {
                    ctl->slot[slot] = nfo;
                    ctl->slot_tile[slot] = tile;
                    st_shared_cluster_v4(peer_slot0 + slot * static_cast<uint32_t>(sizeof(int4)), nfo);
                    st_shared_cluster_u32(peer_tile0 + slot * 4u, static_cast<uint32_t>(tile));
                    mbar_arrive(smem_u32(&ctl->slot_full[slot]));
                    mbar_arrive_cluster(peer_slot_full0 + slot * 8u);
                }
                __syncwarp();
                if (++slot == kPairSlots) {
                    slot = 0;
                    slot_phase ^= 1u;
                }
                if (tile < 0) break;
            }
        } else {
            // ------------------------------------------------ slot-release relay (CTA 1)
            // Once this CTA's producer and epilogue warps have read a slot, one arrive
            // (release at cluster scope, cumulative over theirs) frees it on CTA 0.
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
                if (++slot == kPairSlots) {
                    slot = 0;
                    slot_phase ^= 1u;
                }
                if (e < 0) break;
            }
        }
        if (!ok && leader) {
            raise_abort(ctl, peer);
            report_error(p.status, MK_ERR_TIMEOUT, kSiteGemmProducer);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- epilogue (both CTAs)
        const int sub = warp & 3;  // TMEM lanes [32*sub, 32*sub+32) are this warp's
        const int lane_in_tile = sub * 32 + lane;
        const uint32_t tmem_empty0 = mapa_shared(smem_u32(&ctl->tmem_empty[0]), 0);
        uint32_t acc = 0, acc_phase = 0, slot = 0, slot_phase = 0;
        bool ok = true;
        for (;;) {
            if (!mbar_wait_bounded_cluster(smem_u32(&ctl->slot_full[slot]), slot_phase, abort_word, p.timeout_ns)) {
                ok = false;
                break;
            }
            const int4 info = ctl->slot[slot];
            const int tile_index = ctl->slot_tile[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->slot_empty[slot]));
            if (++slot == kPairSlots) {
                slot = 0;
                slot_phase ^= 1u;
            }
            if (info.x < 0) break;
            if (!mbar_wait_bounded_cluster(smem_u32(&ctl->tmem_full[acc]), acc_phase, abort_word, p.timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) + acc * MMA_N;
            if (p.weight_rows != nullptr) {
                // the row weights were written by the dispatch with the rows: acquire the block's row counters
                const int g0 = sem_tile0(p.offsets, p.mtile_start, info.x, info.y);
                if (lane == 0)
                    for (int q = 0; q < (info.z > BM ? 2 : 1); ++q)
                        if (!wait_count_bounded(p.weight_rows + g0 + q, static_cast<uint32_t>(min(BM, info.z - q * BM)),
                                                abort_word, p.timeout_ns))
                            ok = false;
                __syncwarp();
                if (!__shfl_sync(0xffffffffu, ok ? 1u : 0u, 0)) break;
            }
            if (is_swap(info.z, p)) {
                bf16* oblock = p.out + static_cast<int64_t>(info.y) * p.out_ld;
                if (MODE == 0) {
                    const int col = info.w + static_cast<int>(rank) * (BM / 2) + sub * 16 + (lane & 15);
                    const bool c_ok = col < p.n_valid;
                    epilogue_swiglu_swap(tbase, info.z, oblock + (c_ok ? col : 0), p.out_ld, c_ok);
                } else {
                    const int n = info.w + static_cast<int>(rank) * (MMA_N / 2) + lane_in_tile;
                    const bool n_ok = n < p.n_valid;
                    epilogue_weighted_swap(tbase, info.z, oblock + (n_ok ? n : 0), p.out_ld, n_ok,
                                           p.row_weight != nullptr ? p.row_weight + info.y : nullptr);
                }
            } else {
                // full tile: TMEM lane = row of this CTA's 128
                const bool row_ok = static_cast<int>(rank) * BM + lane_in_tile < info.z;
                const int64_t r = static_cast<int64_t>(info.y) + static_cast<int>(rank) * BM + lane_in_tile;
                bf16* orow = p.out + (row_ok ? r : 0) * p.out_ld;
                if (MODE == 0) {
                    epilogue_swiglu(tbase, row_ok, orow, info.w, p.n_valid);
                } else {
                    const float wr = (row_ok && p.row_weight != nullptr) ? p.row_weight[r] : 1.0f;
                    // paced over ~80 % of a full tile's MMA cycles while more tiles follow
                    const bool more = tile_index + static_cast<int>(gridDim.x / 2) < total_tiles &&
                                      p.k_blocks < kEpiPaceMaxKb;
                    const uint32_t pace = more ? static_cast<uint32_t>(p.k_blocks) * kEpiPacePerKb : 0u;
                    epilogue_weighted(tbase, row_ok, orow, info.w, p.n_valid, wr, pace);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tmem_empty0 + acc * 8u);
            if (p.post != nullptr) {
                // publish this warp's rows: every lane's proxy fence (gemm2 reads h through TMA),
                // the warp barrier (orders the lanes' stores before lane 0's release increment,
                // which is cumulative over them), then one increment per M-tile the warp wrote
                // (a full tile: this CTA's M-tile; a swap tile: every M-tile of the block, since
                // each warp writes all of its rows)
                fence_proxy_async_global();
                __syncwarp();
                if (lane == 0) {
                    const int g0 = sem_tile0(p.offsets, p.mtile_start, info.x, info.y);
                    if (is_swap(info.z, p)) {
                        red_release_gpu_add(p.post + g0, 1u);
                        if (info.z > BM) red_release_gpu_add(p.post + g0 + 1, 1u);
                    } else {
                        red_release_gpu_add(p.post + g0 + static_cast<int>(rank), 1u);
                    }
                }
            }
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (!ok && lane == 0) {
            raise_abort(ctl, peer);
            report_error(p.status, MK_ERR_TIMEOUT, kSiteGemmEpilogue);
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // neither CTA leaves while the other may still use its shared memory
    if (*abort_word != 0u && threadIdx.x == 0) {
        // After a timeout, copies the peer started may still complete on CTA 0's
        // barriers: keep both CTAs resident a little longer (bounded) before exit.
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side

// The tensor maps of one launch.  a*: the activation rows (x_perm or h) in
// boxes of 128 / 16 / 32 / 64 rows; b0, b1: the weights in 128-row boxes
// (gemm1 W1, W3; gemm2 W2 twice); b0q, b1q: 16-row boxes (gemm1 swap tiles).
struct PairMaps {
    CUtensorMap a, b0, b1, a16, a32, a64, b0q, b1q;
};

template <int MODE>
cudaError_t launch_pair_mode(const PairMaps& m, const PairParams& p, int64_t S, cudaStream_t s) {
    static std::atomic<int> configured[64];    // per device: attributes set, max_clusters valid
    static std::atomic<int> max_clusters[64];  // written before `configured` (release / acquire)
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const int slot = dev < 64 ? dev : 0;
    auto fn = grouped_gemm_pair_kernel<MODE>;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(PNUM_THREADS);
    cfg.dynamicSmemBytes = PSMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
        err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(PSMEM_BYTES));
        if (err != cudaSuccess) return err;
        cfg.gridDim = dim3(2 * std::max(1, device_sm_count() / 2));
        int n = 0;
        err = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
        if (err != cudaSuccess) return err;
        if (n < 1) return cudaErrorInvalidConfiguration;
        max_clusters[slot].store(n, std::memory_order_relaxed);
        if (dev < 64) configured[dev].store(1, std::memory_order_release);
    }
    // Upper bound on the pair tiles: every expert adds at most one partial block.
    const int64_t max_tiles = ((S + PAIR_M - 1) / PAIR_M + p.E) * static_cast<int64_t>(p.n_tiles);
    const int64_t resident = max_clusters[slot].load(std::memory_order_relaxed);
    const int clusters = static_cast<int>(std::min<int64_t>(resident, std::max<int64_t>(max_tiles, 1)));
    cfg.gridDim = dim3(2 * clusters);
    LaunchCfg lc(cfg.gridDim, cfg.blockDim, PSMEM_BYTES, s, p.pdl != 0, 2);
    err = cudaLaunchKernelEx(&lc.cfg, fn, m.a, m.b0, m.b1, m.a16, m.a32, m.a64, m.b0q, m.b1q, p);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace

bool make_act_maps(PairMaps* m, const void* act, uint64_t inner, uint64_t rows) {
    return make_map(&m->a, act, inner, rows, BM) && make_map(&m->a16, act, inner, rows, 16) &&
           make_map(&m->a32, act, inner, rows, 32) && make_map(&m->a64, act, inner, rows, 64);
}

cudaError_t launch_gemm1_pair(const FfnArgs& a, cudaStream_t s) {
    PairMaps m;
    const uint64_t wrows = static_cast<uint64_t>(a.E) * a.f;
    if (!make_act_maps(&m, a.x_perm, a.d, a.S) || !make_map(&m.b0, a.w1, a.d, wrows, MMA_N / 2) ||
        !make_map(&m.b1, a.w3, a.d, wrows, MMA_N / 2) || !make_map(&m.b0q, a.w1, a.d, wrows, 16) ||
        !make_map(&m.b1q, a.w3, a.d, wrows, 16))
        return cudaErrorInvalidValue;
    PairParams p;
    p.offsets = a.offsets;
    p.mtile_start = a.mtile_start;
    p.row_weight = nullptr;
    p.out = a.h;
    p.out_ld = a.f;
    p.E = a.E;
    p.tile_n = MMA_N / 2;
    p.n_tiles = (a.f + p.tile_n - 1) / p.tile_n;
    p.n_valid = a.f;
    p.k_blocks = a.d / BK;
    p.b_rows_per_expert = a.f;
    p.b_half_rows = 0;  // full tiles: CTA 1 reads the same rows of W3 through its own map
    p.swap_max_rows = pair_swap_max_rows(1, p.k_blocks);
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    p.stall_first_stage = (a.inject == MK_INJECT_STALL_GEMM1) ? 1 : 0;
    p.ticket = a.tickets;
    p.wait_rows = a.sem.mt_rows;
    p.wait_h = nullptr;
    p.wait_ntiles = 0;
    p.wait_swap_max = 0;
    p.weight_rows = nullptr;
    p.post = a.sem.h_ready;
    p.pdl = a.sem.pdl ? 1 : 0;
    return launch_pair_mode<0>(m, p, a.S, s);
}

cudaError_t launch_gemm2_pair(const FfnArgs& a, cudaStream_t s) {
    PairMaps m;
    if (!make_act_maps(&m, a.h, a.f, a.S) || !make_map(&m.b0, a.w2, a.f, static_cast<uint64_t>(a.E) * a.d, MMA_N / 2))
        return cudaErrorInvalidValue;
    m.b1 = m.b0q = m.b1q = m.b0;  // unused by gemm2
    PairParams p;
    p.offsets = a.offsets;
    p.mtile_start = a.mtile_start;
    p.row_weight = a.row_weight;
    p.out = a.P;
    p.out_ld = a.d;
    p.E = a.E;
    p.tile_n = MMA_N;
    p.n_tiles = (a.d + p.tile_n - 1) / p.tile_n;
    p.n_valid = a.d;
    p.k_blocks = a.f / BK;
    p.b_rows_per_expert = a.d;
    p.b_half_rows = MMA_N / 2;
    p.swap_max_rows = kSwapMaxRows;
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    p.stall_first_stage = 0;
    p.ticket = a.tickets + 1;
    p.wait_rows = nullptr;
    p.wait_h = a.sem.h_ready;
    p.wait_ntiles = (a.f + MMA_N / 2 - 1) / (MMA_N / 2);
    p.wait_swap_max = pair_swap_max_rows(1, a.d / BK);
    p.weight_rows = a.sem.mt_rows;
    p.post = a.sem.p_ready;
    p.pdl = a.sem.pdl ? 2 : 0;
    return launch_pair_mode<1>(m, p, a.S, s);
}

// CTA pairs when experts hold 256 rows or more on average, single CTAs below:
// with a few rows per expert the layer streams weights from HBM and the pair
// tiles' extra rows cost more than the split operands save (same GPU,
// alternating builds: large -6%, skewed -6%, mid -3%, decode +5% on pairs).
bool use_pairs(const FfnArgs& a) { return a.S >= static_cast<int64_t>(PAIR_M) * a.E; }

int pair_swap_max_rows(int gemm, int k_blocks) {
    return (gemm == 1 && k_blocks < 64) ? kSwapMaxRowsShortK : kSwapMaxRows;
}

cudaError_t launch_gemm1_auto(const FfnArgs& a, cudaStream_t s) {
    return use_pairs(a) ? launch_gemm1_pair(a, s) : launch_gemm1(a, s);
}

cudaError_t launch_gemm2_auto(const FfnArgs& a, cudaStream_t s) {
    return use_pairs(a) ? launch_gemm2_pair(a, s) : launch_gemm2(a, s);
}

}  // namespace mk
