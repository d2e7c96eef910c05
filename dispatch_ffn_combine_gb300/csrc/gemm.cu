// gemm.cu -- grouped expert GEMMs on the 5th-generation tensor cores (tcgen05).
//
// The expert FFN of the layer (mKernel README, kernel table, row "MoE Dispatch
// + FFN + Combine": "runs the per-expert FFN (gemm1 -> SwiGLU -> gemm2)") as
// two persistent grouped GEMMs over the expert-contiguous rows:
//   gemm1:  acc = X_e [W1_e ; W3_e]^T  (one 128 x 256 MMA tile: 128 gate
//           columns and the matching 128 up columns), epilogue
//           h = bf16(silu(gate) * up)
//   gemm2:  acc = H_e W2_e^T (128 x 256 tile), epilogue
//           P = bf16(row_weight * acc)
// The paper builds its compute blocks from ThunderKittens tiles on Hopper
// (section 3); here the tile is GB300-native:
//   warp 0      TMA producer: box loads of A (128 x 64) and B (256 x 64) with
//               the 128-byte swizzle into a 4-stage shared-memory ring
//   warp 1      MMA issuer: one thread issues tcgen05.mma (bf16 in, fp32
//               accumulate in TMEM), commits free smem stages and full
//               accumulators to mbarriers
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (each warp owns the
//               32 TMEM lanes its warp index allows), fused SwiGLU or weight
//               scaling, bf16 stores of the valid rows
// Two 256-column accumulators (all 512 TMEM columns) let the epilogue of one
// tile overlap the main loop of the next.  A tile is (expert, 128-row block,
// N block), found from the per-expert tile prefix table with a binary search;
// rows past the expert's end are loaded (TMA fills past the tensor end with
// zeros) but never stored.
//   schedule  persistent CTAs claim tiles in list order, one atomic ticket
//             per tile (decode_tile gives the order: it keeps the readers of a
//             weight block and of a row block close together in time, so both
//             are served from L2).  The producer hands each claimed tile to the
//             MMA and epilogue roles through a small ring of tile slots in
//             shared memory.  Which CTA takes which tile never affects the
//             result.
// Every wait is bounded (see mk_device.cuh): on a timeout the CTA records
// MK_ERR_TIMEOUT, drains its own copies and MMAs, frees TMEM, returns.
#include <atomic>
#include "gemm_impl.cuh"

namespace mk {
namespace {

using namespace gemm_detail;


struct SharedCtl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t drain;
    uint64_t slot_full[4];   // tile slots: producer -> MMA issuer and epilogue
    uint64_t slot_empty[4];  // MMA thread + 4 epilogue warps release a slot
    int4 slot[4];            // {e, row0, rows, n0}; e < 0 ends the CTA's list
    uint32_t tmem_base;
    uint32_t abort_flag;
    uint32_t zero;
};

constexpr int kSlots = 4;

constexpr size_t SMEM_BYTES = static_cast<size_t>(STAGES) * STAGE_BYTES + sizeof(SharedCtl) + 1024;

struct GemmParams {
    const int32_t* offsets;      // [E+1]
    const int32_t* mtile_start;  // [E+1]
    const float* row_weight;     // gemm2 only, may be null
    bf16* out;
    int64_t out_ld;
    int E;
    int n_tiles;    // N blocks per 128-row block
    int tile_n;     // output columns per tile (128 gemm1, 256 gemm2)
    int n_valid;    // output columns of the whole GEMM
    int k_blocks;   // K / 64
    int b_rows_per_expert;
    uint32_t* status;
    uint64_t timeout_ns;
    int stall_first_stage;  // test hook: the CTA that claims tile 0 never loads its first stage
    uint32_t* ticket;       // a zeroed word: tiles claimed so far
    // Tile-synchronised path (all null / 0 otherwise): per-M-tile semaphores.
    const uint32_t* wait_rows;    // gemm1: rows the dispatch has landed per M-tile
    const uint32_t* wait_h;       // gemm2: gemm1 epilogue completions per M-tile (4 per N block)
    int wait_ntiles;              // gemm2: gemm1's N blocks
    const uint32_t* weight_rows;  // gemm2: the dispatch's row counters, acquired before row weights
    uint32_t* post;               // this GEMM's epilogue completions per M-tile
    int pdl;                      // 1: let the next kernel launch after the prologue; 2: once the tiles run out
    const int32_t* row_token;     // gemm1 reading x directly: source token of every dispatched row (else null)
};

struct TileInfo {
    int e;
    int row0;
    int rows;
    int n0;
};

// Tile t -> (expert, 128-row block, N block).  An expert's tiles occupy
// [mtile_start[e] * n_tiles, mtile_start[e + 1] * n_tiles); inside, they run
// in groups of kNGroup N blocks, each group over all of the expert's row
// blocks, N fastest:  (N group, row block, N block in group).  Tiles claimed
// one after another then share a weight block (read by the expert's row blocks
// within a few tile claims) and a row block (read by the group's N blocks
// back to back), so both are still in L2 when their next reader comes.
constexpr int kNGroup = 4;

__device__ __forceinline__ TileInfo decode_tile(int tile, const GemmParams& p) {
    const int g = tile / p.n_tiles;
    int lo = 0, hi = p.E - 1;  // largest e with mtile_start[e] <= g
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.mtile_start[mid] <= g)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int m_e = p.mtile_start[lo + 1] - p.mtile_start[lo];  // row blocks of the expert
    const int l = tile - p.mtile_start[lo] * p.n_tiles;
    const int q = l / (m_e * kNGroup);
    const int nb = min(kNGroup, p.n_tiles - q * kNGroup);  // N blocks in this group
    const int r = l - q * m_e * kNGroup;
    const int mt = r / nb;
    const int nt = q * kNGroup + (r - mt * nb);
    const int off = p.offsets[lo];
    const int cnt = p.offsets[lo + 1] - off;
    TileInfo ti;
    ti.e = lo;
    ti.row0 = off + mt * BM;
    ti.rows = min(BM, cnt - mt * BM);
    ti.n0 = nt * p.tile_n;
    return ti;
}

template <int MODE>  // 0: gemm1 + SwiGLU, 1: gemm2 + row weight
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                        const __grid_constant__ CUtensorMap tmB1, const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    SharedCtl* ctl = reinterpret_cast<SharedCtl*>(smem + STAGES * STAGE_BYTES);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int total_tiles = p.mtile_start[p.E] * p.n_tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&ctl->tmem_full[a]), 1);
            mbar_init(smem_u32(&ctl->tmem_empty[a]), 4);
        }
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(smem_u32(&ctl->slot_full[i]), 1);
            mbar_init(smem_u32(&ctl->slot_empty[i]), 5);
        }
        mbar_init(smem_u32(&ctl->drain), 1);
        ctl->abort_flag = 0;
        ctl->zero = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB0);
        if (MODE == 0) prefetch_tensormap(&tmB1);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (p.pdl == 1) pdl_launch_dependents();
    const uint32_t tmem_base = ctl->tmem_base;
    volatile uint32_t* abort_word = &ctl->abort_flag;
    const volatile uint32_t* never = &ctl->zero;

    if (warp == 0) {
        {
            // ------------------------------------------------ tile claims + TMA producer
            // whole warp; one elected lane claims, writes the slots and issues the copies
            const bool leader = elect_one();
            const int lead = __ffs(__ballot_sync(0xffffffffu, leader)) - 1;
            uint32_t stage = 0, phase = 0, issued = 0, last_par = 0, slot = 0, slot_phase = 0;
            bool ok = true;
            // One ticket per tile.  The elected lane takes the next ticket before this tile's
            // loads and the warp reads it (one shuffle) after them, so the atomic's
            // latency hides behind them.
            uint32_t tk = leader ? atomicAdd(p.ticket, 1u) : 0u;
            for (;;) {
                const uint32_t tkw = __shfl_sync(0xffffffffu, tk, lead);
                const int tile = tkw < static_cast<uint32_t>(total_tiles) ? static_cast<int>(tkw) : -1;
                int4 info = make_int4(-1, 0, 0, 0);
                TileInfo ti{};
                if (tile >= 0) {
                    ti = decode_tile(tile, p);
                    info = make_int4(ti.e, ti.row0, ti.rows, ti.n0);
                }
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&ctl->slot_empty[slot]), slot_phase ^ 1u,
                                                              abort_word, p.timeout_ns))) {
                    ok = false;
                    break;
                }
                if (leader) {
                    ctl->slot[slot] = info;
                    mbar_arrive(smem_u32(&ctl->slot_full[slot]));
                }
                if (++slot == kSlots) {
                    slot = 0;
                    slot_phase ^= 1u;
                }
                if (tile < 0) break;
                if (leader) tk = atomicAdd(p.ticket, 1u);
                if (p.wait_rows != nullptr || p.wait_h != nullptr) {
                    // tile-synchronised path: the M-tile's rows have landed (gemm1) or every gemm1
                    // tile of the M-tile has stored its h rows (gemm2)
                    uint32_t ready = 1u;
                    if (leader) {
                        const int g = sem_tile0(p.offsets, p.mtile_start, ti.e, ti.row0);
                        ready = p.wait_rows != nullptr
                                    ? wait_count_bounded(p.wait_rows + g, static_cast<uint32_t>(ti.rows), abort_word,
                                                         p.timeout_ns)
                                    : wait_count_bounded(p.wait_h + g, static_cast<uint32_t>(4 * p.wait_ntiles),
                                                         abort_word, p.timeout_ns);
                        fence_proxy_async_global();  // the rows are read next through TMA
                    }
                    if (!__shfl_sync(0xffffffffu, ready ? 1u : 0u, lead)) {
                        ok = false;
                        break;
                    }
                }
                const int b_row = ti.e * p.b_rows_per_expert + ti.n0;
                // gemm1 reading x directly: lane i gathers rows 4i .. 4i+3 of the tile by their
                // source tokens (rows past the expert's end reuse a valid token; never stored)
                int tok[4] = {0, 0, 0, 0};
                if (p.row_token != nullptr) {
                    const int first = p.row_token[ti.row0];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int r = 4 * lane + j;
                        tok[j] = (r < ti.rows) ? p.row_token[ti.row0 + r] : first;
                    }
                }
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&ctl->empty[stage]), phase ^ 1u,
                                                                  abort_word, p.timeout_ns))) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&ctl->full[stage]);
                    const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
                    if (p.row_token != nullptr) {
                        // the stage is armed (with its full byte count) before the gathers
                        if (leader) mbar_arrive_expect_tx(fb, STAGE_BYTES);
                        __syncwarp();
                        tma_gather4(sa + 512u * lane, &tmA, kb * BK, tok[0], tok[1], tok[2], tok[3], fb);
                    }
                    if (leader) {
                        const uint32_t sb = sa + A_BYTES;
                        if (p.row_token == nullptr) mbar_arrive_expect_tx(fb, STAGE_BYTES);
                        const bool stall = p.stall_first_stage && tile == 0 && kb == 0;
                        if (!stall) {  // injected stall: the stage is announced but never filled
                            if (p.row_token == nullptr) tma_load_2d(sa, &tmA, kb * BK, ti.row0, fb);
                            if (MODE == 0) {
                                tma_load_2d(sb, &tmB0, kb * BK, b_row, fb);
                                tma_load_2d(sb + B_BYTES / 2, &tmB1, kb * BK, b_row, fb);
                            } else {
                                tma_load_2d(sb, &tmB0, kb * BK, b_row, fb);
                            }
                        }
                    }
                    __syncwarp();
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
            }
            if (p.pdl == 2) pdl_launch_dependents();  // no tile left to claim: the next kernel may launch
            if (leader) {
                if (!ok) {
                    *abort_word = 1u;
                    report_error(p.status, MK_ERR_TIMEOUT, kSiteGemmProducer);
                }
                // Every copy this thread started must land before the CTA exits.
                for (int s = 0; s < STAGES; ++s)
                    if ((issued >> s) & 1u)
                        mbar_wait_bounded(smem_u32(&ctl->full[s]), (last_par >> s) & 1u, never, p.timeout_ns);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        {
            // ------------------------------------------------ MMA issuer
            // The whole warp runs the loop; one elected lane issues the MMAs and
            // commits (a converged issuing warp keeps the tensor pipe's queue
            // fuller than a lone lane); wait results are made warp-uniform.
            const bool leader = elect_one();
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0, slot = 0, slot_phase = 0;
            bool ok = true;
            for (;;) {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&ctl->slot_full[slot]), slot_phase,
                                                              abort_word, p.timeout_ns))) {
                    ok = false;
                    break;
                }
                const int tile_e = ctl->slot[slot].x;
                __syncwarp();
                if (leader) mbar_arrive(smem_u32(&ctl->slot_empty[slot]));
                if (++slot == kSlots) {
                    slot = 0;
                    slot_phase ^= 1u;
                }
                if (tile_e < 0) break;
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&ctl->tmem_empty[acc]), acc_phase ^ 1u,
                                                              abort_word, p.timeout_ns))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * MMA_N;
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait_bounded(smem_u32(&ctl->full[stage]), phase, abort_word, p.timeout_ns))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (leader) {
                        const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
                        const uint32_t sb = sa + A_BYTES;
#pragma unroll
                        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                            const uint64_t ad = sw128_kmajor_desc(sa + kk * UMMA_K * 2);
                            const uint64_t bd = sw128_kmajor_desc(sb + kk * UMMA_K * 2);
                            mma_bf16_ss(d_tmem, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
                        }
                        mma_commit(smem_u32(&ctl->empty[stage]));
                    }
                    __syncwarp();
                    if (++stage == STAGES) {
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
                    report_error(p.status, MK_ERR_TIMEOUT, kSiteGemmMma);
                }
                // All MMAs issued by this thread complete before TMEM is freed.
                mma_commit(smem_u32(&ctl->drain));
                if (!mbar_wait_bounded(smem_u32(&ctl->drain), 0u, never, p.timeout_ns))
                    report_error(p.status, MK_ERR_TIMEOUT, kSiteGemmDrain);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- epilogue
        const int sub = warp & 3;  // TMEM lanes [32*sub, 32*sub+32) are this warp's
        const int row_in_tile = sub * 32 + lane;
        uint32_t acc = 0, acc_phase = 0, slot = 0, slot_phase = 0;
        bool ok = true;
        for (;;) {
            if (!mbar_wait_bounded(smem_u32(&ctl->slot_full[slot]), slot_phase, abort_word, p.timeout_ns)) {
                ok = false;
                break;
            }
            const int4 info = ctl->slot[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->slot_empty[slot]));
            if (++slot == kSlots) {
                slot = 0;
                slot_phase ^= 1u;
            }
            if (info.x < 0) break;
            if (!mbar_wait_bounded(smem_u32(&ctl->tmem_full[acc]), acc_phase, abort_word, p.timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) + acc * MMA_N;
            if (p.weight_rows != nullptr) {
                // the row weights were written by the dispatch with the rows: acquire the M-tile's counter
                if (lane == 0 && !wait_count_bounded(p.weight_rows + sem_tile0(p.offsets, p.mtile_start, info.x, info.y),
                                                     static_cast<uint32_t>(info.z), abort_word, p.timeout_ns))
                    ok = false;
                __syncwarp();
                if (!__shfl_sync(0xffffffffu, ok ? 1u : 0u, 0)) break;
            }
            const bool row_ok = row_in_tile < info.z;
            const int64_t r = static_cast<int64_t>(info.y) + row_in_tile;
            bf16* orow = p.out + (row_ok ? r : 0) * p.out_ld;
            if (MODE == 0) {
                epilogue_swiglu(tbase, row_ok, orow, info.w, p.n_valid);
            } else {
                const float wr = (row_ok && p.row_weight != nullptr) ? p.row_weight[r] : 1.0f;
                epilogue_weighted(tbase, row_ok, orow, info.w, p.n_valid, wr);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->tmem_empty[acc]));
            if (p.post != nullptr) {
                // publish this warp's rows of the M-tile: every lane's proxy fence (gemm2 reads h
                // through TMA), the warp barrier, one release increment (cumulative over the
                // lanes' stores)
                fence_proxy_async_global();
                __syncwarp();
                if (lane == 0) red_release_gpu_add(p.post + sem_tile0(p.offsets, p.mtile_start, info.x, info.y), 1u);
            }
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (!ok && lane == 0) {
            *abort_word = 1u;
            report_error(p.status, MK_ERR_TIMEOUT, kSiteGemmEpilogue);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side

template <int MODE>
cudaError_t launch_mode(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1, const GemmParams& p,
                        int64_t S, cudaStream_t s) {
    static std::atomic<int> configured[64];  // per device: attributes set (repeating them is harmless)
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
        err = cudaFuncSetAttribute(grouped_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(SMEM_BYTES));
        if (err != cudaSuccess) return err;
        if (dev < 64) configured[dev].store(1, std::memory_order_release);
    }
    // Upper bound on the tile count: every expert adds at most one partial block.
    const int64_t max_tiles = ((S + BM - 1) / BM + p.E) * static_cast<int64_t>(p.n_tiles);
    const int grid = static_cast<int>(std::min<int64_t>(device_sm_count(), std::max<int64_t>(max_tiles, 1)));
    LaunchCfg lc(dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, s, p.pdl != 0);
    err = cudaLaunchKernelEx(&lc.cfg, grouped_gemm_kernel<MODE>, a, b0, b1, p);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm1(const FfnArgs& a, cudaStream_t s) {
    CUtensorMap ma, mb0, mb1;
    // A: the dispatched rows in 128-row boxes, or, reading x directly, x's rows one at a time (gather4)
    const bool gather = a.gather_x != nullptr;
    if (!(gather ? make_map(&ma, a.gather_x, a.d, static_cast<uint64_t>(a.gather_T), 1)
                 : make_map(&ma, a.x_perm, a.d, a.S, BM)) ||
        !make_map(&mb0, a.w1, a.d, static_cast<uint64_t>(a.E) * a.f, MMA_N / 2) ||
        !make_map(&mb1, a.w3, a.d, static_cast<uint64_t>(a.E) * a.f, MMA_N / 2))
        return cudaErrorInvalidValue;
    GemmParams p;
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
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    p.stall_first_stage = (a.inject == MK_INJECT_STALL_GEMM1) ? 1 : 0;
    p.ticket = a.tickets;
    p.wait_rows = a.sem.mt_rows;
    p.wait_h = nullptr;
    p.wait_ntiles = 0;
    p.weight_rows = nullptr;
    p.post = a.sem.h_ready;
    p.pdl = a.sem.pdl ? 1 : 0;
    p.row_token = gather ? a.row_token : nullptr;
    return launch_mode<0>(ma, mb0, mb1, p, a.S, s);
}

cudaError_t launch_gemm2(const FfnArgs& a, cudaStream_t s) {
    CUtensorMap ma, mb0;
    if (!make_map(&ma, a.h, a.f, a.S, BM) || !make_map(&mb0, a.w2, a.f, static_cast<uint64_t>(a.E) * a.d, MMA_N))
        return cudaErrorInvalidValue;
    GemmParams p;
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
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    p.stall_first_stage = 0;
    p.ticket = a.tickets + 1;
    p.wait_rows = nullptr;
    p.wait_h = a.sem.h_ready;
    p.wait_ntiles = (a.f + MMA_N / 2 - 1) / (MMA_N / 2);
    p.weight_rows = a.sem.mt_rows;
    p.post = a.sem.p_ready;
    p.pdl = a.sem.pdl ? 2 : 0;
    p.row_token = nullptr;
    return launch_mode<1>(ma, mb0, mb0, p, a.S, s);
}

}  // namespace mk
