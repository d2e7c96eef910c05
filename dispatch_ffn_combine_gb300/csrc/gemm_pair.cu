// gemm_pair.cu -- grouped expert GEMMs on CTA pairs (tcgen05 cta_group::2).
//
// The same two GEMMs as the single-CTA kernels of gemm.cu (the expert FFN of
// the mKernel README's "MoE Dispatch + FFN + Combine" row: gemm1 -> SwiGLU ->
// gemm2), with each output tile computed by a cluster of two CTAs on two SMs:
//
//   pair tile   256 rows of one expert x 256 accumulator columns.  CTA r of
//               the pair holds rows [128 r, 128 r + 128) of A and half of the
//               256 B rows (gemm1: CTA 0 the 128 gate rows of W1, CTA 1 the
//               matching 128 up rows of W3; gemm2: W2 rows n0 + 128 r ...),
//               and receives its 128 rows x 256 columns of the accumulator in
//               its own TMEM.  One thread of CTA 0 issues the MMAs
//               (M = 256, N = 256, K = 16) for both SMs.
//   why         per SM and k-block, 32 KB of operands cross L2 and shared
//               memory instead of 48 KB (B is split, not duplicated), so six
//               pipeline stages fit in shared memory instead of four.
//   copies      each CTA loads its own A and B halves with TMA; all four
//               copies of a stage signal CTA 0's `full` barrier, which CTA 0
//               arms with the byte count of both CTAs.
//   release     the MMA thread's commits arrive on the `empty` barriers of both
//               CTAs (multicast), and on both CTAs' `tmem_full` barriers when
//               an accumulator is complete; the 8 epilogue warps (4 per CTA)
//               release an accumulator on CTA 0's `tmem_empty` barrier.
//   schedule    cluster c walks pair tiles c, c + C, ... of the list ordered
//               by (pair block, N block); a pair block is 256 rows of one
//               expert (the expert's last block may hold fewer valid rows;
//               rows past the expert's end are computed and not stored).
//
// Every wait is bounded.  A CTA whose wait runs out records MK_ERR_TIMEOUT,
// raises the abort word of both CTAs, and both drain and leave through the
// same cluster barrier, so neither exits while the other may still touch its
// shared memory.
#include <algorithm>

#include "gemm_impl.cuh"

namespace mk {
namespace {

using namespace gemm_detail;

constexpr int PSTAGES = 6;
constexpr int PAIR_M = 2 * BM;                          // rows per pair tile
constexpr uint32_t PA_BYTES = BM * BK * 2;              // this CTA's 128 A rows, one k-block
constexpr uint32_t PB_BYTES = (MMA_N / 2) * BK * 2;     // this CTA's 128 of the 256 B rows
constexpr uint32_t PSTAGE_BYTES = PA_BYTES + PB_BYTES;  // 32 KB
constexpr uint32_t PTX_BYTES = 2 * PSTAGE_BYTES;        // both CTAs' copies of one stage
constexpr uint32_t PIDESC = idesc_bf16_f32(PAIR_M, MMA_N);

struct PairCtl {
    uint64_t full[PSTAGES];   // CTA 0: both CTAs' copies of the stage landed
    uint64_t empty[PSTAGES];  // each CTA: the pair MMAs that read the stage are done
    uint64_t tmem_full[2];    // each CTA: accumulator complete
    uint64_t tmem_empty[2];   // CTA 0: all 8 epilogue warps have read the accumulator
    uint64_t drain;           // CTA 0: every MMA issued has completed
    uint32_t tmem_base;
    uint32_t abort_flag;
    uint32_t zero;
    int32_t off[kMaxExperts + 1];     // expert row offsets
    int32_t pstart[kMaxExperts + 1];  // prefix over experts of their pair blocks
};

constexpr size_t PSMEM_BYTES = static_cast<size_t>(PSTAGES) * PSTAGE_BYTES + sizeof(PairCtl) + 1024;

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
    int b_half_rows;    // row offset of CTA 1's half of B in its map (gemm1 0: own map; gemm2 128)
    uint32_t* status;
    uint64_t timeout_ns;
    int stall_first_stage;  // test hook: CTA 0 of cluster 0 never loads its first stage
};

struct PairTile {
    int e;
    int row0;  // first row of the pair block
    int rows;  // valid rows of the pair block (1..256)
    int n0;
};

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ PairTile decode_pair_tile(int tile, const PairCtl* ctl, const PairParams& p) {
    const int g = tile / p.n_tiles;
    const int nt = tile - g * p.n_tiles;
    int lo = 0, hi = p.E - 1;  // largest e with pstart[e] <= g
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ctl->pstart[mid] <= g)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int j = g - ctl->pstart[lo];
    const int off = ctl->off[lo];
    const int cnt = ctl->off[lo + 1] - off;
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
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                             const __grid_constant__ CUtensorMap tmB1, const PairParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    PairCtl* ctl = reinterpret_cast<PairCtl*>(smem + PSTAGES * PSTAGE_BYTES);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int cluster = static_cast<int>(cluster_id_x());
    const int nclusters = static_cast<int>(cluster_count_x());

    // Tile tables in shared memory: row offsets, and the pair-block prefix
    // (an expert with t 128-row tiles has ceil(t / 2) pair blocks).
    for (int i = threadIdx.x; i <= p.E; i += NUM_THREADS) ctl->off[i] = p.offsets[i];
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
        mbar_init(smem_u32(&ctl->drain), 1);
        ctl->abort_flag = 0;
        ctl->zero = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB0);
        if (MODE == 0) prefetch_tensormap(&tmB1);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&ctl->tmem_base), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers exist before any copy or commit targets them
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    volatile uint32_t* abort_word = &ctl->abort_flag;
    const volatile uint32_t* never = &ctl->zero;
    const int total_tiles = ctl->pstart[p.E] * p.n_tiles;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            const uint32_t full0 = mapa_shared(smem_u32(&ctl->full[0]), 0);
            const CUtensorMap* mb = (MODE == 0 && rank == 1) ? &tmB1 : &tmB0;
            uint32_t stage = 0, phase = 0, issued = 0, last_par = 0;
            bool ok = true;
            for (int tile = cluster; ok && tile < total_tiles; tile += nclusters) {
                const PairTile ti = decode_pair_tile(tile, ctl, p);
                const int a_row = ti.row0 + static_cast<int>(rank) * BM;
                const int b_row = ti.e * p.b_rows_per_expert + ti.n0 + static_cast<int>(rank) * p.b_half_rows;
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait_bounded_cluster(smem_u32(&ctl->empty[stage]), phase ^ 1u, abort_word,
                                                   p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full0 + static_cast<uint32_t>(stage) * 8u;
                    const uint32_t sa = smem_u32(smem + stage * PSTAGE_BYTES);
                    const uint32_t sb = sa + PA_BYTES;
                    if (rank == 0) {
                        mbar_arrive_expect_tx(smem_u32(&ctl->full[stage]), PTX_BYTES);
                        issued |= 1u << stage;
                        last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    }
                    const bool stall = p.stall_first_stage && rank == 0 && cluster == 0 && tile == cluster && kb == 0;
                    if (!stall) {  // injected stall: the stage is armed but this CTA's half never comes
                        tma_load_2d_pair(sa, &tmA, kb * BK, a_row, fb);
                        tma_load_2d_pair(sb, mb, kb * BK, b_row, fb);
                    }
                    if (++stage == PSTAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                raise_abort(ctl, peer);
                report_error(p.status, MK_ERR_TIMEOUT, kSiteGemmProducer);
            }
            // CTA 0: every stage it armed completes (or times out) before the CTA exits.
            for (int s = 0; s < PSTAGES; ++s)
                if ((issued >> s) & 1u)
                    mbar_wait_bounded_cluster(smem_u32(&ctl->full[s]), (last_par >> s) & 1u, never, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------------ MMA issuer (CTA 0 only)
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int tile = cluster; ok && tile < total_tiles; tile += nclusters) {
                if (!mbar_wait_bounded_cluster(smem_u32(&ctl->tmem_empty[acc]), acc_phase ^ 1u, abort_word,
                                               p.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * MMA_N;
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait_bounded_cluster(smem_u32(&ctl->full[stage]), phase, abort_word, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * PSTAGE_BYTES);
                    const uint32_t sb = sa + PA_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        const uint64_t ad = sw128_kmajor_desc(sa + kk * UMMA_K * 2);
                        const uint64_t bd = sw128_kmajor_desc(sb + kk * UMMA_K * 2);
                        mma_bf16_ss_pair(d_tmem, ad, bd, PIDESC, (kb | kk) != 0 ? 1u : 0u);
                    }
                    mma_commit_pair_mc(smem_u32(&ctl->empty[stage]), 0x3);
                    if (++stage == PSTAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit_pair_mc(smem_u32(&ctl->tmem_full[acc]), 0x3);
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok) {
                raise_abort(ctl, peer);
                report_error(p.status, MK_ERR_TIMEOUT, kSiteGemmMma);
            }
            // All MMAs issued complete before either CTA frees TMEM or shared memory.
            mma_commit_pair_mc(smem_u32(&ctl->drain), 0x1);
            if (!mbar_wait_bounded_cluster(smem_u32(&ctl->drain), 0u, never, p.timeout_ns))
                report_error(p.status, MK_ERR_TIMEOUT, kSiteGemmDrain);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- epilogue (both CTAs)
        const int sub = warp & 3;  // TMEM lanes [32*sub, 32*sub+32) are this warp's
        const int row_in_tile = sub * 32 + lane;
        const uint32_t tmem_empty0 = mapa_shared(smem_u32(&ctl->tmem_empty[0]), 0);
        uint32_t acc = 0, acc_phase = 0;
        bool ok = true;
        for (int tile = cluster; tile < total_tiles; tile += nclusters) {
            const PairTile ti = decode_pair_tile(tile, ctl, p);
            if (!mbar_wait_bounded_cluster(smem_u32(&ctl->tmem_full[acc]), acc_phase, abort_word, p.timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) + acc * MMA_N;
            const int my_rows = ti.rows - static_cast<int>(rank) * BM;
            const bool row_ok = row_in_tile < my_rows;
            const int64_t r = static_cast<int64_t>(ti.row0) + static_cast<int>(rank) * BM + row_in_tile;
            bf16* orow = p.out + (row_ok ? r : 0) * p.out_ld;
            if (MODE == 0) {
                epilogue_swiglu(tbase, row_ok, orow, ti.n0, p.n_valid);
            } else {
                const float wr = (row_ok && p.row_weight != nullptr) ? p.row_weight[r] : 1.0f;
                epilogue_weighted(tbase, row_ok, orow, ti.n0, p.n_valid, wr);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tmem_empty0 + acc * 8u);
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
        // After a timeout, CTA 1 may have copies in flight that signal CTA 0's
        // barriers: keep both resident a little longer (bounded) before exit.
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

template <int MODE>
cudaError_t launch_pair_mode(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                             const PairParams& p, int64_t S, cudaStream_t s) {
    static int configured[64] = {0};
    static int max_clusters[64] = {0};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    auto fn = grouped_gemm_pair_kernel<MODE>;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = PSMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dev >= 64 || !configured[dev]) {
        err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(PSMEM_BYTES));
        if (err != cudaSuccess) return err;
        cfg.gridDim = dim3(2 * std::max(1, device_sm_count() / 2));
        int n = 0;
        err = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
        if (err != cudaSuccess) return err;
        if (n < 1) return cudaErrorInvalidConfiguration;
        if (dev < 64) {
            max_clusters[dev] = n;
            configured[dev] = 1;
        } else {
            max_clusters[0] = n;
        }
    }
    const int cap = max_clusters[dev < 64 ? dev : 0];
    // Upper bound on the pair tiles: every expert adds at most one partial block.
    const int64_t max_tiles = ((S + PAIR_M - 1) / PAIR_M + p.E) * static_cast<int64_t>(p.n_tiles);
    const int clusters = static_cast<int>(std::min<int64_t>(cap, std::max<int64_t>(max_tiles, 1)));
    cfg.gridDim = dim3(2 * clusters);
    err = cudaLaunchKernelEx(&cfg, fn, a, b0, b1, p);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm1_pair(const FfnArgs& a, cudaStream_t s) {
    CUtensorMap ma, mb0, mb1;
    if (!make_map(&ma, a.x_perm, a.d, a.S, BM) ||
        !make_map(&mb0, a.w1, a.d, static_cast<uint64_t>(a.E) * a.f, MMA_N / 2) ||
        !make_map(&mb1, a.w3, a.d, static_cast<uint64_t>(a.E) * a.f, MMA_N / 2))
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
    p.b_half_rows = 0;  // CTA 1 reads the same rows of W3 through its own map
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    p.stall_first_stage = (a.inject == MK_INJECT_STALL_GEMM1) ? 1 : 0;
    return launch_pair_mode<0>(ma, mb0, mb1, p, a.S, s);
}

cudaError_t launch_gemm2_pair(const FfnArgs& a, cudaStream_t s) {
    CUtensorMap ma, mb0;
    if (!make_map(&ma, a.h, a.f, a.S, BM) ||
        !make_map(&mb0, a.w2, a.f, static_cast<uint64_t>(a.E) * a.d, MMA_N / 2))
        return cudaErrorInvalidValue;
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
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    p.stall_first_stage = 0;
    return launch_pair_mode<1>(ma, mb0, mb0, p, a.S, s);
}

// gemm2 on CTA pairs when experts hold 256 rows or more on average (pair
// tiles then carry little padding: on the large and skewed layer workloads
// this measured 2-7% faster than single-CTA tiles), else on single CTAs.
// gemm1 stays on single-CTA tiles: its longer K makes the padding of the
// 256-row pair blocks cost more than the pairing saves.
cudaError_t launch_gemm2_auto(const FfnArgs& a, cudaStream_t s) {
    return (a.S >= static_cast<int64_t>(PAIR_M) * a.E) ? launch_gemm2_pair(a, s) : launch_gemm2(a, s);
}

}  // namespace mk
