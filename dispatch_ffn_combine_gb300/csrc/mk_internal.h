// mk_internal.h -- workspace layout and kernel launchers shared by the
// translation units of libmkmoe.so (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "mkmoe.h"

namespace mk {

using bf16 = __nv_bfloat16;

constexpr int kChunkTokens = 128;    // tokens per histogram chunk (dispatch)
constexpr int kTileM = 128;          // rows per grouped-GEMM tile
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s

// Device error sites (status[1]).
enum : uint32_t {
    kSiteGemmProducer = 0x100,
    kSiteGemmMma = 0x200,
    kSiteGemmEpilogue = 0x300,
    kSiteGemmDrain = 0x400,
    kSiteCountIds = 0x500,
    kSiteCountRepeat = 0x600,
    kSiteFusedIdle = 0x800,
    kSiteCombineWait = 0x900,
    kSiteRegroup = 0xA00,
};

// Byte offsets of every region of the caller's workspace.  The first 256
// bytes hold the control block: status[0] = first device error code,
// status[1] = its site.
struct WsLayout {
    size_t ctrl = 0;
    size_t logits = 0;        // fp32 [T, E]  gate logits (approximate ones on the candidate-filter path)
    size_t wsplit = 0;        // bf16 [E, 2d]  gate rows split in two bf16 parts, interleaved by 64 columns
    size_t wnorm = 0;         // fp32 [E]      gate row norms, rounded up
    size_t ids = 0;           // int32 [T, k]
    size_t w = 0;             // fp32 [T, k]
    size_t chunk_counts = 0;  // int32 [nchunks, E]
    size_t chunk_base = 0;    // int32 [nchunks, E]  rows of expert e before chunk c
    size_t rank = 0;          // int32 [T, k]        rank of (t, j) inside its chunk and expert
    size_t counts = 0;        // int32 [E]
    size_t offsets = 0;       // int32 [E + 1]
    size_t mtile_start = 0;   // int32 [E + 1]       prefix sum of ceil(count / 128)
    size_t row_token = 0;     // int32 [S]
    size_t row_weight = 0;    // fp32  [S]
    size_t slot_row = 0;      // int32 [S]
    size_t x_perm = 0;        // bf16  [S, d]
    size_t h = 0;             // bf16  [S, f]
    size_t P = 0;             // bf16  [S, d]
    size_t sync = 0;          // fused kernel: tickets, counters and ready flags (zeroed per call)
    size_t tile_sems = 0;     // tile-synchronised path: per-M-tile semaphores (zeroed per call)
    size_t x_stage = 0;       // bf16  [T, d]  host-buffer entry point: staged input
    size_t y_stage = 0;       // bf16  [T, d]  host-buffer entry point: staged output
    size_t y_stage2 = 0;      // bf16  [T, d]  pipelined host-buffer entry point: the second staged output
    size_t total = 0;
};

WsLayout ws_layout(int64_t T, int d, int E, int k, int f);
// The routing and dispatch part of the layout alone (the same offsets, up to
// and including x_perm): the workspace of the Dispatch + GEMM entry point.
WsLayout ws_layout_dispatch(int64_t T, int d, int E, int k);

inline int64_t num_chunks(int64_t T) { return (T + kChunkTokens - 1) / kChunkTokens; }

// Data-tile semaphores of the tile-synchronised path (MK_PATH_TILES): one
// counter per 128-row M-tile of the dispatched rows (the tile table's order),
// zeroed at the start of each call, raised with release semantics by the step
// that fills the tile and read with acquire semantics by the step that reads
// it.
//   mt_rows   rows the dispatch has written into the M-tile; complete at the
//             tile's row count, min(128, expert rows from the tile's first row)
//   h_ready   gemm1 epilogue warps done with the tile, one N block at a time;
//             complete at 4 per N block (8 for a CTA-pair swap tile, whose
//             eight epilogue warps each write every row of the block)
//   p_ready   the same for gemm2
//   tok_done  tokens whose dispatch (slot rows, row tokens, row weights and
//             rows) is written
struct TileSems {
    uint32_t* mt_rows = nullptr;
    uint32_t* h_ready = nullptr;
    uint32_t* p_ready = nullptr;
    uint32_t* tok_done = nullptr;
    bool pdl = false;  // the kernels are launched as programmatic dependents
    bool drop_token0 = false;  // test hook: the dispatch does not publish token 0's rows
};
// Counters per semaphore array: an upper bound on the M-tiles (every expert
// adds at most one partial tile).
inline int64_t tile_sem_units(int64_t S, int E) { return (S + kTileM - 1) / kTileM + E; }
inline size_t tile_sems_bytes(int64_t S, int E) { return 4 * static_cast<size_t>(3 * tile_sem_units(S, E) + 1); }
TileSems tile_sems_at(void* base, int64_t S, int E, bool pdl);

// cudaLaunchKernelEx configuration: `pdl` adds programmatic stream
// serialization (the kernel may be launched before the one ahead of it on the
// stream has finished), cluster_x > 1 a cluster dimension.
struct LaunchCfg {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[2]{};
    LaunchCfg(dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl, unsigned cluster_x = 1) {
        cfg.gridDim = grid;
        cfg.blockDim = block;
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        unsigned n = 0;
        if (cluster_x > 1) {
            attr[n].id = cudaLaunchAttributeClusterDimension;
            attr[n].val.clusterDim.x = cluster_x;
            attr[n].val.clusterDim.y = 1;
            attr[n].val.clusterDim.z = 1;
            ++n;
        }
        if (pdl) {
            attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[n].val.programmaticStreamSerializationAllowed = 1;
            ++n;
        }
        cfg.attrs = attr;
        cfg.numAttrs = n;
    }
};

// ----------------------------------------------------------------- launchers
// `pdl`: launched as a programmatic dependent (the kernel waits for the one
// ahead of it before reading anything, then lets the next one launch).
cudaError_t launch_route_logits(const bf16* x, const float* wg, const float* bias, int64_t T, int d, int E,
                                float* logits, cudaStream_t s, bool pdl = false);
// Router with the tensor-core candidate filter (route_tc.cu): approximate
// logits with an error bound, then the fixed-order fp32 logits of the
// candidates only, top-k and softmax.  Same outputs as launch_route_logits +
// launch_topk, bit for bit.
bool route_tc_supported(int d, int E);
cudaError_t launch_route_approx(const bf16* x, const float* wg, const float* bias, int64_t T, int d, int E,
                                float* approx, bf16* wsplit, float* wnorm, uint32_t* status, uint64_t timeout_ns,
                                cudaStream_t s, bool pdl = false);
cudaError_t launch_route_select(const bf16* x, const float* wg, const float* bias, int64_t T, int d, int E, int k,
                                const float* approx, const float* wnorm, int32_t* ids, float* w, int32_t* counts,
                                uint32_t* fallbacks, bool zero_bound, cudaStream_t s, bool pdl = false);
cudaError_t launch_topk(const float* logits, int64_t T, int E, int k, int32_t* ids, float* w,
                        int32_t* counts_or_null, cudaStream_t s, bool pdl = false);
cudaError_t launch_count(const int32_t* ids, int64_t T, int E, int k, int32_t* chunk_counts, int32_t* rank,
                         uint32_t* status, cudaStream_t s, bool pdl = false);
// `done`: a zeroed word (left zero again) that picks the last block for the expert scan.
cudaError_t launch_scan(const int32_t* chunk_counts, int64_t nchunks, int E, int32_t* chunk_base, int32_t* counts,
                        int32_t* offsets, int32_t* mtile_start, uint32_t* done, cudaStream_t s, bool pdl = false);
cudaError_t launch_scatter(const bf16* x, const int32_t* ids, const float* w, int64_t T, int d, int E, int k,
                           const int32_t* offsets, const int32_t* chunk_base, const int32_t* rank, bf16* x_perm,
                           int32_t* row_token, float* row_weight, int32_t* slot_row, cudaStream_t s,
                           const TileSems* sem = nullptr, const int32_t* mtile_start = nullptr,
                           bool copy_rows = true);
cudaError_t launch_mtile_table(const int32_t* offsets, int E, int64_t S, int32_t* mtile_start, uint32_t* status,
                               cudaStream_t s);
// y[t] = sum_j P[slot_row[t, j]] for t < T; p_rows = rows of P (-1: T * k).
// Copy `bytes` (a multiple of 16; both pointers 16-byte aligned) between
// device memory and mapped page-locked host memory with `blocks` CTAs of plain
// loads and stores.
cudaError_t launch_bulk_copy(const void* src, void* dst, size_t bytes, int blocks, cudaStream_t s);
cudaError_t launch_combine(const bf16* P, const int32_t* slot_row, int64_t T, int d, int k, bf16* y,
                           cudaStream_t s, int64_t p_rows = -1);

// The combine of the tile-synchronised path: token t's rows are summed once
// the dispatch has written its slot rows (tok_done) and gemm2 has published
// every M-tile they lie in (p_ready; `pairs`: gemm2 ran on CTA pairs with
// swap tiles of at most swap_max rows, n_tiles N blocks per tile).
cudaError_t launch_combine_sem(const bf16* P, const int32_t* slot_row, const int32_t* offsets,
                               const int32_t* mtile_start, int64_t T, int d, int E, int k, bf16* y,
                               const TileSems& sem, bool pairs, int n_tiles, int swap_max, uint32_t* status,
                               uint64_t timeout_ns, cudaStream_t s);

struct FfnArgs {
    const bf16* x_perm;
    const int32_t* offsets;      // [E+1]
    const int32_t* mtile_start;  // [E+1]
    const float* row_weight;     // [S] or null
    const bf16* w1;
    const bf16* w3;
    const bf16* w2;
    int64_t S;
    int d, E, f;
    bf16* h;
    bf16* P;
    uint32_t* status;
    uint64_t timeout_ns;
    int inject;                  // MK_INJECT_STALL_GEMM1 or 0
    uint32_t* tickets;           // 2 zeroed words: tile tickets of gemm1 [0] and gemm2 [1]
    TileSems sem{};              // tile-synchronised path only (default: none)
    // gemm1 reading its A rows straight from x (single-CTA kernel, TMA gather4):
    // x [gather_T, d] and the source token of every dispatched row; x_perm unused
    const bf16* gather_x = nullptr;
    int64_t gather_T = 0;
    const int32_t* row_token = nullptr;
};
// The pair kernels' swap-tile thresholds (gemm2's combine readiness needs it).
int pair_swap_max_rows(int gemm, int k_blocks);
bool use_pairs(const FfnArgs& a);
cudaError_t launch_gemm1(const FfnArgs& a, cudaStream_t s);
// The same GEMMs on CTA pairs (tcgen05 cta_group::2; gemm_pair.cu).
cudaError_t launch_gemm1_pair(const FfnArgs& a, cudaStream_t s);
cudaError_t launch_gemm2_pair(const FfnArgs& a, cudaStream_t s);
// Pairs when S >= 256 E (experts of 256+ rows on average), else single CTAs.
cudaError_t launch_gemm1_auto(const FfnArgs& a, cudaStream_t s);
cudaError_t launch_gemm2_auto(const FfnArgs& a, cudaStream_t s);

// Fused persistent kernel: tickets, role accounting and cost sums (followed in
// the workspace by the per-token-group, per-chunk and per-M-tile counters).
struct FusedSync {
    uint32_t route_head;      // next route task (mover queue, ready from the start)
    uint32_t index_head;      // next dispatch task (ready once the scans are done)
    uint32_t comb_head;       // next combine task (ready once every gemm2 quarter is published)
    uint32_t compute_head;    // next compute-queue ticket
    uint32_t movers_active;   // blocks in the mover role (adaptive mode)
    uint32_t target_movers;   // controller target (Eq. 2)
    uint32_t count_done;      // chunks counted
    uint32_t scan_done;       // scans finished (0/1)
    uint32_t index_done;      // dispatch chunks finished
    uint32_t p_done;          // gemm2 epilogue quarters finished
    uint32_t abort_flag;      // set by a block whose bounded wait ran out
    uint32_t ntask[2];        // finished tasks per role (mover, compute)
    uint32_t trace_n;         // trace records claimed
    uint32_t h_tiles;         // CTA-pair kernel: gemm1 epilogue warps finished, all pair blocks
    unsigned long long cyc[2];  // summed task cycles per role
};

struct FusedArgs {
    const bf16* x;
    const float* wg;
    const float* bias;
    const bf16* w1;
    const bf16* w3;
    const bf16* w2;
    int64_t T;
    int d, E, k, f;
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
    void* sync;
    int mover_ctas;   // 0 adaptive; > 0 fixed split; < 0 no block prefers mover tasks
    uint64_t timeout_ns;
    uint32_t* trace;  // optional task trace (8 words per record)
    int trace_cap;
    bool routed = false;  // ids, w, chunk_counts, rank and the scans are already computed
};
size_t fused_sync_bytes(int64_t T, int E, int k);
// The layer as one persistent kernel on CTA pairs (fused_pair.cu).
cudaError_t launch_fused_pair(const FusedArgs& a, cudaStream_t s);
cudaError_t launch_gemm2(const FfnArgs& a, cudaStream_t s);

// Argument checks every entry point shares: sizes within the limits the
// header states (MK_ERR_INVALID_ARG / MK_ERR_UNSUPPORTED), and 16-byte alignment.
mk_status check_sizes(int64_t T, int d, int E, int k, int f_or_64);
bool aligned16(const void* p);

int device_sm_count();      // SMs of the current device (cached per device)
bool device_is_sm103();     // current device is compute capability 10.3

}  // namespace mk
