/*
 * mkmoe.h -- C ABI of the GB300 (sm_103a) fused mixture-of-experts layer.
 *
 * The layer is the one the mKernel README describes in its kernel table, row
 * "MoE Dispatch + FFN + Combine": tokens are routed to experts, each expert
 * runs its FFN (gemm1 -> SwiGLU -> gemm2), and the weighted expert outputs
 * are combined back into each token's row.  The mKernel paper ("mKernel: Fast
 * Multi-GPU, Multi-Node Fused Kernels", section 3 and Figure 2) runs such
 * layers as persistent kernels whose thread blocks take compute or
 * data-movement roles, with per-tile ready flags (section 4, "epoch-stamped
 * readiness flags").  On one GPU the expert-parallel exchanges become a
 * permutation inside HBM (dispatch) and a gather (combine).
 *
 * Conventions for every entry point:
 *   - Pointers to tensors are DEVICE pointers owned by the caller; the library
 *     keeps no reference after the call returns.  All tensors are row-major,
 *     contiguous, 16-byte aligned.  bf16 tensors are passed as void*.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     are asynchronous on that stream; the library allocates nothing per call.
 *   - `ws` is a caller-owned device workspace of at least
 *     mk_moe_workspace_size(...) bytes, 256-byte aligned.  One workspace per
 *     stream in flight: two calls that use one workspace concurrently race.
 *   - Argument errors are returned synchronously, before anything is enqueued.
 *     Errors found on the device (a bounded wait that ran out, an index out of
 *     range in caller-supplied routing) are recorded in the workspace and
 *     reported by mk_moe_last_device_error().  A failed CUDA launch returns
 *     MK_ERR_CUDA.
 *   - T == 0 is a valid no-op.
 *   - Limits: 1 <= E <= 256, 1 <= k <= min(E, 8), d and ffn multiples of 64,
 *     T * k < 2^31, T * k * max(d, ffn) < 2^40.
 *
 * Routing (the pages leave the router open; this is the reading used):
 *   logit[t,e] = sum_i x[t,i] * wg[e,i] (+ bias[e]) in fp32, in a fixed
 *   order: 32 interleaved partial sums s_j over i = j, j+32, ..., each a chain
 *   of correctly rounded fused multiply-adds, then the pairwise tree
 *   s_j += s_{j+off} for off = 16, 8, 4, 2, 1, then + bias[e].  The k largest
 *   logits are chosen, ties to the lower expert id; slot j holds the j-th
 *   largest.  weight_j = exp(l_j - l_0) / sum_j' exp(l_j' - l_0) (softmax over
 *   the chosen k, equal to the full softmax renormalised over the k).
 *   How it is computed (same bits either way): approximate logits with a
 *   rigorous-by-construction error interval come from the tensor cores; only
 *   experts whose interval reaches the k-th largest lower end are candidates,
 *   and only their logits are computed in the fixed order (see
 *   mk_moe_route_fallbacks for the safety net).
 */
#ifndef MKMOE_H
#define MKMOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MK_API __attribute__((visibility("default")))
#else
#define MK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MK_OK = 0,
    MK_ERR_INVALID_ARG = 1,   /* a size, pointer or alignment argument is invalid */
    MK_ERR_WORKSPACE = 2,     /* ws is NULL, misaligned or smaller than required */
    MK_ERR_UNSUPPORTED = 3,   /* valid request outside this build's limits, or no sm_103a device */
    MK_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
    MK_ERR_TIMEOUT = 5,       /* device: a bounded wait ran out (detail = wait site) */
    MK_ERR_BOUNDS = 6         /* device: caller-supplied routing out of range or repeated */
} mk_status;

/* Phases of mk_moe_layer, in launch order (indices into opts->phase_events). */
enum {
    MK_PHASE_ROUTE_LOGITS = 0, /* gate logits, fp32 fixed order                    */
    MK_PHASE_TOPK = 1,         /* top-k + softmax weights                          */
    MK_PHASE_COUNT = 2,        /* per-chunk expert histograms + ranks               */
    MK_PHASE_SCAN = 3,         /* expert offsets, chunk bases, M-tile table          */
    MK_PHASE_SCATTER = 4,      /* token rows -> expert-contiguous rows (dispatch)    */
    MK_PHASE_GEMM1 = 5,        /* grouped x W1^T, x W3^T, SwiGLU -> h                */
    MK_PHASE_GEMM2 = 6,        /* grouped h W2^T, scaled by the routing weight -> P  */
    MK_PHASE_COMBINE = 7,      /* y[t] = sum_j P[slot_row[t,j]] in j order           */
    MK_PHASE_COUNT_ALL = 8
};
/* On the fused and tile-synchronised paths (opts->path = MK_PATH_FUSED or MK_PATH_TILES) the steps
 * overlap: phase_events then gets event 0 before the kernels and events 1..MK_PHASE_COUNT_ALL after them. */

/* Optional per-call settings (pass NULL for defaults). */
typedef struct {
    uint64_t timeout_ns;   /* bound on each device-side wait; 0 = 2 s                       */
    void** phase_events;   /* NULL, or MK_PHASE_COUNT_ALL + 1 cudaEvent_t handles created by
                              the caller; event i is recorded on `stream` before phase i and
                              the last one after the final phase (for per-phase timing)      */
    int inject;            /* test hook, 0 = off.  MK_INJECT_STALL_GEMM1: in the first grouped
                              GEMM, the block that takes tile 0 announces one shared-memory
                              stage but never loads it, so its consumers' bounded waits run
                              out; the call then reports MK_ERR_TIMEOUT (no fault, no hang).
                              Kernel-per-step path only.                                     */
    int path;              /* MK_PATH_STEPS (0, default): one kernel per step, the faster
                              path on GB300 at every workload measured; MK_PATH_FUSED (1): one
                              persistent kernel whose blocks take mover or compute roles
                              (routing, counts and scans included; where the router's
                              tensor-core candidate filter applies -- T >= 2048 and
                              T d E >= 2^32 -- those run first as their own kernels and the
                              persistent kernel starts at the dispatch).
                              Both give bit-identical results.                              */
    int mover_ctas;        /* fused path: 0 = adaptive split (on-GPU controller, paper
                              section 3.2 Eq. 2); n > 0 = fixed split, blocks [0, n) prefer
                              mover tasks; -1 = no block prefers them (compute blocks still
                              help when their input is not ready)                            */
    int trace_cap;         /* fused path: records `trace` can hold (0 = no trace)            */
    uint32_t* trace;       /* fused path, device buffer of trace_cap * 8 words or NULL: one
                              record per task {block, kind, arg, tiles, start_lo, start_hi,
                              end_lo, end_hi} (%globaltimer ns); kinds 2 route, 3 dispatch,
                              5 combine, 6 GEMM session (tiles = tiles it ran, bit 31 set
                              when its first tile is a gemm2 tile).
                              min(trace_cap, tasks run) records are written; the task count
                              is left in the workspace (mk_moe_layer_trace_count).          */
    int gather_rows;       /* kernel-per-step path only, 0 = off: the dispatch writes only its
                              index tables (no copy of x into dispatched rows) and gemm1 loads
                              each tile's rows straight from x by their source tokens (TMA
                              gather4, four rows per copy, single-CTA tiles).  Same bits;
                              slower on GB300 (the gathers, not the MMAs, bound gemm1).     */
} mk_moe_opts;

#define MK_PATH_STEPS 0
#define MK_PATH_FUSED 1
#define MK_PATH_TILES 2  /* one kernel per step, each launched as a programmatic dependent of the one before
                            it, synchronised per 128-row tile of dispatched rows by data-tile semaphores in
                            the workspace (rows landed -> gemm1; h tile stored -> gemm2; P tile stored ->
                            the combine of its tokens), so each step starts on the tiles whose inputs are
                            ready; the MegaOps page's kernel-per-operator design with tile semaphores.
                            Same bits as the other paths.  Test hook: MK_INJECT_DROP_TILE_SIGNAL only.  */

#define MK_INJECT_STALL_GEMM1 1
#define MK_INJECT_DROP_TILE_SIGNAL 3  /* test hook, tile-synchronised path only: the dispatch never
                                         publishes token 0's rows, so the M-tiles holding them never
                                         complete; every wait on them runs out after timeout_ns and the
                                         call reports MK_ERR_TIMEOUT (no fault, no hang).            */
#define MK_INJECT_ROUTE_ZERO_BOUND 2  /* test hook: the router's candidate filter runs with a zero
                                         error bound, so (almost) every token takes the exact
                                         fallback (all E logits in the fixed order); the results
                                         are unchanged.  Kernel-per-step path only.          */

/* Bytes of workspace mk_moe_layer needs for these sizes (also enough for
 * mk_moe_route, mk_moe_dispatch and mk_moe_expert_ffn on the same sizes).
 * Returns 0 if the sizes are invalid. */
MK_API size_t mk_moe_workspace_size(int64_t T, int d, int E, int k, int ffn);

/* Router (routing step of the README's "MoE Dispatch + FFN + Combine" row).
 *   x        bf16 [T, d]            token activations
 *   wg       fp32 [E, d]            gate matrix
 *   bias     fp32 [E] or NULL       per-expert logit offset
 *   topk_ids int32 [T, k] (out)     chosen experts, slot order as above
 *   topk_w   fp32 [T, k] (out)      routing weights, sum to 1 per token
 *   expert_counts int32 [E] (out, may be NULL)  rows routed to each expert */
MK_API mk_status mk_moe_route(const void* x, const float* wg, const float* bias,
                       int64_t T, int d, int E, int k,
                       int32_t* topk_ids, float* topk_w, int32_t* expert_counts,
                       void* ws, size_t ws_bytes, void* stream);

/* The router without a workspace, for callers that cannot allocate device
 * memory (a runtime with a fixed memory plan, a path that may not call
 * cudaMalloc, a plug-in handed only its inputs and outputs).  The paper has no
 * counterpart; this is an addition of this library.  Same arguments, results
 * and slot order as mk_moe_route, minus ws.  Its fp32 logits live in a static
 * device array of 8 MiB that the library keeps on every GPU it runs on until
 * the process exits; T * E above 2,097,152 returns MK_ERR_UNSUPPORTED.  The
 * first call on a device looks up that array's device address, so make the
 * first call on each device before any stream capture.  All calls share the
 * array: calls that overlap on the GPU race.  Allocates nothing.  Its results
 * equal mk_moe_route's bit for bit (the same fixed-order logits, top-k and
 * softmax; it always computes every logit in the fixed order). */
MK_API mk_status mk_moe_route_noalloc(const void* x, const float* wg, const float* bias,
                                      int64_t T, int d, int E, int k,
                                      int32_t* topk_ids, float* topk_w, int32_t* expert_counts,
                                      void* stream);

/* Dispatch: permute token rows into expert-contiguous order (the local form of
 * the README's all-to-all dispatch; paper section 3.1 and Table 3 describe the
 * expert-parallel version that pulls tokens from peers).
 *   x, topk_ids [T,k], topk_w [T,k] (inputs; topk_w may be NULL)
 *   expert_offsets int32 [E+1] (out)  expert e owns rows [off[e], off[e+1])
 *   row_token      int32 [T*k] (out)  source token of each row; ascending within an expert
 *   row_weight     fp32  [T*k] (out, may be NULL)  routing weight of each row
 *   slot_row       int32 [T, k] (out) row that holds (token t, slot j)
 *   x_perm         bf16  [T*k, d] (out) x_perm[slot_row[t,j]] = x[t]
 * Ids outside [0, E) or repeated within a token set MK_ERR_BOUNDS on the device. */
MK_API mk_status mk_moe_dispatch(const void* x, const int32_t* topk_ids, const float* topk_w,
                          int64_t T, int d, int E, int k,
                          int32_t* expert_offsets, int32_t* row_token, float* row_weight,
                          int32_t* slot_row, void* x_perm,
                          void* ws, size_t ws_bytes, void* stream);

/* Grouped expert FFN on dispatched rows (README row: "gemm1 -> SwiGLU -> gemm2",
 * "weighted expert outputs"), on the tensor cores:
 *   h[r]  = bf16( silu(x_perm[r] W1_e^T) * (x_perm[r] W3_e^T) )   (fp32 accumulate)
 *   P[r]  = bf16( row_weight[r] * (h[r] W2_e^T) )                  (fp32 accumulate)
 * for every row r of expert e.
 *   x_perm bf16 [S, d]; expert_offsets int32 [E+1] with off[0] = 0, off[E] = S
 *   row_weight fp32 [S] or NULL (= 1)
 *   w1, w3 bf16 [E, ffn, d]; w2 bf16 [E, d, ffn]   (out x in)
 *   h bf16 [S, ffn] (out), P bf16 [S, d] (out) */
MK_API mk_status mk_moe_expert_ffn(const void* x_perm, const int32_t* expert_offsets, const float* row_weight,
                            const void* w1, const void* w3, const void* w2,
                            int64_t S, int d, int E, int ffn,
                            void* h, void* P,
                            void* ws, size_t ws_bytes, void* stream);

/* Grouped GEMM on dispatched rows: the compute half of the README's "MoE
 * Dispatch + GEMM" row ("runs the per-expert grouped GEMM"; paper section 4,
 * Table 3), on the tensor cores:
 *   out[r] = bf16( row_weight[r] * (x_perm[r] W_e^T) )   (fp32 accumulate)
 * for every row r of expert e.
 *   x_perm bf16 [S, d]; expert_offsets int32 [E+1] with off[0] = 0, off[E] = S
 *   row_weight fp32 [S] or NULL (= 1)
 *   w bf16 [E, n, d] (out x in), n a multiple of 64
 *   out bf16 [S, n] (out)
 *   ws: at least 256 + 4 (E + 1) bytes (control block and tile table).
 * Offsets that are not monotone or do not end at S set MK_ERR_BOUNDS on the
 * device and no row is computed. */
MK_API mk_status mk_moe_grouped_gemm(const void* x_perm, const int32_t* expert_offsets, const float* row_weight,
                              const void* w, int64_t S, int d, int E, int n, void* out,
                              void* ws, size_t ws_bytes, void* stream);

/* Combine (README row: "combines the weighted expert outputs back to each
 * token's source rank"; here: back to the token's row):
 *   y[t] = bf16( sum_{j=0..k-1} P[slot_row[t,j]] ), fp32 sum in ascending j.
 *   P bf16 [T*k, d]; slot_row int32 [T, k]; y bf16 [T, d] (out) */
MK_API mk_status mk_moe_combine(const void* P, const int32_t* slot_row, int64_t T, int d, int k,
                         void* y, void* stream);

/* The whole layer: route -> dispatch -> expert FFN -> combine.
 *   x bf16 [T,d]; wg fp32 [E,d]; bias fp32 [E] or NULL;
 *   w1, w3 bf16 [E,ffn,d]; w2 bf16 [E,d,ffn]; y bf16 [T,d] (out).
 *   opts may be NULL. */
MK_API mk_status mk_moe_layer(const void* x, const float* wg, const float* bias,
                       const void* w1, const void* w3, const void* w2,
                       int64_t T, int d, int E, int k, int ffn,
                       void* y, void* ws, size_t ws_bytes,
                       const mk_moe_opts* opts, void* stream);

/* Bytes of workspace mk_moe_dispatch_gemm needs for these sizes (the routing
 * tables and the dispatched rows; the layer's workspace for the same T, d, E,
 * k is larger and also serves).  Returns 0 if the sizes are invalid. */
MK_API size_t mk_moe_dispatch_gemm_workspace_size(int64_t T, int d, int E, int k);

/* MoE Dispatch + GEMM (README kernel table, row "MoE Dispatch + GEMM"; paper
 * section 4, Table 3, and section 5.3): routes the tokens, sends each
 * token's row to its k experts, and runs every expert's GEMM on the rows it
 * received:
 *   out[r] = bf16( x[row_token[r]] W_e^T )   for every row r of expert e,
 * with the routing, slot order and row order of mk_moe_route and
 * mk_moe_dispatch (on one GPU the exchange is the in-HBM permutation).  The
 * routing weight is not applied here (a later combine applies it); it is
 * returned per row.
 *   x bf16 [T, d]; wg fp32 [E, d]; bias fp32 [E] or NULL; w bf16 [E, n, d]
 *   out            bf16  [T*k, n] (out)  rows grouped by expert
 *   expert_offsets int32 [E+1]  (out)    expert e owns rows [off[e], off[e+1])
 *   row_token      int32 [T*k]  (out)    source token of each row
 *   row_weight     fp32  [T*k]  (out, may be NULL)  routing weight of each row
 *   ws: at least mk_moe_dispatch_gemm_workspace_size(T, d, E, k) bytes.
 * Limits as for the layer, with n in the role of ffn.  T == 0 only zeroes
 * expert_offsets (the other buffers are empty and may be NULL). */
MK_API mk_status mk_moe_dispatch_gemm(const void* x, const float* wg, const float* bias, const void* w,
                               int64_t T, int d, int E, int k, int n,
                               void* out, int32_t* expert_offsets, int32_t* row_token, float* row_weight,
                               void* ws, size_t ws_bytes, void* stream);

/* The layer on HOST buffers: copies x_host (T*d bf16, pinned for an
 * asynchronous copy) into a staging region of `ws`, runs mk_moe_layer, and
 * copies y back into y_host.  Weights stay on the device.  Asynchronous on
 * `stream`; the result is in y_host once the stream has reached this point.
 * On the kernel-per-step path the copies run on two copy streams the library
 * keeps per (device, workspace): the upload of x waits only until the
 * previous call on `ws` has read its staged x, so it overlaps that call's
 * GEMMs (a small kernel's loads when x_host is page-locked memory mapped for
 * the device).  If y_host is page-locked memory mapped for the device, the combine
 * writes y straight into it; otherwise y is combined and downloaded in token
 * chunks (~16 MB each, up to 8) while later chunks are still being combined.
 * The library
 * creates those streams and events on a workspace's first call (and keeps a
 * few sets); device memory is still only the caller's. */
MK_API mk_status mk_moe_layer_host(const void* x_host, const float* wg, const float* bias,
                            const void* w1, const void* w3, const void* w2,
                            int64_t T, int d, int E, int k, int ffn,
                            void* y_host, void* ws, size_t ws_bytes,
                            const mk_moe_opts* opts, void* stream);

/* The layer on HOST buffers for a stream of batches (same operation, inputs
 * and layouts as mk_moe_layer_host), with the output's download left off
 * `stream`: the combine writes y into a staging region of `ws`, a small
 * kernel on the workspace's copy stream stores it into y_host (page-locked
 * and mapped for the device: any cudaHostAlloc / pin_memory buffer; the copy
 * engine otherwise), and the event `y_ready` (a cudaEvent_t created by the
 * caller, passed as void*) is recorded there once y_host holds the output.
 * x's upload is likewise a small kernel's loads when x_host is page-locked
 * and mapped (the copy engine otherwise).  `stream` itself does not wait
 * for the download, so work enqueued on it after this call -- typically the
 * next batch's call on the same workspace -- runs while y is still crossing
 * the host link.  The caller waits for `y_ready` (cudaEventSynchronize, or
 * cudaStreamWaitEvent) before reading y_host, and does not overwrite y_host
 * before then.  x_host is read as for mk_moe_layer_host (its upload may start
 * before earlier work on `stream`; keep it unchanged until `y_ready`).
 * Consecutive calls on a workspace stage y in two alternating regions of it,
 * so a call's combine waits only for the download two calls back (a slow
 * download delays a later step less).  On the
 * fused and tile-synchronised paths the call runs as mk_moe_layer_host and
 * records `y_ready` on `stream`.  Errors as mk_moe_layer_host, plus
 * MK_ERR_INVALID_ARG for a NULL y_ready.  The paper has no host-buffer entry
 * point; this one is for serving loops that feed batches back to back. */
MK_API mk_status mk_moe_layer_host_async(const void* x_host, const float* wg, const float* bias,
                                  const void* w1, const void* w3, const void* w2,
                                  int64_t T, int d, int E, int k, int ffn,
                                  void* y_host, void* ws, size_t ws_bytes,
                                  const mk_moe_opts* opts, void* stream, void* y_ready);

/* Synchronises `stream`, then returns and clears the device-side status of
 * `ws` (MK_OK if no device error).  *detail (may be NULL) receives the site
 * code of the error.  Every call that runs kernels on `ws` starts from a
 * cleared status, so a call's device error is seen only until the next call
 * on `ws` is issued: read it in between. */
MK_API mk_status mk_moe_last_device_error(void* ws, void* stream, uint32_t* detail);

/* Router diagnostics: *count receives the number of tokens of the last router
 * run on `ws` (mk_moe_route, or mk_moe_layer on the kernel-per-step path)
 * whose logits were all computed in the fixed order because the tensor-core
 * candidate filter's error bound did not hold for one of them (expected 0;
 * the routing is exact either way).  Synchronises `stream`.  Returns
 * MK_ERR_WORKSPACE if ws is NULL. */
MK_API mk_status mk_moe_route_fallbacks(void* ws, void* stream, uint32_t* count);

/* Router diagnostics: copies the approximate logits (fp32 [T, E], bias added)
 * that the last run of the tensor-core candidate filter on `ws` left there --
 * mk_moe_route, mk_moe_dispatch_gemm, or mk_moe_layer when the filter applies
 * (T >= 2048 and T d E >= 2^32) -- into `out` (device, T * E floats),
 * asynchronously on `stream`.  Each lies within the filter's error bound of
 * the fixed-order logit.  Returns MK_ERR_WORKSPACE if ws is NULL. */
MK_API mk_status mk_moe_route_approx_logits(const void* ws, int64_t T, int d, int E, int k, float* out, void* stream);

/* Records the last fused mk_moe_layer call on `ws` wrote into its trace buffer
 * (synchronises `stream`).  Returns MK_ERR_WORKSPACE if ws is NULL. */
MK_API mk_status mk_moe_layer_trace_count(void* ws, int64_t T, int d, int E, int k, int ffn, void* stream,
                                          uint32_t* count);

/* Expert parallelism (README kernel table, row "MoE Dispatch + FFN + Combine":
 * tokens go "to their expert ranks" and the weighted outputs "back to each
 * token's source rank"; paper section 3.1 and Table 3).  Over G ranks, rank r
 * owns experts [r E_local, (r + 1) E_local).  After mk_moe_route and
 * mk_moe_dispatch a rank's rows are expert-contiguous, so the rows for rank q
 * are one contiguous range; the ranks exchange them (an all-to-all) and each
 * receives, from every source q, the rows of its local experts grouped by
 * expert: source-major order [q][e][rows].  mk_moe_ep_regroup moves rows
 * between that order and expert-major order [e][q][rows] (what
 * mk_moe_expert_ffn needs), and back (what the return all-to-all needs, so
 * that every source gets its rows in the order it sent them).
 *   rows_in, rows_out  device, `rows` rows of row_bytes bytes (a multiple of 4;
 *                      both 16-byte aligned), distinct buffers
 *   counts   int32 [G, E_local] (device): rows from source q for local expert e
 *   to_expert_major    1: source-major -> expert-major; 0: the inverse
 *   expert_offsets     int32 [E_local + 1] (out, device) or NULL: local expert e
 *                      owns expert-major rows [off[e], off[e+1]) -- the
 *                      offsets mk_moe_expert_ffn takes
 *   ws       at least mk_moe_ep_regroup_workspace_size(G, E_local) bytes,
 *            256-byte aligned (control block and offset tables)
 * Limits: G * E_local <= 2048, rows < 2^31 (rows == 0 writes only the offsets).  Counts below zero or summing to
 * anything but `rows` set MK_ERR_BOUNDS on the device (mk_moe_last_device_error
 * on ws); the rows are then copied unmoved.  A row keeps its position inside
 * its (source, expert) group, so the two directions are inverse permutations. */
MK_API size_t mk_moe_ep_regroup_workspace_size(int G, int E_local);
MK_API mk_status mk_moe_ep_regroup(const void* rows_in, void* rows_out, const int32_t* counts, int G, int E_local,
                                   int64_t rows, int row_bytes, int to_expert_major, int32_t* expert_offsets,
                                   void* ws, size_t ws_bytes, void* stream);

/* Regions of a layer workspace (mk_moe_workspace_size(T, d, E, k, ffn) bytes)
 * that mk_moe_layer leaves filled when its call has finished, for checks and
 * diagnostics; both paths fill the same regions with the same bits.
 *   MK_WS_IDS        int32 [T, k]    chosen experts, slot order
 *   MK_WS_W          fp32  [T, k]    routing weights
 *   MK_WS_OFFSETS    int32 [E + 1]   expert e owns rows [off[e], off[e+1])
 *   MK_WS_ROW_TOKEN  int32 [T * k]   source token of each dispatched row
 *   MK_WS_ROW_WEIGHT fp32  [T * k]   routing weight of each dispatched row
 *   MK_WS_SLOT_ROW   int32 [T, k]    row that holds (token t, slot j)
 *   MK_WS_X_PERM     bf16  [T * k, d]   dispatched token rows
 *   MK_WS_H          bf16  [T * k, ffn] SwiGLU activations
 *   MK_WS_P          bf16  [T * k, d]   weighted expert outputs (combined into y) */
typedef enum {
    MK_WS_IDS = 0,
    MK_WS_W = 1,
    MK_WS_OFFSETS = 2,
    MK_WS_ROW_TOKEN = 3,
    MK_WS_ROW_WEIGHT = 4,
    MK_WS_SLOT_ROW = 5,
    MK_WS_X_PERM = 6,
    MK_WS_H = 7,
    MK_WS_P = 8
} mk_ws_region;

/* Byte offset from the start of the workspace, and size in bytes, of `region`
 * for these sizes.  Host-only arithmetic (no GPU call).  Returns
 * MK_ERR_INVALID_ARG for invalid sizes, an unknown region or NULL outputs. */
MK_API mk_status mk_moe_workspace_region(int64_t T, int d, int E, int k, int ffn, int region, size_t* offset,
                                         size_t* bytes);

/* Static, human-readable name of a status code. */
MK_API const char* mk_moe_status_string(mk_status s);

/* Reads the internal routing tables that mk_moe_layer left in `ws`
 * (asynchronous device-to-device copies on `stream`; any pointer may be NULL):
 * topk_ids [T,k], topk_w [T,k], expert_offsets [E+1], slot_row [T,k]. */
MK_API mk_status mk_moe_layer_routing(const void* ws, int64_t T, int d, int E, int k, int ffn,
                               int32_t* topk_ids, float* topk_w, int32_t* expert_offsets,
                               int32_t* slot_row, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MKMOE_H */
