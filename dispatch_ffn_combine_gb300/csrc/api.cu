// api.cu -- the C ABI (include/mkmoe.h): argument checks, workspace layout,
// and the launch sequence of the layer's steps on the caller's stream.
#include <atomic>
#include <algorithm>
#include <mutex>

#include "mk_internal.h"

namespace mk {

namespace {
constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }
}  // namespace

namespace {
// full: the layer's regions after x_perm (h, P, the fused kernel's flags, the
// host-buffer staging) are laid out too.
WsLayout make_layout(int64_t T, int d, int E, int k, int f, bool full) {
    WsLayout L;
    const size_t S = static_cast<size_t>(T) * k;
    const size_t nch = static_cast<size_t>(num_chunks(T));
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes);
        return at;
    };
    L.ctrl = take(256);
    L.logits = take(static_cast<size_t>(T) * E * 4);
    L.wsplit = take(static_cast<size_t>(E) * d * 4);
    L.wnorm = take(static_cast<size_t>(E) * 4);
    L.ids = take(S * 4);
    L.w = take(S * 4);
    L.chunk_counts = take(nch * E * 4);
    L.chunk_base = take(nch * E * 4);
    L.rank = take(S * 4);
    L.counts = take(static_cast<size_t>(E) * 4);
    L.offsets = take((static_cast<size_t>(E) + 1) * 4);
    L.mtile_start = take((static_cast<size_t>(E) + 1) * 4);
    L.row_token = take(S * 4);
    L.row_weight = take(S * 4);
    L.slot_row = take(S * 4);
    L.x_perm = take(S * d * 2);
    if (!full) {
        L.total = o;
        return L;
    }
    L.h = take(S * f * 2);
    L.P = take(S * d * 2);
    L.sync = take(fused_sync_bytes(T, E, k));
    L.tile_sems = take(tile_sems_bytes(static_cast<int64_t>(S), E));
    L.x_stage = take(static_cast<size_t>(T) * d * 2);
    L.y_stage = take(static_cast<size_t>(T) * d * 2);
    L.y_stage2 = take(static_cast<size_t>(T) * d * 2);
    L.total = o;
    return L;
}
}  // namespace

WsLayout ws_layout(int64_t T, int d, int E, int k, int f) { return make_layout(T, d, E, k, f, true); }

TileSems tile_sems_at(void* base, int64_t S, int E, bool pdl) {
    const int64_t n = tile_sem_units(S, E);
    uint32_t* w = static_cast<uint32_t*>(base);
    TileSems t;
    t.mt_rows = w;
    t.h_ready = w + n;
    t.p_ready = w + 2 * n;
    t.tok_done = w + 3 * n;
    t.pdl = pdl;
    return t;
}

WsLayout ws_layout_dispatch(int64_t T, int d, int E, int k) { return make_layout(T, d, E, k, 64, false); }

int device_sm_count() {
    static std::atomic<int> cache[64];  // per device, 0 until first read (a racing first read repeats the query)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 64) {
        int n = 1;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        return n;
    }
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        n = 1;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

bool device_is_sm103() {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return false;
    return major == 10 && minor == 3;
}

}  // namespace mk

using namespace mk;

namespace mk {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

mk_status check_sizes(int64_t T, int d, int E, int k, int f_or_64) {
    if (T < 0 || d <= 0 || E <= 0 || k <= 0 || f_or_64 <= 0) return MK_ERR_INVALID_ARG;
    if (E > kMaxExperts || k > kMaxTopK || k > E) return MK_ERR_INVALID_ARG;
    if (d % 64 != 0 || f_or_64 % 64 != 0) return MK_ERR_INVALID_ARG;
    if (T * k >= (int64_t(1) << 31)) return MK_ERR_UNSUPPORTED;
    if (T * static_cast<int64_t>(d) >= (int64_t(1) << 31)) return MK_ERR_UNSUPPORTED;
    if (T * k * static_cast<int64_t>(std::max(d, f_or_64)) >= (int64_t(1) << 40)) return MK_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(E) * std::max(d, f_or_64) >= (int64_t(1) << 31)) return MK_ERR_UNSUPPORTED;
    return MK_OK;
}

}  // namespace mk

namespace {

mk_status check_ws(const void* ws, size_t ws_bytes, const WsLayout& L) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < L.total) return MK_ERR_WORKSPACE;
    return MK_OK;
}

mk_status device_ok() { return device_is_sm103() ? MK_OK : MK_ERR_UNSUPPORTED; }

template <typename Tp>
Tp* at(void* ws, size_t off) {
    return reinterpret_cast<Tp*>(static_cast<uint8_t*>(ws) + off);
}

#define MK_TRY(expr)                                 \
    do {                                             \
        const cudaError_t _e = (expr);               \
        if (_e != cudaSuccess) return MK_ERR_CUDA;   \
    } while (0)

// out[r] = row_weight[r] * (x_perm[r] W_e^T): the second GEMM's kernel with
// K = d and N = n (gemm2 of the FFN is the case K = ffn, N = d).
cudaError_t launch_grouped_gemm(const bf16* x_perm, const int32_t* offsets, const int32_t* mtile,
                                const float* row_weight, const bf16* w, int64_t S, int d, int E, int n, bf16* out,
                                uint32_t* status, cudaStream_t s) {
    FfnArgs a{};
    a.offsets = offsets;
    a.mtile_start = mtile;
    a.row_weight = row_weight;
    a.h = const_cast<bf16*>(x_perm);  // the A operand; only read
    a.w2 = w;
    a.S = S;
    a.f = d;
    a.d = n;
    a.E = E;
    a.P = out;
    a.status = status;
    a.timeout_ns = kDefaultTimeoutNs;
    a.inject = 0;
    a.tickets = status + 4;
    return launch_gemm2_auto(a, s);
}

struct PhaseMarks {
    void** ev;
    cudaStream_t s;
    cudaError_t mark(int i) const {
        if (ev == nullptr || ev[i] == nullptr) return cudaSuccess;
        return cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), s);
    }
};

}  // namespace

extern "C" {

size_t mk_moe_workspace_size(int64_t T, int d, int E, int k, int ffn) {
    if (check_sizes(T, d, E, k, ffn) != MK_OK) return 0;
    return ws_layout(T, d, E, k, ffn).total;
}

const char* mk_moe_status_string(mk_status s) {
    switch (s) {
        case MK_OK: return "MK_OK";
        case MK_ERR_INVALID_ARG: return "MK_ERR_INVALID_ARG: invalid size, pointer or alignment";
        case MK_ERR_WORKSPACE: return "MK_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case MK_ERR_UNSUPPORTED: return "MK_ERR_UNSUPPORTED: outside this build's limits or not an sm_103 device";
        case MK_ERR_CUDA: return "MK_ERR_CUDA: a CUDA call or kernel launch failed";
        case MK_ERR_TIMEOUT: return "MK_ERR_TIMEOUT: a bounded device-side wait ran out";
        case MK_ERR_BOUNDS: return "MK_ERR_BOUNDS: routing index out of range or repeated";
    }
    return "unknown mk_status";
}

mk_status mk_moe_route(const void* x, const float* wg, const float* bias, int64_t T, int d, int E, int k,
                       int32_t* topk_ids, float* topk_w, int32_t* expert_counts, void* ws, size_t ws_bytes,
                       void* stream) {
    mk_status st = check_sizes(T, d, E, k, 64);
    if (st != MK_OK) return st;
    if (!x || !wg || !topk_ids || !topk_w) return MK_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(wg)) return MK_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, d, E, k, 64);
    if ((st = check_ws(ws, ws_bytes, L)) != MK_OK) return st;
    if (T == 0) {
        if (expert_counts) MK_TRY(cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * E, (cudaStream_t)stream));
        return MK_OK;
    }
    if ((st = device_ok()) != MK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    MK_TRY(cudaMemsetAsync(at<uint8_t>(ws, L.ctrl), 0, 12, s));  // status, site, router fallbacks
    float* logits = at<float>(ws, L.logits);
    if (expert_counts) MK_TRY(cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * E, s));
    const bf16* xb = static_cast<const bf16*>(x);
    if (route_tc_supported(d, E)) {
        MK_TRY(launch_route_approx(xb, wg, bias, T, d, E, logits, at<bf16>(ws, L.wsplit), at<float>(ws, L.wnorm),
                                   at<uint32_t>(ws, L.ctrl), kDefaultTimeoutNs, s));
        MK_TRY(launch_route_select(xb, wg, bias, T, d, E, k, logits, at<float>(ws, L.wnorm), topk_ids, topk_w,
                                   expert_counts, at<uint32_t>(ws, L.ctrl) + 2, false, s));
    } else {
        MK_TRY(launch_route_logits(xb, wg, bias, T, d, E, logits, s));
        MK_TRY(launch_topk(logits, T, E, k, topk_ids, topk_w, expert_counts, s));
    }
    return MK_OK;
}

mk_status mk_moe_dispatch(const void* x, const int32_t* topk_ids, const float* topk_w, int64_t T, int d, int E, int k,
                          int32_t* expert_offsets, int32_t* row_token, float* row_weight, int32_t* slot_row,
                          void* x_perm, void* ws, size_t ws_bytes, void* stream) {
    mk_status st = check_sizes(T, d, E, k, 64);
    if (st != MK_OK) return st;
    if (!x || !topk_ids || !expert_offsets || !row_token || !slot_row || !x_perm) return MK_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(x_perm)) return MK_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, d, E, k, 64);
    if ((st = check_ws(ws, ws_bytes, L)) != MK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        MK_TRY(cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (E + 1), s));
        return MK_OK;
    }
    if ((st = device_ok()) != MK_OK) return st;
    uint32_t* status = at<uint32_t>(ws, L.ctrl);
    MK_TRY(cudaMemsetAsync(status, 0, 8, s));       // status, site
    MK_TRY(cudaMemsetAsync(status + 3, 0, 4, s));   // scan ticket
    int32_t* chunk_counts = at<int32_t>(ws, L.chunk_counts);
    int32_t* chunk_base = at<int32_t>(ws, L.chunk_base);
    int32_t* rank = at<int32_t>(ws, L.rank);
    MK_TRY(launch_count(topk_ids, T, E, k, chunk_counts, rank, status, s));
    MK_TRY(launch_scan(chunk_counts, num_chunks(T), E, chunk_base, at<int32_t>(ws, L.counts), expert_offsets,
                       at<int32_t>(ws, L.mtile_start), status + 3, s));
    MK_TRY(launch_scatter(static_cast<const bf16*>(x), topk_ids, topk_w, T, d, E, k, expert_offsets, chunk_base, rank,
                          static_cast<bf16*>(x_perm), row_token, row_weight, slot_row, s));
    return MK_OK;
}

mk_status mk_moe_expert_ffn(const void* x_perm, const int32_t* expert_offsets, const float* row_weight, const void* w1,
                            const void* w3, const void* w2, int64_t S, int d, int E, int ffn, void* h, void* P,
                            void* ws, size_t ws_bytes, void* stream) {
    mk_status st = check_sizes(S, d, E, 1, ffn);
    if (st != MK_OK) return st;
    if (S == 0) return MK_OK;
    if (!x_perm || !expert_offsets || !w1 || !w3 || !w2 || !h || !P) return MK_ERR_INVALID_ARG;
    if (!aligned16(x_perm) || !aligned16(w1) || !aligned16(w3) || !aligned16(w2) || !aligned16(h) || !aligned16(P))
        return MK_ERR_INVALID_ARG;
    // Needs only the control block and the tile table that follows it.
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < 256 + 4 * (size_t(E) + 1))
        return MK_ERR_WORKSPACE;
    if (S == 0) return MK_OK;
    if ((st = device_ok()) != MK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t* status = at<uint32_t>(ws, 0);
    int32_t* mtile = at<int32_t>(ws, 256);
    MK_TRY(cudaMemsetAsync(status, 0, 8, s));          // status, site
    MK_TRY(cudaMemsetAsync(status + 4, 0, 16, s));     // GEMM tile tickets
    MK_TRY(launch_mtile_table(expert_offsets, E, S, mtile, status, s));
    FfnArgs a;
    a.x_perm = static_cast<const bf16*>(x_perm);
    a.offsets = expert_offsets;
    a.mtile_start = mtile;
    a.row_weight = row_weight;
    a.w1 = static_cast<const bf16*>(w1);
    a.w3 = static_cast<const bf16*>(w3);
    a.w2 = static_cast<const bf16*>(w2);
    a.S = S;
    a.d = d;
    a.E = E;
    a.f = ffn;
    a.h = static_cast<bf16*>(h);
    a.P = static_cast<bf16*>(P);
    a.status = status;
    a.timeout_ns = kDefaultTimeoutNs;
    a.inject = 0;
    a.tickets = status + 4;
    MK_TRY(launch_gemm1_auto(a, s));
    MK_TRY(launch_gemm2_auto(a, s));
    return MK_OK;
}

mk_status mk_moe_grouped_gemm(const void* x_perm, const int32_t* expert_offsets, const float* row_weight, const void* w,
                              int64_t S, int d, int E, int n, void* out, void* ws, size_t ws_bytes, void* stream) {
    mk_status st = check_sizes(S, d, E, 1, n);
    if (st != MK_OK) return st;
    if (S == 0) return MK_OK;
    if (!x_perm || !expert_offsets || !w || !out) return MK_ERR_INVALID_ARG;
    if (!aligned16(x_perm) || !aligned16(w) || !aligned16(out)) return MK_ERR_INVALID_ARG;
    // Needs only the control block and the tile table that follows it.
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < 256 + 4 * (size_t(E) + 1))
        return MK_ERR_WORKSPACE;
    if ((st = device_ok()) != MK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t* status = at<uint32_t>(ws, 0);
    int32_t* mtile = at<int32_t>(ws, 256);
    MK_TRY(cudaMemsetAsync(status, 0, 8, s));       // status, site
    MK_TRY(cudaMemsetAsync(status + 4, 0, 16, s));  // GEMM tile tickets
    MK_TRY(launch_mtile_table(expert_offsets, E, S, mtile, status, s));
    MK_TRY(launch_grouped_gemm(static_cast<const bf16*>(x_perm), expert_offsets, mtile, row_weight,
                               static_cast<const bf16*>(w), S, d, E, n, static_cast<bf16*>(out), status, s));
    return MK_OK;
}

mk_status mk_moe_combine(const void* P, const int32_t* slot_row, int64_t T, int d, int k, void* y, void* stream) {
    mk_status st = check_sizes(T, d, k, k, 64);
    if (st != MK_OK) return st;
    if (T == 0) return MK_OK;
    if (!P || !slot_row || !y) return MK_ERR_INVALID_ARG;
    if (!aligned16(P) || !aligned16(y)) return MK_ERR_INVALID_ARG;
    if (T == 0) return MK_OK;
    if ((st = device_ok()) != MK_OK) return st;
    MK_TRY(launch_combine(static_cast<const bf16*>(P), slot_row, T, d, k, static_cast<bf16*>(y),
                          static_cast<cudaStream_t>(stream)));
    return MK_OK;
}

}  // extern "C"

namespace {

// Hooks for the host-buffer entry point's pipelined copies (kernel-per-step path).
struct LayerHooks {
    cudaEvent_t after_scatter = nullptr;  // recorded once x has been read for the last time (scatter or gemm1)
    bool skip_combine = false;            // the caller runs the combine itself (in chunks)
};

// The candidate filter pays off once the fixed-order work (T d E fused
// multiply-adds) is large and there are enough 128-token tiles to fill the
// GPU; below that the plain fixed-order router is faster.  Same bits.
bool use_route_filter(int64_t T, int d, int E) {
    return route_tc_supported(d, E) && T >= 2048 && static_cast<double>(T) * d * E >= 4294967296.0;
}

// Where the dispatch step writes (the layer's workspace, or the caller's buffers).
struct DispatchOut {
    int32_t* offsets;    // [E+1]
    int32_t* row_token;  // [S]
    float* row_weight;   // [S]
    int32_t* slot_row;   // [T, k]
    bf16* x_perm;        // [S, d]
};

// Route, count, scan and scatter, one kernel each on `s`: the steps the layer
// and the Dispatch + GEMM entry point share.  The control block is zeroed by
// the caller.
mk_status route_dispatch_steps(const bf16* xb, const float* wg, const float* bias, int64_t T, int d, int E, int k,
                               void* ws, const WsLayout& L, const DispatchOut& o, const mk_moe_opts* opts,
                               const PhaseMarks& pm, cudaStream_t s) {
    uint32_t* status = at<uint32_t>(ws, L.ctrl);
    int32_t* ids = at<int32_t>(ws, L.ids);
    float* w = at<float>(ws, L.w);
    float* logits = at<float>(ws, L.logits);
    int32_t* chunk_counts = at<int32_t>(ws, L.chunk_counts);
    int32_t* chunk_base = at<int32_t>(ws, L.chunk_base);
    int32_t* rank = at<int32_t>(ws, L.rank);
    const uint64_t timeout_ns = (opts && opts->timeout_ns) ? opts->timeout_ns : kDefaultTimeoutNs;
    MK_TRY(pm.mark(MK_PHASE_ROUTE_LOGITS));
    if (use_route_filter(T, d, E) || (opts && opts->inject == MK_INJECT_ROUTE_ZERO_BOUND && route_tc_supported(d, E))) {
        MK_TRY(launch_route_approx(xb, wg, bias, T, d, E, logits, at<bf16>(ws, L.wsplit), at<float>(ws, L.wnorm),
                                   status, timeout_ns, s));
        MK_TRY(pm.mark(MK_PHASE_TOPK));
        MK_TRY(launch_route_select(xb, wg, bias, T, d, E, k, logits, at<float>(ws, L.wnorm), ids, w, nullptr,
                                   status + 2, opts && opts->inject == MK_INJECT_ROUTE_ZERO_BOUND, s));
    } else {
        MK_TRY(launch_route_logits(xb, wg, bias, T, d, E, logits, s));
        MK_TRY(pm.mark(MK_PHASE_TOPK));
        MK_TRY(launch_topk(logits, T, E, k, ids, w, nullptr, s));
    }
    MK_TRY(pm.mark(MK_PHASE_COUNT));
    MK_TRY(launch_count(ids, T, E, k, chunk_counts, rank, status, s));
    MK_TRY(pm.mark(MK_PHASE_SCAN));
    MK_TRY(launch_scan(chunk_counts, num_chunks(T), E, chunk_base, at<int32_t>(ws, L.counts), o.offsets,
                       at<int32_t>(ws, L.mtile_start), status + 3, s));
    MK_TRY(pm.mark(MK_PHASE_SCATTER));
    const bool gather = opts != nullptr && opts->gather_rows != 0;  // gemm1 reads x itself: no row copies
    MK_TRY(launch_scatter(xb, ids, w, T, d, E, k, o.offsets, chunk_base, rank, o.x_perm, o.row_token, o.row_weight,
                          o.slot_row, s, nullptr, nullptr, !gather));
    return MK_OK;
}

mk_status layer_impl(const void* x, const float* wg, const float* bias, const void* w1, const void* w3,
                     const void* w2, int64_t T, int d, int E, int k, int ffn, void* y, void* ws,
                     const WsLayout& L, const mk_moe_opts* opts, cudaStream_t s, const LayerHooks& hk) {
    const PhaseMarks pm{opts ? opts->phase_events : nullptr, s};
    uint32_t* status = at<uint32_t>(ws, L.ctrl);
    int32_t* ids = at<int32_t>(ws, L.ids);
    float* w = at<float>(ws, L.w);
    float* logits = at<float>(ws, L.logits);
    int32_t* chunk_counts = at<int32_t>(ws, L.chunk_counts);
    int32_t* chunk_base = at<int32_t>(ws, L.chunk_base);
    int32_t* rank = at<int32_t>(ws, L.rank);
    int32_t* offsets = at<int32_t>(ws, L.offsets);
    int32_t* mtile = at<int32_t>(ws, L.mtile_start);
    int32_t* slot_row = at<int32_t>(ws, L.slot_row);
    float* row_weight = at<float>(ws, L.row_weight);
    bf16* x_perm = at<bf16>(ws, L.x_perm);

    MK_TRY(cudaMemsetAsync(status, 0, 32, s));  // status, site, router fallbacks, scan ticket, GEMM tickets
    const bool fused = opts && opts->path == MK_PATH_FUSED && opts->inject == 0;
    if (fused) {
        FusedArgs fa;
        fa.x = static_cast<const bf16*>(x);
        fa.wg = wg;
        fa.bias = bias;
        fa.w1 = static_cast<const bf16*>(w1);
        fa.w3 = static_cast<const bf16*>(w3);
        fa.w2 = static_cast<const bf16*>(w2);
        fa.T = T;
        fa.d = d;
        fa.E = E;
        fa.k = k;
        fa.f = ffn;
        fa.logits = logits;
        fa.ids = ids;
        fa.w = w;
        fa.chunk_counts = chunk_counts;
        fa.chunk_base = chunk_base;
        fa.rank = rank;
        fa.counts = at<int32_t>(ws, L.counts);
        fa.offsets = offsets;
        fa.mtile_start = mtile;
        fa.row_token = at<int32_t>(ws, L.row_token);
        fa.row_weight = row_weight;
        fa.slot_row = slot_row;
        fa.x_perm = x_perm;
        fa.h = at<bf16>(ws, L.h);
        fa.P = at<bf16>(ws, L.P);
        fa.y = static_cast<bf16*>(y);
        fa.status = status;
        fa.sync = at<uint8_t>(ws, L.sync);
        fa.mover_ctas = opts ? opts->mover_ctas : 0;
        fa.trace = (opts && opts->trace_cap > 0) ? opts->trace : nullptr;
        fa.trace_cap = (opts && opts->trace) ? opts->trace_cap : 0;
        fa.timeout_ns = (opts && opts->timeout_ns) ? opts->timeout_ns : kDefaultTimeoutNs;
        MK_TRY(pm.mark(0));
        if (use_route_filter(T, d, E)) {
            // The persistent kernel's own router is the plain fixed-order one;
            // where the candidate filter is faster, the routing (and the
            // counts and scans that follow it) run first as their own kernels
            // and the persistent kernel starts at the dispatch.  Same bits.
            const bf16* xb = static_cast<const bf16*>(x);
            MK_TRY(launch_route_approx(xb, wg, bias, T, d, E, logits, at<bf16>(ws, L.wsplit), at<float>(ws, L.wnorm),
                                       status, fa.timeout_ns, s));
            MK_TRY(launch_route_select(xb, wg, bias, T, d, E, k, logits, at<float>(ws, L.wnorm), ids, w, nullptr,
                                       status + 2, false, s));
            MK_TRY(launch_count(ids, T, E, k, chunk_counts, rank, status, s));
            MK_TRY(launch_scan(chunk_counts, num_chunks(T), E, chunk_base, at<int32_t>(ws, L.counts), offsets, mtile,
                               status + 3, s));
            fa.routed = true;
        }
        MK_TRY(launch_fused_pair(fa, s));
        for (int i = 1; i <= MK_PHASE_COUNT_ALL; ++i) MK_TRY(pm.mark(i));
        return MK_OK;
    }
    if (opts && opts->path == MK_PATH_TILES) {
        // Kernel per step, each launched as a programmatic dependent of the one
        // before (it may start before that one has finished).  The routing
        // kernels wait for their predecessor to finish before reading; the
        // scatter, both GEMMs and the combine synchronise per 128-row M-tile
        // through the data-tile semaphores instead (rows landed -> gemm1;
        // every gemm1 N block of the tile stored -> gemm2; every gemm2 N block
        // -> the combine of the tile's tokens), so a step starts on the tiles
        // whose inputs are ready while the step before finishes the others.
        const int64_t S = T * k;
        const TileSems sem = tile_sems_at(at<uint8_t>(ws, L.tile_sems), S, E, true);
        MK_TRY(cudaMemsetAsync(at<uint8_t>(ws, L.tile_sems), 0, tile_sems_bytes(S, E), s));
        const bf16* xb = static_cast<const bf16*>(x);
        const uint64_t timeout_ns = (opts->timeout_ns) ? opts->timeout_ns : kDefaultTimeoutNs;
        MK_TRY(pm.mark(0));
        if (use_route_filter(T, d, E)) {
            MK_TRY(launch_route_approx(xb, wg, bias, T, d, E, logits, at<bf16>(ws, L.wsplit), at<float>(ws, L.wnorm),
                                       status, timeout_ns, s, true));
            MK_TRY(launch_route_select(xb, wg, bias, T, d, E, k, logits, at<float>(ws, L.wnorm), ids, w, nullptr,
                                       status + 2, false, s, true));
        } else {
            MK_TRY(launch_route_logits(xb, wg, bias, T, d, E, logits, s, false));
            MK_TRY(launch_topk(logits, T, E, k, ids, w, nullptr, s, true));
        }
        MK_TRY(launch_count(ids, T, E, k, chunk_counts, rank, status, s, true));
        MK_TRY(launch_scan(chunk_counts, num_chunks(T), E, chunk_base, at<int32_t>(ws, L.counts), offsets, mtile,
                           status + 3, s, true));
        TileSems scatter_sem = sem;
        scatter_sem.drop_token0 = opts->inject == MK_INJECT_DROP_TILE_SIGNAL;
        MK_TRY(launch_scatter(xb, ids, w, T, d, E, k, offsets, chunk_base, rank, x_perm, at<int32_t>(ws, L.row_token),
                              row_weight, slot_row, s, &scatter_sem, mtile));
        if (hk.after_scatter != nullptr) MK_TRY(cudaEventRecord(hk.after_scatter, s));
        FfnArgs a;
        a.x_perm = x_perm;
        a.offsets = offsets;
        a.mtile_start = mtile;
        a.row_weight = row_weight;
        a.w1 = static_cast<const bf16*>(w1);
        a.w3 = static_cast<const bf16*>(w3);
        a.w2 = static_cast<const bf16*>(w2);
        a.S = S;
        a.d = d;
        a.E = E;
        a.f = ffn;
        a.h = at<bf16>(ws, L.h);
        a.P = at<bf16>(ws, L.P);
        a.status = status;
        a.timeout_ns = timeout_ns;
        a.inject = 0;
        a.tickets = status + 4;
        a.sem = sem;
        MK_TRY(launch_gemm1_auto(a, s));
        MK_TRY(launch_gemm2_auto(a, s));
        if (!hk.skip_combine) {
            const bool pairs = use_pairs(a);
            MK_TRY(launch_combine_sem(a.P, slot_row, offsets, mtile, T, d, E, k, static_cast<bf16*>(y), sem, pairs,
                                      (d + 255) / 256, pair_swap_max_rows(2, ffn / 64), status, timeout_ns, s));
        }
        for (int i = 1; i <= MK_PHASE_COUNT_ALL; ++i) MK_TRY(pm.mark(i));
        return MK_OK;
    }
    const DispatchOut dout{offsets, at<int32_t>(ws, L.row_token), row_weight, slot_row, x_perm};
    mk_status st = route_dispatch_steps(static_cast<const bf16*>(x), wg, bias, T, d, E, k, ws, L, dout, opts, pm, s);
    if (st != MK_OK) return st;
    // x is read for the last time by the scatter, or by gemm1 when it gathers its rows from x
    const bool gather = opts != nullptr && opts->gather_rows != 0;
    if (hk.after_scatter != nullptr && !gather) MK_TRY(cudaEventRecord(hk.after_scatter, s));
    FfnArgs a;
    a.x_perm = x_perm;
    a.offsets = offsets;
    a.mtile_start = mtile;
    a.row_weight = row_weight;
    a.w1 = static_cast<const bf16*>(w1);
    a.w3 = static_cast<const bf16*>(w3);
    a.w2 = static_cast<const bf16*>(w2);
    a.S = T * k;
    a.d = d;
    a.E = E;
    a.f = ffn;
    a.h = at<bf16>(ws, L.h);
    a.P = at<bf16>(ws, L.P);
    a.status = status;
    a.timeout_ns = (opts && opts->timeout_ns) ? opts->timeout_ns : kDefaultTimeoutNs;
    a.inject = opts ? opts->inject : 0;  // only MK_INJECT_STALL_GEMM1 acts in the GEMMs
    a.tickets = status + 4;
    if (gather) {  // gemm1 gathers its rows from x by their source tokens (single-CTA tiles)
        a.gather_x = static_cast<const bf16*>(x);
        a.gather_T = T;
        a.row_token = at<int32_t>(ws, L.row_token);
    }
    MK_TRY(pm.mark(MK_PHASE_GEMM1));
    MK_TRY(gather ? launch_gemm1(a, s) : launch_gemm1_auto(a, s));
    if (hk.after_scatter != nullptr && gather) MK_TRY(cudaEventRecord(hk.after_scatter, s));
    MK_TRY(pm.mark(MK_PHASE_GEMM2));
    MK_TRY(gather ? launch_gemm2(a, s) : launch_gemm2_auto(a, s));
    MK_TRY(pm.mark(MK_PHASE_COMBINE));
    if (hk.skip_combine) return MK_OK;
    MK_TRY(launch_combine(a.P, slot_row, T, d, k, static_cast<bf16*>(y), s));
    MK_TRY(pm.mark(MK_PHASE_COUNT_ALL));
    return MK_OK;
}

mk_status validate_layer(const void* x, const float* wg, const void* w1, const void* w3, const void* w2, int64_t T,
                         int d, int E, int k, int ffn, const void* y, void* ws, size_t ws_bytes,
                         const mk_moe_opts* opts, bool device_xy) {
    mk_status st = check_sizes(T, d, E, k, ffn);
    if (st != MK_OK) return st;
    if (!x || !wg || !w1 || !w3 || !w2 || !y) return MK_ERR_INVALID_ARG;
    if (!aligned16(wg) || !aligned16(w1) || !aligned16(w3) || !aligned16(w2)) return MK_ERR_INVALID_ARG;
    if (device_xy && (!aligned16(x) || !aligned16(y))) return MK_ERR_INVALID_ARG;
    if (opts != nullptr) {
        if (opts->trace_cap < 0 || (opts->trace_cap > 0 && opts->trace == nullptr)) return MK_ERR_INVALID_ARG;
        if (opts->inject != 0 && opts->inject != MK_INJECT_STALL_GEMM1 && opts->inject != MK_INJECT_ROUTE_ZERO_BOUND &&
            opts->inject != MK_INJECT_DROP_TILE_SIGNAL)
            return MK_ERR_INVALID_ARG;
        if (opts->path != MK_PATH_FUSED && opts->path != MK_PATH_STEPS && opts->path != MK_PATH_TILES)
            return MK_ERR_INVALID_ARG;
        // the tile-synchronised path takes only its own hook, and that hook only that path
        if (opts->inject == MK_INJECT_DROP_TILE_SIGNAL && opts->path != MK_PATH_TILES) return MK_ERR_INVALID_ARG;
        if (opts->path == MK_PATH_TILES && opts->inject != 0 && opts->inject != MK_INJECT_DROP_TILE_SIGNAL)
            return MK_ERR_INVALID_ARG;
        if (opts->mover_ctas < -1) return MK_ERR_INVALID_ARG;
        if (opts->gather_rows != 0 && (opts->path != MK_PATH_STEPS || opts->inject != 0)) return MK_ERR_INVALID_ARG;
    }
    if ((st = check_ws(ws, ws_bytes, ws_layout(T, d, E, k, ffn))) != MK_OK) return st;
    return device_ok();
}

// Copy streams and events of the host-buffer entry point, one set per
// (device, workspace), created on first use and kept (a few sets, least
// recently used replaced after its copies have drained).
constexpr int kHostChunks = 8;
constexpr int kHostPipes = 8;
constexpr int kCopyOutCtas = 16;  // CTAs of the pipelined entry point's download kernel
constexpr int kCopyInCtas = 32;   // CTAs of the host entry points' upload kernel (its loads wait a link round trip)

// The device address of page-locked host memory mapped for the device, 16-byte
// aligned; null for any other pointer (pageable memory is not an error here).
const void* mapped_host_ptr(const void* p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) == cudaSuccess && a.type == cudaMemoryTypeHost && a.devicePointer != nullptr &&
        aligned16(a.devicePointer))
        return a.devicePointer;
    cudaGetLastError();
    return nullptr;
}

struct HostPipe {
    int dev = -1;
    const void* ws = nullptr;
    uint64_t used = 0;
    cudaStream_t h2d = nullptr, d2h[2] = {nullptr, nullptr};  // output chunks alternate between two copy streams
    cudaEvent_t x_free = nullptr;               // the last read of the staged x (after the scatter)
    cudaEvent_t x_ready = nullptr;              // staged x uploaded
    cudaEvent_t y_ready[kHostChunks] = {};      // combine of output chunk c done
    cudaEvent_t y_done[kHostChunks] = {};       // download of output chunk c done
    uint32_t async_calls = 0;                   // pipelined calls so far: they alternate two staging regions
    cudaEvent_t y_async_done[2] = {};           // download of the last pipelined call from region r done
};

std::mutex g_pipe_mu;
HostPipe g_pipes[kHostPipes];
uint64_t g_pipe_clock = 0;

void release_pipe(HostPipe& p) {
    // The workspace's last call may still run on the caller's stream: wait for
    // every event it recorded there (a no-op once complete or never recorded),
    // so that a later call on this workspace, which gets a new pipe whose events
    // order nothing yet, cannot overwrite its staged x or y under it.
    for (cudaEvent_t e : {p.x_free, p.x_ready})
        if (e) cudaEventSynchronize(e);
    for (int c = 0; c < kHostChunks; ++c) {
        if (p.y_ready[c]) cudaEventSynchronize(p.y_ready[c]);
        if (p.y_done[c]) cudaEventSynchronize(p.y_done[c]);
    }
    for (cudaEvent_t e : p.y_async_done)
        if (e) cudaEventSynchronize(e);
    if (p.h2d) cudaStreamSynchronize(p.h2d);
    for (cudaStream_t q : p.d2h)
        if (q) cudaStreamSynchronize(q);
    cudaEvent_t* evs[] = {&p.x_free, &p.x_ready};
    for (cudaEvent_t* e : evs)
        if (*e) cudaEventDestroy(*e);
    for (int c = 0; c < kHostChunks; ++c) {
        if (p.y_ready[c]) cudaEventDestroy(p.y_ready[c]);
        if (p.y_done[c]) cudaEventDestroy(p.y_done[c]);
    }
    for (cudaEvent_t e : p.y_async_done)
        if (e) cudaEventDestroy(e);
    if (p.h2d) cudaStreamDestroy(p.h2d);
    for (cudaStream_t q : p.d2h)
        if (q) cudaStreamDestroy(q);
    p = HostPipe{};
}

cudaError_t get_pipe(const void* ws, HostPipe** out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    HostPipe* victim = &g_pipes[0];
    for (HostPipe& p : g_pipes) {
        if (p.dev == dev && p.ws == ws) {
            p.used = ++g_pipe_clock;
            *out = &p;
            return cudaSuccess;
        }
        if (p.used < victim->used) victim = &p;
    }
    release_pipe(*victim);
    HostPipe& p = *victim;
    const unsigned ef = cudaEventDisableTiming;
    if ((err = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking)) != cudaSuccess) return err;
    for (cudaStream_t& q : p.d2h)
        if ((err = cudaStreamCreateWithFlags(&q, cudaStreamNonBlocking)) != cudaSuccess) return err;
    if ((err = cudaEventCreateWithFlags(&p.x_free, ef)) != cudaSuccess) return err;
    if ((err = cudaEventCreateWithFlags(&p.x_ready, ef)) != cudaSuccess) return err;
    for (int c = 0; c < kHostChunks; ++c) {
        if ((err = cudaEventCreateWithFlags(&p.y_ready[c], ef)) != cudaSuccess) return err;
        if ((err = cudaEventCreateWithFlags(&p.y_done[c], ef)) != cudaSuccess) return err;
    }
    for (cudaEvent_t& e : p.y_async_done)
        if ((err = cudaEventCreateWithFlags(&e, ef)) != cudaSuccess) return err;
    p.dev = dev;
    p.ws = ws;
    p.used = ++g_pipe_clock;
    *out = &p;
    return cudaSuccess;
}

}  // namespace

extern "C" {

mk_status mk_moe_layer(const void* x, const float* wg, const float* bias, const void* w1, const void* w3,
                       const void* w2, int64_t T, int d, int E, int k, int ffn, void* y, void* ws, size_t ws_bytes,
                       const mk_moe_opts* opts, void* stream) {
    if (T == 0 && check_sizes(T, d, E, k, ffn) == MK_OK) return MK_OK;  // empty batch: nothing to read or write
    mk_status st = validate_layer(x, wg, w1, w3, w2, T, d, E, k, ffn, y, ws, ws_bytes, opts, true);
    if (st != MK_OK) return st;
    return layer_impl(x, wg, bias, w1, w3, w2, T, d, E, k, ffn, y, ws, ws_layout(T, d, E, k, ffn), opts,
                      static_cast<cudaStream_t>(stream), LayerHooks{});
}

size_t mk_moe_dispatch_gemm_workspace_size(int64_t T, int d, int E, int k) {
    if (check_sizes(T, d, E, k, 64) != MK_OK) return 0;
    return ws_layout_dispatch(T, d, E, k).total;
}

mk_status mk_moe_dispatch_gemm(const void* x, const float* wg, const float* bias, const void* w, int64_t T, int d,
                               int E, int k, int n, void* out, int32_t* expert_offsets, int32_t* row_token,
                               float* row_weight, void* ws, size_t ws_bytes, void* stream) {
    mk_status st = check_sizes(T, d, E, k, n);
    if (st != MK_OK) return st;
    const WsLayout L = ws_layout_dispatch(T, d, E, k);
    if ((st = check_ws(ws, ws_bytes, L)) != MK_OK) return st;
    if (!expert_offsets) return MK_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {  // x, out and row_token are empty (and may be NULL)
        MK_TRY(cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (E + 1), s));
        return MK_OK;
    }
    if (!x || !wg || !w || !out || !row_token) return MK_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(wg) || !aligned16(w) || !aligned16(out)) return MK_ERR_INVALID_ARG;
    if ((st = device_ok()) != MK_OK) return st;
    uint32_t* status = at<uint32_t>(ws, L.ctrl);
    MK_TRY(cudaMemsetAsync(status, 0, 32, s));  // status, site, router fallbacks, scan ticket, GEMM tickets
    const DispatchOut dout{expert_offsets, row_token, row_weight, at<int32_t>(ws, L.slot_row), at<bf16>(ws, L.x_perm)};
    const PhaseMarks pm{nullptr, s};
    st = route_dispatch_steps(static_cast<const bf16*>(x), wg, bias, T, d, E, k, ws, L, dout, nullptr, pm, s);
    if (st != MK_OK) return st;
    MK_TRY(launch_grouped_gemm(dout.x_perm, expert_offsets, at<int32_t>(ws, L.mtile_start), nullptr,
                               static_cast<const bf16*>(w), T * k, d, E, n, static_cast<bf16*>(out), status, s));
    return MK_OK;
}

mk_status mk_moe_layer_host(const void* x_host, const float* wg, const float* bias, const void* w1, const void* w3,
                            const void* w2, int64_t T, int d, int E, int k, int ffn, void* y_host, void* ws,
                            size_t ws_bytes, const mk_moe_opts* opts, void* stream) {
    if (T == 0 && check_sizes(T, d, E, k, ffn) == MK_OK) return MK_OK;
    mk_status st = validate_layer(x_host, wg, w1, w3, w2, T, d, E, k, ffn, y_host, ws, ws_bytes, opts, false);
    if (st != MK_OK) return st;
    const WsLayout L = ws_layout(T, d, E, k, ffn);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t bytes = static_cast<size_t>(T) * d * 2;
    bf16* xd = at<bf16>(ws, L.x_stage);
    bf16* yd = at<bf16>(ws, L.y_stage);
    HostPipe* hp = nullptr;
    MK_TRY(get_pipe(ws, &hp));
    if (opts && opts->path == MK_PATH_FUSED) {
        // plain sequence around the persistent kernel, ordered after any
        // earlier call's use of the staging buffers and before any later one
        MK_TRY(cudaStreamWaitEvent(s, hp->x_free, 0));
        for (int c = 0; c < kHostChunks; ++c) MK_TRY(cudaStreamWaitEvent(s, hp->y_done[c], 0));
        MK_TRY(cudaStreamWaitEvent(s, hp->y_async_done[0], 0));
        MK_TRY(cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, s));
        st = layer_impl(xd, wg, bias, w1, w3, w2, T, d, E, k, ffn, yd, ws, L, opts, s, LayerHooks{});
        if (st != MK_OK) return st;
        MK_TRY(cudaEventRecord(hp->x_free, s));
        MK_TRY(cudaMemcpyAsync(y_host, yd, bytes, cudaMemcpyDeviceToHost, s));
        for (int c = 0; c < kHostChunks; ++c) MK_TRY(cudaEventRecord(hp->y_done[c], s));
        return MK_OK;
    }
    // Kernel-per-step path, pipelined copies on the workspace's copy streams:
    //  - the upload of x waits only for the previous call on this workspace to
    //    have read the staged x (its scatter), so it overlaps that call's GEMMs
    //    (from mapped page-locked x_host by a few CTAs' loads, else by the copy
    //    engine);
    //  - the combine runs in chunks of tokens (about 16 MB of output each, at
    //    most kHostChunks) and each chunk is downloaded as soon as it is
    //    combined, alternating between two copy streams (the staged y is
    //    rewritten only once the previous call's downloads are done);
    //  - `stream` waits for the last download, so the output is in y_host once
    //    the stream reaches this point, as for the plain sequence.
    MK_TRY(cudaStreamWaitEvent(hp->h2d, hp->x_free, 0));
    if (const void* xm = mapped_host_ptr(x_host))
        MK_TRY(launch_bulk_copy(xm, xd, bytes, kCopyInCtas, hp->h2d));
    else
        MK_TRY(cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, hp->h2d));
    MK_TRY(cudaEventRecord(hp->x_ready, hp->h2d));
    MK_TRY(cudaStreamWaitEvent(s, hp->x_ready, 0));
    LayerHooks hk;
    hk.after_scatter = hp->x_free;
    hk.skip_combine = true;
    st = layer_impl(xd, wg, bias, w1, w3, w2, T, d, E, k, ffn, yd, ws, L, opts, s, hk);
    if (st != MK_OK) return st;
    const bf16* P = at<bf16>(ws, L.P);
    const int32_t* slot_row = at<int32_t>(ws, L.slot_row);
    // y_host page-locked and mapped for the device: the combine writes it
    // directly over the host link, no staging and no separate download
    cudaPointerAttributes ya{};
    if (cudaPointerGetAttributes(&ya, y_host) == cudaSuccess && ya.type == cudaMemoryTypeHost &&
        ya.devicePointer != nullptr) {
        MK_TRY(launch_combine(P, slot_row, T, d, k, static_cast<bf16*>(ya.devicePointer), s));
        if (opts && opts->phase_events && opts->phase_events[MK_PHASE_COUNT_ALL])
            MK_TRY(cudaEventRecord(static_cast<cudaEvent_t>(opts->phase_events[MK_PHASE_COUNT_ALL]), s));
        return MK_OK;
    }
    cudaGetLastError();  // a pointer unknown to CUDA (pageable memory) is not an error here
    // about 16 MB of output per chunk (1 to kHostChunks chunks): small layers
    // gain nothing from splitting and would pay a launch and a copy per chunk
    const int chunks = static_cast<int>(std::min<int64_t>(kHostChunks, std::max<int64_t>(1, bytes >> 24)));
    const int64_t tc = (T + chunks - 1) / chunks;
    // the staged y is rewritten only after every download of an earlier call
    // (which may have cut it into other chunks) has finished
    for (int c = 0; c < kHostChunks; ++c) MK_TRY(cudaStreamWaitEvent(s, hp->y_done[c], 0));
    MK_TRY(cudaStreamWaitEvent(s, hp->y_async_done[0], 0));
    int last = -1;
    for (int c = 0; c < chunks; ++c) {
        const int64_t t0 = c * tc;
        const int64_t nt = std::min<int64_t>(tc, T - t0);
        if (nt <= 0) break;
        MK_TRY(launch_combine(P, slot_row + t0 * k, nt, d, k, yd + t0 * d, s, T * k));
        MK_TRY(cudaEventRecord(hp->y_ready[c], s));
        cudaStream_t q = hp->d2h[c & 1];
        MK_TRY(cudaStreamWaitEvent(q, hp->y_ready[c], 0));
        MK_TRY(cudaMemcpyAsync(static_cast<bf16*>(y_host) + t0 * d, yd + t0 * d, static_cast<size_t>(nt) * d * 2,
                               cudaMemcpyDeviceToHost, q));
        MK_TRY(cudaEventRecord(hp->y_done[c], q));
        last = c;
    }
    if (opts && opts->phase_events && opts->phase_events[MK_PHASE_COUNT_ALL])
        MK_TRY(cudaEventRecord(static_cast<cudaEvent_t>(opts->phase_events[MK_PHASE_COUNT_ALL]), s));
    for (int c = std::max(0, last - 1); c <= last; ++c)  // the last chunk of each copy stream
        MK_TRY(cudaStreamWaitEvent(s, hp->y_done[c], 0));
    return MK_OK;
}

mk_status mk_moe_layer_host_async(const void* x_host, const float* wg, const float* bias, const void* w1,
                                  const void* w3, const void* w2, int64_t T, int d, int E, int k, int ffn,
                                  void* y_host, void* ws, size_t ws_bytes, const mk_moe_opts* opts, void* stream,
                                  void* y_ready) {
    if (y_ready == nullptr) return MK_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaEvent_t done = static_cast<cudaEvent_t>(y_ready);
    if (T == 0 && check_sizes(T, d, E, k, ffn) == MK_OK) {
        MK_TRY(cudaEventRecord(done, s));
        return MK_OK;
    }
    mk_status st = validate_layer(x_host, wg, w1, w3, w2, T, d, E, k, ffn, y_host, ws, ws_bytes, opts, false);
    if (st != MK_OK) return st;
    if (opts && opts->path != MK_PATH_STEPS) {
        st = mk_moe_layer_host(x_host, wg, bias, w1, w3, w2, T, d, E, k, ffn, y_host, ws, ws_bytes, opts, stream);
        if (st != MK_OK) return st;
        MK_TRY(cudaEventRecord(done, s));
        return MK_OK;
    }
    const WsLayout L = ws_layout(T, d, E, k, ffn);
    const size_t bytes = static_cast<size_t>(T) * d * 2;
    bf16* xd = at<bf16>(ws, L.x_stage);
    HostPipe* hp = nullptr;
    MK_TRY(get_pipe(ws, &hp));
    // consecutive pipelined calls stage y in alternate regions, so a call's
    // combine waits only for the download two calls back
    const int r = static_cast<int>(hp->async_calls++ & 1u);
    bf16* yd = at<bf16>(ws, r ? L.y_stage2 : L.y_stage);
    // upload of x, after the previous call's scatter (as in mk_moe_layer_host):
    // from page-locked memory mapped for the device by a few CTAs' loads
    // (running beside the previous call's GEMMs), else by the copy engine
    MK_TRY(cudaStreamWaitEvent(hp->h2d, hp->x_free, 0));
    if (const void* xm = mapped_host_ptr(x_host))
        MK_TRY(launch_bulk_copy(xm, xd, bytes, kCopyInCtas, hp->h2d));
    else
        MK_TRY(cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, hp->h2d));
    MK_TRY(cudaEventRecord(hp->x_ready, hp->h2d));
    MK_TRY(cudaStreamWaitEvent(s, hp->x_ready, 0));
    LayerHooks hk;
    hk.after_scatter = hp->x_free;
    hk.skip_combine = true;
    st = layer_impl(xd, wg, bias, w1, w3, w2, T, d, E, k, ffn, yd, ws, L, opts, s, hk);
    if (st != MK_OK) return st;
    // the staged y is rewritten only after every earlier download from it
    // (region 0 is also the blocking entry point's staging region)
    if (r == 0)
        for (int c = 0; c < kHostChunks; ++c) MK_TRY(cudaStreamWaitEvent(s, hp->y_done[c], 0));
    MK_TRY(cudaStreamWaitEvent(s, hp->y_async_done[r], 0));
    MK_TRY(launch_combine(at<bf16>(ws, L.P), at<int32_t>(ws, L.slot_row), T, d, k, yd, s));
    if (opts && opts->phase_events && opts->phase_events[MK_PHASE_COUNT_ALL])
        MK_TRY(cudaEventRecord(static_cast<cudaEvent_t>(opts->phase_events[MK_PHASE_COUNT_ALL]), s));
    MK_TRY(cudaEventRecord(hp->y_ready[r], s));
    // the download, off `stream`: into page-locked memory mapped for the device
    // by a few CTAs' stores (running beside the next call's kernels), else by the
    // copy engine
    cudaStream_t q = hp->d2h[0];
    MK_TRY(cudaStreamWaitEvent(q, hp->y_ready[r], 0));
    if (void* ym = const_cast<void*>(mapped_host_ptr(y_host)))
        MK_TRY(launch_bulk_copy(yd, ym, bytes, kCopyOutCtas, q));
    else
        MK_TRY(cudaMemcpyAsync(y_host, yd, bytes, cudaMemcpyDeviceToHost, q));
    MK_TRY(cudaEventRecord(hp->y_async_done[r], q));
    MK_TRY(cudaEventRecord(done, q));
    return MK_OK;
}



mk_status mk_moe_last_device_error(void* ws, void* stream, uint32_t* detail) {
    if (ws == nullptr) return MK_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return MK_ERR_CUDA;
    uint32_t st[2] = {0, 0};
    if (cudaMemcpy(st, ws, sizeof st, cudaMemcpyDeviceToHost) != cudaSuccess) return MK_ERR_CUDA;
    if (cudaMemset(ws, 0, sizeof st) != cudaSuccess) return MK_ERR_CUDA;
    if (detail) *detail = st[1];
    return static_cast<mk_status>(st[0]);
}

mk_status mk_moe_route_fallbacks(void* ws, void* stream, uint32_t* count) {
    if (ws == nullptr) return MK_ERR_WORKSPACE;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MK_ERR_CUDA;
    uint32_t n = 0;
    if (cudaMemcpy(&n, static_cast<uint8_t*>(ws) + 8, sizeof n, cudaMemcpyDeviceToHost) != cudaSuccess)
        return MK_ERR_CUDA;
    if (count) *count = n;
    return MK_OK;
}

mk_status mk_moe_layer_trace_count(void* ws, int64_t T, int d, int E, int k, int ffn, void* stream,
                                   uint32_t* count) {
    if (ws == nullptr) return MK_ERR_WORKSPACE;
    mk_status st = check_sizes(T, d, E, k, ffn);
    if (st != MK_OK) return st;
    if (count == nullptr) return MK_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, d, E, k, ffn);
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MK_ERR_CUDA;
    FusedSync fs;
    if (cudaMemcpy(&fs, at<uint8_t>(ws, L.sync), sizeof fs, cudaMemcpyDeviceToHost) != cudaSuccess) return MK_ERR_CUDA;
    *count = fs.trace_n;
    return MK_OK;
}

mk_status mk_moe_route_approx_logits(const void* ws, int64_t T, int d, int E, int k, float* out, void* stream) {
    mk_status st = check_sizes(T, d, E, k, 64);
    if (st != MK_OK) return st;
    if (ws == nullptr) return MK_ERR_WORKSPACE;
    if (out == nullptr) return MK_ERR_INVALID_ARG;
    if (T == 0) return MK_OK;
    const WsLayout L = ws_layout_dispatch(T, d, E, k);  // the logits sit at the same offset in every layout
    MK_TRY(cudaMemcpyAsync(out, static_cast<const uint8_t*>(ws) + L.logits, static_cast<size_t>(T) * E * 4,
                           cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream)));
    return MK_OK;
}

mk_status mk_moe_workspace_region(int64_t T, int d, int E, int k, int ffn, int region, size_t* offset,
                                  size_t* bytes) {
    if (check_sizes(T, d, E, k, ffn) != MK_OK || offset == nullptr || bytes == nullptr) return MK_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, d, E, k, ffn);
    const size_t S = static_cast<size_t>(T) * k;
    switch (region) {
        case MK_WS_IDS: *offset = L.ids; *bytes = S * 4; break;
        case MK_WS_W: *offset = L.w; *bytes = S * 4; break;
        case MK_WS_OFFSETS: *offset = L.offsets; *bytes = (static_cast<size_t>(E) + 1) * 4; break;
        case MK_WS_ROW_TOKEN: *offset = L.row_token; *bytes = S * 4; break;
        case MK_WS_ROW_WEIGHT: *offset = L.row_weight; *bytes = S * 4; break;
        case MK_WS_SLOT_ROW: *offset = L.slot_row; *bytes = S * 4; break;
        case MK_WS_X_PERM: *offset = L.x_perm; *bytes = S * d * 2; break;
        case MK_WS_H: *offset = L.h; *bytes = S * ffn * 2; break;
        case MK_WS_P: *offset = L.P; *bytes = S * d * 2; break;
        default: return MK_ERR_INVALID_ARG;
    }
    return MK_OK;
}

mk_status mk_moe_layer_routing(const void* ws, int64_t T, int d, int E, int k, int ffn, int32_t* topk_ids,
                               float* topk_w, int32_t* expert_offsets, int32_t* slot_row, void* stream) {
    mk_status st = check_sizes(T, d, E, k, ffn);
    if (st != MK_OK) return st;
    if (ws == nullptr) return MK_ERR_WORKSPACE;
    if (T == 0) return MK_OK;
    const WsLayout L = ws_layout(T, d, E, k, ffn);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* w = const_cast<void*>(ws);
    const size_t tk = static_cast<size_t>(T) * k * 4;
    if (topk_ids) MK_TRY(cudaMemcpyAsync(topk_ids, at<uint8_t>(w, L.ids), tk, cudaMemcpyDeviceToDevice, s));
    if (topk_w) MK_TRY(cudaMemcpyAsync(topk_w, at<uint8_t>(w, L.w), tk, cudaMemcpyDeviceToDevice, s));
    if (expert_offsets)
        MK_TRY(cudaMemcpyAsync(expert_offsets, at<uint8_t>(w, L.offsets), 4 * (E + 1), cudaMemcpyDeviceToDevice, s));
    if (slot_row) MK_TRY(cudaMemcpyAsync(slot_row, at<uint8_t>(w, L.slot_row), tk, cudaMemcpyDeviceToDevice, s));
    return MK_OK;
}

}  // extern "C"
