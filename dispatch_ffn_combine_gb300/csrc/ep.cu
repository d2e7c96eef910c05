// ep.cu -- the row regroup of the expert-parallel layer.
//
// In the expert-parallel form of the layer (mKernel README, kernel table, row
// "MoE Dispatch + FFN + Combine": tokens are routed "to their expert ranks"
// and the weighted outputs combined "back to each token's source rank"; paper
// section 3.1 and Table 3 for the dispatch exchange), each of G ranks owns
// E_l = E / G experts.  A rank receives, from every source rank q, the rows q
// routed to its experts, grouped by local expert: in source-major order
// [q][e][rows].  Its grouped expert FFN needs them expert-major, [e][q][rows];
// its outputs go back in source-major order, so that source q gets its rows in
// the order it sent them.  This file moves rows between the two orders.
//
//   counts[q * E_l + e]  rows from source q for local expert e
//   source-major offset  of (q, e): sum of counts over (q', e') < (q, e) in (q, e) order
//   expert-major offset  of (q, e): sum of counts over (e', q') < (e, q) in (e, q) order
// A row keeps its position inside its (q, e) group.
#include <algorithm>

#include "mk_device.cuh"
#include "mk_internal.h"

namespace mk {
namespace {

constexpr int kMaxGroups = 2048;  // G * E_l

// One block: both prefix tables ([G * E_l + 1] each) from the counts; a count
// below zero or a total different from `rows` is recorded as MK_ERR_BOUNDS and
// the tables are zeroed, so every row is copied to its own position.
__global__ void __launch_bounds__(256) regroup_tables_kernel(const int32_t* __restrict__ counts, int G, int El,
                                                             int64_t rows, int32_t* __restrict__ src_off,
                                                             int32_t* __restrict__ dst_off,
                                                             int32_t* __restrict__ expert_offsets, uint32_t* status) {
    __shared__ int32_t c[kMaxGroups];
    __shared__ int bad;
    const int n = G * El;
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        c[i] = counts[i];
        if (c[i] < 0) atomicExch(&bad, 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int64_t s = 0;
        for (int i = 0; i < n; ++i) s += c[i];
        if (s != rows) bad = 1;
    }
    __syncthreads();
    if (bad) {
        if (threadIdx.x == 0) report_error(status, MK_ERR_BOUNDS, kSiteRegroup);
        for (int i = threadIdx.x; i <= n; i += blockDim.x) src_off[i] = dst_off[i] = 0;
        if (expert_offsets != nullptr)
            for (int e = threadIdx.x; e <= El; e += blockDim.x) expert_offsets[e] = 0;
        return;
    }
    if (threadIdx.x == 0) {  // sequential scans (n <= 2048): fixed order, exact
        int32_t s = 0;
        for (int i = 0; i < n; ++i) {
            src_off[i] = s;
            s += c[i];
        }
        src_off[n] = s;
        s = 0;
        for (int e = 0; e < El; ++e)
            for (int q = 0; q < G; ++q) {
                dst_off[q * El + e] = s;
                s += c[q * El + e];
            }
        dst_off[n] = s;
        if (expert_offsets != nullptr) {  // expert e starts at its source-0 group in expert-major order
            for (int e = 0; e < El; ++e) expert_offsets[e] = dst_off[e];
            expert_offsets[El] = s;
        }
    }
}

// A warp per row: the (q, e) group of source row r by a binary search over the
// source-major offsets, then 16-byte (or 4-byte) copies of the row into its
// expert-major position.  to_expert_major = 0 runs the inverse move (the
// groups are found in the expert-major order and written source-major).
__global__ void __launch_bounds__(256) regroup_rows_kernel(const uint8_t* __restrict__ in, uint8_t* __restrict__ out,
                                                           const int32_t* __restrict__ src_off,
                                                           const int32_t* __restrict__ dst_off, int G, int El,
                                                           int64_t rows, int row_bytes, int to_expert_major) {
    const int lane = threadIdx.x & 31;
    const int n = G * El;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5); r < rows; r += warps) {
        int64_t dst;
        if (to_expert_major) {
            int lo = 0, hi = n - 1;  // last group g with src_off[g] <= r
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (src_off[mid] <= r)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            dst = dst_off[lo] + (r - src_off[lo]);
        } else {
            // r is an expert-major position: find its group in (e, q) order
            int lo = 0, hi = n - 1;  // last (e, q) index with dst_off[q * El + e] <= r
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                const int g = (mid % G) * El + (mid / G);
                if (dst_off[g] <= r)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            const int g = (lo % G) * El + (lo / G);
            dst = src_off[g] + (r - dst_off[g]);
        }
        const uint8_t* src_row = in + r * row_bytes;
        uint8_t* dst_row = out + dst * row_bytes;
        if ((row_bytes & 15) == 0) {
            for (int c = lane; c < row_bytes / 16; c += 32)
                reinterpret_cast<uint4*>(dst_row)[c] = reinterpret_cast<const uint4*>(src_row)[c];
        } else {
            for (int c = lane; c < row_bytes / 4; c += 32)
                reinterpret_cast<uint32_t*>(dst_row)[c] = reinterpret_cast<const uint32_t*>(src_row)[c];
        }
    }
}

}  // namespace
}  // namespace mk

using namespace mk;

extern "C" size_t mk_moe_ep_regroup_workspace_size(int G, int E_local) {
    if (G < 1 || E_local < 1 || G * E_local > kMaxGroups) return 0;
    return 256 + 8 * (static_cast<size_t>(G) * E_local + 1);
}

extern "C" mk_status mk_moe_ep_regroup(const void* rows_in, void* rows_out, const int32_t* counts, int G, int E_local,
                                       int64_t rows, int row_bytes, int to_expert_major, int32_t* expert_offsets,
                                       void* ws, size_t ws_bytes, void* stream) {
    if (G < 1 || E_local < 1 || G * E_local > kMaxGroups || rows < 0 || row_bytes <= 0 || (row_bytes & 3) != 0)
        return MK_ERR_INVALID_ARG;
    if (rows >= (int64_t(1) << 31)) return MK_ERR_UNSUPPORTED;
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 ||
        ws_bytes < mk_moe_ep_regroup_workspace_size(G, E_local))
        return MK_ERR_WORKSPACE;
    if (!counts || (rows > 0 && (!rows_in || !rows_out))) return MK_ERR_INVALID_ARG;
    if (rows > 0 && (!aligned16(rows_in) || !aligned16(rows_out))) return MK_ERR_INVALID_ARG;
    if (!device_is_sm103()) return MK_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t* status = static_cast<uint32_t*>(ws);
    int32_t* src_off = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + 256);
    int32_t* dst_off = src_off + G * E_local + 1;
    if (cudaMemsetAsync(status, 0, 8, s) != cudaSuccess) return MK_ERR_CUDA;
    regroup_tables_kernel<<<1, 256, 0, s>>>(counts, G, E_local, rows, src_off, dst_off, expert_offsets, status);
    if (cudaGetLastError() != cudaSuccess) return MK_ERR_CUDA;
    if (rows == 0) return MK_OK;
    const int64_t blocks = std::min<int64_t>((rows + 7) / 8, 16 * static_cast<int64_t>(device_sm_count()));
    regroup_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        static_cast<const uint8_t*>(rows_in), static_cast<uint8_t*>(rows_out), src_off, dst_off, G, E_local, rows,
        row_bytes, to_expert_major);
    if (cudaGetLastError() != cudaSuccess) return MK_ERR_CUDA;
    return MK_OK;
}
