// route_noalloc.cu -- the router for callers that cannot allocate device memory.
//
// mk_moe_route needs a caller-supplied workspace for its fp32 logits.  Some
// callers cannot provide one: code running where cudaMalloc is not allowed or
// must not be called (inside a region whose memory is fixed up front, such as
// an inference runtime with a static memory plan, a real-time path that may
// not block on the allocator, or a plug-in that receives only its input and
// output buffers), and callers that cannot take a dependency on a caching
// allocator.  This entry point keeps its scratch in a file-scope device array
// instead, so it allocates nothing.
//
// The array holds kNoAllocLogits fp32 logits (8 MiB).  Every GPU on which the
// library is used keeps those 8 MiB until the process exits.  Each call
// writes every logit it later reads, so nothing in the array has to start at
// zero; the array keeps the last call's logits afterwards.  All calls share the
// one array: calls whose kernels overlap on the GPU (for example on two
// streams without ordering between them) race and give wrong results.
#include <mutex>

#include "mk_internal.h"

namespace mk {
namespace {

constexpr int64_t kNoAllocLogits = int64_t(1) << 21;  // T * E <= 2,097,152 (8 MiB of fp32)

static __device__ __align__(256) float g_route_scratch[kNoAllocLogits];

// Device address of g_route_scratch per device, found once per device.  In
// host code the array's name is only a stand-in for the symbol, never a
// device address, so the kernels get the address cudaGetSymbolAddress gives.
std::mutex g_scratch_mu;
float* g_scratch_ptr[64] = {};

cudaError_t scratch_for_current_device(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_route_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace mk

using namespace mk;

extern "C" mk_status mk_moe_route_noalloc(const void* x, const float* wg, const float* bias, int64_t T, int d,
                                          int E, int k, int32_t* topk_ids, float* topk_w, int32_t* expert_counts,
                                          void* stream) {
    // The checks of mk_moe_route (sizes, then pointers, then alignment), plus
    // the size of the static scratch array.
    mk_status st = check_sizes(T, d, E, k, 64);
    if (st != MK_OK) return st;
    if (!x || !wg || !topk_ids || !topk_w) return MK_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(wg)) return MK_ERR_INVALID_ARG;
    if (T * E > kNoAllocLogits) return MK_ERR_UNSUPPORTED;  // more logits than the static scratch holds
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        if (expert_counts && cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * E, s) != cudaSuccess)
            return MK_ERR_CUDA;
        return MK_OK;
    }
    if (!device_is_sm103()) return MK_ERR_UNSUPPORTED;
    float* logits = nullptr;
    if (scratch_for_current_device(&logits) != cudaSuccess) return MK_ERR_CUDA;
    if (launch_route_logits(static_cast<const bf16*>(x), wg, bias, T, d, E, logits, s) != cudaSuccess)
        return MK_ERR_CUDA;
    if (expert_counts && cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * E, s) != cudaSuccess)
        return MK_ERR_CUDA;
    if (launch_topk(logits, T, E, k, topk_ids, topk_w, expert_counts, s) != cudaSuccess) return MK_ERR_CUDA;
    return MK_OK;
}
