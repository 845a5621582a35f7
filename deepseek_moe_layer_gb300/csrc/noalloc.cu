// noalloc.cu -- moe_forward for callers that cannot allocate device memory.
//
// Some callers of this layer have no way to obtain a workspace: a serving engine that
// reserves nearly all of HBM up front for its own pools (KV cache, weights) and hands out
// nothing else, or a host program embedded in a framework that owns the allocator.  For
// them the workspace of the whole layer lives in a fixed array in this library's own device
// memory, sized for decode batches (up to 227 tokens at DeepSeek-V3 shape).  The caller
// still passes its inputs, weights and outputs.
//
// Behaviour a caller must know:
//   - The array is MOE_NOALLOC_SCRATCH_BYTES (64 MiB) on every device that loads the
//     library, held until the process exits.
//   - The first call on a device resolves the array's device address (cudaGetSymbolAddress,
//     with that device current); make that first call before any stream capture.
//   - Every call on a device uses the same array, so calls that overlap on the GPU (two
//     streams, or two host threads) race; serialise them on one stream.
//   - The array keeps whatever the last call left there.  Nothing in it needs to start at
//     zero: every byte the kernels read back is written earlier in the same call (rows the
//     GEMM tiles load past an expert's last token only reach accumulator rows that are
//     never stored).
//   - A configuration whose workspace exceeds the array is rejected with MOE_ERR_INVALID
//     before anything runs.
#include <cstdio>
#include <mutex>

#include "../../include/moe_gb300.h"
#include "launch.h"

namespace {

constexpr size_t kScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once per device).
int scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0)
        return moe::set_error(MOE_ERR_NODEVICE, "no CUDA device is current");
    if (dev >= kMaxDevices) return moe::set_error(MOE_ERR_NODEVICE, "device index too large");
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            char msg[256];
            snprintf(msg, sizeof msg, "scratch set-up failed on device %d: %s", dev,
                     cudaGetErrorString(e));
            return moe::set_error(MOE_ERR_CUDA, msg);
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" int moe_forward_noalloc(const void* x, int64_t T, int32_t d, int32_t I, int32_t E,
                                   const void* w_router, const float* bias,
                                   const float* logit_offset, const moe_route_params_t* params,
                                   const moe_expert_weights_t* experts,
                                   const moe_expert_weights_t* shared, void* y,
                                   int32_t* inds_out, float* scores_out, float* logits_out,
                                   moe_stream_t stream) {
    if (!params) return moe::set_error(MOE_ERR_INVALID, "params is NULL");
    const size_t need =
        moe_forward_workspace_bytes(T, d, I, E, params->top_k, shared != nullptr ? 1 : 0);
    if (need > kScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "this layer needs %zu bytes of workspace; the fixed scratch holds %zu "
                 "(%lld tokens is too many for moe_forward_noalloc: use moe_forward)",
                 need, kScratchBytes, (long long)T);
        return moe::set_error(MOE_ERR_INVALID, msg);
    }
    void* ws = nullptr;
    const int rc = scratch_address(&ws);
    if (rc != MOE_OK) return rc;
    return moe_forward(x, T, d, I, E, w_router, bias, logit_offset, params, experts, shared, y,
                       inds_out, scores_out, logits_out, ws, kScratchBytes, stream);
}
