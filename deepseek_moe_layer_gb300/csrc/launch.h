// launch.h -- host-side launchers of the kernels (internal to the library; the public
// interface is include/moe_gb300.h).  Every launcher assumes its arguments were checked by
// the C-ABI layer and returns the cudaError_t of the launch.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

namespace moe {

// One-time set-up that CUDA keeps per device (a kernel's dynamic shared-memory limit, for
// instance): run() calls fn() the first time it is reached with a given device current and
// remembers a success; a failure is returned and retried on the next call.  Safe to call
// from several host threads.
class DeviceOnce {
  public:
    static constexpr int kMaxDevices = 64;
    template <class F>
    cudaError_t run(F&& fn) {
        int dev = -1;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
        if (done_[dev].load(std::memory_order_acquire)) return cudaSuccess;
        std::lock_guard<std::mutex> lock(mu_);
        if (done_[dev].load(std::memory_order_relaxed)) return cudaSuccess;
        e = fn();
        if (e == cudaSuccess) done_[dev].store(1, std::memory_order_release);
        return e;
    }

  private:
    std::mutex mu_;
    std::atomic<int> done_[kMaxDevices] = {};
};

// ---- gate ---------------------------------------------------------------------------
struct RouteArgs {
    const void* logits;          // [nsplit][rows][E], fp32 (or bf16 when bf16 != 0)
    int bf16;
    int nsplit;                  // partial sums to add, in split order (>= 1)
    long long split_stride;      // elements between splits
    const float* logit_offset;   // [E] or nullptr
    const float* bias;           // [E]
    long long rows;
    int E, top_k, n_group, topk_group, norm;
    float scale;
    int32_t* inds;               // [rows, K]
    float* scores;               // [rows, K]
    float* logits_out;           // [rows, E] copy of the summed logits, or nullptr
    int softmax;                 // 1: softmax route (bias, groups, norm, scale unused)
};
cudaError_t launch_route(const RouteArgs& a, cudaStream_t s);
// logits[t, e] += offset[e] for a [T, E] fp32 matrix.
cudaError_t launch_add_offset(float* logits, long long T, int E, const float* offset,
                              cudaStream_t s);

// ---- dispatch -----------------------------------------------------------------------
cudaError_t launch_permute(const int32_t* inds, long long P, int E, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv, cudaStream_t s,
                           void* scratch = nullptr, size_t scratch_bytes = 0);
// scratch (optional, device): with at least permute_scratch_bytes(E) bytes, batches of at
// least kPermMultiMin pairs are dispatched by many CTAs instead of one.
constexpr long long kPermMultiMin = 8192;
size_t permute_scratch_bytes(int E);
// x_perm[j] = x[perm[j] / K] for the dispatched slots j < offsets[E].
cudaError_t launch_gather_rows(const void* x, const int32_t* perm, const int32_t* offsets, int E,
                               int K, long long P, int d, void* x_perm, cudaStream_t s);

// ---- combine ------------------------------------------------------------------------
// shared_gate: [T] per-token weight of the shared expert's row, or nullptr for weight 1.
cudaError_t launch_combine(const void* expert_out, const float* scores, const int32_t* inv,
                           const void* shared_out, long long T, int K, int d, void* y,
                           cudaStream_t s, const float* shared_gate = nullptr);
// gate[t] = sigmoid(x[t] . w) for bf16 x [T, d] and w [d].
cudaError_t launch_shared_gate(const void* x, long long T, int d, const void* w, float* gate,
                               cudaStream_t s);

// ---- DSA indexer top-k selection -----------------------------------------------------
struct TopkArgs {
    const void* scores;          // [rows, ld] fp32, or bf16 when bf16 != 0
    int bf16;
    long long rows;
    int n;                       // positions per row
    long long ld;                // elements between rows (>= n)
    const int32_t* lengths;      // [rows] valid positions per row, or nullptr (all n)
    int k;                       // index_topk
    int32_t* inds;               // [rows, k] selected positions, ascending, -1 padded
    uint8_t* mask;               // [rows, mask_ld] 1 at the selected positions, or nullptr
    long long mask_ld;
    int nclusters;               // CTAs per row (thread-block cluster size, 1..8)
    int seg;                     // positions per CTA (multiple of 8)
    int cached;                  // keys of a segment held in shared memory
};
// Fills nclusters / seg / cached from n.
void indexer_topk_plan(TopkArgs& a);
// Per-CTA dynamic shared memory of the selection kernel.
size_t indexer_topk_smem(int seg, int cached);
cudaError_t launch_indexer_topk(const TopkArgs& a, cudaStream_t s);

// ---- expert GEMMs (tcgen05) ---------------------------------------------------------
enum GemmMode { kGateUp = 0, kDown = 1, kRouter = 2 };

struct GemmWeights {             // one stacked weight tensor set (bf16 or affine 4/8-bit)
    int bits;                    // 16, 8 or 4
    const void* w0;              // gate (kGateUp) / down (kDown) / router (kRouter)
    const void* w1;              // up (kGateUp only)
    const void* s0; const void* b0;   // quantised: fp16 scale / bias of w0
    const void* s1; const void* b1;   // quantised: fp16 scale / bias of w1
    int group;                   // quantised: inputs per scale (32, 64 or 128)
};

struct GemmArgs {
    GemmMode mode;
    const void* act;             // activation rows (bf16 [rows_total, Kdim])
    long long act_rows;          // rows of `act`
    const void* act_shared;      // rows of the shared group (bf16 [T, Kdim]); may alias act
    long long shared_act_row0;   // first row of the shared group in act_shared
    const int32_t* offsets;      // [E+1] routed group row offsets (device) or nullptr: one
                                 // group of rows [0, single_rows)
    long long single_rows;
    int E;                       // routed groups
    int has_shared;
    long long shared_rows;       // T
    long long shared_out_row0;   // first output row of the shared group
    int Kdim;                    // reduction length
    int F;                       // output features per group
    int ksplit;                  // kRouter only: K-splits, partial sums to out + ks*split_stride
    long long split_stride;
    GemmWeights w;               // routed (or router) weights
    GemmWeights ws;              // shared expert weights (bf16)
    void* out;                   // bf16 [rows, F] (kGateUp: h, kDown: o) or fp32 (kRouter)
    long long out_ld;
    int tok_tile;                // 0: tokens on the M side (128-row tiles); else tokens on
                                 // the N side in tiles of tok_tile (16/32/64/128)
    int pair;                    // bf16, tokens on M: 256-row tiles on CTA pairs
    long long max_tiles;         // host upper bound on the number of tiles
};
cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t s);

// Per-device status word of the kernels with bounded waits.
cudaError_t read_device_status(unsigned int* out, int clear, cudaStream_t s);
// One CTA waits `limit_ns` on an mbarrier nothing completes and records the timeout.
cudaError_t launch_watchdog_selftest(unsigned long long limit_ns, cudaStream_t s);

int num_sms();

// Sets the thread-local text returned by moe_last_error() and returns `code`.
int set_error(int code, const char* msg);

// Programmatic dependent launch for the kernels of one layer call after its first: while set
// (per host thread), the launchers below launch with programmatic stream serialization, so a
// kernel's prologue overlaps the tail of the one before it (each kernel waits with
// griddepcontrol.wait before it reads its predecessor's results or writes global memory).
bool pdl_enabled();

// Launches `kernel` on `s`, with programmatic stream serialization when pdl_enabled().
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, args...);
    return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace moe
