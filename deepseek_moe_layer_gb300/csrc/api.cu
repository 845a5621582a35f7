// api.cu -- the C ABI declared in include/moe_gb300.h: argument checks (all on the host,
// before any CUDA call, so a rejected call touches nothing), workspace layout, and the
// launch sequence of the layer on one stream.
//
// Source of the call contract: "feat(engine): E1 DeepSeek-style MoE gate (sigmoid, group
// top-k, bias) (#108)", sections "API" (precomputed logits [..., E], required bias [E],
// outputs inds / scores [..., K]) and the review's "What looks solid" 4 (outputs left
// unchanged on failure) and "Findings" L1/L2 with the author's reply (the validation
// matrix: null arguments, top_k == 0, top_k > E, E % n_group != 0, topk_group out of
// [1, n_group], n_group > 1 with fewer than two experts per group, bias rank != 1).
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

#include "../../include/moe_gb300.h"
#include "launch.h"

namespace {

thread_local std::string g_err;
thread_local bool g_pdl = false;

// Programmatic dependent launch for the rest of a layer call (restored on return).
struct PdlScope {
    bool prev;
    PdlScope() : prev(g_pdl) {}
    void on() { g_pdl = true; }
    ~PdlScope() { g_pdl = prev; }
};

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char* where) {
    return fail(MOE_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

#define MOE_CHECK(cond, ...)                                  \
    do {                                                      \
        if (!(cond)) return fail(MOE_ERR_INVALID, __VA_ARGS__); \
    } while (0)

#define MOE_CUDA(call, where)                          \
    do {                                               \
        cudaError_t e_ = (call);                       \
        if (e_ != cudaSuccess) return cuda_fail(e_, where); \
    } while (0)

// Host-side fault injection (a test hook; off unless MOE_FAULT is set in the environment or
// moe_set_fault() is called).  MOE_FAULT=launch[:N] makes the N-th kernel launch (0-based,
// default 0) of every API call report MOE_ERR_CUDA instead of launching, so the error path
// after earlier launches can be exercised without making a GPU fail.  The launch count
// restarts at every entry point.
std::atomic<int> g_fault_kind{-1};  // -1: environment not read yet
std::atomic<int> g_fault_at{0};
thread_local int g_launch_no = 0;

void fault_init() {
    int expected = -1;
    if (g_fault_kind.load(std::memory_order_acquire) != -1) return;
    int kind = MOE_FAULT_NONE, at = 0;
    const char* env = getenv("MOE_FAULT");
    if (env && strncmp(env, "launch", 6) == 0 && (env[6] == '\0' || env[6] == ':')) {
        kind = MOE_FAULT_LAUNCH;
        at = env[6] == ':' ? atoi(env + 7) : 0;
        if (at < 0) at = 0;
    }
    g_fault_at.store(at, std::memory_order_relaxed);
    g_fault_kind.compare_exchange_strong(expected, kind, std::memory_order_acq_rel);
}

// True when the launch about to be made is the one the hook fails.
bool fault_this_launch() {
    fault_init();
    const int n = g_launch_no++;
    return g_fault_kind.load(std::memory_order_acquire) == MOE_FAULT_LAUNCH &&
           n == g_fault_at.load(std::memory_order_relaxed);
}

// Start of an entry point: clears the thread's error text and restarts its launch count.
void begin_call() {
    g_err.clear();
    g_launch_no = 0;
}

// A kernel launch through one of the launchers: MOE_ERR_CUDA on a failed launch, or when
// the fault hook selects it (then nothing is launched).
#define MOE_LAUNCH(call, where)                                                        \
    do {                                                                               \
        if (fault_this_launch())                                                       \
            return fail(MOE_ERR_CUDA, "%s: injected launch fault (MOE_FAULT)", where); \
        cudaError_t e_ = (call);                                                       \
        if (e_ != cudaSuccess) return cuda_fail(e_, where);                            \
    } while (0)

constexpr int kMaxExperts = 1024;
constexpr int kMaxPhaseEvents = 8;

cudaEvent_t g_phase_ev[kMaxPhaseEvents];
int g_phase_n = 0;

cudaError_t phase(int i, cudaStream_t s) {
    return i < g_phase_n ? cudaEventRecord(g_phase_ev[i], s) : cudaSuccess;
}
constexpr int kMaxTopK = 32;
constexpr int kMaxGroups = 32;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// The current device must be an sm_103 part (GB300).  Checked once per device.
int check_device() {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(MOE_ERR_NODEVICE, "no CUDA device: %s", cudaGetErrorString(e));
    static std::atomic<int> checked[64] = {};
    if (dev >= 0 && dev < 64 && checked[dev].load(std::memory_order_acquire) == 1) return MOE_OK;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
        return fail(MOE_ERR_NODEVICE, "device %d is sm_%d%d; this library is built for sm_103a",
                    dev, major, minor);
    if (dev >= 0 && dev < 64) checked[dev].store(1, std::memory_order_release);
    return MOE_OK;
}

int check_route_params(int32_t E, const moe_route_params_t* p) {
    MOE_CHECK(p, "params is NULL");
    MOE_CHECK(E >= 1 && E <= kMaxExperts, "E = %d outside [1, %d]", E, kMaxExperts);
    MOE_CHECK(p->top_k >= 1, "top_k = %d < 1", p->top_k);
    MOE_CHECK(p->top_k <= E, "top_k = %d > E = %d", p->top_k, E);
    MOE_CHECK(p->top_k <= kMaxTopK, "top_k = %d > %d", p->top_k, kMaxTopK);
    MOE_CHECK(p->n_group >= 1, "n_group = %d < 1", p->n_group);
    MOE_CHECK(p->n_group <= kMaxGroups, "n_group = %d > %d", p->n_group, kMaxGroups);
    MOE_CHECK(E % p->n_group == 0, "E = %d not divisible by n_group = %d", E, p->n_group);
    MOE_CHECK(p->topk_group >= 1 && p->topk_group <= p->n_group,
              "topk_group = %d outside [1, n_group = %d]", p->topk_group, p->n_group);
    MOE_CHECK(p->n_group == 1 || E / p->n_group >= 2,
              "n_group = %d leaves %d expert(s) per group; the group score needs 2", p->n_group,
              E / p->n_group);
    return MOE_OK;
}

int check_weights(const moe_expert_weights_t* w, const char* what, int shared) {
    MOE_CHECK(w, "%s weights are NULL", what);
    MOE_CHECK(w->bits == 16 || w->bits == 8 || w->bits == 4, "%s weights: bits = %d (16, 8 or 4)",
              what, w->bits);
    MOE_CHECK(!shared || w->bits == 16, "%s weights must be bf16 (bits 16)", what);
    MOE_CHECK(w->gate && w->up && w->down, "%s weights: gate/up/down pointer is NULL", what);
    MOE_CHECK(aligned(w->gate, 16) && aligned(w->up, 16) && aligned(w->down, 16),
              "%s weights: pointers must be 16-byte aligned", what);
    if (w->bits != 16) {
        MOE_CHECK(w->group_size == 32 || w->group_size == 64 || w->group_size == 128,
                  "%s weights: group_size = %d (32, 64 or 128)", what, w->group_size);
        MOE_CHECK(w->gate_scale && w->gate_bias && w->up_scale && w->up_bias && w->down_scale &&
                      w->down_bias,
                  "%s weights: 4-bit scale/bias pointer is NULL", what);
        MOE_CHECK(aligned(w->gate_scale, 2) && aligned(w->gate_bias, 2) &&
                      aligned(w->up_scale, 2) && aligned(w->up_bias, 2) &&
                      aligned(w->down_scale, 2) && aligned(w->down_bias, 2),
                  "%s weights: fp16 scale/bias pointers must be 2-byte aligned", what);
    }
    return MOE_OK;
}

int check_dims(int64_t T, int32_t d, int32_t I, int32_t E, int32_t K) {
    MOE_CHECK(T >= 0, "T = %lld < 0", (long long)T);
    MOE_CHECK(d >= 128 && d % 128 == 0, "d = %d must be a positive multiple of 128", d);
    MOE_CHECK(I >= 128 && I % 128 == 0, "I = %d must be a positive multiple of 128", I);
    MOE_CHECK(E >= 1 && E <= kMaxExperts, "E = %d outside [1, %d]", E, kMaxExperts);
    MOE_CHECK(K >= 1 && K <= kMaxTopK, "K = %d outside [1, %d]", K, kMaxTopK);
    MOE_CHECK(T * (int64_t)K + T < ((int64_t)1 << 31), "T*K = %lld too large",
              (long long)(T * (int64_t)K));
    return MOE_OK;
}

// Token tile of the expert GEMMs.  With tokens on the N side an UMMA (M = 128 weight rows,
// K = 16) costs the same for N = 16 .. 64 (its 128 x 16 A operand sets the pace), so wide
// token tiles are free and avoid streaming a weight tile once per 16 tokens: 64-token tiles
// while the experts see few tokens on average, 128 (bf16 only: the 4-bit TMEM-A path has no
// TMEM room for them) for mid-size batches, else 128-token tiles on the M side.
int expert_tok_tile(int64_t P, int32_t E, int32_t bits) {
    const int64_t avg = (P + E - 1) / E;
    if (avg <= 40) return 64;
    if (avg <= 96 && bits == 16) return 128;
    return 0;
}

// bf16 expert GEMMs with tokens on M run as CTA pairs (256-row tiles, cta_group::2 UMMAs)
// when the experts see many tokens: a pair streams a third fewer operand bytes per unit of
// tensor work and keeps six stages in flight instead of four (measured with 32 experts at
// 8192 tokens: gate/up 2.90 -> 2.76 ms, down 1.47 -> 1.41 ms), but an expert's last tile is
// padded to 256 rows instead of 128, and an UMMA costs the same whatever the share of real
// rows (with 256 experts at 8192 tokens, ~590 rows per expert hit: 3.27 -> 3.43 ms).
int expert_pair_tiles(int64_t P, int32_t E, int tok_tile, int32_t bits) {
    return tok_tile == 0 && bits == 16 && P >= (int64_t)1024 * E ? 1 : 0;
}

struct RouterPlan {
    int tok_tile;
    int ksplit;
    long long tiles;
};

RouterPlan router_plan(int64_t T, int32_t d, int32_t E) {
    RouterPlan rp;
    const int nsm = moe::num_sms();
    long long ttiles, ftiles;
    if (T <= 256) {
        rp.tok_tile = T <= 16 ? 16 : T <= 32 ? 32 : T <= 64 ? 64 : 128;
        ttiles = (T + rp.tok_tile - 1) / rp.tok_tile;
        ftiles = (E + 127) / 128;
    } else {
        rp.tok_tile = 0;
        ttiles = (T + 127) / 128;
        ftiles = (E + 255) / 256;
    }
    // K-split to spread the router weights over the SMs, but at least 8 k-blocks per split:
    // every split adds a partial-logit matrix that the gate must read back
    const int nkb = d / 64;
    rp.ksplit = 1;
    for (int ks = 1; ks <= nkb; ++ks)
        if (nkb % ks == 0 && ttiles * ftiles * ks <= nsm && nkb / ks >= 8) rp.ksplit = ks;
    rp.tiles = ttiles * ftiles * rp.ksplit;
    return rp;
}

// Workspace of the expert SwiGLU: x_perm [P, d] and h [P + T, I].
struct SwigluWs {
    size_t x_perm, h, total;
};
SwigluWs swiglu_ws(int64_t T, int32_t d, int32_t I, int32_t K, int has_shared) {
    SwigluWs w;
    const int64_t P = T * K;
    size_t off = 0;
    w.x_perm = off;
    off += align256((size_t)P * d * 2);
    w.h = off;
    off += align256((size_t)(P + (has_shared ? T : 0)) * I * 2);
    w.total = off;
    return w;
}

// Whole-layer workspace.
struct ForwardWs {
    size_t logits_part, inds, scores, counts, offsets, perm, inv, expert_out, swiglu, total;
};
ForwardWs forward_ws(int64_t T, int32_t d, int32_t I, int32_t E, int32_t K, int has_shared,
                     int ksplit) {
    ForwardWs w;
    const int64_t P = T * K;
    size_t off = 0;
    w.logits_part = off; off += align256((size_t)ksplit * T * E * 4);
    w.inds = off;        off += align256((size_t)P * 4);
    w.scores = off;      off += align256((size_t)P * 4);
    w.counts = off;      off += align256((size_t)E * 4);
    w.offsets = off;     off += align256((size_t)(E + 1) * 4);
    w.perm = off;        off += align256((size_t)P * 4);
    w.inv = off;         off += align256((size_t)P * 4);
    w.expert_out = off;  off += align256((size_t)(P + (has_shared ? T : 0)) * d * 2);
    w.swiglu = off;      off += swiglu_ws(T, d, I, K, has_shared).total;
    w.total = off;
    return w;
}

// Maximum K-split of the router over every device plan (the workspace must not depend on
// the device it is sized on): router_plan keeps at least 8 of the d/64 k-blocks per split,
// so no plan splits more than d/512 ways.
int router_ksplit_bound(int32_t d) { return d / 512 > 1 ? d / 512 : 1; }

int run_swiglu(const void* x, int64_t T, int32_t d, int32_t I, int32_t E, int32_t K,
               const int32_t* offsets, const int32_t* perm, const moe_expert_weights_t* ex,
               const moe_expert_weights_t* sh, void* out, uint8_t* ws, cudaStream_t s) {
    const int64_t P = T * K;
    const SwigluWs lw = swiglu_ws(T, d, I, K, sh != nullptr);
    void* x_perm = ws + lw.x_perm;
    void* h = ws + lw.h;
    const int has_shared = sh != nullptr;
    MOE_LAUNCH(moe::launch_gather_rows(x, perm, offsets, E, K, P, d, x_perm, s), "gather rows");
    MOE_CUDA(phase(4, s), "phase event");
    const int tok = expert_tok_tile(P, E, ex->bits);
    const int tokn = tok ? tok : 128;
    const long long mt_bound = (P + tokn - 1) / tokn + E + (has_shared ? (T + tokn - 1) / tokn : 0);

    moe::GemmArgs g = {};
    g.mode = moe::kGateUp;
    g.act = x_perm;
    g.act_rows = P;
    g.act_shared = x;
    g.shared_act_row0 = 0;
    g.offsets = offsets;
    g.E = E;
    g.has_shared = has_shared;
    g.shared_rows = T;
    g.shared_out_row0 = P;
    g.Kdim = d;
    g.F = I;
    g.ksplit = 1;
    g.w = {ex->bits, ex->gate, ex->up, ex->gate_scale, ex->gate_bias, ex->up_scale, ex->up_bias,
           ex->group_size};
    if (has_shared) g.ws = {16, sh->gate, sh->up, nullptr, nullptr, nullptr, nullptr};
    g.out = h;
    g.out_ld = I;
    g.tok_tile = tok;
    g.pair = expert_pair_tiles(P, E, tok, ex->bits);
    g.max_tiles = mt_bound * (I / 128);
    MOE_LAUNCH(moe::launch_gemm(g, s), "gate/up GEMM");
    MOE_CUDA(phase(5, s), "phase event");

    moe::GemmArgs dn = g;
    dn.mode = moe::kDown;
    dn.act = h;
    dn.act_rows = P + (has_shared ? T : 0);
    dn.act_shared = h;
    dn.shared_act_row0 = P;
    dn.Kdim = I;
    dn.F = d;
    dn.w = {ex->bits, ex->down, nullptr, ex->down_scale, ex->down_bias, nullptr, nullptr,
            ex->group_size};
    if (has_shared) dn.ws = {16, sh->down, nullptr, nullptr, nullptr, nullptr, nullptr};
    dn.out = out;
    dn.out_ld = d;
    // quantised experts: the down GEMM takes its tokens on M at every batch size (256 output
    // rows per tile and UMMA, half the tiles of the tokens-on-N form over the short I-long
    // main loop; measured at decode, 4-bit T=32: 0.336 -> 0.272 ms, 8-bit 0.372 -> 0.302 ms,
    // while the gate/up GEMM stays faster with tokens on N)
    const int tok_dn = ex->bits != 16 ? 0 : tok;
    const long long mt_dn = tok_dn == tok ? mt_bound
                                          : (P + 127) / 128 + E + (has_shared ? (T + 127) / 128 : 0);
    dn.tok_tile = tok_dn;
    dn.pair = expert_pair_tiles(P, E, tok_dn, ex->bits);
    dn.max_tiles = mt_dn * ((d + (tok_dn ? 127 : 255)) / (tok_dn ? 128 : 256));
    MOE_LAUNCH(moe::launch_gemm(dn, s), "down GEMM");
    MOE_CUDA(phase(6, s), "phase event");
    return MOE_OK;
}


// Whole-layer workspace of moe_forward_ex: moe_forward's plus the per-token shared gate.
struct ForwardExWs {
    ForwardWs base;
    size_t gate, total;
};
ForwardExWs forward_ex_ws(const moe_layer_args_t& a) {
    ForwardExWs w;
    w.base = forward_ws(a.T, a.d, a.I, a.E, a.params.top_k, a.shared != nullptr,
                        router_ksplit_bound(a.d));
    w.gate = w.base.total;
    w.total = w.gate + (a.w_shared_gate ? align256((size_t)a.T * 4) : 0);
    return w;
}

// The layer: router linear -> gate -> dispatch -> expert SwiGLU (+ shared) -> combine.
int forward_impl(const moe_layer_args_t& A, void* ws, size_t ws_bytes, cudaStream_t s) {
    const int64_t T = A.T;
    const int32_t d = A.d, I = A.I, E = A.E;
    const moe_route_params_t* params = &A.params;
    const bool softmax = A.route_kind == MOE_ROUTE_SOFTMAX;
    MOE_CHECK(A.route_kind == MOE_ROUTE_DEEPSEEK || softmax, "route_kind %d unknown",
              (int)A.route_kind);
    MOE_CHECK(A.w_router && (softmax || A.bias) && ws && (T == 0 || (A.x && A.y)),
              "NULL pointer argument");
    int rc;
    if (softmax) {
        MOE_CHECK(E >= 1 && E <= kMaxExperts, "E = %d outside [1, %d]", E, kMaxExperts);
        MOE_CHECK(params->top_k >= 1 && params->top_k <= E, "top_k = %d outside [1, E = %d]",
                  params->top_k, E);
    } else {
        rc = check_route_params(E, params);
        if (rc) return rc;
    }
    const int32_t K = params->top_k;
    rc = check_dims(T, d, I, E, K);
    if (rc) return rc;
    rc = check_weights(A.experts, "expert", 0);
    if (rc) return rc;
    if (A.shared) {
        rc = check_weights(A.shared, "shared expert", 1);
        if (rc) return rc;
    }
    MOE_CHECK(!A.w_shared_gate || A.shared, "w_shared_gate given without a shared expert");
    MOE_CHECK(aligned(A.x, 16) && aligned(A.w_router, 16) && aligned(A.y, 16) &&
                  aligned(A.w_shared_gate, 16),
              "x, w_router, w_shared_gate and y must be 16-byte aligned");
    MOE_CHECK(aligned(ws, 256), "ws must be 256-byte aligned");
    const int has_shared = A.shared != nullptr;
    const ForwardExWs lx = forward_ex_ws(A);
    const ForwardWs& lw = lx.base;
    MOE_CHECK(ws_bytes >= lx.total, "ws_bytes = %zu < %zu required", ws_bytes, lx.total);
    if (T == 0) return MOE_OK;
    rc = check_device();
    if (rc) return rc;

    uint8_t* w = static_cast<uint8_t*>(ws);
    const int64_t P = T * K;
    float* lpart = reinterpret_cast<float*>(w + lw.logits_part);
    int32_t* inds = A.inds_out ? A.inds_out : reinterpret_cast<int32_t*>(w + lw.inds);
    float* scores = A.scores_out ? A.scores_out : reinterpret_cast<float*>(w + lw.scores);
    int32_t* counts = reinterpret_cast<int32_t*>(w + lw.counts);
    int32_t* offsets = reinterpret_cast<int32_t*>(w + lw.offsets);
    int32_t* perm = reinterpret_cast<int32_t*>(w + lw.perm);
    int32_t* inv = reinterpret_cast<int32_t*>(w + lw.inv);
    void* eo = w + lw.expert_out;
    float* sgate = A.w_shared_gate ? reinterpret_cast<float*>(w + lx.gate) : nullptr;

    MOE_CUDA(phase(0, s), "phase event");
    // a1: router linear, K-split partial sums
    const RouterPlan rp = router_plan(T, d, E);
    moe::GemmArgs g = {};
    g.mode = moe::kRouter;
    g.act = A.x;
    g.act_rows = T;
    g.offsets = nullptr;
    g.single_rows = T;
    g.E = 1;
    g.Kdim = d;
    g.F = E;
    g.ksplit = rp.ksplit;
    g.split_stride = (long long)T * E;
    g.w = {16, A.w_router, nullptr, nullptr, nullptr, nullptr, nullptr};
    g.out = lpart;
    g.out_ld = E;
    g.tok_tile = rp.tok_tile;
    g.max_tiles = rp.tiles;
    MOE_LAUNCH(moe::launch_gemm(g, s), "router GEMM");
    MOE_CUDA(phase(1, s), "phase event");
    // decode-sized batches: the layer's later kernels start while the one before them
    // finishes (measured at T = 128: 1.099 -> 1.080 ms per layer).  Not for large batches
    // (a programmatic launch of the prefill gate/up GEMM measured 5.49 -> 6.03 ms at T = 8192,
    // where launch gaps are a negligible share anyway), nor while the phase events that time
    // each kernel are recorded between them.
    PdlScope pdl;
    if (g_phase_n == 0 && T * K < moe::kPermMultiMin) pdl.on();

    // a2: gate (sums the partials in split order, adds the offset)
    moe::RouteArgs ra = {};
    ra.logits = lpart;
    ra.bf16 = 0;
    ra.nsplit = rp.ksplit;
    ra.split_stride = (long long)T * E;
    ra.logit_offset = A.logit_offset;
    ra.bias = A.bias;
    ra.rows = T;
    ra.E = E;
    ra.top_k = K;
    ra.n_group = softmax ? 1 : params->n_group;
    ra.topk_group = softmax ? 1 : params->topk_group;
    ra.norm = params->norm_topk_prob != 0;
    ra.scale = params->routed_scaling_factor;
    ra.inds = inds;
    ra.scores = scores;
    ra.logits_out = A.logits_out;
    ra.softmax = softmax ? 1 : 0;
    MOE_LAUNCH(moe::launch_route(ra, s), "route kernel");
    MOE_CUDA(phase(2, s), "phase event");

    // a3: dispatch
    // (the expert-output buffer, written only by the down GEMM, is the dispatch's scratch)
    MOE_LAUNCH(moe::launch_permute(inds, P, E, counts, offsets, perm, inv, s, eo,
                                 (size_t)(P + (has_shared ? T : 0)) * d * 2),
             "permute kernel");
    MOE_CUDA(phase(3, s), "phase event");

    // a4 + a5 (+ a7): expert SwiGLU GEMMs, shared expert as the last group
    rc = run_swiglu(A.x, T, d, I, E, K, offsets, perm, A.experts, A.shared, eo, w + lw.swiglu,
                    s);
    if (rc) return rc;

    // a6: combine (the gated shared expert weighs its row by sigmoid(x . w_shared_gate))
    if (sgate)
        MOE_LAUNCH(moe::launch_shared_gate(A.x, T, d, A.w_shared_gate, sgate, s), "shared gate");
    const void* so = has_shared ? static_cast<const void*>(static_cast<const uint8_t*>(eo) +
                                                           (size_t)P * d * 2)
                                : nullptr;
    MOE_LAUNCH(moe::launch_combine(eo, scores, inv, so, T, K, d, A.y, s, sgate), "combine kernel");
    MOE_CUDA(phase(7, s), "phase event");
    return MOE_OK;
}

}  // namespace

int moe::set_error(int code, const char* msg) {
    g_err = msg;
    return code;
}

bool moe::pdl_enabled() { return g_pdl; }

extern "C" {

const char* moe_last_error(void) { return g_err.c_str(); }

int32_t moe_version(void) { return 100; }

int moe_device_status(int32_t clear, moe_stream_t stream) {
    int rc = check_device();
    if (rc) return rc;
    unsigned int st = 0;
    MOE_CUDA(moe::read_device_status(&st, clear, (cudaStream_t)stream), "status read");
    if (st == 5)
        return fail(MOE_ERR_CUDA, "a CTA pair of an expert GEMM held different TMEM columns "
                                  "(status %u); the GEMM did no work", st);
    if (st != 0) return fail(MOE_ERR_TIMEOUT, "a device-side wait gave up (status %u)", st);
    return MOE_OK;
}

int moe_indexer_topk(const void* scores, moe_dtype_t dtype, int64_t rows, int32_t n,
                     int64_t ld, const int32_t* lengths, int32_t k, int32_t* inds,
                     uint8_t* mask, int64_t mask_ld, moe_stream_t stream) {
    begin_call();
    MOE_CHECK(dtype == MOE_DTYPE_F32 || dtype == MOE_DTYPE_BF16, "dtype %d unknown", (int)dtype);
    MOE_CHECK(rows >= 0, "rows = %lld < 0", (long long)rows);
    MOE_CHECK(n >= 0, "n = %d < 0", n);
    MOE_CHECK(ld >= n, "ld = %lld < n = %d", (long long)ld, n);
    MOE_CHECK(k >= 1 && k <= (1 << 20), "k = %d outside [1, 2^20]", k);
    MOE_CHECK(!mask || mask_ld >= n, "mask_ld = %lld < n = %d", (long long)mask_ld, n);
    MOE_CHECK(rows == 0 || (inds && (n == 0 || scores)), "NULL pointer argument");
    if (rows == 0) return MOE_OK;
    int rc = check_device();
    if (rc) return rc;
    moe::TopkArgs a = {};
    a.scores = scores;
    a.bf16 = dtype == MOE_DTYPE_BF16;
    a.rows = rows;
    a.n = n;
    a.ld = ld;
    a.lengths = lengths;
    a.k = k;
    a.inds = inds;
    a.mask = mask;
    a.mask_ld = mask_ld;
    moe::indexer_topk_plan(a);
    MOE_LAUNCH(moe::launch_indexer_topk(a, (cudaStream_t)stream), "indexer top-k kernel");
    return MOE_OK;
}

int moe_watchdog_selftest(int64_t limit_ns, moe_stream_t stream) {
    begin_call();
    MOE_CHECK(limit_ns >= 1000 && limit_ns <= 1000000000, "limit_ns = %lld outside [1e3, 1e9]",
              (long long)limit_ns);
    int rc = check_device();
    if (rc) return rc;
    MOE_LAUNCH(moe::launch_watchdog_selftest((unsigned long long)limit_ns, (cudaStream_t)stream),
             "watchdog self-test kernel");
    return MOE_OK;
}

int moe_route_deepseek(const void* logits, moe_dtype_t dtype, int64_t rows, int32_t E,
                       const float* bias, const moe_route_params_t* params, int32_t* inds,
                       float* scores, moe_stream_t stream) {
    begin_call();
    MOE_CHECK(bias && (rows == 0 || (logits && inds && scores)), "NULL pointer argument");
    MOE_CHECK(dtype == MOE_DTYPE_F32 || dtype == MOE_DTYPE_BF16, "dtype %d unknown", (int)dtype);
    MOE_CHECK(rows >= 0, "rows = %lld < 0", (long long)rows);
    int rc = check_route_params(E, params);
    if (rc) return rc;
    if (rows == 0) return MOE_OK;
    rc = check_device();
    if (rc) return rc;
    moe::RouteArgs a = {};
    a.logits = logits;
    a.bf16 = dtype == MOE_DTYPE_BF16;
    a.nsplit = 1;
    a.split_stride = 0;
    a.logit_offset = nullptr;
    a.bias = bias;
    a.rows = rows;
    a.E = E;
    a.top_k = params->top_k;
    a.n_group = params->n_group;
    a.topk_group = params->topk_group;
    a.norm = params->norm_topk_prob != 0;
    a.scale = params->routed_scaling_factor;
    a.inds = inds;
    a.scores = scores;
    a.logits_out = nullptr;
    MOE_LAUNCH(moe::launch_route(a, (cudaStream_t)stream), "route kernel");
    return MOE_OK;
}

int moe_permute(const int32_t* inds, int64_t T, int32_t K, int32_t E, int32_t* counts,
                int32_t* offsets, int32_t* perm, int32_t* inv_perm, moe_stream_t stream) {
    begin_call();
    MOE_CHECK(counts && offsets && (T * (int64_t)K == 0 || (inds && perm && inv_perm)),
              "NULL pointer argument");
    MOE_CHECK(T >= 0, "T = %lld < 0", (long long)T);
    MOE_CHECK(K >= 1, "K = %d < 1", K);
    MOE_CHECK(E >= 1 && E <= kMaxExperts, "E = %d outside [1, %d]", E, kMaxExperts);
    MOE_CHECK(T * (int64_t)K < ((int64_t)1 << 31), "T*K too large");
    int rc = check_device();
    if (rc) return rc;
    MOE_LAUNCH(moe::launch_permute(inds, T * K, E, counts, offsets, perm, inv_perm,
                                 (cudaStream_t)stream),
             "permute kernel");
    return MOE_OK;
}

int moe_router_logits(const void* x, int64_t T, int32_t d, const void* w_router, int32_t E,
                      const float* logit_offset, float* logits, moe_stream_t stream) {
    begin_call();
    MOE_CHECK(w_router && (T == 0 || (x && logits)), "NULL pointer argument");
    MOE_CHECK(T >= 0, "T = %lld < 0", (long long)T);
    MOE_CHECK(d >= 64 && d % 64 == 0, "d = %d must be a positive multiple of 64", d);
    MOE_CHECK(E >= 1 && E <= kMaxExperts, "E = %d outside [1, %d]", E, kMaxExperts);
    MOE_CHECK(aligned(x, 16) && aligned(w_router, 16), "x and w_router must be 16-byte aligned");
    if (T == 0) return MOE_OK;
    int rc = check_device();
    if (rc) return rc;
    // one K split, written straight to `logits`, then the offset is added by the gate's
    // reduction kernel only when requested
    moe::GemmArgs g = {};
    g.mode = moe::kRouter;
    g.act = x;
    g.act_rows = T;
    g.offsets = nullptr;
    g.single_rows = T;
    g.E = 1;
    g.Kdim = d;
    g.F = E;
    g.ksplit = 1;
    g.split_stride = 0;
    g.w = {16, w_router, nullptr, nullptr, nullptr, nullptr, nullptr};
    g.out = logits;
    g.out_ld = E;
    g.tok_tile = T <= 256 ? (T <= 16 ? 16 : T <= 32 ? 32 : T <= 64 ? 64 : 128) : 0;
    const int tokn = g.tok_tile ? g.tok_tile : 128;
    g.max_tiles = ((T + tokn - 1) / tokn) * ((E + (g.tok_tile ? 127 : 255)) / (g.tok_tile ? 128 : 256));
    MOE_LAUNCH(moe::launch_gemm(g, (cudaStream_t)stream), "router GEMM");
    if (logit_offset)
        MOE_LAUNCH(moe::launch_add_offset(logits, T, E, logit_offset, (cudaStream_t)stream),
                 "logit offset");
    return MOE_OK;
}

size_t moe_grouped_swiglu_workspace_bytes(int64_t T, int32_t d, int32_t I, int32_t E, int32_t K,
                                          int32_t has_shared) {
    (void)E;
    if (T < 0 || d < 0 || I < 0 || K < 0) return 0;
    return swiglu_ws(T, d, I, K, has_shared != 0).total;
}

int moe_grouped_swiglu(const void* x, int64_t T, int32_t d, int32_t I, int32_t E, int32_t K,
                       const int32_t* offsets, const int32_t* perm,
                       const moe_expert_weights_t* experts, const moe_expert_weights_t* shared,
                       void* out, void* ws, size_t ws_bytes, moe_stream_t stream) {
    begin_call();
    MOE_CHECK(offsets && ws && (T == 0 || (x && perm && out)), "NULL pointer argument");
    int rc = check_dims(T, d, I, E, K);
    if (rc) return rc;
    rc = check_weights(experts, "expert", 0);
    if (rc) return rc;
    if (shared) {
        rc = check_weights(shared, "shared expert", 1);
        if (rc) return rc;
    }
    MOE_CHECK(aligned(x, 16) && aligned(out, 16), "x and out must be 16-byte aligned");
    MOE_CHECK(aligned(ws, 256), "ws must be 256-byte aligned");
    const size_t need = swiglu_ws(T, d, I, K, shared != nullptr).total;
    MOE_CHECK(ws_bytes >= need, "ws_bytes = %zu < %zu required", ws_bytes, need);
    if (T == 0) return MOE_OK;
    rc = check_device();
    if (rc) return rc;
    return run_swiglu(x, T, d, I, E, K, offsets, perm, experts, shared, out,
                      static_cast<uint8_t*>(ws), (cudaStream_t)stream);
}

int moe_combine(const void* expert_out, const float* scores, const int32_t* inv_perm,
                const void* shared_out, int64_t T, int32_t K, int32_t d, void* y,
                moe_stream_t stream) {
    begin_call();
    MOE_CHECK(T == 0 || (expert_out && scores && inv_perm && y), "NULL pointer argument");
    MOE_CHECK(T >= 0, "T = %lld < 0", (long long)T);
    MOE_CHECK(K >= 1, "K = %d < 1", K);
    MOE_CHECK(d >= 8 && d % 8 == 0, "d = %d must be a positive multiple of 8", d);
    MOE_CHECK(aligned(expert_out, 16) && aligned(y, 16) && (!shared_out || aligned(shared_out, 16)),
              "expert_out, shared_out and y must be 16-byte aligned");
    if (T == 0) return MOE_OK;
    int rc = check_device();
    if (rc) return rc;
    MOE_LAUNCH(moe::launch_combine(expert_out, scores, inv_perm, shared_out, T, K, d, y,
                                 (cudaStream_t)stream),
             "combine kernel");
    return MOE_OK;
}

size_t moe_forward_workspace_bytes(int64_t T, int32_t d, int32_t I, int32_t E, int32_t top_k,
                                   int32_t has_shared) {
    if (T < 0 || d < 0 || I < 0 || E < 0 || top_k < 0) return 0;
    return forward_ws(T, d, I, E, top_k, has_shared != 0, router_ksplit_bound(d)).total;
}

int moe_forward(const void* x, int64_t T, int32_t d, int32_t I, int32_t E,
                const void* w_router, const float* bias, const float* logit_offset,
                const moe_route_params_t* params, const moe_expert_weights_t* experts,
                const moe_expert_weights_t* shared, void* y, int32_t* inds_out,
                float* scores_out, float* logits_out, void* ws, size_t ws_bytes,
                moe_stream_t stream) {
    begin_call();
    MOE_CHECK(params, "params is NULL");
    moe_layer_args_t a = {};
    a.route_kind = MOE_ROUTE_DEEPSEEK;
    a.x = x;
    a.T = T;
    a.d = d;
    a.I = I;
    a.E = E;
    a.w_router = w_router;
    a.logit_offset = logit_offset;
    a.bias = bias;
    a.params = *params;
    a.experts = experts;
    a.shared = shared;
    a.w_shared_gate = nullptr;
    a.y = y;
    a.inds_out = inds_out;
    a.scores_out = scores_out;
    a.logits_out = logits_out;
    return forward_impl(a, ws, ws_bytes, (cudaStream_t)stream);
}

size_t moe_forward_ex_workspace_bytes(const moe_layer_args_t* a) {
    if (!a || a->T < 0 || a->d < 0 || a->I < 0 || a->E < 0 || a->params.top_k < 0) return 0;
    return forward_ex_ws(*a).total;
}

int moe_forward_ex(const moe_layer_args_t* args, void* ws, size_t ws_bytes, moe_stream_t stream) {
    begin_call();
    MOE_CHECK(args, "args is NULL");
    return forward_impl(*args, ws, ws_bytes, (cudaStream_t)stream);
}

int moe_route_softmax(const void* logits, moe_dtype_t dtype, int64_t rows, int32_t E,
                      int32_t top_k, int32_t* inds, float* scores, moe_stream_t stream) {
    begin_call();
    MOE_CHECK(rows == 0 || (logits && inds && scores), "NULL pointer argument");
    MOE_CHECK(dtype == MOE_DTYPE_F32 || dtype == MOE_DTYPE_BF16, "dtype %d unknown", (int)dtype);
    MOE_CHECK(rows >= 0, "rows = %lld < 0", (long long)rows);
    MOE_CHECK(E >= 1 && E <= kMaxExperts, "E = %d outside [1, %d]", E, kMaxExperts);
    MOE_CHECK(top_k >= 1 && top_k <= E && top_k <= kMaxTopK, "top_k = %d outside [1, min(E, %d)]",
              top_k, kMaxTopK);
    if (rows == 0) return MOE_OK;
    int rc = check_device();
    if (rc) return rc;
    moe::RouteArgs a = {};
    a.logits = logits;
    a.bf16 = dtype == MOE_DTYPE_BF16;
    a.nsplit = 1;
    a.rows = rows;
    a.E = E;
    a.top_k = top_k;
    a.n_group = 1;
    a.topk_group = 1;
    a.scale = 1.0f;
    a.inds = inds;
    a.scores = scores;
    a.softmax = 1;
    MOE_LAUNCH(moe::launch_route(a, (cudaStream_t)stream), "route kernel");
    return MOE_OK;
}

int moe_shared_gate(const void* x, int64_t T, int32_t d, const void* w_gate, float* gate,
                    moe_stream_t stream) {
    begin_call();
    MOE_CHECK(w_gate && (T == 0 || (x && gate)), "NULL pointer argument");
    MOE_CHECK(T >= 0, "T = %lld < 0", (long long)T);
    MOE_CHECK(d >= 8 && d % 8 == 0, "d = %d must be a positive multiple of 8", d);
    MOE_CHECK(aligned(x, 16) && aligned(w_gate, 16), "x and w_gate must be 16-byte aligned");
    if (T == 0) return MOE_OK;
    int rc = check_device();
    if (rc) return rc;
    MOE_LAUNCH(moe::launch_shared_gate(x, T, d, w_gate, gate, (cudaStream_t)stream), "shared gate");
    return MOE_OK;
}

int moe_combine_gated(const void* expert_out, const float* scores, const int32_t* inv_perm,
                      const void* shared_out, const float* shared_gate, int64_t T, int32_t K,
                      int32_t d, void* y, moe_stream_t stream) {
    begin_call();
    MOE_CHECK(T == 0 || (expert_out && scores && inv_perm && shared_out && shared_gate && y),
              "NULL pointer argument");
    MOE_CHECK(T >= 0, "T = %lld < 0", (long long)T);
    MOE_CHECK(K >= 1, "K = %d < 1", K);
    MOE_CHECK(d >= 8 && d % 8 == 0, "d = %d must be a positive multiple of 8", d);
    MOE_CHECK(aligned(expert_out, 16) && aligned(y, 16) && aligned(shared_out, 16),
              "expert_out, shared_out and y must be 16-byte aligned");
    if (T == 0) return MOE_OK;
    int rc = check_device();
    if (rc) return rc;
    MOE_LAUNCH(moe::launch_combine(expert_out, scores, inv_perm, shared_out, T, K, d, y,
                                 (cudaStream_t)stream, shared_gate),
             "combine kernel");
    return MOE_OK;
}

int moe_set_fault(int32_t kind, int32_t at) {
    begin_call();
    MOE_CHECK(kind == MOE_FAULT_NONE || kind == MOE_FAULT_LAUNCH, "fault kind %d unknown", kind);
    MOE_CHECK(at >= 0, "at = %d < 0", at);
    fault_init();
    g_fault_at.store(at, std::memory_order_relaxed);
    g_fault_kind.store(kind, std::memory_order_release);
    return MOE_OK;
}

int moe_get_fault(int32_t* kind, int32_t* at) {
    begin_call();
    MOE_CHECK(kind && at, "NULL pointer argument");
    fault_init();
    *kind = g_fault_kind.load(std::memory_order_acquire);
    *at = g_fault_at.load(std::memory_order_relaxed);
    return MOE_OK;
}

int moe_set_phase_events(void* const* events, int32_t n) {
    begin_call();
    MOE_CHECK(n >= 0 && n <= kMaxPhaseEvents, "n = %d outside [0, %d]", n, kMaxPhaseEvents);
    MOE_CHECK(n == 0 || events, "events is NULL");
    for (int i = 0; i < n; ++i) g_phase_ev[i] = static_cast<cudaEvent_t>(events[i]);
    g_phase_n = events ? n : 0;
    return MOE_OK;
}

}  // extern "C"
