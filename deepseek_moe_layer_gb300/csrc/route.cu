// route.cu -- the DeepSeek gate (and the softmax route), one warp per token.
//
// Source: "feat(engine): E1 DeepSeek-style MoE gate (sigmoid, group top-k, bias) (#108)",
// section "Algorithm (mlx-lm group_expert_select)": sigmoid of the f32 logits, bias added
// for selection only, group score = sum of the two largest biased scores of the group,
// the worst n_group - topk_group groups zeroed (skipped when that is 0), top-k of the
// biased scores, weights taken from the pre-bias sigmoid, renormalised only for
// top_k > 1 with norm_topk_prob, then scaled by routed_scaling_factor.
//
// Layout: lane l of the warp holds experts [l*EPL, l*EPL + EPL).  Every comparison runs on
// an order-preserving 32-bit key of the fp32 value (NaN lowest, -0 == +0), so a warp-wide
// arg-max is one redux.max on the keys plus one redux.min on the indices of the maxima:
// equal values resolve to the lower expert index, and groups to the lower group index.
#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

MOE_DEV uint32_t okey(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u << 1) == 0u) u = 0u;               // -0.0 -> +0.0
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0u;  // NaN lowest
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
MOE_DEV float okey_value(uint32_t k) {
    uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}

// SOFTMAX: the softmax route instead of the DeepSeek gate: the K largest logits are
// selected (softmax is strictly increasing, so they are the K most probable experts) and
// their weights exp(l_k - l_max) / sum_sel exp(l_j - l_max) are the selected softmax
// probabilities renormalised over the selection, always (no bias, groups or scale).
template <int EPL, bool SOFTMAX>
__global__ void __launch_bounds__(256) route_kernel(const RouteArgs a) {
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= a.rows) return;
    const int E = a.E;
    const int e0 = lane * EPL;

    // ---- logits: sum of the split partials in split order, plus the optional offset ----
    float lg[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) lg[i] = 0.0f;
    if (!a.bf16) {
        const float* base = static_cast<const float*>(a.logits) + row * E;
        int s0 = 0;
        if constexpr (EPL % 4 == 0) {
            // batches of 8 splits: all loads issued before the (in-order) additions
            const bool vec = (E & 3) == 0 && (reinterpret_cast<uintptr_t>(base) & 15) == 0 &&
                             (a.split_stride & 3) == 0;
            if (vec && e0 < E) {
                for (; s0 + 8 <= a.nsplit; s0 += 8) {
                    float4 v[8][EPL / 4];
#pragma unroll
                    for (int u = 0; u < 8; ++u)
#pragma unroll
                        for (int i = 0; i < EPL / 4; ++i)
                            v[u][i] = (e0 + 4 * i < E)  // E % 4 == 0: a vector is all in or out
                                          ? *reinterpret_cast<const float4*>(
                                                base + (long long)(s0 + u) * a.split_stride +
                                                e0 + 4 * i)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
#pragma unroll
                        for (int i = 0; i < EPL / 4; ++i) {
                            lg[4 * i] += v[u][i].x;
                            lg[4 * i + 1] += v[u][i].y;
                            lg[4 * i + 2] += v[u][i].z;
                            lg[4 * i + 3] += v[u][i].w;
                        }
                }
            }
        }
        for (int s = s0; s < a.nsplit; ++s) {
            const float* p = base + (long long)s * a.split_stride;
            if constexpr (EPL % 4 == 0) {
                if ((E & 3) == 0 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
#pragma unroll
                    for (int i = 0; i < EPL; i += 4) {
                        if (e0 + i < E) {
                            const float4 v = *reinterpret_cast<const float4*>(p + e0 + i);
                            lg[i] += v.x; lg[i + 1] += v.y; lg[i + 2] += v.z; lg[i + 3] += v.w;
                        }
                    }
                    continue;
                }
            }
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (e0 + i < E) lg[i] += p[e0 + i];
        }
    } else {
        const __nv_bfloat16_raw* p =
            static_cast<const __nv_bfloat16_raw*>(a.logits) + row * E;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (e0 + i < E) lg[i] = __uint_as_float(((uint32_t)p[e0 + i].x) << 16);
    }

    // ---- sigmoid, bias for selection ----
    float orig[EPL];
    uint32_t key[EPL];
    uint32_t taken = 0;  // bit i: slot i is not selectable (taken, or beyond E)
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = e0 + i;
        if (e < E) {
            float l = lg[i];
            if (a.logit_offset) l = l + a.logit_offset[e];
            if (a.logits_out) a.logits_out[row * E + e] = l;
            if (SOFTMAX) {
                orig[i] = l;  // the logit itself is carried to the weights
                key[i] = okey(l);
            } else {
                const float s = 1.0f / (1.0f + expf(-l));
                orig[i] = s;
                key[i] = okey(s + a.bias[e]);
            }
        } else {
            orig[i] = 0.0f;
            key[i] = 0u;
            taken |= 1u << i;
        }
    }

    // ---- group mask: keep the topk_group groups with the largest top-2 sums ----
    const int G = a.n_group;
    if (!SOFTMAX && G > 1 && G - a.topk_group > 0) {
        const int eg = E / G;
        uint32_t my_gk = 0;  // lane g (< G) holds the key of group g's score
        const int lpg = (eg % EPL == 0) ? eg / EPL : 0;
        if (lpg > 0 && lpg <= 32 && (lpg & (lpg - 1)) == 0) {
            // aligned groups: lanes [g*lpg, (g+1)*lpg) hold exactly group g
            uint32_t t1 = 0, t2 = 0;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                if (taken & (1u << i)) continue;
                const uint32_t k = key[i];
                if (k > t1) { t2 = t1; t1 = k; } else if (k > t2) { t2 = k; }
            }
            for (int off = 1; off < lpg; off <<= 1) {
                const uint32_t o1 = __shfl_xor_sync(kFull, t1, off);
                const uint32_t o2 = __shfl_xor_sync(kFull, t2, off);
                const uint32_t n2 = max(min(t1, o1), max(t2, o2));
                t1 = max(t1, o1);
                t2 = n2;
            }
            const uint32_t gk = okey(okey_value(t1) + okey_value(t2));
            my_gk = __shfl_sync(kFull, gk, min(lane, G - 1) * lpg);
        } else {
            // general layout: one warp-wide top-2 reduction per group
            for (int g = 0; g < G; ++g) {
                uint32_t t1 = 0, t2 = 0;
#pragma unroll
                for (int i = 0; i < EPL; ++i) {
                    const int e = e0 + i;
                    if ((taken & (1u << i)) || e / eg != g) continue;
                    const uint32_t k = key[i];
                    if (k > t1) { t2 = t1; t1 = k; } else if (k > t2) { t2 = k; }
                }
                for (int off = 1; off < 32; off <<= 1) {
                    const uint32_t o1 = __shfl_xor_sync(kFull, t1, off);
                    const uint32_t o2 = __shfl_xor_sync(kFull, t2, off);
                    const uint32_t n2 = max(min(t1, o1), max(t2, o2));
                    t1 = max(t1, o1);
                    t2 = n2;
                }
                if (lane == g) my_gk = okey(okey_value(t1) + okey_value(t2));
            }
        }
        // rank of group `lane` among all groups (larger score first, ties to lower index)
        int rank = 0;
        for (int h = 0; h < G; ++h) {
            const uint32_t hk = __shfl_sync(kFull, my_gk, h);
            rank += (hk > my_gk) || (hk == my_gk && h < lane);
        }
        const int kept = (lane < G) && (rank < a.topk_group);
        const uint32_t zero_key = okey(0.0f);
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int g = min((e0 + i) / eg, 31);
            const int k_i = __shfl_sync(kFull, kept, g);
            if (!(taken & (1u << i)) && !k_i) key[i] = zero_key;
        }
    }

    // ---- top-k selection, one warp arg-max per selected expert ----
    const int K = a.top_k;
    float my_w = 0.0f;
    int my_idx = 0;
    for (int r = 0; r < K; ++r) {
        uint32_t bk = 0, bi = 0xFFFFFFFFu;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            if (taken & (1u << i)) continue;
            if (bi == 0xFFFFFFFFu || key[i] > bk) { bk = key[i]; bi = (uint32_t)(e0 + i); }
        }
        const uint32_t m = __reduce_max_sync(kFull, bi == 0xFFFFFFFFu ? 0u : bk);
        const uint32_t w = __reduce_min_sync(kFull, (bi != 0xFFFFFFFFu && bk == m) ? bi : 0xFFFFFFFFu);
        const int owner = (int)(w / EPL);
        const int slot = (int)(w % EPL);
        float ov = 0.0f;
        if (lane == owner) {
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (i == slot) { ov = orig[i]; taken |= 1u << i; }
        }
        ov = __shfl_sync(kFull, ov, owner);
        if (lane == r) { my_w = ov; my_idx = (int)w; }
    }

    if (SOFTMAX) {
        // exp relative to the largest selected logit, renormalised over the selection
        const float lmax = __shfl_sync(kFull, my_w, 0);
        const float ex = lane < K ? expf(my_w - lmax) : 0.0f;
        float sum = 0.0f;
        for (int k = 0; k < K; ++k) sum += __shfl_sync(kFull, ex, k);
        if (lane < K) {
            a.inds[row * K + lane] = my_idx;
            a.scores[row * K + lane] = ex / sum;
        }
        return;
    }
    // ---- weights: renormalise (K > 1 and norm), then scale ----
    if (K > 1 && a.norm) {
        float sum = 0.0f;
        for (int k = 0; k < K; ++k) sum += __shfl_sync(kFull, my_w, k);
        my_w = my_w / sum;
    }
    my_w = my_w * a.scale;
    if (lane < K) {
        a.inds[row * K + lane] = my_idx;
        a.scores[row * K + lane] = my_w;
    }
}

__global__ void add_offset_kernel(float* __restrict__ logits, long long n, int E,
                                  const float* __restrict__ offset) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) logits[i] = logits[i] + offset[i % E];
}

}  // namespace

cudaError_t launch_add_offset(float* logits, long long T, int E, const float* offset,
                              cudaStream_t s) {
    const long long n = T * E;
    if (n == 0) return cudaSuccess;
    add_offset_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(logits, n, E, offset);
    return cudaGetLastError();
}

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s) {
    if (a.rows == 0) return cudaSuccess;
    const unsigned grid = (unsigned)((a.rows + 7) / 8);
    const int epl = a.E <= 32 ? 1 : a.E <= 64 ? 2 : a.E <= 128 ? 4 : a.E <= 256 ? 8
                  : a.E <= 512 ? 16 : 32;
    if (a.softmax) {
        switch (epl) {
            case 1: route_kernel<1, true><<<grid, 256, 0, s>>>(a); break;
            case 2: route_kernel<2, true><<<grid, 256, 0, s>>>(a); break;
            case 4: route_kernel<4, true><<<grid, 256, 0, s>>>(a); break;
            case 8: route_kernel<8, true><<<grid, 256, 0, s>>>(a); break;
            case 16: route_kernel<16, true><<<grid, 256, 0, s>>>(a); break;
            default: route_kernel<32, true><<<grid, 256, 0, s>>>(a); break;
        }
        return cudaGetLastError();
    }
    switch (epl) {
        case 1: route_kernel<1, false><<<grid, 256, 0, s>>>(a); break;
        case 2: route_kernel<2, false><<<grid, 256, 0, s>>>(a); break;
        case 4: route_kernel<4, false><<<grid, 256, 0, s>>>(a); break;
        case 8: route_kernel<8, false><<<grid, 256, 0, s>>>(a); break;
        case 16: route_kernel<16, false><<<grid, 256, 0, s>>>(a); break;
        default: route_kernel<32, false><<<grid, 256, 0, s>>>(a); break;
    }
    return cudaGetLastError();
}

}  // namespace moe
