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

constexpr uint32_t kEmpty = 0xFFFFFFFFu;

// A lane's two best selectable slots in the route's total order (key descending, expert
// index ascending): key, expert index (kEmpty: none) and the value the weight is made of.
struct Top2 {
    uint32_t k0, k1, i0, i1;
    float v0, v1;
};

// Top2 of the slots of this lane not marked in `skip`.  Slots are visited in increasing
// expert index and only a strictly larger key moves ahead, so equal keys keep the lower
// index first.
template <int EPL>
MOE_DEV Top2 lane_top2(const uint32_t (&key)[EPL], const float (&val)[EPL], uint32_t skip,
                       int e0) {
    Top2 t = {0u, 0u, kEmpty, kEmpty, 0.0f, 0.0f};
#pragma unroll
    for (int s = 0; s < EPL; ++s) {
        if (skip & (1u << s)) continue;
        const uint32_t k = key[s];
        const bool b0 = t.i0 == kEmpty || k > t.k0;
        const bool b1 = t.i1 == kEmpty || k > t.k1;
        if (b1) {
            t.k1 = b0 ? t.k0 : k;
            t.i1 = b0 ? t.i0 : (uint32_t)(e0 + s);
            t.v1 = b0 ? t.v0 : val[s];
        }
        if (b0) {
            t.k0 = k;
            t.i0 = (uint32_t)(e0 + s);
            t.v0 = val[s];
        }
    }
    return t;
}

// SOFTMAX: the softmax route instead of the DeepSeek gate: the K largest logits are
// selected (softmax is strictly increasing, so they are the K most probable experts) and
// their weights exp(l_k - l_max) / sum_sel exp(l_j - l_max) are the selected softmax
// probabilities renormalised over the selection, always (no bias, groups or scale).
//
// Each warp handles rows warp_id, warp_id + nwarps, ... (grid sized to the SMs).
template <int EPL, bool SOFTMAX>
__global__ void __launch_bounds__(256, EPL <= 8 ? 4 : 1) route_kernel(const RouteArgs a) {
    pdl_launch_dependents();
    pdl_wait();  // the logits come from the kernel before
    const int lane = threadIdx.x & 31;
    const long long nwarps = (long long)gridDim.x * 8;
    const int E = a.E;
    const int e0 = lane * EPL;
    // vector access to bias / offset / logits_out when E and the pointers allow it
    const bool vec_e = (EPL % 4 == 0) && (E & 3) == 0;
    const bool bias_vec = vec_e && (reinterpret_cast<uintptr_t>(a.bias) & 15) == 0;
    const bool off_vec = vec_e && (reinterpret_cast<uintptr_t>(a.logit_offset) & 15) == 0;
    const bool lo_vec = vec_e && (reinterpret_cast<uintptr_t>(a.logits_out) & 15) == 0;

    for (long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); row < a.rows;
         row += nwarps) {
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
    if (a.logit_offset) {
        if (off_vec) {
#pragma unroll
            for (int i = 0; i < EPL; i += 4)
                if (e0 + i < E) {
                    const float4 o = *reinterpret_cast<const float4*>(a.logit_offset + e0 + i);
                    lg[i] = lg[i] + o.x; lg[i + 1] = lg[i + 1] + o.y;
                    lg[i + 2] = lg[i + 2] + o.z; lg[i + 3] = lg[i + 3] + o.w;
                }
        } else {
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (e0 + i < E) lg[i] = lg[i] + a.logit_offset[e0 + i];
        }
    }
    if (a.logits_out) {
        float* lo = a.logits_out + row * E;
        if (lo_vec) {
#pragma unroll
            for (int i = 0; i < EPL; i += 4)
                if (e0 + i < E)
                    *reinterpret_cast<float4*>(lo + e0 + i) =
                        make_float4(lg[i], lg[i + 1], lg[i + 2], lg[i + 3]);
        } else {
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (e0 + i < E) lo[e0 + i] = lg[i];
        }
    }

    // ---- selection keys: sigmoid + bias (DeepSeek) or the logit itself (softmax) ----
    float orig[EPL];
    uint32_t key[EPL];
    uint32_t taken = 0;  // bit i: slot i is not selectable (taken, or beyond E)
    float bs[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) bs[i] = 0.0f;
    if (!SOFTMAX) {
        if (bias_vec) {
#pragma unroll
            for (int i = 0; i < EPL; i += 4)
                if (e0 + i < E) {
                    const float4 b = *reinterpret_cast<const float4*>(a.bias + e0 + i);
                    bs[i] = b.x; bs[i + 1] = b.y; bs[i + 2] = b.z; bs[i + 3] = b.w;
                }
        } else {
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (e0 + i < E) bs[i] = a.bias[e0 + i];
        }
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        if (e0 + i < E) {
            const float l = lg[i];
            if (SOFTMAX) {
                orig[i] = l;  // the logit itself is carried to the weights
                key[i] = okey(l);
            } else {
                const float s = 1.0f / (1.0f + expf(-l));
                orig[i] = s;
                key[i] = okey(s + bs[i]);
            }
        } else {
            orig[i] = 0.0f;
            key[i] = 0u;
            taken |= 1u << i;
        }
    }
    Top2 t = lane_top2<EPL>(key, orig, taken, e0);

    // ---- group mask: keep the topk_group groups with the largest top-2 sums ----
    const int G = a.n_group;
    if (!SOFTMAX && G > 1 && G - a.topk_group > 0) {
        const int eg = E / G;
        uint32_t my_gk = 0;  // lane g (< G) holds the key of group g's score
        const int lpg = (eg % EPL == 0) ? eg / EPL : 0;
        const bool aligned = lpg > 0 && lpg <= 32 && (lpg & (lpg - 1)) == 0;
        if (aligned) {
            // lanes [g*lpg, (g+1)*lpg) hold exactly group g: merge the lanes' top-2 keys
            uint32_t t1 = t.i0 == kEmpty ? 0u : t.k0, t2 = t.i1 == kEmpty ? 0u : t.k1;
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
        if (aligned) {
            // the lane's slots are all in group lane / lpg
            if (!__shfl_sync(kFull, kept, lane / lpg)) {
#pragma unroll
                for (int i = 0; i < EPL; ++i)
                    if (!(taken & (1u << i))) key[i] = zero_key;
                // all keys equal: the two lowest selectable slots lead
                t.k0 = t.k1 = zero_key;
                t.i0 = e0 < E ? (uint32_t)e0 : kEmpty;
                t.v0 = orig[0];
                if (EPL > 1) {
                    t.i1 = e0 + 1 < E ? (uint32_t)(e0 + 1) : kEmpty;
                    t.v1 = orig[EPL > 1 ? 1 : 0];
                } else {
                    t.i1 = kEmpty;
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int g = min((e0 + i) / eg, 31);
                const int k_i = __shfl_sync(kFull, kept, g);
                if (!(taken & (1u << i)) && !k_i) key[i] = zero_key;
            }
            t = lane_top2<EPL>(key, orig, taken, e0);
        }
    }

    // ---- top-k selection: one warp arg-max over the lanes' list heads per expert ----
    const int K = a.top_k;
    float my_w = 0.0f;
    int my_idx = 0;
    for (int r = 0; r < K; ++r) {
        const bool has = t.i0 != kEmpty;
        const uint32_t m = __reduce_max_sync(kFull, has ? t.k0 : 0u);
        const uint32_t w = __reduce_min_sync(kFull, (has && t.k0 == m) ? t.i0 : kEmpty);
        const bool owner = t.i0 == w;
        const float ov = __shfl_sync(kFull, t.v0, (int)(w / EPL));
        if (lane == r) { my_w = ov; my_idx = (int)w; }
        if (owner) {
            taken |= 1u << (w - (uint32_t)e0);
            t.k0 = t.k1; t.i0 = t.i1; t.v0 = t.v1;
            t.i1 = kEmpty;
        }
        // a lane whose list ran out while it still holds selectable slots refills it
        const bool refill = owner && t.i0 == kEmpty && taken != (EPL == 32 ? kEmpty : (1u << EPL) - 1u);
        if (r + 1 < K && __any_sync(kFull, refill)) {
            if (refill) t = lane_top2<EPL>(key, orig, taken, e0);
        }
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
        continue;
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
    }  // rows
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
    const int epl = a.E <= 32 ? 1 : a.E <= 64 ? 2 : a.E <= 128 ? 4 : a.E <= 256 ? 8
                  : a.E <= 512 ? 16 : 32;
    // 8 warps per CTA, one row per warp at a time; no more CTAs than fit on the SMs at once
    // (4 per SM up to 8 experts per lane, register-bound to 1 above), rows strided
    const long long want = (a.rows + 7) / 8;
    const long long cap = (long long)(epl <= 8 ? 4 : 1) * num_sms();
    const unsigned grid = (unsigned)(want < cap ? want : cap);
    if (a.softmax) {
        switch (epl) {
            case 1: return launch_kernel(route_kernel<1, true>, dim3(grid), dim3(256), 0, s, a);
            case 2: return launch_kernel(route_kernel<2, true>, dim3(grid), dim3(256), 0, s, a);
            case 4: return launch_kernel(route_kernel<4, true>, dim3(grid), dim3(256), 0, s, a);
            case 8: return launch_kernel(route_kernel<8, true>, dim3(grid), dim3(256), 0, s, a);
            case 16: return launch_kernel(route_kernel<16, true>, dim3(grid), dim3(256), 0, s, a);
            default: return launch_kernel(route_kernel<32, true>, dim3(grid), dim3(256), 0, s, a);
        }
        return cudaGetLastError();
    }
    switch (epl) {
        case 1: return launch_kernel(route_kernel<1, false>, dim3(grid), dim3(256), 0, s, a);
        case 2: return launch_kernel(route_kernel<2, false>, dim3(grid), dim3(256), 0, s, a);
        case 4: return launch_kernel(route_kernel<4, false>, dim3(grid), dim3(256), 0, s, a);
        case 8: return launch_kernel(route_kernel<8, false>, dim3(grid), dim3(256), 0, s, a);
        case 16: return launch_kernel(route_kernel<16, false>, dim3(grid), dim3(256), 0, s, a);
        default: return launch_kernel(route_kernel<32, false>, dim3(grid), dim3(256), 0, s, a);
    }
    return cudaGetLastError();
}

}  // namespace moe
