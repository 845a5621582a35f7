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

template <int EPL>
MOE_DEV void row_logits_tail(const RouteArgs& a, long long row, int e0, bool off_vec,
                             bool lo_vec, bool lo_write, float (&lg)[EPL]);

// The summed logits of `row` for this lane's slots (sum of the split partials in split
// order, plus the optional offset), also copied to logits_out when that is set.
template <int EPL>
MOE_DEV void row_logits(const RouteArgs& a, long long row, int e0, bool off_vec, bool lo_vec,
                        bool lo_write, float (&lg)[EPL]) {
    const int E = a.E;
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
    row_logits_tail<EPL>(a, row, e0, off_vec, lo_vec, lo_write, lg);
}

// Adds the optional offset to the lane's logits of `row` and copies them to logits_out when
// that is set.
template <int EPL>
MOE_DEV void row_logits_tail(const RouteArgs& a, long long row, int e0, bool off_vec,
                             bool lo_vec, bool lo_write, float (&lg)[EPL]) {
    const int E = a.E;
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
    if (a.logits_out && lo_write) {
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
    float lg[EPL];
    row_logits<EPL>(a, row, e0, off_vec, lo_vec, true, lg);

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

// ---- the DeepSeek gate in fewer instructions per token -------------------------------
//
// gate_kernel computes exactly route_kernel<.., false>'s result (the same K experts in the
// same order, weights summed in that order) for up to 8 experts per lane when E % EPL == 0
// and the group mask is off (n_group == 1 or no group dropped) or its groups are a
// power-of-two number of whole lanes: the DeepSeek-V3 shape (256 experts, 8 groups of 32)
// and its relatives.  One warp routes a token; lane l holds experts [l * EPL, l * EPL + EPL).
//  - each lane lists its three best slots (key descending, index ascending) and its
//    fourth-best key; if that fourth entry wins a round (four of the K winners in one lane,
//    rare), the token is redone by exact rounds that re-scan the winner's lane;
//  - the group mask ranks every group's key at once;
//  - the pre-bias sigmoid values and the winners go to shared memory, where lane k reads
//    the k-th winner's value and every lane sums the K values in selection order;
//  - the next token's logits load while this one is routed.

// Key of a biased score s + b with s = sigmoid(l): s is +0 or more, so s + b is never -0 and
// only NaN needs folding; otherwise the same key as okey().  NaN gets 1, still below every
// number (-inf's key is 0x007FFFFF), so that 0 marks an empty list entry and no expert's.
MOE_DEV uint32_t score_key(float f) {
    const uint32_t u = __float_as_uint(f);
    const uint32_t k = u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
    return f != f ? 1u : k;
}

constexpr uint32_t kBound = 0xFFFFFFFEu;  // list entry holding the fourth-best key only

// Inserts slot (key, e) into a lane's list: its best three slots k[0..2] / ix[0..2] (key
// descending, index ascending; an entry at or beyond `filled` may be empty, ix == kEmpty,
// k == 0) and the largest key below them, k[3] (0: none).  Slots arrive in increasing
// index, so an equal key stays behind the entries already listed.
MOE_DEV void list_insert(uint32_t (&k)[4], uint32_t (&ix)[3], uint32_t key, uint32_t e,
                         int filled) {
    bool c[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) c[j] = (j >= filled && ix[j] == kEmpty) || key > k[j];
    k[3] = max(k[3], c[2] ? k[2] : key);  // the slot that leaves (or misses) the best three
#pragma unroll
    for (int j = 2; j >= 0; --j) {
        if (c[j]) {
            const bool up = j > 0 && c[j > 0 ? j - 1 : 0];
            k[j] = up ? k[j > 0 ? j - 1 : 0] : key;
            ix[j] = up ? ix[j > 0 ? j - 1 : 0] : e;
        }
    }
}

// One selection round over the lanes' list heads.  The owner is the lowest lane holding the
// largest head (lanes hold increasing expert ranges and a head is its lane's lowest-index
// maximum, so that is the lowest expert index among the maxima; expert keys are at least 1,
// so an empty entry, key 0, never equals the maximum).  The owner writes its head's index
// to `win` (a shared-memory address), notes in `redo` a fourth-best entry taken, and pops:
// its list moves up and the third place takes the fourth-best key with index kBound.
// Written predicated, without a branch, as the round is the token's critical path.
MOE_DEV void select_round(uint32_t (&k)[4], uint32_t (&ix)[3], uint32_t below, uint32_t win,
                          uint32_t& redo) {
    asm volatile(
        "{\n\t"
        ".reg .u32 m, b, t;\n\t"
        ".reg .pred top, own, bnd;\n\t"
        "redux.sync.max.u32 m, %0, 0xffffffff;\n\t"
        "setp.eq.u32 top, %0, m;\n\t"
        "vote.sync.ballot.b32 b, top, 0xffffffff;\n\t"
        "and.b32 t, b, %8;\n\t"
        "setp.eq.and.u32 own, t, 0, top;\n\t"
        "@own st.shared.u32 [%9], %4;\n\t"
        "setp.eq.and.u32 bnd, %4, %10, own;\n\t"
        "@bnd mov.u32 %7, 1;\n\t"
        "@own mov.u32 %0, %1;\n\t"
        "@own mov.u32 %1, %2;\n\t"
        "@own mov.u32 %2, %3;\n\t"
        "@own mov.u32 %3, 0;\n\t"
        "@own mov.u32 %4, %5;\n\t"
        "@own mov.u32 %5, %6;\n\t"
        "@own mov.u32 %6, %10;\n\t"
        "}"
        : "+r"(k[0]), "+r"(k[1]), "+r"(k[2]), "+r"(k[3]), "+r"(ix[0]), "+r"(ix[1]),
          "+r"(ix[2]), "+r"(redo)
        : "r"(below), "r"(win), "n"(kBound)
        : "memory");
}

constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v / 2); }

// KC: top_k fixed at compile time (0: a.top_k).  GC: n_group fixed at compile time with
// E == 32 * EPL (0: from the arguments).  NW: warps per CTA.  CTA c routes tokens
// [c * rows / grid, (c + 1) * rows / grid), its warps taking one token at a time from a
// shared-memory counter, so that every warp of an SM stays busy until the SM's tokens run
// out (warps given fixed shares finish at very different times: the scheduler favours the
// older ones).
template <int EPL, int KC, int GC, int NW>
__global__ void __launch_bounds__(NW * 32, NW >= 16 ? 1 : 4) gate_kernel(const RouteArgs a) {
    static_assert(EPL >= 1 && EPL <= 8, "one to eight experts per lane");
    constexpr int kNE = 32 * EPL;  // expert slots of a token
    __shared__ __align__(16) float s_val[NW][kNE];
    __shared__ uint32_t s_win[NW][32];
    __shared__ __align__(16) float s_bias[kNE];
    __shared__ int s_next;
    pdl_launch_dependents();
    pdl_wait();  // the logits come from the kernel before
    const int lane = threadIdx.x & 31;
    float* const sv = s_val[threadIdx.x >> 5];
    uint32_t* const swin = s_win[threadIdx.x >> 5];
    const uint32_t swin_s = (uint32_t)__cvta_generic_to_shared(swin);
    const int E = GC ? kNE : a.E;
    const int e0 = lane * EPL;
    const bool live = e0 < E;  // E % EPL == 0: a lane's slots are all experts or none
    const bool vec_e = (EPL % 4 == 0);
    const bool off_vec = vec_e && (reinterpret_cast<uintptr_t>(a.logit_offset) & 15) == 0;
    const bool lo_vec = vec_e && (reinterpret_cast<uintptr_t>(a.logits_out) & 15) == 0;
    for (int e = threadIdx.x; e < kNE; e += NW * 32) s_bias[e] = e < E ? a.bias[e] : 0.0f;
    if (threadIdx.x == 0) s_next = 0;
    __syncthreads();

    // group mask: lanes [g * lpg, (g + 1) * lpg) hold group g (lpg a power of two)
    const int G = GC ? GC : a.n_group;
    const bool grouped = GC ? true : (G > 1 && G > a.topk_group);
    int gshift = GC ? ilog2(32 / (GC ? GC : 1)) : 0;
    if (!GC && grouped) gshift = __ffs((E / G) / EPL) - 1;
    const int grp = lane >> gshift;
    const bool in_group = grouped && live;
    const uint32_t zero_key = 0x80000000u;  // key of +0.0
    const int K = KC ? KC : a.top_k;
    const uint32_t below = (1u << lane) - 1u;

    // one fp32 split with 16-byte rows: the next token's logits load while this one is routed
    constexpr int kV = EPL % 4 == 0 ? EPL / 4 : 1;
    const bool pf = EPL % 4 == 0 && !a.bf16 && a.nsplit == 1 &&
                    (reinterpret_cast<uintptr_t>(a.logits) & 15) == 0;
    const float* const lbase = static_cast<const float*>(a.logits) + e0;
    const long long lo = a.rows * blockIdx.x / gridDim.x;
    const long long hi = a.rows * (blockIdx.x + 1) / gridDim.x;
    auto take = [&]() -> long long {
        int t = 0;
        if (lane == 0) t = atomicAdd(&s_next, 1);
        return lo + __shfl_sync(kFull, t, 0);
    };
    long long row = take();  // the warp's first token
    float4 nx[kV];
    if (pf && live && row < hi) {
#pragma unroll
        for (int v = 0; v < kV; ++v)
            nx[v] = *reinterpret_cast<const float4*>(lbase + row * E + 4 * v);
    }

    while (row < hi) {
        const long long next = take();  // loaded while this token is routed
        float lg[EPL];
        if (pf) {
#pragma unroll
            for (int v = 0; v < kV; ++v) {
                lg[(4 * v) % EPL] = nx[v].x; lg[(4 * v + 1) % EPL] = nx[v].y;
                lg[(4 * v + 2) % EPL] = nx[v].z; lg[(4 * v + 3) % EPL] = nx[v].w;
            }
            if (live && next < hi) {
#pragma unroll
                for (int v = 0; v < kV; ++v)
                    nx[v] = *reinterpret_cast<const float4*>(lbase + next * E + 4 * v);
            }
            row_logits_tail<EPL>(a, row, e0, off_vec, lo_vec, true, lg);
        } else {
            row_logits<EPL>(a, row, e0, off_vec, lo_vec, true, lg);
        }

        // sigmoid (the weights' values, to shared memory) and the biased selection keys
        uint32_t key[EPL];
        float val[EPL], bs[EPL];
        if constexpr (EPL % 4 == 0) {
#pragma unroll
            for (int v = 0; v < EPL / 4; ++v) {
                const float4 b = *reinterpret_cast<const float4*>(s_bias + e0 + 4 * v);
                bs[(4 * v) % EPL] = b.x; bs[(4 * v + 1) % EPL] = b.y;
                bs[(4 * v + 2) % EPL] = b.z; bs[(4 * v + 3) % EPL] = b.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < EPL; ++i) bs[i] = s_bias[e0 + i];
        }
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            val[i] = 1.0f / (1.0f + expf(-lg[i]));
            key[i] = score_key(val[i] + bs[i]);
        }
        if (live) {
            if constexpr (EPL % 4 == 0) {
#pragma unroll
                for (int i = 0; i < EPL; i += 4)
                    *reinterpret_cast<float4*>(sv + e0 + i) =
                        make_float4(val[i], val[i + 1], val[i + 2], val[i + 3]);
            } else {
#pragma unroll
                for (int i = 0; i < EPL; ++i) sv[e0 + i] = val[i];
            }
        }

        // the lane's best three slots and fourth-best key
        uint32_t lk[4] = {0u, 0u, 0u, 0u}, li[3] = {kEmpty, kEmpty, kEmpty};
#pragma unroll
        for (int i = 0; i < EPL; ++i) list_insert(lk, li, key[i], (uint32_t)(e0 + i), i);
        if (!live) {
#pragma unroll
            for (int j = 0; j < 3; ++j) { lk[j] = 0u; li[j] = kEmpty; }
            lk[3] = 0u;
        }

        if (grouped) {
            // group score: the sum of the group's two largest keys' values (a NaN key, 1,
            // reads back as NaN: the sum is NaN and its key 0, the lowest)
            uint32_t t1 = lk[0], t2 = EPL > 1 ? lk[1] : 0u;
#pragma unroll
            for (int off = 1; off < (GC ? 32 / (GC ? GC : 1) : 32); off <<= 1) {
                if (!GC && off >= (1 << gshift)) break;
                const uint32_t o1 = __shfl_xor_sync(kFull, t1, off);
                const uint32_t o2 = __shfl_xor_sync(kFull, t2, off);
                const uint32_t n2 = max(min(t1, o1), max(t2, o2));
                t1 = max(t1, o1);
                t2 = n2;
            }
            const uint32_t gk = okey(okey_value(t1) + okey_value(t2));
            // the group's rank (larger key first, ties to the lower index) from every
            // group's key at once
            int rank = 0;
#pragma unroll
            for (int h = 0; h < (GC ? GC : 32); ++h) {
                if (!GC && h >= G) break;
                const uint32_t hk = __shfl_sync(kFull, gk, h << gshift);
                rank += (hk > gk) || (hk == gk && h < grp);
            }
            if (in_group && rank >= a.topk_group) {
                // a dropped group's scores are all 0: its slots in index order
#pragma unroll
                for (int i = 0; i < EPL; ++i) key[i] = zero_key;
#pragma unroll
                for (int j = 0; j < 3; ++j) {
                    lk[j] = j < EPL ? zero_key : 0u;
                    li[j] = j < EPL ? (uint32_t)(e0 + j) : kEmpty;
                }
                lk[3] = EPL > 3 ? zero_key : 0u;
            }
        }

        // top-k: K rounds over the list heads
        uint32_t redo = 0u;
#pragma unroll
        for (int r = 0; r < (KC ? KC : 32); ++r) {
            if (!KC && r >= K) break;
            select_round(lk, li, below, swin_s + 4u * r, redo);
        }
        if (__any_sync(kFull, redo != 0u)) {
            // exact rounds: the winner's lane re-scans its untaken slots for its next head
            uint32_t hk = 0u, hi_ = kEmpty, taken = 0u;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (live && (hi_ == kEmpty || key[i] > hk)) { hk = key[i]; hi_ = (uint32_t)(e0 + i); }
#pragma unroll 1
            for (int r = 0; r < K; ++r) {
                const uint32_t m = __reduce_max_sync(kFull, hk);
                const bool top = hk == m;
                const unsigned b = __ballot_sync(kFull, top);
                if (top && (b & below) == 0u) {
                    swin[r] = hi_;
                    taken |= 1u << (hi_ - (uint32_t)e0);
                    hk = 0u;
                    hi_ = kEmpty;
#pragma unroll
                    for (int i = 0; i < EPL; ++i)
                        if (!(taken & (1u << i)) && (hi_ == kEmpty || key[i] > hk)) {
                            hk = key[i];
                            hi_ = (uint32_t)(e0 + i);
                        }
                }
            }
        }
        __syncwarp();  // winners and values in shared memory are visible to the whole warp

        // weights: renormalise (K > 1 and norm; summed in selection order), then scale
        const uint32_t my_idx = lane < K ? swin[lane] : 0u;
        float my_w = lane < K ? sv[my_idx] : 0.0f;
        if (K > 1 && a.norm) {
            float sum = 0.0f;
            for (int k = 0; k < K; ++k) sum += sv[swin[k]];
            my_w = my_w / sum;
        }
        my_w = my_w * a.scale;
        if (lane < K) {
            a.inds[row * K + lane] = (int)my_idx;
            a.scores[row * K + lane] = my_w;
        }
        __syncwarp();  // reads done before the next token's values are written
        row = next;
    }  // tokens
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
    // the DeepSeek gate's short form (same result) where its layout conditions hold
    const int G = a.n_group;
    const bool grouped = G > 1 && G > a.topk_group;
    auto groups_fit = [&](int lanes_epl) {
        if (!grouped) return true;
        const int eg = a.E / G;
        const int lpg = eg % lanes_epl == 0 ? eg / lanes_epl : 0;
        return lpg > 0 && (lpg & (lpg - 1)) == 0;
    };
    // one CTA of 32 warps per SM when every warp gets a token (each CTA a contiguous token
    // range), else CTAs of 8 warps, a token per warp
    // one CTA of 32 warps per SM when every warp gets a token (each CTA a contiguous token
    // range), else CTAs of 8 warps, a token per warp
    if (epl <= 8 && a.E % epl == 0 && groups_fit(epl)) {
        const bool wide = a.rows >= 32LL * num_sms();
        const unsigned g32 = (unsigned)num_sms();
        const unsigned g8 = (unsigned)((a.rows + 7) / 8);
#define MOE_GATE(EPL_, KC_, GC_)                                                                  \
    return wide ? launch_kernel(gate_kernel<EPL_, KC_, GC_, 32>, dim3(g32), dim3(1024), 0, s, a) \
                : launch_kernel(gate_kernel<EPL_, KC_, GC_, 8>, dim3(g8), dim3(256), 0, s, a)
        // the DeepSeek-V3 gate: 256 experts, 8 groups, some dropped, top-8
        if (a.E == 256 && G == 8 && grouped && a.top_k == 8) MOE_GATE(8, 8, 8);
        const bool k8 = a.top_k == 8;
        switch (epl) {
            case 1: if (k8) MOE_GATE(1, 8, 0); else MOE_GATE(1, 0, 0);
            case 2: if (k8) MOE_GATE(2, 8, 0); else MOE_GATE(2, 0, 0);
            case 4: if (k8) MOE_GATE(4, 8, 0); else MOE_GATE(4, 0, 0);
            default: if (k8) MOE_GATE(8, 8, 0); else MOE_GATE(8, 0, 0);
        }
#undef MOE_GATE
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
