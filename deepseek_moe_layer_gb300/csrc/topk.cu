// topk.cu -- the DSA indexer's top-k selection: for every query row, the positions of the
// index_topk largest scores among its valid key positions.
//
// Source: SwiftLM issue #139 (stage 2 of the DeepSeek-V3.2 / GLM sparse-attention port),
// "What needs building" item 1 (selection = argPartition(scores, kth: -index_topk)) and
// item 3 (decode gathers the selected positions, prefill ANDs them into the causal mask), and
// the inertness remark (a row with no more than index_topk positions selects them all).
//
// Order: larger score first, equal scores by lower position, NaN below every number,
// -0 == +0.  The selected positions are written in ascending order, padded with -1.
//
// Design: one thread-block cluster per row (1..8 CTAs, each a contiguous segment of the
// row).  Scores become order-preserving 32-bit keys, cached in shared memory.  A radix
// select finds the key of the k-th largest element digit by digit (11-bit digits for long
// rows, 8-bit for short ones): each pass builds a per-CTA histogram of the digit over the keys
// that still match the chosen prefix (shared-memory atomics; warp pre-aggregation with
// match.any measured slower), the cluster's histograms are summed over distributed shared
// memory, and every CTA picks the same digit.  The last pass compacts the selected positions
// in position order (each warp a contiguous range, ballot-free lane scans); elements equal to
// the threshold key are taken lowest position first, across the cluster's segments in order.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

namespace cg = cooperative_groups;

constexpr unsigned kAll = 0xFFFFFFFFu;
constexpr int kSample = 2048;   // keys sampled per row for the threshold window
constexpr int kCandCap = 4096;  // window keys a CTA can hold

// Order-preserving key of an fp32 score: NaN -> 0 (lowest), -0 -> +0.
MOE_DEV uint32_t score_key(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u << 1) == 0u) u = 0u;
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <bool BF16>
MOE_DEV uint32_t load_key(const void* base, long long j) {
    if (BF16) {
        const uint16_t h = static_cast<const uint16_t*>(base)[j];
        return score_key(__uint_as_float(((uint32_t)h) << 16));
    }
    return score_key(static_cast<const float*>(base)[j]);
}

// Exclusive block-wide prefix sum of v over THREADS threads (all call it); *total = sum.
template <int THREADS>
MOE_DEV uint32_t block_excl_scan(uint32_t v, uint32_t* s_warp, uint32_t* total) {
    constexpr int W = THREADS / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kAll, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < W ? s_warp[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kAll, w, o);
            if (lane >= o) w += y;
        }
        if (lane < W) s_warp[lane] = w;  // inclusive warp totals
    }
    __syncthreads();
    const uint32_t before = (warp ? s_warp[warp - 1] : 0u) + x - v;
    *total = s_warp[W - 1];
    __syncthreads();  // s_warp is reused by the next call
    return before;
}

// Four consecutive keys from shared memory starting at i (a multiple of 4); keys at or past
// `end` read as 0 and are flagged invalid by the caller.
MOE_DEV uint4 keys4(const uint32_t* keys, int i, int end) {
    if (i + 3 < end) return *reinterpret_cast<const uint4*>(keys + i);
    uint4 q;
    q.x = i < end ? keys[i] : 0u;
    q.y = i + 1 < end ? keys[i + 1] : 0u;
    q.z = i + 2 < end ? keys[i + 2] : 0u;
    q.w = 0u;
    return q;
}

// THREADS threads per CTA; digits of DBITS bits (the last pass takes the remaining bits).
template <bool BF16, int THREADS, int DBITS, bool CACHED>
__global__ void __launch_bounds__(THREADS) indexer_topk_kernel(const TopkArgs a) {
    constexpr int W = THREADS / 32;
    constexpr int NB = 1 << DBITS;
    cg::cluster_group cl = cg::this_cluster();
    const unsigned nc = cl.num_blocks();
    const unsigned rank = cl.block_rank();
    const long long row = (long long)(blockIdx.x / nc);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    extern __shared__ __align__(16) uint8_t tk_smem[];
    int* hist = reinterpret_cast<int*>(tk_smem);                  // [NB] this CTA's histogram
    int* merged = hist + NB;                                       // [NB] the cluster's sum
    // the threshold window (long rows only): candidates and the sample
    constexpr bool kWin = THREADS == 512;
    uint32_t* cand = reinterpret_cast<uint32_t*>(merged + NB);    // [kCandCap] window keys
    uint32_t* samp = cand + (kWin ? kCandCap : 0);                 // [kSample] (leader's used)
    uint32_t* keys = samp + (kWin ? kSample : 0);                  // [seg] when cached
    __shared__ uint32_t s_warp[W];
    __shared__ uint32_t s_wg[W], s_wq[W];  // per-warp greater / equal counts, then prefixes
    __shared__ int s_pick[2];               // chosen digit, remaining count
    __shared__ int s_counts[2];             // this CTA's (greater, equal) counts
    __shared__ int s_wcnt[2];               // keys above / inside the window
    __shared__ uint32_t s_win[2];           // window (low, high) keys, set by the leader
    __shared__ int s_sel[4];                // leader: the sample's first digits and ranks
    __shared__ int s_cg[8], s_ce[8];        // leader: every CTA's keys above / equal to tau
    __shared__ uint32_t s_res[3];           // from the leader: tau, output base, ties to take

    const int n = a.n, k = a.k;
    int nr = a.lengths ? a.lengths[row] : n;
    nr = nr < 0 ? 0 : (nr > n ? n : nr);
    const int j0 = (int)min((long long)rank * a.seg, (long long)n);
    const int j1 = (int)min((long long)j0 + a.seg, (long long)n);
    const int v1 = j1 < nr ? j1 : nr;
    const int cnt = v1 > j0 ? v1 - j0 : 0;  // valid positions of this CTA's segment
    int32_t* out = a.inds + row * (long long)k;
    uint8_t* mrow = a.mask ? a.mask + row * a.mask_ld : nullptr;
    const bool mvec = mrow && ((reinterpret_cast<uintptr_t>(mrow + j0) & 3u) == 0);

    if (nr <= k) {
        // every valid position is selected: position j goes to slot j, the rest are -1
        for (int j = j0 + tid; j < v1; j += THREADS) out[j] = j;
        if (rank == 0)
            for (int p = nr + tid; p < k; p += THREADS) out[p] = -1;
        if (mrow) {
            if (mvec) {
                for (int j = j0 + 4 * tid; j < j1; j += 4 * THREADS) {
                    uint32_t m = 0;
#pragma unroll
                    for (int e = 0; e < 4; ++e) m |= (uint32_t)(j + e < nr) << (8 * e);
                    if (j + 3 < j1) *reinterpret_cast<uint32_t*>(mrow + j) = m;
                    else
                        for (int e = 0; j + e < j1; ++e) mrow[j + e] = j + e < nr ? 1 : 0;
                }
            } else {
                for (int j = j0 + tid; j < j1; j += THREADS) mrow[j] = j < nr ? 1 : 0;
            }
        }
        return;  // no distributed shared memory was touched: CTAs may leave independently
    }

    const void* srow = BF16 ? (const void*)(static_cast<const uint16_t*>(a.scores) + row * a.ld)
                            : (const void*)(static_cast<const float*>(a.scores) + row * a.ld);
    constexpr bool cached = CACHED;  // keys of the segment held in shared memory
    // short rows (one CTA, no window): the radix select's first histogram (the top DBITS bits
    // of every key) is built while the keys are loaded, which saves a pass over them
    constexpr bool kFuse0 = !kWin && CACHED;
    if (kFuse0) {
        for (int b = tid; b < NB; b += THREADS) hist[b] = 0;
        __syncthreads();
    }
    auto h0 = [&](uint32_t key) {
        if (kFuse0) atomicAdd(&hist[key >> (32 - DBITS)], 1);
    };
    if (cached) {
        // one pass over HBM: 16-byte vectors where the row allows, scalars otherwise
        const int per = BF16 ? 8 : 4;
        const uintptr_t addr = reinterpret_cast<uintptr_t>(srow) +
                               (uintptr_t)j0 * (BF16 ? 2u : 4u);
        const bool vec = (addr & 15u) == 0;
        const int nv = vec ? cnt / per : 0;
        // eight 16-byte loads in flight per thread before any is converted
        constexpr int kU = 8;
        int v0 = tid;
        for (; v0 + (kU - 1) * THREADS < nv; v0 += kU * THREADS) {
            uint4 qq[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u)
                qq[u] = __ldg(reinterpret_cast<const uint4*>(addr) + v0 + u * THREADS);
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int v = v0 + u * THREADS;
                const uint32_t w[4] = {qq[u].x, qq[u].y, qq[u].z, qq[u].w};
                if (BF16) {
                    uint4 lo, hi;
                    lo.x = score_key(__uint_as_float(w[0] << 16));
                    lo.y = score_key(__uint_as_float(w[0] & 0xFFFF0000u));
                    lo.z = score_key(__uint_as_float(w[1] << 16));
                    lo.w = score_key(__uint_as_float(w[1] & 0xFFFF0000u));
                    hi.x = score_key(__uint_as_float(w[2] << 16));
                    hi.y = score_key(__uint_as_float(w[2] & 0xFFFF0000u));
                    hi.z = score_key(__uint_as_float(w[3] << 16));
                    hi.w = score_key(__uint_as_float(w[3] & 0xFFFF0000u));
                    reinterpret_cast<uint4*>(keys)[2 * v] = lo;
                    reinterpret_cast<uint4*>(keys)[2 * v + 1] = hi;
                    h0(lo.x); h0(lo.y); h0(lo.z); h0(lo.w); h0(hi.x); h0(hi.y); h0(hi.z); h0(hi.w);
                } else {
                    uint4 kq;
                    kq.x = score_key(__uint_as_float(w[0]));
                    kq.y = score_key(__uint_as_float(w[1]));
                    kq.z = score_key(__uint_as_float(w[2]));
                    kq.w = score_key(__uint_as_float(w[3]));
                    reinterpret_cast<uint4*>(keys)[v] = kq;
                    h0(kq.x); h0(kq.y); h0(kq.z); h0(kq.w);
                }
            }
        }
        for (int v = v0; v < nv; v += THREADS) {
            const uint4 q = reinterpret_cast<const uint4*>(addr)[v];
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
            if (BF16) {
                uint4 lo, hi;
                lo.x = score_key(__uint_as_float(w[0] << 16));
                lo.y = score_key(__uint_as_float(w[0] & 0xFFFF0000u));
                lo.z = score_key(__uint_as_float(w[1] << 16));
                lo.w = score_key(__uint_as_float(w[1] & 0xFFFF0000u));
                hi.x = score_key(__uint_as_float(w[2] << 16));
                hi.y = score_key(__uint_as_float(w[2] & 0xFFFF0000u));
                hi.z = score_key(__uint_as_float(w[3] << 16));
                hi.w = score_key(__uint_as_float(w[3] & 0xFFFF0000u));
                reinterpret_cast<uint4*>(keys)[2 * v] = lo;
                reinterpret_cast<uint4*>(keys)[2 * v + 1] = hi;
                h0(lo.x); h0(lo.y); h0(lo.z); h0(lo.w); h0(hi.x); h0(hi.y); h0(hi.z); h0(hi.w);
            } else {
                uint4 kq;
                kq.x = score_key(__uint_as_float(w[0]));
                kq.y = score_key(__uint_as_float(w[1]));
                kq.z = score_key(__uint_as_float(w[2]));
                kq.w = score_key(__uint_as_float(w[3]));
                reinterpret_cast<uint4*>(keys)[v] = kq;
                h0(kq.x); h0(kq.y); h0(kq.z); h0(kq.w);
            }
        }
        for (int i = nv * per + tid; i < cnt; i += THREADS) {
            const uint32_t key = load_key<BF16>(srow, j0 + i);
            keys[i] = key;
            h0(key);
        }
    }
    __syncthreads();

    // four keys of this CTA's segment starting at i (a multiple of 4)
    // uncached segments: four keys by one 16-byte (fp32) or 8-byte (bf16) load when the row
    // allows it (j0 and i are multiples of 4 here), else one key at a time
    const bool gvec = ((reinterpret_cast<uintptr_t>(srow) +
                        (uintptr_t)j0 * (BF16 ? 2u : 4u)) & (BF16 ? 7u : 15u)) == 0;
    auto get4 = [&](int i) -> uint4 {
        if constexpr (CACHED) return keys4(keys, i, cnt);
        uint4 q;
        if (gvec && i + 3 < cnt) {
            if (BF16) {
                const uint2 w = __ldg(reinterpret_cast<const uint2*>(
                    static_cast<const uint16_t*>(srow) + j0 + i));
                q.x = score_key(__uint_as_float(w.x << 16));
                q.y = score_key(__uint_as_float(w.x & 0xFFFF0000u));
                q.z = score_key(__uint_as_float(w.y << 16));
                q.w = score_key(__uint_as_float(w.y & 0xFFFF0000u));
            } else {
                const float4 f = __ldg(reinterpret_cast<const float4*>(
                    static_cast<const float*>(srow) + j0 + i));
                q.x = score_key(f.x);
                q.y = score_key(f.y);
                q.z = score_key(f.z);
                q.w = score_key(f.w);
            }
            return q;
        }
        q.x = i < cnt ? load_key<BF16>(srow, j0 + i) : 0u;
        q.y = i + 1 < cnt ? load_key<BF16>(srow, j0 + i + 1) : 0u;
        q.z = i + 2 < cnt ? load_key<BF16>(srow, j0 + i + 2) : 0u;
        q.w = i + 3 < cnt ? load_key<BF16>(srow, j0 + i + 3) : 0u;
        return q;
    };
    auto csync = [&]() {
        if (nc > 1) cl.sync();
        else __syncthreads();
    };

    // ---- a window of keys holding the k-th largest, from a sample (cached rows) ----
    // The leader CTA sorts ~kSample keys taken at a fixed stride of the valid row, takes the
    // keys delta ranks above and below the k-th largest's expected rank, and the cluster
    // counts exactly how many keys lie above and inside that window (register counters, no
    // atomics).  When the k-th largest provably lies inside, only the window's keys (the
    // candidates) enter the radix select.  If all of the row's candidates fit one CTA's
    // buffer, every CTA writes its candidates into the leader's, and the leader alone selects
    // the threshold and hands every CTA its output base and share of the ties (no cluster
    // barrier in its radix passes); otherwise each CTA keeps its own candidates and the
    // cluster merges its histograms pass by pass.  Without a window the cluster's radix
    // select runs over every key.
    bool windowed = false, leader = false;
    int c_above = 0, c_win = 0, c_off = 0;  // leader mode, warp c: CTA c's window counts
    uint32_t wlo = 0u, whi = 0xFFFFFFFFu;  // the window (inclusive), when windowed
    int kk0 = k;               // rank of the threshold among the radix select's keys
    int ccnt = 0;              // candidates of this CTA
    uint32_t above_win = 0;    // this CTA's keys above the window
    static_assert(!kWin || (NB == 2048 && THREADS == 512), "the sample select: 4 bins a thread");
    if (kWin && (long long)k * 8 <= nr) {  // sparse selections (decode-like rows)
        const int stride = (nr + kSample - 1) / kSample;
        const int ns = (nr + stride - 1) / stride;  // <= kSample
        uint32_t* samp0 = nc > 1 ? cl.map_shared_rank(samp, 0) : samp;
        for (int j = (j0 + stride - 1) / stride * stride + tid * stride; j < v1; j += THREADS * stride)
            samp0[j / stride] = CACHED ? keys[j - j0] : load_key<BF16>(srow, j);
        csync();
        if (rank == 0) {
            // the sample's keys of (0-based, descending) ranks r - delta and r + delta, to
            // their top 22 bits: two radix passes of 11 bits, both ranks in the same passes
            // (counts of the two targets packed into the halves of one scanned word)
            const int r = (int)((long long)k * ns / nr);
            const int delta = 3 * (int)sqrtf((float)r) + 8;  // ~3 sigma of the sample rank
            const int kka = r - delta + 1, kkb = r + delta + 1;  // 1-based ranks; a: high end
            for (int b = tid; b < 2048; b += THREADS) hist[b] = 0;
            __syncthreads();
            for (int i = tid; i < ns; i += THREADS) atomicAdd(&hist[samp[i] >> 21], 1);
            __syncthreads();
            {
                const int hi = 2047 - 4 * tid;  // this thread's bins, top-down
                uint32_t mine = 0, total;
#pragma unroll
                for (int q = 0; q < 4; ++q) mine += (uint32_t)hist[hi - q];
                uint32_t acc = block_excl_scan<THREADS>(mine, s_warp, &total);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t c = (uint32_t)hist[hi - q];
                    if ((int)acc < kka && (int)(acc + c) >= kka) { s_sel[0] = hi - q; s_sel[1] = kka - (int)acc; }
                    if ((int)acc < kkb && (int)(acc + c) >= kkb) { s_sel[2] = hi - q; s_sel[3] = kkb - (int)acc; }
                    acc += c;
                }
            }
            __syncthreads();
            const int da = kka >= 1 ? s_sel[0] : -1, db = kkb <= ns ? s_sel[2] : -1;
            for (int b = tid; b < 2048; b += THREADS) { hist[b] = 0; merged[b] = 0; }
            __syncthreads();
            for (int i = tid; i < ns; i += THREADS) {
                const uint32_t key = samp[i];
                const int top = (int)(key >> 21), mid = (int)((key >> 10) & 0x7FFu);
                if (top == da) atomicAdd(&hist[mid], 1);
                if (top == db) atomicAdd(&merged[mid], 1);
            }
            __syncthreads();
            {
                const int hi = 2047 - 4 * tid;
                uint32_t mine = 0, total;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    mine += (uint32_t)hist[hi - q] | ((uint32_t)merged[hi - q] << 16);
                const uint32_t before = block_excl_scan<THREADS>(mine, s_warp, &total);
                int acca = (int)(before & 0xFFFFu), accb = (int)(before >> 16);
                const int ra = s_sel[1], rb = s_sel[3];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int ca = hist[hi - q], cb = merged[hi - q];
                    if (da >= 0 && acca < ra && acca + ca >= ra)
                        s_win[1] = ((uint32_t)da << 21) | ((uint32_t)(hi - q) << 10) | 0x3FFu;
                    if (db >= 0 && accb < rb && accb + cb >= rb)
                        s_win[0] = ((uint32_t)db << 21) | ((uint32_t)(hi - q) << 10);
                    acca += ca;
                    accb += cb;
                }
                if (tid == 0) {
                    if (da < 0) s_win[1] = 0xFFFFFFFFu;  // no high end
                    if (db < 0) s_win[0] = 0u;           // no low end
                }
            }
        }
        csync();
        const uint32_t* w0p = nc > 1 ? cl.map_shared_rank(s_win, 0) : s_win;
        wlo = w0p[0];
        whi = w0p[1];
        uint32_t a = 0, wn = 0;
        for (int base = 0; base < cnt; base += 4 * THREADS) {
            const int i = base + 4 * tid;
            const uint4 q = get4(i);
            const uint32_t kq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool v = i + e < cnt;
                a += v && kq[e] > whi;
                wn += v && kq[e] >= wlo && kq[e] <= whi;
            }
        }
        uint32_t ta, tw;
        block_excl_scan<THREADS>(a, s_warp, &ta);
        const uint32_t wpre = block_excl_scan<THREADS>(wn, s_warp, &tw);  // this thread's slot
        if (tid == 0) { s_wcnt[0] = (int)ta; s_wcnt[1] = (int)tw; }
        csync();
        int ca[8], cw[8];  // every CTA's counts, all remote loads in flight together
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            ca[c] = cw[c] = 0;
            if (c < (int)nc) {
                const int* rc = c == (int)rank ? s_wcnt : cl.map_shared_rank(s_wcnt, c);
                ca[c] = rc[0];
                cw[c] = rc[1];
            }
        }
        long long G = 0, Wt = 0, off = 0;
        int wmax = 0;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            if (c == warp) { c_above = ca[c]; c_win = cw[c]; c_off = (int)Wt; }
            if (c < (int)rank) off += cw[c];
            G += ca[c];
            Wt += cw[c];
            wmax = cw[c] > wmax ? cw[c] : wmax;
        }
        // (s_wcnt, s_win and the sample are never written again: no barrier here)
        windowed = wmax <= kCandCap && G < k && G + Wt >= k;
        leader = windowed && nc > 1 && Wt <= kCandCap;
        if (windowed) {
            kk0 = k - (int)G;
            above_win = ta;
            ccnt = leader ? (int)Wt : (int)tw;
            // this CTA's candidates (thread by thread, each at its prefix of the window counts)
            // into the leader's buffer from `off` on, or into its own
            uint32_t* dst = (leader ? cl.map_shared_rank(cand, 0) + off : cand) + wpre;
            int j = 0;
            for (int base = 0; base < cnt; base += 4 * THREADS) {
                const int i = base + 4 * tid;
                const uint4 q = get4(i);
                const uint32_t kq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (i + e < cnt && kq[e] >= wlo && kq[e] <= whi) dst[j++] = kq[e];
            }
            if (leader) csync();  // every candidate is in the leader's buffer
            else __syncthreads();
        }
    }
    // ---- radix select of the k-th largest key ----
    // run(merge): over the candidates (leader only, merge = false) or over every key of the
    // segment with the cluster's histograms summed through distributed shared memory.  Over
    // the candidates the digits are those of key - wlo, 8 bits at a time, over only the
    // window's significant bits.
    uint32_t tau = 0;
    int kk = kk0;            // elements equal to tau still to take
    uint32_t my_gt = 0;      // this thread's share of the CTA's count of keys above tau
    int last_digit = 0;
    auto radix = [&](bool merge) {
        // (8-bit digits where the cluster merges its histograms over distributed shared memory)
        const int dbits = windowed && merge ? 8 : DBITS;
        const uint32_t kbase = windowed ? wlo : 0u;
        const int nbits = windowed ? (whi == wlo ? 1 : 32 - __clz((int)(whi - wlo))) : 32;
        const int npass = (nbits + dbits - 1) / dbits;
        const int rcnt = windowed ? ccnt : cnt;
        auto getr4 = [&](int i) -> uint4 { return windowed ? keys4(cand, i, ccnt) : get4(i); };
        uint32_t prefix = 0, pmask = 0;
#pragma unroll 1
        for (int pass = 0; pass < npass; ++pass) {
            const int top = nbits - dbits * pass;
            const int shift = top > dbits ? top - dbits : 0;
            const int nb = 1 << (top - shift);
            const bool prebuilt = kFuse0 && pass == 0;  // built during the load
            if (!prebuilt) {
                for (int b = tid; b < nb; b += THREADS) hist[b] = 0;
                __syncthreads();
            }
            for (int base = 0; base < rcnt && !prebuilt; base += 4 * THREADS) {
                const int i = base + 4 * tid;
                const uint4 q = getr4(i);
                const uint32_t kq[4] = {q.x, q.y, q.z, q.w};
                bool want[4];
                bool any = false;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    want[e] = i + e < rcnt && ((kq[e] - kbase) & pmask) == prefix;
                    any |= want[e];
                }
                if (pass == 0 || __any_sync(kAll, any)) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint32_t bin = ((kq[e] - kbase) >> shift) & (uint32_t)(nb - 1);
                        if (want[e]) atomicAdd(&hist[bin], 1);
                    }
                }
            }
            const int* tot = hist;
            if (merge && nc > 1) {
                cl.sync();  // every CTA's histogram is complete
                for (int b = tid; b < nb; b += THREADS) {
                    int sum = 0;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        if (c < (int)nc)
                            sum += c == (int)rank ? hist[b] : cl.map_shared_rank(hist, c)[b];
                    merged[b] = sum;
                }
                cl.sync();  // no CTA reads another's histogram any more
                tot = merged;
            } else {
                __syncthreads();
            }
            // digit: the bin where the count of larger digits < kk <= that count plus the
            // bin; thread t owns bins hi, hi-1, .., hi-per+1 (top-down), hi = nb - 1 - t*per
            const int per = nb >= THREADS ? nb / THREADS : 1;
            const int hi = nb - 1 - tid * per;
            uint32_t mine = 0;
            for (int q = 0; q < per && hi - q >= 0; ++q) mine += (uint32_t)tot[hi - q];
            uint32_t total;
            const uint32_t above = block_excl_scan<THREADS>(mine, s_warp, &total);
            uint32_t acc = above;
            for (int q = 0; q < per && hi - q >= 0; ++q) {
                const uint32_t c = (uint32_t)tot[hi - q];
                if (acc < (uint32_t)kk && acc + c >= (uint32_t)kk) {
                    s_pick[0] = hi - q;
                    s_pick[1] = kk - (int)acc;
                }
                acc += c;
            }
            __syncthreads();
            const int d = s_pick[0];
            // this CTA's keys in the bins above the digit are above the final threshold
            for (int q = 0; q < per && hi - q > d; ++q) my_gt += (uint32_t)hist[hi - q];
            prefix |= (uint32_t)d << shift;
            pmask |= (uint32_t)(nb - 1) << shift;
            kk = s_pick[1];
            last_digit = d;
            __syncthreads();
        }
        tau = prefix + kbase;
    };

    int out_base = 0, take = 0;  // this CTA's first output slot; threshold ties it takes
    if (leader) {
        if (rank == 0) {
            radix(false);
            // CTA c's keys above / equal to tau: its keys above the window plus those of its
            // candidates (warp c counts CTA c's range of the buffer)
            if (warp < (int)nc) {
                uint32_t g = 0, e = 0;
                for (int i = lane; i < c_win; i += 32) {
                    const uint32_t x = cand[c_off + i];
                    g += x > tau;
                    e += x == tau;
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    g += __shfl_xor_sync(kAll, g, o);
                    e += __shfl_xor_sync(kAll, e, o);
                }
                if (lane == 0) { s_cg[warp] = c_above + (int)g; s_ce[warp] = (int)e; }
            }
            __syncthreads();
            if (tid == 0) {  // ties lowest position first: CTAs in rank order
                int rem = kk, base = 0;
                for (int c = 0; c < (int)nc; ++c) {
                    const int t = s_ce[c] < rem ? s_ce[c] : rem;
                    uint32_t* r = c == 0 ? s_res : cl.map_shared_rank(s_res, c);
                    r[0] = tau;
                    r[1] = (uint32_t)base;
                    r[2] = (uint32_t)t;
                    base += s_cg[c] + t;
                    rem -= t;
                }
            }
        }
        cl.sync();  // every CTA's results are in place; no remote access from here on
        tau = s_res[0];
        out_base = (int)s_res[1];
        take = (int)s_res[2];
    } else {
        radix(true);
        uint32_t cta_gt;
        block_excl_scan<THREADS>(my_gt, s_warp, &cta_gt);
        if (tid == 0) {
            s_counts[0] = (int)(cta_gt + above_win);
            s_counts[1] = hist[last_digit];  // keys equal to tau in this CTA
        }
        // each CTA's share of the threshold ties (lowest position first) and its output base
        int rem = kk;
        if (nc > 1) {
            cl.sync();
            int cg_[8], ce_[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                cg_[c] = ce_[c] = 0;
                if (c < (int)nc) {
                    const int* rc = c == (int)rank ? s_counts : cl.map_shared_rank(s_counts, c);
                    cg_[c] = rc[0];
                    ce_[c] = rc[1];
                }
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int t = ce_[c] < rem ? ce_[c] : rem;
                if (c < (int)rank) out_base += cg_[c] + t;
                if (c == (int)rank) take = t;
                rem -= t;
            }
            cl.sync();  // remote counts read: no CTA touches another's shared memory from here on
        } else {
            __syncthreads();
            take = s_counts[1] < rem ? s_counts[1] : rem;
        }
    }

    // ---- compaction in position order: each warp a contiguous range, 4 keys per lane ----
    const int wlen = ((cnt + W - 1) / W + 127) / 128 * 128;
    const int w_lo = min(cnt, warp * wlen), w_hi = min(cnt, w_lo + wlen);
    uint32_t wg = 0, wq = 0;
    for (int b = w_lo; b < w_hi; b += 128) {
        const int i = b + 4 * lane;
        const uint4 q = i < w_hi ? get4(i) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t kq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const bool v = i + e < w_hi;
            wg += v && kq[e] > tau;
            wq += v && kq[e] == tau;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        wg += __shfl_xor_sync(kAll, wg, o);
        wq += __shfl_xor_sync(kAll, wq, o);
    }
    if (lane == 0) { s_wg[warp] = wg; s_wq[warp] = wq; }
    __syncthreads();
    if (tid == 0) {
        uint32_t g = 0, e = 0;
        for (int w = 0; w < W; ++w) {
            const uint32_t tg = s_wg[w], te = s_wq[w];
            s_wg[w] = g; s_wq[w] = e;
            g += tg; e += te;
        }
    }
    __syncthreads();
    uint32_t g_run = s_wg[warp], q_run = s_wq[warp];
    for (int b = w_lo; b < w_hi; b += 128) {
        const int i = b + 4 * lane;
        const uint4 q = i < w_hi ? get4(i) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t kq[4] = {q.x, q.y, q.z, q.w};
        uint32_t fg = 0, fq = 0;  // bit e: key e is above / equal to the threshold
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const bool v = i + e < w_hi;
            fg |= (uint32_t)(v && kq[e] > tau) << e;
            fq |= (uint32_t)(v && kq[e] == tau) << e;
        }
        // lanes' exclusive prefix of (equal, greater) counts within this 128-key step
        const uint32_t packed = (uint32_t)__popc(fg) | ((uint32_t)__popc(fq) << 16);
        uint32_t x = packed;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kAll, x, o);
            if (lane >= o) x += y;
        }
        const uint32_t step_tot = __shfl_sync(kAll, x, 31);
        const uint32_t before = x - packed;
        uint32_t gb = g_run + (before & 0xFFFFu), qb = q_run + (before >> 16);
        uint32_t mbits = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const bool isg = (fg >> e) & 1u, isq = (fq >> e) & 1u;
            const bool sel = isg || (isq && qb < (uint32_t)take);
            const uint32_t pos = (uint32_t)out_base + gb + min(qb, (uint32_t)take);
            if (sel && pos < (uint32_t)k) out[pos] = j0 + i + e;  // exactly k are selected
            mbits |= (uint32_t)sel << (8 * e);
            gb += isg;
            qb += isq;
        }
        if (mrow && i < w_hi) {
            if (mvec && i + 3 < w_hi) *reinterpret_cast<uint32_t*>(mrow + j0 + i) = mbits;
            else
                for (int e = 0; e < 4 && i + e < w_hi; ++e)
                    mrow[j0 + i + e] = (uint8_t)((mbits >> (8 * e)) & 1u);
        }
        g_run += step_tot & 0xFFFFu;
        q_run += step_tot >> 16;
    }
    if (mrow) {  // positions of this segment past the row's valid length
        const int z0 = v1 > j0 ? v1 : j0;
        for (int j = z0 + tid; j < j1; j += THREADS) mrow[j] = 0;
    }
}

}  // namespace

constexpr int kShortRow = 8192;  // segments up to this many keys take the short-row kernel

void indexer_topk_plan(TopkArgs& a) {
    // segments of at most kSegMax keys (64 KB of shared memory) per CTA, up to 8 CTAs per
    // row; longer rows keep 8 CTAs and re-read their keys from global memory (L2 after the
    // first pass) in every pass.  (Re-reading was also measured for many rows of cacheable
    // length: slower, as registers hold the kernel to 2 CTAs per SM either way.)
    constexpr int kSegMax = 16384;
    long long nc = (a.n + kSegMax - 1) / kSegMax;
    nc = nc < 1 ? 1 : (nc > 8 ? 8 : nc);
    long long seg = (a.n + nc - 1) / nc;
    seg = (seg + 7) / 8 * 8;
    a.nclusters = (int)nc;
    a.seg = (int)seg;
    a.cached = seg <= kSegMax;
}

size_t indexer_topk_smem(int seg, int cached) {
    const bool shortrow = seg <= kShortRow;
    const int nb = shortrow ? 256 : 2048;
    return (size_t)2 * nb * sizeof(int) +
           (shortrow ? 0 : (size_t)(kCandCap + kSample) * sizeof(uint32_t)) +
           (cached ? (size_t)seg * sizeof(uint32_t) : 0);
}

namespace {
template <bool BF16, int THREADS, int DBITS, bool CACHED>
cudaError_t launch_topk_t(const TopkArgs& a, cudaStream_t s) {
    const size_t smem = indexer_topk_smem(a.seg, a.cached);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.rows * a.nclusters), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)a.nclusters;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err = cudaFuncSetAttribute(indexer_topk_kernel<BF16, THREADS, DBITS, CACHED>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    err = cudaLaunchKernelEx(&cfg, indexer_topk_kernel<BF16, THREADS, DBITS, CACHED>, a);
    return err != cudaSuccess ? err : cudaGetLastError();
}
}  // namespace

cudaError_t launch_indexer_topk(const TopkArgs& a, cudaStream_t s) {
    if (a.rows == 0) return cudaSuccess;
    // short rows (one CTA, few keys): 256 threads and 8-bit digits keep the fixed cost of a
    // pass small; long rows: 512 threads and 11-bit digits (three passes)
    // (short rows are always cached: kShortRow <= the 16384-key segment cap)
    const bool shortrow = a.seg <= kShortRow;
    if (a.bf16) {
        if (shortrow) return launch_topk_t<true, 256, 8, true>(a, s);
        return a.cached ? launch_topk_t<true, 512, 11, true>(a, s)
                        : launch_topk_t<true, 512, 11, false>(a, s);
    }
    if (shortrow) return launch_topk_t<false, 256, 8, true>(a, s);
    return a.cached ? launch_topk_t<false, 512, 11, true>(a, s)
                    : launch_topk_t<false, 512, 11, false>(a, s);
}

}  // namespace moe
