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
// select over three digits (11, 11, 10 bits) finds the key of the k-th largest element: each
// pass builds a per-CTA histogram of the digit over the keys that still match the chosen
// prefix (warp-aggregated shared-memory atomics), the cluster's histograms are summed over
// distributed shared memory, and every CTA picks the same digit.  The final pass compacts the
// selected positions in position order with block scans; elements equal to the threshold key
// are taken lowest position first, across the cluster's segments in order.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

namespace cg = cooperative_groups;

constexpr int kTkThreads = 512;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kBins = 2048;  // histogram size of the 11-bit digits
constexpr unsigned kAll = 0xFFFFFFFFu;

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

// Exclusive block-wide prefix sum of v (all kTkThreads threads call it); *total gets the sum.
MOE_DEV uint32_t block_excl_scan(uint32_t v, uint32_t* s_warp, uint32_t* total) {
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
        uint32_t w = lane < kTkWarps ? s_warp[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kAll, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kTkWarps) s_warp[lane] = w;  // inclusive warp totals
    }
    __syncthreads();
    const uint32_t before = (warp ? s_warp[warp - 1] : 0u) + x - v;
    *total = s_warp[kTkWarps - 1];
    __syncthreads();  // s_warp is reused by the next call
    return before;
}

template <bool BF16>
__global__ void __launch_bounds__(kTkThreads) indexer_topk_kernel(const TopkArgs a) {
    cg::cluster_group cl = cg::this_cluster();
    const unsigned nc = cl.num_blocks();
    const unsigned rank = cl.block_rank();
    const long long row = (long long)(blockIdx.x / nc);
    const int tid = threadIdx.x, lane = tid & 31;

    extern __shared__ __align__(16) uint8_t tk_smem[];
    int* hist = reinterpret_cast<int*>(tk_smem);            // [kBins] this CTA's histogram
    int* merged = hist + kBins;                              // [kBins] the cluster's sum
    uint32_t* keys = reinterpret_cast<uint32_t*>(merged + kBins);  // [seg] when cached
    __shared__ uint32_t s_warp[kTkWarps];
    __shared__ int s_pick[2];       // chosen digit, remaining count
    __shared__ int s_counts[2];     // this CTA's (greater, equal) counts, read by the cluster

    const int n = a.n, k = a.k;
    int nr = a.lengths ? a.lengths[row] : n;
    nr = nr < 0 ? 0 : (nr > n ? n : nr);
    const int j0 = (int)min((long long)rank * a.seg, (long long)n);
    const int j1 = (int)min((long long)j0 + a.seg, (long long)n);
    const int v1 = j1 < nr ? j1 : nr;
    const int cnt = v1 > j0 ? v1 - j0 : 0;  // valid positions of this CTA's segment
    int32_t* out = a.inds + row * (long long)k;
    uint8_t* mrow = a.mask ? a.mask + row * a.mask_ld : nullptr;

    if (nr <= k) {
        // every valid position is selected: position j goes to slot j, the rest are -1
        for (int j = j0 + tid; j < j1; j += kTkThreads) {
            if (j < nr) out[j] = j;
            if (mrow) mrow[j] = j < nr ? 1 : 0;
        }
        if (rank == 0)
            for (int p = nr + tid; p < k; p += kTkThreads) out[p] = -1;
        return;  // no distributed shared memory was touched: CTAs may leave independently
    }

    const void* srow = BF16 ? (const void*)(static_cast<const uint16_t*>(a.scores) + row * a.ld)
                            : (const void*)(static_cast<const float*>(a.scores) + row * a.ld);
    const bool cached = a.cached != 0;
    if (cached) {
        // one pass over HBM: 16-byte vectors where the row allows, scalars otherwise
        const int per = BF16 ? 8 : 4;
        const uintptr_t addr = reinterpret_cast<uintptr_t>(srow) +
                               (uintptr_t)j0 * (BF16 ? 2u : 4u);
        const bool vec = (addr & 15u) == 0;
        const int nv = vec ? cnt / per : 0;
        for (int v = tid; v < nv; v += kTkThreads) {
            const uint4 q = reinterpret_cast<const uint4*>(addr)[v];
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
            if (BF16) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    keys[v * 8 + 2 * e] = score_key(__uint_as_float(w[e] << 16));
                    keys[v * 8 + 2 * e + 1] = score_key(__uint_as_float(w[e] & 0xFFFF0000u));
                }
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) keys[v * 4 + e] = score_key(__uint_as_float(w[e]));
            }
        }
        for (int i = nv * per + tid; i < cnt; i += kTkThreads)
            keys[i] = load_key<BF16>(srow, j0 + i);
    }
    __syncthreads();

    // ---- radix select of the k-th largest key over the cluster ----
    uint32_t prefix = 0, pmask = 0;
    int kk = k;  // elements still to take among those matching the prefix
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int nb = pass == 2 ? 1024 : 2048;
        for (int b = tid; b < kBins; b += kTkThreads) hist[b] = 0;
        __syncthreads();
        for (int base = 0; base < cnt; base += kTkThreads) {
            const int i = base + tid;
            uint32_t key = 0;
            if (i < cnt) key = cached ? keys[i] : load_key<BF16>(srow, j0 + i);
            const bool want = i < cnt && (key & pmask) == prefix;
            const uint32_t bin = (key >> shift) & (uint32_t)(nb - 1);
            const unsigned grp = __match_any_sync(kAll, want ? bin : 0xFFFFFFFFu);
            if (want && lane == __ffs(grp) - 1) atomicAdd(&hist[bin], __popc(grp));
        }
        cl.sync();  // every CTA's histogram is complete
        for (int b = tid; b < nb; b += kTkThreads) {
            int s = 0;
            for (unsigned c = 0; c < nc; ++c) s += c == rank ? hist[b] : cl.map_shared_rank(hist, c)[b];
            merged[b] = s;
        }
        cl.sync();  // no CTA reads another's histogram any more
        // digit: the bin where the count of larger digits < kk <= that count plus the bin
        const int per = nb / kTkThreads;  // 4 or 2 bins per thread, thread t owns the top-down
        const int hi = nb - 1 - tid * per;  // chunk [hi - per + 1, hi]
        uint32_t mine = 0;
        for (int q = 0; q < per; ++q) mine += (uint32_t)merged[hi - q];
        uint32_t total;
        const uint32_t above = block_excl_scan(mine, s_warp, &total);
        uint32_t acc = above;
        for (int q = 0; q < per; ++q) {
            const uint32_t c = (uint32_t)merged[hi - q];
            if (acc < (uint32_t)kk && acc + c >= (uint32_t)kk) {
                s_pick[0] = hi - q;
                s_pick[1] = kk - (int)acc;
            }
            acc += c;
        }
        __syncthreads();
        prefix |= (uint32_t)s_pick[0] << shift;
        pmask |= (uint32_t)(nb - 1) << shift;
        kk = s_pick[1];
        __syncthreads();
    }
    const uint32_t tau = prefix;  // key of the k-th largest; kk of the keys equal to it are taken

    // ---- counts per CTA, then each CTA's share of the threshold ties and its output base ----
    uint32_t gt = 0, eq = 0;
    for (int i = tid; i < cnt; i += kTkThreads) {
        const uint32_t key = cached ? keys[i] : load_key<BF16>(srow, j0 + i);
        gt += key > tau;
        eq += key == tau;
    }
    uint32_t tot_gt, tot_eq;
    block_excl_scan(gt, s_warp, &tot_gt);
    block_excl_scan(eq, s_warp, &tot_eq);
    if (tid == 0) {
        s_counts[0] = (int)tot_gt;
        s_counts[1] = (int)tot_eq;
    }
    cl.sync();
    int rem = kk, out_base = 0, take = 0;
    for (unsigned c = 0; c < nc; ++c) {
        const int* rc = c == rank ? s_counts : cl.map_shared_rank(s_counts, c);
        const int g = rc[0], e = rc[1];
        const int t = e < rem ? e : rem;
        if (c < rank) out_base += g + t;
        if (c == rank) take = t;
        rem -= t;
    }
    cl.sync();  // remote counts read: from here on no CTA touches another's shared memory

    // ---- compaction in position order ----
    uint32_t gt_run = 0, eq_run = 0;
    for (int base = 0; base < cnt; base += kTkThreads) {
        const int i = base + tid;
        uint32_t key = 0;
        if (i < cnt) key = cached ? keys[i] : load_key<BF16>(srow, j0 + i);
        const uint32_t g = (i < cnt) && key > tau;
        const uint32_t e = (i < cnt) && key == tau;
        uint32_t chunk;
        // per-chunk counts are at most kTkThreads: both fit one word
        const uint32_t before = block_excl_scan(g | (e << 16), s_warp, &chunk);
        const uint32_t gb = gt_run + (before & 0xFFFFu);
        const uint32_t eb = eq_run + (before >> 16);  // equal keys before this position
        const bool sel = g || (e && eb < (uint32_t)take);
        const uint32_t pos = (uint32_t)out_base + gb + min(eb, (uint32_t)take);
        if (sel && pos < (uint32_t)k) out[pos] = j0 + i;  // exactly k are selected
        if (mrow && i < cnt) mrow[j0 + i] = sel ? 1 : 0;
        gt_run += chunk & 0xFFFFu;
        eq_run += chunk >> 16;
    }
    if (mrow)  // positions of this segment past the row's valid length
        for (int j = (v1 > j0 ? v1 : j0) + tid; j < j1; j += kTkThreads) mrow[j] = 0;
}

}  // namespace

void indexer_topk_plan(TopkArgs& a) {
    // segments of at most kSegMax keys (64 KB of shared memory) per CTA, up to 8 CTAs per
    // row; longer rows keep 8 CTAs and re-read their keys from global memory in every pass
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
    return (size_t)2 * kBins * sizeof(int) + (cached ? (size_t)seg * sizeof(uint32_t) : 0);
}

cudaError_t launch_indexer_topk(const TopkArgs& a, cudaStream_t s) {
    if (a.rows == 0) return cudaSuccess;
    const size_t smem = indexer_topk_smem(a.seg, a.cached);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.rows * a.nclusters), 1, 1);
    cfg.blockDim = dim3(kTkThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)a.nclusters;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err;
    if (a.bf16) {
        err = cudaFuncSetAttribute(indexer_topk_kernel<true>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        err = cudaLaunchKernelEx(&cfg, indexer_topk_kernel<true>, a);
    } else {
        err = cudaFuncSetAttribute(indexer_topk_kernel<false>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        err = cudaLaunchKernelEx(&cfg, indexer_topk_kernel<false>, a);
    }
    return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace moe
