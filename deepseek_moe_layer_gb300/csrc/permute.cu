// permute.cu -- token-to-expert dispatch: expert histogram, exclusive scan, stable
// permutation and its inverse, and the gather of the dispatched token rows.
//
// Source: "Epic: Engine Inference Core Stage E - MoE + hybrid families", first paragraph:
// the MoE forward dispatches tokens to experts for gather_mm / gather_qmm.  The grouping
// those calls consume is made explicit here: slot j of expert e holds pair p = t*K + k,
// slots sorted by (expert, p).
//
// One CTA of 32 warps.  Warp w owns the contiguous chunk w of the P pairs.  Pass 1 builds
// a per-warp histogram in shared memory, pass 2 turns (expert, warp) counts into slot
// bases (experts in order, warps in order inside an expert), pass 3 replays each chunk in
// pair order, ranking equal experts inside a 32-pair step with __match_any_sync.  Chunks
// are ordered and each step is in pair order, so the permutation is stable and
// deterministic without any global atomics.
#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

constexpr int kPermWarps = 32;

__global__ void __launch_bounds__(1024) permute_kernel(const int32_t* __restrict__ inds,
                                                       long long P, int E,
                                                       int32_t* __restrict__ counts,
                                                       int32_t* __restrict__ offsets,
                                                       int32_t* __restrict__ perm,
                                                       int32_t* __restrict__ inv) {
    extern __shared__ int32_t sh[];
    int32_t* hist = sh;                      // [kPermWarps][E]
    int32_t* wsum = sh + kPermWarps * E;     // [32] scan carries
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_launch_dependents();

    for (int i = threadIdx.x; i < kPermWarps * E; i += blockDim.x) hist[i] = 0;
    pdl_wait();  // the expert ids come from the kernel before
    __syncthreads();

    const long long chunk = (P + kPermWarps - 1) / kPermWarps;
    const long long c0 = min(P, (long long)warp * chunk);
    const long long c1 = min(P, c0 + chunk);
    int32_t* my = hist + warp * E;

    // pass 1: per-warp histogram (four loads in flight per lane)
    for (long long p0 = c0 + lane; p0 < c1; p0 += 128) {
        int ev[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) ev[u] = p0 + 32 * u < c1 ? __ldg(inds + p0 + 32 * u) : -1;
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (ev[u] >= 0 && ev[u] < E) atomicAdd(&my[ev[u]], 1);
    }
    __syncthreads();

    // pass 2: counts, exclusive scan over experts, per-(warp, expert) bases
    const int per = (E + blockDim.x - 1) / blockDim.x;  // experts per thread (1 for E <= 1024)
    int local = 0;
    for (int q = 0; q < per; ++q) {
        const int e = threadIdx.x * per + q;
        if (e < E) {
            int c = 0;
            for (int w = 0; w < kPermWarps; ++w) c += hist[w * E + e];
            counts[e] = c;
            local += c;
        }
    }
    int incl = local;
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = wsum[lane];
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xFFFFFFFFu, v, off);
            if (lane >= off) v += u;
        }
        wsum[lane] = v;  // inclusive over warps
    }
    __syncthreads();
    int run = (warp > 0 ? wsum[warp - 1] : 0) + incl - local;
    for (int q = 0; q < per; ++q) {
        const int e = threadIdx.x * per + q;
        if (e < E) {
            offsets[e] = run;
            for (int w = 0; w < kPermWarps; ++w) {
                const int h = hist[w * E + e];
                hist[w * E + e] = run;
                run += h;
            }
        }
    }
    if (threadIdx.x == blockDim.x - 1) offsets[E] = wsum[31];
    __syncthreads();

    // pass 3: stable placement, 32 pairs a step in pair order (the next three steps' expert
    // ids already in flight)
    const unsigned lt_mask = (1u << lane) - 1u;
    int ahead[3];
#pragma unroll
    for (int u = 0; u < 3; ++u) {
        const long long q = c0 + 32 * (u + 1) + lane;
        ahead[u] = q < c1 ? __ldg(inds + q) : -1;
    }
    int cur = c0 + lane < c1 ? __ldg(inds + c0 + lane) : -1;
    for (long long base = c0; base < c1; base += 32) {
        const long long p = base + lane;
        const bool active = p < c1;
        const int e = active ? cur : -1;
        cur = ahead[0];
        ahead[0] = ahead[1];
        ahead[1] = ahead[2];
        const long long q = base + 128 + lane;
        ahead[2] = q < c1 ? __ldg(inds + q) : -1;
        const bool valid = active && e >= 0 && e < E;
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, valid ? e : -1 - lane);
        int pos = 0;
        if (valid) pos = my[e] + __popc(peers & lt_mask);
        __syncwarp();
        if (valid && (__ffs(peers) - 1) == lane) my[e] += __popc(peers);
        __syncwarp();
        if (valid) {
            perm[pos] = (int32_t)p;
            inv[p] = pos;
        } else if (active) {
            inv[p] = -1;
        }
    }
}

// ---- large batches: the same dispatch spread over kPermCtas CTAs ----
// CTA b owns the contiguous chunk b of the pairs.  permute_count_kernel writes the chunk's
// expert counts cnt[b][e]; permute_place_kernel turns the count matrix into this chunk's
// slot base per expert (the slots of expert e: chunks in order, inside a chunk warps in
// order, inside a warp pairs in order: the same stable order as the one-CTA kernel), then
// places its chunk as that kernel does.  The scattered slot stores are spread over many SMs
// (from one SM they set the pace of the one-CTA kernel at large batches).
constexpr int kPermCtas = 64;

__global__ void __launch_bounds__(1024) permute_count_kernel(const int32_t* __restrict__ inds,
                                                             long long P, int E, long long chunk,
                                                             int32_t* __restrict__ cnt) {
    extern __shared__ int32_t sh[];  // [E]
    pdl_launch_dependents();
    for (int i = threadIdx.x; i < E; i += blockDim.x) sh[i] = 0;
    pdl_wait();
    __syncthreads();
    const long long c0 = min(P, (long long)blockIdx.x * chunk);
    const long long c1 = min(P, c0 + chunk);
    for (long long p = c0 + threadIdx.x; p < c1; p += blockDim.x) {
        const int e = __ldg(inds + p);
        if (e >= 0 && e < E) atomicAdd(&sh[e], 1);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < E; i += blockDim.x) cnt[(long long)blockIdx.x * E + i] = sh[i];
}

__global__ void __launch_bounds__(1024) permute_place_kernel(
    const int32_t* __restrict__ inds, long long P, int E, long long chunk,
    const int32_t* __restrict__ cnt, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
    extern __shared__ int32_t sh[];
    int32_t* hist = sh;                      // [kPermWarps][E]
    int32_t* wsum = sh + kPermWarps * E;     // [32] scan carries
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x, nb = gridDim.x;
    pdl_launch_dependents();

    for (int i = threadIdx.x; i < kPermWarps * E; i += blockDim.x) hist[i] = 0;
    pdl_wait();  // the per-chunk counts come from the kernel before
    // expert e (thread e, E <= 1024): its pairs in all chunks and in the chunks before b
    const int e_t = threadIdx.x;
    int tot = 0, pre = 0;
    if (e_t < E)
        for (int c = 0; c < nb; ++c) {
            const int v = __ldg(cnt + (long long)c * E + e_t);
            tot += v;
            pre += c < b ? v : 0;
        }
    // exclusive scan of the totals over the experts
    int incl = tot;
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = wsum[lane];
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xFFFFFFFFu, v, off);
            if (lane >= off) v += u;
        }
        wsum[lane] = v;  // inclusive over warps
    }
    __syncthreads();
    const int off_e = (warp > 0 ? wsum[warp - 1] : 0) + incl - tot;  // slot of expert e's first pair
    if (b == 0) {
        if (e_t < E) {
            counts[e_t] = tot;
            offsets[e_t] = off_e;
        }
        if (threadIdx.x == blockDim.x - 1) offsets[E] = wsum[31];
    }

    // this chunk's per-warp histograms
    const long long c0 = min(P, (long long)b * chunk);
    const long long c1 = min(P, c0 + chunk);
    const long long wch = (c1 - c0 + kPermWarps - 1) / kPermWarps;
    const long long w0 = min(c1, c0 + (long long)warp * wch);
    const long long w1 = min(c1, w0 + wch);
    int32_t* my = hist + warp * E;
    for (long long p0 = w0 + lane; p0 < w1; p0 += 128) {
        int ev[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) ev[u] = p0 + 32 * u < w1 ? __ldg(inds + p0 + 32 * u) : -1;
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (ev[u] >= 0 && ev[u] < E) atomicAdd(&my[ev[u]], 1);
    }
    __syncthreads();
    // per-(warp, expert) slot bases
    if (e_t < E) {
        int run = off_e + pre;
        for (int w = 0; w < kPermWarps; ++w) {
            const int h = hist[w * E + e_t];
            hist[w * E + e_t] = run;
            run += h;
        }
    }
    __syncthreads();

    // stable placement of the warp's pairs, 32 a step in pair order
    const unsigned lt_mask = (1u << lane) - 1u;
    for (long long base = w0; base < w1; base += 32) {
        const long long p = base + lane;
        const bool active = p < w1;
        const int e = active ? __ldg(inds + p) : -1;
        const bool valid = active && e >= 0 && e < E;
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, valid ? e : -1 - lane);
        int pos = 0;
        if (valid) pos = my[e] + __popc(peers & lt_mask);
        __syncwarp();
        if (valid && (__ffs(peers) - 1) == lane) my[e] += __popc(peers);
        __syncwarp();
        if (valid) {
            perm[pos] = (int32_t)p;
            inv[p] = pos;
        } else if (active) {
            inv[p] = -1;
        }
    }
}

// x_perm[j] = x[perm[j] / K], 16-byte vectors.  Warp w takes piece w % pieces (128 vectors,
// 2 KB) of slot w / pieces: four 16-byte loads in flight per lane, all before the stores, and
// many warps per row, so that a small batch is not one warp's serial walk along a 14 KB row.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x,
                                                          const int32_t* __restrict__ perm,
                                                          const int32_t* __restrict__ offsets,
                                                          int E, int K, long long P, int vec_per_row,
                                                          int pieces, uint4* __restrict__ x_perm) {
    const long long wg = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const long long j = wg / pieces;
    const int v0 = (int)(wg % pieces) * 128;
    const int lane = threadIdx.x & 31;
    pdl_launch_dependents();
    pdl_wait();  // the dispatch comes from the kernel before
    if (j >= P || j >= offsets[E]) return;
    const long long t = perm[j] / K;
    const uint4* src = x + t * vec_per_row;
    uint4* dst = x_perm + j * vec_per_row;
    // the gathered rows are streamed out (evict-first) so that x, read K times, stays in L2
    uint4 q[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int v = v0 + 32 * u + lane;
        if (v < vec_per_row) q[u] = __ldg(src + v);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int v = v0 + 32 * u + lane;
        if (v < vec_per_row) __stcs(dst + v, q[u]);
    }
}

}  // namespace

size_t permute_scratch_bytes(int E) { return sizeof(int32_t) * (size_t)kPermCtas * E; }

cudaError_t launch_permute(const int32_t* inds, long long P, int E, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv, cudaStream_t s,
                           void* scratch, size_t scratch_bytes) {
    const size_t smem = sizeof(int32_t) * ((size_t)kPermWarps * E + 32);
    static DeviceOnce attr_once;
    const cudaError_t attr_err = attr_once.run([] {
        const int most = (int)(sizeof(int32_t) * (kPermWarps * 1024 + 32));
        cudaError_t err = cudaFuncSetAttribute(permute_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, most);
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(permute_place_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, most);
        return err;
    });
    if (attr_err != cudaSuccess) return attr_err;
    if (P >= kPermMultiMin && scratch && scratch_bytes >= permute_scratch_bytes(E)) {
        const long long chunk = (P + kPermCtas - 1) / kPermCtas;
        int32_t* cnt = static_cast<int32_t*>(scratch);
        cudaError_t err = launch_kernel(permute_count_kernel, dim3(kPermCtas), dim3(1024),
                                        sizeof(int32_t) * (size_t)E, s, inds, P, E, chunk, cnt);
        if (err != cudaSuccess) return err;
        return launch_kernel(permute_place_kernel, dim3(kPermCtas), dim3(1024), smem, s, inds, P, E,
                             chunk, (const int32_t*)cnt, counts, offsets, perm, inv);
    }
    return launch_kernel(permute_kernel, dim3(1), dim3(1024), smem, s, inds, P, E, counts, offsets,
                         perm, inv);
}

cudaError_t launch_gather_rows(const void* x, const int32_t* perm, const int32_t* offsets, int E,
                               int K, long long P, int d, void* x_perm, cudaStream_t s) {
    if (P == 0) return cudaSuccess;
    const int vpr = d / 8;
    const int pieces = (vpr + 127) / 128;
    const unsigned grid = (unsigned)((P * pieces + 7) / 8);
    return launch_kernel(gather_rows_kernel, dim3(grid), dim3(256), 0, s,
                         static_cast<const uint4*>(x), perm, offsets, E, K, P, vpr, pieces,
                         static_cast<uint4*>(x_perm));
}

}  // namespace moe
