// combine.cu -- weighted combine of the expert outputs plus the shared expert.
//
// Source: "feat(engine): E1 DeepSeek-style MoE gate (sigmoid, group top-k, bias) (#108)",
// review section "Architecture and design": route -> switch_glu -> combine, the combine
// taking the always-active, ungated shared expert:
//     y[t] = sum_k scores[t,k] * expert_out[slot(t,k)] + shared_out[t].
//
// With the gated shared expert (the combine's has_shared_expert_gate) the shared row is
// weighted by a per-token sigmoid gate instead of 1.
//
// Grid (d / (8 * 128), min(T, 65535)): each thread owns 8 consecutive features of a token
// and reads K + 1 16-byte vectors, so the kernel streams the expert rows once at full width;
// the blocks of one grid row stride over the tokens (grid.y is capped at 65535).
#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

__global__ void __launch_bounds__(128) combine_kernel(const uint4* __restrict__ eo,
                                                      const float* __restrict__ scores,
                                                      const int32_t* __restrict__ inv,
                                                      const uint4* __restrict__ so,
                                                      const float* __restrict__ sgate, long long T,
                                                      int K, int vec_per_row, uint4* __restrict__ y) {
    const int v = blockIdx.x * blockDim.x + threadIdx.x;
    pdl_launch_dependents();
    pdl_wait();  // the expert outputs come from the kernels before
    if (v >= vec_per_row) return;
    for (long long t = blockIdx.y; t < T; t += gridDim.y) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        // K rows in chunks of 4: the chunk's slot ids, then its rows, all in flight together;
        // the sum still runs k = 0, 1, .., K-1
        for (int k0 = 0; k0 < K; k0 += 4) {
            int jj[4];
            float ww[4];
            uint4 qq[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                jj[c] = k0 + c < K ? __ldg(inv + t * K + k0 + c) : -1;
                ww[c] = k0 + c < K ? __ldg(scores + t * K + k0 + c) : 0.0f;
            }
#pragma unroll
            for (int c = 0; c < 4; ++c)
                qq[c] = jj[c] >= 0 ? __ldg(eo + (long long)jj[c] * vec_per_row + v)
                                   : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (jj[c] < 0) continue;
                const uint32_t u[4] = {qq[c].x, qq[c].y, qq[c].z, qq[c].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] = fmaf(ww[c], bf16_lo(u[i]), acc[2 * i]);
                    acc[2 * i + 1] = fmaf(ww[c], bf16_hi(u[i]), acc[2 * i + 1]);
                }
            }
        }
        if (so) {
            const uint4 q = __ldg(so + t * vec_per_row + v);
            const uint32_t u[4] = {q.x, q.y, q.z, q.w};
            const float gw = sgate ? sgate[t] : 1.0f;  // gated shared expert: sigmoid weight
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] = fmaf(gw, bf16_lo(u[i]), acc[2 * i]);
                acc[2 * i + 1] = fmaf(gw, bf16_hi(u[i]), acc[2 * i + 1]);
            }
        }
        uint4 r;
        r.x = pack_bf16x2(acc[0], acc[1]);
        r.y = pack_bf16x2(acc[2], acc[3]);
        r.z = pack_bf16x2(acc[4], acc[5]);
        r.w = pack_bf16x2(acc[6], acc[7]);
        y[t * vec_per_row + v] = r;
    }
}

// gate[t] = sigmoid(x[t] . w): one warp per token, 16-byte loads, fp32 products summed by
// lane then across the warp.  The gated shared expert's per-token weight.
__global__ void __launch_bounds__(256) shared_gate_kernel(const uint4* __restrict__ x,
                                                          const uint4* __restrict__ w,
                                                          long long T, int vec_per_row,
                                                          float* __restrict__ gate) {
    const long long t = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    pdl_launch_dependents();
    pdl_wait();  // writes nothing before the kernel before has finished
    if (t >= T) return;
    float acc = 0.0f;
    for (int v = lane; v < vec_per_row; v += 32) {
        const uint4 a = __ldg(x + t * vec_per_row + v);
        const uint4 b = __ldg(w + v);
        const uint32_t ua[4] = {a.x, a.y, a.z, a.w}, ub[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc = fmaf(bf16_lo(ua[i]), bf16_lo(ub[i]), acc);
            acc = fmaf(bf16_hi(ua[i]), bf16_hi(ub[i]), acc);
        }
    }
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    if (lane == 0) gate[t] = 1.0f / (1.0f + expf(-acc));
}

}  // namespace

cudaError_t launch_shared_gate(const void* x, long long T, int d, const void* w, float* gate,
                               cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    return launch_kernel(shared_gate_kernel, dim3((unsigned)((T + 7) / 8)), dim3(256), 0, s,
                         static_cast<const uint4*>(x), static_cast<const uint4*>(w), T, d / 8, gate);
}

cudaError_t launch_combine(const void* expert_out, const float* scores, const int32_t* inv,
                           const void* shared_out, long long T, int K, int d, void* y,
                           cudaStream_t s, const float* shared_gate) {
    if (T == 0) return cudaSuccess;
    const int vpr = d / 8;
    dim3 grid((unsigned)((vpr + 127) / 128), (unsigned)(T < 65535 ? T : 65535));
    return launch_kernel(combine_kernel, grid, dim3(128), 0, s,
                         static_cast<const uint4*>(expert_out), scores, inv,
                         static_cast<const uint4*>(shared_out), shared_gate, T, K, vpr,
                         static_cast<uint4*>(y));
}

}  // namespace moe
