// combine.cu -- weighted combine of the expert outputs plus the shared expert.
//
// Source: "feat(engine): E1 DeepSeek-style MoE gate (sigmoid, group top-k, bias) (#108)",
// review section "Architecture and design": route -> switch_glu -> combine, the combine
// taking the always-active, ungated shared expert:
//     y[t] = sum_k scores[t,k] * expert_out[slot(t,k)] + shared_out[t].
//
// Grid (d / (8 * 128), T): each thread owns 8 consecutive features of one token and reads
// K + 1 16-byte vectors, so the kernel streams the expert rows once at full width.
#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

__global__ void __launch_bounds__(128) combine_kernel(const uint4* __restrict__ eo,
                                                      const float* __restrict__ scores,
                                                      const int32_t* __restrict__ inv,
                                                      const uint4* __restrict__ so, long long T,
                                                      int K, int vec_per_row, uint4* __restrict__ y) {
    const long long t = blockIdx.y;
    const int v = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T || v >= vec_per_row) return;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int k = 0; k < K; ++k) {
        const int j = inv[t * K + k];
        if (j < 0) continue;
        const float w = scores[t * K + k];
        const uint4 q = __ldg(eo + (long long)j * vec_per_row + v);
        const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[2 * i] = fmaf(w, bf16_lo(u[i]), acc[2 * i]);
            acc[2 * i + 1] = fmaf(w, bf16_hi(u[i]), acc[2 * i + 1]);
        }
    }
    if (so) {
        const uint4 q = __ldg(so + t * vec_per_row + v);
        const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[2 * i] += bf16_lo(u[i]);
            acc[2 * i + 1] += bf16_hi(u[i]);
        }
    }
    uint4 r;
    r.x = pack_bf16x2(acc[0], acc[1]);
    r.y = pack_bf16x2(acc[2], acc[3]);
    r.z = pack_bf16x2(acc[4], acc[5]);
    r.w = pack_bf16x2(acc[6], acc[7]);
    y[t * vec_per_row + v] = r;
}

}  // namespace

cudaError_t launch_combine(const void* expert_out, const float* scores, const int32_t* inv,
                           const void* shared_out, long long T, int K, int d, void* y,
                           cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int vpr = d / 8;
    dim3 grid((unsigned)((vpr + 127) / 128), (unsigned)T);
    combine_kernel<<<grid, 128, 0, s>>>(static_cast<const uint4*>(expert_out), scores, inv,
                                        static_cast<const uint4*>(shared_out), T, K, vpr,
                                        static_cast<uint4*>(y));
    return cudaGetLastError();
}

}  // namespace moe
