// Output gate of the shared expert: gate[t] = sigmoid(hidden[t] . w) scales
// the shared expert's output of token t ("core.transformer.moe.megakernel.mok.
// runtime", _MoKAutograd.forward: shared_output_gate_weight; the pages name the
// weight, the per-token sigmoid gate is the layer's reading of it).
//
// Backward: with dgate[t] = <grad_out[t], y_shared[t]> (the shared dgrad-down
// GEMM's dprob partials, summed in a fixed order) and dz = gate (1 - gate) dgate,
// main_grad_w[h] += sum_t dz[t] hidden[t,h] in two deterministic passes (per
// 128-token chunk, then over chunks); dhidden[t] += dz[t] w is added by the
// un-permute kernel.
#include "device_common.cuh"
#include "internal.h"

namespace moe {

namespace {

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
    unpack_bf16x2(v.x, f[0], f[1]);
    unpack_bf16x2(v.y, f[2], f[3]);
    unpack_bf16x2(v.z, f[4], f[5]);
    unpack_bf16x2(v.w, f[6], f[7]);
}

// one warp per token: fp32 dot product of the bf16 row with w, lane partials
// combined by a fixed butterfly
__global__ void __launch_bounds__(256) gate_forward_kernel(const uint4* __restrict__ x, const uint4* __restrict__ w,
                                                           int T, int vec_per_row, float* __restrict__ gate) {
    pdl_wait();
    pdl_trigger();
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    float acc = 0.0f;
    for (int v = lane; v < vec_per_row; v += 32) {
        float xf[8], wf[8];
        unpack8(__ldg(x + int64_t(t) * vec_per_row + v), xf);
        unpack8(__ldg(w + v), wf);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc = fmaf(xf[j], wf[j], acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) gate[t] = sigmoidf_(acc);
}

// block c: tokens [c*128, c*128+128). dz of each token from its n_part
// partials (in order), then gpart[c][h] = sum over the chunk's tokens (in
// order) of dz[t] hidden[t,h]; 8 columns per thread
__global__ void __launch_bounds__(256) gate_grad_chunk_kernel(const uint4* __restrict__ x,
                                                              const float* __restrict__ gate,
                                                              const float* __restrict__ partial, int n_part, int T,
                                                              int vec_per_row, float* __restrict__ dz,
                                                              float4* __restrict__ gpart) {
    pdl_wait();
    pdl_trigger();
    __shared__ float s_dz[kGateChunk];
    const int t0 = blockIdx.x * kGateChunk;
    const int nt = min(kGateChunk, T - t0);
    for (int i = threadIdx.x; i < nt; i += blockDim.x) {
        const float* p = partial + int64_t(t0 + i) * n_part;
        float sum = 0.0f;
        for (int j = 0; j < n_part; ++j) sum += p[j];
        const float g = gate[t0 + i];
        const float d = g * (1.0f - g) * sum;
        s_dz[i] = d;
        dz[t0 + i] = d;
    }
    __syncthreads();
    for (int v = threadIdx.x; v < vec_per_row; v += blockDim.x) {
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int i = 0; i < nt; ++i) {
            float xf[8];
            unpack8(__ldg(x + int64_t(t0 + i) * vec_per_row + v), xf);
            const float d = s_dz[i];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = fmaf(d, xf[j], acc[j]);
        }
        float4* o = gpart + (int64_t(blockIdx.x) * vec_per_row + v) * 2;
        o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

// mg[h] += sum over chunks c (in order) of gpart[c][h]; bf16 main_grad:
// mg[h] = bf16(mg[h] + bf16(sum))
__global__ void __launch_bounds__(256) gate_grad_reduce_kernel(const float* __restrict__ gpart, int chunks, int H,
                                                               void* __restrict__ mg, int mg_bf16) {
    pdl_wait();
    pdl_trigger();
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= H) return;
    float sum = 0.0f;
    for (int c = 0; c < chunks; ++c) sum += gpart[int64_t(c) * H + h];
    if (mg_bf16) {
        __nv_bfloat16* m = static_cast<__nv_bfloat16*>(mg) + h;
        *m = __float2bfloat16_rn(__bfloat162float(*m) + __bfloat162float(__float2bfloat16_rn(sum)));
    } else {
        static_cast<float*>(mg)[h] += sum;
    }
}

}  // namespace

cudaError_t launch_gate_forward(const __nv_bfloat16* hidden, const __nv_bfloat16* w, int T, int H, float* gate,
                                cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const int blocks = (T * 32 + 255) / 256;
    const cudaError_t e = launch_pdl(gate_forward_kernel, dim3(blocks), dim3(256), 0, st,
                                     reinterpret_cast<const uint4*>(hidden), reinterpret_cast<const uint4*>(w), T,
                                     H / 8, gate);
    count_launch();
    return e;
}

cudaError_t launch_gate_backward(const __nv_bfloat16* hidden, const float* gate, const float* partial, int n_part,
                                 int T, int H, float* dz, float* gpart, void* mg_gate, bool mg_bf16, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const int chunks = (T + kGateChunk - 1) / kGateChunk;
    cudaError_t e = launch_pdl(gate_grad_chunk_kernel, dim3(chunks), dim3(256), 0, st,
                               reinterpret_cast<const uint4*>(hidden), gate, partial, n_part, T, H / 8, dz,
                               reinterpret_cast<float4*>(gpart));
    count_launch();
    if (e != cudaSuccess) return e;
    e = launch_pdl(gate_grad_reduce_kernel, dim3((H + 255) / 256), dim3(256), 0, st, gpart, chunks, H, mg_gate,
                   mg_bf16 ? 1 : 0);
    count_launch();
    return e;
}

}  // namespace moe
