// Bandwidth-bound kernels of the MoE layer: the dispatch gather, the combine
// (un-permute + prob-weighted sum + shared expert), and the backward
// un-permute reduction with the dense dprobs scatter.
//
// "feat(moe): add a megakernel backend with MOK integration", Summary
// (dispatch, combine) and Design > Authoritative routing maps (the backward
// adapter scatters router-weight gradients into the dense prob tensor).
//
// Rows are moved as vectors of 8 elements; the experts' outputs and input
// gradients (fp32, or bf16 with bf16 activations) are summed in fp32 in slot
// order, so the results are deterministic and rounded to bf16 once.
#include "device_common.cuh"
#include "internal.h"

namespace moe {

namespace {

// The grad gather, walked from the token side: item t*k + s copies row t of src
// to the permuted row row_of[t,s] of dst (nothing for a missing route); items
// past T*k zero the padding rows at the end of each expert's segment
// (offs_pad[e] + counts[e] up to the next multiple of 64: the weight gradients' K
// ranges end there, and the padding rows after it are read by nothing). Consecutive warps
// take the slots of one token, so each source row leaves DRAM once however its
// slots are spread over the experts. One warp per item, 16-byte vectors; with
// dst_q the row is also quantised to MXFP8 along H.
// QUANT: dst_q / dst_sf are set (MXFP8 routed weights); a build of its own (see route_place)
template <bool QUANT>
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ src,
                                                          const int* __restrict__ row_of,
                                                          const int* __restrict__ counts,
                                                          const int* __restrict__ offs_pad, int T, int E, int k,
                                                          int vec_per_row, uint4* __restrict__ dst,
                                                          uint8_t* __restrict__ dst_q, uint8_t* __restrict__ dst_sf) {
    pdl_wait();
    pdl_trigger();
    const int64_t item = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int64_t n_routes = int64_t(T) * k;
    const uint4* from = nullptr;
    int64_t pos;
    if (item < n_routes) {
        pos = __ldg(row_of + item);
        if (pos < 0) return;
        from = src + (item / k) * vec_per_row;
    } else {
        const int64_t j = item - n_routes;
        if (j >= int64_t(E) * kBM) return;
        const int e = int(j / kBM);
        const int r = int(j % kBM);
        const int cnt = __ldg(counts + e);
        if (r >= (cnt + kBK - 1) / kBK * kBK - cnt) return;
        pos = __ldg(offs_pad + e) + cnt + r;
    }
    uint4* d = dst + pos * vec_per_row;
    if constexpr (QUANT)  // the routed dgrad-down GEMM's operand
        copy_quant_row(from, d, dst_q, dst_sf, pos, vec_per_row);
    else
        copy_row(from, d, vec_per_row);
}

// 8 elements of a row, element index 8 * i: one 16-byte vector of bf16 or two of fp32
template <bool F32>
struct Vec8 {
    uint4 v[F32 ? 2 : 1];
    __device__ __forceinline__ void load(const void* base, int64_t i) {
        const uint4* p = reinterpret_cast<const uint4*>(base) + i * (F32 ? 2 : 1);
        v[0] = __ldg(p);
        if (F32) v[F32 ? 1 : 0] = __ldg(p + 1);
    }
    __device__ __forceinline__ void to_float(float (&f)[8]) const {
        if (F32) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint4 w = v[F32 ? j : 0];
                f[4 * j] = __uint_as_float(w.x);
                f[4 * j + 1] = __uint_as_float(w.y);
                f[4 * j + 2] = __uint_as_float(w.z);
                f[4 * j + 3] = __uint_as_float(w.w);
            }
        } else {
            unpack_bf16x2(v[0].x, f[0], f[1]);
            unpack_bf16x2(v[0].y, f[2], f[3]);
            unpack_bf16x2(v[0].z, f[4], f[5]);
            unpack_bf16x2(v[0].w, f[6], f[7]);
        }
    }
};

// acc += w * (8 elements at vector i of base)
template <bool F32>
__device__ __forceinline__ void fma_x8(float (&acc)[8], const void* base, int64_t i, float w) {
    Vec8<F32> x;
    x.load(base, i);
    float f[8];
    x.to_float(f);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = fmaf(w, f[j], acc[j]);
}

// acc += 8 elements at vector i of base
template <bool F32>
__device__ __forceinline__ void add_x8(float (&acc)[8], const void* base, int64_t i) {
    Vec8<F32> x;
    x.load(base, i);
    float f[8];
    x.to_float(f);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] += f[j];
}

// acc += sum over the valid slots s (row_of_t[s] >= 0) of pp_t[s] * (8 elements of
// row row_of_t[s] at column vector v), in slot order: the indices and weights of up
// to four slots, then their rows, are loaded before any is used
template <bool F32>
__device__ __forceinline__ void acc_slots(float (&acc)[8], const void* __restrict__ rows, int vec_per_row, int v,
                                          const int* __restrict__ row_of_t, const float* __restrict__ pp_t, int k) {
    constexpr int B = 4;
    for (int s0 = 0; s0 < k; s0 += B) {
        int r[B];
        float w[B];
        Vec8<F32> val[B];
#pragma unroll
        for (int j = 0; j < B; ++j) {
            r[j] = s0 + j < k ? __ldg(row_of_t + s0 + j) : -1;
            w[j] = s0 + j < k ? __ldg(pp_t + s0 + j) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < B; ++j)
            if (r[j] >= 0) val[j].load(rows, int64_t(r[j]) * vec_per_row + v);
#pragma unroll
        for (int j = 0; j < B; ++j) {
            if (r[j] < 0) continue;
            float f[8];
            val[j].to_float(f);
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = fmaf(w[j], f[q], acc[q]);
        }
    }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&acc)[8]) {
    return make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                      pack_bf16x2(acc[6], acc[7]));
}

// out[t] = gate[t] y_shared[t] + sum over valid slots s of pp[t,s] y[row_of[t,s]]
// (gate 1 without a shared output gate): expert outputs in fp32 (or bf16), fp32 sum
// in slot order, one bf16 rounding at the end; 8 columns per thread
template <bool F32>
__global__ void __launch_bounds__(256) combine_kernel(const void* __restrict__ ys, const float* __restrict__ gate,
                                                      const void* __restrict__ y, const int* __restrict__ row_of,
                                                      const float* __restrict__ pp, int T, int vec_per_row, int k,
                                                      uint4* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    const int64_t total = int64_t(T) * vec_per_row;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
        const int t = int(i / vec_per_row);
        const int v = int(i - int64_t(t) * vec_per_row);
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (ys) fma_x8<F32>(acc, ys, i, gate ? __ldg(gate + t) : 1.0f);  // no shared expert: ys null
        acc_slots<F32>(acc, y, vec_per_row, v, row_of + int64_t(t) * k, pp + int64_t(t) * k, k);
        out[i] = pack_bf16x8(acc);
    }
}

// acc += sum over the valid slots s of (8 elements of row row_of_t[s] at column vector
// v), in slot order: the row indices of up to four slots, then their rows, are loaded
// before any is added
template <bool F32>
__device__ __forceinline__ void add_slots(float (&acc)[8], const void* __restrict__ rows, int vec_per_row, int v,
                                          const int* __restrict__ row_of_t, int k) {
    constexpr int B = 4;
    for (int s0 = 0; s0 < k; s0 += B) {
        int r[B];
        Vec8<F32> val[B];
#pragma unroll
        for (int j = 0; j < B; ++j) r[j] = s0 + j < k ? __ldg(row_of_t + s0 + j) : -1;
#pragma unroll
        for (int j = 0; j < B; ++j)
            if (r[j] >= 0) val[j].load(rows, int64_t(r[j]) * vec_per_row + v);
#pragma unroll
        for (int j = 0; j < B; ++j) {
            if (r[j] < 0) continue;
            float f[8];
            val[j].to_float(f);
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] += f[q];
        }
    }
}

// the dprob of route row r: the sum of its n_part partial dot products, in order
__device__ __forceinline__ float route_dprob(const float* __restrict__ partial, int n_part, int r) {
    const float* p = partial + int64_t(r) * n_part;
    float val = 0.0f;
    for (int j = 0; j < n_part; ++j) val += __ldg(p + j);
    return val;
}

// dhidden[t] = dx_shared[t] (+ dz[t] w, the shared output gate's term) + sum
// over valid slots of dx_perm[row_of[t,s]];
// dprobs[t,e] = sum of the dprob partials of the route (t,e), 0 off the map; with
// slot_dprobs, dprobs[t,s] of slot s instead (0 for an empty slot); written by a
// second grid-stride pass over the dprobs entries
template <bool F32>
__global__ void __launch_bounds__(256) unpermute_kernel(const void* __restrict__ dxs, const void* __restrict__ dxp,
                                                        const int* __restrict__ row_of, const int* __restrict__ ids,
                                                        const float* __restrict__ partial, int n_part, int T,
                                                        int vec_per_row, int k, int E, const float* __restrict__ dz,
                                                        const uint4* __restrict__ gate_w,
                                                        uint4* __restrict__ dhidden, float* __restrict__ dprobs,
                                                        int slot_dprobs) {
    pdl_wait();
    pdl_trigger();
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    const int64_t total = int64_t(T) * vec_per_row;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total; i += stride) {
        const int t = int(i / vec_per_row);
        const int v = int(i - int64_t(t) * vec_per_row);
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (dxs) add_x8<F32>(acc, dxs, i);  // no shared expert: dxs null
        if (dz) {
            const float d = __ldg(dz + t);
            const uint4 wv = __ldg(gate_w + v);
            float wf[8];
            unpack_bf16x2(wv.x, wf[0], wf[1]);
            unpack_bf16x2(wv.y, wf[2], wf[3]);
            unpack_bf16x2(wv.z, wf[4], wf[5]);
            unpack_bf16x2(wv.w, wf[6], wf[7]);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = fmaf(d, wf[j], acc[j]);
        }
        add_slots<F32>(acc, dxp, vec_per_row, v, row_of + int64_t(t) * k, k);
        dhidden[i] = pack_bf16x8(acc);
    }
    if (slot_dprobs) {
        for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < int64_t(T) * k; i += stride) {
            const int r = __ldg(row_of + i);
            dprobs[i] = r >= 0 ? route_dprob(partial, n_part, r) : 0.0f;
        }
        return;
    }
    const int64_t total_p = int64_t(T) * E;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total_p; i += stride) {
        const int t = int(i / E);
        const int e = int(i - int64_t(t) * E);
        float val = 0.0f;
        for (int s = 0; s < k; ++s)
            if (__ldg(ids + int64_t(t) * k + s) == e)
                val = route_dprob(partial, n_part, __ldg(row_of + int64_t(t) * k + s));
        dprobs[i] = val;
    }
}

int grid_for(int64_t work, int threads, int num_sms) {
    int64_t g = (work + threads - 1) / threads;
    const int64_t cap = int64_t(num_sms) * 8;
    if (g > cap) g = cap;
    return g < 1 ? 1 : int(g);
}

}  // namespace

cudaError_t launch_gather_rows(const __nv_bfloat16* src, const int* row_of, const int* counts, const int* offs_pad,
                               int T, int E, int k, int H, __nv_bfloat16* dst, uint8_t* dst_q, uint8_t* dst_sf,
                               cudaStream_t st) {
    const int64_t items = int64_t(T) * k + int64_t(E) * kBM;
    const int64_t blocks = (items + 7) / 8;
    const cudaError_t e = launch_pdl(dst_q ? gather_rows_kernel<true> : gather_rows_kernel<false>,
                                     dim3(unsigned(blocks)), dim3(256), 0, st,
                                     reinterpret_cast<const uint4*>(src), row_of, counts, offs_pad, T, E, k, H / 8,
                                     reinterpret_cast<uint4*>(dst), dst_q, dst_sf);
    count_launch();
    return e;
}

cudaError_t launch_combine(const void* ys, const float* gate, const void* y, bool f32, const int* row_of,
                           const float* pp, int T, int H, int k, __nv_bfloat16* out, int num_sms, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const int grid = grid_for(int64_t(T) * (H / 8), 256, num_sms);
    const cudaError_t e =
        launch_pdl(f32 ? combine_kernel<true> : combine_kernel<false>, dim3(grid), dim3(256), 0, st, ys, gate, y,
                   row_of, pp, T, H / 8, k, reinterpret_cast<uint4*>(out));
    count_launch();
    return e;
}

cudaError_t launch_unpermute(const void* dxs, const void* dxp, bool f32, const int* row_of, const int* ids,
                             const float* partial, int n_part, int T, int H, int k, int E, const float* dz,
                             const __nv_bfloat16* gate_w, __nv_bfloat16* dhidden, float* dprobs, bool slot_dprobs,
                             int num_sms, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const int grid = grid_for(int64_t(T) * (H / 8), 256, num_sms);
    const cudaError_t e = launch_pdl(f32 ? unpermute_kernel<true> : unpermute_kernel<false>, dim3(grid), dim3(256), 0,
                                     st, dxs, dxp, row_of, ids, partial, n_part, T, H / 8, k, E, dz,
                                     reinterpret_cast<const uint4*>(gate_w), reinterpret_cast<uint4*>(dhidden), dprobs,
                                     slot_dprobs ? 1 : 0);
    count_launch();
    return e;
}

}  // namespace moe
