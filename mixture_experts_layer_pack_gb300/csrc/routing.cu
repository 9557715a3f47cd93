// Routing kernels: dense routing map -> fixed-width expert ids, then the
// dispatch permutation (per-expert token segments), all on the device.
//
// "feat(moe): add a megakernel backend with MOK integration", Design >
// Authoritative routing maps: the router's dense map is converted into a
// fixed-width top-k representation, missing routes are expert id -1, the
// matching probabilities are gathered. Dispatch on one GPU is a local
// permutation (same page, Summary).
//
// Order is deterministic: slots list a token's experts in ascending id order;
// within an expert, routes are ordered by token index. Each expert segment is
// padded to a multiple of 128 rows so that a GEMM row tile never spans two
// experts; padding rows have source token -1 and prob 0.
//
// Three launches: (1) pack + per-chunk expert histogram (smem atomics),
// (2) one block scans the histogram over chunks and experts, writes the
// segment offsets and the expert of every 128-row tile, (3) each chunk places
// its routes at their stable positions.
#include "device_common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kPackThreads = 256;

__global__ void __launch_bounds__(kPackThreads) route_pack_kernel(const uint8_t* __restrict__ map,
                                                                  const float* __restrict__ probs, int T, int E,
                                                                  int k, int* __restrict__ ids, float* __restrict__ pp,
                                                                  int* __restrict__ row_of, int* __restrict__ hist,
                                                                  int* status) {
    extern __shared__ int s_hist[];  // [E]
    const int chunk = blockIdx.x;
    const int t0 = chunk * kChunk;
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const unsigned lt_mask = (1u << lane) - 1u;
    const int t_end = min(t0 + kChunk, T);
    for (int t = t0 + warp; t < t_end; t += nwarps) {
        const uint8_t* row = map + int64_t(t) * E;
        // pass 1: count the row's routes
        int cnt = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            const bool on = e < E && row[e] != 0;
            cnt += __popc(__ballot_sync(0xffffffffu, on));
        }
        int* ids_t = ids + int64_t(t) * k;
        float* pp_t = pp + int64_t(t) * k;
        int* ro_t = row_of + int64_t(t) * k;
        if (cnt > k) {
            // more routes than slots: flag it and drop the row's routes
            if (lane == 0) atomicOr(status, kStatusRouting);
            for (int s = lane; s < k; s += 32) {
                ids_t[s] = -1;
                pp_t[s] = 0.0f;
                ro_t[s] = -1;
            }
            continue;
        }
        // pass 2: write slots in ascending expert order
        int slot_base = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            const bool on = e < E && row[e] != 0;
            const unsigned m = __ballot_sync(0xffffffffu, on);
            if (on) {
                const int slot = slot_base + __popc(m & lt_mask);
                ids_t[slot] = e;
                pp_t[slot] = probs[int64_t(t) * E + e];
                atomicAdd(&s_hist[e], 1);
            }
            slot_base += __popc(m);
        }
        for (int s = cnt + lane; s < k; s += 32) {
            ids_t[s] = -1;
            pp_t[s] = 0.0f;
            ro_t[s] = -1;
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[int64_t(chunk) * E + e] = s_hist[e];
}

// block-wide exclusive scan of one int per thread (blockDim.x <= 1024)
__device__ int block_excl_scan(int v, int* s_warp, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        int w = lane < nw ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < nw) s_warp[lane] = w;  // inclusive prefix of warp sums
    }
    __syncthreads();
    const int warp_prefix = warp > 0 ? s_warp[warp - 1] : 0;
    total = s_warp[(blockDim.x >> 5) - 1];
    __syncthreads();
    return warp_prefix + x - v;
}

__global__ void __launch_bounds__(1024) route_scan_kernel(int* __restrict__ hist, int nchunks, int E,
                                                          int* __restrict__ counts, int* __restrict__ offsets,
                                                          int* __restrict__ offs_pad, int* __restrict__ mtile_expert,
                                                          int* __restrict__ meta, int* __restrict__ perm_src,
                                                          float* __restrict__ pp_perm) {
    __shared__ int s_warp[32];
    const int e = threadIdx.x;
    int cnt = 0;
    if (e < E) {
        // exclusive scan over chunks, in place: hist[c][e] becomes the chunk's base
        for (int c = 0; c < nchunks; ++c) {
            const int v = hist[int64_t(c) * E + e];
            hist[int64_t(c) * E + e] = cnt;
            cnt += v;
        }
    }
    const int padded = (cnt + kBM - 1) / kBM * kBM;
    int total_cnt, total_pad;
    const int off = block_excl_scan(cnt, s_warp, total_cnt);
    const int offp = block_excl_scan(padded, s_warp, total_pad);
    if (e < E) {
        counts[e] = cnt;
        offsets[e] = off;
        offs_pad[e] = offp;
        for (int j = 0; j < padded / kBM; ++j) mtile_expert[offp / kBM + j] = e;
        for (int j = cnt; j < padded; ++j) {
            perm_src[offp + j] = -1;
            pp_perm[offp + j] = 0.0f;
        }
    }
    if (e == 0) {
        offsets[E] = total_cnt;
        offs_pad[E] = total_pad;
        meta[0] = total_pad / kBM;  // number of 128-row tiles
        meta[1] = total_cnt;        // R, valid routes
        meta[2] = total_pad;        // rows including padding
    }
}

__global__ void __launch_bounds__(512) route_place_kernel(const int* __restrict__ ids, const float* __restrict__ pp,
                                                          int T, int E, int k, const int* __restrict__ hist,
                                                          const int* __restrict__ offs_pad,
                                                          int* __restrict__ perm_src, float* __restrict__ pp_perm,
                                                          int* __restrict__ row_of) {
    extern __shared__ int s_ids[];  // [kChunk * k]
    const int chunk = blockIdx.x;
    const int t0 = chunk * kChunk;
    const int n = kChunk * k;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int t = t0 + i / k;
        s_ids[i] = t < T ? ids[int64_t(t0) * k + i] : -1;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int pos = offs_pad[e] + hist[int64_t(chunk) * E + e];
        for (int i = 0; i < n; ++i) {
            if (s_ids[i] == e) {
                const int t = t0 + i / k;
                const int64_t ts = int64_t(t0) * k + i;
                perm_src[pos] = t;
                pp_perm[pos] = pp[ts];
                row_of[ts] = pos;
                ++pos;
            }
        }
    }
}

__global__ void export_routing_kernel(const int* __restrict__ ids, const int* __restrict__ row_of,
                                      const int* __restrict__ perm_src_pad, const int* __restrict__ counts,
                                      const int* __restrict__ offsets, const int* __restrict__ offs_pad,
                                      const int* __restrict__ mtile_expert, const int* __restrict__ meta, int T,
                                      int k, int max_rows, int32_t* __restrict__ perm_out,
                                      int32_t* __restrict__ row_of_out) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    const int rows = meta[2];
    if (perm_out) {
        for (int64_t r = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; r < rows && r < max_rows; r += stride) {
            const int e = mtile_expert[r / kBM];
            const int j = int(r) - offs_pad[e];
            if (j < counts[e]) perm_out[offsets[e] + j] = perm_src_pad[r];
        }
    }
    if (row_of_out) {
        for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < int64_t(T) * k; i += stride) {
            const int rp = row_of[i];
            row_of_out[i] = rp < 0 ? -1 : rp - offs_pad[ids[i]] + offsets[ids[i]];
        }
    }
}

}  // namespace

cudaError_t launch_route_pack(const uint8_t* map, const float* probs, int T, int E, int k, int* ids, float* pp,
                              int* row_of, int* hist, int* status, cudaStream_t st) {
    const int nchunks = (T + kChunk - 1) / kChunk;
    if (nchunks == 0) return cudaSuccess;
    route_pack_kernel<<<nchunks, kPackThreads, E * sizeof(int), st>>>(map, probs, T, E, k, ids, pp, row_of, hist,
                                                                      status);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_route_scan(int* hist, int nchunks, int E, int* counts, int* offsets, int* offs_pad,
                              int* mtile_expert, int* meta, int* perm_src, float* pp_perm, cudaStream_t st) {
    const int threads = (E + 31) / 32 * 32;
    route_scan_kernel<<<1, threads, 0, st>>>(hist, nchunks, E, counts, offsets, offs_pad, mtile_expert, meta,
                                             perm_src, pp_perm);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_route_place(const int* ids, const float* pp, int T, int E, int k, const int* hist,
                               const int* offs_pad, int* perm_src, float* pp_perm, int* row_of, cudaStream_t st) {
    const int nchunks = (T + kChunk - 1) / kChunk;
    if (nchunks == 0) return cudaSuccess;
    const int threads = E < 512 ? (E + 31) / 32 * 32 : 512;
    route_place_kernel<<<nchunks, threads, kChunk * k * sizeof(int), st>>>(ids, pp, T, E, k, hist, offs_pad,
                                                                           perm_src, pp_perm, row_of);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_export_routing(const int* ids, const int* row_of, const int* perm_src_pad, const int* counts,
                                  const int* offsets, const int* offs_pad, const int* mtile_expert, const int* meta,
                                  int T, int k, int max_rows, int32_t* perm_src_out, int32_t* row_of_out,
                                  cudaStream_t st) {
    export_routing_kernel<<<256, 256, 0, st>>>(ids, row_of, perm_src_pad, counts, offsets, offs_pad, mtile_expert,
                                               meta, T, k, max_rows, perm_src_out, row_of_out);
    count_launch();
    return cudaGetLastError();
}

}  // namespace moe
