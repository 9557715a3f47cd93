// Routing kernels: dense routing map -> fixed-width expert ids, then the
// dispatch permutation (per-expert token segments) and the dispatch gather,
// all on the device.
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
// experts; padding rows have source token -1 and prob 0, and zero activations up
// to the end of the expert's last 64-row block that holds a route (the weight
// gradients' K ranges end there; the padding rows after it are read by nothing).
//
// The forward's three launches:
//   pack+rank  one thread per token, 128-token blocks: ids[t,:], pp[t,:], -1 slots;
//              flags rows with > k routes; a ballot per expert ranks the routes
//              inside the block and counts them per expert
//   scan       one block: each expert's chunk counts scanned in token order (the
//              chunk's rank offset, the expert's count), then exclusive scans of
//              counts (compact and 128-padded), the expert of every 128-row tile
//   place      one warp per route (and per padding row): writes the permutation
//              entries and copies the token's hidden row into its permuted row
// moe_route_noalloc (end of file) ranks with one block per expert instead
// (route_pack_kernel, route_rank_kernel), whose only scratch is one int per route.
#include "../../include/moe.h"
#include "device_common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kRankThreads = 1024;

__global__ void __launch_bounds__(32 * kWarpsPerBlock) route_pack_kernel(const uint8_t* __restrict__ map,
                                                                       const float* __restrict__ probs, int T, int E,
                                                                       int k, int* __restrict__ ids,
                                                                       float* __restrict__ pp,
                                                                       int* __restrict__ row_of, int* status) {
    const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (t >= T) return;
    const int lane = threadIdx.x & 31;
    const unsigned lt_mask = (1u << lane) - 1u;
    const uint8_t* row = map + int64_t(t) * E;
    // lane holds experts lane, lane+32, ...: bit j of `mine` = map[t, lane + 32 j]
    uint32_t mine = 0;
    const int rounds = (E + 31) >> 5;
    for (int j = 0; j < rounds; ++j) {
        const int e = lane + 32 * j;
        if (e < E && __ldg(row + e) != 0) mine |= 1u << j;
    }
    int cnt = 0;
    for (int j = 0; j < rounds; ++j) cnt += __popc(__ballot_sync(0xffffffffu, (mine >> j) & 1u));
    int* ids_t = ids + int64_t(t) * k;
    float* pp_t = pp + int64_t(t) * k;
    int* ro_t = row_of + int64_t(t) * k;
    if (cnt > k) {  // more routes than slots: flag it, drop the row's routes
        if (lane == 0) atomicOr(status, kStatusRouting);
        cnt = 0;
        mine = 0;
    }
    int base = 0;
    for (int j = 0; j < rounds; ++j) {
        const bool on = (mine >> j) & 1u;
        const unsigned m = __ballot_sync(0xffffffffu, on);
        if (on) {
            const int slot = base + __popc(m & lt_mask);
            const int e = lane + 32 * j;
            ids_t[slot] = e;
            pp_t[slot] = __ldg(probs + int64_t(t) * E + e);
        }
        base += __popc(m);
    }
    for (int s = cnt + lane; s < k; s += 32) {
        ids_t[s] = -1;
        pp_t[s] = 0.0f;
        ro_t[s] = -1;
    }
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

// block e: thread i owns tokens [i*C, (i+1)*C); a stable block scan of their
// routes to expert e gives each one its rank; rank[t*k + s] for ids[t,s] == e
__global__ void __launch_bounds__(kRankThreads) route_rank_kernel(const uint8_t* __restrict__ map,
                                                                  const int* __restrict__ ids, int T, int E, int k,
                                                                  int* __restrict__ rank, int* __restrict__ counts) {
    __shared__ int s_warp[32];
    const int e = blockIdx.x;
    const int C = (T + blockDim.x - 1) / blockDim.x;
    const int t0 = threadIdx.x * C;
    const int t1 = min(t0 + C, T);
    uint64_t bits = 0;  // C <= 64 is checked on the host
    int n = 0;
    for (int t = t0; t < t1; ++t) {
        // a row with more than k routes was dropped by the pack kernel: ids decide
        if (__ldg(map + int64_t(t) * E + e) != 0) bits |= 1ull << (t - t0);
    }
    for (int t = t0; t < t1; ++t) {
        if ((bits >> (t - t0)) & 1ull) {
            const int* ids_t = ids + int64_t(t) * k;
            bool found = false;
            for (int s = 0; s < k; ++s) found |= (ids_t[s] == e);
            if (!found) bits &= ~(1ull << (t - t0));
        }
    }
    n = __popcll(bits);
    int total;
    int r = block_excl_scan(n, s_warp, total);
    for (int t = t0; t < t1; ++t) {
        if ((bits >> (t - t0)) & 1ull) {
            const int* ids_t = ids + int64_t(t) * k;
            for (int s = 0; s < k; ++s)
                if (ids_t[s] == e) rank[int64_t(t) * k + s] = r;
            ++r;
        }
    }
    if (threadIdx.x == 0) counts[e] = total;
}

// Fused route-pack and chunk-local rank (the forward's routing). Block c owns
// tokens [c*C, c*C+C) (C = kRankChunk), one thread per token, warp w its 32
// tokens. The block first copies its C map rows (one contiguous, coalesced
// range of the map) into shared memory, rows padded to an odd number of words
// so that the threads' row reads fall in distinct banks. Each thread counts its
// row: more than k routes flags the status and drops the row; otherwise its
// experts, ascending, fill ids/pp (-1 / 0 / row_of -1 pad the slots). One ballot
// per expert gives the warp's tokens routed to it: a route's rank among them
// (earlier lanes = earlier tokens) and the warp's count. The counts' exclusive
// prefix over the block's warps is added to every rank, and the block's totals
// go to hist[c][e]; a later scan over blocks completes the stable (expert,
// token) order.
// With topk_ids set (the router's top-k output instead of the dense map), the
// map rows are built in shared memory from topk_ids[T,k] (-1 = no route); a row
// with an id outside [-1, E) or a repeated id flags the status and is dropped;
// the slots keep the caller's order, with probs from topk_probs[T,k].
__global__ void __launch_bounds__(kRankChunk) route_pack_rank_kernel(const uint8_t* __restrict__ map,
                                                                     const float* __restrict__ probs, int T, int E,
                                                                     int k, int* __restrict__ ids,
                                                                     float* __restrict__ pp, int* __restrict__ row_of,
                                                                     int* __restrict__ rank, int* __restrict__ hist,
                                                                     int words_aligned, int* status,
                                                                     const int* __restrict__ topk_ids,
                                                                     const float* __restrict__ topk_probs) {
    pdl_wait();
    pdl_trigger();
    constexpr int W = kRankChunk / 32;
    extern __shared__ int s_dyn[];
    int* s_cnt = s_dyn;                                           // [W][E]: warp counts, then warp offsets
    int* s_e = s_cnt + W * E;                                     // [kRankChunk][k]: a token's experts
    int* s_r = s_e + kRankChunk * k;                              // [kRankChunk][k]: their ranks in the warp
    const int RW = (E + 3) / 4 + (((E + 3) / 4) % 2 == 0 ? 1 : 0);  // row stride in words (odd)
    uint32_t* s_rows = reinterpret_cast<uint32_t*>(s_r + kRankChunk * k);  // [kRankChunk][RW]
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const int t0 = blockIdx.x * kRankChunk;
    const int nt = min(kRankChunk, T - t0);
    const int t = t0 + threadIdx.x;
    const bool in = threadIdx.x < nt;

    // the chunk's rows: bytes [t0*E, (t0+nt)*E) of the map
    const uint8_t* src = topk_ids ? nullptr : map + int64_t(t0) * E;
    bool bad_ids = false;  // top-k input: an id out of range or repeated in this thread's row
    if (topk_ids) {
        for (int i = threadIdx.x; i < kRankChunk * RW; i += blockDim.x) s_rows[i] = 0u;
        __syncthreads();
        if (in) {
            uint8_t* row8 = reinterpret_cast<uint8_t*>(s_rows + threadIdx.x * RW);
            int n_ids = 0, n_set = 0;
            for (int s = 0; s < k; ++s) {
                const int e = __ldg(topk_ids + int64_t(t) * k + s);
                if (e < -1 || e >= E) {
                    bad_ids = true;
                } else if (e >= 0) {
                    ++n_ids;
                    n_set += row8[e] == 0 ? 1 : 0;
                    row8[e] = 1;
                }
            }
            bad_ids = bad_ids || n_set != n_ids;
        }
    } else if (words_aligned == 4) {  // E % 16 == 0 and a 16-byte aligned map: 16-byte loads, 8 in flight
        const int eq = E / 16;
        const int nq = nt * eq;
        const uint4* s4 = reinterpret_cast<const uint4*>(src);
        for (int i0 = threadIdx.x; i0 < nq; i0 += 8 * blockDim.x) {
            uint4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = i0 + j * blockDim.x;
                if (i < nq) v[j] = __ldg(s4 + i);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = i0 + j * blockDim.x;
                if (i < nq) {
                    const int r = i / eq;
                    uint32_t* d = s_rows + r * RW + 4 * (i - r * eq);
                    d[0] = v[j].x;
                    d[1] = v[j].y;
                    d[2] = v[j].z;
                    d[3] = v[j].w;
                }
            }
        }
    } else if (words_aligned) {  // E % 4 == 0 and a 4-byte aligned map
        const int ew = E / 4;
        const int nw = nt * ew;
        for (int i = threadIdx.x; i < nw; i += blockDim.x) {
            const int r = i / ew;
            s_rows[r * RW + (i - r * ew)] = __ldg(reinterpret_cast<const uint32_t*>(src) + i);
        }
    } else {
        uint8_t* rows8 = reinterpret_cast<uint8_t*>(s_rows);
        const int nb = nt * E;
        for (int i = threadIdx.x; i < nb; i += blockDim.x) {
            const int r = i / E;
            rows8[r * RW * 4 + (i - r * E)] = __ldg(src + i);
        }
        // zero the tail bytes of each row's last word
        for (int r = threadIdx.x; r < nt; r += blockDim.x)
            for (int b = E; b < ((E + 3) / 4) * 4; ++b) rows8[r * RW * 4 + b] = 0;
    }
    __syncthreads();

    const uint32_t* my = s_rows + threadIdx.x * RW;
    const int EW = (E + 3) / 4;
    int cnt = 0;
    if (in)
        for (int j = 0; j < EW; ++j) {
            const uint32_t v = my[j];
            cnt += ((v & 0xffu) != 0) + ((v & 0xff00u) != 0) + ((v & 0xff0000u) != 0) + ((v & 0xff000000u) != 0);
        }
    bool valid = in;
    if (in && (cnt > k || bad_ids)) {  // more routes than slots, or bad ids: flag it, drop the row's routes
        atomicOr(status, kStatusRouting);
        valid = false;
    }
    // one ballot per expert; only shared memory is touched inside the loop
    const unsigned lt = (1u << lane) - 1u;
    int* my_e = s_e + threadIdx.x * k;
    int* my_r = s_r + threadIdx.x * k;
    int sl = 0;
    for (int j = 0; j < EW; ++j) {
        const uint32_t v = valid ? my[j] : 0u;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int e = 4 * j + b;
            if (e >= E) break;
            const bool on = ((v >> (8 * b)) & 0xffu) != 0;
            const unsigned m = __ballot_sync(0xffffffffu, on);
            if (lane == 0) s_cnt[w * E + e] = __popc(m);
            if (on) {
                my_e[sl] = e;
                my_r[sl] = __popc(m & lt);
                ++sl;
            }
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
#pragma unroll
        for (int ww = 0; ww < W; ++ww) {
            const int c = s_cnt[ww * E + e];
            s_cnt[ww * E + e] = run;
            run += c;
        }
        hist[int64_t(blockIdx.x) * E + e] = run;
    }
    __syncthreads();
    if (!in) return;
    int* ids_t = ids + int64_t(t) * k;
    float* pp_t = pp + int64_t(t) * k;
    int* rk_t = rank + int64_t(t) * k;
    if (topk_ids) {  // the caller's slot order: find each slot's expert among the ranked ones
        for (int s = 0; s < k; ++s) {
            const int e = valid ? __ldg(topk_ids + int64_t(t) * k + s) : -1;
            int j = 0;
            while (j < sl && my_e[j] != e) ++j;
            if (e >= 0 && j < sl) {
                ids_t[s] = e;
                pp_t[s] = __ldg(topk_probs + int64_t(t) * k + s);
                rk_t[s] = my_r[j] + s_cnt[w * E + e];
            } else {
                ids_t[s] = -1;
                pp_t[s] = 0.0f;
                row_of[int64_t(t) * k + s] = -1;
            }
        }
        return;
    }
    for (int s0 = 0; s0 < k; s0 += 8) {  // the probs of eight slots in flight at a time
        float pv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            pv[j] = (s0 + j < sl) ? __ldg(probs + int64_t(t) * E + my_e[s0 + j]) : 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int s = s0 + j;
            if (s >= k) break;
            if (s < sl) {
                const int e = my_e[s];
                ids_t[s] = e;
                pp_t[s] = pv[j];
                rk_t[s] = my_r[s] + s_cnt[w * E + e];
            } else {
                ids_t[s] = -1;
                pp_t[s] = 0.0f;
                row_of[int64_t(t) * k + s] = -1;
            }
        }
    }
}

size_t pack_rank_smem(int E, int k) {
    const int RW = (E + 3) / 4 + (((E + 3) / 4) % 2 == 0 ? 1 : 0);
    return size_t(kRankChunk / 32) * E * sizeof(int) + 2 * size_t(kRankChunk) * k * sizeof(int) +
           size_t(kRankChunk) * RW * 4;
}

// One block, thread e per expert: exclusive scan of the chunk totals of
// expert e in chunk order (hist[c][e] becomes the expert's rank offset of
// chunk c) and the expert's count, then exclusive scans of the counts
// (compact and 128-padded), the expert of every 128-row tile and the totals.
__global__ void __launch_bounds__(1024) route_scan_chunks_kernel(int* __restrict__ hist, int chunks, int E,
                                                                 int* __restrict__ counts, int* __restrict__ offsets,
                                                                 int* __restrict__ offs_pad,
                                                                 int* __restrict__ mtile_expert,
                                                                 int* __restrict__ meta, int shared_tiles,
                                                                 int* __restrict__ mtile_x, int* __restrict__ seg_x) {
    pdl_wait();
    pdl_trigger();
    __shared__ int s_warp[32];
    const int e = threadIdx.x;
    int cnt = 0;
    if (e < E) {
        int c = 0;
        for (; c + 8 <= chunks; c += 8) {  // eight loads in flight per step
            int h[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) h[j] = hist[int64_t(c + j) * E + e];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                hist[int64_t(c + j) * E + e] = cnt;
                cnt += h[j];
            }
        }
        for (; c < chunks; ++c) {
            const int h = hist[int64_t(c) * E + e];
            hist[int64_t(c) * E + e] = cnt;
            cnt += h;
        }
        counts[e] = cnt;
    }
    const int padded = (cnt + kBM - 1) / kBM * kBM;
    int total_cnt, total_pad;
    const int off = block_excl_scan(cnt, s_warp, total_cnt);
    const int offp = block_excl_scan(padded, s_warp, total_pad);
    if (e < E) {
        offsets[e] = off;
        offs_pad[e] = offp;
        for (int j = 0; j < padded / kBM; ++j) mtile_expert[offp / kBM + j] = e;
    }
    if (e == 0) {
        offsets[E] = total_cnt;
        offs_pad[E] = total_pad;
        meta[0] = total_pad / kBM;
        meta[1] = total_cnt;
        meta[2] = total_pad;
    }
    if (!mtile_x) return;
    // the shared expert and the routed experts as one grouped GEMM: group 0 is the
    // shared expert over rows [0, 128 * shared_tiles), group e + 1 routed expert e
    // at its segment shifted by those rows
    const int r0 = shared_tiles * kBM;
    for (int j = threadIdx.x; j < shared_tiles; j += blockDim.x) mtile_x[j] = 0;
    if (e < E) {
        for (int j = 0; j < padded / kBM; ++j) mtile_x[shared_tiles + offp / kBM + j] = e + 1;
        seg_x[e + 1] = r0 + offp;
    }
    if (e == 0) {
        seg_x[0] = 0;
        seg_x[E + 1] = r0 + total_pad;
        meta[3] = shared_tiles + total_pad / kBM;
        meta[4] = r0 + total_pad;
    }
}

// items [0, T*k): routes; items [T*k, T*k + E*128): padding rows (expert j/128, row
// j%128); with shared_rows > 0, items [T*k + E*128, ... + shared_rows): the shared
// expert's rows, which sit before the routed segments at rows -shared_rows + t
// (token t for t < T, a zero row after it). With x_q set, the copied row is also quantised to MXFP8 along H (the routed
// gate/up GEMM's operand): E4M3 codes to x_q, scales to x_sf in the MMA's
// scale-factor layout.
// QUANT: x_q / x_sf are set (MXFP8 routed weights); a build of its own, so that the
// bf16-only copy keeps its smaller register footprint and twice the resident warps
template <bool QUANT>
__global__ void __launch_bounds__(32 * kWarpsPerBlock) route_place_kernel(
    const int* __restrict__ ids, const float* __restrict__ pp, const int* __restrict__ rank,
    const int* __restrict__ chunk_base, const int* __restrict__ counts, const int* __restrict__ offs_pad, int T,
    int E, int k, int shared_rows, int copy_shared,
    const uint4* __restrict__ hidden, int vec_per_row, int* __restrict__ perm_src, float* __restrict__ pp_perm,
    int* __restrict__ row_of, uint4* __restrict__ x_perm, uint8_t* __restrict__ x_q, uint8_t* __restrict__ x_sf) {
    pdl_wait();
    pdl_trigger();
    const int64_t item = int64_t(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int64_t n_routes = int64_t(T) * k;
    if (item < n_routes) {
        const int e = __ldg(ids + item);
        if (e < 0) return;
        const int t = int(item / k);
        const int pos = __ldg(offs_pad + e) + __ldg(rank + item) +
                        (chunk_base ? __ldg(chunk_base + int64_t(t / kRankChunk) * E + e) : 0);
        if (lane == 0) {
            perm_src[pos] = t;
            pp_perm[pos] = __ldg(pp + item);
            row_of[item] = pos;
        }
        const uint4* src = hidden + int64_t(t) * vec_per_row;
        uint4* dst = x_perm + int64_t(pos) * vec_per_row;
        if constexpr (QUANT)
            copy_quant_row(src, dst, x_q, x_sf, pos, vec_per_row);
        else
            copy_row(src, dst, vec_per_row);
        return;
    }
    const int64_t j = item - n_routes;
    if (j >= int64_t(E) * kBM) {
        const int t = int(j - int64_t(E) * kBM);
        if (t >= shared_rows) return;
        const int64_t pos = int64_t(t) - shared_rows;
        const bool tok = t < T;
        if (lane == 0) {
            perm_src[pos] = tok ? t : -1;
            pp_perm[pos] = tok ? 1.0f : 0.0f;  // the shared output gate, when there is one, overwrites it
        }
        if (!copy_shared) return;  // the GEMMs read the shared rows from hidden itself
        copy_row(tok ? hidden + int64_t(t) * vec_per_row : nullptr, x_perm + pos * vec_per_row, vec_per_row);
        return;
    }
    const int e = int(j / kBM);
    const int r = int(j % kBM);
    const int cnt = __ldg(counts + e);
    const int pad = (cnt + kBM - 1) / kBM * kBM - cnt;
    if (r >= pad) return;
    const int pos = __ldg(offs_pad + e) + cnt + r;
    if (lane == 0) {
        perm_src[pos] = -1;
        pp_perm[pos] = 0.0f;
    }
    if (r >= (cnt + kBK - 1) / kBK * kBK - cnt) return;  // past the last 64-row block with a route
    uint4* dst = x_perm + int64_t(pos) * vec_per_row;
    if constexpr (QUANT)
        copy_quant_row(nullptr, dst, x_q, x_sf, pos, vec_per_row);
    else
        copy_row(nullptr, dst, vec_per_row);
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

int route_rank_max_tokens() { return kRankThreads * 64; }

cudaError_t launch_route_pack(const uint8_t* map, const float* probs, int T, int E, int k, int* ids, float* pp,
                              int* row_of, int* status, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    route_pack_kernel<<<(T + kWarpsPerBlock - 1) / kWarpsPerBlock, 32 * kWarpsPerBlock, 0, st>>>(
        map, probs, T, E, k, ids, pp, row_of, status);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_route_rank(const uint8_t* map, const int* ids, int T, int E, int k, int* rank, int* counts,
                              cudaStream_t st) {
    route_rank_kernel<<<E, kRankThreads, 0, st>>>(map, ids, T, E, k, rank, counts);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_route_pack_rank(const uint8_t* map, const float* probs, const int* topk_ids,
                                   const float* topk_probs, int T, int E, int k, int* ids, float* pp, int* row_of,
                                   int* rank, int* hist, int* status, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const size_t smem = pack_rank_smem(E, k);
    static size_t smem_set = 48 * 1024;
    if (smem > smem_set) {
        const cudaError_t e = cudaFuncSetAttribute(route_pack_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   int(pack_rank_smem(1024, 32)));
        if (e != cudaSuccess) return e;
        smem_set = pack_rank_smem(1024, 32);
    }
    // 4: 16-byte loads (E % 16 == 0, 16-byte aligned map); 1: 4-byte loads; 0: bytes
    const uintptr_t mp = reinterpret_cast<uintptr_t>(map);
    const int words = (E % 16 == 0 && (mp & 15) == 0) ? 4 : ((E % 4 == 0 && (mp & 3) == 0) ? 1 : 0);
    const cudaError_t e = launch_pdl(route_pack_rank_kernel, dim3((T + kRankChunk - 1) / kRankChunk),
                                     dim3(kRankChunk), smem, st, map, probs, T, E, k, ids, pp, row_of, rank, hist,
                                     words, status, topk_ids, topk_probs);
    count_launch();
    return e;
}

cudaError_t launch_route_scan_chunks(int* hist, int T, int E, int* counts, int* offsets, int* offs_pad,
                                     int* mtile_expert, int* meta, int shared_tiles, int* mtile_x, int* seg_x,
                                     cudaStream_t st) {
    const int threads = (E + 31) / 32 * 32;
    const cudaError_t e = launch_pdl(route_scan_chunks_kernel, dim3(1), dim3(threads), 0, st, hist,
                                     (T + kRankChunk - 1) / kRankChunk, E, counts, offsets, offs_pad, mtile_expert,
                                     meta, shared_tiles, mtile_x, seg_x);
    count_launch();
    return e;
}


cudaError_t launch_route_place(const int* ids, const float* pp, const int* rank, const int* chunk_base,
                               const int* counts, const int* offs_pad, int T, int E, int k, int shared_rows,
                               bool copy_shared, const __nv_bfloat16* hidden, int H, int* perm_src, float* pp_perm,
                               int* row_of, __nv_bfloat16* x_perm, uint8_t* x_q, uint8_t* x_sf, cudaStream_t st) {
    const int64_t items = int64_t(T) * k + int64_t(E) * kBM + shared_rows;
    const int64_t blocks = (items + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const cudaError_t e = launch_pdl(x_q ? route_place_kernel<true> : route_place_kernel<false>, dim3(unsigned(blocks)),
                                     dim3(32 * kWarpsPerBlock), 0, st,
                                     ids, pp, rank, chunk_base, counts, offs_pad, T, E, k, shared_rows,
                                     copy_shared ? 1 : 0, reinterpret_cast<const uint4*>(hidden), H / 8, perm_src,
                                     pp_perm, row_of, reinterpret_cast<uint4*>(x_perm), x_q, x_sf);
    count_launch();
    return e;
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

// ======================================================================
// Routing without any device allocation (moe_route_noalloc).
//
// Its only scratch -- the rank of every route inside its expert -- is this
// file-scope device array, which every GPU that loads the library holds until
// the process exits. Every call shares it; nothing in it has to start at zero
// (each call writes the rank of every route it later reads), and calls whose
// kernels overlap on the GPU race on it.
// ======================================================================
namespace moe {
namespace {

constexpr int64_t kNoAllocMaxRoutes = int64_t(1) << 17;  // T * k, 512 KB of int32
static __device__ __align__(256) int g_noalloc_rank[kNoAllocMaxRoutes];

// device address of the scratch array on the current device, resolved on every
// call (cheap once the library's device code is loaded on the device, and never
// stale after a device reset or a new primary context)
int* noalloc_scratch() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_rank) != cudaSuccess || !p) return nullptr;
    return static_cast<int*>(p);
}

__global__ void __launch_bounds__(1024) route_scan_compact_kernel(const int* __restrict__ counts, int E,
                                                                  int* __restrict__ offsets) {
    __shared__ int s_warp[32];
    const int e = threadIdx.x;
    const int cnt = e < E ? counts[e] : 0;
    int total;
    const int off = block_excl_scan(cnt, s_warp, total);
    if (e < E) offsets[e] = off;
    if (e == 0) offsets[E] = total;
}

__global__ void __launch_bounds__(256) route_place_compact_kernel(const int* __restrict__ ids,
                                                                  const int* __restrict__ rank,
                                                                  const int* __restrict__ offsets, int T, int k,
                                                                  int* __restrict__ perm_src,
                                                                  int* __restrict__ row_of) {
    const int64_t item = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (item >= int64_t(T) * k) return;
    const int e = ids[item];
    if (e < 0) return;  // the pack kernel already wrote row_of = -1
    const int pos = offsets[e] + rank[item];
    perm_src[pos] = int(item / k);
    row_of[item] = pos;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_route_noalloc(int64_t T, int64_t E, int64_t k, const uint8_t* routing_map,
                                        const float* probs, int32_t* ids, float* pp, int32_t* counts,
                                        int32_t* offsets, int32_t* perm_src, int32_t* row_of,
                                        int32_t* routing_error, void* stream) {
    using namespace moe;
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E) return MOE_ERR_INVALID_ARG;
    if (T * k > kNoAllocMaxRoutes || T > route_rank_max_tokens()) return MOE_ERR_UNSUPPORTED;
    if (!counts || !offsets || !routing_error) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!routing_map || !probs || !ids || !pp || !perm_src || !row_of)) return MOE_ERR_INVALID_ARG;
    int* rank = noalloc_scratch();
    if (!rank) return MOE_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(routing_error, 0, sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
    if (T == 0) {
        if (cudaMemsetAsync(counts, 0, E * sizeof(int32_t), st) != cudaSuccess ||
            cudaMemsetAsync(offsets, 0, (E + 1) * sizeof(int32_t), st) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    const int Ti = int(T), Ei = int(E), ki = int(k);
    if (launch_route_pack(routing_map, probs, Ti, Ei, ki, ids, pp, row_of, routing_error, st) != cudaSuccess ||
        launch_route_rank(routing_map, ids, Ti, Ei, ki, rank, counts, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    route_scan_compact_kernel<<<1, (Ei + 31) / 32 * 32, 0, st>>>(counts, Ei, offsets);
    count_launch();
    const int64_t n = T * k;
    route_place_compact_kernel<<<unsigned((n + 255) / 256), 256, 0, st>>>(ids, rank, offsets, Ti, ki, perm_src,
                                                                          row_of);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
