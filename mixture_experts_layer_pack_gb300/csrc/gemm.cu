// Grouped GEMMs of the MoE layer on the 5th-generation tensor cores (sm_103a).
//
// One persistent kernel template serves the five GEMM shapes of the layer
// (expert computation of "feat(moe): add a megakernel backend with MOK
// integration", Summary: routed and shared expert computation; backward per
// "core.transformer.moe.megakernel.mok.runtime", _MoKAutograd.backward):
//
//   OP_FWD_GU   [R,2I] = X_perm[R,H] . W_fc1[e]^T     epilogue g,u -> bf16 (kept), a = silu(g)*u (bf16)
//   OP_FWD_DOWN [R,H]  = a[R,I] . W_down[e]^T          epilogue y -> bf16 (the combine weights it)
//   OP_BWD_DOWN [R,I]  = go_perm[R,H] . W_down[e]      epilogue SwiGLU backward, dprob partials
//   OP_BWD_GU   [R,H]  = [dg|du][R,2I] . W_fc1[e]      epilogue dx -> bf16
//   OP_WGRAD    [M,N] += A[seg,M]^T . B[seg,N]        epilogue fp32 load-add-store of main_grad
//
// Rows of the routed GEMMs are the dispatch permutation, each expert's
// segment padded to a multiple of 128 rows (zero rows), so a 128-row tile
// never straddles two experts; the expert of each tile comes from a device
// table, so nothing is read back to the host.
//
// Block = 10 warps: warp 0 issues TMA loads into a STAGES-deep shared-memory
// ring, warp 1 owns TMEM and issues tcgen05.mma (M=128, N=BN, K=16 steps),
// warps 2..9 drain the double-buffered TMEM accumulator through tcgen05.ld
// (two warps per 32-lane quarter, alternating 32-column chunks) and run the
// fused epilogue while the next tile accumulates. Operands use the 128-byte
// swizzle: K-major tiles are 128 rows x 128 bytes; M/N-major tiles are
// 64-element (128-byte) columns x 64 K-rows, 8 KB apart. The weight-gradient
// epilogue moves main_grad in TMA boxes of 32 x 32 fp32: each box is loaded
// one box ahead into a double buffer, gets the accumulator added in shared
// memory and is stored back (a TMA reduce-add into L2 streams main_grad at
// only ~3/4 of the rate of a plain load and store on this part).
#include "device_common.cuh"
#include "internal.h"

#include <climits>

namespace moe {

namespace {

constexpr uint32_t kSwizzleAtom = 1024;   // 8 rows x 128 bytes
constexpr uint32_t kMnChunkBytes = 8192;  // 64 K-rows x 128 bytes

constexpr uint32_t kStageTileBytes = 32 * 32 * 4;  // fp32 staging box of one epilogue warp (32 rows x 32 cols)
constexpr int kRing = 4;  // weight gradient: depth of the claimed-tile ring
constexpr int kRingInts = 6;  // a ring slot: the tile index, then its decoded mt, nt, e, k_lo, kblocks

// SPLIT: one operand comes as hi + lo bf16 terms (the A operand of the down
// projection and of the dgrad through gate/up; A or B of the weight gradients) and
// its lo tile rides in the same stage (L_BYTES: an A tile, or for the weight
// gradient the larger of A and B), so the other operand's tile crosses L2 once for
// both products
template <int OP, int BN, bool SPLIT = false, bool DEEP = false>
struct Cfg {
    static constexpr uint32_t A_BYTES = kBM * kBK * 2;
    static constexpr uint32_t B_BYTES = BN * kBK * 2;
    // (DEEP weight gradient: the A operand is the split one, its lo tile an A tile)
    static constexpr uint32_t L_BYTES = SPLIT ? ((OP == OP_WGRAD && B_BYTES > A_BYTES && !DEEP) ? B_BYTES : A_BYTES) : 0;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES + L_BYTES;
    // the weight-gradient epilogue double-buffers its main_grad boxes, so it
    // gives up operand stages (its K per tile is one expert's short segment); the
    // SwiGLU-backward epilogue (dgrad-down) moves more bytes than its mainloop, and
    // three stages leave it more of the memory system than four (measured)
    // A DEEP weight gradient (long K per tile: the mainloop, not the main_grad stream, is the
    // bound) gives the epilogue one box buffer per warp and the operands a third stage.
    static constexpr int BUFS = (OP == OP_WGRAD) ? (DEEP ? 1 : 2) : 1;
    static constexpr int STAGES =
        (OP == OP_WGRAD) ? (SPLIT ? ((BN == 256) ? (DEEP ? 3 : 2) : 3) : ((BN == 256) ? 3 : (BN == 128 ? 5 : 6)))
                         : (SPLIT ? ((BN == 256) ? 3 : 4)
                                  : ((BN == 256) ? (OP == OP_BWD_DOWN && !DEEP ? 3 : 4) : (BN == 128 ? 6 : 8)));
    static constexpr uint32_t TMEM_COLS = 2 * BN;  // two accumulators; 128/256/512 are legal sizes
    static constexpr uint32_t STAGING = kEpiWarps * BUFS * kStageTileBytes;
    static constexpr size_t SMEM = size_t(STAGES) * STAGE_BYTES + STAGING + 1024 + 512;
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

// tcgen05 shared-memory matrix descriptor, 128-byte swizzle
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= uint64_t((addr >> 4) & 0x3FFF);
    d |= uint64_t((lbo >> 4) & 0x3FFF) << 16;
    d |= uint64_t((sbo >> 4) & 0x3FFF) << 32;
    d |= 1ull << 46;  // descriptor version for tcgen05
    d |= 2ull << 61;  // SWIZZLE_128B
    return d;
}

// instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, M = 128
template <int BN, bool A_MN, bool B_MN>
__host__ __device__ constexpr uint32_t instr_desc() {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((A_MN ? 1u : 0u) << 15) | ((B_MN ? 1u : 0u) << 16) |
           (uint32_t(BN >> 3) << 17) | (uint32_t(kBM >> 4) << 24);
}

struct Tile {
    int mt, nt, e, k_lo, kblocks;
};

template <int OP>
__device__ __forceinline__ Tile decode_tile(int tile, const GemmArgs& a) {
    Tile t;
    if (OP == OP_WGRAD) {
        const int per = a.m_tiles * a.n_tiles;
        t.e = tile / per;
        const int r = tile - t.e * per;
        t.mt = r / a.n_tiles;
        t.nt = r - t.mt * a.n_tiles;
        const int lo = a.seg_off ? a.seg_off[t.e] : 0;
        const int hi = a.seg_off ? a.seg_off[t.e + 1] : a.seg_len;
        int len = hi - lo;
        if (a.seg_off && a.seg_rows) {
            const int valid = (a.group0_shared && t.e == 0) ? a.g0_rows : a.seg_rows[t.e - a.group0_shared];
            len = min(len, valid);
        }
        t.k_lo = lo;
        t.kblocks = (len + kBK - 1) / kBK;
    } else {
        t.mt = tile / a.n_tiles;
        t.nt = tile - t.mt * a.n_tiles;
        t.e = a.mtile_expert ? a.mtile_expert[t.mt] : 0;
        t.k_lo = 0;
        t.kblocks = a.k_blocks;
    }
    return t;
}

// block-scaled GEMM tile `tile` when a CTA tile is NH adjacent 128-column tiles:
// its m tile, expert, and its first 128-column tile (nt in units of 128 columns)
template <int NH>
__device__ __forceinline__ Tile decode_mx_tile(int tile, const GemmArgs& a) {
    const int pairs = a.n_tiles / NH;
    Tile t;
    t.mt = tile / pairs;
    t.nt = (tile - t.mt * pairs) * NH;
    t.e = a.mtile_expert ? a.mtile_expert[t.mt] : 0;
    t.k_lo = 0;
    t.kblocks = a.k_blocks;
    return t;
}

// bounded wait that ignores the abort flag (used while winding down)
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, int* status) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
    return true;
}

// sl: the stage's lo tile of the split operand (SPLIT builds; a.split 1: A, 2: B)
// mG: group 0's token rows (a.g0_operand 1: in place of A, 2: of B), at the same
// row coordinates (group 0's rows are tokens 0 .. T-1, then zero rows)
template <int OP, int BN, bool SPLIT>
__device__ __forceinline__ void issue_loads(const Tile& t, int kb, uint8_t* sa, uint8_t* sb, uint8_t* sl,
                                            const CUtensorMap* mA, const CUtensorMap* mB0, const CUtensorMap* mB1,
                                            const CUtensorMap* mS0, const CUtensorMap* mS1, const CUtensorMap* mL,
                                            const CUtensorMap* mG, uint64_t* bar, const GemmArgs& a) {
    const bool g0 = a.g0_operand && a.group0_shared && t.e == 0;
    if (g0 && a.g0_operand == 1) mA = mG;
    if (OP == OP_WGRAD) {
        if (g0 && a.g0_operand == 2) mB0 = mG;
        const int krow = t.k_lo + kb * kBK;
#pragma unroll
        for (int c = 0; c < kBM / 64; ++c) tma_load_2d(sa + c * kMnChunkBytes, mA, bar, t.mt * kBM + 64 * c, krow);
#pragma unroll
        for (int c = 0; c < BN / 64; ++c) tma_load_2d(sb + c * kMnChunkBytes, mB0, bar, t.nt * BN + 64 * c, krow);
        if (SPLIT) {
            if (a.split == 2) {
#pragma unroll
                for (int c = 0; c < BN / 64; ++c)
                    tma_load_2d(sl + c * kMnChunkBytes, mL, bar, t.nt * BN + 64 * c, krow);
            } else {
#pragma unroll
                for (int c = 0; c < kBM / 64; ++c)
                    tma_load_2d(sl + c * kMnChunkBytes, mL, bar, t.mt * kBM + 64 * c, krow);
            }
        }
        return;
    }
    const int k0 = kb * kBK;
    tma_load_2d(sa, mA, bar, k0, t.mt * kBM);
    if (SPLIT) tma_load_2d(sl, mL, bar, k0, t.mt * kBM);
    // an expert's weights: group 0's own maps when it is the shared expert, else
    // routed expert re's descriptor (z = 0) from a per-expert table or the 3D map at z = re
    const bool sh = a.group0_shared && t.e == 0;
    const int re = t.e - a.group0_shared;
    const CUtensorMap* B0 = sh ? mS0 : (a.b0_tab ? a.b0_tab + re : mB0);
    const CUtensorMap* B1 = sh ? mS1 : (a.b1_tab ? a.b1_tab + re : mB1);
    const int z0 = (sh || a.b0_tab) ? 0 : re;
    const int z1 = (sh || a.b1_tab) ? 0 : re;
    if (OP == OP_FWD_GU) {
        const int j0 = t.nt * (BN / 2);
        tma_load_3d(sb, B0, bar, k0, j0, z0);
        tma_load_3d(sb + (BN / 2) * 128, B1, bar, k0, j0, z1);
    } else if (OP == OP_FWD_DOWN) {
        tma_load_3d(sb, B0, bar, k0, t.nt * BN, z0);
    } else if (OP == OP_BWD_DOWN) {
#pragma unroll
        for (int c = 0; c < BN / 64; ++c) tma_load_3d(sb + c * kMnChunkBytes, B0, bar, t.nt * BN + 64 * c, k0, z0);
    } else {  // OP_BWD_GU: K rows [0,I) come from the gate view, [I,2I) from the up view
        const bool up = k0 >= a.gate_up_split;
        const CUtensorMap* m = up ? B1 : B0;
        const int z = up ? z1 : z0;
        const int kk = up ? k0 - a.gate_up_split : k0;
#pragma unroll
        for (int c = 0; c < BN / 64; ++c) tma_load_3d(sb + c * kMnChunkBytes, m, bar, t.nt * BN + 64 * c, kk, z);
    }
}

// Writes a warp's 32x32 fp32 chunk (lane = row) into its 4 KB staging buffer,
// 128-byte swizzled (16-byte unit j of row r at j ^ (r % 8)): conflict-free
// both for this write and for the transposed read below, and the layout a TMA
// box with 128-byte swizzle expects.
__device__ __forceinline__ void stage_chunk(float* staging, const float (&v)[32]) {
    const int lane = threadIdx.x & 31;
    float4* srow = reinterpret_cast<float4*>(staging + lane * 32);
#pragma unroll
    for (int j = 0; j < 8; ++j) srow[j ^ (lane & 7)] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    __syncwarp();
}

// step i of the transposed read: row i*4 + lane/8, columns 4*(lane%8) .. +3
__device__ __forceinline__ float4 staged(const float* staging, int i) {
    const int lane = threadIdx.x & 31;
    const int r = i * 4 + (lane >> 3);
    return reinterpret_cast<const float4*>(staging + r * 32)[(lane & 7) ^ (r & 7)];
}

// Quantises the 32-column block that 8 consecutive lanes hold (4 columns each,
// same row) to MXFP8: returns the E4M3 codes of this lane's 4 values and the
// block's E8M0 code (the block amax is reduced over the 8 lanes).
__device__ __forceinline__ uint32_t mx_quant_lane4(const float (&v)[4], uint32_t& code) {
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    code = e8m0_code(amax);
    const float mul = e8m0_inv_scale(code);
    return e4m3x4(v[0] * mul, v[1] * mul, v[2] * mul, v[3] * mul);
}

// Stores 4 consecutive values as bf16 hi = bf16(v) and, where lo is given,
// lo = bf16(v - hi) (v - hi is exact in fp32): hi + lo carries 16 significant bits
__device__ __forceinline__ void store_split4(__nv_bfloat16* hi, __nv_bfloat16* lo, const float (&v)[4]) {
    const uint32_t h0 = pack_bf16x2(v[0], v[1]), h1 = pack_bf16x2(v[2], v[3]);
    *reinterpret_cast<uint2*>(hi) = make_uint2(h0, h1);
    if (lo) {
        float r[4];
        unpack_bf16x2(h0, r[0], r[1]);
        unpack_bf16x2(h1, r[2], r[3]);
        *reinterpret_cast<uint2*>(lo) =
            make_uint2(pack_bf16x2(v[0] - r[0], v[1] - r[1]), pack_bf16x2(v[2] - r[2], v[3] - r[3]));
    }
}

template <int OP, int BN, bool MX = false, bool CLAMP = false>
__device__ __forceinline__ void epilogue_tile(const Tile& t, uint32_t t_row, int q, int half, const GemmArgs& a,
                                              float* staging) {
    const int lane = threadIdx.x & 31;
    // The warp owns rows [m_base, m_base+32) of the tile. Each 32x32 fp32 chunk
    // read from TMEM (lane = row) is transposed through the warp's staging
    // buffer so that global loads and stores cover whole row segments: in step
    // i a lane holds row i*4 + lane/8, columns 4*(lane%8) .. +3.
    const int m_base = t.mt * kBM + q * 32;
    const int sub_row = lane >> 3;
    const int sub_col = 4 * (lane & 7);
    // rows a later kernel reads: below rows_valid and, with group row counts, below the end
    // of the tile's group's last 64-row block that holds a valid row
    int row_lim = a.rows_valid;
    if (a.seg_off && a.seg_rows) {
        const int valid = (a.group0_shared && t.e == 0) ? a.g0_rows : a.seg_rows[t.e - a.group0_shared];
        row_lim = min(row_lim, a.seg_off[t.e] + (valid + kBK - 1) / kBK * kBK);
    }
    const bool lane_row_valid = m_base + lane < row_lim;

    if (OP == OP_FWD_GU) {
        const int j0 = t.nt * (BN / 2);
#pragma unroll 1
        for (int c = half; c < BN / 64; c += kEpiHalves) {
            float g[32], u[32];
            tmem_ld32(t_row + c * 32, g);
            tmem_ld32(t_row + BN / 2 + c * 32, u);
            float4 gv[8], uv[8];
            stage_chunk(staging, g);
#pragma unroll
            for (int i = 0; i < 8; ++i) gv[i] = staged(staging, i);
            __syncwarp();
            stage_chunk(staging, u);
#pragma unroll
            for (int i = 0; i < 8; ++i) uv[i] = staged(staging, i);
            __syncwarp();
            const int col = j0 + c * 32 + sub_col;
            if (a.outf) {
                // fp32 activations: g, u are kept as accumulated, a is computed from them
                // and leaves as two bf16 terms (the down projection's split operand)
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int row = m_base + i * 4 + sub_row;
                    const float4 g4 = gv[i], u4 = uv[i];
                    float gc[4] = {g4.x, g4.y, g4.z, g4.w}, uc[4] = {u4.x, u4.y, u4.z, u4.w};
                    if (CLAMP) {
#pragma unroll
                        for (int z = 0; z < 4; ++z) {
                            gc[z] = fminf(gc[z], a.swiglu_limit);
                            uc[z] = fminf(fmaxf(uc[z], -a.swiglu_limit), a.swiglu_limit);
                        }
                    }
                    float av[4];
#pragma unroll
                    for (int z = 0; z < 4; ++z) av[z] = gc[z] * sigmoidf_(gc[z]) * uc[z];
                    if (MX) {  // the routed down projection's operand: a quantised along I
                        uint32_t code;
                        const uint32_t qv = mx_quant_lane4(av, code);
                        if (row < row_lim) {
                            *reinterpret_cast<uint32_t*>(a.q_out + int64_t(row) * a.ld_q + col) = qv;
                            if ((lane & 7) == 0) a.q_sf[sf_atom_offset(row, col >> 5, a.q_kblocks)] = uint8_t(code);
                        }
                    }
                    if (row >= row_lim) continue;
                    float* gu = a.outf + int64_t(row) * a.ld_outf;
                    *reinterpret_cast<float4*>(gu + col) = g4;
                    *reinterpret_cast<float4*>(gu + a.inter + col) = u4;
                    if (a.out0) store_split4(a.out0 + int64_t(row) * a.ld_out0 + col,
                                             a.out0lo ? a.out0lo + int64_t(row) * a.ld_out0lo + col : nullptr, av);
                }
                continue;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int row = m_base + i * 4 + sub_row;
                const float4 g4 = gv[i], u4 = uv[i];
                // g, u are passed on in bf16; a is computed from those values
                const uint2 gb = make_uint2(pack_bf16x2(g4.x, g4.y), pack_bf16x2(g4.z, g4.w));
                const uint2 ub = make_uint2(pack_bf16x2(u4.x, u4.y), pack_bf16x2(u4.z, u4.w));
                float gc[4], uc[4];
                unpack_bf16x2(gb.x, gc[0], gc[1]);
                unpack_bf16x2(gb.y, gc[2], gc[3]);
                unpack_bf16x2(ub.x, uc[0], uc[1]);
                unpack_bf16x2(ub.y, uc[2], uc[3]);
                if (CLAMP) {  // clamped SwiGLU inputs; g, u are saved unclamped
#pragma unroll
                    for (int z = 0; z < 4; ++z) {
                        gc[z] = fminf(gc[z], a.swiglu_limit);
                        uc[z] = fminf(fmaxf(uc[z], -a.swiglu_limit), a.swiglu_limit);
                    }
                }
                float av[4];
#pragma unroll
                for (int z = 0; z < 4; ++z) av[z] = gc[z] * sigmoidf_(gc[z]) * uc[z];
                if (MX) {
                    // the down projection's operand: a quantised along I (this chunk is one
                    // 32-column block); a itself becomes its exact dequantised value
                    uint32_t code;
                    const uint32_t qv = mx_quant_lane4(av, code);
                    if (row < row_lim) {
                        *reinterpret_cast<uint32_t*>(a.q_out + int64_t(row) * a.ld_q + col) = qv;
                        if ((lane & 7) == 0) a.q_sf[sf_atom_offset(row, col >> 5, a.q_kblocks)] = uint8_t(code);
                    }
                    const float sc = e8m0_scale(code);
#pragma unroll
                    for (int z = 0; z < 4; ++z) av[z] = e4m3_value(qv >> (8 * z)) * sc;
                }
                if (row >= row_lim) continue;
                *reinterpret_cast<uint2*>(a.out0 + int64_t(row) * a.ld_out0 + col) =
                    make_uint2(pack_bf16x2(av[0], av[1]), pack_bf16x2(av[2], av[3]));
                __nv_bfloat16* gu = a.outh + int64_t(row) * a.ld_outh;
                *reinterpret_cast<uint2*>(gu + col) = gb;
                *reinterpret_cast<uint2*>(gu + a.inter + col) = ub;
            }
        }
    } else if (OP == OP_FWD_DOWN || OP == OP_BWD_GU) {
#pragma unroll 1
        for (int c = half; c < BN / 32; c += kEpiHalves) {
            float v[32];
            tmem_ld32(t_row + c * 32, v);
            stage_chunk(staging, v);
            const int col = t.nt * BN + c * 32 + sub_col;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 x = staged(staging, i);
                const int row = m_base + i * 4 + sub_row;
                if (row >= row_lim) continue;
                if (a.outf)
                    *reinterpret_cast<float4*>(a.outf + int64_t(row) * a.ld_outf + col) = x;
                else
                    *reinterpret_cast<uint2*>(a.outh + int64_t(row) * a.ld_outh + col) =
                        make_uint2(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w));
            }
            __syncwarp();
        }
    } else {  // OP_BWD_DOWN: acc = da_u = go . W_down[e] for columns i of the tile
        const float lane_p = (a.row_scale && lane_row_valid) ? a.row_scale[m_base + lane] : 1.0f;
        float part[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) part[i] = 0.0f;
#pragma unroll 1
        for (int c = half; c < BN / 32; c += kEpiHalves) {
            float d[32];
            tmem_ld32(t_row + c * 32, d);
            stage_chunk(staging, d);
            const int col = t.nt * BN + c * 32 + sub_col;
            if (a.inf) {
                // fp32 activations: g, u load in fp32 and a is recomputed from them (the
                // value the forward's down projection took as hi + lo terms); the dprob
                // partial, p * a and the SwiGLU gradients come from these fp32 values, and
                // [dg|du] and p * a leave as hi + lo bf16 terms
                float4 gq[8], uq[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int row = m_base + i * 4 + sub_row;
                    if (row < row_lim) {
                        const float* gu = a.inf + int64_t(row) * a.ld_inf;
                        gq[i] = __ldg(reinterpret_cast<const float4*>(gu + col));
                        uq[i] = __ldg(reinterpret_cast<const float4*>(gu + a.inter + col));
                    } else {
                        gq[i] = uq[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r_local = i * 4 + sub_row;
                    const float p = __shfl_sync(0xffffffffu, lane_p, r_local);
                    const float4 d4 = staged(staging, i);
                    const int row = m_base + r_local;
                    const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
                    const float gv[4] = {gq[i].x, gq[i].y, gq[i].z, gq[i].w};
                    const float uv[4] = {uq[i].x, uq[i].y, uq[i].z, uq[i].w};
                    float dg[4], du[4], ap[4];
#pragma unroll
                    for (int z = 0; z < 4; ++z) {
                        float g = gv[z], u = uv[z], mg = 1.0f, mu = 1.0f;
                        if (CLAMP) {
                            const float L = a.swiglu_limit;
                            mg = g <= L ? 1.0f : 0.0f;
                            mu = (u >= -L && u <= L) ? 1.0f : 0.0f;
                            g = fminf(g, L);
                            u = fminf(fmaxf(u, -L), L);
                        }
                        const float sg = sigmoidf_(g);
                        const float av = g * sg * u;
                        part[i] = fmaf(av, dv[z], part[i]);
                        const float da = p * dv[z];
                        dg[z] = da * u * (sg * (1.0f + g * (1.0f - sg))) * mg;
                        du[z] = da * (g * sg) * mu;
                        ap[z] = p * av;
                    }
                    if (MX) {
                        uint32_t cg, cu;
                        const uint32_t qg = mx_quant_lane4(dg, cg);
                        const uint32_t qu = mx_quant_lane4(du, cu);
                        if (row < row_lim) {
                            uint8_t* qo = a.q_out + int64_t(row) * a.ld_q;
                            *reinterpret_cast<uint32_t*>(qo + col) = qg;
                            *reinterpret_cast<uint32_t*>(qo + a.inter + col) = qu;
                            if ((lane & 7) == 0) {
                                a.q_sf[sf_atom_offset(row, col >> 5, a.q_kblocks)] = uint8_t(cg);
                                a.q_sf[sf_atom_offset(row, (a.inter + col) >> 5, a.q_kblocks)] = uint8_t(cu);
                            }
                        }
                    }
                    if (row >= row_lim) continue;
                    const int64_t o = int64_t(row) * a.ld_out0 + col;
                    const int64_t ol = int64_t(row) * a.ld_out0lo + col;
                    store_split4(a.out0 + o, a.out0lo ? a.out0lo + ol : nullptr, dg);
                    store_split4(a.out0 + o + a.inter, a.out0lo ? a.out0lo + ol + a.inter : nullptr, du);
                    if (a.out1)
                        store_split4(a.out1 + int64_t(row) * a.ld_out1 + col,
                                     a.out1lo ? a.out1lo + int64_t(row) * a.ld_out1lo + col : nullptr, ap);
                }
                __syncwarp();
                continue;
            }
            // load phase: every input of the chunk is requested before any result
            // is stored, so the eight row steps share one memory latency
            uint2 aw[8], gw[8], uw[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int row = m_base + i * 4 + sub_row;
                if (row < row_lim) {
                    aw[i] = __ldg(reinterpret_cast<const uint2*>(a.in0 + int64_t(row) * a.ld_in0 + col));
                    const __nv_bfloat16* gu = a.inh + int64_t(row) * a.ld_inh;
                    gw[i] = __ldg(reinterpret_cast<const uint2*>(gu + col));
                    uw[i] = __ldg(reinterpret_cast<const uint2*>(gu + a.inter + col));
                } else {
                    aw[i] = gw[i] = uw[i] = make_uint2(0, 0);
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r_local = i * 4 + sub_row;
                const float p = __shfl_sync(0xffffffffu, lane_p, r_local);
                const float4 d4 = staged(staging, i);
                const int row = m_base + r_local;
                float av[4];
                unpack_bf16x2(aw[i].x, av[0], av[1]);
                unpack_bf16x2(aw[i].y, av[2], av[3]);
                const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
                float gv[4], uv[4];
                unpack_bf16x2(gw[i].x, gv[0], gv[1]);
                unpack_bf16x2(gw[i].y, gv[2], gv[3]);
                unpack_bf16x2(uw[i].x, uv[0], uv[1]);
                unpack_bf16x2(uw[i].y, uv[2], uv[3]);
                float dg[4], du[4], ap[4];
#pragma unroll
                for (int z = 0; z < 4; ++z) {
                    part[i] = fmaf(av[z], dv[z], part[i]);
                    float g = gv[z], u = uv[z], mg = 1.0f, mu = 1.0f;
                    if (CLAMP) {  // gradients pass only where the clamp is inactive
                        const float L = a.swiglu_limit;
                        mg = g <= L ? 1.0f : 0.0f;
                        mu = (u >= -L && u <= L) ? 1.0f : 0.0f;
                        g = fminf(g, L);
                        u = fminf(fmaxf(u, -L), L);
                    }
                    const float sg = sigmoidf_(g);
                    const float da = p * dv[z];
                    dg[z] = da * u * (sg * (1.0f + g * (1.0f - sg))) * mg;
                    du[z] = da * (g * sg) * mu;
                    ap[z] = p * av[z];
                }
                if (MX) {
                    // the gate/up dgrad operand [dg|du] quantised along 2I (32-column blocks)
                    uint32_t cg, cu;
                    const uint32_t qg = mx_quant_lane4(dg, cg);
                    const uint32_t qu = mx_quant_lane4(du, cu);
                    if (row < row_lim) {
                        uint8_t* qo = a.q_out + int64_t(row) * a.ld_q;
                        *reinterpret_cast<uint32_t*>(qo + col) = qg;
                        *reinterpret_cast<uint32_t*>(qo + a.inter + col) = qu;
                        if ((lane & 7) == 0) {
                            a.q_sf[sf_atom_offset(row, col >> 5, a.q_kblocks)] = uint8_t(cg);
                            a.q_sf[sf_atom_offset(row, (a.inter + col) >> 5, a.q_kblocks)] = uint8_t(cu);
                        }
                    }
                }
                if (row >= row_lim) continue;
                __nv_bfloat16* o = a.out0 + int64_t(row) * a.ld_out0;
                *reinterpret_cast<uint2*>(o + col) = make_uint2(pack_bf16x2(dg[0], dg[1]), pack_bf16x2(dg[2], dg[3]));
                *reinterpret_cast<uint2*>(o + a.inter + col) =
                    make_uint2(pack_bf16x2(du[0], du[1]), pack_bf16x2(du[2], du[3]));
                if (a.out1)
                    *reinterpret_cast<uint2*>(a.out1 + int64_t(row) * a.ld_out1 + col) =
                        make_uint2(pack_bf16x2(ap[0], ap[1]), pack_bf16x2(ap[2], ap[3]));
            }
            __syncwarp();
        }
        // the 8 lanes holding one row's columns add up their partial dot products
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float v = part[i];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            const int row = m_base + i * 4 + sub_row;
            if ((lane & 7) == 0 && row < row_lim && a.partial)
                a.partial[(int64_t(row) * a.n_tiles + t.nt) * kEpiHalves + half] = v;
        }
    }
}

// Weight-gradient epilogue of one warp: main_grad[e][m][n] += acc for its
// 32-row quarter of every tile and its share of the tile's boxes (fp32
// main_grad: 32 x 32 boxes, bf16: 32 rows x 64 columns -- 4 KB and 128-byte
// rows either way; the two warps of a quarter take alternate boxes). Each box
// is TMA-loaded into one of two 4 KB buffers one box ahead (the next tile's
// first box is fetched while this tile's last box is added), the accumulator
// columns read from TMEM (lane = row) are added in shared memory, and the box
// is TMA-stored back: one add per element, so the result is
// fl32(main_grad + dW), or bf16(main_grad + bf16(dW)) for bf16 main_grad,
// whatever the schedule.
template <int BN, int BUFS>
__device__ __forceinline__ void wgrad_epilogue(const GemmArgs& args, uint32_t tmem_base, int q, int half,
                                               float* bufs, uint64_t* mg_bar, uint64_t* tfull, uint64_t* tempty,
                                               const uint64_t* ring_full, uint64_t* ring_empty,
                                               const int* ring_tile, volatile int* abort_flag,
                                               const CUtensorMap* mC0, const CUtensorMap* mC1,
                                               const CUtensorMap* mS0, const CUtensorMap* mS1) {
    const int lane = threadIdx.x & 31;
    const bool bf = args.mg_bf16 != 0;
    const int bw = bf ? 64 : 32;                           // box width in elements
    const int nb = (BN / bw - half + kEpiHalves - 1) / kEpiHalves;  // boxes of this warp per tile
    // tile at ring position pos (-1: no more tiles, -2: the wait gave up) and its
    // decoded coordinates, as the producer published them; the position is released
    // to the producer as soon as it has been read
    auto ring_take = [&](int pos, Tile& tt) -> int {
        int v[kRingInts] = {-2, 0, 0, 0, 0, 0};
        if (lane == 0) {
            const int slot = pos % kRing;
            if (mbar_wait(const_cast<uint64_t*>(&ring_full[slot]), (pos / kRing) & 1, abort_flag, args.status)) {
#pragma unroll
                for (int j = 0; j < kRingInts; ++j) v[j] = ring_tile[slot * kRingInts + j];
                mbar_arrive(&ring_empty[slot]);
            }
        }
#pragma unroll
        for (int j = 0; j < kRingInts; ++j) v[j] = __shfl_sync(0xffffffffu, v[j], 0);
        tt.mt = v[1];
        tt.nt = v[2];
        tt.e = v[3];
        tt.k_lo = v[4];
        tt.kblocks = v[5];
        return v[0];
    };
    // box (tile t, c-th box of this warp): destination map and coordinates (group
    // 0's own maps when it is the shared expert; a routed expert's own descriptor
    // at z = 0 when main_grad comes as a per-expert table, else the 3D map)
    auto box = [&](const Tile& t, int c, const CUtensorMap*& mc, int& x, int& y, int& z) {
        const int m0 = t.mt * kBM + q * 32;
        if (args.mg_trans) {  // main_grad row = accumulator column, main_grad column = accumulator row
            const bool sh = args.group0_shared && t.e == 0;
            const int re = t.e - args.group0_shared;
            mc = sh ? mS0 : (args.c0_tab ? args.c0_tab + re : mC0);
            z = (sh || args.c0_tab) ? 0 : re;
            x = m0;
            y = t.nt * BN + (half + c * kEpiHalves) * bw;
            return;
        }
        const bool hi = m0 >= args.m_split;
        const bool sh = args.group0_shared && t.e == 0;
        const int re = t.e - args.group0_shared;
        const CUtensorMap* tab = hi ? args.c1_tab : args.c0_tab;
        mc = sh ? (hi ? mS1 : mS0) : (tab ? tab + re : (hi ? mC1 : mC0));
        z = (sh || tab) ? 0 : re;
        y = hi ? m0 - args.m_split : m0;
        x = t.nt * BN + (half + c * kEpiHalves) * bw;
    };
    auto load_box = [&](const Tile& t, int c, int b) {
        const CUtensorMap* mc;
        int x, y, z;
        box(t, c, mc, x, y, z);
        mbar_arrive_expect_tx(&mg_bar[b], kStageTileBytes);
        tma_load_3d(bufs + b * (kStageTileBytes / 4), mc, &mg_bar[b], x, y, z);
    };

    // add accumulator column chunk `col` into the box in buffer b (its row `lane`: 128 bytes,
    // 16-byte unit j at j ^ (lane % 8), the 128-byte swizzle)
    auto add_box = [&](const float (&v)[32], const float (&v2)[32], int b) {
        uint4* srow = reinterpret_cast<uint4*>(bufs + b * (kStageTileBytes / 4) + lane * 32);
        if (bf) {
            // bf16(main_grad + bf16(dW)) as one packed rounding of the exact sum of two
            // bf16 values: that sum is exact in fp32 unless their exponents differ by
            // more than 15, and then the smaller lies below half a bf16 ulp of the
            // larger either way, so this equals the fp32 add followed by rounding
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint4 m = srow[j ^ (lane & 7)];
                uint32_t* mw = reinterpret_cast<uint32_t*>(&m);
#pragma unroll
                for (int z = 0; z < 4; ++z) {
                    const int cidx = 8 * (j & 3) + 2 * z;
                    const float d0 = j < 4 ? v[cidx] : v2[cidx];
                    const float d1 = j < 4 ? v[cidx + 1] : v2[cidx + 1];
                    const __nv_bfloat162 sum =
                        __hadd2(*reinterpret_cast<const __nv_bfloat162*>(&mw[z]), __floats2bfloat162_rn(d0, d1));
                    mw[z] = *reinterpret_cast<const uint32_t*>(&sum);
                }
                srow[j ^ (lane & 7)] = m;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float4 m = reinterpret_cast<float4*>(srow)[j ^ (lane & 7)];
                m.x += v[4 * j];
                m.y += v[4 * j + 1];
                m.z += v[4 * j + 2];
                m.w += v[4 * j + 3];
                reinterpret_cast<float4*>(srow)[j ^ (lane & 7)] = m;
            }
        }
    };

    // the transposed add (mg_trans, fp32 main_grad): box row r (a main_grad row) gets
    // accumulator column r of this lane's row, element (r, lane) of the 128-byte-swizzled box
    auto add_box_t = [&](const float (&v)[32], int b) {
        float* base = bufs + b * (kStageTileBytes / 4);
#pragma unroll
        for (int r = 0; r < 32; ++r) base[r * 32 + ((((lane >> 2) ^ (r & 7)) << 2) | (lane & 3))] += v[r];
    };

    if constexpr (BUFS == 1) {
        // one box buffer: load, add, store, one box after the other (the tile's mainloop,
        // long for these tiles, runs meanwhile on the other accumulator)
        int rpos = 0;
        Tile t;
        int cur = ring_take(rpos++, t);
        uint32_t parity = 0;
        int it = 0;
        bool ok = true;
        while (ok && cur >= 0) {
            const int acc = it & 1;
            const uint32_t use = uint32_t(it >> 1);
            ++it;
            int w = 0;
            if (lane == 0) w = mbar_wait(&tfull[acc], use & 1, abort_flag, args.status) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, w, 0)) break;
            __syncwarp();
            tc_fence_after();
            const uint32_t t_row = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(acc * BN);
            Tile tn;
            const int nxt = ring_take(rpos++, tn);
            if (nxt == -2) break;
#pragma unroll 1
            for (int c = 0; c < nb; ++c) {
                if (lane == 0) {
                    bulk_wait_read<0>();  // the previous store has read the buffer out
                    load_box(t, c, 0);
                }
                const uint32_t col = uint32_t((half + c * kEpiHalves) * bw);
                float v[32], v2[32];
                tmem_ld32(t_row + col, v);
                if (bf) tmem_ld32(t_row + col + 32, v2);
                if (lane == 0) w = mbar_wait(&mg_bar[0], parity & 1, abort_flag, args.status) ? 1 : 0;
                if (!__shfl_sync(0xffffffffu, w, 0)) {
                    ok = false;
                    break;
                }
                (void)mbar_try_wait(&mg_bar[0], parity & 1);  // every lane acquires the box
                __syncwarp();
                parity ^= 1u;
                if (args.mg_trans)
                    add_box_t(v, 0);
                else
                    add_box(v, v2, 0);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const CUtensorMap* mc;
                    int x, y, z;
                    box(t, c, mc, x, y, z);
                    tma_store_3d(mc, bufs, x, y, z);
                    bulk_commit();
                }
            }
            if (!ok) {
                // a box load may be in flight: let it land before the buffer is given up
                if (lane == 0) mbar_wait_drain(&mg_bar[0], parity & 1, args.status);
                break;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            cur = nxt;
            t = tn;
        }
        if (lane == 0) bulk_wait<0>();  // every store completes
        __syncwarp();
        return;
    }

    int rpos = 0;
    Tile t;
    int cur = ring_take(rpos++, t);
    uint32_t pending = 0, parity = 0;  // per buffer: a load in flight / parity of its next completion
    if (nb > 0 && cur >= 0 && lane == 0) {
        load_box(t, 0, 0);
        pending = 1;
    }
    int jb = 0, it = 0;
    bool ok = true;
    while (ok && cur >= 0) {
        const int acc = it & 1;
        const uint32_t use = uint32_t(it >> 1);
        ++it;
        int w = 0;
        if (lane == 0) w = mbar_wait(&tfull[acc], use & 1, abort_flag, args.status) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, w, 0)) break;
        __syncwarp();
        tc_fence_after();
        const uint32_t t_row = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(acc * BN);
        // the producer publishes the next tile once this one's loads are issued
        Tile tn;
        const int nxt = ring_take(rpos++, tn);
        if (nxt == -2) break;
#pragma unroll 1
        for (int c = 0; c < nb; ++c) {
            const int b = jb & 1;
            if (lane == 0) {
                // prefetch the box after this one into the other buffer, once the
                // store that last used it has read it out
                const bool more = c + 1 < nb || nxt >= 0;
                if (more) {
                    bulk_wait_read<0>();
                    load_box(c + 1 < nb ? t : tn, c + 1 < nb ? c + 1 : 0, b ^ 1);
                    pending |= 1u << (b ^ 1);
                }
            }
            const uint32_t col = uint32_t((half + c * kEpiHalves) * bw);
            float v[32], v2[32];
            tmem_ld32(t_row + col, v);
            if (bf) tmem_ld32(t_row + col + 32, v2);
            if (lane == 0) w = mbar_wait(&mg_bar[b], (parity >> b) & 1, abort_flag, args.status) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, w, 0)) {
                ok = false;
                break;
            }
            // the phase has completed: every lane's own successful test acquires the box
            (void)mbar_try_wait(&mg_bar[b], (parity >> b) & 1);
            __syncwarp();
            pending &= ~(1u << b);
            parity ^= 1u << b;
            if (args.mg_trans)
                add_box_t(v, b);
            else
                add_box(v, v2, b);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                const CUtensorMap* mc;
                int x, y, z;
                box(t, c, mc, x, y, z);
                tma_store_3d(mc, bufs + b * (kStageTileBytes / 4), x, y, z);
                bulk_commit();
            }
            ++jb;
        }
        if (!ok) break;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        cur = nxt;
        t = tn;
    }
    if (lane == 0) {
        // wind down: loads still in flight land, every store completes
        for (int b = 0; b < 2; ++b)
            if (pending & (1u << b)) mbar_wait_drain(&mg_bar[b], (parity >> b) & 1, args.status);
        bulk_wait<0>();
    }
    __syncwarp();
}

template <int OP, int BN, bool CLAMP, bool SPLIT, bool DEEP>
__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmC0,
                    const __grid_constant__ CUtensorMap tmC1, const __grid_constant__ CUtensorMap tmS0,
                    const __grid_constant__ CUtensorMap tmS1, const __grid_constant__ CUtensorMap tmL,
                    const __grid_constant__ CUtensorMap tmG, const GemmArgs args) {
    using C = Cfg<OP, BN, SPLIT, DEEP>;
    constexpr bool A_MN = (OP == OP_WGRAD);
    constexpr bool B_MN = (OP == OP_BWD_DOWN || OP == OP_BWD_GU || OP == OP_WGRAD);
    constexpr uint32_t IDESC = instr_desc<BN, A_MN, B_MN>();
    constexpr int STAGES = C::STAGES;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* staging = reinterpret_cast<float*>(smem + STAGES * C::STAGE_BYTES);  // 1024-byte aligned
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES + C::STAGING);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint64_t* mg_bar = drain + 1;  // weight gradient: two box buffers per epilogue warp
    // weight gradient: ring of claimed tiles (dynamic scheduling), producer -> MMA and epilogue warps
    uint64_t* ring_full = mg_bar + 2 * kEpiWarps;
    uint64_t* ring_empty = ring_full + kRing;
    int* ring_tile = reinterpret_cast<int*>(ring_empty + kRing);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ring_tile + kRing * kRingInts);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], kEpiWarps);
        }
        mbar_init(drain, 1);
        if (OP == OP_WGRAD) {
            for (int b = 0; b < 2 * kEpiWarps; ++b) mbar_init(&mg_bar[b], 1);
            for (int r = 0; r < kRing; ++r) {
                mbar_init(&ring_full[r], 1);
                mbar_init(&ring_empty[r], 1 + kEpiWarps);  // the MMA thread and every epilogue warp
            }
        }
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB0);
        if (OP == OP_FWD_GU || OP == OP_BWD_GU) tma_prefetch_map(&tmB1);
        if (OP == OP_WGRAD) {
            tma_prefetch_map(&tmC0);
            tma_prefetch_map(&tmC1);
        }
        if (SPLIT) tma_prefetch_map(&tmL);
        if (args.g0_operand) tma_prefetch_map(&tmG);
        if (args.group0_shared) {
            tma_prefetch_map(&tmS0);
            if (OP == OP_FWD_GU || OP == OP_BWD_GU || OP == OP_WGRAD) tma_prefetch_map(&tmS1);
        }
    }
    if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();  // from here on the predecessor's writes are visible (prologue above touched no global memory)
    pdl_trigger();

    int total_tiles;
    if (OP == OP_WGRAD)
        total_tiles = args.groups * args.m_tiles * args.n_tiles;
    else
        total_tiles = (args.num_mtiles_dev ? *args.num_mtiles_dev : args.num_mtiles) * args.n_tiles;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            int stage = 0;
            uint32_t phase = 0;
            uint32_t filled = 0, fill_parity = 0;  // per stage: ever filled / parity of its last fill
            bool ok = true;
            int claimed = 0;  // weight gradient: tiles published into the ring so far
            // weight gradient: the tile claimed for the next turn; its claim (an atomic on
            // the launch's counter) is issued a turn ahead, so its round trip overlaps the
            // current tile's loads
            int ahead = (OP == OP_WGRAD) ? atomicAdd(args.tile_counter, 1) : 0;
            for (int next = blockIdx.x; ok; next += gridDim.x) {
                int tile = next;
                Tile tw{};  // weight gradient: the claimed tile, decoded once here
                if (OP == OP_WGRAD) {
                    // publish the claimed tile with work (-1 once the counter has passed
                    // the last tile), then claim the next one
                    const int slot = claimed % kRing;
                    if (!mbar_wait(&ring_empty[slot], ((claimed / kRing) & 1) ^ 1, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    tile = ahead;
                    Tile tt = decode_tile<OP>(tile < total_tiles ? tile : 0, args);
                    while (tile < total_tiles && tt.kblocks == 0) {
                        tile = atomicAdd(args.tile_counter, 1);
                        tt = decode_tile<OP>(tile < total_tiles ? tile : 0, args);
                    }
                    int* rs = ring_tile + slot * kRingInts;
                    rs[0] = tile < total_tiles ? tile : -1;
                    rs[1] = tt.mt;
                    rs[2] = tt.nt;
                    rs[3] = tt.e;
                    rs[4] = tt.k_lo;
                    rs[5] = tt.kblocks;
                    mbar_arrive(&ring_full[slot]);
                    ++claimed;
                    if (tile < total_tiles) ahead = atomicAdd(args.tile_counter, 1);
                    tw = tt;
                }
                if (tile >= total_tiles) break;
                const Tile t = (OP == OP_WGRAD) ? tw : decode_tile<OP>(tile, args);
                for (int kb = 0; kb < t.kblocks; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + stage * C::STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[stage], C::A_BYTES + C::B_BYTES +
                                                            (SPLIT ? (args.split == 2 ? C::B_BYTES : C::A_BYTES) : 0));
                    issue_loads<OP, BN, SPLIT>(t, kb, sa, sa + C::A_BYTES, sa + C::A_BYTES + C::B_BYTES, &tmA, &tmB0,
                                               &tmB1, &tmS0, &tmS1, &tmL, &tmG, &full[stage], args);
                    filled |= 1u << stage;
                    fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok) {
                // wind down: let every copy this thread issued land before the CTA exits
                for (int s = 0; s < STAGES; ++s)
                    if (filled & (1u << s)) mbar_wait_drain(&full[s], (fill_parity >> s) & 1, args.status);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            int rpos = 0;  // weight gradient: ring positions read so far
            bool ok = true;
            for (int next = blockIdx.x; ok; next += gridDim.x) {
                int tile = next;
                Tile t;
                if (OP == OP_WGRAD) {  // the next claimed tile, in the producer's order, decoded there
                    const int slot = rpos % kRing;
                    if (!mbar_wait(&ring_full[slot], (rpos / kRing) & 1, abort_flag, args.status)) break;
                    const int* rs = ring_tile + slot * kRingInts;
                    tile = rs[0];
                    t.mt = rs[1];
                    t.nt = rs[2];
                    t.e = rs[3];
                    t.k_lo = rs[4];
                    t.kblocks = rs[5];
                    mbar_arrive(&ring_empty[slot]);
                    ++rpos;
                    if (tile < 0) break;
                } else {
                    if (tile >= total_tiles) break;
                    t = decode_tile<OP>(tile, args);
                }
                if (tile >= total_tiles) break;
                if (t.kblocks == 0) continue;
                const int buf = it & 1;
                const uint32_t use = uint32_t(it >> 1);
                ++it;
                if (!mbar_wait(&tempty[buf], (use & 1) ^ 1, abort_flag, args.status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + uint32_t(buf * BN);
                for (int kb = 0; kb < t.kblocks; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint64_t ad = A_MN ? smem_desc(a_addr + kk * 2048, kMnChunkBytes, kSwizzleAtom)
                                                 : smem_desc(a_addr + kk * 32, 16, kSwizzleAtom);
                        const uint64_t bd = B_MN ? smem_desc(b_addr + kk * 2048, kMnChunkBytes, kSwizzleAtom)
                                                 : smem_desc(b_addr + kk * 32, 16, kSwizzleAtom);
                        mma_bf16(d_tmem, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
                    }
                    if (SPLIT) {
                        const uint32_t l_addr = b_addr + C::B_BYTES;
                        const bool lo_b = args.split == 2;
                        const uint32_t a2 = lo_b ? a_addr : l_addr;
                        const uint32_t b2 = lo_b ? l_addr : b_addr;
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk) {
                            const uint64_t ad = A_MN ? smem_desc(a2 + kk * 2048, kMnChunkBytes, kSwizzleAtom)
                                                     : smem_desc(a2 + kk * 32, 16, kSwizzleAtom);
                            const uint64_t bd = B_MN ? smem_desc(b2 + kk * 2048, kMnChunkBytes, kSwizzleAtom)
                                                     : smem_desc(b2 + kk * 32, 16, kSwizzleAtom);
                            mma_bf16(d_tmem, ad, bd, IDESC, 1u);
                        }
                    }
                    mma_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (ok) mma_commit(&tfull[buf]);
            }
            // every MMA issued by this thread completes before TMEM is released
            mma_commit(drain);
            mbar_wait_drain(drain, 0, args.status);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue warps 2..: TMEM lane quarter = warp % 4, column half = (warp - 2) / 4
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        float* my_staging = staging + (warp - 2) * C::BUFS * (kStageTileBytes / 4);
        if constexpr (OP == OP_WGRAD) {
            wgrad_epilogue<BN, C::BUFS>(args, tmem_base, q, half, my_staging, mg_bar + 2 * (warp - 2), tfull, tempty,
                               ring_full, ring_empty, ring_tile, abort_flag, &tmC0, &tmC1,
                               &tmS0, &tmS1);
        } else {
            int it = 0;
            for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
                const Tile t = decode_tile<OP>(tile, args);
                if (t.kblocks == 0) continue;
                const int buf = it & 1;
                const uint32_t use = uint32_t(it >> 1);
                ++it;
                int ok = 0;
                if (lane == 0) ok = mbar_wait(&tfull[buf], use & 1, abort_flag, args.status) ? 1 : 0;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                __syncwarp();
                tc_fence_after();
                const uint32_t t_row = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(buf * BN);
                epilogue_tile<OP, BN, false, CLAMP>(t, t_row, q, half, args, my_staging);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[buf]);
            }
        }
        __syncwarp();
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}


// ---------------------------------------------------------------- block-scaled MXFP8 GEMM
// Same roles and pipeline as moe_gemm_kernel; operands are E4M3 (K stage = 128
// elements = one 128-byte swizzle row), each stage also brings the 512-byte
// scale-factor atoms of A (128 rows x 4 K blocks) and B, which the MMA warp
// copies into a per-stage TMEM slot with tcgen05.cp; the four K=32 MMAs of a
// stage select their K block through the scale-factor id of the instruction
// descriptor.
// NH = 2: a CTA's tile is two adjacent 128-column tiles of the same rows, which
// share the stage's A tile (their B halves, scale atoms and accumulators side by
// side), so that a stage brings 48 KB for the work two 32 KB stages did: the
// operand fill rate of an SM from L2, not the tensor pipe, bounds these GEMMs.
// The accumulator pair then takes 256 TMEM columns, so it is single-buffered (the
// loads of the next tile go on while the epilogue drains it).
// The dgrad-down's SwiGLU-backward epilogue moves more bytes than its mainloop:
// it keeps NH = 1 and three stages (206 against 235 us with five at T=4096,
// H=2048, E=96 top-6, I=1024) unless its K is long (DEEP: five stages, 1.88 ->
// 1.67 ms at H=7168); the other ops stream operands: five stages at NH = 1,
// three (as many as fit) at NH = 2.
template <int OP, int NH, bool DEEP = false>
struct MxCfg {
    static constexpr uint32_t A_BYTES = kBM * kMxBK;
    static constexpr uint32_t B_HALF = kMxBN * kMxBK;          // one 128-column tile's B
    static constexpr uint32_t B_BYTES = NH * B_HALF;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t SF_BYTES = 512 * (1 + NH);       // A atom + NH B atoms
    static constexpr int STAGES = (OP == OP_BWD_DOWN && !DEEP) ? 3 : (NH == 1 ? 5 : 3);
    static constexpr int ACC = NH == 1 ? 2 : 1;                // accumulator buffers of NH x 128 columns
    static constexpr uint32_t STAGING = kEpiWarps * kStageTileBytes;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t SF_TMEM = 2 * kMxBN;             // scale slots after the accumulators
    static constexpr uint32_t SF_COLS = 4 * (1 + NH);          // TMEM columns of a stage's scale slot
    static constexpr uint32_t SF_REGION = (STAGES * SF_BYTES + 1023) / 1024 * 1024;  // keeps the staging 1 KB aligned
    static_assert(SF_TMEM + STAGES * SF_COLS <= TMEM_COLS, "tensor memory");
    static_assert(ACC * NH * kMxBN <= SF_TMEM, "accumulators");
    static constexpr size_t SMEM = size_t(STAGES) * STAGE_BYTES + SF_REGION + STAGING + 1024 + 256;
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

// instruction descriptor of kind::mxf8f6f4 with E4M3 A and B, UE8M0 scales, M = 128, N = 128
template <bool B_MN>
__device__ __forceinline__ uint32_t mx_idesc(uint32_t sf_id) {
    return (sf_id << 4) | ((B_MN ? 1u : 0u) << 16) | (uint32_t(kMxBN >> 3) << 17) | (1u << 23) |
           (uint32_t(kBM >> 4) << 24) | (sf_id << 29);
}

// shared-memory descriptor of a 32-row x 16-byte scale atom (no swizzle, 8-row groups 128 B apart)
__device__ __forceinline__ uint64_t sf_smem_desc(uint32_t addr) {
    return uint64_t((addr >> 4) & 0x3FFF) | (uint64_t(128 >> 4) << 32) | (1ull << 46);
}

__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

template <int OP, bool CLAMP, int NH, bool DEEP>
__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                       const __grid_constant__ CUtensorMap tmB1, const GemmArgs args) {
    using C = MxCfg<OP, NH, DEEP>;
    constexpr bool B_MN = (OP == OP_BWD_DOWN || OP == OP_BWD_GU);
    constexpr int STAGES = C::STAGES;
    constexpr int BN = kMxBN;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sf_smem = smem + STAGES * C::STAGE_BYTES;
    float* staging = reinterpret_cast<float*>(sf_smem + C::SF_REGION);  // 1024-byte aligned
    uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(staging) + C::STAGING);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], kEpiWarps);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB0);
        if (OP == OP_FWD_GU || OP == OP_BWD_GU) tma_prefetch_map(&tmB1);
    }
    if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();  // from here on the predecessor's writes are visible (prologue above touched no global memory)
    pdl_trigger();
    // a.n_tiles counts 128-column tiles; a CTA tile is NH of them (tile index in units of NH)
    const int total_tiles = (args.num_mtiles_dev ? *args.num_mtiles_dev : args.num_mtiles) * (args.n_tiles / NH);

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t filled = 0, fill_parity = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
                const Tile t = decode_mx_tile<NH>(tile, args);
                for (int kb = 0; kb < t.kblocks; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + stage * C::STAGE_BYTES;
                    uint8_t* ssf = sf_smem + stage * C::SF_BYTES;
                    uint64_t* bar = &full[stage];
                    const int k0 = kb * kMxBK;
                    mbar_arrive_expect_tx(bar, C::STAGE_BYTES + C::SF_BYTES);
                    tma_load_2d(sa, &tmA, bar, k0, t.mt * kBM);
                    bulk_load(ssf, args.sfa + (int64_t(t.mt) * args.sfa_kgroups + kb) * 512, 512, bar);
                    // an expert's payload: its own descriptor (z = 0) from a per-expert table, or the 3D map at z = e
                    const CUtensorMap* B0 = args.b0_tab ? args.b0_tab + t.e : &tmB0;
                    const CUtensorMap* B1 = args.b1_tab ? args.b1_tab + t.e : &tmB1;
                    const int z0 = args.b0_tab ? 0 : t.e;
                    const int z1 = args.b1_tab ? 0 : t.e;
#pragma unroll
                    for (int hf = 0; hf < NH; ++hf) {  // the B tile and scale atom of 128-column tile nt
                        const int nt = t.nt + hf;
                        uint8_t* sb = sa + C::A_BYTES + hf * C::B_HALF;
                        if (OP == OP_FWD_GU) {
                            tma_load_3d(sb, B0, bar, k0, nt * (kMxBN / 2), z0);
                            tma_load_3d(sb + (kMxBN / 2) * kMxBK, B1, bar, k0, nt * (kMxBN / 2), z1);
                        } else if (OP == OP_FWD_DOWN) {
                            tma_load_3d(sb, B0, bar, k0, nt * kMxBN, z0);
                        } else if (OP == OP_BWD_DOWN) {
                            tma_load_3d(sb, B0, bar, nt * kMxBN, k0, z0);
                        } else {
                            const bool up = k0 >= args.gate_up_split;
                            tma_load_3d(sb, up ? B1 : B0, bar, nt * kMxBN, up ? k0 - args.gate_up_split : k0,
                                        up ? z1 : z0);
                        }
                        bulk_load(ssf + 512 * (1 + hf),
                                  args.sfb + ((int64_t(t.e) * args.sfb_ntiles + nt) * args.sfb_kgroups + kb) * 512,
                                  512, bar);
                    }
                    filled |= 1u << stage;
                    fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok) {
                for (int s = 0; s < STAGES; ++s)
                    if (filled & (1u << s)) mbar_wait_drain(&full[s], (fill_parity >> s) & 1, args.status);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
                const Tile t = decode_mx_tile<NH>(tile, args);
                const int buf = C::ACC == 2 ? (it & 1) : 0;
                const uint32_t use = uint32_t(C::ACC == 2 ? (it >> 1) : it);
                ++it;
                if (!mbar_wait(&tempty[buf], (use & 1) ^ 1, abort_flag, args.status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + uint32_t(buf * NH * BN);
                for (int kb = 0; kb < t.kblocks; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t sf_addr = smem_u32(sf_smem + stage * C::SF_BYTES);
                    const uint32_t sfa_t = tmem_base + C::SF_TMEM + uint32_t(stage) * C::SF_COLS;
                    tmem_cp_sf(sfa_t, sf_smem_desc(sf_addr));
#pragma unroll
                    for (int hf = 0; hf < NH; ++hf) tmem_cp_sf(sfa_t + 4 * (1 + hf), sf_smem_desc(sf_addr + 512 * (1 + hf)));
#pragma unroll
                    for (int hf = 0; hf < NH; ++hf) {  // 128-column tile nt + hf: its B half, scales, accumulator
                        const uint32_t b_addr = a_addr + C::A_BYTES + hf * C::B_HALF;
                        const uint32_t sfb_t = sfa_t + 4 * (1 + hf);
#pragma unroll
                        for (int kk = 0; kk < kMxBK / 32; ++kk) {
                            const uint64_t ad = smem_desc(a_addr + kk * 32, 16, kSwizzleAtom);
                            const uint64_t bd = B_MN ? smem_desc(b_addr + kk * 32 * 128, 16384, kSwizzleAtom)
                                                     : smem_desc(b_addr + kk * 32, 16, kSwizzleAtom);
                            mma_mx(d_tmem + hf * BN, ad, bd, mx_idesc<B_MN>(uint32_t(kk)), sfa_t, sfb_t,
                                   (kb | kk) != 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (ok) mma_commit(&tfull[buf]);
            }
            mma_commit(drain);
            mbar_wait_drain(drain, 0, args.status);
        }
        __syncwarp();
    } else {
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        float* my_staging = staging + (warp - 2) * (kStageTileBytes / 4);
        int it = 0;
        for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
            const Tile t = decode_mx_tile<NH>(tile, args);
            const int buf = C::ACC == 2 ? (it & 1) : 0;
            const uint32_t use = uint32_t(C::ACC == 2 ? (it >> 1) : it);
            ++it;
            int ok = 0;
            if (lane == 0) ok = mbar_wait(&tfull[buf], use & 1, abort_flag, args.status) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            __syncwarp();
            tc_fence_after();
#pragma unroll 1
            for (int hf = 0; hf < NH; ++hf) {  // each 128-column tile as its own epilogue tile
                Tile th = t;
                th.nt = t.nt + hf;
                const uint32_t t_row = tmem_base + (uint32_t(q * 32) << 16) + uint32_t((buf * NH + hf) * BN);
                epilogue_tile<OP, BN, true, CLAMP>(th, t_row, q, half, args, my_staging);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[buf]);
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <int OP, bool CLAMP, int NH, bool DEEP = false>
cudaError_t launch_mx_one(const GemmMaps& m, const GemmArgs& a, int sms, cudaStream_t st) {
    static bool attr_set = false;
    using C = MxCfg<OP, NH, DEEP>;
    auto kern = moe_gemm_mx_kernel<OP, CLAMP, NH, DEEP>;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::SMEM));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int64_t tiles = int64_t(a.num_mtiles) * (a.n_tiles / NH);
    const int grid = int(tiles < sms ? tiles : sms);
    if (grid <= 0) return cudaSuccess;
    const cudaError_t e = launch_pdl(kern, dim3(grid), dim3(kGemmThreads), C::SMEM, st, m.a, m.b0, m.b1, a);
    count_launch();
    return e;
}

template <int OP, bool CLAMP>
cudaError_t launch_mx_nh(int nh, const GemmMaps& m, const GemmArgs& a, int sms, cudaStream_t st) {
    if (nh == 2 && OP != OP_BWD_DOWN && a.n_tiles % 2 == 0) return launch_mx_one<OP, CLAMP, (OP == OP_BWD_DOWN ? 1 : 2)>(m, a, sms, st);
    return launch_mx_one<OP, CLAMP, 1>(m, a, sms, st);
}

template <int OP, int BN, bool CLAMP, bool SPLIT, bool DEEP = false>
cudaError_t launch_one(const GemmMaps& m, const GemmArgs& a, int grid, cudaStream_t st) {
    static bool attr_set = false;
    using C = Cfg<OP, BN, SPLIT, DEEP>;
    static_assert(C::SMEM <= 227 * 1024, "shared memory per CTA");
    auto kern = moe_gemm_kernel<OP, BN, CLAMP, SPLIT, DEEP>;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::SMEM));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const cudaError_t e = launch_pdl(kern, dim3(grid), dim3(kGemmThreads), C::SMEM, st, m.a, m.b0, m.b1, m.c0, m.c1,
                                     m.s0, m.s1, m.lo, m.g0, a);
    count_launch();
    return e;
}

// the split builds exist for the GEMMs that take a two-term operand
template <int OP, bool CLAMP = false>
cudaError_t launch_bn(int bn, const GemmMaps& m, const GemmArgs& a, int grid, cudaStream_t st) {
    constexpr bool CAN_SPLIT = OP == OP_FWD_DOWN || OP == OP_BWD_GU || OP == OP_WGRAD;
    if (a.split && !CAN_SPLIT) return cudaErrorInvalidValue;
    if constexpr (OP == OP_WGRAD)  // long K per tile, A the split operand: the deep build
        if (bn == 256 && a.split == 1 && a.deep_stages) return launch_one<OP, 256, CLAMP, true, true>(m, a, grid, st);
    if (CAN_SPLIT && a.split) {
        switch (bn) {
            case 256: return launch_one<OP, 256, CLAMP, CAN_SPLIT>(m, a, grid, st);
            case 128: return launch_one<OP, 128, CLAMP, CAN_SPLIT>(m, a, grid, st);
            case 64: return launch_one<OP, 64, CLAMP, CAN_SPLIT>(m, a, grid, st);
            default: return cudaErrorInvalidValue;
        }
    }
    // the dgrad-down with a long K (a.deep_stages): four stages, its epilogue a smaller share
    if constexpr (OP == OP_BWD_DOWN)
        if (bn == 256 && a.deep_stages) return launch_one<OP, 256, CLAMP, false, true>(m, a, grid, st);
    switch (bn) {
        case 256: return launch_one<OP, 256, CLAMP, false>(m, a, grid, st);
        case 128: return launch_one<OP, 128, CLAMP, false>(m, a, grid, st);
        case 64: return launch_one<OP, 64, CLAMP, false>(m, a, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

namespace {
// thread 0 waits on a barrier of phase 0 that nothing arrives at: mbar_wait gives up after
// kWaitLimitNs, setting the abort flag and the timeout bit of *status
__global__ void wait_selftest_kernel(int* status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
        (void)mbar_wait(&bar, 0, &abort_flag, status);
    }
}
}  // namespace

cudaError_t launch_wait_selftest(int* status, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(status);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_gemm_mx(int op, const GemmMaps& m, const GemmArgs& a, int nh, int sms, cudaStream_t st) {
    const bool clamp = a.swiglu_limit > 0.0f;
    switch (op) {
        // the SwiGLU epilogues come in a clamped and an unclamped build
        case OP_FWD_GU:
            return clamp ? launch_mx_nh<OP_FWD_GU, true>(nh, m, a, sms, st)
                         : launch_mx_nh<OP_FWD_GU, false>(nh, m, a, sms, st);
        case OP_FWD_DOWN: return launch_mx_nh<OP_FWD_DOWN, false>(nh, m, a, sms, st);
        case OP_BWD_DOWN:
            if (a.deep_stages)
                return clamp ? launch_mx_one<OP_BWD_DOWN, true, 1, true>(m, a, sms, st)
                             : launch_mx_one<OP_BWD_DOWN, false, 1, true>(m, a, sms, st);
            return clamp ? launch_mx_one<OP_BWD_DOWN, true, 1>(m, a, sms, st)
                         : launch_mx_one<OP_BWD_DOWN, false, 1>(m, a, sms, st);
        case OP_BWD_GU: return launch_mx_nh<OP_BWD_GU, false>(nh, m, a, sms, st);
        default: return cudaErrorInvalidValue;
    }
}

int pick_bn(int64_t n, bool split_gate_up) {
    // split_gate_up: n is 2I and each half of the tile must divide I
    const int cands[3] = {256, 128, 64};
    for (int bn : cands) {
        if (split_gate_up) {
            if (bn >= 128 && (n / 2) % (bn / 2) == 0) return bn;
        } else if (n % bn == 0) {
            return bn;
        }
    }
    return 0;
}

cudaError_t launch_gemm(int op, int bn, const GemmMaps& m, const GemmArgs& a, int grid, cudaStream_t st) {
    if (grid <= 0) return cudaSuccess;
    const bool clamp = a.swiglu_limit > 0.0f;
    switch (op) {
        case OP_FWD_GU:
            return clamp ? launch_bn<OP_FWD_GU, true>(bn, m, a, grid, st) : launch_bn<OP_FWD_GU>(bn, m, a, grid, st);
        case OP_FWD_DOWN: return launch_bn<OP_FWD_DOWN>(bn, m, a, grid, st);
        case OP_BWD_DOWN:
            return clamp ? launch_bn<OP_BWD_DOWN, true>(bn, m, a, grid, st)
                         : launch_bn<OP_BWD_DOWN>(bn, m, a, grid, st);
        case OP_BWD_GU: return launch_bn<OP_BWD_GU>(bn, m, a, grid, st);
        case OP_WGRAD: return launch_bn<OP_WGRAD>(bn, m, a, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

// ------------------------------------------------------------------ tensor maps
namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}
}  // namespace

bool encode_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                const uint32_t* box, int type) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t d[3], s[2];
    cuuint32_t b[3], es[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
    }
    for (int i = 0; i < rank - 1; ++i) s[i] = strides_bytes[i];
    const CUtensorMapDataType dt = type == MAP_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : type == MAP_U8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                    : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUresult r = fn(m, dt, cuuint32_t(rank), const_cast<void*>(base), d, s, b, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace moe
