// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kBM = 128;        // GEMM tile rows (= TMEM lanes) and expert segment padding
constexpr int kBK = 64;         // GEMM K block (64 bf16 = one 128-byte swizzle row)
constexpr int kEpiWarps = 8;    // epilogue warps: two per TMEM lane quarter, alternating 32-column chunks
constexpr int kEpiHalves = kEpiWarps / 4;
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;

// device status word bits (read back by moe_device_status)
constexpr int kStatusRouting = 1;  // a routing_map row had more than k routes
constexpr int kStatusTimeout = 2;  // a bounded wait gave up

// the five GEMM shapes of the layer
enum GemmOp : int {
    OP_FWD_GU = 0,    // [a | g,u] = SwiGLU(X W_fc1^T): A K-major rows, B = gate/up rows (K-major)
    OP_FWD_DOWN = 1,  // y = a W_down^T: A K-major, B = W_down rows (K-major)
    OP_BWD_DOWN = 2,  // da_u = go W_down; SwiGLU backward epilogue: A K-major, B = W_down (N-major)
    OP_BWD_GU = 3,    // dx = [dg|du] W_fc1: A K-major (K = 2I), B = gate/up (N-major)
    OP_WGRAD = 4,     // main_grad += A^T B over a token segment: A, B both M/N-major
};

struct GemmArgs {
    // row-tile scheduling (OP 0..3)
    const int* mtile_expert;    // expert of each 128-row tile; null: expert 0 for every tile
    const int* num_mtiles_dev;  // device-resident tile count; null: use num_mtiles
    int num_mtiles;
    int n_tiles;                // N / BN
    int k_blocks;               // K / 64
    int rows_valid;             // output rows >= rows_valid are not stored
    int gate_up_split;          // I: offset of the up half (N for FWD_GU, K for BWD_GU)
    // segment scheduling (OP_WGRAD)
    const int* seg_off;         // [groups+1] row offsets of each group's K range; null: [0, seg_len)
                                // (OP 0..3: each group's first row, for the row limits below)
    int seg_len;
    const int* seg_rows;        // with seg_off: valid rows of each routed group (its token count). OP_WGRAD:
                                // a group's K range ends with its last 64-row block that holds a valid row
                                // (the padding rows after it are zero and add nothing); OP 0..3: the
                                // epilogue stores only rows below that block's end (the padding past it
                                // is read by nothing). null: every row
    int g0_rows;                // with seg_rows and group0_shared: valid rows of group 0 (the tokens)
    int groups;
    int m_tiles;                // M / 128
    // epilogue operands
    __nv_bfloat16* out0;        // bf16 GEMM operands produced here: a, [dg|du]
    int64_t ld_out0;
    __nv_bfloat16* out1;        // p * a
    int64_t ld_out1;
    __nv_bfloat16* outh;        // bf16 GEMM results passed on: [g|u] (kept for backward), y, dx
    int64_t ld_outh;
    const __nv_bfloat16* in0;   // a
    int64_t ld_in0;
    const __nv_bfloat16* inh;   // [g|u]
    int64_t ld_inh;
    // fp32 activations (the default precision): results kept in fp32 and the
    // derived GEMM operands given as two bf16 terms, hi = bf16(v), lo = bf16(v - hi)
    float* outf;                // fp32 results (replace outh): FWD_GU [g|u], FWD_DOWN y, BWD_GU dx
    int64_t ld_outf;
    const float* inf;           // BWD_DOWN: fp32 [g|u], a recomputed from them (replaces in0, inh)
    int64_t ld_inf;
    __nv_bfloat16* out0lo;      // lo terms of out0 (a, [dg|du])
    int64_t ld_out0lo;
    __nv_bfloat16* out1lo;      // lo terms of out1 (p * a)
    int64_t ld_out1lo;
    int split;                  // 1: A, 2: B operand comes as hi (its map) + lo (map lo) terms
    int deep_stages;            // long K: dgrad-down more stages (BF16 N tile 256: four; MXFP8: five); gate/up
                                // weight gradient with a two-term A: three stages, one main_grad box buffer
    int g0_operand;             // group 0 (the shared expert) reads its token rows through map g0:
                                // 1: the A operand, 2: the B operand (0: the row buffer like the others)
    const float* row_scale;     // BWD_DOWN: per-row prob (null: 1)
    float* partial;             // per row: n_tiles * kEpiHalves partial dot products (null: skip)
    int m_split;                // WGRAD rows >= m_split go to the second main_grad map at row - m_split
    int mg_trans;               // WGRAD (deep build, fp32 main_grad): the accumulator tile is the
                                // transpose of the main_grad tile (its rows are main_grad columns)
    int inter;
    float swiglu_limit;         // > 0: SwiGLU inputs clamped, g <= L, |u| <= L (FWD_GU, BWD_DOWN epilogues)
    int mg_bf16;                // WGRAD: main_grad is bf16 (bf16(mg + bf16(dW))), else fp32 (mg + dW)
    int* tile_counter;          // WGRAD: zeroed before the launch; CTAs claim tiles from it in order
    // per-expert descriptor tables in device memory (null: the 3D maps, expert = z);
    // entry e is expert e's own map (z = 0)
    const CUtensorMap* b0_tab;
    const CUtensorMap* b1_tab;
    const CUtensorMap* c0_tab;
    const CUtensorMap* c1_tab;
    // 1: group (expert) 0 is the shared expert, with its own maps (GemmMaps s0, s1),
    // and group e >= 1 routed expert e - 1 (the tables' entry e - 1, or z = e - 1)
    int group0_shared;
    int* status;
    // MXFP8 (block-scaled) GEMMs
    uint8_t* q_out;             // E4M3 copy of the epilogue's GEMM-operand output (a, or [dg|du])
    int64_t ld_q;
    uint8_t* q_sf;              // its scale atoms (K blocks of 32 = q_kblocks)
    int q_kblocks;
    const uint8_t* sfa;         // A operand scale atoms [m tiles][K/128][512 B]
    int sfa_kgroups;
    const uint8_t* sfb;         // B operand scale atoms [E][n tiles][K/128][512 B]
    int sfb_ntiles, sfb_kgroups;
};

struct GemmMaps {
    CUtensorMap a, b0, b1;
    CUtensorMap lo;      // split operand: the lo terms of A (split 1) or B (split 2), same box as its hi map
    CUtensorMap g0;      // group 0's token rows (hidden or grad_out, T rows; rows past T read as zeros)
    CUtensorMap c0, c1;  // OP_WGRAD: main_grad destinations (rows < m_split, rows >= m_split)
    // group0_shared: the shared expert's b0, b1 (OP 0..3) or c0, c1 (OP_WGRAD)
    CUtensorMap s0, s1;
};

// tensor-map construction (driver entry point resolved at first use), 128-byte swizzle
enum MapType : int { MAP_BF16 = 0, MAP_F32 = 1, MAP_U8 = 2 };
bool encode_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                const uint32_t* box, int type = MAP_BF16);

// picks the N tile (256, 128 or 64) for an output width
int pick_bn(int64_t n, bool split_gate_up);

cudaError_t launch_gemm(int op, int bn, const GemmMaps& maps, const GemmArgs& args, int grid, cudaStream_t st);
// one block waiting on an mbarrier that nothing completes (the bounded wait gives up and
// sets the timeout bit of *status): the test of the timeout path
cudaError_t launch_wait_selftest(int* status, cudaStream_t st);
// block-scaled MXFP8 GEMM (N tile 128, K stage 128); ops FWD_GU, FWD_DOWN, BWD_DOWN, BWD_GU
// nh = 2: a CTA tile is two adjacent 128-column tiles sharing the A stage (the
// gate/up forward, down forward and dgrad through gate/up; n_tiles even); else 1.
// The grid is min(tiles, sms).
cudaError_t launch_gemm_mx(int op, const GemmMaps& maps, const GemmArgs& args, int nh, int sms, cudaStream_t st);
constexpr int kMxBN = 128;
constexpr int kMxBK = 128;

// routing
constexpr int kRankChunk = 128;  // tokens per block of the fused pack/rank kernel
int route_rank_max_tokens();
// the dense routing map + probs, or (topk_ids set) the router's top-k ids + probs
cudaError_t launch_route_pack_rank(const uint8_t* map, const float* probs, const int* topk_ids,
                                   const float* topk_probs, int T, int E, int k, int* ids, float* pp, int* row_of,
                                   int* rank, int* hist, int* status, cudaStream_t st);
// mtile_x (optional): tile experts of the shared-first grouped GEMM (shared_tiles
// tiles of group 0, then routed expert e as group e + 1), seg_x its E + 2 row
// offsets, meta[3] its tile count and meta[4] its row count
cudaError_t launch_route_scan_chunks(int* hist, int T, int E, int* counts, int* offsets, int* offs_pad,
                                     int* mtile_expert, int* meta, int shared_tiles, int* mtile_x, int* seg_x,
                                     cudaStream_t st);
cudaError_t launch_route_pack(const uint8_t* map, const float* probs, int T, int E, int k, int* ids, float* pp,
                              int* row_of, int* status, cudaStream_t st);
cudaError_t launch_route_rank(const uint8_t* map, const int* ids, int T, int E, int k, int* rank, int* counts,
                              cudaStream_t st);
// shared_rows > 0: also writes the shared expert's rows, which sit at rows
// [-shared_rows, 0) of perm_src, pp_perm and x_perm (no MXFP8 copy)
// copy_shared: also copy the shared rows' hidden rows (else only their source and scale)
cudaError_t launch_route_place(const int* ids, const float* pp, const int* rank, const int* chunk_base,
                               const int* counts, const int* offs_pad, int T, int E, int k, int shared_rows,
                               bool copy_shared,
                               const __nv_bfloat16* hidden, int H, int* perm_src, float* pp_perm, int* row_of,
                               __nv_bfloat16* x_perm, uint8_t* x_q, uint8_t* x_sf, cudaStream_t st);
// tab0 / tab1: device arrays of E source pointers, expert e's scales at tab[e]
// with row stride src_rs
cudaError_t launch_swizzle_scales(int mode, const uint8_t* const* tab0, const uint8_t* const* tab1, int64_t src_rs,
                                  int E, int n_tiles, int k_blocks, int kb_split, uint8_t* dst, cudaStream_t st);
cudaError_t launch_export_routing(const int* ids, const int* row_of, const int* perm_src_pad, const int* counts,
                                  const int* offsets, const int* offs_pad, const int* mtile_expert, const int* meta,
                                  int T, int k, int max_rows, int32_t* perm_src_out, int32_t* row_of_out,
                                  cudaStream_t st);

// elementwise / copy
// dst row r (r < row0 + *n_dev, r < max_rows) = src row perm_src[r], a zero row where it is -1
// dst[row_of[t,s]] = src[t] for every valid route, zero padding rows (counts, offs_pad:
// the routed segments); with dst_q also the rows' MXFP8 quantisation along H
cudaError_t launch_gather_rows(const __nv_bfloat16* src, const int* row_of, const int* counts, const int* offs_pad,
                               int T, int E, int k, int H, __nv_bfloat16* dst, uint8_t* dst_q, uint8_t* dst_sf,
                               cudaStream_t st);
// ys, y (and dxs, dxp): fp32 rows when f32, else bf16
cudaError_t launch_combine(const void* ys, const float* gate, const void* y, bool f32, const int* row_of,
                           const float* pp, int T, int H, int k, __nv_bfloat16* out, int num_sms, cudaStream_t st);
cudaError_t launch_unpermute(const void* dxs, const void* dxp, bool f32, const int* row_of, const int* ids,
                             const float* partial, int n_part, int T, int H, int k, int E, const float* dz,
                             const __nv_bfloat16* gate_w, __nv_bfloat16* dhidden, float* dprobs, bool slot_dprobs,
                             int num_sms, cudaStream_t st);

// shared-expert output gate
constexpr int kGateChunk = 128;  // tokens per partial sum of the gate weight's gradient
cudaError_t launch_gate_forward(const __nv_bfloat16* hidden, const __nv_bfloat16* w, int T, int H, float* gate,
                                cudaStream_t st);
cudaError_t launch_gate_backward(const __nv_bfloat16* hidden, const float* gate, const float* partial, int n_part,
                                 int T, int H, float* dz, float* gpart, void* mg_gate, bool mg_bf16, cudaStream_t st);

void count_launch(int n = 1);

// launches kernel<<<grid, block, smem, st>>>(args...) with programmatic stream
// serialisation (the kernel calls pdl_wait before touching global memory)
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace moe
