// C ABI of the MoE layer library: argument checks, memory carving, tensor
// maps and the launch sequence of forward and backward. Declarations and the
// contract of every entry point are in include/moe.h.
#include "../../include/moe.h"
#include "internal.h"

#include <algorithm>
#include <array>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

namespace moe {
static std::atomic<uint64_t> g_launches{0};
void count_launch(int n) { g_launches.fetch_add(uint64_t(n), std::memory_order_relaxed); }
}  // namespace moe

using namespace moe;

namespace {

constexpr size_t kAlign = 256;

// per-expert descriptor tables: one TMA descriptor per expert for each use of a
// routed weight (each GEMM loads its own box shape) and of a routed main_grad
enum TableId : int {
    TB_FWD_GU_G = 0, TB_FWD_GU_U, TB_FWD_DOWN, TB_BWD_DOWN, TB_BWD_GU_G, TB_BWD_GU_U,
    TB_MG_G, TB_MG_U, TB_MG_D, kTables
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Shape {
    int64_t Tmax, H, E, k, I;
    int64_t rows;     // permuted rows incl. padding, worst case
    int64_t srows;    // rows of the shared expert's region (Tmax rounded up to 128)
    int bn_gu, bn_down, bn_bd, bn_bgu, bn_wfc1, bn_wd;
    int n_part;       // dprob partials per row (= N tiles of the dgrad-down GEMM x epilogue halves)
    int n_part_s;     // the same for the shared expert's (always BF16) dgrad-down GEMM
    bool mx;          // routed weights MXFP8: block-scaled fprop and dgrad GEMMs
    bool recompute;   // recompute_dispatch: the backward redoes placement and gate/up
    bool act32;       // MOE_ACT_FP32: fp32 g|u, y, dx; derived GEMM operands as hi + lo bf16 terms
    float limit;      // swiglu_limit (0: none)
    bool shared;      // the layer has the shared expert (no_shared_expert = 0)
    // block-scaled GEMMs: 128-column tiles per CTA tile (1 or 2) of the gate/up forward, the
    // down forward and the dgrad through gate/up
    int mx_nh_gu, mx_nh_down, mx_nh_bgu;
};

// carves consecutive 256-byte aligned pieces out of one block
struct Carver {
    uint8_t* base;
    size_t off = 0;
    template <typename T>
    T* take(size_t count) {
        off = align_up(off, kAlign);
        T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
        off += count * sizeof(T);
        return p;
    }
};

moe_status check_config(const moe_config* c, Shape* s) {
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->max_tokens < 0 || c->hidden <= 0 || c->num_experts <= 0 || c->topk <= 0 || c->inter <= 0)
        return MOE_ERR_INVALID_ARG;
    if (!(c->swiglu_limit >= 0.0f) || !std::isfinite(c->swiglu_limit)) return MOE_ERR_INVALID_ARG;
    if (c->recompute_dispatch != 0 && c->recompute_dispatch != 1) return MOE_ERR_INVALID_ARG;
    if (c->act_precision != MOE_ACT_FP32 && c->act_precision != MOE_ACT_BF16) return MOE_ERR_INVALID_ARG;
    if (c->no_shared_expert != 0 && c->no_shared_expert != 1) return MOE_ERR_INVALID_ARG;
    s->shared = c->no_shared_expert == 0;
    s->recompute = c->recompute_dispatch != 0;
    s->act32 = c->act_precision == MOE_ACT_FP32;
    s->limit = c->swiglu_limit;
    if (c->routed_wtype != MOE_W_BF16 && c->routed_wtype != MOE_W_MXFP8) return MOE_ERR_UNSUPPORTED;
    s->mx = c->routed_wtype == MOE_W_MXFP8;
    if (s->mx && (c->hidden % 128 || c->inter % 128)) return MOE_ERR_UNSUPPORTED;
    if (c->num_experts > 1024 || c->topk > 32 || c->topk > c->num_experts) return MOE_ERR_UNSUPPORTED;
    if (c->hidden % 128 || c->inter % 64) return MOE_ERR_UNSUPPORTED;
    s->Tmax = c->max_tokens;
    s->H = c->hidden;
    s->E = c->num_experts;
    s->k = c->topk;
    s->I = c->inter;
    s->rows = align_up(size_t(s->Tmax * s->k + s->E * (kBM - 1)), kBM);
    s->srows = s->shared ? align_up(size_t(s->Tmax), kBM) : 0;
    if (s->rows + s->srows >= INT_MAX / 2 || s->Tmax * s->k >= INT_MAX / 2) return MOE_ERR_UNSUPPORTED;
    if (s->Tmax > route_rank_max_tokens()) return MOE_ERR_UNSUPPORTED;
    s->bn_gu = pick_bn(2 * s->I, true);
    s->bn_down = pick_bn(s->H, false);
    s->bn_bd = pick_bn(s->I, false);
    s->bn_bgu = pick_bn(s->H, false);
    s->bn_wfc1 = pick_bn(s->H, false);
    s->bn_wd = pick_bn(s->I, false);
    if (!s->bn_gu || !s->bn_down || !s->bn_bd || !s->bn_bgu || !s->bn_wfc1 || !s->bn_wd) return MOE_ERR_UNSUPPORTED;
    s->n_part = int(s->I / (s->mx ? kMxBN : s->bn_bd)) * kEpiHalves;
    s->n_part_s = int(s->I / s->bn_bd) * kEpiHalves;
    // Pairs of 128-column tiles share a stage's A tile (a quarter fewer bytes a stage) but
    // get three stages instead of five and a single-buffered accumulator: measured at
    // T=4096 H=2048 E=96 top-6 I=1024 and T=8192 H=7168 E=384 top-6 I=2048, the dgrad
    // through gate/up gains at both (178 -> 172, 2554 -> 2420 us), the gate/up forward
    // only with a long K (2590 -> 2484 us at H = 7168; 192 -> 213 us at H = 2048), the
    // down forward at neither
    s->mx_nh_gu = s->H / kMxBK >= 32 ? 2 : 1;
    s->mx_nh_down = 1;
    s->mx_nh_bgu = 2;
    return MOE_OK;
}

// Row buffers (per-row operands of the grouped GEMMs) hold the shared expert's
// rows first, rows [0, R0) with R0 = T rounded up to 128 (token t at row t, zero
// rows after T), and the routed segments from row R0 on; srows + rows rows each.
struct Workspace {
    int* status;
    int* tile_counters;  // one per weight-gradient launch of a backward (dynamic tile scheduling)
    __nv_bfloat16 *go_all, *dgdu_all, *ap_all;  // grad_out rows, [dg|du] (hi terms), prob (or gate) * a (hi)
    __nv_bfloat16* yx_all;  // bf16 activations -- forward: y; backward: dx
    float* yx32;            // fp32 activations -- forward: y; backward: dx
    // fp32 activations: lo terms of a (forward only), [dg|du] and prob * a
    __nv_bfloat16 *alo_all, *dgdulo_all, *aplo_all;
    float* partial_all;     // dgrad-down partial dot products (n_part per row)
    // MXFP8 routed weights: the shared expert's own dgrad-down partials (n_part_s per row)
    float* partial_s;
    // shared output gate: dz and the chunk sums of the gate weight's gradient
    float *dz, *gpart;
    // per-expert TMA descriptors of the tables (kTables x E)
    CUtensorMap* tabs;
    // recompute_dispatch: the GEMM input rows, a and [g|u] (and their MXFP8 copies)
    // live here, shared by every saved state of the handle, instead of in each
    __nv_bfloat16 *x_all, *a_all, *gu_all;
    float* gu32;
    uint8_t *x_q, *x_sf, *a_q, *a_sf;
    // MXFP8 only: quantised backward operands and the swizzled weight scales
    uint8_t *go_q, *go_sf, *dgdu_q, *dgdu_sf;
    uint8_t *sf_fc1_row, *sf_down_row, *sf_down_col, *sf_fc1_col;
    // MXFP8: per-expert source scale pointers of the swizzle (gate, up, down rowwise;
    // down, gate, up columnwise; E each)
    const uint8_t** sf_src;
};

struct SavedBufs {
    int *ids, *row_of, *counts, *offsets, *offs_pad, *mtile_expert;  // routed segments (relative to row R0)
    int* rank;  // rank of each route inside its expert
    int* hist;  // per 128-token chunk and expert: route count, then the chunk's rank offset
    int* meta;  // [0..2] routed tiles, routes, rows; [3], [4] tiles and rows of the shared-first GEMMs
    int *mtile_x, *seg_x;  // shared-first grouped GEMMs: group of each 128-row tile, E + 2 group row offsets
    int* perm_src_all;     // source token of each row (-1: zero row)
    float* pp;
    float* pp_all;         // per row: the shared output gate (1 without one), the route's prob, 0 for padding
    __nv_bfloat16 *x_all, *a_all, *gu_all;  // GEMM input rows, SwiGLU output a (hi terms), bf16 [g|u]
    float* gu32;                            // fp32 activations: [g|u] (kept for backward), gu_all unused
    uint8_t *x_q, *x_sf, *a_q, *a_sf;  // MXFP8 only: routed rows (relative to row R0)
};

// the routed part of the row buffers for a call with T tokens
struct Views {
    int R0;  // rows of the shared expert's region
    int* perm_src;
    float* pp_perm;
    __nv_bfloat16 *x_perm, *a, *gu, *go_perm, *dgdu, *ap, *yx;
    float *gu32, *yx32;
    __nv_bfloat16 *dgdulo, *aplo;
    float* partial;
};

// bytes of MXFP8 scale atoms for R rows (multiple of 128) and K columns (multiple of 128)
size_t sf_atoms_bytes(int64_t rows, int64_t K) { return size_t(rows / 128) * size_t(K / 128) * 512; }

size_t carve_workspace(const Shape& s, uint8_t* base, Workspace* w) {
    Carver c{base};
    w->status = c.take<int>(64);
    w->tile_counters = c.take<int>(4);
    const size_t ra = size_t(s.srows + s.rows);
    w->go_all = c.take<__nv_bfloat16>(ra * s.H);
    w->dgdu_all = c.take<__nv_bfloat16>(ra * 2 * s.I);
    w->ap_all = c.take<__nv_bfloat16>(ra * s.I);
    w->yx_all = w->alo_all = w->dgdulo_all = w->aplo_all = nullptr;
    w->yx32 = nullptr;
    if (s.act32) {
        w->yx32 = c.take<float>(ra * s.H);
        w->alo_all = c.take<__nv_bfloat16>(ra * s.I);
        w->dgdulo_all = c.take<__nv_bfloat16>(ra * 2 * s.I);
        w->aplo_all = c.take<__nv_bfloat16>(ra * s.I);
    } else {
        w->yx_all = c.take<__nv_bfloat16>(ra * s.H);
    }
    w->partial_all = c.take<float>(ra * s.n_part);
    w->partial_s = s.mx ? c.take<float>(size_t(s.Tmax) * s.n_part_s) : nullptr;
    w->dz = c.take<float>(size_t(s.Tmax));
    w->gpart = c.take<float>(size_t((s.Tmax + kGateChunk - 1) / kGateChunk) * s.H);
    w->tabs = c.take<CUtensorMap>(size_t(kTables) * s.E);
    w->x_all = w->a_all = w->gu_all = nullptr;
    w->gu32 = nullptr;
    w->x_q = w->x_sf = w->a_q = w->a_sf = nullptr;
    if (s.recompute) {
        w->x_all = c.take<__nv_bfloat16>(ra * s.H);
        w->a_all = c.take<__nv_bfloat16>(ra * s.I);
        if (s.act32)
            w->gu32 = c.take<float>(ra * 2 * s.I);
        else
            w->gu_all = c.take<__nv_bfloat16>(ra * 2 * s.I);
        if (s.mx) {
            w->x_q = c.take<uint8_t>(size_t(s.rows) * s.H);
            w->x_sf = c.take<uint8_t>(sf_atoms_bytes(s.rows, s.H));
            w->a_q = c.take<uint8_t>(size_t(s.rows) * s.I);
            w->a_sf = c.take<uint8_t>(sf_atoms_bytes(s.rows, s.I));
        }
    }
    if (s.mx) {
        w->go_q = c.take<uint8_t>(size_t(s.rows) * s.H);
        w->go_sf = c.take<uint8_t>(sf_atoms_bytes(s.rows, s.H));
        w->dgdu_q = c.take<uint8_t>(size_t(s.rows) * 2 * s.I);
        w->dgdu_sf = c.take<uint8_t>(sf_atoms_bytes(s.rows, 2 * s.I));
        w->sf_fc1_row = c.take<uint8_t>(size_t(s.E) * sf_atoms_bytes(2 * s.I, s.H));
        w->sf_down_row = c.take<uint8_t>(size_t(s.E) * sf_atoms_bytes(s.H, s.I));
        w->sf_down_col = c.take<uint8_t>(size_t(s.E) * sf_atoms_bytes(s.I, s.H));
        w->sf_fc1_col = c.take<uint8_t>(size_t(s.E) * sf_atoms_bytes(s.H, 2 * s.I));
        w->sf_src = c.take<const uint8_t*>(6 * size_t(s.E));
    } else {
        w->go_q = w->go_sf = w->dgdu_q = w->dgdu_sf = nullptr;
        w->sf_fc1_row = w->sf_down_row = w->sf_down_col = w->sf_fc1_col = nullptr;
        w->sf_src = nullptr;
    }
    return align_up(c.off, kAlign);
}

size_t carve_saved(const Shape& s, uint8_t* base, SavedBufs* b) {
    Carver c{base};
    const size_t tk = size_t(s.Tmax * s.k);
    b->ids = c.take<int>(tk);
    b->pp = c.take<float>(tk);
    b->row_of = c.take<int>(tk);
    b->rank = c.take<int>(tk);
    b->hist = c.take<int>(size_t((s.Tmax + kRankChunk - 1) / kRankChunk) * s.E);
    b->counts = c.take<int>(s.E);
    b->offsets = c.take<int>(s.E + 1);
    b->offs_pad = c.take<int>(s.E + 1);
    b->meta = c.take<int>(8);
    b->mtile_expert = c.take<int>(s.rows / kBM);
    const size_t ra = size_t(s.srows + s.rows);
    b->mtile_x = c.take<int>(ra / kBM);
    b->seg_x = c.take<int>(s.E + 2);
    b->perm_src_all = c.take<int>(ra);
    b->pp_all = c.take<float>(ra);
    b->x_all = b->a_all = b->gu_all = nullptr;  // recompute_dispatch: the workspace's (moe_saved_create)
    b->gu32 = nullptr;
    b->x_q = b->x_sf = b->a_q = b->a_sf = nullptr;
    if (!s.recompute) {
        b->x_all = c.take<__nv_bfloat16>(ra * s.H);
        b->a_all = c.take<__nv_bfloat16>(ra * s.I);
        if (s.act32)
            b->gu32 = c.take<float>(ra * 2 * s.I);
        else
            b->gu_all = c.take<__nv_bfloat16>(ra * 2 * s.I);
        if (s.mx) {
            b->x_q = c.take<uint8_t>(size_t(s.rows) * s.H);
            b->x_sf = c.take<uint8_t>(sf_atoms_bytes(s.rows, s.H));
            b->a_q = c.take<uint8_t>(size_t(s.rows) * s.I);
            b->a_sf = c.take<uint8_t>(sf_atoms_bytes(s.rows, s.I));
        }
    }
    return align_up(c.off, kAlign);
}

Views views_of(const Shape& s, const SavedBufs& b, const Workspace& w, int64_t T) {
    Views v;
    v.R0 = s.shared ? int(align_up(size_t(T), kBM)) : 0;
    const int64_t r = v.R0;
    v.perm_src = b.perm_src_all + r;
    v.pp_perm = b.pp_all + r;
    v.x_perm = b.x_all + r * s.H;
    v.a = b.a_all + r * s.I;
    v.gu = s.act32 ? nullptr : b.gu_all + r * 2 * s.I;
    v.gu32 = s.act32 ? b.gu32 + r * 2 * s.I : nullptr;
    v.go_perm = w.go_all + r * s.H;
    v.dgdu = w.dgdu_all + r * 2 * s.I;
    v.ap = w.ap_all + r * s.I;
    v.yx = s.act32 ? nullptr : w.yx_all + r * s.H;
    v.yx32 = s.act32 ? w.yx32 + r * s.H : nullptr;
    v.dgdulo = s.act32 ? w.dgdulo_all + r * 2 * s.I : nullptr;
    v.aplo = s.act32 ? w.aplo_all + r * s.I : nullptr;
    v.partial = w.partial_all + r * s.n_part;
    return v;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// a weight view of N rows x K columns (per expert when routed)
bool check_view(const moe_wview& v, int64_t N, int64_t K, bool routed) {
    if (v.row_stride < K || (v.row_stride * 2) % 16) return false;
    if (routed && v.expert_ptrs) return true;  // per-expert pointers: checked as they are encoded
    if (!v.data || !aligned16(v.data)) return false;
    if (routed && (v.expert_stride < N * v.row_stride || (v.expert_stride * 2) % 16)) return false;
    return true;
}

// an MXFP8 view of N rows x K columns per expert: E4M3 payloads (row stride in bytes), scales
// indexed with the payload strides (see include/moe.h)
bool check_mx_view(const moe_wview& v, int64_t N, int64_t K) {
    if (v.expert_ptrs) return v.row_stride >= K && v.row_stride % 32 == 0;  // pointers checked as they are used
    if (!v.data || !v.col_data || !v.scale || !v.col_scale) return false;
    if (!aligned16(v.data) || !aligned16(v.col_data)) return false;
    if (v.row_stride < K || v.row_stride % 32 || v.expert_stride < N * v.row_stride || v.expert_stride % 32)
        return false;
    return true;
}

bool check_weights(const Shape& s, const moe_weights* w) {
    if (!w) return false;
    const bool shared = !s.shared || (check_view(w->shared_gate, s.I, s.H, false) &&
                                      check_view(w->shared_up, s.I, s.H, false) &&
                                      check_view(w->shared_down, s.H, s.I, false));
    if (s.mx)
        return shared && check_mx_view(w->routed_gate, s.I, s.H) && check_mx_view(w->routed_up, s.I, s.H) &&
               check_mx_view(w->routed_down, s.H, s.I);
    return shared && check_view(w->routed_gate, s.I, s.H, true) && check_view(w->routed_up, s.I, s.H, true) &&
           check_view(w->routed_down, s.H, s.I, true);
}

// 2D K-major E4M3 operand: rows x K bytes, box 128 x 128 rows
bool map_u8_kmajor(CUtensorMap* m, const void* base, int64_t rows, int64_t K, int64_t ld) {
    const uint64_t dims[2] = {uint64_t(K), uint64_t(rows)};
    const uint64_t strides[1] = {uint64_t(ld)};
    const uint32_t box[2] = {128, uint32_t(kBM)};
    return encode_map(m, base, 2, dims, strides, box, MAP_U8);
}

// 3D E4M3 weight view [E][rows][cols] (strides in bytes), box (128 cols, box_rows rows, 1 expert)
bool map_u8_weight(CUtensorMap* m, const void* data, const moe_wview& v, int64_t E, int64_t rows, int64_t cols,
                   uint32_t box_rows) {
    const uint64_t dims[3] = {uint64_t(cols), uint64_t(rows), uint64_t(E)};
    const uint64_t strides[2] = {uint64_t(v.row_stride), uint64_t(v.expert_stride)};
    const uint32_t box[3] = {128, box_rows, 1};
    return encode_map(m, data, 3, dims, strides, box, MAP_U8);
}

bool check_mg(const moe_main_grads* m, bool shared) {
    if (!m) return false;
    if (m->dtype != MOE_G_FP32 && m->dtype != MOE_G_BF16) return false;
    const int64_t q = m->dtype == MOE_G_BF16 ? 8 : 4;  // elements per 16 bytes
    void* const p[6] = {m->shared_gate, m->shared_up, m->shared_down, m->routed_gate, m->routed_up, m->routed_down};
    for (int i = 0; i < 6; ++i) {
        if (i < 3 && !shared) continue;                  // no shared expert: ignored
        if (m->strides[i][1] % q || m->strides[i][1] <= 0) return false;
        if (i >= 3 && m->expert_ptrs[i - 3]) continue;  // per-expert table: checked as it is encoded
        if (!p[i] || !aligned16(p[i])) return false;
        if (i >= 3 && (m->strides[i][0] % q || m->strides[i][0] <= 0)) return false;
    }
    return true;
}

// 2D K-major operand: rows x K bf16 matrix, box 64 x 128 rows
bool map_kmajor(CUtensorMap* m, const void* base, int64_t rows, int64_t K, int64_t ld) {
    const uint64_t dims[2] = {uint64_t(K), uint64_t(rows)};
    const uint64_t strides[1] = {uint64_t(ld) * 2};
    const uint32_t box[2] = {64, uint32_t(kBM)};
    return encode_map(m, base, 2, dims, strides, box);
}

// 2D M/N-major operand: K-rows x MN bf16 matrix (MN contiguous), box 64 x 64
bool map_mnmajor(CUtensorMap* m, const void* base, int64_t rows, int64_t mn, int64_t ld) {
    const uint64_t dims[2] = {uint64_t(mn), uint64_t(rows)};
    const uint64_t strides[1] = {uint64_t(ld) * 2};
    const uint32_t box[2] = {64, 64};
    return encode_map(m, base, 2, dims, strides, box);
}

// 3D main_grad view [E][rows][cols] (expert stride es, row stride rs, elements)
// as a TMA load and store map with 128-byte box rows: 32 fp32 or 64 bf16
// columns x 32 rows
bool map_main_grad(CUtensorMap* m, void* base, int64_t E, int64_t rows, int64_t cols, int64_t es, int64_t rs,
                   bool bf16) {
    if (E <= 1) es = rows * rs;
    const uint64_t eb = bf16 ? 2 : 4;
    const uint64_t dims[3] = {uint64_t(cols), uint64_t(rows), uint64_t(E)};
    const uint64_t strides[2] = {uint64_t(rs) * eb, uint64_t(es) * eb};
    const uint32_t box[3] = {bf16 ? 64u : 32u, 32, 1};
    return encode_map(m, base, 3, dims, strides, box, bf16 ? MAP_BF16 : MAP_F32);
}

// 3D weight view [E][rows][cols] with a box of (64 cols, box_rows rows, 1 expert)
bool map_weight(CUtensorMap* m, const moe_wview& v, int64_t E, int64_t rows, int64_t cols, uint32_t box_cols,
                uint32_t box_rows) {
    const int64_t es = E > 1 ? v.expert_stride : rows * v.row_stride;
    const uint64_t dims[3] = {uint64_t(cols), uint64_t(rows), uint64_t(E)};
    const uint64_t strides[2] = {uint64_t(v.row_stride) * 2, uint64_t(es) * 2};
    const uint32_t box[3] = {box_cols, box_rows, 1};
    return encode_map(m, v.data, 3, dims, strides, box);
}

// Without a shared expert the grouped BF16 GEMMs keep their group 0 empty (no
// tiles, an empty K range): its weight and main_grad descriptors are encoded
// but never used, so they are pointed at any 16-byte aligned device memory.
moe_wview unused_view(const void* any16, const Shape& s) {
    moe_wview v;
    std::memset(&v, 0, sizeof(v));
    v.data = any16;
    v.row_stride = std::max(s.H, s.I);
    return v;
}

void set_unused_shared_main_grads(moe_main_grads* mg, void* any16, const Shape& s) {
    mg->shared_gate = mg->shared_up = mg->shared_down = any16;
    for (int i = 0; i < 3; ++i) {
        mg->strides[i][0] = 0;
        mg->strides[i][1] = std::max(s.H, s.I);
    }
}

GemmArgs base_args(int* status, const Shape& s) {
    GemmArgs a;
    std::memset(&a, 0, sizeof(a));
    a.rows_valid = INT_MAX;
    a.m_split = INT_MAX;
    a.inter = int(s.I);
    a.swiglu_limit = s.limit;
    a.status = status;
    return a;
}

int grid_of(int64_t tiles, int sms) { return int(tiles < sms ? tiles : sms); }

// Row tiles of the routed GEMMs (gate/up, down, dgrad-down, dgrad through gate/up):
// a group's rows past its last 64-row block that holds a valid row are padding that
// nothing reads -- the weight gradients' K ranges end at that block, the combine,
// the un-permute and the dprob scatter read valid rows only -- so the epilogues store
// (and the dgrad-down loads) rows below that bound only. start: each group's first
// row; rows: each routed group's valid rows; g0_rows: group 0's when it is the shared
// expert (group0_shared).
void set_row_limits(GemmArgs& a, const int* start, const int* rows, int g0_rows) {
    a.seg_off = start;
    a.seg_rows = rows;
    a.g0_rows = g0_rows;
}

// Gate/up epilogue outputs: a (hi terms; with fp32 activations also the lo terms,
// where a_lo is given) and [g|u] (bf16, or fp32 with fp32 activations).
void set_gu_outputs(const Shape& s, GemmArgs& a, __nv_bfloat16* a_hi, __nv_bfloat16* a_lo, __nv_bfloat16* gu,
                    float* gu32) {
    a.out0 = a_hi;
    a.ld_out0 = s.I;
    if (s.act32) {
        a.outf = gu32;
        a.ld_outf = 2 * s.I;
        a.out0lo = a_lo;
        a.ld_out0lo = s.I;
    } else {
        a.outh = gu;
        a.ld_outh = 2 * s.I;
    }
}

// Down / dgrad-gate-up epilogue output rows of width H: y or dx
void set_row_output(const Shape& s, GemmArgs& a, __nv_bfloat16* bf, float* f32) {
    if (s.act32) {
        a.outf = f32;
        a.ld_outf = s.H;
    } else {
        a.outh = bf;
        a.ld_outh = s.H;
    }
}

// Dgrad-down epilogue: its inputs (bf16 a and [g|u], or fp32 [g|u]) and outputs
// ([dg|du] and, where ap is given, scale * a; each with lo terms under fp32 activations)
void set_bwd_down_io(const Shape& s, GemmArgs& a, const __nv_bfloat16* a_in, const __nv_bfloat16* gu,
                     const float* gu32, __nv_bfloat16* dgdu, __nv_bfloat16* dgdu_lo, __nv_bfloat16* ap,
                     __nv_bfloat16* ap_lo) {
    if (s.act32) {
        a.inf = gu32;
        a.ld_inf = 2 * s.I;
        a.out0lo = dgdu_lo;
        a.ld_out0lo = 2 * s.I;
        a.out1lo = ap ? ap_lo : nullptr;
        a.ld_out1lo = s.I;
    } else {
        a.in0 = a_in;
        a.ld_in0 = s.I;
        a.inh = gu;
        a.ld_inh = 2 * s.I;
    }
    a.out0 = dgdu;
    a.ld_out0 = 2 * s.I;
    a.out1 = ap;
    a.ld_out1 = s.I;
}

}  // namespace

struct moe_handle {
    moe_config cfg;
    Shape s;
    Workspace ws;
    int device;
    int sms;
    bool weights_prepared = false;  // MXFP8: moe_prepare_weights has run
    // host copies of the per-expert descriptor tables last uploaded to ws.tabs
    struct Table {
        bool valid = false;
        std::array<int64_t, 4> key{};        // what else the descriptors encode (strides, box, dtype)
        std::vector<const void*> ptrs;
        std::vector<CUtensorMap> maps;
    };
    Table tables[kTables];
    std::vector<const uint8_t*> sf_src_host;  // MXFP8: the scale pointers last uploaded to ws.sf_src
    // per-kernel timing (moe_profile_enable, moe_profile_select)
    bool profiling = false;
    uint32_t profile_mask = ~0u;  // kernel classes bracketed by events
    struct Rec {
        int cls;
        cudaEvent_t start, stop;
    };
    std::vector<Rec> recs;        // recorded, not yet read
    std::vector<cudaEvent_t> pool;  // free events
};

namespace {

cudaEvent_t take_event(moe_handle* h) {
    if (!h->pool.empty()) {
        cudaEvent_t e = h->pool.back();
        h->pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Per-expert descriptor table `id`: encodes one descriptor per routed expert
// with enc(map, expert pointer) when the pointers or `key` (what else the
// descriptors encode) changed since the last upload, and uploads them into the
// workspace; *tab = their device address, *first = expert 0's descriptor (a
// valid map for the kernel's own map parameter).
template <class Enc>
moe_status expert_table(moe_handle* h, int id, const void* const* ptrs, const std::array<int64_t, 4>& key, Enc enc,
                        cudaStream_t st, const CUtensorMap** tab, CUtensorMap* first) {
    moe_handle::Table& tb = h->tables[id];
    const int64_t E = h->s.E;
    CUtensorMap* dev = h->ws.tabs + size_t(id) * size_t(E);
    if (!(tb.valid && tb.key == key && std::equal(ptrs, ptrs + E, tb.ptrs.begin()))) {
        tb.valid = false;
        tb.ptrs.assign(ptrs, ptrs + E);
        tb.maps.resize(size_t(E));
        for (int64_t e = 0; e < E; ++e)
            if (!ptrs[e] || (reinterpret_cast<uintptr_t>(ptrs[e]) & 15) || !enc(&tb.maps[size_t(e)], ptrs[e]))
                return MOE_ERR_INVALID_ARG;
        // pageable source: the copy is staged before the call returns, so the host copy may change later
        if (cudaMemcpyAsync(dev, tb.maps.data(), size_t(E) * sizeof(CUtensorMap), cudaMemcpyHostToDevice, st) !=
            cudaSuccess)
            return MOE_ERR_CUDA;
        tb.key = key;
        tb.valid = true;
    }
    *tab = dev;
    *first = tb.maps[0];
    return MOE_OK;
}

// B-operand map of a routed BF16 weight view: the 3D map over all experts, or,
// for a per-expert table, expert descriptors (box of 64 columns x box_rows rows)
moe_status routed_map(moe_handle* h, int id, const moe_wview& v, int64_t rows, int64_t cols, uint32_t box_rows,
                      cudaStream_t st, CUtensorMap* m, const CUtensorMap** tab) {
    *tab = nullptr;
    if (!v.expert_ptrs)
        return map_weight(m, v, h->s.E, rows, cols, 64, box_rows) ? MOE_OK : MOE_ERR_INVALID_ARG;
    return expert_table(
        h, id, v.expert_ptrs, {v.row_stride, rows, cols, int64_t(box_rows)},
        [&](CUtensorMap* mm, const void* p) {
            moe_wview one = v;
            one.data = p;
            return map_weight(mm, one, 1, rows, cols, 64, box_rows);
        },
        st, tab, m);
}

// B-operand map of a routed MXFP8 payload (rowwise, or columnwise with col): the
// 3D map over all experts, or, for a per-expert table (expert_ptrs holds the
// rowwise payloads at [0, E) and the columnwise ones at [E, 2E)), expert
// descriptors; box of 128 columns x box_rows rows
moe_status routed_map_u8(moe_handle* h, int id, const moe_wview& v, bool col, int64_t rows, int64_t cols,
                         uint32_t box_rows, cudaStream_t st, CUtensorMap* m, const CUtensorMap** tab) {
    *tab = nullptr;
    if (!v.expert_ptrs)
        return map_u8_weight(m, col ? v.col_data : v.data, v, h->s.E, rows, cols, box_rows) ? MOE_OK
                                                                                           : MOE_ERR_INVALID_ARG;
    return expert_table(
        h, id, v.expert_ptrs + (col ? h->s.E : 0), {v.row_stride, rows, cols, int64_t(box_rows) + (col ? 1 << 20 : 0)},
        [&](CUtensorMap* mm, const void* p) {
            moe_wview one = v;
            one.expert_stride = rows * v.row_stride;
            return map_u8_weight(mm, p, one, 1, rows, cols, box_rows);
        },
        st, tab, m);
}

// map of a routed main_grad: the 3D map, or per-expert descriptors from a table
moe_status routed_mg_map(moe_handle* h, int id, void* base, void* const* table, int64_t rows, int64_t cols,
                         int64_t es, int64_t rs, bool bf16, cudaStream_t st, CUtensorMap* m, const CUtensorMap** tab) {
    *tab = nullptr;
    if (!table)
        return map_main_grad(m, base, h->s.E, rows, cols, es, rs, bf16) ? MOE_OK : MOE_ERR_INVALID_ARG;
    return expert_table(
        h, id, const_cast<const void* const*>(table), {rs, rows, cols, bf16 ? 1 : 0},
        [&](CUtensorMap* mm, const void* p) { return map_main_grad(mm, const_cast<void*>(p), 1, rows, cols, 0, rs, bf16); },
        st, tab, m);
}

// brackets the launches of one kernel class with events while profiling
struct Timed {
    moe_handle* h;
    int cls;
    cudaStream_t st;
    cudaEvent_t start = nullptr;
    Timed(moe_handle* h_, int cls_, cudaStream_t st_) : h(h_), cls(cls_), st(st_) {
        if (h->profiling && ((h->profile_mask >> cls) & 1u) && (start = take_event(h)) != nullptr)
            cudaEventRecord(start, st);
    }
    ~Timed() {
        if (!start) return;
        cudaEvent_t stop = take_event(h);
        if (!stop) {
            h->pool.push_back(start);
            return;
        }
        cudaEventRecord(stop, st);
        h->recs.push_back({cls, start, stop});
    }
};

const char* const kKernelNames[MOE_K_COUNT] = {
    "route_pack", "route_scan", "route_place", "gather_rows",
    "gemm_fwd_gu_routed", "gemm_fwd_gu_shared", "gemm_fwd_down_routed", "gemm_fwd_down_shared", "combine",
    "gemm_bwd_down_routed", "gemm_bwd_down_shared", "gemm_bwd_gu_routed", "gemm_bwd_gu_shared",
    "gemm_wgrad_fc1_routed", "gemm_wgrad_down_routed", "gemm_wgrad_fc1_shared", "gemm_wgrad_down_shared",
    "unpermute", "shared_gate_fwd", "shared_gate_bwd"};

}  // namespace

struct moe_saved {
    moe_handle* h;
    SavedBufs b;
    int64_t T;
    const void* hidden;
    moe_weights w;
    bool valid;
    bool gated;  // the forward had a shared output gate
    bool topk;   // the forward took top-k ids + probs: dprobs per slot [T,k]
};

extern "C" {

const char* moe_status_string(moe_status st) {
    switch (st) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
        case MOE_ERR_ROUTING: return "a routing_map row has more than topk routes";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_TIMEOUT: return "a device-side wait timed out";
        case MOE_ERR_STATE: return "invalid call order";
    }
    return "unknown status";
}

uint64_t moe_launch_count(void) { return g_launches.load(); }

moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes) {
    Shape s;
    moe_status st = check_config(cfg, &s);
    if (st != MOE_OK) return st;
    if (!bytes) return MOE_ERR_INVALID_ARG;
    Workspace w;
    *bytes = carve_workspace(s, nullptr, &w);
    return MOE_OK;
}

moe_status moe_saved_size(const moe_config* cfg, size_t* bytes) {
    Shape s;
    moe_status st = check_config(cfg, &s);
    if (st != MOE_OK) return st;
    if (!bytes) return MOE_ERR_INVALID_ARG;
    SavedBufs b;
    *bytes = carve_saved(s, nullptr, &b);
    return MOE_OK;
}

moe_status moe_create(const moe_config* cfg, void* workspace, size_t workspace_bytes, moe_handle** out) {
    if (!out) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    Shape s;
    moe_status st = check_config(cfg, &s);
    if (st != MOE_OK) return st;
    Workspace w;
    const size_t need = carve_workspace(s, nullptr, &w);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) % kAlign))
        return MOE_ERR_INVALID_ARG;
    moe_handle* h = new (std::nothrow) moe_handle;
    if (!h) return MOE_ERR_INVALID_ARG;
    h->cfg = *cfg;
    h->s = s;
    carve_workspace(s, static_cast<uint8_t*>(workspace), &h->ws);
    if (cudaGetDevice(&h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess ||
        cudaMemset(h->ws.status, 0, sizeof(int)) != cudaSuccess) {
        delete h;
        return MOE_ERR_CUDA;
    }
    *out = h;
    return MOE_OK;
}

moe_status moe_handle_config(const moe_handle* h, moe_config* cfg) {
    if (!h || !cfg) return MOE_ERR_INVALID_ARG;
    *cfg = h->cfg;
    return MOE_OK;
}

void moe_destroy(moe_handle* h) {
    if (!h) return;
    for (auto& r : h->recs) {
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.stop);
    }
    for (cudaEvent_t e : h->pool) cudaEventDestroy(e);
    delete h;
}

moe_status moe_saved_create(moe_handle* h, void* memory, size_t bytes, moe_saved** out) {
    if (!h || !out) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    SavedBufs b;
    const size_t need = carve_saved(h->s, nullptr, &b);
    if (!memory || bytes < need || (reinterpret_cast<uintptr_t>(memory) % kAlign)) return MOE_ERR_INVALID_ARG;
    moe_saved* sv = new (std::nothrow) moe_saved;
    if (!sv) return MOE_ERR_INVALID_ARG;
    std::memset(sv, 0, sizeof(*sv));
    sv->h = h;
    carve_saved(h->s, static_cast<uint8_t*>(memory), &sv->b);
    if (h->s.recompute) {
        sv->b.x_all = h->ws.x_all;
        sv->b.a_all = h->ws.a_all;
        sv->b.gu_all = h->ws.gu_all;
        sv->b.gu32 = h->ws.gu32;
        sv->b.x_q = h->ws.x_q;
        sv->b.x_sf = h->ws.x_sf;
        sv->b.a_q = h->ws.a_q;
        sv->b.a_sf = h->ws.a_sf;
    }
    *out = sv;
    return MOE_OK;
}

void moe_saved_destroy(moe_saved* s) { delete s; }

#define MOE_CU(x)                                        \
    do {                                                 \
        if ((x) != cudaSuccess) return MOE_ERR_CUDA;     \
    } while (0)

#define MOE_TRY(x)                                       \
    do {                                                 \
        const moe_status st_ = (x);                      \
        if (st_ != MOE_OK) return st_;                   \
    } while (0)

// Row placement (the routed rows; with BF16 routed weights also the shared
// expert's rows), the shared output gate's values, and the gate/up GEMMs with
// the SwiGLU epilogue: the part of the forward that a backward runs again under
// recompute_dispatch, from the saved routing, hidden and weights.
static moe_status redispatch(moe_handle* h, const moe_saved* saved, cudaStream_t st) {
    const Shape& s = h->s;
    const SavedBufs& b = saved->b;
    const Workspace& ws = h->ws;
    const moe_weights* w = &saved->w;
    const void* hidden = saved->hidden;
    const bool mx = s.mx;
    const int64_t T = saved->T;
    const int Ti = int(T), E = int(s.E), k = int(s.k), H = int(s.H), I = int(s.I);
    const int rows = int(s.rows);
    const Views v = views_of(s, b, ws, T);
    const int rows_all = v.R0 + rows;
    { Timed tm_(h, MOE_K_ROUTE_PLACE, st);
    MOE_CU(launch_route_place(b.ids, b.pp, b.rank, b.hist, b.counts, b.offs_pad, Ti, E, k, mx ? 0 : v.R0, false,
                              static_cast<const __nv_bfloat16*>(hidden), H, v.perm_src, v.pp_perm, b.row_of, v.x_perm,
                              mx ? b.x_q : nullptr, mx ? b.x_sf : nullptr, st)); }

    // shared output gate: gate[t] = sigmoid(hidden[t] . w), the shared rows' scale
    if (saved->gated) {
        Timed tm_(h, MOE_K_SHARED_GATE_FWD, st);
        MOE_CU(launch_gate_forward(static_cast<const __nv_bfloat16*>(hidden),
                                   static_cast<const __nv_bfloat16*>(w->shared_output_gate), Ti, H, b.pp_all, st));
    }
    GemmMaps m{};
    // gate/up + SwiGLU
    if (mx) {
        GemmArgs a = base_args(ws.status, s);
        if (!map_u8_kmajor(&m.a, b.x_q, rows, H, H) ||
            routed_map_u8(h, TB_FWD_GU_G, w->routed_gate, false, I, H, kMxBN / 2, st, &m.b0, &a.b0_tab) != MOE_OK ||
            routed_map_u8(h, TB_FWD_GU_U, w->routed_up, false, I, H, kMxBN / 2, st, &m.b1, &a.b1_tab) != MOE_OK)
            return MOE_ERR_INVALID_ARG;
        a.mtile_expert = b.mtile_expert;
        a.num_mtiles_dev = b.meta;
        set_row_limits(a, b.offs_pad, b.counts, 0);
        a.num_mtiles = rows / kBM;
        a.n_tiles = 2 * I / kMxBN;
        a.k_blocks = H / kMxBK;
        a.gate_up_split = I;
        // the routed down projection takes a quantised (a_q); a bf16 copy of a is read only by
        // the bf16-activation dgrad-down (the fp32 one recomputes a from g, u)
        set_gu_outputs(s, a, s.act32 ? nullptr : v.a, nullptr, v.gu, v.gu32);
        a.q_out = b.a_q;
        a.ld_q = I;
        a.q_sf = b.a_sf;
        a.q_kblocks = I / 32;
        a.sfa = b.x_sf;
        a.sfa_kgroups = H / 128;
        a.sfb = ws.sf_fc1_row;
        a.sfb_ntiles = 2 * I / 128;
        a.sfb_kgroups = H / 128;
        Timed tm_(h, MOE_K_FWD_GU_ROUTED, st);
        MOE_CU(launch_gemm_mx(OP_FWD_GU, m, a, s.mx_nh_gu, h->sms, st));
    } else {  // shared expert (group 0) and routed experts in one launch
        GemmArgs a = base_args(ws.status, s);
        const int bn = s.bn_gu;
        // the shared expert's rows are hidden itself (rows past T read as zeros)
        if (!map_kmajor(&m.a, b.x_all, rows_all, H, H) || !map_kmajor(&m.g0, hidden, Ti, H, H))
            return MOE_ERR_INVALID_ARG;
        a.g0_operand = 1;
        MOE_TRY(routed_map(h, TB_FWD_GU_G, w->routed_gate, I, H, bn / 2, st, &m.b0, &a.b0_tab));
        MOE_TRY(routed_map(h, TB_FWD_GU_U, w->routed_up, I, H, bn / 2, st, &m.b1, &a.b1_tab));
        if (!map_weight(&m.s0, w->shared_gate, 1, I, H, 64, bn / 2) ||
            !map_weight(&m.s1, w->shared_up, 1, I, H, 64, bn / 2))
            return MOE_ERR_INVALID_ARG;
        a.group0_shared = 1;
        a.mtile_expert = b.mtile_x;
        a.num_mtiles_dev = b.meta + 3;
        set_row_limits(a, b.seg_x, b.counts, s.shared ? Ti : 0);
        a.num_mtiles = rows_all / kBM;
        a.n_tiles = 2 * I / bn;
        a.k_blocks = H / kBK;
        a.gate_up_split = I;
        set_gu_outputs(s, a, b.a_all, ws.alo_all, b.gu_all, b.gu32);
        Timed tm_(h, MOE_K_FWD_GU_ROUTED, st);
        MOE_CU(launch_gemm(OP_FWD_GU, bn, m, a, grid_of(int64_t(a.num_mtiles) * a.n_tiles, h->sms), st));
    }
    if (mx && s.shared) {  // shared gate/up + SwiGLU (BF16) into the shared rows
        GemmArgs a = base_args(ws.status, s);
        const int bn = s.bn_gu;
        if (!map_kmajor(&m.a, hidden, Ti, H, H) || !map_weight(&m.b0, w->shared_gate, 1, I, H, 64, bn / 2) ||
            !map_weight(&m.b1, w->shared_up, 1, I, H, 64, bn / 2))
            return MOE_ERR_INVALID_ARG;
        a.num_mtiles = (Ti + kBM - 1) / kBM;
        a.n_tiles = 2 * I / bn;
        a.k_blocks = H / kBK;
        a.rows_valid = Ti;
        a.gate_up_split = I;
        set_gu_outputs(s, a, b.a_all, ws.alo_all, b.gu_all, b.gu32);
        Timed tm_(h, MOE_K_FWD_GU_SHARED, st);
        MOE_CU(launch_gemm(OP_FWD_GU, bn, m, a, grid_of(int64_t(a.num_mtiles) * a.n_tiles, h->sms), st));
    }
    return MOE_OK;
}

// the forward from the dense routing map + probs, or (topk_ids set) from the
// router's top-k ids + probs
static moe_status forward_impl(moe_handle* h, int64_t T, const void* hidden, const float* probs,
                               const uint8_t* routing_map, const int32_t* topk_ids, const float* topk_probs,
                               const moe_weights* w, void* out, moe_saved* saved, void* stream) {
    if (!h || !saved || saved->h != h) return MOE_ERR_INVALID_ARG;
    const Shape& s = h->s;
    if (T < 0 || T > s.Tmax) return MOE_ERR_INVALID_ARG;
    if (!check_weights(s, w)) return MOE_ERR_INVALID_ARG;
    const bool topk = topk_ids != nullptr;
    if (T > 0 && (!hidden || !out || !aligned16(hidden) || !aligned16(out))) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (topk ? !topk_probs : (!probs || !routing_map))) return MOE_ERR_INVALID_ARG;
    const bool mx = s.mx;
    if (mx && !h->weights_prepared) return MOE_ERR_STATE;
    const bool gated = w->shared_output_gate != nullptr;
    if (gated && (!aligned16(w->shared_output_gate) || !s.shared)) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const SavedBufs& b = saved->b;
    const Workspace& ws = h->ws;
    saved->T = T;
    saved->hidden = hidden;
    saved->w = *w;
    if (!s.shared && T > 0) {
        const moe_wview u = unused_view(hidden, s);
        saved->w.shared_gate = saved->w.shared_up = saved->w.shared_down = u;
    }
    w = &saved->w;
    saved->valid = true;
    saved->gated = gated;
    saved->topk = topk;
    if (T == 0) return MOE_OK;

    const int Ti = int(T), E = int(s.E), k = int(s.k), H = int(s.H), I = int(s.I);
    const int rows = int(s.rows);
    const Views v = views_of(s, b, ws, T);
    const int rows_all = v.R0 + rows;  // rows of the shared-first grouped GEMMs (BF16 routed weights)

    // dispatch: route-pack, per-expert ranks, segment scan, placement + row gather
    // (with BF16 routed weights also the shared expert's rows, as group 0 of the GEMMs)
    { Timed tm_(h, MOE_K_ROUTE_PACK, st);
    MOE_CU(launch_route_pack_rank(routing_map, probs, topk_ids, topk_probs, Ti, E, k, b.ids, b.pp, b.row_of, b.rank,
                                  b.hist, ws.status, st)); }
    { Timed tm_(h, MOE_K_ROUTE_SCAN, st);
    MOE_CU(launch_route_scan_chunks(b.hist, Ti, E, b.counts, b.offsets, b.offs_pad, b.mtile_expert, b.meta,
                                    v.R0 / kBM, b.mtile_x, b.seg_x, st)); }
    MOE_TRY(redispatch(h, saved, st));
    GemmMaps m{};
    // down projection (y in bf16; the combine weights it by the route's prob or the gate)
    if (mx) {
        GemmArgs a = base_args(ws.status, s);
        if (!map_u8_kmajor(&m.a, b.a_q, rows, I, I) ||
            routed_map_u8(h, TB_FWD_DOWN, w->routed_down, false, H, I, kMxBN, st, &m.b0, &a.b0_tab) != MOE_OK)
            return MOE_ERR_INVALID_ARG;
        m.b1 = m.b0;
        a.mtile_expert = b.mtile_expert;
        a.num_mtiles_dev = b.meta;
        set_row_limits(a, b.offs_pad, b.counts, 0);
        a.num_mtiles = rows / kBM;
        a.n_tiles = H / kMxBN;
        a.k_blocks = I / kMxBK;
        set_row_output(s, a, v.yx, v.yx32);
        a.sfa = b.a_sf;
        a.sfa_kgroups = I / 128;
        a.sfb = ws.sf_down_row;
        a.sfb_ntiles = H / 128;
        a.sfb_kgroups = I / 128;
        Timed tm_(h, MOE_K_FWD_DOWN_ROUTED, st);
        MOE_CU(launch_gemm_mx(OP_FWD_DOWN, m, a, s.mx_nh_down, h->sms, st));
    } else {
        GemmArgs a = base_args(ws.status, s);
        const int bn = s.bn_down;
        if (!map_kmajor(&m.a, b.a_all, rows_all, I, I)) return MOE_ERR_INVALID_ARG;
        if (s.act32) {  // a as hi + lo terms
            if (!map_kmajor(&m.lo, ws.alo_all, rows_all, I, I)) return MOE_ERR_INVALID_ARG;
            a.split = 1;
        }
        MOE_TRY(routed_map(h, TB_FWD_DOWN, w->routed_down, H, I, bn, st, &m.b0, &a.b0_tab));
        if (!map_weight(&m.s0, w->shared_down, 1, H, I, 64, bn)) return MOE_ERR_INVALID_ARG;
        m.b1 = m.b0;
        m.s1 = m.s0;
        a.group0_shared = 1;
        a.mtile_expert = b.mtile_x;
        a.num_mtiles_dev = b.meta + 3;
        set_row_limits(a, b.seg_x, b.counts, s.shared ? Ti : 0);
        a.num_mtiles = rows_all / kBM;
        a.n_tiles = H / bn;
        a.k_blocks = I / kBK;
        set_row_output(s, a, ws.yx_all, ws.yx32);
        Timed tm_(h, MOE_K_FWD_DOWN_ROUTED, st);
        MOE_CU(launch_gemm(OP_FWD_DOWN, bn, m, a, grid_of(int64_t(a.num_mtiles) * a.n_tiles, h->sms), st));
    }
    if (mx && s.shared) {  // shared down projection (BF16)
        GemmArgs a = base_args(ws.status, s);
        const int bn = s.bn_down;
        if (!map_kmajor(&m.a, b.a_all, Ti, I, I) || !map_weight(&m.b0, w->shared_down, 1, H, I, 64, bn))
            return MOE_ERR_INVALID_ARG;
        if (s.act32) {
            if (!map_kmajor(&m.lo, ws.alo_all, Ti, I, I)) return MOE_ERR_INVALID_ARG;
            a.split = 1;
        }
        m.b1 = m.b0;
        a.num_mtiles = (Ti + kBM - 1) / kBM;
        a.n_tiles = H / bn;
        a.k_blocks = I / kBK;
        a.rows_valid = Ti;
        set_row_output(s, a, ws.yx_all, ws.yx32);
        Timed tm_(h, MOE_K_FWD_DOWN_SHARED, st);
        MOE_CU(launch_gemm(OP_FWD_DOWN, bn, m, a, grid_of(int64_t(a.num_mtiles) * a.n_tiles, h->sms), st));
    }
    // combine
    Timed tm_(h, MOE_K_COMBINE, st);
    const void* ys = s.shared ? (s.act32 ? static_cast<const void*>(ws.yx32) : ws.yx_all) : nullptr;
    MOE_CU(launch_combine(ys, gated ? b.pp_all : nullptr,
                          s.act32 ? static_cast<const void*>(v.yx32) : v.yx, s.act32, b.row_of, b.pp, Ti, H, k,
                          static_cast<__nv_bfloat16*>(out), h->sms, st));
    return MOE_OK;
}

moe_status moe_forward(moe_handle* h, int64_t T, const void* hidden, const float* probs, const uint8_t* routing_map,
                       const moe_weights* w, void* out, moe_saved* saved, void* stream) {
    return forward_impl(h, T, hidden, probs, routing_map, nullptr, nullptr, w, out, saved, stream);
}

moe_status moe_forward_topk(moe_handle* h, int64_t T, const void* hidden, const int32_t* topk_ids,
                            const float* topk_probs, const moe_weights* w, void* out, moe_saved* saved,
                            void* stream) {
    if (T > 0 && !topk_ids) return MOE_ERR_INVALID_ARG;
    static const int32_t kNone = -1;  // any non-null marker selects the top-k input when T == 0
    return forward_impl(h, T, hidden, nullptr, nullptr, T > 0 ? topk_ids : &kNone, topk_probs, w, out, saved,
                        stream);
}

moe_status moe_backward(moe_handle* h, const void* grad_out, const moe_saved* saved, void* dhidden, float* dprobs,
                        const moe_main_grads* mg, void* stream) {
    if (!h || !saved || saved->h != h) return MOE_ERR_INVALID_ARG;
    if (!saved->valid) return MOE_ERR_STATE;
    if (!check_mg(mg, h->s.shared)) return MOE_ERR_INVALID_ARG;
    const bool gated = saved->gated;
    if (gated && (!mg->shared_output_gate || !aligned16(mg->shared_output_gate))) return MOE_ERR_INVALID_ARG;
    const bool mg_bf16 = mg->dtype == MOE_G_BF16;
    const Shape& s = h->s;
    const int64_t T = saved->T;
    if (T == 0) return MOE_OK;
    if (!grad_out || !dhidden || !dprobs || !aligned16(grad_out) || !aligned16(dhidden)) return MOE_ERR_INVALID_ARG;
    const bool mx = s.mx;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const SavedBufs& b = saved->b;
    const Workspace& ws = h->ws;
    const moe_weights* w = &saved->w;
    const int Ti = int(T), E = int(s.E), k = int(s.k), H = int(s.H), I = int(s.I);
    const int rows = int(s.rows);
    const Views v = views_of(s, b, ws, T);
    const int rows_all = v.R0 + rows;
    const __nv_bfloat16* go = static_cast<const __nv_bfloat16*>(grad_out);
    moe_main_grads mg_local = *mg;  // without a shared expert: its (ignored) buffers point at the workspace
    if (!s.shared) set_unused_shared_main_grads(&mg_local, ws.go_all, s);
    mg = &mg_local;

    // the weight-gradient launches claim their tiles from these counters
    MOE_CU(cudaMemsetAsync(ws.tile_counters, 0, 4 * sizeof(int), st));
    if (mx && v.R0 > Ti) {
        // the shared expert's separate dgrad-down launch writes rows [0, T); the grouped
        // weight gradients read its region up to R0, so the rows past T hold zeros
        const size_t tail = size_t(v.R0 - Ti);
        MOE_CU(cudaMemsetAsync(ws.dgdu_all + size_t(Ti) * 2 * I, 0, tail * 2 * I * sizeof(__nv_bfloat16), st));
        MOE_CU(cudaMemsetAsync(ws.ap_all + size_t(Ti) * I, 0, tail * I * sizeof(__nv_bfloat16), st));
        if (s.act32) {
            MOE_CU(cudaMemsetAsync(ws.dgdulo_all + size_t(Ti) * 2 * I, 0, tail * 2 * I * sizeof(__nv_bfloat16), st));
            MOE_CU(cudaMemsetAsync(ws.aplo_all + size_t(Ti) * I, 0, tail * I * sizeof(__nv_bfloat16), st));
        }
    }
    // recompute_dispatch: the rows, the gate values and a, [g|u] again, into the workspace
    if (s.recompute) MOE_TRY(redispatch(h, saved, st));
    { Timed tm_(h, MOE_K_GATHER, st);
    // routed rows only: the GEMMs read the shared expert's rows from grad_out itself
    MOE_CU(launch_gather_rows(go, b.row_of, b.counts, b.offs_pad, Ti, E, k, H, v.go_perm, mx ? ws.go_q : nullptr,
                              mx ? ws.go_sf : nullptr, st)); }

    GemmMaps m{};
    // dgrad through the down projection + SwiGLU backward + dprob partials
    if (mx) {
        GemmArgs a = base_args(ws.status, s);
        if (!map_u8_kmajor(&m.a, ws.go_q, rows, H, H) ||
            routed_map_u8(h, TB_BWD_DOWN, w->routed_down, true, H, I, 128, st, &m.b0, &a.b0_tab) != MOE_OK)
            return MOE_ERR_INVALID_ARG;
        m.b1 = m.b0;
        a.mtile_expert = b.mtile_expert;
        a.num_mtiles_dev = b.meta;
        set_row_limits(a, b.offs_pad, b.counts, 0);
        a.num_mtiles = rows / kBM;
        a.n_tiles = I / kMxBN;
        a.k_blocks = H / kMxBK;
        set_bwd_down_io(s, a, v.a, v.gu, v.gu32, v.dgdu, v.dgdulo, v.ap, v.aplo);
        a.row_scale = v.pp_perm;
        a.partial = v.partial;
        a.q_out = ws.dgdu_q;
        a.ld_q = 2 * I;
        a.q_sf = ws.dgdu_sf;
        a.q_kblocks = 2 * I / 32;
        a.sfa = ws.go_sf;
        a.sfa_kgroups = H / 128;
        a.sfb = ws.sf_down_col;
        a.sfb_ntiles = I / 128;
        a.sfb_kgroups = H / 128;
        a.deep_stages = s.H >= 4096 ? 1 : 0;  // five stages with a long K (H = 7168: 1.88 -> 1.67 ms)
        Timed tm_(h, MOE_K_BWD_DOWN_ROUTED, st);
        MOE_CU(launch_gemm_mx(OP_BWD_DOWN, m, a, 1, h->sms, st));
    } else {  // shared expert (group 0: its rows' scale is the gate, or 1) and routed experts
        GemmArgs a = base_args(ws.status, s);
        const int bn = s.bn_bd;
        if (!map_kmajor(&m.a, ws.go_all, rows_all, H, H) || !map_kmajor(&m.g0, go, Ti, H, H))
            return MOE_ERR_INVALID_ARG;
        a.g0_operand = 1;
        MOE_TRY(routed_map(h, TB_BWD_DOWN, w->routed_down, H, I, 64, st, &m.b0, &a.b0_tab));
        if (!map_weight(&m.s0, w->shared_down, 1, H, I, 64, 64)) return MOE_ERR_INVALID_ARG;
        m.b1 = m.b0;
        m.s1 = m.s0;
        a.group0_shared = 1;
        a.mtile_expert = b.mtile_x;
        a.num_mtiles_dev = b.meta + 3;
        set_row_limits(a, b.seg_x, b.counts, s.shared ? Ti : 0);
        a.num_mtiles = rows_all / kBM;
        a.n_tiles = I / bn;
        a.k_blocks = H / kBK;
        set_bwd_down_io(s, a, b.a_all, b.gu_all, b.gu32, ws.dgdu_all, ws.dgdulo_all, ws.ap_all, ws.aplo_all);
        a.row_scale = b.pp_all;
        a.partial = ws.partial_all;
        // four stages with a long K (H = 4096, I = 1536: 1.77 -> 1.63 ms); at H = 2048 three stay
        // faster (229 against 237 us)
        a.deep_stages = s.H >= 4096 ? 1 : 0;
        Timed tm_(h, MOE_K_BWD_DOWN_ROUTED, st);
        MOE_CU(launch_gemm(OP_BWD_DOWN, bn, m, a, grid_of(int64_t(a.num_mtiles) * a.n_tiles, h->sms), st));
    }
    if (mx && s.shared) {  // shared dgrad through the down projection + SwiGLU backward (BF16)
        GemmArgs a = base_args(ws.status, s);
        const int bn = s.bn_bd;
        if (!map_kmajor(&m.a, go, Ti, H, H) || !map_weight(&m.b0, w->shared_down, 1, H, I, 64, 64))
            return MOE_ERR_INVALID_ARG;
        m.b1 = m.b0;
        a.num_mtiles = (Ti + kBM - 1) / kBM;
        a.n_tiles = I / bn;
        a.k_blocks = H / kBK;
        a.rows_valid = Ti;
        // (gate *) a for the down projection's weight gradient (its shared rows)
        set_bwd_down_io(s, a, b.a_all, b.gu_all, b.gu32, ws.dgdu_all, ws.dgdulo_all, ws.ap_all, ws.aplo_all);
        if (gated) {  // the gate acts as the shared rows' prob: dgate partials, gate * a_shared
            a.row_scale = b.pp_all;
            a.partial = ws.partial_s;
        }
        a.deep_stages = s.H >= 4096 ? 1 : 0;
        Timed tm_(h, MOE_K_BWD_DOWN_SHARED, st);
        MOE_CU(launch_gemm(OP_BWD_DOWN, bn, m, a, grid_of(int64_t(a.num_mtiles) * a.n_tiles, h->sms), st));
    }
    if (gated) {
        Timed tm_(h, MOE_K_SHARED_GATE_BWD, st);
        MOE_CU(launch_gate_backward(static_cast<const __nv_bfloat16*>(saved->hidden), b.pp_all,
                                    mx ? ws.partial_s : ws.partial_all, mx ? s.n_part_s : s.n_part, Ti, H, ws.dz,
                                    ws.gpart, mg->shared_output_gate, mg_bf16, st));
    }
    // dgrad through gate/up
    if (mx) {
        GemmArgs a = base_args(ws.status, s);
        if (!map_u8_kmajor(&m.a, ws.dgdu_q, rows, 2 * I, 2 * I) ||
            routed_map_u8(h, TB_BWD_GU_G, w->routed_gate, true, I, H, 128, st, &m.b0, &a.b0_tab) != MOE_OK ||
            routed_map_u8(h, TB_BWD_GU_U, w->routed_up, true, I, H, 128, st, &m.b1, &a.b1_tab) != MOE_OK)
            return MOE_ERR_INVALID_ARG;
        a.mtile_expert = b.mtile_expert;
        a.num_mtiles_dev = b.meta;
        set_row_limits(a, b.offs_pad, b.counts, 0);
        a.num_mtiles = rows / kBM;
        a.n_tiles = H / kMxBN;
        a.k_blocks = 2 * I / kMxBK;
        a.gate_up_split = I;
        set_row_output(s, a, v.yx, v.yx32);
        a.sfa = ws.dgdu_sf;
        a.sfa_kgroups = 2 * I / 128;
        a.sfb = ws.sf_fc1_col;
        a.sfb_ntiles = H / 128;
        a.sfb_kgroups = 2 * I / 128;
        Timed tm_(h, MOE_K_BWD_GU_ROUTED, st);
        MOE_CU(launch_gemm_mx(OP_BWD_GU, m, a, s.mx_nh_bgu, h->sms, st));
    } else {
        GemmArgs a = base_args(ws.status, s);
        const int bn = s.bn_bgu;
        if (!map_kmajor(&m.a, ws.dgdu_all, rows_all, 2 * I, 2 * I)) return MOE_ERR_INVALID_ARG;
        if (s.act32) {  // [dg|du] as hi + lo terms
            if (!map_kmajor(&m.lo, ws.dgdulo_all, rows_all, 2 * I, 2 * I)) return MOE_ERR_INVALID_ARG;
            a.split = 1;
        }
        MOE_TRY(routed_map(h, TB_BWD_GU_G, w->routed_gate, I, H, 64, st, &m.b0, &a.b0_tab));
        MOE_TRY(routed_map(h, TB_BWD_GU_U, w->routed_up, I, H, 64, st, &m.b1, &a.b1_tab));
        if (!map_weight(&m.s0, w->shared_gate, 1, I, H, 64, 64) || !map_weight(&m.s1, w->shared_up, 1, I, H, 64, 64))
            return MOE_ERR_INVALID_ARG;
        a.group0_shared = 1;
        a.mtile_expert = b.mtile_x;
        a.num_mtiles_dev = b.meta + 3;
        set_row_limits(a, b.seg_x, b.counts, s.shared ? Ti : 0);
        a.num_mtiles = rows_all / kBM;
        a.n_tiles = H / bn;
        a.k_blocks = 2 * I / kBK;
        a.gate_up_split = I;
        set_row_output(s, a, ws.yx_all, ws.yx32);
        Timed tm_(h, MOE_K_BWD_GU_ROUTED, st);
        MOE_CU(launch_gemm(OP_BWD_GU, bn, m, a, grid_of(int64_t(a.num_mtiles) * a.n_tiles, h->sms), st));
    }
    if (mx && s.shared) {  // shared dgrad through gate/up (BF16)
        GemmArgs a = base_args(ws.status, s);
        const int bn = s.bn_bgu;
        if (!map_kmajor(&m.a, ws.dgdu_all, Ti, 2 * I, 2 * I) || !map_weight(&m.b0, w->shared_gate, 1, I, H, 64, 64) ||
            !map_weight(&m.b1, w->shared_up, 1, I, H, 64, 64))
            return MOE_ERR_INVALID_ARG;
        if (s.act32) {
            if (!map_kmajor(&m.lo, ws.dgdulo_all, Ti, 2 * I, 2 * I)) return MOE_ERR_INVALID_ARG;
            a.split = 1;
        }
        a.num_mtiles = (Ti + kBM - 1) / kBM;
        a.n_tiles = H / bn;
        a.k_blocks = 2 * I / kBK;
        a.rows_valid = Ti;
        a.gate_up_split = I;
        set_row_output(s, a, ws.yx_all, ws.yx32);
        Timed tm_(h, MOE_K_BWD_GU_SHARED, st);
        MOE_CU(launch_gemm(OP_BWD_GU, bn, m, a, grid_of(int64_t(a.num_mtiles) * a.n_tiles, h->sms), st));
    }
    // wgrad of gate/up: main_grad[e] += [dg|du]_e^T X_e, the shared expert as group 0
    // (its long K range is claimed first); both weight gradients are BF16 GEMMs with
    // either routed weight type
    {
        GemmArgs a = base_args(ws.status, s);
        const int bn = s.bn_wfc1;
        a.m_tiles = 2 * I / kBM;
        a.n_tiles = H / bn;
        a.m_split = I;
        a.mg_bf16 = mg_bf16;
        a.tile_counter = ws.tile_counters + 0;
        MOE_TRY(routed_mg_map(h, TB_MG_G, mg->routed_gate, mg->expert_ptrs[0], I, H, mg->strides[3][0],
                              mg->strides[3][1], mg_bf16, st, &m.c0, &a.c0_tab));
        MOE_TRY(routed_mg_map(h, TB_MG_U, mg->routed_up, mg->expert_ptrs[1], I, H, mg->strides[4][0],
                              mg->strides[4][1], mg_bf16, st, &m.c1, &a.c1_tab));
        if (s.act32) {  // [dg|du] as hi + lo terms
            if (!map_mnmajor(&m.lo, ws.dgdulo_all, rows_all, 2 * I, 2 * I)) return MOE_ERR_INVALID_ARG;
            a.split = 1;
            // with ~512 or more rows per expert a tile's mainloop outlasts its main_grad
            // read-add-store: a third operand stage beats the second box buffer
            a.deep_stages = int64_t(Ti) * k >= 512 * int64_t(E) ? 1 : 0;
        }
        // the shared expert is group 0 (its x rows: hidden), with either routed weight type
        if (!map_mnmajor(&m.a, ws.dgdu_all, rows_all, 2 * I, 2 * I) || !map_mnmajor(&m.b0, b.x_all, rows_all, H, H) ||
            !map_mnmajor(&m.g0, saved->hidden, Ti, H, H) ||
            !map_main_grad(&m.s0, mg->shared_gate, 1, I, H, 0, mg->strides[0][1], mg_bf16) ||
            !map_main_grad(&m.s1, mg->shared_up, 1, I, H, 0, mg->strides[1][1], mg_bf16))
            return MOE_ERR_INVALID_ARG;
        a.seg_off = b.seg_x;
        a.seg_rows = b.counts;
        a.g0_rows = s.shared ? Ti : 0;
        a.groups = E + 1;
        a.group0_shared = 1;
        a.g0_operand = 2;
        m.b1 = m.b0;
        Timed tm_(h, MOE_K_WGRAD_FC1_ROUTED, st);
        MOE_CU(launch_gemm(OP_WGRAD, bn, m, a, grid_of(int64_t(a.groups) * a.m_tiles * a.n_tiles, h->sms), st));
    }
    // wgrad of down: main_grad[e] += go_e^T (p a)_e. With long tiles (the deep build, fp32
    // main_grad) it runs transposed: the accumulator tile is (p a)_e^T go_e, whose split operand
    // (p a as two terms) is A, so that its lo tile is the smaller one, and the epilogue adds
    // it into main_grad's boxes transposed. (With short tiles the main_grad stream is the
    // bound and the transposed add slows it: config 2 317 -> 323 us, config 4 7.26 -> 7.88 ms.)
    const bool down_deep = int64_t(Ti) * k >= 512 * int64_t(E);
    const bool down_trans = s.act32 && !mg_bf16 && H % 256 == 0 && down_deep;
    if (down_trans) {
        GemmArgs a = base_args(ws.status, s);
        a.m_tiles = I / kBM;
        a.n_tiles = H / 256;
        a.mg_bf16 = 0;
        a.tile_counter = ws.tile_counters + 1;
        MOE_TRY(routed_mg_map(h, TB_MG_D, mg->routed_down, mg->expert_ptrs[2], H, I, mg->strides[5][0],
                              mg->strides[5][1], false, st, &m.c0, &a.c0_tab));
        if (!map_mnmajor(&m.a, ws.ap_all, rows_all, I, I) || !map_mnmajor(&m.lo, ws.aplo_all, rows_all, I, I) ||
            !map_mnmajor(&m.b0, ws.go_all, rows_all, H, H) || !map_mnmajor(&m.g0, go, Ti, H, H) ||
            !map_main_grad(&m.s0, mg->shared_down, 1, H, I, 0, mg->strides[2][1], false))
            return MOE_ERR_INVALID_ARG;
        a.split = 1;
        a.deep_stages = 1;
        a.mg_trans = 1;
        a.seg_off = b.seg_x;
        a.seg_rows = b.counts;
        a.g0_rows = s.shared ? Ti : 0;
        a.groups = E + 1;
        a.group0_shared = 1;
        a.g0_operand = 2;  // group 0's B: grad_out rows
        m.b1 = m.b0;
        m.c1 = m.c0;
        m.s1 = m.s0;
        Timed tm_(h, MOE_K_WGRAD_DOWN_ROUTED, st);
        MOE_CU(launch_gemm(OP_WGRAD, 256, m, a, grid_of(int64_t(a.groups) * a.m_tiles * a.n_tiles, h->sms), st));
    } else {
        GemmArgs a = base_args(ws.status, s);
        const int bn = s.bn_wd;
        a.m_tiles = H / kBM;
        a.n_tiles = I / bn;
        a.mg_bf16 = mg_bf16;
        a.tile_counter = ws.tile_counters + 1;
        MOE_TRY(routed_mg_map(h, TB_MG_D, mg->routed_down, mg->expert_ptrs[2], H, I, mg->strides[5][0],
                              mg->strides[5][1], mg_bf16, st, &m.c0, &a.c0_tab));
        if (s.act32) {  // p * a as hi + lo terms
            if (!map_mnmajor(&m.lo, ws.aplo_all, rows_all, I, I)) return MOE_ERR_INVALID_ARG;
            a.split = 2;
        }
        // the shared expert is group 0 (its grad_out rows: grad_out), with either routed weight type
        if (!map_mnmajor(&m.a, ws.go_all, rows_all, H, H) || !map_mnmajor(&m.b0, ws.ap_all, rows_all, I, I) ||
            !map_mnmajor(&m.g0, go, Ti, H, H) ||
            !map_main_grad(&m.s0, mg->shared_down, 1, H, I, 0, mg->strides[2][1], mg_bf16))
            return MOE_ERR_INVALID_ARG;
        a.seg_off = b.seg_x;
        a.seg_rows = b.counts;
        a.g0_rows = s.shared ? Ti : 0;
        a.groups = E + 1;
        a.group0_shared = 1;
        a.g0_operand = 1;
        m.b1 = m.b0;
        m.c1 = m.c0;
        m.s1 = m.s0;
        Timed tm_(h, MOE_K_WGRAD_DOWN_ROUTED, st);
        MOE_CU(launch_gemm(OP_WGRAD, bn, m, a, grid_of(int64_t(a.groups) * a.m_tiles * a.n_tiles, h->sms), st));
    }
    // dhidden = shared + un-permuted routed dgrad; dense dprobs
    Timed tm_(h, MOE_K_UNPERMUTE, st);
    const void* dxs = s.shared ? (s.act32 ? static_cast<const void*>(ws.yx32) : ws.yx_all) : nullptr;
    MOE_CU(launch_unpermute(dxs,
                            s.act32 ? static_cast<const void*>(v.yx32) : v.yx, s.act32, b.row_of, b.ids, v.partial,
                            s.n_part, Ti, H, k, E,
                            gated ? ws.dz : nullptr,
                            gated ? static_cast<const __nv_bfloat16*>(w->shared_output_gate) : nullptr,
                            static_cast<__nv_bfloat16*>(dhidden), dprobs, saved->topk, h->sms, st));
    return MOE_OK;
}

moe_status moe_prepare_weights(moe_handle* h, const moe_weights* w, void* stream) {
    if (!h) return MOE_ERR_INVALID_ARG;
    const Shape& s = h->s;
    if (!s.mx) return MOE_OK;
    if (!w) return MOE_ERR_INVALID_ARG;
    if (!check_weights(s, w)) return MOE_ERR_INVALID_ARG;
    const moe_wview &g = w->routed_gate, &u = w->routed_up, &d = w->routed_down;
    if (g.row_stride != u.row_stride) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int E = int(s.E), H = int(s.H), I = int(s.I);
    const Workspace& ws = h->ws;
    // every expert's rowwise and columnwise scale base, from its table entries
    // (scales at [2E, 3E) and [3E, 4E)) or from the strided view
    std::vector<const uint8_t*>& src = h->sf_src_host;
    src.assign(6 * size_t(E), nullptr);
    const moe_wview* views[3] = {&g, &u, &d};
    for (int i = 0; i < 3; ++i) {
        const moe_wview& v = *views[i];
        for (int e = 0; e < E; ++e) {
            const uint8_t* row = v.expert_ptrs ? static_cast<const uint8_t*>(v.expert_ptrs[2 * E + e])
                                               : v.scale + int64_t(e) * (v.expert_stride / 32);
            const uint8_t* colp = v.expert_ptrs ? static_cast<const uint8_t*>(v.expert_ptrs[3 * E + e])
                                                : v.col_scale + int64_t(e) * (v.expert_stride / 32);
            if (!row || !colp) return MOE_ERR_INVALID_ARG;
            src[size_t(i) * E + e] = row;              // rowwise: gate, up, down
            src[size_t(3 + (i + 1) % 3) * E + e] = colp;  // columnwise: down, gate, up
        }
    }
    // pageable source: the copy is staged before the call returns
    MOE_CU(cudaMemcpyAsync(ws.sf_src, src.data(), src.size() * sizeof(const uint8_t*), cudaMemcpyHostToDevice, st));
    const uint8_t* const* t = ws.sf_src;
    MOE_CU(launch_swizzle_scales(1 /*rows, gate|up tiles*/, t, t + E, g.row_stride / 32, E, 2 * I / 128, H / 32, 0,
                                 ws.sf_fc1_row, st));
    MOE_CU(launch_swizzle_scales(0 /*rows*/, t + 2 * E, nullptr, d.row_stride / 32, E, H / 128, I / 32, 0,
                                 ws.sf_down_row, st));
    MOE_CU(launch_swizzle_scales(2 /*columns*/, t + 3 * E, nullptr, d.row_stride, E, I / 128, H / 32, 0,
                                 ws.sf_down_col, st));
    MOE_CU(launch_swizzle_scales(3 /*columns, gate then up*/, t + 4 * E, t + 5 * E, g.row_stride, E, H / 128,
                                 2 * I / 32, I / 32, ws.sf_fc1_col, st));
    h->weights_prepared = true;
    return MOE_OK;
}

moe_status moe_export_routing(moe_handle* h, const moe_saved* saved, int32_t* ids, float* pp, int32_t* counts,
                              int32_t* offsets, int32_t* perm_src, int32_t* row_of, void* stream) {
    if (!h || !saved || saved->h != h) return MOE_ERR_INVALID_ARG;
    if (!saved->valid) return MOE_ERR_STATE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const Shape& s = h->s;
    const SavedBufs& b = saved->b;
    const int64_t T = saved->T;
    if (T == 0) {
        if (counts) MOE_CU(cudaMemsetAsync(counts, 0, s.E * sizeof(int32_t), st));
        if (offsets) MOE_CU(cudaMemsetAsync(offsets, 0, (s.E + 1) * sizeof(int32_t), st));
        return MOE_OK;
    }
    const size_t tk = size_t(T * s.k);
    if (ids) MOE_CU(cudaMemcpyAsync(ids, b.ids, tk * sizeof(int32_t), cudaMemcpyDeviceToDevice, st));
    if (pp) MOE_CU(cudaMemcpyAsync(pp, b.pp, tk * sizeof(float), cudaMemcpyDeviceToDevice, st));
    if (counts) MOE_CU(cudaMemcpyAsync(counts, b.counts, s.E * sizeof(int32_t), cudaMemcpyDeviceToDevice, st));
    if (offsets)
        MOE_CU(cudaMemcpyAsync(offsets, b.offsets, (s.E + 1) * sizeof(int32_t), cudaMemcpyDeviceToDevice, st));
    if (perm_src || row_of)
        MOE_CU(launch_export_routing(b.ids, b.row_of, views_of(s, b, h->ws, T).perm_src, b.counts, b.offsets,
                                     b.offs_pad, b.mtile_expert,
                                     b.meta, int(T), int(s.k), int(s.rows), perm_src, row_of, st));
    return MOE_OK;
}

moe_status moe_profile_select(moe_handle* h, uint32_t class_mask) {
    if (!h) return MOE_ERR_INVALID_ARG;
    h->profile_mask = class_mask;
    return MOE_OK;
}

moe_status moe_profile_enable(moe_handle* h, int enable) {
    if (!h) return MOE_ERR_INVALID_ARG;
    h->profiling = enable != 0;
    return MOE_OK;
}

moe_status moe_profile_read(moe_handle* h, double* total_ms, int64_t* launches, int n) {
    if (!h || n < 0 || n > MOE_K_COUNT || (n > 0 && (!total_ms || !launches))) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        total_ms[i] = 0.0;
        launches[i] = 0;
    }
    moe_status st = MOE_OK;
    for (auto& r : h->recs) {
        float ms = 0.0f;
        if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
            st = MOE_ERR_CUDA;
        if (r.cls < n) {
            total_ms[r.cls] += ms;
            launches[r.cls] += 1;
        }
        h->pool.push_back(r.start);
        h->pool.push_back(r.stop);
    }
    h->recs.clear();
    return st;
}

const char* moe_kernel_name(int kernel_class) {
    return (kernel_class >= 0 && kernel_class < MOE_K_COUNT) ? kKernelNames[kernel_class] : nullptr;
}

moe_status moe_selftest_timeout(moe_handle* h, void* stream) {
    if (!h) return MOE_ERR_INVALID_ARG;
    MOE_CU(moe::launch_wait_selftest(h->ws.status, static_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

moe_status moe_device_status(moe_handle* h, void* stream) {
    if (!h) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int v = 0;
    MOE_CU(cudaStreamSynchronize(st));
    MOE_CU(cudaMemcpy(&v, h->ws.status, sizeof(int), cudaMemcpyDeviceToHost));
    MOE_CU(cudaMemset(h->ws.status, 0, sizeof(int)));
    if (v & kStatusTimeout) return MOE_ERR_TIMEOUT;
    if (v & kStatusRouting) return MOE_ERR_ROUTING;
    return MOE_OK;
}

}  // extern "C"
