/*
 * moe.h -- C ABI of the GB300 (sm_103a) MoE layer library (libmoe.so).
 *
 * The library runs the post-router Mixture-of-Experts layer on one GPU,
 * forward and backward: route-pack, dispatch (a local permutation), routed
 * SwiGLU experts, the shared SwiGLU expert, prob-weighted combine; then
 * dgrad of the hidden states, router-prob gradients scattered into the dense
 * [T,E] tensor, and weight gradients accumulated into fp32 main_grad buffers.
 * Sources: "feat(moe): add a megakernel backend with MOK integration"
 * (Megatron-LM PR #6572), Summary and Design; "Add Mixture-of-Kittens MoE
 * backend on main" (PR #8210), What does this PR do; API pages
 * "core.transformer.moe.megakernel.mok.backend" (MoKMegakernel.forward) and
 * "core.transformer.moe.megakernel.mok.runtime" (_MoKWeightArguments,
 * _gate_up_weight_arguments, _gate_up_main_grad_arguments, _MoKAutograd).
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers unless a comment says otherwise;
 *    the caller owns them. Weights and main_grads are non-owning views: nothing
 *    is copied or registered (runtime page, _MoKWeightArguments).
 *  - Layouts are row-major; strides are in ELEMENTS. bf16 is passed as void*.
 *  - `stream` is a cudaStream_t passed as void*; every call is asynchronous on
 *    it and performs no host synchronisation, except moe_device_status.
 *  - Argument errors are reported synchronously, before anything is launched.
 *    Errors found by kernels (a routing row with more than k routes, a
 *    bounded wait that gave up) are recorded in a device status word that
 *    moe_device_status reads; the outputs of such a call are undefined.
 *  - The library allocates no device memory: workspace and saved-state
 *    memory come from the caller (sizes from the *_size queries).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null pointer, size out of range, misaligned view */
    MOE_ERR_UNSUPPORTED = 2,  /* a configuration the pages' backend also rejects, or a shape the kernels do not tile */
    MOE_ERR_ROUTING = 3,      /* a routing_map row has more than k routes (device-detected) */
    MOE_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    MOE_ERR_TIMEOUT = 5,      /* a bounded device-side wait gave up (device-detected) */
    MOE_ERR_STATE = 6         /* call order violated (e.g. backward without a forward into `saved`) */
} moe_status;

typedef enum { MOE_W_BF16 = 0, MOE_W_MXFP8 = 1 } moe_wtype;

/* dtype of the main_grad buffers (PR #8210 review thread on wgrad precision:
 * main_grad.dtype selects the accumulation, one dtype for all buffers). */
typedef enum { MOE_G_FP32 = 0, MOE_G_BF16 = 1 } moe_gtype;

/* Precision of the activations between an expert's GEMMs (the pages fix the
 * weights, BF16 or MXFP8, and the FP32 accumulator -- PR #6572, Supported
 * configurations; PR #8210 review thread on wgrad precision -- but not this).
 * MOE_ACT_FP32 (the default): the gate/up results g, u, the expert outputs y
 * and the expert input gradients dx stay fp32, and every GEMM operand the layer
 * derives (a = silu(g) u, [dg|du], p a) reaches the tensor cores as two bf16
 * terms hi = bf16(v), lo = bf16(v - hi) whose products add in the same fp32
 * accumulator (the GEMM runs its K range twice, once per term); results then
 * follow the layer's exact definition to within fp32 accumulation and the final
 * bf16 roundings of out and dhidden. MXFP8 routed GEMMs take their operands
 * quantised as the MXFP8 method does, unsplit. MOE_ACT_BF16: g, u, y, dx and
 * every derived operand are single bf16 values (faster: no second K pass,
 * half the bytes; each rounding adds a relative error of up to 2^-8). */
typedef enum { MOE_ACT_FP32 = 0, MOE_ACT_BF16 = 1 } moe_act;

/* Layer shape. Routed and shared experts share `inter` (PR #6572, Supported
 * configurations: MOK limitations). hidden must be a multiple of 128, inter of 64;
 * 1 <= topk <= 32; 1 <= num_experts <= 1024.
 * swiglu_limit (PR #8210 review: the backend's swiglu_limit, taken from the
 * layer's activation clamp value; the pages give no formula): 0 disables it;
 * L > 0 clamps the SwiGLU inputs of every expert, routed and shared, before
 * the activation: a = silu(min(g, L)) * min(max(u, -L), L) for g = x Wg^T,
 * u = x Wu^T. Gradients pass where the clamp is inactive, bounds included
 * (dg = 0 where g > L, du = 0 where |u| > L). Negative or non-finite values are
 * MOE_ERR_INVALID_ARG. */
typedef struct {
    int64_t max_tokens;   /* largest T any call will pass */
    int64_t hidden;       /* H */
    int64_t num_experts;  /* E, routed experts */
    int64_t topk;         /* k, fixed route width */
    int64_t inter;        /* I, intermediate size of routed and shared experts */
    int32_t routed_wtype; /* moe_wtype of the routed weights; shared weights are always bf16 */
    float swiglu_limit;   /* 0: no clamp; L > 0: SwiGLU input clamp (above) */
    int32_t recompute_dispatch; /* 0 or 1; see below */
    int32_t act_precision; /* moe_act: MOE_ACT_FP32 (0, default) or MOE_ACT_BF16 */
    int32_t no_shared_expert; /* 0 (default): the layer has the shared expert; 1: see below */
} moe_config;
/* no_shared_expert = 1: routed experts only. out[t] = sum_s pp[t,s] y[t,s],
 * dhidden the routed part alone; the shared weight views, the shared main_grad
 * buffers and the output gate are ignored (NULL is fine; an output gate is
 * MOE_ERR_INVALID_ARG). This is the owner-side step of expert parallelism
 * (PR #6572, Validation: EP16 / EP64; "core.transformer.moe.megakernel.mok.backend",
 * MoKMegakernel: ep_group): a rank that owns experts [e0, e1) runs them on the
 * token rows it received, in expert order, through moe_forward_topk on a handle
 * with num_experts = e1 - e0 and topk = 1 (ids = local expert, probs = the
 * route's prob): out rows come back prob-weighted, and the matching
 * moe_backward gives the rows' dx (prob-weighted), the per-route dprob in
 * dprobs[n,1] and the local experts' main_grad accumulation. The token side
 * keeps the shared expert and sums the returned rows. */
/* recompute_dispatch = 1 (redispatch in backward: PR #8210 review thread on
 * CUDA graphs, per-layer replay needs the saved schedule and activations to
 * survive pending microbatches, which a redispatch in backward provides): a
 * moe_saved then keeps only the routing (a few bytes per route and per row);
 * the dispatched rows and the SwiGLU intermediates live in the handle's
 * workspace, and moe_backward first runs the row placement, the shared output
 * gate and the gate/up GEMMs again from the saved routing, hidden and weights.
 * Results are bitwise those of recompute_dispatch = 0, for any interleaving of
 * forwards and backwards over several moe_saved states of one handle on one
 * stream. Costs one more gate/up GEMM per backward. */

/* One weight argument in the external ABI order (runtime page,
 * _MoKWeightArguments: shared_gate, shared_up, shared_down, routed_gate,
 * routed_up, routed_down). Gate/up are [I,H] (routed [E,I,H]), down is [H,I]
 * (routed [E,H,I]). A combined FC1 [.., 2I, H] is passed as two views whose
 * data pointers differ by I rows (runtime page, _gate_up_weight_arguments).
 * data must be 16-byte aligned and row_stride*elem_size a multiple of 16.
 * MXFP8 routed views (PR #6572, Supported configurations; PR #8210 review on
 * rowwise/columnwise payloads and scales): data is the E4M3 payload quantised
 * in blocks of 32 along K (the row), col_data the payload quantised in blocks
 * of 32 down the rows (N), both with expert_stride/row_stride in bytes
 * (multiples of 32). E8M0 scales are indexed with those strides:
 * scale[e][n][kb] at e*expert_stride/32 + n*row_stride/32 + kb, and
 * col_scale[e][nb][k] at e*expert_stride/32 + nb*row_stride + k -- for a
 * compact payload these are the compact [E,N,K/32] and [E,N/32,K] arrays. */
typedef struct {
    const void* data;         /* bf16 elements (MXFP8: e4m3 rowwise payload) */
    int64_t expert_stride;    /* elements between experts (routed views) */
    int64_t row_stride;       /* elements between rows */
    const uint8_t* scale;     /* MXFP8 only: E8M0 rowwise scales [E, N, K/32], compact */
    const void* col_data;     /* MXFP8 only: e4m3 columnwise payload, same shape/strides as data */
    const uint8_t* col_scale; /* MXFP8 only: E8M0 columnwise scales [E, N/32, K], compact */
    /* Optional per-expert descriptor table of a routed BF16 view (PR #6572,
     * Design > MCore-owned parameters: non-single expert weights are described
     * expert by expert): a HOST array of E device pointers, expert e's [N,K]
     * matrix at expert_ptrs[e] with row_stride (each 16-byte aligned); data and
     * expert_stride are then ignored. NULL: the strided view above. Read during
     * the call only. For an MXFP8 view the array holds 4*E pointers: rowwise
     * payloads [0, E), columnwise payloads [E, 2E) (16-byte aligned, row stride
     * row_stride bytes), rowwise scales [2E, 3E) ([N, K/32], row stride
     * row_stride/32) and columnwise scales [3E, 4E) ([N/32, K], row stride
     * row_stride); data, col_data, scale, col_scale and expert_stride are then
     * ignored. moe_prepare_weights reads the scales, the forward and backward
     * the payloads. */
    const void* const* expert_ptrs;
} moe_wview;

typedef struct {
    /* (with no_shared_expert the three shared views are ignored) */
    moe_wview shared_gate, shared_up, shared_down, routed_gate, routed_up, routed_down;
    /* Optional output gate of the shared expert ("core.transformer.moe.megakernel.
     * mok.runtime", _MoKAutograd.forward: shared_output_gate_weight;
     * "...mok.backend", _register_shared_weights(use_output_gate)): bf16 [H],
     * 16-byte aligned, or NULL for an ungated shared expert. The pages name the
     * weight without its formula; the layer reads it as a per-token scalar
     * gate on the shared expert's output: y_shared[t] *= sigmoid(hidden[t] . w). */
    const void* shared_output_gate;
} moe_weights;

/* main_grad buffers in the six-buffer order (runtime page,
 * _gate_up_main_grad_arguments). Shapes as the matching weights.
 * strides[i] = {expert_stride, row_stride} in elements (expert_stride unused
 * for the shared three). Fused accumulation is mandatory (PR #6572, Design >
 * Gradient accumulation): every pointer must be non-null, 16-byte aligned,
 * strides multiples of 16 bytes (with no_shared_expert the shared three are
 * ignored and may be NULL). shared_output_gate is the [H] main_grad of
 * the shared expert's output gate: required (16-byte aligned) when the forward
 * recorded in `saved` had a gate, ignored otherwise.
 * dtype (moe_gtype) applies to every buffer. MOE_G_FP32: main_grad += dW in
 * fp32, one add per element. MOE_G_BF16 (PR #8210 review: with BF16 main_grad
 * each contribution is rounded to BF16 before the BF16 reduction-store):
 * main_grad = bf16(main_grad + bf16(dW)), dW the fp32 GEMM accumulator, both
 * roundings to nearest even. */
typedef struct {
    void *shared_gate, *shared_up, *shared_down, *routed_gate, *routed_up, *routed_down;
    int64_t strides[6][2];
    void* shared_output_gate;
    int32_t dtype;
    /* Optional per-expert descriptor tables of the routed gate, up and down
     * main_grads ("core.transformer.moe.megakernel.mok.runtime",
     * main_grad_arguments: logical main grads and optional per-expert
     * descriptors): HOST arrays of E device pointers (16-byte aligned), expert
     * e's buffer at expert_ptrs[i][e] with row stride strides[3+i][1]; the
     * matching routed_* pointer and expert stride are then ignored. NULL: the
     * strided buffer. Read during the call only. */
    void* const* expert_ptrs[3];
} moe_main_grads;

typedef struct moe_handle moe_handle;
typedef struct moe_saved moe_saved;

/* Bytes of device workspace a handle needs for `cfg` (worst case R = T*k). */
moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes);

/* Creates a handle over caller-owned device workspace (256-byte aligned,
 * >= moe_workspace_size bytes, kept alive and unused by others until
 * moe_destroy). The handle itself is host memory owned by the library. The
 * current CUDA device at this call is the device of every later call.
 * Weight and main_grad views become per-expert TMA descriptor tables in this
 * workspace (with BF16 routed weights every view, the shared expert's as entry
 * 0; with MXFP8 ones the main_grad views given as moe_main_grads.expert_ptrs).
 * A table is re-encoded and uploaded only when its pointers, strides or dtype
 * change; such an upload (a host-to-device copy from library host memory)
 * waits for the work already queued on `stream` before it starts, and cannot
 * be captured into a CUDA graph: run one call with the same buffers before
 * capturing. */
moe_status moe_create(const moe_config* cfg, void* workspace, size_t workspace_bytes, moe_handle** out);
void moe_destroy(moe_handle* h);

/* Saved forward state (routing, permuted activations, SwiGLU intermediates;
 * with recompute_dispatch the routing only) lives in caller-owned device memory
 * of moe_saved_size bytes. A handle serves any number of saved states; their
 * forwards and backwards may interleave on the handle's stream. */
moe_status moe_saved_size(const moe_config* cfg, size_t* bytes);
moe_status moe_saved_create(moe_handle* h, void* memory, size_t bytes, moe_saved** out);
void moe_saved_destroy(moe_saved* s);

/* Forward: out[T,H] = gate[t] * SharedSwiGLU(hidden) + sum_s pp[t,s] * RoutedSwiGLU_{ids[t,s]}(hidden),
 * gate[t] = sigmoid(hidden[t] . w->shared_output_gate) (1 without a gate)
 * ("core.transformer.moe.megakernel.mok.backend", MoKMegakernel.forward;
 * PR #6572 Summary: dispatch, routed and shared experts, combine).
 *   hidden[T,H] bf16, probs[T,E] fp32, routing_map[T,E] bytes (0/1, e.g.
 *   torch.bool), out[T,H] bf16. 0 <= T <= max_tokens.
 * The routing map is authoritative (PR #6572, Design > Authoritative routing
 * maps): a token's experts are its map's true entries in ascending id order;
 * fewer than k leaves -1 slots that contribute nothing; probs off the map are
 * ignored; more than k is MOE_ERR_ROUTING (device status).
 * `saved` receives what backward needs. It keeps `hidden` and the weight
 * views BY POINTER: they must stay alive and unchanged until the matching
 * moe_backward. */
moe_status moe_forward(moe_handle* h, int64_t T, const void* hidden, const float* probs,
                       const uint8_t* routing_map, const moe_weights* w, void* out,
                       moe_saved* saved, void* stream);

/* The same forward fed by the router's top-k output instead of the dense map
 * (PR #6572, Possible feature work: consuming the router's output directly).
 *   topk_ids[T,k] int32: expert ids, -1 for an empty slot; topk_probs[T,k]
 *   fp32: the matching probs (ignored where the id is -1). Device memory, any
 *   alignment. Slots keep this order (the combine sums them in it). A row with
 *   an id outside [-1, E) or the same id twice is MOE_ERR_ROUTING (device
 *   status) and contributes nothing, like a map row with more than k routes.
 * The matching moe_backward writes dprobs as [T,k] fp32 in the same slot
 * order (0 for an empty slot) instead of the dense [T,E]. */
moe_status moe_forward_topk(moe_handle* h, int64_t T, const void* hidden, const int32_t* topk_ids,
                            const float* topk_probs, const moe_weights* w, void* out,
                            moe_saved* saved, void* stream);

/* Backward of L = sum(grad_out * out) for the forward recorded in `saved`
 * (runtime page, _MoKAutograd.backward; PR #6572, Design > Authoritative
 * routing maps (backward adapter) and > Gradient accumulation).
 *   grad_out[T,H] bf16 -> dhidden[T,H] bf16, dprobs[T,E] fp32 (dense: every
 *   element written; 0 where the map is false; after moe_forward_topk, [T,k]
 *   per slot), and main_grad += dW for all
 *   six buffers, one add per element in mg->dtype (deterministic). Experts that
 *   received no tokens keep their main_grad bitwise. `saved` is not consumed.
 *   With a shared output gate, also main_grad_gate[h] += sum_t dz[t] hidden[t,h]
 *   and dhidden[t] += dz[t] w, dz[t] = gate[t] (1 - gate[t]) <grad_out[t], y_shared[t]>
 *   (y_shared before the gate), summed in fp32 in a fixed order. */
moe_status moe_backward(moe_handle* h, const void* grad_out, const moe_saved* saved,
                        void* dhidden, float* dprobs, const moe_main_grads* mg, void* stream);

/* The configuration a handle was created with. */
moe_status moe_handle_config(const moe_handle* h, moe_config* cfg);

/* ---- Steps fed from HOST memory ----
 * A forward + backward step whose inputs and results live in host memory
 * (the pages' backend is called with device tensors; this pipeline is the
 * library's own entry for callers that hold a batch on the host). Each step
 * copies hidden, probs, routing_map and grad_out to the device, runs
 * moe_forward and moe_backward on them, and copies out, dhidden and dprobs
 * back. The copies run on two streams of the pipeline's own, joined to the
 * compute stream by events, into two alternating device staging sets, so that
 * one step's uploads and downloads overlap the kernels of its neighbours. */
typedef struct moe_host_pipe moe_host_pipe;

/* Bytes of device memory a pipeline for steps of exactly T tokens needs (two
 * staging sets of hidden, probs, routing_map, grad_out, out, dhidden, dprobs,
 * and one saved state); 1 <= T <= cfg->max_tokens. */
moe_status moe_host_pipe_size(const moe_config* cfg, int64_t T, size_t* bytes);

/* Creates a pipeline of `h` over caller-owned device memory (256-byte aligned,
 * >= moe_host_pipe_size bytes for h's configuration, kept alive and unused by
 * others until moe_host_pipe_destroy). The pipeline owns two non-blocking CUDA
 * streams and six events (host-side objects, released by destroy); it
 * allocates no device memory. */
moe_status moe_host_pipe_create(moe_handle* h, int64_t T, void* memory, size_t bytes, moe_host_pipe** out);

/* Enqueues one step and returns. HOST pointers: hidden[T,H] bf16, probs[T,E]
 * fp32, routing_map[T,E] bytes, grad_out[T,H] bf16 in; out[T,H] bf16,
 * dhidden[T,H] bf16, dprobs[T,E] fp32 receive the results (dense dprobs, as
 * moe_backward after moe_forward). w and mg as for moe_forward / moe_backward
 * (device weights and main_grads: main_grad += dW every step, steps applied in
 * call order). Inputs must stay unchanged, and results unread, until the step
 * is complete (moe_host_pipe_sync). Page-locked host memory (cudaHostAlloc,
 * cudaHostRegister) gives asynchronous copies; pageable memory works but the
 * call then returns only after the step's downloads are done. `stream` is the
 * compute stream (any stream; the pipeline orders its steps itself).
 * Argument errors return before anything is enqueued; the device status
 * (moe_device_status) reports kernel-detected errors as for moe_forward. */
moe_status moe_host_step(moe_host_pipe* p, const void* hidden, const float* probs, const uint8_t* routing_map,
                         const void* grad_out, const moe_weights* w, const moe_main_grads* mg, void* out,
                         void* dhidden, float* dprobs, void* stream);

/* Blocks until every enqueued step's results are in host memory. */
moe_status moe_host_pipe_sync(moe_host_pipe* p);

/* Waits for the pipeline's steps, then releases its streams and events. */
void moe_host_pipe_destroy(moe_host_pipe* p);

/* MXFP8 weight preparation (PR #6572, Design > MCore-owned parameters:
 * converted scale layouts refreshed once per optimizer iteration at stable
 * addresses; PR #8210 review on _swizzle_mxfp8_scale): converts the routed
 * weights' compact E8M0 scales (rowwise and columnwise, all experts in one
 * launch each) into the scale-factor layout of the block-scaled MMA, in the
 * handle's workspace. Call after every change of the routed weights' scales
 * and before moe_forward; payloads are read in place. No-op for BF16 handles.
 * moe_forward on an MXFP8 handle before the first call returns MOE_ERR_STATE. */
moe_status moe_prepare_weights(moe_handle* h, const moe_weights* w, void* stream);

/* MXFP8 quantisation of a bf16 matrix x[rows, cols] (row stride ld elements):
 * E4M3 elements (round to nearest even, saturating at +-448) and one E8M0
 * shared exponent per 32 elements, floor(log2 amax) - 8 + 127 clamped to
 * [0, 254] (OCP MX v1.0; the pages name MXFP8 without restating it).
 * axis 1: blocks along each row (cols % 32 == 0), scales[rows, cols/32];
 * axis 0: blocks down each column (rows % 32 == 0), scales[rows/32, cols].
 * q[rows, cols] E4M3 bytes with row stride ldq; all device pointers. */
moe_status moe_quantize_mxfp8(const void* x, int64_t rows, int64_t cols, int64_t ld, int32_t axis, uint8_t* q,
                              int64_t ldq, uint8_t* scales, void* stream);

/* Test hook: copies the routing of `saved` into caller device buffers.
 * ids[T,k] int32 (-1 = missing), pp[T,k] fp32, counts[E] int32,
 * offsets[E+1] int32 (exclusive scan of counts), perm_src[T*k] int32 (token of
 * each permuted route, compact, first offsets[E] entries written), row_of[T,k]
 * int32 (compact permuted row of each slot, -1 = missing). Any pointer may be
 * NULL to skip it. */
moe_status moe_export_routing(moe_handle* h, const moe_saved* saved, int32_t* ids, float* pp,
                              int32_t* counts, int32_t* offsets, int32_t* perm_src,
                              int32_t* row_of, void* stream);

/* Routing without any device allocation, for callers that cannot allocate
 * device memory: code that runs where cudaMalloc is not allowed or not
 * wanted, such as a plugin called from a host framework that owns all device
 * memory through its own pool, a serving loop that forbids allocation after
 * start-up, or a memory budget that must stay fixed. The pages have no
 * counterpart to this call.
 * It computes the same routing as moe_forward and moe_export_routing, in the
 * same compact form, into caller device buffers: ids[T,k] int32 (-1 =
 * missing), pp[T,k] fp32, counts[E] int32, offsets[E+1] int32, perm_src[T*k]
 * int32 (first offsets[E] entries), row_of[T,k] int32, and routing_error[1]
 * int32 (1 when a row has more than k routes; such rows are dropped).
 * Its only scratch is a library-owned device array of 2^17 int32 (512 KB)
 * that every GPU loading the library keeps until the process exits, so
 * T*k must not exceed 131072 (and T not 65536): larger sizes return
 * MOE_ERR_UNSUPPORTED. The array is shared by every call and keeps the last
 * call's contents; calls whose kernels overlap on the GPU (two streams, two
 * threads) race on it. Every call resolves the array's device address on the
 * current device (cudaGetSymbolAddress; valid again after a device reset); the
 * first call on a device loads the library's device code there, so make that
 * first call before any stream capture. Cost: the per-expert ranking reads the
 * routing map column by column (about 32 * T * E bytes of L2 traffic, 67 MB at
 * T = 16384, E = 128), several times the forward's fused routing; it is meant
 * for callers that cannot allocate, not for the hot path. Asynchronous on
 * `stream`; nothing is allocated or freed. */
moe_status moe_route_noalloc(int64_t T, int64_t E, int64_t k, const uint8_t* routing_map, const float* probs,
                             int32_t* ids, float* pp, int32_t* counts, int32_t* offsets, int32_t* perm_src,
                             int32_t* row_of, int32_t* routing_error, void* stream);

/* Synchronises `stream`, returns the device status recorded since the last
 * call (MOE_OK, MOE_ERR_ROUTING or MOE_ERR_TIMEOUT) and clears it. */
moe_status moe_device_status(moe_handle* h, void* stream);

/* Test hook for the timeout path: enqueues one block that waits on an mbarrier
 * nothing completes, with the same bounded wait the GEMM kernels use; the wait
 * gives up after the library's limit (2 s), records MOE_ERR_TIMEOUT in the
 * handle's device status (read by moe_device_status) and the block exits, so
 * the context and the handle stay usable. Asynchronous on `stream`. */
moe_status moe_selftest_timeout(moe_handle* h, void* stream);

/* Number of kernels this library has launched in this process. */
uint64_t moe_launch_count(void);

/* Kernel classes of the layer, in the order moe_profile_read reports them.
 * With BF16 routed weights the shared expert runs as group 0 of the ROUTED
 * classes' grouped GEMMs (its rows before the routed segments), so the
 * *_SHARED GEMM classes launch only with MXFP8 routed weights. */
enum {
    MOE_K_ROUTE_PACK = 0, MOE_K_ROUTE_SCAN, MOE_K_ROUTE_PLACE, MOE_K_GATHER,
    MOE_K_FWD_GU_ROUTED, MOE_K_FWD_GU_SHARED, MOE_K_FWD_DOWN_ROUTED, MOE_K_FWD_DOWN_SHARED, MOE_K_COMBINE,
    MOE_K_BWD_DOWN_ROUTED, MOE_K_BWD_DOWN_SHARED, MOE_K_BWD_GU_ROUTED, MOE_K_BWD_GU_SHARED,
    MOE_K_WGRAD_FC1_ROUTED, MOE_K_WGRAD_DOWN_ROUTED, MOE_K_WGRAD_FC1_SHARED, MOE_K_WGRAD_DOWN_SHARED,
    MOE_K_UNPERMUTE, MOE_K_SHARED_GATE_FWD, MOE_K_SHARED_GATE_BWD, MOE_K_COUNT
};

/* Per-kernel timing for measurement. While enabled, every kernel the handle
 * launches is bracketed by a pair of CUDA events recorded on the launch
 * stream: no extra GPU work and no host synchronisation. */
moe_status moe_profile_enable(moe_handle* h, int enable);

/* Restricts the timing to the kernel classes whose bits are set in class_mask
 * (bit i = class i; all classes by default), so that a measurement can time one
 * kernel without events between the others. Host-only. */
moe_status moe_profile_select(moe_handle* h, uint32_t class_mask);

/* Synchronises the recorded events and writes, per kernel class (n entries,
 * n <= MOE_K_COUNT), the summed device time in milliseconds and the number of
 * launches since the previous read; then forgets them. Host arrays. */
moe_status moe_profile_read(moe_handle* h, double* total_ms, int64_t* launches, int n);

/* Name of a kernel class ("gemm_wgrad_fc1_routed", ...), or NULL. */
const char* moe_kernel_name(int kernel_class);

const char* moe_status_string(moe_status s);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
