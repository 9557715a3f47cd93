"""Thin ctypes binding of libmoe.so (include/moe.h): same names, argument marshalling only.

Every step of the layer runs in the library's CUDA kernels; PyTorch only
supplies device memory (tensors) and streams. There is no other code path: if
the library cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

c_int64, c_int32, c_float, c_void_p, c_size_t = (ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                                                 ctypes.c_void_p, ctypes.c_size_t)

MOE_OK = 0
MOE_ERR_ROUTING, MOE_ERR_TIMEOUT = 3, 5    # device-detected errors (moe_device_status)
MOE_W_BF16, MOE_W_MXFP8 = 0, 1
MOE_G_FP32, MOE_G_BF16 = 0, 1
MOE_ACT_FP32, MOE_ACT_BF16 = 0, 1   # activations between the expert GEMMs (include/moe.h, moe_act)
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_ROUTING",
                4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_STATE"}
WEIGHT_NAMES = ("shared_gate", "shared_up", "shared_down", "routed_gate", "routed_up", "routed_down")


class moe_config(ctypes.Structure):
    _fields_ = [("max_tokens", c_int64), ("hidden", c_int64), ("num_experts", c_int64), ("topk", c_int64),
                ("inter", c_int64), ("routed_wtype", c_int32), ("swiglu_limit", c_float),
                ("recompute_dispatch", c_int32), ("act_precision", c_int32), ("no_shared_expert", c_int32)]


class moe_wview(ctypes.Structure):
    _fields_ = [("data", c_void_p), ("expert_stride", c_int64), ("row_stride", c_int64), ("scale", c_void_p),
                ("col_data", c_void_p), ("col_scale", c_void_p), ("expert_ptrs", c_void_p)]


class moe_weights(ctypes.Structure):
    _fields_ = [(n, moe_wview) for n in WEIGHT_NAMES] + [("shared_output_gate", c_void_p)]


class moe_main_grads(ctypes.Structure):
    _fields_ = ([(n, c_void_p) for n in WEIGHT_NAMES] + [("strides", (c_int64 * 2) * 6)] +
                [("shared_output_gate", c_void_p), ("dtype", c_int32), ("expert_ptrs", c_void_p * 3)])


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({_status_string(status)})")


_LIB = None
_LOCK = threading.Lock()
EXPORTED = ("moe_workspace_size", "moe_create", "moe_destroy", "moe_saved_size", "moe_saved_create",
            "moe_saved_destroy", "moe_forward", "moe_backward", "moe_export_routing", "moe_device_status",
            "moe_launch_count", "moe_status_string", "moe_profile_enable", "moe_profile_read", "moe_kernel_name",
            "moe_route_noalloc", "moe_prepare_weights", "moe_quantize_mxfp8", "moe_profile_select",
            "moe_forward_topk", "moe_handle_config", "moe_host_pipe_size", "moe_host_pipe_create", "moe_host_step",
            "moe_host_pipe_sync", "moe_host_pipe_destroy", "moe_selftest_timeout")
MOE_K_COUNT = 20


def lib_path() -> str:
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libmoe.so")


def load(build_if_missing: bool = True):
    """Loads libmoe.so (building it first if it is absent)."""
    global _LIB
    with _LOCK:
        if _LIB is not None:
            return _LIB
        path = lib_path()
        if not os.path.exists(path):
            if not build_if_missing:
                raise OSError(f"{path} is not built")
            from . import build_lib
            build_lib.build()
        L = ctypes.CDLL(path)
        P = ctypes.POINTER
        L.moe_workspace_size.argtypes = [P(moe_config), P(c_size_t)]
        L.moe_saved_size.argtypes = [P(moe_config), P(c_size_t)]
        L.moe_create.argtypes = [P(moe_config), c_void_p, c_size_t, P(c_void_p)]
        L.moe_destroy.argtypes = [c_void_p]
        L.moe_destroy.restype = None
        L.moe_saved_create.argtypes = [c_void_p, c_void_p, c_size_t, P(c_void_p)]
        L.moe_saved_destroy.argtypes = [c_void_p]
        L.moe_saved_destroy.restype = None
        L.moe_forward.argtypes = [c_void_p, c_int64, c_void_p, c_void_p, c_void_p, P(moe_weights), c_void_p,
                                  c_void_p, c_void_p]
        L.moe_forward_topk.argtypes = [c_void_p, c_int64, c_void_p, c_void_p, c_void_p, P(moe_weights), c_void_p,
                                       c_void_p, c_void_p]
        L.moe_backward.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, P(moe_main_grads), c_void_p]
        L.moe_export_routing.argtypes = [c_void_p, c_void_p] + [c_void_p] * 6 + [c_void_p]
        L.moe_device_status.argtypes = [c_void_p, c_void_p]
        L.moe_selftest_timeout.argtypes = [c_void_p, c_void_p]
        L.moe_launch_count.argtypes = []
        L.moe_launch_count.restype = ctypes.c_uint64
        L.moe_profile_enable.argtypes = [c_void_p, c_int32]
        L.moe_profile_select.argtypes = [c_void_p, ctypes.c_uint32]
        L.moe_profile_read.argtypes = [c_void_p, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(c_int64), c_int32]
        L.moe_kernel_name.argtypes = [c_int32]
        L.moe_kernel_name.restype = ctypes.c_char_p
        L.moe_route_noalloc.argtypes = [c_int64, c_int64, c_int64] + [c_void_p] * 10
        L.moe_prepare_weights.argtypes = [c_void_p, P(moe_weights), c_void_p]
        L.moe_quantize_mxfp8.argtypes = [c_void_p, c_int64, c_int64, c_int64, c_int32, c_void_p, c_int64, c_void_p,
                                         c_void_p]
        L.moe_status_string.argtypes = [c_int32]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_handle_config.argtypes = [c_void_p, P(moe_config)]
        L.moe_host_pipe_size.argtypes = [P(moe_config), c_int64, P(c_size_t)]
        L.moe_host_pipe_create.argtypes = [c_void_p, c_int64, c_void_p, c_size_t, P(c_void_p)]
        L.moe_host_step.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, P(moe_weights),
                                    P(moe_main_grads), c_void_p, c_void_p, c_void_p, c_void_p]
        L.moe_host_pipe_sync.argtypes = [c_void_p]
        L.moe_host_pipe_destroy.argtypes = [c_void_p]
        L.moe_host_pipe_destroy.restype = None
        for name in ("moe_workspace_size", "moe_saved_size", "moe_create", "moe_saved_create", "moe_forward",
                     "moe_backward", "moe_export_routing", "moe_device_status", "moe_profile_enable",
                     "moe_profile_read", "moe_route_noalloc", "moe_prepare_weights", "moe_quantize_mxfp8",
                     "moe_profile_select", "moe_handle_config", "moe_host_pipe_size", "moe_host_pipe_create",
                     "moe_host_step", "moe_host_pipe_sync", "moe_selftest_timeout"):
            getattr(L, name).restype = c_int32
        _LIB = L
        return L


def _status_string(status: int) -> str:
    try:
        return load().moe_status_string(status).decode()
    except Exception:  # pragma: no cover
        return "?"


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ------------------------------------------------------------------ the C ABI, same names
def moe_workspace_size(cfg: moe_config) -> int:
    n = c_size_t(0)
    _check(load().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def moe_saved_size(cfg: moe_config) -> int:
    n = c_size_t(0)
    _check(load().moe_saved_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_saved_size")
    return n.value


def moe_create(cfg: moe_config, workspace) -> c_void_p:
    h = c_void_p()
    _check(load().moe_create(ctypes.byref(cfg), _ptr(workspace), workspace.numel() * workspace.element_size(),
                             ctypes.byref(h)), "moe_create")
    return h


def moe_destroy(h):
    load().moe_destroy(h)


def moe_saved_create(h, memory) -> c_void_p:
    s = c_void_p()
    _check(load().moe_saved_create(h, _ptr(memory), memory.numel() * memory.element_size(), ctypes.byref(s)),
           "moe_saved_create")
    return s


def moe_saved_destroy(s):
    load().moe_saved_destroy(s)


def moe_forward(h, T, hidden, probs, routing_map, weights: moe_weights, out, saved, stream=None):
    _check(load().moe_forward(h, int(T), _ptr(hidden), _ptr(probs), _ptr(routing_map), ctypes.byref(weights),
                              _ptr(out), saved, _stream_ptr(stream)), "moe_forward")


def moe_forward_topk(h, T, hidden, topk_ids, topk_probs, weights: moe_weights, out, saved, stream=None):
    _check(load().moe_forward_topk(h, int(T), _ptr(hidden), _ptr(topk_ids), _ptr(topk_probs), ctypes.byref(weights),
                                   _ptr(out), saved, _stream_ptr(stream)), "moe_forward_topk")


def moe_backward(h, grad_out, saved, dhidden, dprobs, main_grads: moe_main_grads, stream=None):
    _check(load().moe_backward(h, _ptr(grad_out), saved, _ptr(dhidden), _ptr(dprobs), ctypes.byref(main_grads),
                               _stream_ptr(stream)), "moe_backward")


def moe_handle_config(h) -> moe_config:
    c = moe_config()
    _check(load().moe_handle_config(h, ctypes.byref(c)), "moe_handle_config")
    return c


def moe_host_pipe_size(cfg: moe_config, T: int) -> int:
    n = c_size_t(0)
    _check(load().moe_host_pipe_size(ctypes.byref(cfg), int(T), ctypes.byref(n)), "moe_host_pipe_size")
    return n.value


def moe_host_pipe_create(h, T: int, memory) -> c_void_p:
    p = c_void_p()
    _check(load().moe_host_pipe_create(h, int(T), _ptr(memory), memory.numel() * memory.element_size(),
                                       ctypes.byref(p)), "moe_host_pipe_create")
    return p


def moe_host_step(p, hidden, probs, routing_map, grad_out, weights: moe_weights, main_grads: moe_main_grads,
                  out, dhidden, dprobs, stream=None):
    """One forward + backward step from HOST tensors (include/moe.h, moe_host_step)."""
    _check(load().moe_host_step(p, _ptr(hidden), _ptr(probs), _ptr(routing_map), _ptr(grad_out),
                                ctypes.byref(weights), ctypes.byref(main_grads), _ptr(out), _ptr(dhidden),
                                _ptr(dprobs), _stream_ptr(stream)), "moe_host_step")


def moe_host_pipe_sync(p):
    _check(load().moe_host_pipe_sync(p), "moe_host_pipe_sync")


def moe_host_pipe_destroy(p):
    load().moe_host_pipe_destroy(p)


def moe_export_routing(h, saved, ids=None, pp=None, counts=None, offsets=None, perm_src=None, row_of=None,
                       stream=None):
    _check(load().moe_export_routing(h, saved, _ptr(ids), _ptr(pp), _ptr(counts), _ptr(offsets), _ptr(perm_src),
                                     _ptr(row_of), _stream_ptr(stream)), "moe_export_routing")


def moe_device_status(h, stream=None) -> int:
    return int(load().moe_device_status(h, _stream_ptr(stream)))


def moe_selftest_timeout(h, stream=None):
    """Enqueues the timeout-path test: one bounded wait that gives up (2 s) and records
    MOE_ERR_TIMEOUT in the handle's device status."""
    _check(load().moe_selftest_timeout(h, _stream_ptr(stream)), "moe_selftest_timeout")


def moe_route_noalloc(T, E, k, routing_map, probs, ids, pp, counts, offsets, perm_src, row_of, routing_error,
                      stream=None):
    """Routing into caller buffers with no device allocation (see include/moe.h)."""
    _check(load().moe_route_noalloc(int(T), int(E), int(k), _ptr(routing_map), _ptr(probs), _ptr(ids), _ptr(pp),
                                    _ptr(counts), _ptr(offsets), _ptr(perm_src), _ptr(row_of), _ptr(routing_error),
                                    _stream_ptr(stream)), "moe_route_noalloc")


def moe_prepare_weights(h, weights: moe_weights, stream=None):
    _check(load().moe_prepare_weights(h, ctypes.byref(weights), _stream_ptr(stream)), "moe_prepare_weights")


def moe_quantize_mxfp8(x, axis, q, scales, stream=None):
    """MXFP8-quantise a 2-D bf16 tensor x into q (uint8, same shape) and compact scales."""
    rows, cols = x.shape
    _check(load().moe_quantize_mxfp8(_ptr(x), rows, cols, x.stride(0), int(axis), _ptr(q), q.stride(0),
                                     _ptr(scales), _stream_ptr(stream)), "moe_quantize_mxfp8")


def mxfp8_weight(w):
    """Quantises a bf16 weight [E, N, K] (or a combined-FC1 row view of one) on the
    device with moe_quantize_mxfp8: returns (rowwise payload, compact row scales,
    columnwise payload, compact column scales) as [E, N, K], [E, N, K/32],
    [E, N, K], [E, N/32, K] uint8 tensors."""
    import torch
    E, N, K = w.shape
    x = w.reshape(E * N, K).contiguous()
    q = torch.empty((E * N, K), dtype=torch.uint8, device=w.device)
    s = torch.empty((E * N, K // 32), dtype=torch.uint8, device=w.device)
    moe_quantize_mxfp8(x, 1, q, s)
    qc = torch.empty((E * N, K), dtype=torch.uint8, device=w.device)
    sc = torch.empty((E * N // 32, K), dtype=torch.uint8, device=w.device)
    moe_quantize_mxfp8(x, 0, qc, sc)
    return q.view(E, N, K), s.view(E, N, K // 32), qc.view(E, N, K), sc.view(E, N // 32, K)


def mxfp8_view(payload, scale, col_payload, col_scale) -> moe_wview:
    """moe_wview of an MXFP8 routed weight ([E, N, K] payloads, strides in bytes)."""
    return moe_wview(payload.data_ptr(), payload.stride(0), payload.stride(1), scale.data_ptr(),
                     col_payload.data_ptr(), col_scale.data_ptr())


def moe_launch_count() -> int:
    return int(load().moe_launch_count())


def moe_profile_enable(h, enable: bool = True):
    _check(load().moe_profile_enable(h, 1 if enable else 0), "moe_profile_enable")


def moe_profile_select(h, classes=None):
    """Time only the given kernel classes (names or indices); None: all of them."""
    if classes is None:
        mask = 0xFFFFFFFF
    else:
        names = [moe_kernel_name(i) for i in range(MOE_K_COUNT)]
        mask = 0
        for c in classes:
            mask |= 1 << (names.index(c) if isinstance(c, str) else int(c))
    _check(load().moe_profile_select(h, mask), "moe_profile_select")


def moe_profile_read(h) -> dict:
    """{kernel name: (summed ms, launches)} since the previous read."""
    ms = (ctypes.c_double * MOE_K_COUNT)()
    n = (c_int64 * MOE_K_COUNT)()
    _check(load().moe_profile_read(h, ms, n, MOE_K_COUNT), "moe_profile_read")
    return {moe_kernel_name(i): (ms[i], n[i]) for i in range(MOE_K_COUNT)}


def moe_kernel_name(i: int) -> str:
    r = load().moe_kernel_name(i)
    return r.decode() if r else None


# ------------------------------------------------------------------ marshalling helpers
def wview(t, scale=None, col_data=None, col_scale=None) -> moe_wview:
    """View of a 2-D [N,K] or 3-D [E,N,K] tensor (strides taken from the tensor)."""
    if t.dim() == 3:
        es, rs = t.stride(0), t.stride(1)
    else:
        es, rs = 0, t.stride(0)
    return moe_wview(t.data_ptr(), es, rs, None if scale is None else scale.data_ptr(),
                     None if col_data is None else col_data.data_ptr(),
                     None if col_scale is None else col_scale.data_ptr())


def weights_from_combined(shared_fc1, shared_fc2, routed_fc1, routed_fc2, shared_output_gate=None) -> moe_weights:
    """Gate/up views of combined FC1 weights ([2I,H], [E,2I,H]): rows [0,I) gate, [I,2I) up;
    optional bf16 [H] shared-expert output gate. shared_fc1 / shared_fc2 None: no shared
    views (a layer without a shared expert ignores them)."""
    inter = routed_fc1.shape[1] // 2
    shared = (moe_wview(), moe_wview(), moe_wview()) if shared_fc1 is None else \
        (wview(shared_fc1[:inter]), wview(shared_fc1[inter:]), wview(shared_fc2))
    return moe_weights(*shared, wview(routed_fc1[:, :inter]), wview(routed_fc1[:, inter:]), wview(routed_fc2),
                       None if shared_output_gate is None else shared_output_gate.data_ptr())


def main_grads_from_combined(shared_fc1, shared_fc2, routed_fc1, routed_fc2, shared_output_gate=None) -> moe_main_grads:
    """Six-buffer main_grad order over combined FC1/FC2 buffers, all fp32 or all
    bf16 (plus the optional [H] main_grad of the shared-expert output gate)."""
    import torch
    inter = routed_fc1.shape[1] // 2
    shared = (None, None, None) if shared_fc1 is None else (shared_fc1[:inter], shared_fc1[inter:], shared_fc2)
    views = shared + (routed_fc1[:, :inter], routed_fc1[:, inter:], routed_fc2)
    present = [v for v in views if v is not None]
    dtypes = {v.dtype for v in present} | ({shared_output_gate.dtype} if shared_output_gate is not None else set())
    if dtypes not in ({torch.float32}, {torch.bfloat16}):
        raise ValueError(f"main_grad buffers must be all fp32 or all bf16, got {dtypes}")
    m = moe_main_grads(*[None if v is None else v.data_ptr() for v in views])
    m.dtype = MOE_G_BF16 if dtypes == {torch.bfloat16} else MOE_G_FP32
    m.shared_output_gate = None if shared_output_gate is None else shared_output_gate.data_ptr()
    for i, v in enumerate(views):
        if v is None:
            continue
        if v.dim() == 3:
            m.strides[i][0], m.strides[i][1] = v.stride(0), v.stride(1)
        else:
            m.strides[i][0], m.strides[i][1] = 0, v.stride(0)
    return m


def _pointer_table(tensors):
    """HOST array of the tensors' device pointers (ctypes), one per expert."""
    return (c_void_p * len(tensors))(*[t.data_ptr() for t in tensors])


def set_expert_tables(weights: moe_weights, gate=None, up=None, down=None) -> moe_weights:
    """Describes routed BF16 weights expert by expert: each argument a list of E
    [N,K] tensors sharing one row stride (PR #6572 per-expert non-single
    weights). The host pointer arrays are kept alive on ``weights``."""
    keep = list(getattr(weights, "_tables", []))
    for name, ts in (("routed_gate", gate), ("routed_up", up), ("routed_down", down)):
        if ts is None:
            continue
        arr = _pointer_table(ts)
        v = getattr(weights, name)
        v.expert_ptrs = ctypes.cast(arr, c_void_p).value
        v.row_stride = ts[0].stride(0)
        v.data = None
        v.expert_stride = 0
        keep.append(arr)
    weights._tables = keep
    return weights


def set_mx_expert_tables(weights: moe_weights, gate=None, up=None, down=None) -> moe_weights:
    """Describes MXFP8 routed weights expert by expert: each argument a tuple of four
    lists of E tensors -- rowwise payloads [N,K] uint8, columnwise payloads [N,K],
    rowwise scales [N,K/32], columnwise scales [N/32,K] -- with the row strides the
    C ABI expects (payload row stride R; scales R/32 and R). The host pointer
    arrays are kept alive on ``weights``."""
    keep = list(getattr(weights, "_tables", []))
    for name, parts in (("routed_gate", gate), ("routed_up", up), ("routed_down", down)):
        if parts is None:
            continue
        q, cq, sc, csc = parts
        r = q[0].stride(0)
        if any(t.stride(0) != r for t in list(q) + list(cq)) or any(t.stride(0) * 32 != r for t in sc) or \
                any(t.stride(0) != r for t in csc):
            raise ValueError("per-expert MXFP8 tensors with inconsistent row strides")
        arr = _pointer_table(list(q) + list(cq) + list(sc) + list(csc))
        v = getattr(weights, name)
        v.expert_ptrs = ctypes.cast(arr, c_void_p).value
        v.row_stride = r
        v.data = v.col_data = v.scale = v.col_scale = None
        v.expert_stride = 0
        keep.append(arr)
    weights._tables = keep
    return weights


def set_main_grad_tables(main_grads: moe_main_grads, gate=None, up=None, down=None) -> moe_main_grads:
    """Describes the routed main_grads expert by expert: lists of E [N,K] tensors
    (one row stride per list). The host pointer arrays are kept alive on ``main_grads``."""
    keep = list(getattr(main_grads, "_tables", []))
    for i, ts in enumerate((gate, up, down)):
        if ts is None:
            continue
        arr = _pointer_table(ts)
        main_grads.expert_ptrs[i] = ctypes.cast(arr, c_void_p).value
        main_grads.strides[3 + i][1] = ts[0].stride(0)
        keep.append(arr)
    main_grads._tables = keep
    return main_grads


class MoELayer:
    """Holds a handle, its workspace and one saved-state block (all torch device memory)."""

    def __init__(self, max_tokens, hidden, num_experts, topk, inter, device="cuda", routed_wtype=MOE_W_BF16,
                 swiglu_limit=0.0, recompute_dispatch=False, act_precision=None, shared_expert=True, fill=None):
        """fill: a byte value written over the workspace and saved-state memory before the
        handle is created (None: left as allocated); no result may depend on it."""
        import torch
        self.cfg = moe_config(max_tokens, hidden, num_experts, topk, inter, routed_wtype, float(swiglu_limit),
                              int(bool(recompute_dispatch)),
                              MOE_ACT_FP32 if act_precision is None else int(act_precision),
                              0 if shared_expert else 1)
        self.device = torch.device(device)
        ws = moe_workspace_size(self.cfg)
        sv = moe_saved_size(self.cfg)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=self.device)
        self.saved_mem = torch.empty(sv, dtype=torch.uint8, device=self.device)
        if fill is not None:
            self.workspace.fill_(int(fill))
            self.saved_mem.fill_(int(fill))
        with torch.cuda.device(self.device):
            self.handle = moe_create(self.cfg, self.workspace)
            self.saved = moe_saved_create(self.handle, self.saved_mem)

    def prepare_weights(self, weights: moe_weights, stream=None):
        moe_prepare_weights(self.handle, weights, stream)

    def forward(self, hidden, probs, routing_map, weights: moe_weights, out=None, stream=None):
        import torch
        if out is None:
            out = torch.empty_like(hidden)
        moe_forward(self.handle, hidden.shape[0], hidden, probs, routing_map, weights, out, self.saved, stream)
        self._topk = False
        return out

    def forward_topk(self, hidden, topk_ids, topk_probs, weights: moe_weights, out=None, stream=None):
        """Forward from the router's top-k output: int32 ids [T,k] (-1 = empty slot), fp32 probs [T,k]."""
        import torch
        if out is None:
            out = torch.empty_like(hidden)
        moe_forward_topk(self.handle, hidden.shape[0], hidden, topk_ids, topk_probs, weights, out, self.saved, stream)
        self._topk = True
        return out

    def backward(self, grad_out, main_grads: moe_main_grads, dhidden=None, dprobs=None, stream=None):
        import torch
        T = grad_out.shape[0]
        if dhidden is None:
            dhidden = torch.empty_like(grad_out)
        if dprobs is None:  # [T,k] per slot after forward_topk, else dense [T,E]
            n = self.cfg.topk if getattr(self, "_topk", False) else self.cfg.num_experts
            dprobs = torch.empty((T, n), dtype=torch.float32, device=grad_out.device)
        moe_backward(self.handle, grad_out, self.saved, dhidden, dprobs, main_grads, stream)
        return dhidden, dprobs

    def device_status(self, stream=None) -> int:
        return moe_device_status(self.handle, stream)

    def host_pipe(self, T):
        """A HostPipe of forward + backward steps of T tokens from host buffers."""
        return HostPipe(self, T)

    def close(self):
        if getattr(self, "handle", None) is not None:
            moe_saved_destroy(self.saved)
            moe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class HostPipe:
    """Forward + backward steps of a layer fed from host buffers, through the C
    ABI's host pipeline (moe_host_pipe_create / moe_host_step): every step
    uploads its inputs and downloads its results, the copies overlapped with the
    kernels of the neighbouring steps. Device staging memory is a torch buffer
    held here; the steps apply to main_grad in call order."""

    def __init__(self, layer: "MoELayer", T: int):
        import torch
        self.layer = layer
        self.T = int(T)
        self.compute = torch.cuda.Stream(layer.device)
        self.memory = torch.empty(moe_host_pipe_size(layer.cfg, self.T), dtype=torch.uint8, device=layer.device)
        with torch.cuda.device(layer.device):
            self.pipe = moe_host_pipe_create(layer.handle, self.T, self.memory)

    def step(self, hidden, probs, routing_map, grad_out, weights: moe_weights, main_grads: moe_main_grads,
             out, dhidden, dprobs):
        """Enqueues one step: host hidden[T,H] bf16, probs[T,E] f32, routing_map[T,E]
        (bool or uint8), grad_out[T,H] bf16 in; host out[T,H], dhidden[T,H] bf16 and
        dprobs[T,E] f32 receive the results once `synchronize` returns. Page-locked
        tensors only (pageable ones would make every call wait for its step)."""
        import torch
        for t in (hidden, probs, routing_map, grad_out, out, dhidden, dprobs):
            if t.is_cuda or not t.is_pinned() or not t.is_contiguous():
                raise ValueError("HostPipe.step takes contiguous pinned host tensors")
        if hidden.shape[0] != self.T:
            raise ValueError("token count differs from the pipeline's")
        H, E = self.layer.cfg.hidden, self.layer.cfg.num_experts
        for t, shape, dt in ((hidden, (self.T, H), torch.bfloat16), (grad_out, (self.T, H), torch.bfloat16),
                             (out, (self.T, H), torch.bfloat16), (dhidden, (self.T, H), torch.bfloat16),
                             (probs, (self.T, E), torch.float32), (dprobs, (self.T, E), torch.float32)):
            if tuple(t.shape) != shape or t.dtype != dt:
                raise ValueError("host tensor of the wrong shape or dtype")
        if tuple(routing_map.shape) != (self.T, E) or routing_map.element_size() != 1:
            raise ValueError("routing_map must be [T,E] bytes")
        moe_host_step(self.pipe, hidden, probs, routing_map, grad_out, weights, main_grads, out, dhidden, dprobs,
                      self.compute)

    def synchronize(self):
        """Waits until every enqueued step's results are in host memory."""
        moe_host_pipe_sync(self.pipe)

    def close(self):
        if getattr(self, "pipe", None) is not None:
            moe_host_pipe_destroy(self.pipe)   # waits for the steps in flight
            self.pipe = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

