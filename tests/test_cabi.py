"""The C-ABI library builds, loads without a GPU, exports every symbol that
include/moe.h declares, and rejects bad configurations on the host."""
import ctypes
import os
import re

import pytest

import mixture_experts_layer_pack_gb300 as M
from mixture_experts_layer_pack_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(moe_\w+)\s*\(", src))
    return names


def test_library_exports_every_declared_symbol():
    L = M.load()
    declared = _declared_functions()
    assert {"moe_forward", "moe_backward", "moe_create"} <= declared
    for name in sorted(declared):
        assert hasattr(L, name), name
    assert set(B.EXPORTED) <= declared


def test_status_strings():
    L = M.load()
    for s in range(7):
        assert L.moe_status_string(s)


def _cfg(**kw):
    base = dict(max_tokens=4096, hidden=2048, num_experts=96, topk=6, inter=1024, routed_wtype=0, swiglu_limit=0.0)
    base.update(kw)
    return B.moe_config(**base)


def test_workspace_sizes_scale_with_config():
    a = M.moe_workspace_size(_cfg())
    b = M.moe_workspace_size(_cfg(max_tokens=8192))
    assert 0 < a < b
    assert M.moe_saved_size(_cfg()) > 0


@pytest.mark.parametrize("kw,status", [
    (dict(swiglu_limit=-1.0), 1),         # the clamp bound must be >= 0 (0 = off)
    (dict(swiglu_limit=float("nan")), 1),
    (dict(swiglu_limit=float("inf")), 1),
    (dict(hidden=2000), 2),               # H not a multiple of 128
    (dict(inter=1000), 2),                # I not a multiple of 64
    (dict(topk=0), 1),
    (dict(num_experts=2048), 2),
    (dict(topk=8, num_experts=4), 2),
    (dict(max_tokens=-1), 1),
])
def test_bad_configs_rejected(kw, status):
    with pytest.raises(B.MoeError) as ei:
        M.moe_workspace_size(_cfg(**kw))
    assert ei.value.status == status


def test_swiglu_limit_accepted():
    assert M.moe_workspace_size(_cfg(swiglu_limit=7.0)) == M.moe_workspace_size(_cfg())


def test_null_arguments_rejected():
    L = M.load()
    assert L.moe_workspace_size(None, None) == 1
    h = ctypes.c_void_p()
    assert L.moe_create(ctypes.byref(_cfg()), None, 0, ctypes.byref(h)) == 1
    assert L.moe_forward(None, 0, None, None, None, None, None, None, None) == 1
    assert L.moe_backward(None, None, None, None, None, None, None) == 1
    p = ctypes.c_void_p()
    assert L.moe_host_pipe_create(None, 16, None, 0, ctypes.byref(p)) == 1
    assert L.moe_host_step(None, *([None] * 10)) == 1
    assert L.moe_host_pipe_sync(None) == 1
    assert L.moe_handle_config(None, ctypes.byref(_cfg())) == 1
    assert L.moe_selftest_timeout(None, None) == 1


def test_host_pipe_sizes():
    """Two staging sets of T rows and one saved state: the size grows with T by
    2 x (4 [T,H] bf16 + 2 [T,E] fp32 + 1 [T,E] byte) per token, and T must lie in
    [1, max_tokens]."""
    c = _cfg()
    a, b = M.moe_host_pipe_size(c, 1024), M.moe_host_pipe_size(c, 2048)
    per_token = 2 * (4 * c.hidden * 2 + 2 * c.num_experts * 4 + c.num_experts)
    assert b - a == pytest.approx(1024 * per_token, abs=2 * 14 * 256)   # 256-byte rounding of 14 buffers
    assert a > M.moe_saved_size(c)
    for T in (0, c.max_tokens + 1):
        with pytest.raises(B.MoeError) as ei:
            M.moe_host_pipe_size(c, T)
        assert ei.value.status == 1


def _c_layout(tmp_path):
    """sizeof / offsetof of the ABI structs as a C compiler lays them out from include/moe.h."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = {
        "moe_config": ["max_tokens", "hidden", "num_experts", "topk", "inter", "routed_wtype", "swiglu_limit",
                       "recompute_dispatch", "act_precision", "no_shared_expert"],
        "moe_wview": ["data", "expert_stride", "row_stride", "scale", "col_data", "col_scale", "expert_ptrs"],
        "moe_weights": ["shared_gate", "shared_up", "shared_down", "routed_gate", "routed_up", "routed_down",
                        "shared_output_gate"],
        "moe_main_grads": [n for n, _ in B.moe_main_grads._fields_],
    }
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "moe.h"', "int main(void) {"]
    for s, fs in fields.items():
        lines.append(f'printf("{s} size %zu\\n", sizeof({s}));')
        for f in fs:
            lines.append(f'printf("{s} {f} %zu\\n", offsetof({s}, {f}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    return {tuple(l.split()[:2]): int(l.split()[2]) for l in out.splitlines()}


def test_ctypes_structs_match_the_c_header(tmp_path):
    """The binding's ctypes structs have the size and field offsets the C header
    gives, so every argument is marshalled where the library reads it."""
    c = _c_layout(tmp_path)
    for s in (B.moe_config, B.moe_wview, B.moe_weights, B.moe_main_grads):
        assert c[(s.__name__, "size")] == ctypes.sizeof(s), s.__name__
        for f, _ in s._fields_:
            assert c[(s.__name__, f)] == getattr(s, f).offset, (s.__name__, f)


def test_no_shared_expert_flag():
    """Without a shared expert the row buffers lose their shared region (T rows of
    every per-row buffer); 0 and 1 are the only values."""
    c = _cfg()
    assert M.moe_workspace_size(_cfg(no_shared_expert=1)) < M.moe_workspace_size(c)
    assert M.moe_saved_size(_cfg(no_shared_expert=1)) < M.moe_saved_size(c)
    with pytest.raises(M.MoeError) as ei:
        M.moe_workspace_size(_cfg(no_shared_expert=2))
    assert ei.value.status == 1


def test_recompute_dispatch_flag():
    full = M.moe_saved_size(_cfg())
    small = M.moe_saved_size(_cfg(recompute_dispatch=1))
    assert 0 < small * 100 < full                    # the saved state keeps only the routing
    assert M.moe_workspace_size(_cfg(recompute_dispatch=1)) > M.moe_workspace_size(_cfg())
    with pytest.raises(M.MoeError) as ei:
        M.moe_saved_size(_cfg(recompute_dispatch=2))
    assert ei.value.status == 1


def test_act_precision_flag():
    """fp32 activations (the default) keep [g|u] in fp32 in the saved state and need
    the lo-term and fp32 row buffers in the workspace; other values are rejected."""
    fp32 = _cfg()
    bf16 = _cfg(act_precision=M.binding.MOE_ACT_BF16)
    assert M.moe_saved_size(fp32) > M.moe_saved_size(bf16)
    assert M.moe_workspace_size(fp32) > M.moe_workspace_size(bf16)
    with pytest.raises(M.MoeError) as ei:
        M.moe_saved_size(_cfg(act_precision=2))
    assert ei.value.status == 1


def test_mx_expert_tables_pointer_layout():
    """set_mx_expert_tables: 4E pointers per view in the ABI order (rowwise payloads,
    columnwise payloads, rowwise scales, columnwise scales), strides checked."""
    import torch
    E, N, K = 3, 64, 128
    q = [torch.zeros((N, K), dtype=torch.uint8) for _ in range(E)]
    cq = [torch.zeros((N, K), dtype=torch.uint8) for _ in range(E)]
    sc = [torch.zeros((N, K // 32), dtype=torch.uint8) for _ in range(E)]
    csc = [torch.zeros((N // 32, K), dtype=torch.uint8) for _ in range(E)]
    w = B.moe_weights()
    M.set_mx_expert_tables(w, gate=(q, cq, sc, csc))
    v = w.routed_gate
    assert v.row_stride == K and v.data is None and v.expert_stride == 0
    arr = ctypes.cast(v.expert_ptrs, ctypes.POINTER(ctypes.c_void_p))
    want = [t.data_ptr() for t in q + cq + sc + csc]
    assert [arr[i] for i in range(4 * E)] == want
    bad = [torch.zeros((N, K // 16), dtype=torch.uint8) for _ in range(E)]   # wrong scale row stride
    with pytest.raises(ValueError):
        M.set_mx_expert_tables(B.moe_weights(), up=(q, cq, bad, csc))


def test_a_c_program_links_and_calls_the_library(tmp_path):
    """A plain C caller: compiled against include/moe.h, linked against libmoe.so,
    it queries sizes, gets the argument errors of the header's contract and the
    kernel names -- everything that needs no GPU."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    M.load()
    lib = B.lib_path()
    src = tmp_path / "caller.c"
    src.write_text(r"""
#include <stdio.h>
#include "moe.h"
int main(void) {
    moe_config c = {4096, 2048, 96, 6, 1024, MOE_W_BF16, 0.0f, 0, MOE_ACT_FP32, 0};
    size_t ws = 0, sv = 0, pipe = 0;
    if (moe_workspace_size(&c, &ws) != MOE_OK || ws == 0) return 1;
    if (moe_saved_size(&c, &sv) != MOE_OK || sv == 0) return 2;
    if (moe_host_pipe_size(&c, 4096, &pipe) != MOE_OK || pipe <= sv) return 3;
    if (moe_workspace_size(NULL, &ws) != MOE_ERR_INVALID_ARG) return 4;
    c.hidden = 2000;                                   /* not a multiple of 128 */
    if (moe_workspace_size(&c, &ws) != MOE_ERR_UNSUPPORTED) return 5;
    if (moe_forward(NULL, 0, NULL, NULL, NULL, NULL, NULL, NULL, NULL) != MOE_ERR_INVALID_ARG) return 6;
    for (int i = 0; i < MOE_K_COUNT; ++i)
        if (!moe_kernel_name(i)) return 7;
    printf("%s %s\n", moe_kernel_name(MOE_K_WGRAD_FC1_ROUTED), moe_status_string(MOE_ERR_ROUTING));
    return 0;
}
""")
    exe = tmp_path / "caller"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), lib,
                    "-Wl,-rpath," + os.path.dirname(lib), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, (r.returncode, r.stderr)
    assert r.stdout.split()[0] == "gemm_wgrad_fc1_routed"
