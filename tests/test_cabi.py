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
