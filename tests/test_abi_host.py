"""C-ABI checks that need no GPU: the library loads, exports every function the header
declares, and rejects invalid host arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

pytest.importorskip("torch")
import variable_length_packed_gb300 as vlp  # noqa: E402
from variable_length_packed_gb300 import build as vbuild  # noqa: E402


@pytest.fixture(scope="module")
def lib():
    vbuild.build()
    return vlp.load_library()


def header_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(inc, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(thd_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_exports_every_declared_symbol(lib):
    names = header_functions()
    assert {"thd_attn_fwd", "thd_padding_mask", "thd_attn_workspace_size", "thd_status_string"} <= names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_workspace(lib):
    assert vlp.thd_attn_workspace_size() >= 16
    for s in (0, -1, -2, -3, -4):
        assert vlp.thd_status_string(s).startswith("THD_")


def call_fwd(lib, **over):
    args = dict(q=16, k=16, v=16, cu_q=16, cu_kv=16, pq=None, pkv=None, causal=None, B=1, S=8, scale=0.125,
                out=16, lse=None, T=8, Hq=2, Hkv=2, d=64, dtype=0, ws=16, ws_bytes=256, stream=None)
    args.update(over)
    P = ctypes.c_void_p
    return lib.thd_attn_fwd(P(args["q"]), P(args["k"]), P(args["v"]), P(args["cu_q"]), P(args["cu_kv"]),
                            P(args["pq"]), P(args["pkv"]), P(args["causal"]), args["B"], args["S"],
                            args["scale"], P(args["out"]), P(args["lse"]), args["T"], args["Hq"],
                            args["Hkv"], args["d"], args["dtype"], P(args["ws"]), args["ws_bytes"],
                            P(args["stream"]))


@pytest.mark.parametrize("over,status", [
    (dict(B=-1), -1), (dict(T=-1), -1), (dict(S=-1), -1), (dict(Hq=0), -1), (dict(Hkv=0), -1),
    (dict(scale=float("nan")), -1), (dict(scale=0.0), -1), (dict(scale=-1.0), -1),
    (dict(scale=float("inf")), -1), (dict(dtype=7), -2), (dict(d=4), -2), (dict(d=136), -2),
    (dict(d=60), -2), (dict(Hq=3, Hkv=2), -2), (dict(q=None), -1), (dict(out=None), -1),
    (dict(cu_q=None), -1), (dict(q=24), -1), (dict(out=12), -1), (dict(lse=6), -1),
    (dict(ws=None), -4), (dict(ws=8), -4), (dict(ws_bytes=8), -4),
    (dict(T=2**31 - 1, Hq=256, Hkv=256), -2),
])
def test_invalid_arguments_rejected_before_launch(lib, over, status):
    assert call_fwd(lib, **over) == status


def test_trivial_calls_launch_nothing(lib):
    # no rows: nothing to write, returns OK without any CUDA call (works without a GPU)
    assert call_fwd(lib, T=0, q=None, k=None, v=None, out=None) == 0
    P = ctypes.c_void_p
    assert lib.thd_padding_mask(P(None), 0, 8, P(None), P(None)) == 0
    assert lib.thd_padding_mask(P(16), 4, 0, P(16), P(None)) == 0
    assert lib.thd_padding_mask(P(16), -1, 8, P(16), P(None)) == -1
    assert lib.thd_padding_mask(P(16), 4, -2, P(16), P(None)) == -1
    assert lib.thd_padding_mask(P(None), 4, 8, P(16), P(None)) == -1
    assert lib.thd_padding_mask(P(16), 4, 8, P(None), P(None)) == -1
    assert lib.thd_padding_mask(P(18), 4, 8, P(16), P(None)) == -1


def test_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros(4, 1, 64, dtype=torch.bfloat16)
    cu = torch.tensor([0, 4], dtype=torch.int32)
    with pytest.raises(TypeError):
        vlp.thd_attn_fwd(x, x, x, cu, cu)
    with pytest.raises(TypeError):
        vlp.thd_padding_mask(cu, 1, 4)


def test_bwd_and_merge_arguments_rejected_before_launch(lib):
    P = ctypes.c_void_p
    assert lib.thd_attn_bwd_workspace_size(100, 4, 128) == 256 + 1792 + 204800
    assert lib.thd_attn_bwd_workspace_size(-1, 4, 128) == 0

    def bwd(**over):
        a = dict(ptr=16, B=1, S=8, scale=0.1, T=100, Hq=4, Hkv=2, d=128, dtype=0, ws=256,
                 ws_bytes=lib.thd_attn_bwd_workspace_size(100, 4, 128), lse=16)
        a.update(over)
        x = a["ptr"]
        return lib.thd_attn_bwd(P(x), P(x), P(x), P(x), P(a["lse"]), P(x), P(x), P(x), P(None), P(None), P(None),
                                a["B"], a["S"], ctypes.c_float(a["scale"]), P(x), P(x), P(x), a["T"], a["Hq"],
                                a["Hkv"], a["d"], a["dtype"], P(a["ws"]), ctypes.c_size_t(a["ws_bytes"]), P(None))
    assert bwd(d=96) == -2 and bwd(d=40) == -2 and bwd(Hq=3) == -2 and bwd(dtype=5) == -2
    assert bwd(B=-1) == -1 and bwd(scale=0.0) == -1 and bwd(lse=None) == -1 and bwd(ptr=24) == -1
    assert bwd(ws=128) == -4 and bwd(ws_bytes=1024) == -4 and bwd(ws=None) == -4
    assert bwd(T=0, ptr=None, lse=None) == 0

    def merge(**over):
        a = dict(ptr=16, lse=16, T=10, H=2, d=64, dtype=0)
        a.update(over)
        return lib.thd_attn_merge(P(a["ptr"]), P(a["lse"]), P(a["ptr"]), P(a["lse"]), P(a["ptr"]), P(a["lse"]),
                                  a["T"], a["H"], a["d"], a["dtype"], P(None))
    assert merge(d=4) == -2 and merge(d=136) == -2 and merge(dtype=3) == -2
    assert merge(T=-1) == -1 and merge(H=0) == -1 and merge(ptr=8) == -1 and merge(lse=2) == -1
    assert merge(ptr=None) == -1 and merge(T=0, ptr=None, lse=None) == 0
    assert lib.thd_padding_mask_cross(P(16), P(16), -1, 4, 4, P(16), P(16), P(None)) == -1
    assert lib.thd_padding_mask_cross(P(16), P(16), 0, 4, 4, P(None), P(None), P(None)) == 0
    assert lib.thd_padding_mask_cross(P(None), P(16), 2, 4, 4, P(16), P(16), P(None)) == -1


def test_window_arguments_rejected_before_launch(lib):
    P = ctypes.c_void_p
    F = ctypes.c_float

    def fwd(left, right, T=8):
        return lib.thd_attn_fwd_window(P(16), P(16), P(16), P(16), P(16), P(None), P(None), P(None), 1, 8, F(0.125),
                                       P(16), P(None), T, 2, 2, 64, 0, left, right, P(16), ctypes.c_size_t(256),
                                       P(None))
    assert fwd(-2, -1) == -1 and fwd(0, -5) == -1
    assert fwd(-1, -1, T=0) == 0 and fwd(3, 0, T=0) == 0      # valid windows, nothing to do

    def bwd(left, right):
        ws = lib.thd_attn_bwd_workspace_size(100, 4, 128)
        return lib.thd_attn_bwd_window(P(16), P(16), P(16), P(16), P(16), P(16), P(16), P(16), P(None), P(None),
                                       P(None), 1, 8, F(0.1), P(16), P(16), P(16), 100, 4, 2, 128, 0, left, right,
                                       P(256), ctypes.c_size_t(ws), P(None))
    assert bwd(-3, 0) == -1 and bwd(2, -2) == -1
    with pytest.raises(ValueError):
        vlp._window_args((-2, 0))


def _qkv_cpu(T=16, Hq=2, Hkv=2, d=64, dtype=None):
    import torch
    dtype = dtype or torch.bfloat16
    return (torch.zeros((T, Hq, d), dtype=dtype), torch.zeros((T, Hkv, d), dtype=dtype),
            torch.zeros((T, Hkv, d), dtype=dtype))


@pytest.mark.parametrize("fn", ["thd_attn_fwd", "thd_attn_fwd_noalloc"])
def test_binding_refuses_bad_qkv_before_any_launch(fn):
    """Both forward wrappers check q/k/v shapes and dtypes, and the metadata dtypes, before
    anything reaches the library: a k or v with fewer tokens than q (the library would read
    past its end), a head_dim mismatch, mixed or fp32 dtypes, int64 cu_seqlens, a float
    per-sequence flag.  The tensors here are on the CPU; each case fails on its own check,
    ahead of the CUDA-tensor check."""
    import torch
    call = getattr(vlp, fn)
    cu = torch.tensor([0, 16], dtype=torch.int32)

    def run(q, k, v, cu_q=cu, flags=None):
        if fn == "thd_attn_fwd":
            return call(q, k, v, cu_q, cu_q, None, None, flags, 1, 16, 0.125)
        return call(q, k, v, cu_q, cu_q, None, None, flags, 1, 16, 0.125, torch.empty_like(q))

    q, k, v = _qkv_cpu()
    with pytest.raises(ValueError, match="k and v"):
        run(q, k[:8], v)                                # short k
    with pytest.raises(ValueError, match="k and v"):
        run(q, k, v[:15])                               # short v
    with pytest.raises(ValueError, match="k and v"):
        run(q, k[:, :, :32], v)                         # head_dim mismatch
    with pytest.raises(ValueError, match=r"\[T, heads, head_dim\]"):
        run(q, k.reshape(16, 128), v)
    with pytest.raises(TypeError, match="dtype"):
        run(q, k.half(), v)                             # mixed dtypes
    with pytest.raises(TypeError, match="dtype"):
        run(*(t.float() for t in (q, k, v)))            # fp32
    with pytest.raises(TypeError, match="int32"):
        run(q, k, v, cu_q=cu.long())                    # int64 metadata
    with pytest.raises(TypeError, match="seq_is_causal"):
        run(q, k, v, flags=torch.zeros(1, dtype=torch.float32))
    with pytest.raises(TypeError, match="CUDA tensor"):
        run(q, k, v)                                    # valid shapes, but no CPU path


def test_noalloc_status_rejects_null(lib):
    assert lib.thd_attn_noalloc_status(None, None) == vlp.THD_ERR_ARG


def test_wait_injection_setter_round_trip():
    """The failure-path test setting is off by default and returns its previous value
    (host state only: no launch)."""
    assert vlp.thd_set_wait_injection(True) is False
    assert vlp.thd_set_wait_injection(False) is True
    assert vlp.thd_set_wait_injection(False) is False
