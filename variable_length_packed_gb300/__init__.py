"""Packed variable-length (THD) attention forward and padding mask on GB300 (sm_103a).

A thin ctypes binding over ``libthdattn.so`` (``include/thd_attn.h``): it only
marshals torch tensors into pointers, sizes and the current CUDA stream, and
allocates outputs / workspace through torch.  Every step of the computation
runs in the library's CUDA kernels; there is no CPU or PyTorch fallback, and a
missing library or a non-CUDA tensor raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

__all__ = ["thd_attn_fwd", "thd_attn_fwd_noalloc", "thd_padding_mask", "thd_attn_workspace_size", "thd_status_string",
           "ThdError", "library_path", "load_library", "STATUS_WAIT_TIMEOUT"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

THD_OK, THD_ERR_ARG, THD_ERR_UNSUPPORTED, THD_ERR_CUDA, THD_ERR_WORKSPACE = 0, -1, -2, -3, -4
THD_BF16, THD_FP16 = 0, 1
STATUS_WAIT_TIMEOUT = 0x1


class ThdError(RuntimeError):
    def __init__(self, status, what):
        super().__init__(f"{what}: {_lib().thd_status_string(status).decode()} ({status})")
        self.status = status


def library_path():
    return os.path.join(_HERE, "libthdattn.so")


def load_library():
    """Load libthdattn.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with variable_length_packed_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.thd_attn_fwd.restype = I
    lib.thd_attn_fwd.argtypes = [P, P, P, P, P, P, P, P, I, I, F, P, P, I, I, I, I, I, P, SZ, P]
    lib.thd_attn_fwd_noalloc.restype = I
    lib.thd_attn_fwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, I, I, F, P, P, I, I, I, I, I, P]
    lib.thd_padding_mask.restype = I
    lib.thd_padding_mask.argtypes = [P, I, I, P, P]
    lib.thd_attn_workspace_size.restype = SZ
    lib.thd_attn_workspace_size.argtypes = []
    lib.thd_status_string.restype = ctypes.c_char_p
    lib.thd_status_string.argtypes = [I]
    _LIB = lib
    return lib


_lib = load_library


def thd_attn_workspace_size():
    return int(_lib().thd_attn_workspace_size())


def thd_status_string(status):
    return _lib().thd_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _cuda(t, name):
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream_handle(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def thd_attn_fwd(q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded=None,
                 cu_seqlens_kv_padded=None, seq_is_causal=None, batch_size=None, max_seqlen=0,
                 softmax_scale=None, out=None, lse=None, return_lse=True, workspace=None):
    """Packed THD self-attention forward on the current CUDA stream.

    q: [T, Hq, d], k/v: [T, Hkv, d] (bf16 or fp16, CUDA, contiguous).  cu_seqlens_*:
    int32 CUDA tensors with >= batch_size + 1 entries; *_padded: slot starts or None;
    seq_is_causal: bool/uint8 CUDA tensor [>= batch_size] or None (all full-context).
    Returns (out [T, Hq, d], lse [Hq, T] float32 or None).
    """
    for name, t in (("q", q), ("k", k), ("v", v), ("cu_seqlens_q", cu_seqlens_q),
                    ("cu_seqlens_kv", cu_seqlens_kv), ("cu_seqlens_q_padded", cu_seqlens_q_padded),
                    ("cu_seqlens_kv_padded", cu_seqlens_kv_padded), ("seq_is_causal", seq_is_causal),
                    ("out", out), ("lse", lse), ("workspace", workspace)):
        _cuda(t, name)
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise ValueError("q, k, v must be [T, heads, head_dim]")
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (T, Hkv, d) or v.shape != (T, Hkv, d):
        raise ValueError("k and v must be [T, Hkv, head_dim] with q's T and head_dim")
    if q.dtype not in (torch.bfloat16, torch.float16) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share dtype bf16 or fp16")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_kv", cu_seqlens_kv),
                    ("cu_seqlens_q_padded", cu_seqlens_q_padded),
                    ("cu_seqlens_kv_padded", cu_seqlens_kv_padded)):
        if t is not None and t.dtype != torch.int32:
            raise TypeError(f"{name} must be int32")
    if seq_is_causal is not None and seq_is_causal.dtype not in (torch.bool, torch.uint8):
        raise TypeError("seq_is_causal must be bool or uint8")
    if batch_size is None:
        batch_size = cu_seqlens_q.numel() - 1
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(thd_attn_workspace_size(), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        st = _lib().thd_attn_fwd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv),
            _ptr(cu_seqlens_q_padded), _ptr(cu_seqlens_kv_padded), _ptr(seq_is_causal),
            int(batch_size), int(max_seqlen), float(softmax_scale), _ptr(out), _ptr(lse),
            int(T), int(Hq), int(Hkv), int(d), THD_BF16 if q.dtype == torch.bfloat16 else THD_FP16,
            _ptr(workspace), workspace.numel(), _stream_handle(q.device))
    if st != THD_OK:
        raise ThdError(st, "thd_attn_fwd")
    return out, lse


def thd_attn_fwd_noalloc(q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded,
                         seq_is_causal, batch_size, max_seqlen, softmax_scale, out, lse=None):
    """thd_attn_fwd without a workspace: the library uses its fixed per-device buffer.

    For callers that cannot allocate device memory; the caller passes every input and
    output tensor, and nothing is allocated here either.  Calls on one device must not
    overlap on the GPU (they share the buffer).
    """
    for name, t in (("q", q), ("k", k), ("v", v), ("cu_seqlens_q", cu_seqlens_q),
                    ("cu_seqlens_kv", cu_seqlens_kv), ("cu_seqlens_q_padded", cu_seqlens_q_padded),
                    ("cu_seqlens_kv_padded", cu_seqlens_kv_padded), ("seq_is_causal", seq_is_causal),
                    ("out", out), ("lse", lse)):
        _cuda(t, name)
    if out is None:
        raise ValueError("out must be provided")
    T, Hq, d = q.shape
    with torch.cuda.device(q.device):
        st = _lib().thd_attn_fwd_noalloc(
            _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv),
            _ptr(cu_seqlens_q_padded), _ptr(cu_seqlens_kv_padded), _ptr(seq_is_causal),
            int(batch_size), int(max_seqlen), float(softmax_scale), _ptr(out), _ptr(lse),
            int(T), int(Hq), int(k.shape[1]), int(d), THD_BF16 if q.dtype == torch.bfloat16 else THD_FP16,
            _stream_handle(q.device))
    if st != THD_OK:
        raise ThdError(st, "thd_attn_fwd_noalloc")
    return out, lse


def thd_padding_mask(cu_seqlens, batch_size, max_seqlen, mask=None):
    """Boolean padding mask [B, 1, 1, S] (True = padded position), built on the device."""
    _cuda(cu_seqlens, "cu_seqlens")
    _cuda(mask, "mask")
    if cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    if mask is None:
        mask = torch.empty((batch_size, 1, 1, max_seqlen), dtype=torch.bool, device=cu_seqlens.device)
    with torch.cuda.device(cu_seqlens.device):
        st = _lib().thd_padding_mask(_ptr(cu_seqlens), int(batch_size), int(max_seqlen), _ptr(mask),
                                     _stream_handle(cu_seqlens.device))
    if st != THD_OK:
        raise ThdError(st, "thd_padding_mask")
    return mask
