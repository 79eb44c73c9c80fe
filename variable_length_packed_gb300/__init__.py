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

__all__ = ["thd_attn_fwd", "thd_attn_bwd", "thd_attn_fwd_noalloc", "thd_attn_noalloc_status", "thd_attn_merge", "thd_padding_mask",
           "thd_padding_mask_cross", "MASK_PADDING", "MASK_PADDING_CAUSAL", "MASK_PADDING_CAUSAL_BOTTOM_RIGHT", "thd_attn_workspace_size", "thd_set_wait_limit_ns", "thd_set_wait_injection", "thd_status_string",
           "ThdError", "library_path", "load_library", "STATUS_WAIT_TIMEOUT"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

THD_OK, THD_ERR_ARG, THD_ERR_UNSUPPORTED, THD_ERR_CUDA, THD_ERR_WORKSPACE = 0, -1, -2, -3, -4
THD_BF16, THD_FP16 = 0, 1
STATUS_WAIT_TIMEOUT = 0x1
# per-sequence mask type codes accepted in seq_is_causal (a bool tensor is codes 0 / 1)
MASK_PADDING, MASK_PADDING_CAUSAL, MASK_PADDING_CAUSAL_BOTTOM_RIGHT = 0, 1, 2


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
    lib.thd_attn_fwd_window.restype = I
    lib.thd_attn_fwd_window.argtypes = [P, P, P, P, P, P, P, P, I, I, F, P, P, I, I, I, I, I, I, I, P, SZ, P]
    lib.thd_attn_fwd_noalloc.restype = I
    lib.thd_attn_fwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, I, I, F, P, P, I, I, I, I, I, P]
    lib.thd_attn_noalloc_status.restype = I
    lib.thd_attn_noalloc_status.argtypes = [P, P]
    lib.thd_attn_bwd.restype = I
    lib.thd_attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, I, I, F, P, P, P, I, I, I, I, I, P, SZ, P]
    lib.thd_attn_bwd_window.restype = I
    lib.thd_attn_bwd_window.argtypes = [P, P, P, P, P, P, P, P, P, P, P, I, I, F, P, P, P, I, I, I, I, I, I, I, P, SZ,
                                        P]
    lib.thd_attn_bwd_workspace_size.restype = SZ
    lib.thd_attn_bwd_workspace_size.argtypes = [I, I, I]
    lib.thd_attn_merge.restype = I
    lib.thd_attn_merge.argtypes = [P, P, P, P, P, P, I, I, I, I, P]
    lib.thd_padding_mask_cross.restype = I
    lib.thd_padding_mask_cross.argtypes = [P, P, I, I, I, P, P, P]
    lib.thd_padding_mask.restype = I
    lib.thd_padding_mask.argtypes = [P, I, I, P, P]
    lib.thd_attn_workspace_size.restype = SZ
    lib.thd_attn_workspace_size.argtypes = []
    lib.thd_set_wait_limit_ns.restype = ctypes.c_uint64
    lib.thd_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.thd_set_wait_injection.restype = ctypes.c_int
    lib.thd_set_wait_injection.argtypes = [ctypes.c_int]
    lib.thd_status_string.restype = ctypes.c_char_p
    lib.thd_status_string.argtypes = [I]
    _LIB = lib
    return lib


_lib = load_library


def thd_attn_workspace_size():
    return int(_lib().thd_attn_workspace_size())


def thd_set_wait_limit_ns(ns):
    """Time limit of one pipeline wait inside the kernels for later calls (0: the default,
    2 s); returns the previous limit.  A short limit makes waits run out on purpose: the
    call then sets STATUS_WAIT_TIMEOUT in its status word and its output is unspecified."""
    return int(_lib().thd_set_wait_limit_ns(int(ns)))


def thd_set_wait_injection(enable):
    """Test setting of the failure path (see include/thd_attn.h): with enable true, every
    CTA of a later attention call makes one wait that runs out, so the call reports
    STATUS_WAIT_TIMEOUT.  Returns the previous setting."""
    return bool(_lib().thd_set_wait_injection(1 if enable else 0))


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


def _check_metadata(batch_size, cu_q, cu_kv=None, pad_q=None, pad_kv=None, flags=None):
    """The kernels read entries 0..batch_size of cu_seqlens*, 0..batch_size-1 of the padded
    starts and the per-sequence flags: the buffers must hold them (longer is fine)."""
    if int(batch_size) < 0:
        raise ValueError("batch_size must be >= 0")
    if int(batch_size) == 0:
        return
    for name, t, need in (("cu_seqlens_q", cu_q, batch_size + 1), ("cu_seqlens_kv", cu_kv, batch_size + 1),
                          ("cu_seqlens_q_padded", pad_q, batch_size), ("cu_seqlens_kv_padded", pad_kv, batch_size),
                          ("seq_is_causal", flags, batch_size)):
        if t is not None and t.numel() < need:
            raise ValueError(f"{name} holds {t.numel()} entries, batch_size {batch_size} needs {need}")


def _check_qkv(q, k, v):
    """q [T, Hq, d], k / v [T, Hkv, d] with q's T and d, one dtype (bf16 or fp16).  The library
    encodes its tensor maps from these sizes, so a k or v shorter than q would be read past
    its end: refused here, before anything is launched.  Returns (T, Hq, Hkv, d)."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch tensor")
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise ValueError("q, k, v must be [T, heads, head_dim]")
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (T, Hkv, d) or tuple(v.shape) != (T, Hkv, d):
        raise ValueError("k and v must be [T, Hkv, head_dim] with q's T and head_dim")
    if q.dtype not in (torch.bfloat16, torch.float16) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share dtype bf16 or fp16")
    return T, Hq, Hkv, d


def _check_metadata_dtypes(cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded, seq_is_causal):
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_kv", cu_seqlens_kv),
                    ("cu_seqlens_q_padded", cu_seqlens_q_padded),
                    ("cu_seqlens_kv_padded", cu_seqlens_kv_padded)):
        if t is not None and (not isinstance(t, torch.Tensor) or t.dtype != torch.int32):
            raise TypeError(f"{name} must be an int32 tensor")
    if seq_is_causal is not None and (not isinstance(seq_is_causal, torch.Tensor)
                                      or seq_is_causal.dtype not in (torch.bool, torch.uint8)):
        raise TypeError("seq_is_causal must be a bool or uint8 tensor")


def _check_out(t, name, shape, dtype, device):
    if t is not None and (tuple(t.shape) != tuple(shape) or t.dtype != dtype or t.device != device):
        raise ValueError(f"{name} must be a {dtype} tensor of shape {tuple(shape)} on {device}")


def _stream_handle(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _window_args(window):
    left, right = (int(window[0]), int(window[1]))
    if left < -1 or right < -1:
        raise ValueError("window extents must be >= -1 (-1: unbounded)")
    return left, right


def thd_attn_fwd(q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded=None,
                 cu_seqlens_kv_padded=None, seq_is_causal=None, batch_size=None, max_seqlen=0,
                 softmax_scale=None, out=None, lse=None, return_lse=True, workspace=None, window=(-1, -1)):
    """Packed THD self-attention forward on the current CUDA stream.

    q: [T, Hq, d], k/v: [T, Hkv, d] (bf16 or fp16, CUDA, contiguous).  cu_seqlens_*:
    int32 CUDA tensors with >= batch_size + 1 entries; *_padded: slot starts or None;
    seq_is_causal: bool/uint8 CUDA tensor [>= batch_size] or None (all full-context), the
    per-sequence mask type: MASK_PADDING (0), MASK_PADDING_CAUSAL (1, top-left) or
    MASK_PADDING_CAUSAL_BOTTOM_RIGHT (2).  q and k/v sequences may differ in length.
    window: (left, right) sliding window around the mask type's diagonal, -1 = unbounded.
    max_seqlen: a hint (never trusted for correctness); 1..256 selects the kernel that packs
    runs of short sequences into shared tiles (see thd_attn_fwd in include/thd_attn.h).
    Returns (out [T, Hq, d], lse [Hq, T] float32 or None).
    """
    T, Hq, Hkv, d = _check_qkv(q, k, v)
    _check_metadata_dtypes(cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded, seq_is_causal)
    for name, t in (("q", q), ("k", k), ("v", v), ("cu_seqlens_q", cu_seqlens_q),
                    ("cu_seqlens_kv", cu_seqlens_kv), ("cu_seqlens_q_padded", cu_seqlens_q_padded),
                    ("cu_seqlens_kv_padded", cu_seqlens_kv_padded), ("seq_is_causal", seq_is_causal),
                    ("out", out), ("lse", lse), ("workspace", workspace)):
        _cuda(t, name)
    if batch_size is None:
        batch_size = cu_seqlens_q.numel() - 1
    _check_metadata(batch_size, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded,
                    seq_is_causal)
    _check_out(out, "out", q.shape, q.dtype, q.device)
    _check_out(lse, "lse", (Hq, T), torch.float32, q.device)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(thd_attn_workspace_size(), dtype=torch.uint8, device=q.device)
    left, right = _window_args(window)
    with torch.cuda.device(q.device):
        st = _lib().thd_attn_fwd_window(
            _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv),
            _ptr(cu_seqlens_q_padded), _ptr(cu_seqlens_kv_padded), _ptr(seq_is_causal),
            int(batch_size), int(max_seqlen), float(softmax_scale), _ptr(out), _ptr(lse),
            int(T), int(Hq), int(Hkv), int(d), THD_BF16 if q.dtype == torch.bfloat16 else THD_FP16,
            left, right, _ptr(workspace), workspace.numel(), _stream_handle(q.device))
    if st != THD_OK:
        raise ThdError(st, "thd_attn_fwd")
    return out, lse


def thd_attn_fwd_noalloc(q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded,
                         seq_is_causal, batch_size, max_seqlen, softmax_scale, out, lse=None):
    """thd_attn_fwd without a workspace: the library uses its fixed per-device buffer.

    For callers that cannot allocate device memory; the caller passes every input and
    output tensor, and nothing is allocated here either.  Calls on one device must not
    overlap on the GPU (they share the buffer).  The argument checks are those of
    thd_attn_fwd.  thd_attn_noalloc_status() reads the buffer's device status word.
    """
    T, Hq, Hkv, d = _check_qkv(q, k, v)
    _check_metadata_dtypes(cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded, seq_is_causal)
    if out is None:
        raise ValueError("out must be provided")
    for name, t in (("q", q), ("k", k), ("v", v), ("cu_seqlens_q", cu_seqlens_q),
                    ("cu_seqlens_kv", cu_seqlens_kv), ("cu_seqlens_q_padded", cu_seqlens_q_padded),
                    ("cu_seqlens_kv_padded", cu_seqlens_kv_padded), ("seq_is_causal", seq_is_causal),
                    ("out", out), ("lse", lse)):
        _cuda(t, name)
    _check_metadata(batch_size, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded,
                    seq_is_causal)
    _check_out(out, "out", q.shape, q.dtype, q.device)
    _check_out(lse, "lse", (Hq, T), torch.float32, q.device)
    with torch.cuda.device(q.device):
        st = _lib().thd_attn_fwd_noalloc(
            _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv),
            _ptr(cu_seqlens_q_padded), _ptr(cu_seqlens_kv_padded), _ptr(seq_is_causal),
            int(batch_size), int(max_seqlen), float(softmax_scale), _ptr(out), _ptr(lse),
            int(T), int(Hq), int(Hkv), int(d), THD_BF16 if q.dtype == torch.bfloat16 else THD_FP16,
            _stream_handle(q.device))
    if st != THD_OK:
        raise ThdError(st, "thd_attn_fwd_noalloc")
    return out, lse


def thd_attn_noalloc_status(device=None):
    """Device status word (STATUS_* bits) of the last thd_attn_fwd_noalloc call on `device`
    that ran before this read: waits for the work queued so far on the current stream."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    word = ctypes.c_uint32(0)
    with torch.cuda.device(dev):
        st = _lib().thd_attn_noalloc_status(ctypes.byref(word), _stream_handle(dev))
    if st != THD_OK:
        raise ThdError(st, "thd_attn_noalloc_status")
    return int(word.value)


def thd_padding_mask(cu_seqlens, batch_size, max_seqlen, mask=None):
    """Boolean padding mask [B, 1, 1, S] (True = padded position), built on the device."""
    _cuda(cu_seqlens, "cu_seqlens")
    _cuda(mask, "mask")
    if cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    _check_metadata(batch_size, cu_seqlens)
    if mask is not None and (mask.numel() != int(batch_size) * int(max_seqlen) or mask.element_size() != 1):
        raise ValueError("mask must hold batch_size * max_seqlen one-byte elements")
    if mask is None:
        mask = torch.empty((batch_size, 1, 1, max_seqlen), dtype=torch.bool, device=cu_seqlens.device)
    with torch.cuda.device(cu_seqlens.device):
        st = _lib().thd_padding_mask(_ptr(cu_seqlens), int(batch_size), int(max_seqlen), _ptr(mask),
                                     _stream_handle(cu_seqlens.device))
    if st != THD_OK:
        raise ThdError(st, "thd_padding_mask")
    return mask


def thd_attn_merge(out_a, lse_a, out_b, lse_b, out=None, lse=None):
    """Merge two partial attention results over disjoint key sets (see thd_attn_merge in
    include/thd_attn.h).  out_*: [T, H, d] bf16/fp16; lse_*: [H, T] float32.  out / lse may
    be out_a / lse_a (in place)."""
    for name, t in (("out_a", out_a), ("lse_a", lse_a), ("out_b", out_b), ("lse_b", lse_b),
                    ("out", out), ("lse", lse)):
        _cuda(t, name)
    if out_a.shape != out_b.shape or out_a.dtype != out_b.dtype or out_a.dim() != 3:
        raise ValueError("out_a and out_b must be [T, H, d] of one dtype")
    T, H, d = out_a.shape
    if lse_a.shape != (H, T) or lse_b.shape != (H, T) or lse_a.dtype != torch.float32 \
            or lse_b.dtype != torch.float32:
        raise ValueError("lse_a and lse_b must be float32 [H, T]")
    _check_out(out, "out", out_a.shape, out_a.dtype, out_a.device)
    _check_out(lse, "lse", (H, T), torch.float32, out_a.device)
    if out is None:
        out = torch.empty_like(out_a)
    if lse is None:
        lse = torch.empty_like(lse_a)
    with torch.cuda.device(out_a.device):
        st = _lib().thd_attn_merge(_ptr(out_a), _ptr(lse_a), _ptr(out_b), _ptr(lse_b), _ptr(out), _ptr(lse),
                                   int(T), int(H), int(d),
                                   THD_BF16 if out_a.dtype == torch.bfloat16 else THD_FP16,
                                   _stream_handle(out_a.device))
    if st != THD_OK:
        raise ThdError(st, "thd_attn_merge")
    return out, lse


def thd_padding_mask_cross(cu_seqlens_q, cu_seqlens_kv, batch_size, max_seqlen_q, max_seqlen_kv,
                           mask_q=None, mask_kv=None):
    """Cross-attention padding masks ([B,1,1,Sq], [B,1,1,Skv]; True = padded position)."""
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_kv", cu_seqlens_kv),
                    ("mask_q", mask_q), ("mask_kv", mask_kv)):
        _cuda(t, name)
    if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_kv.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    dev = cu_seqlens_q.device
    _check_metadata(batch_size, cu_seqlens_q, cu_seqlens_kv)
    for name, m, sl in (("mask_q", mask_q, max_seqlen_q), ("mask_kv", mask_kv, max_seqlen_kv)):
        if m is not None and (m.numel() != int(batch_size) * int(sl) or m.element_size() != 1):
            raise ValueError(f"{name} must hold batch_size * max_seqlen one-byte elements")
    if mask_q is None:
        mask_q = torch.empty((batch_size, 1, 1, max_seqlen_q), dtype=torch.bool, device=dev)
    if mask_kv is None:
        mask_kv = torch.empty((batch_size, 1, 1, max_seqlen_kv), dtype=torch.bool, device=dev)
    with torch.cuda.device(dev):
        st = _lib().thd_padding_mask_cross(_ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), int(batch_size),
                                           int(max_seqlen_q), int(max_seqlen_kv), _ptr(mask_q), _ptr(mask_kv),
                                           _stream_handle(dev))
    if st != THD_OK:
        raise ThdError(st, "thd_padding_mask_cross")
    return mask_q, mask_kv


def thd_attn_bwd(q, k, v, out, lse, dout, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded=None,
                 cu_seqlens_kv_padded=None, seq_is_causal=None, batch_size=None, max_seqlen=0,
                 softmax_scale=None, dq=None, dk=None, dv=None, workspace=None, window=(-1, -1)):
    """Gradients (dq, dk, dv) of thd_attn_fwd for the same batch and window; out / lse are
    the forward's outputs.  head_dim 64 or 128."""
    T, Hq, Hkv, d = _check_qkv(q, k, v)
    _check_metadata_dtypes(cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded, seq_is_causal)
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("lse", lse), ("dout", dout),
                    ("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_kv", cu_seqlens_kv),
                    ("cu_seqlens_q_padded", cu_seqlens_q_padded),
                    ("cu_seqlens_kv_padded", cu_seqlens_kv_padded), ("seq_is_causal", seq_is_causal),
                    ("dq", dq), ("dk", dk), ("dv", dv), ("workspace", workspace)):
        _cuda(t, name)
    if out.dtype != q.dtype or dout.dtype != q.dtype:
        raise TypeError("out and dout must have q's dtype")
    if out.shape != q.shape or dout.shape != q.shape or lse.shape != (Hq, T) or lse.dtype != torch.float32:
        raise ValueError("out / dout must match q; lse must be float32 [Hq, T]")
    if batch_size is None:
        batch_size = cu_seqlens_q.numel() - 1
    _check_metadata(batch_size, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded,
                    seq_is_causal)
    _check_out(dq, "dq", q.shape, q.dtype, q.device)
    _check_out(dk, "dk", k.shape, k.dtype, k.device)
    _check_out(dv, "dv", v.shape, v.dtype, v.device)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = int(_lib().thd_attn_bwd_workspace_size(int(T), int(Hq), int(d)))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    left, right = _window_args(window)
    with torch.cuda.device(q.device):
        st = _lib().thd_attn_bwd_window(
            _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv),
            _ptr(cu_seqlens_q_padded), _ptr(cu_seqlens_kv_padded), _ptr(seq_is_causal), int(batch_size),
            int(max_seqlen), float(softmax_scale), _ptr(dq), _ptr(dk), _ptr(dv), int(T), int(Hq), int(Hkv), int(d),
            THD_BF16 if q.dtype == torch.bfloat16 else THD_FP16, left, right, _ptr(workspace), workspace.numel(),
            _stream_handle(q.device))
    if st != THD_OK:
        raise ThdError(st, "thd_attn_bwd")
    return dq, dk, dv
