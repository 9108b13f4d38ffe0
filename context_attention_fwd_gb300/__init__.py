"""Ring-chunked exact attention for GB300 (sm_103a): thin Python binding.

Every computation runs in the CUDA library ``_build/libctxattn.so`` through
its C ABI (``include/ctx_attn.h``); this module only marshals torch tensors
into ``ctx_tensor_t`` descriptors, allocates outputs and workspace with torch,
and passes the current CUDA stream.  There is no CPU path: if the library is
missing or a call fails, an exception is raised.

Tensors are *logical* ``[B, S, H, D]`` views (``.permute(1, 0, 2, 3)`` of a
sequence-first ``[S, B, H, D]`` tensor is one); their strides tell the
library how they are stored.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

__all__ = [
    "attn_fwd", "attn_bwd", "seq_head_exchange", "exchanged_view", "workspace_size",
    "chunk_offsets", "device_status", "selftest_wait_timeout", "library_path", "load_library",
    "profile_enable", "profile_read", "launch_plan", "debug_set", "kernel_binary_version",
    "CtxError", "FLAG_MATERIALIZE_PARTIALS", "FLAG_KV_ALLGATHER", "DEBUG_SKIP_ARRIVAL",
]

FLAG_MATERIALIZE_PARTIALS = 1
FLAG_KV_ALLGATHER = 2
DEBUG_SKIP_ARRIVAL = 1
LAYOUT_BSHD, LAYOUT_SBHD = 0, 1
_lock = threading.Lock()
_lib = None


class CtxError(RuntimeError):
    def __init__(self, code: int, what: str):
        msg = _status_text(code)
        super().__init__(f"{what}: {msg} (status {code})")
        self.code = code


class _Tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("B", ctypes.c_int64), ("S", ctypes.c_int64),
                ("H", ctypes.c_int64), ("D", ctypes.c_int64), ("stride_b", ctypes.c_int64),
                ("stride_s", ctypes.c_int64), ("stride_h", ctypes.c_int64)]


class _Plan(ctypes.Structure):
    _fields_ = [("fwd_ctas", ctypes.c_int64), ("bwd_ctas", ctypes.c_int64), ("fwd_head_major", ctypes.c_int),
                ("bwd_head_major", ctypes.c_int), ("bwd_group_split", ctypes.c_int)]


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = True):
    """Load libctxattn.so (building it first if asked and it is missing/stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if build_if_missing and not _build.up_to_date():
                _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library not built: {path} (run build())")
            lib = ctypes.CDLL(path)
            P, I, F, SZ, V = ctypes.POINTER, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p
            T = P(_Tensor)
            lib.ctx_attn_fwd.argtypes = [T, T, T, I, P(I), I, I, F, T, V, V, SZ, I, V]
            lib.ctx_attn_bwd.argtypes = [T, T, T, T, V, T, I, P(I), I, I, F, T, T, T, V, SZ, V]
            lib.ctx_seq_head_exchange.argtypes = [T, V, I, I, I, I, V]
            lib.ctx_attn_workspace_size.argtypes = [I, I, I, I, I, I, I]
            lib.ctx_attn_workspace_size.restype = SZ
            lib.ctx_chunk_offsets.argtypes = [I, I, P(I)]
            lib.ctx_exchange_padded_len.argtypes = [ctypes.c_int64, I, I]
            lib.ctx_exchange_padded_len.restype = ctypes.c_int64
            lib.ctx_get_device_status.argtypes = [V]
            lib.ctx_selftest_wait_timeout.argtypes = [ctypes.c_uint, V]
            lib.ctx_selftest_exp2.argtypes = [V, V, V, ctypes.c_int64, V]
            lib.ctx_profile_enable.argtypes = [I]
            lib.ctx_profile_read.argtypes = [I, P(ctypes.c_double), P(I)]
            lib.ctx_attn_launch_plan.argtypes = [I, I, I, I, I, I, P(I), I, P(_Plan)]
            lib.ctx_debug_set.argtypes = [ctypes.c_uint, ctypes.c_uint]
            lib.ctx_kernel_binary_version.argtypes = [P(I)]
            lib.ctx_status_string.argtypes = [I]
            lib.ctx_status_string.restype = ctypes.c_char_p
            for n in ("ctx_attn_fwd", "ctx_attn_bwd", "ctx_seq_head_exchange", "ctx_chunk_offsets",
                      "ctx_get_device_status", "ctx_selftest_wait_timeout", "ctx_profile_enable",
                      "ctx_profile_read", "ctx_selftest_exp2", "ctx_attn_launch_plan", "ctx_debug_set",
                      "ctx_kernel_binary_version"):
                getattr(lib, n).restype = I
            _lib = lib
    return _lib


def _status_text(code: int) -> str:
    try:
        return load_library(False).ctx_status_string(code).decode()
    except Exception:  # library unavailable while formatting an error
        return "error"


def _check(rc: int, what: str):
    if rc != 0:
        raise CtxError(rc, what)


def _desc(t: torch.Tensor, name: str = "tensor", bits16: bool = False) -> _Tensor:
    """ctx_tensor_t of a logical [B,S,H,D] tensor.  The C ABI carries no
    element type (bf16 throughout), so the type is checked here; the
    exchange (bits16) only moves 16-bit elements and takes any such type."""
    if t.dim() != 4:
        raise ValueError(f"{name}: expected a logical [B,S,H,D] tensor, got {t.dim()} dims")
    if bits16 and t.element_size() != 2:
        raise ValueError(f"{name}: the exchange moves 16-bit elements, got {t.dtype}")
    if not bits16 and t.dtype != torch.bfloat16:
        raise ValueError(f"{name}: dtype must be torch.bfloat16, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: tensor must be on a CUDA device")
    if t.stride(3) != 1:
        raise ValueError(f"{name}: the D dimension must be contiguous")
    B, S, H, D = t.shape
    return _Tensor(t.data_ptr(), B, S, H, D, t.stride(0), t.stride(1), t.stride(2))


def _check_types(named):
    """Ranks and element types of a call's [B,S,H,D] tensors."""
    for name, t in named:
        if t.dim() != 4:
            raise ValueError(f"{name}: expected a logical [B,S,H,D] tensor, got {t.dim()} dims")
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name}: dtype must be torch.bfloat16, got {t.dtype}")


def _check_inputs(named, device, lse=None, lse_shape=None):
    """A call's tensors before anything is allocated or launched: ranks and
    element types, the lse buffer, then devices."""
    _check_types(named)
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != tuple(lse_shape)
                            or not lse.is_contiguous()):
        raise ValueError(f"lse: expected a contiguous float32 tensor of shape {tuple(lse_shape)}, "
                         f"got {lse.dtype} {tuple(lse.shape)}")
    for name, t in named + ([("lse", lse)] if lse is not None else []):
        if not t.is_cuda:
            raise ValueError(f"{name}: tensor must be on a CUDA device")
        if t.device != device:
            raise ValueError(f"{name}: on {t.device}, the other tensors are on {device}")


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _offsets(P, offsets):
    if offsets is None:
        return None
    off = list(offsets)
    if len(off) != P + 1:
        raise ValueError("chunk offsets need P+1 entries")
    return (ctypes.c_int * (P + 1))(*off)


def _like_layout(t: torch.Tensor, H: int) -> torch.Tensor:
    """An empty bf16 [B,S,H,D] tensor stored in the same order as t."""
    B, S, _, D = t.shape
    if t.stride(0) >= t.stride(1):  # [B,S,H,D] storage
        return torch.empty(B, S, H, D, dtype=torch.bfloat16, device=t.device)
    return torch.empty(S, B, H, D, dtype=torch.bfloat16, device=t.device).permute(1, 0, 2, 3)


def launch_plan(B, S, Hq, Hkv, D, P, chunk_offsets=None, causal=False) -> dict:
    """How the attention calls of these sizes will be launched (host only):
    CTA counts, launch order (heads first or not) and the D=256 backward's
    GQA group split."""
    plan = _Plan()
    _check(load_library().ctx_attn_launch_plan(B, S, Hq, Hkv, D, P, _offsets(P, chunk_offsets), int(causal),
                                               ctypes.byref(plan)), "ctx_attn_launch_plan")
    return {name: getattr(plan, name) for name, _ in _Plan._fields_}


def workspace_size(B, S, Hq, Hkv, D, P, flags=0) -> int:
    return int(load_library().ctx_attn_workspace_size(B, S, Hq, Hkv, D, P, flags))


def chunk_offsets(S: int, P: int):
    """array_split chunk offsets computed by the library's host code."""
    arr = (ctypes.c_int * (P + 1))()
    _check(load_library().ctx_chunk_offsets(S, P, arr), "ctx_chunk_offsets")
    return list(arr)


def _workspace(nbytes: int, device, workspace):
    if nbytes == 0:
        return None, 0
    if workspace is not None:
        return workspace, workspace.numel() * workspace.element_size()
    return torch.empty(nbytes, dtype=torch.uint8, device=device), nbytes


def attn_fwd(q, k, v, P, chunk_offsets=None, causal=False, scale=None, out=None, lse=None,
             flags=0, workspace=None):
    """Ring-chunked attention forward -> (out bf16 [B,S,Hq,D] like q, lse fp32 [B,Hq,S])."""
    lib = load_library()
    named = [("q", q), ("k", k), ("v", v)] + ([("out", out)] if out is not None else [])
    _check_types(named)
    B, S, Hq, D = q.shape
    _check_inputs(named, q.device, lse, (B, Hq, S))
    out = _like_layout(q, Hq) if out is None else out
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device=q.device) if lse is None else lse
    nbytes = (lib.ctx_attn_workspace_size(B, S, Hq, k.shape[2], D, P, flags)
              if flags & FLAG_MATERIALIZE_PARTIALS else 0)
    ws, wsb = _workspace(nbytes, q.device, workspace)
    rc = lib.ctx_attn_fwd(ctypes.byref(_desc(q)), ctypes.byref(_desc(k)), ctypes.byref(_desc(v)), P,
                          _offsets(P, chunk_offsets), LAYOUT_BSHD, int(causal),
                          float(scale) if scale else 0.0, ctypes.byref(_desc(out)),
                          ctypes.c_void_p(lse.data_ptr()),
                          ctypes.c_void_p(ws.data_ptr() if ws is not None else 0), wsb, flags,
                          _stream(q))
    _check(rc, "ctx_attn_fwd")
    return out, lse


def attn_bwd(q, k, v, out, lse, dout, P, chunk_offsets=None, causal=False, scale=None,
             dq=None, dk=None, dv=None, workspace=None):
    """Ring-chunked attention backward -> (dq, dk, dv) bf16, stored like q / k."""
    lib = load_library()
    named = [("q", q), ("k", k), ("v", v), ("out", out), ("dout", dout)]
    named += [(n, t) for n, t in (("dq", dq), ("dk", dk), ("dv", dv)) if t is not None]
    _check_types(named)
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    _check_inputs(named, q.device, lse, (B, Hq, S))
    dq = _like_layout(q, Hq) if dq is None else dq
    dk = _like_layout(k, Hkv) if dk is None else dk
    dv = _like_layout(k, Hkv) if dv is None else dv
    nbytes = lib.ctx_attn_workspace_size(B, S, Hq, Hkv, D, P, 0)
    ws, wsb = _workspace(nbytes, q.device, workspace)
    rc = lib.ctx_attn_bwd(ctypes.byref(_desc(q)), ctypes.byref(_desc(k)), ctypes.byref(_desc(v)),
                          ctypes.byref(_desc(out)), ctypes.c_void_p(lse.data_ptr()),
                          ctypes.byref(_desc(dout)), P, _offsets(P, chunk_offsets), LAYOUT_BSHD,
                          int(causal), float(scale) if scale else 0.0, ctypes.byref(_desc(dq)),
                          ctypes.byref(_desc(dk)), ctypes.byref(_desc(dv)),
                          ctypes.c_void_p(ws.data_ptr()), wsb, _stream(q))
    _check(rc, "ctx_attn_bwd")
    return dq, dk, dv


def exchanged_shape(B, S, H, D, ring, ulysses, layout):
    Sp = int(load_library().ctx_exchange_padded_len(S, ring, ulysses))
    if layout == "bshd":
        return (ulysses, B, Sp, H // ulysses, D)
    return (ulysses, Sp, B, H // ulysses, D)


def seq_head_exchange(x, ring, ulysses, direction, layout, y=None, S=None, B=None, H=None):
    """Ulysses exchange through the library.

    direction 0: x is a logical [B,S,H,D] view stored in `layout` order;
    returns y (dense, ``exchanged_shape``).  direction 1: x is y; returns the
    logical [B,S,H,D] tensor stored in `layout` order (S, B, H required)."""
    lib = load_library()
    lay = LAYOUT_BSHD if layout == "bshd" else LAYOUT_SBHD
    if direction == 0:
        B_, S_, H_, D = x.shape
        y = torch.empty(exchanged_shape(B_, S_, H_, D, ring, ulysses, layout), dtype=x.dtype,
                        device=x.device) if y is None else y
        rc = lib.ctx_seq_head_exchange(ctypes.byref(_desc(x, "x", bits16=True)), ctypes.c_void_p(y.data_ptr()),
                                       ring, ulysses, 0, lay, _stream(x))
        _check(rc, "ctx_seq_head_exchange")
        return y
    D = x.shape[-1]
    if y is None:
        if layout == "bshd":
            y = torch.empty(B, S, H, D, dtype=x.dtype, device=x.device)
        else:
            y = torch.empty(S, B, H, D, dtype=x.dtype, device=x.device).permute(1, 0, 2, 3)
    if not x.is_contiguous():
        raise ValueError("the exchanged buffer must be dense")
    rc = lib.ctx_seq_head_exchange(ctypes.byref(_desc(y, "y", bits16=True)), ctypes.c_void_p(x.data_ptr()),
                                   ring, ulysses, 1, lay, _stream(x))
    _check(rc, "ctx_seq_head_exchange")
    return y


def exchanged_view(y, S, layout):
    """Logical [U*B, S, H/U, D] view of an exchanged [U,B,Sp,H/U,D] buffer
    (layout "bshd"): every head group's whole sequence, as the attention
    calls consume it.  Pad rows past S are not part of the view."""
    if layout != "bshd":
        raise ValueError("the batched view exists for [B,S,H,D] storage; use y[u] per group")
    U, B, Sp, Hu, D = y.shape
    return y.view(U * B, Sp, Hu, D)[:, :S]


def device_status(stream=None) -> int:
    """Synchronise and read/clear the device status word (0 = ok, 5 = a wait timed out)."""
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    return int(load_library().ctx_get_device_status(ctypes.c_void_p(s)))


def profile_enable(on: bool = True):
    """Start (clearing earlier records) or stop per-launch event timing of the
    attention kernels inside the library."""
    _check(load_library().ctx_profile_enable(int(on)), "ctx_profile_enable")


def profile_read(kernel: str):
    """(total device ms, launches) of the 'fwd' or 'bwd' attention kernel since profile_enable."""
    ms, n = ctypes.c_double(), ctypes.c_int()
    _check(load_library().ctx_profile_read(0 if kernel == "fwd" else 1, ctypes.byref(ms), ctypes.byref(n)),
           "ctx_profile_read")
    return ms.value, n.value


def selftest_exp2(x: torch.Tensor):
    """(polynomial 2^x, SFU 2^x) for a CUDA fp32 tensor x, as the kernels compute them."""
    x = x.contiguous()
    yp, ys = torch.empty_like(x), torch.empty_like(x)
    _check(load_library().ctx_selftest_exp2(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(yp.data_ptr()),
                                            ctypes.c_void_p(ys.data_ptr()), x.numel(), _stream(x)),
           "ctx_selftest_exp2")
    return yp, ys


def selftest_wait_timeout(timeout_us: int = 20000):
    s = torch.cuda.current_stream().cuda_stream
    _check(load_library().ctx_selftest_wait_timeout(timeout_us, ctypes.c_void_p(s)),
           "ctx_selftest_wait_timeout")


def debug_set(flags: int = 0, wait_limit_ms: int = 0):
    """Test-only switches of the library (``ctx_debug_set``): DEBUG_SKIP_ARRIVAL
    makes every attention kernel's producer leave out one load step so that a
    bounded device wait runs out; wait_limit_ms overrides the wait limit
    (0 = default).  ``debug_set()`` restores normal operation."""
    _check(load_library().ctx_debug_set(flags, wait_limit_ms), "ctx_debug_set")


def kernel_binary_version() -> int:
    """cudaFuncAttributes.binaryVersion of the attention kernels on the current device (103 = sm_103a)."""
    v = ctypes.c_int()
    _check(load_library().ctx_kernel_binary_version(ctypes.byref(v)), "ctx_kernel_binary_version")
    return v.value
