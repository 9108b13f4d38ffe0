"""fp64 CPU oracle for ring-chunked exact attention and the Ulysses exchange.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference legs of ``bench.py`` call this package; the
product path (``context_attention_fwd_gb300``) never imports it and shares
no code with it.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over rows); this
module compiles it with gcc on first use and marshals torch CPU tensors to it.
Every tensor argument is a *logical* ``[B, S, H, D]`` view; its strides say
how it is stored, so ``[B,S,H,D]`` and sequence-first ``[S,B,H,D]`` storage
go through the same routine (``.permute(1, 0, 2, 3)`` of an ``[S,B,H,D]``
tensor is such a view).

Parity status of each routine (what pins it is in ``tests/test_oracle_pins.py``):
  attn_fwd, attn_bwd, ring_fwd, ring_bwd, lse_merge, fwd_rows, dq_rows,
  dkv_rows, seq_head_exchange -- all pinned; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.c_void_p
_i = ctypes.c_int
_d = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, -fopenmp)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            for name in ("oracle_attn_fwd", "oracle_attn_bwd", "oracle_attn_fwd_rows",
                         "oracle_attn_dq_rows", "oracle_attn_dkv_rows", "oracle_ring_fwd",
                         "oracle_lse_merge", "oracle_ring_bwd", "oracle_seq_head_exchange"):
                getattr(lib, name).restype = ctypes.c_int
            lib.oracle_set_threads.restype = None
            _lib = lib
    return _lib


def set_threads(n: int) -> None:
    """OpenMP threads for the oracle's loops run from this thread (the
    arithmetic does not depend on it)."""
    _load().oracle_set_threads(int(n))


def _f64(t: torch.Tensor) -> torch.Tensor:
    """Exact fp64 copy of a [B,S,H,D] view, keeping its storage order."""
    assert t.dim() == 4 and t.stride(3) == 1, "D must be the contiguous dimension"
    return t.detach().to("cpu").to(torch.float64)


def _strides(t: torch.Tensor):
    assert t.stride(3) == 1
    return (ctypes.c_long * 3)(t.stride(0), t.stride(1), t.stride(2))


def _ptr(t: torch.Tensor):
    return ctypes.c_void_p(t.data_ptr())


def _like(t: torch.Tensor) -> torch.Tensor:
    return torch.empty_strided(t.shape, t.stride(), dtype=torch.float64)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments (rc={rc})")


def default_scale(D: int) -> float:
    """1/sqrt(D): the scaled-dot-product default the pages' reference uses."""
    return 1.0 / math.sqrt(D)


def chunk_offsets(S: int, P: int):
    """array_split chunking: the first S mod P chunks are one row longer."""
    if P < 1 or P > S:
        raise ValueError("need 1 <= P <= S")
    base, extra = divmod(S, P)
    off = [0]
    for c in range(P):
        off.append(off[-1] + base + (1 if c < extra else 0))
    return off


def _dims(q, k):
    B, S, Hq, D = q.shape
    assert k.shape[0] == B and k.shape[1] == S and k.shape[3] == D
    return B, S, Hq, k.shape[2], D


def attn_fwd(q, k, v, scale=None, causal=False):
    """Full-sequence attention forward -> (out fp64 [B,S,Hq,D] in q's storage order, lse [B,Hq,S])."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    assert k.stride() == v.stride()
    B, S, Hq, Hkv, D = _dims(q, k)
    scale = default_scale(D) if scale is None else scale
    out = _like(q)
    lse = torch.empty(B, Hq, S, dtype=torch.float64)
    rc = lib.oracle_attn_fwd(_i(B), _i(S), _i(Hq), _i(Hkv), _i(D), _d(scale), _i(int(causal)),
                             _ptr(q), _strides(q), _ptr(k), _ptr(v), _strides(k),
                             _ptr(out), _strides(out), _ptr(lse))
    _check(rc, "attn_fwd")
    return out, lse


def attn_bwd(q, k, v, dout, scale=None, causal=False):
    """Analytic backward of the full-sequence definition -> (dq, dk, dv) fp64."""
    lib = _load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    assert k.stride() == v.stride()
    B, S, Hq, Hkv, D = _dims(q, k)
    scale = default_scale(D) if scale is None else scale
    dq, dk, dv = _like(q), _like(k), _like(k)
    rc = lib.oracle_attn_bwd(_i(B), _i(S), _i(Hq), _i(Hkv), _i(D), _d(scale), _i(int(causal)),
                             _ptr(q), _strides(q), _ptr(k), _ptr(v), _strides(k),
                             _ptr(dout), _strides(dout), _ptr(dq), _strides(dq),
                             _ptr(dk), _ptr(dv), _strides(dk))
    _check(rc, "attn_bwd")
    return dq, dk, dv


def _index_arrays(rows):
    n = len(rows)
    cols = list(zip(*rows)) if n else ([], [], [])
    return n, [(ctypes.c_int * n)(*c) for c in cols]


def fwd_rows(q, k, v, rows, scale=None, causal=False):
    """out and lse of sampled query rows; rows = [(b, h, s), ...]."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, S, Hq, Hkv, D = _dims(q, k)
    scale = default_scale(D) if scale is None else scale
    n, (bi, hi, si) = _index_arrays(rows)
    out = torch.empty(n, D, dtype=torch.float64)
    lse = torch.empty(n, dtype=torch.float64)
    rc = lib.oracle_attn_fwd_rows(_i(B), _i(S), _i(Hq), _i(Hkv), _i(D), _d(scale), _i(int(causal)),
                                  _ptr(q), _strides(q), _ptr(k), _ptr(v), _strides(k),
                                  _i(n), bi, hi, si, _ptr(out), _ptr(lse))
    _check(rc, "fwd_rows")
    return out, lse


def dq_rows(q, k, v, dout, rows, scale=None, causal=False):
    """dq of sampled query rows; rows = [(b, h, s), ...]."""
    lib = _load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, S, Hq, Hkv, D = _dims(q, k)
    scale = default_scale(D) if scale is None else scale
    n, (bi, hi, si) = _index_arrays(rows)
    dq = torch.empty(n, D, dtype=torch.float64)
    rc = lib.oracle_attn_dq_rows(_i(B), _i(S), _i(Hq), _i(Hkv), _i(D), _d(scale), _i(int(causal)),
                                 _ptr(q), _strides(q), _ptr(k), _ptr(v), _strides(k),
                                 _ptr(dout), _strides(dout), _i(n), bi, hi, si, _ptr(dq))
    _check(rc, "dq_rows")
    return dq


def dkv_rows(q, k, v, dout, rows, scale=None, causal=False):
    """dk, dv of sampled key rows; rows = [(b, h_kv, s), ...]."""
    lib = _load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, S, Hq, Hkv, D = _dims(q, k)
    scale = default_scale(D) if scale is None else scale
    n, (bi, hi, si) = _index_arrays(rows)
    dk = torch.empty(n, D, dtype=torch.float64)
    dv = torch.empty(n, D, dtype=torch.float64)
    rc = lib.oracle_attn_dkv_rows(_i(B), _i(S), _i(Hq), _i(Hkv), _i(D), _d(scale), _i(int(causal)),
                                  _ptr(q), _strides(q), _ptr(k), _ptr(v), _strides(k),
                                  _ptr(dout), _strides(dout), _i(n), bi, hi, si,
                                  _ptr(dk), _ptr(dv))
    _check(rc, "dkv_rows")
    return dk, dv


def _offsets_arg(S, P, offsets):
    off = chunk_offsets(S, P) if offsets is None else list(offsets)
    if len(off) != P + 1:
        raise ValueError("offsets must have P+1 entries")
    return (ctypes.c_int * (P + 1))(*off)


def ring_fwd(q, k, v, P, offsets=None, scale=None, causal=False, partials=False):
    """Ring-scheduled forward with the LSE merge.  Returns (out, lse) and, with
    partials=True, also (part_o [P,B,Hq,S,D], part_lse [P,B,Hq,S]) where
    index i is ring iteration i of each query row's chunk."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, S, Hq, Hkv, D = _dims(q, k)
    scale = default_scale(D) if scale is None else scale
    out = _like(q)
    lse = torch.empty(B, Hq, S, dtype=torch.float64)
    po = torch.empty(P, B, Hq, S, D, dtype=torch.float64) if partials else None
    pl = torch.empty(P, B, Hq, S, dtype=torch.float64) if partials else None
    rc = lib.oracle_ring_fwd(_i(B), _i(S), _i(Hq), _i(Hkv), _i(D), _d(scale), _i(int(causal)),
                             _i(P), _offsets_arg(S, P, offsets), _ptr(q), _strides(q),
                             _ptr(k), _ptr(v), _strides(k), _ptr(out), _strides(out), _ptr(lse),
                             _ptr(po) if partials else None, _ptr(pl) if partials else None)
    _check(rc, "ring_fwd")
    return (out, lse, po, pl) if partials else (out, lse)


def lse_merge(part_o, part_lse, out_like=None):
    """Merge partials [P,B,H,S,D] / [P,B,H,S] -> (out [B,S,H,D], lse [B,H,S])."""
    lib = _load()
    part_o = part_o.to(torch.float64).contiguous()
    part_lse = part_lse.to(torch.float64).contiguous()
    P, B, H, S, D = part_o.shape
    out = torch.empty(B, S, H, D, dtype=torch.float64) if out_like is None else _like(_f64(out_like))
    lse = torch.empty(B, H, S, dtype=torch.float64)
    rc = lib.oracle_lse_merge(_i(B), _i(S), _i(H), _i(D), _i(P), _ptr(part_o), _ptr(part_lse),
                              _ptr(out), _strides(out), _ptr(lse))
    _check(rc, "lse_merge")
    return out, lse


def ring_bwd(q, k, v, out, lse, dout, P, offsets=None, scale=None, causal=False, stale=False):
    """Ring-scheduled backward; stale=True plants the iteration-0 K/V defect."""
    lib = _load()
    q, k, v, out, dout = _f64(q), _f64(k), _f64(v), _f64(out), _f64(dout)
    lse = lse.to(torch.float64).contiguous()
    B, S, Hq, Hkv, D = _dims(q, k)
    scale = default_scale(D) if scale is None else scale
    dq, dk, dv = _like(q), _like(k), _like(k)
    rc = lib.oracle_ring_bwd(_i(B), _i(S), _i(Hq), _i(Hkv), _i(D), _d(scale), _i(int(causal)),
                             _i(P), _offsets_arg(S, P, offsets), _ptr(q), _strides(q),
                             _ptr(k), _ptr(v), _strides(k), _ptr(out), _strides(out), _ptr(lse),
                             _ptr(dout), _strides(dout), _i(int(stale)), _ptr(dq), _strides(dq),
                             _ptr(dk), _ptr(dv), _strides(dk))
    _check(rc, "ring_bwd")
    return dq, dk, dv


def exchanged_shape(B, S, H, D, ring, ulysses, layout):
    W = ring * ulysses
    Sp = -(-S // W) * W
    if layout == "bshd":
        return (ulysses, B, Sp, H // ulysses, D)
    return (ulysses, Sp, B, H // ulysses, D)


def seq_head_exchange(x, ring, ulysses, direction, layout, S=None, B=None, H=None):
    """Bitwise Ulysses exchange of 16-bit data.

    direction 0: x is a logical [B,S,H,D] view (storage order = layout) ->
    returns y of ``exchanged_shape`` (same dtype as x).
    direction 1: x is y -> returns the [B,S,H,D]-shaped tensor stored in
    ``layout`` order (S, B, H must then be given)."""
    lib = _load()
    assert x.element_size() == 2
    if direction == 0:
        B_, S_, H_, D = x.shape
        xs = x.detach().to("cpu")
        ys = exchanged_shape(B_, S_, H_, D, ring, ulysses, layout)
        y = torch.empty(ys, dtype=x.dtype)
        rc = lib.oracle_seq_head_exchange(_i(B_), _i(S_), _i(H_), _i(D), _i(ring), _i(ulysses),
                                          _i(0), _i(0 if layout == "bshd" else 1),
                                          _ptr(xs), _ptr(y), _strides(xs))
        _check(rc, "seq_head_exchange")
        return y
    D = x.shape[-1]
    ys = x.detach().to("cpu").contiguous()
    if layout == "bshd":
        out = torch.zeros(B, S, H, D, dtype=x.dtype)
        view = out
    else:
        out = torch.zeros(S, B, H, D, dtype=x.dtype)
        view = out.permute(1, 0, 2, 3)
    rc = lib.oracle_seq_head_exchange(_i(B), _i(S), _i(H), _i(D), _i(ring), _i(ulysses),
                                      _i(1), _i(0 if layout == "bshd" else 1),
                                      _ptr(ys), _ptr(out), _strides(view))
    _check(rc, "seq_head_exchange")
    return out
