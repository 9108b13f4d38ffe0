"""The backward entry point that allocates nothing (ctx_attn_bwd_noalloc).

Some callers cannot allocate device memory themselves (a framework owns the
memory pool, or the implicit synchronisation of cudaFree is not allowed on
their path); this entry point takes its scratch from a fixed device array
inside the library.  The test calls it through the C ABI twice in a row and
compares each result with the regular ctx_attn_bwd, which gets a workspace
allocated by the caller, and checks that an oversized problem is refused.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

import context_attention_fwd_gb300 as ctx
from seeded_inputs import AttnShape, attn_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-2  # the tolerance the parity tests use


def _close(got, ref, name):
    g, r = got.double().cpu(), ref.double().cpu()
    nrm = ((g - r).norm() / r.norm()).item()
    mx = ((g - r).abs().max() / r.abs().max()).item()
    assert nrm <= TOL and mx <= TOL, f"{name}: norm-rel {nrm:.3e}, max-rel {mx:.3e}"


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = ctx.load_library(build_if_missing=True)
    lib.ctx_attn_bwd_noalloc.argtypes = [ctypes.POINTER(ctx._Tensor)] * 4 + [
        ctypes.c_void_p, ctypes.POINTER(ctx._Tensor), ctypes.c_int, ctypes.POINTER(ctypes.c_int),
        ctypes.c_int, ctypes.c_int, ctypes.c_float] + [ctypes.POINTER(ctx._Tensor)] * 3 + [ctypes.c_void_p]
    lib.ctx_attn_bwd_noalloc.restype = ctypes.c_int
    return lib


def _noalloc(lib, q, k, v, out, lse, do, P, causal=False):
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    d = ctx._desc
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.ctx_attn_bwd_noalloc(ctypes.byref(d(q)), ctypes.byref(d(k)), ctypes.byref(d(v)),
                                  ctypes.byref(d(out)), ctypes.c_void_p(lse.data_ptr()),
                                  ctypes.byref(d(do)), P, None, 0, int(causal), 0.0, ctypes.byref(d(dq)),
                                  ctypes.byref(d(dk)), ctypes.byref(d(dv)), stream)
    return rc, (dq, dk, dv)


def test_noalloc_backward_matches_regular_backward_twice(lib):
    sh = AttnShape(B=2, S=1001, Hq=4, Hkv=2, D=128, P=4)
    q, k, v, do = (t.cuda() for t in attn_inputs(sh, seed=31))
    out, lse = ctx.attn_fwd(q, k, v, sh.P)
    ref = ctx.attn_bwd(q, k, v, out, lse, do, sh.P)  # workspace allocated by the caller
    torch.cuda.synchronize()
    for call in range(2):  # the second call finds the first call's data in the array
        rc, got = _noalloc(lib, q, k, v, out, lse, do, sh.P)
        assert rc == 0, ctx._status_text(rc)
        torch.cuda.synchronize()
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            _close(g, r, f"{name} (call {call + 1})")
    assert ctx.device_status() == 0


def test_noalloc_refuses_problems_beyond_its_scratch(lib):
    # S=32760, H=24, D=128 needs ~420 MB of scratch, above the 64 MiB array;
    # the call is refused before any launch, so placeholder pointers suffice.
    fake = 1 << 20
    q = ctx._Tensor(fake, 1, 32760, 24, 128, 0, 0, 0)
    lse = ctypes.c_void_p(fake)
    rc = lib.ctx_attn_bwd_noalloc(ctypes.byref(q), ctypes.byref(q), ctypes.byref(q), ctypes.byref(q),
                                  lse, ctypes.byref(q), 8, None, 0, 0, 0.0, ctypes.byref(q),
                                  ctypes.byref(q), ctypes.byref(q), None)
    assert rc == 3  # CTX_ERR_WORKSPACE
    need = lib.ctx_attn_workspace_size(1, 32760, 24, 24, 128, 8, 0)
    assert need > 64 * 1024 * 1024


def test_noalloc_backward_d256_group_split(lib):
    """Head dimension 256 at 1024 tokens: the backward splits each GQA group
    over CTAs and keeps their partial dK/dV in the scratch as well."""
    sh = AttnShape(B=1, S=1024, Hq=24, Hkv=4, D=256, P=2)
    assert lib.ctx_attn_workspace_size(1, 1024, 24, 4, 256, 2, 0) <= 64 * 1024 * 1024
    q, k, v, do = (t.cuda() for t in attn_inputs(sh, seed=32))
    out, lse = ctx.attn_fwd(q, k, v, sh.P)
    ref = ctx.attn_bwd(q, k, v, out, lse, do, sh.P)
    rc, got = _noalloc(lib, q, k, v, out, lse, do, sh.P)
    assert rc == 0, ctx._status_text(rc)
    torch.cuda.synchronize()
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        _close(g, r, name)
    assert ctx.device_status() == 0


# (shape, causal): every head dimension, causal or not; the D=256 cases split
# the GQA group over CTAs and keep the partial dK/dV in the scratch as well
CASES = [(AttnShape(B=1, S=777, Hq=4, Hkv=2, D=64, P=3), True),
         (AttnShape(B=2, S=600, Hq=2, Hkv=2, D=128, P=2), True),
         (AttnShape(B=1, S=1024, Hq=24, Hkv=4, D=256, P=2), True),
         (AttnShape(B=1, S=1000, Hq=12, Hkv=2, D=256, P=3), False)]


def test_noalloc_calls_in_a_row_leave_nothing_behind(lib):
    """The scratch keeps the last call's contents.  Calls of different head
    dimensions, causal or not, made one after the other (each problem twice,
    and the first problem again at the end) must each give what the regular
    backward gives: nothing a previous call left in the array may leak into
    the next."""
    refs = []
    for i, (sh, causal) in enumerate(CASES):
        assert lib.ctx_attn_workspace_size(sh.B, sh.S, sh.Hq, sh.Hkv, sh.D, sh.P, 0) <= 64 * 1024 * 1024
        q, k, v, do = (t.cuda() for t in attn_inputs(sh, seed=40 + i))
        out, lse = ctx.attn_fwd(q, k, v, sh.P, causal=causal)
        ref = ctx.attn_bwd(q, k, v, out, lse, do, sh.P, causal=causal)
        refs.append(((q, k, v, out, lse, do), ref))
    torch.cuda.synchronize()
    order = [0, 0, 1, 1, 2, 2, 3, 3, 0]
    for n, i in enumerate(order):
        (q, k, v, out, lse, do), ref = refs[i]
        sh, causal = CASES[i]
        rc, got = _noalloc(lib, q, k, v, out, lse, do, sh.P, causal)
        assert rc == 0, ctx._status_text(rc)
        torch.cuda.synchronize()
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            _close(g, r, f"{name} (call {n + 1}: D={sh.D}, causal={causal})")
    assert ctx.device_status() == 0
