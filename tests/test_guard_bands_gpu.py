"""Out-of-bounds write checks with guard bands (sentinel canaries).

Every output (out, lse, dq, dk, dv, and the exchange's y) is carved out of
a larger device buffer filled with a sentinel pattern: a band before and
after it, and gaps inside each row (a head stride larger than D, a row
stride larger than the heads) so that the output is a strided view.  After the
call every byte outside the view must still hold the sentinel, and the view
must hold the oracle's values.  The cases are the ones where tails and
strides are awkward: uneven chunks (sequence-first 1001 rows in 4 chunks),
the 4095-row chunks of the long-context workload (tile tail of 127 rows),
64 single-tile chunks, strided head-group views of the fused exchange, and
padded exchange shards.  Padding changes results unless it is masked
(diffusers PR #12443, "Fix Flux Context Parallel Bug ...", the padding
discussion); these checks make sure no padded row or column is written
either.
"""
import pytest
import torch

import context_attention_fwd_gb300 as ctx
import oracle
from seeded_inputs import AttnShape, attn_inputs, exchange_input
from test_parity_gpu import LSE_TOL, check

pytestmark = pytest.mark.gpu

GUARD = 4096  # elements of sentinel before and after every output
SENT16 = -12345  # int16 sentinel for bf16 buffers (a NaN-free bf16 bit pattern)
SENT32 = -7.25e30  # fp32 sentinel for lse


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ctx.load_library(build_if_missing=True)
    yield
    assert ctx.device_status() == 0


class Guarded:
    """A strided logical [B,S,H,D] bf16 view inside a sentinel-filled buffer.

    Storage is `order` ("bshd" or "sbhd") with gaps: each (b, s) row holds H
    heads at a stride of D + pad_d elements, plus pad_row extra elements."""

    def __init__(self, B, S, H, D, order="bshd", pad_d=16, pad_row=8):
        dh = D + pad_d
        row = H * dh + pad_row
        n = B * S * row
        self.buf = torch.full((GUARD + n + GUARD,), SENT16, dtype=torch.int16, device="cuda")
        base = self.buf[GUARD:GUARD + n].view(torch.bfloat16)
        if order == "bshd":
            strides = (S * row, row, dh, 1)
        else:
            strides = (row, B * row, dh, 1)
        self.view = base.as_strided((B, S, H, D), strides)
        mark = torch.zeros(GUARD + n + GUARD, dtype=torch.int16, device="cuda")
        mark[GUARD:GUARD + n].as_strided((B, S, H, D), strides).fill_(1)
        self.mask = mark.bool()

    def untouched(self):
        return bool((self.buf[~self.mask] == SENT16).all().item())


class GuardedLse:
    def __init__(self, B, H, S):
        n = B * H * S
        self.buf = torch.full((GUARD + n + GUARD,), SENT32, dtype=torch.float32, device="cuda")
        self.view = self.buf[GUARD:GUARD + n].view(B, H, S)

    def untouched(self):
        return bool((self.buf[:GUARD] == SENT32).all().item() and (self.buf[-GUARD:] == SENT32).all().item())


@pytest.mark.parametrize("sh,causal", [
    (AttnShape(B=1, S=1001, Hq=4, Hkv=2, D=64, P=4, layout="sbhd"), False),
    (AttnShape(B=2, S=1001, Hq=2, Hkv=2, D=128, P=4, layout="sbhd"), True),
    (AttnShape(B=1, S=8190, Hq=2, Hkv=2, D=128, P=2), False),  # two 4095-row chunks: tile tail 127
    (AttnShape(B=1, S=1000, Hq=2, Hkv=1, D=64, P=64), True),   # 64 chunks of one partial tile each
    (AttnShape(B=1, S=777, Hq=4, Hkv=2, D=256, P=3), False),
    (AttnShape(B=1, S=1000, Hq=12, Hkv=2, D=256, P=3), True),  # D=256 backward with the group split
])
def test_outputs_stay_inside_their_views(sh, causal):
    q, k, v, do = attn_inputs(sh)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    out = Guarded(sh.B, sh.S, sh.Hq, sh.D, sh.layout)
    dq = Guarded(sh.B, sh.S, sh.Hq, sh.D, sh.layout)
    dk = Guarded(sh.B, sh.S, sh.Hkv, sh.D, sh.layout, pad_d=32, pad_row=16)
    dv = Guarded(sh.B, sh.S, sh.Hkv, sh.D, sh.layout, pad_d=32, pad_row=16)
    lse = GuardedLse(sh.B, sh.Hq, sh.S)
    ctx.attn_fwd(qd, kd, vd, sh.P, causal=causal, out=out.view, lse=lse.view)
    ctx.attn_bwd(qd, kd, vd, out.view, lse.view, dod, sh.P, causal=causal, dq=dq.view, dk=dk.view, dv=dv.view)
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    for name, g in (("out", out), ("dq", dq), ("dk", dk), ("dv", dv), ("lse", lse)):
        assert g.untouched(), f"{name}: a byte outside the output view was written"
    o_ref, l_ref = oracle.attn_fwd(q, k, v, causal=causal)
    check("out", out.view, o_ref)
    assert (lse.view.double().cpu() - l_ref).abs().max() < LSE_TOL
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), oracle.attn_bwd(q, k, v, do, causal=causal)):
        check(name, g.view, r)


def test_fused_head_group_views_stay_inside():
    """Fused exchange + attention: one call over strided head-group views
    ([U, S, H/U, D] of the un-exchanged tensors, the head group as batch)
    writes each group's out, dq, dk, dv only into its own heads' columns."""
    sh = AttnShape(B=1, S=2000, Hq=8, Hkv=4, D=128, P=4)
    U = 2
    Hu, Hku = sh.Hq // U, sh.Hkv // U
    q, k, v, do = attn_inputs(sh)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    gview = lambda t, Hg: t[0].view(sh.S, U, Hg, sh.D).permute(1, 0, 2, 3)
    out = Guarded(1, sh.S, sh.Hq, sh.D, pad_d=0, pad_row=24)
    dq = Guarded(1, sh.S, sh.Hq, sh.D, pad_d=0, pad_row=24)
    dk = Guarded(1, sh.S, sh.Hkv, sh.D, pad_d=0, pad_row=40)
    dv = Guarded(1, sh.S, sh.Hkv, sh.D, pad_d=0, pad_row=40)
    gv = lambda g, Hg: g.view[0].unflatten(1, (U, Hg)).permute(1, 0, 2, 3)
    lse = GuardedLse(U, Hu, sh.S)
    ctx.attn_fwd(gview(qd, Hu), gview(kd, Hku), gview(vd, Hku), sh.P, out=gv(out, Hu), lse=lse.view)
    ctx.attn_bwd(gview(qd, Hu), gview(kd, Hku), gview(vd, Hku), gv(out, Hu), lse.view, gview(dod, Hu), sh.P,
                 dq=gv(dq, Hu), dk=gv(dk, Hku), dv=gv(dv, Hku))
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    for name, g in (("out", out), ("dq", dq), ("dk", dk), ("dv", dv), ("lse", lse)):
        assert g.untouched(), f"{name}: a byte outside the output view was written"
    o_ref, _ = oracle.attn_fwd(q, k, v)
    check("out", out.view, o_ref)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), oracle.attn_bwd(q, k, v, do)):
        check(name, g.view, r)


@pytest.mark.parametrize("B,S,H,D,ring,U,layout", [(1, 1001, 8, 64, 4, 2, "bshd"), (2, 37, 6, 128, 1, 3, "sbhd")])
def test_exchange_stays_inside(B, S, H, D, ring, U, layout):
    """The exchange writes its padded output buffer exactly (pad rows as
    zeros) and nothing around it; the inverse writes only the view's
    elements of a padded [B,S,H,D] destination."""
    x = exchange_input(B, S, H, D, layout=layout, seed=11)
    shape = ctx.exchanged_shape(B, S, H, D, ring, U, layout)
    n = 1
    for e in shape:
        n *= e
    ybuf = torch.full((GUARD + n + GUARD,), SENT16, dtype=torch.int16, device="cuda")
    y = ybuf[GUARD:GUARD + n].view(torch.bfloat16).view(shape)
    ctx.seq_head_exchange(x.cuda(), ring, U, 0, layout, y=y)
    torch.cuda.synchronize()
    assert (ybuf[:GUARD] == SENT16).all() and (ybuf[-GUARD:] == SENT16).all()
    y_ref = oracle.seq_head_exchange(x, ring, U, 0, layout)
    assert torch.equal(y.view(torch.int16).cpu(), y_ref.view(torch.int16))
    back = Guarded(B, S, H, D, layout)
    ctx.seq_head_exchange(y, ring, U, 1, layout, y=back.view, S=S, B=B, H=H)
    torch.cuda.synchronize()
    assert back.untouched()
    assert torch.equal(back.view.contiguous().view(torch.int16).cpu(), x.contiguous().view(torch.int16))
