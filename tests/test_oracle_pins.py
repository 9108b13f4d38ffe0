"""Pins of the fp64 oracle against things other than itself.

Each test ties one oracle routine to a fact the pages or the mathematics fix:
a library routine (torch fp64 SDPA + autograd), brute-force finite
differences, closed forms, invariants, and the worked shapes printed on the
pages (tests/golden/).  A dropped term, a wrong sign, a wrong index or a
transposed operand anywhere in oracle.c fails at least one of them.
"""
import json
import math
import os

import pytest
import torch
import torch.nn.functional as F

import oracle
from seeded_inputs import AttnShape, attn_inputs, exchange_input

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rel(a, b):
    return ((a - b).norm() / b.norm()).item()


def _sdpa_ref(q, k, v, dout, causal=False, scale=None):
    """torch fp64 SDPA + autograd on logical [B,S,H,D] inputs (GQA by repeating k, v)."""
    G = q.shape[2] // k.shape[2]
    qd = q.double().clone().requires_grad_(True)
    kd = k.double().clone().requires_grad_(True)
    vd = v.double().clone().requires_grad_(True)
    kr = kd.repeat_interleave(G, dim=2)
    vr = vd.repeat_interleave(G, dim=2)
    o = F.scaled_dot_product_attention(qd.transpose(1, 2), kr.transpose(1, 2), vr.transpose(1, 2),
                                       is_causal=causal, scale=scale).transpose(1, 2)
    dq, dk, dv = torch.autograd.grad(o, (qd, kd, vd), dout.double())
    # lse by the textbook formula on the same library matmul
    sc = (1.0 / math.sqrt(q.shape[-1])) if scale is None else scale
    s = torch.einsum("bihd,bjhd->bhij", qd.detach(), kr.detach()) * sc
    if causal:
        S = q.shape[1]
        s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    return o.detach(), lse, dq, dk, dv


SMALL = [
    AttnShape(B=2, S=37, Hq=4, Hkv=4, D=16, P=1, layout="bshd"),
    AttnShape(B=1, S=29, Hq=6, Hkv=2, D=8, P=1, layout="bshd"),
    AttnShape(B=2, S=23, Hq=4, Hkv=1, D=16, P=1, layout="sbhd"),
    # the head dimensions the kernels implement, at the GQA group size of the
    # 24/4-head model
    AttnShape(B=1, S=33, Hq=6, Hkv=1, D=64, P=1, layout="bshd"),
    AttnShape(B=1, S=21, Hq=6, Hkv=1, D=128, P=1, layout="sbhd"),
    AttnShape(B=1, S=17, Hq=6, Hkv=1, D=256, P=1, layout="bshd"),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: f"B{s.B}S{s.S}H{s.Hq}/{s.Hkv}D{s.D}{s.layout}")
@pytest.mark.parametrize("causal", [False, True])
def test_fwd_bwd_match_torch_fp64(shape, causal):
    q, k, v, do = attn_inputs(shape, seed=11)
    o_ref, lse_ref, dq_ref, dk_ref, dv_ref = _sdpa_ref(q, k, v, do, causal=causal)
    o, lse = oracle.attn_fwd(q, k, v, causal=causal)
    assert torch.allclose(o, o_ref, rtol=0, atol=1e-12)
    assert torch.allclose(lse, lse_ref, rtol=0, atol=1e-12)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal=causal)
    for got, ref in ((dq, dq_ref), (dk, dk_ref), (dv, dv_ref)):
        assert torch.allclose(got, ref, rtol=0, atol=1e-11)


def test_custom_scale_matches_torch():
    sh = AttnShape(B=1, S=19, Hq=2, Hkv=2, D=8, P=1)
    q, k, v, do = attn_inputs(sh, seed=5)
    o_ref, _, dq_ref, dk_ref, dv_ref = _sdpa_ref(q, k, v, do, scale=0.3)
    o, _ = oracle.attn_fwd(q, k, v, scale=0.3)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, scale=0.3)
    assert torch.allclose(o, o_ref, atol=1e-12)
    for got, ref in ((dq, dq_ref), (dk, dk_ref), (dv, dv_ref)):
        assert torch.allclose(got, ref, atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_central_finite_differences(causal):
    """Brute force: d/dx sum(out * G) by central differences, every element."""
    torch.manual_seed(3)
    B, S, Hq, Hkv, D = 1, 5, 2, 1, 3
    q = torch.randn(B, S, Hq, D, dtype=torch.float64)
    k = torch.randn(B, S, Hkv, D, dtype=torch.float64)
    v = torch.randn(B, S, Hkv, D, dtype=torch.float64)
    G = torch.randn(B, S, Hq, D, dtype=torch.float64)
    dq, dk, dv = oracle.attn_bwd(q, k, v, G, causal=causal)
    h = 1e-6

    def loss(qq, kk, vv):
        o, _ = oracle.attn_fwd(qq, kk, vv, causal=causal)
        return float((o * G).sum())

    for name, base, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = torch.zeros_like(base)
        for idx in range(base.numel()):
            xp = base.clone().view(-1); xp[idx] += h
            xm = base.clone().view(-1); xm[idx] -= h
            ap = {"q": q, "k": k, "v": v, name: xp.view_as(base)}
            am = {"q": q, "k": k, "v": v, name: xm.view_as(base)}
            fd.view(-1)[idx] = (loss(ap["q"], ap["k"], ap["v"]) - loss(am["q"], am["k"], am["v"])) / (2 * h)
        assert torch.allclose(grad, fd, rtol=1e-6, atol=1e-8), name


def test_closed_form_equal_keys():
    """All keys equal: softmax is uniform, o_i = mean_j v_j, lse_i = log S + scale <q_i, k>."""
    torch.manual_seed(4)
    B, S, H, D = 1, 13, 2, 8
    q = torch.randn(B, S, H, D, dtype=torch.float64)
    k = torch.randn(B, 1, H, D, dtype=torch.float64).expand(B, S, H, D).contiguous()
    v = torch.randn(B, S, H, D, dtype=torch.float64)
    o, lse = oracle.attn_fwd(q, k, v)
    sc = 1 / math.sqrt(D)
    assert torch.allclose(o, v.mean(dim=1, keepdim=True).expand_as(o), atol=1e-13)
    want = math.log(S) + sc * (q * k).sum(-1).transpose(1, 2)
    assert torch.allclose(lse, want, atol=1e-13)


def test_closed_form_single_key():
    """S = 1: out = v, dq = dk = 0, dv = dout."""
    torch.manual_seed(6)
    q, k, v, do = (torch.randn(2, 1, 3, 4, dtype=torch.float64) for _ in range(4))
    o, lse = oracle.attn_fwd(q, k, v)
    assert torch.equal(o, v)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do)
    assert dq.abs().max() == 0 and dk.abs().max() == 0
    assert torch.allclose(dv, do, atol=1e-15)


def test_gradient_sum_rules():
    """Rows of P sum to one, rows of dS sum to zero, hence per kv head:
    sum_j dv_j = sum over the group's query rows of do_i and sum_j dk_j = 0."""
    sh = AttnShape(B=2, S=31, Hq=6, Hkv=3, D=8, P=1)
    q, k, v, do = attn_inputs(sh, seed=9)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do)
    G = sh.Hq // sh.Hkv
    do_grp = do.double().reshape(sh.B, sh.S, sh.Hkv, G, sh.D).sum(dim=(1, 3))
    assert torch.allclose(dv.sum(dim=1), do_grp, atol=1e-11)
    assert dk.sum(dim=1).abs().max() < 1e-11


def test_gqa_equals_mha_with_repeated_kv():
    sh = AttnShape(B=1, S=21, Hq=8, Hkv=2, D=8, P=1)
    q, k, v, do = attn_inputs(sh, seed=12)
    G = sh.Hq // sh.Hkv
    kr, vr = k.repeat_interleave(G, dim=2), v.repeat_interleave(G, dim=2)
    o1, l1 = oracle.attn_fwd(q, k, v)
    o2, l2 = oracle.attn_fwd(q, kr, vr)
    assert torch.allclose(o1, o2, atol=1e-14) and torch.allclose(l1, l2, atol=1e-14)
    dq1, dk1, dv1 = oracle.attn_bwd(q, k, v, do)
    dq2, dk2, dv2 = oracle.attn_bwd(q, kr, vr, do)
    assert torch.allclose(dq1, dq2, atol=1e-13)
    assert torch.allclose(dk1, dk2.reshape(1, sh.S, sh.Hkv, G, sh.D).sum(3), atol=1e-12)
    assert torch.allclose(dv1, dv2.reshape(1, sh.S, sh.Hkv, G, sh.D).sum(3), atol=1e-12)


def test_layouts_agree():
    """[S,B,H,D] storage read through strides gives the [B,S,H,D] result."""
    a = AttnShape(B=2, S=17, Hq=4, Hkv=2, D=8, P=1, layout="bshd")
    b = AttnShape(B=2, S=17, Hq=4, Hkv=2, D=8, P=1, layout="sbhd")
    qa, ka, va, da = attn_inputs(a, seed=2)
    qb, kb, vb, db = attn_inputs(b, seed=2)
    assert torch.equal(qa, qb) and qb.stride(1) == 2 * 4 * 8
    oa, la = oracle.attn_fwd(qa, ka, va)
    ob, lb = oracle.attn_fwd(qb, kb, vb)
    assert ob.stride() == qb.stride()
    assert torch.equal(oa, ob) and torch.equal(la, lb)
    ga = oracle.attn_bwd(qa, ka, va, da)
    gb = oracle.attn_bwd(qb, kb, vb, db)
    for x, y in zip(ga, gb):
        assert torch.equal(x, y)


def test_chunk_offsets_array_split():
    off = oracle.chunk_offsets(1001, 4)
    assert [b - a for a, b in zip(off[:-1], off[1:])] == [251, 250, 250, 250]
    off = oracle.chunk_offsets(32760, 8)
    assert all(b - a == 4095 for a, b in zip(off[:-1], off[1:]))
    assert oracle.chunk_offsets(512, 2) == [0, 256, 512]
    assert oracle.chunk_offsets(4608, 4) == [0, 1152, 2304, 3456, 4608]
    with pytest.raises(ValueError):
        oracle.chunk_offsets(3, 4)


RING_CASES = [(5, p) for p in range(1, 6)] + [(17, p) for p in range(1, 9)] + [(1001, 4), (1001, 7)]


@pytest.mark.parametrize("S,P", RING_CASES)
def test_ring_merge_equals_full_attention(S, P):
    """LSE-merge of the ring partials equals full attention, every P, uneven splits."""
    sh = AttnShape(B=1, S=S, Hq=2, Hkv=1, D=4 if S > 100 else 8, P=P)
    q, k, v, _ = attn_inputs(sh, seed=S * 31 + P)
    o_full, l_full = oracle.attn_fwd(q, k, v)
    o_ring, l_ring = oracle.ring_fwd(q, k, v, P)
    assert torch.allclose(o_ring, o_full, rtol=0, atol=1e-12)
    assert torch.allclose(l_ring, l_full, rtol=0, atol=1e-12)


def test_ring_merge_equals_full_attention_long_sequence():
    """The long-video workload's chunking (S=32760 as 8 chunks of 4095 rows),
    on one head with a narrow head dimension to keep the fp64 work small."""
    sh = AttnShape(B=1, S=32760, Hq=1, Hkv=1, D=8, P=8)
    q, k, v, _ = attn_inputs(sh, seed=32760)
    o_full, l_full = oracle.attn_fwd(q, k, v)
    o_ring, l_ring = oracle.ring_fwd(q, k, v, 8)
    assert torch.allclose(o_ring, o_full, rtol=0, atol=1e-12)
    assert torch.allclose(l_ring, l_full, rtol=0, atol=1e-12)


def test_ring_merge_custom_offsets_and_causal():
    sh = AttnShape(B=2, S=23, Hq=2, Hkv=2, D=8, P=3)
    q, k, v, do = attn_inputs(sh, seed=1)
    for causal in (False, True):
        o_full, l_full = oracle.attn_fwd(q, k, v, causal=causal)
        o_ring, l_ring = oracle.ring_fwd(q, k, v, 3, offsets=[0, 3, 20, 23], causal=causal)
        assert torch.allclose(o_ring, o_full, atol=1e-12) and torch.allclose(l_ring, l_full, atol=1e-12)


def test_lse_merge_of_partials():
    sh = AttnShape(B=1, S=29, Hq=2, Hkv=1, D=8, P=4)
    q, k, v, _ = attn_inputs(sh, seed=8)
    o_ring, l_ring, po, pl = oracle.ring_fwd(q, k, v, 4, partials=True)
    o_m, l_m = oracle.lse_merge(po, pl)
    assert torch.allclose(o_m, o_ring, atol=1e-14) and torch.allclose(l_m, l_ring, atol=1e-14)
    # a single partial is the full answer when P = 1
    o1, l1, po1, pl1 = oracle.ring_fwd(q, k, v, 1, partials=True)
    assert torch.allclose(po1[0].permute(0, 2, 1, 3), o1, atol=1e-14)
    # the partial of iteration i covers only chunk (r - i) mod P: its lse is the
    # log-sum-exp over that chunk alone
    off = oracle.chunk_offsets(29, 4)
    s = torch.einsum("bihd,bjhd->bhij", q.double(), k.double().repeat_interleave(2, 2)) / math.sqrt(8)
    row, r = 10, 1  # row 10 lies in chunk 1
    for it in range(4):
        c = (r - it) % 4
        want = torch.logsumexp(s[0, 0, row, off[c]:off[c + 1]], dim=0)
        assert abs(pl[it, 0, 0, row] - want) < 1e-12


@pytest.mark.parametrize("P", [1, 2, 3, 4, 8])
def test_ring_bwd_equals_full_bwd(P):
    sh = AttnShape(B=1, S=37, Hq=4, Hkv=2, D=8, P=P)
    q, k, v, do = attn_inputs(sh, seed=40 + P)
    o, lse = oracle.ring_fwd(q, k, v, P)
    got = oracle.ring_bwd(q, k, v, o, lse, do, P)
    ref = oracle.attn_bwd(q, k, v, do)
    for g, r in zip(got, ref):
        assert torch.allclose(g, r, rtol=0, atol=1e-11)


def test_ring_bwd_causal_equals_full():
    sh = AttnShape(B=1, S=19, Hq=2, Hkv=1, D=8, P=3)
    q, k, v, do = attn_inputs(sh, seed=77)
    o, lse = oracle.ring_fwd(q, k, v, 3, causal=True)
    got = oracle.ring_bwd(q, k, v, o, lse, do, 3, causal=True)
    ref = oracle.attn_bwd(q, k, v, do, causal=True)
    for g, r in zip(got, ref):
        assert torch.allclose(g, r, atol=1e-11)


@pytest.mark.parametrize("P", [2, 4])
def test_stale_kv_negative_control(P):
    """The defect the issue reports (every backward iteration reads the
    iteration-0 K/V) fails parity by an O(1) margin on the issue's workload
    shape; the correct ring backward passes it.  Smaller S keeps it quick."""
    with open(os.path.join(GOLDEN, "stale_kv_defect.json")) as f:
        gold = json.load(f)
    tol = gold["tolerance_used_on_the_page"]
    sh = AttnShape(B=2, S=128, Hq=8, Hkv=8, D=64, P=P)
    q, k, v, do = attn_inputs(sh, seed=gold["workload"]["seed"])
    o, lse = oracle.ring_fwd(q, k, v, P)
    ref = oracle.attn_bwd(q, k, v, do)
    good = oracle.ring_bwd(q, k, v, o, lse, do, P)
    bad = oracle.ring_bwd(q, k, v, o, lse, do, P, stale=True)
    for g, b, r in zip(good, bad, ref):
        assert _rel(g, r) < 1e-12
        assert _rel(b, r) > 0.5 > 10 * tol


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_rows_equal_full(causal):
    """The sampled-row routines used at full size agree with the full routines."""
    sh = AttnShape(B=2, S=41, Hq=6, Hkv=2, D=8, P=1, layout="sbhd")
    q, k, v, do = attn_inputs(sh, seed=21)
    o, lse = oracle.attn_fwd(q, k, v, causal=causal)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal=causal)
    qrows = [(0, 0, 0), (1, 5, 40), (0, 3, 17), (1, 1, 1)]
    o_r, l_r = oracle.fwd_rows(q, k, v, qrows, causal=causal)
    dq_r = oracle.dq_rows(q, k, v, do, qrows, causal=causal)
    for t, (b, h, s) in enumerate(qrows):
        assert torch.allclose(o_r[t], o[b, s, h], atol=1e-14)
        assert abs(l_r[t] - lse[b, h, s]) < 1e-14
        assert torch.allclose(dq_r[t], dq[b, s, h], atol=1e-13)
    krows = [(0, 0, 0), (1, 1, 40), (0, 1, 22)]
    dk_r, dv_r = oracle.dkv_rows(q, k, v, do, krows, causal=causal)
    for t, (b, h, s) in enumerate(krows):
        assert torch.allclose(dk_r[t], dk[b, s, h], atol=1e-13)
        assert torch.allclose(dv_r[t], dv[b, s, h], atol=1e-13)


# ---------------------------------------------------------------- exchange

def test_exchange_worked_example_shapes():
    with open(os.path.join(GOLDEN, "exchange_worked_example.json")) as f:
        gold = json.load(f)
    W = gold["world_size"]
    S_loc, B, H, D = gold["local_input_shape"]
    x = exchange_input(B, S_loc * W, H, D, layout="sbhd", seed=3)   # the whole sequence
    y = oracle.seq_head_exchange(x, ring=1, ulysses=W, direction=0, layout="sbhd")
    # rank (0, u)'s local tensor: rows [0, W*S_loc) of head group u
    for u in range(W):
        local = y[u]
        assert list(local.shape) == gold["exchanged_shape"]
    back = oracle.seq_head_exchange(y, 1, W, 1, "sbhd", S=S_loc * W, B=B, H=H)
    for rho in range(W):
        shard = back[rho * S_loc:(rho + 1) * S_loc]
        assert list(shard.shape) == gold["restored_shape"]
    diff = (back.float() - x.permute(1, 0, 2, 3).float()).abs().max().item()
    assert diff == gold["max_abs_diff_after_round_trip"]


@pytest.mark.parametrize("layout", ["bshd", "sbhd"])
@pytest.mark.parametrize("B,S,H,ring,U", [(1, 16, 4, 2, 2), (2, 1001, 8, 4, 2), (1, 7, 6, 1, 3), (2, 10, 4, 3, 1)])
def test_exchange_roundtrip_and_slots(layout, B, S, H, ring, U):
    D = 8
    x = exchange_input(B, S, H, D, layout=layout, seed=S)
    y = oracle.seq_head_exchange(x, ring, U, 0, layout)
    W = ring * U
    Ssh = -(-S // W)
    Hu = H // U
    xb = x.contiguous() if layout == "bshd" else x  # logical [B,S,H,D]
    yb = y if layout == "bshd" else y.permute(0, 2, 1, 3, 4)  # [U,B,Sp,Hu,D]
    # slot rule: slot u' of rank (r,u)'s output = rank (r*U+u')'s input rows, head group u
    for r in range(ring):
        for u in range(U):
            local = yb[u][:, r * U * Ssh:(r + 1) * U * Ssh]
            for up in range(U):
                rho = r * U + up
                rows = range(rho * Ssh, min((rho + 1) * Ssh, S))
                for t, s in enumerate(rows):
                    assert torch.equal(local[:, up * Ssh + t], xb[:, s, u * Hu:(u + 1) * Hu])
                # pad rows are zero
                for t in range(len(rows), Ssh):
                    assert local[:, up * Ssh + t].abs().max() == 0
    back = oracle.seq_head_exchange(y, ring, U, 1, layout, S=S, B=B, H=H)
    back_b = back if layout == "bshd" else back.permute(1, 0, 2, 3)
    assert torch.equal(back_b.view(torch.int16), xb.contiguous().view(torch.int16))


def test_exchange_gradient_is_2x():
    """The exchange is a permutation (plus zero pads), so the gradient of
    sum(exchange(x)^2) is exactly 2x.  The Jacobian of the oracle's map is
    materialised on basis vectors, then grad = J^T (2 J x)."""
    B, S, H, D, ring, U = 1, 5, 4, 2, 1, 2
    n = B * S * H * D
    cols = []
    for idx in range(n):
        e = torch.zeros(n, dtype=torch.float64)
        e[idx] = 1.0
        xe = e.to(torch.bfloat16).view(B, S, H, D)
        cols.append(oracle.seq_head_exchange(xe, ring, U, 0, "bshd").double().reshape(-1))
    J = torch.stack(cols, dim=1)           # [m, n]
    assert torch.equal(J.sum(dim=0), torch.ones(n, dtype=torch.float64))   # every input lands once
    assert J.sum(dim=1).max() <= 1                                           # no output gets two
    x = exchange_input(B, S, H, D, seed=1).double().reshape(-1)
    y = J @ x
    grad = J.t() @ (2 * y)
    assert torch.equal(grad, 2 * x)
