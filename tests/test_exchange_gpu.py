"""GPU checks of the Ulysses exchange (bit-exact) and of the hybrid
ring x Ulysses composition, through the C ABI."""
import pytest
import torch

import context_attention_fwd_gb300 as ctx
import oracle
from seeded_inputs import HYBRID_RING, HYBRID_S65536, HYBRID_ULYSSES, AttnShape, attn_inputs, exchange_input

pytestmark = pytest.mark.gpu

CASES = [(1, 1000, 8, 64, 4, 2, "bshd"), (2, 1001, 16, 64, 4, 2, "sbhd"), (8, 10, 8, 64, 1, 2, "sbhd"),
         (2, 37, 6, 128, 1, 3, "bshd"), (3, 64, 4, 64, 2, 1, "sbhd")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ctx.load_library(build_if_missing=True)


def bits(t):
    return t.contiguous().view(torch.int16).cpu()


@pytest.mark.parametrize("B,S,H,D,ring,U,layout", CASES)
def test_exchange_bit_exact_and_inverse(B, S, H, D, ring, U, layout):
    x = exchange_input(B, S, H, D, layout=layout, seed=S + H)
    y = ctx.seq_head_exchange(x.cuda(), ring, U, 0, layout)
    y_ref = oracle.seq_head_exchange(x, ring, U, 0, layout)
    assert y.shape == y_ref.shape
    assert torch.equal(bits(y), bits(y_ref))
    back = ctx.seq_head_exchange(y, ring, U, 1, layout, S=S, B=B, H=H)
    assert back.stride() == x.stride()
    assert torch.equal(bits(back), bits(x))
    # the transposed exchange is the gradient: grad of sum(y^2) = inv(2 y) = 2 x, exactly
    g = ctx.seq_head_exchange(2 * y, ring, U, 1, layout, S=S, B=B, H=H)
    assert torch.equal(bits(g), bits(2 * x))


def test_exchange_worked_example_shapes():
    """Sequence-first (10, 8, 8, 64) on two ulysses ranks: each rank gets
    (10, 8, 4, 64) and the inverse restores (5, 8, 8, 64) per rank."""
    x = exchange_input(8, 10, 8, 64, layout="sbhd", seed=3)
    y = ctx.seq_head_exchange(x.cuda(), 1, 2, 0, "sbhd")
    assert tuple(y[0].shape) == (10, 8, 4, 64) and tuple(y[1].shape) == (10, 8, 4, 64)
    back = ctx.seq_head_exchange(y, 1, 2, 1, "sbhd", S=10, B=8, H=8)
    restored = back.permute(1, 0, 2, 3)  # [S,B,H,D] storage
    assert tuple(restored[:5].shape) == (5, 8, 8, 64)
    assert (restored.float().cpu() - x.permute(1, 0, 2, 3).float()).abs().max().item() == 0.0


def test_exchange_full_size_hybrid_q():
    """q of the ring 4 x ulysses 2 hybrid, [1, 65536, 32, 128], bit-exact."""
    sh = HYBRID_S65536
    x = exchange_input(sh.B, sh.S, sh.Hq, sh.D, seed=5)
    y = ctx.seq_head_exchange(x.cuda(), HYBRID_RING, HYBRID_ULYSSES, 0, "bshd")
    y_ref = oracle.seq_head_exchange(x, HYBRID_RING, HYBRID_ULYSSES, 0, "bshd")
    assert torch.equal(bits(y), bits(y_ref))
    back = ctx.seq_head_exchange(y, HYBRID_RING, HYBRID_ULYSSES, 1, "bshd", S=sh.S, B=sh.B, H=sh.Hq)
    assert torch.equal(bits(back), bits(x))


def hybrid(q, k, v, do, ring, U):
    """exchange -> ring attention over the exchanged view -> inverse exchange;
    backward: exchange(dout) -> ring backward -> inverse exchange."""
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    W = ring * U
    Ssh = -(-S // W)
    offs = [min(r * U * Ssh, S) for r in range(ring)] + [S]  # rank (r, u) holds these rows
    ex = lambda t: ctx.seq_head_exchange(t, ring, U, 0, "bshd")
    yq, yk, yv, ydo = ex(q), ex(k), ex(v), ex(do)
    vq, vk, vv, vdo = (ctx.exchanged_view(t, S, "bshd") for t in (yq, yk, yv, ydo))
    out_v, lse_v = ctx.attn_fwd(vq, vk, vv, ring, chunk_offsets=offs)
    dq_v, dk_v, dv_v = ctx.attn_bwd(vq, vk, vv, out_v, lse_v, vdo, ring, chunk_offsets=offs)

    def inv(view, H):
        full = torch.zeros(U, B, W * Ssh, H // U, D, dtype=view.dtype, device=view.device)
        full.view(U * B, W * Ssh, H // U, D)[:, :S] = view
        return ctx.seq_head_exchange(full, ring, U, 1, "bshd", S=S, B=B, H=H)

    return inv(out_v, Hq), inv(dq_v, Hq), inv(dk_v, Hkv), inv(dv_v, Hkv), offs


@pytest.mark.parametrize("S", [1000, 4096])
def test_hybrid_ring_x_ulysses_matches_plain_ring(S):
    sh = AttnShape(B=1, S=S, Hq=8, Hkv=4, D=128, P=4)
    q, k, v, do = attn_inputs(sh)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    out_h, dq_h, dk_h, dv_h, offs = hybrid(qd, kd, vd, dod, ring=4, U=2)
    out_p, lse_p = ctx.attn_fwd(qd, kd, vd, 4, chunk_offsets=offs)
    # same chunks, same kernel, values moved bit-exactly: the forward is identical
    assert torch.equal(bits(out_h), bits(out_p))
    o_ref, _ = oracle.attn_fwd(q, k, v)
    g_ref = oracle.attn_bwd(q, k, v, do)
    from test_parity_gpu import check
    check("out", out_h, o_ref)
    check("dq", dq_h, g_ref[0])
    check("dk", dk_h, g_ref[1])
    check("dv", dv_h, g_ref[2])
    assert ctx.device_status() == 0


def test_head_group_views_read_the_unexchanged_layout():
    """Fused exchange + attention: a head group's attention reads the
    pre-exchange tensor through a strided view (no copy) and gives bit for
    bit what it gives on the exchanged buffer."""
    sh = AttnShape(B=1, S=2000, Hq=8, Hkv=4, D=128, P=4)
    q, k, v, _ = (t.cuda() for t in attn_inputs(sh))
    ring, U = 4, 2
    Hu, Hku = sh.Hq // U, sh.Hkv // U
    ex = lambda t: ctx.seq_head_exchange(t, ring, U, 0, "bshd")
    yq, yk, yv = ex(q), ex(k), ex(v)
    for u in range(U):
        o_view, l_view = ctx.attn_fwd(q[:, :, u * Hu:(u + 1) * Hu], k[:, :, u * Hku:(u + 1) * Hku],
                                      v[:, :, u * Hku:(u + 1) * Hku], ring)
        o_ex, l_ex = ctx.attn_fwd(yq[u][:, :sh.S], yk[u][:, :sh.S], yv[u][:, :sh.S], ring)
        assert torch.equal(bits(o_view), bits(o_ex))
        assert torch.equal(l_view.cpu(), l_ex.cpu())


def test_hybrid_ring4_ulysses2_full_size_sampled():
    """The ring 4 x ulysses 2 hybrid at full size: exchange of
    [1,65536,32,128] (k, v with 8 heads), GQA 32/8 attention over 4 ring
    chunks on the exchanged tensors, inverse exchange; forward and backward.
    Sampled query rows (out, dq) and key rows of one key/value head (dk, dv:
    every row of its four query heads enters them) at rank and chunk edges
    against the oracle; the sum rules for dk and dv over every head."""
    from test_parity_gpu import check
    sh = HYBRID_S65536
    q, k, v, do = attn_inputs(sh)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    out, dq, dk, dv, offs = hybrid(qd, kd, vd, dod, ring=HYBRID_RING, U=HYBRID_ULYSSES)
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    g = torch.Generator().manual_seed(2)
    rows = [(0, int(h), int(s)) for h, s in zip(torch.randint(0, sh.Hq, (24,), generator=g),
                                                torch.randint(0, sh.S, (24,), generator=g))]
    rows += [(0, 17, s) for s in (0, 16383, 16384, 32767, 32768, 49152, 65535)]  # rank edges
    o_ref, _ = oracle.fwd_rows(q, k, v, rows)
    check("out rows", torch.stack([out[b, s, h].cpu() for b, h, s in rows]), o_ref)
    g2 = torch.Generator().manual_seed(3)
    qrows = rows + [(0, int(h), int(s)) for h, s in zip(torch.randint(0, sh.Hq, (17,), generator=g2),
                                                        torch.randint(0, sh.S, (17,), generator=g2))]
    dq_ref = oracle.dq_rows(q, k, v, do, qrows)
    check("dq rows", torch.stack([dq[b, s, h].cpu() for b, h, s in qrows]), dq_ref)
    # kv head 5 lives in head group 1 after the exchange (kv heads 4..7)
    krows = [(0, 5, s) for s in (0, 1, 8191, 8192, 16383, 16384, 24575, 32767, 32768, 40960, 49151,
                                 49152, 57344, 65534, 65535)]
    dk_ref, dv_ref = oracle.dkv_rows(q, k, v, do, krows)
    check("dk rows", torch.stack([dk[b, s, h].cpu() for b, h, s in krows]), dk_ref)
    check("dv rows", torch.stack([dv[b, s, h].cpu() for b, h, s in krows]), dv_ref)
    G = sh.Hq // sh.Hkv
    do_grp = do.float().reshape(sh.B, sh.S, sh.Hkv, G, sh.D).sum(dim=(1, 3)).to(dv.device)
    dv_sum = dv.float().sum(dim=1)
    assert ((dv_sum - do_grp).norm() / do_grp.norm()).item() < 2e-2
    assert (dk.float().sum(dim=1).abs().max() / dk.float().abs().sum(dim=1).max()).item() < 2e-2


def test_fused_single_call_over_head_group_views():
    """Fused exchange + attention in one call: a strided view that turns the
    head group into the batch index ([U, S, H/U, D] for B = 1) runs both
    groups' attention on the un-exchanged tensors and writes out, dq, dk, dv
    straight into the un-exchanged layout; equals the explicit pipeline
    (exchange, attention, inverse exchange) - the forward bit for bit."""
    sh = AttnShape(B=1, S=4096, Hq=8, Hkv=4, D=128, P=4)
    ring, U = 4, 2
    q, k, v, do = (t.cuda() for t in attn_inputs(sh))
    out_h, dq_h, dk_h, dv_h, offs = hybrid(q, k, v, do, ring=ring, U=U)
    gview = lambda t, Hg: t[0].view(sh.S, U, Hg, sh.D).permute(1, 0, 2, 3)
    Hu, Hku = sh.Hq // U, sh.Hkv // U
    out, dq = torch.empty_like(q), torch.empty_like(q)
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    lse = torch.empty(U, Hu, sh.S, dtype=torch.float32, device="cuda")
    fq, fk, fv, fdo = gview(q, Hu), gview(k, Hku), gview(v, Hku), gview(do, Hu)
    ctx.attn_fwd(fq, fk, fv, ring, chunk_offsets=offs, out=gview(out, Hu), lse=lse)
    ctx.attn_bwd(fq, fk, fv, gview(out, Hu), lse, fdo, ring, chunk_offsets=offs,
                 dq=gview(dq, Hu), dk=gview(dk, Hku), dv=gview(dv, Hku))
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    assert torch.equal(bits(out), bits(out_h))
    from test_parity_gpu import check
    for name, a, b in (("dq", dq, dq_h), ("dk", dk, dk_h), ("dv", dv, dv_h)):
        check(name, a, b, tol=1e-2)
