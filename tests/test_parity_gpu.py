"""GPU parity of the ring-chunked attention forward and backward against the
fp64 oracle, through the C ABI.

Tolerance (bf16 inputs, fp32 accumulation, bf16 outputs): per tensor both
  ||got - ref||_2 / ||ref||_2 <= 2e-2   and   max|got - ref| / max|ref| <= 2e-2.
lse (fp32 output) is held to 1e-3 absolute.
"""
import pytest
import torch

import context_attention_fwd_gb300 as ctx
import oracle
from seeded_inputs import (FLUX_GQA_S4608_P4, MHA_B2_S512_P2, SEQFIRST_S1001_P4, VIDEO_S32760_P8,
                           AttnShape, attn_inputs)

pytestmark = pytest.mark.gpu
TOL = 2e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ctx.load_library(build_if_missing=True)
    yield
    assert ctx.device_status() == 0


def check(name, got, ref, tol=TOL):
    g, r = got.double().cpu(), ref.double().cpu()
    assert torch.isfinite(g).all(), f"{name}: non-finite values"
    if r.abs().max().item() == 0:
        # an identically zero reference (one key: dq = dk = 0 exactly) has no
        # relative error; the kernels' fp32 arithmetic leaves rounding noise
        assert g.abs().max().item() < 1e-3, f"{name}: {g.abs().max().item():.3e} against exact zero"
        return 0.0, 0.0
    nrm = ((g - r).norm() / r.norm()).item()
    mx = ((g - r).abs().max() / r.abs().max()).item()
    assert nrm <= tol and mx <= tol, f"{name}: norm-rel {nrm:.3e}, max-rel {mx:.3e}"
    return nrm, mx


def run_gpu(shape, P=None, offsets=None, flags=0, causal=False):
    q, k, v, do = attn_inputs(shape)
    qd, kd, vd, dod = (t.to("cuda") for t in (q, k, v, do))  # .to() keeps the storage order
    if shape.layout == "sbhd" and shape.B > 1:
        assert qd.stride(1) > qd.stride(0)
    P = shape.P if P is None else P
    out, lse = ctx.attn_fwd(qd, kd, vd, P, chunk_offsets=offsets, flags=flags, causal=causal)
    dq, dk, dv = ctx.attn_bwd(qd, kd, vd, out, lse, dod, P, chunk_offsets=offsets, causal=causal)
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    return (q, k, v, do), (out, lse, dq, dk, dv)


def check_full(inputs, outputs, causal=False):
    q, k, v, do = inputs
    out, lse, dq, dk, dv = outputs
    o_ref, l_ref = oracle.attn_fwd(q, k, v, causal=causal)
    check("out", out, o_ref)
    assert (lse.double().cpu() - l_ref).abs().max() < LSE_TOL
    dq_r, dk_r, dv_r = oracle.attn_bwd(q, k, v, do, causal=causal)
    check("dq", dq, dq_r)
    check("dk", dk, dk_r)
    check("dv", dv, dv_r)


def test_mha_b2_s512_p2():
    check_full(*run_gpu(MHA_B2_S512_P2))


def test_seqfirst_s1001_p4_uneven():
    """Sequence-first storage, chunks 251/250/250/250 (not tile multiples)."""
    inputs, outputs = run_gpu(SEQFIRST_S1001_P4)
    assert outputs[0].stride(1) == 16 * 64  # output kept sequence-first
    check_full(inputs, outputs)


@pytest.mark.parametrize("P", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_every_p_gqa(P, D):
    sh = AttnShape(B=1, S=777, Hq=4, Hkv=2, D=D, P=P)
    check_full(*run_gpu(sh))


@pytest.mark.parametrize("causal", [False, True])
def test_max_chunks_p64(causal):
    """The largest chunk table: 64 ring chunks of 15-16 rows (every chunk a
    single partial tile)."""
    sh = AttnShape(B=1, S=1000, Hq=4, Hkv=2, D=64, P=64)
    check_full(*run_gpu(sh, causal=causal), causal=causal)


def test_custom_chunk_offsets():
    sh = AttnShape(B=2, S=700, Hq=2, Hkv=1, D=128, P=4)
    check_full(*run_gpu(sh, offsets=[0, 1, 300, 429, 700]))


@pytest.mark.parametrize("S,P", [(1, 1), (5, 5), (130, 1), (257, 2), (128, 1), (129, 3)])
def test_edge_sizes(S, P):
    """Single rows, one-row chunks (P == S), tile tails of 1 and 2 rows."""
    sh = AttnShape(B=1, S=S, Hq=2, Hkv=2, D=64, P=P)
    inputs, outputs = run_gpu(sh)
    if S == 1:
        # closed form: one key, out = v, dq = dk = 0, dv = dout
        q, k, v, do = inputs
        out, lse, dq, dk, dv = outputs
        assert torch.equal(out.cpu(), v.expand_as(out))
        # dP - delta is zero up to fp32 summation order
        assert dq.abs().max().item() < 1e-3 and dk.abs().max().item() < 1e-3
        assert torch.equal(dv.cpu(), do)
    else:
        check_full(inputs, outputs)


def test_materialized_partials_match_online():
    """Per-iteration partials + the LSE-merge kernel give the oracle's result."""
    sh = AttnShape(B=1, S=1001, Hq=4, Hkv=4, D=64, P=4, layout="sbhd")
    inputs, outputs = run_gpu(sh, flags=ctx.FLAG_MATERIALIZE_PARTIALS)
    check_full(inputs, outputs)
    sh2 = AttnShape(B=2, S=600, Hq=4, Hkv=2, D=128, P=5)
    check_full(*run_gpu(sh2, flags=ctx.FLAG_MATERIALIZE_PARTIALS))


def test_results_independent_of_p():
    """Every P computes the same attention: compare P=1 with P=8 on the GPU."""
    sh = AttnShape(B=1, S=2048, Hq=4, Hkv=4, D=128, P=1)
    _, o1 = run_gpu(sh, P=1)
    inputs, o8 = run_gpu(sh, P=8)
    for name, a, b in zip(("out", "lse", "dq", "dk", "dv"), o1, o8):
        if name == "lse":
            assert (a - b).abs().max().item() < LSE_TOL
        else:
            check(name, a, b, tol=1e-2)


def test_flux_gqa_s4608_p4_full():
    """Flux-like joint sequence (4096 image + 512 text tokens), GQA 24/8,
    D=128, P=4: every element of out, lse, dq, dk and dv against the oracle's
    full forward and analytic backward."""
    check_full(*run_gpu(FLUX_GQA_S4608_P4))


def _head(t, h):
    """Head h of a logical [B,S,H,D] tensor as a one-head [B,S,1,D] view."""
    return t[:, :, h:h + 1]


def test_video_s32760_p8_full_size():
    """The long-context workload at full size, in the launch configuration
    the bench times.  One whole head (all 32760 rows) of all four outputs and
    lse against the oracle: heads are independent in MHA, so the oracle's
    full-sequence forward and backward of that head alone are the full
    problem's values for it.  Then sampled rows of other heads at chunk and
    tile edges, and the sum rules over every head."""
    sh = VIDEO_S32760_P8
    inputs, outputs = run_gpu(sh)
    q, k, v, do = inputs
    out, lse, dq, dk, dv = outputs
    h = 11
    qh, kh, vh, doh = (_head(t, h) for t in (q, k, v, do))
    o_ref, l_ref = oracle.attn_fwd(qh, kh, vh)
    check("out head", _head(out, h), o_ref)
    assert (lse[:, h:h + 1].double().cpu() - l_ref).abs().max() < LSE_TOL
    dq_r, dk_r, dv_r = oracle.attn_bwd(qh, kh, vh, doh)
    check("dq head", _head(dq, h), dq_r)
    check("dk head", _head(dk, h), dk_r)
    check("dv head", _head(dv, h), dv_r)
    off = oracle.chunk_offsets(sh.S, sh.P)
    edges = sorted({o + d for o in off for d in (-1, 0, 127, 128) if 0 <= o + d < sh.S})
    rows = [(0, hh, s) for hh, s in zip([0, 7, 13, 23] * 16, edges[:64])]
    o_ref, l_ref = oracle.fwd_rows(q, k, v, rows)
    check("out rows", torch.stack([out[b, s, hh].cpu() for b, hh, s in rows]), o_ref)
    assert max(abs(lse[b, hh, s].item() - l_ref[i].item()) for i, (b, hh, s) in enumerate(rows)) < LSE_TOL
    qrows = rows[:24]
    check("dq rows", torch.stack([dq[b, s, hh].cpu() for b, hh, s in qrows]),
          oracle.dq_rows(q, k, v, do, qrows))
    # at any size: sum_j dk_j = 0 and sum_j dv_j = sum_i do_i per head (fp32 sums)
    dv_sum = dv.float().sum(dim=1)
    do_sum = do.float().sum(dim=1).to(dv_sum.device)
    assert ((dv_sum - do_sum).norm() / do_sum.norm()).item() < 2e-2
    assert (dk.float().sum(dim=1).abs().max() / dk.float().abs().sum(dim=1).max()).item() < 2e-2


def test_video_s32760_p8_causal_full_size_sampled():
    """The long-context shape with causal masking, as the bench times it:
    sampled rows at chunk and tile edges against the oracle, one head's
    key rows, and the sum rules (every row's probabilities still sum to
    one, so they hold under the mask)."""
    sh = VIDEO_S32760_P8
    inputs, outputs = run_gpu(sh, causal=True)
    q, k, v, do = inputs
    out, lse, dq, dk, dv = outputs
    off = oracle.chunk_offsets(sh.S, sh.P)
    edges = sorted({o + d for o in off for d in (-1, 0, 1, 127, 128) if 0 <= o + d < sh.S})
    rows = [(0, h, s) for h, s in zip([2, 9, 16, 21] * 12, edges[:48])]
    o_ref, l_ref = oracle.fwd_rows(q, k, v, rows, causal=True)
    check("out rows", torch.stack([out[b, s, h].cpu() for b, h, s in rows]), o_ref)
    assert max(abs(lse[b, h, s].item() - l_ref[i].item()) for i, (b, h, s) in enumerate(rows)) < LSE_TOL
    check("dq rows", torch.stack([dq[b, s, h].cpu() for b, h, s in rows[:24]]),
          oracle.dq_rows(q, k, v, do, rows[:24], causal=True))
    krows = [(0, 5, s) for s in edges[:16]]
    dk_ref, dv_ref = oracle.dkv_rows(q, k, v, do, krows, causal=True)
    check("dk rows", torch.stack([dk[b, s, h].cpu() for b, h, s in krows]), dk_ref)
    check("dv rows", torch.stack([dv[b, s, h].cpu() for b, h, s in krows]), dv_ref)
    dv_sum = dv.float().sum(dim=1)
    do_sum = do.float().sum(dim=1).to(dv_sum.device)
    assert ((dv_sum - do_sum).norm() / do_sum.norm()).item() < 2e-2
    assert (dk.float().sum(dim=1).abs().max() / dk.float().abs().sum(dim=1).max()).item() < 2e-2


@pytest.mark.parametrize("P", [1, 3, 5])
@pytest.mark.parametrize("D", [64, 128])
def test_causal_every_p_gqa(P, D):
    """Causal masking on global indices: later chunks skipped, diagonal masked."""
    sh = AttnShape(B=1, S=777, Hq=4, Hkv=2, D=D, P=P)
    check_full(*run_gpu(sh, causal=True), causal=True)


@pytest.mark.parametrize("S,P,layout,offsets", [(1001, 4, "sbhd", None), (130, 1, "bshd", None),
                                                 (700, 4, "bshd", [0, 1, 300, 429, 700]),
                                                 (2048, 8, "bshd", None), (5, 5, "bshd", None)])
def test_causal_layouts_and_edges(S, P, layout, offsets):
    sh = AttnShape(B=2, S=S, Hq=4, Hkv=4, D=64, P=P, layout=layout)
    check_full(*run_gpu(sh, offsets=offsets, causal=True), causal=True)


def test_causal_many_waves_sampled():
    """Causal masking on grids of many waves (over four per SM: each head's
    tiles are launched together); the cases above have grids of a few waves,
    which are launched heavy tiles of every head first.  Sampled rows at
    chunk and tile edges against the oracle."""
    sh = AttnShape(B=2, S=8192, Hq=24, Hkv=8, D=128, P=4)
    inputs, outputs = run_gpu(sh, causal=True)
    q, k, v, do = inputs
    out, lse, dq, dk, dv = outputs
    off = oracle.chunk_offsets(sh.S, sh.P)
    edges = sorted({o + d for o in off for d in (-1, 0, 1, 127, 128) if 0 <= o + d < sh.S})
    rows = [(b, h, s) for b, h, s in zip([0, 1] * 12, [0, 5, 17, 23] * 6, edges[:24])]
    o_ref, l_ref = oracle.fwd_rows(q, k, v, rows, causal=True)
    check("out rows", torch.stack([out[b, s, h].cpu() for b, h, s in rows]), o_ref)
    assert max(abs(lse[b, h, s].item() - l_ref[i].item()) for i, (b, h, s) in enumerate(rows)) < LSE_TOL
    check("dq rows", torch.stack([dq[b, s, h].cpu() for b, h, s in rows]),
          oracle.dq_rows(q, k, v, do, rows, causal=True))
    krows = [(1, 6, s) for s in edges[:12]]
    dk_ref, dv_ref = oracle.dkv_rows(q, k, v, do, krows, causal=True)
    check("dk rows", torch.stack([dk[b, s, h].cpu() for b, h, s in krows]), dk_ref)
    check("dv rows", torch.stack([dv[b, s, h].cpu() for b, h, s in krows]), dv_ref)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("allgather", [False, True])
def test_causal_materialized_partials(D, allgather):
    """Causal masking with materialised partials: per-chunk partials (the
    query's own chunk ends at its diagonal tile) merged over the iterations
    that meet chunks at or before the query's; equals the online merge and
    the oracle."""
    sh = AttnShape(B=1, S=1001, Hq=4, Hkv=2, D=D, P=4)
    flags = ctx.FLAG_MATERIALIZE_PARTIALS | (ctx.FLAG_KV_ALLGATHER if allgather else 0)
    inputs, outputs = run_gpu(sh, flags=flags, causal=True)
    check_full(inputs, outputs, causal=True)
    q, k, v, _ = (t.cuda() for t in inputs)
    o_online, l_online = ctx.attn_fwd(q, k, v, sh.P, causal=True)
    check("partials vs online", outputs[0], o_online, tol=1e-2)
    assert (outputs[1] - l_online).abs().max().item() < 1e-4


@pytest.mark.parametrize("causal", [False, True])
def test_kv_allgather_order_matches_ring(causal):
    """All-gather chunk order (every query shard over the concatenated K/V)
    computes the same attention as the ring order."""
    sh = AttnShape(B=1, S=1500, Hq=4, Hkv=2, D=128, P=4)
    q, k, v, do = attn_inputs(sh)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o_ring, l_ring = ctx.attn_fwd(qd, kd, vd, 4, causal=causal)
    o_ag, l_ag = ctx.attn_fwd(qd, kd, vd, 4, causal=causal, flags=ctx.FLAG_KV_ALLGATHER)
    o_ref, l_ref = oracle.attn_fwd(q, k, v, causal=causal)
    check("out ring", o_ring, o_ref)
    check("out allgather", o_ag, o_ref)
    assert (l_ag.double().cpu() - l_ref).abs().max() < LSE_TOL
    check("ring vs allgather", o_ag, o_ring, tol=1e-2)


def test_exp2_polynomial_and_sfu_accuracy():
    """The two exponentials the kernels use, against torch's exp2 in fp64:
    the FMA-pipe polynomial within its 7.5e-5 design bound (plus fp32
    rounding), the SFU within 2^-20 relative; both far below bf16's 3.9e-3."""
    x = torch.cat([torch.linspace(-125.0, 8.0, 1 << 20), torch.linspace(-1.0, 1.0, 1 << 16)]).cuda()
    yp, ys = ctx.selftest_exp2(x)
    ref = torch.exp2(x.double())
    rel_p = ((yp.double() - ref).abs() / ref).max().item()
    rel_s = ((ys.double() - ref).abs() / ref).max().item()
    assert rel_p < 1e-4, rel_p
    assert rel_s < 2 ** -20, rel_s
    # below the clamp the polynomial returns 2^-125, a negligible weight
    yp2, _ = ctx.selftest_exp2(torch.tensor([-126.0, -500.0, float("-inf")], device="cuda"))
    assert (yp2.double() <= 2.0 ** -124).all() and (yp2 > 0).all()


def test_timeout_selftest_reports_status():
    """A device wait that nothing satisfies gives up and reports CTX_ERR_TIMEOUT."""
    assert ctx.device_status() == 0
    ctx.selftest_wait_timeout(20000)
    assert ctx.device_status() == 5
    assert ctx.device_status() == 0  # reading clears it
    # the context is still usable
    sh = AttnShape(B=1, S=300, Hq=2, Hkv=2, D=64, P=2)
    check_full(*run_gpu(sh))


@pytest.mark.parametrize("D", [64, 128, 256])
def test_gqa_equals_mha_with_repeated_kv(D):
    """GQA reads kv head h // (Hq/Hkv): running MHA on K/V with each kv head
    repeated for its query heads gives the same forward bit for bit, and the
    GQA dk/dv equal the group sums of the MHA dk/dv."""
    sh = AttnShape(B=1, S=900, Hq=6, Hkv=2, D=D, P=3)
    q, k, v, do = (t.cuda() for t in attn_inputs(sh))
    G = sh.Hq // sh.Hkv
    k_rep, v_rep = k.repeat_interleave(G, dim=2), v.repeat_interleave(G, dim=2)
    o_g, l_g = ctx.attn_fwd(q, k, v, sh.P)
    o_m, l_m = ctx.attn_fwd(q, k_rep, v_rep, sh.P)
    assert torch.equal(o_g, o_m) and torch.equal(l_g, l_m)
    dq_g, dk_g, dv_g = ctx.attn_bwd(q, k, v, o_g, l_g, do, sh.P)
    dq_m, dk_m, dv_m = ctx.attn_bwd(q, k_rep, v_rep, o_m, l_m, do, sh.P)
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    check("dq", dq_g, dq_m, tol=1e-2)
    sum_groups = lambda t: t.float().reshape(sh.B, sh.S, sh.Hkv, G, sh.D).sum(dim=3)
    check("dk", dk_g, sum_groups(dk_m), tol=1e-2)
    check("dv", dv_g, sum_groups(dv_m), tol=1e-2)


@pytest.mark.parametrize("D,scale,causal", [(64, 0.05, False), (128, 0.2, True), (256, 0.03, False)])
def test_custom_scale(D, scale, causal):
    """A caller-given softmax scale (instead of 1/sqrt(D)) in both passes."""
    sh = AttnShape(B=1, S=600, Hq=4, Hkv=2, D=D, P=3)
    q, k, v, do = attn_inputs(sh)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    out, lse = ctx.attn_fwd(qd, kd, vd, sh.P, causal=causal, scale=scale)
    dq, dk, dv = ctx.attn_bwd(qd, kd, vd, out, lse, dod, sh.P, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    o_ref, l_ref = oracle.attn_fwd(q, k, v, scale=scale, causal=causal)
    check("out", out, o_ref)
    assert (lse.double().cpu() - l_ref).abs().max() < LSE_TOL
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), oracle.attn_bwd(q, k, v, do, scale=scale, causal=causal)):
        check(name, g, r)


def test_binding_refuses_wrong_types_on_the_gpu():
    """Device tensors of another element type, a malformed lse buffer or a
    host tensor among device ones are refused before any launch."""
    q = torch.zeros(1, 128, 2, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="bfloat16"):
        ctx.attn_fwd(q.half(), q, q, 1)
    with pytest.raises(ValueError, match="lse"):
        ctx.attn_fwd(q, q, q, 1, lse=torch.empty(1, 2, 127, device="cuda"))
    with pytest.raises(ValueError, match="CUDA device"):
        ctx.attn_fwd(q, q.cpu(), q, 1)
    out, lse = ctx.attn_fwd(q, q, q, 1)
    with pytest.raises(ValueError, match="bfloat16"):
        ctx.attn_bwd(q, q, q, out, lse, q.float(), 1)
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
