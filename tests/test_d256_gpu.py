"""GPU parity of the head-dimension-256 kernels (forward and backward)
against the fp64 oracle, through the C ABI.

The workload is the causal language model of the DeepSpeed Ulysses pull
request's end-to-end check (24 query heads, 4 key/value heads, head
dimension 256, 1024 tokens, sequence parallelism 2 and 8), plus ragged and
degenerate sizes.  Tolerances as in test_parity_gpu.py.
"""
import pytest
import torch

import context_attention_fwd_gb300 as ctx
import oracle
from seeded_inputs import GQA_D256_S1024, AttnShape, attn_inputs
from test_parity_gpu import LSE_TOL, check, check_full, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ctx.load_library(build_if_missing=True)
    yield
    assert ctx.device_status() == 0


@pytest.mark.parametrize("P", [2, 8])
@pytest.mark.parametrize("causal", [True, False])
def test_gqa_d256_s1024(P, causal):
    check_full(*run_gpu(GQA_D256_S1024, P=P, causal=causal), causal=causal)


@pytest.mark.parametrize("P", [1, 3, 5])
def test_every_p_ragged(P):
    """777 rows: ragged chunks and tile tails; GQA 4/2."""
    sh = AttnShape(B=1, S=777, Hq=4, Hkv=2, D=256, P=P)
    check_full(*run_gpu(sh))


@pytest.mark.parametrize("P", [1, 3])
def test_causal_ragged(P):
    sh = AttnShape(B=2, S=777, Hq=4, Hkv=2, D=256, P=P, layout="sbhd")
    check_full(*run_gpu(sh, causal=True), causal=True)


@pytest.mark.parametrize("S,P", [(1, 1), (5, 5), (129, 3), (64, 1), (65, 1)])
def test_edge_sizes(S, P):
    """Single rows, one-row chunks, tiles whose rows fit in the first or second
    64-row half of the V tile."""
    sh = AttnShape(B=1, S=S, Hq=2, Hkv=1, D=256, P=P)
    inputs, outputs = run_gpu(sh)
    if S == 1:
        q, k, v, do = inputs
        out, lse, dq, dk, dv = outputs
        assert torch.equal(out.cpu(), v.expand_as(out))
        assert dq.abs().max().item() < 1e-3 and dk.abs().max().item() < 1e-3
    else:
        check_full(inputs, outputs)


def test_partials_and_allgather():
    sh = AttnShape(B=1, S=1001, Hq=4, Hkv=2, D=256, P=4)
    check_full(*run_gpu(sh, flags=ctx.FLAG_MATERIALIZE_PARTIALS))
    q, k, v, _ = attn_inputs(sh)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    for causal in (False, True):
        o_ag, l_ag = ctx.attn_fwd(qd, kd, vd, 4, causal=causal, flags=ctx.FLAG_KV_ALLGATHER)
        o_ref, l_ref = oracle.attn_fwd(q, k, v, causal=causal)
        check("out allgather", o_ag, o_ref)
        assert (l_ag.double().cpu() - l_ref).abs().max() < LSE_TOL


def test_d256_equals_two_d128_halves_of_v():
    """P and the LSE depend on q, k only, and every output column is its own
    dot product: running with one column half of V zeroed reproduces the
    other half of the full output bit for bit (and zeros).  Checks the
    kernel's V column blocks against each other without the oracle."""
    sh = AttnShape(B=1, S=640, Hq=2, Hkv=2, D=256, P=2)
    q, k, v, do = (t.cuda() for t in attn_inputs(sh))
    out, lse = ctx.attn_fwd(q, k, v, 2)
    for half in range(2):
        vh = v.clone()
        vh[..., (1 - half) * 128:(2 - half) * 128] = 0
        oh, lh = ctx.attn_fwd(q, k, vh, 2)
        assert torch.equal(lh, lse)
        sl = slice(half * 128, (half + 1) * 128)
        assert torch.equal(oh[..., sl], out[..., sl])
        assert oh[..., (1 - half) * 128:(2 - half) * 128].abs().max().item() == 0


@pytest.mark.parametrize("B,S,Hq,Hkv,P", [(2, 1300, 8, 4, 2),   # enough KV tiles: one CTA per group
                                          (1, 1000, 12, 2, 3),  # short: the group of 6 split 3 ways
                                          (1, 600, 6, 1, 1)])   # a single KV head: split 6 ways
def test_gqa_group_split(B, S, Hq, Hkv, P):
    """The backward splits a GQA group's query heads over several CTAs when
    the sequence is short (partial dK/dV summed afterwards) and keeps one CTA
    per group otherwise; both give the oracle's gradients."""
    sh = AttnShape(B=B, S=S, Hq=Hq, Hkv=Hkv, D=256, P=P)
    check_full(*run_gpu(sh))


def test_long_context_s16384_causal_sampled():
    """The same heads at 16384 tokens, P=8, causal, as the bench times them:
    sampled query rows (out, lse, dq) and key rows of one key/value head
    (dk, dv: every query row of its six-head group enters them) at chunk and
    tile edges against the oracle, plus the sum rules for dk and dv over
    every key/value head's group."""
    sh = AttnShape(B=1, S=16384, Hq=24, Hkv=4, D=256, P=8)
    inputs, outputs = run_gpu(sh, causal=True)
    q, k, v, do = inputs
    out, lse, dq, dk, dv = outputs
    off = oracle.chunk_offsets(sh.S, sh.P)
    edges = sorted({o + d for o in off for d in (-1, 0, 1, 127, 128) if 0 <= o + d < sh.S})
    rows = [(0, h, s) for h, s in zip([0, 7, 13, 23] * 12, edges[:40])]
    o_ref, l_ref = oracle.fwd_rows(q, k, v, rows, causal=True)
    check("out rows", torch.stack([out[b, s, h].cpu() for b, h, s in rows]), o_ref)
    assert max(abs(lse[b, h, s].item() - l_ref[i].item()) for i, (b, h, s) in enumerate(rows)) < LSE_TOL
    check("dq rows", torch.stack([dq[b, s, h].cpu() for b, h, s in rows[:24]]),
          oracle.dq_rows(q, k, v, do, rows[:24], causal=True))
    # key rows at chunk and tile edges, the sequence's first and last rows
    krows = [(0, 2, s) for s in sorted(set(edges[:14]) | {sh.S - 1})]
    dk_ref, dv_ref = oracle.dkv_rows(q, k, v, do, krows, causal=True)
    check("dk rows", torch.stack([dk[b, s, h].cpu() for b, h, s in krows]), dk_ref)
    check("dv rows", torch.stack([dv[b, s, h].cpu() for b, h, s in krows]), dv_ref)
    G = sh.Hq // sh.Hkv
    dv_sum = dv.float().sum(dim=1)  # [B, Hkv, D]
    do_sum = do.float().sum(dim=1).view(sh.B, sh.Hkv, G, sh.D).sum(dim=2).to(dv_sum.device)
    assert ((dv_sum - do_sum).norm() / do_sum.norm()).item() < 2e-2
    assert (dk.float().sum(dim=1).abs().max() / dk.float().abs().sum(dim=1).max()).item() < 2e-2
