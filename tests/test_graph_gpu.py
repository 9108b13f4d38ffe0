"""The library makes no allocation, no synchronisation and no host round
trip inside a call, so a whole forward + backward step can be captured in a
CUDA graph and replayed: the replay must give the eager results (the
forward bit for bit; the gradients up to the order of the fp32 dQ
reductions) and match the oracle."""
import pytest
import torch

import context_attention_fwd_gb300 as ctx
import oracle
from seeded_inputs import AttnShape, attn_inputs
from test_parity_gpu import check

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D,causal", [(128, False), (256, True)])
def test_step_captured_in_a_cuda_graph(D, causal):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ctx.load_library(build_if_missing=True)
    sh = AttnShape(B=1, S=1024, Hq=8, Hkv=2, D=D, P=2)
    q_h, k_h, v_h, do_h = attn_inputs(sh, seed=41)
    q, k, v, do = (t.cuda() for t in (q_h, k_h, v_h, do_h))
    # eager step (also does the one-time per-kernel setup outside the capture)
    out_e, lse_e = ctx.attn_fwd(q, k, v, sh.P, causal=causal)
    dq_e, dk_e, dv_e = ctx.attn_bwd(q, k, v, out_e, lse_e, do, sh.P, causal=causal)
    # static buffers for the graph
    out, lse = torch.empty_like(out_e), torch.empty_like(lse_e)
    dq, dk, dv = torch.empty_like(dq_e), torch.empty_like(dk_e), torch.empty_like(dv_e)
    ws = torch.empty(ctx.workspace_size(sh.B, sh.S, sh.Hq, sh.Hkv, sh.D, sh.P), dtype=torch.uint8,
                     device="cuda")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ctx.attn_fwd(q, k, v, sh.P, causal=causal, out=out, lse=lse)
        ctx.attn_bwd(q, k, v, out, lse, do, sh.P, causal=causal, dq=dq, dk=dk, dv=dv, workspace=ws)
    for _ in range(3):  # replays reuse the same buffers
        g.replay()
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    assert torch.equal(out, out_e) and torch.equal(lse, lse_e)
    for name, a, b in (("dq", dq, dq_e), ("dk", dk, dk_e), ("dv", dv, dv_e)):
        check(name + " replay vs eager", a, b, tol=1e-2)
    o_ref, _ = oracle.attn_fwd(q_h, k_h, v_h, causal=causal)
    check("out", out, o_ref)
    g_ref = oracle.attn_bwd(q_h, k_h, v_h, do_h, causal=causal)
    for name, a, r in zip(("dq", "dk", "dv"), (dq, dk, dv), g_ref):
        check(name, a, r)
