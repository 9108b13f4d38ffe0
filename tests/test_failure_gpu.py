"""Failure detection in the attention kernels themselves, on the GPU.

Every device-side wait of the attention kernels is bounded.  With the
test-only switch CTX_DEBUG_SKIP_ARRIVAL the TMA producers of each kernel
issue no loads (and so no mbarrier arrivals) from their second load step on,
so a consumer's wait runs out: the kernel must record CTX_ERR_TIMEOUT in the
device status word, leave its loops, wait (bounded) for its own copies and
products in flight, free its tensor memory and return.  Nothing faults,
traps or hangs; the test then runs the same call normally and holds it to
the oracle, which shows the context and the tensor memory are usable again.

The lesson comes from DeepSpeed issue #7842 ("[BUG] DistributedAttention
produces numerically incorrect results ..."): a harness whose timed barrier
never actually times out.  Here the timeouts are made to run out on purpose
and their report is checked.
"""
import pytest
import torch

import context_attention_fwd_gb300 as ctx
import oracle
from seeded_inputs import AttnShape, attn_inputs
from test_parity_gpu import LSE_TOL, check, check_full

pytestmark = pytest.mark.gpu

TIMEOUT = 5  # CTX_ERR_TIMEOUT
LIMIT_MS = 100  # device wait limit while the injection is on


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ctx.load_library(build_if_missing=True)
    assert ctx.device_status() == 0
    yield
    ctx.debug_set()
    assert ctx.device_status() == 0


def _inject():
    ctx.debug_set(ctx.DEBUG_SKIP_ARRIVAL, LIMIT_MS)


def _restore():
    ctx.debug_set()


# (D, causal, shape): few CTAs each (one wave), at least two load steps per CTA
CASES = [
    (64, False, AttnShape(B=1, S=600, Hq=2, Hkv=2, D=64, P=2)),
    (128, False, AttnShape(B=1, S=777, Hq=4, Hkv=2, D=128, P=3)),
    (128, True, AttnShape(B=2, S=1001, Hq=2, Hkv=1, D=128, P=4, layout="sbhd")),
    (256, False, AttnShape(B=1, S=700, Hq=4, Hkv=2, D=256, P=2)),
    (256, True, AttnShape(B=1, S=1024, Hq=6, Hkv=1, D=256, P=2)),
]


@pytest.mark.parametrize("D,causal,sh", CASES)
def test_forward_wait_timeout_is_reported_and_recovered(D, causal, sh):
    q, k, v, do = attn_inputs(sh)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    _inject()
    try:
        ctx.attn_fwd(qd, kd, vd, sh.P, causal=causal)
        assert ctx.device_status() == TIMEOUT
    finally:
        _restore()
    assert ctx.device_status() == 0  # reading cleared it
    out, lse = ctx.attn_fwd(qd, kd, vd, sh.P, causal=causal)
    assert ctx.device_status() == 0
    o_ref, l_ref = oracle.attn_fwd(q, k, v, causal=causal)
    check("out after recovery", out, o_ref)
    assert (lse.double().cpu() - l_ref).abs().max() < LSE_TOL


@pytest.mark.parametrize("D,causal,sh", CASES)
def test_backward_wait_timeout_is_reported_and_recovered(D, causal, sh):
    q, k, v, do = attn_inputs(sh)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    out, lse = ctx.attn_fwd(qd, kd, vd, sh.P, causal=causal)
    assert ctx.device_status() == 0
    _inject()
    try:
        ctx.attn_bwd(qd, kd, vd, out, lse, dod, sh.P, causal=causal)
        assert ctx.device_status() == TIMEOUT
    finally:
        _restore()
    dq, dk, dv = ctx.attn_bwd(qd, kd, vd, out, lse, dod, sh.P, causal=causal)
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    check_full((q, k, v, do), (out, lse, dq, dk, dv), causal=causal)


def test_injection_switch_is_off_by_default_and_refuses_unknown_bits():
    with pytest.raises(ctx.CtxError):
        ctx.debug_set(0x80)
    with pytest.raises(ctx.CtxError):
        ctx.debug_set(0, 10 ** 6)
    sh = AttnShape(B=1, S=300, Hq=2, Hkv=2, D=128, P=2)
    q, k, v, do = (t.cuda() for t in attn_inputs(sh))
    ctx.attn_fwd(q, k, v, sh.P)
    assert ctx.device_status() == 0


def test_kernels_are_sm103a_machine_code():
    """The attention kernels carry machine code for compute capability 10.3
    (sm_103a), queried from the runtime, and the device is one."""
    major, minor = torch.cuda.get_device_capability()
    assert (major, minor) == (10, 3)
    assert ctx.kernel_binary_version() == 103


def test_launch_plan_at_the_devices_sm_count():
    """The D=256 backward's GQA split on the 24/4-head, 1024-token model at
    this device's SM count: a divisor of the group size, no larger than the
    smallest split that gives one CTA per SM (what the workspace is sized
    for), and the CTA count that follows from it."""
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    for causal in (False, True):
        plan = ctx.launch_plan(1, 1024, 24, 4, 256, 2, causal=causal)
        G, tiles = 6, 8
        base = tiles * 4 * 2
        cap = next((d for d in range(1, G) if G % d == 0 and base * d >= nsm), G)
        d = plan["bwd_group_split"]
        assert G % d == 0 and 1 <= d <= cap
        assert plan["bwd_ctas"] == base * d
        assert plan["bwd_head_major"] == (1 if causal and base * d <= 4 * nsm else 0)
