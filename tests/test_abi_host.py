"""Host-side checks of the C ABI library (no GPU needed): it builds for
sm_103a, loads, exports every function include/ctx_attn.h declares, and its
host-only logic (chunk table, workspace sizing, argument validation that
happens before any launch) behaves as documented."""
import ctypes
import os
import re

import pytest

import context_attention_fwd_gb300 as ctx
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ctx_attn.h")


@pytest.fixture(scope="module")
def lib():
    return ctx.load_library(build_if_missing=True)


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(ctx_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert {"ctx_attn_fwd", "ctx_attn_bwd", "ctx_seq_head_exchange"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in ctx_attn.h but not exported"


def test_library_is_built_for_sm103a():
    """The build compiles every translation unit and links for sm_103a
    only (one -gencode, no PTX for other targets), and the library on disk
    is up to date with the sources.  On a GPU the runtime's binaryVersion
    of the kernels is checked too (tests/test_failure_gpu.py)."""
    from context_attention_fwd_gb300 import build as b
    assert b.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert os.path.exists(ctx.library_path()) and b.up_to_date()


def test_debug_switches_validate_their_arguments(lib):
    assert lib.ctx_debug_set(0x80, 0) == 1       # unknown flag bit
    assert lib.ctx_debug_set(0, 60001) == 1      # wait limit above 60 s
    assert lib.ctx_debug_set(1, 100) == 0
    assert lib.ctx_debug_set(0, 0) == 0          # back to normal operation


@pytest.mark.parametrize("S,P", [(1001, 4), (32760, 8), (512, 2), (4608, 4), (5, 5), (17, 3), (65536, 4)])
def test_chunk_table_matches_array_split(S, P):
    assert ctx.chunk_offsets(S, P) == oracle.chunk_offsets(S, P)


def test_chunk_table_examples():
    off = ctx.chunk_offsets(1001, 4)
    assert [b - a for a, b in zip(off[:-1], off[1:])] == [251, 250, 250, 250]
    off = ctx.chunk_offsets(32760, 8)
    assert all(b - a == 4095 for a, b in zip(off[:-1], off[1:]))


def test_chunk_table_rejects_empty_chunks(lib):
    arr = (ctypes.c_int * 8)()
    assert lib.ctx_chunk_offsets(3, 4, arr) == 1
    assert lib.ctx_chunk_offsets(3, 0, arr) == 1


def test_workspace_size(lib):
    # backward: two fp32 row-statistics arrays + the fp32 dq accumulator over
    # 128-row tiles (each chunk padded to whole tiles)
    n = lib.ctx_attn_workspace_size(1, 32760, 24, 24, 128, 8, 0)
    slots = 24 * (8 * 32) * 128
    assert n >= slots * 4 * 2 + slots * 128 * 4
    assert lib.ctx_attn_workspace_size(1, 10, 6, 4, 64, 2, 0) == 0  # Hq % Hkv != 0
    assert lib.ctx_attn_workspace_size(1, 10, 4, 4, 64, 11, 0) == 0  # P > S
    # materialised partials need P * rows * (D + 1) fp32
    n2 = lib.ctx_attn_workspace_size(1, 1000, 4, 4, 64, 4, 1)
    assert n2 >= 4 * 4 * 1000 * 65 * 4


def test_exchange_padded_len(lib):
    assert lib.ctx_exchange_padded_len(65536, 4, 2) == 65536
    assert lib.ctx_exchange_padded_len(1001, 4, 2) == 1008
    assert lib.ctx_exchange_padded_len(10, 1, 2) == 10
    assert lib.ctx_exchange_padded_len(0, 1, 2) == -1


def test_status_strings(lib):
    for code in range(6):
        assert lib.ctx_status_string(code)
    assert b"timed out" in lib.ctx_status_string(5)


def _t(data, B, S, H, D):
    return ctx._Tensor(data, B, S, H, D, 0, 0, 0)


def test_invalid_arguments_fail_before_launch(lib):
    """Validation runs on the host and writes nothing; these calls need no GPU."""
    fake = 1 << 20  # never dereferenced: validation fails first
    lse = ctypes.c_void_p(fake)
    q = _t(fake, 1, 64, 4, 64)
    kv = _t(fake, 1, 64, 2, 64)
    out = _t(fake, 1, 64, 4, 64)
    call = lambda **kw: lib.ctx_attn_fwd(
        ctypes.byref(kw.get("q", q)), ctypes.byref(kw.get("k", kv)), ctypes.byref(kw.get("v", kv)),
        kw.get("P", 2), None, kw.get("layout", 0), kw.get("causal", 0), 0.0,
        ctypes.byref(kw.get("out", out)), kw.get("lse", lse), None, 0, kw.get("flags", 0), None)
    assert call(P=0) == 1                               # P < 1
    assert call(P=65) == 1                              # P > S
    big_q, big_kv, big_o = _t(fake, 1, 1000, 4, 64), _t(fake, 1, 1000, 2, 64), _t(fake, 1, 1000, 4, 64)
    assert call(q=big_q, k=big_kv, v=big_kv, out=big_o, P=65) == 1  # more chunks than the table holds
    for empty in ((0, 64, 4, 64), (1, 0, 4, 64), (1, 64, 0, 64), (1, 64, 4, 0)):  # empty inputs
        B_, S_, H_, D_ = empty
        e = _t(fake, B_, S_, H_, D_)
        assert call(q=e, k=e, v=e, out=e) == 1, empty
    assert call(k=_t(fake, 1, 64, 3, 64), v=_t(fake, 1, 64, 3, 64)) == 1  # Hq % Hkv
    assert call(layout=7) == 1
    assert call(lse=None) == 1
    assert call(q=_t(fake, 1, 64, 4, 96), k=_t(fake, 1, 64, 2, 96), v=_t(fake, 1, 64, 2, 96),
                out=_t(fake, 1, 64, 4, 96)) == 2        # D = 96 unsupported
    assert call(causal=1, flags=1) == 3                 # causal with materialised partials: needs a workspace
    assert call(out=_t(fake, 1, 63, 4, 64)) == 1        # shape mismatch
    assert call(q=_t(fake + 2, 1, 64, 4, 64)) == 2      # misaligned for TMA
    assert call(flags=1) == 3                           # partials need a workspace
    assert call(flags=4) == 1                           # unknown flag
    assert call(flags=3) == 3                           # all-gather order + partials: needs a workspace
    offs = (ctypes.c_int * 3)(0, 40, 63)                # must end at S
    assert lib.ctx_attn_fwd(ctypes.byref(q), ctypes.byref(kv), ctypes.byref(kv), 2, offs, 0, 0, 0.0,
                            ctypes.byref(out), lse, None, 0, 0, None) == 1
    offs = (ctypes.c_int * 3)(0, 0, 64)                 # empty chunk
    assert lib.ctx_attn_fwd(ctypes.byref(q), ctypes.byref(kv), ctypes.byref(kv), 2, offs, 0, 0, 0.0,
                            ctypes.byref(out), lse, None, 0, 0, None) == 1


def test_bwd_invalid_arguments(lib):
    fake = 1 << 20
    q = _t(fake, 1, 64, 4, 64)
    kv = _t(fake, 1, 64, 2, 64)
    lse = ctypes.c_void_p(fake)
    args = [ctypes.byref(q), ctypes.byref(kv), ctypes.byref(kv), ctypes.byref(q), lse,
            ctypes.byref(q), 2, None, 0, 0, 0.0, ctypes.byref(q), ctypes.byref(kv), ctypes.byref(kv)]
    assert lib.ctx_attn_bwd(*args, None, 0, None) == 3                 # no workspace
    assert lib.ctx_attn_bwd(*args, ctypes.c_void_p(fake), 16, None) == 3  # too small
    need = lib.ctx_attn_workspace_size(1, 64, 4, 2, 64, 2, 0)
    assert lib.ctx_attn_bwd(*args, ctypes.c_void_p(fake + 16), need, None) == 3  # misaligned
    bad = list(args)
    bad[6] = 0
    assert lib.ctx_attn_bwd(*bad, ctypes.c_void_p(fake), need, None) == 1


def test_exchange_invalid_arguments(lib):
    fake = 1 << 20
    x = _t(fake, 1, 16, 6, 64)
    assert lib.ctx_seq_head_exchange(ctypes.byref(x), ctypes.c_void_p(fake), 2, 4, 0, 0, None) == 1  # H % U
    assert lib.ctx_seq_head_exchange(ctypes.byref(x), ctypes.c_void_p(fake), 2, 2, 3, 0, None) == 1  # dir
    assert lib.ctx_seq_head_exchange(ctypes.byref(x), None, 2, 2, 0, 0, None) == 1
    assert lib.ctx_seq_head_exchange(ctypes.byref(x), ctypes.c_void_p(fake + 8), 2, 2, 0, 0, None) == 2


def test_product_path_does_not_import_the_oracle():
    """The library package never routes through oracle/ (no CPU fallback)."""
    pkg = os.path.join(ROOT, "context_attention_fwd_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f


def test_chunk_table_random_splits():
    """Random (S, P): the library's chunk table is numpy's array_split, and
    every workspace size covers the backward's fixed parts."""
    hyp = pytest.importorskip("hypothesis")
    st = hyp.strategies

    @hyp.settings(max_examples=200, deadline=None)
    @hyp.given(S=st.integers(1, 200000), P=st.integers(1, 64))
    def check(S, P):
        if P > S:
            return
        assert ctx.chunk_offsets(S, P) == oracle.chunk_offsets(S, P)

    check()


@pytest.mark.parametrize("D", [64, 128, 256])
def test_workspace_grows_with_the_problem(lib, D):
    sizes = [lib.ctx_attn_workspace_size(1, S, 8, 2, D, 4, 0) for S in (512, 1024, 4096, 16384)]
    assert all(a < b for a, b in zip(sizes, sizes[1:]))
    assert lib.ctx_attn_workspace_size(2, 4096, 8, 2, D, 4, 0) > sizes[2]



def test_missing_library_fails_loudly():
    """No CPU path: without the compiled library every entry point raises."""
    code = (
        "import context_attention_fwd_gb300 as ctx, context_attention_fwd_gb300.build as b\n"
        "b.LIB = '/nonexistent/libctxattn.so'\n"
        "try:\n"
        "    ctx.load_library(build_if_missing=False)\n"
        "except RuntimeError as e:\n"
        "    print('raised', e)\n"
    )
    import subprocess
    import sys
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT, timeout=120)
    assert r.returncode == 0 and r.stdout.startswith("raised"), r.stdout + r.stderr


def test_binding_checks_element_types_before_any_call(lib):
    """The C ABI carries no element type (bf16 throughout, fp32 lse): the
    binding refuses other types and host tensors with a ValueError before it
    allocates or calls anything, so no call can read the wrong bytes."""
    import torch
    q32 = torch.zeros(1, 8, 2, 64, dtype=torch.float32)
    with pytest.raises(ValueError, match="bfloat16"):
        ctx.attn_fwd(q32, q32, q32, 1)
    qb = q32.bfloat16()
    with pytest.raises(ValueError, match="bfloat16"):
        ctx.attn_fwd(qb, q32.half(), qb, 1)
    with pytest.raises(ValueError, match="CUDA device"):
        ctx.attn_fwd(qb, qb, qb, 1)
    with pytest.raises(ValueError, match="bfloat16"):
        ctx.attn_bwd(qb, qb, qb, qb, torch.zeros(1, 2, 8), q32, 1)
    with pytest.raises(ValueError, match="lse"):
        ctx.attn_bwd(qb, qb, qb, qb, torch.zeros(1, 2, 8, dtype=torch.float64), qb, 1)
    with pytest.raises(ValueError, match=r"\[B,S,H,D\]"):
        ctx.attn_fwd(qb[0], qb[0], qb[0], 1)
    with pytest.raises(ValueError, match="16-bit"):
        ctx.seq_head_exchange(q32, 2, 1, 0, "bshd")


def test_plain_c_client_links_and_runs(lib, tmp_path):
    """tests/c_client/abi_client.c includes only ctx_attn.h (as C99, with
    warnings as errors), links the shared library and checks the host-side
    entry points and early refusals: the boundary needs neither C++ nor
    Python."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    libdir = os.path.dirname(ctx.library_path())
    src = os.path.join(os.path.dirname(__file__), "c_client", "abi_client.c")
    exe = str(tmp_path / "abi_client")
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.dirname(HEADER), src,
           "-L", libdir, "-lctxattn", f"-Wl,-rpath,{libdir}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and "abi client ok" in r.stdout, r.stdout + r.stderr


def test_launch_plan(lib):
    """Launch decisions, on the host.  Without a GPU the library takes 148
    SMs."""
    # not causal: each head's tiles together, no group split
    p = ctx.launch_plan(1, 32760, 24, 24, 128, 8)
    assert (p["fwd_head_major"], p["bwd_head_major"], p["bwd_group_split"]) == (0, 0, 1)
    assert p["fwd_ctas"] == 8 * 16 * 24 and p["bwd_ctas"] == 8 * 32 * 24  # 16 tile pairs, 32 tiles per chunk
    # causal on a grid of many waves: still tile-major
    p = ctx.launch_plan(1, 32760, 24, 24, 128, 8, causal=True)
    assert (p["fwd_head_major"], p["bwd_head_major"]) == (0, 0)
    # causal on a small grid: heads first
    p = ctx.launch_plan(1, 777, 4, 2, 128, 3, causal=True)
    assert (p["fwd_head_major"], p["bwd_head_major"], p["bwd_group_split"]) == (1, 1, 1)
    # the 24/4-head D=256 causal model at 1024 tokens: heads first, group split in three
    p = ctx.launch_plan(1, 1024, 24, 4, 256, 2, causal=True)
    assert (p["fwd_head_major"], p["bwd_head_major"], p["bwd_group_split"]) == (1, 1, 3)
    assert p["fwd_ctas"] == 8 * 24 and p["bwd_ctas"] == 8 * 4 * 2 * 3
    # the same heads not causal: split in two, one wave
    p = ctx.launch_plan(1, 1024, 24, 4, 256, 2)
    assert (p["bwd_group_split"], p["bwd_head_major"], p["bwd_ctas"]) == (2, 0, 128)
    # refusals as in the attention calls
    with pytest.raises(ctx.CtxError) as e:
        ctx.launch_plan(1, 1024, 24, 4, 96, 2)
    assert e.value.code == 2
    with pytest.raises(ctx.CtxError) as e:
        ctx.launch_plan(1, 3, 1, 1, 64, 4)
    assert e.value.code == 1


@pytest.mark.parametrize("causal", [False, True])
def test_group_split_fits_the_workspace(lib, causal):
    """Whatever split the backward picks, its fp32 partial rows fit in the
    workspace that ctx_attn_workspace_size reports (any chunking of S)."""
    import random
    rng = random.Random(5 + causal)
    for _ in range(40):
        B, Hkv = rng.choice([1, 2]), rng.choice([1, 2, 4])
        Hq = Hkv * rng.choice([1, 2, 3, 4, 6, 8])
        S = rng.randint(1, 5000)
        P = rng.randint(1, min(S, 16))
        p = ctx.launch_plan(B, S, Hq, Hkv, 256, P, causal=causal)
        ntiles_max = sum(-(-(S // P + (c < S % P)) // 128) for c in range(P))
        need = 2 * B * Hq * ntiles_max * 128 * 4 + B * Hq * ntiles_max * 128 * 256 * 4
        if p["bwd_group_split"] > 1:
            need += p["bwd_group_split"] * B * Hkv * S * 2 * 256 * 4
        assert lib.ctx_attn_workspace_size(B, S, Hq, Hkv, 256, P, 0) >= need
        assert (Hq // Hkv) % p["bwd_group_split"] == 0


@pytest.mark.parametrize("D", [64, 128, 256])
def test_launch_order_rule(lib, D):
    """Heads first exactly for causal calls on grids of at most four CTAs per
    SM (148 SMs without a GPU), for both kernels."""
    for S in (64, 500, 1024, 3000, 8192, 20000):
        for Hq, Hkv in ((24, 24), (24, 4), (4, 2)):
            for causal in (False, True):
                p = ctx.launch_plan(1, S, Hq, Hkv, D, 4, causal=causal)
                assert p["fwd_head_major"] == int(causal and p["fwd_ctas"] <= 4 * 148)
                assert p["bwd_head_major"] == int(causal and p["bwd_ctas"] <= 4 * 148)
