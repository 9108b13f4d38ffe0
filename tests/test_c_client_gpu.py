"""A plain C program runs the forward and backward on the GPU through the C
ABI alone (tests/c_client/gpu_client.c: CUDA runtime C API for memory and
stream, no Python, no torch).  Its outputs are held against the fp64 oracle
and, for the forward, against the Python binding's bit for bit (the same
kernels on the same inputs)."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import context_attention_fwd_gb300 as ctx
from seeded_inputs import AttnShape, attn_inputs
from test_parity_gpu import check_full

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    ctx.load_library(build_if_missing=True)
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    libdir = os.path.dirname(ctx.library_path())
    exe = str(tmp_path_factory.mktemp("c_client") / "gpu_client")
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), os.path.join(HERE, "c_client", "gpu_client.c"),
           "-L", libdir, "-lctxattn", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def _bits(t):
    return t.contiguous().view(torch.int16).numpy()


@pytest.mark.parametrize("sh,causal", [(AttnShape(B=2, S=777, Hq=4, Hkv=2, D=128, P=3), True),
                                       (AttnShape(B=1, S=1024, Hq=24, Hkv=4, D=256, P=2), True),
                                       (AttnShape(B=1, S=600, Hq=8, Hkv=8, D=64, P=4), False)])
def test_c_client_fwd_bwd(client, tmp_path, sh, causal):
    q, k, v, do = attn_inputs(sh)
    fin, fout = str(tmp_path / "in.bin"), str(tmp_path / "out.bin")
    with open(fin, "wb") as f:
        for t in (q, k, v, do):
            _bits(t).tofile(f)
    r = subprocess.run([client, fin, fout, str(sh.B), str(sh.S), str(sh.Hq), str(sh.Hkv), str(sh.D),
                        str(sh.P), str(int(causal))], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "gpu client ok" in r.stdout, r.stdout + r.stderr
    raw = np.fromfile(fout, dtype=np.uint8)
    nq, nk, nl = sh.B * sh.S * sh.Hq * sh.D, sh.B * sh.S * sh.Hkv * sh.D, sh.B * sh.Hq * sh.S
    sizes = [2 * nq, 4 * nl, 2 * nq, 2 * nk, 2 * nk]
    assert raw.size == sum(sizes)
    parts, at = [], 0
    for n in sizes:
        parts.append(torch.from_numpy(raw[at:at + n].copy()))
        at += n
    bf = lambda b, H: b.view(torch.bfloat16).view(sh.B, sh.S, H, sh.D)
    out, lse = bf(parts[0], sh.Hq), parts[1].view(torch.float32).view(sh.B, sh.Hq, sh.S)
    dq, dk, dv = bf(parts[2], sh.Hq), bf(parts[3], sh.Hkv), bf(parts[4], sh.Hkv)
    check_full((q, k, v, do), (out, lse, dq, dk, dv), causal=causal)
    o_py, l_py = ctx.attn_fwd(q.cuda(), k.cuda(), v.cuda(), sh.P, causal=causal)
    assert torch.equal(o_py.cpu().view(torch.int16), out.view(torch.int16))
    assert torch.equal(l_py.cpu(), lse)
