"""The C ABI from a plain C program on the GPU (no Python or torch in the program): it
allocates device buffers with the CUDA runtime, runs cca_pool and cca_attn_fwd on a stream
it created, and writes its inputs and outputs to a file, which this test checks against the
fp64 oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from parity import check_out
from sparse_long_context_cca_gb300 import api

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
B, HQ, HKV, N, D, G, W = 1, 4, 2, 768, 128, 16, 200  # as in c_abi_prefill.c


def _cuda_home():
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.isdir(os.path.join(c, "include")):
            return c
    nvcc = shutil.which("nvcc")
    return os.path.dirname(os.path.dirname(nvcc)) if nvcc else None


def test_c_program_prefill(tmp_path):
    cc, cuda = shutil.which("gcc") or shutil.which("cc"), _cuda_home()
    if cc is None or cuda is None:
        pytest.skip("no C compiler or CUDA toolkit")
    libdir = os.path.dirname(api.library_path())
    exe = tmp_path / "c_abi_prefill"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-I", os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c_abi_prefill.c"),
                        "-L", libdir, "-lcca", "-L", os.path.join(cuda, "lib64"), "-lcudart",
                        "-Wl,-rpath," + libdir, "-Wl,-rpath," + os.path.join(cuda, "lib64"), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = tmp_path / "io.bin"
    r = subprocess.run([str(exe), str(out)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    raw = np.fromfile(out, dtype=np.uint8)
    nq, nk = B * HQ * N * D, B * HKV * N * D
    sizes = [nq * 2, nk * 2, nk * 2, nq * 2, B * HQ * N * 4]
    assert raw.size == sum(sizes)
    parts, at = [], 0
    for n in sizes:
        parts.append(raw[at:at + n])
        at += n

    def bf16(buf, shape):
        return torch.from_numpy(buf.view(np.int16).copy()).view(torch.bfloat16).reshape(shape)

    Q = bf16(parts[0], (B, HQ, N, D))
    K = bf16(parts[1], (B, HKV, N, D))
    V = bf16(parts[2], (B, HKV, N, D))
    O = bf16(parts[3], (B, HQ, N, D))
    L = torch.from_numpy(parts[4].view(np.float32).copy()).reshape(B, HQ, N)
    Or, Lr, _, _ = oracle.prefill(Q, K, V, G, W)
    check_out(O, L, Or, Lr, torch.bfloat16, "C program")
