"""The library from plain C: tests/c/decode_from_c.c includes only include/gqa_decode.h, allocates
its buffers with cudaMalloc, sizes the workspace with gqa_workspace_size and runs one gqa_decode
step -- no Python, no torch on that side.  Its output is checked against the CPU float64 oracle."""
from __future__ import annotations

import os
import subprocess

import numpy as np
import pytest

import gqa_inputs as gi
import oracle

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    from decode_attention_03_gb300 import build
    lib = build.build()
    exe = str(tmp_path_factory.mktemp("c_caller") / "decode_from_c")
    cmd = [build.nvcc(), "-O2", "-I" + os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "decode_from_c.c"),
           "-o", exe, "-L" + os.path.dirname(lib), "-lgqa_decode", "-Xlinker", "-rpath=" + os.path.dirname(lib)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


@pytest.mark.parametrize("shape", [(1, 1, 4096, 8, 2, 64), (2, 2, 5000, 32, 8, 128), (1, 16, 3001, 64, 8, 128)])
def test_c_caller_matches_oracle(program, tmp_path, shape):
    B, T, S, hq, hkv, D = shape
    x = gi.make_contiguous(gi.custom(B, T, S, hq, hkv, D, 7070 + S))
    for n in ("q", "k", "v"):
        np.ascontiguousarray(x[n]).tofile(tmp_path / f"{n}.bin")
    r = subprocess.run([program, str(tmp_path), str(B), str(T), str(S), str(hq), str(hkv), str(D), repr(x["scale"])],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    o = np.fromfile(tmp_path / "o.bin", dtype=np.float16).astype(np.float64).reshape(B, T, hq * D)
    ref = oracle.decode(x["q"], x["k"], x["v"], hq, hkv, D, x["scale"]).numpy()
    err = np.abs(o - ref)
    assert (err <= 2e-3 + 2e-3 * np.abs(ref)).all(), f"max err {err.max():.3e}"
    assert np.linalg.norm(o - ref) / np.linalg.norm(ref) <= 5e-3
