"""gqa_decode_noalloc -- the decode entry point for callers that cannot allocate device memory.

Some callers cannot give the library a workspace: a plugin whose device memory is owned
and budgeted by its host framework, a latency-critical loop that cannot take cudaMalloc's
implicit synchronisation, a C / FFI caller without a device allocator.  For them
gqa_decode_noalloc uses a device array the library owns (8 MiB per GPU).  These tests
call it through the C ABI and check it, on two calls in a row, against the CPU float64
oracle and against gqa_decode (the regular entry point, with a caller workspace), within
the tolerance the parity tests use; gqa_decode_noalloc_check then reports a clean status.
This file is collected last on purpose and also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import gqa_inputs as gi
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from decode_attention_03_gb300 import build
    build.build()
    import decode_attention_03_gb300._binding as b
    assert torch.cuda.is_available()
    return b


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _within(a, b):
    a, b = a.double().cpu().reshape(b.shape), b.double().cpu()
    return bool(((a - b).abs() <= 2e-3 + 2e-3 * b.abs()).all())


def _rel_l2(a, b):
    a, b = a.double().cpu().reshape(b.shape), b.double().cpu()
    return float((a - b).norm() / b.norm())


@pytest.mark.parametrize("shape", [(2, 1, 5000, 32, 8, 128), (1, 4, 131071, 64, 8, 128), (1, 1, 4096, 8, 2, 64),
                                   (1, 1, 19 * 48 * 64 + 37, 32, 8, 128)])   # 152 SMs: the deep ring + merge kernel
def test_noalloc_matches_regular_entry_point_twice(lib, shape):
    B, T_q, S, hq, hkv, D = shape
    x = gi.make_contiguous(gi.custom(B, T_q, S, hq, hkv, D, 1234 + S))
    q, k, v = (torch.from_numpy(x[n]).cuda() for n in ("q", "k", "v"))
    scale = 1.0 / np.sqrt(D)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    nbytes = lib.lib.gqa_decode_workspace_size(B, T_q, S, hq, hkv, D, 0)
    assert 0 < nbytes <= lib.GQA_NOALLOC_SCRATCH_BYTES
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    ref = torch.empty_like(q)
    st = lib.lib.gqa_decode(_p(q), _p(k), _p(v), _p(ref), B, T_q, S, hq, hkv, D, scale, _p(ws), nbytes, stream)
    assert st == lib.GQA_OK

    exact = oracle.decode(x["q"], x["k"], x["v"], hq, hkv, D, scale)
    for call in range(2):                       # the array keeps the previous call's contents
        out = torch.full_like(q, float("nan"))
        st = lib.lib.gqa_decode_noalloc(_p(q), _p(k), _p(v), _p(out), B, T_q, S, hq, hkv, D, scale, stream)
        assert st == lib.GQA_OK, lib.gqa_status_string(st)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        assert _within(out, exact), f"call {call} against the oracle"
        assert _rel_l2(out, exact) <= 5e-3, f"call {call} against the oracle"
        assert _within(out, ref), f"call {call} against gqa_decode"
    assert lib.lib.gqa_decode_noalloc_check(stream) == lib.GQA_OK


def test_noalloc_rejects_shapes_beyond_its_array(lib):
    # 40000 sequences x 64 KV heads need 10 MB of arrival counters alone (> 8 MiB)
    B, T_q, S, hq, hkv, D = 40000, 1, 1, 64, 64, 64
    need = lib.lib.gqa_decode_workspace_size(B, T_q, S, hq, hkv, D, 0)
    assert need > lib.GQA_NOALLOC_SCRATCH_BYTES
    q = torch.zeros(B, T_q, hq * D, dtype=torch.float16, device="cuda")
    k = torch.zeros(B, S, hkv * D, dtype=torch.float16, device="cuda")
    out = torch.zeros_like(q)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.lib.gqa_decode_noalloc(_p(q), _p(k), _p(k), _p(out), B, T_q, S, hq, hkv, D, 0.125, stream)
    assert st == lib.GQA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert (out == 0).all()                     # nothing was launched
