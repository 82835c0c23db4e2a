"""The bounds-checked build (libgqa_decode_checked.so, compiled with GQA_BOUNDS_CHECK=1): every
computed global- and shared-memory offset of the kernels is range-checked on the device, and a
failure would set GQA_ERR_BOUNDS in the status word instead of making the access.

Run over the small ragged shapes -- key counts around the tile and block edges, every kernel
(mma.sync split kernel with each merge, its cluster and deep-ring variants, the tcgen05 kernel,
the paged kernel over both cache layouts, the merge kernels) -- each call must leave the status
word clean and match the CPU float64 oracle at the parity tolerance.  Calls go through the C ABI of the checked
library.
"""
from __future__ import annotations

import ctypes
import math

import numpy as np
import pytest
import torch

import gqa_inputs as gi
import oracle
from test_gpu_parity import assert_close

pytestmark = pytest.mark.gpu

LENGTHS = [1, 2, 63, 64, 65, 127, 129, 511, 513, 4097]


@pytest.fixture(scope="module")
def chk():
    from decode_attention_03_gb300 import build
    path = build.build(checked=True)
    import decode_attention_03_gb300._binding as b
    assert torch.cuda.is_available()
    lib = b.open_library(path)
    assert lib.gqa_build_flags() == b.GQA_BUILD_BOUNDS_CHECK
    return b, lib


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() else None


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ws(lib, nbytes):
    ws = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device="cuda")
    return ws


def _decode(b, lib, x, **opt):
    q, k, v = (torch.from_numpy(x[n]).cuda() for n in ("q", "k", "v"))
    B, T_q, _ = q.shape
    S = k.shape[1]
    hq, hkv, D = x["h_q"], x["h_kv"], x["d_head"]
    o = torch.full_like(q, float("nan"))
    ws = _ws(lib, lib.gqa_decode_workspace_size(B, T_q, S, hq, hkv, D, opt.get("n_splits", 0)))
    op = b._opts(**opt)
    st = lib.gqa_decode_ex(_p(q), _p(k), _p(v), _p(o), B, T_q, S, hq, hkv, D, x["scale"], _p(ws), ws.numel(),
                           _stream(), ctypes.byref(op))
    assert st == b.GQA_OK, b.gqa_status_string(st)
    assert lib.gqa_workspace_check(_p(ws), _stream()) == b.GQA_OK
    return o


@pytest.mark.parametrize("S", LENGTHS)
@pytest.mark.parametrize("D", [64, 128])
def test_checked_contiguous(chk, S, D):
    b, lib = chk
    x = gi.make_contiguous(gi.custom(2, 1, S, 8, 2, D, 9100 + S + D))
    ref = oracle.decode(x["q"], x["k"], x["v"], 8, 2, D, x["scale"])
    for opt in ({}, {"n_splits": 3, "merge_mode": 1}, {"n_splits": 5, "merge_mode": 2},
                {"n_splits": 7, "merge_mode": 3}):
        assert_close(_decode(b, lib, x, **opt), ref, f"checked S={S} D={D} {opt}")


def test_checked_deep_ring(chk):
    """The split kernel's deep-ring variant (one CTA per SM), which the plan takes for 8 units where the
    SMs divide into more than 16 splits of at least 48 tiles."""
    b, lib = chk
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms % 8 or sms // 8 <= 16:
        pytest.skip("no deep-ring grid for 8 units on this GPU")
    S = (sms // 8) * 48 * 64 + 37
    x = gi.make_contiguous(gi.custom(1, 1, S, 32, 8, 128, 9500))
    ref = oracle.decode(x["q"], x["k"], x["v"], 32, 8, 128, x["scale"])
    assert_close(_decode(b, lib, x), ref, "checked deep ring")


@pytest.mark.parametrize("S", [1, 65, 513, 4097])
@pytest.mark.parametrize("T_q,hq,hkv", [(4, 64, 8), (2, 32, 2), (16, 64, 8)])
def test_checked_many_rows(chk, S, T_q, hq, hkv):
    """16 to 128 query rows per KV head: the tcgen05 kernel (and the mma.sync kernel's larger row
    classes where they fit), plain and causal."""
    b, lib = chk
    x = gi.make_contiguous(gi.custom(1, T_q, S, hq, hkv, 128, 9200 + S + T_q))
    ref = oracle.decode(x["q"], x["k"], x["v"], hq, hkv, 128, x["scale"])
    rows = hq // hkv * T_q
    paths = [2] + ([1] if rows <= 64 else [])
    for path in paths:
        for n in (1, 4):
            assert_close(_decode(b, lib, x, n_splits=n, mma_path=path), ref, f"checked rows={rows} path={path}")
    refc = oracle.decode(x["q"], x["k"], x["v"], hq, hkv, 128, x["scale"], causal=True)
    assert_close(_decode(b, lib, x, n_splits=3, mma_path=2, causal=True), refc, "checked causal tcgen05")


@pytest.mark.parametrize("rng", [(0, 513), (100, 0), (63, 65), (4000, 97)])
def test_checked_partial_and_merge(chk, rng):
    b, lib = chk
    s0, n = rng
    x = gi.make_contiguous(gi.custom(2, 2, 4097, 16, 4, 64, 9300))
    q, k, v = (torch.from_numpy(x[c]).cuda() for c in ("q", "k", "v"))
    R, D = 2 * 2 * 16, 64
    m = torch.empty(R, device="cuda")
    l = torch.empty(R, device="cuda")
    op = torch.empty(R, D, device="cuda")
    ws = _ws(lib, lib.gqa_decode_workspace_size(2, 2, max(n, 1), 16, 4, D, 0))
    st = lib.gqa_decode_partial(_p(q), _p(k), _p(v), _p(m), _p(l), _p(op), 2, 2, 4097, s0, n, 16, 4, D,
                                x["scale"], _p(ws), ws.numel(), _stream())
    assert st == b.GQA_OK
    assert lib.gqa_workspace_check(_p(ws), _stream()) == b.GQA_OK
    rm, rl, ro = oracle.decode_partial(x["q"], x["k"], x["v"], 16, 4, D, x["scale"], s0, n)
    if n == 0:
        assert torch.isneginf(m).all() and (l == 0).all() and (op == 0).all()
        return
    rl, ro = rl.reshape(-1), ro.reshape(-1, D)
    assert_close(op.double().cpu() / l.double().cpu()[:, None], oracle.normalize(rl, ro), f"checked partial {rng}")
    # the public merge over two copies of the partial: the same normalised result
    o = torch.empty(R, D, dtype=torch.float16, device="cuda")
    m2, l2, op2 = torch.stack([m, m]), torch.stack([l, l]), torch.stack([op, op])   # alive across the call
    st = lib.gqa_merge(_p(m2), _p(l2), _p(op2), 2, R, D, _p(o), _stream())
    assert st == b.GQA_OK
    torch.cuda.synchronize()
    assert_close(o, oracle.normalize(rl, ro), f"checked merge {rng}")


@pytest.mark.parametrize("bs,part", [(16, 512), (8, 64), (64, 512)])
@pytest.mark.parametrize("vllm", [False, True])
def test_checked_paged(chk, bs, part, vllm):
    b, lib = chk
    hq, hkv, D = 32, 8, 128
    lens = np.array([0, 1, 15, 16, 17, 511, 512, 513, 1000, 64, 2049], dtype=np.int32)
    N = len(lens)
    nblk = (lens + bs - 1) // bs
    num_blocks = int(nblk.sum()) + 3
    perm = np.random.Generator(np.random.PCG64(bs + part)).permutation(num_blocks).astype(np.int32)
    tab = np.full((N, int(nblk.max())), -1, dtype=np.int32)
    off = 0
    for i in range(N):
        tab[i, :nblk[i]] = perm[off:off + nblk[i]]
        off += nblk[i]
    qn = gi.normal_f16(9400 + bs, 0, (N, 1, hq * D))
    kp = gi.normal_f16(9400 + bs, 1, (num_blocks, bs, hkv * D))
    vp = gi.normal_f16(9400 + bs, 2, (num_blocks, bs, hkv * D))
    scale = 1 / math.sqrt(D)
    ref = oracle.decode_paged(qn, kp, vp, tab, lens, hq, hkv, D, scale, bs).reshape(N, -1)
    if vllm:
        kc, vc = gi.to_vllm_layout(kp, vp, hkv, D)
    else:
        kc, vc = kp, vp
    q, k, v, t, ln = (torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (qn.reshape(N, -1), kc, vc, tab, lens))
    o = torch.full_like(q, float("nan"))
    ws = _ws(lib, lib.gqa_paged_workspace_size(N, hq, hkv, D, int(lens.max()), part))
    fn = lib.gqa_decode_paged_vllm if vllm else lib.gqa_decode_paged
    st = fn(_p(q), _p(k), _p(v), _p(t), _p(ln), _p(o), N, tab.shape[1], num_blocks, bs, part, hq, hkv, D, scale,
            int(lens.max()), _p(ws), ws.numel(), _stream())
    assert st == b.GQA_OK, b.gqa_status_string(st)
    assert lib.gqa_workspace_check(_p(ws), _stream()) == b.GQA_OK
    assert bool((ref[0] == 0).all()) and (o[0].float() == 0).all()
    assert_close(o, ref, f"checked paged bs={bs} part={part} vllm={vllm}")
