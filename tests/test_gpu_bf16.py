"""GPU parity of the bfloat16 variant against the CPU float64 oracle.

The oracle takes the exact values of the bfloat16 inputs.  Tolerance, derived from the
arithmetic: the output is rounded to bfloat16 (8 significand bits: half an ulp is at most
2^-8 = 3.9e-3 relative) and P is rounded to bfloat16 for the P.V MMA (at most 2^-8 per
weight); so every element must satisfy |o - o_ref| <= 2e-3 + 8e-3 * |o_ref|, and the
relative L2 error must stay below 1e-2 (rounding noise alone is about 2.3e-3).
"""
from __future__ import annotations


import numpy as np
import pytest
import torch

import gqa_inputs as gi
import oracle

pytestmark = pytest.mark.gpu

ABS_TOL = 2e-3
REL_TOL = 8e-3
REL_L2 = 1e-2


@pytest.fixture(scope="module")
def gqa():
    from decode_attention_03_gb300 import build
    build.build()
    import decode_attention_03_gb300._binding as b
    assert torch.cuda.is_available()
    return b


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def val(a):
    return gi.values(a, "bf16")


def assert_close(got, ref, where):
    got = got.detach().float().double().cpu().reshape(ref.shape)
    ref = ref.double()
    mask = ~torch.isnan(ref)
    g, r = got[mask], ref[mask]
    assert torch.isfinite(g).all(), f"{where}: non-finite output"
    err = (g - r).abs()
    bad = err > ABS_TOL + REL_TOL * r.abs()
    assert not bad.any(), f"{where}: {int(bad.sum())} of {g.numel()} outside tolerance, max err {float(err.max()):.3e}"
    rl2 = float((g - r).norm() / r.norm().clamp_min(1e-30))
    assert rl2 <= REL_L2, f"{where}: relative L2 error {rl2:.3e}"


def contig(B, T, S, hq, hkv, D, seed, **kw):
    return gi.make_contiguous(gi.custom(B, T, S, hq, hkv, D, seed, elem="bf16", **kw))


@pytest.mark.parametrize("B,T,S,hq,hkv,D", [(1, 1, 4096, 8, 2, 64), (2, 1, 20000, 32, 8, 128), (1, 4, 9000, 64, 8, 128),
                                            (2, 2, 777, 16, 2, 128), (3, 1, 65, 8, 8, 64)])
@pytest.mark.parametrize("n_splits", [0, 1, 5])
@pytest.mark.parametrize("path", [1, 2])
def test_bf16_decode(gqa, B, T, S, hq, hkv, D, n_splits, path):
    x = contig(B, T, S, hq, hkv, D, 2000 + S + T, v_dist="uniform", spike_frac=0.01, spike_mult=8.0)
    ref = oracle.decode(val(x["q"]), val(x["k"]), val(x["v"]), hq, hkv, D, x["scale"])
    o = gqa.gqa_decode(dev(x["q"]), dev(x["k"]), dev(x["v"]), hq, hkv, x["scale"], n_splits=n_splits, mma_path=path)
    torch.cuda.synchronize()
    assert o.dtype == torch.bfloat16
    assert_close(o, ref, f"bf16 B={B} T={T} S={S} hq={hq} hkv={hkv} D={D} splits={n_splits} path={path}")


def test_bf16_causal_and_merge_mode(gqa):
    x = contig(2, 4, 3000, 32, 8, 128, 2101)
    q, k, v = dev(x["q"]), dev(x["k"]), dev(x["v"])
    ref = oracle.decode(val(x["q"]), val(x["k"]), val(x["v"]), 32, 8, 128, x["scale"], causal=True)
    assert_close(gqa.gqa_decode(q, k, v, 32, 8, x["scale"], causal=True), ref, "bf16 causal")
    ref2 = oracle.decode(val(x["q"]), val(x["k"]), val(x["v"]), 32, 8, 128, x["scale"])
    assert_close(gqa.gqa_decode(q, k, v, 32, 8, x["scale"], n_splits=6, merge_mode=1), ref2, "bf16 merge kernel")


def test_bf16_partial(gqa):
    x = contig(2, 1, 3000, 16, 4, 64, 2201)
    m, l, op = gqa.gqa_decode_partial(dev(x["q"]), dev(x["k"]), dev(x["v"]), 16, 4, 100, 2000, x["scale"])
    torch.cuda.synchronize()
    rm, rl, ro = oracle.decode_partial(val(x["q"]), val(x["k"]), val(x["v"]), 16, 4, 64, x["scale"], 100, 2000)
    rm, rl, ro = rm.reshape(-1), rl.reshape(-1), ro.reshape(-1, 64)
    m, l, op = m.double().cpu(), l.double().cpu(), op.double().cpu()
    assert ((m - rm).abs() <= 1e-5 * (1 + rm.abs())).all()
    assert ((l - rl).abs() <= 8e-3 * rl).all()
    assert_close(op / l[:, None], oracle.normalize(rl, ro), "bf16 partial O/l")


@pytest.mark.parametrize("hg", [0, 1, 2])
@pytest.mark.parametrize("bs", [16, 32])
def test_bf16_paged(gqa, hg, bs):
    w = gi.custom(12, 1, 3000, 32, 8, 128, 2300 + bs, kind="paged", block_size=bs, partition_size=512,
                  len_lo=1, len_hi=3000, elem="bf16")
    p = gi.make_paged(w, tail_fill="nan")
    o = gqa.gqa_decode_paged(dev(p["q"]).reshape(12, -1), dev(p["k_pool"]), dev(p["v_pool"]), dev(p["block_tables"]),
                             dev(p["seq_lens"]), 32, 8, p["scale"], max_seq_len=p["max_seq_len"], head_group=hg)
    torch.cuda.synchronize()
    assert o.dtype == torch.bfloat16
    pf = gi.make_paged(w)                                   # same draws, finite tails, for the oracle
    ref = oracle.decode_paged(val(pf["q"]), val(pf["k_pool"]), val(pf["v_pool"]), p["block_tables"], p["seq_lens"],
                              32, 8, 128, p["scale"], bs)
    assert_close(o, ref.reshape(12, -1), f"bf16 paged hg={hg} bs={bs}")


def test_bf16_rejects_mixed_dtypes(gqa):
    x = contig(1, 1, 64, 8, 2, 64, 2401)
    q = dev(x["q"])
    k = dev(x["k"]).float().half()
    with pytest.raises(ValueError):
        gqa.gqa_decode(q, k, k, 8, 2)


def test_bf16_public_merge(gqa):
    """gqa_merge writing bfloat16: the fold of fp32 partials, rounded to bf16 (the binding picks
    gqa_merge_ex with the bf16 option from the output's dtype)."""
    x = contig(2, 1, 2000, 8, 2, 128, 3900)
    cuts = [0, 700, 701, 2000]
    parts = [oracle.decode_partial(val(x["q"]), val(x["k"]), val(x["v"]), 8, 2, 128, x["scale"], a, b - a)
             for a, b in zip(cuts[:-1], cuts[1:])]
    m = torch.stack([p[0].reshape(-1).float() for p in parts]).cuda()
    l = torch.stack([p[1].reshape(-1).float() for p in parts]).cuda()
    o = torch.stack([p[2].reshape(-1, 128).float() for p in parts]).cuda()
    out = gqa.gqa_merge(m, l, o, dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert out.dtype == torch.bfloat16
    ref = oracle.decode(val(x["q"]), val(x["k"]), val(x["v"]), 8, 2, 128, x["scale"])
    assert_close(out, ref.reshape(-1, 128), "bf16 merge")
