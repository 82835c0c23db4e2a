"""Batch-size edges, against the CPU float64 oracle on sampled sequences.

* paged decode with more than 1024 sequences runs as consecutive launches of at most 1024
  sequences sharing one workspace (each launch's partition pass and merge pass);
* contiguous decode with far more (sequence, KV head) units than SMs takes one split per unit
  (no partials), with the grid's z extent in the thousands.
Tolerance as in the f16 parity tests: |o - o_ref| <= 2e-3 + 2e-3 |o_ref|, relative L2 <= 5e-3.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gqa_inputs as gi
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gqa():
    from decode_attention_03_gb300 import build
    build.build()
    import decode_attention_03_gb300._binding as b
    assert torch.cuda.is_available()
    return b


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_close(got, ref, where):
    got = got.detach().double().cpu().reshape(ref.shape)
    mask = ~torch.isnan(ref)
    g, r = got[mask], ref[mask].double()
    assert torch.isfinite(g).all(), where
    err = (g - r).abs()
    assert not (err > 2e-3 + 2e-3 * r.abs()).any(), f"{where}: max err {float(err.max()):.3e}"
    assert float((g - r).norm() / r.norm()) <= 5e-3, where


@pytest.mark.parametrize("layout", ["rows", "vllm"])
def test_paged_more_than_1024_sequences(gqa, layout):
    N = 2300
    w = gi.custom(N, 1, 1200, 16, 4, 64, 5000, kind="paged", block_size=16, partition_size=512,
                  len_lo=1, len_hi=1200, layout=layout)
    p = gi.make_paged(w)
    fn = gqa.gqa_decode_paged_vllm if layout == "vllm" else gqa.gqa_decode_paged
    part, hg, launches = gqa.gqa_paged_plan(N, 16, 4, 64, p["max_seq_len"], 512, vllm_layout=layout == "vllm")
    assert launches == 6                                  # 3 launches of <= 1024 sequences, 2 passes each
    o = fn(cuda(p["q"]).reshape(N, -1), cuda(p["k_pool"]), cuda(p["v_pool"]), cuda(p["block_tables"]),
           cuda(p["seq_lens"]), 16, 4, p["scale"], max_seq_len=p["max_seq_len"], partition_size=512)
    torch.cuda.synchronize()
    lens = p["seq_lens"]
    seqs = sorted(set([0, 1, 1023, 1024, 1025, 2047, 2048, N - 1, int(np.argmax(lens)), int(np.argmin(lens))]))
    ref = oracle.decode_paged(p["q"], p["k_pool"], p["v_pool"], p["block_tables"], lens, 16, 4, 64, p["scale"], 16,
                              seqs=seqs, layout=layout).reshape(N, -1)
    assert_close(o, ref, f"{N} sequences ({layout})")


def test_contiguous_many_units(gqa):
    B, T, S, hq, hkv, D = 3000, 1, 200, 8, 8, 64            # 24000 units, one split each
    n, path, launches = gqa.gqa_decode_plan(B, T, S, hq, hkv, D)
    assert n == 1 and launches == 1
    x = gi.make_contiguous(gi.custom(B, T, S, hq, hkv, D, 5100))
    o = gqa.gqa_decode(cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), hq, hkv, x["scale"])
    torch.cuda.synchronize()
    units = [(b, g) for b in (0, 1, 1499, 2998, 2999) for g in (0, 7)]
    ref = oracle.decode(x["q"], x["k"], x["v"], hq, hkv, D, x["scale"], units=units)
    assert_close(o, ref, "3000 sequences")
