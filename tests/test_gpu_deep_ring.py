"""The split kernel's deep-ring variant: one CTA per SM with a ring of four 32 KB stages, which the
automatic plan takes for single-sequence decode at d_head 128 with up to 8 query rows per KV head
where the (sequence, KV head) units divide the SMs into more splits than a cluster holds, each of at
least 48 64-key tiles (the long workload: 8 KV heads, 152 SMs -> 19 splits).  Every call goes
through the C ABI and is checked against the CPU float64 oracle at the parity tolerance."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gqa_inputs as gi
import oracle
from test_gpu_bf16 import assert_close as assert_close_bf16
from test_gpu_parity import assert_close, cuda, ref_contig, run_contig

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gqa():
    from decode_attention_03_gb300 import build
    build.build()
    import decode_attention_03_gb300._binding as b
    assert torch.cuda.is_available()
    return b


def _deep_splits(units):
    """Splits the deep-ring variant gives `units` units on this GPU (None where it does not apply)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return sms // units if sms % units == 0 and sms // units > 16 else None


def _long_enough(units):
    # keys for at least 48 tiles per split, plus a ragged tail
    n = _deep_splits(units)
    return None if n is None else n * 48 * 64 + 37


def test_plan_takes_the_deep_ring_where_it_applies(gqa):
    n = _deep_splits(8)
    if n is None:
        pytest.skip("the SM count does not divide into more than 16 splits per unit for 8 units")
    # the long workload's shape: one CTA per SM, the merge kernel after it
    assert gqa.gqa_decode_plan(1, 1, 1 << 20, 32, 8, 128) == (n, 1, 2)
    assert gqa.gqa_decode_plan(1, 2, 1 << 20, 32, 8, 128) == (n, 1, 2)        # 8 rows
    # not with the causal tail, a forced split count or merge mode, d_head 64, 16 rows, or short splits
    h = gqa.gqa_decode_plan(1, 2, 1 << 20, 32, 8, 128, causal=True)[0]
    assert h != n
    assert gqa.gqa_decode_plan(1, 1, 1 << 20, 32, 8, 128, n_splits=24)[0] == 24
    assert gqa.gqa_decode_plan(1, 1, 1 << 20, 32, 8, 128, merge_mode=1)[0] != n
    assert gqa.gqa_decode_plan(1, 1, 1 << 20, 32, 8, 64)[0] != n
    assert gqa.gqa_decode_plan(1, 1, n * 27 * 64, 32, 8, 128)[0] != n
    assert gqa.gqa_decode_plan(1, 1, _long_enough(8), 32, 8, 128)[0] == n


@pytest.mark.parametrize("hq,T", [(32, 1), (32, 2), (64, 1), (8, 1)])
def test_deep_ring_parity(gqa, hq, T):
    S = _long_enough(8)
    if S is None:
        pytest.skip("no deep-ring grid for 8 units on this GPU")
    x = gi.make_contiguous(gi.custom(1, T, S, hq, 8, 128, 8800 + hq + T))
    assert gqa.gqa_decode_plan(1, T, S, hq, 8, 128)[0] == _deep_splits(8)
    assert_close(run_contig(gqa, x), ref_contig(x), f"deep ring hq={hq} T={T}")


def test_deep_ring_one_unit_and_bf16(gqa):
    S = _long_enough(1)
    if S is None:
        pytest.skip("no deep-ring grid for one unit on this GPU")
    x = gi.make_contiguous(gi.custom(1, 1, S, 4, 1, 128, 8900, elem="bf16"))
    vals = {c: gi.values(x[c], "bf16") for c in ("q", "k", "v")}
    ref = oracle.decode(vals["q"], vals["k"], vals["v"], 4, 1, 128, x["scale"])
    q, k, v = (torch.from_numpy(np.ascontiguousarray(x[c]).view(np.int16)).cuda().view(torch.bfloat16)
               for c in ("q", "k", "v"))
    assert gqa.gqa_decode_plan(1, 1, S, 4, 1, 128)[0] == _deep_splits(1)
    o = gqa.gqa_decode(q, k, v, 4, 1, x["scale"])
    torch.cuda.synchronize()
    assert_close_bf16(o, ref, "deep ring, one unit, bf16")


def test_deep_ring_partial(gqa):
    S = _long_enough(8)
    if S is None:
        pytest.skip("no deep-ring grid for 8 units on this GPU")
    x = gi.make_contiguous(gi.custom(1, 1, S + 5000, 32, 8, 128, 9000))
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    m, l, op = gqa.gqa_decode_partial(q, k, v, 32, 8, 3000, S, x["scale"])
    torch.cuda.synchronize()
    rm, rl, ro = oracle.decode_partial(x["q"], x["k"], x["v"], 32, 8, 128, x["scale"], 3000, S)
    rl, ro = rl.reshape(-1), ro.reshape(-1, 128)
    assert_close(op.double().cpu() / l.double().cpu()[:, None], oracle.normalize(rl, ro), "deep ring partial")


def test_deep_ring_timeout_is_reported_not_hung(gqa):
    S = _long_enough(8)
    if S is None:
        pytest.skip("no deep-ring grid for 8 units on this GPU")
    x = gi.make_contiguous(gi.custom(1, 1, S, 32, 8, 128, 9100))
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    ws = torch.zeros(gqa.gqa_decode_workspace_size(1, 1, S, 32, 8, 128, 0), dtype=torch.uint8, device="cuda")
    gqa.gqa_decode(q, k, v, 32, 8, x["scale"], workspace_tensor=ws, timeout_us=20000, test_stall_cta=3 + 8 * 5)
    assert gqa.gqa_workspace_check(ws) == gqa.GQA_ERR_TIMEOUT
    gqa.gqa_workspace_init(ws)
    o = gqa.gqa_decode(q, k, v, 32, 8, x["scale"], workspace_tensor=ws)
    assert gqa.gqa_workspace_check(ws) == gqa.GQA_OK
    assert_close(o, ref_contig(x), "deep ring after a timeout")


@pytest.mark.parametrize("seed", range(6))
def test_deep_ring_random_shapes(gqa, seed):
    """Seeded random shapes the deep ring serves: (sequences, KV heads) giving 1, 2, 4 or 8 units,
    G * T_q up to 8 rows, f16 or bf16, a ragged number of keys of at least 48 tiles per split."""
    rng = np.random.default_rng(7300 + seed)
    B, hkv = [(1, 1), (2, 1), (1, 2), (1, 4), (2, 2), (4, 2), (8, 1), (2, 4)][rng.integers(8)]
    n = _deep_splits(B * hkv)
    if n is None:
        pytest.skip("no deep-ring grid for these units on this GPU")
    G, T = [(1, 1), (2, 1), (4, 1), (8, 1), (2, 2), (4, 2), (1, 8)][rng.integers(7)]
    S = n * 64 * int(rng.integers(48, 56)) + int(rng.integers(0, 64))
    elem = "bf16" if rng.integers(2) else "f16"
    x = gi.make_contiguous(gi.custom(B, T, S, G * hkv, hkv, 128, 7400 + seed, elem=elem))
    assert gqa.gqa_decode_plan(B, T, S, G * hkv, hkv, 128)[0] == n
    where = f"deep ring B={B} h_kv={hkv} G={G} T={T} S={S} {elem}"
    if elem == "f16":
        assert_close(run_contig(gqa, x), ref_contig(x), where)
    else:
        vals = {c: gi.values(x[c], "bf16") for c in ("q", "k", "v")}
        ref = oracle.decode(vals["q"], vals["k"], vals["v"], G * hkv, hkv, 128, x["scale"])
        q, k, v = (torch.from_numpy(np.ascontiguousarray(x[c]).view(np.int16)).cuda().view(torch.bfloat16)
                   for c in ("q", "k", "v"))
        o = gqa.gqa_decode(q, k, v, G * hkv, hkv, x["scale"])
        torch.cuda.synchronize()
        assert_close_bf16(o, ref, where)


def test_plan_names_the_kernel_and_fold_of_each_workload(gqa):
    """gqa_decode_plan_ex: the kernel variant and fold the automatic plan picks for the workloads."""
    def plan(name, **kw):
        w = gi.WORKLOADS[name]
        return gqa.gqa_decode_plan(w.batch, w.T_q, w.S_kv, w.h_q, w.h_kv, w.d_head, detail=True, **kw)
    assert plan("tiny")["kernel"] == "split-cluster" and plan("tiny")["fold"] == "cluster"
    assert plan("llama8b")["kernel"] == "split-cluster" and plan("llama8b")["fold"] == "cluster"
    for name in ("ragged", "verify16"):
        assert plan(name)["kernel"] == "tcgen05" and plan(name)["fold"] == "merge-kernel"
    long = plan("long")
    assert long["fold"] == "merge-kernel"
    assert long["kernel"] == ("split-deep-ring" if _deep_splits(8) else "split")
    assert plan("long", merge_mode=2)["fold"] == "last-cta" and plan("long", merge_mode=2)["kernel"] == "split"
    assert plan("long", n_splits=1)["fold"] == "none"
