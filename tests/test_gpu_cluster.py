"""The split kernel's cluster variant (merge_mode 3): the splits of a (sequence, KV head) unit run as
one thread-block cluster and fold their partials -- the page's _merge_running over the splits in
order, then O / l (page "kernbench2 ... _gqa_attention_decode_long.py") -- through distributed
shared memory, in one launch.  Checked against the CPU float64 oracle at the parity tolerance."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gqa_inputs as gi
import oracle
from test_gpu_parity import assert_close, cuda, ref_contig, run_contig

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gqa():
    from decode_attention_03_gb300 import build
    build.build()
    import decode_attention_03_gb300._binding as b
    assert torch.cuda.is_available()
    return b


@pytest.mark.parametrize("n_splits", [2, 3, 4, 8, 11, 16])
def test_cluster_tiny(gqa, n_splits):
    x = gi.make("tiny")
    ref = ref_contig(x)
    assert gqa.gqa_decode_plan(1, 1, 4096, 8, 2, 64, n_splits=n_splits, merge_mode=3) == (n_splits, 1, 1)
    assert_close(run_contig(gqa, x, n_splits=n_splits, merge_mode=3), ref, f"tiny, cluster of {n_splits}")


def test_cluster_caps_at_sixteen(gqa):
    x = gi.make("tiny")
    assert gqa.gqa_decode_plan(1, 1, 4096, 8, 2, 64, n_splits=64, merge_mode=3) == (16, 1, 1)
    assert gqa.gqa_decode_plan(1, 1, 4096, 8, 2, 64, merge_mode=3)[0] <= 16
    assert_close(run_contig(gqa, x, n_splits=64, merge_mode=3), ref_contig(x), "tiny, 64 splits capped")
    assert_close(run_contig(gqa, x, merge_mode=3), ref_contig(x), "tiny, heuristic splits capped")


@pytest.mark.parametrize("shape", [
    (2, 1, 5000, 32, 8, 128),     # 4 rows per unit, d 128
    (1, 2, 3001, 16, 2, 64),      # 16 rows (two n-tiles)
    (1, 4, 2999, 32, 4, 128),     # 32 rows (two warp columns)
    (1, 8, 1500, 64, 8, 64),      # 64 rows (four warp columns)
    (1, 8, 2500, 64, 8, 128),     # 64 rows at d_head 128 (the cluster variant's shorter ring)
    (3, 1, 65, 8, 2, 64),         # two tiles, ragged
    (1, 1, 1, 8, 1, 128),         # one key
])
@pytest.mark.parametrize("n_splits", [2, 7, 16])
def test_cluster_shapes(gqa, shape, n_splits):
    B, T_q, S, hq, hkv, D = shape
    x = gi.make_contiguous(gi.custom(B, T_q, S, hq, hkv, D, 7300 + S + n_splits))
    assert_close(run_contig(gqa, x, n_splits=n_splits, merge_mode=3, mma_path=1), ref_contig(x),
                 f"cluster {shape} splits {n_splits}")


@pytest.mark.parametrize("n_splits", [2, 5, 16])
def test_cluster_causal(gqa, n_splits):
    x = gi.make_contiguous(gi.custom(2, 4, 3000, 32, 4, 128, 7400 + n_splits))
    ref = oracle.decode(x["q"], x["k"], x["v"], 32, 4, 128, x["scale"], causal=True)
    assert_close(run_contig(gqa, x, n_splits=n_splits, merge_mode=3, causal=True), ref, f"causal {n_splits}")


def test_cluster_bf16(gqa):
    x = gi.make_contiguous(gi.custom(2, 1, 4096, 16, 4, 64, 7500, elem="bf16"))
    q, k, v = (torch.from_numpy(x[n].view(np.int16)).view(torch.bfloat16).cuda() for n in ("q", "k", "v"))
    o = gqa.gqa_decode(q, k, v, 16, 4, x["scale"], n_splits=12, merge_mode=3)
    torch.cuda.synchronize()
    assert o.dtype == torch.bfloat16
    vals = {n: gi.values(x[n], "bf16") for n in ("q", "k", "v")}
    ref = oracle.decode(vals["q"], vals["k"], vals["v"], 16, 4, 64, x["scale"])
    got = o.double().cpu().reshape(ref.shape)
    assert bool(((got - ref).abs() <= 2e-3 + 8e-3 * ref.abs()).all())
    assert float((got - ref).norm() / ref.norm()) <= 1e-2


@pytest.mark.parametrize("rng", [(0, 3000), (100, 1000), (2999, 1), (64, 128)])
def test_cluster_partial(gqa, rng):
    s0, n = rng
    x = gi.make_contiguous(gi.custom(2, 2, 3000, 16, 4, 64, 7600))
    m, l, op = gqa.gqa_decode_partial(cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), 16, 4, s0, n, x["scale"],
                                      n_splits=8, merge_mode=3)
    torch.cuda.synchronize()
    rm, rl, ro = oracle.decode_partial(x["q"], x["k"], x["v"], 16, 4, 64, x["scale"], s0, n)
    rm, rl, ro = rm.reshape(-1), rl.reshape(-1), ro.reshape(-1, 64)
    m, l, op = m.double().cpu(), l.double().cpu(), op.double().cpu()
    assert ((m - rm).abs() <= 1e-5 * (1 + rm.abs())).all()
    assert ((l - rl).abs() <= 2e-3 * rl).all()
    assert_close(op / l[:, None], oracle.normalize(rl, ro), f"cluster partial {rng}")


def test_cluster_is_deterministic(gqa):
    x = gi.make_contiguous(gi.custom(1, 1, 60000, 32, 8, 128, 7700))
    a = run_contig(gqa, x, n_splits=16, merge_mode=3)
    b = run_contig(gqa, x, n_splits=16, merge_mode=3)
    assert torch.equal(a, b)


def test_cluster_timeout_is_reported_not_hung(gqa):
    """One CTA of a cluster withholds a tile: its waits give up, it still pushes its completion
    flag and joins the cluster barrier, the cluster writes nothing for that unit, the status word says timeout, and the
    next call succeeds."""
    x = gi.make_contiguous(gi.custom(1, 1, 8192, 8, 2, 128, 7800))
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    nbytes = gqa.gqa_decode_workspace_size(1, 1, 8192, 8, 2, 128, 8)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.zeros_like(q)
    gqa.gqa_decode(q, k, v, 8, 2, x["scale"], out=out, n_splits=8, merge_mode=3, workspace_tensor=ws,
                   timeout_us=20000, test_stall_cta=0 + 2 * 3)     # KV head 0, split 3 (x + X*y)
    assert gqa.gqa_workspace_check(ws) == gqa.GQA_ERR_TIMEOUT
    o = out.double().cpu()
    assert bool((o[..., :4 * 128] == 0).all())        # the stalled unit (KV head 0) wrote nothing
    gqa.gqa_workspace_init(ws)
    o2 = gqa.gqa_decode(q, k, v, 8, 2, x["scale"], n_splits=8, merge_mode=3, workspace_tensor=ws)
    assert gqa.gqa_workspace_check(ws) == gqa.GQA_OK
    assert_close(o2, ref_contig(x), "after a timeout")


def test_cluster_not_on_tcgen05(gqa):
    x = gi.make_contiguous(gi.custom(1, 16, 1000, 64, 8, 64, 7900))      # 128 rows: tcgen05 only
    with pytest.raises(gqa.GQAError) as e:
        run_contig(gqa, x, merge_mode=3)
    assert e.value.status == gqa.GQA_ERR_UNSUPPORTED
    y = gi.make_contiguous(gi.custom(1, 4, 1000, 32, 4, 64, 7901))       # 32 rows: either kernel
    with pytest.raises(gqa.GQAError):
        run_contig(gqa, y, merge_mode=3, mma_path=2)
    assert gqa.gqa_decode_plan(1, 4, 1000, 32, 4, 64, merge_mode=3)[1] == 1   # automatic: mma.sync
    assert_close(run_contig(gqa, y, merge_mode=3), ref_contig(y), "32 rows, cluster, automatic path")


def test_automatic_choice_takes_the_cluster_for_short_sweeps(gqa):
    # tiny workload: 64 one-tile splits would need the merge kernel; one cluster of 16 instead
    assert gqa.gqa_decode_plan(1, 1, 4096, 8, 2, 64) == (16, 1, 1)
    assert gqa.gqa_decode_plan(1, 1, 2048, 8, 2, 64) == (16, 1, 1)
    assert gqa.gqa_decode_plan(1, 1, 8192, 8, 2, 64) == (16, 1, 1)
    # a longer sweep keeps the heuristic's splits (and its bandwidth)
    n, path, launches = gqa.gqa_decode_plan(1, 1, 65536, 8, 2, 64)
    assert n > 16 and launches == 2
    # many units, 3 splits each: one cluster per unit (one launch)
    assert gqa.gqa_decode_plan(8, 1, 32768, 32, 8, 128) == (3, 1, 1)


def test_automatic_choice_between_cluster_and_merge_kernel(gqa):
    """merge_mode 0 on the mma.sync kernel: 2 to 16 splits fold in a cluster (one launch), more in the
    merge kernel (two); at d_head 128 with 64 rows, where the cluster variant's receiving area costs a
    ring stage, the merge kernel too.  Each choice matches the oracle."""
    for n, launches in [(2, 1), (5, 1), (16, 1), (17, 2), (24, 2)]:   # 2 units: their clusters fit at once
        assert gqa.gqa_decode_plan(1, 1, 20000, 8, 2, 128, n_splits=n) == (n, 1, launches)
    assert gqa.gqa_decode_plan(1, 1, 20000, 32, 8, 64, n_splits=7) == (7, 1, 1)
    assert gqa.gqa_decode_plan(1, 16, 20000, 32, 8, 128, n_splits=3, mma_path=1) == (3, 1, 2)   # 64 rows
    assert gqa.gqa_decode_plan(1, 16, 20000, 32, 8, 64, n_splits=3, mma_path=1) == (3, 1, 1)
    # only while every unit's cluster is resident at once: at d_head 64 with 64 rows the variant
    # holds one CTA per SM, so 64 units of 2-CTA clusters fit in one wave and 160 do not
    assert gqa.gqa_decode_plan(8, 16, 4096, 32, 8, 64, n_splits=2, mma_path=1) == (2, 1, 1)
    assert gqa.gqa_decode_plan(20, 16, 4096, 32, 8, 64, n_splits=2, mma_path=1) == (2, 1, 2)
    for (T, D, n) in [(1, 128, 5), (1, 128, 24), (16, 128, 3), (16, 64, 3), (2, 64, 11)]:
        y = gi.make_contiguous(gi.custom(2, T, 3000, 32, 8, D, 7900 + T + D + n))
        assert_close(run_contig(gqa, y, n_splits=n, mma_path=1), ref_contig(y), f"automatic T={T} D={D} n={n}")
