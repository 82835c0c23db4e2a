"""GPU parity of the tcgen05 kernel (tensor-memory accumulators, M = 128 query rows) against
the CPU float64 oracle, through the C ABI.

The path serves G*T_q up to 128 query rows per KV head (automatically above 64) and can be
forced on smaller units (mma_path=2).  Same tolerance as the f16 parity tests: every element
within 2e-3 + 2e-3 * |o_ref| and relative L2 error below 5e-3 (bf16: 2e-3 + 8e-3 * |o_ref|,
1e-2).  Spiked keys (logits of tens) make rows rescale their accumulators mid-sweep.
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


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def assert_close(got, ref, where, abs_tol=2e-3, rel_tol=2e-3, rel_l2=5e-3):
    got = got.detach().float().double().cpu().reshape(ref.shape)
    ref = ref.double()
    assert torch.isfinite(got).all(), f"{where}: non-finite output"
    mask = ~torch.isnan(ref)                 # heads the oracle did not compute
    got, ref = got[mask], ref[mask]
    err = (got - ref).abs()
    bad = err > abs_tol + rel_tol * ref.abs()
    assert not bad.any(), f"{where}: {int(bad.sum())} of {got.numel()} outside tolerance, max {float(err.max()):.3e}"
    rl2 = float((got - ref).norm() / ref.norm().clamp_min(1e-30))
    assert rl2 <= rel_l2, f"{where}: relative L2 error {rl2:.3e}"


def run(gqa, x, **kw):
    o = gqa.gqa_decode(dev(x["q"]), dev(x["k"]), dev(x["v"]), x["h_q"], x["h_kv"], x["scale"], **kw)
    torch.cuda.synchronize()
    return o


def ref(x, causal=False, units=None, elem="f16"):
    q, k, v = (gi.values(x[n], elem) for n in ("q", "k", "v"))
    return oracle.decode(q, k, v, x["h_q"], x["h_kv"], x["d_head"], x["scale"], units=units, causal=causal)


# (batch, T_q, S_kv, h_q, h_kv, d_head, n_splits, merge_mode): G*T_q from 72 to 128, ragged
# tails, one tile, one key, a single KV head, the merge modes (0 automatic, 1 separate kernel,
# 2 last-arriving CTA)
SHAPES = [
    (1, 16, 5000, 64, 8, 128, 0, 0),
    (1, 16, 5000, 64, 8, 128, 0, 2),
    (2, 12, 3001, 64, 8, 64, 0, 0),
    (1, 9, 777, 8, 1, 128, 1, 0),
    (1, 16, 4097, 64, 8, 128, 7, 1),
    (3, 5, 2000, 16, 1, 128, 3, 0),
    (1, 2, 1, 64, 1, 64, 0, 0),
    (1, 16, 64, 64, 8, 128, 0, 0),
    (1, 16, 65, 64, 8, 128, 1, 0),
    (2, 8, 9000, 128, 8, 64, 5, 0),
    (3, 5, 2000, 16, 1, 128, 3, 2),
    (2, 8, 9000, 128, 8, 64, 5, 2),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_tc_parity(gqa, shape):
    B, T, S, hq, hkv, D, n, mm = shape
    x = gi.make_contiguous(gi.custom(B, T, S, hq, hkv, D, 2000 + S + T, v_dist="uniform",
                                     spike_frac=0.01, spike_mult=8.0))
    o = run(gqa, x, n_splits=n, merge_mode=mm)
    assert_close(o, ref(x), f"tc {shape}")


@pytest.mark.parametrize("rows", [(1, 4, 1), (2, 8, 1), (1, 8, 4), (4, 16, 1), (2, 16, 4)])
def test_tc_forced_on_small_units(gqa, rows):
    """mma_path=2 on units the mma.sync kernel also serves: same result."""
    hkv, G, T = rows
    x = gi.make_contiguous(gi.custom(2, T, 3333, G * hkv, hkv, 128, 2100 + G * T))
    r = ref(x)
    assert_close(run(gqa, x, mma_path=2), r, f"tc forced G={G} T={T}")
    assert_close(run(gqa, x, mma_path=1), r, f"mma.sync G={G} T={T}")


@pytest.mark.parametrize("hq,T", [(20, 1), (33, 1), (16, 3), (8, 6), (64, 1)])
@pytest.mark.parametrize("D", [64, 128])
def test_tc_odd_row_counts(gqa, hq, T, D):
    """Row counts that are not multiples of a warp (20, 33, 48) and that leave warps of a
    warpgroup idle, with a ragged key tail, plain and causal."""
    x = gi.make_contiguous(gi.custom(2, T, 1000 + 7 * hq, hq, 1, D, 2150 + hq * T + D))
    assert_close(run(gqa, x, mma_path=2), ref(x), f"rows hq={hq} T={T} D={D}")
    assert_close(run(gqa, x, mma_path=2, n_splits=3, causal=True), ref(x, causal=True),
                 f"rows causal hq={hq} T={T} D={D}")


def test_tc_forced_on_ragged_workload(gqa):
    x = gi.make("ragged")
    assert_close(run(gqa, x, mma_path=2), ref(x), "ragged on tcgen05")


def test_verify16_workload(gqa):
    # full size, the benchmark's launch configuration; every KV head against the oracle
    x = gi.make("verify16")
    o = run(gqa, x)
    r = ref(x)
    assert not bool(torch.isnan(r).any())
    assert_close(o, r, "verify16 (all 8 KV heads)")


@pytest.mark.parametrize("n_splits", [0, 1, 5])
def test_tc_causal(gqa, n_splits):
    x = gi.make_contiguous(gi.custom(2, 16, 3000, 64, 8, 128, 2200 + n_splits))
    assert_close(run(gqa, x, causal=True, n_splits=n_splits), ref(x, causal=True), f"tc causal {n_splits}")


@pytest.mark.parametrize("rng", [(0, 3000), (100, 1000), (2999, 1), (5, 0)])
@pytest.mark.parametrize("T", [16, 2])
def test_tc_partial(gqa, rng, T):
    """The partial a split emits is the exact-max partial (m = the row max, l and O relative to it),
    with all 128 TMEM lanes holding rows (T = 16) and with only 16 of them (T = 2)."""
    s0, n = rng
    B, hq, hkv, D = 2, 64, 8, 64
    x = gi.make_contiguous(gi.custom(B, T, 3000, hq, hkv, D, 2300, spike_frac=0.01, spike_mult=8.0))
    k, v = x["k"].copy(), x["v"].copy()
    mask = np.ones(3000, dtype=bool)
    mask[s0:s0 + n] = False
    k[:, mask] = np.float16(np.nan)          # keys outside the range must not be read
    v[:, mask] = np.float16(np.nan)
    m, l, op = gqa.gqa_decode_partial(dev(x["q"]), dev(k), dev(v), hq, hkv, s0, n, x["scale"], mma_path=2)
    torch.cuda.synchronize()
    rm, rl, ro = oracle.decode_partial(x["q"], x["k"], x["v"], hq, hkv, D, x["scale"], s0, n)
    rm, rl, ro = rm.reshape(-1), rl.reshape(-1), ro.reshape(-1, D)
    m, l, op = m.double().cpu(), l.double().cpu(), op.double().cpu()
    if n == 0:
        assert torch.isneginf(m).all() and (l == 0).all() and (op == 0).all()
        return
    assert ((m - rm).abs() <= 1e-5 * (1 + rm.abs())).all()
    assert ((l - rl).abs() <= 2e-3 * rl).all()
    assert_close(op / l[:, None], oracle.normalize(rl, ro), f"tc partial {rng}")


@pytest.mark.parametrize("causal", [False, True])
def test_tc_bf16(gqa, causal):
    x = gi.make_contiguous(gi.custom(1, 16, 5000, 64, 8, 128, 2400, elem="bf16", v_dist="uniform",
                                     spike_frac=0.01, spike_mult=8.0))
    o = run(gqa, x, causal=causal)
    assert o.dtype == torch.bfloat16
    assert_close(o, ref(x, causal=causal, elem="bf16"), f"tc bf16 causal={causal}", rel_tol=8e-3, rel_l2=1e-2)


@pytest.mark.parametrize("merge_mode", [0, 2])
def test_tc_timeout_is_reported_not_hung(gqa, merge_mode):
    """A CTA whose producer withholds a tile: every wait of the tcgen05 kernel gives up after
    ~20 ms, the tensor memory is released, the status word says so and the context stays usable
    (splits folded by the merge kernel, or by the unit's last CTA)."""
    x = gi.make_contiguous(gi.custom(1, 16, 8192, 64, 8, 128, 2500))
    q, k, v = dev(x["q"]), dev(x["k"]), dev(x["v"])
    nbytes = gqa.gqa_decode_workspace_size(1, 16, 8192, 64, 8, 128, 4)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    gqa.gqa_decode(q, k, v, 64, 8, x["scale"], n_splits=4, merge_mode=merge_mode, workspace_tensor=ws,
                   timeout_us=20000, test_stall_cta=9)
    assert gqa.gqa_workspace_check(ws) == gqa.GQA_ERR_TIMEOUT
    gqa.gqa_workspace_init(ws)
    o = gqa.gqa_decode(q, k, v, 64, 8, x["scale"], n_splits=4, merge_mode=merge_mode, workspace_tensor=ws)
    assert gqa.gqa_workspace_check(ws) == gqa.GQA_OK
    assert_close(o, ref(x), "after a timeout")


def test_tc_determinism(gqa):
    x = gi.make_contiguous(gi.custom(1, 16, 20000, 64, 8, 128, 2600))
    a = run(gqa, x)
    b = run(gqa, x)
    assert torch.equal(a, b)


def test_plan_query(gqa):
    """gqa_decode_plan reports the kernel path, the split count and the launches of a call."""
    w = gi.WORKLOADS["verify16"]
    n, path, launches = gqa.gqa_decode_plan(w.batch, w.T_q, w.S_kv, w.h_q, w.h_kv, w.d_head)
    assert path == 2 and n > 1 and launches == 2          # tcgen05: the splits fold in the merge kernel
    assert gqa.gqa_decode_plan(w.batch, w.T_q, w.S_kv, w.h_q, w.h_kv, w.d_head, merge_mode=2)[2] == 1
    w = gi.WORKLOADS["ragged"]                          # 32 rows: tcgen05 automatically
    n, path, launches = gqa.gqa_decode_plan(w.batch, w.T_q, w.S_kv, w.h_q, w.h_kv, w.d_head)
    assert path == 2
    # the same split count on the mma.sync kernel, more than a cluster holds: the merge kernel
    assert n > 16 and gqa.gqa_decode_plan(w.batch, w.T_q, w.S_kv, w.h_q, w.h_kv, w.d_head, mma_path=1) == (n, 1, 2)
    w = gi.WORKLOADS["llama8b"]                         # 4 rows: mma.sync, 3 splits folded in a cluster
    n, path, launches = gqa.gqa_decode_plan(w.batch, w.T_q, w.S_kv, w.h_q, w.h_kv, w.d_head)
    assert path == 1 and launches == 1
    assert gqa.gqa_decode_plan(1, 1, 100, 8, 2, 64, n_splits=1) == (1, 1, 1)


@pytest.mark.parametrize("rows", [(4, 4), (8, 2), (16, 4), (16, 1)])
def test_workspace_query_serves_every_path(gqa, rows):
    """gqa_decode_workspace_size (automatic split count) covers both MMA paths and every merge mode:
    the two kernels' occupancies, and so their heuristic split counts, differ."""
    G, T = rows
    hq, hkv = G * 8, 8
    x = gi.make_contiguous(gi.custom(1, T, 3000, hq, hkv, 128, 2300 + G * T))
    nbytes = gqa.gqa_decode_workspace_size(1, T, 3000, hq, hkv, 128, 0)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    r = ref(x)
    for path in (1, 2):
        for mode in (0, 1, 2, 3):
            if mode == 3 and path == 2:
                continue
            o = run(gqa, x, mma_path=path, merge_mode=mode, workspace_tensor=ws)
            assert_close(o, r, f"rows {G * T}, path {path}, merge {mode}")
