"""GPU parity: the CUDA library (through its C ABI) against the CPU float64 oracle.

Tolerance (stated for f16 output with fp32 accumulation): every element must
satisfy |o - o_ref| <= 2e-3 + 2e-3 * |o_ref|; in addition the relative L2 error
||o - o_ref|| / ||o_ref|| must stay below 5e-3, because at long context the
outputs shrink toward the absolute term (|O| ~ sqrt(e / S_kv)) and the
element-wise bound alone would accept a zero output.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import gqa_inputs as gi
import oracle

pytestmark = pytest.mark.gpu

ABS_TOL = 2e-3
REL_TOL = 2e-3
REL_L2 = 5e-3


@pytest.fixture(scope="module")
def gqa():
    from decode_attention_03_gb300 import build
    build.build()
    import decode_attention_03_gb300._binding as b
    assert torch.cuda.is_available()
    return b


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_close(got, ref, where, rel_l2=REL_L2):
    got = got.detach().double().cpu().reshape(ref.shape)
    ref = ref.double()
    mask = ~torch.isnan(ref)
    assert mask.any(), where
    g, r = got[mask], ref[mask]
    assert torch.isfinite(g).all(), f"{where}: non-finite output"
    err = (g - r).abs()
    bad = err > ABS_TOL + REL_TOL * r.abs()
    assert not bad.any(), f"{where}: {int(bad.sum())} of {g.numel()} outside tolerance, max err {float(err.max()):.3e}"
    rl2 = float((g - r).norm() / r.norm().clamp_min(1e-30))
    assert rl2 <= rel_l2, f"{where}: relative L2 error {rl2:.3e}"
    return float(err.max()), rl2


def run_contig(gqa, x, **kw):
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    o = gqa.gqa_decode(q, k, v, x["h_q"], x["h_kv"], x["scale"], **kw)
    torch.cuda.synchronize()
    return o


def ref_contig(x, units=None):
    return oracle.decode(x["q"], x["k"], x["v"], x["h_q"], x["h_kv"], x["d_head"], x["scale"], units=units)


# ---------------------------------------------------------------- the five workloads
def test_workload_tiny(gqa):
    x = gi.make("tiny")
    ref = ref_contig(x)
    for kw in [{}, {"n_splits": 1}, {"n_splits": 2}, {"n_splits": 16}, {"n_splits": 64},
               {"n_splits": 16, "merge_mode": 1}]:
        assert_close(run_contig(gqa, x, **kw), ref, f"tiny {kw}")


def test_workload_llama8b(gqa):
    x = gi.make("llama8b")
    ref = ref_contig(x)
    assert_close(run_contig(gqa, x), ref, "llama8b")


def test_workload_long(gqa):
    # full size, the launch configuration the benchmark times; every KV head against the oracle
    x = gi.make("long")
    o = run_contig(gqa, x)
    assert torch.isfinite(o.float()).all()
    ref = ref_contig(x)
    assert not bool(torch.isnan(ref).any())
    assert_close(o, ref, "long (all 8 KV heads)")


def test_workload_ragged(gqa):
    x = gi.make("ragged")
    ref = ref_contig(x)
    # spiked keys drive logits to tens: the online rescale and the masked tail tile are exercised
    assert_close(run_contig(gqa, x), ref, "ragged")
    assert_close(run_contig(gqa, x, n_splits=1), ref, "ragged, one split")
    assert_close(run_contig(gqa, x, mma_path=1), ref, "ragged on the mma.sync kernel")


def run_paged(gqa, p, **kw):
    o = gqa.gqa_decode_paged(cuda(p["q"]).reshape(p["q"].shape[0], -1), cuda(p["k_pool"]), cuda(p["v_pool"]),
                             cuda(p["block_tables"]), cuda(p["seq_lens"]), p["h_q"], p["h_kv"], p["scale"],
                             max_seq_len=p["max_seq_len"], partition_size=p["partition_size"], **kw)
    torch.cuda.synchronize()
    return o


def ref_paged(p, seqs=None):
    return oracle.decode_paged(p["q"], p["k_pool"], p["v_pool"], p["block_tables"], p["seq_lens"], p["h_q"],
                               p["h_kv"], p["d_head"], p["scale"], p["block_size"], seqs=seqs)


_PAGED_REF = {}


@pytest.mark.parametrize("hg", [0, 1, 2])
def test_workload_paged(gqa, hg):
    w = gi.WORKLOADS["paged"]
    p = gi.make_paged(w)
    o = run_paged(gqa, p, head_group=hg)
    if "paged" not in _PAGED_REF:                            # every one of the 64 sequences
        _PAGED_REF["paged"] = ref_paged(p)
    ref = _PAGED_REF["paged"]
    assert not bool(torch.isnan(ref).any())
    assert_close(o, ref.reshape(64, -1), f"paged (all sequences, head group {hg})")
    # unused tail slots of every last block filled with NaN: identical output, bit for bit
    pn = gi.make_paged(w, tail_fill="nan")
    o2 = run_paged(gqa, pn, head_group=hg)
    assert torch.equal(o, o2)


# ---------------------------------------------------------------- splits, shapes, edges
@pytest.mark.parametrize("n_splits", [1, 2, 7, 37, 79])
@pytest.mark.parametrize("merge_mode", [0, 1, 2])
def test_split_sweep(gqa, n_splits, merge_mode):
    # automatic (a cluster up to 16 splits, else the merge kernel), the merge kernel, the last CTA's fold
    x = gi.make_contiguous(gi.custom(2, 1, 5000, 8, 2, 128, 101))
    ref = ref_contig(x)
    assert_close(run_contig(gqa, x, n_splits=n_splits, merge_mode=merge_mode), ref,
                 f"splits={n_splits} mode={merge_mode}")


@pytest.mark.parametrize("S", [1, 2, 63, 64, 65, 511, 513, 4097])
@pytest.mark.parametrize("D", [64, 128])
def test_ragged_lengths(gqa, S, D):
    x = gi.make_contiguous(gi.custom(2, 1, S, 8, 2, D, 200 + S))
    ref = ref_contig(x)
    assert_close(run_contig(gqa, x), ref, f"S={S} D={D}")
    if S >= 2:
        assert_close(run_contig(gqa, x, n_splits=2), ref, f"S={S} D={D} 2 splits")


@pytest.mark.parametrize("hq,hkv,T", [(8, 8, 1), (32, 8, 1), (24, 2, 1), (16, 2, 2), (32, 4, 3), (64, 8, 4),
                                      (64, 4, 3), (64, 2, 2), (16, 16, 4)])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("path", [1, 2])
def test_row_classes(gqa, hq, hkv, T, D, path):
    # every row class of the mma.sync kernel (path 1) and the same units on the tcgen05 kernel
    x = gi.make_contiguous(gi.custom(2, T, 777, hq, hkv, D, 300 + hq + T))
    ref = ref_contig(x)
    assert_close(run_contig(gqa, x, mma_path=path), ref, f"hq={hq} hkv={hkv} T={T} D={D} path={path}")
    assert_close(run_contig(gqa, x, n_splits=3, mma_path=path), ref, f"hq={hq} hkv={hkv} T={T} D={D} 3 splits")
    if path == 1:   # the last CTA's fold, which the automatic choice leaves to explicit requests
        assert_close(run_contig(gqa, x, n_splits=3, merge_mode=2, mma_path=1), ref,
                     f"hq={hq} hkv={hkv} T={T} D={D} 3 splits, last-CTA fold")


def test_constant_scores_and_shift(gqa):
    # K = 0: every output row is the mean of V; large logit shifts (|logit| ~ 60) change nothing
    x = gi.make_contiguous(gi.custom(1, 2, 3000, 16, 4, 128, 401))
    x0 = dict(x)
    x0["k"] = np.zeros_like(x["k"])
    ref0 = ref_contig(x0)
    assert_close(run_contig(gqa, x0), ref0, "K = 0")
    xs = dict(x)
    k = x["k"].astype(np.float32) * 6.0
    xs["k"] = k.astype(np.float16)
    assert_close(run_contig(gqa, xs), ref_contig(xs), "logits ~ +-60")


def test_determinism(gqa):
    x = gi.make_contiguous(gi.custom(2, 1, 20000, 32, 8, 128, 501))
    a = run_contig(gqa, x)
    b = run_contig(gqa, x)
    assert torch.equal(a, b)


# ---------------------------------------------------------------- partial / merge calls
@pytest.mark.parametrize("rng", [(0, 3000), (100, 1000), (2999, 1), (64, 128), (5, 0)])
def test_partial_matches_oracle(gqa, rng):
    s0, n = rng
    x = gi.make_contiguous(gi.custom(2, 2, 3000, 16, 4, 64, 601))
    B, T, hq, D = 2, 2, 16, 64
    # keys outside the range are NaN: the partial must not see them
    k = x["k"].copy()
    v = x["v"].copy()
    mask = np.ones(3000, dtype=bool)
    mask[s0:s0 + n] = False
    k[:, mask] = np.float16(np.nan)
    v[:, mask] = np.float16(np.nan)
    m, l, op = gqa.gqa_decode_partial(cuda(x["q"]), cuda(k), cuda(v), hq, 4, s0, n, x["scale"])
    torch.cuda.synchronize()
    rm, rl, ro = oracle.decode_partial(x["q"], x["k"], x["v"], hq, 4, D, x["scale"], s0, n)
    rm, rl, ro = rm.reshape(-1), rl.reshape(-1), ro.reshape(-1, D)
    m, l, op = m.double().cpu(), l.double().cpu(), op.double().cpu()
    if n == 0:
        assert torch.isneginf(m).all() and (l == 0).all() and (op == 0).all()
        return
    assert ((m - rm).abs() <= 1e-5 * (1 + rm.abs())).all()
    assert ((l - rl).abs() <= 2e-3 * rl).all()
    assert_close(op / l[:, None], oracle.normalize(rl, ro), f"partial {rng} O/l")


def test_merge_api(gqa):
    x = gi.make_contiguous(gi.custom(2, 1, 2000, 8, 2, 128, 701))
    D = 128
    cuts = [0, 1, 300, 301, 1500, 2000]
    parts = [oracle.decode_partial(x["q"], x["k"], x["v"], 8, 2, D, x["scale"], a, b - a)
             for a, b in zip(cuts[:-1], cuts[1:])]
    # plus one empty partial
    parts.append(oracle.decode_partial(x["q"], x["k"], x["v"], 8, 2, D, x["scale"], 7, 0))
    ms = torch.stack([p[0].reshape(-1) for p in parts]).float()
    ls = torch.stack([p[1].reshape(-1) for p in parts]).float()
    os_ = torch.stack([p[2].reshape(-1, D) for p in parts]).float()
    o = gqa.gqa_merge(ms.cuda(), ls.cuda(), os_.cuda())
    mo, lo, oo = gqa.gqa_merge_partial(ms.cuda(), ls.cuda(), os_.cuda())
    torch.cuda.synchronize()
    full = ref_contig(x).reshape(-1, D)
    assert_close(o, full, "gqa_merge")
    assert_close(oo.cpu().double() / lo.cpu().double()[:, None], full, "gqa_merge_partial")
    # all-empty rows give zeros
    e = gqa.gqa_merge(torch.full((2, 3), float("-inf")).cuda(), torch.zeros(2, 3).cuda(),
                      torch.zeros(2, 3, 64).cuda())
    torch.cuda.synchronize()
    assert (e.float() == 0).all()


def test_chain_reduce_equals_full(gqa):
    """The page's reduce-to-root: 4 ranks each hold an S_kv slice, partials are merged hop by
    hop toward the root (merge_partial) and normalised at the root (merge)."""
    x = gi.make_contiguous(gi.custom(1, 1, 8192, 32, 8, 128, 801))
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    parts = [gqa.gqa_decode_partial(q, k, v, 32, 8, r * 2048, 2048, x["scale"]) for r in range(4)]
    m, l, o = parts[3]
    for r in (2, 1):
        m, l, o = gqa.gqa_merge_partial(torch.stack([parts[r][0], m]), torch.stack([parts[r][1], l]),
                                        torch.stack([parts[r][2], o]))
    out = gqa.gqa_merge(torch.stack([parts[0][0], m]), torch.stack([parts[0][1], l]),
                        torch.stack([parts[0][2], o]))
    torch.cuda.synchronize()
    assert_close(out, ref_contig(x).reshape(-1, 128), "chain reduce")


# ---------------------------------------------------------------- paged edges
@pytest.mark.parametrize("bs,part", [(16, 512), (8, 64), (32, 128), (64, 512), (16, 64)])
@pytest.mark.parametrize("hq,hkv,hg,D", [(8, 2, 1, 128), (8, 2, 2, 128), (32, 8, 4, 128), (16, 4, 4, 64),
                                         (32, 8, 2, 64), (64, 4, 1, 128)])
def test_paged_edges(gqa, bs, part, hq, hkv, hg, D):
    lens = np.array([0, 1, 15, 16, 17, 511, 512, 513, 1000, 64], dtype=np.int32)
    N = len(lens)
    nblk = (lens + bs - 1) // bs
    num_blocks = int(nblk.sum()) + 3
    perm = np.random.Generator(np.random.PCG64(bs + part)).permutation(num_blocks).astype(np.int32)
    maxb = int(nblk.max())
    tab = np.full((N, maxb), -1, dtype=np.int32)
    off = 0
    for b in range(N):
        tab[b, :nblk[b]] = perm[off:off + nblk[b]]
        off += nblk[b]
    q = gi.normal_f16(900 + bs, 0, (N, 1, hq * D))
    kp = gi.normal_f16(900 + bs, 1, (num_blocks, bs, hkv * D))
    vp = gi.normal_f16(900 + bs, 2, (num_blocks, bs, hkv * D))
    p = dict(q=q, k_pool=kp, v_pool=vp, block_tables=tab, seq_lens=lens, num_seqs=N, h_q=hq, h_kv=hkv,
             d_head=D, scale=1 / math.sqrt(D), block_size=bs, partition_size=part, max_seq_len=int(lens.max()))
    o = run_paged(gqa, p, head_group=hg)
    ref = ref_paged(p)
    assert bool((ref[0] == 0).all())                         # the oracle's empty sequence: exact zeros
    assert (o[0].float() == 0).all()                         # and the kernel's
    assert_close(o, ref.reshape(N, -1), f"paged bs={bs} part={part} hq={hq} hkv={hkv} hg={hg} D={D}")


def test_paged_bad_block_is_reported(gqa):
    lens = np.array([100, 40], dtype=np.int32)
    tab = np.array([[0, 1, 2, 3, 4, 5, 6], [7, 8, 99, -1, -1, -1, -1]], dtype=np.int32)   # 99 >= num_blocks
    hq, hkv, D, bs = 8, 2, 64, 16
    q = gi.normal_f16(1, 0, (2, hq * D))
    kp = gi.normal_f16(1, 1, (10, bs, hkv * D))
    vp = gi.normal_f16(1, 2, (10, bs, hkv * D))
    ws = torch.zeros(gqa.gqa_paged_workspace_size(2, hq, hkv, D, 100, 512), dtype=torch.uint8, device="cuda")
    o = gqa.gqa_decode_paged(cuda(q), cuda(kp), cuda(vp), cuda(tab), cuda(lens), hq, hkv, max_seq_len=100,
                             workspace_tensor=ws)
    assert gqa.gqa_workspace_check(ws) == gqa.GQA_ERR_INVALID_ARG
    # sequence 0 is unaffected
    p = dict(q=q[:1], k_pool=kp, v_pool=vp, block_tables=tab[:1], seq_lens=lens[:1], h_q=hq, h_kv=hkv, d_head=D,
             scale=1 / 8, block_size=bs)
    ref = ref_paged(p)
    assert_close(o[:1], ref.reshape(1, -1), "paged seq 0 next to a bad table")
    assert gqa.gqa_workspace_check(ws) == gqa.GQA_OK


def test_timeout_is_reported_not_hung(gqa):
    """A CTA whose producer withholds a tile: its bounded waits give up after ~20 ms and the
    status word says so; the context stays usable (the last-CTA fold; the cluster variant and the
    merge kernel have their own such tests)."""
    x = gi.make_contiguous(gi.custom(1, 1, 8192, 8, 2, 128, 1001))
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    nbytes = gqa.gqa_decode_workspace_size(1, 1, 8192, 8, 2, 128, 4)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    gqa.gqa_decode(q, k, v, 8, 2, x["scale"], n_splits=4, merge_mode=2, workspace_tensor=ws, timeout_us=20000,
                   test_stall_cta=1)
    assert gqa.gqa_workspace_check(ws) == gqa.GQA_ERR_TIMEOUT
    gqa.gqa_workspace_init(ws)
    o = gqa.gqa_decode(q, k, v, 8, 2, x["scale"], n_splits=4, merge_mode=2, workspace_tensor=ws)
    assert gqa.gqa_workspace_check(ws) == gqa.GQA_OK
    assert_close(o, ref_contig(x), "after a timeout")


def test_paged_repeated_calls_reset_the_queue(gqa):
    """The persistent paged kernel's item queue is reset by its last CTA: back-to-back
    calls on one workspace give identical results."""
    w = gi.custom(16, 1, 5000, 32, 8, 128, 1101, kind="paged", block_size=16, partition_size=512,
                  len_lo=1, len_hi=5000)
    p = gi.make_paged(w)
    ws = torch.zeros(gqa.gqa_paged_workspace_size(16, 32, 8, 128, p["max_seq_len"], 512), dtype=torch.uint8,
                     device="cuda")
    outs = [run_paged(gqa, p, workspace_tensor=ws) for _ in range(3)]
    assert gqa.gqa_workspace_check(ws) == gqa.GQA_OK
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    assert_close(outs[2], ref_paged(p).reshape(16, -1), "paged, third call")


def test_paged_timeout_is_reported_not_hung(gqa):
    w = gi.custom(8, 1, 4000, 16, 4, 128, 1201, kind="paged", block_size=16, partition_size=512,
                  len_lo=2000, len_hi=4000)
    p = gi.make_paged(w)
    ws = torch.zeros(gqa.gqa_paged_workspace_size(8, 16, 4, 128, p["max_seq_len"], 512), dtype=torch.uint8,
                     device="cuda")
    run_paged(gqa, p, workspace_tensor=ws, timeout_us=20000, test_stall_cta=0)
    assert gqa.gqa_workspace_check(ws) == gqa.GQA_ERR_TIMEOUT
    gqa.gqa_workspace_init(ws)
    o = run_paged(gqa, p, workspace_tensor=ws)
    assert gqa.gqa_workspace_check(ws) == gqa.GQA_OK
    assert_close(o, ref_paged(p).reshape(8, -1), "paged after a timeout")


# ---------------------------------------------------------------- causal tail (speculative verify)
@pytest.mark.parametrize("hq,hkv,T,S,D", [(32, 8, 4, 5000, 128), (64, 8, 4, 20000, 128), (16, 16, 3, 777, 64),
                                          (8, 2, 2, 64, 128), (32, 4, 8, 3000, 128), (16, 2, 4, 5, 64)])
@pytest.mark.parametrize("n_splits", [0, 1, 7])
@pytest.mark.parametrize("path", [1, 2])
def test_causal_tail(gqa, hq, hkv, T, S, D, n_splits, path):
    x = gi.make_contiguous(gi.custom(2, T, S, hq, hkv, D, 1300 + S + T))
    ref = oracle.decode(x["q"], x["k"], x["v"], hq, hkv, D, x["scale"], causal=True)
    o = run_contig(gqa, x, causal=True, n_splits=n_splits, mma_path=path)
    assert_close(o, ref, f"causal hq={hq} hkv={hkv} T={T} S={S} D={D} splits={n_splits} path={path}")


def test_causal_partial_with_empty_rows(gqa):
    """A key range past some tokens' causal limit: those rows get the empty partial."""
    T, S, hq, hkv, D = 4, 600, 16, 4, 128
    x = gi.make_contiguous(gi.custom(1, T, S, hq, hkv, D, 1401))
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    for s0, n in [(S - 3, 3), (0, S), (100, 400), (S - 1, 1)]:
        m, l, op = gqa.gqa_decode_partial(q, k, v, hq, hkv, s0, n, x["scale"], causal=True)
        torch.cuda.synchronize()
        rm, rl, ro = oracle.decode_partial(x["q"], x["k"], x["v"], hq, hkv, D, x["scale"], s0, n, causal=True)
        rm, rl, ro = rm.reshape(-1), rl.reshape(-1), ro.reshape(-1, D)
        m, l, op = m.double().cpu(), l.double().cpu(), op.double().cpu()
        empty = torch.isneginf(rm)
        assert torch.equal(torch.isneginf(m), empty)
        assert (l[empty] == 0).all() and (op[empty] == 0).all()
        keep = ~empty
        assert ((m[keep] - rm[keep]).abs() <= 1e-5 * (1 + rm[keep].abs())).all()
        assert ((l[keep] - rl[keep]).abs() <= 2e-3 * rl[keep]).all()
        assert_close(op[keep] / l[keep][:, None], oracle.normalize(rl[keep], ro[keep]), f"causal partial {s0},{n}")


@pytest.mark.parametrize("path", [1, 2])
def test_merge_kernel_path(gqa, path):
    """The separate merge kernel after either decode kernel: parity on repeated calls with the
    counters left at 0, and a withheld tile reported (the workspace then re-initialised)."""
    x = gi.make_contiguous(gi.custom(3, 2, 3000, 16, 4, 128, 1101))
    ref = ref_contig(x)
    units = 3 * 4
    nbytes = gqa.gqa_decode_workspace_size(3, 2, 3000, 16, 4, 128, 6)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        o = run_contig(gqa, x, n_splits=6, merge_mode=1, mma_path=path, workspace_tensor=ws)
        assert_close(o, ref, f"merge kernel, path {path}")
        assert gqa.gqa_workspace_check(ws) == gqa.GQA_OK
        assert bool((ws[256:256 + 4 * units] == 0).all())          # counters back to 0
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    gqa.gqa_decode(q, k, v, 16, 4, x["scale"], n_splits=6, merge_mode=1, mma_path=path, workspace_tensor=ws,
                   timeout_us=20000, test_stall_cta=5)
    assert gqa.gqa_workspace_check(ws) == gqa.GQA_ERR_TIMEOUT
    gqa.gqa_workspace_init(ws)
    assert_close(run_contig(gqa, x, n_splits=6, merge_mode=1, mma_path=path, workspace_tensor=ws), ref,
                 "after a timeout")
    assert gqa.gqa_workspace_check(ws) == gqa.GQA_OK


@pytest.mark.parametrize("bs,part", [(16, 512), (8, 64), (64, 1024)])
def test_paged_matches_contiguous_on_gathered_kv(gqa, bs, part):
    """Paged decode over a shuffled pool equals contiguous decode over the same keys gathered into
    (sequences, keys, h_kv*d) -- two different kernels -- and both match the oracle."""
    N, L, hq, hkv, D = 3, 3000, 32, 8, 128
    nb = (L + bs - 1) // bs
    num_blocks = N * nb + 5
    perm = np.random.Generator(np.random.PCG64(bs + part)).permutation(num_blocks).astype(np.int32)
    tab = perm[:N * nb].reshape(N, nb).copy()
    q = gi.normal_f16(6100 + bs, 0, (N, 1, hq * D))
    kp = gi.normal_f16(6100 + bs, 1, (num_blocks, bs, hkv * D))
    vp = gi.normal_f16(6100 + bs, 2, (num_blocks, bs, hkv * D))
    lens = np.full(N, L, dtype=np.int32)
    j = np.arange(L)
    kc = np.stack([kp[tab[b, j // bs], j % bs] for b in range(N)])       # (N, L, h_kv*D), gathered
    vc = np.stack([vp[tab[b, j // bs], j % bs] for b in range(N)])
    scale = 1 / math.sqrt(D)
    op = gqa.gqa_decode_paged(cuda(q).reshape(N, -1), cuda(kp), cuda(vp), cuda(tab), cuda(lens), hq, hkv, scale,
                              max_seq_len=L, partition_size=part)
    oc = gqa.gqa_decode(cuda(q), cuda(kc), cuda(vc), hq, hkv, scale)
    torch.cuda.synchronize()
    ref = oracle.decode(q, kc, vc, hq, hkv, D, scale)
    assert_close(op, ref.reshape(N, -1), f"paged bs={bs} part={part}")
    assert_close(oc, ref, "contiguous on the gathered keys")
    d = (op.double().cpu().reshape(-1) - oc.double().cpu().reshape(-1)).abs()
    assert float(d.max()) <= 2e-3, f"paged vs contiguous: {float(d.max()):.3e}"
