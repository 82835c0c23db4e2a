"""Seeded random configurations of every compute entry point against the CPU float64 oracle.

Each case draws its shape and options from a fixed seed (the same cases on every run), across
the whole supported space: batch, query tokens T_q, KV heads, group size G (G*T_q up to 128
rows), d_head 64 / 128, key counts from 1 to a few thousand, the split count and merge mode,
the kernel (mma.sync, tcgen05, automatic), the split kernel's cluster variant (merge mode 3),
the causal tail, float16 / bfloat16, partial key ranges, and for paged calls both cache layouts, block sizes 8-64, partitions of 64 keys up to
single pass, head groups, empty sequences and NaN in the unused tail slots.  Every output
element is checked: |o - o_ref| <= 2e-3 + 2e-3 |o_ref| and the relative L2 error <= 5e-3.

bfloat16: P enters the P.V product rounded to bfloat16 (unit roundoff u = 2^-9) while l sums
the unrounded p, so an output element can be off by up to u * A, A = sum_j p_j |v_j| / l (the
softmax-weighted mean of |V|), before its own rounding (u |o|).  With one or two visible keys
and values of opposite sign this exceeds any bound relative to |o| alone; the bfloat16 bound
is 2e-3 + 8e-3 |o_ref| + 4e-3 A (2u per term of A), and the L2 check divides by
|| max(|o_ref|, A) ||.
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


def assert_close(got, ref, where, elem, aref=None):
    """aref (bfloat16 only): the oracle's output with |V| in place of V, the A of the bound."""
    got = got.detach().float().double().cpu().reshape(ref.shape)
    ref = ref.double()
    assert torch.isfinite(got).all(), f"{where}: non-finite output"
    err = (got - ref).abs()
    if elem == "f16":
        tol, scale, rl2_tol = 2e-3 + 2e-3 * ref.abs(), ref, 5e-3
    else:
        a = aref.double().reshape(ref.shape)
        tol, scale, rl2_tol = 2e-3 + 8e-3 * ref.abs() + 4e-3 * a, torch.maximum(ref.abs(), a), 1e-2
    bad = err > tol
    assert not bad.any(), f"{where}: {int(bad.sum())} of {got.numel()} outside tolerance, max {float(err.max()):.3e}"
    rl2 = float((got - ref).norm() / scale.norm().clamp_min(1e-30))
    assert rl2 <= rl2_tol or float(scale.norm()) == 0.0, f"{where}: relative L2 error {rl2:.3e}"


def _contig_cases(n, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    cases = []
    while len(cases) < n:
        D = int(rng.choice([64, 128]))
        h_kv = int(rng.choice([1, 2, 4, 8]))
        G = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
        T = int(rng.choice([1, 1, 2, 3, 4, 8, 16]))
        if G * T > 128:
            continue
        path = int(rng.choice([0, 1, 2]))
        if path == 1 and G * T > 64:
            path = 2            # the mma.sync kernel holds at most 64 rows
        S = int(np.exp(rng.uniform(0, np.log(6000))))
        S = max(S, 1)
        B = int(rng.choice([1, 1, 2, 3]))
        causal = bool(T > 1 and rng.random() < 0.4)
        partial = bool(rng.random() < 0.25)
        s0 = int(rng.integers(0, S)) if partial else 0
        sl = int(rng.integers(0, S - s0 + 1)) if partial else S
        cases.append(dict(B=B, T=T, S=S, h_q=G * h_kv, h_kv=h_kv, D=D, path=path,
                          n_splits=int(rng.choice([0, 0, 1, 2, 5, 19, 40])),
                          merge_mode=int(rng.choice([0, 1, 2])), causal=causal,
                          elem=str(rng.choice(["f16", "bf16"])), partial=partial, s0=s0, sl=sl,
                          seed=int(rng.integers(10_000, 20_000))))
    return cases


CONTIG = _contig_cases(300, 4242)


def _cluster_cases(n, seed):
    """The split kernel's cluster variant (merge_mode 3): up to 64 rows per KV head, split counts
    up to 40 (capped at 16 by the call), the automatic or the mma.sync path."""
    rng = np.random.Generator(np.random.PCG64(seed))
    cases = []
    while len(cases) < n:
        D = int(rng.choice([64, 128]))
        h_kv = int(rng.choice([1, 2, 4, 8]))
        G = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
        T = int(rng.choice([1, 1, 2, 3, 4]))
        if G * T > 64:
            continue
        S = max(int(np.exp(rng.uniform(0, np.log(9000)))), 1)
        partial = bool(rng.random() < 0.25)
        s0 = int(rng.integers(0, S)) if partial else 0
        sl = int(rng.integers(0, S - s0 + 1)) if partial else S
        cases.append(dict(B=int(rng.choice([1, 2, 3])), T=T, S=S, h_q=G * h_kv, h_kv=h_kv, D=D,
                          path=int(rng.choice([0, 1])), n_splits=int(rng.choice([0, 2, 3, 7, 16, 40])),
                          merge_mode=3, causal=bool(T > 1 and rng.random() < 0.4),
                          elem=str(rng.choice(["f16", "bf16"])), partial=partial, s0=s0, sl=sl,
                          seed=int(rng.integers(30_000, 40_000))))
    return cases


CLUSTER = _cluster_cases(100, 4545)


@pytest.mark.parametrize("c", CONTIG + CLUSTER,
                         ids=[f"c{i:02d}" for i in range(len(CONTIG))] + [f"k{i:02d}" for i in range(len(CLUSTER))])
def test_fuzz_contiguous(gqa, c):
    w = gi.custom(c["B"], c["T"], c["S"], c["h_q"], c["h_kv"], c["D"], c["seed"], elem=c["elem"],
                  spike_frac=0.02, spike_mult=6.0)
    x = gi.make_contiguous(w)
    q, k, v = (gi.values(x[n], c["elem"]) for n in ("q", "k", "v"))
    kw = dict(n_splits=c["n_splits"], merge_mode=c["merge_mode"], causal=c["causal"], mma_path=c["path"])
    where = str(c)
    if not c["partial"]:
        o = gqa.gqa_decode(dev(x["q"]), dev(x["k"]), dev(x["v"]), c["h_q"], c["h_kv"], x["scale"], **kw)
        torch.cuda.synchronize()
        ref = oracle.decode(q, k, v, c["h_q"], c["h_kv"], c["D"], x["scale"], causal=c["causal"])
        aref = oracle.decode(q, k, np.abs(v), c["h_q"], c["h_kv"], c["D"], x["scale"], causal=c["causal"])
        assert_close(o, ref, where, c["elem"], aref)
        return
    m, l, op = gqa.gqa_decode_partial(dev(x["q"]), dev(x["k"]), dev(x["v"]), c["h_q"], c["h_kv"], c["s0"],
                                      c["sl"], x["scale"], **kw)
    torch.cuda.synchronize()
    rm, rl, ro = oracle.decode_partial(q, k, v, c["h_q"], c["h_kv"], c["D"], x["scale"], c["s0"], c["sl"],
                                       causal=c["causal"])
    _, _, ra = oracle.decode_partial(q, k, np.abs(v), c["h_q"], c["h_kv"], c["D"], x["scale"], c["s0"], c["sl"],
                                     causal=c["causal"])
    rm, rl, ro, ra = rm.reshape(-1), rl.reshape(-1), ro.reshape(-1, c["D"]), ra.reshape(-1, c["D"])
    m, l, op = m.double().cpu(), l.double().cpu(), op.double().cpu()
    empty = rl == 0
    assert torch.equal(torch.isneginf(m), empty), f"{where}: empty rows"
    assert (l[empty] == 0).all() and (op[empty] == 0).all(), f"{where}: empty rows"
    keep = ~empty
    if keep.any():
        assert ((m[keep] - rm[keep]).abs() <= 1e-5 * (1 + rm[keep].abs())).all(), f"{where}: m"
        assert ((l[keep] - rl[keep]).abs() <= 4e-3 * rl[keep]).all(), f"{where}: l"
        assert_close(op[keep] / l[keep][:, None], oracle.normalize(rl[keep], ro[keep]), where + " O/l", c["elem"],
                     oracle.normalize(rl[keep], ra[keep]))


def _paged_workload(c):
    return gi.custom(c["N"], 1, c["len_hi"], c["h_q"], c["h_kv"], c["D"], c["seed"], kind="paged",
                     block_size=c["bs"], partition_size=c["part"], len_lo=0, len_hi=c["len_hi"],
                     layout=c["layout"], elem=c["elem"])


def _paged_cases(n, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    cases = []
    while len(cases) < n:
        D = int(rng.choice([64, 128]))
        h_kv = int(rng.choice([1, 2, 4, 8]))
        G = int(rng.choice([1, 2, 4, 6, 8, 16, 32]))
        bs = int(rng.choice([8, 16, 32, 64]))
        layout = str(rng.choice(["rows", "vllm"]))
        N = int(rng.integers(1, 41))
        hi = int(np.exp(rng.uniform(np.log(2), np.log(5000))))
        hg_max = 4 if layout == "rows" else min(4, 64 // bs)
        hg = int(rng.choice([0, 0, 1, 2, 4]))
        if hg and (hg > hg_max or h_kv % hg or (hg > 1 and G > 16)):
            hg = 0
        part = int(rng.choice([0, 64, 128, 512, 1024, 8192]))
        if part and part // min(bs, 16) > 1024:
            part = 0
        c = dict(N=N, h_q=G * h_kv, h_kv=h_kv, D=D, bs=bs, layout=layout, len_hi=hi, hg=hg, part=part,
                 elem=str(rng.choice(["f16", "bf16"])), seed=int(rng.integers(20_000, 30_000)))
        if gi.paged_layout(_paged_workload(c))[2] == 0:
            continue            # every sequence empty: no pool to address
        cases.append(c)
    return cases


PAGED = _paged_cases(150, 4343)


@pytest.mark.parametrize("c", PAGED, ids=[f"p{i:02d}" for i in range(len(PAGED))])
def test_fuzz_paged(gqa, c):
    p = gi.make_paged(_paged_workload(c), tail_fill="nan")
    N = c["N"]
    fn = gqa.gqa_decode_paged_vllm if c["layout"] == "vllm" else gqa.gqa_decode_paged
    o = fn(dev(p["q"]).reshape(N, -1), dev(p["k_pool"]), dev(p["v_pool"]), dev(p["block_tables"]),
           dev(p["seq_lens"]), c["h_q"], c["h_kv"], p["scale"], max_seq_len=max(p["max_seq_len"], 1),
           partition_size=c["part"], head_group=c["hg"])
    torch.cuda.synchronize()
    q, kc, vc = (gi.values(p[n], c["elem"]) for n in ("q", "k_pool", "v_pool"))
    args = (p["block_tables"], p["seq_lens"], c["h_q"], c["h_kv"], c["D"], p["scale"], c["bs"])
    ref = oracle.decode_paged(q, kc, vc, *args, layout=c["layout"]).reshape(N, -1)
    aref = oracle.decode_paged(q, kc, np.abs(vc), *args, layout=c["layout"]).reshape(N, -1)
    assert_close(o, ref, str(c), c["elem"], aref)
