"""Decode calls captured in CUDA graphs and run concurrently on several streams.

Serving stacks capture the decode step in a CUDA graph and run independent batches on separate
streams.  A call that launches two kernels (split pass + merge kernel, launched as a
programmatic dependent) must replay correctly from a graph, and calls with separate workspaces
on separate streams must not interfere.  Checked against the CPU float64 oracle with the f16
parity tolerance (|o - o_ref| <= 2e-3 + 2e-3 |o_ref|, relative L2 <= 5e-3).
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


@pytest.mark.parametrize("shape,kw", [((1, 16, 6000, 64, 8, 128), {}),                  # tcgen05 + merge kernel
                                      ((2, 1, 4096, 8, 2, 64), {"n_splits": 64}),       # one-tile splits + merge
                                      ((2, 1, 9000, 32, 8, 128), {}),                   # cluster
                                      ((2, 1, 9000, 32, 8, 128), {"merge_mode": 2})])   # last-CTA fold
def test_graph_replay_contiguous(gqa, shape, kw):
    B, T, S, hq, hkv, D = shape
    x = gi.make_contiguous(gi.custom(B, T, S, hq, hkv, D, 4000 + S))
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    out = torch.empty_like(q)
    ws = torch.zeros(gqa.gqa_decode_workspace_size(B, T, S, hq, hkv, D, kw.get("n_splits", 0)), dtype=torch.uint8,
                     device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        gqa.gqa_decode(q, k, v, hq, hkv, x["scale"], out=out, workspace_tensor=ws, **kw)   # warm-up, outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        gqa.gqa_decode(q, k, v, hq, hkv, x["scale"], out=out, workspace_tensor=ws, **kw)
    ref = oracle.decode(x["q"], x["k"], x["v"], hq, hkv, D, x["scale"])
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_close(out, ref, f"graph replay {shape}")
    # new inputs in the captured buffers: the replay computes on them
    x2 = gi.make_contiguous(gi.custom(B, T, S, hq, hkv, D, 4100 + S))
    q.copy_(cuda(x2["q"])), k.copy_(cuda(x2["k"])), v.copy_(cuda(x2["v"]))
    g.replay()
    torch.cuda.synchronize()
    assert_close(out, oracle.decode(x2["q"], x2["k"], x2["v"], hq, hkv, D, x2["scale"]), "graph replay, new inputs")
    assert gqa.gqa_workspace_check(ws) == gqa.GQA_OK


def test_graph_replay_paged(gqa):
    w = gi.custom(16, 1, 3000, 32, 8, 128, 4200, kind="paged", block_size=16, partition_size=512,
                  len_lo=1, len_hi=3000)
    p = gi.make_paged(w)
    q = cuda(p["q"]).reshape(16, -1)
    kp, vp, tb, ln = cuda(p["k_pool"]), cuda(p["v_pool"]), cuda(p["block_tables"]), cuda(p["seq_lens"])
    out = torch.empty_like(q)
    ws = torch.zeros(gqa.gqa_paged_workspace_size(16, 32, 8, 128, p["max_seq_len"], 512), dtype=torch.uint8,
                     device="cuda")
    s = torch.cuda.Stream()
    call = lambda: gqa.gqa_decode_paged(q, kp, vp, tb, ln, 32, 8, p["scale"], max_seq_len=p["max_seq_len"],
                                        out=out, workspace_tensor=ws)
    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    ref = oracle.decode_paged(p["q"], p["k_pool"], p["v_pool"], p["block_tables"], p["seq_lens"], 32, 8, 128,
                              p["scale"], 16).reshape(16, -1)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_close(out, ref, "paged graph replay")
    assert gqa.gqa_workspace_check(ws) == gqa.GQA_OK


def test_concurrent_streams(gqa):
    """Four calls on four streams at once (different shapes and kernels), each with its own workspace."""
    cases = [(1, 16, 5000, 64, 8, 128), (2, 1, 7000, 32, 8, 128), (1, 4, 3000, 64, 8, 64), (3, 2, 2500, 16, 2, 128)]
    xs, outs, wss, streams = [], [], [], []
    for i, (B, T, S, hq, hkv, D) in enumerate(cases):
        x = gi.make_contiguous(gi.custom(B, T, S, hq, hkv, D, 4300 + i))
        xs.append((x, cuda(x["q"]), cuda(x["k"]), cuda(x["v"])))
        wss.append(torch.zeros(gqa.gqa_decode_workspace_size(B, T, S, hq, hkv, D, 0), dtype=torch.uint8,
                               device="cuda"))
        streams.append(torch.cuda.Stream())
    torch.cuda.synchronize()
    for rep in range(3):
        outs = []
        for (x, q, k, v), ws, s, c in zip(xs, wss, streams, cases):
            with torch.cuda.stream(s):
                outs.append(gqa.gqa_decode(q, k, v, c[3], c[4], x["scale"], workspace_tensor=ws, stream=s))
        torch.cuda.synchronize()
        for (x, _, _, _), o, c in zip(xs, outs, cases):
            assert_close(o, oracle.decode(x["q"], x["k"], x["v"], c[3], c[4], c[5], x["scale"]), f"stream {c} rep {rep}")
    for ws in wss:
        assert gqa.gqa_workspace_check(ws) == gqa.GQA_OK


def test_cached_workspace_on_a_side_stream(gqa):
    """Without a workspace argument the binding keeps one per (device, stream); one created for a
    stream other than the current one is ready (zero-filled) before the call's kernels run there."""
    x = gi.make_contiguous(gi.custom(1, 4, 30000, 64, 8, 128, 4400))
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    ref = oracle.decode(x["q"], x["k"], x["v"], 64, 8, 128, x["scale"])
    for _ in range(2):
        s = torch.cuda.Stream()
        o = gqa.gqa_decode(q, k, v, 64, 8, x["scale"], stream=s)
        s.synchronize()
        assert_close(o, ref, "cached workspace, side stream")


# ---------------------------------------------------------------- programmatic dependent launches
@pytest.mark.parametrize("kw", [{}, {"n_splits": 64, "merge_mode": 1}, {"merge_mode": 3}, {"mma_path": 2},
                                {"mma_path": 1}, {"mma_path": 1, "n_splits": 5, "merge_mode": 2}])
def test_dependent_launch_reads_the_previous_kernels_output(gqa, kw):
    """Every decode kernel may begin while the previous kernel in the stream finishes, and waits
    (griddepcontrol.wait) before it reads global memory.  Chain the library's own kernels -- the merge
    kernel and the decode kernels signal their dependents early -- so that each call's Q is the
    output the previous kernel has just written: gqa_merge -> gqa_decode -> gqa_decode.  A read
    before the wait would see the NaN the buffers were filled with, or stale values."""
    B, T, S, hq, hkv, D = 1, 4, 3000, 32, 8, 64
    x = gi.make_contiguous(gi.custom(B, T, S, hq, hkv, D, 4400))
    k, v = cuda(x["k"]), cuda(x["v"])
    rows = B * T * hq
    parts = [oracle.decode_partial(x["q"], x["k"], x["v"], hq, hkv, D, x["scale"], a, b - a)
             for a, b in [(0, 1000), (1000, 3000)]]
    m = torch.stack([p[0].reshape(-1).float() for p in parts]).cuda()
    l = torch.stack([p[1].reshape(-1).float() for p in parts]).cuda()
    o = torch.stack([p[2].reshape(-1, D).float() for p in parts]).cuda()
    q1 = torch.full((B, T, hq * D), float("nan"), dtype=torch.float16, device="cuda")
    q2 = torch.full_like(q1, float("nan"))
    q3 = torch.full_like(q1, float("nan"))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):   # set-up outside the chain: the stream's cached workspace, first use
        gqa.gqa_decode(q1, k, v, hq, hkv, x["scale"], out=q3, stream=s, **kw)
    torch.cuda.synchronize()
    q3.fill_(float("nan"))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        # a long sleep first, so that the three calls are all queued before the first one runs:
        # each dependent kernel can then launch while its predecessor is still at work
        torch.cuda._sleep(20_000_000)
        gqa.gqa_merge(m, l, o, out=q1.view(rows, D), stream=s)
        gqa.gqa_decode(q1, k, v, hq, hkv, x["scale"], out=q2, stream=s, **kw)
        gqa.gqa_decode(q2, k, v, hq, hkv, x["scale"], out=q3, stream=s, **kw)
    torch.cuda.synchronize()
    # each stage against the oracle applied to the previous stage's (device-computed) values
    r1 = oracle.decode(x["q"], x["k"], x["v"], hq, hkv, D, x["scale"])
    assert_close(q1, r1, "merge output")
    a1 = q1.cpu().numpy()
    r2 = oracle.decode(a1, x["k"], x["v"], hq, hkv, D, x["scale"])
    assert_close(q2, r2, f"decode of the merge output {kw}")
    r3 = oracle.decode(q2.cpu().numpy(), x["k"], x["v"], hq, hkv, D, x["scale"])
    assert_close(q3, r3, f"decode of the decode output {kw}")


@pytest.mark.parametrize("shape", ["deep", (1, 4, 20000, 64, 8, 128), (8, 1, 4096, 32, 8, 128)])
def test_keys_written_by_the_previous_kernel(gqa, shape):
    """The split and tcgen05 kernels prefetch their first K/V boxes into L2 before their dependency
    wait, while the previous kernel may still run.  Here that kernel (gqa_merge, which signals its
    dependents at its start) writes the very K buffer the decode reads, over NaN: the decode must
    see the written keys.  Shapes: the deep-ring split kernel, the tcgen05 kernel, the cluster."""
    if shape == "deep":
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        if sms % 8 or sms // 8 <= 16:
            pytest.skip("no deep-ring grid for 8 units on this GPU")
        shape = (1, 1, (sms // 8) * 48 * 64 + 37, 32, 8, 128)
    B, T, S, hq, hkv, D = shape
    x = gi.make_contiguous(gi.custom(B, T, S, hq, hkv, D, 4500 + S))
    ref = oracle.decode(x["q"], x["k"], x["v"], hq, hkv, D, x["scale"])
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    R = B * S * hkv
    # one partial per row with m = 0, l = 1: the merge writes O = the keys (f16 -> f32 -> f16 exact)
    m = torch.zeros(1, R, device="cuda")
    l = torch.ones(1, R, device="cuda")
    op = k.float().reshape(1, R, D)
    kbuf = torch.empty_like(k)
    out = torch.empty_like(q)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):   # set-up outside the chain: the stream's cached workspace, first use
        gqa.gqa_decode(q, k, v, hq, hkv, x["scale"], out=out, stream=s)
    torch.cuda.synchronize()
    for it in range(3):
        with torch.cuda.stream(s):
            kbuf.fill_(float("nan"))
            out.fill_(float("nan"))
            torch.cuda._sleep(5_000_000)   # queue both calls before the merge runs
            gqa.gqa_merge(m, l, op, out=kbuf.view(R, D), stream=s)
            gqa.gqa_decode(q, kbuf, v, hq, hkv, x["scale"], out=out, stream=s)
        torch.cuda.synchronize()
        assert torch.equal(kbuf, k), "merge output"
        assert_close(out, ref, f"decode of keys written just before it, {shape}, pass {it}")
