"""GPU parity of paged decode over vLLM's cache layout (key cache [blocks, h_kv, D/8, block, 8],
value cache [blocks, h_kv, D, block]), read in place, against the CPU float64 oracle, which
gathers the keys and values from the same caches by its own indexing.

Also: the partition plan (automatic v2 with 512-token partitions; the page's single-pass v1 as a
partition covering whole sequences), agreement with the
row-layout path on the same values (identical arithmetic, so identical bits), NaN in the unused
tail slots, bfloat16, bad block ids and the bounded waits.  Same tolerance as the f16 parity
tests: |o - o_ref| <= 2e-3 + 2e-3 |o_ref| and relative L2 error <= 5e-3 (bf16: 8e-3, 1e-2).
"""
from __future__ import annotations

import math

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


def assert_close(got, ref, where, rel_tol=2e-3, rel_l2=5e-3):
    got = got.detach().float().double().cpu().reshape(ref.shape)
    ref = ref.double()
    mask = ~torch.isnan(ref)
    g, r = got[mask], ref[mask]
    assert torch.isfinite(g).all(), f"{where}: non-finite output"
    err = (g - r).abs()
    bad = err > 2e-3 + rel_tol * r.abs()
    assert not bad.any(), f"{where}: {int(bad.sum())} of {g.numel()} outside tolerance, max {float(err.max()):.3e}"
    rl2 = float((g - r).norm() / r.norm().clamp_min(1e-30))
    assert rl2 <= rel_l2, f"{where}: relative L2 error {rl2:.3e}"


def run(gqa, p, **kw):
    N = p["q"].shape[0]
    o = gqa.gqa_decode_paged_vllm(dev(p["q"]).reshape(N, -1), dev(p["k_pool"]), dev(p["v_pool"]),
                                  dev(p["block_tables"]), dev(p["seq_lens"]), p["h_q"], p["h_kv"], p["scale"],
                                  max_seq_len=p["max_seq_len"], **kw)
    torch.cuda.synchronize()
    return o


def ref(p, seqs=None):
    e = p.get("elem", "f16")
    q, kc, vc = (gi.values(p[n], e) for n in ("q", "k_pool", "v_pool"))
    N = p["q"].shape[0]
    return oracle.decode_paged(q, kc, vc, p["block_tables"], p["seq_lens"], p["h_q"], p["h_kv"], p["d_head"],
                               p["scale"], p["block_size"], seqs=seqs, layout="vllm").reshape(N, -1)


def edge_case(bs, hq, hkv, D, seed, elem="f16", lens=None):
    """Sequences of 0, 1, block +- 1, partition +- 1 ... keys (or `lens`); NaN in every unused
    tail slot."""
    if lens is None:
        lens = np.array([0, 1, 15, 16, 17, 511, 512, 513, 1000, 64, 2049], dtype=np.int32)
    N = len(lens)
    nblk = (lens + bs - 1) // bs
    num_blocks = int(nblk.sum()) + 3
    perm = np.random.Generator(np.random.PCG64(seed)).permutation(num_blocks).astype(np.int32)
    tab = np.full((N, int(nblk.max())), -1, dtype=np.int32)
    off = 0
    for b in range(N):
        tab[b, :nblk[b]] = perm[off:off + nblk[b]]
        off += nblk[b]
    q = gi.normal_f16(seed, 0, (N, 1, hq * D), elem)
    kp = gi.normal_f16(seed, 1, (num_blocks, bs, hkv * D), elem)
    vp = gi.normal_f16(seed, 2, (num_blocks, bs, hkv * D), elem)
    nan = np.float16(np.nan) if elem == "f16" else np.uint16(0x7FC0)
    for b in range(N):
        L = int(lens[b])
        if L % bs:
            kp[tab[b, L // bs], L % bs:] = nan
            vp[tab[b, L // bs], L % bs:] = nan
    kc, vc = gi.to_vllm_layout(kp, vp, hkv, D)
    return dict(q=q, k_pool=kc, v_pool=vc, block_tables=tab, seq_lens=lens, h_q=hq, h_kv=hkv, d_head=D,
                scale=1 / math.sqrt(D), block_size=bs, max_seq_len=int(lens.max()), elem=elem,
                rows=(kp, vp))


@pytest.mark.parametrize("bs,part", [(16, 512), (8, 64), (32, 128), (64, 512), (16, 0), (8, 2112)])
@pytest.mark.parametrize("hq,hkv,hg,D", [(8, 2, 1, 128), (8, 2, 2, 128), (32, 8, 4, 128), (16, 4, 4, 64),
                                         (32, 8, 2, 64), (64, 4, 1, 128)])
def test_vllm_edges(gqa, bs, part, hq, hkv, hg, D):
    p = edge_case(bs, hq, hkv, D, 3000 + bs + part + hq + D)
    if hg > 64 // bs:
        # a TMA box holds whole blocks: a work item spans at most 64 / block_size KV heads
        with pytest.raises(gqa.GQAError):
            run(gqa, p, partition_size=part, head_group=hg)
        hg = 0
    o = run(gqa, p, partition_size=part, head_group=hg)
    r = ref(p)
    assert bool((r[0] == 0).all())                           # the oracle's empty sequence: exact zeros
    assert (o[0].float() == 0).all()                         # and the kernel's
    assert_close(o, r, f"vllm bs={bs} part={part} hq={hq} hkv={hkv} hg={hg} D={D}")


@pytest.mark.parametrize("bs", [8, 16, 64])
def test_vllm_matches_row_layout_bitwise(gqa, bs):
    """The same values in the two layouts go through the same arithmetic."""
    p = edge_case(bs, 32, 8, 128, 3100 + bs)
    kp, vp = p["rows"]
    N = p["q"].shape[0]
    hg = min(4, 64 // bs)            # the same work items in both (the vLLM layout caps the head group)
    o_rows = gqa.gqa_decode_paged(dev(p["q"]).reshape(N, -1), dev(kp), dev(vp), dev(p["block_tables"]),
                                  dev(p["seq_lens"]), 32, 8, p["scale"], max_seq_len=p["max_seq_len"],
                                  partition_size=512, head_group=hg)
    o_vllm = run(gqa, p, partition_size=512, head_group=hg)
    assert torch.equal(o_rows, o_vllm)


def test_partition_plan(gqa):
    """Automatic: v2 with 512-token partitions (partition pass + merge pass); a partition of at
    least max_seq_len is the single-pass v1 (one launch)."""
    part, hg, launches = gqa.gqa_paged_plan(384, 32, 8, 128, 2048, 0, vllm_layout=True)
    assert part == 512 and hg == 4 and launches == 2
    part, hg, launches = gqa.gqa_paged_plan(384, 32, 8, 128, 2048, 2048, vllm_layout=True)
    assert part == 2048 and launches == 1
    assert gqa.gqa_paged_plan(384, 32, 8, 128, 500, 0, vllm_layout=True)[2] == 1   # one partition anyway
    assert gqa.gqa_paged_plan(2000, 32, 8, 128, 2048, 0)[2] == 4                   # two launches of <= 1024 seqs
    # whole blocks per box: at most 64 / block_size heads per item over the vLLM layout
    assert gqa.gqa_paged_plan(64, 32, 8, 128, 16384, 0, block_size=32, vllm_layout=True)[1] == 2
    assert gqa.gqa_paged_plan(64, 32, 8, 128, 16384, 0, block_size=64, vllm_layout=True)[1] == 1
    assert gqa.gqa_paged_plan(64, 32, 8, 128, 16384, 0, block_size=64)[1] == 4


def test_v1_workload(gqa):
    """The paged_v1 workload (384 sequences of at most 2048 keys): single pass (partition 2048)
    and the automatic 512-token partitions, every sequence."""
    p = gi.make("paged_v1")
    r = ref(p)
    assert not bool(torch.isnan(r).any())
    assert_close(run(gqa, p, partition_size=2048), r, "paged_v1, single pass")
    assert_close(run(gqa, p), r, "paged_v1, 512-token partitions")


def test_single_pass_takes_every_sequence_once(gqa):
    """A single-pass launch hands its sequences out longest first (a counting sort in every CTA):
    300 sequences whose lengths repeat (ties), include 0, 1 and the partition itself, and span
    every length class; every output row is checked, on both cache layouts."""
    rng = np.random.Generator(np.random.PCG64(3500))
    lens = np.concatenate([np.array([0, 1, 2048, 2048, 2047, 0, 32, 33, 31, 1024] * 6),
                           rng.integers(1, 2049, 240)]).astype(np.int32)
    rng.shuffle(lens)
    p = edge_case(16, 8, 2, 64, 3501, lens=lens)
    assert gqa.gqa_paged_plan(len(lens), 8, 2, 64, 2048, 2048, block_size=16, vllm_layout=True)[2] == 1
    r = ref(p)
    assert_close(run(gqa, p, partition_size=2048), r, "single pass, vLLM caches")
    kp, vp = p["rows"]
    N = len(lens)
    o = gqa.gqa_decode_paged(dev(p["q"]).reshape(N, -1), dev(kp), dev(vp), dev(p["block_tables"]),
                             dev(p["seq_lens"]), 8, 2, p["scale"], max_seq_len=2048, partition_size=2048)
    torch.cuda.synchronize()
    assert_close(o, r, "single pass, row pools")


def test_vllm_workload(gqa):
    # full size, the benchmark's launch configuration; every sequence against the oracle
    p = gi.make("paged_vllm")
    o = run(gqa, p)
    r = ref(p)
    assert not bool(torch.isnan(r).any())
    assert_close(o, r, "paged_vllm (all 64 sequences)")


@pytest.mark.parametrize("bs,part", [(16, 0), (32, 512)])
def test_vllm_bf16(gqa, bs, part):
    p = edge_case(bs, 32, 8, 128, 3200 + bs, elem="bf16")
    o = run(gqa, p, partition_size=part)
    assert o.dtype == torch.bfloat16
    r = ref(p)
    assert bool((r[0] == 0).all())                  # the oracle's empty sequence: exact zeros
    assert_close(o, r, f"vllm bf16 bs={bs}", rel_tol=8e-3, rel_l2=1e-2)


def test_vllm_bad_block_is_reported(gqa):
    hq, hkv, D, bs = 8, 2, 64, 16
    lens = np.array([100, 40], dtype=np.int32)
    tab = np.array([[0, 1, 2, 3, 4, 5, 6], [7, 8, 99, -1, -1, -1, -1]], dtype=np.int32)   # 99 >= num_blocks
    q = gi.normal_f16(2, 0, (2, hq * D))
    kp = gi.normal_f16(2, 1, (10, bs, hkv * D))
    vp = gi.normal_f16(2, 2, (10, bs, hkv * D))
    kc, vc = gi.to_vllm_layout(kp, vp, hkv, D)
    ws = torch.zeros(gqa.gqa_paged_workspace_size(2, hq, hkv, D, 100, 0), dtype=torch.uint8, device="cuda")
    o = gqa.gqa_decode_paged_vllm(dev(q), dev(kc), dev(vc), dev(tab), dev(lens), hq, hkv, max_seq_len=100,
                                  workspace_tensor=ws)
    assert gqa.gqa_workspace_check(ws) == gqa.GQA_ERR_INVALID_ARG
    p = dict(q=q[:1], k_pool=kc, v_pool=vc, block_tables=tab[:1], seq_lens=lens[:1], h_q=hq, h_kv=hkv, d_head=D,
             scale=1 / 8, block_size=bs)
    assert_close(o[:1], ref(p), "vllm seq 0 next to a bad table")


def test_vllm_timeout_is_reported_not_hung(gqa):
    w = gi.custom(8, 1, 4000, 16, 4, 128, 3300, kind="paged", block_size=16, partition_size=512,
                  len_lo=2000, len_hi=4000, layout="vllm")
    p = gi.make_paged(w)
    N = 8
    ws = torch.zeros(gqa.gqa_paged_workspace_size(N, 16, 4, 128, p["max_seq_len"], 512), dtype=torch.uint8,
                     device="cuda")
    run(gqa, p, partition_size=512, workspace_tensor=ws, timeout_us=20000, test_stall_cta=3)
    assert gqa.gqa_workspace_check(ws) == gqa.GQA_ERR_TIMEOUT
    gqa.gqa_workspace_init(ws)
    o = run(gqa, p, partition_size=512, workspace_tensor=ws)
    assert gqa.gqa_workspace_check(ws) == gqa.GQA_OK
    assert_close(o, ref(p), "vllm after a timeout")


@pytest.mark.parametrize("layout", ["rows", "vllm"])
def test_partition_at_the_box_table_limit(gqa, layout):
    """Block size 8 and an 8192-key single-pass partition: 1024 TMA boxes in one work item, the
    most the scheduler's per-item table holds (one more block per partition is rejected)."""
    N, bs = 6, 8
    w = gi.custom(N, 1, 8192, 16, 4, 64, 3400, kind="paged", block_size=bs, partition_size=8192,
                  len_lo=7000, len_hi=8192, layout=layout)
    p = gi.make_paged(w)
    fn = gqa.gqa_decode_paged_vllm if layout == "vllm" else gqa.gqa_decode_paged
    args = (dev(p["q"]).reshape(N, -1), dev(p["k_pool"]), dev(p["v_pool"]), dev(p["block_tables"]),
            dev(p["seq_lens"]), 16, 4, p["scale"])
    o = fn(*args, max_seq_len=8192, partition_size=8192, head_group=1 if layout == "vllm" else 0)
    torch.cuda.synchronize()
    assert gqa.gqa_paged_plan(N, 16, 4, 64, 8192, 8192, block_size=bs)[2] == 1     # single pass
    assert_close(o, ref(p) if layout == "vllm" else
                 torch.from_numpy(np.asarray(oracle.decode_paged(p["q"], p["k_pool"], p["v_pool"], p["block_tables"],
                                                                 p["seq_lens"], 16, 4, 64, p["scale"], bs)))
                 .reshape(N, -1), f"8192-key partition, block 8 ({layout})")
    with pytest.raises(gqa.GQAError):
        fn(*args, max_seq_len=8192, partition_size=8256)
