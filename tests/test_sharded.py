"""The key axis sharded across ranks (the method's own multi-device form, page "kernbench2 ...
_gqa_attention_decode_long.py": every rank sweeps a contiguous slice of S_kv, the (m, l, O)
partials meet at the root, are merged with _merge_running and divided by l).

CPU tests (gloo, spawned ranks): ``shard_range`` covers every key once; ``exchange_partials``
delivers every rank's partial in rank order, to all ranks or to one root.  The partials in
those tests are the oracle's (test infrastructure), cast to fp32 as the kernels emit them.

GPU test: ranks as processes on cuda:0, exchanging over gloo (nothing on the device waits on
another rank), each running ``sharded_decode`` on its own uneven (sometimes empty) shard; every
rank's output is checked against the oracle on the whole sequence.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import gqa_inputs as gi


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _run_ranks(target, world, *extra, timeout=300):
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=target, args=(r, world, port, out) + extra) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=timeout)
        codes = [p.exitcode for p in procs]
        res = dict(out)
    assert codes == [0] * world, f"rank exit codes {codes}, results {res}"
    return res


def _init(rank, world, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)


@pytest.mark.parametrize("S,world", [(0, 1), (1, 2), (5, 8), (1000, 3), (4096, 2), (131071, 7)])
def test_shard_range_covers_every_key_once(S, world):
    from decode_attention_03_gb300.sharded import shard_range
    seen = np.zeros(S, dtype=np.int64)
    lens = []
    prev_end = 0
    for r in range(world):
        b, n = shard_range(S, r, world)
        assert b == prev_end                      # contiguous, in rank order
        seen[b:b + n] += 1
        prev_end = b + n
        lens.append(n)
    assert prev_end == S and (seen == 1).all()
    assert max(lens) - min(lens) <= 1


def _exchange_worker(rank, world, port, out, root):
    _init(rank, world, port)
    import oracle
    from decode_attention_03_gb300.sharded import exchange_partials, shard_range
    x = gi.make_contiguous(gi.custom(2, 2, 301, 8, 2, 16, 4242))
    b, n = shard_range(301, rank, world)
    m, l, o = oracle.decode_partial(x["q"], x["k"], x["v"], 8, 2, 16, 0.25, b, n)
    ms, ls, os_ = exchange_partials(m.float().reshape(-1), l.float().reshape(-1), o.float().reshape(-1, 16),
                                    root=root)
    if ms is None:
        out[rank] = None
    else:
        assert ms.shape == (world, 2 * 2 * 8) and os_.shape == (world, 2 * 2 * 8, 16)
        mm, ll, oo = oracle.merge_parts(list(ms), list(ls), list(os_))
        got = oracle.normalize(ll, oo).reshape(2, 2, 8 * 16)
        ref = oracle.decode(x["q"], x["k"], x["v"], 8, 2, 16, 0.25)
        out[rank] = float((got - ref).abs().max())
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,root", [(2, None), (2, 0), (3, 1), (4, None)])
def test_exchange_partials_gloo(world, root):
    res = _run_ranks(_exchange_worker, world, root)
    for r in range(world):
        if root is None or r == root:
            assert res[r] is not None and res[r] < 1e-5, res     # fp32 transport of fp64 partials
        else:
            assert res[r] is None


# ---------------------------------------------------------------- on the GPU
def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:                       # bfloat16 bit patterns
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def _gpu_worker(rank, world, port, out, cuts, root, shape, elem="f16"):
    _init(rank, world, port)
    torch.cuda.set_device(0)
    from decode_attention_03_gb300 import build
    build.build()
    from decode_attention_03_gb300.sharded import sharded_decode
    B, T_q, S, hq, hkv, D, seed = shape
    x = gi.make_contiguous(gi.custom(B, T_q, S, hq, hkv, D, seed, elem=elem))
    a, b = cuts[rank], cuts[rank + 1]
    q = _dev(x["q"])
    k = _dev(x["k"][:, a:b])
    v = _dev(x["v"][:, a:b])
    o = sharded_decode(q, k, v, hq, hkv, x["scale"], root=root)
    torch.cuda.synchronize()
    assert o is None or o.dtype == q.dtype
    out[rank] = None if o is None else o.double().cpu().numpy()
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.gpu
@pytest.mark.parametrize("world,cuts,root", [
    (2, [0, 2048, 5000], None),          # even-ish
    (2, [0, 4937, 5000], 0),             # uneven, reduce to a root
    (2, [0, 0, 5000], None),             # rank 0 holds no key
    (3, [0, 1, 1, 5000], 2),             # one key, one empty shard, the rest
])
def test_sharded_decode_matches_oracle(world, cuts, root):
    import oracle
    shape = (2, 1, 5000, 32, 8, 128, 5150)
    res = _run_ranks(_gpu_worker, world, cuts, root, shape, timeout=600)
    B, T_q, S, hq, hkv, D, seed = shape
    x = gi.make_contiguous(gi.custom(B, T_q, S, hq, hkv, D, seed))
    ref = oracle.decode(x["q"], x["k"], x["v"], hq, hkv, D, x["scale"]).numpy()
    for r in range(world):
        if root is not None and r != root:
            assert res[r] is None
            continue
        got = res[r].reshape(ref.shape)
        err = np.abs(got - ref)
        assert (err <= 2e-3 + 2e-3 * np.abs(ref)).all(), f"rank {r}: max err {err.max():.3e}"
        assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 5e-3


@pytest.mark.gpu
def test_sharded_decode_bf16():
    """bfloat16 inputs: the partials stay fp32, gqa_merge writes bfloat16 (tolerance of the bf16 path)."""
    import oracle
    shape = (1, 2, 3000, 16, 4, 64, 5160)
    cuts = [0, 1234, 3000]
    res = _run_ranks(_gpu_worker, 2, cuts, None, shape, "bf16", timeout=600)
    B, T_q, S, hq, hkv, D, seed = shape
    x = gi.make_contiguous(gi.custom(B, T_q, S, hq, hkv, D, seed, elem="bf16"))
    vals = {n: gi.values(x[n], "bf16") for n in ("q", "k", "v")}
    ref = oracle.decode(vals["q"], vals["k"], vals["v"], hq, hkv, D, x["scale"]).numpy()
    for r in range(2):
        got = res[r].reshape(ref.shape)
        err = np.abs(got - ref)
        assert (err <= 2e-3 + 8e-3 * np.abs(ref)).all(), f"rank {r}: max err {err.max():.3e}"
        assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 1e-2
