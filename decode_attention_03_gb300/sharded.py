"""Decode over a key axis sharded across ranks (one process per GPU).

The method's own multi-device form (page "kernbench2 ... _gqa_attention_decode_long.py",
module docstring: each of the C*P ranks sweeps a contiguous ``S_local`` slice of S_kv;
section "Communication: chain reduce-to-root at PE 0 of CUBE 0"): every rank computes the
partial ``(m, l, O)`` of all query rows over the keys it holds, the partials meet at the
root and are folded with ``_merge_running``, and the root divides by ``l``.

Here a rank's partial is one ``gqa_decode_partial`` call on its own device, the partials
are exchanged in ONE collective (an all-gather, or a gather to one root: the page's chain of
point-to-point hops is a latency-bound way of doing the same reduction), and ``gqa_merge``
folds them in rank order and normalises.  Every arithmetic step runs in the library's CUDA
kernels; this module only slices, packs and moves fp32 partials.

Readings:
  * the page gives each rank ``S_kv // (C*P)`` keys and drops the remainder; here every key is
    attended exactly once: :func:`shard_range` gives the first ``S_kv % world`` ranks one key
    more, and a rank may hold no key at all (its partial is the empty one, ``(-inf, 0, 0)``);
  * the page exchanges the partials as f16; here they stay fp32 (as the paged v2 row's
    ``exp_sum`` / ``max_logits`` on page "muh_kernel_map.py");
  * every query token attends to all keys of all shards (no causal tail across shards).
"""
from __future__ import annotations

import math
from typing import Optional, Tuple

import torch
import torch.distributed as dist


def shard_range(S_kv: int, rank: int, world: int) -> Tuple[int, int]:
    """Keys ``[begin, begin + length)`` of rank ``rank`` out of ``world``: contiguous, in rank
    order, every key exactly once; lengths differ by at most one (0 when S_kv < world)."""
    if world < 1 or not 0 <= rank < world or S_kv < 0:
        raise ValueError("need 0 <= rank < world and S_kv >= 0")
    base, rem = divmod(int(S_kv), int(world))
    begin = rank * base + min(rank, rem)
    return begin, base + (1 if rank < rem else 0)


def _pack(m: torch.Tensor, l: torch.Tensor, o: torch.Tensor) -> torch.Tensor:
    return torch.cat([m.reshape(-1), l.reshape(-1), o.reshape(-1)])


def _unpack(flat: torch.Tensor, world: int, rows: int, d_head: int):
    per = rows * (d_head + 2)
    parts = flat.reshape(world, per)
    m = parts[:, :rows]
    l = parts[:, rows:2 * rows]
    o = parts[:, 2 * rows:].reshape(world, rows, d_head)
    return m.contiguous(), l.contiguous(), o.contiguous()


def exchange_partials(m: torch.Tensor, l: torch.Tensor, o: torch.Tensor, *, group=None,
                      root: Optional[int] = None):
    """Collect every rank's fp32 partial ``m, l (rows)``, ``o (rows, d_head)`` in rank order.

    ``root=None``: every rank receives them (one all-gather); ``root=r``: only rank ``r`` does
    (one gather) and the others get ``(None, None, None)``.  Returned shapes ``(world, rows)``,
    ``(world, rows)``, ``(world, rows, d_head)`` on the partials' device.  The three tensors
    travel packed in one message per rank.  NCCL moves device tensors directly; any other
    backend (gloo) is handed host copies."""
    rows, d_head = o.shape
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size(group) == 1:
        return m.reshape(1, rows), l.reshape(1, rows), o.reshape(1, rows, d_head)   # a single rank
    world = dist.get_world_size(group)
    flat = _pack(m, l, o)
    device_ok = dist.get_backend(group) == "nccl" and flat.is_cuda
    send = flat if device_ok else flat.cpu()
    if root is None:
        recv = torch.empty(world * send.numel(), dtype=send.dtype, device=send.device)
        if device_ok:
            dist.all_gather_into_tensor(recv, send, group=group)
        else:
            dist.all_gather(list(recv.chunk(world)), send, group=group)
    else:
        me = dist.get_rank(group)
        recv = torch.empty(world * send.numel(), dtype=send.dtype, device=send.device) if me == root else None
        dst = dist.get_global_rank(group, root) if group is not None else root
        dist.gather(send, list(recv.chunk(world)) if recv is not None else None, dst=dst, group=group)
        if recv is None:
            return None, None, None
    recv = recv.to(flat.device, non_blocking=True)
    return _unpack(recv, world, rows, d_head)


def sharded_decode(q: torch.Tensor, k_shard: torch.Tensor, v_shard: torch.Tensor, h_q: int, h_kv: int,
                   scale: Optional[float] = None, *, group=None, root: Optional[int] = None,
                   out: Optional[torch.Tensor] = None, stream=None) -> Optional[torch.Tensor]:
    """Attention output of ``q (B, T_q, h_q*D)`` over the keys of all ranks' shards.

    Every rank passes the same ``q`` and its own ``k_shard, v_shard (B, s_local, h_kv*D)``: the
    rank's contiguous slice of each sequence's keys, in rank order (``shard_range``), possibly
    empty.  Returns ``O (B, T_q, h_q*D)`` on every rank (``root=None``) or on rank ``root`` only
    (``None`` elsewhere).  float16 or bfloat16 inputs and output (q's dtype), fp32 partials."""
    from . import _binding as b

    if q.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("sharded_decode takes float16 or bfloat16 inputs")
    B, T_q, qc = q.shape
    D = qc // h_q
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    s_local = k_shard.shape[1]
    st = torch.cuda.current_stream(q.device) if stream is None else stream
    with torch.cuda.stream(st):   # the partial, the exchange and the merge in stream order
        m, l, o = b.gqa_decode_partial(q, k_shard, v_shard, h_q, h_kv, 0, s_local, scale, stream=st)
        ms, ls, os_ = exchange_partials(m, l, o, group=group, root=root)
        if ms is None:
            return None
        rows = B * T_q * h_q
        res = torch.empty(rows, D, dtype=q.dtype, device=q.device) if out is None else out.view(rows, D)
        b.gqa_merge(ms, ls, os_, out=res, stream=st)
    return res.view(B, T_q, qc)
