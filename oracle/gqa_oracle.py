"""Plain float64 GQA decode attention on the CPU -- test infrastructure only.

Definition (page "kernbench2 ... _gqa_attention_decode_long.py", "GQA
fused-attention decode kernel -- long context"; kernel docstring "Tensor
layout" and the local-attention tile math), for every sequence ``b``, query
token ``t`` and query head ``h``, with ``G = h_q // h_kv`` and KV head
``g = h // G``:

    s_j  = scale * sum_d Q[b, t, h*D + d] * K[b, j, g*D + d]        j < S_kv
    m    = max_j s_j
    p_j  = exp(s_j - m)
    l    = sum_j p_j
    O[b, t, h*D + d] = (sum_j p_j * V[b, j, g*D + d]) / l

Readings where the pages are silent or differ from this (each is listed in the
design notes with its reason):

* ``scale`` multiplies the dot product (the page's kernel applies none);
* K is used with a true transpose (the page's reshape is a simulator
  shortcut valid only for zero / symmetric inputs, per its own caveat);
* query head ``h`` reads KV head ``h // G`` (contiguous groups, matching the
  page's contiguous ``(G*T_q, d_head)`` query load per KV head);
* every query token attends to all keys, no causal mask -- unless ``causal`` is
  asked for (the speculative-verification variant): then query token ``t`` of
  ``T_q`` sees the keys ``j <= S_kv - T_q + t`` only;
* every key is attended exactly once (the page's ``S_kv // n_ranks`` drops a
  remainder; the method does not);
* an empty key range gives the partial ``(m, l, O) = (-inf, 0, 0)``; merging
  it contributes nothing; normalising ``l = 0`` gives ``O = 0``.

No blocking, fusion or reordering: one full softmax per query row over its
whole key range; a torch float64 matmul is the only library primitive.
"""
from __future__ import annotations

from typing import Iterable, Optional, Sequence, Tuple

import numpy as np
import torch

__all__ = [
    "partial_rows", "merge_pair", "merge_parts", "normalize",
    "decode", "decode_unit", "decode_partial", "gather_paged", "gather_paged_vllm", "decode_paged",
    "decode_paged_seq",
]

NEG_INF = float("-inf")


def _f64(a) -> torch.Tensor:
    if isinstance(a, np.ndarray):
        a = torch.from_numpy(np.ascontiguousarray(a))
    return a.to(device="cpu", dtype=torch.float64)


# ---------------------------------------------------------------------------
# One set of query rows against one key range (the page's local attention)
# ---------------------------------------------------------------------------

def partial_rows(q_rows, k_rows, v_rows, scale: float):
    """Unnormalised partial ``(m, l, O)`` of query rows against a key range.

    Follows the page's local attention of one tile: ``scores = Q . K^T``
    (here times ``scale``), ``m`` = row max, ``exp(scores - m)``, ``l`` = row
    sum, ``O = exp(scores - m) . V``.  ``q_rows`` is ``(n, D)``, ``k_rows`` and
    ``v_rows`` are ``(S, D)``.  An empty key range gives ``(-inf, 0, 0)``.
    """
    q = _f64(q_rows)
    k = _f64(k_rows)
    v = _f64(v_rows)
    n, D = q.shape
    if k.shape[0] == 0:
        return (torch.full((n,), NEG_INF, dtype=torch.float64),
                torch.zeros(n, dtype=torch.float64),
                torch.zeros(n, D, dtype=torch.float64))
    s = float(scale) * (q @ k.T)                 # (n, S)
    m = s.max(dim=1).values                      # row max
    p = torch.exp(s - m[:, None])
    l = p.sum(dim=1)
    o = p @ v                                    # (n, D), not yet divided by l
    return m, l, o


def normalize(l, o):
    """Final normalise ``O / l`` (page: "Final normalise + store"); ``l = 0`` gives 0."""
    l = _f64(l)
    o = _f64(o)
    safe = torch.where(l > 0, l, torch.ones_like(l))
    out = o / safe[..., None]
    return torch.where((l > 0)[..., None], out, torch.zeros_like(out))


# ---------------------------------------------------------------------------
# The online-softmax merge (page: ``_merge_running``)
# ---------------------------------------------------------------------------

def merge_pair(m_a, l_a, o_a, m_b, l_b, o_b):
    """Merge two partials: ``m = max(m_a, m_b)``, each side rescaled by
    ``exp(m_side - m)``, ``l`` and ``O`` summed.  A side with ``m = -inf``
    (empty range) contributes nothing; two empty sides stay empty."""
    m_a, l_a, o_a = _f64(m_a), _f64(l_a), _f64(o_a)
    m_b, l_b, o_b = _f64(m_b), _f64(l_b), _f64(o_b)
    m_new = torch.maximum(m_a, m_b)
    both_empty = torch.isneginf(m_new)
    ref = torch.where(both_empty, torch.zeros_like(m_new), m_new)
    scale_old = torch.exp(m_a - ref)             # exp(-inf) = 0 for an empty side
    scale_new = torch.exp(m_b - ref)
    l_new = l_a * scale_old + l_b * scale_new
    o_new = o_a * scale_old[..., None] + o_b * scale_new[..., None]
    return m_new, l_new, o_new


def merge_parts(ms: Sequence, ls: Sequence, os_: Sequence):
    """Fold a list of partials left to right with :func:`merge_pair`
    (the page's sweep: the first partial seeds the running state, every later
    one is merged into it)."""
    assert len(ms) == len(ls) == len(os_) and len(ms) > 0
    m, l, o = _f64(ms[0]), _f64(ls[0]), _f64(os_[0])
    for i in range(1, len(ms)):
        m, l, o = merge_pair(m, l, o, ms[i], ls[i], os_[i])
    return m, l, o


# ---------------------------------------------------------------------------
# Contiguous layout: Q (B, T_q, h_q*D), K/V (B, S_kv, h_kv*D)
# ---------------------------------------------------------------------------

def _unit_rows(q, b: int, g: int, T_q: int, G: int, D: int):
    """Query rows of KV head ``g`` of sequence ``b``: heads ``g*G .. g*G+G-1``
    of every token, ordered (t, head) -> shape ``(T_q*G, D)``."""
    rows = q[b, :, g * G * D:(g + 1) * G * D]          # (T_q, G*D)
    return np.asarray(rows).reshape(T_q * G, D)


def decode_unit(q, k, v, b: int, g: int, h_q: int, h_kv: int, D: int, scale: float,
                s_begin: int = 0, s_len: Optional[int] = None, causal: bool = False):
    """Partial ``(m, l, O)`` of all query rows of KV head ``g`` of sequence ``b``
    over keys ``[s_begin, s_begin + s_len)``; shapes ``(T_q, G)`` and ``(T_q, G, D)``.
    With ``causal``, token ``t`` uses only the keys ``j <= S_kv - T_q + t`` of that range."""
    B, T_q, _ = q.shape
    S = k.shape[1]
    G = h_q // h_kv
    if s_len is None:
        s_len = S - s_begin
    qr = _unit_rows(q, b, g, T_q, G, D)
    if not causal:
        kr = k[b, s_begin:s_begin + s_len, g * D:(g + 1) * D]
        vr = v[b, s_begin:s_begin + s_len, g * D:(g + 1) * D]
        m, l, o = partial_rows(qr, kr, vr, scale)
        return m.reshape(T_q, G), l.reshape(T_q, G), o.reshape(T_q, G, D)
    m = torch.empty(T_q, G, dtype=torch.float64)
    l = torch.empty(T_q, G, dtype=torch.float64)
    o = torch.empty(T_q, G, D, dtype=torch.float64)
    for t in range(T_q):
        hi = max(s_begin, min(s_begin + s_len, S - T_q + t + 1))      # keys [s_begin, hi) visible
        kr = k[b, s_begin:hi, g * D:(g + 1) * D]
        vr = v[b, s_begin:hi, g * D:(g + 1) * D]
        mt, lt, ot = partial_rows(qr[t * G:(t + 1) * G], kr, vr, scale)
        m[t], l[t], o[t] = mt, lt, ot
    return m, l, o


def decode_partial(q, k, v, h_q: int, h_kv: int, D: int, scale: float,
                   s_begin: int = 0, s_len: Optional[int] = None, causal: bool = False):
    """Partials of every query row over keys ``[s_begin, s_begin + s_len)``.

    Returns ``m, l`` of shape ``(B, T_q, h_q)`` and unnormalised ``O`` of shape
    ``(B, T_q, h_q, D)`` (row order = the order of Q's rows and heads)."""
    B, T_q, _ = q.shape
    G = h_q // h_kv
    m = torch.empty(B, T_q, h_q, dtype=torch.float64)
    l = torch.empty(B, T_q, h_q, dtype=torch.float64)
    o = torch.empty(B, T_q, h_q, D, dtype=torch.float64)
    for b in range(B):
        for g in range(h_kv):
            mu, lu, ou = decode_unit(q, k, v, b, g, h_q, h_kv, D, scale, s_begin, s_len, causal)
            m[b, :, g * G:(g + 1) * G] = mu
            l[b, :, g * G:(g + 1) * G] = lu
            o[b, :, g * G:(g + 1) * G, :] = ou
    return m, l, o


def decode(q, k, v, h_q: int, h_kv: int, D: int, scale: float,
           units: Optional[Iterable[Tuple[int, int]]] = None, causal: bool = False):
    """Attention output ``(B, T_q, h_q*D)`` in float64.

    ``units`` restricts the work to the listed ``(b, g)`` pairs (sequence, KV
    head); rows of other units are NaN.  Each unit is an independent full
    softmax, so computing a subset changes nothing in the rows computed."""
    B, T_q, _ = q.shape
    G = h_q // h_kv
    out = torch.full((B, T_q, h_q * D), float("nan"), dtype=torch.float64)
    todo = [(b, g) for b in range(B) for g in range(h_kv)] if units is None else list(units)
    for b, g in todo:
        _, l, o = decode_unit(q, k, v, b, g, h_q, h_kv, D, scale, causal=causal)
        res = normalize(l, o)                                  # (T_q, G, D)
        out[b, :, g * G * D:(g + 1) * G * D] = res.reshape(T_q, G * D)
    return out


# ---------------------------------------------------------------------------
# Paged layout (page "muh_kernel_map.py", paged_attention_v1 / v2 rows):
# pools (num_blocks, block_size, h_kv*D); token j of sequence b lives in
# block block_tables[b, j // block_size], slot j % block_size.
# ---------------------------------------------------------------------------

def gather_paged(pool, table_row, length: int, block_size: int):
    """The ``length`` rows of one sequence, gathered from the pool in token order."""
    j = np.arange(int(length))
    blocks = np.asarray(table_row)[j // block_size]
    slots = j % block_size
    return np.asarray(pool)[blocks, slots]                 # (length, h_kv*D)


def gather_paged_vllm(k_cache, v_cache, table_row, length: int, block_size: int):
    """Keys and values of one sequence in token order, read from vLLM's cache layout (page
    "muh_kernel_map.py", VLLM_KERNEL_MAP 'paged_attention_v1': key_cache [num_blocks,
    num_kv_heads, head_dim/x, block_size, x]; the page gives no value layout, and the same
    serving stack's [num_blocks, num_kv_heads, head_dim, block_size] is taken).  Token j
    lives in block ``table_row[j // block_size]``, slot ``j % block_size``; dimension
    ``c*x + e`` of KV head g is ``k_cache[block, g, c, slot, e]`` and value dimension ``e`` is
    ``v_cache[block, g, e, slot]``.  Returns both as ``(length, h_kv*D)`` in head-major order."""
    kc, vc = np.asarray(k_cache), np.asarray(v_cache)
    _, h_kv, dx, _, x = kc.shape
    j = np.arange(int(length))
    blocks = np.asarray(table_row)[j // block_size]
    slots = j % block_size
    k = kc[blocks, :, :, slots, :]                        # (length, h_kv, D/x, x)
    v = vc[blocks, :, :, slots]                           # (length, h_kv, D)
    return k.reshape(len(j), h_kv * dx * x), v.reshape(len(j), h_kv * dx * x)


def decode_paged_seq(q, k_pool, v_pool, block_tables, seq_lens, b: int,
                     h_q: int, h_kv: int, D: int, scale: float, block_size: int, layout: str = "rows"):
    """Output ``(T_q, h_q*D)`` of sequence ``b``: the contiguous definition on
    its gathered keys and values.  ``seq_len = 0`` gives zeros.  ``layout``: "rows" for
    pools ``(num_blocks, block_size, h_kv*D)``, "vllm" for vLLM's caches."""
    L = int(seq_lens[b])
    if layout == "vllm":
        kb, vb = gather_paged_vllm(k_pool, v_pool, block_tables[b], L, block_size)
        kb, vb = kb[None], vb[None]
    else:
        kb = gather_paged(k_pool, block_tables[b], L, block_size)[None]
        vb = gather_paged(v_pool, block_tables[b], L, block_size)[None]
    qb = np.asarray(q[b:b + 1])
    if qb.ndim == 2:
        qb = qb[:, None, :]
    T_q = qb.shape[1]
    G = h_q // h_kv
    out = torch.empty(T_q, h_q * D, dtype=torch.float64)
    for g in range(h_kv):
        _, l, o = decode_unit(qb, kb, vb, 0, g, h_q, h_kv, D, scale)
        out[:, g * G * D:(g + 1) * G * D] = normalize(l, o).reshape(T_q, G * D)
    return out


def decode_paged(q, k_pool, v_pool, block_tables, seq_lens, h_q: int, h_kv: int, D: int,
                 scale: float, block_size: int, seqs: Optional[Iterable[int]] = None, layout: str = "rows"):
    """Paged attention output ``(num_seqs, T_q, h_q*D)``; ``seqs`` restricts the
    work to some sequences (others are NaN).  ``layout`` as in ``decode_paged_seq``."""
    q = np.asarray(q)
    if q.ndim == 2:
        q = q[:, None, :]
    N, T_q, _ = q.shape
    out = torch.full((N, T_q, h_q * D), float("nan"), dtype=torch.float64)
    for b in (range(N) if seqs is None else seqs):
        out[b] = decode_paged_seq(q, k_pool, v_pool, block_tables, seq_lens, b,
                                  h_q, h_kv, D, scale, block_size, layout)
    return out

