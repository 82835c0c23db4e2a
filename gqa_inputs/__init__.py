"""Seeded synthetic inputs for GQA decode attention.

This module is the one piece of code that both sides of the parity check use:
the CPU oracle (``oracle/``) and the CUDA library (``decode_attention_03_gb300``)
are fed the very same arrays from here.  It therefore holds no attention
arithmetic at all -- only random draws, shapes and index bookkeeping.

Generator convention (frozen; regression constants live in
``tests/test_inputs.py``):

* every tensor is identified by ``(seed, stream)``; a tensor is viewed as a
  2-D array of ``rows x cols`` (its last dimension is ``cols``) and drawn in
  chunks of ``CHUNK_ROWS`` rows; chunk ``c`` uses its own
  ``numpy.random.Generator(PCG64(SeedSequence([seed, stream, c])))``.  Chunks
  are independent, so the draw is the same whatever the number of threads
  and on any platform (numpy's bit-stream guarantee for PCG64 and
  ``standard_normal``/``random``);
* normals are drawn as float32 and rounded to float16 (round-to-nearest-even);
* uniforms in ``[lo, hi)`` are float32 ``lo + (hi-lo)*U`` rounded to float16;
* bfloat16 workloads round the same float32 draws to bfloat16 (nearest even) instead;
  numpy has no bfloat16, so they are held as their 16-bit patterns (``uint16``) and
  decoded exactly with :func:`bf16_to_f32`;
* integer draws (sequence lengths, permutations) use the stream's
  un-chunked generator ``SeedSequence([seed, stream])``.

Workloads follow the shapes the pages give for the decode kernel (contiguous
``(S_kv, h_kv*d_head)`` K/V and ``(T_q, h_q*d_head)`` Q, "GQA fused-attention
decode kernel -- long context", kernel docstring) and the vLLM paged
attention v2 shape (16-token KV blocks, 512-token partitions;
"muh_kernel_map.py", ``VLLM_KERNEL_MAP['paged_attention_v1'/'v2']``).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, asdict
from typing import Dict, Optional

import numpy as np

CHUNK_ROWS = 65536

# stream ids
S_Q, S_K, S_V, S_LENS, S_PERM, S_SPIKE = 0, 1, 2, 3, 4, 5


def _gen(seed: int, stream: int, chunk: Optional[int] = None) -> np.random.Generator:
    key = [int(seed), int(stream)] if chunk is None else [int(seed), int(stream), int(chunk)]
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(key)))


def _threads() -> int:
    return max(1, min(os.cpu_count() or 1, 32))


def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bfloat16, nearest even; returns the bit patterns."""
    bits = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounded = (bits + np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact float32 values of bfloat16 bit patterns."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _draw_2d(seed: int, stream: int, rows: int, cols: int, kind: str,
             lo: float = -1.0, hi: float = 1.0, elem: str = "f16") -> np.ndarray:
    out = np.empty((rows, cols), dtype=np.float16 if elem == "f16" else np.uint16)
    n_chunks = (rows + CHUNK_ROWS - 1) // CHUNK_ROWS

    def one(c: int) -> None:
        r0 = c * CHUNK_ROWS
        r1 = min(rows, r0 + CHUNK_ROWS)
        g = _gen(seed, stream, c)
        if kind == "normal":
            a = g.standard_normal((r1 - r0, cols), dtype=np.float32)
        elif kind == "uniform":
            a = g.random((r1 - r0, cols), dtype=np.float32)
            a *= np.float32(hi - lo)
            a += np.float32(lo)
        else:
            raise ValueError(kind)
        out[r0:r1] = a.astype(np.float16) if elem == "f16" else f32_to_bf16(a)

    if n_chunks <= 1:
        for c in range(n_chunks):
            one(c)
    else:
        with ThreadPoolExecutor(min(_threads(), n_chunks)) as ex:
            list(ex.map(one, range(n_chunks)))
    return out


def normal_f16(seed: int, stream: int, shape, elem: str = "f16") -> np.ndarray:
    """N(0,1) float32 draws rounded to float16 (or to bfloat16 bit patterns with
    ``elem='bf16'``), shape ``shape``."""
    shape = tuple(int(s) for s in shape)
    cols = shape[-1]
    rows = int(np.prod(shape[:-1])) if len(shape) > 1 else 1
    return _draw_2d(seed, stream, rows, cols, "normal", elem=elem).reshape(shape)


def uniform_f16(seed: int, stream: int, shape, lo: float = -1.0, hi: float = 1.0, elem: str = "f16") -> np.ndarray:
    """Uniform ``[lo, hi)`` float32 draws rounded to float16 (or bfloat16 bit patterns),
    shape ``shape``."""
    shape = tuple(int(s) for s in shape)
    cols = shape[-1]
    rows = int(np.prod(shape[:-1])) if len(shape) > 1 else 1
    return _draw_2d(seed, stream, rows, cols, "uniform", lo, hi, elem=elem).reshape(shape)


# ---------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    """One synthetic decode workload.

    ``kind`` is ``"contiguous"`` (K/V ``(batch, S_kv, h_kv*d_head)``) or
    ``"paged"`` (K/V pools ``(num_blocks, block_size, h_kv*d_head)`` addressed
    through per-sequence block tables).  ``spike_frac``/``spike_mult`` scale a
    seeded fraction of whole key rows (all heads) to create large logits;
    ``v_dist`` is ``"normal"`` or ``"uniform"`` (on ``[-1, 1)``).
    """
    name: str
    kind: str
    batch: int
    T_q: int
    S_kv: int            # contiguous: keys per sequence; paged: max length bound
    h_q: int
    h_kv: int
    d_head: int
    seed: int
    v_dist: str = "normal"
    spike_frac: float = 0.0
    spike_mult: float = 1.0
    block_size: int = 16
    partition_size: int = 512
    len_lo: int = 0      # paged: inclusive bounds of the per-sequence length
    len_hi: int = 0
    elem: str = "f16"    # element type of Q, K, V: "f16" or "bf16" (bit patterns)
    layout: str = "rows"  # paged: "rows" pools (num_blocks, block_size, h_kv*d) or "vllm" caches
                          # k (num_blocks, h_kv, d/8, block_size, 8), v (num_blocks, h_kv, d, block_size)

    @property
    def G(self) -> int:
        return self.h_q // self.h_kv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d_head)

    def asdict(self) -> dict:
        return asdict(self)


WORKLOADS: Dict[str, Workload] = {
    # T_q=1, S_kv=4096, h_q=8, h_kv=2 (G=4), d_head=64, one sequence, seed 0
    "tiny": Workload("tiny", "contiguous", 1, 1, 4096, 8, 2, 64, seed=0),
    # Llama-3-8B-shaped decode step: 8 sequences of 32768, h_q=32, h_kv=8, d=128, seed 1
    "llama8b": Workload("llama8b", "contiguous", 8, 1, 32768, 32, 8, 128, seed=1),
    # one sequence of 2^20 keys (~4 GiB of f16 K+V), seed 2
    "long": Workload("long", "contiguous", 1, 1, 1048576, 32, 8, 128, seed=2),
    # paged v2 shape: 64 sequences, lengths uniform in [1024, 16384], block 16, partition 512, seed 3
    "paged": Workload("paged", "paged", 64, 1, 16384, 32, 8, 128, seed=3,
                      block_size=16, partition_size=512, len_lo=1024, len_hi=16384),
    # stability / ragged stress: T_q=4, S_kv=131071, h_q=64, h_kv=8 (G=8); 1% of key rows x8;
    # V uniform in [-1, 1); seed 4
    "ragged": Workload("ragged", "contiguous", 1, 4, 131071, 64, 8, 128, seed=4,
                       v_dist="uniform", spike_frac=0.01, spike_mult=8.0),
    # speculative verification of 16 draft tokens (G*T_q = 128 query rows per KV head, the
    # tcgen05 path): T_q=16, S_kv=262143, h_q=64, h_kv=8; the ragged stress's value
    # distributions (1% of key rows x8, V uniform in [-1, 1)); seed 5
    "verify16": Workload("verify16", "contiguous", 1, 16, 262143, 64, 8, 128, seed=5,
                         v_dist="uniform", spike_frac=0.01, spike_mult=8.0),
    # the paged workload's values (seed 3) in vLLM's cache layout, partitions chosen automatically
    "paged_vllm": Workload("paged_vllm", "paged", 64, 1, 16384, 32, 8, 128, seed=3,
                           block_size=16, partition_size=0, len_lo=1024, len_hi=16384, layout="vllm"),
    # many short sequences (<= 8192 keys: the page's single-pass v1 regime), vLLM layout, run as
    # v1 (one partition of 2048 keys per sequence): 384 sequences, lengths uniform in [128, 2048],
    # block 16; seed 6
    "paged_v1": Workload("paged_v1", "paged", 384, 1, 2048, 32, 8, 128, seed=6,
                         block_size=16, partition_size=2048, len_lo=128, len_hi=2048, layout="vllm"),
}


def custom(batch: int, T_q: int, S_kv: int, h_q: int, h_kv: int, d_head: int, seed: int,
           **kw) -> Workload:
    """A contiguous (or, with ``kind='paged'``, paged) workload of any shape."""
    kind = kw.pop("kind", "contiguous")
    name = kw.pop("name", f"custom_b{batch}_t{T_q}_s{S_kv}_hq{h_q}_hkv{h_kv}_d{d_head}_seed{seed}")
    return Workload(name, kind, batch, T_q, S_kv, h_q, h_kv, d_head, seed, **kw)


def make_contiguous(w: Workload) -> dict:
    """Q ``(batch, T_q, h_q*d)``, K/V ``(batch, S_kv, h_kv*d)`` float16 arrays."""
    assert w.kind == "contiguous"
    e = w.elem
    q = normal_f16(w.seed, S_Q, (w.batch, w.T_q, w.h_q * w.d_head), e)
    k = normal_f16(w.seed, S_K, (w.batch, w.S_kv, w.h_kv * w.d_head), e)
    if w.v_dist == "normal":
        v = normal_f16(w.seed, S_V, (w.batch, w.S_kv, w.h_kv * w.d_head), e)
    else:
        v = uniform_f16(w.seed, S_V, (w.batch, w.S_kv, w.h_kv * w.d_head), -1.0, 1.0, e)
    spike_rows = np.zeros((0,), dtype=np.int64)
    if w.spike_frac > 0.0:
        n_spike = int(round(w.spike_frac * w.S_kv))
        spike_rows = _gen(w.seed, S_SPIKE).permutation(w.S_kv)[:n_spike].astype(np.int64)
        if e == "f16":
            k[:, spike_rows, :] *= np.float16(w.spike_mult)   # x8 is exact in float16
        else:
            k[:, spike_rows, :] = f32_to_bf16(bf16_to_f32(k[:, spike_rows, :]) * np.float32(w.spike_mult))
    return dict(workload=w, q=q, k=k, v=v, spike_rows=spike_rows, elem=e,
                batch=w.batch, T_q=w.T_q, S_kv=w.S_kv, h_q=w.h_q, h_kv=w.h_kv,
                d_head=w.d_head, scale=w.scale)


def paged_layout(w: Workload):
    """Sequence lengths, block tables and pool size of a paged workload.

    Lengths are uniform integers in ``[len_lo, len_hi]``; sequence ``b`` owns
    ``ceil(len_b / block_size)`` blocks, taken in order from a seeded random
    permutation of the pool.  Unused table entries are ``-1``.
    """
    assert w.kind == "paged"
    lens = _gen(w.seed, S_LENS).integers(w.len_lo, w.len_hi + 1, size=w.batch).astype(np.int64)
    nblk = (lens + w.block_size - 1) // w.block_size
    num_blocks = int(nblk.sum())
    perm = _gen(w.seed, S_PERM).permutation(num_blocks).astype(np.int32)
    max_blocks = int(nblk.max()) if w.batch > 0 else 0
    tables = np.full((w.batch, max(1, max_blocks)), -1, dtype=np.int32)
    off = 0
    for b in range(w.batch):
        tables[b, : nblk[b]] = perm[off: off + nblk[b]]
        off += int(nblk[b])
    return lens.astype(np.int32), tables, num_blocks


def to_vllm_layout(k_pool: np.ndarray, v_pool: np.ndarray, h_kv: int, d_head: int):
    """The same keys and values rearranged into vLLM's caches: k (num_blocks, h_kv, d/8,
    block_size, 8), v (num_blocks, h_kv, d, block_size)."""
    nb, bs, _ = k_pool.shape
    k = k_pool.reshape(nb, bs, h_kv, d_head // 8, 8).transpose(0, 2, 3, 1, 4)
    v = v_pool.reshape(nb, bs, h_kv, d_head).transpose(0, 2, 3, 1)
    return np.ascontiguousarray(k), np.ascontiguousarray(v)


def make_paged(w: Workload, tail_fill: str = "normal") -> dict:
    """Q ``(num_seqs, h_q*d)``, K/V pools ``(num_blocks, block_size, h_kv*d)`` (``layout='vllm'``:
    the same values in vLLM's caches, under the same keys).

    ``tail_fill='nan'`` overwrites the pool slots past each sequence's end (the
    unused tail of its last block) with float16 NaN in both K and V; a correct
    kernel must not read them into the result.
    """
    lens, tables, num_blocks = paged_layout(w)
    e = w.elem
    q = normal_f16(w.seed, S_Q, (w.batch, w.T_q, w.h_q * w.d_head), e)
    kp = normal_f16(w.seed, S_K, (num_blocks, w.block_size, w.h_kv * w.d_head), e)
    vp = normal_f16(w.seed, S_V, (num_blocks, w.block_size, w.h_kv * w.d_head), e)
    if tail_fill == "nan":
        nan = np.float16(np.nan) if e == "f16" else np.uint16(0x7FC0)
        for b in range(w.batch):
            L = int(lens[b])
            if L % w.block_size:
                last = tables[b, L // w.block_size]
                kp[last, L % w.block_size:, :] = nan
                vp[last, L % w.block_size:, :] = nan
    elif tail_fill != "normal":
        raise ValueError(tail_fill)
    if w.layout == "vllm":
        kp, vp = to_vllm_layout(kp, vp, w.h_kv, w.d_head)
    elif w.layout != "rows":
        raise ValueError(w.layout)
    return dict(workload=w, q=q, k_pool=kp, v_pool=vp, block_tables=tables, seq_lens=lens, elem=e, layout=w.layout,
                num_seqs=w.batch, T_q=w.T_q, h_q=w.h_q, h_kv=w.h_kv, d_head=w.d_head,
                scale=w.scale, num_blocks=num_blocks, block_size=w.block_size,
                partition_size=w.partition_size, max_blocks_per_seq=tables.shape[1],
                max_seq_len=int(lens.max()) if w.batch else 0)


def make(w) -> dict:
    """Inputs of a workload given by name or as a :class:`Workload`."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    return make_contiguous(w) if w.kind == "contiguous" else make_paged(w)


def kv_bytes(inp: dict) -> int:
    """Bytes the decode step must move: K + V + Q + O (+ block tables and lengths when paged).

    For a paged workload only the K/V rows of the sequences' own tokens count.
    """
    if "k" in inp:
        k = inp["k"]
        q = inp["q"]
        return 2 * k.nbytes + 2 * q.nbytes
    row = inp["h_kv"] * inp["d_head"] * 2
    tokens = int(np.asarray(inp["seq_lens"], dtype=np.int64).sum())
    nblk_used = int(((np.asarray(inp["seq_lens"], dtype=np.int64) + inp["block_size"] - 1)
                     // inp["block_size"]).sum())
    return (2 * tokens * row + 2 * inp["q"].nbytes + nblk_used * 4 + inp["seq_lens"].nbytes)


def values(a: np.ndarray, elem: str) -> np.ndarray:
    """Exact float32 values of an input array (float16 as is, bfloat16 bit patterns decoded)."""
    return a.astype(np.float32) if elem == "f16" else bf16_to_f32(a)
