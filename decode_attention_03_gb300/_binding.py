"""ctypes binding of ``libgqa_decode.so`` -- argument marshalling only.

Every function here has the name of the C entry point it calls (see
``include/gqa_decode.h``), takes torch tensors where the C call takes device
pointers, reads sizes off the tensors' shapes, and raises :class:`GQAError`
when the call returns a non-OK status.  All compute runs in the library's CUDA
kernels; there is no other code path.  If the library has not been built,
importing this module raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgqa_decode.so")

GQA_OK = 0
GQA_ERR_INVALID_ARG = 1
GQA_ERR_UNSUPPORTED = 2
GQA_ERR_WORKSPACE = 3
GQA_ERR_CUDA = 4
GQA_ERR_TIMEOUT = 5
GQA_ERR_BOUNDS = 6
GQA_BUILD_BOUNDS_CHECK = 1


class GQAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {gqa_status_string(status)} (status {status})")


class gqa_options(ctypes.Structure):
    _fields_ = [("n_splits", ctypes.c_int), ("merge_mode", ctypes.c_int),
                ("timeout_us", ctypes.c_uint32), ("test_stall_cta", ctypes.c_int),
                ("paged_head_group", ctypes.c_int), ("causal", ctypes.c_int), ("bf16", ctypes.c_int),
                ("mma_path", ctypes.c_int)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    return ctypes.CDLL(LIB_PATH)


lib = _load()

_p, _i, _i64, _sz, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
_opt = ctypes.POINTER(gqa_options)
_SIGS = {
    "gqa_default_options": ([], gqa_options),
    "gqa_status_string": ([_i], ctypes.c_char_p),
    "gqa_version": ([], _i),
    "gqa_build_flags": ([], _i),
    "gqa_decode_num_splits": ([_i, _i, _i64, _i, _i, _i], _i),
    "gqa_decode_plan": ([_i, _i, _i64, _i, _i, _i, _opt, _p, _p, _p], _i),
    "gqa_decode_plan_ex": ([_i, _i, _i64, _i, _i, _i, _opt, _p, _p, _p, _p, _p], _i),
    "gqa_paged_plan": ([_i, _i, _i, _i, _i, _i, _i, _i, _opt, _p, _p, _p], _i),
    "gqa_decode_workspace_size": ([_i, _i, _i64, _i, _i, _i, _i], _sz),
    "gqa_workspace_size": ([_i, _i, _i64, _i, _i, _i], _sz),
    "gqa_paged_workspace_size": ([_i, _i, _i, _i, _i, _i], _sz),
    "gqa_workspace_init": ([_p, _sz, _p], _i),
    "gqa_workspace_check": ([_p, _p], _i),
    "gqa_decode": ([_p, _p, _p, _p, _i, _i, _i64, _i, _i, _i, _f, _p, _sz, _p], _i),
    "gqa_decode_ex": ([_p, _p, _p, _p, _i, _i, _i64, _i, _i, _i, _f, _p, _sz, _p, _opt], _i),
    "gqa_decode_partial": ([_p, _p, _p, _p, _p, _p, _i, _i, _i64, _i64, _i64, _i, _i, _i, _f, _p, _sz, _p], _i),
    "gqa_decode_partial_ex": ([_p, _p, _p, _p, _p, _p, _i, _i, _i64, _i64, _i64, _i, _i, _i, _f, _p, _sz, _p,
                               _opt], _i),
    "gqa_merge": ([_p, _p, _p, _i, _i64, _i, _p, _p], _i),
    "gqa_merge_ex": ([_p, _p, _p, _i, _i64, _i, _p, _p, _opt], _i),
    "gqa_merge_partial": ([_p, _p, _p, _i, _i64, _i, _p, _p, _p, _p], _i),
    "gqa_decode_paged": ([_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i, _p, _sz, _p], _i),
    "gqa_decode_paged_ex": ([_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i, _p, _sz, _p, _opt],
                            _i),
    "gqa_decode_noalloc": ([_p, _p, _p, _p, _i, _i, _i64, _i, _i, _i, _f, _p], _i),
    "gqa_decode_noalloc_check": ([_p], _i),
    "gqa_decode_paged_vllm": ([_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i, _p, _sz, _p], _i),
    "gqa_decode_paged_vllm_ex": ([_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i, _p, _sz, _p,
                                  _opt], _i),
}
def _bind(cdll):
    for name, (args, res) in _SIGS.items():
        fn = getattr(cdll, name)
        fn.argtypes = args
        fn.restype = res
    return cdll


_bind(lib)


def open_library(path: str):
    """Another build of the library (e.g. the bounds-checked ``libgqa_decode_checked.so``) as a
    ctypes handle with every entry point's signature set; its functions are called directly."""
    return _bind(ctypes.CDLL(path))

EXPORTED = tuple(_SIGS)


def gqa_status_string(status: int) -> str:
    return lib.gqa_status_string(int(status)).decode()


def gqa_version() -> int:
    return lib.gqa_version()


def _check(status: int, where: str) -> None:
    if status != GQA_OK:
        raise GQAError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _f16(t: torch.Tensor, name: str) -> None:
    if not (t.is_cuda and t.dtype == torch.float16 and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous float16 CUDA tensor")


def _h16(t: torch.Tensor, name: str, dtype=None) -> None:
    """float16 or bfloat16 (and equal to ``dtype`` when given)."""
    if not (t.is_cuda and t.dtype in (torch.float16, torch.bfloat16) and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous float16 or bfloat16 CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}")


def _f32(t: torch.Tensor, name: str) -> None:
    if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")


def _opts(n_splits=0, merge_mode=0, timeout_us=0, test_stall_cta=-1, paged_head_group=0, causal=False,
          bf16=False, mma_path=0):
    o = gqa_options()
    o.n_splits, o.merge_mode, o.timeout_us, o.test_stall_cta = int(n_splits), int(merge_mode), int(timeout_us), \
        int(test_stall_cta)
    o.paged_head_group = int(paged_head_group)
    o.causal = 1 if causal else 0
    o.bf16 = 1 if bf16 else 0
    o.mma_path = int(mma_path)
    return o


# ---------------------------------------------------------------- workspaces
_ws_lock = threading.Lock()
_ws_cache = {}


def workspace(nbytes: int, device=None, stream=None) -> torch.Tensor:
    """A zero-initialised workspace of at least ``nbytes``, cached per (device, stream).

    Calls that share a workspace must not overlap on the GPU: keep one per stream."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    sid = _stream(stream).value or 0
    key = (dev.index, sid)
    with _ws_lock:
        t = _ws_cache.get(key)
        if t is None or t.numel() < nbytes:
            # growing the cache (rare): the replaced workspace may still be in use on `stream`, and
            # the new one is zero-filled on the current stream, which need not be `stream`; a device
            # synchronisation orders both (not while a graph is being captured: there the fill is
            # captured on the capturing stream)
            capturing = torch.cuda.is_current_stream_capturing()
            if not capturing:
                torch.cuda.synchronize(dev)
            t = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=dev)
            if not capturing:
                torch.cuda.synchronize(dev)
            _ws_cache[key] = t
        return t


def gqa_decode_num_splits(batch, T_q, S_kv, h_q, h_kv, d_head) -> int:
    return lib.gqa_decode_num_splits(batch, T_q, S_kv, h_q, h_kv, d_head)


def gqa_paged_plan(num_seqs, h_q, h_kv, d_head, max_seq_len, partition_size=0, *, block_size=16,
                   vllm_layout=False, head_group=0):
    """(partition_size, head_group, launches) a paged call with these shapes makes on the current device
    (partition_size 0 resolved to the automatic choice)."""
    opt = _opts(0, 0, paged_head_group=head_group)
    part, hg, launches = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    st = lib.gqa_paged_plan(num_seqs, h_q, h_kv, d_head, int(block_size), int(max_seq_len), int(partition_size),
                            1 if vllm_layout else 0, ctypes.byref(opt), ctypes.byref(part), ctypes.byref(hg),
                            ctypes.byref(launches))
    _check(st, "gqa_paged_plan")
    return part.value, hg.value, launches.value


KERNELS = {0: "split", 1: "split-cluster", 2: "split-deep-ring", 3: "tcgen05"}   # GQA_KERNEL_*
FOLDS = {0: "none", 1: "cluster", 2: "merge-kernel", 3: "last-cta"}                # GQA_FOLD_*


def gqa_decode_plan(batch, T_q, S_kv, h_q, h_kv, d_head, *, n_splits=0, merge_mode=0, mma_path=0, causal=False,
                    detail=False):
    """(n_splits, mma_path, launches) of a gqa_decode call with these shapes and options on the current
    device: mma_path 1 = mma.sync split kernel, 2 = tcgen05 kernel; launches 2 with the merge kernel.
    ``detail``: a dict with those and the kernel variant and fold (names from KERNELS and FOLDS)."""
    opt = _opts(n_splits, merge_mode, causal=causal, mma_path=mma_path)
    n, path, launches, kernel, fold = (ctypes.c_int(0) for _ in range(5))
    st = lib.gqa_decode_plan_ex(batch, T_q, S_kv, h_q, h_kv, d_head, ctypes.byref(opt), ctypes.byref(n),
                                ctypes.byref(path), ctypes.byref(launches), ctypes.byref(kernel), ctypes.byref(fold))
    _check(st, "gqa_decode_plan_ex")
    if detail:
        return {"n_splits": n.value, "mma_path": path.value, "launches": launches.value,
                "kernel": KERNELS[kernel.value], "fold": FOLDS[fold.value]}
    return n.value, path.value, launches.value


def gqa_decode_workspace_size(batch, T_q, S_kv, h_q, h_kv, d_head, n_splits=0) -> int:
    return lib.gqa_decode_workspace_size(batch, T_q, S_kv, h_q, h_kv, d_head, n_splits)


def gqa_workspace_size(batch, T_q, S_kv, h_q, h_kv, d_head) -> int:
    """Workspace bytes of a gqa_decode call with the automatic split count (0: invalid shape)."""
    return lib.gqa_workspace_size(batch, T_q, S_kv, h_q, h_kv, d_head)


def gqa_paged_workspace_size(num_seqs, h_q, h_kv, d_head, max_seq_len, partition_size=512) -> int:
    return lib.gqa_paged_workspace_size(num_seqs, h_q, h_kv, d_head, max_seq_len, partition_size)


def gqa_workspace_init(ws: torch.Tensor, stream=None) -> None:
    _check(lib.gqa_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "gqa_workspace_init")


def gqa_workspace_check(ws: torch.Tensor, stream=None) -> int:
    """Status word of the last calls on this workspace (synchronises ``stream``)."""
    return lib.gqa_workspace_check(_ptr(ws), _stream(stream))


# ---------------------------------------------------------------- calls
def _shape_qkv(q, k, v, h_q, h_kv):
    _h16(q, "q"), _h16(k, "k", q.dtype), _h16(v, "v", q.dtype)
    if q.dim() != 3 or k.dim() != 3 or k.shape != v.shape or k.shape[0] != q.shape[0]:
        raise ValueError("q must be (batch, T_q, h_q*d_head), k and v (batch, S_kv, h_kv*d_head)")
    B, T_q, qc = q.shape
    S = k.shape[1]
    if qc % h_q or k.shape[2] % h_kv or qc // h_q != k.shape[2] // h_kv:
        raise ValueError("inconsistent head sizes")
    return B, T_q, S, qc // h_q


def gqa_decode(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, h_q: int, h_kv: int,
               scale: Optional[float] = None, *, out: Optional[torch.Tensor] = None,
               workspace_tensor: Optional[torch.Tensor] = None, stream=None, n_splits: int = 0,
               merge_mode: int = 0, timeout_us: int = 0, test_stall_cta: int = -1,
               causal: bool = False, mma_path: int = 0) -> torch.Tensor:
    """O = softmax(scale Q K^T) V for GQA decode; q (B, T_q, h_q*D), k/v (B, S_kv, h_kv*D) float16 or
    bfloat16 (all the same; the output has that dtype too).
    ``causal``: query token t sees keys j <= S_kv - T_q + t only.
    ``mma_path``: 0 automatic, 1 the mma.sync split kernel (G*T_q <= 64), 2 the tcgen05 kernel
    (G*T_q <= 128).
    ``merge_mode``: 0 automatic, 1 separate merge kernel, 2 last-arriving CTA, 3 the splits of a
    (sequence, KV head) as one thread-block cluster (at most 16) merging in distributed shared memory."""
    B, T_q, S, D = _shape_qkv(q, k, v, h_q, h_kv)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    _h16(out, "out", q.dtype)
    nbytes = gqa_decode_workspace_size(B, T_q, S, h_q, h_kv, D, n_splits)
    if nbytes == 0:
        raise GQAError(GQA_ERR_INVALID_ARG, "gqa_decode_workspace_size")
    ws = workspace(nbytes, q.device, stream) if workspace_tensor is None else workspace_tensor
    opt = _opts(n_splits, merge_mode, timeout_us, test_stall_cta, causal=causal, bf16=q.dtype == torch.bfloat16,
                mma_path=mma_path)
    st = lib.gqa_decode_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, T_q, S, h_q, h_kv, D, scale,
                           _ptr(ws), ws.numel(), _stream(stream), ctypes.byref(opt))
    _check(st, "gqa_decode")
    return out


def gqa_decode_partial(q, k, v, h_q: int, h_kv: int, s_begin: int, s_len: int, scale: Optional[float] = None, *,
                       m=None, l=None, o_part=None, workspace_tensor=None, stream=None, n_splits: int = 0,
                       merge_mode: int = 0, causal: bool = False,
                       mma_path: int = 0) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Partial (m, l, O) over keys [s_begin, s_begin+s_len): m, l (B*T_q*h_q) and O (B*T_q*h_q, D) fp32."""
    B, T_q, S, D = _shape_qkv(q, k, v, h_q, h_kv)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    R = B * T_q * h_q
    dev = q.device
    m = torch.empty(R, dtype=torch.float32, device=dev) if m is None else m
    l = torch.empty(R, dtype=torch.float32, device=dev) if l is None else l
    o_part = torch.empty(R, D, dtype=torch.float32, device=dev) if o_part is None else o_part
    _f32(m, "m"), _f32(l, "l"), _f32(o_part, "o_part")
    nbytes = gqa_decode_workspace_size(B, T_q, max(int(s_len), 1), h_q, h_kv, D, n_splits)
    if nbytes == 0:
        raise GQAError(GQA_ERR_INVALID_ARG, "gqa_decode_workspace_size")
    ws = workspace(nbytes, dev, stream) if workspace_tensor is None else workspace_tensor
    opt = _opts(n_splits, merge_mode, causal=causal, bf16=q.dtype == torch.bfloat16, mma_path=mma_path)
    st = lib.gqa_decode_partial_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(m), _ptr(l), _ptr(o_part), B, T_q, S,
                                   int(s_begin), int(s_len), h_q, h_kv, D, scale, _ptr(ws), ws.numel(),
                                   _stream(stream), ctypes.byref(opt))
    _check(st, "gqa_decode_partial")
    return m, l, o_part


def gqa_merge(m: torch.Tensor, l: torch.Tensor, o_part: torch.Tensor, *, out=None, stream=None,
              dtype=torch.float16) -> torch.Tensor:
    """Merge partials m, l (n_parts, rows), o_part (n_parts, rows, D) into o (rows, D), float16 or
    bfloat16 (the dtype of ``out`` when given, else ``dtype``)."""
    _f32(m, "m"), _f32(l, "l"), _f32(o_part, "o_part")
    n_parts, rows, D = o_part.shape
    out = torch.empty(rows, D, dtype=dtype, device=o_part.device) if out is None else out
    _h16(out, "out")
    opt = _opts(bf16=out.dtype == torch.bfloat16)
    _check(lib.gqa_merge_ex(_ptr(m), _ptr(l), _ptr(o_part), n_parts, rows, D, _ptr(out), _stream(stream),
                            ctypes.byref(opt)), "gqa_merge")
    return out


def gqa_merge_partial(m, l, o_part, *, m_out=None, l_out=None, o_out=None, stream=None):
    """Merge partials into one partial (m, l, O), all fp32."""
    _f32(m, "m"), _f32(l, "l"), _f32(o_part, "o_part")
    n_parts, rows, D = o_part.shape
    dev = o_part.device
    m_out = torch.empty(rows, dtype=torch.float32, device=dev) if m_out is None else m_out
    l_out = torch.empty(rows, dtype=torch.float32, device=dev) if l_out is None else l_out
    o_out = torch.empty(rows, D, dtype=torch.float32, device=dev) if o_out is None else o_out
    _check(lib.gqa_merge_partial(_ptr(m), _ptr(l), _ptr(o_part), n_parts, rows, D, _ptr(m_out), _ptr(l_out),
                                 _ptr(o_out), _stream(stream)), "gqa_merge_partial")
    return m_out, l_out, o_out


def gqa_decode_paged(q, k_pool, v_pool, block_tables, seq_lens, h_q: int, h_kv: int, scale: Optional[float] = None,
                     *, max_seq_len: int, partition_size: int = 512, out=None, workspace_tensor=None,
                     stream=None, timeout_us: int = 0, test_stall_cta: int = -1,
                     head_group: int = 0) -> torch.Tensor:
    """Paged decode; q (N, h_q*D), pools (num_blocks, block_size, h_kv*D) float16 or bfloat16,
    tables (N, max_blocks) int32."""
    _h16(q, "q"), _h16(k_pool, "k_pool", q.dtype), _h16(v_pool, "v_pool", q.dtype)
    if not (block_tables.is_cuda and block_tables.dtype == torch.int32 and block_tables.is_contiguous()):
        raise ValueError("block_tables must be a contiguous int32 CUDA tensor")
    if not (seq_lens.is_cuda and seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()):
        raise ValueError("seq_lens must be a contiguous int32 CUDA tensor")
    q2 = q.reshape(q.shape[0], -1)
    N, qc = q2.shape
    num_blocks, block_size, kc = k_pool.shape
    if qc % h_q or kc % h_kv or qc // h_q != kc // h_kv or v_pool.shape != k_pool.shape:
        raise ValueError("inconsistent head sizes")
    D = qc // h_q
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    out = torch.empty_like(q2) if out is None else out
    _h16(out, "out", q.dtype)
    nbytes = gqa_paged_workspace_size(N, h_q, h_kv, D, max_seq_len, partition_size)
    if nbytes == 0:
        raise GQAError(GQA_ERR_INVALID_ARG, "gqa_paged_workspace_size")
    ws = workspace(nbytes, q.device, stream) if workspace_tensor is None else workspace_tensor
    opt = _opts(0, 0, timeout_us, test_stall_cta, head_group, bf16=q.dtype == torch.bfloat16)
    st = lib.gqa_decode_paged_ex(_ptr(q2), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(seq_lens),
                                 _ptr(out), N, block_tables.shape[1], num_blocks, block_size, partition_size,
                                 h_q, h_kv, D, scale, int(max_seq_len), _ptr(ws), ws.numel(), _stream(stream),
                                 ctypes.byref(opt))
    _check(st, "gqa_decode_paged")
    return out


def gqa_decode_paged_vllm(q, k_cache, v_cache, block_tables, seq_lens, h_q: int, h_kv: int,
                          scale: Optional[float] = None, *, max_seq_len: int, partition_size: int = 0, out=None,
                          workspace_tensor=None, stream=None, timeout_us: int = 0, test_stall_cta: int = -1,
                          head_group: int = 0) -> torch.Tensor:
    """Paged decode over vLLM's cache layout, read in place: q (N, h_q*D); k_cache
    (num_blocks, h_kv, D/8, block_size, 8), v_cache (num_blocks, h_kv, D, block_size), float16 or
    bfloat16; tables (N, max_blocks) int32.  partition_size 0: automatic (512-token partitions);
    partition_size >= max_seq_len: single pass (one launch)."""
    _h16(q, "q"), _h16(k_cache, "k_cache", q.dtype), _h16(v_cache, "v_cache", q.dtype)
    if not (block_tables.is_cuda and block_tables.dtype == torch.int32 and block_tables.is_contiguous()):
        raise ValueError("block_tables must be a contiguous int32 CUDA tensor")
    if not (seq_lens.is_cuda and seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()):
        raise ValueError("seq_lens must be a contiguous int32 CUDA tensor")
    q2 = q.reshape(q.shape[0], -1)
    N, qc = q2.shape
    if k_cache.dim() != 5 or k_cache.shape[4] != 8 or v_cache.dim() != 4:
        raise ValueError("k_cache must be (num_blocks, h_kv, D/8, block_size, 8), v_cache (num_blocks, h_kv, D, block_size)")
    num_blocks, hk, d8, block_size, _ = k_cache.shape
    D = d8 * 8
    if hk != h_kv or qc != h_q * D or tuple(v_cache.shape) != (num_blocks, h_kv, D, block_size):
        raise ValueError("inconsistent head sizes")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    out = torch.empty_like(q2) if out is None else out
    _h16(out, "out", q.dtype)
    nbytes = gqa_paged_workspace_size(N, h_q, h_kv, D, max_seq_len, partition_size)
    if nbytes == 0:
        raise GQAError(GQA_ERR_INVALID_ARG, "gqa_paged_workspace_size")
    ws = workspace(nbytes, q.device, stream) if workspace_tensor is None else workspace_tensor
    opt = _opts(0, 0, timeout_us, test_stall_cta, head_group, bf16=q.dtype == torch.bfloat16)
    st = lib.gqa_decode_paged_vllm_ex(_ptr(q2), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(seq_lens),
                                      _ptr(out), N, block_tables.shape[1], num_blocks, block_size, partition_size,
                                      h_q, h_kv, D, scale, int(max_seq_len), _ptr(ws), ws.numel(), _stream(stream),
                                      ctypes.byref(opt))
    _check(st, "gqa_decode_paged_vllm")
    return out


GQA_NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024


def gqa_decode_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, h_q: int, h_kv: int,
                       scale: Optional[float] = None, *, out: Optional[torch.Tensor] = None,
                       stream=None) -> torch.Tensor:
    """gqa_decode without a caller workspace: the library's own per-GPU device array is used.

    For callers that cannot allocate device memory.  Calls on one device share that array,
    so they must not overlap on the GPU; shapes needing more than 8 MiB of workspace raise."""
    B, T_q, S, D = _shape_qkv(q, k, v, h_q, h_kv)
    _f16(q, "q")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    _f16(out, "out")
    st = lib.gqa_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, T_q, S, h_q, h_kv, D, scale,
                                _stream(stream))
    _check(st, "gqa_decode_noalloc")
    return out


def gqa_decode_noalloc_check(stream=None) -> int:
    """Status of the gqa_decode_noalloc calls on the current device since the last check
    (synchronises ``stream``; GQA_OK or GQA_ERR_TIMEOUT); clears it."""
    return lib.gqa_decode_noalloc_check(_stream(stream))
