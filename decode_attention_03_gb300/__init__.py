"""GB300-native (sm_103a) GQA split-KV decode attention.

The compute lives in ``libgqa_decode.so`` (C ABI, ``include/gqa_decode.h``):
hand-written CUDA kernels for the split-KV partial pass (mma.sync with TMA, and
tcgen05 with tensor memory), the online-softmax merge of its splits (inside a
thread-block cluster, or a merge kernel), the paged (block-table) variant and the
standalone merge.
This package is the thin Python binding (``_binding``), loaded on first use of
any of its names; it raises if the library has not been built -- there is no
fallback path.  ``build`` compiles the library in-tree.
"""
from __future__ import annotations

import importlib

_BINDING_NAMES = (
    "gqa_decode", "gqa_decode_noalloc", "gqa_decode_noalloc_check", "gqa_decode_partial", "gqa_merge", "gqa_merge_partial", "gqa_decode_paged",
    "gqa_decode_paged_vllm",
    "gqa_decode_workspace_size", "gqa_workspace_size", "gqa_paged_workspace_size", "gqa_decode_num_splits",
    "gqa_decode_plan", "gqa_paged_plan",
    "gqa_workspace_init", "gqa_workspace_check", "gqa_status_string", "gqa_version",
    "GQAError", "gqa_options", "workspace", "lib", "LIB_PATH", "EXPORTED",
    "GQA_OK", "GQA_ERR_INVALID_ARG", "GQA_ERR_UNSUPPORTED", "GQA_ERR_WORKSPACE", "GQA_ERR_CUDA",
    "GQA_ERR_TIMEOUT", "GQA_ERR_BOUNDS", "GQA_BUILD_BOUNDS_CHECK", "GQA_NOALLOC_SCRATCH_BYTES", "open_library",
)

__all__ = list(_BINDING_NAMES)


def __getattr__(name):
    if name in _BINDING_NAMES:
        mod = importlib.import_module("._binding", __name__)
        return getattr(mod, name)
    raise AttributeError(name)
