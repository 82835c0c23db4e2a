"""The C-ABI library builds, loads and exports every declared symbol; host-side
validation returns the documented status codes without touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa_decode.h")


@pytest.fixture(scope="module")
def binding():
    from decode_attention_03_gb300 import build
    build.build()
    import decode_attention_03_gb300._binding as b
    return b


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(gqa_\w+)\s*\(", text)
    return sorted(set(n for n in names if not n.startswith("gqa_status\b")))


def test_header_declares_the_four_calls():
    names = declared_functions()
    for n in ("gqa_decode", "gqa_decode_partial", "gqa_merge", "gqa_decode_paged"):
        assert n in names


def test_every_declared_symbol_is_exported(binding):
    lib = ctypes.CDLL(binding.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding wraps each of them under the same name
    assert set(declared_functions()) == set(binding.EXPORTED)


def test_version_and_status_strings(binding):
    assert binding.gqa_version() == 10000
    for s in range(7):
        assert binding.gqa_status_string(s) != "unknown status"
    assert binding.lib.gqa_build_flags() == 0                       # the regular build checks no bounds
    assert binding.gqa_status_string(99) == "unknown status"


def test_default_options(binding):
    o = binding.lib.gqa_default_options()
    assert (o.n_splits, o.merge_mode, o.timeout_us, o.test_stall_cta, o.paged_head_group, o.causal) == \
        (0, 0, 0, -1, 0, 0)


def _fake(n=1 << 12):
    # host buffers standing in for device pointers: validation must reject before any access
    buf = ctypes.create_string_buffer(n + 64)
    addr = (ctypes.addressof(buf) + 15) & ~15
    return buf, ctypes.c_void_p(addr)


def test_validation_codes_without_gpu(binding):
    lib = binding.lib
    _b, p = _fake()
    st = ctypes.c_void_p(0)
    s = 1.0 / 8

    def dec(B=1, T=1, S=16, hq=8, hkv=2, d=64, ws=p, wsb=1 << 12, q=p):
        return lib.gqa_decode(q, p, p, p, B, T, S, hq, hkv, d, s, ws, wsb, st)

    assert dec(hq=6, hkv=4) == binding.GQA_ERR_INVALID_ARG          # h_q % h_kv != 0
    assert dec(d=96) == binding.GQA_ERR_UNSUPPORTED                 # d_head not in {64, 128}
    assert dec(hq=129, hkv=1) == binding.GQA_ERR_UNSUPPORTED         # G*T_q > 128
    assert dec(hq=16, hkv=1, T=9) == binding.GQA_ERR_UNSUPPORTED     # G*T_q = 144
    assert dec(S=0) == binding.GQA_ERR_INVALID_ARG                   # no keys
    assert dec(B=-1) == binding.GQA_ERR_INVALID_ARG
    assert dec(T=0) == binding.GQA_ERR_INVALID_ARG
    assert dec(q=None) == binding.GQA_ERR_INVALID_ARG                # null pointer
    assert dec(q=ctypes.c_void_p(p.value + 2)) == binding.GQA_ERR_INVALID_ARG   # misaligned
    # the plan query validates before it asks the device
    outs = [ctypes.c_int(-7) for _ in range(5)]
    assert lib.gqa_decode_plan_ex(1, 1, 0, 8, 2, 64, None, *(ctypes.byref(o) for o in outs)) == \
        binding.GQA_ERR_INVALID_ARG
    bad = binding._opts(merge_mode=4)
    assert lib.gqa_decode_plan_ex(1, 1, 16, 8, 2, 64, ctypes.byref(bad), *(ctypes.byref(o) for o in outs)) == \
        binding.GQA_ERR_INVALID_ARG
    assert all(o.value == -7 for o in outs)                          # nothing written on an error
    assert dec(B=0) == binding.GQA_OK                                # empty batch: no-op
    assert dec(B=2, S=(1 << 30)) == binding.GQA_ERR_INVALID_ARG      # batch*S_kv >= 2^31
    assert lib.gqa_decode(p, p, p, p, 1, 1, 16, 8, 2, 64, float("nan"), p, 4096, st) == binding.GQA_ERR_INVALID_ARG
    # the mma.sync path stops at 64 query rows per KV head; the tcgen05 path at 128
    def dec_path(path, T, hq=16, hkv=1):
        opt = binding.gqa_options(0, 0, 0, -1, 0, 0, 0, path)
        return lib.gqa_decode_ex(p, p, p, p, 1, T, 16, hq, hkv, 64, s, p, 1 << 12, st, ctypes.byref(opt))

    assert dec_path(1, 5) == binding.GQA_ERR_UNSUPPORTED             # G*T_q = 80 on mma.sync
    assert dec_path(2, 9) == binding.GQA_ERR_UNSUPPORTED             # G*T_q = 144
    assert dec_path(3, 1) == binding.GQA_ERR_INVALID_ARG             # no such path
    assert dec_path(-1, 1) == binding.GQA_ERR_INVALID_ARG
    # merge modes 0-3 only
    for mm in (-1, 4):
        opt = binding.gqa_options(0, mm, 0, -1, 0, 0)
        r = lib.gqa_decode_ex(p, p, p, p, 1, 1, 16, 8, 2, 64, s, p, 1 << 12, st, ctypes.byref(opt))
        assert r == binding.GQA_ERR_INVALID_ARG
    # workspace too small (forced split count: sized without a device)
    opt = binding.gqa_options(8, 0, 0, -1, 0, 0)
    need = lib.gqa_decode_workspace_size(1, 1, 4096, 8, 2, 64, 8)
    assert need > 256
    r = lib.gqa_decode_ex(p, p, p, p, 1, 1, 4096, 8, 2, 64, s, p, need - 1, st, ctypes.byref(opt))
    assert r == binding.GQA_ERR_WORKSPACE


def test_partial_and_merge_validation(binding):
    lib = binding.lib
    _b, p = _fake()
    st = ctypes.c_void_p(0)
    # s_begin + s_len beyond S_kv
    r = lib.gqa_decode_partial(p, p, p, p, p, p, 1, 1, 100, 90, 20, 8, 2, 64, 0.125, p, 4096, st)
    assert r == binding.GQA_ERR_INVALID_ARG
    r = lib.gqa_decode_partial(p, p, p, p, p, p, 1, 1, 100, -1, 20, 8, 2, 64, 0.125, p, 4096, st)
    assert r == binding.GQA_ERR_INVALID_ARG
    assert lib.gqa_merge(p, p, p, 0, 4, 64, p, st) == binding.GQA_ERR_INVALID_ARG       # n_parts < 1
    assert lib.gqa_merge(p, p, p, 2, 4, 80, p, st) == binding.GQA_ERR_UNSUPPORTED
    assert lib.gqa_merge(p, p, p, 2, 0, 64, p, st) == binding.GQA_OK                    # no rows
    assert lib.gqa_merge(None, p, p, 2, 4, 64, p, st) == binding.GQA_ERR_INVALID_ARG


def test_paged_validation(binding):
    lib = binding.lib
    _b, p = _fake()
    st = ctypes.c_void_p(0)

    def paged(bs=16, part=512, N=2, hq=8, hkv=2, d=128, maxlen=1000, maxblk=64, nblk=100, wsb=1 << 20):
        return lib.gqa_decode_paged(p, p, p, p, p, p, N, maxblk, nblk, bs, part, hq, hkv, d, 0.1, maxlen,
                                    p, wsb, st)

    assert paged(bs=12) == binding.GQA_ERR_INVALID_ARG
    assert paged(part=500) == binding.GQA_ERR_INVALID_ARG            # not a multiple of 64
    assert paged(bs=8, part=16384) == binding.GQA_ERR_INVALID_ARG    # > 1024 blocks per partition
    assert paged(part=-64) == binding.GQA_ERR_INVALID_ARG
    assert paged(d=256) == binding.GQA_ERR_UNSUPPORTED
    assert paged(maxlen=-1) == binding.GQA_ERR_INVALID_ARG
    assert paged(N=0) == binding.GQA_OK
    assert paged(wsb=255) == binding.GQA_ERR_WORKSPACE
    opt = binding.gqa_options(0, 0, 0, -1, 3, 0)                        # head group must be 1, 2 or 4
    assert lib.gqa_decode_paged_ex(p, p, p, p, p, p, 2, 64, 100, 16, 512, 8, 2, 128, 0.1, 1000, p, 1 << 20, st,
                                   ctypes.byref(opt)) == binding.GQA_ERR_INVALID_ARG
    opt = binding.gqa_options(0, 0, 0, -1, 4, 0)                        # ... and divide h_kv
    assert lib.gqa_decode_paged_ex(p, p, p, p, p, p, 2, 64, 100, 16, 512, 8, 2, 128, 0.1, 1000, p, 1 << 20, st,
                                   ctypes.byref(opt)) == binding.GQA_ERR_INVALID_ARG
    assert lib.gqa_paged_workspace_size(64, 32, 8, 128, 16384, 512) > 0
    assert lib.gqa_paged_workspace_size(64, 32, 8, 128, 16384, 500) == 0
    # partition 0 (automatic v1 / v2) is sized as v2 with 512-token partitions
    assert lib.gqa_paged_workspace_size(64, 32, 8, 128, 16384, 0) == lib.gqa_paged_workspace_size(64, 32, 8, 128,
                                                                                                16384, 512)


def test_paged_vllm_validation(binding):
    """The vLLM-layout entry point rejects bad shapes on the host, before any device access."""
    lib = binding.lib
    _b, p = _fake()
    st = ctypes.c_void_p(0)

    def paged(bs=16, part=0, N=2, hq=8, hkv=2, d=128, maxlen=1000, maxblk=64, nblk=100, wsb=1 << 20):
        return lib.gqa_decode_paged_vllm(p, p, p, p, p, p, N, maxblk, nblk, bs, part, hq, hkv, d, 0.1, maxlen,
                                         p, wsb, st)

    assert paged(bs=12) == binding.GQA_ERR_INVALID_ARG
    assert paged(part=500) == binding.GQA_ERR_INVALID_ARG
    assert paged(d=96) == binding.GQA_ERR_UNSUPPORTED
    assert paged(hq=9, hkv=2) == binding.GQA_ERR_INVALID_ARG          # h_q % h_kv
    assert paged(hq=130, hkv=1) == binding.GQA_ERR_UNSUPPORTED        # G > 64
    assert paged(N=0) == binding.GQA_OK
    assert paged(wsb=255) == binding.GQA_ERR_WORKSPACE
    assert paged(nblk=1 << 27, hkv=2, hq=8) == binding.GQA_ERR_INVALID_ARG   # blocks * h_kv * d/8 >= 2^31


def test_workspace_layout_sizes(binding):
    lib = binding.lib
    # one split: header + counters only; S splits: + S * R * (D + 2) fp32 partials (256-aligned)
    one = lib.gqa_decode_workspace_size(1, 1, 1 << 20, 32, 8, 128, 1)
    assert one == 256 + 256
    n = 38
    R = 32
    many = lib.gqa_decode_workspace_size(1, 1, 1 << 20, 32, 8, 128, n)
    al = lambda x: (x + 255) // 256 * 256
    assert many == 256 + 256 + 2 * al(n * R * 4) + al(n * R * 128 * 4)


def test_workspace_size_alias(binding):
    """gqa_workspace_size(batch, T_q, S_kv, h_q, h_kv, d_head) is the automatic-split size query."""
    assert binding.gqa_workspace_size(1, 1, 100, 8, 3, 128) == 0        # h_q % h_kv != 0
    assert binding.gqa_workspace_size(1, 1, 100, 8, 2, 96) == 0         # unsupported d_head
    for shape in [(1, 1, 4096, 8, 2, 64), (8, 1, 32768, 32, 8, 128), (1, 4, 131071, 64, 8, 128)]:
        assert binding.gqa_workspace_size(*shape) == binding.gqa_decode_workspace_size(*shape, 0)
