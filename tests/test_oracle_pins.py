"""Pins of the CPU oracle to things other than itself (CPU only).

Each ``pin_*`` function checks the oracle module passed to it against a fact
fixed by the mathematics or by an independent library routine and returns
``True`` when it holds.  The tests run every pin on the real oracle; the
mutation tests at the end plant plausible mistakes in copies of the oracle
(a dropped scale, a wrong head mapping, K reshaped instead of transposed, a
sign flip or a dropped term in the merge, a missing normalise, an unshifted
exp, an off-by-one paged gather) and check that some pin catches each one.

Passages pinned (page "kernbench2 ... _gqa_attention_decode_long.py"): the
tile math (scores, row max, exp, row sum, exp@V), ``_merge_running``, the
final ``O / l``; (page "muh_kernel_map.py", ``paged_attention_v1/v2``): the
paged KV cache addressed through block tables.
"""
from __future__ import annotations

import math
import os
import types

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import gqa_inputs
import oracle
from oracle import gqa_oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _close(a, b, tol=1e-12) -> bool:
    a = torch.as_tensor(np.asarray(a, dtype=np.float64)) if not torch.is_tensor(a) else a
    b = torch.as_tensor(np.asarray(b, dtype=np.float64)) if not torch.is_tensor(b) else b
    if a.shape != b.shape:
        return False
    if not torch.isfinite(a).all():
        return False
    return bool(((a - b).abs() <= tol * (1.0 + b.abs())).all())


def _inputs(B, T_q, S, h_q, h_kv, D, seed):
    w = gqa_inputs.custom(B, T_q, S, h_q, h_kv, D, seed)
    return gqa_inputs.make_contiguous(w)


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

def brute_force(q, k, v, h_q, h_kv, D, scale):
    """Triple loop in plain Python floats with math.exp: the definition itself."""
    B, T_q, _ = q.shape
    S = k.shape[1]
    G = h_q // h_kv
    out = np.zeros((B, T_q, h_q * D))
    for b in range(B):
        for t in range(T_q):
            for h in range(h_q):
                g = h // G
                s = []
                for j in range(S):
                    acc = 0.0
                    for d in range(D):
                        acc += float(q[b, t, h * D + d]) * float(k[b, j, g * D + d])
                    s.append(scale * acc)
                mx = max(s)
                p = [math.exp(x - mx) for x in s]
                tot = sum(p)
                for d in range(D):
                    num = 0.0
                    for j in range(S):
                        num += p[j] * float(v[b, j, g * D + d])
                    out[b, t, h * D + d] = num / tot
    return out


def pin_brute_force(orc) -> bool:
    ok = True
    for (B, T_q, S, h_q, h_kv, D, seed) in [(2, 2, 7, 4, 2, 4, 11), (1, 1, 5, 3, 1, 3, 12),
                                            (1, 2, 8, 4, 4, 2, 13), (2, 1, 1, 2, 1, 4, 14)]:
        x = _inputs(B, T_q, S, h_q, h_kv, D, seed)
        scale = 0.37
        ref = brute_force(x["q"], x["k"], x["v"], h_q, h_kv, D, scale)
        got = orc.decode(x["q"], x["k"], x["v"], h_q, h_kv, D, scale)
        ok &= _close(got, ref)
    return ok


def pin_sdpa(orc) -> bool:
    """GQA reduces to PyTorch's scaled_dot_product_attention with
    ``enable_gqa`` (float64, no mask): pins the scale, K's transpose and the
    head mapping ``h -> h // G``."""
    ok = True
    for (B, T_q, S, h_q, h_kv, D, seed) in [(2, 3, 37, 8, 2, 16, 21), (1, 4, 129, 16, 2, 8, 22),
                                            (3, 1, 50, 6, 3, 4, 23)]:
        x = _inputs(B, T_q, S, h_q, h_kv, D, seed)
        scale = 1.0 / math.sqrt(D)
        q = torch.from_numpy(x["q"]).double().view(B, T_q, h_q, D).permute(0, 2, 1, 3)
        k = torch.from_numpy(x["k"]).double().view(B, S, h_kv, D).permute(0, 2, 1, 3)
        v = torch.from_numpy(x["v"]).double().view(B, S, h_kv, D).permute(0, 2, 1, 3)
        ref = F.scaled_dot_product_attention(q, k, v, scale=scale, enable_gqa=True)
        ref = ref.permute(0, 2, 1, 3).reshape(B, T_q, h_q * D)
        got = orc.decode(x["q"], x["k"], x["v"], h_q, h_kv, D, scale)
        ok &= _close(got, ref, 1e-11)
    return ok


def pin_constant_scores(orc) -> bool:
    """K = 0 (or Q = 0): every score is 0, the output is the mean of V."""
    x = _inputs(2, 2, 33, 8, 2, 8, 31)
    k0 = np.zeros_like(x["k"])
    got = orc.decode(x["q"], k0, x["v"], 8, 2, 8, 0.5)
    mean_v = x["v"].astype(np.float64).mean(axis=1)              # (B, h_kv*D)
    ref = np.empty((2, 2, 8 * 8))
    for h in range(8):
        ref[:, :, h * 8:(h + 1) * 8] = mean_v[:, None, (h // 4) * 8:(h // 4 + 1) * 8]
    q0 = np.zeros_like(x["q"])
    got2 = orc.decode(q0, x["k"], x["v"], 8, 2, 8, 0.5)
    return _close(got, ref) and _close(got2, ref)


def pin_one_hot(orc) -> bool:
    """A key with a logit gap >= 40 over all others returns its V row
    (to within S * exp(-40))."""
    B, T_q, S, h_q, h_kv, D = 1, 1, 64, 1, 1, 16
    x = _inputs(B, T_q, S, h_q, h_kv, D, 41)
    q = x["q"].astype(np.float64)
    k = x["k"].astype(np.float64) * 0.01
    jstar = 37
    qn = q[0, 0] / np.linalg.norm(q[0, 0])
    k[0, jstar] = 64.0 * qn
    scale = 1.0
    s = scale * (k[0] @ q[0, 0])
    gap = s[jstar] - np.max(np.delete(s, jstar))
    assert gap >= 40
    got = orc.decode(q, k, x["v"], h_q, h_kv, D, scale)
    ref = x["v"].astype(np.float64)[0, jstar]
    return _close(got[0, 0], ref, S * math.exp(-40) * 10)


def pin_single_key(orc) -> bool:
    """S_kv = 1: the output is that key's V row, whatever Q and K are."""
    x = _inputs(2, 3, 1, 8, 4, 8, 51)
    got = orc.decode(x["q"], x["k"], x["v"], 8, 4, 8, 0.125)
    v = x["v"].astype(np.float64)[:, 0]                          # (B, h_kv*D)
    ref = np.empty((2, 3, 64))
    for h in range(8):
        ref[:, :, h * 8:(h + 1) * 8] = v[:, None, (h // 2) * 8:(h // 2 + 1) * 8]
    return _close(got, ref)


def pin_split_merge(orc) -> bool:
    """Any split of the key range, merged with the page's merge and then
    normalised, equals the unsplit result (including size-1 and empty splits)."""
    B, T_q, S, h_q, h_kv, D = 2, 2, 100, 8, 2, 8
    x = _inputs(B, T_q, S, h_q, h_kv, D, 61)
    scale = 0.3
    full = orc.decode(x["q"], x["k"], x["v"], h_q, h_kv, D, scale)
    ok = True
    for cuts in ([0, 1, 2, 50, 99, 100], [0, 37, 37, 100], [0, 100], [0, 10, 20, 30, 40, 100]):
        ms, ls, os_ = [], [], []
        for a, b in zip(cuts[:-1], cuts[1:]):
            m, l, o = orc.decode_partial(x["q"], x["k"], x["v"], h_q, h_kv, D, scale, a, b - a)
            ms.append(m), ls.append(l), os_.append(o)
        m, l, o = orc.merge_parts(ms, ls, os_)
        got = orc.normalize(l, o).reshape(B, T_q, h_q * D)
        ok &= _close(got, full)
    # one unit (sequence b, KV head g) over a key range is the slice of the all-rows partial
    G = h_q // h_kv
    mp, lp, op = orc.decode_partial(x["q"], x["k"], x["v"], h_q, h_kv, D, scale, 13, 41)
    for b in range(B):
        for g in range(h_kv):
            mu, lu, ou = orc.decode_unit(x["q"], x["k"], x["v"], b, g, h_q, h_kv, D, scale, 13, 41)
            ok &= _close(mu, mp[b, :, g * G:(g + 1) * G]) and _close(lu, lp[b, :, g * G:(g + 1) * G])
            ok &= _close(ou, op[b, :, g * G:(g + 1) * G])
    return ok


def pin_merge_closed_form(orc) -> bool:
    """Two single-key partials ``(s_a, 1, v_a)`` and ``(s_b, 1, v_b)`` merge to
    the two-key softmax: weights ``1/(1+e^(s_b-s_a))`` and the complement."""
    ok = True
    for sa, sb in [(0.0, math.log(3.0)), (5.0, -2.0), (-60.0, 60.0), (1.5, 1.5)]:
        va = torch.tensor([[1.0, -2.0, 4.0]], dtype=torch.float64)
        vb = torch.tensor([[3.0, 5.0, -1.0]], dtype=torch.float64)
        f64 = torch.float64
        m, l, o = orc.merge_pair(torch.tensor([sa], dtype=f64), torch.ones(1, dtype=f64), va,
                                 torch.tensor([sb], dtype=f64), torch.ones(1, dtype=f64), vb)
        wa = 1.0 / (1.0 + math.exp(sb - sa))
        ref = wa * va + (1.0 - wa) * vb
        ok &= _close(orc.normalize(l, o), ref) and abs(float(m[0]) - max(sa, sb)) == 0.0
        # empty partials contribute nothing; two empties stay empty
        e_m = torch.tensor([float("-inf")], dtype=f64)
        e_l, e_o = torch.zeros(1, dtype=f64), torch.zeros(1, 3, dtype=f64)
        m2, l2, o2 = orc.merge_pair(e_m, e_l, e_o, m, l, o)
        ok &= _close(orc.normalize(l2, o2), ref)
        m3, l3, o3 = orc.merge_pair(e_m, e_l, e_o, e_m, e_l, e_o)
        ok &= bool(torch.isneginf(m3).all()) and float(l3[0]) == 0.0 and bool((o3 == 0).all())
    return ok


def pin_empty(orc) -> bool:
    """Empty key ranges (reading R7 of the pages' merge): an empty partial is (-inf, 0, 0),
    normalising l = 0 gives exactly 0 while the other rows are still divided by their l, an
    all-empty merge normalises to 0, and a length-0 paged sequence has an all-zero output
    (its neighbours unchanged)."""
    f64 = torch.float64
    ok = True
    # closed form, mixed rows: O / l where l > 0, exactly 0 where l = 0
    l = torch.tensor([2.0, 0.0, 4.0], dtype=f64)
    o = torch.tensor([[2.0, -4.0], [0.0, 0.0], [4.0, 8.0]], dtype=f64)
    got = orc.normalize(l, o)
    ok &= _close(got, torch.tensor([[1.0, -2.0], [0.0, 0.0], [1.0, 2.0]], dtype=f64), 0.0)
    # an empty key range through the partial path
    x = _inputs(1, 2, 9, 4, 2, 8, 131)
    m, l0, o0 = orc.decode_partial(x["q"], x["k"], x["v"], 4, 2, 8, 0.5, 3, 0)
    ok &= bool(torch.isneginf(m).all()) and bool((l0 == 0).all()) and bool((o0 == 0).all())
    ok &= _close(orc.normalize(l0, o0), torch.zeros(1, 2, 4, 8, dtype=f64), 0.0)
    # merging only empty partials, then normalising: zeros
    mm, lm, om = orc.merge_parts([m, m, m], [l0, l0, l0], [o0, o0, o0])
    ok &= _close(orc.normalize(lm, om), torch.zeros(1, 2, 4, 8, dtype=f64), 0.0)
    # a length-0 paged sequence among non-empty ones
    w = gqa_inputs.custom(3, 1, 40, 4, 2, 8, 132, kind="paged", block_size=8, partition_size=64,
                          len_lo=1, len_hi=40)
    p = gqa_inputs.make_paged(w)
    lens = p["seq_lens"].copy()
    lens[1] = 0
    one = orc.decode_paged_seq(p["q"], p["k_pool"], p["v_pool"], p["block_tables"], lens, 1, 4, 2, 8, 0.3, 8)
    ok &= _close(one, torch.zeros(1, 4 * 8, dtype=f64), 0.0)
    allp = orc.decode_paged(p["q"], p["k_pool"], p["v_pool"], p["block_tables"], lens, 4, 2, 8, 0.3, 8)
    ok &= _close(allp[1], torch.zeros(1, 4 * 8, dtype=f64), 0.0)
    for b in (0, 2):
        L = int(lens[b])
        kb = orc.gather_paged(p["k_pool"], p["block_tables"][b], L, 8)[None]
        vb = orc.gather_paged(p["v_pool"], p["block_tables"][b], L, 8)[None]
        ok &= _close(allp[b], orc.decode(p["q"][b:b + 1].reshape(1, 1, -1), kb, vb, 4, 2, 8, 0.3)[0])
    return ok


def pin_permutation(orc) -> bool:
    """Permuting the key rows (K and V together) leaves the output unchanged;
    permuting the query tokens permutes the output rows."""
    B, T_q, S, h_q, h_kv, D = 1, 3, 80, 4, 2, 8
    x = _inputs(B, T_q, S, h_q, h_kv, D, 71)
    base = orc.decode(x["q"], x["k"], x["v"], h_q, h_kv, D, 0.4)
    perm = np.random.Generator(np.random.PCG64(5)).permutation(S)
    got = orc.decode(x["q"], x["k"][:, perm], x["v"][:, perm], h_q, h_kv, D, 0.4)
    tp = [2, 0, 1]
    got_t = orc.decode(x["q"][:, tp], x["k"], x["v"], h_q, h_kv, D, 0.4)
    return _close(got, base) and _close(got_t, base[:, tp])


def pin_shift(orc) -> bool:
    """Adding a constant to every logit of a row leaves the output unchanged
    and shifts m by that constant (large shifts exercise the max subtraction)."""
    D, S = 16, 50
    x = _inputs(1, 1, S, 1, 1, D, 81)
    q = x["q"][0].astype(np.float64)                      # (1, D)
    k = x["k"][0].astype(np.float64)
    v = x["v"][0].astype(np.float64)
    scale = 0.25
    m0, l0, o0 = orc.partial_rows(q, k, v, scale)
    ok = True
    for c in (1000.0, -1000.0, 60.0):
        k2 = k + (c / scale) * q / float((q @ q.T)[0, 0])    # s_j -> s_j + c
        m1, l1, o1 = orc.partial_rows(q, k2, v, scale)
        ok &= _close(orc.normalize(l1, o1), orc.normalize(l0, o0), 1e-9)
        ok &= abs(float(m1[0]) - float(m0[0]) - c) < 1e-9 * (1 + abs(c))
    return ok


def pin_paged(orc) -> bool:
    """Paged = contiguous on the gathered rows; shuffling the pool's blocks
    (table remapped) or NaN in the unused tail slots changes nothing."""
    w = gqa_inputs.custom(5, 1, 100, 8, 2, 8, 91, kind="paged", block_size=16, partition_size=64,
                          len_lo=1, len_hi=100)
    p = gqa_inputs.make_paged(w)
    lens, tab, bs = p["seq_lens"], p["block_tables"], 16
    got = orc.decode_paged(p["q"], p["k_pool"], p["v_pool"], tab, lens, 8, 2, 8, 0.3, bs)
    ok = True
    for b in range(5):
        L = int(lens[b])
        kb = np.stack([p["k_pool"][tab[b, j // bs], j % bs] for j in range(L)])[None]
        vb = np.stack([p["v_pool"][tab[b, j // bs], j % bs] for j in range(L)])[None]
        ref = orc.decode(p["q"][b:b + 1], kb, vb, 8, 2, 8, 0.3)
        ok &= _close(got[b:b + 1], ref)
    nb = p["num_blocks"]
    perm = np.random.Generator(np.random.PCG64(6)).permutation(nb)     # new position of block i
    kp2 = np.empty_like(p["k_pool"]); kp2[perm] = p["k_pool"]
    vp2 = np.empty_like(p["v_pool"]); vp2[perm] = p["v_pool"]
    tab2 = np.where(tab >= 0, perm[np.clip(tab, 0, None)], -1).astype(np.int32)
    got2 = orc.decode_paged(p["q"], kp2, vp2, tab2, lens, 8, 2, 8, 0.3, bs)
    ok &= _close(got2, got)
    pn = gqa_inputs.make_paged(w, tail_fill="nan")
    got3 = orc.decode_paged(pn["q"], pn["k_pool"], pn["v_pool"], tab, lens, 8, 2, 8, 0.3, bs)
    ok &= _close(got3, got)
    return ok


def pin_paged_vllm(orc) -> bool:
    """vLLM's cache layout (key cache [blocks, h_kv, D/x, block, x], x = 8; value cache
    [blocks, h_kv, D, block]) holding the same keys and values as a row pool gives the same
    output: the caches are filled here element by element from the layout statement."""
    w = gqa_inputs.custom(4, 1, 70, 8, 2, 16, 93, kind="paged", block_size=8, partition_size=64,
                          len_lo=1, len_hi=70)
    p = gqa_inputs.make_paged(w)
    kp, vp, lens, tab = p["k_pool"], p["v_pool"], p["seq_lens"], p["block_tables"]
    nb, bs, h_kv, D, x = p["num_blocks"], 8, 2, 16, 8
    kc = np.empty((nb, h_kv, D // x, bs, x), dtype=kp.dtype)
    vc = np.empty((nb, h_kv, D, bs), dtype=vp.dtype)
    for n in range(nb):
        for slot in range(bs):
            for g in range(h_kv):
                for dd in range(D):
                    kc[n, g, dd // x, slot, dd % x] = kp[n, slot, g * D + dd]
                    vc[n, g, dd, slot] = vp[n, slot, g * D + dd]
    rows = orc.decode_paged(p["q"], kp, vp, tab, lens, 8, 2, D, 0.3, bs)
    got = orc.decode_paged(p["q"], kc, vc, tab, lens, 8, 2, D, 0.3, bs, layout="vllm")
    ok = True
    for b in range(4):   # the gathered rows themselves, key by key, from the layout statement
        L = int(lens[b])
        kg, vg = orc.gather_paged_vllm(kc, vc, tab[b], L, bs)
        kr = np.stack([kp[tab[b, j // bs], j % bs] for j in range(L)])
        vr = np.stack([vp[tab[b, j // bs], j % bs] for j in range(L)])
        ok &= np.array_equal(kg, kr) and np.array_equal(vg, vr)
    k2, v2 = gqa_inputs.to_vllm_layout(kp, vp, h_kv, D)      # the input module's rearrangement agrees
    return ok and _close(got, rows) and np.array_equal(k2, kc) and np.array_equal(v2, vc)


def pin_causal(orc) -> bool:
    """Causal tail (token t of T_q sees keys j <= S - T_q + t): equals PyTorch SDPA with the
    explicit bottom-right mask, equals the plain decode of each token over its visible
    prefix, and is the plain decode when T_q = 1."""
    ok = True
    for (B, T_q, S, h_q, h_kv, D, seed) in [(2, 4, 37, 8, 2, 16, 121), (1, 3, 5, 4, 1, 8, 122)]:
        x = _inputs(B, T_q, S, h_q, h_kv, D, seed)
        scale = 1.0 / math.sqrt(D)
        got = orc.decode(x["q"], x["k"], x["v"], h_q, h_kv, D, scale, causal=True)
        q = torch.from_numpy(x["q"]).double().view(B, T_q, h_q, D).permute(0, 2, 1, 3)
        k = torch.from_numpy(x["k"]).double().view(B, S, h_kv, D).permute(0, 2, 1, 3)
        v = torch.from_numpy(x["v"]).double().view(B, S, h_kv, D).permute(0, 2, 1, 3)
        mask = torch.arange(S)[None, :] <= (S - T_q + torch.arange(T_q))[:, None]
        ref = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale, enable_gqa=True)
        ok &= _close(got, ref.permute(0, 2, 1, 3).reshape(B, T_q, h_q * D), 1e-11)
        for t in range(T_q):
            hi = S - T_q + t + 1
            one = orc.decode(x["q"][:, t:t + 1], x["k"][:, :hi], x["v"][:, :hi], h_q, h_kv, D, scale)
            ok &= _close(got[:, t:t + 1], one)
    x = _inputs(2, 1, 20, 4, 2, 8, 123)
    ok &= _close(orc.decode(x["q"], x["k"], x["v"], 4, 2, 8, 0.3, causal=True),
                 orc.decode(x["q"], x["k"], x["v"], 4, 2, 8, 0.3))
    return ok


def pin_golden(orc) -> bool:
    """Hand-worked examples under ``tests/golden/``."""
    ok = True
    for fn in sorted(os.listdir(GOLDEN)):
        if not fn.endswith(".txt"):
            continue
        case = _read_golden(os.path.join(GOLDEN, fn))
        if case["kind"] == "decode":
            got = orc.decode(case["q"], case["k"], case["v"], case["h_q"], case["h_kv"],
                             case["d_head"], case["scale"])
            ok &= _close(got.reshape(-1), case["expect"].reshape(-1), 1e-13)
        elif case["kind"] == "merge":
            m, l, o = orc.merge_pair(case["m_a"], case["l_a"], case["o_a"],
                                     case["m_b"], case["l_b"], case["o_b"])
            ok &= _close(m, case["expect_m"], 1e-13) and _close(l, case["expect_l"], 1e-13)
            ok &= _close(orc.normalize(l, o).reshape(-1), case["expect"].reshape(-1), 1e-13)
    return ok


def _read_golden(path: str) -> dict:
    """Plain ``key: values`` text; ``#`` starts a comment."""
    out = {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = line.split(":", 1)
            key, val = key.strip(), val.strip()
            if key == "kind":
                out[key] = val
            elif key == "shape":
                out[key] = [int(x) for x in val.split()]
            elif key in ("h_q", "h_kv", "d_head"):
                out[key] = int(val)
            elif key == "scale":
                out[key] = float(val)
            else:
                out[key] = np.array([float(x) for x in val.split()], dtype=np.float64)
    if out["kind"] == "decode":
        B, T_q, S = out["shape"]
        out["q"] = out["q"].reshape(B, T_q, out["h_q"] * out["d_head"])
        out["k"] = out["k"].reshape(B, S, out["h_kv"] * out["d_head"])
        out["v"] = out["v"].reshape(B, S, out["h_kv"] * out["d_head"])
    else:
        for key in ("o_a", "o_b"):
            out[key] = out[key].reshape(1, -1)
    return out


PINS = [pin_brute_force, pin_sdpa, pin_constant_scores, pin_one_hot, pin_single_key,
        pin_split_merge, pin_merge_closed_form, pin_empty, pin_permutation, pin_shift, pin_paged, pin_paged_vllm, pin_causal,
        pin_golden]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin_holds(pin):
    assert pin(gqa_oracle)


def test_every_exported_function_is_pinned():
    """Each function the oracle exports is called by name in at least one pin."""
    import inspect
    src = "\n".join(inspect.getsource(p) for p in PINS)
    missing = [n for n in oracle.__all__ if f"orc.{n}(" not in src]
    assert not missing, f"oracle functions no pin calls: {missing}"
    assert sorted(oracle.__all__) == sorted(gqa_oracle.__all__)


def test_golden_files_present():
    names = [f for f in os.listdir(GOLDEN) if f.endswith(".txt")]
    assert len(names) >= 2


# ---------------------------------------------------------------------------
# planted mistakes: each must be caught by at least one pin
# ---------------------------------------------------------------------------

def _mutant(**overrides):
    """A copy of the oracle module with some functions replaced."""
    mod = types.ModuleType("oracle_mutant")
    mod.__dict__.update(gqa_oracle.__dict__)
    for name, fn in overrides.items():
        mod.__dict__[name] = types.FunctionType(fn.__code__, mod.__dict__, name,
                                                fn.__defaults__, fn.__closure__)
    # re-bind every original function to the mutant namespace so internal calls see the mutation
    for name, obj in list(gqa_oracle.__dict__.items()):
        if isinstance(obj, types.FunctionType) and name not in overrides and obj.__module__ == gqa_oracle.__name__:
            mod.__dict__[name] = types.FunctionType(obj.__code__, mod.__dict__, name,
                                                    obj.__defaults__, obj.__closure__)
    return mod


def _m_no_scale(q_rows, k_rows, v_rows, scale):
    q, k, v = _f64(q_rows), _f64(k_rows), _f64(v_rows)
    if k.shape[0] == 0:
        n, D = q.shape
        return torch.full((n,), NEG_INF, dtype=torch.float64), torch.zeros(n, dtype=torch.float64), torch.zeros(n, D, dtype=torch.float64)
    s = q @ k.T
    m = s.max(dim=1).values
    p = torch.exp(s - m[:, None])
    return m, p.sum(dim=1), p @ v


def _m_reshape_k(q_rows, k_rows, v_rows, scale):
    q, k, v = _f64(q_rows), _f64(k_rows), _f64(v_rows)
    if k.shape[0] == 0:
        n, D = q.shape
        return torch.full((n,), NEG_INF, dtype=torch.float64), torch.zeros(n, dtype=torch.float64), torch.zeros(n, D, dtype=torch.float64)
    s = float(scale) * (q @ k.reshape(k.shape[1], k.shape[0]))
    m = s.max(dim=1).values
    p = torch.exp(s - m[:, None])
    return m, p.sum(dim=1), p @ v


def _m_no_shift(q_rows, k_rows, v_rows, scale):
    q, k, v = _f64(q_rows), _f64(k_rows), _f64(v_rows)
    if k.shape[0] == 0:
        n, D = q.shape
        return torch.full((n,), NEG_INF, dtype=torch.float64), torch.zeros(n, dtype=torch.float64), torch.zeros(n, D, dtype=torch.float64)
    s = float(scale) * (q @ k.T)
    m = s.max(dim=1).values
    p = torch.exp(s)
    return m, p.sum(dim=1), p @ v


def _m_head_mod(q, b, g, T_q, G, D):
    h_kv = q.shape[2] // (G * D)
    heads = [g + i * h_kv for i in range(G)]
    rows = np.stack([q[b, :, h * D:(h + 1) * D] for h in heads], axis=1)
    return np.asarray(rows).reshape(T_q * G, D)


def _m_merge_sign(m_a, l_a, o_a, m_b, l_b, o_b):
    m_a, l_a, o_a = _f64(m_a), _f64(l_a), _f64(o_a)
    m_b, l_b, o_b = _f64(m_b), _f64(l_b), _f64(o_b)
    m_new = torch.maximum(m_a, m_b)
    ref = torch.where(torch.isneginf(m_new), torch.zeros_like(m_new), m_new)
    so = torch.exp(ref - m_a)
    sn = torch.exp(m_b - ref)
    return m_new, l_a * so + l_b * sn, o_a * so[..., None] + o_b * sn[..., None]


def _m_merge_drop_l(m_a, l_a, o_a, m_b, l_b, o_b):
    m_a, l_a, o_a = _f64(m_a), _f64(l_a), _f64(o_a)
    m_b, l_b, o_b = _f64(m_b), _f64(l_b), _f64(o_b)
    m_new = torch.maximum(m_a, m_b)
    ref = torch.where(torch.isneginf(m_new), torch.zeros_like(m_new), m_new)
    so = torch.exp(m_a - ref)
    sn = torch.exp(m_b - ref)
    return m_new, l_a * so, o_a * so[..., None] + o_b * sn[..., None]


def _m_no_normalize(l, o):
    return _f64(o)


def _m_normalize_nan_when_empty(l, o):
    l, o = _f64(l), _f64(o)
    return o / l[..., None]


def _m_vllm_chunk_swap(k_cache, v_cache, table_row, length, block_size):
    # reads the key's d as (x, D/x) instead of (D/x, x)
    kc, vc = np.asarray(k_cache), np.asarray(v_cache)
    _, h_kv, dx, _, x = kc.shape
    j = np.arange(int(length))
    blocks = np.asarray(table_row)[j // block_size]
    slots = j % block_size
    k = kc[blocks, :, :, slots, :].transpose(0, 1, 3, 2)
    v = vc[blocks, :, :, slots]
    return k.reshape(len(j), h_kv * dx * x), v.reshape(len(j), h_kv * dx * x)


def _m_vllm_v_transposed(k_cache, v_cache, table_row, length, block_size):
    # takes the value cache as [blocks, h_kv, block, D] (the key's slot-major order)
    kc, vc = np.asarray(k_cache), np.asarray(v_cache)
    _, h_kv, dx, bs, x = kc.shape
    j = np.arange(int(length))
    blocks = np.asarray(table_row)[j // block_size]
    slots = j % block_size
    k = kc[blocks, :, :, slots, :]
    vr = vc.reshape(vc.shape[0], h_kv, bs, dx * x)
    v = vr[blocks, :, slots, :]
    return k.reshape(len(j), h_kv * dx * x), v.reshape(len(j), h_kv * dx * x)


def _m_gather_off_by_one(pool, table_row, length, block_size):
    j = np.arange(int(length))
    blocks = np.asarray(table_row)[j // block_size]
    slots = (j + 1) % block_size
    return np.asarray(pool)[blocks, slots]


def _m_causal_off_by_one(q, k, v, b, g, h_q, h_kv, D, scale, s_begin=0, s_len=None, causal=False):
    B, T_q, _ = q.shape
    S = k.shape[1]
    G = h_q // h_kv
    if s_len is None:
        s_len = S - s_begin
    qr = _unit_rows(q, b, g, T_q, G, D)
    m = torch.empty(T_q, G, dtype=torch.float64)
    l = torch.empty(T_q, G, dtype=torch.float64)
    o = torch.empty(T_q, G, D, dtype=torch.float64)
    for t in range(T_q):
        hi = s_begin + s_len if not causal else max(s_begin, min(s_begin + s_len, S - T_q + t))
        mt, lt, ot = partial_rows(qr[t * G:(t + 1) * G], k[b, s_begin:hi, g * D:(g + 1) * D],
                                  v[b, s_begin:hi, g * D:(g + 1) * D], scale)
        m[t], l[t], o[t] = mt, lt, ot
    return m, l, o


MUTANTS = {
    "no_scale": dict(partial_rows=_m_no_scale),
    "k_reshaped_not_transposed": dict(partial_rows=_m_reshape_k),
    "exp_without_max_shift": dict(partial_rows=_m_no_shift),
    "head_mapping_h_mod_hkv": dict(_unit_rows=_m_head_mod),
    "merge_sign_flip": dict(merge_pair=_m_merge_sign),
    "merge_drops_l_term": dict(merge_pair=_m_merge_drop_l),
    "no_normalize": dict(normalize=_m_no_normalize),
    "normalize_nan_for_empty_rows": dict(normalize=_m_normalize_nan_when_empty),
    "paged_slot_off_by_one": dict(gather_paged=_m_gather_off_by_one),
    "vllm_key_chunk_order_swapped": dict(gather_paged_vllm=_m_vllm_chunk_swap),
    "vllm_value_transposed": dict(gather_paged_vllm=_m_vllm_v_transposed),
    "causal_limit_off_by_one": dict(decode_unit=_m_causal_off_by_one),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    mod = _mutant(**MUTANTS[name])
    caught = [p.__name__ for p in PINS if not _safe(p, mod)]
    assert caught, f"mutant {name} passed every pin"


def _safe(pin, mod) -> bool:
    try:
        with np.errstate(all="ignore"):
            return bool(pin(mod))
    except Exception:
        return False


# these names are referenced by the mutant bodies (resolved in the mutant namespace)
_f64 = gqa_oracle._f64
NEG_INF = gqa_oracle.NEG_INF
_unit_rows = gqa_oracle._unit_rows
partial_rows = gqa_oracle.partial_rows
