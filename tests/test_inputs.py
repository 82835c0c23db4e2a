"""The seeded input generators: frozen draws and workload structure (CPU only)."""
import numpy as np

import gqa_inputs as gi


def test_regression_constants():
    # first draws of three streams, frozen: any change to the convention fails here
    a = gi.normal_f16(0, 0, (1, 8)).astype(np.float32).tolist()[0]
    assert a == [1.1171875, -1.38671875, -0.426513671875, -0.8037109375, 0.6015625,
                 -0.07501220703125, 0.0596923828125, -0.032012939453125]
    b = gi.normal_f16(2, 1, (2, 4)).astype(np.float32).tolist()
    assert b == [[0.37646484375, 1.755859375, -0.72705078125, 1.2490234375],
                 [0.2021484375, -0.09527587890625, 0.09918212890625, 1.5087890625]]
    c = gi.uniform_f16(4, 2, (1, 6)).astype(np.float32).tolist()[0]
    assert c == [-0.42529296875, 0.2236328125, 0.62646484375, 0.443115234375,
                 -0.26953125, -0.69189453125]


def test_chunking_is_thread_independent():
    rows = gi.CHUNK_ROWS + 77
    x = gi.normal_f16(9, 1, (rows, 4))
    # chunk c depends only on (seed, stream, c): the second chunk equals a fresh draw of it
    g = gi._gen(9, 1, 1)
    tail = g.standard_normal((77, 4), dtype=np.float32).astype(np.float16)
    assert np.array_equal(x[gi.CHUNK_ROWS:], tail)


def test_paged_layout_structure():
    w = gi.WORKLOADS["paged"]
    lens, tab, nb = gi.paged_layout(w)
    assert lens.shape == (64,) and lens.min() >= 1024 and lens.max() <= 16384
    assert lens[:4].tolist() == [5867, 2603, 5602, 5938]
    nblk = (lens.astype(np.int64) + 15) // 16
    assert nb == int(nblk.sum())
    used = np.concatenate([tab[b, :nblk[b]] for b in range(64)])
    assert np.array_equal(np.sort(used), np.arange(nb))          # every pool block used exactly once
    for b in range(64):
        assert (tab[b, nblk[b]:] == -1).all()


def test_ragged_spikes():
    w = gi.custom(1, 4, 1000, 16, 2, 8, 4, v_dist="uniform", spike_frac=0.01, spike_mult=8.0)
    x = gi.make_contiguous(w)
    assert len(x["spike_rows"]) == 10
    assert x["v"].min() >= -1.0 and x["v"].max() <= 1.0
    base = gi.normal_f16(4, gi.S_K, (1, 1000, 16))
    assert np.array_equal(x["k"][0, x["spike_rows"]], base[0, x["spike_rows"]] * np.float16(8))


def test_workloads_match_stated_shapes():
    W = gi.WORKLOADS
    assert (W["tiny"].S_kv, W["tiny"].h_q, W["tiny"].h_kv, W["tiny"].d_head) == (4096, 8, 2, 64)
    assert (W["llama8b"].batch, W["llama8b"].S_kv, W["llama8b"].G) == (8, 32768, 4)
    assert W["long"].S_kv == 1 << 20 and W["long"].G == 4
    assert (W["ragged"].T_q, W["ragged"].S_kv, W["ragged"].G) == (4, 131071, 8)
    assert W["paged"].block_size == 16 and W["paged"].partition_size == 512


def test_bf16_draws_round_the_same_float32_values():
    # the bfloat16 workload rounds the very float32 draws the float16 workload rounds
    f32 = gi._gen(7, 1, 0).standard_normal((3, 5), dtype=np.float32)
    b = gi.normal_f16(7, 1, (3, 5), elem="bf16")
    assert b.dtype == np.uint16
    assert np.array_equal(b, gi.f32_to_bf16(f32))
    back = gi.bf16_to_f32(b)
    assert np.all(np.abs(back - f32) <= np.abs(f32) * 2.0 ** -8)
    # round to nearest even on exact ties
    ties = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8], dtype=np.float32)
    assert gi.bf16_to_f32(gi.f32_to_bf16(ties)).tolist() == [1.0, 1.0 + 2.0 ** -6]
