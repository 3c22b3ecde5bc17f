"""The seeded input generators: determinism and the structure each workload promises."""
import numpy as np
import pytest

import workloads as W


def test_same_seed_same_inputs():
    a, b = W.make_config(2, B=4, ctx_lo=20, ctx_hi=200), W.make_config(2, B=4, ctx_lo=20, ctx_hi=200)
    for f in ("q", "k_pool", "v_pool", "block_tables", "context_lens", "slot_mapping", "k_new"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    c = W.make_config(2, seed=99, B=4, ctx_lo=20, ctx_hi=200)
    assert not np.array_equal(a.q, c.q)


@pytest.mark.parametrize("cfg", [1, 2, 4, 5])
def test_tables_are_shuffled_unique_blocks(cfg):
    kw = {} if cfg == 1 else dict(B=6, ctx_lo=16, ctx_hi=200)
    w = W.make_config(cfg, **kw)
    used = w.block_tables[w.block_tables >= 0]
    assert used.max() < w.NB
    if w.shared_prefix_blocks == 0:
        assert len(np.unique(used)) == len(used)  # no block referenced twice
        assert (w.ref_count[used] == 1).all()
    # every context token has a table entry, and none beyond the context
    for b in range(w.B):
        nblk = -(-int(w.context_lens[b]) // 16)
        assert (w.block_tables[b, :nblk] >= 0).all() and (w.block_tables[b, nblk:] < 0).all()
    # the new token's slot is the sequence's last logical position
    for b in range(w.B):
        n = int(w.context_lens[b])
        assert w.slot_mapping[b] == w.block_tables[b, (n - 1) // 16] * 16 + (n - 1) % 16


def test_tiny_config_matches_its_description():
    w = W.make_config(1)
    assert list(w.context_lens) == [1, 17, 33, 100]
    assert (w.Hq, w.Hkv, w.D, w.NB, w.kv_dtype, w.scale) == (4, 4, 64, 64, "f32", 0.125)


def test_prefix_shared_refcounts():
    w = W.make_config(5, B=7, ctx_lo=16, ctx_hi=64, prefix_tokens=128)
    pre = w.block_tables[:, :8]
    assert (pre == pre[0]).all()
    assert (w.ref_count[pre[0]] == 7).all()
    c = W.unshare_prefix(w)
    assert c.ref_count.max() == 1 and c.NB == w.NB + 7 * 8
    for b in range(w.B):
        for j in range(8):
            np.testing.assert_array_equal(c.k_pool[c.block_tables[b, j]], w.k_pool[pre[0, j]])


def test_permutation_moves_data_consistently():
    w = W.make_config(4, B=3, ctx_lo=17, ctx_hi=90)
    p = W.permute_blocks(w, seed=5)
    for b in range(w.B):
        for j in range(-(-int(w.context_lens[b]) // 16)):
            np.testing.assert_array_equal(p.k_pool[p.block_tables[b, j]], w.k_pool[w.block_tables[b, j]])
            np.testing.assert_array_equal(p.v_scales[p.block_tables[b, j]], w.v_scales[w.block_tables[b, j]])
    assert (p.slot_mapping // 16 == p.block_tables[np.arange(w.B), (w.context_lens - 1) // 16]).all()


def test_int8_input_recipe_round_trip():
    x = np.random.default_rng(0).standard_normal((50, 128)).astype(np.float32)
    qv, s = W.quantize_int8_rows(x)
    assert np.abs(qv).max() <= 127
    err = np.abs(qv.astype(np.float64) * s[:, None] - x)
    assert (err <= s[:, None] * 0.5 * (1 + 1e-6)).all()


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 1e-3], np.float32)
    bits = W.f32_to_bf16_bits(vals)
    back = W.bf16_bits_to_f32(bits)
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == 1.0 + 2**-6 and back[3] == -2.5
    assert abs(back[4] - 1e-3) <= 1e-3 * 2**-8


def test_dead_slot_map_on_a_hand_made_table():
    """The dead-slot rule the GPU sentinel tests fill with NaN: two sequences sharing block 0,
    lengths 20 and 16."""
    from _gpu import dead_slots
    bt = np.array([[0, 2, -1], [0, -1, -1]], dtype=np.int32)
    dead = dead_slots(bt, np.array([20, 16]), NB=4, BS=16)
    assert not dead[0].any()                       # full, shared
    assert not dead[2, :4].any() and dead[2, 4:].all()
    assert dead[1].all() and dead[3].all()         # referenced by no table
