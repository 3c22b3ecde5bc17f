"""Pins of the fp64 oracle to facts fixed outside itself (CPU only).

Each test targets a plausible mistake: a dropped softmax term or normalisation (one token,
identical keys), a wrong sign / base / missing scale in the exponent (two-key logistic), a
transposed or mis-indexed gather (permutation, library comparison, one-hot keys), a wrong GQA
head map, a wrong bf16 decode, a wrong INT8 scale index, a wrong merge weight.
"""
import math

import numpy as np
import pytest

import workloads as W

F64_TOL = 1e-12


def _pool_from_contiguous(K, V, perm_seed=None):
    """Lay contiguous per-sequence K/V [B, n, Hkv, D] (all n equal) into a 16-token block pool
    with either identity or shuffled block tables. Built here, independently of workloads."""
    B, n, Hkv, D = K.shape
    BS = 16
    nb = -(-n // BS)
    NB = B * nb
    ids = np.arange(NB, dtype=np.int32)
    if perm_seed is not None:
        ids = np.random.default_rng(perm_seed).permutation(NB).astype(np.int32)
    bt = ids.reshape(B, nb)
    kp = np.zeros((NB, Hkv, BS, D), K.dtype)
    vp = np.zeros((NB, Hkv, BS, D), V.dtype)
    for b in range(B):
        for t in range(n):
            kp[bt[b, t // BS], :, t % BS, :] = K[b, t]
            vp[bt[b, t // BS], :, t % BS, :] = V[b, t]
    return kp, vp, bt, np.full(B, n, np.int32)


def test_bf16_bit_patterns(orc):
    cases = {0x3F80: 1.0, 0xC000: -2.0, 0x3E80: 0.25, 0x0000: 0.0, 0x3F81: 1.0 + 2.0 ** -7,
             0x4049: 3.140625, 0x0001: 2.0 ** -133, 0x7F7F: (2 - 2.0 ** -7) * 2.0 ** 127}
    for bits, val in cases.items():
        assert orc.bf16_to_double(bits) == val, hex(bits)
    assert math.isinf(orc.bf16_to_double(0x7F80))
    assert math.copysign(1.0, orc.bf16_to_double(0x8000)) == -1.0


@pytest.mark.parametrize("kv", ["f32", "bf16", "i8"])
def test_single_token_returns_v(orc, kv):
    """context_len 1: softmax over one score is exactly 1, so out = v_0."""
    w = W.make_decode(name="t", B=3, Hq=4, Hkv=2, D=64, context_lens=[1, 1, 1], kv_dtype=kv,
                      q_dtype="f32" if kv == "f32" else "bf16", seed=7)
    out = orc.paged_decode_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                     w.scale, w.k_scales, w.v_scales)
    for b in range(w.B):
        blk = w.block_tables[b, 0]
        for h in range(w.Hq):
            v = w.v_pool[blk, h // 2, 0]
            if kv == "bf16":
                v = W.bf16_bits_to_f32(v).astype(np.float64)
            elif kv == "i8":
                v = v.astype(np.float64) * np.float64(w.v_scales[blk, h // 2, 0])
            np.testing.assert_array_equal(out[b, h], np.asarray(v, np.float64))


def test_identical_keys_give_mean_of_v(orc):
    """All keys equal -> uniform weights -> out = mean_t v_t."""
    rng = np.random.default_rng(3)
    B, n, Hkv, D = 2, 37, 2, 64
    K = np.broadcast_to(rng.standard_normal((1, 1, Hkv, D)), (B, n, Hkv, D)).astype(np.float32)
    V = rng.standard_normal((B, n, Hkv, D)).astype(np.float32)
    kp, vp, bt, cl = _pool_from_contiguous(K, V, perm_seed=1)
    q = rng.standard_normal((B, 4, D)).astype(np.float32)
    out = orc.paged_decode_attention(q, kp, vp, bt, cl, 0.125)
    for b in range(B):
        for h in range(4):
            np.testing.assert_allclose(out[b, h], V[b, :, h // 2].astype(np.float64).mean(0),
                                       rtol=0, atol=F64_TOL)


def test_two_key_logistic_weights(orc):
    """Keys e_0 and 0, query a*e_0: scores scale*a and 0, so the weight of key 0 is the
    logistic 1 / (1 + exp(-scale*a)) (natural base, scale applied once)."""
    D = 64
    K = np.zeros((1, 2, 1, D), np.float32)
    K[0, 0, 0, 0] = 1.0
    V = np.zeros((1, 2, 1, D), np.float32)
    V[0, 0, 0, :] = np.arange(D)
    V[0, 1, 0, :] = -1.0
    kp, vp, bt, cl = _pool_from_contiguous(K, V)
    for a, scale in [(2.0, 0.5), (3.0, 1.0 / 8.0), (-4.0, 0.25)]:
        q = np.zeros((1, 1, D), np.float32)
        q[0, 0, 0] = a
        out = orc.paged_decode_attention(q, kp, vp, bt, cl, scale)
        w0 = 1.0 / (1.0 + math.exp(-scale * a))
        expect = w0 * np.arange(D) + (1.0 - w0) * -1.0
        np.testing.assert_allclose(out[0, 0], expect, rtol=0, atol=F64_TOL)


def test_one_hot_keys_select_value(orc):
    """Orthogonal keys and a query aligned with key j at a large scale: out -> v_j."""
    D, n = 64, 40
    K = np.zeros((1, n, 1, D), np.float32)
    for t in range(n):
        K[0, t, 0, t] = 1.0
    V = np.random.default_rng(5).standard_normal((1, n, 1, D)).astype(np.float32)
    kp, vp, bt, cl = _pool_from_contiguous(K, V, perm_seed=4)
    for j in (0, 15, 16, 39):
        q = np.zeros((1, 1, D), np.float32)
        q[0, 0, j] = 1.0
        out = orc.paged_decode_attention(q, kp, vp, bt, cl, 60.0)
        # every other weight is exp(-60) relative: far below the tolerance
        np.testing.assert_allclose(out[0, 0], V[0, j, 0], rtol=0, atol=1e-20)


def test_gqa_head_map_is_contiguous_groups(orc):
    """Hq=8, Hkv=2: query heads 0-3 read kv head 0 and 4-7 read kv head 1."""
    D, n = 64, 20
    rng = np.random.default_rng(9)
    K = rng.standard_normal((1, n, 2, D)).astype(np.float32)
    V = np.empty((1, n, 2, D), np.float32)
    V[:, :, 0, :] = 1.0
    V[:, :, 1, :] = 2.0
    kp, vp, bt, cl = _pool_from_contiguous(K, V)
    q = rng.standard_normal((1, 8, D)).astype(np.float32)
    out = orc.paged_decode_attention(q, kp, vp, bt, cl, 0.125)
    for h in range(8):
        np.testing.assert_allclose(out[0, h], np.full(D, 1.0 + h // 4), rtol=0, atol=F64_TOL)


@pytest.mark.parametrize("g,D,n", [(1, 64, 1), (4, 128, 33), (2, 64, 100), (8, 128, 47)])
def test_matches_library_attention_on_contiguous_kv(orc, g, D, n):
    """Against torch's scaled_dot_product_attention in float64 on CPU (a library routine the
    oracle does not use), with the K/V laid out through shuffled block tables."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(g * 1000 + n)
    B, Hkv = 3, 2
    Hq = Hkv * g
    K = rng.standard_normal((B, n, Hkv, D)).astype(np.float32)
    V = rng.standard_normal((B, n, Hkv, D)).astype(np.float32)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    kp, vp, bt, cl = _pool_from_contiguous(K, V, perm_seed=n)
    scale = 1.0 / math.sqrt(D)
    out = orc.paged_decode_attention(q, kp, vp, bt, cl, scale)
    tq = torch.from_numpy(q.astype(np.float64)).unsqueeze(2)             # [B, Hq, 1, D]
    tk = torch.from_numpy(K.astype(np.float64)).permute(0, 2, 1, 3)      # [B, Hkv, n, D]
    tv = torch.from_numpy(V.astype(np.float64)).permute(0, 2, 1, 3)
    tk = tk.repeat_interleave(g, dim=1)
    tv = tv.repeat_interleave(g, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)
    np.testing.assert_allclose(out, ref[:, :, 0].numpy(), rtol=0, atol=1e-12)


def test_block_permutation_is_bit_identical(orc):
    w = W.make_config(2, B=4, ctx_lo=40, ctx_hi=300)
    p = W.permute_blocks(w, seed=77)
    assert not np.array_equal(w.block_tables, p.block_tables)
    a = orc.paged_decode_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens, w.scale)
    b = orc.paged_decode_attention(p.q, p.k_pool, p.v_pool, p.block_tables, p.context_lens, p.scale)
    assert np.array_equal(a, b)


def test_shared_prefix_equals_copy_on_write(orc):
    w = W.make_config(5, B=5, ctx_lo=16, ctx_hi=70, prefix_tokens=64)
    assert (w.ref_count[w.block_tables[0, :4]] == 5).all()
    c = W.unshare_prefix(w)
    assert c.ref_count.max() == 1
    a = orc.paged_decode_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens, w.scale)
    b = orc.paged_decode_attention(c.q, c.k_pool, c.v_pool, c.block_tables, c.context_lens, c.scale)
    assert np.array_equal(a, b)


def test_int8_dequant_uses_per_token_scales(orc):
    """Two tokens; K zero so weights are 1/2 each; out = (v0*s0 + v1*s1) / 2 with each token's
    own V scale (a wrong scale index -- K's, or the other token's -- fails)."""
    D = 64
    kp = np.zeros((2, 1, 16, D), np.int8)
    vp = np.zeros((2, 1, 16, D), np.int8)
    vp[1, 0, 0, :] = np.arange(D) - 32
    vp[0, 0, 0, :] = 7
    ks = np.full((2, 1, 16), 3.0, np.float32)
    vs = np.zeros((2, 1, 16), np.float32)
    vs[1, 0, 0] = 0.5
    vs[0, 0, 0] = 0.25
    bt = np.array([[1, 0]], np.int32)  # token 0 -> block 1, token 16 -> block 0
    cl = np.array([17], np.int32)
    q = W.f32_to_bf16_bits(np.ones((1, 1, D), np.float32))
    # tokens 1..15 of block 1 are zero K and zero V with scale 0: they carry weight too
    out = orc.paged_decode_attention(q, kp, vp, bt, cl, 1.0, ks, vs)
    expect = ((np.arange(D) - 32) * 0.5 + 7 * 0.25) / 17.0
    np.testing.assert_allclose(out[0, 0], expect, rtol=0, atol=F64_TOL)


def test_int8_scores_use_each_tokens_k_scale(orc):
    """Two tokens with int8 K codes 1 and 2 under K scales 0.05 and 0.01 and V codes 10 and -10
    under V scales 0.1 and 0.2: scores are 64 * 0.05 / 8 = 0.4 and 64 * 0.02 / 8 = 0.16, so the
    output is the two-key logistic mix w * 1.0 + (1 - w) * (-2.0) with w = 1 / (1 + e^-0.24).
    Dequantising K with the V scales (or V with the K scales) gives other scores or values."""
    D = 64
    kp = np.zeros((1, 1, 16, D), np.int8)
    vp = np.zeros((1, 1, 16, D), np.int8)
    kp[0, 0, 0, :], kp[0, 0, 1, :] = 1, 2
    vp[0, 0, 0, :], vp[0, 0, 1, :] = 10, -10
    ks = np.zeros((1, 1, 16), np.float32)
    vs = np.zeros((1, 1, 16), np.float32)
    ks[0, 0, :2] = [0.05, 0.01]
    vs[0, 0, :2] = [0.1, 0.2]
    q = W.f32_to_bf16_bits(np.ones((1, 1, D), np.float32))
    out = orc.paged_decode_attention(q, kp, vp, np.array([[0]], np.int32), np.array([2], np.int32),
                                     1.0 / 8.0, ks, vs)
    s0 = D * float(np.float32(0.05)) / 8.0
    s1 = D * 2 * float(np.float32(0.01)) / 8.0
    w = 1.0 / (1.0 + math.exp(-(s0 - s1)))
    expect = w * 10 * float(np.float32(0.1)) + (1.0 - w) * (-10) * float(np.float32(0.2))
    np.testing.assert_allclose(out[0, 0], expect, rtol=0, atol=F64_TOL)


def test_context_len_zero_gives_zeros(orc):
    w = W.make_decode(name="z", B=3, Hq=2, Hkv=1, D=64, context_lens=[0, 5, 0], kv_dtype="f32",
                      q_dtype="f32", seed=1)
    out = orc.paged_decode_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens, w.scale)
    assert np.all(out[0] == 0) and np.all(out[2] == 0) and np.all(np.isfinite(out))
    assert np.any(out[1] != 0)


@pytest.mark.parametrize("chunk", [16, 48, 64, 256, 512])
def test_split_merge_equals_unsplit(orc, chunk):
    w = W.make_config(2, B=5, ctx_lo=1, ctx_hi=700, seed=11)
    w.context_lens[0] = 0
    maxn = w.max_context_len
    S = max(1, maxn // chunk)
    m, l, acc, ns = orc.paged_decode_partials(w.q, w.k_pool, w.v_pool, w.block_tables,
                                              w.context_lens, w.scale, chunk, S)
    merged = orc.merge_partials(m, l, acc, ns)
    full = orc.paged_decode_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens, w.scale)
    np.testing.assert_allclose(merged, full, rtol=1e-12, atol=1e-13)
    for b, n in enumerate(w.context_lens):
        assert ns[b] == orc.split_count(n, chunk, S)[0]


def test_split_rule_closed_forms(orc):
    """split_num = max(1, n // chunk) from the FlashDecoding notes, whole blocks per split,
    no empty split, capped by the grid extent."""
    assert orc.split_count(0, 512, 8) == (1, 0)
    assert orc.split_count(100, 512, 8) == (1, 112)
    assert orc.split_count(511, 512, 8) == (1, 512)
    assert orc.split_count(512, 512, 8) == (1, 512)
    assert orc.split_count(2560, 512, 8) == (5, 512)
    assert orc.split_count(2561, 512, 8) == (5, 528)
    assert orc.split_count(131072, 512, 256) == (256, 512)
    assert orc.split_count(131072, 512, 64) == (64, 2048)  # capped
    for n in range(1, 400):
        for chunk in (16, 32, 48, 256):
            ns, per = orc.split_count(n, chunk, 1 << 20)
            assert per % 16 == 0 and per > 0
            assert ns <= max(1, n // chunk)
            assert (ns - 1) * per < n <= ns * per  # covers [0, n), last split non-empty


def test_kv_write_hand_offsets(orc):
    """Slot s goes to block s // 16, row s % 16 of every kv head; nothing else changes;
    negative slots are skipped; out-of-range slots are reported."""
    NB, Hkv, BS, D = 4, 2, 16, 64
    sentinel = np.float32(-777.0)
    kp = np.full((NB, Hkv, BS, D), sentinel, np.float32)
    vp = np.full((NB, Hkv, BS, D), sentinel, np.float32)
    kn = np.arange(3 * Hkv * D, dtype=np.float32).reshape(3, Hkv, D)
    vn = -kn
    slots = np.array([17, -1, 63], np.int64)
    k2, v2, _, _ = orc.kv_cache_write(kn, vn, kp, vp, slots)
    flat_k = k2.reshape(-1)
    row = lambda blk, h, off: ((blk * Hkv + h) * BS + off) * D  # noqa: E731
    np.testing.assert_array_equal(flat_k[row(1, 0, 1):row(1, 0, 1) + D], kn[0, 0])
    np.testing.assert_array_equal(flat_k[row(1, 1, 1):row(1, 1, 1) + D], kn[0, 1])
    np.testing.assert_array_equal(flat_k[row(3, 1, 15):row(3, 1, 15) + D], kn[2, 1])
    changed = np.argwhere(np.any(k2 != sentinel, axis=-1))
    assert sorted(map(tuple, changed)) == [(1, 0, 1), (1, 1, 1), (3, 0, 15), (3, 1, 15)]
    np.testing.assert_array_equal(v2[1, :, 1], vn[0])
    with pytest.raises(RuntimeError, match="slot"):
        orc.kv_cache_write(kn, vn, kp, vp, np.array([0, 64, 1], np.int64))


def test_kv_write_int8_moves_scales(orc):
    NB, Hkv, BS, D = 2, 1, 16, 64
    kp = np.zeros((NB, Hkv, BS, D), np.int8)
    vp = np.zeros_like(kp)
    ks = np.zeros((NB, Hkv, BS), np.float32)
    vs = np.zeros_like(ks)
    kn = np.full((1, Hkv, D), 5, np.int8)
    vn = np.full((1, Hkv, D), -3, np.int8)
    k2, v2, ks2, vs2 = orc.kv_cache_write(kn, vn, kp, vp, np.array([20], np.int64),
                                          np.array([[0.5]], np.float32),
                                          np.array([[0.25]], np.float32), ks, vs)
    assert (k2[1, 0, 4] == 5).all() and (v2[1, 0, 4] == -3).all()
    assert ks2[1, 0, 4] == 0.5 and vs2[1, 0, 4] == 0.25
    assert np.count_nonzero(ks2) == 1 and np.count_nonzero(k2) == D


def test_write_then_attend_sees_new_token(orc):
    """Ordering: the step writes the new token, then attends over context_lens that count it."""
    w = W.make_config(1)
    kp, vp, _, _ = orc.kv_cache_write(w.k_new, w.v_new, w.k_pool, w.v_pool, w.slot_mapping)
    out = orc.paged_decode_attention(w.q, kp, vp, w.block_tables, w.context_lens, w.scale)
    # sequence 0 has one token: the new one
    np.testing.assert_array_equal(out[0], w.v_new[0].astype(np.float64))


# ---- quantising INT8 write (EchoLLMServing notes, section 3: per-token scale) -------------------

def test_quantize_rounds_half_to_even_at_unit_scale(orc):
    """amax 127 makes the scale exactly 1, so codes are rint(x): halves go to the even code."""
    x = np.zeros((1, 64), np.float32)
    vals = [127.0, -127.0, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5, 126.5, 0.0]
    x[0, :len(vals)] = vals
    codes, scale = orc.quantize_rows_int8(x)
    assert scale[0] == 1.0
    assert list(codes[0, :len(vals)]) == [127, -127, 2, 4, -2, 0, 2, 0, 126, 0]


def test_quantize_zero_row_and_power_of_two_scaling(orc):
    codes, scale = orc.quantize_rows_int8(np.zeros((1, 128), np.float32))
    assert scale[0] == 1.0 and not codes.any()
    x = np.random.default_rng(2).standard_normal((6, 128)).astype(np.float32)
    c0, s0 = orc.quantize_rows_int8(x)
    for k in (-3, 5):  # a power-of-two factor scales the scale exactly and leaves the codes
        c1, s1 = orc.quantize_rows_int8((x * np.float32(2.0 ** k)).astype(np.float32))
        assert np.array_equal(c0, c1) and np.array_equal(s1, s0 * np.float32(2.0 ** k))


def test_quantize_error_bound_and_extremes(orc):
    x = np.random.default_rng(4).standard_normal((50, 128)).astype(np.float32) * 3
    codes, scale = orc.quantize_rows_int8(x)
    err = np.abs(codes.astype(np.float64) * scale[:, None] - x)
    assert (err <= scale[:, None].astype(np.float64) * (0.5 + 1e-5)).all()
    amax_at = np.argmax(np.abs(x), axis=1)
    assert (np.abs(codes[np.arange(50), amax_at]) == 127).all()
    assert codes.min() >= -127


def test_quantize_matches_generator_recipe_bit_exact(orc):
    """The numpy input recipe (workloads) is an independent statement of the same rule."""
    x = np.random.default_rng(6).standard_normal((40, 128)).astype(np.float32)
    c_np, s_np = W.quantize_int8_rows(x)
    c_or, s_or = orc.quantize_rows_int8(x)
    assert np.array_equal(c_np, c_or) and np.array_equal(s_np, s_or)
    xb = W.f32_to_bf16_bits(x)  # bf16 source rows widen exactly before quantising
    c_b, s_b = orc.quantize_rows_int8(xb)
    c_n2, s_n2 = W.quantize_int8_rows(W.bf16_bits_to_f32(xb))
    assert np.array_equal(c_b, c_n2) and np.array_equal(s_b, s_n2)


def test_kv_write_quant_places_rows_like_the_copy_write(orc):
    NB, Hkv, BS, D = 3, 2, 16, 64
    kn = np.random.default_rng(8).standard_normal((2, Hkv, D)).astype(np.float32)
    vn = -kn
    slots = np.array([20, 47], np.int64)
    kp = np.zeros((NB, Hkv, BS, D), np.int8)
    ks = np.zeros((NB, Hkv, BS), np.float32)
    k2, v2, ks2, vs2 = orc.kv_cache_write_quant(kn, vn, kp, kp.copy(), ks, ks.copy(), slots)
    c, sc = orc.quantize_rows_int8(kn)
    assert np.array_equal(k2[1, :, 4], c[0]) and np.array_equal(ks2[1, :, 4], sc[0])
    assert np.array_equal(k2[2, :, 15], c[1]) and np.array_equal(ks2[2, :, 15], sc[1])
    assert np.array_equal(v2[1, :, 4], -c[0])
    assert np.count_nonzero(ks2) == 4


# ---- multi-token decode (ATOM page, section 4: num_new_tokens = mtp_k + 1) ------------------------

def test_multi_token_with_one_token_is_decode(orc):
    w = W.make_config(2, B=3, ctx_lo=20, ctx_hi=200, seed=3)
    m = W.make_multi_token(w, 1, seed=5)
    a = orc.paged_decode_attention_multi(m.q, m.k_pool, m.v_pool, m.block_tables, m.context_lens, m.scale)
    b = orc.paged_decode_attention(m.q[:, 0], m.k_pool, m.v_pool, m.block_tables, m.context_lens, m.scale)
    assert np.array_equal(a[:, 0], b)


def test_multi_token_is_causal_over_the_new_tokens(orc):
    """Query token l sees exactly the first n - (L - 1 - l) tokens: changing the rows after that
    leaves it unchanged, and token l equals a plain decode with that context length."""
    L = 4
    w = W.make_config(2, B=3, ctx_lo=30, ctx_hi=90, seed=9)
    m = W.make_multi_token(w, L, seed=2)
    base = orc.paged_decode_attention_multi(m.q, m.k_pool, m.v_pool, m.block_tables, m.context_lens, m.scale)
    for l in range(L):
        cut = m.context_lens - (L - 1 - l)
        ref = orc.paged_decode_attention(m.q[:, l], m.k_pool, m.v_pool, m.block_tables, cut, m.scale)
        assert np.array_equal(base[:, l], ref)
    # perturb the last new token of sequence 0: only its own query (l = L - 1) may change
    kp = m.k_pool.copy()
    t = int(m.context_lens[0]) - 1
    kp[m.block_tables[0, t // 16], :, t % 16, :] ^= np.uint16(0x4000)
    pert = orc.paged_decode_attention_multi(m.q, kp, m.v_pool, m.block_tables, m.context_lens, m.scale)
    assert np.array_equal(pert[0, :L - 1], base[0, :L - 1]) and not np.array_equal(pert[0, L - 1], base[0, L - 1])
    assert np.array_equal(pert[1:], base[1:])


def test_multi_token_matches_library_masked_attention(orc):
    """Against torch scaled_dot_product_attention (fp64, CPU) with an explicit causal mask."""
    torch = pytest.importorskip("torch")
    L, n, D, Hkv, g = 3, 40, 64, 2, 2
    rng = np.random.default_rng(12)
    K = rng.standard_normal((2, n, Hkv, D)).astype(np.float32)
    V = rng.standard_normal((2, n, Hkv, D)).astype(np.float32)
    q = rng.standard_normal((2, L, Hkv * g, D)).astype(np.float32)
    kp, vp, bt, cl = _pool_from_contiguous(K, V, perm_seed=7)
    out = orc.paged_decode_attention_multi(q, kp, vp, bt, cl, 0.125)
    tq = torch.from_numpy(q.astype(np.float64)).permute(0, 2, 1, 3)                  # [B, Hq, L, D]
    tk = torch.from_numpy(K.astype(np.float64)).permute(0, 2, 1, 3).repeat_interleave(g, 1)
    tv = torch.from_numpy(V.astype(np.float64)).permute(0, 2, 1, 3).repeat_interleave(g, 1)
    mask = torch.tensor([[t <= n - L + l for t in range(n)] for l in range(L)])
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=0.125)
    np.testing.assert_allclose(out, ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)


def test_multi_token_needs_context_for_every_new_token(orc):
    w = W.make_config(2, B=2, ctx_lo=3, ctx_hi=3, seed=1)
    q = np.zeros((2, 4, w.Hq, w.D), np.uint16)
    with pytest.raises(RuntimeError):
        orc.paged_decode_attention_multi(q, w.k_pool, w.v_pool, w.block_tables, w.context_lens, w.scale)


# ---- paged prefill (varlen causal) --------------------------------------------------------------

def test_prefill_with_uniform_lengths_is_multi_token_decode(orc):
    w = W.make_prefill(name="p", query_lens=[3, 3, 3], cached_lens=[10, 0, 40], Hq=4, Hkv=2, D=64, seed=3)
    a = orc.paged_prefill_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                    w.query_start, w.scale)
    b = orc.paged_decode_attention_multi(w.q.reshape(3, 3, 4, 64), w.k_pool, w.v_pool,
                                         w.block_tables, w.context_lens, w.scale)
    assert np.array_equal(a.reshape(3, 3, 4, 64), b)


def test_prefill_matches_library_causal_attention(orc):
    """Whole-prompt prefill (nothing cached) is ordinary causal attention: torch SDPA with
    is_causal on the gathered K/V, fp64 on CPU."""
    torch = pytest.importorskip("torch")
    w = W.make_prefill(name="p", query_lens=[37, 1, 20], cached_lens=[0, 0, 0], Hq=4, Hkv=2, D=64, seed=5)
    out = orc.paged_prefill_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                      w.query_start, w.scale)
    kf = W.bf16_bits_to_f32(w.k_pool).astype(np.float64)
    vf = W.bf16_bits_to_f32(w.v_pool).astype(np.float64)
    qf = W.bf16_bits_to_f32(w.q).astype(np.float64)
    for b in range(w.B):
        n = int(w.context_lens[b])
        rows = [(w.block_tables[b, t // 16], t % 16) for t in range(n)]
        K = np.stack([kf[blk, :, off] for blk, off in rows], 1)  # [Hkv, n, D]
        V = np.stack([vf[blk, :, off] for blk, off in rows], 1)
        Q = qf[w.query_start[b]:w.query_start[b + 1]].transpose(1, 0, 2)  # [Hq, n, D]
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(Q), torch.from_numpy(K).repeat_interleave(2, 0),
            torch.from_numpy(V).repeat_interleave(2, 0), is_causal=True, scale=w.scale)
        np.testing.assert_allclose(out[w.query_start[b]:w.query_start[b + 1]],
                                   ref.numpy().transpose(1, 0, 2), rtol=0, atol=1e-12)


def _int8_prefill_with_pow2_scales(seed, query_lens, cached_lens, Hq=4, Hkv=2, D=64):
    """An INT8 prefill whose scales are powers of two that differ per block, kv head, token and
    between K and V, so code * scale is exact in fp32."""
    w = W.make_prefill(name="p8", query_lens=query_lens, cached_lens=cached_lens, Hq=Hq, Hkv=Hkv,
                       D=D, seed=seed, kv_dtype="i8")
    idx = np.arange(w.k_scales.size).reshape(w.k_scales.shape)
    ks = np.ldexp(np.float32(1.0), -(3 + idx % 5)).astype(np.float32)
    vs = np.ldexp(np.float32(1.0), -(2 + (idx * 3) % 7)).astype(np.float32)
    return w, ks, vs


def test_prefill_int8_is_prefill_on_the_dequantised_values(orc):
    """"EchoLLMServing notes" section 3 with the prefill of section 2: an INT8 cache attends as
    the cache of its dequantised values K = code * k_scale, V = code * v_scale (per token and kv
    head). With power-of-two scales those values are exact in fp32, so the INT8 prefill must equal
    the fp32-pool prefill bit for bit -- swapping the K and V scales, or taking another token's or
    head's scale, does not."""
    w, ks, vs = _int8_prefill_with_pow2_scales(11, [5, 1, 40, 17], [30, 0, 7, 100])
    a = orc.paged_prefill_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                    w.query_start, w.scale, ks, vs)
    kf = (w.k_pool.astype(np.float32) * ks[..., None]).astype(np.float32)
    vf = (w.v_pool.astype(np.float32) * vs[..., None]).astype(np.float32)
    assert np.array_equal(kf.astype(np.float64), w.k_pool.astype(np.float64) * ks[..., None].astype(np.float64))
    b = orc.paged_prefill_attention(w.q, kf, vf, w.block_tables, w.context_lens, w.query_start, w.scale)
    assert np.array_equal(a, b)
    swapped = orc.paged_prefill_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                          w.query_start, w.scale, vs, ks)
    assert not np.allclose(a, swapped, atol=1e-6)


def test_prefill_int8_matches_library_causal_attention(orc):
    """Whole-prompt INT8 prefill is causal attention over the dequantised K/V: torch SDPA with
    is_causal, fp64 on CPU, on values gathered here from the codes and scales."""
    torch = pytest.importorskip("torch")
    w = W.make_prefill(name="p8", query_lens=[33, 1, 18], cached_lens=[0, 0, 0], Hq=4, Hkv=2, D=64,
                       seed=13, kv_dtype="i8")
    out = orc.paged_prefill_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                      w.query_start, w.scale, w.k_scales, w.v_scales)
    kf = w.k_pool.astype(np.float64) * w.k_scales[..., None].astype(np.float64)
    vf = w.v_pool.astype(np.float64) * w.v_scales[..., None].astype(np.float64)
    qf = W.bf16_bits_to_f32(w.q).astype(np.float64)
    for b in range(w.B):
        n = int(w.context_lens[b])
        rows = [(w.block_tables[b, t // 16], t % 16) for t in range(n)]
        K = np.stack([kf[blk, :, off] for blk, off in rows], 1)
        V = np.stack([vf[blk, :, off] for blk, off in rows], 1)
        Q = qf[w.query_start[b]:w.query_start[b + 1]].transpose(1, 0, 2)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(Q), torch.from_numpy(K).repeat_interleave(2, 0),
            torch.from_numpy(V).repeat_interleave(2, 0), is_causal=True, scale=w.scale)
        np.testing.assert_allclose(out[w.query_start[b]:w.query_start[b + 1]],
                                   ref.numpy().transpose(1, 0, 2), rtol=0, atol=1e-12)


@pytest.mark.parametrize("kv", ["bf16", "i8"])
def test_prefill_rows_are_decode_queries_at_their_causal_limits(orc, kv):
    """Each prefill row is, by definition, one decode query: row i of a sequence with L new tokens
    attends to the first context_len - (L - 1 - i) tokens of its table. The prefill equals the
    decode oracle run row by row with those limits, bit for bit (this is also how the full-size GPU
    tests get their sampled rows)."""
    from _gpu import prefill_rows_by_decode
    w = W.make_prefill(name="p", query_lens=[37, 1, 20, 5], cached_lens=[5, 0, 30, 16], Hq=4, Hkv=2,
                       D=64, seed=21, kv_dtype=kv)
    full = orc.paged_prefill_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                       w.query_start, w.scale, w.k_scales, w.v_scales)
    assert np.array_equal(full, prefill_rows_by_decode(w, np.arange(w.q.shape[0]), orc=orc))


@pytest.mark.parametrize("kv", ["f32", "bf16", "i8"])
def test_oracle_reads_no_slot_past_a_context(orc, kv):
    """The oracle reads only the first context_len positions of each table: NaN in every other slot
    and in every unreferenced block (rows, or INT8 scales) leaves its decode, multi-token and
    prefill answers bit-identical and finite. The GPU sentinel tests compare against exactly this."""
    from _gpu import poisoned
    q_dtype = "f32" if kv == "f32" else "bf16"
    w = W.make_decode(name="d", B=4, Hq=8, Hkv=2, D=64, context_lens=[5, 33, 250, 17], kv_dtype=kv,
                      q_dtype=q_dtype, seed=90)
    pw = poisoned(w)
    a = orc.paged_decode_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens, w.scale,
                                   w.k_scales, w.v_scales)
    b = orc.paged_decode_attention(pw.q, pw.k_pool, pw.v_pool, pw.block_tables, pw.context_lens,
                                   pw.scale, pw.k_scales, pw.v_scales)
    assert np.all(np.isfinite(a)) and np.array_equal(a, b)
    m = W.make_multi_token(w, 3, seed=91)
    pm = poisoned(m)
    a = orc.paged_decode_attention_multi(m.q, m.k_pool, m.v_pool, m.block_tables, m.context_lens,
                                         m.scale, m.k_scales, m.v_scales)
    b = orc.paged_decode_attention_multi(pm.q, pm.k_pool, pm.v_pool, pm.block_tables, pm.context_lens,
                                         pm.scale, pm.k_scales, pm.v_scales)
    assert np.all(np.isfinite(a)) and np.array_equal(a, b)
    if kv != "f32":
        p = W.make_prefill(name="p", query_lens=[20, 1, 7], cached_lens=[13, 40, 0], Hq=4, Hkv=2, D=64,
                           seed=92, kv_dtype=kv)
        pp = poisoned(p)
        a = orc.paged_prefill_attention(p.q, p.k_pool, p.v_pool, p.block_tables, p.context_lens,
                                        p.query_start, p.scale, p.k_scales, p.v_scales)
        b = orc.paged_prefill_attention(pp.q, pp.k_pool, pp.v_pool, pp.block_tables, pp.context_lens,
                                        pp.query_start, pp.scale, pp.k_scales, pp.v_scales)
        assert np.all(np.isfinite(a)) and np.array_equal(a, b)
