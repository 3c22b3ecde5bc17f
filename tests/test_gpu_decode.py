"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the same seeded inputs.

Element-by-element at sizes the oracle finishes in seconds (several splits, ragged tails), on
every sequence and head of the five full workloads, plus the invariants and edge cases.
"""
import math
import os

import numpy as np
import pytest

import oracle
import paged_kv_decode_reshape_gb300 as P
import workloads as W
from _gpu import DevWorkload, assert_close, oracle_step, to_dev, to_f64, to_host_raw

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

REDUCED = {
    1: dict(),
    2: dict(B=6, ctx_lo=1, ctx_hi=1500),
    3: dict(B=2, ctx_lo=3000, ctx_hi=9000),
    4: dict(B=5, ctx_lo=17, ctx_hi=3000),
    5: dict(B=6, ctx_lo=16, ctx_hi=300, prefix_tokens=256),
}


@pytest.fixture(scope="module", autouse=True)
def _lib(pkv):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return pkv


def status_tensor():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_kv_write_bit_exact(cfg):
    w = W.make_config(cfg, **REDUCED[cfg])
    d = DevWorkload(w)
    st = status_tensor()
    d.write(st)
    torch.cuda.synchronize()
    kp, vp, ks, vs = oracle.kv_cache_write(w.k_new, w.v_new, w.k_pool, w.v_pool, w.slot_mapping,
                                           w.k_new_scales, w.v_new_scales, w.k_scales, w.v_scales)
    assert np.array_equal(to_host_raw(d.k_pool), kp)
    assert np.array_equal(to_host_raw(d.v_pool), vp)
    if ks is not None:
        assert np.array_equal(d.k_scales.cpu().numpy(), ks)
        assert np.array_equal(d.v_scales.cpu().numpy(), vs)
    assert int(st.item()) == 0


def test_kv_write_skips_padding_and_flags_bad_slots():
    w = W.make_config(2, B=4, ctx_lo=20, ctx_hi=60)
    sm = w.slot_mapping.copy()
    sm[1] = -1                       # padding token: not written
    sm[2] = w.NB * 16 + 5            # outside the pool: not written, flagged
    w2 = W.DecodeWorkload(**{**w.__dict__, "slot_mapping": sm})
    d = DevWorkload(w2)
    st = status_tensor()
    d.write(st)
    torch.cuda.synchronize()
    kp, vp, _, _ = oracle.kv_cache_write(w2.k_new, w2.v_new, w2.k_pool, w2.v_pool, sm, check=False)
    assert np.array_equal(to_host_raw(d.k_pool), kp)
    assert np.array_equal(to_host_raw(d.v_pool), vp)
    assert int(st.item()) & 1


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_decode_step_matches_oracle(cfg):
    w = W.make_config(cfg, **REDUCED[cfg])
    d = DevWorkload(w)
    st = status_tensor()
    got = to_f64(d.step(status=st))
    ref = oracle_step(w)
    assert_close(got, ref, w.kv_dtype, f"config {cfg}")
    assert int(st.item()) == 0


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_full_size_every_sequence(cfg):
    """The full workload, in the launch configuration the bench times (auto chunk, write then
    attention on one stream; the shared-prefix batch also through the cascade call the bench
    uses), compared with the oracle element by element over every sequence and every head."""
    w = W.make_config(cfg)
    d = DevWorkload(w)
    st = status_tensor()
    got = to_f64(d.step(status=st))
    ref = oracle_step(w, num_threads=os.cpu_count() or 8)
    assert got.shape == (w.B, w.Hq, w.D)
    assert_close(got, ref, w.kv_dtype, f"config {cfg}, all {w.B} sequences")
    if w.shared_prefix_blocks:
        prefix = w.shared_prefix_blocks * w.BS
        nbytes = P.decode_shared_prefix_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, w.max_context_len,
                                                        prefix, 0)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        out = torch.empty_like(d.q)
        P.paged_decode_attention_shared_prefix(out, d.q, d.k_pool, d.v_pool, d.block_tables,
                                               d.context_lens, w.max_context_len, w.scale, prefix,
                                               0, ws, st)
        assert_close(to_f64(out), ref, "bf16", f"config {cfg} cascade call, all sequences")
    torch.cuda.synchronize()
    assert int(st.item()) == 0


@pytest.mark.parametrize("chunk", [16, 48, 64, 256, 4096])
def test_forced_split_sizes(chunk):
    w = W.make_config(2, B=5, ctx_lo=1, ctx_hi=900, seed=21)
    ref = oracle_step(w)
    d = DevWorkload(w)
    got = to_f64(d.step(chunk=chunk))
    assert_close(got, ref, "bf16", f"chunk {chunk}")


def test_split_partials_match_oracle_partials():
    """The workspace holds each split's (m, l, acc), m in base-2 units. m is a reference max
    (the kernel only raises it when scores exceed it by more than 2^8), so a split's state is
    compared through what does not depend on the reference: the log-sum-exp m + log(l) and the
    normalised accumulator acc / l."""
    w = W.make_config(2, B=3, ctx_lo=100, ctx_hi=700, seed=4)
    chunk = 64
    d = DevWorkload(w)
    d.write()
    maxc = w.max_context_len
    S = max(1, maxc // chunk)
    nbytes = w.B * w.Hq * S * (w.D + 2) * 4
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    d.attend(chunk=chunk, workspace=ws)
    torch.cuda.synchronize()
    f = ws.view(torch.float32).cpu().numpy().astype(np.float64)
    acc = f[: w.B * w.Hq * S * w.D].reshape(w.B, w.Hq, S, w.D)
    ml = f[w.B * w.Hq * S * w.D:].reshape(w.B, w.Hq, S, 2)
    kp, vp, _, _ = oracle.kv_cache_write(w.k_new, w.v_new, w.k_pool, w.v_pool, w.slot_mapping)
    m, l, oacc, ns = oracle.paged_decode_partials(w.q, kp, vp, w.block_tables, w.context_lens,
                                                  w.scale, chunk, S)
    for b in range(w.B):
        k = int(ns[b])
        assert k > 1
        gm, gl = ml[b, :, :k, 0] * math.log(2), ml[b, :, :k, 1]
        assert np.all(gm <= m[b, :, :k] + 1e-3)                      # never above the true max
        assert np.all(gm >= m[b, :, :k] - 8 * math.log(2) - 1e-3)    # within 2^8 of it
        np.testing.assert_allclose(gm + np.log(gl), m[b, :, :k] + np.log(l[b, :, :k]), atol=2e-3)
        np.testing.assert_allclose(acc[b, :, :k] / gl[..., None],
                                   oacc[b, :, :k] / l[b, :, :k, None], atol=5e-3)


@pytest.mark.parametrize("kv", ["bf16", "i8", "f32"])
def test_workspace_contents_on_entry_do_not_matter(kv):
    """A workspace full of random bytes, one left by a call with other lengths (more splits per
    sequence), and a repeat of the same call must all give the oracle's answer, the repeat bit for
    bit: the merge reads only partial states the same call wrote."""
    lens_a = [700, 33, 1500, 64, 1023, 257]
    lens_b = [1500, 1400, 16, 900, 1024, 600]
    mk = lambda lens, seed: W.make_decode(name="ws", B=6, Hq=16, Hkv=2, D=128, context_lens=lens,
                                          kv_dtype=kv, q_dtype="f32" if kv == "f32" else "bf16",
                                          seed=seed)
    wa, wb = mk(lens_a, 51), mk(lens_b, 52)
    chunk = 64
    nbytes = max(P.decode_workspace_bytes(6, 16, 2, 128, max(l), chunk) for l in (lens_a, lens_b))
    g = torch.Generator(device="cuda").manual_seed(5)
    ws = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda", generator=g)

    def ref(w):
        return oracle.paged_decode_attention(w.q, w.k_pool, w.v_pool, w.block_tables,
                                             w.context_lens, w.scale, w.k_scales, w.v_scales)
    da, db = DevWorkload(wa), DevWorkload(wb)
    first = da.attend(chunk=chunk, workspace=ws).clone()
    assert_close(to_f64(first), ref(wa), kv, "random workspace")
    got_b = db.attend(chunk=chunk, workspace=ws)
    assert_close(to_f64(got_b), ref(wb), kv, "workspace left by another batch")
    again = da.attend(chunk=chunk, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(again, first)


@pytest.mark.parametrize("cfg", [2, 4])
def test_block_permutation_bit_identical(cfg):
    w = W.make_config(cfg, B=6, ctx_lo=30, ctx_hi=1200)
    p = W.permute_blocks(w, seed=123)
    a = DevWorkload(w).step()
    b = DevWorkload(p).step()
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_shared_prefix_equals_copy_on_write_bit_identical():
    w = W.make_config(5, B=8, ctx_lo=16, ctx_hi=500, prefix_tokens=512)
    c = W.unshare_prefix(w)
    a = DevWorkload(w).step()
    b = DevWorkload(c).step()
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert_close(to_f64(a), oracle_step(w), "bf16", "prefix-shared")


@pytest.mark.parametrize("kv", ["f32", "bf16", "i8"])
def test_edge_context_lengths(kv):
    lens = [0, 1, 2, 15, 16, 17, 31, 32, 33, 511, 512, 513, 1024, 1025]
    w = W.make_decode(name="edges", B=len(lens), Hq=8, Hkv=2, D=128, context_lens=lens,
                      kv_dtype=kv, q_dtype="f32" if kv == "f32" else "bf16", seed=31)
    d = DevWorkload(w)
    for chunk in (0, 16, 512):
        got = to_f64(d.attend(chunk=chunk))
        ref = oracle.paged_decode_attention(w.q, w.k_pool, w.v_pool, w.block_tables,
                                            w.context_lens, w.scale, w.k_scales, w.v_scales)
        assert np.all(got[0] == 0.0)  # empty context -> zeros
        assert_close(got, ref, kv, f"{kv} chunk {chunk}")
    if kv == "bf16":  # one token: out is that token's V row exactly
        got = to_f64(d.attend())
        blk = w.block_tables[1, 0]
        for h in range(8):
            np.testing.assert_array_equal(got[1, h], W.bf16_bits_to_f32(w.v_pool[blk, h // 4, 0]))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("g", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("kv", ["f32", "bf16"])
def test_head_groups_and_dims(D, g, kv):
    Hkv = 2
    w = W.make_decode(name="groups", B=3, Hq=Hkv * g, Hkv=Hkv, D=D, context_lens=[5, 100, 700],
                      kv_dtype=kv, q_dtype=kv, seed=g * 10 + D)
    got = to_f64(DevWorkload(w).attend(chunk=256))
    ref = oracle.paged_decode_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens, w.scale)
    assert_close(got, ref, kv, f"g={g} D={D}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("g", [1, 4, 8])
def test_int8_head_groups_and_dims(D, g):
    w = W.make_decode(name="i8groups", B=3, Hq=2 * g, Hkv=2, D=D, context_lens=[9, 300, 1100],
                      kv_dtype="i8", q_dtype="bf16", seed=g + D)
    got = to_f64(DevWorkload(w).attend(chunk=256))
    ref = oracle.paged_decode_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                        w.scale, w.k_scales, w.v_scales)
    assert_close(got, ref, "i8", f"int8 g={g} D={D}")


def test_int8_every_byte_value_converts_exactly():
    """Single-token contexts with unit V scales: out = the int8 V row, exact in bf16."""
    D, Hkv = 128, 1
    NB = 2
    kp = np.zeros((NB, Hkv, 16, D), np.int8)
    vp = np.zeros((NB, Hkv, 16, D), np.int8)
    allv = np.arange(-128, 128, dtype=np.int16).astype(np.int8)
    vp[0, 0, 0] = allv[:128]
    vp[1, 0, 0] = allv[128:]
    ks = np.ones((NB, Hkv, 16), np.float32)
    vs = np.ones((NB, Hkv, 16), np.float32)
    q = W.f32_to_bf16_bits(np.ones((2, 1, D), np.float32))
    w = W.DecodeWorkload(name="bytes", B=2, Hq=1, Hkv=1, D=D, BS=16, NB=NB, kv_dtype="i8",
                         q_dtype="bf16", q=q, k_pool=kp, v_pool=vp,
                         block_tables=np.array([[0], [1]], np.int32),
                         context_lens=np.array([1, 1], np.int32),
                         slot_mapping=np.array([-1, -1], np.int64),
                         k_new=np.zeros((2, 1, D), np.int8), v_new=np.zeros((2, 1, D), np.int8),
                         scale=0.1, ref_count=np.ones(NB, np.int32), k_scales=ks, v_scales=vs,
                         k_new_scales=np.ones((2, 1), np.float32),
                         v_new_scales=np.ones((2, 1), np.float32))
    got = to_f64(DevWorkload(w).attend())
    np.testing.assert_array_equal(got[:, 0].reshape(-1), allv.astype(np.float64))


def test_identical_keys_give_mean_of_v():
    w = W.make_config(2, B=3, ctx_lo=200, ctx_hi=800, seed=8)
    kp = w.k_pool.copy()
    kp[:] = kp[0, :, 0:1, :]  # every row of every block: the same key per kv head
    w2 = W.DecodeWorkload(**{**w.__dict__, "k_pool": kp})
    got = to_f64(DevWorkload(w2).attend())
    vf = W.bf16_bits_to_f32(w.v_pool).astype(np.float64)
    for b in range(w.B):
        n = int(w.context_lens[b])
        rows = np.stack([vf[w.block_tables[b, t // 16], :, t % 16] for t in range(n)])
        mean = rows.mean(0)  # [Hkv, D]
        for h in range(w.Hq):
            np.testing.assert_allclose(got[b, h], mean[h // w.group], atol=4e-3)


def _ranged_workload(kv, case):
    """Scores far from the unit range. "wide": scale x8 on N(0, 1) data, so the running max is
    raised many times. "below_zero": every key points away from its sequence's query (scale x16),
    so all scores lie ~170 base-2 units below zero and 2^s underflows unless the reference is the
    running max. "late_spike": one key near the end of each context is aligned with the query, so
    the max jumps by tens of units in a late, partial block."""
    lens = [1, 40, 700, 2100]
    w = W.make_decode(name="ranges", B=len(lens), Hq=16, Hkv=2, D=128, context_lens=lens,
                      kv_dtype=kv, q_dtype="bf16", seed=55 if kv == "bf16" else 56)
    G = w.group
    q = W.bf16_bits_to_f32(w.q).copy()
    kp = w.k_pool.copy()
    kf = W.bf16_bits_to_f32(kp) if kv == "bf16" else kp.astype(np.float32)
    scale = w.scale * (8.0 if case == "wide" else 16.0)
    if case != "wide":
        for b, n in enumerate(lens):
            for h in range(w.Hkv):
                q[b, h * G:(h + 1) * G] = q[b, h * G]      # one query per group
                sgn = np.where(q[b, h * G] < 0, -1.0, 1.0)
                rows = [t for t in range(n)] if case == "below_zero" else [max(0, n - 3)]
                for t in rows:
                    blk, off = w.block_tables[b, t // 16], t % 16
                    mag = np.abs(kf[blk, h, off]) + (0.0 if kv == "i8" else 0.25)
                    kf[blk, h, off] = (-sgn if case == "below_zero" else sgn) * mag
        if case == "late_spike":
            scale = w.scale * 2.0
    if kv == "bf16":
        kp = W.f32_to_bf16_bits(kf)
    else:
        kp = np.clip(kf, -127, 127).astype(np.int8)
    return W.DecodeWorkload(**{**w.__dict__, "q": W.f32_to_bf16_bits(q), "k_pool": kp,
                               "scale": scale})


@pytest.mark.parametrize("kv", ["bf16", "i8"])
@pytest.mark.parametrize("case", ["wide", "below_zero", "late_spike"])
def test_extreme_score_ranges(kv, case):
    w = _ranged_workload(kv, case)
    ref = oracle.paged_decode_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                        w.scale, w.k_scales, w.v_scales)
    d = DevWorkload(w)
    for chunk in (0, 64):
        got = to_f64(d.attend(chunk=chunk))
        assert np.all(np.isfinite(got))
        assert_close(got, ref, kv, f"{kv} {case} chunk {chunk}")


def _outlier_workload(kv, mag, ndims, k_mult, seed):
    """A G = 8 batch (Hq 16, Hkv 2) whose queries carry `ndims` outlier dims of magnitude `mag`
    (signs random, bf16-rounded; ndims = 128 scales the whole query by `mag` instead), with every
    key multiplied by k_mult (bf16 pools: the values, re-rounded; INT8 pools: the K scales)."""
    lens = [1, 40, 700, 2100]
    w = W.make_decode(name="outliers", B=len(lens), Hq=16, Hkv=2, D=128, context_lens=lens,
                      kv_dtype=kv, q_dtype="bf16", seed=seed)
    rng = np.random.default_rng(seed)
    q = W.bf16_bits_to_f32(w.q).copy()
    if ndims == w.D:
        q *= np.float32(mag)
    else:
        for b in range(w.B):
            for h in range(w.Hq):
                dims = rng.choice(w.D, ndims, replace=False)
                q[b, h, dims] = np.float32(mag) * np.sign(rng.standard_normal(ndims)).astype(np.float32)
    changes = {"q": W.f32_to_bf16_bits(q)}
    if kv == "bf16":
        changes["k_pool"] = W.f32_to_bf16_bits(W.bf16_bits_to_f32(w.k_pool) * np.float32(k_mult))
    else:
        changes["k_scales"] = (w.k_scales * np.float32(k_mult)).astype(np.float32)
    return W.DecodeWorkload(**{**w.__dict__, **changes})


@pytest.mark.parametrize("kv", ["bf16", "i8"])
@pytest.mark.parametrize("mag,ndims,k_mult", [
    (1e2, 4, 1.0), (1e3, 2, 1.0), (1e4, 1, 1.0), (1e4, 4, 1.0),   # outlier dims, N(0, 1) keys
    (1e6, 3, 1e-4), (1e6, 128, 1e-5),  # |q * scale| past fp16's range, logits of ordinary size
    (1e-6, 128, 1.0),                  # tiny queries: near-uniform weights
    (1e-4, 128, 1e4),                  # q * scale below fp16's normal range, logits of ordinary size
])
def test_outlier_query_magnitudes(kv, mag, ndims, k_mult):
    """Queries with a few outlier dims of the magnitudes LLM activations reach (10^2 - 10^4), and
    queries whose magnitude times the softmax scale falls outside fp16's normal range while the
    keys keep the logits of ordinary size: the INT8 kernel's fp16 operands must neither overflow
    nor lose precision there. Same bars as every other parity case.

    Not covered, by design: logits of 10^5 and more (|q| ~ 10^6 against unit keys). An fp32 score
    of that size resolves only ~|s| * 2^-24, and a dot product whose terms span 10^6 down to 1
    loses the small ones in any fp32 accumulation, so no fp32 kernel meets the bf16 bar there."""
    seed = int(round(np.log10(mag) * 10)) + ndims + int(round(np.log10(k_mult))) * 7 + (0 if kv == "bf16" else 500)
    w = _outlier_workload(kv, mag, ndims, k_mult, seed=seed)
    ref = oracle.paged_decode_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                        w.scale, w.k_scales, w.v_scales)
    d = DevWorkload(w)
    for chunk in (0, 64):
        st = status_tensor()
        got = to_f64(d.attend(chunk=chunk, status=st))
        assert np.all(np.isfinite(got))
        assert_close(got, ref, kv, f"{kv} |q| {mag} in {ndims} dims, keys x {k_mult}, chunk {chunk}")
        assert int(st.item()) == 0


def test_bad_block_ids_are_skipped_and_flagged():
    w = W.make_config(2, B=4, ctx_lo=100, ctx_hi=400, seed=3)
    bt = w.block_tables.copy()
    bt[1, 2] = w.NB + 1000
    bt[2, 0] = -7
    w2 = W.DecodeWorkload(**{**w.__dict__, "block_tables": bt})
    st = status_tensor()
    got = to_f64(DevWorkload(w2).attend(status=st))
    assert int(st.item()) & 2
    ref = oracle.paged_decode_attention(w.q[[0, 3]], w.k_pool, w.v_pool, w.block_tables[[0, 3]],
                                        w.context_lens[[0, 3]], w.scale)
    assert np.all(np.isfinite(got))
    assert_close(got[[0, 3]], ref, "bf16", "untouched sequences")


def test_understated_max_context_len_is_still_correct():
    w = W.make_config(2, B=4, ctx_lo=600, ctx_hi=3000, seed=12)
    st = status_tensor()
    got = to_f64(DevWorkload(w).attend(status=st, max_context_len=1024))
    assert int(st.item()) & 8
    ref = oracle.paged_decode_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens, w.scale)
    assert_close(got, ref, "bf16", "long context")


def test_context_beyond_table_is_clamped_and_flagged():
    w = W.make_config(2, B=2, ctx_lo=40, ctx_hi=60, seed=2)
    lens = w.context_lens.copy()
    lens[0] = w.MBPS * 16 + 100
    w2 = W.DecodeWorkload(**{**w.__dict__, "context_lens": lens})
    st = status_tensor()
    d = DevWorkload(w2)
    d.attend(status=st, max_context_len=w.MBPS * 16)
    torch.cuda.synchronize()
    assert int(st.item()) & 4


def test_runs_on_the_callers_stream():
    w = W.make_config(2, B=8, ctx_lo=500, ctx_hi=2000, seed=9)
    d = DevWorkload(w)
    ref = to_f64(d.step())
    d2 = DevWorkload(w)
    torch.cuda.synchronize()  # uploads ran on the default stream
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = d2.step()
    s.synchronize()
    assert np.array_equal(to_f64(out), ref)


@pytest.mark.parametrize("kv", ["bf16", "i8"])
@pytest.mark.parametrize("shape", [
    dict(B=1, Hq=32, Hkv=8, lens="131072"),            # one sequence at the longest context
    dict(B=512, Hq=32, Hkv=8, lens="1-200"),           # many short sequences
    dict(B=16, Hq=64, Hkv=8, lens="100-3000"),         # 8 query heads per kv head
    dict(B=16, Hq=16, Hkv=16, lens="100-3000"),        # MHA: one query head per kv head
    dict(B=8, Hq=32, Hkv=2, lens="100-3000"),          # 16 query heads per kv head: two CTA groups
    dict(B=12, Hq=20, Hkv=5, lens="1-2000"),           # odd kv-head count, G = 4
], ids=["B1_131k", "B512_short", "G8", "MHA", "G16", "Hkv5"])
def test_shape_sweep_sampled_rows(shape, kv):
    """Shapes beyond the five workloads, in the auto launch configuration, checked against the
    oracle on a sample of sequences (every head), including the longest."""
    rng = np.random.default_rng(shape["B"] * 7 + shape["Hkv"])
    lo_hi = shape["lens"].split("-")
    if len(lo_hi) == 1:
        lens = np.full(shape["B"], int(lo_hi[0]))
    else:
        lens = rng.integers(int(lo_hi[0]), int(lo_hi[1]) + 1, size=shape["B"])
    w = W.make_decode(name="sweep", B=shape["B"], Hq=shape["Hq"], Hkv=shape["Hkv"], D=128,
                      context_lens=lens, kv_dtype=kv, q_dtype="bf16", seed=int(lens.sum() % 1000))
    rows = sorted({0, shape["B"] - 1, shape["B"] // 2, int(np.argmax(w.context_lens))})
    d = DevWorkload(w)
    st = status_tensor()
    got = to_f64(d.step(status=st))[rows]
    ref = oracle_step(w, rows=rows, num_threads=16)
    assert_close(got, ref, kv, f"{shape} {kv} rows {rows}")
    assert int(st.item()) == 0
