"""GPU parity of the paged prefill over an INT8 cache (pkv_paged_prefill_attention_int8) against the
fp64 oracle on the dequantised values: the query-length mix of a chunked-prefill / mixed batch
(decode rows of one token beside prompt chunks of several 128-row tiles), cached prefixes, GQA
groups, missing blocks and extreme scales, at the INT8 bar ("EchoLLMServing inference framework
notes", section 3: per-token dequantisation fused into the FlashAttention prefill)."""
import numpy as np
import pytest

import oracle
import paged_kv_decode_reshape_gb300 as P
import workloads as W
from _gpu import assert_close, prefill_rows_by_decode, to_dev, to_f64

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib(pkv):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_prefill_i8(w, status=None, bt=None):
    bt = w.block_tables if bt is None else bt
    out = torch.zeros((w.q.shape[0], w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    P.paged_prefill_attention_int8(out, to_dev(w.q), to_dev(w.k_pool), to_dev(w.v_pool),
                                   to_dev(w.k_scales), to_dev(w.v_scales), to_dev(bt),
                                   to_dev(w.context_lens), to_dev(w.query_start), w.max_query_len,
                                   w.scale, status)
    return to_f64(out)


def reference(w):
    return oracle.paged_prefill_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                          w.query_start, w.scale, w.k_scales, w.v_scales)


@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 8), (16, 2), (6, 2), (4, 2), (32, 2)])
def test_prefill_int8_matches_oracle(hq, hkv):
    w = W.make_prefill(name="pf8", query_lens=[1, 5, 127, 128, 129, 300],
                       cached_lens=[0, 17, 64, 200, 5, 1000], Hq=hq, Hkv=hkv, D=128,
                       seed=hq + hkv + 100, kv_dtype="i8")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_prefill_i8(w, st)
    assert_close(got, reference(w), "i8", f"INT8 prefill Hq={hq} Hkv={hkv}")
    assert int(st.item()) == 0


def test_prefill_int8_mixed_batch_decode_rows_equal_decode():
    """A mixed batch: one-token rows (decode) beside prompt chunks; the decode rows must equal the
    INT8 decode oracle and the chunks the prefill oracle."""
    w = W.make_prefill(name="pfm8", query_lens=[1, 200, 1, 1, 64], cached_lens=[900, 30, 15, 0, 333],
                       Hq=32, Hkv=8, D=128, seed=41, kv_dtype="i8")
    got = run_prefill_i8(w)
    ref = reference(w)
    assert_close(got, ref, "i8", "mixed INT8 batch")
    dec = [0, 2, 3]
    rows = w.query_start[dec]
    ref_dec = oracle.paged_decode_attention(w.q[rows], w.k_pool, w.v_pool, w.block_tables[dec],
                                            w.context_lens[dec], w.scale, w.k_scales, w.v_scales)
    assert_close(got[rows], ref_dec, "i8", "decode rows")


def test_prefill_int8_long_prompt_and_empty_sequences():
    w = W.make_prefill(name="pfl8", query_lens=[1000, 0, 37], cached_lens=[2048, 10, 3000], Hq=32,
                       Hkv=8, D=128, seed=8, kv_dtype="i8")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_prefill_i8(w, st)
    assert_close(got, reference(w), "i8", "long INT8 prompt")
    assert int(st.item()) == 0


def test_prefill_int8_missing_block_is_skipped_and_flagged():
    w = W.make_prefill(name="pfb8", query_lens=[40, 70], cached_lens=[100, 30], Hq=16, Hkv=4, D=128,
                       seed=9, kv_dtype="i8")
    bt = w.block_tables.copy()
    bt[0, 2] = w.NB + 5
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_prefill_i8(w, st, bt)
    assert int(st.item()) & P.FLAG_BAD_BLOCK
    assert np.all(np.isfinite(got))
    s1 = slice(w.query_start[1], w.query_start[2])
    assert_close(got[s1], reference(w)[s1], "i8", "untouched sequence")


@pytest.mark.parametrize("scale", [-0.3, 2.0, 0.0])
def test_prefill_int8_scale_sign_and_running_max_rescale(scale):
    w = W.make_prefill(name="pfs8", query_lens=[300, 129], cached_lens=[700, 0], Hq=8, Hkv=2,
                       D=128, seed=17, kv_dtype="i8")
    w.scale = scale
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_prefill_i8(w, st)
    assert_close(got, reference(w), "i8", f"INT8 prefill scale={scale}")
    assert int(st.item()) == 0


def test_prefill_int8_every_byte_value():
    """One visible key per row (L = 1, context 1) with unit V scale: out = that key's int8 V row,
    exact in bf16 for every code -128..127 across two sequences."""
    D, Hkv = 128, 1
    NB = 2
    kp = np.zeros((NB, Hkv, 16, D), np.int8)
    vp = np.zeros((NB, Hkv, 16, D), np.int8)
    allv = np.arange(-128, 128, dtype=np.int16).astype(np.int8)
    vp[0, 0, 0], vp[1, 0, 0] = allv[:128], allv[128:]
    ones = np.ones((NB, Hkv, 16), np.float32)
    w = W.PrefillWorkload(name="bytes8", Hq=1, Hkv=1, D=D, BS=16, NB=NB,
                          q=W.f32_to_bf16_bits(np.ones((2, 1, D), np.float32)), k_pool=kp, v_pool=vp,
                          block_tables=np.array([[0], [1]], np.int32),
                          context_lens=np.array([1, 1], np.int32),
                          query_start=np.array([0, 1, 2], np.int32), scale=0.1, kv_dtype="i8",
                          k_scales=ones, v_scales=ones)
    got = run_prefill_i8(w)
    np.testing.assert_array_equal(got[:, 0].reshape(-1), allv.astype(np.float64))


def test_prefill_int8_argument_errors():
    w = W.make_prefill(name="pfe8", query_lens=[3], cached_lens=[5], Hq=8, Hkv=2, D=128, seed=2,
                       kv_dtype="i8")
    out = torch.zeros((3, 8, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(P.PkvError):  # scales missing
        P.paged_prefill_attention_int8(out, to_dev(w.q), to_dev(w.k_pool), to_dev(w.v_pool), None,
                                       to_dev(w.v_scales), to_dev(w.block_tables),
                                       to_dev(w.context_lens), to_dev(w.query_start), 3, w.scale)


@pytest.mark.parametrize("mag,ndims,k_mult", [
    (1e2, 4, 1.0), (1e3, 2, 1.0), (1e4, 1, 1.0),  # outlier dims, N(0, 1) keys
    (1e6, 3, 1e-4),                               # |q| past fp16's range, logits of ordinary size
    (1e-4, 128, 1e4),                             # |q| below fp16's normal range, same logits
    (1e-6, 128, 1.0),                             # tiny queries: near-uniform weights
])
def test_prefill_int8_outlier_query_magnitudes(mag, ndims, k_mult):
    """The INT8 prefill runs fp16 products with q scaled by one power of two per CTA: queries with a
    few outlier dims (the magnitudes LLM activations reach), or whose magnitude falls outside fp16's
    normal range while the keys (K scales times k_mult) keep the logits of ordinary size, must
    neither overflow nor lose precision. The same INT8 bar as every other case."""
    w = W.make_prefill(name="pfo", query_lens=[1, 40, 200], cached_lens=[0, 300, 100], Hq=16,
                       Hkv=2, D=128, seed=int(np.log10(mag) * 10) + ndims, kv_dtype="i8")
    rng = np.random.default_rng(ndims)
    q = W.bf16_bits_to_f32(w.q).copy()
    if ndims == w.D:
        q *= np.float32(mag)
    else:
        for t in range(q.shape[0]):
            for h in range(w.Hq):
                dims = rng.choice(w.D, ndims, replace=False)
                q[t, h, dims] = np.float32(mag) * np.sign(rng.standard_normal(ndims)).astype(np.float32)
    w.q = W.f32_to_bf16_bits(q)
    w.k_scales = (w.k_scales * np.float32(k_mult)).astype(np.float32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_prefill_i8(w, st)
    assert np.all(np.isfinite(got))
    assert_close(got, reference(w), "i8", f"INT8 prefill |q| {mag} in {ndims} dims, keys x {k_mult}")
    assert int(st.item()) == 0


def test_prefill_int8_full_size_sampled_rows():
    """The bench's INT8 prefill workload at full size (4 x 4096 new tokens after 2048 cached,
    Llama-3-8B heads) through the call the bench times, every head of sampled rows of every
    sequence (first, middle and last query tiles and their edges) against the oracle."""
    import os
    w = W.make_prefill(name="prefill_llama3_8b_int8", query_lens=[4096] * 4, cached_lens=[2048] * 4,
                       Hq=32, Hkv=8, D=128, seed=7, kv_dtype="i8")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_prefill_i8(w, st)
    qs = np.asarray(w.query_start)
    rows = np.concatenate([qs[b] + np.asarray([0, 1, 2, 127, 128, 129, 2047, 2048, 4094, 4095])
                           for b in range(w.B)])
    ref = prefill_rows_by_decode(w, rows, num_threads=os.cpu_count() or 8)
    assert_close(got[rows], ref, "i8", f"full-size INT8 prefill, {rows.size} rows x 32 heads")
    assert np.all(np.isfinite(got))
    assert int(st.item()) == 0
