"""GPU parity of the shared-prefix (cascade) decode: the prefix every sequence shares goes through the
tcgen05 prefix kernel once per kv head, each suffix through the split-K kernel, and the merge
combines them. The answer is the plain decode attention, so it is held to the oracle like the
regular path, on shared-prefix batches ("LLM Primer VI, Chapter 8", section 8.1: one physical copy
of the prompt's blocks referenced by every sequence's table)."""
import numpy as np
import pytest

import oracle
import paged_kv_decode_reshape_gb300 as P
import workloads as W
from _gpu import DevWorkload, assert_close, to_dev, to_f64

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib(pkv):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def cascade(d: DevWorkload, prefix, chunk=0, status=None, max_context_len=None):
    w = d.w
    maxc = w.max_context_len if max_context_len is None else max_context_len
    nbytes = P.decode_shared_prefix_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, maxc, prefix, chunk)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.empty(d.q.shape, dtype=d.q.dtype, device="cuda")
    P.paged_decode_attention_shared_prefix(out, d.q, d.k_pool, d.v_pool, d.block_tables,
                                           d.context_lens, maxc, w.scale, prefix, chunk, ws, status)
    return out


def reference(w):
    return oracle.paged_decode_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                         w.scale)


@pytest.mark.parametrize("B,prefix,lo,hi", [(12, 512, 16, 500), (7, 144, 1, 300), (40, 2048, 16, 200),
                                            (3, 16, 1, 40)])
def test_shared_prefix_matches_oracle(B, prefix, lo, hi):
    w = W.make_config(5, B=B, ctx_lo=lo, ctx_hi=hi, prefix_tokens=prefix, seed=B + prefix)
    d = DevWorkload(w)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = to_f64(cascade(d, prefix, status=st))
    assert int(st.item()) == 0
    assert_close(got, reference(w), "bf16", f"cascade B={B} prefix={prefix}")
    # and close to the regular path on the same inputs (another summation order)
    reg = to_f64(d.attend())
    assert np.abs(got - reg).max() <= 2e-2



def test_shared_prefix_reference_raised_on_alternate_tiles():
    """Prefix keys whose magnitude grows with their position: most 128-key tiles of the prefix raise
    each row's reference maximum past the lazy margin, so the prefix kernel's two softmax warps of
    a row hand a raised reference to each other on almost every tile. The partial states it writes
    (m, l, acc) must stay consistent for the merge with the suffixes."""
    prefix = 1024
    w = W.make_config(5, B=10, ctx_lo=16, ctx_hi=300, prefix_tokens=prefix, seed=91)
    k = W.bf16_bits_to_f32(w.k_pool)
    for pos in range(prefix):  # the shared blocks: row 0's first prefix / 16 entries
        k[w.block_tables[0][pos // w.BS], :, pos % w.BS, :] *= np.float32(1.0 + 6.0 * pos / 128.0)
    w.k_pool = W.f32_to_bf16_bits(k)
    d = DevWorkload(w)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = to_f64(cascade(d, prefix, status=st))
    assert int(st.item()) == 0
    assert_close(got, reference(w), "bf16", "cascade with rising prefix keys")

@pytest.mark.parametrize("g", [1, 2, 8, 16])
def test_shared_prefix_head_groups(g):
    Hkv = 2
    base = W.make_config(5, B=9, ctx_lo=16, ctx_hi=400, prefix_tokens=256, seed=70 + g)
    w = W.make_decode(name="casc_g", B=9, Hq=Hkv * g, Hkv=Hkv, D=128,
                      context_lens=base.context_lens, kv_dtype="bf16", q_dtype="bf16",
                      seed=80 + g, shared_prefix_tokens=256)
    d = DevWorkload(w)
    got = to_f64(cascade(d, 256, chunk=64))
    assert_close(got, reference(w), "bf16", f"cascade g={g}")


def test_shared_prefix_with_empty_suffixes_and_one_token_suffixes():
    w = W.make_config(5, B=6, ctx_lo=16, ctx_hi=300, prefix_tokens=384, seed=5)
    lens = w.context_lens.copy()
    lens[0] = 384        # the whole context is the prefix
    lens[3] = 385        # one private token
    w.context_lens = lens.astype(np.int32)
    d = DevWorkload(w)
    got = to_f64(cascade(d, 384))
    assert_close(got, reference(w), "bf16", "cascade empty suffix")


def test_shared_prefix_flags_a_sequence_that_does_not_share():
    w = W.make_config(5, B=5, ctx_lo=16, ctx_hi=200, prefix_tokens=256, seed=9)
    bt = w.block_tables.copy()
    spare = int(bt[2, 16])   # a private block of sequence 2, swapped into its prefix
    bt[2, 3] = spare
    w.block_tables = bt
    d = DevWorkload(w)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cascade(d, 256, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & P.FLAG_BAD_PREFIX


def test_shared_prefix_argument_errors():
    w = W.make_config(5, B=4, ctx_lo=16, ctx_hi=100, prefix_tokens=128, seed=2)
    d = DevWorkload(w)
    out = torch.empty(d.q.shape, dtype=d.q.dtype, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    for bad in (0, 40, w.max_context_len + 16):  # none, not a block multiple, beyond the context
        with pytest.raises(P.PkvError):
            P.paged_decode_attention_shared_prefix(out, d.q, d.k_pool, d.v_pool, d.block_tables,
                                                   d.context_lens, w.max_context_len, w.scale,
                                                   bad, 0, ws)
    with pytest.raises(P.PkvError) as e:  # workspace too small
        P.paged_decode_attention_shared_prefix(out, d.q, d.k_pool, d.v_pool, d.block_tables,
                                               d.context_lens, w.max_context_len, w.scale, 128,
                                               0, ws[:256])
    assert e.value.status == P.ERR_WORKSPACE


def _int8_shared_prefix(B, prefix, lo, hi, Hq, Hkv, seed):
    rng = np.random.default_rng(seed)
    lens = prefix + rng.integers(lo, hi + 1, size=B)
    return W.make_decode(name="casc_i8", B=B, Hq=Hq, Hkv=Hkv, D=128, context_lens=lens, kv_dtype="i8",
                         q_dtype="bf16", seed=seed, shared_prefix_tokens=prefix)


def cascade_i8(d: DevWorkload, prefix, chunk=0, status=None):
    w = d.w
    maxc = w.max_context_len
    nbytes = P.decode_shared_prefix_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, maxc, prefix, chunk)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.empty(d.q.shape, dtype=d.q.dtype, device="cuda")
    P.paged_decode_attention_shared_prefix_int8(out, d.q, d.k_pool, d.v_pool, d.k_scales, d.v_scales,
                                                d.block_tables, d.context_lens, maxc, w.scale, prefix,
                                                chunk, ws, status)
    return out


@pytest.mark.parametrize("B,prefix,lo,hi,Hq,Hkv", [(12, 512, 1, 500, 64, 8), (40, 2048, 1, 200, 64, 8),
                                                   (7, 144, 1, 300, 32, 8), (9, 256, 1, 400, 16, 1),
                                                   (3, 16, 1, 40, 8, 4)])
def test_shared_prefix_int8_matches_oracle(B, prefix, lo, hi, Hq, Hkv):
    """The cascade over an INT8 cache: the prefix through the INT8 prefill kernel's machinery, the
    suffixes through the INT8 split-K kernel, one merge; against the INT8 oracle and close to the
    plain INT8 decode call."""
    w = _int8_shared_prefix(B, prefix, lo, hi, Hq, Hkv, seed=B * 7 + prefix)
    d = DevWorkload(w)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = to_f64(cascade_i8(d, prefix, status=st))
    assert int(st.item()) == 0
    ref = oracle.paged_decode_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                        w.scale, w.k_scales, w.v_scales)
    assert_close(got, ref, "i8", f"INT8 cascade B={B} prefix={prefix} G={Hq // Hkv}")
    plain = to_f64(d.attend())
    assert np.abs(got - plain).max() <= 5e-2


def test_shared_prefix_int8_empty_suffix_and_bad_prefix():
    w = _int8_shared_prefix(6, 384, 1, 300, 64, 8, seed=5)
    lens = w.context_lens.copy()
    lens[0] = 384        # the whole context is the prefix
    lens[3] = 385        # one private token
    w.context_lens = lens.astype(np.int32)
    d = DevWorkload(w)
    got = to_f64(cascade_i8(d, 384))
    ref = oracle.paged_decode_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                        w.scale, w.k_scales, w.v_scales)
    assert_close(got, ref, "i8", "INT8 cascade with empty suffix")
    bt = w.block_tables.copy()
    bt[2, 3] = int(bt[2, 24])  # a private block of sequence 2 swapped into its prefix
    w.block_tables = bt
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cascade_i8(DevWorkload(w), 384, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & P.FLAG_BAD_PREFIX
