"""GPU parity of multi-token decode (MTP verification: L new tokens per sequence, causal among
themselves) against the fp64 oracle, for the bf16 / INT8 tensor-core kernel and the fp32
CUDA-core kernel."""
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


def _base(kind):
    if kind == "bf16":
        return W.make_config(2, B=5, ctx_lo=4, ctx_hi=1300, seed=17)
    if kind == "i8":
        return W.make_config(4, B=4, ctx_lo=4, ctx_hi=1300, seed=18)
    return W.make_decode(name="f32_d64", B=4, Hq=8, Hkv=2, D=64, context_lens=[4, 33, 250, 700],
                         kv_dtype="f32", q_dtype="f32", seed=19)


def _run(m, chunk, status=None):
    d = DevWorkload(m)
    d.write()
    out = torch.empty(m.q.shape, dtype=d.q.dtype, device="cuda")
    nbytes = P.decode_workspace_bytes(m.B * m.q.shape[1], m.Hq, m.Hkv, m.D, m.max_context_len, chunk)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda") if nbytes else None
    P.paged_decode_attention_multi(out, d.q, d.k_pool, d.v_pool, d.block_tables, d.context_lens,
                                   m.max_context_len, m.scale, d.k_scales, d.v_scales, chunk, ws,
                                   status)
    return to_f64(out)


def _oracle(m):
    kp, vp, ks, vs = oracle.kv_cache_write(m.k_new, m.v_new, m.k_pool, m.v_pool, m.slot_mapping,
                                           m.k_new_scales, m.v_new_scales, m.k_scales, m.v_scales)
    return oracle.paged_decode_attention_multi(m.q, kp, vp, m.block_tables, m.context_lens, m.scale,
                                               ks, vs)


@pytest.mark.parametrize("kind", ["bf16", "i8", "f32"])
@pytest.mark.parametrize("L", [1, 2, 4])
@pytest.mark.parametrize("chunk", [0, 64])
def test_multi_token_matches_oracle(kind, L, chunk):
    m = W.make_multi_token(_base(kind), L, seed=100 + L)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _run(m, chunk, st)
    assert_close(got, _oracle(m), kind, f"{kind} L={L} chunk={chunk}")
    assert int(st.item()) == 0


def test_one_query_token_equals_decode_bitwise():
    w = W.make_config(2, B=6, ctx_lo=20, ctx_hi=900, seed=23)
    m = W.make_multi_token(w, 1, seed=5)
    a = _run(m, 0)
    d = DevWorkload(W.DecodeWorkload(**{**m.__dict__, "q": m.q[:, 0]}))
    d.write()
    b = to_f64(d.attend())
    assert np.array_equal(a[:, 0], b)


def test_context_shorter_than_new_tokens_is_flagged():
    w = W.make_config(2, B=3, ctx_lo=2, ctx_hi=2, seed=29)
    L = 3
    q = W.f32_to_bf16_bits(np.ones((w.B, L, w.Hq, w.D), np.float32))
    d = DevWorkload(w)
    out = torch.empty((w.B, L, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    P.paged_decode_attention_multi(out, to_dev(q), d.k_pool, d.v_pool, d.block_tables,
                                   d.context_lens, 2, w.scale, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & P.FLAG_BAD_CONTEXT
    got = to_f64(out)
    assert np.all(got[:, 0] == 0) and np.all(np.isfinite(got))  # token 0 sees no context


@pytest.mark.parametrize("kv", ["bf16", "i8"])
@pytest.mark.parametrize("g,L", [(1, 3), (2, 4), (3, 3), (4, 2), (4, 5), (6, 2), (1, 8), (8, 2), (8, 4),
                                 (16, 2)])
def test_multi_token_packed_columns(kv, g, L):
    """When L * G query rows of a sequence's kv head fit the kernel's columns (8 or 16 per CTA)
    better than one token at a time, the tensor-core kernel packs (token, head) pairs as columns,
    each masked at its own causal limit; L * G not a multiple of the column count leaves a partial
    last column group. G = 8 with L = 2 or 4 takes the 16-column kernel, as G = 16 does."""
    Hkv = 2
    base = W.make_decode(name="mtp_pack", B=5, Hq=Hkv * g, Hkv=Hkv, D=128,
                         context_lens=[L, L + 1, 17, 300, 900], kv_dtype=kv, q_dtype="bf16",
                         seed=200 + 10 * g + L)
    m = W.make_multi_token(base, L, seed=300 + L)
    for chunk in (0, 64):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        got = _run(m, chunk, st)
        assert_close(got, _oracle(m), kv, f"{kv} G={g} L={L} chunk={chunk}")
        assert int(st.item()) == 0
