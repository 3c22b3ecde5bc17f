"""Pool contents the kernels must not let through, and output bytes they must not touch.

Every pool position that no sequence's context reaches is filled with NaN before the call: the
tail of each sequence's last block (the slots past its length) and every block no table
references. For bf16 / fp32 pools that is the K and V rows; for an INT8 cache the K and V scales
(the codes are bytes, finite whatever they hold). A paged cache reuses blocks, so such slots hold
stale or never-written data ("LLM Primer VI, Chapter 8", section 8.1: a block's slots past the
sequence's length hold no token of it). The oracle reads only the first context_len positions of
each table, so the results must equal its answer, finite. The output buffer is framed by guard rows
of a fixed bit pattern, which must come back unchanged.
"""
import numpy as np
import pytest

import oracle
import paged_kv_decode_reshape_gb300 as P
import workloads as W
from _gpu import DevWorkload, assert_close, oracle_step, poisoned, to_dev, to_f64

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

GUARD = 3                # guard rows before and after the output


@pytest.fixture(scope="module", autouse=True)
def _lib(pkv):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def guarded(shape, dtype):
    """An output of `shape` inside a buffer with GUARD rows of a bit pattern on either side."""
    full = torch.empty((shape[0] + 2 * GUARD,) + tuple(shape[1:]), dtype=dtype, device="cuda")
    bits = full.view(torch.int16) if full.element_size() == 2 else full.view(torch.int32)
    bits.fill_(0x5A5A if full.element_size() == 2 else 0x5A5A5A5A)
    return full, full[GUARD:GUARD + shape[0]]


def assert_guards_intact(full, n):
    bits = full.view(torch.int16) if full.element_size() == 2 else full.view(torch.int32)
    pat = 0x5A5A if full.element_size() == 2 else 0x5A5A5A5A
    assert bool((bits[:GUARD] == pat).all()), "guard rows before the output were written"
    assert bool((bits[GUARD + n:] == pat).all()), "guard rows after the output were written"


REDUCED = {
    1: dict(),
    2: dict(B=6, ctx_lo=1, ctx_hi=1500),
    3: dict(B=2, ctx_lo=3000, ctx_hi=9000),
    4: dict(B=5, ctx_lo=17, ctx_hi=3000),
    5: dict(B=6, ctx_lo=16, ctx_hi=300, prefix_tokens=256),
}


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("chunk", [0, 64])
def test_decode_ignores_dead_slots_and_keeps_guards(cfg, chunk):
    w = poisoned(W.make_config(cfg, seed=40 + cfg, **REDUCED[cfg]))
    d = DevWorkload(w)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    full, out = guarded(d.q.shape, d.q.dtype)
    d.write(st)
    d.attend(chunk, st, out=out)
    torch.cuda.synchronize()
    assert_close(to_f64(out), oracle_step(w), w.kv_dtype, f"config {cfg} chunk {chunk}, NaN in dead slots")
    assert_guards_intact(full, w.B)
    assert int(st.item()) == 0


@pytest.mark.parametrize("kind", ["bf16", "i8"])
def test_shared_prefix_cascade_ignores_dead_slots(kind):
    prefix = 256
    if kind == "bf16":
        w = W.make_config(5, B=7, ctx_lo=1, ctx_hi=300, prefix_tokens=prefix, seed=61)
    else:
        rng = np.random.default_rng(62)
        lens = prefix + rng.integers(1, 301, size=7)
        w = W.make_decode(name="casc_i8", B=7, Hq=16, Hkv=2, D=128, context_lens=lens, kv_dtype="i8",
                          q_dtype="bf16", seed=62, shared_prefix_tokens=prefix)
    w = poisoned(w)
    d = DevWorkload(w)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    nbytes = P.decode_shared_prefix_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, w.max_context_len, prefix, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    full, out = guarded(d.q.shape, d.q.dtype)
    if kind == "bf16":
        P.paged_decode_attention_shared_prefix(out, d.q, d.k_pool, d.v_pool, d.block_tables,
                                               d.context_lens, w.max_context_len, w.scale, prefix, 0,
                                               ws, st)
    else:
        P.paged_decode_attention_shared_prefix_int8(out, d.q, d.k_pool, d.v_pool, d.k_scales,
                                                    d.v_scales, d.block_tables, d.context_lens,
                                                    w.max_context_len, w.scale, prefix, 0, ws, st)
    torch.cuda.synchronize()
    ref = oracle.paged_decode_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                        w.scale, w.k_scales, w.v_scales)
    assert_close(to_f64(out), ref, kind, f"{kind} cascade, NaN in dead slots")
    assert_guards_intact(full, w.B)
    assert int(st.item()) == 0


@pytest.mark.parametrize("kind", ["bf16", "i8", "f32"])
@pytest.mark.parametrize("L", [2, 4])
def test_multi_token_ignores_dead_slots_and_keeps_guards(kind, L):
    if kind == "bf16":
        base = W.make_config(2, B=5, ctx_lo=4, ctx_hi=1300, seed=71)
    elif kind == "i8":
        base = W.make_config(4, B=4, ctx_lo=4, ctx_hi=1300, seed=72)
    else:
        base = W.make_decode(name="f32_d64", B=4, Hq=8, Hkv=2, D=64, context_lens=[5, 33, 250, 700],
                             kv_dtype="f32", q_dtype="f32", seed=73)
    m = poisoned(W.make_multi_token(base, L, seed=74 + L))
    d = DevWorkload(m)
    d.write()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    nbytes = P.decode_workspace_bytes(m.B * m.q.shape[1], m.Hq, m.Hkv, m.D, m.max_context_len, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda") if nbytes else None
    full, out = guarded(d.q.shape, d.q.dtype)
    P.paged_decode_attention_multi(out, d.q, d.k_pool, d.v_pool, d.block_tables, d.context_lens,
                                   m.max_context_len, m.scale, d.k_scales, d.v_scales, 0, ws, st)
    torch.cuda.synchronize()
    kp, vp, ks, vs = oracle.kv_cache_write(m.k_new, m.v_new, m.k_pool, m.v_pool, m.slot_mapping,
                                           m.k_new_scales, m.v_new_scales, m.k_scales, m.v_scales)
    ref = oracle.paged_decode_attention_multi(m.q, kp, vp, m.block_tables, m.context_lens, m.scale, ks, vs)
    assert_close(to_f64(out), ref, kind, f"{kind} L={L}, NaN in dead slots")
    assert_guards_intact(full, m.B)
    assert int(st.item()) == 0


@pytest.mark.parametrize("kind", ["bf16", "i8"])
def test_prefill_ignores_dead_slots_and_keeps_guards(kind):
    # query lengths with ragged last tiles and a decode row; contexts ending mid-block
    w = poisoned(W.make_prefill(name="sentinel", query_lens=[300, 1, 77, 129], cached_lens=[21, 500, 0, 7],
                                Hq=8, Hkv=2, D=128, seed=81, kv_dtype=kind))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = to_dev(w.q)
    full, out = guarded((w.q.shape[0], w.Hq, w.D), torch.bfloat16)
    args = (to_dev(w.block_tables), to_dev(w.context_lens), to_dev(w.query_start), w.max_query_len,
            w.scale, st)
    if kind == "bf16":
        P.paged_prefill_attention(out, q, to_dev(w.k_pool), to_dev(w.v_pool), *args)
    else:
        P.paged_prefill_attention_int8(out, q, to_dev(w.k_pool), to_dev(w.v_pool), to_dev(w.k_scales),
                                       to_dev(w.v_scales), *args)
    torch.cuda.synchronize()
    ref = oracle.paged_prefill_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                         w.query_start, w.scale, w.k_scales, w.v_scales)
    tol = "bf16" if kind == "bf16" else "i8"
    assert_close(to_f64(out), ref, tol, f"{kind} prefill, NaN in dead slots")
    assert_guards_intact(full, w.q.shape[0])
    assert int(st.item()) == 0

