"""GPU parity of the tcgen05 paged prefill kernel against the fp64 oracle: variable query lengths
(1 to several 128-row tiles, ragged), cached prefixes, GQA groups, and missing blocks."""
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


def run_prefill(w, status=None, bt=None):
    bt = w.block_tables if bt is None else bt
    out = torch.zeros((w.q.shape[0], w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    P.paged_prefill_attention(out, to_dev(w.q), to_dev(w.k_pool), to_dev(w.v_pool), to_dev(bt),
                              to_dev(w.context_lens), to_dev(w.query_start), w.max_query_len,
                              w.scale, status)
    return to_f64(out)


# G = 4, 1, 8, 3, 2, 16: the kernel runs one query head per CTA (no clusters); each GQA group size
# changes which kv head a CTA's head reads and how the heads of a group fall on the grid
@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 8), (16, 2), (6, 2), (4, 2), (32, 2)])
def test_prefill_matches_oracle(hq, hkv):
    w = W.make_prefill(name="pf", query_lens=[1, 5, 127, 128, 129, 300],
                       cached_lens=[0, 17, 64, 200, 5, 1000], Hq=hq, Hkv=hkv, D=128, seed=hq + hkv)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_prefill(w, st)
    ref = oracle.paged_prefill_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                         w.query_start, w.scale)
    assert_close(got, ref, "bf16", f"prefill Hq={hq} Hkv={hkv}")
    assert int(st.item()) == 0


def test_prefill_batch_with_empty_sequences():
    """Sequences with no new tokens (one of them with no context at all) own no rows and launch no
    work; the others are unaffected."""
    w = W.make_prefill(name="pfz", query_lens=[0, 130, 0, 7], cached_lens=[5, 20, 0, 300], Hq=8,
                       Hkv=2, D=128, seed=3)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_prefill(w, st)
    ref = oracle.paged_prefill_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                         w.query_start, w.scale)
    assert_close(got, ref, "bf16", "prefill with empty sequences")
    assert int(st.item()) == 0


def test_prefill_single_token_rows_equal_decode():
    """A prefill chunk of one token per sequence is a decode step."""
    w = W.make_prefill(name="pf1", query_lens=[1, 1, 1, 1], cached_lens=[0, 15, 16, 700], Hq=32,
                       Hkv=8, D=128, seed=4)
    got = run_prefill(w)
    ref = oracle.paged_decode_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens, w.scale)
    assert_close(got, ref, "bf16", "prefill L=1")


def test_prefill_long_prompt():
    w = W.make_prefill(name="pfl", query_lens=[1000, 37], cached_lens=[2048, 3000], Hq=32, Hkv=8,
                       D=128, seed=8)
    got = run_prefill(w)
    rows = np.r_[0:64, 480:560, 936:1037]
    sub_q = w.q[rows]
    ref = oracle.paged_prefill_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                         w.query_start, w.scale)
    assert_close(got[rows], ref[rows], "bf16", "long prompt rows")
    assert sub_q.shape[0] == rows.size


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 4), (32, 4)])
def test_prefill_missing_block_is_skipped_and_flagged(hq, hkv):
    w = W.make_prefill(name="pfb", query_lens=[40, 70], cached_lens=[100, 30], Hq=hq, Hkv=hkv, D=128,
                       seed=9)
    bt = w.block_tables.copy()
    bt[0, 2] = w.NB + 5  # a block of sequence 0 outside the pool
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_prefill(w, st, bt)
    assert int(st.item()) & P.FLAG_BAD_BLOCK
    assert np.all(np.isfinite(got))
    ref = oracle.paged_prefill_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                         w.query_start, w.scale)
    s1 = slice(w.query_start[1], w.query_start[2])
    assert_close(got[s1], ref[s1], "bf16", "untouched sequence")


@pytest.mark.parametrize("scale", [-0.3, 2.0, 0.0])
def test_prefill_scale_sign_and_running_max_rescale(scale):
    """A negative scale flips which key dominates; a large one makes the running maximum jump by
    far more than the kernel's lazy-rescale margin across key tiles (the O rescale path); zero
    gives uniform weights over the visible keys."""
    w = W.make_prefill(name="pfs", query_lens=[300, 129], cached_lens=[700, 0], Hq=8, Hkv=2,
                       D=128, seed=17)
    w.scale = scale
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_prefill(w, st)
    ref = oracle.paged_prefill_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                         w.query_start, w.scale)
    assert_close(got, ref, "bf16", f"prefill scale={scale}")
    assert int(st.item()) == 0


@pytest.mark.parametrize("growth", [2.0, 6.0])
def test_prefill_reference_raised_on_alternate_tiles(growth):
    """Keys whose magnitude grows with their position, so that most 128-key tiles raise a row's
    reference maximum by more than the kernel's lazy margin of 2^8. The two softmax warps of a row
    take alternate tiles, so the raised reference is handed from one to the other on almost every
    tile, and O is rescaled on almost every tile, by either warp; query tiles with odd and even
    numbers of key tiles, a ragged last tile."""
    w = W.make_prefill(name="pfg", query_lens=[300, 129, 77], cached_lens=[700, 0, 333], Hq=8,
                       Hkv=2, D=128, seed=23)
    k = W.bf16_bits_to_f32(w.k_pool)
    for b in range(len(w.context_lens)):
        for pos in range(int(w.context_lens[b])):
            blk = w.block_tables[b][pos // w.BS]
            k[blk, :, pos % w.BS, :] *= np.float32(1.0 + growth * pos / 128.0)
    w.k_pool = W.f32_to_bf16_bits(k)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_prefill(w, st)
    ref = oracle.paged_prefill_attention(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                         w.query_start, w.scale)
    assert_close(got, ref, "bf16", f"prefill rising keys x{growth}")
    assert int(st.item()) == 0


def full_size_rows(w, per_seq=(0, 1, 2, 127, 128, 129, 2047, 2048, 4094, 4095)):
    """Rows of every sequence spread over the first, a middle and the last query tile (the tile
    edges, where the causal limit and the tile split meet)."""
    qs = np.asarray(w.query_start)
    return np.concatenate([qs[b] + np.asarray([i for i in per_seq if i < qs[b + 1] - qs[b]])
                           for b in range(len(qs) - 1)])


def test_prefill_full_size_sampled_rows():
    """The bench's prefill workload at full size (4 sequences x 4096 new tokens after 2048 cached,
    Llama-3-8B heads) through the same call the bench times, every head of sampled rows of every
    sequence against the oracle (each row as the decode query it is)."""
    import os
    w = W.make_prefill(name="prefill_llama3_8b", query_lens=[4096] * 4, cached_lens=[2048] * 4,
                       Hq=32, Hkv=8, D=128, seed=7)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_prefill(w, st)
    rows = full_size_rows(w)
    ref = prefill_rows_by_decode(w, rows, num_threads=os.cpu_count() or 8)
    assert_close(got[rows], ref, "bf16", f"full-size prefill, {rows.size} rows x 32 heads")
    assert np.all(np.isfinite(got))
    assert int(st.item()) == 0
