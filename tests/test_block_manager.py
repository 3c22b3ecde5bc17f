"""The native host block manager (pkv_bm_*) against its plain-Python oracle and the pages' facts:
XXH64 against the system xxHash library, the chained block hash as the ATOM page defines it
(section 5.2), the best-of-8 token-slot count of the Chapter 8 primer (section 8.1), and the
manager's tables / slots / reference counts against the oracle on random operation scripts."""
import ctypes
import ctypes.util
import os

import numpy as np
import pytest

import paged_kv_decode_reshape_gb300 as P
from oracle import block_manager as O

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _system_xxh64():
    for name in ("libxxhash.so.0", ctypes.util.find_library("xxhash")):
        if not name:
            continue
        try:
            lib = ctypes.CDLL(name)
            lib.XXH64.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint64]
            lib.XXH64.restype = ctypes.c_uint64
            return lambda b, seed=0: int(lib.XXH64(ctypes.create_string_buffer(b, len(b)), len(b), seed))
        except OSError:
            continue
    return None


SYS_XXH64 = _system_xxh64()


def test_xxh64_empty_input_published_value(pkv):
    # the value the xxHash documentation gives for empty input, seed 0
    assert O.xxh64(b"") == 0xEF46DB3751D8E999
    assert P.xxh64(b"") == 0xEF46DB3751D8E999


@pytest.mark.skipif(SYS_XXH64 is None, reason="no system xxHash library")
def test_xxh64_matches_system_library_on_every_length_path(pkv):
    rng = np.random.default_rng(0)
    for n in list(range(0, 70)) + [95, 96, 97, 127, 128, 129, 255, 1000]:
        data = rng.integers(0, 256, n, dtype=np.uint8).tobytes()
        for seed in (0, 12345, 2**63 + 7):
            ref = SYS_XXH64(data, seed)
            assert P.xxh64(data, seed) == ref, (n, seed)
            assert O.xxh64(data, seed) == ref, (n, seed)


@pytest.mark.skipif(SYS_XXH64 is None, reason="no system xxHash library")
def test_block_hash_is_xxh64_of_prefix_then_int64_tokens(pkv):
    """ATOM section 5.2: h.update(prefix.to_bytes(8, 'little')) when prefix != -1, then
    h.update(np.array(token_ids).tobytes()), h.intdigest()."""
    toks = np.arange(100, 116, dtype=np.int64)
    first = SYS_XXH64(toks.tobytes())
    assert P.block_hash(toks) == first == O.compute_hash(toks)
    second = SYS_XXH64(first.to_bytes(8, "little") + (toks + 16).tobytes())
    assert P.block_hash(toks + 16, first) == second == O.compute_hash(toks + 16, first)
    # the same tokens under a different prefix hash differently
    assert P.block_hash(toks + 16, first) != P.block_hash(toks + 16)


def _read_gold(name):
    vals = {}
    for line in open(os.path.join(GOLD, name)):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            vals[k] = int(v)
    return vals


@pytest.mark.parametrize("prefix_cache,slots_key", [(True, "slots_with_sharing"),
                                                    (False, "slots_without_sharing")])
def test_best_of_8_token_slots_through_the_manager(pkv, prefix_cache, slots_key):
    g = _read_gold("best_of_8_token_slots.txt")
    n, prompt, new = g["samples"], g["prompt_tokens"], g["new_tokens_per_sample"]
    bm = P.BlockManager(4096, 16, prefix_cache)
    toks = np.random.default_rng(1).integers(0, 32000, prompt)
    cached = [bm.allocate(s, toks) for s in range(n)]
    assert cached == [0] + [prompt if prefix_cache else 0] * (n - 1)
    for s in range(n):
        bm.append(s, np.full(new, 7 + s))
    used_blocks = 4096 - bm.num_free_blocks
    token_slots = (prompt if prefix_cache else n * prompt) + n * new
    assert token_slots == g[slots_key]
    # whole blocks in use: the shared prompt once (125 blocks) plus each sample's own tail blocks
    per_tail = -(-new // 16)
    assert used_blocks == (prompt // 16 if prefix_cache else n * prompt // 16) + n * per_tail
    if prefix_cache:
        bt, cl = bm.batch_tables(list(range(n)), 140)
        assert (bt[:, :prompt // 16] == bt[0, :prompt // 16]).all()
        assert all(bm.ref_count(b) == n for b in bt[0, :prompt // 16])


def _compare(bm, ob, live):
    assert bm.num_free_blocks == len(ob.free)
    if live:
        mb = max(len(ob.seqs[s]["table"]) for s in live)
        a, ca = bm.batch_tables(live, mb)
        b, cb = ob.batch_tables(live, mb)
        assert np.array_equal(a, b) and np.array_equal(ca, cb)
    for i, blk in enumerate(ob.blocks):
        assert bm.ref_count(i) == blk.ref_count


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("prefix_cache", [True, False])
def test_manager_matches_oracle_on_random_scripts(pkv, seed, prefix_cache):
    rng = np.random.default_rng(seed)
    NB = 300
    bm, ob = P.BlockManager(NB, 16, prefix_cache), O.BlockManager(NB, 16, prefix_cache)
    system = rng.integers(0, 1000, 64)  # shared prompt prefixes of 0..4 blocks
    live, next_id = [], 0
    for _ in range(250):
        op = rng.random()
        if op < 0.35 or not live:
            n = int(rng.integers(1, 120))
            pre = int(rng.integers(0, 5)) * 16
            toks = np.concatenate([system[:pre], rng.integers(0, 1000, n)])
            ok = ob.can_allocate(len(toks))
            assert bm.can_allocate(len(toks)) == ok
            if ok:
                assert bm.allocate(next_id, toks) == ob.allocate(next_id, toks)
                live.append(next_id)
            else:
                with pytest.raises(P.PkvError):
                    bm.allocate(next_id, toks)
            next_id += 1
        elif op < 0.8:
            sid = live[int(rng.integers(len(live)))]
            k = int(rng.integers(1, 20))
            toks = rng.integers(0, 1000, k)
            ok = ob.can_append(sid, k)
            assert bm.can_append(sid, k) == ok
            if ok:
                assert np.array_equal(bm.append(sid, toks), ob.append(sid, toks))
                assert bm.context_len(sid) == len(ob.seqs[sid]["tokens"])
        else:
            sid = live.pop(int(rng.integers(len(live))))
            bm.free(sid)
            ob.free_seq(sid)
        _compare(bm, ob, live)


def test_exhaustion_and_errors_change_nothing(pkv):
    bm = P.BlockManager(4, 16)
    bm.allocate(1, np.arange(40))  # 3 blocks
    assert not bm.can_allocate(17)
    with pytest.raises(P.PkvError) as e:
        bm.allocate(2, np.arange(40))
    assert e.value.status == P.ERR_NO_BLOCKS and bm.num_free_blocks == 1
    assert bm.append(1, np.arange(8)).tolist() == [bm.batch_tables([1], 3)[0][0, 2] * 16 + 8 + i for i in range(8)]
    assert not bm.can_append(1, 17)  # 48 + 17 tokens need 5 blocks
    with pytest.raises(P.PkvError):
        bm.allocate(1, np.arange(3))   # known id
    with pytest.raises(P.PkvError):
        bm.free(99)                    # unknown id
    bm.free(1)
    assert bm.num_free_blocks == 4


def test_freed_prefix_blocks_are_found_again(pkv):
    bm = P.BlockManager(64, 16)
    toks = np.arange(200, 264)  # 4 full blocks
    bm.allocate(1, toks)
    first = bm.batch_tables([1], 4)[0][0].tolist()
    bm.free(1)
    assert bm.allocate(2, toks) == 64  # every block still cached on the free list
    assert bm.batch_tables([2], 4)[0][0].tolist() == first
