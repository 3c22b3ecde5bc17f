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
    assert P.block_hash(toks) == first == O.chain_hash(toks)
    second = SYS_XXH64(first.to_bytes(8, "little") + (toks + 16).tobytes())
    assert P.block_hash(toks + 16, first) == second == O.chain_hash(toks + 16, first)
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
    for i in range(len(ob.users)):
        assert bm.ref_count(i) == ob.ref_count(i)
    for s in live:
        assert bm.context_len(s) == len(ob.seqs[s]["tokens"])


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
@pytest.mark.parametrize("prefix_cache", [True, False])
def test_manager_matches_oracle_on_random_scripts(pkv, seed, prefix_cache):
    """Random allocate / fork / append / free scripts: the native manager's answers (cache hits,
    slots, copy-on-write copies, errors) and state (tables, lengths, reference counts, free
    count) equal the oracle's after every operation."""
    rng = np.random.default_rng(seed)
    NB = 300
    bm, ob = P.BlockManager(NB, 16, prefix_cache), O.BlockManager(NB, 16, prefix_cache)
    system = rng.integers(0, 1000, 64)  # shared prompt prefixes of 0..4 blocks
    live, next_id, copies_seen = [], 0, 0
    for _ in range(300):
        op = rng.random()
        if op < 0.3 or not live:
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
        elif op < 0.4:
            parent = live[int(rng.integers(len(live)))]
            bm.fork(parent, next_id)
            ob.fork(parent, next_id)
            live.append(next_id)
            next_id += 1
        elif op < 0.85:
            sid = live[int(rng.integers(len(live)))]
            k = int(rng.integers(1, 20))
            toks = rng.integers(0, 1000, k)
            ok = ob.can_append(sid, k)
            assert bm.can_append(sid, k) == ok
            if ok:
                slots, copies = bm.append_cow(sid, toks)
                oslots, ocopies = ob.append(sid, toks)
                assert np.array_equal(slots, oslots) and copies == ocopies
                copies_seen += len(copies)
                assert bm.context_len(sid) == len(ob.seqs[sid]["tokens"])
        else:
            sid = live.pop(int(rng.integers(len(live))))
            bm.free(sid)
            ob.free_seq(sid)
        _compare(bm, ob, live)
    assert copies_seen > 0  # the scripts do reach copy-on-write


def test_best_of_8_by_fork_through_the_manager(pkv):
    """Chapter 8 primer, section 8.1, through pkv_bm_*: one 2,000-token prompt, seven forks, 100
    new tokens per sample -> 2,800 token slots (16,800 unshared), the prompt's 125 blocks shared
    by all eight, each sample with 7 blocks of its own; with a 2,001-token prompt the shared tail
    block is copied for all but the last sample to write into it."""
    g = _read_gold("best_of_8_token_slots.txt")
    n, prompt, new = g["samples"], g["prompt_tokens"], g["new_tokens_per_sample"]
    for plen in (prompt, prompt + 1):
        bm = P.BlockManager(4096, 16)
        toks = np.random.default_rng(plen).integers(0, 32000, plen)
        assert bm.allocate(0, toks) == 0
        for c in range(1, n):
            bm.fork(0, c)
        slots, copies = set(), []
        for s in range(n):
            sl, cp = bm.append_cow(s, np.full(new, 7 + s))
            copies += cp
        for s in range(n):
            bt, cl = bm.batch_tables([s], 140)
            assert cl[0] == plen + new
            slots |= {int(bt[0, t // 16]) * 16 + t % 16 for t in range(plen + new)}
        # each copy holds its own duplicate of the prompt tokens in the shared tail block
        assert len(slots) == plen + n * new + (n - 1) * (plen % 16)
        if plen == prompt:
            assert len(slots) == g["slots_with_sharing"] and copies == []
            assert 4096 - bm.num_free_blocks == prompt // 16 + n * -(-new // 16)
        else:
            assert len(copies) == n - 1 and len({src for src, _ in copies}) == 1
        bt, _ = bm.batch_tables(list(range(n)), 140)
        assert (bt[:, :prompt // 16] == bt[0, :prompt // 16]).all()
        assert all(bm.ref_count(int(b)) == n for b in bt[0, :prompt // 16])
        for s in range(n):
            bm.free(s)
        assert bm.num_free_blocks == 4096


def test_fork_errors_and_append_without_copy_output(pkv):
    bm = P.BlockManager(8, 16)
    bm.allocate(1, np.arange(20))          # tail block holds 4 tokens
    with pytest.raises(P.PkvError):
        bm.fork(9, 2)                       # unknown parent
    bm.fork(1, 2)
    with pytest.raises(P.PkvError):
        bm.fork(1, 2)                       # known child id
    free = bm.num_free_blocks
    with pytest.raises(P.PkvError) as e:    # a copy is needed but the plain append cannot report it
        bm.append(2, [5])
    assert e.value.status == P.ERR_INVALID_ARG
    assert bm.num_free_blocks == free and bm.context_len(2) == 20
    slots, copies = bm.append_cow(2, [5])
    assert len(copies) == 1 and bm.num_free_blocks == free - 1
    assert bm.append(1, [6]).tolist() == [copies[0][0] * 16 + 4]  # the last user writes in place


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


# ---- fork and copy-on-write: pins of the oracle itself ------------------------------------------

def _read_slots(pool, table, n, bs=16):
    """The tokens a sequence sees: logical position t read through its table from the pool."""
    return [pool[table[t // bs] * bs + t % bs] for t in range(n)]


def _play(ob, pool, seq_id, toks):
    """Append through the oracle and apply what it reports to a token-per-slot pool: the copies
    first (whole blocks), then the new tokens into their slots."""
    slots, copies = ob.append(seq_id, toks)
    for src, dst in copies:
        pool[dst * 16:(dst + 1) * 16] = pool[src * 16:(src + 1) * 16]
    for sl, t in zip(slots, toks):
        pool[int(sl)] = int(t)
    return copies


@pytest.mark.parametrize("prompt_len", [2000, 2001, 2013, 15, 16, 1])
def test_oracle_fork_and_copy_on_write_keep_every_sequence_its_own_tokens(prompt_len):
    """Best-of-8 by forking: whatever the prompt length, every sample must read back exactly its
    own tokens through its table after all samples appended (in interleaved order) -- which
    fails if a sample writes into a block another sample still references, or if a copy goes the
    wrong way -- and the prompt's full blocks stay shared."""
    rng = np.random.default_rng(prompt_len)
    ob = O.BlockManager(2048, 16)
    pool = [None] * (2048 * 16)
    prompt = [int(t) for t in rng.integers(0, 32000, prompt_len)]
    ob.allocate(0, prompt)
    for sl, t in zip(range(prompt_len), prompt):
        tb = ob.seqs[0]["table"]
        pool[tb[sl // 16] * 16 + sl % 16] = t
    for c in range(1, 8):
        ob.fork(0, c)
    own = {s: list(prompt) for s in range(8)}
    ncopies = 0
    for step in range(100):
        for s in rng.permutation(8):
            t = int(rng.integers(0, 32000))
            ncopies += len(_play(ob, pool, int(s), [t]))
            own[int(s)].append(t)
    for s in range(8):
        rec = ob.seqs[s]
        assert rec["tokens"] == own[s]
        assert _read_slots(pool, rec["table"], len(own[s])) == own[s]
    partial = prompt_len % 16 != 0
    assert ncopies == (7 if partial else 0)     # all but the last writer of the shared tail copy
    full = prompt_len // 16
    for j in range(full):                        # full prompt blocks: still one shared copy
        assert len({ob.seqs[s]["table"][j] for s in range(8)}) == 1
        assert ob.ref_count(ob.seqs[0]["table"][j]) == 8
    for s in range(8):
        ob.free_seq(s)
    assert len(ob.free) == 2048 and all(u == 0 for u in ob.users)


def test_oracle_best_of_8_by_fork_gives_the_pages_token_slots():
    """Chapter 8 primer, section 8.1: best-of-8 on a 2,000-token prompt holds 2,800 token slots
    instead of 16,800 (tests/golden/best_of_8_token_slots.txt), here by forking one prompt."""
    g = _read_gold("best_of_8_token_slots.txt")
    n, prompt, new = g["samples"], g["prompt_tokens"], g["new_tokens_per_sample"]
    ob = O.BlockManager(4096, 16)
    ob.allocate(0, list(range(prompt)))
    for c in range(1, n):
        ob.fork(0, c)
    copies = []
    for s in range(n):
        copies += ob.append(s, [7 + s] * new)[1]
    assert copies == []                        # 2,000 tokens fill 125 blocks: nothing to copy
    slots = set()
    for s in range(n):
        rec = ob.seqs[s]
        slots |= {rec["table"][t // 16] * 16 + t % 16 for t in range(len(rec["tokens"]))}
    assert len(slots) == g["slots_with_sharing"]
    assert n * (prompt + new) == g["slots_without_sharing"]
    assert 4096 - len(ob.free) == prompt // 16 + n * -(-new // 16)


def test_oracle_can_append_counts_the_copy():
    ob = O.BlockManager(4, 16)
    ob.allocate(0, list(range(20)))             # 2 blocks, the second holds 4 tokens
    ob.fork(0, 1)
    assert ob.can_append(0, 1)                  # 2 free: the copy takes one
    ob.allocate(2, list(range(100, 117)))       # takes the last 2
    assert not ob.can_append(0, 1)              # the copy needs a block, none is free
    assert not ob.can_append(1, 12)
    ob.free_seq(2)
    slots, copies = ob.append(1, [5])
    assert len(copies) == 1 and copies[0][0] == ob.seqs[0]["table"][1]
    slots, copies = ob.append(0, [6])           # now the only user: writes in place
    assert copies == [] and int(slots[0]) == ob.seqs[0]["table"][1] * 16 + 4


def test_oracle_chain_hash_links_blocks():
    """Section 5.2: a block's hash covers the previous block's hash, so equal tokens in another
    context hash differently; the first block of a sequence hashes its tokens alone."""
    toks = list(range(500, 516))
    first = O.chain_hash(toks)
    assert first == O.xxh64(np.asarray(toks, dtype="<i8").tobytes())
    assert O.chain_hash(toks, first) == O.xxh64(first.to_bytes(8, "little") + np.asarray(toks, dtype="<i8").tobytes())
    assert O.chain_hash(toks, first) != first
    if SYS_XXH64 is not None:
        assert first == SYS_XXH64(np.asarray(toks, dtype="<i8").tobytes())


def test_oracle_prefix_hits_count_their_references():
    """A second prompt with the same first blocks shares them (section 5.2 with the reference
    counts of section 5.1): each shared block has two users, and freeing one sequence keeps them
    out of the free list until the other goes too."""
    ob = O.BlockManager(16, 16)
    prompt = list(range(1000, 1040))            # 2 full blocks + 8 tokens
    assert ob.allocate(0, prompt) == 0
    assert ob.allocate(1, prompt) == 32
    t0, t1 = ob.seqs[0]["table"], ob.seqs[1]["table"]
    assert t0[:2] == t1[:2] and t0[2] != t1[2]
    assert [ob.ref_count(b) for b in t0] == [2, 2, 1]
    ob.free_seq(0)
    assert t1[0] not in ob.free and t1[1] not in ob.free and len(ob.free) == 16 - 3
    ob.free_seq(1)
    assert len(ob.free) == 16 and all(u == 0 for u in ob.users)


@pytest.mark.parametrize("prefix_cache", [True, False])
def test_decode_loop_preempting_from_the_tail_matches_oracle(pkv, prefix_cache):
    """Decode scheduling on a small pool ("AMD ATOM inference engine", section 5: can_append before
    each decode step, preemption when the KV blocks run out): every running sequence appends one
    token per step; when the pool cannot take a sequence's token, the most recently admitted
    running sequence (the tail of the running queue) is preempted -- its blocks freed -- until it
    can, or until the sequence itself is the one preempted. The native manager and the oracle
    agree on every decision and on every slot, table and free count; preempted sequences are
    admitted again (recomputed from their tokens) when the whole prompt fits."""
    rng = np.random.default_rng(11)
    NB = 14
    bm, ob = P.BlockManager(NB, 16, prefix_cache), O.BlockManager(NB, 16, prefix_cache)
    tokens = {sid: list(rng.integers(0, 1000, int(rng.integers(5, 40)))) for sid in range(8)}
    waiting, running, preemptions, next_id, ids = list(range(8)), [], 0, 100, {}
    for step in range(80):
        # admit waiting sequences (first come, first served) while their tokens fit
        while waiting and ob.can_allocate(len(tokens[waiting[0]])):
            s = waiting.pop(0)
            assert bm.can_allocate(len(tokens[s]))
            ids[s], next_id = next_id, next_id + 1   # a re-admitted sequence gets a fresh id
            assert bm.allocate(ids[s], tokens[s]) == ob.allocate(ids[s], tokens[s])
            running.append(s)
        if waiting:
            assert not bm.can_allocate(len(tokens[waiting[0]]))
        for s in list(running):
            if s not in running:
                continue
            while not ob.can_append(ids[s], 1):
                assert not bm.can_append(ids[s], 1)
                victim = running.pop()                # the tail of the running queue
                bm.free(ids[victim])
                ob.free_seq(ids[victim])
                waiting.insert(0, victim)             # back to the head of the waiting queue
                preemptions += 1
                if victim == s:
                    break
            if s not in running:
                continue
            assert bm.can_append(ids[s], 1)
            t = [int(rng.integers(0, 1000))]
            slots, copies = bm.append_cow(ids[s], t)
            oslots, ocopies = ob.append(ids[s], t)
            assert np.array_equal(slots, oslots) and copies == ocopies
            tokens[s] += t
        _compare(bm, ob, [ids[s] for s in running])
    assert preemptions > 0 and running   # the pool did run out, and decoding went on
