"""Plain-Python statement of the host block manager -- TEST INFRASTRUCTURE ONLY.

What it states, from the pages:
- "AMD ATOM inference engine", section 5.1: the KV cache is managed as fixed blocks of 16 tokens;
  every sequence keeps a table of the blocks it occupies; a block records how many sequences use
  it (its reference count), and a block taken from the free list starts with one user and no
  cached contents.
- Same page, section 5.2: prefix caching identifies a full block by a chained xxhash64 -- the
  hash of the block before it (8 bytes, little-endian; absent for a sequence's first block)
  followed by the block's token ids as 64-bit little-endian integers -- so that equal tokens in a
  different context hash differently.
- "LLM Primer VI, Chapter 8", section 8.1: sequences share physical blocks by reference count;
  best-of-n sampling on one prompt holds the prompt once.

Readings where the pages are silent (each listed in the design notes): free blocks are taken
first-in first-out starting at block 0; a freed block goes to the back of the free list (tail
block of a sequence first) and keeps its hash until it is taken again; only full blocks are
hashed and shared through the cache. Forking (parallel sampling) makes the child reference every
block of its parent. Copy-on-write: a sequence about to write into a block that other sequences
also reference (only a partly filled tail block can be, after a fork) first takes a free block,
drops its reference to the shared one and reports the copy (source, destination) that the
caller makes on the device; the last sequence still referencing the block writes in place.

XXH64 is written out here from the algorithm's published definition.
"""
import struct
from collections import deque

import numpy as np

_M = (1 << 64) - 1
P1, P2, P3, P4, P5 = (0x9E3779B185EBCA87, 0xC2B2AE3D27D4EB4F, 0x165667B19E3779F9,
                      0x85EBCA77C2B2AE63, 0x27D4EB2F165667C5)


def _rotl(x, r):
    return ((x << r) | (x >> (64 - r))) & _M


def _round(acc, lane):
    return (_rotl((acc + lane * P2) & _M, 31) * P1) & _M


def xxh64(data: bytes, seed: int = 0) -> int:
    n = len(data)
    i = 0
    if n >= 32:
        v = [(seed + P1 + P2) & _M, (seed + P2) & _M, seed & _M, (seed - P1) & _M]
        while i + 32 <= n:
            for j in range(4):
                v[j] = _round(v[j], int.from_bytes(data[i + 8 * j:i + 8 * j + 8], "little"))
            i += 32
        h = (_rotl(v[0], 1) + _rotl(v[1], 7) + _rotl(v[2], 12) + _rotl(v[3], 18)) & _M
        for j in range(4):
            h = ((h ^ _round(0, v[j])) * P1 + P4) & _M
    else:
        h = (seed + P5) & _M
    h = (h + n) & _M
    while i + 8 <= n:
        h = (_rotl(h ^ _round(0, int.from_bytes(data[i:i + 8], "little")), 27) * P1 + P4) & _M
        i += 8
    if i + 4 <= n:
        h = (_rotl(h ^ ((int.from_bytes(data[i:i + 4], "little") * P1) & _M), 23) * P2 + P3) & _M
        i += 4
    while i < n:
        h = (_rotl(h ^ ((data[i] * P5) & _M), 11) * P1) & _M
        i += 1
    h ^= h >> 33
    h = (h * P2) & _M
    h ^= h >> 29
    h = (h * P3) & _M
    h ^= h >> 32
    return h


def chain_hash(token_ids, previous=None) -> int:
    """The chained block hash: XXH64 (seed 0) of the previous full block's hash as 8 little-endian
    bytes (nothing when the block is the sequence's first) followed by the tokens as int64 LE."""
    head = b"" if previous is None else struct.pack("<Q", previous & _M)
    return xxh64(head + struct.pack(f"<{len(token_ids)}q", *[int(t) for t in token_ids]))


class BlockManager:
    """The manager's state is three per-block arrays (users, cache key, cached tokens), a FIFO of
    free block ids, a map from cache key to block, and one record per live sequence: its block
    table, its tokens and the key of its last full block (the link of its hash chain)."""

    def __init__(self, num_blocks, block_size=16, prefix_cache=True):
        self.block_size = block_size
        self.prefix_cache = prefix_cache
        self.users = [0] * num_blocks        # sequences whose table holds the block
        self.key = [None] * num_blocks       # chained hash of a full cached block, else None
        self.cached_tokens = [None] * num_blocks
        self.free = deque(range(num_blocks))
        self.by_key = {}
        self.seqs = {}                       # id -> {"table": [...], "tokens": [...], "link": key}

    def ref_count(self, block):
        return self.users[block]

    # -- free list ---------------------------------------------------------------------------
    def _take(self):
        """Front of the free list; whatever the block cached is forgotten; one user."""
        b = self.free.popleft()
        k = self.key[b]
        if k is not None and self.by_key.get(k) == b:
            del self.by_key[k]
        self.key[b] = None
        self.cached_tokens[b] = None
        self.users[b] = 1
        return b

    def _filled(self, rec, b, toks):
        """Block b of sequence rec just became full: it enters the cache under its chained key."""
        if not self.prefix_cache:
            return
        k = chain_hash(toks, rec["link"])
        self.key[b] = k
        self.cached_tokens[b] = list(toks)
        self.by_key[k] = b
        rec["link"] = k

    # -- prefill -----------------------------------------------------------------------------
    def can_allocate(self, n):
        return len(self.free) >= -(-n // self.block_size)

    def allocate(self, seq_id, token_ids):
        assert seq_id not in self.seqs
        if not self.can_allocate(len(token_ids)):
            raise MemoryError("no blocks")
        rec = {"table": [], "tokens": [int(t) for t in token_ids], "link": None}
        bs, hits = self.block_size, 0
        for start in range(0, len(token_ids), bs):
            toks = rec["tokens"][start:start + bs]
            full = len(toks) == bs
            if full and self.prefix_cache:
                k = chain_hash(toks, rec["link"])
                b = self.by_key.get(k)
                if b is not None and self.cached_tokens[b] == toks:  # a hit: share the block
                    if self.users[b] == 0:
                        self.free.remove(b)
                    self.users[b] += 1
                    rec["table"].append(b)
                    rec["link"] = k
                    hits += bs
                    continue
            b = self._take()
            if full:
                self._filled(rec, b, toks)
            rec["table"].append(b)
        self.seqs[seq_id] = rec
        return hits

    # -- parallel sampling ---------------------------------------------------------------------
    def fork(self, parent_id, child_id):
        assert parent_id in self.seqs and child_id not in self.seqs
        par = self.seqs[parent_id]
        for b in par["table"]:
            self.users[b] += 1
        self.seqs[child_id] = {"table": list(par["table"]), "tokens": list(par["tokens"]),
                               "link": par["link"]}

    # -- decode ------------------------------------------------------------------------------
    def _blocks_needed(self, rec, k):
        n, bs = len(rec["tokens"]), self.block_size
        need = -(-(n + k) // bs) - len(rec["table"])
        if k > 0 and n % bs != 0 and self.users[rec["table"][-1]] > 1:
            need += 1  # the shared, partly filled tail block is copied first
        return need

    def can_append(self, seq_id, k):
        need = self._blocks_needed(self.seqs[seq_id], k)
        return need <= 0 or len(self.free) >= need

    def append(self, seq_id, token_ids):
        """Slots of the new tokens (block * block_size + offset) and the copies [(src, dst)]
        the caller must make on the device before writing them."""
        if not self.can_append(seq_id, len(token_ids)):
            raise MemoryError("no blocks")
        rec, bs = self.seqs[seq_id], self.block_size
        slots, copies = [], []
        for t in token_ids:
            pos = len(rec["tokens"])
            if pos % bs == 0:
                rec["table"].append(self._take())
            elif self.users[rec["table"][-1]] > 1:  # copy-on-write of the shared tail block
                src = rec["table"][-1]
                dst = self._take()
                self.users[src] -= 1
                rec["table"][-1] = dst
                copies.append((src, dst))
            b = rec["table"][-1]
            slots.append(b * bs + pos % bs)
            rec["tokens"].append(int(t))
            if pos % bs == bs - 1:
                self._filled(rec, b, rec["tokens"][pos + 1 - bs:])
        return np.array(slots, dtype=np.int64), copies

    def free_seq(self, seq_id):
        for b in reversed(self.seqs.pop(seq_id)["table"]):
            self.users[b] -= 1
            if self.users[b] == 0:
                self.free.append(b)

    def batch_tables(self, seq_ids, mbps):
        bt = np.full((len(seq_ids), mbps), -1, dtype=np.int32)
        cl = np.zeros(len(seq_ids), dtype=np.int32)
        for i, sid in enumerate(seq_ids):
            t = self.seqs[sid]["table"]
            bt[i, :len(t)] = t
            cl[i] = len(self.seqs[sid]["tokens"])
        return bt, cl
