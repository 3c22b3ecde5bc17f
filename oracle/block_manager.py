"""Plain-Python statement of the host block manager -- TEST INFRASTRUCTURE ONLY.

Follows the "AMD ATOM inference engine" page, section 5.1 (Block with block_id, ref_count,
hash = -1 and token_ids; reset() sets ref_count to 1; a block_table per sequence) and section 5.2
(compute_hash: xxhash64 over the previous block's hash as 8 little-endian bytes, when there is
one, then the token ids as int64 bytes), and "LLM Primer VI, Chapter 8", section 8.1 (blocks
shared through reference counts). Readings where the pages are silent: free blocks are taken
first-in first-out starting at block 0; a freed block goes to the back of the free list (tail
block of a sequence first) and keeps its hash until it is taken again; only full blocks are
hashed and shared. XXH64 is written out here from the algorithm's published definition.
"""
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


def compute_hash(token_ids, prefix: int = -1) -> int:
    data = b""
    if prefix != -1:
        data += int(prefix).to_bytes(8, "little")
    data += np.asarray(token_ids, dtype=np.int64).tobytes()
    return xxh64(data)


class Block:
    def __init__(self, block_id):
        self.block_id = block_id
        self.ref_count = 0
        self.hash = -1
        self.token_ids = []

    def update(self, h, token_ids):
        self.hash = h
        self.token_ids = list(token_ids)

    def reset(self):
        self.ref_count = 1
        self.hash = -1
        self.token_ids = []


class BlockManager:
    def __init__(self, num_blocks, block_size=16, prefix_cache=True):
        self.block_size = block_size
        self.prefix_cache = prefix_cache
        self.blocks = [Block(i) for i in range(num_blocks)]
        self.free = deque(range(num_blocks))
        self.hash_to_block = {}
        self.seqs = {}  # id -> dict(table, tokens, last_hash)

    def _take_free(self):
        bid = self.free.popleft()
        blk = self.blocks[bid]
        if blk.hash != -1 and self.hash_to_block.get(blk.hash) == bid:
            del self.hash_to_block[blk.hash]
        blk.reset()
        return bid

    def _seal(self, s, bid, toks):
        if not self.prefix_cache:
            return
        h = compute_hash(toks, s["last_hash"])
        self.blocks[bid].update(h, toks)
        self.hash_to_block[h] = bid
        s["last_hash"] = h

    def can_allocate(self, n):
        return len(self.free) >= -(-n // self.block_size)

    def allocate(self, seq_id, token_ids):
        assert seq_id not in self.seqs
        if not self.can_allocate(len(token_ids)):
            raise MemoryError("no blocks")
        s = dict(table=[], tokens=list(token_ids), last_hash=-1)
        bs, cached = self.block_size, 0
        for i in range(0, len(token_ids), bs):
            toks = list(token_ids[i:i + bs])
            bid = None
            if len(toks) == bs and self.prefix_cache:
                h = compute_hash(toks, s["last_hash"])
                hit = self.hash_to_block.get(h)
                if hit is not None and self.blocks[hit].token_ids == toks:
                    bid = hit
                    if self.blocks[bid].ref_count == 0:
                        self.free.remove(bid)
                    self.blocks[bid].ref_count += 1
                    cached += bs
                    s["last_hash"] = h
            if bid is None:
                bid = self._take_free()
                if len(toks) == bs:
                    self._seal(s, bid, toks)
            s["table"].append(bid)
        self.seqs[seq_id] = s
        return cached

    def can_append(self, seq_id, k):
        s = self.seqs[seq_id]
        need = -(-(len(s["tokens"]) + k) // self.block_size) - len(s["table"])
        return need <= 0 or len(self.free) >= need

    def append(self, seq_id, token_ids):
        if not self.can_append(seq_id, len(token_ids)):
            raise MemoryError("no blocks")
        s, bs, slots = self.seqs[seq_id], self.block_size, []
        for t in token_ids:
            pos = len(s["tokens"])
            if pos % bs == 0:
                s["table"].append(self._take_free())
            bid = s["table"][pos // bs]
            slots.append(bid * bs + pos % bs)
            s["tokens"].append(int(t))
            if pos % bs == bs - 1:
                self._seal(s, bid, s["tokens"][pos + 1 - bs:pos + 1])
        return np.array(slots, dtype=np.int64)

    def free_seq(self, seq_id):
        for bid in reversed(self.seqs.pop(seq_id)["table"]):
            self.blocks[bid].ref_count -= 1
            if self.blocks[bid].ref_count == 0:
                self.free.append(bid)

    def batch_tables(self, seq_ids, mbps):
        bt = np.full((len(seq_ids), mbps), -1, dtype=np.int32)
        cl = np.zeros(len(seq_ids), dtype=np.int32)
        for i, sid in enumerate(seq_ids):
            t = self.seqs[sid]["table"]
            bt[i, :len(t)] = t
            cl[i] = len(self.seqs[sid]["tokens"])
        return bt, cl
