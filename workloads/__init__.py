"""Seeded synthetic inputs for the paged-KV decode path.

This module is shared by the oracle side (tests, cpu baseline) and the CUDA side (tests,
bench). It draws random numbers and lays out pools and block tables; it holds none of the
method's arithmetic (no attention, no dequantisation, no split rule).

Workload shapes follow the pages' settings: 16-token blocks in a flat physical pool with
per-sequence block tables ("LLM Primer VI, Chapter 8", section 8.1); Llama-class GQA decode;
long contexts served by split-K ("EchoLLMServing inference framework notes", section 2);
an INT8 KV cache with per-token scales (same page, section 3); a shared system-prompt prefix
referenced by every sequence with a reference count (Chapter 8, sections 8.1 and 8.3, and the
"AMD ATOM inference engine" page, section 5.1, Block.ref_count).

Element encodings: fp32 -> float32 arrays; bf16 -> uint16 arrays of bf16 bit patterns
(round-to-nearest-even from float32); int8 -> int8 arrays plus float32 scales.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

BLOCK_SIZE = 16


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bf16 (ties to even); returns uint16 bit patterns.
    Inputs here are finite normal draws, so no NaN handling is needed."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def quantize_int8_rows(x: np.ndarray):
    """Per-row symmetric int8 input recipe: scale = absmax / 127 (float32), value =
    clip(rint(x / scale), -127, 127). Rows with absmax 0 get scale 1."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1)
    scale = (amax / np.float32(127.0)).astype(np.float32)
    scale = np.where(scale == 0, np.float32(1.0), scale).astype(np.float32)
    qv = np.clip(np.rint(x / scale[..., None]), -127, 127).astype(np.int8)
    return qv, scale


@dataclass
class BlockPool:
    """Host-side block-pool fixture: hands out physical block ids in a seeded random order and
    counts references per block (a block shared by k tables has ref_count k)."""
    num_blocks: int
    rng: np.random.Generator
    free: list = field(default_factory=list)
    ref_count: Optional[np.ndarray] = None

    def __post_init__(self):
        self.free = list(self.rng.permutation(self.num_blocks).astype(np.int64))
        self.ref_count = np.zeros(self.num_blocks, dtype=np.int32)

    def allocate(self, n: int) -> np.ndarray:
        if n > len(self.free):
            raise MemoryError(f"pool exhausted: need {n}, have {len(self.free)}")
        ids = np.array(self.free[:n], dtype=np.int32)
        del self.free[:n]
        self.ref_count[ids] += 1
        return ids

    def share(self, ids: np.ndarray):
        self.ref_count[ids] += 1

    @property
    def used(self) -> int:
        return int(np.count_nonzero(self.ref_count))


@dataclass
class DecodeWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    BS: int
    NB: int
    kv_dtype: str            # "f32" | "bf16" | "i8"
    q_dtype: str             # "f32" | "bf16"
    q: np.ndarray            # [B, Hq, D]
    k_pool: np.ndarray       # [NB, Hkv, BS, D]
    v_pool: np.ndarray
    block_tables: np.ndarray  # int32 [B, MBPS], unused entries -1
    context_lens: np.ndarray  # int32 [B], counts the new token
    slot_mapping: np.ndarray  # int64 [T]
    k_new: np.ndarray        # [T, Hkv, D]
    v_new: np.ndarray
    scale: float
    ref_count: np.ndarray    # int32 [NB]
    k_scales: Optional[np.ndarray] = None     # float32 [NB, Hkv, BS] (int8 only)
    v_scales: Optional[np.ndarray] = None
    k_new_scales: Optional[np.ndarray] = None  # float32 [T, Hkv]
    v_new_scales: Optional[np.ndarray] = None
    shared_prefix_blocks: int = 0
    k_new_src: Optional[np.ndarray] = None     # bf16 bits [T, Hkv, D]: unquantised new rows (int8)
    v_new_src: Optional[np.ndarray] = None

    @property
    def MBPS(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def T(self) -> int:
        return int(self.slot_mapping.shape[0])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.B else 0

    @property
    def group(self) -> int:
        return self.Hq // self.Hkv


def _draw(rng, shape, kind):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if kind == "f32":
        return x
    if kind == "bf16":
        return f32_to_bf16_bits(x)
    raise ValueError(kind)


def _draw_kv(rng, shape, kv_dtype):
    """Pool-shaped K or V draws; int8 pools are quantised per (block, head, token) row."""
    if kv_dtype == "i8":
        x = rng.standard_normal(size=shape, dtype=np.float32)
        return quantize_int8_rows(x)
    return _draw(rng, shape, kv_dtype), None


def make_decode(*, name, B, Hq, Hkv, D, context_lens, kv_dtype, q_dtype, seed,
                shared_prefix_tokens=0, pool_slack=0.10, min_pool_blocks=0, scale=None,
                block_size=BLOCK_SIZE, mbps=None) -> DecodeWorkload:
    """Lay out a paged decode step: sequence b has context_lens[b] tokens (the last one is the
    token this step writes). Physical blocks come from a shuffled pool; the first
    shared_prefix_tokens (a whole number of blocks) are one set of blocks referenced by every
    sequence."""
    rng = np.random.Generator(np.random.PCG64(seed))
    BS = block_size
    lens = np.asarray(context_lens, dtype=np.int64)
    assert lens.shape == (B,)
    assert shared_prefix_tokens % BS == 0
    npre = shared_prefix_tokens // BS
    if npre:
        assert np.all(lens > shared_prefix_tokens), "the new token must land in a private block"
    need = [(-(-int(n) // BS)) for n in lens]
    private = sum(max(0, n - npre) for n in need)
    unique = private + npre
    NB = max(int(math.ceil(unique * (1.0 + pool_slack))), unique, min_pool_blocks, 1)
    MBPS = mbps if mbps is not None else max(1, max(need) if B else 1)
    pool = BlockPool(NB, rng)
    prefix = pool.allocate(npre) if npre else np.zeros(0, np.int32)
    if npre:
        pool.ref_count[prefix] -= 1  # counted once per referencing table below
    bt = np.full((B, MBPS), -1, dtype=np.int32)
    for b in range(B):
        if npre:
            bt[b, :npre] = prefix
            pool.share(prefix)
        nb = need[b] - npre if npre else need[b]
        if nb > 0:
            bt[b, npre:npre + nb] = pool.allocate(nb)
    k_pool, k_scales = _draw_kv(rng, (NB, Hkv, BS, D), kv_dtype)
    v_pool, v_scales = _draw_kv(rng, (NB, Hkv, BS, D), kv_dtype)
    q = _draw(rng, (B, Hq, D), q_dtype)
    # one new token per sequence, at logical position n - 1
    slots = np.full(B, -1, dtype=np.int64)
    for b in range(B):
        n = int(lens[b])
        if n > 0:
            slots[b] = int(bt[b, (n - 1) // BS]) * BS + (n - 1) % BS
    if kv_dtype == "i8":
        # new rows arrive from the model in bf16; the pre-quantised copies follow the same recipe
        k_new_src = f32_to_bf16_bits(rng.standard_normal(size=(B, Hkv, D), dtype=np.float32))
        v_new_src = f32_to_bf16_bits(rng.standard_normal(size=(B, Hkv, D), dtype=np.float32))
        k_new, k_new_scales = quantize_int8_rows(bf16_bits_to_f32(k_new_src))
        v_new, v_new_scales = quantize_int8_rows(bf16_bits_to_f32(v_new_src))
    else:
        k_new_src = v_new_src = None
        k_new, k_new_scales = _draw_kv(rng, (B, Hkv, D), kv_dtype)
        v_new, v_new_scales = _draw_kv(rng, (B, Hkv, D), kv_dtype)
    return DecodeWorkload(
        name=name, B=B, Hq=Hq, Hkv=Hkv, D=D, BS=BS, NB=NB, kv_dtype=kv_dtype,
        q_dtype=q_dtype, q=q, k_pool=k_pool, v_pool=v_pool, block_tables=bt,
        context_lens=lens.astype(np.int32), slot_mapping=slots, k_new=k_new, v_new=v_new,
        scale=float(scale if scale is not None else 1.0 / math.sqrt(D)),
        ref_count=pool.ref_count, k_scales=k_scales, v_scales=v_scales,
        k_new_scales=k_new_scales, v_new_scales=v_new_scales, shared_prefix_blocks=npre,
        k_new_src=k_new_src, v_new_src=v_new_src)


# --- the five workloads (sizes as the pages' settings suggest; see the design notes) ----------

CONFIGS = {
    1: "tiny paged decode: 4 seqs, ctx {1,17,33,100}, 4q/4kv, D=64, fp32, 64-block pool",
    2: "Llama-3-8B-shaped GQA decode: B=64, 32q/8kv, D=128, bf16, ctx U[512,4096]",
    3: "long-context split-K decode: B=8, 32q/8kv, D=128, bf16, ctx U[32768,131072]",
    4: "INT8 KV decode: B=128, 64q/8kv, D=128, int8 K/V + fp32 per-token scales, ctx U[1024,8192]",
    5: "prefix-shared decode: B=256, 32q/8kv, D=128, bf16, 2048-token shared prefix + U[16,2048]",
}


def make_config(cfg: int, seed: Optional[int] = None, *, B=None, ctx_lo=None, ctx_hi=None,
                prefix_tokens=None) -> DecodeWorkload:
    """Config `cfg` at full size, or reduced by overriding B / the context range / the prefix
    (parity runs at sizes the oracle finishes in seconds)."""
    seed = cfg if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(10_000 + seed))
    if cfg == 1:
        lens = [1, 17, 33, 100] if B is None else list(
            rng.integers(ctx_lo or 1, (ctx_hi or 100) + 1, size=B))
        return make_decode(name="tiny", B=len(lens), Hq=4, Hkv=4, D=64, context_lens=lens,
                           kv_dtype="f32", q_dtype="f32", seed=seed, min_pool_blocks=64,
                           pool_slack=0.0, scale=1.0 / 8.0)
    if cfg == 2:
        B = 64 if B is None else B
        lens = rng.integers(ctx_lo or 512, (ctx_hi or 4096) + 1, size=B)
        return make_decode(name="llama3_8b_gqa", B=B, Hq=32, Hkv=8, D=128, context_lens=lens,
                           kv_dtype="bf16", q_dtype="bf16", seed=seed)
    if cfg == 3:
        B = 8 if B is None else B
        lens = rng.integers(ctx_lo or 32768, (ctx_hi or 131072) + 1, size=B)
        return make_decode(name="long_splitk", B=B, Hq=32, Hkv=8, D=128, context_lens=lens,
                           kv_dtype="bf16", q_dtype="bf16", seed=seed)
    if cfg == 4:
        B = 128 if B is None else B
        lens = rng.integers(ctx_lo or 1024, (ctx_hi or 8192) + 1, size=B)
        return make_decode(name="int8_kv", B=B, Hq=64, Hkv=8, D=128, context_lens=lens,
                           kv_dtype="i8", q_dtype="bf16", seed=seed)
    if cfg == 5:
        B = 256 if B is None else B
        pre = 2048 if prefix_tokens is None else prefix_tokens
        suffix = rng.integers(ctx_lo or 16, (ctx_hi or 2048) + 1, size=B)
        return make_decode(name="prefix_shared", B=B, Hq=32, Hkv=8, D=128,
                           context_lens=pre + suffix, kv_dtype="bf16", q_dtype="bf16",
                           seed=seed, shared_prefix_tokens=pre)
    raise ValueError(f"unknown config {cfg}")


def permute_blocks(w: DecodeWorkload, seed: int) -> DecodeWorkload:
    """Same logical contents, physical blocks moved by a random permutation (data moved, tables
    rewritten)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    perm = rng.permutation(w.NB).astype(np.int32)  # old id -> new id
    inv = np.empty_like(perm)
    inv[perm] = np.arange(w.NB, dtype=np.int32)
    def move(a):
        return None if a is None else np.ascontiguousarray(a[inv])
    bt = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    slots = np.where(w.slot_mapping >= 0,
                     perm[np.maximum(w.slot_mapping // w.BS, 0)].astype(np.int64) * w.BS
                     + w.slot_mapping % w.BS, -1)
    return DecodeWorkload(**{**w.__dict__, "k_pool": move(w.k_pool), "v_pool": move(w.v_pool),
                             "k_scales": move(w.k_scales), "v_scales": move(w.v_scales),
                             "block_tables": bt, "slot_mapping": slots,
                             "ref_count": move(w.ref_count)})


def unshare_prefix(w: DecodeWorkload) -> DecodeWorkload:
    """Copy-on-write duplicate: every sequence gets private copies of the shared prefix blocks
    (appended to the pool), so no block is referenced twice."""
    npre = w.shared_prefix_blocks
    assert npre > 0
    pre = w.block_tables[0, :npre]
    new_ids = (w.NB + np.arange(w.B * npre, dtype=np.int32)).reshape(w.B, npre)
    def grow(a):
        if a is None:
            return None
        extra = np.concatenate([a[pre]] * w.B, axis=0)
        return np.ascontiguousarray(np.concatenate([a, extra], axis=0))
    bt = w.block_tables.copy()
    bt[:, :npre] = new_ids
    rc = np.concatenate([w.ref_count, np.ones(w.B * npre, np.int32)])
    rc[pre] = 0
    return DecodeWorkload(**{**w.__dict__, "NB": w.NB + w.B * npre, "k_pool": grow(w.k_pool),
                             "v_pool": grow(w.v_pool), "k_scales": grow(w.k_scales),
                             "v_scales": grow(w.v_scales), "block_tables": bt,
                             "ref_count": rc, "shared_prefix_blocks": 0})


def kv_bytes(w: DecodeWorkload, unique: bool = True) -> int:
    """Algorithmic HBM bytes of one decode step (write + attention), counted once per byte the
    step must move: K and V of every context token (the shared prefix once when unique=True),
    INT8 scales, q, out, the block-table entries in use, context_lens and the written tokens."""
    elem = {"f32": 4, "bf16": 2, "i8": 1}[w.kv_dtype]
    qe = {"f32": 4, "bf16": 2}[w.q_dtype]
    lens = w.context_lens.astype(np.int64)
    tokens = int(lens.sum())
    if unique and w.shared_prefix_blocks:
        tokens -= (w.B - 1) * w.shared_prefix_blocks * w.BS
    per_tok = w.Hkv * w.D * elem * 2 + (w.Hkv * 4 * 2 if w.kv_dtype == "i8" else 0)
    kv = tokens * per_tok
    qo = 2 * w.B * w.Hq * w.D * qe
    tables = 4 * int(((lens + w.BS - 1) // w.BS).sum()) + 4 * w.B
    written = int((w.slot_mapping >= 0).sum())
    wr = written * per_tok * 2 + 8 * w.T  # read new rows + write pool rows; slot ids
    return kv + qo + tables + wr


def make_multi_token(w: DecodeWorkload, L: int, seed: int) -> DecodeWorkload:
    """A multi-token decode step built on workload w: every sequence's last L context positions
    are new tokens (written this step, verified together, as MTP speculative decoding does with
    mtp_k + 1 tokens). q becomes [B, L, Hq, D]; slot_mapping / k_new / v_new cover the B * L
    new tokens, sequence-major. Needs context_lens >= L."""
    assert L >= 1 and (w.context_lens >= L).all()
    rng = np.random.Generator(np.random.PCG64(seed))
    B, Hkv, D = w.B, w.Hkv, w.D
    q = _draw(rng, (B, L, w.Hq, D), w.q_dtype)
    slots = np.empty(B * L, dtype=np.int64)
    for b in range(B):
        n = int(w.context_lens[b])
        for l in range(L):
            t = n - L + l
            slots[b * L + l] = int(w.block_tables[b, t // w.BS]) * w.BS + t % w.BS
    extra = {}
    if w.kv_dtype == "i8":
        ks = f32_to_bf16_bits(rng.standard_normal(size=(B * L, Hkv, D), dtype=np.float32))
        vs = f32_to_bf16_bits(rng.standard_normal(size=(B * L, Hkv, D), dtype=np.float32))
        kn, kns = quantize_int8_rows(bf16_bits_to_f32(ks))
        vn, vns = quantize_int8_rows(bf16_bits_to_f32(vs))
        extra = dict(k_new_src=ks, v_new_src=vs, k_new_scales=kns, v_new_scales=vns)
    else:
        kn, _ = _draw_kv(rng, (B * L, Hkv, D), w.kv_dtype)
        vn, _ = _draw_kv(rng, (B * L, Hkv, D), w.kv_dtype)
    return DecodeWorkload(**{**w.__dict__, "name": f"{w.name}_mtp{L}", "q": q,
                             "slot_mapping": slots, "k_new": kn, "v_new": vn, **extra})


@dataclass
class PrefillWorkload:
    """A paged (chunked) prefill step: sequence b has context_lens[b] tokens in the pool, of
    which its last L_b (query_start[b + 1] - query_start[b]) are this step's queries."""
    name: str
    Hq: int
    Hkv: int
    D: int
    BS: int
    NB: int
    q: np.ndarray             # bf16 bits [total, Hq, D]
    k_pool: np.ndarray        # bf16 bits [NB, Hkv, BS, D]
    v_pool: np.ndarray
    block_tables: np.ndarray  # int32 [B, MBPS]
    context_lens: np.ndarray  # int32 [B]
    query_start: np.ndarray   # int32 [B + 1]
    scale: float
    kv_dtype: str = "bf16"    # "bf16" or "i8"
    k_scales: Optional[np.ndarray] = None   # float32 [NB, Hkv, BS] (int8 only)
    v_scales: Optional[np.ndarray] = None

    @property
    def B(self):
        return int(self.context_lens.shape[0])

    @property
    def max_query_len(self):
        return int(np.diff(self.query_start).max()) if self.B else 0


def make_prefill(*, name, query_lens, cached_lens, Hq, Hkv, D, seed, pool_slack=0.10,
                 kv_dtype="bf16") -> PrefillWorkload:
    """Sequences with cached_lens[b] tokens already in the cache and query_lens[b] new prompt
    tokens (also in the cache, written before attention), blocks from a shuffled pool. An INT8
    cache ("i8") holds per-row quantised codes and fp32 scales (the decode workloads' recipe)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ql = np.asarray(query_lens, np.int64)
    cl = ql + np.asarray(cached_lens, np.int64)
    B = len(ql)
    need = [-(-int(n) // BLOCK_SIZE) for n in cl]
    NB = max(1, int(math.ceil(sum(need) * (1 + pool_slack))))
    pool = BlockPool(NB, rng)
    MBPS = max(1, max(need))
    bt = np.full((B, MBPS), -1, np.int32)
    for b in range(B):
        if need[b]:
            bt[b, :need[b]] = pool.allocate(need[b])
    kp, ks = _draw_kv(rng, (NB, Hkv, BLOCK_SIZE, D), kv_dtype)
    vp, vs = _draw_kv(rng, (NB, Hkv, BLOCK_SIZE, D), kv_dtype)
    qs = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    q = _draw(rng, (int(qs[-1]), Hq, D), "bf16")
    return PrefillWorkload(name=name, Hq=Hq, Hkv=Hkv, D=D, BS=BLOCK_SIZE, NB=NB, q=q, k_pool=kp,
                           v_pool=vp, block_tables=bt, context_lens=cl.astype(np.int32),
                           query_start=qs, scale=1.0 / math.sqrt(D), kv_dtype=kv_dtype,
                           k_scales=ks, v_scales=vs)
