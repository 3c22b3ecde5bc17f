"""Paged KV-cache decode for GB300: Python binding of libpkv.so.

Argument marshalling only: every step of the path runs in the library's CUDA kernels. Tensors
are torch CUDA tensors (device memory and streams come from PyTorch); the calls and their
semantics are those of include/pkv.h. There is no CPU fallback: if libpkv.so cannot be loaded
(or built), every call raises.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA = range(5)
F32, BF16, I8 = 0, 1, 2
FLAG_BAD_SLOT, FLAG_BAD_BLOCK, FLAG_BAD_CONTEXT, FLAG_LONG_CONTEXT, FLAG_TIMEOUT = 1, 2, 4, 8, 16
FLAG_BAD_PREFIX = 32
BLOCK_SIZE = 16

# every exported symbol, with its ctypes signature (mirrors include/pkv.h)
_P, _I, _SZ, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
SIGNATURES = {
    "pkv_status_string": ([_I], ctypes.c_char_p),
    "pkv_version": ([], ctypes.c_char_p),
    "pkv_kv_cache_write": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "pkv_kv_cache_write_int8": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "pkv_decode_workspace_bytes": ([_I, _I, _I, _I, _I, _I], _SZ),
    "pkv_decode_workspace_bytes_dtype": ([_I, _I, _I, _I, _I, _I, _I], _SZ),
    "pkv_decode_split_chunk": ([_I, _I, _I, _I, _I, _I], _I),
    "pkv_paged_decode_attention": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F,
                                    _I, _I, _P, _SZ, _P, _P], _I),
    "pkv_paged_decode_attention_int8": ([_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                         _I, _I, _F, _I, _P, _SZ, _P, _P], _I),
    "pkv_paged_decode_attention_multi": ([_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                          _I, _I, _I, _F, _I, _I, _P, _SZ, _P, _P], _I),
    "pkv_paged_prefill_attention": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                     _I, _F, _P, _P], _I),
    "pkv_paged_prefill_attention_int8": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                          _I, _I, _I, _I, _F, _P, _P], _I),
    "pkv_paged_decode_attention_static_ws": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                              _I, _F, _I, _I, _P, _P], _I),
    "pkv_paged_decode_attention_shared_prefix": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                                  _I, _I, _F, _I, _I, _P, _SZ, _P, _P], _I),
    "pkv_decode_shared_prefix_workspace_bytes": ([_I, _I, _I, _I, _I, _I, _I], _SZ),
    "pkv_paged_decode_attention_shared_prefix_int8": ([_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I,
                                                       _I, _I, _I, _I, _I, _F, _I, _I, _P, _SZ, _P,
                                                       _P], _I),
    "pkv_kv_cache_copy_blocks": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P], _I),
}
STATIC_WORKSPACE_BYTES = 32 << 20  # PKV_STATIC_WORKSPACE_BYTES

_lib = None


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libpkv.so (building it in-tree first if it is missing or stale)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if build_if_missing and not _build.up_to_date():
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"libpkv.so not found at {path}: run __graft_entry__.build()")
        L = ctypes.CDLL(path)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def library_path() -> str:
    return _build.LIB


def status_string(status: int) -> str:
    return load().pkv_status_string(status).decode()


def version() -> str:
    return load().pkv_version().decode()


def _check(status: int, what: str):
    if status != OK:
        raise PkvError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _kv_code(t) -> int:
    import torch
    return {torch.float32: F32, torch.bfloat16: BF16, torch.int8: I8}[t.dtype]


def kv_cache_write(k_new, v_new, k_pool, v_pool, slot_mapping, k_new_scales=None,
                   v_new_scales=None, k_scales=None, v_scales=None, status=None, stream=None):
    """pkv_kv_cache_write on torch tensors: k_new/v_new [T, Hkv, D], pools [NB, Hkv, 16, D],
    slot_mapping int64 [T]; INT8 pools also take the four scale tensors."""
    T, Hkv, D = k_new.shape
    NB, _, BS, _ = k_pool.shape
    rc = load().pkv_kv_cache_write(
        _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool), _ptr(k_new_scales),
        _ptr(v_new_scales), _ptr(k_scales), _ptr(v_scales), _ptr(slot_mapping), T, Hkv, D, BS,
        NB, _kv_code(k_pool), _ptr(status), _stream(stream))
    _check(rc, "kv_cache_write")


def kv_cache_write_int8(k_new, v_new, k_pool, v_pool, k_scales, v_scales, slot_mapping,
                        status=None, stream=None):
    """pkv_kv_cache_write_int8: quantise fp32/bf16 rows k_new/v_new [T, Hkv, D] into int8 pools
    [NB, Hkv, 16, D] and fp32 scales [NB, Hkv, 16] at their slots."""
    T, Hkv, D = k_new.shape
    NB, _, BS, _ = k_pool.shape
    rc = load().pkv_kv_cache_write_int8(
        _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool), _ptr(k_scales), _ptr(v_scales),
        _ptr(slot_mapping), T, Hkv, D, BS, NB, _kv_code(k_new), _ptr(status), _stream(stream))
    _check(rc, "kv_cache_write_int8")


def kv_cache_copy_blocks(k_pool, v_pool, block_pairs, k_scales=None, v_scales=None, status=None,
                         stream=None):
    """pkv_kv_cache_copy_blocks: block_pairs is an int32 CUDA tensor [n, 2] of (src, dst)."""
    NB, Hkv, BS, D = k_pool.shape
    n = int(block_pairs.shape[0]) if block_pairs is not None else 0
    rc = load().pkv_kv_cache_copy_blocks(
        _ptr(k_pool), _ptr(v_pool), _ptr(k_scales), _ptr(v_scales), _ptr(block_pairs), n, Hkv, D,
        BS, NB, _kv_code(k_pool), _ptr(status), _stream(stream))
    _check(rc, "kv_cache_copy_blocks")


def decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len,
                           split_chunk_tokens=0) -> int:
    return int(load().pkv_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                 max_context_len, split_chunk_tokens))


def decode_workspace_bytes_dtype(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len,
                                 split_chunk_tokens=0, kv_dtype=BF16) -> int:
    """The exact workspace bytes of one decode call whose K/V pools have element type kv_dtype."""
    return int(load().pkv_decode_workspace_bytes_dtype(num_seqs, num_q_heads, num_kv_heads,
                                                       head_dim, max_context_len,
                                                       split_chunk_tokens, kv_dtype))


def decode_split_chunk(num_seqs, num_kv_heads, head_dim, max_context_len, split_chunk_tokens=0,
                       kv_dtype=BF16) -> int:
    """The chunk a decode call uses; kv_dtype is F32, BF16 or I8 (the pool's element type)."""
    return int(load().pkv_decode_split_chunk(num_seqs, num_kv_heads, head_dim, max_context_len,
                                             split_chunk_tokens, kv_dtype))


def paged_decode_attention(out, q, k_pool, v_pool, block_tables, context_lens, max_context_len,
                           scale, split_chunk_tokens=0, workspace=None, status=None,
                           stream=None):
    """pkv_paged_decode_attention: out/q [B, Hq, D] (fp32 or bf16), pools [NB, Hkv, 16, D] of
    the same dtype, block_tables int32 [B, MBPS], context_lens int32 [B]; workspace a uint8
    CUDA tensor of at least decode_workspace_bytes(...) bytes (None if that is 0)."""
    B, Hq, D = q.shape
    NB, Hkv, BS, _ = k_pool.shape
    rc = load().pkv_paged_decode_attention(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(context_lens),
        B, Hq, Hkv, D, BS, NB, block_tables.shape[1], int(max_context_len), float(scale),
        _kv_code(q), int(split_chunk_tokens), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _ptr(status),
        _stream(stream))
    _check(rc, "paged_decode_attention")


def decode_shared_prefix_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                         max_context_len, shared_prefix_tokens,
                                         split_chunk_tokens=0) -> int:
    return int(load().pkv_decode_shared_prefix_workspace_bytes(
        num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len, shared_prefix_tokens,
        split_chunk_tokens))


def paged_decode_attention_shared_prefix(out, q, k_pool, v_pool, block_tables, context_lens,
                                         max_context_len, scale, shared_prefix_tokens,
                                         split_chunk_tokens=0, workspace=None, status=None,
                                         stream=None):
    """pkv_paged_decode_attention_shared_prefix: bf16 q/out [B, Hq, 128], bf16 pools; the first
    shared_prefix_tokens tokens of every sequence are the blocks of block_tables row 0."""
    B, Hq, D = q.shape
    NB, Hkv, BS, _ = k_pool.shape
    rc = load().pkv_paged_decode_attention_shared_prefix(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(context_lens),
        B, Hq, Hkv, D, BS, NB, block_tables.shape[1], int(max_context_len), float(scale),
        int(shared_prefix_tokens), int(split_chunk_tokens), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _ptr(status),
        _stream(stream))
    _check(rc, "paged_decode_attention_shared_prefix")


def paged_decode_attention_shared_prefix_int8(out, q, k_pool, v_pool, k_scales, v_scales,
                                              block_tables, context_lens, max_context_len, scale,
                                              shared_prefix_tokens, split_chunk_tokens=0,
                                              workspace=None, status=None, stream=None):
    """pkv_paged_decode_attention_shared_prefix_int8: the cascade decode over an INT8 cache."""
    B, Hq, D = q.shape
    NB, Hkv, BS, _ = k_pool.shape
    rc = load().pkv_paged_decode_attention_shared_prefix_int8(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scales), _ptr(v_scales),
        _ptr(block_tables), _ptr(context_lens), B, Hq, Hkv, D, BS, NB, block_tables.shape[1],
        int(max_context_len), float(scale), int(shared_prefix_tokens), int(split_chunk_tokens),
        _ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(),
        _ptr(status), _stream(stream))
    _check(rc, "paged_decode_attention_shared_prefix_int8")


def paged_decode_attention_int8(out, q, k_pool, v_pool, k_scales, v_scales, block_tables,
                                context_lens, max_context_len, scale, split_chunk_tokens=0,
                                workspace=None, status=None, stream=None):
    """pkv_paged_decode_attention_int8: q/out bf16, pools int8, scales fp32 [NB, Hkv, 16]."""
    B, Hq, D = q.shape
    NB, Hkv, BS, _ = k_pool.shape
    rc = load().pkv_paged_decode_attention_int8(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scales), _ptr(v_scales),
        _ptr(block_tables), _ptr(context_lens), B, Hq, Hkv, D, BS, NB, block_tables.shape[1],
        int(max_context_len), float(scale), int(split_chunk_tokens), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _ptr(status),
        _stream(stream))
    _check(rc, "paged_decode_attention_int8")


def paged_decode_attention_multi(out, q, k_pool, v_pool, block_tables, context_lens,
                                 max_context_len, scale, k_scales=None, v_scales=None,
                                 split_chunk_tokens=0, workspace=None, status=None, stream=None):
    """pkv_paged_decode_attention_multi: q/out [B, L, Hq, D]; query token l of sequence b sees its
    first context_lens[b] - (L - 1 - l) tokens. INT8 pools take k_scales / v_scales."""
    B, L, Hq, D = q.shape
    NB, Hkv, BS, _ = k_pool.shape
    rc = load().pkv_paged_decode_attention_multi(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scales), _ptr(v_scales),
        _ptr(block_tables), _ptr(context_lens), B, L, Hq, Hkv, D, BS, NB, block_tables.shape[1],
        int(max_context_len), float(scale), _kv_code(k_pool), int(split_chunk_tokens),
        _ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(),
        _ptr(status), _stream(stream))
    _check(rc, "paged_decode_attention_multi")


def paged_prefill_attention(out, q, k_pool, v_pool, block_tables, context_lens, query_start,
                            max_query_len, scale, status=None, stream=None):
    """pkv_paged_prefill_attention: q/out [total, Hq, 128] bf16; sequence b's rows are
    query_start[b] .. query_start[b + 1] - 1, its last tokens, attending causally."""
    T, Hq, D = q.shape
    NB, Hkv, BS, _ = k_pool.shape
    rc = load().pkv_paged_prefill_attention(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(context_lens),
        _ptr(query_start), context_lens.shape[0], T, Hq, Hkv, D, BS, NB, block_tables.shape[1],
        int(max_query_len), float(scale), _ptr(status), _stream(stream))
    _check(rc, "paged_prefill_attention")


def paged_prefill_attention_int8(out, q, k_pool, v_pool, k_scales, v_scales, block_tables,
                                 context_lens, query_start, max_query_len, scale, status=None,
                                 stream=None):
    """pkv_paged_prefill_attention_int8: as paged_prefill_attention over int8 pools with their
    fp32 per-token scales [NB, Hkv, 16]."""
    T, Hq, D = q.shape
    NB, Hkv, BS, _ = k_pool.shape
    rc = load().pkv_paged_prefill_attention_int8(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scales), _ptr(v_scales),
        _ptr(block_tables), _ptr(context_lens), _ptr(query_start), context_lens.shape[0], T, Hq,
        Hkv, D, BS, NB, block_tables.shape[1], int(max_query_len), float(scale), _ptr(status),
        _stream(stream))
    _check(rc, "paged_prefill_attention_int8")


def paged_decode_attention_static_ws(out, q, k_pool, v_pool, block_tables, context_lens,
                                     max_context_len, scale, split_chunk_tokens=0, status=None,
                                     stream=None):
    """pkv_paged_decode_attention_static_ws: as paged_decode_attention, with the split-K partial
    states in the library's fixed device array instead of a caller-allocated workspace (for
    callers that cannot allocate device memory). Calls that overlap on the GPU race on that
    array."""
    B, Hq, D = q.shape
    NB, Hkv, BS, _ = k_pool.shape
    rc = load().pkv_paged_decode_attention_static_ws(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(context_lens),
        B, Hq, Hkv, D, BS, NB, block_tables.shape[1], int(max_context_len), float(scale),
        _kv_code(q), int(split_chunk_tokens), _ptr(status), _stream(stream))
    _check(rc, "paged_decode_attention_static_ws")


# ---- host block manager (ctypes marshalling of the pkv_bm_* calls) ---------------------------
ERR_NO_BLOCKS = 5
_BM_SIGNATURES = {
    "pkv_bm_create": ([_I, _I, _I], _P),
    "pkv_bm_destroy": ([_P], None),
    "pkv_bm_num_free_blocks": ([_P], _I),
    "pkv_bm_ref_count": ([_P, _I], _I),
    "pkv_xxh64": ([_P, _SZ, ctypes.c_uint64], ctypes.c_uint64),
    "pkv_block_hash": ([_P, _I, ctypes.c_int64], ctypes.c_uint64),
    "pkv_bm_can_allocate": ([_P, _I], _I),
    "pkv_bm_allocate": ([_P, ctypes.c_int64, _P, _I, _P], _I),
    "pkv_bm_can_append": ([_P, ctypes.c_int64, _I], _I),
    "pkv_bm_append": ([_P, ctypes.c_int64, _P, _I, _P], _I),
    "pkv_bm_append_cow": ([_P, ctypes.c_int64, _P, _I, _P, _P, _P], _I),
    "pkv_bm_fork": ([_P, ctypes.c_int64, ctypes.c_int64], _I),
    "pkv_bm_free": ([_P, ctypes.c_int64], _I),
    "pkv_bm_context_len": ([_P, ctypes.c_int64], _I),
    "pkv_bm_batch_tables": ([_P, _P, _I, _I, _P, _P], _I),
}
SIGNATURES.update(_BM_SIGNATURES)


def _np_ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def xxh64(data: bytes, seed: int = 0) -> int:
    buf = ctypes.create_string_buffer(bytes(data), len(data))
    return int(load().pkv_xxh64(buf, len(data), seed))


def block_hash(token_ids, prefix_hash: int = -1) -> int:
    import numpy as np
    t = np.ascontiguousarray(token_ids, dtype=np.int64)
    p = prefix_hash if prefix_hash < 2**63 else prefix_hash - 2**64  # int64 view of the uint64
    return int(load().pkv_block_hash(_np_ptr(t), t.size, p))


class BlockManager:
    """Host block manager (include/pkv.h, pkv_bm_*): allocate prompts with prefix sharing, append
    decode tokens (returning their slots), free sequences, and emit batch block tables."""

    def __init__(self, num_blocks: int, block_size: int = BLOCK_SIZE, prefix_cache: bool = True):
        self._h = load().pkv_bm_create(num_blocks, block_size, int(prefix_cache))
        if not self._h:
            raise PkvError(ERR_INVALID_ARG, "pkv_bm_create")
        self.block_size = block_size

    def close(self):
        if self._h:
            load().pkv_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def num_free_blocks(self) -> int:
        return load().pkv_bm_num_free_blocks(self._h)

    def ref_count(self, block_id: int) -> int:
        return load().pkv_bm_ref_count(self._h, block_id)

    def can_allocate(self, num_tokens: int) -> bool:
        return bool(load().pkv_bm_can_allocate(self._h, num_tokens))

    def allocate(self, seq_id: int, token_ids) -> int:
        import numpy as np
        t = np.ascontiguousarray(token_ids, dtype=np.int64)
        cached = ctypes.c_int(0)
        _check(load().pkv_bm_allocate(self._h, seq_id, _np_ptr(t), t.size, ctypes.byref(cached)),
               "pkv_bm_allocate")
        return cached.value

    def can_append(self, seq_id: int, num_new_tokens: int) -> bool:
        return bool(load().pkv_bm_can_append(self._h, seq_id, num_new_tokens))

    def append(self, seq_id: int, token_ids):
        import numpy as np
        t = np.ascontiguousarray(token_ids, dtype=np.int64)
        slots = np.zeros(t.size, dtype=np.int64)
        _check(load().pkv_bm_append(self._h, seq_id, _np_ptr(t), t.size, _np_ptr(slots)),
               "pkv_bm_append")
        return slots

    def append_cow(self, seq_id: int, token_ids):
        """Append with copy-on-write: (slots, copies) where copies is a list of (src, dst) block
        pairs to copy on the device (pkv_kv_cache_copy_blocks) before writing the slots."""
        import numpy as np
        t = np.ascontiguousarray(token_ids, dtype=np.int64)
        slots = np.zeros(t.size, dtype=np.int64)
        pair = np.zeros(2, dtype=np.int32)
        n = ctypes.c_int(0)
        _check(load().pkv_bm_append_cow(self._h, seq_id, _np_ptr(t), t.size, _np_ptr(slots),
                                        _np_ptr(pair), ctypes.byref(n)), "pkv_bm_append_cow")
        return slots, [(int(pair[0]), int(pair[1]))] * n.value

    def fork(self, parent_id: int, child_id: int):
        _check(load().pkv_bm_fork(self._h, parent_id, child_id), "pkv_bm_fork")

    def free(self, seq_id: int):
        _check(load().pkv_bm_free(self._h, seq_id), "pkv_bm_free")

    def context_len(self, seq_id: int) -> int:
        return load().pkv_bm_context_len(self._h, seq_id)

    def batch_tables(self, seq_ids, max_blocks_per_seq: int):
        import numpy as np
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        bt = np.zeros((ids.size, max_blocks_per_seq), dtype=np.int32)
        cl = np.zeros(ids.size, dtype=np.int32)
        _check(load().pkv_bm_batch_tables(self._h, _np_ptr(ids), ids.size, max_blocks_per_seq,
                                          _np_ptr(bt), _np_ptr(cl)), "pkv_bm_batch_tables")
        return bt, cl
