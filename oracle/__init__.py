"""fp64 CPU oracle for the paged-KV decode path -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg may import
this package. The product (paged_kv_decode_reshape_gb300) never does, and this package never
imports the product. The arithmetic lives in pkv_oracle.c (plain C, fp64); this module only
marshals numpy arrays.

Element codes: F32 = 0, BF16 = 1 (arrays of uint16 bit patterns), I8 = 2.
"""
import ctypes
import os

import numpy as np

from . import build as _build

F32, BF16, I8 = 0, 1, 2
_STATUS = {0: "ok", 1: "bad argument", 2: "block id out of range", 3: "slot out of range",
           4: "out of memory"}

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        L.orc_kv_cache_write.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I]
        L.orc_kv_cache_write.restype = I
        L.orc_split_count.argtypes = [I, I, I, I, ctypes.POINTER(ctypes.c_int)]
        L.orc_split_count.restype = I
        L.orc_paged_decode_attention.argtypes = [P, P, I, P, P, I, P, P, P, P,
                                                 I, I, I, I, I, I, I, D, I]
        L.orc_paged_decode_attention.restype = I
        L.orc_paged_decode_attention_multi.argtypes = [P, P, I, P, P, I, P, P, P, P,
                                                       I, I, I, I, I, I, I, I, D]
        L.orc_paged_decode_attention_multi.restype = I
        L.orc_paged_prefill_attention.argtypes = [P, P, I, P, P, I, P, P, P, P, P, I, I, I, I, I, I, I, D]
        L.orc_paged_prefill_attention.restype = I
        L.orc_paged_decode_partials.argtypes = [P, P, P, P, P, I, P, P, I, P, P, P, P,
                                                I, I, I, I, I, I, I, D, I, I]
        L.orc_paged_decode_partials.restype = I
        L.orc_merge_partials.argtypes = [P, P, P, P, P, I, I, I, I]
        L.orc_merge_partials.restype = I
        L.orc_kv_cache_write_quant.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I]
        L.orc_kv_cache_write_quant.restype = I
        L.orc_quantize_row_int8.argtypes = [P, ctypes.c_size_t, I, I, P, P]
        L.orc_quantize_row_int8.restype = None
        L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_double.restype = D
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _check(rc):
    if rc != 0:
        raise RuntimeError(f"oracle: {_STATUS.get(rc, rc)}")


def _code(arr):
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.uint16:
        return BF16
    if arr.dtype == np.int8:
        return I8
    raise TypeError(f"unsupported element type {arr.dtype}")


def bf16_to_double(bits: int) -> float:
    return lib().orc_bf16_to_double(bits)


def kv_cache_write(k_new, v_new, k_pool, v_pool, slot_mapping, k_new_scales=None,
                   v_new_scales=None, k_scales=None, v_scales=None, check=True, inplace=False):
    """Write new tokens into copies of the pools (or, with inplace=True, into the given
    C-contiguous arrays); returns (k_pool, v_pool, k_scales, v_scales).
    Pools are [NB, Hkv, BS, D]; k_new/v_new [T, Hkv, D]; slot_mapping int64 [T]."""
    if inplace:
        for a in (k_pool, v_pool, k_scales, v_scales):
            assert a is None or a.flags.c_contiguous
        kp, vp, ks, vs = k_pool, v_pool, k_scales, v_scales
    else:
        kp, vp = np.array(k_pool, copy=True), np.array(v_pool, copy=True)
        ks = None if k_scales is None else np.array(k_scales, dtype=np.float32, copy=True)
        vs = None if v_scales is None else np.array(v_scales, dtype=np.float32, copy=True)
    kn, vn = np.ascontiguousarray(k_new), np.ascontiguousarray(v_new)
    sm = _c(slot_mapping, np.int64)
    NB, Hkv, BS, D = kp.shape
    T = sm.shape[0]
    rc = lib().orc_kv_cache_write(_ptr(kn), _ptr(vn), _ptr(kp), _ptr(vp),
                                  _ptr(_c(k_new_scales, np.float32)),
                                  _ptr(_c(v_new_scales, np.float32)), _ptr(ks), _ptr(vs),
                                  _ptr(sm), T, Hkv, D, BS, NB, _code(kp))
    if check:
        _check(rc)
    return kp, vp, ks, vs


def copy_blocks(k_pool, v_pool, pairs, k_scales=None, v_scales=None):
    """Copy-on-write for forked sequences ("LLM Primer VI, Chapter 8", section 8.1, blocks
    shared by reference count; the copy itself is a reading, listed in the design notes): for
    each (src, dst) in order, block dst of both pools -- every kv head, every slot -- and, for
    INT8 pools, its rows of scales become a copy of block src. Returns new arrays."""
    kp, vp = np.array(k_pool, copy=True), np.array(v_pool, copy=True)
    ks = None if k_scales is None else np.array(k_scales, copy=True)
    vs = None if v_scales is None else np.array(v_scales, copy=True)
    for src, dst in pairs:
        for a in (kp, vp, ks, vs):
            if a is not None:
                a[dst] = a[src]
    return kp, vp, ks, vs


def quantize_rows_int8(x):
    """int8 codes and fp32 scales of each last-axis row of x (float32 or bf16 bits)."""
    x = np.ascontiguousarray(x)
    D = x.shape[-1]
    rows = x.reshape(-1, D)
    codes = np.zeros(rows.shape, np.int8)
    scales = np.zeros(rows.shape[0], np.float32)
    for r in range(rows.shape[0]):
        lib().orc_quantize_row_int8(_ptr(rows), r * D, D, _code(rows),
                                    _ptr(codes[r:r + 1]), _ptr(scales[r:r + 1]))
    return codes.reshape(x.shape), scales.reshape(x.shape[:-1])


def kv_cache_write_quant(k_new, v_new, k_pool, v_pool, k_scales, v_scales, slot_mapping,
                         check=True):
    """Quantise new rows (float32 or bf16 bits, [T, Hkv, D]) into copies of the int8 pools and
    scale arrays; returns (k_pool, v_pool, k_scales, v_scales)."""
    kp, vp = np.array(k_pool, dtype=np.int8, copy=True), np.array(v_pool, dtype=np.int8, copy=True)
    ks = np.array(k_scales, dtype=np.float32, copy=True)
    vs = np.array(v_scales, dtype=np.float32, copy=True)
    kn, vn = np.ascontiguousarray(k_new), np.ascontiguousarray(v_new)
    sm = _c(slot_mapping, np.int64)
    NB, Hkv, BS, D = kp.shape
    rc = lib().orc_kv_cache_write_quant(_ptr(kn), _ptr(vn), _ptr(kp), _ptr(vp), _ptr(ks),
                                        _ptr(vs), _ptr(sm), sm.shape[0], Hkv, D, BS, NB,
                                        _code(kn))
    if check:
        _check(rc)
    return kp, vp, ks, vs


def split_count(n, chunk, max_splits, block_size=16):
    """(number of splits, tokens per split) for a context of n tokens."""
    per = ctypes.c_int(0)
    ns = lib().orc_split_count(int(n), int(chunk), int(max_splits), int(block_size),
                               ctypes.byref(per))
    return ns, per.value


def paged_decode_attention(q, k_pool, v_pool, block_tables, context_lens, scale,
                           k_scales=None, v_scales=None, num_threads=1):
    """fp64 out [B, Hq, D] = softmax(scale * q K^T) V gathered through the block tables."""
    q = np.ascontiguousarray(q)
    kp, vp = np.ascontiguousarray(k_pool), np.ascontiguousarray(v_pool)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    B, Hq, D = q.shape
    NB, Hkv, BS, _ = kp.shape
    out = np.zeros((B, Hq, D), dtype=np.float64)
    rc = lib().orc_paged_decode_attention(
        _ptr(out), _ptr(q), _code(q), _ptr(kp), _ptr(vp), _code(kp),
        _ptr(_c(k_scales, np.float32)), _ptr(_c(v_scales, np.float32)), _ptr(bt), _ptr(cl),
        B, Hq, Hkv, D, BS, NB, bt.shape[1], float(scale), int(num_threads))
    _check(rc)
    return out


def paged_decode_attention_multi(q, k_pool, v_pool, block_tables, context_lens, scale,
                                 k_scales=None, v_scales=None):
    """Multi-token decode: q [B, L, Hq, D]; query token l of sequence b sees its first
    context_lens[b] - (L - 1 - l) tokens. Returns fp64 [B, L, Hq, D]."""
    q = np.ascontiguousarray(q)
    kp, vp = np.ascontiguousarray(k_pool), np.ascontiguousarray(v_pool)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    B, L, Hq, D = q.shape
    NB, Hkv, BS, _ = kp.shape
    out = np.zeros((B, L, Hq, D), dtype=np.float64)
    rc = lib().orc_paged_decode_attention_multi(
        _ptr(out), _ptr(q), _code(q), _ptr(kp), _ptr(vp), _code(kp),
        _ptr(_c(k_scales, np.float32)), _ptr(_c(v_scales, np.float32)), _ptr(bt), _ptr(cl),
        B, L, Hq, Hkv, D, BS, NB, bt.shape[1], float(scale))
    _check(rc)
    return out


def paged_prefill_attention(q, k_pool, v_pool, block_tables, context_lens, query_start, scale,
                            k_scales=None, v_scales=None):
    """Paged (chunked) prefill: q [total, Hq, D]; sequence b owns rows query_start[b] ..
    query_start[b + 1] - 1, its last L_b context tokens, attending causally. INT8 pools come with
    their per-token scales [NB, Hkv, BS]. fp64 [total, Hq, D]."""
    q = np.ascontiguousarray(q)
    kp, vp = np.ascontiguousarray(k_pool), np.ascontiguousarray(v_pool)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    qs = _c(query_start, np.int32)
    ks, vs = _c(k_scales, np.float32), _c(v_scales, np.float32)
    T, Hq, D = q.shape
    NB, Hkv, BS, _ = kp.shape
    out = np.zeros((T, Hq, D), dtype=np.float64)
    rc = lib().orc_paged_prefill_attention(
        _ptr(out), _ptr(q), _code(q), _ptr(kp), _ptr(vp), _code(kp), _ptr(ks), _ptr(vs), _ptr(bt),
        _ptr(cl), _ptr(qs), cl.shape[0], Hq, Hkv, D, BS, NB, bt.shape[1], float(scale))
    _check(rc)
    return out


def paged_decode_partials(q, k_pool, v_pool, block_tables, context_lens, scale, chunk,
                          max_splits, k_scales=None, v_scales=None):
    """Per-split partial states: (m [B,Hq,S], l [B,Hq,S], acc [B,Hq,S,D], n_splits [B])."""
    q = np.ascontiguousarray(q)
    kp, vp = np.ascontiguousarray(k_pool), np.ascontiguousarray(v_pool)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    B, Hq, D = q.shape
    NB, Hkv, BS, _ = kp.shape
    S = int(max_splits)
    m = np.zeros((B, Hq, S)); l = np.zeros((B, Hq, S)); acc = np.zeros((B, Hq, S, D))
    ns = np.zeros(B, dtype=np.int32)
    rc = lib().orc_paged_decode_partials(
        _ptr(m), _ptr(l), _ptr(acc), _ptr(ns), _ptr(q), _code(q), _ptr(kp), _ptr(vp),
        _code(kp), _ptr(_c(k_scales, np.float32)), _ptr(_c(v_scales, np.float32)),
        _ptr(bt), _ptr(cl), B, Hq, Hkv, D, BS, NB, bt.shape[1], float(scale), int(chunk), S)
    _check(rc)
    return m, l, acc, ns


def merge_partials(m, l, acc, n_splits):
    """Merge per-split states into fp64 out [B, Hq, D]."""
    m, l, acc = (np.ascontiguousarray(x, dtype=np.float64) for x in (m, l, acc))
    ns = _c(n_splits, np.int32)
    B, Hq, S, D = acc.shape
    out = np.zeros((B, Hq, D))
    _check(lib().orc_merge_partials(_ptr(out), _ptr(m), _ptr(l), _ptr(acc), _ptr(ns),
                                    B, Hq, D, S))
    return out


def library_path():
    return os.path.abspath(_build.LIB)
