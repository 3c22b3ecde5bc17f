"""The C ABI without a GPU: the library loads, exports every symbol include/pkv.h declares, and
host-side argument checks reject bad calls before any CUDA call is made."""
import ctypes
import os
import re

import pytest

import paged_kv_decode_reshape_gb300 as P

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pkv.h")

# Fake, never-dereferenced device addresses: every call below fails validation before launch.
# Host-logic tests for a machine without a GPU; skipped where a GPU exists, so that a
# validation regression can never launch a kernel on fake pointers.
A = 0x7F0000000000


def _no_gpu():
    try:
        import torch
        return not torch.cuda.is_available()
    except Exception:
        return True


fake_ptrs = pytest.mark.skipif(not _no_gpu(), reason="fake-pointer checks run on CPU-only hosts")
FAKE = [ctypes.c_void_p(A + i * 0x1000000) for i in range(12)]


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(pkv):
    names = declared_functions()
    assert {"pkv_kv_cache_write", "pkv_paged_decode_attention",
            "pkv_paged_decode_attention_int8", "pkv_decode_workspace_bytes"} <= set(names)
    lib = ctypes.CDLL(P.library_path())
    for n in names:
        assert hasattr(lib, n), f"{n} declared in pkv.h but not exported"
        assert n in P.SIGNATURES, f"{n} has no binding signature"


def test_status_strings(pkv):
    assert P.status_string(P.OK) == "ok"
    assert "workspace" in P.status_string(P.ERR_WORKSPACE)
    assert P.status_string(99) == "unknown status"
    assert "sm_103a" in P.version()


def test_workspace_arithmetic(pkv):
    L = P.load()
    # 8 seqs x 32 q / 8 kv heads, 131072 tokens: the workspace bound takes the smallest auto chunk
    # of any dtype (fp32's, 2048) -> 64 splits x (128 acc + m + l); the INT8 kernel keeps the
    # longest sequence at <= 32 splits (chunk 4096)
    assert L.pkv_decode_split_chunk(8, 8, 128, 131072, 0, P.I8) == 4096
    assert L.pkv_decode_split_chunk(8, 8, 128, 131072, 0, P.F32) == 2048
    assert L.pkv_decode_split_chunk(8, 8, 128, 131072, 0, P.BF16) == 4096
    assert L.pkv_decode_workspace_bytes(8, 32, 8, 128, 131072, 0) == 8 * 32 * 64 * 130 * 4
    assert L.pkv_decode_workspace_bytes(8, 32, 8, 128, 131072, 1024) == 8 * 32 * 128 * 130 * 4
    assert L.pkv_decode_workspace_bytes(4, 4, 4, 64, 100, 0) == 0    # one split: no workspace
    assert L.pkv_decode_workspace_bytes(4, 4, 4, 64, 100, 17) == 0   # chunk not a block multiple
    # auto chunk: ~1024 units (bf16 tensor-core kernel) or ~4096 (INT8, CUDA-core), powers of
    # two in [256, 4096], more only to keep splits <= 8192
    BF, I8, F32 = P.BF16, P.I8, P.F32
    assert L.pkv_decode_split_chunk(64, 8, 128, 4055, 0, BF) == 1024     # Llama-3-8B GQA batch
    assert L.pkv_decode_split_chunk(8, 8, 128, 130882, 0, BF) == 4096    # 131k-context batch
    assert L.pkv_decode_split_chunk(128, 8, 128, 8083, 0, I8) == 1024    # INT8 batch
    assert L.pkv_decode_split_chunk(64, 8, 128, 4055, 0, I8) == 512      # INT8: at least 512
    assert L.pkv_decode_split_chunk(512, 8, 128, 8083, 0, I8) == 4096    # 128 seqs x 4 tokens
    assert L.pkv_decode_split_chunk(256, 8, 128, 4090, 0, BF) == 4096    # shared-prefix batch
    assert L.pkv_decode_split_chunk(64, 8, 64, 4055, 0, BF) == 256       # head_dim 64: CUDA cores
    assert L.pkv_decode_split_chunk(64, 8, 128, 4055, 0, F32) == 256     # fp32: CUDA cores
    assert L.pkv_decode_split_chunk(4, 4, 64, 100, 0, F32) == 256
    assert L.pkv_decode_split_chunk(1024, 64, 128, 1 << 20, 0, BF) == 4096
    assert L.pkv_decode_split_chunk(1, 1, 128, 1 << 30, 0, BF) >= 4096
    assert (1 << 30) // L.pkv_decode_split_chunk(1, 1, 128, 1 << 30, 0, BF) <= 8192
    assert L.pkv_decode_split_chunk(4, 4, 64, 100, 48, F32) == 48        # explicit request kept
    assert L.pkv_decode_split_chunk(4, 4, 64, 100, 0, 7) == 0            # unknown dtype
    # shared-prefix decode: suffix splits (auto chunk over the longest suffix) + prefix key splits
    # (about 64 CTAs over (row tile of 128, kv head, split); whole 128-key tiles).
    # 256 seqs x 32/8 heads, prefix 2048 of max 4090: suffix chunk 2048 (bf16) or 512 (INT8, the
    # bound) -> 3 splits; 8 row tiles x 8 kv heads = 64 -> 1 prefix split; 4 slots x 130 floats
    assert L.pkv_decode_shared_prefix_workspace_bytes(256, 32, 8, 128, 4090, 2048, 0) == 256 * 32 * 4 * 130 * 4
    # 8 seqs: suffix chunk 256 -> 2042 // 256 = 7 splits; 1 row tile x 8 kv heads -> 8 prefix
    # splits of 256 tokens; 15 slots
    assert L.pkv_decode_shared_prefix_workspace_bytes(8, 32, 8, 128, 4090, 2048, 0) == 8 * 32 * 15 * 130 * 4
    assert L.pkv_decode_shared_prefix_workspace_bytes(256, 32, 8, 128, 4090, 40, 0) == 0    # not a block multiple
    assert L.pkv_decode_shared_prefix_workspace_bytes(256, 32, 8, 64, 4090, 2048, 0) == 0   # head_dim 128 only
    assert L.pkv_decode_shared_prefix_workspace_bytes(256, 32, 8, 128, 1000, 2048, 0) == 0  # prefix > context
    # the workspace bound covers the bf16 call (fewer splits) too
    assert L.pkv_decode_workspace_bytes(64, 32, 8, 128, 4055, 0) == 64 * 32 * (4055 // 256) * 130 * 4
    # the exact per-dtype size: the split extent at that dtype's own auto chunk
    WB = L.pkv_decode_workspace_bytes_dtype
    assert WB(64, 32, 8, 128, 4055, 0, BF) == 64 * 32 * (4055 // 1024) * 130 * 4
    assert WB(8, 32, 8, 128, 131072, 0, BF) == 8 * 32 * 32 * 130 * 4           # chunk 4096
    assert WB(8, 32, 8, 128, 131072, 0, I8) == 8 * 32 * 32 * 130 * 4         # chunk 4096
    assert WB(8, 32, 8, 128, 131072, 0, F32) == L.pkv_decode_workspace_bytes(8, 32, 8, 128, 131072, 0)
    assert WB(128, 64, 8, 128, 8083, 0, I8) == 128 * 64 * (8083 // 1024) * 130 * 4
    assert WB(64, 32, 8, 64, 4055, 0, BF) == 64 * 32 * (4055 // 256) * 66 * 4   # CUDA-core kernel
    assert WB(8, 32, 8, 128, 131072, 1024, BF) == 8 * 32 * 128 * 130 * 4        # forced chunk
    assert WB(4, 4, 4, 64, 100, 0, F32) == 0                                     # one split
    assert WB(4, 4, 4, 64, 100, 0, 7) == 0                                       # unknown dtype
    for shape in [(64, 32, 8, 128, 4055), (8, 32, 8, 128, 131072), (3, 8, 2, 128, 700),
                  (256, 32, 8, 128, 4090), (1, 64, 8, 128, 1 << 17)]:
        for c in (0, 16, 512):
            for dt in (F32, BF, I8):  # never above the dtype-free bound
                assert WB(*shape, c, dt) <= L.pkv_decode_workspace_bytes(*shape, c)


def _attn(L, **kw):
    a = dict(out=FAKE[0], q=FAKE[1], k=FAKE[2], v=FAKE[3], bt=FAKE[4], cl=FAKE[5], B=2, Hq=8,
             Hkv=2, D=128, BS=16, NB=64, MBPS=8, maxc=100, scale=0.1, dtype=P.BF16, chunk=0,
             ws=None, wsb=0, status=None, stream=None)
    a.update(kw)
    return L.pkv_paged_decode_attention(a["out"], a["q"], a["k"], a["v"], a["bt"], a["cl"], a["B"],
                                        a["Hq"], a["Hkv"], a["D"], a["BS"], a["NB"], a["MBPS"],
                                        a["maxc"], a["scale"], a["dtype"], a["chunk"], a["ws"],
                                        a["wsb"], a["status"], a["stream"])


@fake_ptrs
@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), P.ERR_INVALID_ARG),
    (dict(out=None), P.ERR_INVALID_ARG),
    (dict(Hq=6, Hkv=4), P.ERR_INVALID_ARG),
    (dict(D=96), P.ERR_UNSUPPORTED),
    (dict(BS=32), P.ERR_UNSUPPORTED),
    (dict(maxc=8 * 16 + 1), P.ERR_INVALID_ARG),
    (dict(maxc=-1), P.ERR_INVALID_ARG),
    (dict(chunk=20), P.ERR_INVALID_ARG),
    (dict(scale=float("nan")), P.ERR_INVALID_ARG),
    (dict(dtype=P.I8), P.ERR_INVALID_ARG),
    (dict(q=ctypes.c_void_p(A + 8)), P.ERR_INVALID_ARG),               # misaligned
    (dict(out=FAKE[1]), P.ERR_INVALID_ARG),                            # out aliases q
    (dict(maxc=128, MBPS=8, chunk=16), P.ERR_WORKSPACE),               # 8 splits, no workspace
    (dict(maxc=128, MBPS=8, chunk=16, ws=FAKE[6], wsb=100), P.ERR_WORKSPACE),
    (dict(maxc=128, MBPS=8, chunk=16, ws=ctypes.c_void_p(A + 0x6000010), wsb=1 << 30),
     P.ERR_INVALID_ARG),                                               # workspace misaligned
    (dict(B=70000), P.ERR_UNSUPPORTED),
])
def test_decode_argument_checks(pkv, kw, expect):
    assert _attn(P.load(), **kw) == expect


@fake_ptrs
def test_empty_batch_is_a_no_op(pkv):
    assert _attn(P.load(), B=0, out=None, q=None) == P.OK


@fake_ptrs
def test_int8_requires_scales(pkv):
    L = P.load()
    rc = L.pkv_paged_decode_attention_int8(FAKE[0], FAKE[1], FAKE[2], FAKE[3], None, FAKE[5],
                                           FAKE[6], FAKE[7], 2, 8, 2, 128, 16, 64, 8, 100, 0.1,
                                           0, None, 0, None, None)
    assert rc == P.ERR_INVALID_ARG


def _write(L, **kw):
    a = dict(kn=FAKE[0], vn=FAKE[1], kp=FAKE[2], vp=FAKE[3], kns=None, vns=None, ks=None,
             vs=None, sm=FAKE[8], T=4, Hkv=8, D=128, BS=16, NB=64, dtype=P.BF16)
    a.update(kw)
    return L.pkv_kv_cache_write(a["kn"], a["vn"], a["kp"], a["vp"], a["kns"], a["vns"], a["ks"],
                                a["vs"], a["sm"], a["T"], a["Hkv"], a["D"], a["BS"], a["NB"],
                                a["dtype"], None, None)


@fake_ptrs
@pytest.mark.parametrize("kw,expect", [
    (dict(kn=None), P.ERR_INVALID_ARG),
    (dict(sm=None), P.ERR_INVALID_ARG),
    (dict(D=80), P.ERR_UNSUPPORTED),
    (dict(BS=8), P.ERR_UNSUPPORTED),
    (dict(dtype=P.I8), P.ERR_INVALID_ARG),                              # int8 without scales
    (dict(ks=FAKE[9]), P.ERR_INVALID_ARG),                              # scales for bf16
    (dict(vp=FAKE[2]), P.ERR_INVALID_ARG),                              # K and V pools alias
    (dict(kp=ctypes.c_void_p(A + 0x2000004)), P.ERR_INVALID_ARG),      # misaligned
    (dict(T=-1), P.ERR_INVALID_ARG),
    (dict(T=0, kn=None, sm=None), P.OK),                               # nothing to write
])
def test_write_argument_checks(pkv, kw, expect):
    assert _write(P.load(), **kw) == expect


@fake_ptrs
@pytest.mark.parametrize("kw,expect", [
    (dict(kn=None), P.ERR_INVALID_ARG),
    (dict(ks=None), P.ERR_INVALID_ARG),
    (dict(src=P.I8), P.ERR_INVALID_ARG),                               # source must be fp32/bf16
    (dict(D=96), P.ERR_UNSUPPORTED),
    (dict(vp=FAKE[2]), P.ERR_INVALID_ARG),                              # K and V pools alias
    (dict(vs=FAKE[4]), P.ERR_INVALID_ARG),                              # K and V scales alias
    (dict(T=0, kn=None), P.OK),
])
def test_quant_write_argument_checks(pkv, kw, expect):
    a = dict(kn=FAKE[0], vn=FAKE[1], kp=FAKE[2], vp=FAKE[3], ks=FAKE[4], vs=FAKE[5], sm=FAKE[6],
             T=4, Hkv=8, D=128, BS=16, NB=64, src=P.BF16)
    a.update(kw)
    rc = P.load().pkv_kv_cache_write_int8(a["kn"], a["vn"], a["kp"], a["vp"], a["ks"], a["vs"],
                                          a["sm"], a["T"], a["Hkv"], a["D"], a["BS"], a["NB"],
                                          a["src"], None, None)
    assert rc == expect


@fake_ptrs
@pytest.mark.parametrize("kw,expect", [
    (dict(L=0), P.ERR_INVALID_ARG),
    (dict(ks=FAKE[8]), P.ERR_INVALID_ARG),                             # scales with bf16 pools
    (dict(dtype=P.I8), P.ERR_INVALID_ARG),                             # INT8 without scales
    (dict(B=20000, L=4), P.ERR_UNSUPPORTED),                           # B * L rows over grid.z
    (dict(maxc=128, chunk=16), P.ERR_WORKSPACE),
    (dict(B=0, out=None, q=None), P.OK),
])
def test_multi_token_argument_checks(pkv, kw, expect):
    a = dict(out=FAKE[0], q=FAKE[1], k=FAKE[2], v=FAKE[3], ks=None, vs=None, bt=FAKE[4], cl=FAKE[5],
             B=2, L=3, Hq=8, Hkv=2, D=128, BS=16, NB=64, MBPS=8, maxc=100, scale=0.1,
             dtype=P.BF16, chunk=0, ws=None, wsb=0)
    a.update(kw)
    rc = P.load().pkv_paged_decode_attention_multi(
        a["out"], a["q"], a["k"], a["v"], a["ks"], a["vs"], a["bt"], a["cl"], a["B"], a["L"],
        a["Hq"], a["Hkv"], a["D"], a["BS"], a["NB"], a["MBPS"], a["maxc"], a["scale"], a["dtype"],
        a["chunk"], a["ws"], a["wsb"], None, None)
    assert rc == expect


@fake_ptrs
@pytest.mark.parametrize("kw,expect", [
    (dict(D=64), P.ERR_UNSUPPORTED),
    (dict(Hq=6, Hkv=4), P.ERR_INVALID_ARG),
    (dict(qs=None), P.ERR_INVALID_ARG),
    (dict(out=FAKE[1]), P.ERR_INVALID_ARG),                             # out aliases q
    (dict(T=0), P.OK),
])
def test_prefill_argument_checks(pkv, kw, expect):
    a = dict(out=FAKE[0], q=FAKE[1], k=FAKE[2], v=FAKE[3], bt=FAKE[4], cl=FAKE[5], qs=FAKE[6],
             B=2, T=10, Hq=8, Hkv=2, D=128, BS=16, NB=64, MBPS=8, maxq=8, scale=0.1)
    a.update(kw)
    rc = P.load().pkv_paged_prefill_attention(
        a["out"], a["q"], a["k"], a["v"], a["bt"], a["cl"], a["qs"], a["B"], a["T"], a["Hq"],
        a["Hkv"], a["D"], a["BS"], a["NB"], a["MBPS"], a["maxq"], a["scale"], None, None)
    assert rc == expect
