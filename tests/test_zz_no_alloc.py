"""pkv_paged_decode_attention_static_ws: the entry point for callers that cannot allocate device
memory (a plugin inside another runtime's memory plan, a loop where an allocation's implicit
synchronisation is not acceptable). It takes the split-K scratch from a fixed array inside the
library. It runs the same kernels at the same chunk as the entry point that takes a
caller-allocated workspace, so its answers must equal that entry point's bit for bit, and match
the oracle at the bf16 bar.

Collected last on purpose (file name), so a run that stops at the first failure has already run
every other test; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import oracle
import paged_kv_decode_reshape_gb300 as P
import workloads as W

torch = pytest.importorskip("torch")

BF16_BAR = (2e-2, 2e-3)  # max-abs, mean-abs against the fp64 oracle (the parity tests' bf16 bar)


def _call_static(w, dev, out, chunk, status, stream):
    L = P.load()
    return L.pkv_paged_decode_attention_static_ws(
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(dev["q"].data_ptr()),
        ctypes.c_void_p(dev["k"].data_ptr()), ctypes.c_void_p(dev["v"].data_ptr()),
        ctypes.c_void_p(dev["bt"].data_ptr()), ctypes.c_void_p(dev["cl"].data_ptr()),
        w.B, w.Hq, w.Hkv, w.D, w.BS, w.NB, w.MBPS, w.max_context_len, w.scale,
        P.BF16 if w.kv_dtype == "bf16" else P.F32, chunk, ctypes.c_void_p(status.data_ptr()),
        ctypes.c_void_p(stream.cuda_stream))


def _upload(w):
    def up(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
        return torch.from_numpy(a).cuda()
    return dict(q=up(w.q), k=up(w.k_pool), v=up(w.v_pool), bt=up(w.block_tables),
                cl=up(w.context_lens))


def _splits(w, chunk):
    c = P.decode_split_chunk(w.B, w.Hkv, w.D, w.max_context_len, chunk, P.BF16)
    return max(1, w.max_context_len // c)


@pytest.mark.gpu
@pytest.mark.parametrize("chunk_first,chunk_second", [(64, 128), (0, 0)], ids=["forced", "auto"])
def test_static_workspace_matches_caller_workspace_on_two_calls_in_a_row(chunk_first, chunk_second):
    """Two different batches back to back on one stream, sharing the one static array; the second
    needs fewer split slots than the first, so partial states the first call left behind sit in
    the array while the second runs and would show if the merge read them."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    P.load()
    stream = torch.cuda.current_stream()
    cases = [(W.make_config(2, seed=41, B=6, ctx_lo=300, ctx_hi=2500), chunk_first),
             (W.make_config(2, seed=42, B=9, ctx_lo=50, ctx_hi=1100), chunk_second)]
    s0, s1 = (_splits(w, c) for w, c in cases)
    assert s0 > s1 > 1, (s0, s1)  # both use the scratch; the second fewer slots per head
    for w, chunk in cases:
        need = P.decode_workspace_bytes_dtype(w.B, w.Hq, w.Hkv, w.D, w.max_context_len, chunk, P.BF16)
        assert 0 < need <= P.STATIC_WORKSPACE_BYTES
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    results = []
    for w, chunk in cases:
        dev = _upload(w)
        torch.cuda.synchronize()
        out = torch.empty_like(dev["q"])
        assert _call_static(w, dev, out, chunk, status, stream) == P.OK
        results.append((w, chunk, dev, out))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for w, chunk, dev, out in results:
        ref = torch.empty_like(dev["q"])
        nbytes = P.decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, w.max_context_len, chunk)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        P.paged_decode_attention(ref, dev["q"], dev["k"], dev["v"], dev["bt"], dev["cl"],
                                 w.max_context_len, w.scale, chunk, ws, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        # same kernels, same chunk, same summation order: identical bits
        assert torch.equal(out, ref)
        got = out.float().cpu().numpy().astype(np.float64)
        exp = oracle.paged_decode_attention(w.q, w.k_pool, w.v_pool, w.block_tables,
                                            w.context_lens, w.scale)
        err = np.abs(got - exp)
        assert err.max() <= BF16_BAR[0] and err.mean() <= BF16_BAR[1], (err.max(), err.mean())


def test_static_workspace_refuses_batches_beyond_its_size():
    """Partial states larger than the fixed array are refused before anything is enqueued (no
    CUDA call is made on this path, so it runs without a GPU)."""
    L = P.load()
    fake = [ctypes.c_void_p(0x7F0000000000 + i * 0x1000000) for i in range(6)]
    # 64 seqs x 64 heads x 512 splits (chunk 16, 8192 tokens) x 130 floats >> 32 MiB
    need = P.decode_workspace_bytes_dtype(64, 64, 8, 128, 8192, 16, P.BF16)
    assert need > P.STATIC_WORKSPACE_BYTES
    rc = L.pkv_paged_decode_attention_static_ws(*fake, 64, 64, 8, 128, 16, 40000, 512, 8192, 0.1,
                                                P.BF16, 16, None, None)
    assert rc == P.ERR_WORKSPACE
