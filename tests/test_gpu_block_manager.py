"""A decode step whose block tables, context lengths and slots come from the host block manager:
prompts sharing a system prefix are allocated (prefix blocks shared by reference), each sequence
appends its new token, and the CUDA write + attention must match the oracle on those tables."""
import numpy as np
import pytest

import oracle
import paged_kv_decode_reshape_gb300 as P
import workloads as W
from _gpu import assert_close, to_dev, to_f64

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib(pkv):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("kv", ["bf16", "i8"])
def test_decode_step_on_manager_tables(kv):
    rng = np.random.default_rng(31)
    B, Hq, Hkv, D, NB = 6, 32, 8, 128, 400
    bm = P.BlockManager(NB, 16, prefix_cache=True)
    system = rng.integers(0, 32000, 96)  # 6 shared blocks
    for b in range(B):
        toks = np.concatenate([system, rng.integers(0, 32000, int(rng.integers(5, 700)))])
        cached = bm.allocate(b, toks)
        assert cached == (0 if b == 0 else 96)
    slots = np.concatenate([bm.append(b, [int(rng.integers(0, 32000))]) for b in range(B)])
    mbps = 64
    bt, cl = bm.batch_tables(list(range(B)), mbps)
    assert (bt[:, :6] == bt[0, :6]).all()  # the prefix is shared, not copied
    # pool contents as a prefill would have left them, plus this step's new rows
    if kv == "bf16":
        kp = W.f32_to_bf16_bits(rng.standard_normal((NB, Hkv, 16, D), dtype=np.float32))
        vp = W.f32_to_bf16_bits(rng.standard_normal((NB, Hkv, 16, D), dtype=np.float32))
        kn = W.f32_to_bf16_bits(rng.standard_normal((B, Hkv, D), dtype=np.float32))
        vn = W.f32_to_bf16_bits(rng.standard_normal((B, Hkv, D), dtype=np.float32))
        ks = vs = kns = vns = None
    else:
        kp, ks = W.quantize_int8_rows(rng.standard_normal((NB, Hkv, 16, D), dtype=np.float32))
        vp, vs = W.quantize_int8_rows(rng.standard_normal((NB, Hkv, 16, D), dtype=np.float32))
        kn, kns = W.quantize_int8_rows(rng.standard_normal((B, Hkv, D), dtype=np.float32))
        vn, vns = W.quantize_int8_rows(rng.standard_normal((B, Hkv, D), dtype=np.float32))
    q = W.f32_to_bf16_bits(rng.standard_normal((B, Hq, D), dtype=np.float32))
    scale = 1 / np.sqrt(D)
    d_kp, d_vp, d_ks, d_vs = to_dev(kp), to_dev(vp), to_dev(ks), to_dev(vs)
    P.kv_cache_write(to_dev(kn), to_dev(vn), d_kp, d_vp, to_dev(slots), to_dev(kns), to_dev(vns),
                     d_ks, d_vs)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    maxc = int(cl.max())
    nbytes = P.decode_workspace_bytes(B, Hq, Hkv, D, maxc, 64)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    if kv == "bf16":
        P.paged_decode_attention(out, to_dev(q), d_kp, d_vp, to_dev(bt), to_dev(cl), maxc, scale, 64, ws)
    else:
        P.paged_decode_attention_int8(out, to_dev(q), d_kp, d_vp, d_ks, d_vs, to_dev(bt),
                                      to_dev(cl), maxc, scale, 64, ws)
    got = to_f64(out)
    okp, ovp, oks, ovs = oracle.kv_cache_write(kn, vn, kp, vp, slots, kns, vns, ks, vs)
    ref = oracle.paged_decode_attention(q, okp, ovp, bt, cl, scale, oks, ovs)
    assert_close(got, ref, kv, f"manager tables {kv}")


@pytest.mark.parametrize("kv", ["f32", "bf16", "i8"])
def test_copy_blocks_bit_exact(kv):
    """pkv_kv_cache_copy_blocks against the oracle's block copy, every byte of both pools (and
    the INT8 scales); a pair with a bad id is skipped and flagged."""
    rng = np.random.default_rng(3)
    NB, Hkv, D = 40, 4, 128 if kv != "f32" else 64
    if kv == "i8":
        kp, ks = W.quantize_int8_rows(rng.standard_normal((NB, Hkv, 16, D), dtype=np.float32))
        vp, vs = W.quantize_int8_rows(rng.standard_normal((NB, Hkv, 16, D), dtype=np.float32))
    else:
        conv = (lambda x: x) if kv == "f32" else W.f32_to_bf16_bits
        kp = conv(rng.standard_normal((NB, Hkv, 16, D), dtype=np.float32))
        vp = conv(rng.standard_normal((NB, Hkv, 16, D), dtype=np.float32))
        ks = vs = None
    pairs = [(3, 17), (5, 6), (39, 0), (11, 12)]
    bad = [(2, NB + 4), (-1, 9), (8, 8)]
    d_kp, d_vp, d_ks, d_vs = to_dev(kp), to_dev(vp), to_dev(ks), to_dev(vs)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev_pairs = torch.tensor(pairs + bad, dtype=torch.int32, device="cuda")
    P.kv_cache_copy_blocks(d_kp, d_vp, dev_pairs, d_ks, d_vs, status=st)
    torch.cuda.synchronize()
    okp, ovp, oks, ovs = oracle.copy_blocks(kp, vp, pairs, ks, vs)
    from _gpu import to_host_raw
    assert np.array_equal(to_host_raw(d_kp), okp) and np.array_equal(to_host_raw(d_vp), ovp)
    if kv == "i8":
        assert np.array_equal(d_ks.cpu().numpy(), oks) and np.array_equal(d_vs.cpu().numpy(), ovs)
    assert int(st.item()) & P.FLAG_BAD_BLOCK


@pytest.mark.parametrize("kv", ["bf16", "i8"])
@pytest.mark.parametrize("prompt_len", [2001, 2000, 37])
def test_forked_decode_step_with_copy_on_write(kv, prompt_len):
    """Best-of-4 sampling through the block manager: one prompt, three forks, each sample appends
    its own new token (append_cow), the device copies the shared partial tail block for all but
    the last writer (pkv_kv_cache_copy_blocks), writes the new tokens and runs attention on the
    samples' tables. The oracle applies the same copies and writes to its own pools."""
    rng = np.random.default_rng(prompt_len + (0 if kv == "bf16" else 7))
    n, Hq, Hkv, D, NB = 4, 32, 8, 128, 200
    bm = P.BlockManager(NB, 16)
    bm.allocate(0, rng.integers(0, 32000, prompt_len))
    for c in range(1, n):
        bm.fork(0, c)
    slots, copies = [], []
    for s in range(n):
        sl, cp = bm.append_cow(s, [int(rng.integers(0, 32000))])
        slots.append(sl)
        copies += cp
    slots = np.concatenate(slots)
    assert len(copies) == (n - 1 if prompt_len % 16 else 0)
    bt, cl = bm.batch_tables(list(range(n)), 140)
    if kv == "bf16":
        kp = W.f32_to_bf16_bits(rng.standard_normal((NB, Hkv, 16, D), dtype=np.float32))
        vp = W.f32_to_bf16_bits(rng.standard_normal((NB, Hkv, 16, D), dtype=np.float32))
        kn = W.f32_to_bf16_bits(rng.standard_normal((n, Hkv, D), dtype=np.float32))
        vn = W.f32_to_bf16_bits(rng.standard_normal((n, Hkv, D), dtype=np.float32))
        ks = vs = kns = vns = None
    else:
        kp, ks = W.quantize_int8_rows(rng.standard_normal((NB, Hkv, 16, D), dtype=np.float32))
        vp, vs = W.quantize_int8_rows(rng.standard_normal((NB, Hkv, 16, D), dtype=np.float32))
        kn, kns = W.quantize_int8_rows(rng.standard_normal((n, Hkv, D), dtype=np.float32))
        vn, vns = W.quantize_int8_rows(rng.standard_normal((n, Hkv, D), dtype=np.float32))
    q = W.f32_to_bf16_bits(rng.standard_normal((n, Hq, D), dtype=np.float32))
    scale = 1 / np.sqrt(D)
    d_kp, d_vp, d_ks, d_vs = to_dev(kp), to_dev(vp), to_dev(ks), to_dev(vs)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    if copies:
        P.kv_cache_copy_blocks(d_kp, d_vp, torch.tensor(copies, dtype=torch.int32, device="cuda"),
                               d_ks, d_vs, status=st)
    P.kv_cache_write(to_dev(kn), to_dev(vn), d_kp, d_vp, to_dev(slots), to_dev(kns), to_dev(vns),
                     d_ks, d_vs, status=st)
    out = torch.empty((n, Hq, D), dtype=torch.bfloat16, device="cuda")
    maxc = int(cl.max())
    ws = torch.empty(max(256, P.decode_workspace_bytes(n, Hq, Hkv, D, maxc, 0)), dtype=torch.uint8,
                     device="cuda")
    if kv == "bf16":
        P.paged_decode_attention(out, to_dev(q), d_kp, d_vp, to_dev(bt), to_dev(cl), maxc, scale, 0, ws, st)
    else:
        P.paged_decode_attention_int8(out, to_dev(q), d_kp, d_vp, d_ks, d_vs, to_dev(bt), to_dev(cl),
                                      maxc, scale, 0, ws, st)
    got = to_f64(out)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ckp, cvp, cks, cvs = oracle.copy_blocks(kp, vp, copies, ks, vs)
    okp, ovp, oks, ovs = oracle.kv_cache_write(kn, vn, ckp, cvp, slots, kns, vns, cks, cvs)
    ref = oracle.paged_decode_attention(q, okp, ovp, bt, cl, scale, oks, ovs)
    assert_close(got, ref, kv, f"forked samples {kv} prompt {prompt_len}")
    # the prompt's full blocks stay one shared copy
    assert (bt[:, :prompt_len // 16] == bt[0, :prompt_len // 16]).all()
