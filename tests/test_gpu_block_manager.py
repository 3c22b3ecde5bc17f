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
