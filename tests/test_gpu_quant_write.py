"""GPU parity of the quantising INT8 KV write: codes and scales bit-exact against the oracle, and
a decode step that quantises its new token before the INT8 attention."""
import numpy as np
import pytest

import oracle
import paged_kv_decode_reshape_gb300 as P
import workloads as W
from _gpu import DevWorkload, assert_close, to_dev, to_f64

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib(pkv):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("src", ["f32", "bf16"])
def test_quant_write_bit_exact(D, src):
    rng = np.random.default_rng(D + (1 if src == "bf16" else 0))
    T, Hkv, NB = 40, 4, 12
    x = (rng.standard_normal((2, T, Hkv, D)) * rng.uniform(0.01, 30, (2, T, Hkv, 1))).astype(np.float32)
    x[0, 3] = 0.0                       # an all-zero row: scale 1, codes 0
    x[1, 5, 0, :4] = [127, -2.5, 3.5, 0.5]  # exact halves at unit scale
    x[1, 5, 0, 4:] = 0
    kn, vn = (x[0], x[1]) if src == "f32" else (W.f32_to_bf16_bits(x[0]), W.f32_to_bf16_bits(x[1]))
    slots = rng.permutation(NB * 16)[:T].astype(np.int64)
    slots[7] = -1                        # padding
    slots[9] = NB * 16 + 3               # outside the pool: skipped and flagged
    kp = rng.integers(-100, 100, (NB, Hkv, 16, D)).astype(np.int8)  # old contents stay elsewhere
    vp = rng.integers(-100, 100, (NB, Hkv, 16, D)).astype(np.int8)
    ks = rng.uniform(0, 1, (NB, Hkv, 16)).astype(np.float32)
    vs = rng.uniform(0, 1, (NB, Hkv, 16)).astype(np.float32)
    d_kp, d_vp, d_ks, d_vs = to_dev(kp), to_dev(vp), to_dev(ks), to_dev(vs)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    P.kv_cache_write_int8(to_dev(kn), to_dev(vn), d_kp, d_vp, d_ks, d_vs, to_dev(slots), status=st)
    torch.cuda.synchronize()
    ekp, evp, eks, evs = oracle.kv_cache_write_quant(kn, vn, kp, vp, ks, vs, slots, check=False)
    assert np.array_equal(d_kp.cpu().numpy(), ekp) and np.array_equal(d_vp.cpu().numpy(), evp)
    assert np.array_equal(d_ks.cpu().numpy(), eks) and np.array_equal(d_vs.cpu().numpy(), evs)
    assert int(st.item()) & P.FLAG_BAD_SLOT


def test_decode_step_with_quantising_write():
    """INT8 step as a server runs it: the new token arrives in bf16, is quantised into its slot,
    then the INT8 attention reads it back with the rest of the context."""
    w = W.make_config(4, B=5, ctx_lo=17, ctx_hi=1500, seed=13)
    d = DevWorkload(w)
    P.kv_cache_write_int8(to_dev(w.k_new_src), to_dev(w.v_new_src), d.k_pool, d.v_pool,
                          d.k_scales, d.v_scales, d.slot_mapping)
    got = to_f64(d.attend(chunk=256))
    kp, vp, ks, vs = oracle.kv_cache_write_quant(w.k_new_src, w.v_new_src, w.k_pool, w.v_pool,
                                                 w.k_scales, w.v_scales, w.slot_mapping)
    ref = oracle.paged_decode_attention(w.q, kp, vp, w.block_tables, w.context_lens, w.scale, ks, vs)
    assert_close(got, ref, "i8", "quantising write + INT8 attention")
    # the generator's pre-quantised rows are the same codes: the copy write gives the same pools
    assert np.array_equal(kp[w.slot_mapping // 16, :, w.slot_mapping % 16], w.k_new)
