"""Helpers for the GPU parity tests: move a seeded workload to the device, run one decode step
through the C ABI binding, and compute the oracle's answer for the same inputs (also for sampled
rows of a prefill, each as the decode query it is); the dead-slot map of a batch's tables and a
copy of a workload with NaN in those slots."""
import numpy as np

import oracle
import paged_kv_decode_reshape_gb300 as P
import workloads as W

# (max-abs, mean-abs, relative L2) against the fp64 oracle. bf16 and INT8 bars as the pages'
# task statement fixes them; fp32 is held to a tighter internal bar; the relative-L2 guard
# keeps long contexts (|out| ~ 1e-2) honest.
TOL = {"f32": (1e-5, 1e-6, 1e-5), "bf16": (2e-2, 2e-3, 2e-2), "i8": (5e-2, 5e-3, 2e-2)}


def _torch():
    import torch
    return torch


def to_dev(a, kind=None):
    torch = _torch()
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:  # bf16 bit patterns
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def to_f64(t):
    torch = _torch()
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def to_host_raw(t):
    """Device tensor -> numpy array in the generator's encoding (bf16 as uint16 bits)."""
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


class DevWorkload:
    def __init__(self, w: W.DecodeWorkload):
        self.w = w
        self.q = to_dev(w.q)
        self.k_pool, self.v_pool = to_dev(w.k_pool), to_dev(w.v_pool)
        self.k_scales, self.v_scales = to_dev(w.k_scales), to_dev(w.v_scales)
        self.block_tables = to_dev(w.block_tables)
        self.context_lens = to_dev(w.context_lens)
        self.slot_mapping = to_dev(w.slot_mapping)
        self.k_new, self.v_new = to_dev(w.k_new), to_dev(w.v_new)
        self.k_new_scales, self.v_new_scales = to_dev(w.k_new_scales), to_dev(w.v_new_scales)

    def write(self, status=None):
        P.kv_cache_write(self.k_new, self.v_new, self.k_pool, self.v_pool, self.slot_mapping,
                         self.k_new_scales, self.v_new_scales, self.k_scales, self.v_scales,
                         status=status)

    def attend(self, chunk=0, status=None, max_context_len=None, workspace=None, out=None):
        torch = _torch()
        w = self.w
        maxc = w.max_context_len if max_context_len is None else max_context_len
        nbytes = P.decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, maxc, chunk)
        if workspace is None and nbytes:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        if out is None:
            out = torch.empty(self.q.shape, dtype=self.q.dtype, device="cuda")
        if w.kv_dtype == "i8":
            P.paged_decode_attention_int8(out, self.q, self.k_pool, self.v_pool, self.k_scales,
                                          self.v_scales, self.block_tables, self.context_lens,
                                          maxc, w.scale, chunk, workspace, status)
        else:
            P.paged_decode_attention(out, self.q, self.k_pool, self.v_pool, self.block_tables,
                                     self.context_lens, maxc, w.scale, chunk, workspace, status)
        return out

    def step(self, chunk=0, status=None):
        self.write(status)
        return self.attend(chunk, status)


def oracle_step(w: W.DecodeWorkload, rows=None, num_threads=8):
    """Oracle answer of one step (write, then attention) for all or the sampled sequences."""
    kp, vp, ks, vs = oracle.kv_cache_write(w.k_new, w.v_new, w.k_pool, w.v_pool, w.slot_mapping,
                                           w.k_new_scales, w.v_new_scales, w.k_scales, w.v_scales)
    rows = np.arange(w.B) if rows is None else np.asarray(rows)
    return oracle.paged_decode_attention(w.q[rows], kp, vp, w.block_tables[rows],
                                         w.context_lens[rows], w.scale, ks, vs,
                                         num_threads=num_threads)


def assert_close(got, ref, kind, what=""):
    mx, mean, rel = TOL[kind]
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    m, a = float(err.max()), float(err.mean())
    r = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    assert m <= mx and a <= mean and r <= rel, (
        f"{what}: max-abs {m:.3g} (<= {mx}), mean-abs {a:.3g} (<= {mean}), rel-L2 {r:.3g} (<= {rel})")
    return m, a, r


def dead_slots(block_tables, context_lens, NB, BS):
    """[NB, BS] True where no sequence's context reaches (the first context_lens[b] positions of
    table b are live; every other slot of every block is dead)."""
    live = np.zeros((NB, BS), dtype=bool)
    for b, n in enumerate(np.asarray(context_lens)):
        for t0 in range(0, int(n), BS):
            live[int(block_tables[b][t0 // BS]), :min(BS, int(n) - t0)] = True
    return ~live


def prefill_rows_by_decode(w, rows, num_threads=8, orc=None):
    """Oracle rows of a paged prefill, each computed as the decode query it is by definition:
    query row i of sequence b attends to the first context_lens[b] - (L_b - 1 - i) tokens of its
    table. `rows` are flat query-token rows; returns fp64 [len(rows), Hq, D]. `orc`: the oracle
    module to use (default: the oracle)."""
    orc = oracle if orc is None else orc
    rows = np.asarray(rows)
    qs = np.asarray(w.query_start)
    b = np.searchsorted(qs, rows, side="right") - 1
    L = qs[b + 1] - qs[b]
    i = rows - qs[b]
    n = np.asarray(w.context_lens)[b] - (L - 1 - i)
    return orc.paged_decode_attention(w.q[rows], w.k_pool, w.v_pool, np.asarray(w.block_tables)[b],
                                         n.astype(np.int32), w.scale, w.k_scales, w.v_scales,
                                         num_threads=num_threads)


def poisoned(w):
    """A copy of workload w with NaN in every dead slot (dead_slots): bf16 / fp32 K and V rows, or
    for an INT8 cache the K and V scales."""
    NB, Hkv, BS, D = w.k_pool.shape
    dead = dead_slots(w.block_tables, w.context_lens, NB, BS)
    rep = {}
    if w.kv_dtype == "i8":
        m = np.broadcast_to(dead[:, None, :], w.k_scales.shape)
        for name in ("k_scales", "v_scales"):
            a = getattr(w, name).copy()
            a[m] = np.nan
            rep[name] = a
    else:
        m = np.broadcast_to(dead[:, None, :, None], w.k_pool.shape)
        nan = np.uint16(0x7FC0) if w.k_pool.dtype == np.uint16 else np.float32(np.nan)
        for name in ("k_pool", "v_pool"):
            a = getattr(w, name).copy()
            a[m] = nan
            rep[name] = a
    assert dead.any(), "the workload leaves no slot dead"
    return type(w)(**{**w.__dict__, **rep})
