"""The oracle's pins must catch a planted mistake.

Each case copies pkv_oracle.c, plants one plausible mistake by a textual substitution (a dropped
term, a wrong sign, index or operand, an off-by-one limit, a wrong rounding rule), compiles the
copy on the CPU, points the oracle binding at it, and runs the pin tests of test_oracle_pins.py
and test_golden.py. At least one pin must fail for every mutant; the unmutated source must pass
all of them. The oracle source itself carries no switches: mistakes are only ever planted in a
temporary copy.
"""
import inspect
import subprocess

import pytest

import oracle
from oracle import build as oracle_build

import test_golden
import test_oracle_pins

# (name, [(text, replacement, occurrences)]) -- every text must occur exactly `occurrences` times
MUTANTS = [
    ("gqa head map by modulo", [("int kvh = h / (P->Hq / P->Hkv);", "int kvh = h % P->Hkv;", 2)]),
    ("block index from the offset",
     [("P->block_tables[(size_t)b * P->MBPS + t / P->BS]", "P->block_tables[(size_t)b * P->MBPS + t % P->BS]", 1)]),
    ("row offset shifted", [("int off = t % P->BS;", "int off = (t + 1) % P->BS;", 1)]),
    ("scale dropped", [("s[t - lo] = P->scale * dot;", "s[t - lo] = dot;", 1)]),
    ("K dequantised with the V scale",
     [("sc = (double)(which_v ? P->v_scales : P->k_scales)[r];", "sc = (double)P->v_scales[r];", 1)]),
    ("scores against V instead of K",
     [("int rc = gather_row(P, b, kvh, t, 0, row);", "int rc = gather_row(P, b, kvh, t, 1, row);", 1)]),
    ("softmax not normalised", [("for (int d = 0; d < P->D; ++d) o[d] = acc[d] / l;",
                                 "for (int d = 0; d < P->D; ++d) o[d] = acc[d];", 1)]),
    ("context one short", [("int rc = partial(P, b, h, 0, n, &m, &l, acc, s, row);",
                            "int rc = partial(P, b, h, 0, n - 1, &m, &l, acc, s, row);", 1)]),
    ("exponent sign flipped", [("double p = exp(s[t - lo] - m);", "double p = exp(m - s[t - lo]);", 1)]),
    ("merge weight inverted", [("double w = exp(m[base + j] - M);", "double w = exp(M - m[base + j]);", 1)]),
    ("split count rounded up", [("int s0 = n / chunk;", "int s0 = (n + chunk - 1) / chunk;", 1)]),
    ("splits not whole blocks", [("per = ((per + BS - 1) / BS) * BS;", "per = per + 0;", 1)]),
    ("quantiser rounds half away from zero", [("rintf(", "roundf(", 1)]),
    ("quantiser scale over 128", [("float scale = amax / 127.0f;", "float scale = amax / 128.0f;", 1)]),
    ("multi-token causal limit off", [("int n_l = context_lens[b] - (L - 1 - l);",
                                       "int n_l = context_lens[b] - l;", 1)]),
    ("prefill causal limit one short", [("int n_i = context_lens[b] - (L - 1 - i);",
                                         "int n_i = context_lens[b] - (L - i);", 1)]),
    ("written to the next slot", [("int64_t blk = s / BS, off = s % BS;",
                                   "int64_t blk = s / BS, off = (s + 1) % BS;", 2)]),
    ("bf16 decoded with the wrong shift", [("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;", 1)]),
    ("merge sum not weighted", [("L += l[base + j] * w;", "L += l[base + j];", 1)]),
    ("split ranges overlap by a token", [("int lo = j * per, hi = lo + per < n ? lo + per : n;",
                                          "int lo = j * per, hi = lo + per + 1 < n ? lo + per + 1 : n;", 1)]),
    ("prefill query row from the sequence index", [("size_t r = (size_t)(query_start[b] + i) * Hq + h;",
                                                   "size_t r = (size_t)(b + i) * Hq + h;", 1)]),
    ("multi-token rows transposed", [("size_t r = (size_t)(b * L + l) * Hq + h;",
                                      "size_t r = (size_t)(l * B + b) * Hq + h;", 1)]),
    ("prefill skips the first key", [("rc = partial_q(&P, r * D, b, h, 0, n_i, &m, &lsum, acc, s, row);",
                                      "rc = partial_q(&P, r * D, b, h, 1, n_i, &m, &lsum, acc, s, row);", 1)]),
    ("prefill output not normalised",
     [("rc = partial_q(&P, r * D, b, h, 0, n_i, &m, &lsum, acc, s, row);\n"
       "                if (rc) break;\n"
       "                double* o = out + r * D;\n"
       "                for (int d = 0; d < D; ++d) o[d] = acc[d] / lsum;",
       "rc = partial_q(&P, r * D, b, h, 0, n_i, &m, &lsum, acc, s, row);\n"
       "                if (rc) break;\n"
       "                double* o = out + r * D;\n"
       "                for (int d = 0; d < D; ++d) o[d] = acc[d];", 1)]),
]


def _pins():
    """(name, callable taking the oracle module) for every pin test, parametrisations expanded."""
    out = []
    for mod in (test_oracle_pins, test_golden):
        for name, fn in sorted(vars(mod).items()):
            if not name.startswith("test_") or not callable(fn):
                continue
            marks = getattr(fn, "pytestmark", [])
            params = [m for m in marks if m.name == "parametrize"]
            sig = inspect.signature(fn)
            combos = [dict()]
            for m in params:
                names = [s.strip() for s in m.args[0].split(",")] if isinstance(m.args[0], str) else list(m.args[0])
                new = []
                for c in combos:
                    for v in m.args[1]:
                        vals = v if len(names) > 1 else (v,)
                        new.append({**c, **dict(zip(names, vals))})
                combos = new
            for c in combos:
                kw = dict(c)
                if "orc" in sig.parameters:
                    kw["orc"] = oracle
                missing = [p for p in sig.parameters if p not in kw]
                if missing:
                    continue  # needs a fixture this harness does not provide
                out.append((f"{mod.__name__}.{name}{c}", fn, kw))
    return out


def _build(src_text, path):
    with open(path + ".c", "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O1", "-std=c99", "-D_POSIX_C_SOURCE=200809L", "-fPIC", "-shared",
                    "-w", "-o", path, path + ".c", "-lm", "-lpthread"], check=True)


def _run_pins(lib_path):
    saved_build, saved_lib = oracle._build.build, oracle._lib
    oracle._build.build = lambda *a, **k: lib_path
    oracle._lib = None
    failed = []
    try:
        for name, fn, kw in _pins():
            try:
                fn(**kw)
            except Exception as e:  # any failure of a pin counts (assertion, error status)
                failed.append((name, type(e).__name__))
    finally:
        oracle._build.build, oracle._lib = saved_build, saved_lib
    return failed


@pytest.fixture(scope="module")
def source():
    with open(oracle_build.SRC) as f:
        return f.read()


def test_unmutated_copy_passes_every_pin(source, tmp_path):
    path = str(tmp_path / "liborc_clean.so")
    _build(source, path)
    assert _run_pins(path) == []
    assert len(_pins()) >= 25


@pytest.mark.parametrize("name,subs", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(source, tmp_path, name, subs):
    text = source
    for old, new, count in subs:
        assert text.count(old) == count, f"mutation site moved: {old!r}"
        text = text.replace(old, new)
    path = str(tmp_path / "liborc_mutant.so")
    _build(text, path)
    failed = _run_pins(path)
    assert failed, f"no pin caught the planted mistake: {name}"


# ---- the block manager's oracle (oracle/block_manager.py): same idea, Python source ------------

import importlib.util  # noqa: E402

import test_block_manager  # noqa: E402
from oracle import block_manager as oracle_bm  # noqa: E402

BM_MUTANTS = [
    ("copy-on-write skipped", [('elif self.users[rec["table"][-1]] > 1:', "elif False:", 1)]),
    ("copy reported the wrong way", [("copies.append((src, dst))", "copies.append((dst, src))", 1)]),
    ("fork does not count its references",
     [('for b in par["table"]:\n            self.users[b] += 1', 'for b in par["table"]:\n            pass', 1)]),
    ("can_append ignores the copy", [("need += 1", "need += 0", 1)]),
    ("hash chain broken", [('head = b"" if previous is None else struct.pack("<Q", previous & _M)',
                            'head = b""', 1)]),
    ("shared prompt blocks taken fresh", [("if self.users[b] == 0:\n                        self.free.remove(b)\n"
                                           "                    self.users[b] += 1",
                                           "if self.users[b] == 0:\n                        self.free.remove(b)\n"
                                           "                    self.users[b] += 0", 1)]),
]


def _bm_pins():
    return [fn for name, fn in sorted(vars(test_block_manager).items())
            if name.startswith("test_oracle_") and callable(fn)]


def _run_bm_pins(module):
    saved = test_block_manager.O
    test_block_manager.O = module
    failed = []
    try:
        for fn in _bm_pins():
            marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
            combos = [dict(zip([m.args[0]], [v])) for m in marks for v in m.args[1]] or [{}]
            for kw in combos:
                try:
                    fn(**kw)
                except Exception as e:
                    failed.append((fn.__name__, kw, type(e).__name__))
    finally:
        test_block_manager.O = saved
    return failed


def _load_bm(text, path):
    with open(path, "w") as f:
        f.write(text)
    spec = importlib.util.spec_from_file_location("bm_mutant", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.fixture(scope="module")
def bm_source():
    with open(oracle_bm.__file__) as f:
        return f.read()


def test_block_manager_oracle_unmutated_copy_passes_every_pin(bm_source, tmp_path):
    assert _run_bm_pins(_load_bm(bm_source, str(tmp_path / "bm_clean.py"))) == []
    assert len(_bm_pins()) >= 4


@pytest.mark.parametrize("name,subs", BM_MUTANTS, ids=[m[0] for m in BM_MUTANTS])
def test_block_manager_oracle_planted_mistake_fails_a_pin(bm_source, tmp_path, name, subs):
    text = bm_source
    for old, new, count in subs:
        assert text.count(old) == count, f"mutation site moved: {old!r}"
        text = text.replace(old, new)
    failed = _run_bm_pins(_load_bm(text, str(tmp_path / "bm_mutant.py")))
    assert failed, f"no pin caught the planted mistake: {name}"
