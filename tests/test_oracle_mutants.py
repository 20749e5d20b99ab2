"""The oracle's pins have teeth.

Each mutant below plants one plausible mistake in a copy of the oracle's C
source: a dropped term, a wrong sign, index or operand, a reversed order, a
swapped argument.  The copy is compiled on the CPU into a temporary directory
(the oracle itself is never modified), every pin of test_oracle_pins runs
against it, and at least one pin must fail.  A mutant that survives means a
mistake of that kind could sit in the oracle unnoticed.
"""
import importlib
import importlib.util
import inspect
import os
import pathlib
import shutil
import subprocess

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")
HDR = os.path.join(ROOT, "oracle", "oracle.h")

# (name, text in oracle.c, replacement); each text occurs exactly once.  Every
# replacement keeps all memory accesses in bounds.
MUTANTS = [
    ("bf16 rounds ties away from zero",
     "u = (u + 0x7fffu + keep_lsb) & 0xffff0000u;", "u = (u + 0x8000u + 0u * keep_lsb) & 0xffff0000u;"),
    ("serial sum runs right to left",
     "for (int64_t i = 1; i < n; ++i) acc = acc + x[i];", "for (int64_t i = n - 1; i >= 1; --i) acc = acc + x[i];"),
    ("rmsnorm mean over d - 1", "float mean = ss / (float)d;", "float mean = ss / (float)(d - 1);"),
    ("rmsnorm drops eps", "float rinv = 1.0f / sqrtf(mean + eps);", "float rinv = 1.0f / sqrtf(mean);"),
    ("rmsnorm drops gamma", "float v = (xr[i] * rinv) * gamma[i];", "float v = xr[i] * rinv;"),
    ("matmul reads W transposed",
     "for (int32_t k = 0; k < K; ++k) acc = acc + a[k] * w[k];",
     "for (int32_t k = 0; k < K; ++k) acc = acc + a[k] * W[((int64_t)k * N + n) % ((int64_t)N * K)];"),
    ("softmax skips the max shift", "p[j] = expf(s[j] - m);", "p[j] = expf(s[j]);"),
    ("softmax skips normalisation",
     "for (int32_t j = 0; j < n; ++j) p[j] = p[j] / z;", "for (int32_t j = 0; j < n; ++j) p[j] = p[j] * 1.0f;"),
    ("silu sign", "float silu = g[i] / (1.0f + expf(-g[i]));", "float silu = g[i] / (1.0f + expf(g[i]));"),
    ("gate and up swapped in the layer", "orc_swiglu(g, u, g, T * F, rb);", "orc_swiglu(u, g, g, T * F, rb);"),
    ("argmax ties go to the last index", "if (c_nan || c > b) best = j;", "if (c_nan || c >= b) best = j;"),
    ("argmax: a later NaN displaces the first", "if (b_nan) break; ", "if (b_nan && 0) break; "),
    ("log_softmax drops log z",
     "lp[r * (int64_t)n + j] = ((double)xr[j] - m) - lz;", "lp[r * (int64_t)n + j] = ((double)xr[j] - m);"),
    ("log_softmax shifts by the first logit, not the max",
     "for (int32_t j = 1; j < n; ++j) if ((double)xr[j] > m) m = (double)xr[j];",
     "for (int32_t j = 1; j < n; ++j) if (0) m = (double)xr[j];"),
    ("murmur3 block constant", "h = h * 5u + 0xe6546b64u;", "h = h * 5u + 0xe6546b65u;"),
    ("murmur3 tail byte shift", "case 3: k ^= (uint32_t)tail[2] << 16;", "case 3: k ^= (uint32_t)tail[2] << 8;"),
    ("murmur3 drops the length", "h ^= (uint32_t)len;", "h ^= 0u;"),
    ("exponential instead of Gumbel noise", "const double g = -log(-log(u));", "const double g = -log(u);"),
    ("logits multiplied by the temperature",
     "const double sc = (double)x[j] / (double)t + g;", "const double sc = (double)x[j] * (double)t + g;"),
    ("rope sign", "xv[i] = a - b;", "xv[i] = a + b;"),
    ("rope pairs neighbours, not halves",
     "float x0 = xv[i], x1 = xv[i + half];", "float x0 = xv[i], x1 = xv[(i ^ 1) + half];"),
    ("rope frequency exponent", "double inv_freq = pow(theta, -(double)(2 * i) / (double)Dh);",
     "double inv_freq = pow(theta, -(double)(i) / (double)Dh);"),
    ("attention drops the scale",
     "s[j] = dot_serial(q, k + (int64_t)j * kv_stride, Dh) * scale;",
     "s[j] = dot_serial(q, k + (int64_t)j * kv_stride, Dh);"),
    ("attention pairs p with the wrong value row",
     "acc = acc + p[j] * v[(int64_t)j * kv_stride + d];",
     "acc = acc + p[j] * v[(int64_t)(n_keys - 1 - j) * kv_stride + d];"),
    ("split merge drops the rescale of l",
     "L = L + l[c] * expf(m[c] - M);", "L = L + l[c];"),
    ("GQA maps heads round robin", "int32_t kvh = h / group;", "int32_t kvh = h % Hkv;"),
    ("attention skips the diagonal key",
     "p + 1, (int64_t)Hkv * Dh, Dh, scale,", "(p > 0 ? p : 1), (int64_t)Hkv * Dh, Dh, scale,"),
    ("attention residual dropped",
     "x_out[j] = maybe_round(x_in[j] + tmp[j], rb);", "x_out[j] = maybe_round(tmp[j], rb);"),
    ("rope applied to v as well", "for (int32_t h = 0; h < H + Hkv; ++h)", "for (int32_t h = 0; h < H + 2 * Hkv; ++h)"),
    ("lm head skips the final norm",
     "orc_matmul(y, w_lm, logits, R, V, d);", "orc_matmul(xr, w_lm, logits, R, V, d);"),
    ("lm head takes rows 0..R-1",
     "memcpy(xr + (int64_t)r * d, x + (int64_t)rows[r] * d,", "memcpy(xr + (int64_t)r * d, x + (int64_t)r * d,"),
    ("embedding row off by one",
     "E + (int64_t)ids[t] * d,", "E + (int64_t)(ids[t] > 0 ? ids[t] - 1 : 0) * d,"),
]


# Conventions the pages state only in words, with no printed value to pin them:
# a mutant here passes every pin, and the oracle's header and the design notes
# say so.  The pages name the hash's inputs (seed, position, column) but not the
# byte layout of the key; the reading is le32(position) followed by le32(column).
UNPINNED = [
    ("hash key: column before position",
     "key[b] = (uint8_t)(p >> (8 * b));\n            key[4 + b] = (uint8_t)(c >> (8 * b));",
     "key[b] = (uint8_t)(c >> (8 * b));\n            key[4 + b] = (uint8_t)(p >> (8 * b));"),
]


# Mistakes planted in the oracle's Python wrapper (argument marshalling): the
# mutated copy of the package reuses the unmutated compiled library.
PY_MUTANTS = [
    ("history rows shifted by one position",
     "k_pool[row0[i]:row0[i] + pos0[i]] = k_hist[i][:pos0[i]]",
     "k_pool[row0[i]:row0[i] + pos0[i]] = np.roll(k_hist[i][:pos0[i]], 1, axis=0)"),
    ("pool offsets from query lengths, not context lengths",
     "row0[1:] = np.cumsum(rows)[:-1]", "row0[1:] = np.cumsum(q_lens)[:-1]"),
    ("returned caches start one row late",
     "k_new = [k_pool[row0[i]:row0[i] + rows[i]] for i in range(B)]",
     "k_new = [k_pool[row0[i] + 1:row0[i] + rows[i] + 1] for i in range(B)]"),
    ("default attention scale 1/Dh",
     "scale = np.float32(1.0) / np.sqrt(np.float32(Dh)) if scale is None else scale\n    out = np.empty(Dh, np.float32)\n"
     "    _check(lib().orc_attention_head(",
     "scale = np.float32(1.0) / np.float32(Dh) if scale is None else scale\n    out = np.empty(Dh, np.float32)\n"
     "    _check(lib().orc_attention_head("),
    ("rope table one position short", "n_pos = int(pos.max()) + 1 if pos.size else 1",
     "n_pos = int(pos.max()) if pos.size else 1"),
]


@pytest.fixture
def build_dir(request):
    """Where this test's copies are built: the oracle's own (git-ignored) build folder, emptied afterwards."""
    d = pathlib.Path(ROOT) / "oracle" / "_build" / "mutants" / request.node.name
    shutil.rmtree(d, ignore_errors=True)
    d.mkdir(parents=True)
    yield d
    shutil.rmtree(d, ignore_errors=True)


def _pin_cases():
    """Every (pin, arguments) of test_oracle_pins, parametrisations expanded."""
    mod = importlib.import_module("tests.test_oracle_pins")
    golden = os.path.join(ROOT, "tests", "golden")
    cases = []
    for name, fn in inspect.getmembers(mod, inspect.isfunction):
        if not name.startswith("test_") or fn.__module__ != mod.__name__:
            continue
        params = [{}]
        for mark in getattr(fn, "pytestmark", []):
            if mark.name != "parametrize":
                continue
            names = [s.strip() for s in mark.args[0].split(",")]
            params = [{**p, **dict(zip(names, vals if len(names) > 1 else (vals,)))}
                      for p in params for vals in mark.args[1]]
        for p in params:
            if "golden_dir" in inspect.signature(fn).parameters:
                p = {**p, "golden_dir": golden}
            cases.append((name, fn, p))
    return cases


def _compile(tmp, text, repl):
    src = open(SRC).read()
    assert src.count(text) == 1, text
    d = os.path.join(tmp, "m")
    os.makedirs(d, exist_ok=True)
    shutil.copy(HDR, d)
    with open(os.path.join(d, "oracle.c"), "w") as fh:
        fh.write(src.replace(text, repl))
    so = os.path.join(d, "liboracle_mutant.so")
    cc = shutil.which("gcc") or shutil.which("cc")
    subprocess.run([cc, "-O1", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                    os.path.join(d, "oracle.c"), "-o", so, "-lm"], check=True, capture_output=True, text=True)
    return so


def _killed(cases) -> bool:
    for _, fn, kw in cases:
        try:
            fn(**kw)
        except Exception:  # an assertion, or the oracle reporting an error
            return True
    return False


def _survivors(mutants, folder, monkeypatch):
    cases = _pin_cases()
    assert len(cases) > 40
    survivors = []
    for i, (name, text, repl) in enumerate(mutants):
        so = _compile(str(folder / str(i)), text, repl)
        monkeypatch.setattr(oracle, "_lib", oracle.bind(so))
        if not _killed(cases):
            survivors.append(name)
    monkeypatch.undo()
    return survivors


def _py_mutant(tmp, name, text, repl):
    """A copy of the oracle package with one wrapper mistake, bound to the unmutated library."""
    src = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    assert src.count(text) == 1, text
    d = os.path.join(tmp, "pkg")
    os.makedirs(d, exist_ok=True)
    path = os.path.join(d, "__init__.py")
    with open(path, "w") as fh:
        fh.write(src.replace(text, repl))
    spec = importlib.util.spec_from_file_location(f"oracle_mutant_{abs(hash(name))}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._lib = mod.bind(oracle.build())  # its own handle: argument types name the copy's structures
    return mod


def test_unmutated_oracle_passes_every_pin():
    for _, fn, kw in _pin_cases():
        fn(**kw)


def test_every_mutant_fails_a_pin(build_dir, monkeypatch):
    # control: an unchanged copy built the way the mutants are passes every pin
    text = MUTANTS[0][1]
    assert _survivors([("copy", text, text)], build_dir / "copy", monkeypatch) == ["copy"]
    survivors = _survivors(MUTANTS, build_dir, monkeypatch)
    assert not survivors, f"mutants no pin catches: {survivors}"


def test_unpinned_readings_are_still_unpinned(build_dir, monkeypatch):
    """If a pin comes to catch one of these, move it to MUTANTS and drop its "parity unpinned" notes."""
    assert _survivors(UNPINNED, build_dir, monkeypatch) == [m[0] for m in UNPINNED]


def test_every_wrapper_mutant_fails_a_pin(build_dir, monkeypatch):
    pins = importlib.import_module("tests.test_oracle_pins")
    cases = _pin_cases()
    text = PY_MUTANTS[0][1]
    monkeypatch.setattr(pins, "oracle", _py_mutant(str(build_dir / "copy"), "copy", text, text))
    assert not _killed(cases), "an unmutated copy of the wrapper fails a pin"
    monkeypatch.undo()
    survivors = []
    for i, (name, text, repl) in enumerate(PY_MUTANTS):
        monkeypatch.setattr(pins, "oracle", _py_mutant(str(build_dir / str(i)), name, text, repl))
        if not _killed(cases):
            survivors.append(name)
        monkeypatch.undo()
    assert not survivors, f"wrapper mutants no pin catches: {survivors}"
