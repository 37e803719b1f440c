"""The oracle's pins have teeth: each plausible mistake planted in a copy of the oracle (a
dropped term, a wrong sign, a transposed operand, a wrong index, an off-by-one, a step in the
wrong order) makes at least one pin in tests/test_oracle_*.py fail.

The mistakes are planted on the host only, in throwaway copies: the C oracle is copied to a
temporary directory, edited as text and compiled with the oracle's own gcc flags; the Python
modules are edited as text and executed into fresh module objects whose functions replace the
real ones for the duration of one check.  The real oracle is never modified.  An unmodified
copy passes every pin, so a failure below comes from the planted mistake, not the harness.
"""
import importlib.util
import itertools
import os
import subprocess
import types

import numpy as np
import pytest

import oracle
from oracle import policy, q8

HERE = os.path.dirname(os.path.abspath(__file__))
ORACLE_DIR = os.path.dirname(os.path.abspath(oracle.__file__))
PIN_FILES = {
    "recurrence": "test_oracle_recurrence.py",
    "policy": "test_oracle_policy.py",
    "q8": "test_oracle_q8.py",
}


def _load_pins(key):
    path = os.path.join(HERE, PIN_FILES[key])
    spec = importlib.util.spec_from_file_location(f"_pins_{key}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _cases(mod):
    """Every (name, function, kwargs) a pin module defines, parametrizations expanded."""
    out = []
    for name in sorted(n for n in dir(mod) if n.startswith("test_")):
        fn = getattr(mod, name)
        grids = []
        for m in getattr(fn, "pytestmark", []):
            if m.name != "parametrize":
                continue
            names, values = m.args[0], m.args[1]
            names = [x.strip() for x in names.split(",")] if isinstance(names, str) else list(names)
            rows = [v if len(names) > 1 else (v,) for v in values]
            grids.append([dict(zip(names, row)) for row in rows])
        for combo in itertools.product(*grids) if grids else [()]:
            kw = {}
            for part in combo:
                kw.update(part)
            out.append((name, fn, kw))
    return out


def _first_failing_pin(keys, stop=True):
    """Run the pins of the given modules; return the names of the ones that fail."""
    failed = []
    for key in keys:
        for name, fn, kw in _cases(_load_pins(key)):
            try:
                fn(**kw)
            except (AssertionError, pytest.fail.Exception):
                failed.append(f"{PIN_FILES[key]}::{name}{kw or ''}")
                if stop:
                    return failed
    return failed


def _edit(src, edits):
    for old, new in edits:
        assert src.count(old) >= 1, f"planting site not found: {old!r}"
        src = src.replace(old, new)
    return src


# ------------------------------------------------------------------ the C oracle
_DECAY = ("        /* decay: row i scaled by alpha_t[i] */\n"
          "        for (int32_t i = 0; i < d; ++i)\n"
          "            for (int32_t j = 0; j < d; ++j)\n"
          "                S[(int64_t)i * d + j] *= at[i];\n")
_READ = ("        /* read o = S^T q */\n"
         "        if (o) {\n"
         "            for (int32_t j = 0; j < d; ++j) {\n"
         "                double acc = 0.0;\n"
         "                for (int32_t i = 0; i < d; ++i)\n"
         "                    acc += S[(int64_t)i * d + j] * qt[i];\n"
         "                o[t * o_ld + j] = acc;\n"
         "            }\n"
         "        }\n")
_WRITE_START = "        /* delta-rule write vector w = beta (v - S^T k) */\n"

C_MUTANTS = {
    # recurrence step
    "write without beta": [("w[j] = bt * (vt[j] - acc);", "w[j] = (vt[j] - acc);")],
    "write with the prediction added": [("w[j] = bt * (vt[j] - acc);", "w[j] = bt * (vt[j] + acc);")],
    "prediction S k instead of S^T k": [("acc += S[(int64_t)i * d + j] * kt[i];",
                                         "acc += S[(int64_t)j * d + i] * kt[i];")],
    "read S q instead of S^T q": [("acc += S[(int64_t)i * d + j] * qt[i];",
                                   "acc += S[(int64_t)j * d + i] * qt[i];")],
    "decay along the value channel": [("S[(int64_t)i * d + j] *= at[i];",
                                       "S[(int64_t)i * d + j] *= at[j];")],
    "update w k^T instead of k w^T": [("S[(int64_t)i * d + j] += kt[i] * w[j];",
                                       "S[(int64_t)i * d + j] += kt[j] * w[i];")],
    "decay after the write": [(_DECAY, ""), (_READ, _DECAY + _READ)],
    "read before the update": [(_READ, ""), (_DECAY, _READ + _DECAY)],
    "decay skipped": [(_DECAY, "")],
    # explicit segment map
    "segment map decays the wrong side": [
        ("- bt * kt[i] * kt[m]) * at[m];", "- bt * kt[i] * kt[m]) * at[i];")],
    "segment maps composed in the wrong order": [
        ("acc += Mt[(size_t)i * d + m] * M[(size_t)m * d + j];",
         "acc += M[(size_t)i * d + m] * Mt[(size_t)m * d + j];")],
    "segment offset not carried through M_t": [
        ("tmp[(size_t)i * d + j] = acc + bt * kt[i] * vt[j];",
         "tmp[(size_t)i * d + j] = b[(size_t)i * d + j] + bt * kt[i] * vt[j];")],
    "segment offset k k^T instead of k v^T": [
        ("tmp[(size_t)i * d + j] = acc + bt * kt[i] * vt[j];",
         "tmp[(size_t)i * d + j] = acc + bt * kt[i] * kt[j];")],
    "segment map starts from zero": [("M[(size_t)i * d + i] = 1.0;", "M[(size_t)i * d + i] = 0.0;")],
    # full path: conv, indexing, checkpoints
    "conv taps reversed": [
        ("xc[c] = wk[0] * win[c] + wk[1] * win[C + c] + wk[2] * win[2 * C + c] + wk[3] * xr[c];",
         "xc[c] = wk[3] * win[c] + wk[2] * win[C + c] + wk[1] * win[2 * C + c] + wk[0] * xr[c];")],
    "conv window never shifted": [("memmove(win, win + C, sizeof(double) * 2 * (size_t)C);", "")],
    "conv window keeps post-conv values": [
        ("memcpy(win + 2 * C, xr, sizeof(double) * (size_t)C);",
         "memcpy(win + 2 * C, xc, sizeof(double) * (size_t)C);")],
    "conv weights of head 0 for every head": [
        ("const double *wc = conv_w + (int64_t)h * C * 4;", "const double *wc = conv_w;")],
    "q and k channels swapped": [
        ("xr[c] = q[row * d + c];\n                xr[d + c] = k[row * d + c];",
         "xr[c] = k[row * d + c];\n                xr[d + c] = q[row * d + c];")],
    "beta of head 0 for every head": [("beta + row, 0,", "beta + (t0 + t) * H, 0,")],
    "decay of the next token": [("alpha + row * d, 0,", "alpha + (row + (t + 1 < T ? H : 0)) * d, 0,")],
    "checkpoint one token late": [("ck_at[ck] == t + 1", "ck_at[ck] == t")],
    "initial state ignored": [
        ("if (S0) memcpy(S, S0 + ((int64_t)s * H + h) * d * d, sizeof(double) * (size_t)d * d);", "")],
    "initial window ignored": [
        ("if (win0) memcpy(win, win0 + ((int64_t)s * H + h) * 3 * C, sizeof(double) * 3 * (size_t)C);", "")],
}


def _build_c(src, path):
    with open(path + ".c", "w") as f:
        f.write(src)
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared",
                    "-fPIC", "-std=c11", "-o", path, path + ".c"], check=True)


def _with_c_library(monkeypatch, so):
    monkeypatch.setattr(oracle, "_lib", None)
    monkeypatch.setattr(oracle, "_SO", so)
    monkeypatch.setattr(oracle, "build", lambda force=False: so)


@pytest.fixture(scope="module")
def c_source():
    with open(os.path.join(ORACLE_DIR, "kda_oracle.c")) as f:
        return f.read()


def test_unmodified_c_copy_passes_every_pin(c_source, tmp_path, monkeypatch):
    so = str(tmp_path / "liboracle_copy.so")
    _build_c(c_source, so)
    _with_c_library(monkeypatch, so)
    assert _first_failing_pin(["recurrence"], stop=False) == []


@pytest.mark.parametrize("name", sorted(C_MUTANTS))
def test_c_mistake_is_caught(name, c_source, tmp_path, monkeypatch):
    so = str(tmp_path / "liboracle_mutant.so")
    _build_c(_edit(c_source, C_MUTANTS[name]), so)
    _with_c_library(monkeypatch, so)
    assert _first_failing_pin(["recurrence"]), f"no pin catches: {name}"


# ------------------------------------------------------------------ the Python oracle
POLICY_MUTANTS = {
    "positions start at the resume point": [
        ("first = (start // step + 1) * step", "first = (start // step) * step")],
    "positions exclude the end": [("out = list(range(first, end + 1, step))",
                                   "out = list(range(first, end, step))")],
    "last aligned position rounded up": [("last = (end // hash_block) * hash_block",
                                          "last = -(-end // hash_block) * hash_block")],
    "hit strictly below the matched length": [("if p <= matched and p > best:",
                                               "if p < matched and p > best:")],
    "decode checkpoint one step early": [("return pos > 0 and pos % interval == 0",
                                          "return pos > 0 and (pos + 1) % interval == 0")],
    "records padded to 128 bytes": [("raw = d * d * 4 + 3 * 3 * d * DTYPE_SIZE[dtype]\n    return (raw + 255) // 256 * 256",
                                     "raw = d * d * 4 + 3 * 3 * d * DTYPE_SIZE[dtype]\n    return (raw + 127) // 128 * 128")],
    "state stored column-major": [
        ("body = np.ascontiguousarray(S, dtype=np.float64).astype(np.float32).tobytes()",
         "body = np.ascontiguousarray(S.T, dtype=np.float64).astype(np.float32).tobytes()"),
        ("S = np.frombuffer(buf[:nS], dtype=np.float32).astype(np.float64).reshape(d, d)",
         "S = np.frombuffer(buf[:nS], dtype=np.float32).astype(np.float64).reshape(d, d).T")],
    "window stored channel-major": [
        ("body += _window_bytes(np.asarray(win).reshape(3, 3 * d), dtype)",
         "body += _window_bytes(np.asarray(win).reshape(3, 3 * d).T, dtype)"),
        ("return S, win.reshape(3, 3 * d)", "return S, win.reshape(3 * d, 3).T")],
    "pages of an object in reverse order": [
        ("p = pages[x0 // page_bytes]", "p = pages[len(pages) - 1 - x0 // page_bytes]")],
    "highest free page first": [("ids = free[:n]", "ids = free[len(free) - n:]")],
    "checkpoint pages in position-major order": [
        ("    return [(s, p, pool.alloc(pages_per_object)) for s, p in items]",
         "    items.sort(key=lambda x: (x[1], x[0]))\n"
         "    return [(s, p, pool.alloc(pages_per_object)) for s, p in items]")],
    "ping-pong pages for requests that are not due": [
        ("due = [r for r, p in enumerate(pos) if decode_ckpt_due(p, interval)]",
         "due = [r for r, p in enumerate(pos) if not decode_ckpt_due(p, interval)]")],
}

Q8_MUTANTS = {
    "scale max / 128": [("QMAX = 127", "QMAX = 128")],
    "rounding half up": [("q = np.rint((S / safe[:, None]).astype(np.float32))",
                          "q = np.floor((S / safe[:, None]).astype(np.float32) + np.float32(0.5))")],
    "rounding toward zero": [("q = np.rint((S / safe[:, None]).astype(np.float32))",
                              "q = np.trunc((S / safe[:, None]).astype(np.float32))")],
    "scale per value channel": [("amax = np.max(np.abs(S), axis=1)", "amax = np.max(np.abs(S), axis=0)")],
    "dequantised with the transposed scale": [
        ("np.asarray(codes, dtype=np.int8).astype(np.float32) * scale[:, None]",
         "np.asarray(codes, dtype=np.int8).astype(np.float32) * scale[None, :]")],
    "codes before scales in the record": [
        ("body = scale.tobytes() + q.tobytes() + policy._window_bytes",
         "body = q.tobytes() + scale.tobytes() + policy._window_bytes"),
        ("scale = np.frombuffer(buf[:4 * d], dtype=np.float32).copy()\n"
         "    codes = np.frombuffer(buf[4 * d:4 * d + d * d], dtype=np.int8).reshape(d, d).copy()",
         "scale = np.frombuffer(buf[d * d:d * d + 4 * d], dtype=np.float32).copy()\n"
         "    codes = np.frombuffer(buf[:d * d], dtype=np.int8).reshape(d, d).copy()")],
}


def _module_from(src, name):
    mod = types.ModuleType(name)
    mod.__dict__["__name__"] = name
    exec(compile(src, name, "exec"), mod.__dict__)
    return mod


def _patch_module(monkeypatch, real, fake):
    for attr, val in vars(real).items():
        if attr.startswith("__") or isinstance(val, types.ModuleType):
            continue
        if callable(val) and getattr(val, "__module__", None) == real.__name__:
            monkeypatch.setattr(real, attr, getattr(fake, attr))
    for attr in ("QMAX", "DTYPE_SIZE"):
        if hasattr(real, attr):
            monkeypatch.setattr(real, attr, getattr(fake, attr))


def _py_source(fname):
    with open(os.path.join(ORACLE_DIR, fname)) as f:
        return f.read().replace("from . import policy", "from oracle import policy")


def test_unmodified_python_copies_pass_every_pin(monkeypatch):
    _patch_module(monkeypatch, policy, _module_from(_py_source("policy.py"), "_copy_policy"))
    _patch_module(monkeypatch, q8, _module_from(_py_source("q8.py"), "_copy_q8"))
    assert _first_failing_pin(["policy", "q8"], stop=False) == []


@pytest.mark.parametrize("name", sorted(POLICY_MUTANTS))
def test_policy_mistake_is_caught(name, monkeypatch):
    fake = _module_from(_edit(_py_source("policy.py"), POLICY_MUTANTS[name]), "_mutant_policy")
    _patch_module(monkeypatch, policy, fake)
    assert _first_failing_pin(["policy", "q8"]), f"no pin catches: {name}"


@pytest.mark.parametrize("name", sorted(Q8_MUTANTS))
def test_q8_mistake_is_caught(name, monkeypatch):
    fake = _module_from(_edit(_py_source("q8.py"), Q8_MUTANTS[name]), "_mutant_q8")
    _patch_module(monkeypatch, q8, fake)
    assert _first_failing_pin(["q8"]), f"no pin catches: {name}"
