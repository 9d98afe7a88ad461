"""Mutation check of the oracle's pins: each entry plants one plausible mistake
in a scratch copy of oracle/cconv_oracle.c (a flipped tap, a dropped term, an
off-by-one index, a wrong rounding, an ignored argument), builds it, points the
oracle module at the mutant and runs the pin tests (tests/test_oracle_pins.py,
tests/test_oracle_fused_pins.py, tests/test_oracle_state_dtype.py) over all
their parameters. Every mutant must fail at least one of them. The stored
fixtures are left out: they were written by the oracle and would catch any
change for that reason alone. CPU only; every mutant keeps its memory accesses
in bounds.
"""
import ctypes
import itertools
import os
import subprocess
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle
from tests import test_oracle_fused_pins, test_oracle_pins, test_oracle_state_dtype

SRC = os.path.join(os.path.dirname(oracle.__file__), "cconv_oracle.c")

# (name, text in the oracle, replacement, replace every occurrence)
MUTANTS = [
    ("tap orientation", "xt[S + j - (W - 1 - k) * D]", "xt[S + j - k * D]", False),
    ("dropped bias", "float acc = bias ? orc_get(bias, c, dtype) : 0.0f;", "float acc = 0.0f;",
     False),
    ("state columns reversed",
     "orc_state_put(pool, slot * s_slot + c * s_chan + i * s_col, sdtype, dtype, xt[L + i]);",
     "orc_state_put(pool, slot * s_slot + c * s_chan + i * s_col, sdtype, dtype,"
     " xt[L + S - 1 - i]);", False),
    ("decode shift", "sdtype, dtype, xt[1 + i]);", "sdtype, dtype, xt[i]);", False),
    ("spec prior offset", "xt[i] = Bc[off + i];", "xt[i] = Bc[i];", False),
    ("spec kept columns", "Bc[off + 1 + i]", "Bc[off + i]", False),
    ("has_init ignored", "const int h = (has_init ? has_init[s] != 0 : 1) && slot >= 0;",
     "const int h = slot >= 0;", True),
    ("SiLU sign", "expf(-v)", "expf(v)", False),
    ("truncating bf16", "u += 0x7fffu + ((u >> 16) & 1u);", "u += 0u;", False),
    ("truncating state conversion", "  return orc_f32_to_bf16(v);\n}",
     "  uint32_t t;\n  memcpy(&t, &v, 4);\n  return (uint16_t)(t >> 16);\n}", False),
    ("CCA depthwise tap", "xc[n + p - (T0 - 1 - k)]", "xc[n + p - k]", False),
    ("CCA grouped tap", "(o * gs + i) * T1 + k", "(o * gs + i) * T1 + (T1 - 1 - k)", False),
    ("CCA unrounded intermediate", "r = orc_bf16_to_f32(orc_f32_to_bf16(acc));", "r = acc;",
     False),
    ("delayed shift", "(start + j - 1) * delayed_rs", "(start + j) * delayed_rs", False),
    ("delayed state from the first token", "(start + L - 1) * delayed_rs", "(start) * delayed_rs",
     False),
    ("outer residual sign", "v = v + orc_get(outer", "v = v - orc_get(outer", False),
    ("token_indices ignored", "prow[i] = tidx ? tidx[start + i] : start + i;",
     "prow[i] = start + i;", False),
    ("checkpoint window one late", "cu_seqlens[s] + off - S + i;",
     "cu_seqlens[s] + off - S + i + 1;", False),
    ("key residual mean", "sum / (float)kvg", "sum / (float)(kvg + 1)", False),
]


def _cases():
    for mod in (test_oracle_pins, test_oracle_fused_pins, test_oracle_state_dtype):
        for name in sorted(dir(mod)):
            fn = getattr(mod, name)
            if not name.startswith("test_") or not callable(fn):
                continue
            grids = []
            for m in getattr(fn, "pytestmark", []):
                if m.name != "parametrize":
                    continue
                names = m.args[0]
                if isinstance(names, str):
                    names = [n.strip() for n in names.split(",")]
                names = list(names)
                rows = [v if len(names) > 1 else (v,) for v in m.args[1]]
                grids.append([dict(zip(names, r)) for r in rows])
            for combo in itertools.product(*grids):
                kw = {}
                for d in combo:
                    kw.update(d)
                yield f"{mod.__name__.split('.')[-1]}::{name}", fn, kw


def _build(tmp, k, text):
    c = os.path.join(tmp, f"m{k}.c")
    so = os.path.join(tmp, f"m{k}.so")
    with open(c, "w") as f:
        f.write(text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-fno-fast-math", c, "-o", so, "-lm"], check=True)
    return so


def _killed_by(lib):
    saved = oracle._lib
    oracle._lib = lib
    try:
        for where, fn, kw in _cases():
            try:
                fn(**kw)
            except pytest.skip.Exception:
                continue
            except Exception:            # a failed pin, or the oracle rejecting its own state
                return where
        return None
    finally:
        oracle._lib = saved


def test_every_planted_mistake_fails_a_pin():
    src = open(SRC).read()
    texts = []
    for name, a, b, every in MUTANTS:
        assert a in src, f"{name}: text not found in the oracle"
        texts.append(src.replace(a, b) if every else src.replace(a, b, 1))
    with tempfile.TemporaryDirectory() as tmp:
        with ThreadPoolExecutor(8) as ex:
            paths = list(ex.map(lambda kt: _build(tmp, *kt), enumerate(texts + [src])))
        # control: the unchanged oracle, built the same way, passes every pin
        where = _killed_by(oracle._configure(ctypes.CDLL(paths.pop())))
        assert where is None, f"the unchanged oracle fails {where}"
        survivors = []
        for (name, *_), path in zip(MUTANTS, paths):
            if _killed_by(oracle._configure(ctypes.CDLL(path))) is None:
                survivors.append(name)
    assert not survivors, f"mutants no pin catches: {survivors}"
