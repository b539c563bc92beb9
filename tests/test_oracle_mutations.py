"""Strength of the oracle's pins: plant one plausible mistake at a time in a
copy of the oracle (or of the seeded input generator), on the CPU, and check
that the CPU pins then fail.  Nothing here touches the CUDA library.

Each entry is (name, file, text to replace, replacement); the text must occur
exactly once, so a refactor that moves it makes the entry fail loudly rather
than pass silently.
"""
import shutil
import subprocess
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]

MUTATIONS = [
    ("relu-drops-bias", "oracle/ffn.py",
     "a[t] = np.maximum(0.0, _rowdots(L.W_up, S, x[t]) + b)",
     "a[t] = np.maximum(0.0, _rowdots(L.W_up, S, x[t]))"),
    ("threshold-ge", "oracle/ffn.py",
     "return np.asarray(l) > 0.0", "return np.asarray(l) >= 0.0"),
    ("logits-drop-c_p", "oracle/ffn.py",
     "l = l + _f64(L.c_p)[None, :]", "l = l"),
    ("reglu-gate-up-swapped", "oracle/ffn.py",
     "g = np.maximum(0.0, _rowdots(L.W_gate, S, x[t]) + b)\n            a[t] = g * _rowdots(L.W_up, S, x[t])",
     "g = np.maximum(0.0, _rowdots(L.W_up, S, x[t]) + b)\n            a[t] = g * _rowdots(L.W_gate, S, x[t])"),
    ("silu-negative-branch", "oracle/ffn.py",
     "np.where(z >= 0, z / (1.0 + e), z * e / (1.0 + e))",
     "np.where(z >= 0, z / (1.0 + e), z / (1.0 + e))"),
    ("down-sign", "oracle/ffn.py",
     "y += a[:, s + k:s + k + 1] * cols[k][None, :]",
     "y -= a[:, s + k:s + k + 1] * cols[k][None, :]"),
    ("hidden-without-relu", "oracle/ffn.py",
     "return np.maximum(0.0, x @ _f64(L.W_p1).T)", "return x @ _f64(L.W_p1).T"),
    ("intersection-not-union", "oracle/ffn.py",
     "np.flatnonzero(m.any(axis=0))", "np.flatnonzero(m.all(axis=0))"),
    ("ties-by-descending-index", "oracle/ffn.py",
     'return np.argsort(-c, kind="stable").astype(np.int64)',
     "return np.lexsort((-np.arange(c.size), -c)).astype(np.int64)"),
    ("permute-skips-W_down", "oracle/ffn.py",
     "        W_down=L.W_down[:, p],", "        W_down=L.W_down,"),
    ("logit-band-drops-h-error", "oracle/ffn.py",
     "tau = _gamma(L.rank + 1) * ((h + e) @ A2.T + cabs) + e @ A2.T",
     "tau = _gamma(L.rank + 1) * (h @ A2.T + cabs)"),
    ("fp16-pair-drops-subnormal-term", "oracle/ffn.py",
     "return 2.0 ** -22 * np.abs(_f64(v)) + 2.0 ** -25", "return 2.0 ** -22 * np.abs(_f64(v))"),
    ("preact-band-drops-bias", "oracle/ffn.py",
     "s = np.abs(x) @ np.abs(_f64(Wg)).T + np.abs(_f64(L.b))[None, :]",
     "s = np.abs(x) @ np.abs(_f64(Wg)).T"),
    ("profile-band-zero", "oracle/ffn.py",
     "band += (np.abs(z) <= tau).sum(axis=0)", "band += 0"),
    ("e4m3-round-half-up", "oracle/quant.py",
     "val = np.round(a / quantum) * quantum", "val = np.floor(a / quantum + 0.5) * quantum"),
    ("e4m3-exponent-bias", "oracle/quant.py",
     "(1.0 + mf / 8.0) * np.ldexp(1.0, ef - 7)", "(1.0 + mf / 8.0) * np.ldexp(1.0, ef - 8)"),
    ("generator-sigma-from-up", "workload/gen.py",
     "gated = W_gate if W_gate is not None else W_up", "gated = W_up"),
    ("generator-arc-cosine", "workload/gen.py",
     "(torch.sin(t) + (math.pi - t) * cos_t)", "(torch.sin(t) + (math.pi + t) * cos_t)"),
]


@pytest.mark.parametrize("name,path,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_a_planted_mistake(tmp_path, name, path, old, new):
    for d in ("oracle", "workload", "tests"):
        shutil.copytree(ROOT / d, tmp_path / d, ignore=shutil.ignore_patterns("__pycache__"))
    f = tmp_path / path
    src = f.read_text()
    assert src.count(old) == 1, f"{name}: the text to replace must occur exactly once in {path}"
    f.write_text(src.replace(old, new))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py", "tests/test_oracle_fp8.py"],
                       cwd=tmp_path, capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"the pins did not catch '{name}':\n{r.stdout[-3000:]}\n{r.stderr[-2000:]}"
