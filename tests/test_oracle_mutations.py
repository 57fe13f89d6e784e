"""Planted mistakes in the oracle: each case compiles a copy of the fp64 oracle
(``oracle/gdn_oracle.c``) with one plausible error -- a dropped term, a wrong
sign, a wrong operand, index or tap order -- and checks that the oracle's pins
(``tests/test_oracle_pins.py``, every parametrisation) reject it: at least one
pin must fail against the mutant. The mutants are built with gcc in a
temporary directory; the oracle itself is untouched.

Not planted: dropping the q scale. The output o_t = S_t q_t is linear in q and
the gated RMSNorm divides by the RMS of o, so the scale reaches the layer's
outputs only through the RMSNorm's epsilon; no output-level check can see it.
"""
import importlib.util
import inspect
import itertools
from pathlib import Path

import pytest

from tests import test_oracle_pins as pins

ROOT = Path(__file__).resolve().parent.parent
SRC = ROOT / "oracle" / "gdn_oracle.c"
WRAPPER = ROOT / "oracle" / "oracle.py"

# name -> (exact text in the oracle, replacement)
MUTATIONS = {
    "prediction error with the wrong sign": ("u[c] = vt[c] - acc;", "u[c] = vt[c] + acc;"),
    "write without beta": ("St[(size_t)r * dv + c] += beta[t] * kt[r] * u[c];",
                           "St[(size_t)r * dv + c] += kt[r] * u[c];"),
    "no decay": ("double decay = exp(g[t]);", "double decay = 1.0;"),
    "decay with the wrong sign": ("double decay = exp(g[t]);", "double decay = exp(-g[t]);"),
    "output reads k instead of q": ("acc += St[(size_t)r * dv + c] * qt[r];",
                                    "acc += St[(size_t)r * dv + c] * kt[r];"),
    "gate without exp(A_log)": ("double gt = -exp(A_log[h]) * softplus(", "double gt = -A_log[h] * softplus("),
    "beta with the wrong sign": ("double bt = sigmoid(b[t * nv + h]);", "double bt = sigmoid(-b[t * nv + h]);"),
    "mask not applied to g": ("g[t * nv + h] = gt * m;", "g[t * nv + h] = gt;"),
    "conv taps reversed": ("acc += w[(size_t)c * K + j] * xin", "acc += w[(size_t)c * K + (K - 1 - j)] * xin"),
    "conv tail taken at the padded end": ("memcpy(conv_state, xin + (size_t)Lr * C,",
                                          "memcpy(conv_state, xin + (size_t)T * C,"),
    "L2 norm without the square root": ("double r = 1.0 / sqrt(ss + eps);", "double r = 1.0 / (ss + eps);"),
    "RMSNorm over the sum instead of the mean": ("double r = 1.0 / sqrt(ss / n + eps);",
                                                 "double r = 1.0 / sqrt(ss + eps);"),
    "RMSNorm gate sigmoid(z) instead of silu(z)": ("out[i] = o[i] * r * w[i] * silu(z[i]);",
                                                   "out[i] = o[i] * r * w[i] * sigmoid(z[i]);"),
    "GQA heads interleaved instead of grouped": ("int kh = h / (nv / nk);", "int kh = h % nk;"),
}


def _mutant(tmp: Path, tag: str, old: str, new: str):
    """A separate instance of the oracle wrapper bound to a mutated, freshly
    compiled copy of the C oracle."""
    src = SRC.read_text()
    assert src.count(old) == 1, f"mutation site not unique: {old!r}"
    (tmp / "gdn_oracle.c").write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"oracle_mutant_{tag}", WRAPPER)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC = tmp / "gdn_oracle.c"
    mod._SO = tmp / "_build" / "libgdn_oracle.so"
    mod._lib = None
    mod.build(force=True)
    return mod


def _pin_calls():
    """(name, function, kwargs) for every pin and parametrisation that needs no
    fixture other than the oracle module."""
    calls = []
    for name, fn in sorted(vars(pins).items()):
        if not (name.startswith("test_") and callable(fn)):
            continue
        grids = []
        for mark in getattr(fn, "pytestmark", []):
            if mark.name == "parametrize":
                names = [n.strip() for n in mark.args[0].split(",")] if isinstance(mark.args[0], str) \
                    else list(mark.args[0])
                values = [v if len(names) > 1 else (v,) for v in mark.args[1]]
                grids.append([dict(zip(names, v)) for v in values])
        params = set(inspect.signature(fn).parameters) - {"oracle_mod"}
        for combo in itertools.product(*grids) if grids else [()]:
            kw = {}
            for d in combo:
                kw.update(d)
            if set(kw) == params:
                calls.append((name, fn, kw))
    return calls


PIN_CALLS = _pin_calls()


def test_pins_are_collected():
    assert len({n for n, _, _ in PIN_CALLS}) >= 15


def test_harness_control_unmutated_copy_passes_every_pin(tmp_path):
    """The same harness on an unchanged copy: no pin may fail, so a caught
    mutant is caught by its mistake, not by the harness."""
    mod = _mutant(tmp_path, "control", "u[c] = vt[c] - acc;", "u[c] = vt[c] - acc;")
    for pin, fn, kw in PIN_CALLS:
        fn(mod, **kw)


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_pins_reject_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    mod = _mutant(tmp_path, str(abs(hash(name))), old, new)
    caught = []
    for pin, fn, kw in PIN_CALLS:
        try:
            fn(mod, **kw)
        except Exception:  # an assertion, or a check the mutant makes impossible
            caught.append(pin)
    assert caught, f"no pin of the oracle fails when it has: {name}"
