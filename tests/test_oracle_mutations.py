"""Planted mistakes in the oracle: each one must make at least one pin fail (CPU).

Each case copies the oracle package to a temporary directory, makes one plausible mistake in its C
source (a wrong rounding mode, an off-by-one in the exponent search, an inverted scale, a
transposed index, a wrong constant, ...), builds and imports the copy, and runs the pins of
test_oracle_pins.py against it, stopping at the first that fails.  The unchanged copy must pass
them all, so a caught mistake is the mistake and not the harness.
"""
import importlib.util
import inspect
import os
import shutil

import pytest

import test_oracle_pins as pins

ORACLE_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")

MUTATIONS = [
    ("rounding ties away from zero", "r = nearbyint(a / quantum) * quantum;", "r = round(a / quantum) * quantum;"),
    ("floor(log2(amax / Fmax)) + 1 instead of the ceiling",
     "while (amax > ldexp(fmax, k))\n        k++;\n    while (amax <= ldexp(fmax, k - 1))",
     "while (amax >= ldexp(fmax, k))\n        k++;\n    while (amax < ldexp(fmax, k - 1))"),
    ("E8M0 bias off by one", "e = k + 127;", "e = k + 126;"),
    ("scale applied inverted", "const double s = ldexp(1.0, 127 - e);\n                scale_row",
     "const double s = ldexp(1.0, e - 127);\n                scale_row"),
    ("all-zero block gets exponent 0", "if (amax == 0.0)\n        return 127;", "if (amax == 0.0)\n        return 0;"),
    ("lower clamp dropped", "if (e < 0)\n        e = 0;", "if (e < -1000)\n        e = 0;"),
    ("dbias accumulated in fp32", "double acc = 0.0;", "float acc = 0.0f;"),
    ("columnwise scale index transposed", "scale_col[r * N + j] = (uint8_t)e;",
     "scale_col[j * ((M + 31) / 32) + r] = (uint8_t)e;"),
    ("BF16 subnormal exponent off by one", "mag = ldexp((double)m, 1 - 127 - 7);", "mag = ldexp((double)m, 0 - 127 - 7);"),
    ("E5M2 maximum wrong", "448.0 : 57344.0", "448.0 : 49152.0"),
    ("FP8 subnormal mantissa step wrong", "m = (int)(r / ldexp(1.0, emin - mbits));",
     "m = (int)(r / ldexp(1.0, emin - mbits + 1));"),
    ("swizzle row split transposed", "(rr % 32) * 16 + (rr / 32) * 4 + cc", "(rr % 32) * 4 + (rr / 32) * 16 + cc"),
    ("GeLU cubic coefficient wrong", "(x + 0.044715 * x * x * x));", "(x + 0.04715 * x * x * x));"),
    ("dGeLU derivative of the cubic wrong", "dt = c * (1.0 + 3.0 * 0.044715 * x * x)", "dt = c * (1.0 + 0.044715 * x * x)"),
    ("dSiLU factor sign", "return s * (1.0 + x * oms);", "return s * (1.0 - x * oms);"),
    ("grouped columnwise scales at the flat call's row", "scale_col ? scale_col + s0 * N : 0",
     "scale_col ? scale_col + (r0 / MXO_BLOCK) * N : 0"),
    ("grouped scale rows counted with floor", "s0 += (rows + MXO_BLOCK - 1) / MXO_BLOCK;",
     "s0 += rows / MXO_BLOCK;"),
    ("gated halves swapped", "const double a = mxo_bf16_to_double(x[i * 2 * N + j]);",
     "const double a = mxo_bf16_to_double(x[i * 2 * N + N + j]);"),
    ("gated backward's da without the derivative", "(float)(gv * b * mxo_dactivation_f64(a, act));",
     "(float)(gv * b * mxo_activation_f64(a, act));"),
]


def pin_calls():
    """(name, function, kwargs) for every pin that takes the oracle, in file order."""
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_") or "oracle_mod" not in inspect.signature(fn).parameters:
            continue
        line = fn.__code__.co_firstlineno
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not marks:
            calls.append((line, name, fn, {}))
            continue
        names = [n.strip() for n in marks[0].args[0].split(",")]
        for v in marks[0].args[1]:
            calls.append((line, name, fn, dict(zip(names, v if len(names) > 1 else (v,)))))
    return [c[1:] for c in sorted(calls, key=lambda c: c[0])]


def load_copy(tmp_path, tag, mutate=None):
    dst = tmp_path / "oracle_copy"
    shutil.copytree(ORACLE_DIR, dst, ignore=shutil.ignore_patterns("_build", "__pycache__"))
    if mutate is not None:
        old, new = mutate
        src = (dst / "mxfp8_oracle.c").read_text()
        assert old in src, f"mutation site not found: {old!r}"
        (dst / "mxfp8_oracle.c").write_text(src.replace(old, new, 1))
    spec = importlib.util.spec_from_file_location(f"oracle_copy_{tag}", dst / "__init__.py",
                                                  submodule_search_locations=[str(dst)])
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    return mod


def first_failing_pin(mod):
    for name, fn, kw in pin_calls():
        try:
            fn(oracle_mod=mod, **kw)
        except Exception:  # an assertion, or the oracle rejecting its own output
            return f"{name}{kw or ''}"
    return None


def test_unchanged_copy_passes_every_pin(tmp_path):
    assert len(pin_calls()) >= 50
    assert first_failing_pin(load_copy(tmp_path, "clean")) is None


@pytest.mark.parametrize("what,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(tmp_path, what, old, new):
    caught = first_failing_pin(load_copy(tmp_path, abs(hash(what)), (old, new)))
    assert caught is not None, f"no pin caught: {what}"
