"""Planted mistakes in a copy of the layout oracle must each fail at least one pin.

The copy is made from oracle/layout.py's source text with one plausible error
inserted; it runs on the CPU only.  The pins re-run here are those of
test_oracle_layout (hand-derived values and brute force).
"""
import os
import types

import pytest

import test_oracle_layout as pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "layout.py")

MUTATIONS = {
    "padding_entry_numbered": ("            if x == padding_value:\n                continue\n",
                               "            if x == padding_value:\n                x = 0\n"),
    "zero_length_skipped": ("            cu.append(cu[-1] + int(x))",
                            "            if x > 0:\n                cu.append(cu[-1] + int(x))"),
    "positions_from_one": ("                pos[b, p] = p - start", "                pos[b, p] = p - start + 1"),
    "gap_may_resume": ("            else:\n                ok = x == 0\n",
                       "            else:\n                ok = x == 0 or x == ps[b, prev] + 1\n"),
    "first_must_be_zero": ("            if prev < 0:\n                ok = x >= 0",
                           "            if prev < 0:\n                ok = x == 0"),
    "range_from_first_query": ("            lo = seg_start if lo is None else lo",
                               "            lo = t if lo is None else lo"),
    "range_end_inclusive": ("            hi = t + 1", "            hi = t"),
}


def _mutant(name):
    src = open(SRC).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found"
    src = src.replace(old, new).replace("from .blockdiag import", "from oracle.blockdiag import")
    mod = types.ModuleType(f"layout_mutant_{name}")
    exec(compile(src, SRC, "exec"), mod.__dict__)
    return mod


PIN_FUNCS = [getattr(pins, n) for n in dir(pins)
             if n.startswith("test_") and callable(getattr(pins, n))]


def _run_pins(mod, monkeypatch):
    monkeypatch.setattr(pins, "lay", mod)
    failures = 0
    for f in PIN_FUNCS:
        marks = getattr(f, "pytestmark", [])
        cases = [()]
        for m in marks:
            if m.name == "parametrize":
                cases = [c if isinstance(c, tuple) else (c,) for c in m.args[1]]
        for c in cases:
            try:
                f(*c)
            except Exception:  # noqa: BLE001 - a failed assertion or a crash counts as caught
                failures += 1
    return failures


def test_unmutated_copy_passes(monkeypatch):
    src = open(SRC).read().replace("from .blockdiag import", "from oracle.blockdiag import")
    clean = types.ModuleType("layout_clean")
    exec(compile(src, SRC, "exec"), clean.__dict__)
    assert _run_pins(clean, monkeypatch) == 0


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, monkeypatch):
    assert _run_pins(_mutant(name), monkeypatch) > 0, f"no pin catches {name}"
