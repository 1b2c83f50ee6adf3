"""Planted mistakes in the conv1d + SiLU oracle: each must fail at least one of its pins.

As for the recurrence oracle: one plausible mistake at a time (a reversed tap order, a dropped
term of the SiLU derivative, an off-by-one read position, an ignored halo, a wrong reduction)
is planted into a copy of oracle/conv1d.py, the copy is loaded as a module, and every pin of
tests/test_conv_pins.py runs against it; at least one must fail.  The real source is never
modified.
"""
import importlib.util
import os
import sys
import tempfile

import pytest

import test_conv_pins as pins
from oracle import conv1d

SRC = conv1d.__file__

MUTANTS = [
    ("taps reversed", "acc = acc + w[:, j] * xp[t + j]", "acc = acc + w[:, 3 - j] * xp[t + j]"),
    ("read one token late", "acc = acc + w[:, j] * xp[t + j]",
     "acc = acc + w[:, j] * xp[min(t + j + 1, len(xp) - 1)]"),
    ("SiLU derivative without its second term", "dz = dy * s * (1.0 + z * (1.0 - s))",
     "dz = dy * s"),
    ("SiLU derivative sign", "dz = dy * s * (1.0 + z * (1.0 - s))",
     "dz = dy * s * (1.0 - z * (1.0 - s))"),
    ("dx read position off by one", "src = t + j - (WIDTH - 1)", "src = t + j - WIDTH"),
    ("halo ignored", "        xp[:WIDTH - 1] = halo_n\n", "        pass\n"),
    ("dw from the wrong row", "dw[:, j] += dz[a + t] * xp[t + j]",
     "dw[:, j] += dz[a + t] * xp[max(t + j - 1, 0)]"),
    ("db from dy", "db=dz.sum(axis=0)", "db=dy.sum(axis=0)"),
    ("no bias", "acc = np.zeros(C) if bias is None else np.array(bias, dtype=np.float64)",
     "acc = np.zeros(C)"),
]

PINS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_")]


def _load(text, tag):
    d = tempfile.mkdtemp(prefix="conv_mutant_")
    path = os.path.join(d, f"conv1d_{tag}.py")
    with open(path, "w") as f:
        f.write(text)
    spec = importlib.util.spec_from_file_location(f"conv1d_{tag}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _run_pins(mod, monkeypatch):
    failed = []
    monkeypatch.setattr(pins, "conv1d", mod)
    for pin in PINS:
        params = [1, 2, 3, 6] if pin.__name__ == "test_halo_split_equals_whole_document" else [None]
        for p in params:
            try:
                pin(p) if p is not None else pin()
            except AssertionError:
                failed.append(pin.__name__)
                break
    return failed


def test_clean_copy_passes_every_pin(monkeypatch):
    with open(SRC) as f:
        mod = _load(f.read(), "clean")
    assert _run_pins(mod, monkeypatch) == []


@pytest.mark.parametrize("name,line,bad", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(name, line, bad, monkeypatch):
    with open(SRC) as f:
        text = f.read()
    assert text.count(line) >= 1, f"line of mutant {name!r} not found"
    mod = _load(text.replace(line, bad, 1), name.replace(" ", "_"))
    assert _run_pins(mod, monkeypatch), f"mutant {name!r} passed every pin"
