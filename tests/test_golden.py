"""The oracle and the seeded generator still reproduce the stored tiny-workload samples.

Fixture: tests/golden/tiny_oracle.txt, written by tests/golden/make_golden.py
(which calls only the oracle).  A change here means the oracle's arithmetic or
the input stream changed; such a change must name the passage that justifies it.
"""
import importlib.util
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_golden_samples():
    spec = importlib.util.spec_from_file_location("make_golden",
                                                  os.path.join(HERE, "golden", "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    stored = {}
    with open(os.path.join(HERE, "golden", "tiny_oracle.txt")) as f:
        for line in f:
            if line.startswith("#"):
                continue
            name, i, val = line.split()
            stored.setdefault(name, []).append((int(i), float(val)))
    got = dict(mg.cases())
    assert set(got) == set(stored)
    for name, items in stored.items():
        flat = got[name].reshape(-1)
        for i, val in items:
            assert abs(flat[i] - val) <= 1e-12 * max(1.0, abs(val)), (name, i)
