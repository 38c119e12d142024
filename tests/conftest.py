"""Shared pytest setup: the ``gpu`` marker, golden-file loading and seeds."""
from __future__ import annotations

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libqsa.so")


def load_golden(name: str) -> dict:
    """Parse a ``key: v v v`` fixture into {key: [float|int, ...]}."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, _, rest = line.partition(":")
            vals = []
            for tok in rest.split():
                vals.append(float(tok) if any(c in tok for c in ".e") else int(tok))
            out[key.strip()] = vals
    return out


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.lib()
    return oracle
