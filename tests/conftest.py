"""Shared test fixtures.

Markers:
  gpu  -- needs a CUDA device (a GB300); runs the CUDA library through its C ABI
          and compares it with the CPU oracle.  Everything else runs on CPU.
"""
from __future__ import annotations

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a library)")


def golden(name: str) -> dict:
    """Parse a `key = value` fixture under tests/golden (comments start with #)."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            if "," in v:
                out[k] = [float(t) for t in v.split(",")]
            else:
                try:
                    out[k] = int(v)
                except ValueError:
                    try:
                        out[k] = float(v)
                    except ValueError:
                        out[k] = v
    return out


@pytest.fixture(scope="session")
def oracle():
    import oracle as o
    o.build()
    o.lib()
    return o


@pytest.fixture(scope="session")
def native_lib():
    """The CUDA library, built here if needed (compiling needs no GPU)."""
    from fp8_scaled_quantization_gb300 import build as b
    b.build()
    import fp8_scaled_quantization_gb300 as f
    return f.library()


@pytest.fixture(scope="session")
def cuda():
    """A CUDA device; a GPU test without one fails rather than skips."""
    import torch
    assert torch.cuda.is_available(), "this test needs a CUDA GPU"
    from fp8_scaled_quantization_gb300 import build as b
    b.build()
    torch.cuda.init()
    return torch.device("cuda:0")
