import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def read_golden(name):
    """Rows of whitespace-separated fields of a fixture, comments dropped."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# The oracle's two implementations: the C++ FP64 one (oracle/moe_oracle.cpp,
# the reference every GPU parity test uses) and the numpy one it is
# cross-checked against.  The pins run against both.
ORACLES = ("native", "numpy")


def oracle_ns(name):
    import importlib
    return importlib.import_module("oracle.native" if name == "native" else "oracle")


def swap_oracle(module_name, request, monkeypatch, names):
    """Rebind the test module's oracle modules (``formats``, ``quant``,
    ``layer``) and ``SlotTable`` to the implementation the fixture
    parameter names."""
    mod = sys.modules[module_name]
    ns = oracle_ns(request.param)
    for n in names:
        monkeypatch.setattr(mod, n, ns.lru.SlotTable if n == "SlotTable" else getattr(ns, n))
    return request.param
