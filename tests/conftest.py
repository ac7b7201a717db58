import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) and the CUDA library")
    config.addinivalue_line("markers", "slow: large-size parity case")


def pytest_sessionstart(session):
    # Importing the binding needs the in-tree library; build it when stale
    # (nvcc cross-compiles without a GPU).
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_csa2_build", os.path.join(ROOT, "sparse_attention_fp4_mxfp4_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
