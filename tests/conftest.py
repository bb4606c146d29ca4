import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def _ensure_built():
    lib = os.path.join(ROOT, "rank_decomposed_gb300", "liblr.so")
    gen = os.path.join(ROOT, "synth", "libsynth.so")
    host = os.path.join(ROOT, "synth", "libsynth_host.so")
    if not (os.path.exists(lib) and os.path.exists(gen) and os.path.exists(host)):
        sys.path.insert(0, ROOT)
        import __graft_entry__
        __graft_entry__.build()


_ensure_built()
