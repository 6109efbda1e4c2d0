import importlib.util
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _build_library():
    """Build libengram.so in-tree if it is missing or stale (a no-op otherwise).
    The build script is loaded by path: the package itself loads the library."""
    spec = importlib.util.spec_from_file_location(
        "_engram_build", os.path.join(ROOT, "hashed_gram_memory_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    _build_library()
