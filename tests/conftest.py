import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _ensure_library():
    lib = os.path.join(ROOT, "sparse_attention_fp4_02_b300", "libcsa2.so")
    if not os.path.exists(lib):
        import importlib.util     # load the build script by path: the package imports the library
        spec = importlib.util.spec_from_file_location("_csa2_build", os.path.join(os.path.dirname(lib), "build.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        mod.build()


_ensure_library()


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
