import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _ensure_library():
    lib = os.path.join(ROOT, "sparse_attention_fp4_02_b300", "libcsa2.so")
    if not os.path.exists(lib):
        from sparse_attention_fp4_02_b300.build import build
        build()


_ensure_library()


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
