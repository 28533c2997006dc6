import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GB300 (sm_103a); run with -m gpu")


def pytest_sessionstart(session):
    # Build the CUDA library and the C oracle if missing or stale (nvcc and
    # gcc are needed; nothing here runs GPU code).
    import importlib.util
    for rel in ("implicit_gemm_convolution_conv_gb300/build.py",
                "oracle/build.py"):
        spec = importlib.util.spec_from_file_location(
            "_b", os.path.join(ROOT, rel))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        mod.build()
