import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    # the binding loads libsv.so at import; build it (incrementally) before collection
    import importlib.util
    spec = importlib.util.spec_from_file_location("_sv_build", os.path.join(ROOT, "verify_step_02_b300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload; takes minutes")
