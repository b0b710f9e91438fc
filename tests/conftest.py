import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the CUDA library")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="session")
def golden_dir():
    return GOLDEN


@pytest.fixture(autouse=True)
def _index_checks_clear(request):
    """Under KIVI_DEBUG_BOUNDS=1 (the index-checking library), a GPU test must
    leave bit 4 of the device fault word clear: no kernel index left its bh
    slice.  Other tests and builds are not affected."""
    yield
    if os.environ.get("KIVI_DEBUG_BOUNDS") != "1" or request.node.get_closest_marker("gpu") is None:
        return
    import kv_cache_quantization_kivi_gb300 as K
    import torch
    torch.cuda.synchronize()
    fault = K.kivi_device_fault()
    assert not (fault & 16), f"index check failed in {request.node.nodeid} (fault word {fault:#x})"


def pytest_report_header(config):
    if os.environ.get("KIVI_DEBUG_BOUNDS") == "1":
        import kv_cache_quantization_kivi_gb300 as K
        return f"kivi library: {os.path.basename(K.library_path())} (index checks)"
    return None
