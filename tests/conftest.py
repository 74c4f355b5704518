import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# The mutation check (test_oracle_mutations.py) runs the pins against a copy
# of the oracle package with one planted mistake: this variable names that
# copy's directory, which is then imported as `oracle` in place of ROOT/oracle.
_UNDER_TEST = os.environ.get("PHOTON_ORACLE_UNDER_TEST")
if _UNDER_TEST:
    import importlib.util
    _spec = importlib.util.spec_from_file_location(
        "oracle", os.path.join(_UNDER_TEST, "__init__.py"),
        submodule_search_locations=[_UNDER_TEST])
    _mod = importlib.util.module_from_spec(_spec)
    sys.modules["oracle"] = _mod
    _spec.loader.exec_module(_mod)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA library)")
    config.addinivalue_line("markers", "slow: larger CPU cases")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(params=[1, 2], ids=["cuda_cores", "tensor_cores"])
def consumer(request):
    """Runs a decode test on each attention consumer of the library: 1 = the
    CUDA-core one, 2 = the tensor-core one (16-bit storage; f32 stays on CUDA
    cores).  Restores the default selection afterwards."""
    import paged_kv_attention_photon_gb300 as P
    P.photon_debug_set_decode_consumer(request.param)
    yield request.param
    P.photon_debug_set_decode_consumer(0)
