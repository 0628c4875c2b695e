import pytest


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    """GPU tests are skipped, with a reason, on a machine without a CUDA
    device; on a GPU machine they build and load the CUDA library and fail
    loudly if it is missing."""
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except ImportError:
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device on this machine")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def cuda_lib():
    from fully_sharded_state_gb300 import build, capi
    build.build()
    return capi.load()
