import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: large workload; still bounded to a minute or two")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library; a GPU test fails (not skips) if it is missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    from tiled_attention_10_gb300 import binding
    return binding.load()


@pytest.fixture(scope="session")
def built_lib():
    """The C-ABI library for host-only tests (no kernel launch): built here if
    nvcc is available, else the one already built; skipped on a host that has
    neither (a CPU machine without the CUDA toolkit)."""
    import shutil
    from tiled_attention_10_gb300 import binding, build
    have_nvcc = shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")
    if have_nvcc:
        build.build()
    elif not os.path.exists(build.LIB):
        pytest.skip("no nvcc and no built library on this host")
    return binding.load()
