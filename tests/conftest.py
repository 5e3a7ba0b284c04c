import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def cuda_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library, built in-tree if it is missing (or the prebuilt one
    that Q8ATTN_LIBRARY names, which is loaded as it is)."""
    if not os.environ.get("Q8ATTN_LIBRARY"):
        from chunked_prefill_attention_gb300 import _build
        _build.ensure_built()
    from chunked_prefill_attention_gb300 import q8attn
    return q8attn.load()
