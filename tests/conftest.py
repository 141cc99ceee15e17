import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(scope="session")
def oracle_pool():
    """The oracle on all host cores (worker processes started with spawn, so
    it is safe to create after the GPU is in use)."""
    from oracle_par import OraclePool
    pool = OraclePool()
    yield pool
    pool.close()


# every string of up to five code points over this alphabet goes through the
# pre-tokenizer in the brute-force tests: letters (ASCII lower and upper case,
# contraction letters in both cases, a 3-byte caseless one), the apostrophe,
# numbers (ASCII and not), the whitespace the patterns treat apart (space,
# tab, LF, CR, a 2-byte one) and '/' (an ASCII symbol that the o200k-style
# pattern also takes into a symbol run's tail)
BRUTE_ALPHABET = ["a", "s", "S", "l", "'", "1", "\u00b2", " ", "\t", "\n", "\r", "/", "\u4e2d", "\u00a0"]
