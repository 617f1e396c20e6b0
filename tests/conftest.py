import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the built CUDA library")
    config.addinivalue_line("markers", "slow: larger oracle runs (still CPU)")


@pytest.fixture(scope="session")
def full_table():
    import workloads
    return workloads.full_table()


@pytest.fixture(scope="session")
def full_enc(full_table):
    import oracle
    import workloads
    return oracle.Encoding(full_table, workloads.SPECIALS)


@pytest.fixture(scope="session")
def tiny_table():
    """256 byte tokens + 4,096 merges from the oracle's plain trainer on the
    seeded 2 MiB tiny corpus."""
    import oracle
    import workloads
    merges = oracle.train(workloads.tiny_corpus(), 4096)
    return [bytes([b]) for b in range(256)] + merges


@pytest.fixture(scope="session")
def tiny_enc(tiny_table):
    import oracle
    return oracle.Encoding(tiny_table)
