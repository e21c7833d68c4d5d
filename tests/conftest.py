"""Shared pytest set-up: the ``gpu`` marker and building the two native libraries.

``-m "not gpu"`` runs everything that needs no GPU: the oracle against its
pins, host-side validation of the C ABI and the library's exported symbols.
``-m gpu`` runs the parity tests proper (CUDA path vs the oracle).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def wq():
    from weight_only_bit_pack_b300 import build as wqbuild
    wqbuild.build()
    import weight_only_bit_pack_b300 as pkg
    return pkg
