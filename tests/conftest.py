import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libmmq.so")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle


@pytest.fixture(scope="session")
def oracle_ref(orc):
    """Oracle results for synthetic GEMMs (synth.Gemm), computed once per
    session on every host core: (qs, ds, Y) of the q8_1-quantised input and
    the method-form output, shared by the tests that check different kernels
    on the same configuration."""
    cache = {}

    def ref(g):
        key = (g.fmt, g.T, g.K, g.O, g.w_seed, g.x_seed, g.outliers)
        if key not in cache:
            qs, ds = orc.quantize_q8_1(g.x())
            cache[key] = (qs, ds, orc.gemm(g.fmt, g.weights(), qs, ds, g.O))
        return cache[key]

    return ref
