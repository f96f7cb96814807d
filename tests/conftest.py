import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running case")


@pytest.fixture(scope="session")
def built_lib():
    """Build (or reuse) libeagle3.so for sm_103a and load it."""
    from eagle_speculative_decode_gb300 import binding, build
    build.build()
    return binding.load()


@pytest.fixture(scope="session")
def full_drafter(built_lib):
    """Seeded weights of the full drafter geometry (n_embd 4096, draft vocab 32000 ->
    target vocab 248320) and the oracle's float64 view of them, built once per session
    (the widening alone takes tens of seconds)."""
    from eagle_speculative_decode_gb300 import synth
    from oracle import eagle3_oracle as O
    wts = synth.make_weights(synth.FULL, seed=0)
    return wts, O.Drafter(synth.FULL, wts.bits, wts.d2t)
