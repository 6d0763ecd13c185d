"""The package entry's smoke() (one tiny pass of every hot-path call, checked against
the oracle and against the number of kernels it should launch) runs under pytest too."""
import os
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_smoke():
    sys.path.insert(0, ROOT)
    import __graft_entry__
    __graft_entry__.smoke()
