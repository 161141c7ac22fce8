"""The build-and-smoke entry point's smoke() (one small forward and decode step
per variant against the fp64 oracle) runs clean on the GPU."""

import pytest

pytestmark = pytest.mark.gpu


def test_graft_entry_smoke():
    import __graft_entry__

    __graft_entry__.smoke()
