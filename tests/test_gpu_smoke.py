"""The package's smoke entry point (one small decode run on cuda:0, checked
against the oracle) runs as a GPU test too."""
import pytest


@pytest.mark.gpu
def test_smoke_entry_point():
    import __graft_entry__ as g
    g.smoke()
