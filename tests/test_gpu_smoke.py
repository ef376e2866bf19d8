"""The build entry's smoke run (one small call of each hot-path family on cuda:0, each checked
against the oracle inside smoke()), so that every GPU test run also covers it."""
import pytest

pytestmark = pytest.mark.gpu


def test_smoke_runs(lib, cuda):
    import __graft_entry__

    __graft_entry__.smoke()
    lib.ein_status()
