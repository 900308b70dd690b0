"""The round-trip check the build entry point runs on a GPU (needs a GB300)."""
import pytest

pytestmark = pytest.mark.gpu


def test_smoke_runs_and_matches_the_oracle():
    import __graft_entry__
    __graft_entry__.build()
    __graft_entry__.smoke()
