"""The tracing build: one token of a 2-layer 8B-shaped stack with phase stamps."""
import pytest

from weight_streaming_q4_gb300 import timeline

pytestmark = pytest.mark.gpu


def test_timeline_of_a_stack_is_ordered():
    r = timeline.run("8b", 2)
    assert r["status"] == 0
    assert len(r["phases"]) == 9 and len(r["layers"]) == 2
    for p in r["phases"][:-1]:
        assert p["reached"][0] <= p["staged"][0] <= p["last unit"][0] <= p["last store"][1] + 1e-3
        assert p["last unit"][1] <= p["last store"][1] + 1e-3
    for lay in r["layers"]:
        assert 0 < lay["unit_loop_frac"] < 1 and lay["boundaries_us"] > 0
