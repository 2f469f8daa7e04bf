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


def test_timeline_of_a_batched_stack_is_ordered():
    """The batched engine at batch 4: every product phase's first stage lands
    after its input chunk was issued and before its last unit, and every
    RMSNorm is published after its rows were formed."""
    r = timeline.run("8b", 3, batch=4)
    assert r["status"] == 0
    assert len(r["phases"]) == 19 and len(r["layers"]) == 2
    for p in r["phases"][1:]:
        if p["kind"] == "norm":
            assert p["landed/formed"][0] <= p["published"][1] + 1e-3
            continue
        assert p["input"][0] <= p["landed/formed"][0] <= p["last unit"][0] + 1e-3
    for lay in r["layers"]:
        assert 0 < lay["unit_loops_us"] < lay["us"] and lay["rest_us"] > 0
