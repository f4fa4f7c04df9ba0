"""Host-side schedule logic (CPU): which steps are dense, anchor or reuse, and the
anchor overhead as equivalent extra density on hand-made step times."""
import pytest

from sparse_attention_diffusion_gb300 import schedule


def test_step_kinds_follow_warmup_and_period():
    s = schedule.Schedule(steps=50, warmup=5, period=10)
    kinds = [s.kind(t) for t in range(s.steps)]
    assert kinds[:5] == ["dense"] * 5
    anchors = [t for t, k in enumerate(kinds) if k == "anchor"]
    assert anchors == [5, 15, 25, 35, 45]
    assert kinds.count("reuse") == 50 - 5 - 5


def test_anchor_overhead_on_hand_made_times():
    # 2 dense warm-up steps of 100 ms, then per period of 4: one anchor (250 ms) and three reuse steps (20 ms)
    R = schedule.StepRecord
    recs = [R("dense", 100.0), R("dense", 100.0)] + [R("anchor", 250.0), R("reuse", 20.0), R("reuse", 20.0),
                                                     R("reuse", 20.0)] * 2
    rho_eq, extra = schedule.anchor_overhead(recs, 100.0, 0.2, 2)
    # post-warm-up time 2 * (250 + 60) = 620 ms against 8 dense steps = 800 ms
    assert rho_eq == pytest.approx(620.0 / 800.0)
    assert extra == pytest.approx(620.0 / 800.0 - 0.2)
    # all-reuse trajectory at exactly the density's cost has no overhead
    rho_eq, extra = schedule.anchor_overhead([R("reuse", 20.0)] * 10, 100.0, 0.2, 0)
    assert rho_eq == pytest.approx(0.2) and extra == pytest.approx(0.0)
