"""Sizing of the benchmark's CPU baseline sample, on CPU with a stand-in oracle forward and a
stand-in clock.  The sample of tokens grows, at least doubling each time, until one run takes
three quarters of the budget, covers every token, or the number of sizes tried reaches its
limit; a run is repeated only while the float64 weight cache still keeps the conversions it
makes (conversions past the cache's cap recur on every run)."""
import sys
import types

import pytest

from tests.conftest import ROOT


def _bench():
    sys.path.insert(0, ROOT)
    import bench
    return bench


@pytest.fixture
def stand_in(monkeypatch):
    """Returns (bench, calls, set_forward): set_forward(fn) installs fn(S, n_call) -> seconds
    as the oracle's layer forward; the stand-in clock advances by what fn returns."""
    bench = _bench()
    import oracle
    now = [0.0]
    monkeypatch.setattr(bench, "time", types.SimpleNamespace(perf_counter=lambda: now[0]))
    monkeypatch.setattr(bench.ExpertsF64, "conversions", 0)
    monkeypatch.setattr(bench.ExpertsF64, "held", 0)
    calls = []

    def set_forward(fn):
        def forward(spec, d):
            assert len(d["x"]) == spec.T   # the first spec.T tokens
            now[0] += fn(spec.T, len(calls))
            calls.append(spec.T)
        monkeypatch.setattr(oracle, "moe_forward", forward)

    return bench, calls, set_forward


def _spec(T):
    from workloads import CONFIGS
    return CONFIGS["tiny"].replace(T=T)


def test_sample_grows_until_three_quarters_of_the_budget(stand_in):
    bench, calls, set_forward = stand_in
    set_forward(lambda S, n: 0.01 * S)                # 10 ms per token
    S, t = bench.time_oracle(_spec(8192), {"x": list(range(8192))}, budget_s=12.0)
    assert calls[0] == 64 and calls[-1] == S
    assert t >= 0.75 * 12.0 and t == pytest.approx(0.01 * S)
    assert all(b >= 2 * a for a, b in zip(calls, calls[1:]))
    # the step before the last stayed below the stopping point
    assert 0.01 * calls[-2] < 0.75 * 12.0


def test_sample_stops_at_the_size_limit_when_time_grows_slowly(stand_in):
    bench, calls, set_forward = stand_in
    set_forward(lambda S, n: 4.0 + 1e-4 * S)          # dominated by a fixed cost
    S, t = bench.time_oracle(_spec(1 << 20), {"x": list(range(1 << 20))}, budget_s=12.0,
                             max_sizes=5)
    assert len(calls) == 5 and S == calls[-1]
    assert t < 0.75 * 12.0
    assert all(b >= 2 * a for a, b in zip(calls, calls[1:]))


def test_sample_stops_at_every_token(stand_in):
    bench, calls, set_forward = stand_in
    set_forward(lambda S, n: 1e-3 * S)
    S, t = bench.time_oracle(_spec(256), {"x": list(range(256))}, budget_s=12.0)
    assert S == 256 and calls == [64, 256]


@pytest.mark.parametrize("kept_by_cache, expect_runs", [
    ([], 1),                   # no conversions: one run
    ([True, False], 2),        # the first run filled the cache, the second converted past it
    ([False], 1),              # the cache is already full: a repeat would convert again
    ([True, True, True], 3),   # still filling after two repeats: at most three runs
])
def test_runs_repeat_only_while_the_cache_keeps_conversions(stand_in, kept_by_cache, expect_runs):
    bench, calls, set_forward = stand_in

    def forward(S, n):
        if n < len(kept_by_cache):
            bench.ExpertsF64.conversions += 3
            if kept_by_cache[n]:
                bench.ExpertsF64.held += 1 << 20
        return 1.0 + n          # each run a different length: the last one is returned
    set_forward(forward)
    t = bench.oracle_seconds(_spec(64), {"x": list(range(64))}, 64)
    assert len(calls) == expect_runs
    assert t == pytest.approx(float(expect_runs))
    last_converted = 3 if expect_runs <= len(kept_by_cache) else 0
    assert bench.oracle_seconds.converted == last_converted
