"""bench.py's clock record: only samples taken inside the timed window count,
the nearest one stands in for a window shorter than the sampling period, and
throttle reasons are the union over the window (host logic, no GPU)."""


def _sampler(samples, t0, t1):
    import bench
    c = bench.ClockSampler(0)
    c.source, c.smax = "nvml", 2070.0
    c.samples = samples
    c.t0, c.t1 = t0, t1
    return c


def test_only_samples_inside_the_window_count():
    s = [(0.0, 1200.0, {"sw_power_cap"}), (1.0, 2070.0, set()), (1.5, 2040.0, set()),
         (2.0, 1900.0, {"hw_slowdown"}), (9.0, 300.0, {"hw_thermal_slowdown"})]
    r = _sampler(s, 0.9, 2.1).summary()
    assert r["samples"] == 3
    assert r["sm_mhz"] == 2040.0
    assert r["reasons"] == ["hw_slowdown"]
    assert r["sm_max_mhz"] == 2070.0


def test_short_window_takes_the_nearest_sample():
    s = [(0.0, 1000.0, set()), (1.0, 2070.0, set()), (3.0, 1500.0, {"sw_power_cap"})]
    r = _sampler(s, 1.2, 1.25).summary()
    assert r["samples"] == 1 and r["sm_mhz"] == 2070.0 and r["reasons"] == []


def test_no_source_reports_nothing():
    import bench
    r = bench.ClockSampler(0).stop()
    assert r["sm_mhz"] is None and r["samples"] == 0


def test_roofline_terms_of_the_1b_workload():
    """The two roofline terms of the 1B-layer step: 26,112 algorithmic bytes per
    token (the packed row once, the output once) and the chunked scan's MMA work
    2 (Q (N + P) + 2 P N) H = 1.835 MFLOP per token at Q = 64."""
    import bench
    from selective_state_space_mamba3_gb300 import inputs as gen
    w = gen.SISO_1B
    assert bench.bytes_per_token_packed(w) == 26112
    assert bench.mma_flops_per_token_chunked(w) == 2 * (64 * (128 + 64) + 2 * 64 * 128) * 32
    assert bench.mma_flops_per_token_chunked(w) == 1835008
    peak, kind = bench.tf32_peak()
    assert 400.0 < peak < 1200.0 and "1.1/2.25" in kind
