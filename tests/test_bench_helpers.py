"""The host-side arithmetic behind bench.py's line (CPU only): which kernel a plan names,
the committed ncu traffic lookup, the cache replicas that keep the KV reads out of L2, and
the clock record taken during the timed region."""
import json
import os

import bench
import workloads as W


def test_kernel_name_follows_the_plan():
    # the key-major decode tile: four consumer warps (2), eight (32), two kv-heads a CTA (64)
    for k in (2, 32, 64):
        assert bench.kernel_name({"kernel": k}, 128) == "ua_decode_kernel"
    assert bench.kernel_name({"kernel": 1}, 256) == "ua_attn_tile_kernel"
    assert bench.kernel_name({"kernel": 4}, 64) == "ua_attn_tile_kernel"
    for k in (8, 16):
        assert bench.kernel_name({"kernel": k}, 64) == "ua_prefill_tm_kernel"
        assert bench.kernel_name({"kernel": k}, 128) == "ua_prefill_tm_kernel"
        assert bench.kernel_name({"kernel": k}, 256) == "ua_prefill_wide_kernel"


def test_recorded_traffic_only_for_unchanged_kernel_sources():
    with open(os.path.join(bench.ROOT, "profiles", "dram_traffic.json")) as f:
        recs = json.load(f)
    for key, rec in recs.items():
        if key.startswith("_"):
            continue
        kernel, workload = key.split("/")
        assert kernel in bench.KERNEL_SOURCES
        assert os.path.exists(os.path.join(bench.ROOT, rec["capture"])), rec["capture"]
        got = bench.recorded_traffic(kernel, workload)
        if rec["source_hash"] == bench.kernel_source_hash(kernel):
            assert got == float(rec["dram_bytes_per_launch"])
        else:
            assert got is None
    assert bench.recorded_traffic("ua_decode_kernel", "no_such_workload") is None


def test_cache_replicas_keep_every_step_out_of_l2():
    for spec in W.WORKLOADS.values():
        r = bench.n_replicas(spec)
        assert 1 <= r <= 64
        if spec.name in ("swdecode_bf16", "swdecode_fp8", "swdecode_fp8_tok"):
            keys = sum(kv - max(0, kv - a - (spec.window - 1)) for a, kv in spec.seqs)
            esz = 1 if "fp8" in spec.name else 2
            per_step = keys * spec.num_kv_heads * spec.head_dim * esz * 2
            assert r * per_step >= 3 * bench.L2_BYTES


def _row(ts, sm, sm_max=2070.0, hw="Not Active", swpc="Not Active"):
    # timestamp, index, clocks.sm, clocks.max.sm, power, active, hw, hwt, swt, swpc
    return (ts, f"2026/01/01 00:00:00.000, 0, {sm}, {sm_max}, 900.0, 0x0, {hw}, Not Active, "
                f"Not Active, {swpc}")


def test_clock_record_uses_the_timed_window_and_names_throttle_reasons():
    s = bench.ClockSampler(0)
    s.proc = None
    s.marks = {"timed_start": 10.0, "timed_end": 11.0}
    s.lines = [_row(9.0, 1000.0), _row(10.2, 2070.0), _row(10.5, 2060.0, swpc="Active"),
               _row(10.9, 2050.0), _row(12.0, 900.0, hw="Active")]

    class _P:  # a finished sampler process
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    s.proc = _P()
    rec = s.stop()
    assert rec["window"] == "timed" and rec["samples"] == 3
    assert rec["sm_mhz"] == 2060.0 and rec["sm_max_mhz"] == 2070.0
    # the hw_slowdown sample lies outside the timed window
    assert rec["reasons"] == ["sw_power_cap"]


def test_peaks_are_positive_and_name_their_source():
    hbm, tc, tc_sustained, src = bench.peaks()
    assert hbm > 0 and tc > 0 and tc_sustained > 0
    assert src in ("measured", "fallback")


def test_cpu_sample_heads_are_whole_rounds_of_threads():
    import bench
    assert bench.sample_heads(32, 16, 19) == 16
    assert bench.sample_heads(32, 16, 40) == 32
    assert bench.sample_heads(32, 16, 1) == 16      # at least one round
    assert bench.sample_heads(8, 16, 3) == 8        # fewer heads than threads: every head
    assert bench.sample_heads(24, 16, 100) == 16    # never past the heads there are
    for heads, threads, budget in ((32, 16, 19), (24, 8, 9), (16, 4, 13)):
        assert bench.sample_heads(heads, threads, budget) % threads == 0


def test_both_arms_share_one_config_dict():
    import bench
    import workloads as W
    cfg = bench.workload_config(W.SWDECODE_BF16, 1)
    assert cfg["workload"] == "swdecode_bf16" and "l2" in cfg
    assert cfg == bench.workload_config(W.SWDECODE_BF16, 1)
