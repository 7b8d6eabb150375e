"""The benchmark's host-side pieces on CPU: the reference arm's JSON line and
the clock sampler's window (with a stand-in for nvidia-smi)."""
import json
import os
import stat
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_complete_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3",
                          "--warmup", "3"], cwd=ROOT, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["host"]["nproc"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    # value is the metric's all_reduce rows; the whole step is reported beside it
    assert d["config"]["value_rows"] == ["all_reduce_sum", "all_reduce_mean", "all_reduce_max"]
    assert d["step_algbw_gbs"] > 0


def test_openmp_baseline_computes_the_oracles_all_reduce():
    """The second CPU baseline (all host cores) reduces exactly as the
    single-threaded oracle does, so the two timings measure the same work."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import oracle
    import oracle.omp as omp
    from gradient_sync_rcc_gb300 import synth
    oracle.build.build()
    xs = synth.rank_buffers("grad", 5, 100003, 4, 4)
    xs[2][17] = np.nan
    outs = [np.empty(100003, np.float32) for _ in range(5)]
    for op in ("sum", "mean", "max", "min"):
        omp.all_reduce(xs, outs, op, 4)
        want = oracle.reduce_f32(xs, op)
        for o in outs:
            assert o.tobytes() == want.tobytes(), op


def test_clock_sampler_keeps_only_the_timed_window(tmp_path, monkeypatch):
    fake = tmp_path / "nvidia-smi"
    fake.write_text("#!/bin/sh\n"
                    "i=0\n"
                    "while true; do\n"
                    "  echo \"$((1000+i)), 2070, 0x0000000000000000\"\n"
                    "  i=$((i+1)); sleep 0.05\n"
                    "done\n")
    fake.chmod(fake.stat().st_mode | stat.S_IEXEC)
    monkeypatch.setenv("PATH", str(tmp_path) + os.pathsep + os.environ["PATH"])
    sys.path.insert(0, ROOT)
    import bench
    s = bench.ClockSampler(0)
    s.start()
    t0 = time.time()
    while s.lines() < 3 and time.time() - t0 < 10:
        time.sleep(0.02)
    first = s.lines()
    assert first >= 3
    time.sleep(0.3)
    c = s.stop(first)
    assert c["window"] == "timed region" and c["samples"] >= 2
    assert c["sm_mhz"] >= 1000 + first        # none of the pre-roll samples counted
    assert c["sm_max_mhz"] == 2070 and c["reasons"] == []


def test_clock_sampler_decodes_the_reasons_bitmask(tmp_path):
    """NVML's clocks-event reason bits: 0x4 software power cap, 0x8 hardware
    slowdown, 0x20 software thermal, 0x40 hardware thermal, 0x80 power brake;
    the idle bit (0x1) is not a throttle reason."""
    sys.path.insert(0, ROOT)
    import bench
    s = bench.ClockSampler(0)
    s.f = open(tmp_path / "samples.csv", "w+")
    s.f.write("2070, 2070, 0x0000000000000001\n"
              "2055, 2070, 0x0000000000000004\n"
              "1800, 2070, 0x00000000000000E8\n")
    s.f.flush()

    class Done:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            pass

    s.proc = Done()
    c = s.stop(0)
    assert c["samples"] == 3 and c["sm_mhz"] == 2055.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["hw_power_brake_slowdown", "hw_slowdown", "hw_thermal_slowdown",
                            "sw_power_cap", "sw_thermal_slowdown"]
