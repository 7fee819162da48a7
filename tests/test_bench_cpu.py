"""The benchmark's reference arm on CPU: the JSON line the contract asks for.

`bench.py --impl reference` times the CPU oracle (the reference arm of this
path), so it runs here without a GPU; the test checks the keys and units of its
one line on the tiny workload.
"""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, cwd=ROOT, env=env, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == "drafted tokens/s"
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    assert d["config"]["workload"] == "tiny"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


class _FakeSmi:
    """Stands in for the nvidia-smi child: three samples 20 ms apart."""
    OUT = ("2026/12/02 18:00:00.000, 0, 2070, 2070, 900, 0x0, Not Active, Not Active, "
           "Not Active, Not Active\n"
           "2026/12/02 18:00:00.020, 0, 1800, 2070, 1300, 0x4, Not Active, Not Active, "
           "Not Active, Active\n"
           "2026/12/02 18:00:00.040, 0, 1700, 2070, 1350, 0x4, Not Active, Not Active, "
           "Not Active, Active\n")

    def terminate(self):
        pass

    def kill(self):
        pass

    def communicate(self, timeout=None):
        return self.OUT, ""


def test_clock_sampler_keeps_the_samples_of_the_timed_region():
    import datetime
    sys.path.insert(0, ROOT)
    import bench
    t = lambda ms: datetime.datetime(2026, 12, 2, 18, 0, 0, ms * 1000)
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.proc, c.gpu, c.t0, c.t1 = _FakeSmi(), 0, None, None
    c.region(t(15), t(45))  # the last two samples
    d = c.stop()
    assert d["samples"] == 2 and d["sm_mhz"] == 1750.0 and d["reasons"] == ["sw_power_cap"]
    assert d["window_ms"] == 30.0
    c.proc = _FakeSmi()
    c.region(t(1), t(6))  # shorter than the period: the sample nearest its middle
    d = c.stop()
    assert d["samples"] == 1 and d["sm_mhz"] == 2070.0 and d["reasons"] == []
