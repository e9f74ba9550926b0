"""The benchmark's host logic on CPU: the JSON line carries every key of the contract,
the kernel count per step, the expert-FFN path the library picks, the recorded DRAM
traffic lookup, and the reference arm (the oracle) printing on rank 0 only."""
import json
from types import SimpleNamespace

import numpy as np

import bench
from synth import CONFIGS, make_layer


def _args(**kw):
    a = dict(steps=20, warmup=3, ffn_path="auto", ref_tokens=64)
    a.update(kw)
    return SimpleNamespace(**a)


def test_result_line_has_every_contract_key():
    L = make_layer(**CONFIGS["tiny"])
    cfg = {"workload": "tiny layer"}
    roof = {"bound": "hbm", "achieved": 1.0, "peak": 2.0, "unit": "GB/s", "frac": 0.5, "traffic": None}
    cpu = {"value": 10.0, "unit": "tokens/s", "cores": 4, "kind": "oracle", "sample": "64 tokens"}
    clocks = {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0, "reasons": []}
    line = bench.result_line(_args(), 1, cfg, L, value=1e5, step_ms=[0.1, 0.2], eager_ms=0.3,
                             roofline=roof, cpu=cpu, e2e_serial=9e4, e2e_pipelined=9.5e4,
                             clocks=clocks, extras={"gate": None})
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert key in line, key
    assert line["config"]["workload"] == "tiny layer" and line["scaling"] == "weak"
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in line["roofline"]
    for key in ("value", "unit", "cores", "kind", "sample"):
        assert key in line["cpu_baseline"]
    e2e = line["e2e"]
    assert e2e["value"] == 9e4 and e2e["h2d_bytes_per_step"] == L.T * L.H * 2 + L.T * L.E * 4
    assert e2e["d2h_bytes_per_step"] == L.T * L.H * 2
    assert line["gpu_launches"] == 5 * 20 and line["ms_per_step"] == np.mean([0.1, 0.2])
    json.dumps(line)  # serialisable as one line


def test_launches_and_paths():
    assert bench.launches_per_step(512, False) == 5
    assert bench.launches_per_step(32768, True) == 9
    E = 128
    assert bench.ffn_path_used(8 * E - 1, E, "auto") == "gemv"
    assert bench.ffn_path_used(8 * E, E, "auto") == "gemm_decode"
    assert bench.ffn_path_used(32 * E, E, "auto") == "gemm"
    assert bench.ffn_path_used(10, E, "gemm") == "gemm"


def test_recorded_traffic_only_for_its_workload_and_sources():
    got = bench.recorded_traffic("expert_ffn_gemv", "decode layer H2048 I768 E128 top-8 q4_0 T64")
    assert got is None or got > 3e8  # the headline pair reads ~341 MB when recorded
    assert bench.recorded_traffic("expert_ffn_gemv", "some other workload") is None


def test_reference_arm_prints_on_rank_zero_only(capsys):
    L = make_layer(**CONFIGS["tiny"])
    cfg = {"workload": "tiny layer"}
    bench.run_reference(_args(steps=1), cfg, L, 2, 1)
    assert capsys.readouterr().out == ""
    bench.run_reference(_args(steps=1), cfg, L, 1, 0)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_scalars_flattens_nested_numbers_for_the_one_line_record():
    d = {"q4_0": {"tokens_per_s": 5.0, "workload": "w", "roofline": {"frac": 0.3, "unit": "TFLOP/s"}},
         "n": 3, "flag": True, "none": None}
    assert bench.scalars(d) == {"q4_0_tokens_per_s": 5.0, "q4_0_roofline_frac": 0.3, "n": 3}
    assert bench.scalars(None) == {}


def test_every_bank_format_is_a_bench_format():
    assert set(CONFIGS["decode"]["qtypes"]) == {"q4_0", "mxfp4", "nvfp4", "mxfp8"}
    assert set(CONFIGS["prefill"]["qtypes"]) == {"q4_0", "mxfp4", "nvfp4", "mxfp8"}
    assert CONFIGS["stream"]["steps"] == 2048


def test_clock_sampler_reads_nvml_often_and_maps_reasons(monkeypatch):
    """The sampler takes NVML readings every 10 ms (a short timed region still gets several
    samples) and reports the throttle reasons that were active, from a fake NVML."""
    import sys
    import time
    import types
    calls = {"n": 0}
    fake = types.SimpleNamespace(
        NVML_CLOCK_SM=1,
        nvmlInit=lambda: None,
        nvmlDeviceGetHandleByIndex=lambda i: ("gpu", i),
        nvmlDeviceGetHandleByPciBusId=lambda b: ("gpu", b),
        nvmlDeviceGetClockInfo=lambda h, c: 1965,
        nvmlDeviceGetMaxClockInfo=lambda h, c: 2032,
        nvmlDeviceGetPowerUsage=lambda h: 850000,
        nvmlClocksEventReasonSwPowerCap=0x4, nvmlClocksEventReasonHwSlowdown=0x8,
        nvmlClocksEventReasonSwThermalSlowdown=0x20, nvmlClocksEventReasonHwThermalSlowdown=0x40)

    def reasons(h):
        calls["n"] += 1
        return 0x4 if calls["n"] % 2 else 0x0  # sw_power_cap on every other reading
    fake.nvmlDeviceGetCurrentClocksEventReasons = reasons
    monkeypatch.setitem(sys.modules, "pynvml", fake)
    clk = bench.ClockSampler(0, "00000000:1B:00.0")
    with clk:
        time.sleep(0.15)
    s = clk.summary()
    assert s["source"] == "nvml" and s["samples"] >= 5
    assert s["sm_mhz"] == 1965.0 and s["sm_max_mhz"] == 2032.0
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_sampler_falls_back_without_nvml(monkeypatch):
    """Without NVML the sampler reads one nvidia-smi process in loop mode (a fake here)
    until the timed region ends, then ends that process."""
    import sys
    import time
    monkeypatch.setitem(sys.modules, "pynvml", None)  # import fails
    line = "0, 2032, 2032, 800.00, 0x4, Not Active, Not Active, Not Active, Active\n"
    ended = {"terminated": False}

    class FakeProc:
        def __init__(self, argv, **kw):
            assert argv[0] == "nvidia-smi" and "-lms" in argv
            self.stdout = self._lines()

        def _lines(self):
            for _ in range(1000):
                if ended["terminated"]:
                    return
                time.sleep(0.005)
                yield line

        def terminate(self):
            ended["terminated"] = True

        def wait(self, timeout=None):
            return 0
    monkeypatch.setattr(bench.subprocess, "Popen", FakeProc)
    clk = bench.ClockSampler(0)
    with clk:
        time.sleep(0.05)
    s = clk.summary()
    assert ended["terminated"]
    assert s["source"] == "nvidia-smi" and s["samples"] >= 3 and s["reasons"] == ["sw_power_cap"]
    assert s["sm_mhz"] == 2032.0
