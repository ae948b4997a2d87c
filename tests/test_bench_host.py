"""Host logic of bench.py that needs no GPU: the clock record of a timed
region (nvidia-smi samples kept only inside the region's wall-clock window)
and the rule that voids a number measured under a slowdown or a clock lock,
and the guard that reports DRAM traffic only for unchanged kernel sources."""
import datetime
import json

import bench

UUID = "GPU-0000"


def _line(t, sm, smax=2070, reasons=("Not Active",) * 4, uuid=UUID, power=1300.0):
    stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    active = "0x0000000000000004" if "Active" in reasons else "0x0000000000000000"
    return ", ".join([stamp, uuid, str(sm), str(smax), f"{power:.2f}", active, *reasons])


def _sampler(lines, windows):
    s = bench.ClockSampler(UUID)
    s.lines = list(lines)
    s.windows = list(windows)
    return s


def test_summary_keeps_samples_inside_the_windows_only():
    t0 = 1_700_000_000.0
    lines = [_line(t0 + 0.05 * i, 1000 if i < 10 else 1900) for i in range(30)]
    lines.append(_line(t0 + 0.6, 100, uuid="GPU-other"))      # another GPU's sample
    s = _sampler(lines, [(t0 + 0.5, t0 + 1.2)])
    out = s.summary()
    assert out["sm_mhz"] == 1900.0
    assert out["sm_max_mhz"] == 2070.0
    assert out["samples_in_timed_regions"] == 15
    assert out["reasons"] == []
    # an explicit window list overrides the recorded one
    early = s.summary(windows=[(t0, t0 + 0.45)], span="early")
    assert early["sm_mhz"] == 1000.0 and early["span"] == "early"


def test_summary_collects_active_reasons():
    t0 = 1_700_000_000.0
    cap = ("Not Active", "Not Active", "Not Active", "Active")
    thermal = ("Not Active", "Active", "Not Active", "Not Active")
    lines = [_line(t0 + 0.05 * i, 1850, reasons=cap) for i in range(10)]
    lines.append(_line(t0 + 0.2, 1500, reasons=thermal))
    out = _sampler(lines, [(t0, t0 + 1.0)]).summary()
    assert out["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_rejection_rule():
    ok = {"sm_mhz": 1852.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    assert bench.clock_rejection(ok) == []
    # a power cap explains a lower clock: the number stands
    assert bench.clock_rejection({**ok, "sm_mhz": 1200.0}) == []
    for r in bench.REJECTING_REASONS:
        assert bench.clock_rejection({**ok, "reasons": ["sw_power_cap", r]}) == [r]
    # a low clock with no reason reported reads as a leftover clock lock
    locked = {"sm_mhz": 1100.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert len(bench.clock_rejection(locked)) == 1
    assert bench.clock_rejection({**locked, "sm_mhz": 2000.0}) == []
    # no samples at all voids nothing (and says so in the record itself)
    assert bench.clock_rejection({"sm_mhz": None, "sm_max_mhz": None,
                                  "reasons": ["unsampled"]}) == []


def test_recorded_traffic_follows_the_source_digest(tmp_path, monkeypatch):
    digest = "a" * 64
    rec = {"quant2d_tile_rows": {"bytes_per_launch": 123, "source_sha256": digest}}
    path = tmp_path / "profiles" / "roofline_traffic.json"
    path.parent.mkdir()
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_digest", lambda key: digest)
    assert bench.recorded_traffic("quant2d_tile_rows") == 123
    rec["quant2d_tile_rows"]["source_sha256"] = "0" * 64      # the kernel changed since
    path.write_text(json.dumps(rec))
    assert bench.recorded_traffic("quant2d_tile_rows") is None
    assert bench.recorded_traffic("gemm_mx_kernel") is None      # no record at all


def test_every_committed_traffic_record_is_complete():
    with open(f"{bench.ROOT}/profiles/roofline_traffic.json") as f:
        recs = json.load(f)
    assert set(bench.KERNEL_SOURCES) <= set(recs)
    for key, r in recs.items():
        assert r["bytes_per_launch"] > 0
        assert len(r["source_sha256"]) == 64
        assert "ncu" in r["command"] and "--clock-control none" in r["command"]


def test_reference_arm_prints_its_line_on_the_host():
    """`bench.py --impl reference` times the oracle on the host cores and
    prints one JSON line with the bench contract's keys (one short step)."""
    import subprocess
    import sys
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=bench.ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 1 and line["n_gpus"] == 1
    assert line["value"] > 0 and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == line["value"]
    assert cpu["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert line["config"]["workload"]


def test_reference_arm_under_torchrun_prints_once():
    """With two ranks (gloo on the CPU) rank 0 alone runs the reference arm and
    prints its line; the other rank exits 0 without work."""
    import socket
    import subprocess
    import sys
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port",
                        str(port), "bench.py", "--impl", "reference", "--gpus", "2", "--steps",
                        "1", "--warmup", "0"], cwd=bench.ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0


def test_profile_summaries_name_runnable_cases():
    """Every ncu summary under profiles/ gives a command that runs committed
    files only: each `--profile-case` it names exists in bench.py (templates
    such as layer_<recipe>_<linear> expand to existing cases), and every ncu
    command leaves the clocks alone."""
    import glob
    import itertools
    import os
    import re
    paths = sorted(glob.glob(os.path.join(bench.ROOT, "profiles", "*.md")) +
                   glob.glob(os.path.join(bench.ROOT, "profiles", "*.json")))
    assert paths
    fill = {"<recipe>": ("tensor", "block", "mx"),
            "<linear>": ("qkv", "attn_out", "mlp_up", "mlp_down")}
    for path in paths:
        text = open(path).read()
        for case in re.findall(r"--profile-case ([a-z_<>]+)", text):
            slots = [s for s in fill if s in case]
            for combo in itertools.product(*(fill[s] for s in slots)):
                name = case
                for s, v in zip(slots, combo):
                    name = name.replace(s, v)
                assert name in bench.PROFILE_CASES, (os.path.basename(path), name)
        for cmd in re.findall(r"ncu [^\n]*", text):
            if "--metrics" in cmd or "--set" in cmd or "--section" in cmd:
                block = text[text.index(cmd):text.index(cmd) + 400]
                assert "--clock-control none" in block, (os.path.basename(path), cmd)
