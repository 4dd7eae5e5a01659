"""Host-side behaviour of bench.py (no GPU).

* A timed region after which the library's device status word is not zero
  (a staged kernel whose bounded wait ran out, recorded a code and returned
  early) yields no value: the bench raises, prints no JSON line and exits
  with a non-zero code.
* The reference arm (the CPU oracle) runs without the library in its
  address space and prints its JSON line.
"""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_check_device_status_passes_zero_and_refuses_a_code():
    assert bench.check_device_status(lambda: 0, "a region") == 0
    with pytest.raises(bench.DeviceStatusError) as e:
        bench.check_device_status(lambda: 2, "the timed steps")
    assert "2" in str(e.value) and "the timed steps" in str(e.value)


class _FakeEvent:
    def __init__(self, enable_timing=False):
        pass

    def record(self, stream=None):
        pass

    def elapsed_time(self, other):
        return 1.0


class _FakeCuda:
    Event = _FakeEvent

    @staticmethod
    def synchronize(dev=None):
        pass


class _FakeTorch:
    cuda = _FakeCuda


def test_timed_region_with_a_device_code_yields_no_time():
    calls = []
    codes = iter([3])

    def status(where):
        return bench.check_device_status(lambda: next(codes), where)

    with pytest.raises(bench.DeviceStatusError):
        bench.timed_on_stream(_FakeTorch, lambda: calls.append(1), 2, 1, None, None, None, status, "a point")
    assert len(calls) == 3                        # the region ran; its time was refused


def test_main_prints_no_line_and_fails_when_the_status_is_set(monkeypatch, capsys):
    def fake_run(args, ws, rank, local):
        bench.check_device_status(lambda: 1, "the timed steps")
        print(json.dumps({"value": 1.0}))         # never reached
        return 0

    monkeypatch.setattr(bench, "run_ours", fake_run)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--steps", "1", "--warmup", "3"])
    rc = bench.main()
    out = capsys.readouterr()
    assert rc != 0
    assert out.out.strip() == ""
    assert "device status 1" in out.err


def test_reference_arm_runs_without_the_library():
    proc = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                           "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert proc.returncode == 0, proc.stderr[-3000:]
    lines = [ln for ln in proc.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"


def test_walk_launch_counts_match_the_recorded_launch_lists():
    """The launch counts bench.py reports for walked calls follow the library's piece cutting; pinned
    to the counts ncu's launch lists of the benchmarked steps show (profiles/launches_*.md): one
    dynamic-order launch per Llama-1.3B ZeRO-2 step and for the update alone on its shard arrays, 360
    walked launches for the step bucket by bucket over its 103 buckets, 66 gathers + 33 updates per
    Llama-7B ZeRO-3 step (one dynamic-order launch per unit and phase)."""
    import fsdp_sharded_optimizer_flatparameter_gb300 as zs
    import synth

    shapes, _ = synth.workload_params("llama-1.3b")
    plan13 = zs.Plan(shapes, 8, stage=2, bucket_bytes=25 << 20)
    P = plan13.padded
    assert bench.walk_launches([(0, P)], 8) == 1
    assert bench.staged_walk_launches([(0, P)]) == 1
    br = [plan13.bucket(b)[1:] for b in reversed(range(plan13.n_buckets))]
    assert plan13.n_buckets == 103 and bench.walk_launches(br, 8) == 360
    shapes, units = synth.workload_params("llama-7b")
    plan = zs.Plan(shapes, 16, stage=3, unit_of_param=units)
    assert bench.zero3_launches(plan, 16) == 99
    assert bench.zero3_launches(plan, 16, reshard=False) == 66
    flat32 = zs.Plan([((1 << 28) + 7,)], 32, stage=3)                 # N_d = 32 keeps the walk
    assert bench.zero3_launches(flat32, 32) == 32 * 3
    # short, ragged and unaligned ranges
    assert bench.staged_walk_launches([(0, 1000)]) == 1
    assert bench.staged_walk_launches([(3, (1 << 21) + 5)]) == 3          # body plus two ragged ends
    assert bench.staged_walk_launches([(0, 3 * (1 << 22) + 8)]) == 3
    assert bench.staged_walk_launches([(5, (1 << 24) + 21)]) == 3         # one dynamic-order launch + two ends
    assert bench.staged_walk_launches([(0, (1 << 24) - 8)]) == 4          # just under 2^24: walked
