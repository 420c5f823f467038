"""Host-side logic of bench.py: byte model, rotation, step split, clocks, ranks."""

import json
import os
import socket
import subprocess
import sys

import pytest

import bench
import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_byte_model_matches_oracle_counts():
    orc = oracle.load()
    for name, w in synth.WORKLOADS.items():
        assert bench.algorithmic_bytes(w.dtype, w.M, w.N) == orc.bytes(w.dtype, w.M, w.N), name
    # the headline workload: 2MN + 2N + 4M
    assert bench.algorithmic_bytes("f16", 4096, 14336) == 2 * 4096 * 14336 + 2 * 14336 + 4 * 4096


def test_rotation_covers_l2_and_256mib():
    l2 = 126 << 20
    wb = bench.a_bytes("f16", 4096, 14336)
    c = bench.rotation_copies(wb, l2)
    assert c * wb >= max(256 << 20, 4 * l2) and (c - 1) * wb < max(256 << 20, 4 * l2)
    assert bench.rotation_copies(1 << 40, l2) == 2  # never fewer than two copies


def test_split_steps_is_exact():
    for steps in (1, 7, 100, 30000, 30001):
        for batch in (1, 5, 100, 105):
            full, tail = bench.split_steps(steps, batch)
            assert full * batch + tail == steps and 0 <= tail < batch


def test_mbu_arithmetic_reproduces_the_published_row():
    # membound "Results": 4096x14336 vec at 0.2817 ms is 417.0 GB/s
    b = bench.algorithmic_bytes("f16", 4096, 14336)
    assert abs(bench.gbs(b, 0.2817e-3) - 417.0) < 0.1


def test_parse_clock_line():
    s = bench.parse_clock_line("0, 1965, 2070, 612.3, 0x0000000000000004, Not Active, Not Active, "
                               "Not Active, Active")
    assert s == {"sm": 1965.0, "sm_max": 2070.0, "reasons": ["sw_power_cap"]}
    assert bench.parse_clock_line("garbage") is None


def test_kernel_source_hash_is_stable():
    assert bench.kernel_source_hash() == bench.kernel_source_hash()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


_RANK_SCRIPT = r"""
import os, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
r = dist.get_rank()
m = bench.max_over_ranks(1.5 + r)
bench.barrier()
print("RESULT", r, m, flush=True)
dist.destroy_process_group()
"""


def test_max_over_ranks_gloo_world_size_2(tmp_path):
    pytest.importorskip("torch")
    script = tmp_path / "rank.py"
    script.write_text(_RANK_SCRIPT.format(root=ROOT))
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (out, err) in zip(procs, outs):
        assert p.returncode == 0, err
        assert "RESULT" in out
        assert float(out.split()[-1]) == 2.5


def test_reference_arm_prints_one_json_line_on_cpu():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "1", "--reference-seconds", "1"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["metric"] == bench.METRIC
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "1"], capture_output=True, text=True,
                       timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_cli_rejects_aux_without_profile_and_bad_arguments():
    """`--op aux` launches kernels for a profiler only; it and other bad argument sets are refused
    by the argument parser (exit code 2) before anything touches a GPU."""
    for argv in (["--op", "aux"], ["--steps", "0"], ["--warmup", "-1"],
                 ["--op", "softmax", "--workload", "f16_4096"], ["--workload", "no_such_workload"]):
        with pytest.raises(SystemExit) as e:
            bench.main(argv)
        assert e.value.code == 2, argv
