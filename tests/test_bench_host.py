"""bench.py on the host, no GPU: the reference arm (the fp64 oracle timed on the host
cores) prints one JSON line with the contract's keys, alone and as rank 0 of two gloo
ranks (the other rank exits without work), and the max-over-ranks timing helper
agrees across two gloo processes."""
import json
import os
import socket
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def env_cpu():
    env = dict(os.environ)
    env["CUDA_VISIBLE_DEVICES"] = ""
    env["OMP_NUM_THREADS"] = "2"
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    return env


def json_lines(out: str):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def check_reference_line(d, n, steps, warmup):
    assert d["impl"] == "reference" and d["n_gpus"] == n
    assert d["steps"] == steps and d["warmup"] == warmup
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["unit"] == "block-steps/s" and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["dtype"] == "f64" and d["data"] == "synthetic" and d["config"]["workload"].startswith("clover_layer")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_one_process():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "clover_layer", "--steps", "2",
                        "--warmup", "1"], cwd=ROOT, env=env_cpu(), capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = json_lines(r.stdout)
    assert len(lines) == 1
    check_reference_line(lines[0], 1, 2, 1)


def test_reference_arm_two_gloo_ranks():
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py", "--gpus", "2",
                        "--impl", "reference", "--config", "clover_layer", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, env=env_cpu(), capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = json_lines(r.stdout)
    assert len(lines) == 1          # rank 0 alone prints
    check_reference_line(lines[0], 2, 1, 0)


def test_dist_max_over_two_gloo_ranks(tmp_path):
    script = tmp_path / "dist_max.py"
    script.write_text(textwrap.dedent(f"""
        import sys
        sys.path.insert(0, {ROOT!r})
        import bench
        d = bench.Dist("gloo")
        d.barrier()
        v = d.max(1.5 + 2.0 * d.rank)
        import os
        os.write(1, f"RANK {{d.rank}} WORLD {{d.world}} MAX {{v}}\\n".encode())   # one write: lines never interleave
        d.close()
    """))
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(free_port()), str(script)],
                       cwd=ROOT, env=env_cpu(), capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    got = sorted(l.split() for l in r.stdout.splitlines() if l.startswith("RANK"))
    assert [g[1] for g in got] == ["0", "1"] and all(g[3] == "2" for g in got)
    assert all(float(g[5]) == 3.5 for g in got)


@pytest.mark.parametrize("argv", [["--impl", "gpu", "--gpus", "1", "--steps", "3", "--warmup", "3"]])
def test_bench_arguments_parse(argv, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setattr(sys, "argv", ["bench.py"] + argv)
    a = bench.parse()
    assert a.steps == 3 and a.warmup == 3 and a.layer_head is None
