"""Host-side pieces of bench.py without a GPU: the max-over-ranks timing
with two gloo ranks, the workload description, the oracle timing legs."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


WORKER = r"""
import os, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
rank = dist.get_rank()
t = bench.max_over_ranks(10.0 + 5.0 * rank, dist.get_world_size())
print("RESULT", rank, t, flush=True)
dist.destroy_process_group()
"""


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    """Each rank reports its own time; every rank gets the slowest one."""
    script = tmp_path / "worker.py"
    script.write_text(WORKER.format(root=ROOT))
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2",
                   LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env,
                                      stdout=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120)[0] for p in procs]
    assert all(p.returncode == 0 for p in procs)
    got = sorted(line.split()[1:] for o in outs for line in o.splitlines()
                 if line.startswith("RESULT"))
    assert got == [["0", "15.0"], ["1", "15.0"]]


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_workload_description_and_bytes():
    import bench
    from spec_verify_paged_gb300 import workloads as W
    wl = W.make_attention(W.CONFIGS["tiny-decode"], poison=False)
    conf, tr = bench.workload_config(wl)
    assert conf["workload"] == "tiny-decode"
    assert conf["kv_bytes_per_step"] == 2 * 4 * 64 * 4 * 256 == 524288
    json.dumps(conf)


def test_reference_arm_prints_one_line(capsys):
    """--impl reference times the CPU oracle and prints the contract line."""
    import bench
    bench.main(["--impl", "reference", "--workload", "tiny-decode",
                "--steps", "2", "--warmup", "3"])
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle"


def test_warmup_floor():
    import bench
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "1"])


def test_code_hash_ignores_comments_and_traffic_lookup(tmp_path, monkeypatch):
    """A comment-only edit keeps a source's code hash (so a committed ncu
    summary stays valid); a code edit changes it (so the traffic figure is
    dropped)."""
    import bench
    src = tmp_path / "k.cu"
    src.write_text("int f() {  // one\n  return 1;\n}\n")
    h0 = bench.code_hash(str(src))
    src.write_text("// a new header comment\nint f() {  // two\n\n  return 1;\n}\n")
    assert bench.code_hash(str(src)) == h0
    src.write_text("int f() {\n  return 2;\n}\n")
    assert bench.code_hash(str(src)) != h0
    # a summary line with the file hash appended still parses
    root = tmp_path / "root"
    (root / "profiles").mkdir(parents=True)
    csrc = tmp_path / "csrc"
    csrc.mkdir()
    (csrc / "k.cu").write_text("int f() {\n  return 2;\n}\n")
    h = bench.code_hash(str(csrc / "k.cu"))
    (root / "profiles" / "ncu_kern_wl.md").write_text(
        f"- k.cu code sha256 prefix: `{h}` (file `0123`)\n"
        "- dram bytes per launch: `12345`\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    monkeypatch.setattr(bench, "CSRC", str(csrc))
    assert bench.kernel_traffic("kern", "k.cu", "wl") == 12345
    (csrc / "k.cu").write_text("int f() {\n  return 3;\n}\n")
    assert bench.kernel_traffic("kern", "k.cu", "wl") is None
