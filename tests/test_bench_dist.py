"""The N>1 bench path on CPU: gloo ranks, max-over-ranks time, sum of units,
and the reference arm under torchrun (rank 0 prints one line, others none)."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    torch.distributed.init_process_group("gloo")
    bench.barrier(ws)
    t, u = bench.reduce_max_sum(ws, float(rank + 1), 10.0 * (rank + 1), torch.device("cpu"))
    q.put((rank, t, u))
    torch.distributed.destroy_process_group()


def test_reduce_max_sum_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [2.0, 2.0]        # max over ranks
    assert [r[2] for r in res] == [30.0, 30.0]      # sum of units


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "2", "--warmup", "3", "--ref-seconds", "2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def _load_bench(root):
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    b.ROOT = root
    return b


def test_kernel_hash_ignores_comments_and_sees_code(tmp_path):
    # the recorded DRAM counters stay valid across comment edits, not code edits
    import shutil
    src = os.path.join(ROOT, "bit_codebook_quantized_gb300", "csrc")
    dst = tmp_path / "bit_codebook_quantized_gb300" / "csrc"
    shutil.copytree(src, dst)
    b = _load_bench(str(tmp_path))
    h0 = b.kernel_source_hash("gemv_kernel")
    f = dst / "cbq_gemv.cu"
    text = f.read_text()
    f.write_text(text.replace("namespace cbq {", "namespace cbq {  // an added comment\n// and a comment line", 1))
    assert b.kernel_source_hash("gemv_kernel") == h0
    f.write_text(text.replace("constexpr int kStages = 4;", "constexpr int kStages = 5;", 1))
    assert b.kernel_source_hash("gemv_kernel") != h0
    assert b.kernel_source_hash("sk_kernel") != b.kernel_source_hash("umma_kernel")


def test_profiled_traffic_needs_a_matching_hash(tmp_path):
    import shutil
    shutil.copytree(os.path.join(ROOT, "bit_codebook_quantized_gb300", "csrc"),
                    tmp_path / "bit_codebook_quantized_gb300" / "csrc")
    (tmp_path / "profiles").mkdir()
    b = _load_bench(str(tmp_path))
    h = b.kernel_source_hash("gemv_kernel")
    prof = tmp_path / "profiles" / "cbq_gemm_decode_4096x12288.md"
    prof.write_text(f"kernel_source_sha256[gemv_kernel]: {h}\n"
                    "dram_bytes_per_launch[gemv_kernel] M=1: 100\n"
                    "dram_bytes_per_launch[gemv_kernel] M=8: 200\n")
    assert b.profiled_traffic("gemv_kernel") == {"1": 100.0, "8": 200.0}
    assert b.profiled_traffic("sk_kernel") is None                 # no counters recorded for it
    prof.write_text(prof.read_text().replace(h, "0" * 16))
    assert b.profiled_traffic("gemv_kernel") is None                # sources changed since
