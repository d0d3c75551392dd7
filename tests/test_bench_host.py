"""bench.py's host logic without a GPU: the N > 1 aggregation over two gloo
ranks, the reference arm under torchrun (rank 0 prints, rank 1 exits 0), and
the small parsers (traffic summary, peaks, nvidia-smi samples)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        elapsed = [0.25, 0.5][rank]                 # rank 1 is the slowest
        elems = 1000.0 * (rank + 1)
        t = bench.max_over_ranks(elapsed)
        total = bench.sum_over_ranks(elems)
        out.put((r, w, local, bench.emulated_rank(r, 8), t, total, total / t))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1] and all(x[1] == 2 for x in res)
    assert [x[3] for x in res] == [0, 1]                 # distinct emulated ranks
    for x in res:
        assert x[4] == 0.5 and x[5] == 3000.0          # max time, summed work
        assert x[6] == 6000.0                          # whole-job throughput


def test_emulated_rank_wraps():
    assert [bench.emulated_rank(g, 4) for g in range(9)] == [0, 1, 2, 3, 0, 1, 2, 3, 0]
    assert [bench.emulated_rank(g, 4, 3) for g in range(5)] == [3, 0, 1, 2, 3]


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "3",
           "--warmup", "3", "--workload", "tiny"]
    p = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [json.loads(x) for x in p.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = lines[0]
    assert line["impl"] == "reference" and line["unit"] == "elements/s" and line["value"] > 0
    assert line["metric"] == bench.METRIC and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_loads_only_the_oracle_and_generator():
    """The reference arm sizes its sample with the oracle's own plan: the CUDA
    path's library is never loaded, and its config is the dict the GPU arm
    prints for the same run; ms_per_step is the measured sample's."""
    code = ("import json, sys; sys.argv = ['bench.py', '--impl', 'reference', '--steps', '3', "
            "'--warmup', '3', '--workload', 'gpt2-small', '--buckets']; import bench; "
            "bench.main(sys.argv[1:]); "
            "maps = open('/proc/self/maps').read(); "
            "print('LIBS', json.dumps(sorted({l.split()[-1].rsplit('/', 1)[-1] for l in "
            "maps.splitlines() if l.endswith('.so') and '/repo' in l or 'libzs' in l "
            "or 'liboracle' in l})))")
    p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    line = json.loads(next(x for x in p.stdout.splitlines() if x.startswith("{")))
    libs = json.loads(next(x for x in p.stdout.splitlines() if x.startswith("LIBS"))[5:])
    assert "liboracle.so" in libs and not any(x.startswith("libzs.") or
                                               x.startswith("libzs_checked") for x in libs), libs
    from synth.workloads import WORKLOADS
    import oracle
    w = WORKLOADS["gpt2-small"]
    op = oracle.default().plan(w.numels, w.tied_to, world=w.world, align=w.align,
                               bucket_elems=w.bucket_elems)
    args = bench.argparse.Namespace(pipeline="step", step_path="auto", micro_steps=4,
                                    no_overlap=False)
    # rank 0's shard lies inside one bucket (the one holding wte): one call
    want = bench.run_config(args, w, op["S"], op["P"], op["P_pad"], 1, 0, 1)
    assert line["config"] == want
    n = line["sample_elems_per_step"]
    assert abs(line["value"] * line["ms_per_step"] / 1e3 - n) <= 1e-6 * n


def test_traffic_summary_matches_kernel_sha(tmp_path, monkeypatch):
    f = tmp_path / "traffic.txt"
    sha = bench.kernel_sha()
    f.write_text(f"# c\ntraffic llama-7b kernel_sha={sha} bytes_per_elem=41.97\n"
                 f"traffic qwen2.5-3b kernel_sha=0000000000000000 bytes_per_elem=33.9\n")
    monkeypatch.setattr(bench, "TRAFFIC_SUMMARY", str(f))
    assert bench.committed_traffic("llama-7b") == 41.97
    assert bench.committed_traffic("qwen2.5-3b") is None      # taken on other code
    assert bench.committed_traffic("gpt2-small") is None


def test_clock_sampler_parses_nvidia_smi(monkeypatch):
    s = bench.ClockSampler()

    class FakeProc:
        def terminate(self):
            pass

        def communicate(self, timeout=None):
            rows = ["0, 2070, 2070, 900.5, Not Active, Not Active, Not Active, Not Active",
                    "0, 1980, 2070, 1390.0, Not Active, Not Active, Not Active, Active",
                    "0, 2070, 2070, 1000.0, Not Active, Not Active, Not Active, Not Active"]
            return "\n".join(rows) + "\n", ""

    s.proc = FakeProc()
    c = s.stop()
    assert c["sm_mhz"] == 2070.0 and c["sm_max_mhz"] == 2070.0 and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"]


def test_peak_fallback(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peak() == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 1234.5}))
    assert bench.measured_peak() == (1234.5, "measured")


def test_warmup_below_three_rejected():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2", "--impl", "reference"])
