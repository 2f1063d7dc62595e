"""The N > 1 paths of bench.py on the CPU: two ranks over gloo on 127.0.0.1.

The path shards as independent replicas (no collective on the data path); what the ranks
share is the barrier and the max-over-ranks reduction of the timed interval, and the
reference arm, which only rank 0 runs and prints.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist(world)
    assert d.pg is not None and d.world == world and d.rank == rank
    d.barrier()
    # each rank's "elapsed ms"; every rank must see the slowest one
    got = d.max(10.0 + 5.0 * rank)
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
        f.write(repr(got))
    d.close()


def test_dist_barrier_and_max_over_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    vals = [float((tmp_path / f"r{r}.txt").read_text()) for r in range(2)]
    assert vals == [15.0, 15.0]


def test_reference_arm_under_torchrun_prints_once(tmp_path):
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0", "--cpu-tokens", "96", "--prefill-workload", "pair"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = lines[0]
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["n_gpus"] == 2 and line["steps"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    # the rest of the JSON-line contract
    for key in ("metric", "unit", "ms_per_step", "higher_is_better", "scaling", "vs_baseline",
                "dtype", "data", "config", "warmup"):
        assert key in line, key
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["dtype"] == "f64" and line["vs_baseline"] is None
    assert line["config"]["workload"] and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["unit"] == line["unit"]
    # the same config dict as the GPU arm prints for these arguments
    sys.path.insert(0, ROOT)
    import bench
    args = _parse(bench, cmd[cmd.index("--impl"):])
    assert line["config"] == bench.line_config(args, 2)


def _parse(bench, argv):
    saved = sys.argv
    sys.argv = ["bench.py"] + list(argv)
    try:
        return bench.parse()
    finally:
        sys.argv = saved


def test_both_arms_name_the_same_stack28_workload_and_sample():
    """The headline workload is the 28-layer T = 8192 stack; both arms build their config from
    one function, and the oracle's default sample is a stated prefix of that sequence."""
    sys.path.insert(0, ROOT)
    import bench
    args = _parse(bench, ["--impl", "reference"])
    assert args.prefill_workload == "stack28"
    cfg = bench.line_config(args, 1)
    assert cfg["seq_len"] == 8192 and cfg["global_batch"] == 1 and cfg["parallelism"] == "single"
    assert cfg["workload"].startswith("stack28_bf16_T8192: 28-layer")
    assert "3.41 GB of layer weights" in cfg["l2"]
    wl, what = bench.cpu_sample("stack28")
    assert wl.shape.num_layers == 28 and wl.seq_lens == [bench.CPU_SAMPLE_TOKENS["stack28"]]
    assert "every layer and the head" in what
    wl4 = bench.make_workload("stack28", 4)
    assert wl4.shape.num_layers == 4 and wl4.shape.layer_types[3] == "full_attention"
