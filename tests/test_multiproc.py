"""The N > 1 launch path of bench.py on CPU: two gloo ranks under
torch.distributed.run; rank 0 alone prints the JSON line of the reference
(oracle) arm and every rank exits 0."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_reference_arm_two_ranks_gloo():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", "--master-port=29531", "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3", "--config", "c1"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def _owner_rank(rank, world, port, outdir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    from newton_schulz_gb300 import binding
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    # each rank's own measurement of the per-shape NS times (here synthetic:
    # a common table with rank-dependent noise), then the median across ranks
    base = {(4096, 4096): 4.0, (1024, 4096): 1.5, (4096, 14336): 11.0}
    noise = 1.0 + 0.05 * ((rank * 7919) % 11 - 5) / 5.0
    mine = {k: v * noise for k, v in base.items()}
    tables = [None] * world
    dist.all_gather_object(tables, mine)
    import statistics
    cost = {k: statistics.median(t[k] for t in tables) for k in base}
    # Llama-like units: 32 layers x (q, k, v, o, gate, up, down)
    shapes = [(4096, 4096), (1024, 4096), (1024, 4096), (4096, 4096),
              (4096, 14336), (4096, 14336), (4096, 14336)]
    units = [(l, s) for l in range(32) for s in shapes]
    owner = binding.muon_assign_owners([cost[s] for _, s in units], world,
                                       nbytes=[s[0] * s[1] * 10 for _, s in units],
                                       elems=[s[0] * s[1] for _, s in units],
                                       layers=[l for l, _ in units], eps=0.1)
    with open(os.path.join(outdir, f"owner{rank}.json"), "w") as f:
        json.dump(owner, f)
    dist.destroy_process_group()


def test_owner_assignment_agrees_across_gloo_ranks(tmp_path):
    """Two gloo ranks aggregate their cost tables (median) and compute the
    owner assignment independently: the same owners on every rank, each
    matrix owned exactly once, every rank with a share."""
    import torch.multiprocessing as mp
    mp.spawn(_owner_rank, args=(2, 29533, str(tmp_path)), nprocs=2, join=True)
    a = json.load(open(tmp_path / "owner0.json"))
    b = json.load(open(tmp_path / "owner1.json"))
    assert a == b
    assert set(a) == {0, 1} and len(a) == 32 * 7
