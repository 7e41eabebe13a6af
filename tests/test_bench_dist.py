"""bench.py's multi-rank host logic on the CPU, world_size 2 over gloo: the timing
reduction every GPU arm uses (the job's time is its slowest rank's), the partition of
the (batch, head) pairs across ranks, the --gpus / WORLD_SIZE agreement, and the
reference arm launched by torchrun (rank 0 alone runs and prints one line; the other
rank exits 0 without work).  The forward itself has no collective: heads are
independent."""
import json
import os
import socket
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_gloo_world_size_2(tmp_path):
    script = tmp_path / "rank.py"
    script.write_text(textwrap.dedent(f"""
        import json, sys
        sys.path.insert(0, {ROOT!r})
        import torch.distributed as dist
        import bench
        dist.init_process_group("gloo", init_method="env://")
        rank = dist.get_rank()
        # rank r reports (r + 1, 10 - r) ms: the job takes (2, 10)
        vals = bench.max_over_ranks([rank + 1.0, 10.0 - rank], dist, "cpu")
        local = bench.max_over_ranks([rank + 1.0], None, "cpu")
        print(json.dumps({{"rank": rank, "vals": vals, "local": local}}))
        dist.destroy_process_group()
    """))
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()),
               WORLD_SIZE="2")
    procs = [subprocess.Popen([sys.executable, str(script)], env=dict(env, RANK=str(r)),
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for r in range(2)]
    outs = []
    for pr in procs:
        out, err = pr.communicate(timeout=300)
        assert pr.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["vals"] == [2.0, 10.0]
        assert o["local"] == [o["rank"] + 1.0]


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                        "--master-port", str(port), "bench.py", "--gpus", "2", "--impl",
                        "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1  # rank 0 only
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0


def test_head_partition_gloo_world_size_2(tmp_path):
    """Every rank computes its own slice; gathered over gloo, the slices tile the
    (batch, head) pairs exactly once, in rank order, balanced within one head."""
    script = tmp_path / "part.py"
    script.write_text(textwrap.dedent(f"""
        import json, sys
        sys.path.insert(0, {ROOT!r})
        import torch, torch.distributed as dist
        import bench
        dist.init_process_group("gloo", init_method="env://")
        rank, world = dist.get_rank(), dist.get_world_size()
        res = {{}}
        for bh in (1, 2, 3, 32, 33, 1024):
            lo, hi = bench.head_slice(bh, world, rank)
            t = torch.tensor([lo, hi], dtype=torch.int64)
            allv = [torch.zeros(2, dtype=torch.int64) for _ in range(world)]
            dist.all_gather(allv, t)
            res[bh] = [v.tolist() for v in allv]
        print(json.dumps({{"rank": rank, "res": res}}))
        dist.destroy_process_group()
    """))
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()),
               WORLD_SIZE="2")
    procs = [subprocess.Popen([sys.executable, str(script)], env=dict(env, RANK=str(r)),
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for r in range(2)]
    outs = []
    for pr in procs:
        out, err = pr.communicate(timeout=300)
        assert pr.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    assert outs[0]["res"] == outs[1]["res"]
    for bh, slices in outs[0]["res"].items():
        bh = int(bh)
        covered = [i for lo, hi in slices for i in range(lo, hi)]
        assert covered == list(range(bh))  # every head once, contiguous, in rank order
        sizes = [hi - lo for lo, hi in slices]
        assert max(sizes) - min(sizes) <= 1


def test_head_partition_larger_worlds():
    sys.path.insert(0, ROOT)
    import bench
    for world in (1, 3, 4, 8):
        for bh in (1, 5, 32, 100):
            slices = [bench.head_slice(bh, world, r) for r in range(world)]
            assert [i for lo, hi in slices for i in range(lo, hi)] == list(range(bh))
            sizes = [hi - lo for lo, hi in slices]
            assert max(sizes) - min(sizes) <= 1


def test_gpus_must_match_world_size():
    """Run under a launcher with WORLD_SIZE=1 but --gpus 2: bench.py refuses."""
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, "bench.py", "--gpus", "2", "--impl", "reference",
                        "--steps", "1"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode != 0 and "WORLD_SIZE" in (r.stderr + r.stdout)
