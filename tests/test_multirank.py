"""The N > 1 host logic of bench.py on CPU with the gloo backend (world size
2): the timing reduction takes the max over ranks, and a torchrun launch of
the reference arm prints exactly one JSON line (rank 0) while the other rank
exits without work."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    q.put((rank, bench.max_over_ranks(1.5 + 2.0 * rank, world)))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 3.5, 1: 3.5}


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3", "--ref-budget-s", "0.5"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["unit"] == "GB/s" and j["value"] > 0
    assert j["cpu_baseline"]["kind"] == "oracle"
    assert j["steps"] == 2 and j["warmup"] == 3   # the requested timed and untimed steps
    assert j["e2e"]["h2d_bytes_per_step"] == 0


def test_shard_rows_covers_the_batch_once():
    from gated_deltanet_linear_04_gb300 import gdn
    for B in (0, 1, 5, 8, 128, 131):
        for world in (1, 2, 3, 8):
            spans = [gdn.shard_rows(B, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == B
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1


def _shard_worker(rank, world, port, q):
    """Rank `rank` runs a few decode steps of its rows of a small batch (the
    oracle stands in for the device path on CPU), then the ranks gather."""
    import numpy as np
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from gated_deltanet_linear_04_gb300 import gdn, workloads as wl
    d = wl.Dims(B=5, T=1, Hk=1, Hv=2, Dk=32, Dv=32, K=4)
    w = wl.Workload("shard", 0, d, 3, "normal", "normal", False, 1, 1)
    inp = wl.workload_inputs(w)
    steps = [wl.decode_step_inputs(w, i) for i in range(3)]
    b0, b1 = gdn.shard_rows(d.B, world, rank)
    dl = d.with_(B=b1 - b0)
    sb = [{k: wl.bf16_bits(s[k][b0:b1]) for k in ("qkv", "a", "b")} for s in steps]
    ys, st, _ = oracle.decode(dl, sb, wl.bf16_bits(inp["conv_w"]), inp["A_log"].numpy(), inp["dt_bias"].numpy(),
                              wl.bf16_bits(inp["conv_state"][b0:b1]), inp["state"][b0:b1].numpy().astype(np.float64))
    sizes = [gdn.shard_rows(d.B, world, r) for r in range(world)]
    rows = max(e - s for s, e in sizes)
    y_pad = torch.zeros((3, rows, d.Hv, d.Dv), dtype=torch.float64)
    s_pad = torch.zeros((rows, d.Hv, d.Dv, d.Dk), dtype=torch.float64)
    y_pad[:, :b1 - b0] = torch.from_numpy(np.stack(ys))
    s_pad[:b1 - b0] = torch.from_numpy(st)
    gy = [torch.zeros_like(y_pad) for _ in range(world)]
    gs = [torch.zeros_like(s_pad) for _ in range(world)]
    dist.all_gather(gy, y_pad)
    dist.all_gather(gs, s_pad)
    if rank == 0:
        y_full = torch.cat([g[:, :e - s] for g, (s, e) in zip(gy, sizes)], dim=1).numpy()
        s_full = torch.cat([g[:e - s] for g, (s, e) in zip(gs, sizes)], dim=0).numpy()
        sbf = [{k: wl.bf16_bits(s[k]) for k in ("qkv", "a", "b")} for s in steps]
        yr, sr, _ = oracle.decode(d, sbf, wl.bf16_bits(inp["conv_w"]), inp["A_log"].numpy(), inp["dt_bias"].numpy(),
                                  wl.bf16_bits(inp["conv_state"]), inp["state"].numpy().astype(np.float64))
        q.put(bool(np.array_equal(y_full, np.stack(yr)) and np.array_equal(s_full, sr)))
    dist.barrier()
    dist.destroy_process_group()


def test_batch_split_over_two_ranks_equals_one_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    assert q.get(timeout=10) is True
