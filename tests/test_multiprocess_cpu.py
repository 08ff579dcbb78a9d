"""The benchmark's multi-process path on CPU (gloo, world size 2): the barrier and the
max-over-ranks timing reduction, and the reference arm under torchrun, where rank 0 alone runs
and prints one line and the other rank exits 0.  Replicas share nothing on the data path, so
these host-side pieces are the whole N>1 path."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    got = bench.max_over_ranks(1.5 + rank, world, torch.device("cpu"))
    bench.barrier(world)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(repr(got))


def test_max_over_ranks_gloo_two_ranks(tmp_path):
    mp.start_processes(_rank_main, args=(2, free_port(), str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        assert float((tmp_path / f"rank{r}.txt").read_text()) == 2.5


def test_reference_arm_under_torchrun_two_ranks():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py",
           "--impl", "reference", "--config", "1", "--gpus", "2", "--steps", "2", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def _syncbn_rank_main(rank, world, port, out_dir):
    """One rank of the synchronised-BN host path: this rank's share of the batch, its moments and
    backward sums (computed here by the oracle, standing in for the GPU half-calls), then the
    binding's two collectives."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import numpy as np

    import oracle
    from conv_batchnorm_relu_gb300 import cbr
    from conv_batchnorm_relu_gb300.inputs import CONFIGS, make_inputs

    dist.init_process_group("gloo", rank=rank, world_size=world)
    spec = CONFIGS[1].with_(n=4)
    inp = {k: v.double().numpy() for k, v in make_inputs(spec, 4242).items()}
    share = slice(rank * 2, rank * 2 + 2)               # rank r holds images 2r, 2r+1
    z = oracle.conv2d_fwd(inp["x"][share], inp["w"], spec.stride, spec.pad).reshape(-1, spec.c_out)
    mean, var = oracle.bn_batch_stats(z)
    mom = torch.tensor(np.concatenate([mean, var * z.shape[0], [z.shape[0]]]), dtype=torch.float32)
    gathered = cbr.gather_moments(mom)
    g = inp["dy"][share].reshape(-1, spec.c_out)  # mask-free sums suffice to check the reduction
    sums = torch.tensor(np.concatenate([g.sum(0), (g * z).sum(0)]), dtype=torch.float32)
    total = cbr.reduce_sums(sums)
    dist.destroy_process_group()
    np.save(os.path.join(out_dir, f"gathered{rank}.npy"), gathered.numpy())
    np.save(os.path.join(out_dir, f"total{rank}.npy"), total.numpy())


def test_syncbn_collectives_gloo_two_ranks(tmp_path):
    """Both ranks receive every rank's moments in rank order and the element-wise total of the
    backward sums; merging the gathered moments in that order reproduces the whole batch's
    two-pass mean and variance (the oracle on all four images)."""
    import numpy as np

    import oracle
    from conv_batchnorm_relu_gb300.inputs import CONFIGS, make_inputs

    mp.start_processes(_syncbn_rank_main, args=(2, free_port(), str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    spec = CONFIGS[1].with_(n=4)
    inp = {k: v.double().numpy() for k, v in make_inputs(spec, 4242).items()}
    K = spec.c_out
    g0, g1 = (np.load(tmp_path / f"gathered{r}.npy") for r in range(2))
    assert np.array_equal(g0, g1) and g0.shape == (2, 2 * K + 1)
    per_rank = []
    for r in range(2):
        z = oracle.conv2d_fwd(inp["x"][2 * r:2 * r + 2], inp["w"], spec.stride, spec.pad).reshape(-1, K)
        per_rank.append(z)
        assert np.allclose(g0[r, :K], z.mean(0), rtol=1e-6, atol=1e-6)   # rank order kept
    # Chan's merge of the two sets, as cbr_forward_train_finish does on the device
    n_a, n_b = g0[0, -1], g0[1, -1]
    d = g0[1, :K] - g0[0, :K]
    mean = g0[0, :K] + d * n_b / (n_a + n_b)
    var = (g0[0, K:2 * K] + g0[1, K:2 * K] + d * d * n_a * n_b / (n_a + n_b)) / (n_a + n_b)
    z_all = oracle.conv2d_fwd(inp["x"], inp["w"], spec.stride, spec.pad).reshape(-1, K)
    want_mean, want_var = oracle.bn_batch_stats(z_all)
    assert np.allclose(mean, want_mean, rtol=1e-5, atol=1e-5)
    assert np.allclose(var, want_var, rtol=1e-5)
    t0, t1 = (np.load(tmp_path / f"total{r}.npy") for r in range(2))
    g_all = inp["dy"].reshape(-1, K)
    want = np.concatenate([g_all.sum(0), (g_all * z_all).sum(0)])
    assert np.array_equal(t0, t1) and np.allclose(t0, want, rtol=1e-5, atol=1e-4)
