"""The staged collectives across processes on the GPU: ranks as separate
processes on one GPU, each staging buffer a device allocation that the other
processes map through CUDA IPC, the gather or the fixed-order fold the
library's kernel over the mapped buffers.  Every rank's output is compared
with the oracle, bit for bit (NaN by class), over several epochs, at aligned,
unaligned and multi-tile sizes and for every element type.

No kernel waits for another process: the handshakes are host barriers (the
node-local shared-memory counters, and the gloo process group's monitored
barrier), so the processes' launches never depend on one another.
The failure cases (a rank that never arrives or dies) are covered on CPU.

Page, by title: "perf(cuda): vectorize the deterministic all-gather copy and
right-size its single-block path" (the author's replies: the collective over
CUDA IPC, stage, gather, complete).
"""
from __future__ import annotations

import json
import os
import shutil
import socket
import subprocess

import numpy as np
import pytest
import torch.multiprocessing as mp

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

SIZES = [4099, 1 << 20, (3 << 20) + 5]


def _port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, handshake, outdir, op="gather"):
    import torch
    import torch.distributed as dist

    import reduce_copy_rank_gb300 as dc
    from reduce_copy_rank_gb300.ipc import CudaIpcTransport, StagedAllGather

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    res = {"rank": rank, "ok": [], "launches": 0}
    try:
        n0 = dc.launch_count()
        if op == "gathermany":
            _gather_many(rank, world, handshake, res)
            res["launches"] = dc.launch_count() - n0
            dc.check_device()
            return
        if op != "gather":
            _reductions(rank, world, handshake, op, res)
            res["launches"] = dc.launch_count() - n0
            dc.check_device()
            return
        for si, B in enumerate(SIZES):
            coll = StagedAllGather(None, B, CudaIpcTransport(), timeout=30.0, handshake=handshake)
            for epoch in range(1, 4):
                payloads = [W.random_bytes(W.seed_for(3, 900 + 10 * si + epoch), q, B)
                            for q in range(world)]
                mine = torch.from_numpy(payloads[rank]).cuda()
                out = torch.full((world * B,), 0xA5, dtype=torch.uint8, device="cuda")
                coll.all_gather(mine, out)
                res["ok"].append(bool(np.array_equal(out.cpu().numpy(), oracle.all_gather(payloads))))
            coll.close()
        res["launches"] = dc.launch_count() - n0
        dc.check_device()
    except Exception as e:  # reported through the result file
        res["error"] = repr(e)
    finally:
        with open(os.path.join(outdir, f"r{rank}.json"), "w") as fh:
            json.dump(res, fh)
        dist.destroy_process_group()


MANY_SIZES = [0, 1, 15, 4099, 256, 70001, (1 << 20) + 3]


def _gather_many(rank, world, handshake, res):
    """all_gather_many over CUDA IPC (one staging buffer per rank), three
    epochs, against the oracle."""
    import torch

    from reduce_copy_rank_gb300.ipc import CudaIpcTransport, StagedAllGatherMany

    coll = StagedAllGatherMany(None, MANY_SIZES, CudaIpcTransport(), timeout=30.0, handshake=handshake)
    for epoch in range(1, 4):
        tensors = [[W.random_bytes(W.seed_for(5, 940 + epoch), q, B, tensor=t) for q in range(world)]
                   for t, B in enumerate(MANY_SIZES)]
        mine = [torch.from_numpy(tensors[t][rank]).cuda() for t in range(len(MANY_SIZES))]
        outs = [torch.full((world * B,), 0xA5, dtype=torch.uint8, device="cuda") for B in MANY_SIZES]
        coll.all_gather_many(mine, outs)
        want = oracle.all_gather_many(tensors)
        res["ok"].append(all(bool(np.array_equal(o.cpu().numpy(), w)) for o, w in zip(outs, want)))
    coll.close()


RED_CASES = [("bf16", "linear", 4099), ("f16", "tree", 1 << 18), ("f32", "linear", (1 << 18) + 3)]


def _reductions(rank, world, handshake, op, res):
    """all_reduce / reduce_scatter over CUDA IPC for each (dtype, order, n),
    three epochs each, against the oracle's fold and the single-process
    entry point's output for this rank."""
    import torch

    from gpu_util import NP_OF, is_nan_typed, torch_dtype, typed_bits, typed_tensor
    from reduce_copy_rank_gb300.ipc import CudaIpcTransport, StagedAllReduce, StagedReduceScatter

    for ci, (dtype, order, n) in enumerate(RED_CASES):
        if op == "allreduce":
            coll = StagedAllReduce(None, n, dtype, CudaIpcTransport(), order=order, timeout=30.0,
                                   handshake=handshake)
            total = n
        else:
            coll = StagedReduceScatter(None, n, dtype, CudaIpcTransport(), order=order, timeout=30.0,
                                       handshake=handshake)
            total = world * n
        for epoch in range(1, 4):
            cols = []
            for q in range(world):
                g = np.random.default_rng(np.random.SeedSequence([W.seed_for(4, 930 + 10 * ci + epoch), q]))
                hi = np.iinfo(NP_OF[dtype]).max
                cols.append(g.integers(0, hi, total, dtype=np.uint64).astype(NP_OF[dtype]))
            mine = typed_tensor(cols[rank], dtype)
            out = torch.empty(n, dtype=torch_dtype(dtype), device="cuda")
            if op == "allreduce":
                coll.all_reduce(mine, out)
                want = oracle.all_reduce(cols, dtype, order)
            else:
                coll.reduce_scatter(mine, out)
                want = oracle.reduce_scatter(cols, dtype, order)[rank]
            got, w = typed_bits(out, dtype), want.view(NP_OF[dtype])
            gn, wn = is_nan_typed(got, dtype), is_nan_typed(w, dtype)  # NaN compared by class
            res["ok"].append(bool(np.array_equal(gn, wn) and np.array_equal(got[~wn], w[~wn])))
        coll.close()


def _compute_mode_default():
    smi = shutil.which("nvidia-smi")
    if smi is None:
        return True
    try:
        out = subprocess.run([smi, "--query-gpu=compute_mode", "--format=csv,noheader", "-i", "0"],
                             capture_output=True, text=True, timeout=30).stdout.strip()
    except (OSError, subprocess.SubprocessError):
        return True
    return out in ("", "Default")


@pytest.mark.parametrize("handshake", ["shm", "gloo"])
@pytest.mark.parametrize("world", [2, 3])
def test_staged_all_gather_over_cuda_ipc(world, handshake, tmp_path):
    if not _compute_mode_default():
        pytest.skip("GPU 0 is not in the default compute mode: one process per GPU only")
    mp.spawn(_worker, args=(world, _port(), handshake, str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        res = json.load(open(tmp_path / f"r{r}.json"))
        assert "error" not in res, res
        assert res["ok"] == [True] * (3 * len(SIZES)), res
        assert res["launches"] == 2 * 3 * len(SIZES), res  # per epoch: the staging copy and the gather


@pytest.mark.parametrize("world", [2, 3])
def test_staged_all_gather_many_over_cuda_ipc(world, tmp_path):
    if not _compute_mode_default():
        pytest.skip("GPU 0 is not in the default compute mode: one process per GPU only")
    mp.spawn(_worker, args=(world, _port(), "shm", str(tmp_path), "gathermany"), nprocs=world, join=True)
    for r in range(world):
        res = json.load(open(tmp_path / f"r{r}.json"))
        assert "error" not in res, res
        assert res["ok"] == [True] * 3, res
        assert res["launches"] == 2 * 3, res  # per epoch: one staging launch, one gather launch


@pytest.mark.parametrize("op", ["allreduce", "reducescatter"])
@pytest.mark.parametrize("world", [2, 3])
def test_staged_reductions_over_cuda_ipc(world, op, tmp_path):
    if not _compute_mode_default():
        pytest.skip("GPU 0 is not in the default compute mode: one process per GPU only")
    mp.spawn(_worker, args=(world, _port(), "shm", str(tmp_path), op), nprocs=world, join=True)
    for r in range(world):
        res = json.load(open(tmp_path / f"r{r}.json"))
        assert "error" not in res, res
        assert res["ok"] == [True] * (3 * len(RED_CASES)), res
        assert res["launches"] == 2 * 3 * len(RED_CASES), res  # per epoch: the staging copy and the fold
