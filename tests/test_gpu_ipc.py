"""The staged all-gather across processes on the GPU: ranks as separate
processes on one GPU, each staging buffer a device allocation that the other
processes map through CUDA IPC, the gather the library's kernel over the
mapped buffers.  Every rank's output is compared with the oracle, bit for bit,
over several epochs and at aligned, unaligned and multi-tile sizes.

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


def _worker(rank, world, port, handshake, outdir):
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
        assert res["launches"] == 3 * len(SIZES), res  # one gather kernel per epoch
