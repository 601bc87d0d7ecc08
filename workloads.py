"""Seeded synthetic inputs for the deterministic gather / reduction workloads.

This module only draws random inputs and lists the workload shapes.  It holds
none of the method's arithmetic (no gather, no fold, no rounding of results),
so both the oracle side and the CUDA side may use it.

Workloads (KiB = 1024 B):

1. all-gather, P=2, 1 KiB per rank of BF16 bit patterns, 16-byte aligned
   (2 KiB output: the single-CTA path).
2. all-gather sweep, P=8 and P=2, per-rank sizes 1, 8, 32, 64, 128 KiB,
   1 MiB, 4 MiB of BF16 bit patterns, 16-byte aligned.  The per-rank sizes
   are the rows of the results table of "perf(cuda): vectorize the
   deterministic all-gather copy and right-size its single-block path"
   (section "Results"), plus 64 KiB from its H100 table.
3. misaligned / odd all-gather: P in {2, 3, 8}, uint8 payloads of 1, 15, 17,
   65535, 65537, 262145, 1048577 bytes, input and output base offsets in
   {0, 1, 8, 15} (all 16 pairs).
4. all_reduce BF16, P=8, per-rank element counts 131072 (256 KiB),
   262144 (512 KiB), 8x8192, 8627x8192, 16384x8192, values N(0,1).
5. reduce_scatter BF16, P=8, 16384x8192 per rank, values N(0,1); and
   all_gather_many of 6 tensors per rank, sizes {3 B, 4 KiB, 100000 B, 1 MiB,
   7 MiB+5 B, 32 MiB}, random bytes, P=8.

Seeds: ``0xDC0000 + 1000*config + case``; each rank r (and tensor t) draws
from ``numpy.random.default_rng(SeedSequence([seed, r, t]))``.  BF16 values
for the reductions are binary32 N(0,1) draws converted by torch's own
float->bfloat16 cast (a library conversion, not the method's rounding).
Full-size inputs may instead be drawn on the GPU with a torch generator
seeded from the same SeedSequence (``*_device`` helpers).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Iterator

import numpy as np

KiB = 1024
MiB = 1024 * 1024

# ---------------------------------------------------------------- shapes ---

CONFIG1 = dict(P=2, bytes_per_rank=1 * KiB)

CONFIG2_SIZES = [1 * KiB, 8 * KiB, 32 * KiB, 64 * KiB, 128 * KiB, 1 * MiB, 4 * MiB]
CONFIG2_PS = [8, 2]

CONFIG3_PS = [2, 3, 8]
CONFIG3_SIZES = [1, 15, 17, 65535, 65537, 262145, 1048577]
CONFIG3_OFFSETS = [0, 1, 8, 15]

CONFIG4_P = 8
CONFIG4_COUNTS = {
    "256KiB": 131072,
    "512KiB": 262144,
    "8x8192": 8 * 8192,
    "8627x8192": 8627 * 8192,
    "16384x8192": 16384 * 8192,
}

CONFIG5_RS = dict(P=8, rows=16384, cols=8192)
CONFIG5_MANY_P = 8
CONFIG5_MANY_SIZES = [3, 4 * KiB, 100000, 1 * MiB, 7 * MiB + 5, 32 * MiB]


def seed_for(config: int, case: int) -> int:
    return 0xDC0000 + 1000 * config + case


@dataclass(frozen=True)
class GatherCase:
    config: int
    case: int
    P: int
    bytes_per_rank: int
    in_offset: int = 0
    out_offset: int = 0

    @property
    def seed(self) -> int:
        return seed_for(self.config, self.case)


def config2_cases() -> list[GatherCase]:
    out, case = [], 0
    for P in CONFIG2_PS:
        for B in CONFIG2_SIZES:
            out.append(GatherCase(2, case, P, B))
            case += 1
    return out


def config3_cases() -> Iterator[GatherCase]:
    case = 0
    for P in CONFIG3_PS:
        for B in CONFIG3_SIZES:
            for io in CONFIG3_OFFSETS:
                for oo in CONFIG3_OFFSETS:
                    yield GatherCase(3, case, P, B, io, oo)
                    case += 1


# ------------------------------------------------------------ generators ---

def _rng(seed: int, rank: int, tensor: int = 0) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([seed, rank, tensor]))


def random_bytes(seed: int, rank: int, nbytes: int, tensor: int = 0) -> np.ndarray:
    """Uniform random bytes for one rank's payload."""
    return _rng(seed, rank, tensor).integers(0, 256, nbytes, dtype=np.uint8)


def random_bf16_patterns(seed: int, rank: int, count: int, tensor: int = 0) -> np.ndarray:
    """Uniform random 16-bit patterns (BF16 bit patterns, NaNs included)."""
    return _rng(seed, rank, tensor).integers(0, 65536, count, dtype=np.uint16)


def normal_bf16(seed: int, rank: int, count: int, tensor: int = 0) -> np.ndarray:
    """N(0,1) binary32 draws cast to BF16 by torch; returned as uint16 bits."""
    import torch

    f = _rng(seed, rank, tensor).standard_normal(count, dtype=np.float32)
    return torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def device_seed(seed: int, rank: int, tensor: int = 0) -> int:
    """A 63-bit integer seed for a torch generator, derived like the numpy
    streams so that each (workload, rank, tensor) gets its own stream."""
    s = np.random.SeedSequence([seed, rank, tensor]).generate_state(1, np.uint64)[0]
    return int(s & np.uint64(0x7FFF_FFFF_FFFF_FFFF))


def normal_bf16_device(seed: int, rank: int, count: int, device, tensor: int = 0):
    """N(0,1) BF16 drawn directly on ``device`` with a seeded torch generator
    (for the full-size reductions, where drawing on the host is slow).
    Returns a torch.bfloat16 tensor; the same seed gives the same values."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(device_seed(seed, rank, tensor))
    return torch.randn(count, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def normal_device(seed: int, rank: int, count: int, device, dtype, tensor: int = 0):
    """N(0,1) drawn on ``device`` in FP32 and cast by torch to ``dtype``
    (torch.bfloat16, torch.float16 or torch.float32); same stream as
    normal_bf16_device for the same seed, rank and tensor."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(device_seed(seed, rank, tensor))
    return torch.randn(count, generator=g, device=device, dtype=torch.float32).to(dtype)


def random_bytes_device(seed: int, rank: int, nbytes: int, device, tensor: int = 0):
    """Uniform random bytes drawn on ``device`` with a seeded torch generator."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(device_seed(seed, rank, tensor))
    return torch.randint(0, 256, (nbytes,), generator=g, device=device, dtype=torch.uint8)
