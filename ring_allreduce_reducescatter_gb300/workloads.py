"""Seeded synthetic workloads of the ring collectives.

This module describes the benchmark and test workloads (shapes, formats,
value distributions, seeds) and generates their inputs.  It contains none of
the collectives' arithmetic, so the CUDA path and the CPU oracle can both be
fed from it without sharing any of the method.

Workloads (values drawn in binary32 on the given device with a
``torch.Generator`` seeded ``1000 * workload_id + r`` for rank r, then rounded
to the storage format by torch's round-to-nearest-even conversion):

  1  AllReduce / ReduceScatter / AllGather, R = 4, binary32, N = 1,048,576,
     uniform in [-1, 1)
  2  AllReduce, R = 8, binary16 storage and wire, per-rank messages of 1, 16,
     128 and 512 MiB (N = 524,288 ... 268,435,456), normal with sigma 1e-3
     (gradient-like; about 5 % of the values are binary16 subnormals)
  3  AllReduce, R = 8, binary32 storage on a bfloat16 wire, N = 50,000,017
     (prime: chunks of 6,250,002 x 7 and 6,250,003), standard normal
  4  two-level AllReduce, R = 16 = 2 groups x 8, binary32, N = 16,777,216
     (64 MiB per rank), uniform in [-1, 1)
  5  fusion-bucket AllReduce, R = 8, bfloat16 storage and wire: the gradients
     of 32 layers of a 4096-hidden decoder (q, k, v, o 4096x4096; gate, up
     4096x11008; down 11008x4096) packed flat, in that order, into 256 MiB
     buckets: 48 buckets of 134,217,728 elements and one of 33,554,432;
     normal with sigma 1e-2; bucket b of rank r seeded 5000 + 100 b + r.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional

import torch

MIB = 1 << 20


@dataclass(frozen=True)
class Workload:
    wid: int
    name: str
    op: str            # "allreduce" | "reduce_scatter" | "allgather"
    R: int
    dtype: torch.dtype  # storage format
    wire: Optional[str]  # None = same as storage
    count: int
    dist: str          # "uniform" | "normal" | "grad1e-3" | "grad1e-2"
    group_size: int = 0


def config1(op: str = "allreduce") -> Workload:
    return Workload(1, f"{op} R=4 fp32 N=1048576", op, 4, torch.float32, None, 1_048_576, "uniform")


def config2(msg_mib: int = 512, wire: Optional[str] = None) -> Workload:
    """Workload 2; wire="f32" is its binary32-accumulation variant (same inputs)."""
    count = msg_mib * MIB // 2
    how = "per-hop fp16" if wire is None else f"{wire} accumulation"
    return Workload(2, f"allreduce R=8 fp16 {how} msg={msg_mib}MiB", "allreduce", 8,
                    torch.float16, wire, count, "grad1e-3")


CONFIG2_SIZES_MIB = (1, 16, 128, 512)


def config3() -> Workload:
    return Workload(3, "allreduce R=8 fp32 storage bf16 wire N=50000017", "allreduce", 8,
                    torch.float32, "bf16", 50_000_017, "normal")


def config4() -> Workload:
    return Workload(4, "two-level allreduce R=16 (2x8) fp32 N=16777216", "allreduce", 16,
                    torch.float32, None, 16_777_216, "uniform", group_size=8)


def decoder_bucket_counts(layers: int = 32, hidden: int = 4096, ffn: int = 11008,
                          bucket_bytes: int = 256 * MIB, elem_bytes: int = 2) -> List[int]:
    """Element counts of the flat gradient buckets of workload 5 (tensors may
    straddle buckets; the last bucket holds the remainder)."""
    per_layer = 4 * hidden * hidden + 3 * hidden * ffn
    total = layers * per_layer
    per_bucket = bucket_bytes // elem_bytes
    counts = [per_bucket] * (total // per_bucket)
    if total % per_bucket:
        counts.append(total % per_bucket)
    return counts


def config5(bucket: int) -> Workload:
    counts = decoder_bucket_counts()
    return Workload(5, f"bucket {bucket} of {len(counts)}: allreduce R=8 bf16 per-hop bf16",
                    "allreduce", 8, torch.bfloat16, None, counts[bucket], "grad1e-2")


def seed(wid: int, r: int, bucket: int = 0) -> int:
    return 1000 * wid + 100 * bucket + r


def rank_values(wid: int, r: int, count: int, dtype: torch.dtype, dist: str, device,
                bucket: int = 0, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Rank r's input vector of a workload (deterministic for a given device type)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed(wid, r, bucket))
    if dist == "uniform":
        x = torch.rand(count, generator=g, device=device, dtype=torch.float32).mul_(2).sub_(1)
    elif dist == "normal":
        x = torch.randn(count, generator=g, device=device, dtype=torch.float32)
    elif dist == "grad1e-3":
        x = torch.randn(count, generator=g, device=device, dtype=torch.float32).mul_(1e-3)
    elif dist == "grad1e-2":
        x = torch.randn(count, generator=g, device=device, dtype=torch.float32).mul_(1e-2)
    else:
        raise ValueError(dist)
    if out is not None:
        out.copy_(x)
        return out
    return x.to(dtype)


def inputs(w: Workload, device, bucket: int = 0, lengths: Optional[List[int]] = None) -> List[torch.Tensor]:
    """The R input vectors of workload w; ``lengths`` overrides the per-rank
    lengths (the AllGather inputs are the chunks, whose lengths the caller
    takes from the chunk table)."""
    lengths = lengths if lengths is not None else [w.count] * w.R
    return [rank_values(w.wid, r, lengths[r], w.dtype, w.dist, device, bucket) for r in range(w.R)]
