"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws random tensors with
the shapes, dtypes and value distributions of the workloads (bf16 values from
a standard normal, optionally scaled; integer key lengths drawn uniformly).
Both the CUDA path and the oracle are fed the very same tensors.

Seeds follow one fixed recipe: q = 1000 + tag, k = 2000 + tag, v = 3000 + tag,
key lengths = 4000 (+ tag for non-default cases), where ``tag`` identifies the
workload.  Generation runs on the requested device with a torch.Generator of
that device, so a given (tag, device type) pair always yields the same data.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch


@dataclass
class AttentionInputs:
    q: torch.Tensor                    # [B, Hq, Sq, d] bf16
    k: torch.Tensor                    # [B, Hkv, Sk, d] bf16
    v: torch.Tensor                    # [B, Hkv, Sk, d] bf16
    seqlens_k: Optional[torch.Tensor]  # [B] int32 or None


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, seed, device="cpu", scale=1.0):
    """bf16(scale * N(0, 1)) drawn from a generator seeded with ``seed``."""
    x = torch.randn(shape, generator=_gen(device, seed), device=device,
                    dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(torch.bfloat16)


def uniform_lengths(batch, lo, hi, seed, device="cpu"):
    """int32 lengths drawn uniformly from the inclusive range [lo, hi]."""
    g = _gen("cpu", seed)
    lens = torch.randint(lo, hi + 1, (batch,), generator=g, dtype=torch.int64)
    return lens.to(torch.int32).to(device)


def make_inputs(B, Hq, Hkv, Sq, Sk, d, *, tag, device="cpu", k_scale=1.0,
                lengths=None, length_seed=4000):
    """Q, K, V ~ bf16(N(0,1)) (K optionally scaled) plus optional key lengths.

    ``lengths``: None (every batch entry uses all Sk keys), a (lo, hi) pair to
    draw lengths uniformly from [lo, hi], or an explicit sequence of ints.
    """
    q = randn_bf16((B, Hq, Sq, d), 1000 + tag, device)
    k = randn_bf16((B, Hkv, Sk, d), 2000 + tag, device, scale=k_scale)
    v = randn_bf16((B, Hkv, Sk, d), 3000 + tag, device)
    sl = None
    if lengths is not None:
        if isinstance(lengths, tuple) and len(lengths) == 2:
            sl = uniform_lengths(B, lengths[0], lengths[1], length_seed, device)
        else:
            sl = torch.tensor(list(lengths), dtype=torch.int32, device=device)
    return AttentionInputs(q, k, v, sl)


def poison_beyond_lengths(t, seqlens_k, value=float("nan")):
    """Fill key rows j >= L_b of a [B, H, Sk, d] tensor with ``value``.

    Used by tests to prove that rows past each sequence's length are never
    read: any read of them would surface as a non-finite output.
    """
    B, _, Sk, _ = t.shape
    lens = seqlens_k.to("cpu").tolist()
    for b in range(B):
        L = max(0, min(int(lens[b]), Sk))
        if L < Sk:
            t[b, :, L:, :] = value
    return t


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 array of its bit patterns (host copy)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
