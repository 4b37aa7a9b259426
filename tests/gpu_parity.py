"""Shared helpers of the GPU parity tests: run the CUDA path and the oracle on
the very same seeded inputs and compare element by element."""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle
from attention_forward_blackwell_gb300 import inputs

# Tolerances of the parity gate (max-abs over all compared elements).
TOL_O = 2e-2
TOL_LSE = 1e-3
THREADS = max(1, min(32, os.cpu_count() or 1))


def oracle_for(x: inputs.AttentionInputs, scale, causal, rows=None):
    lens = None if x.seqlens_k is None else x.seqlens_k.cpu().tolist()
    return oracle.attention_fwd(inputs.bf16_bits(x.q), inputs.bf16_bits(x.k),
                                inputs.bf16_bits(x.v), scale=scale, causal=causal,
                                seqlens_k=lens, rows=rows, threads=THREADS)


def max_abs(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    same_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        d = np.where(same_inf, 0.0, np.abs(a - b))
    if np.isnan(d).any():
        return float("nan")
    return float(d.max()) if d.size else 0.0


def compare(o_gpu, lse_gpu, o_ref, lse_ref, what="", tol_o=TOL_O, tol_lse=TOL_LSE):
    """o_gpu/lse_gpu: torch (any device); o_ref/lse_ref: float64 numpy of the
    same element count.  Asserts the gate, returns (err_o, err_lse, cos)."""
    og = o_gpu.detach().float().cpu().numpy().astype(np.float64).reshape(o_ref.shape)
    lg = lse_gpu.detach().cpu().numpy().astype(np.float64).reshape(lse_ref.shape)
    eo = max_abs(og, o_ref)
    el = max_abs(lg, lse_ref)
    a, b = og.reshape(-1), o_ref.reshape(-1)
    den = np.linalg.norm(a) * np.linalg.norm(b)
    cos = float(a @ b / den) if den > 0 else 1.0
    print(f"{what}: max|dO|={eo:.3e} max|dLSE|={el:.3e} cos(O)={cos:.7f}")
    assert eo == eo and eo <= tol_o, f"{what}: O error {eo}"
    assert el == el and el <= tol_lse, f"{what}: LSE error {el}"
    return eo, el, cos


def sample_rows(B, Hq, Sq, n_random=384, seed=0):
    """Flattened row ids: tile edges of a few heads plus uniform samples."""
    rng = np.random.default_rng(seed)
    rows = set()
    edges = [0, 1, 127, 128, 255, 256, Sq // 2, Sq - 129, Sq - 128, Sq - 2, Sq - 1]
    for (b, h) in [(0, 0), (B - 1, Hq - 1), (B // 2, Hq // 2)]:
        for i in edges:
            if 0 <= i < Sq:
                rows.add((b * Hq + h) * Sq + i)
    total = B * Hq * Sq
    rows.update(int(r) for r in rng.integers(0, total, size=min(n_random, total)))
    return np.array(sorted(rows), dtype=np.int64)


def check_device_error():
    from attention_forward_blackwell_gb300 import binding
    st, word = binding.get_device_error_word()
    assert st == binding.FA_OK, f"device error {binding.status_string(st)} word=0x{word:x}"


def free_cuda():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def to_pages(k, v, lens, page_size, seed, spare=3):
    """Scatter K, V [B, Hkv, Sk, d] into shuffled pages [num_pages, Hkv, P, d].
    Rows past each length and every unused page hold NaN (never read)."""
    B, Hkv, Sk, d = k.shape
    max_pages = math.ceil(Sk / page_size)
    need = [math.ceil(L / page_size) for L in lens]
    num_pages = sum(need) + spare
    perm = np.random.default_rng(seed).permutation(num_pages)
    kc = torch.full((num_pages, Hkv, page_size, d), float("nan"), device=k.device,
                    dtype=k.dtype)
    vc = kc.clone()
    table = torch.zeros(B, max_pages, dtype=torch.int32)
    nxt = 0
    for b in range(B):
        for i in range(need[b]):
            pg = int(perm[nxt])
            nxt += 1
            table[b, i] = pg
            lo, hi = i * page_size, min((i + 1) * page_size, lens[b])
            kc[pg, :, :hi - lo] = k[b, :, lo:hi]
            vc[pg, :, :hi - lo] = v[b, :, lo:hi]
    return kc, vc, table.cuda(), num_pages
