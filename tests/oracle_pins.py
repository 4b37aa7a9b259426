"""Checks that pin the fp64 oracle to facts fixed outside the oracle itself.

Each ``pin_*`` function takes ``attn`` -- a callable with the signature of
``oracle.attention_fwd`` -- and raises AssertionError if the result disagrees
with a closed form, a hand-derived golden value, an invariant of the
definition, a brute-force evaluation on tiny inputs, or an independent
library routine.  ``test_oracle_pins.py`` runs them against the oracle;
``test_oracle_mutations.py`` runs them against deliberately broken builds of
the oracle source and requires every planted mistake to be caught.

The definition being pinned: "b200-flash-attention4-planner", section E
step 1 (math semantics) and section A1 (the streamed result is O / row_sum,
i.e. softmax(scale * Q K^T + mask) V with LSE = ln sum exp(scale * q.k)).
"""
from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
_EXPR_NS = {"log": math.log, "exp": math.exp, "sqrt": math.sqrt,
            "inf": math.inf, "__builtins__": {}}


def parse_closed_forms(path=os.path.join(GOLDEN, "closed_forms.txt")):
    cases, cur = [], None
    for raw in open(path):
        line = raw.strip()
        if not line or line.startswith("#"):
            continue
        key, _, rest = line.partition(" ")
        if key == "case":
            cur = {"name": rest.strip()}
        elif key == "end":
            cases.append(cur)
            cur = None
        elif key == "shape":
            cur["shape"] = [int(x) for x in rest.split()]
        elif key == "seqlens":
            cur["seqlens"] = (None if rest.strip() == "none"
                              else [int(x) for x in rest.split()])
        elif key == "causal":
            cur["causal"] = bool(int(rest))
        else:
            cur[key] = np.array([float(eval(x, _EXPR_NS)) for x in rest.split()])
    return cases


def _rand(rng, shape, lo=-1.0, hi=1.0):
    return rng.uniform(lo, hi, size=shape).astype(np.float64)


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    same_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        diff = np.where(same_inf, 0.0, np.abs(a - b))
    assert not np.isnan(diff).any(), f"{what}: NaN"
    err = float(diff.max()) if diff.size else 0.0
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.1e}"


def visible_counts(B, Hq, Sq, Sk, causal, seqlens):
    """Number of visible keys per (b, h, i): the mask reading, written out."""
    n = np.zeros((B, Hq, Sq), dtype=np.int64)
    for b in range(B):
        L = Sk if seqlens is None else max(0, min(int(seqlens[b]), Sk))
        for i in range(Sq):
            last = L - 1
            if causal:
                last = min(last, i + L - Sq)
            n[b, :, i] = max(0, last + 1)
    return n


# ---------------------------------------------------------------- pins ----

def pin_golden_closed_forms(attn):
    for c in parse_closed_forms():
        B, Hq, Hkv, Sq, Sk, d = c["shape"]
        q = c["q"].reshape(B, Hq, Sq, d)
        k = c["k"].reshape(B, Hkv, Sk, d)
        v = c["v"].reshape(B, Hkv, Sk, d)
        o, lse = attn(q, k, v, scale=float(c["scale"][0]), causal=c["causal"],
                      seqlens_k=c["seqlens"])
        _close(o.reshape(-1), c["o"], 1e-12, c["name"] + " O")
        _close(lse.reshape(-1), c["lse"], 1e-12, c["name"] + " LSE")


def pin_zero_query_gives_mean_of_values(attn):
    """Q = 0 makes every score 0: O is the plain mean of the visible value
    rows and LSE = ln(number of visible keys)."""
    rng = np.random.default_rng(11)
    for (B, Hq, Hkv, Sq, Sk, d, causal, seqlens) in [
            (1, 2, 2, 9, 9, 4, True, None),
            (2, 4, 2, 5, 12, 3, True, [12, 7]),    # Sq < L: bottom-right shift
            (2, 3, 1, 7, 6, 2, False, [6, 2]),
            (1, 2, 1, 6, 4, 3, True, None),         # Sq > Sk: empty top rows
    ]:
        q = np.zeros((B, Hq, Sq, d))
        k = _rand(rng, (B, Hkv, Sk, d), -3, 3)
        v = _rand(rng, (B, Hkv, Sk, d), -3, 3)
        o, lse = attn(q, k, v, scale=0.7, causal=causal, seqlens_k=seqlens)
        n = visible_counts(B, Hq, Sq, Sk, causal, seqlens)
        G = Hq // Hkv
        for b in range(B):
            for h in range(Hq):
                for i in range(Sq):
                    cnt = n[b, h, i]
                    if cnt == 0:
                        exp_o, exp_l = np.zeros(d), -math.inf
                    else:
                        exp_o = v[b, h // G, :cnt, :].mean(axis=0)
                        exp_l = math.log(cnt)
                    _close(o[b, h, i], exp_o, 1e-12, "Q=0 mean O")
                    _close([lse[b, h, i]], [exp_l], 1e-12, "Q=0 LSE")


def pin_single_key(attn):
    """Sk = 1: the only key gets weight 1, so O = v_0 and LSE = scale*q.k_0."""
    rng = np.random.default_rng(12)
    B, Hq, Hkv, Sq, d = 2, 4, 2, 3, 5
    q = _rand(rng, (B, Hq, Sq, d), -2, 2)
    k = _rand(rng, (B, Hkv, 1, d), -2, 2)
    v = _rand(rng, (B, Hkv, 1, d), -2, 2)
    scale = 0.37
    o, lse = attn(q, k, v, scale=scale, causal=False)
    for b in range(B):
        for h in range(Hq):
            for i in range(Sq):
                _close(o[b, h, i], v[b, h // 2, 0], 1e-12, "Sk=1 O")
                dot = math.fsum(q[b, h, i, c] * k[b, h // 2, 0, c] for c in range(d))
                _close([lse[b, h, i]], [scale * dot], 1e-12, "Sk=1 LSE")


def pin_causal_first_row(attn):
    """Causal with Sq = Sk: row 0 sees key 0 only, so O_0 = v_0."""
    rng = np.random.default_rng(13)
    B, H, S, d = 1, 3, 10, 4
    q = _rand(rng, (B, H, S, d), -2, 2)
    k = _rand(rng, (B, H, S, d), -2, 2)
    v = _rand(rng, (B, H, S, d), -2, 2)
    o, lse = attn(q, k, v, scale=0.5, causal=True)
    for h in range(H):
        _close(o[0, h, 0], v[0, h, 0], 1e-12, "causal row 0 O")
        dot = math.fsum(q[0, h, 0, c] * k[0, h, 0, c] for c in range(d))
        _close([lse[0, h, 0]], [0.5 * dot], 1e-12, "causal row 0 LSE")


def pin_shift_invariance(attn):
    """Adding one vector u to every key adds scale*q_i.u to every score of row
    i: O is unchanged and LSE_i moves by exactly that amount.  Adding a
    constant c to every score (through an extra coordinate, q = c/scale and
    k = 1) leaves O unchanged and adds c to LSE."""
    rng = np.random.default_rng(14)
    B, Hq, Hkv, Sq, Sk, d = 2, 4, 2, 7, 11, 6
    q = _rand(rng, (B, Hq, Sq, d), -2, 2)
    k = _rand(rng, (B, Hkv, Sk, d), -2, 2)
    v = _rand(rng, (B, Hkv, Sk, d), -2, 2)
    u = _rand(rng, (d,), -3, 3)
    scale = 0.8
    for causal in (False, True):
        o1, l1 = attn(q, k, v, scale=scale, causal=causal, seqlens_k=[11, 9])
        o2, l2 = attn(q, k + u, v, scale=scale, causal=causal, seqlens_k=[11, 9])
        _close(o2, o1, 1e-11, "key shift O")
        _close(l2 - l1, scale * (q @ u), 1e-11, "key shift LSE")
        c = 2.5
        qa = np.concatenate([q, np.full((B, Hq, Sq, 1), c / scale)], axis=-1)
        ka = np.concatenate([k, np.ones((B, Hkv, Sk, 1))], axis=-1)
        va = np.concatenate([v, np.zeros((B, Hkv, Sk, 1))], axis=-1)
        o3, l3 = attn(qa, ka, va, scale=scale, causal=causal, seqlens_k=[11, 9])
        _close(o3[..., :d], o1, 1e-11, "score shift O")
        _close(l3 - l1, np.full_like(l1, c), 1e-11, "score shift LSE")


def pin_bruteforce_tiny(attn):
    """Tiny inputs with |s| <= 5: evaluate the definition directly (no max
    subtraction, exact fsum) with Python loops."""
    rng = np.random.default_rng(15)
    for (B, Hq, Hkv, Sq, Sk, d, causal, seqlens) in [
            (1, 1, 1, 3, 5, 2, False, None),
            (2, 2, 1, 4, 4, 3, True, None),
            (1, 4, 2, 2, 6, 2, True, [5]),
            (2, 2, 2, 5, 3, 1, True, [3, 2]),
    ]:
        q = _rand(rng, (B, Hq, Sq, d), -1.5, 1.5)
        k = _rand(rng, (B, Hkv, Sk, d), -1.5, 1.5)
        v = _rand(rng, (B, Hkv, Sk, d), -2, 2)
        scale = 0.9
        o, lse = attn(q, k, v, scale=scale, causal=causal, seqlens_k=seqlens)
        n = visible_counts(B, Hq, Sq, Sk, causal, seqlens)
        G = Hq // Hkv
        for b in range(B):
            for h in range(Hq):
                for i in range(Sq):
                    cnt = int(n[b, h, i])
                    s = [scale * math.fsum(q[b, h, i, c] * k[b, h // G, j, c]
                                           for c in range(d)) for j in range(cnt)]
                    assert all(abs(x) <= 5 for x in s)
                    if cnt == 0:
                        _close([lse[b, h, i]], [-math.inf], 0, "empty LSE")
                        _close(o[b, h, i], np.zeros(d), 0, "empty O")
                        continue
                    w = [math.exp(x) for x in s]
                    tot = math.fsum(w)
                    _close([lse[b, h, i]], [math.log(tot)], 1e-12, "brute LSE")
                    ref = [math.fsum(w[j] * v[b, h // G, j, c] for j in range(cnt)) / tot
                           for c in range(d)]
                    _close(o[b, h, i], ref, 1e-12, "brute O")


def pin_library_sdpa(attn):
    """Independent library routine: torch CPU float64 scaled_dot_product_attention
    with an explicit boolean mask and repeat_interleave for GQA, and
    torch.logsumexp of the masked scaled scores for LSE."""
    import torch
    rng = np.random.default_rng(16)
    for (B, Hq, Hkv, Sq, Sk, d, causal, seqlens) in [
            (1, 1, 1, 128, 128, 64, False, None),
            (2, 4, 2, 33, 47, 16, True, [47, 30]),
            (1, 8, 1, 20, 20, 8, True, None),
            (2, 6, 3, 17, 29, 12, False, [29, 5]),
    ]:
        q = _rand(rng, (B, Hq, Sq, d), -2, 2)
        k = _rand(rng, (B, Hkv, Sk, d), -2, 2)
        v = _rand(rng, (B, Hkv, Sk, d), -2, 2)
        scale = 1.0 / math.sqrt(d)
        o, lse = attn(q, k, v, scale=scale, causal=causal, seqlens_k=seqlens)
        G = Hq // Hkv
        tq = torch.from_numpy(q)
        tk = torch.from_numpy(k).repeat_interleave(G, dim=1)
        tv = torch.from_numpy(v).repeat_interleave(G, dim=1)
        mask = torch.zeros(B, 1, Sq, Sk, dtype=torch.bool)
        for b in range(B):
            L = Sk if seqlens is None else seqlens[b]
            for i in range(Sq):
                last = L - 1
                if causal:
                    last = min(last, i + L - Sq)
                mask[b, 0, i, :max(0, last + 1)] = True
        ref_o = torch.nn.functional.scaled_dot_product_attention(
            tq, tk, tv, attn_mask=mask, scale=scale)
        scores = (tq @ tk.transpose(-1, -2)) * scale
        scores = scores.masked_fill(~mask, -math.inf)
        ref_l = torch.logsumexp(scores, dim=-1)
        has = mask.any(dim=-1).expand(B, Hq, Sq)
        ref_o = torch.where(has[..., None], ref_o, torch.zeros_like(ref_o))
        _close(o, ref_o.numpy(), 1e-10, "sdpa O")
        _close(lse, ref_l.numpy(), 1e-10, "sdpa LSE")


def pin_permutation_invariance(attn):
    """Non-causal: permuting key rows together with their value rows is
    invisible to the result."""
    rng = np.random.default_rng(17)
    B, Hq, Hkv, Sq, Sk, d = 2, 2, 1, 5, 13, 4
    q = _rand(rng, (B, Hq, Sq, d), -2, 2)
    k = _rand(rng, (B, Hkv, Sk, d), -2, 2)
    v = _rand(rng, (B, Hkv, Sk, d), -2, 2)
    perm = rng.permutation(Sk)
    o1, l1 = attn(q, k, v, scale=0.6, causal=False)
    o2, l2 = attn(q, k[:, :, perm], v[:, :, perm], scale=0.6, causal=False)
    _close(o2, o1, 1e-12, "perm O")
    _close(l2, l1, 1e-12, "perm LSE")


def pin_gqa_equals_repeated_heads(attn):
    """GQA equals MHA over key/value heads repeated G times in place
    (repeat_interleave order: query head h uses kv head h // G)."""
    rng = np.random.default_rng(18)
    B, Hq, Hkv, Sq, Sk, d = 2, 6, 2, 4, 7, 3
    q = _rand(rng, (B, Hq, Sq, d), -2, 2)
    k = _rand(rng, (B, Hkv, Sk, d), -2, 2)
    v = _rand(rng, (B, Hkv, Sk, d), -2, 2)
    G = Hq // Hkv
    o1, l1 = attn(q, k, v, scale=0.5, causal=True)
    o2, l2 = attn(q, np.repeat(k, G, axis=1), np.repeat(v, G, axis=1),
                  scale=0.5, causal=True)
    _close(o1, o2, 0, "gqa O")
    _close(l1, l2, 0, "gqa LSE")


def pin_bf16_decoding(attn):
    """bf16 inputs are decoded exactly: with Sk = 1 and Q = 0 the output row
    is the value row itself, so known bit patterns must come back as their
    exact values."""
    patterns = {0x3F80: 1.0, 0xC020: -2.5, 0x3E20: 0.15625, 0x4780: 65536.0,
                0x0001: 2.0 ** -133, 0x8000: -0.0, 0x7F7F: 3.3895313892515355e38,
                0x3F81: 1.0078125}
    bits = np.array(list(patterns.keys()), dtype=np.uint16)
    d = bits.size
    q = np.zeros((1, 1, 1, d), dtype=np.uint16)
    k = np.zeros((1, 1, 1, d), dtype=np.uint16)
    v = bits.reshape(1, 1, 1, d)
    o, lse = attn(q, k, v, scale=1.0, causal=False)
    _close(o.reshape(-1), list(patterns.values()), 0, "bf16 decode")
    # a non-trivial score: q = 1.5 (0x3FC0), k = -0.75 (0xBF40) -> s = -1.125
    q1 = np.array([0x3FC0], dtype=np.uint16).reshape(1, 1, 1, 1)
    k1 = np.array([0xBF40], dtype=np.uint16).reshape(1, 1, 1, 1)
    v1 = np.array([0x4040], dtype=np.uint16).reshape(1, 1, 1, 1)
    o, lse = attn(q1, k1, v1, scale=2.0, causal=False)
    _close(lse.reshape(-1), [-2.25], 0, "bf16 score")
    _close(o.reshape(-1), [3.0], 0, "bf16 value")


def pin_row_subset(attn):
    """Computing a subset of rows gives exactly the corresponding full rows."""
    rng = np.random.default_rng(19)
    B, Hq, Hkv, Sq, Sk, d = 2, 4, 2, 9, 9, 3
    q = _rand(rng, (B, Hq, Sq, d))
    k = _rand(rng, (B, Hkv, Sk, d))
    v = _rand(rng, (B, Hkv, Sk, d))
    o, lse = attn(q, k, v, scale=0.5, causal=True, seqlens_k=[9, 4])
    rows = np.array([0, 5, 17, 40, 71, B * Hq * Sq - 1])
    os_, ls_ = attn(q, k, v, scale=0.5, causal=True, seqlens_k=[9, 4], rows=rows)
    _close(os_, o.reshape(-1, d)[rows], 0, "subset O")
    _close(ls_, lse.reshape(-1)[rows], 0, "subset LSE")


ALL_PINS = [pin_golden_closed_forms, pin_zero_query_gives_mean_of_values,
            pin_single_key, pin_causal_first_row, pin_shift_invariance,
            pin_bruteforce_tiny, pin_library_sdpa, pin_permutation_invariance,
            pin_gqa_equals_repeated_heads, pin_bf16_decoding, pin_row_subset]
