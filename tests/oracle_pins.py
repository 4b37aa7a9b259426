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


# ------------------------------------------- sliding window and sinks ----
# Readings: "2026-05-28_STATUS.md" items D3/D4 (window mask, with causal) and
# D5c (one softmax over the scores and the sink); see oracle.c.


def pin_window_covering_all_keys(attn):
    """A window wider than every row's key range changes nothing (exactly)."""
    rng = np.random.default_rng(21)
    B, Hq, Hkv, Sq, Sk, d = 2, 2, 1, 7, 9, 3
    q, k, v = (_rand(rng, s) for s in ((B, Hq, Sq, d), (B, Hkv, Sk, d), (B, Hkv, Sk, d)))
    for causal in (False, True):
        o0, l0 = attn(q, k, v, scale=0.7, causal=causal, seqlens_k=[9, 5])
        o1, l1 = attn(q, k, v, scale=0.7, causal=causal, seqlens_k=[9, 5], window=Sk + Sq)
        _close(o1, o0, 0, "wide window O")
        _close(l1, l0, 0, "wide window LSE")


def pin_window_one_is_own_key(attn):
    """Causal with a window of one key: row i sees only key p = i + L - Sq, so
    O_i = v_p and LSE_i = scale q_i . k_p; rows with p < 0 see nothing."""
    rng = np.random.default_rng(22)
    B, Hq, Hkv, Sq, Sk, d = 2, 2, 2, 6, 6, 4
    q, k, v = (_rand(rng, s) for s in ((B, Hq, Sq, d), (B, Hkv, Sk, d), (B, Hkv, Sk, d)))
    lens = [6, 3]
    o, lse = attn(q, k, v, scale=0.3, causal=True, seqlens_k=lens, window=1)
    for b in range(B):
        for h in range(Hq):
            for i in range(Sq):
                p = i + lens[b] - Sq
                if p < 0:
                    _close(o[b, h, i], np.zeros(d), 0, "empty row O")
                    assert lse[b, h, i] == -math.inf, "empty row LSE"
                else:
                    _close(o[b, h, i], v[b, h, p], 1e-15, "own-key O")
                    _close(lse[b, h, i], 0.3 * float(np.dot(q[b, h, i], k[b, h, p])), 1e-14,
                           "own-key LSE")


def pin_window_equals_sliced_keys(attn):
    """Row i with window W sees keys [p - W + 1, p] (causal) or [p - W + 1, L)
    (not causal), p = i + L - Sq: the same as the unwindowed definition on K, V
    sliced to those keys, for that row alone."""
    rng = np.random.default_rng(23)
    B, Hq, Hkv, Sq, Sk, d = 1, 2, 1, 5, 12, 3
    q, k, v = (_rand(rng, s) for s in ((B, Hq, Sq, d), (B, Hkv, Sk, d), (B, Hkv, Sk, d)))
    L, W = 10, 4
    for causal in (False, True):
        o, lse = attn(q, k, v, scale=0.9, causal=causal, seqlens_k=[L], window=W)
        for i in range(Sq):
            p = i + L - Sq
            lo, hi = max(0, p - W + 1), (p + 1 if causal else L)
            ks, vs = k[:, :, lo:hi], v[:, :, lo:hi]
            o1, l1 = attn(q[:, :, i:i + 1], np.ascontiguousarray(ks), np.ascontiguousarray(vs),
                          scale=0.9)
            _close(o[:, :, i], o1[:, :, 0], 1e-14, f"sliced window O row {i}")
            _close(lse[:, :, i], l1[:, :, 0], 1e-14, f"sliced window LSE row {i}")


def pin_sink_zero_query(attn):
    """Q = 0: every score is 0, so O = sum_j v_j / (e^sigma + n) and
    LSE = ln(e^sigma + n) (n visible keys)."""
    rng = np.random.default_rng(24)
    B, Hq, Hkv, Sq, Sk, d = 1, 3, 1, 2, 5, 3
    q = np.zeros((B, Hq, Sq, d))
    k, v = _rand(rng, (B, Hkv, Sk, d)), _rand(rng, (B, Hkv, Sk, d))
    sig = np.array([-2.0, 0.5, 3.0])
    o, lse = attn(q, k, v, scale=1.0, sinks=sig)
    for h in range(Hq):
        den = math.exp(sig[h]) + Sk
        _close(o[0, h], np.broadcast_to(v[0, 0].sum(axis=0) / den, (Sq, d)), 1e-15, "sink O")
        _close(lse[0, h], np.full(Sq, math.log(den)), 1e-15, "sink LSE")


def pin_sink_is_a_zero_value_key(attn):
    """A sink equals one more key whose score is exactly sigma and whose value
    row is zero."""
    rng = np.random.default_rng(25)
    B, H, Sq, Sk, d = 1, 2, 1, 6, 4
    q = _rand(rng, (B, H, Sq, d), 0.5, 1.0)
    k, v = _rand(rng, (B, H, Sk, d)), _rand(rng, (B, H, Sk, d))
    sig = np.array([0.75, -1.25])
    scale = 0.5
    k2 = np.concatenate([k, np.zeros((B, H, 1, d))], axis=2)
    v2 = np.concatenate([v, np.zeros((B, H, 1, d))], axis=2)
    for h in range(H):
        k2[0, h, Sk, 0] = sig[h] / (scale * q[0, h, 0, 0])   # score = sigma (to rounding)
    o, lse = attn(q, k, v, scale=scale, sinks=sig)
    o2, l2 = attn(q, k2, v2, scale=scale)
    _close(o, o2, 1e-14, "sink as a key O")
    _close(lse, l2, 1e-14, "sink as a key LSE")


def pin_sink_extremes(attn):
    """sigma = -inf is no sink (exactly); sigma = 1000 takes all the weight
    (O = 0, LSE = 1000); a row without keys has LSE = sigma."""
    rng = np.random.default_rng(26)
    B, Hq, Hkv, Sq, Sk, d = 2, 2, 1, 4, 4, 3
    q, k, v = (_rand(rng, s) for s in ((B, Hq, Sq, d), (B, Hkv, Sk, d), (B, Hkv, Sk, d)))
    o0, l0 = attn(q, k, v, scale=0.8, causal=True, seqlens_k=[4, 2])
    o1, l1 = attn(q, k, v, scale=0.8, causal=True, seqlens_k=[4, 2],
                  sinks=[-math.inf, -math.inf])
    _close(o1, o0, 0, "-inf sink O")
    _close(l1, l0, 0, "-inf sink LSE")
    o2, l2 = attn(q, k, v, scale=0.8, causal=True, seqlens_k=[4, 2], sinks=[1000.0, 1000.0])
    _close(o2, np.zeros_like(o2), 1e-300, "huge sink O")
    _close(l2, np.full_like(l2, 1000.0), 1e-12, "huge sink LSE")
    o3, l3 = attn(q, k, v, scale=0.8, causal=True, seqlens_k=[4, 2], sinks=[0.25, -0.5])
    # batch entry 1 has L = 2 < Sq = 4: rows 0 and 1 see no key
    _close(o3[1, :, :2], np.zeros((Hq, 2, d)), 0, "sink empty-row O")
    _close(l3[1, :, :2], np.array([[0.25, 0.25], [-0.5, -0.5]]), 0, "sink empty-row LSE")


ALL_PINS = [pin_golden_closed_forms, pin_zero_query_gives_mean_of_values,
            pin_single_key, pin_causal_first_row, pin_shift_invariance,
            pin_bruteforce_tiny, pin_library_sdpa, pin_permutation_invariance,
            pin_gqa_equals_repeated_heads, pin_bf16_decoding, pin_row_subset,
            pin_window_covering_all_keys, pin_window_one_is_own_key,
            pin_window_equals_sliced_keys, pin_sink_zero_query,
            pin_sink_is_a_zero_value_key, pin_sink_extremes]
