"""Parity tests whose inputs force the online softmax to move its basis.

The streaming recurrence ("b200-flash-attention4-planner" A1; E.8 says the
rescale of the old row_sum and O when a new maximum appears cannot be left
out) multiplies O and row_sum by alpha = 2^(m_old - m_new) whenever the
running max grows.  The kernels do it lazily: the basis moves only when a key
block's max exceeds it by more than 8 log2 units (prefill per 128-key block,
decode per 16-key slice of each warp).  With N(0,1) inputs that almost never
happens after the first block, so these tests build inputs where it must:

* a ramp on head coordinate 0 -- q[i, 0] = a_i (a per-row slope) and
  k[j, 0] = c * level(j) with c = 1 / (scale * log2 e) -- adds a_i * level(j)
  log2 units to every score, so each later key block's max beats the running
  max by about a_i;
* "mixed" slopes give some rows of every warp a steep ramp (rebase at every
  block), others a shallow one (rebase every few blocks, with P up to 2^8
  in between) and others a falling one (never), so a rebase factor applied to
  the wrong row shows up;
* a dominant key placed in a later key block (scores ~60 above the rest, K
  scaled by 8);
* a query block computed in pieces whose later piece holds the larger scores,
  so the merge of the pieces rescales the earlier ones.

Each test first checks on the host, from the inputs alone (fp64 scores of the
bf16 values and the kernels' block order), that the rows it compares really do
move their basis after their first block -- so the test cannot silently stop
exercising the path -- and then compares every output element with the fp64
oracle.
"""
import math

import numpy as np
import pytest
import torch

from gpu_parity import check_device_error, compare, free_cuda, oracle_for

pytestmark = pytest.mark.gpu

LOG2E = 1.4426950408889634
THRESHOLD = 8.0      # the kernels' lazy-rebase threshold, log2 units


@pytest.fixture(scope="module", autouse=True)
def built():
    from attention_forward_blackwell_gb300 import build
    build.build()
    yield
    free_cuda()


# ----------------------------------------------------------- inputs ----

def _row_slopes(B, Hq, Sq, mode, seed):
    """Per-row slope a_i (log2 units per ramp step), a pattern that changes
    from row to row inside every warp."""
    rng = np.random.default_rng(seed)
    n = B * Hq * Sq
    if mode == "steep":
        a = rng.uniform(14.0, 18.0, size=n)
    elif mode == "mixed":
        # a third falling, a third shallow (1.5-4), a third steep (10-16)
        kind = rng.integers(0, 3, size=n)
        a = np.where(kind == 0, rng.uniform(-3.0, -0.5, size=n),
                     np.where(kind == 1, rng.uniform(1.5, 4.0, size=n),
                              rng.uniform(10.0, 16.0, size=n)))
    else:
        raise ValueError(mode)
    return a.reshape(B, Hq, Sq)


def ramp_inputs(B, Hq, Hkv, Sq, Sk, d, *, tag, mode, step_keys, lengths=None, device="cuda"):
    """N(0,1) inputs plus a ramp on coordinate 0: score(i, j) gains
    a_i * floor(j / step_keys) log2 units.  V gets a per-128-key-block offset
    (-0.75, 0, +0.75 in turn) so that mixing up blocks shows in O."""
    from attention_forward_blackwell_gb300 import inputs
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=tag, device=device, lengths=lengths)
    scale = 1.0 / math.sqrt(d)
    c = 1.0 / (scale * LOG2E)
    a = _row_slopes(B, Hq, Sq, mode, seed=tag)
    x.q[..., 0] = torch.from_numpy(a).to(device=device, dtype=torch.float32).to(torch.bfloat16)
    lvl = torch.arange(Sk, device=device, dtype=torch.float32).div(step_keys).floor()
    x.k[..., 0] = (c * lvl).to(torch.bfloat16).expand(B, Hkv, Sk)
    off = (torch.arange(Sk, device=device) // 128 % 3 - 1).float() * 0.75
    x.v.copy_((x.v.float() + off[None, None, :, None]).to(torch.bfloat16))
    if lengths is not None:
        inputs.poison_beyond_lengths(x.k, x.seqlens_k)
        inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    return x, scale


# -------------------------------------------- host-side rebase schedule ----

def scores_log2(x, scale, causal):
    """fp64 scores in log2 units, [B, Hq, Sq, Sk], -inf where a key is not
    visible (key length, bottom-right causal alignment)."""
    q = x.q.float().cpu().double().numpy()
    k = x.k.float().cpu().double().numpy()
    B, Hq, Sq, _ = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    G = Hq // Hkv
    lens = [Sk] * B if x.seqlens_k is None else x.seqlens_k.cpu().tolist()
    t = np.empty((B, Hq, Sq, Sk))
    j = np.arange(Sk)[None, :]
    i = np.arange(Sq)[:, None]
    for b in range(B):
        L = max(0, min(int(lens[b]), Sk))
        vis = j < L
        if causal:
            vis = vis & (j <= i + (L - Sq))
        for h in range(Hq):
            s = np.nan_to_num(q[b, h] @ np.nan_to_num(k[b, h // G]).T) * (scale * LOG2E)
            t[b, h] = np.where(vis, s, -np.inf)
    return t


def lazy_rebases(t, groups):
    """Number of times the lazy rule moves a finite running max, per row.
    t: [rows, keys] log2 scores; groups: list of key-index arrays visited in
    order (one per block or slice).  The first visited group with a finite
    max sets the basis (alpha = 0 on an empty O: not counted)."""
    m = np.full(t.shape[0], -np.inf)
    count = np.zeros(t.shape[0], dtype=np.int64)
    for g in groups:
        if len(g) == 0:
            continue
        mx = t[:, g].max(axis=1)
        mn = np.maximum(m, mx)
        move = mn > m + THRESHOLD
        count += (move & np.isfinite(m)).astype(np.int64)
        m = np.where(move, mn, m)
    return count


def prefill_blocks(Sk, kb=0, ke=None, bs=128):
    """Key blocks of bs keys, [kb, ke) of them."""
    ke = (Sk + bs - 1) // bs if ke is None else ke
    return [np.arange(j * bs, min((j + 1) * bs, Sk)) for j in range(kb, ke)]


def block_keys(B, Hq, Sq, Sk, d, causal, paged=False):
    """Keys per score block of the kernel that runs this launch (256 for the
    256-key kernel, else 128)."""
    from attention_forward_blackwell_gb300 import binding
    return binding.debug_prefill_plan_ex(B, Hq, Sq, Sk, d, causal, 152,
                                         paged=paged).keys_per_block


def decode_warp_slices(k_lo, k_hi, warp):
    """Keys of the 16-key slices one decode warp visits in its split."""
    out = []
    s = k_lo + 16 * warp
    while s < k_hi:
        out.append(np.arange(s, min(s + 16, k_hi)))
        s += 64
    return out


def _run_prefill(x, scale, causal):
    from attention_forward_blackwell_gb300 import binding
    o, lse = binding.prefill(x.q, x.k, x.v, scale=scale, causal=causal, seqlens_k=x.seqlens_k)
    torch.cuda.synchronize()
    check_device_error()
    return o, lse


# ----------------------------------------------------------- prefill ----

PREFILL = [
    # B, Hq, Hkv, S, d: whole units (no split: few key blocks), ragged tails
    (1, 2, 1, 1100, 64),
    (1, 2, 2, 1100, 96),
    (1, 2, 1, 1100, 128),
    (1, 4, 2, 1100, 256),
    (1, 2, 2, 700, 512),
]


@pytest.mark.parametrize("mode", ["steep", "mixed"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,S,d", PREFILL, ids=[f"d{c[4]}" for c in PREFILL])
def test_prefill_rebase_ramp(B, Hq, Hkv, S, d, causal, mode):
    from attention_forward_blackwell_gb300 import binding
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert binding.debug_prefill_plan(B, Hq, S, S, d, causal, n_sms)[2] == 1   # whole units
    x, scale = ramp_inputs(B, Hq, Hkv, S, S, d, tag=7000 + d + 3 * causal, mode=mode,
                           step_keys=128)
    bs = block_keys(B, Hq, S, S, d, causal)
    t = scores_log2(x, scale, causal).reshape(-1, S)
    n = lazy_rebases(t, prefill_blocks(S, bs=bs))
    # key blocks of the kernel, and 128-key ramp steps, that each row sees
    vis_kblocks = np.array([len({j // bs for j in np.flatnonzero(np.isfinite(r))}) for r in t])
    vis_blocks = np.array([len({j // 128 for j in np.flatnonzero(np.isfinite(r))}) for r in t])
    multi = vis_kblocks >= 2
    if mode == "steep":
        # every row that sees two or more key blocks moves its basis; with a
        # causal mask a row that sees only a few keys of its second block
        # may not, so there the bar is 95 % of them
        frac = n[multi].astype(bool).mean()
        assert frac >= (0.95 if causal else 1.0), frac
        assert n[multi].mean() >= 2.0
    else:
        slope = x.q[..., 0].float().cpu().numpy().reshape(-1)
        steep = (vis_blocks >= 3) & (slope > 9)
        shallow = (vis_blocks >= 6) & (slope >= 2.5) & (slope < 5)
        # (with 256-key blocks and a causal mask a steep row that sees only a
        # few keys of its last block may stay below the threshold: there the
        # bar is 95 % of them, as for the causal steep ramp)
        assert steep.any()
        assert n[steep].astype(bool).mean() >= (0.95 if causal and bs > 128 else 1.0)
        assert not n[slope < 0].any()                   # falling: never
        assert shallow.any() and n[shallow].astype(bool).mean() >= 0.9
    o, lse = _run_prefill(x, scale, causal)
    ro, rl = oracle_for(x, scale, causal)
    compare(o, lse, ro, rl, f"rebase ramp d={d} causal={causal} {mode} "
                            f"({int(n.astype(bool).sum())}/{n.size} rows rebase)")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 96, 128, 256, 512])
@pytest.mark.parametrize("pos", [300, 1000])
def test_prefill_dominant_key_in_a_later_block(d, causal, pos):
    """K*8 gives scores spread ~8.5 (max ~25 over 1,100 keys); key `pos`
    (a middle block or the last block, for 128- and 256-key blocks alike)
    scores ~60 for every query, so every row that sees it jumps by more than
    30 log2 units at that block and O ~ v_pos."""
    from attention_forward_blackwell_gb300 import inputs
    S = 1100
    Hq = 2
    x = inputs.make_inputs(1, Hq, Hq, S, S, d, tag=7100 + d + pos, device="cuda", k_scale=8.0)
    x.q[..., 0] = 4.0
    x.k[..., pos, :] = 0.0
    x.k[..., pos, 0] = 60.0 * math.sqrt(d) / 4.0
    scale = 1.0 / math.sqrt(d)
    t = scores_log2(x, scale, causal).reshape(-1, S)
    n = lazy_rebases(t, prefill_blocks(S, bs=block_keys(1, Hq, S, S, d, causal)))
    sees = np.isfinite(t[:, pos])
    assert n[sees].astype(bool).all() and sees.sum() >= Hq * (S - pos)
    o, lse = _run_prefill(x, scale, causal)
    ro, rl = oracle_for(x, scale, causal)
    compare(o, lse, ro, rl, f"dominant key {pos} d={d} causal={causal}")
    rows = torch.from_numpy(np.flatnonzero(sees)).cuda()
    assert float(lse.view(-1)[rows].min()) > 55.0
    dv = (o.view(-1, d)[rows].float() - x.v[0, :, pos:pos + 1].float().expand(Hq, S, d)
          .reshape(-1, d)[rows]).abs().max().item()
    assert dv < 2e-2, dv


@pytest.mark.parametrize("mode", ["steep", "mixed"])
@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,d,paged", [
    (1, 2, 2, 2048, 2048, 64, False),
    (1, 2, 1, 2048, 2304, 96, True),
    (1, 2, 2, 2048, 2048, 128, True),
    (1, 2, 1, 1024, 2048, 256, False),
], ids=["d64", "d96", "d128", "d256"])
def test_split_unit_merge_rebases(B, Hq, Hkv, Sq, Sk, d, paged, mode):
    """Query blocks computed in pieces along the key axis: with the ramp the
    later piece holds the larger scores (steep: every row's later piece beats
    the first by far more than 8 log2 units; mixed: in both directions), so
    the merge of the pieces rescales the earlier partial O and row_sum, and
    every piece also rebases inside itself.  (Head_dim 96 and 128 split on
    paged caches: their contiguous non-causal launches run the persistent
    256-key kernel, which does not split.)"""
    from attention_forward_blackwell_gb300 import binding
    from gpu_parity import to_pages
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    n_full, n_tail, split = binding.debug_prefill_plan_ex(B, Hq, Sq, Sk, d, False, n_sms,
                                                          paged=paged)[:3]
    assert n_full == 0 and split > 1, (n_full, n_tail, split)
    nk = (Sk + 127) // 128
    x, scale = ramp_inputs(B, Hq, Hkv, Sq, Sk, d, tag=7200 + d, mode=mode, step_keys=128)
    t = scores_log2(x, scale, False).reshape(-1, Sk)
    bounds = [(k * nk // split, (k + 1) * nk // split) for k in range(split)]
    inside = sum(lazy_rebases(t, prefill_blocks(Sk, kb, ke)) for kb, ke in bounds)
    piece_max = np.stack([t[:, kb * 128:min(ke * 128, Sk)].max(axis=1) for kb, ke in bounds], 1)
    jump = piece_max.max(axis=1) - piece_max[:, 0]
    if mode == "steep":
        assert inside.astype(bool).all()
        assert (jump > 4 * THRESHOLD).all()
    else:
        slope = x.q[..., 0].float().cpu().numpy().reshape(-1)
        assert (jump[slope > 9] > THRESHOLD).all()
        # falling rows: the first piece dominates, the later ones are scaled down
        assert (piece_max[slope < -1, 0] > piece_max[slope < -1, -1] + 4).all()
    if paged:
        kc, vc, table, _ = to_pages(x.k, x.v, [Sk] * B, 256, seed=d)
        lens = torch.full((B,), Sk, dtype=torch.int32, device="cuda")
        o, lse = binding.prefill_paged(x.q, kc, vc, table, lens, scale=scale)
        torch.cuda.synchronize()
        check_device_error()
    else:
        o, lse = _run_prefill(x, scale, False)
    ro, rl = oracle_for(x, scale, False)
    compare(o, lse, ro, rl, f"split merge d={d} split={split} {mode}")


# ------------------------------------------------------------ decode ----

@pytest.mark.parametrize("num_splits", [1, 7])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("mode,causal,Sq", [("steep", False, 1), ("mixed", False, 1),
                                            ("steep", True, 4)])
def test_decode_rebase_ramp(d, num_splits, mode, causal, Sq):
    """Decode over a ramp that rises 14-18 log2 units (steep) every 64 keys --
    one step of each warp's walk over its 16-key slices -- so every warp of
    every split rebases at each slice, and the combine merges splits whose
    LSEs differ by hundreds of log2 units."""
    from attention_forward_blackwell_gb300 import binding
    B, Hq, Hkv, Sk = 3, 8, 2, 2000
    lengths = [2000, 1300, 700]
    x, scale = ramp_inputs(B, Hq, Hkv, Sq, Sk, d, tag=7300 + d + Sq, mode=mode, step_keys=64,
                           lengths=lengths)
    t = scores_log2(x, scale, causal)
    span = Sk
    chunk = -(-span // num_splits)
    chunk = -(-chunk // 64) * 64
    n_splits = -(-span // chunk)
    counts = np.zeros(t.shape[:3], dtype=np.int64)
    for b in range(B):
        for s in range(n_splits):
            lo, hi = s * chunk, min((s + 1) * chunk, lengths[b])
            for w in range(4):
                counts[b] += lazy_rebases(t[b].reshape(-1, Sk), decode_warp_slices(lo, hi, w)) \
                    .reshape(Hq, Sq)
    if mode == "steep":
        assert counts.astype(bool).all()
    else:
        slope = x.q[..., 0].float().cpu().numpy()
        assert counts[slope > 9].astype(bool).all() and not counts[slope < 0].any()
    o, lse = binding.decode(x.q, x.k, x.v, scale=scale, causal=causal, seqlens_k=x.seqlens_k,
                            num_splits=num_splits)
    torch.cuda.synchronize()
    check_device_error()
    ro, rl = oracle_for(x, scale, causal)
    compare(o, lse, ro, rl, f"decode rebase d={d} splits={num_splits} {mode} Sq={Sq}")
