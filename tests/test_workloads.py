"""The benchmark's FLOP convention against the throughput table printed on
the "fa4-sm120-research" page (CPU only)."""
import os

from attention_forward_blackwell_gb300 import workloads

TABLE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                     "fwd_tflops_table.txt")


def _rows():
    for line in open(TABLE):
        line = line.strip()
        if line and not line.startswith("#"):
            b, s, h, d, ms, tf = line.split()
            yield int(b), int(s), int(h), int(d), float(ms), float(tf)


def test_flop_convention_reproduces_printed_table():
    rows = list(_rows())
    assert len(rows) == 4
    for b, s, h, d, ms, tf in rows:
        f = workloads.prefill_flops(b, h, s, s, d, causal=False)
        # "Fwd ms" is printed to 3 decimals and TFLOPS to 1: the printed TFLOPS
        # must lie in the range the printed time allows.
        lo = f / ((ms + 0.0005) * 1e-3) / 1e12 - 0.05
        hi = f / ((ms - 0.0005) * 1e-3) / 1e12 + 0.05
        assert lo <= tf <= hi, (b, s, h, d, f / (ms * 1e-3) / 1e12, tf)
        # a factor-2 slip (counting one GEMM, or halving as if causal) fails
        assert not (lo / 2 <= tf / 1 <= hi / 2)


def test_causal_halves_and_decode_counts():
    assert workloads.prefill_flops(2, 16, 4096, 4096, 128, True) == 137438953472.0
    assert workloads.prefill_flops(2, 16, 4096, 4096, 128, False) == 274877906944.0
    # two sequences of 3 and 5 keys, Hkv=1, d=2: K+V rows 2*(3+5)*2*2 bytes
    assert workloads.decode_bytes(1, 2, 2, [3, 5]) == 2 * 8 * 2 * 2 + 2 * (2 * 2 * 2) * 2 + 2 * 2 * 4


def test_workload_shapes_match_configuration():
    w = workloads
    assert (w.TINY.B, w.TINY.Hq, w.TINY.Sq, w.TINY.d, w.TINY.causal) == (1, 1, 128, 64, False)
    assert (w.GQA_D256.Hq // w.GQA_D256.Hkv, w.GQA_D256.k_scale) == (8, 0.5)
    assert w.DECODE.lengths == (1024, 16384) and w.DECODE.Sk == 16384
    assert abs(w.PREFILL_D128.scale - 128 ** -0.5) < 1e-15


def test_prefill_bytes_counts_each_tensor_once():
    """K and V once per kv head (not per query head), Q and O in bf16, LSE fp32:
    the chunked GQA workload's 8 query heads per kv head add no K/V bytes."""
    w = workloads.CHUNKED_GQA
    kv = 2 * w.B * w.Hkv * w.Sk * w.d * 2
    qo = 2 * w.B * w.Hq * w.Sq * w.d * 2
    assert workloads.prefill_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d) == \
        kv + qo + w.B * w.Hq * w.Sq * 4
    assert workloads.prefill_bytes(1, 8, 1, 1, 100, 64) < workloads.prefill_bytes(1, 8, 8, 1, 100, 64)
