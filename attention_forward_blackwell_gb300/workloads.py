"""The benchmark workloads and their algorithmic work counts.

FLOPs follow the convention of the "fa4-sm120-research" page's throughput
table: a forward pass over B*H heads of Sq queries and Sk keys at head
dimension d costs 4*B*Hq*Sq*Sk*d floating-point operations (two GEMMs of
2*Sq*Sk*d each per head), halved when a causal mask removes half the score
matrix.  The four rows of that table are reproduced by this formula to four
significant digits (checked by the golden test of the table).

Decode is memory-bound; its algorithmic bytes are the valid key and value
rows read once (each key/value head is read once for all of its query heads),
plus Q read once and O and LSE written once.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Tuple


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    d: int
    causal: bool
    tag: int                               # seed tag for the input generator
    k_scale: float = 1.0
    lengths: Optional[Tuple[int, int]] = None   # uniform [lo, hi] key lengths
    decode: bool = False
    description: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        return 1.0 / (self.d ** 0.5)


def prefill_flops(B, Hq, Sq, Sk, d, causal):
    f = 4.0 * B * Hq * Sq * Sk * d
    return f * 0.5 if causal else f


def prefill_bytes(B, Hq, Hkv, Sq, Sk, d):
    """Algorithmic HBM bytes of one prefill pass without key lengths: K and V
    once per kv head, Q and O once (bf16), LSE (fp32)."""
    return 2 * B * Hkv * Sk * d * 2 + 2 * B * Hq * Sq * d * 2 + B * Hq * Sq * 4


def decode_bytes(Hkv, Hq, d, lengths, Sq=1):
    """Algorithmic HBM bytes of one decode pass (bf16 K/V/Q/O, fp32 LSE)."""
    B = len(lengths)
    kv = sum(2 * Hkv * int(L) * d * 2 for L in lengths)
    q = B * Hq * Sq * d * 2
    o = B * Hq * Sq * d * 2
    lse = B * Hq * Sq * 4
    return kv + q + o + lse


def decode_flops(Hq, d, lengths, Sq=1):
    return sum(4.0 * Hq * Sq * int(L) * d for L in lengths)


TINY = Workload("tiny_mha_b1_h1_s128_d64", 1, 1, 1, 128, 128, 64, False, 1,
                description="tiny non-causal MHA B=1 H=1 Sq=Sk=128 d=64")
PREFILL_D128 = Workload("prefill_mha_b2_h16_s4096_d128", 2, 16, 16, 4096, 4096,
                        128, False, 2,
                        description="prefill MHA B=2 H=16 Sq=Sk=4096 d=128 non-causal")
PREFILL_D128_CAUSAL = Workload("prefill_mha_b2_h16_s4096_d128_causal", 2, 16,
                               16, 4096, 4096, 128, True, 2,
                               description="prefill MHA B=2 H=16 Sq=Sk=4096 d=128 causal")
LONG_D128 = Workload("long_prefill_b1_h16_s8192_d128", 1, 16, 16, 8192, 8192,
                     128, False, 3,
                     description="long prefill MHA B=1 H=16 Sq=Sk=8192 d=128 non-causal")
LONG_D96 = Workload("prefill_b2_h16_s4096_d96", 2, 16, 16, 4096, 4096, 96,
                    False, 6,
                    description="prefill MHA B=2 H=16 Sq=Sk=4096 d=96 non-causal")
# head_dim 64 at the shape of the last row of the "fa4-sm120-research" table
PREFILL_D64 = Workload("prefill_b4_h32_s2048_d64", 4, 32, 32, 2048, 2048, 64, False, 8,
                       description="prefill MHA B=4 H=32 Sq=Sk=2048 d=64 non-causal")
GQA_D256 = Workload("causal_gqa_b4_hq32_hkv4_s2048_d256", 4, 32, 4, 2048, 2048,
                    256, True, 4, k_scale=0.5,
                    description="causal GQA B=4 Hq=32 Hkv=4 Sq=Sk=2048 d=256, K*0.5")
# head_dim 512 (no configuration of the pages uses it): the FLOPs of the
# 8K-key d=128 shape at a quarter of the heads times four the head dimension
PREFILL_D512 = Workload("prefill_b2_h8_s4096_d512", 2, 8, 8, 4096, 4096, 512,
                        False, 7,
                        description="prefill MHA B=2 H=8 Sq=Sk=4096 d=512 non-causal")
PREFILL_D512_CAUSAL = Workload("prefill_b2_h8_s4096_d512_causal", 2, 8, 8, 4096,
                               4096, 512, True, 7,
                               description="prefill MHA B=2 H=8 Sq=Sk=4096 d=512 causal")
DECODE = Workload("decode_gqa_b64_hq64_hkv8_d128", 64, 64, 8, 1, 16384, 128,
                  False, 5, lengths=(1024, 16384), decode=True,
                  description="decode GQA B=64 Hq=64 Hkv=8 Sq=1 d=128, "
                              "L_b~U[1024,16384], KV padded to 16384")

# short-query GQA prefill (chunked prefill: 16 new queries per sequence over
# its cached keys), where the 256-key kernel packs the 8 query heads of a kv
# group into one tile (not a configuration of the pages)
CHUNKED_GQA = Workload("chunked_prefill_gqa_b64_hq32_hkv4_q16_k4096_d128", 64, 32, 4, 16, 4096,
                       128, True, 9,
                       description="chunked prefill GQA B=64 Hq=32 Hkv=4 Sq=16 Sk=4096 d=128 "
                                   "causal")

# few units over long keys (32 units of 128 rows on 152 SMs), where the
# 256-key kernel splits each unit along the keys (not a configuration of the
# pages)
SPLIT_FEW = Workload("split_prefill_b1_h8_q512_k16384_d128", 1, 8, 8, 512, 16384, 128, False, 10,
                     description="prefill B=1 H=8 Sq=512 Sk=16384 d=128 non-causal (few units)")

ALL = [TINY, PREFILL_D128, PREFILL_D128_CAUSAL, LONG_D128, LONG_D96, PREFILL_D64, GQA_D256,
       PREFILL_D512, PREFILL_D512_CAUSAL, DECODE, CHUNKED_GQA, SPLIT_FEW]
