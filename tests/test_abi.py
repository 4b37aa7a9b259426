"""The C-ABI library loads and exports every declared entry point; host-side
argument validation rejects bad calls before any GPU work (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    from attention_forward_blackwell_gb300 import binding, build
    build.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("fa_fwd_prefill", "fa_fwd_decode", "fa_status_string",
                     "fa_get_device_error", "fa_version"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from attention_forward_blackwell_gb300 import binding
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in binding.SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    from attention_forward_blackwell_gb300 import binding
    assert binding.status_string(0) == "FA_OK"
    assert binding.status_string(5) == "FA_ERR_TIMEOUT"
    assert binding.status_string(99) == "FA_ERR_UNKNOWN"
    assert binding.version() >= 100


P16 = ctypes.c_void_p(1 << 12)      # a 16-byte aligned (never dereferenced) address
P_ODD = ctypes.c_void_p((1 << 12) + 8)


@pytest.mark.parametrize("fn", ["fa_fwd_prefill", "fa_fwd_decode"])
@pytest.mark.parametrize("args,expect", [
    # (q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, seqlens, d, scale, causal), status
    ((P16, P16, P16, P16, P16, -1, 1, 1, 1, 1, None, 64, 1.0, 0), 1),     # negative batch
    ((P16, P16, P16, P16, P16, 1, 3, 2, 1, 1, None, 64, 1.0, 0), 1),      # hq % hkv
    ((P16, P16, P16, P16, P16, 1, 1, 1, 1, 1, None, 64, 0.0, 0), 1),      # scale 0
    ((P16, P16, P16, P16, P16, 1, 1, 1, 1, 1, None, 64, float("nan"), 0), 1),
    ((None, P16, P16, P16, P16, 1, 1, 1, 1, 1, None, 64, 1.0, 0), 1),     # null q
    ((P16, None, P16, P16, P16, 1, 1, 1, 1, 4, None, 64, 1.0, 0), 1),     # null k
    ((P_ODD, P16, P16, P16, P16, 1, 1, 1, 1, 1, None, 64, 1.0, 0), 3),    # misaligned q
    ((P16, P16, P16, P16, P16, 1, 1, 1, 1, 1, None, 80, 1.0, 0), 2),      # head_dim
    ((P16, P16, P16, P16, P16, 70000, 1, 1, 1, 1, None, 64, 1.0, 0), 1),  # batch too big
    ((None, None, None, None, None, 0, 4, 2, 8, 8, None, 64, 1.0, 0), 0),  # empty batch
    ((None, None, None, None, None, 2, 4, 2, 0, 8, None, 64, 1.0, 1), 0),  # no queries
])
def test_host_validation(lib, fn, args, expect):
    assert getattr(lib, fn)(*args, None) == expect


def test_decode_specific_validation(lib):
    # sq above the decode limit, and head_dims 96 and 512 (prefill only)
    assert lib.fa_fwd_decode(P16, P16, P16, P16, P16, 1, 1, 1, 17, 8, None, 64, 1.0, 0,
                             None) == 1
    assert lib.fa_fwd_decode(P16, P16, P16, P16, P16, 1, 1, 1, 1, 8, None, 96, 1.0, 0,
                             None) == 2
    assert lib.fa_fwd_decode(P16, P16, P16, P16, P16, 1, 1, 1, 1, 8, None, 512, 1.0, 0,
                             None) == 2


def test_prefill_head_dims(lib):
    """head_dim 512 passes the prefill argument checks exactly as 64 does (on
    a machine without the GPU both then stop at the same device check); head
    dimensions outside {64, 96, 128, 256, 512} are rejected first."""
    def call(d):
        return lib.fa_fwd_prefill(P16, P16, P16, P16, P16, 1, 1, 1, 8, 8, None, d, 1.0, 0, None)
    import torch
    if not torch.cuda.is_available():   # (with a GPU the fake pointers would be read)
        assert call(512) == call(64) != 2
    for d in (384, 1024, 32, 80):
        assert call(d) == 2
    out = (ctypes.c_int * 3)()
    # two CTAs per unit, never split along the keys
    assert lib.fa_debug_prefill_plan(2, 8, 4096, 4096, 512, 0, 152, out) == 0
    assert list(out) == [2 * 8 * 32, 0, 1]
    assert lib.fa_debug_prefill_plan(2, 8, 4096, 4096, 384, 0, 152, out) == 1


P_MIS4 = ctypes.c_void_p((1 << 12) + 2)   # not 4-byte aligned


@pytest.mark.parametrize("args,expect", [
    # (q, k, v, o, lse, cu_q, cu_k, B, max_q, max_k, total_q, total_k, Hq, Hkv, d, scale,
    #  causal, window, sinks), status
    ((P16, P16, P16, P16, P16, P16, P16, -1, 8, 8, 8, 8, 2, 1, 64, 1.0, 0, 0, None), 1),
    ((P16, P16, P16, P16, P16, P16, P16, 2, 0, 8, 8, 8, 2, 1, 64, 1.0, 0, 0, None), 1),
    ((P16, P16, P16, P16, P16, P16, P16, 2, 8, 0, 8, 8, 2, 1, 64, 1.0, 0, 0, None), 1),
    ((P16, P16, P16, P16, P16, None, P16, 2, 8, 8, 8, 8, 2, 1, 64, 1.0, 0, 0, None), 1),
    ((P16, P16, P16, P16, P16, P_MIS4, P16, 2, 8, 8, 8, 8, 2, 1, 64, 1.0, 0, 0, None), 3),
    ((P16, P16, P16, P16, P16, P16, P16, 2, 8, 8, 8, 8, 3, 2, 64, 1.0, 0, 0, None), 1),
    ((P16, P16, P16, P16, P16, P16, P16, 2, 8, 8, 8, 8, 2, 1, 80, 1.0, 0, 0, None), 2),
    ((P_ODD, P16, P16, P16, P16, P16, P16, 2, 8, 8, 8, 8, 2, 1, 64, 1.0, 0, 0, None), 3),
    ((None, None, None, None, None, None, None, 0, 0, 0, 0, 0, 2, 1, 64, 1.0, 0, 0, None), 0),
    ((None, None, None, None, None, None, None, 3, 0, 0, 0, 0, 2, 1, 64, 1.0, 0, 0, None), 0),
])
def test_varlen_host_validation(lib, args, expect):
    """Packed-sequence argument checks run on the host, before any launch."""
    assert lib.fa_fwd_prefill_varlen(*args, None) == expect


def test_paged_host_validation(lib):
    # (q, kc, vc, o, lse, B, Hq, Hkv, Sq, seqlens, table, max_pages, page, pages, d, scale, causal)
    ok = (P16, P16, P16, P16, P16, 1, 2, 1, 4, P16, P16, 2, 128, 4, 64, 1.0, 0)
    bad_table = ok[:10] + (None,) + ok[11:]
    bad_page = ok[:12] + (100,) + ok[13:]
    assert lib.fa_fwd_prefill_paged(*bad_table, None) == 1           # no block table
    assert lib.fa_fwd_prefill_paged(*bad_page, None) == 2            # tile must fit a page
    assert lib.fa_fwd_decode_paged(*(ok[:13] + (0,) + ok[14:]), None) == 1   # no pages


def test_varlen_paged_host_validation(lib):
    # (q, kc, vc, o, lse, cu_q, seqlens, table, max_pages, page, pages, B, max_q, total_q,
    #  Hq, Hkv, d, scale, causal, window, sinks)
    ok = [P16, P16, P16, P16, P16, P16, P16, P16, 2, 128, 4, 1, 8, 8, 2, 1, 64, 1.0, 0, 0, None]
    def call(**kw):
        a = list(ok)
        for i, val in kw.items():
            a[int(i[1:])] = val
        return lib.fa_fwd_prefill_varlen_paged(*a, None)
    assert call(a5=None) == 1              # no query offsets
    assert call(a6=None) == 1              # no key lengths
    assert call(a7=None) == 1              # no block table
    assert call(a9=100) == 2               # a key tile must fit a page
    assert call(a12=0) == 1                # max_seqlen_q = 0 with tokens present
    assert call(a5=P_MIS4) == 3            # misaligned offsets
    assert call(a11=0, a13=0) == 0         # nothing to compute


def test_binding_rejects_bad_tensors():
    import torch
    from attention_forward_blackwell_gb300 import binding
    q = torch.zeros(1, 2, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        binding.prefill(q, q, q)          # CPU tensors: no fallback, refused
    with pytest.raises(TypeError):
        binding.prefill(q.float(), q, q)


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "attention_forward_blackwell_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "liboracle" not in text, f
