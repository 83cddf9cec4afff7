"""The C ABI on the CPU: the library loads, exports every declared symbol, and
rejects every host-checkable error before any CUDA call (no GPU needed).

Pointers passed here are fake but 16-byte aligned; every call below fails its
host-side validation first, so none is dereferenced and nothing is launched.
"""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
HEADER = ROOT / "include" / "pagedkv.h"


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_275_gb300 import build
    build.build(quiet=True)
    from paged_kv_cache_275_gb300 import _capi
    return _capi.load()


def declared_functions() -> list[str]:
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_calls():
    names = declared_functions()
    for required in ("pkv_kv_append", "pkv_paged_decode_attention", "pkv_decode_workspace_size",
                     "pkv_get_and_clear_device_error", "pkv_last_error_message"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from paged_kv_cache_275_gb300 import EXPORTS
    names = declared_functions()
    assert sorted(EXPORTS) == names
    for name in names:
        assert hasattr(lib, name), name


def test_exported_symbols_are_c_linkage():
    import subprocess
    from paged_kv_cache_275_gb300 import LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", str(LIB_PATH)], capture_output=True, text=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in syms, f"{name} is not exported unmangled"


FAKE = 0x10000  # aligned, never dereferenced


def msg(lib) -> str:
    return lib.pkv_last_error_message().decode()


def append(lib, **kw):
    args = dict(k=FAKE, v=FAKE, slots=FAKE, n=4, hkv=8, d=128, kc=FAKE, vc=FAKE, nb=10, bs=16, stream=None)
    args.update(kw)
    return lib.pkv_kv_append(args["k"], args["v"], args["slots"], args["n"], args["hkv"], args["d"], args["kc"],
                             args["vc"], args["nb"], args["bs"], args["stream"])


def test_append_rejects_bad_arguments(lib):
    assert append(lib, d=96) == 2 and "head_dim" in msg(lib)
    assert append(lib, bs=32) == 2 and "block_size" in msg(lib)
    assert append(lib, hkv=0) == 1
    assert append(lib, n=-1) == 1
    assert append(lib, nb=0) == 1
    assert append(lib, k=None) == 1 and "null" in msg(lib)
    assert append(lib, kc=FAKE + 8) == 1 and "aligned" in msg(lib)
    assert append(lib, slots=FAKE + 4) == 1


def test_append_zero_tokens_is_a_noop(lib):
    assert append(lib, n=0, k=None, v=None) == 0
    assert msg(lib) == ""


def attention(lib, **kw):
    a = dict(q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, W=8, cl=FAKE, B=4, hq=32, hkv=8, d=128, nb=100, bs=16, scale=0.088,
             out=FAKE, ws=FAKE, wsb=16, parts=64, phases=3, stream=None)
    a.update(kw)
    return lib.pkv_paged_decode_attention_split(a["q"], a["kc"], a["vc"], a["bt"], a["W"], a["cl"], a["B"], a["hq"],
                                                a["hkv"], a["d"], a["nb"], a["bs"], a["scale"], a["out"], a["ws"],
                                                a["wsb"], a["parts"], a["phases"], a["stream"])


def test_attention_rejects_bad_arguments(lib):
    assert attention(lib, hq=30) == 1 and "multiple" in msg(lib)
    assert attention(lib, hq=24, hkv=2) == 2 and "group" in msg(lib)        # G = 12
    assert attention(lib, d=256) == 2
    assert attention(lib, bs=8) == 2
    assert attention(lib, B=-1) == 1
    assert attention(lib, B=5000, phases=1) == 2 and "PKV_MAX_SEQS" in msg(lib)   # split phases: one slice only
    assert attention(lib, B=5000) == 1 and "workspace too small" in msg(lib)        # sliced, checked as a whole
    assert attention(lib, W=0) == 1
    assert attention(lib, nb=0) == 1
    assert attention(lib, scale=float("inf")) == 1
    assert attention(lib, phases=0) == 1 and attention(lib, phases=4) == 1
    assert attention(lib, parts=-3) == 1
    assert attention(lib, out=None) == 1
    assert attention(lib, q=FAKE + 2) == 1
    assert attention(lib, ws=FAKE + 8) == 1
    assert attention(lib, wsb=16) == 1 and "workspace too small" in msg(lib)


def prefill(lib, **kw):
    a = dict(q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, W=8, cl=FAKE, qs=FAKE, mql=512, B=4, hq=32, hkv=8, d=128, nb=100,
             bs=16, scale=0.088, out=FAKE, stream=None)
    a.update(kw)
    return lib.pkv_paged_prefill_attention(a["q"], a["kc"], a["vc"], a["bt"], a["W"], a["cl"], a["qs"], a["mql"], a["B"],
                                           a["hq"], a["hkv"], a["d"], a["nb"], a["bs"], a["scale"], a["out"],
                                           a["stream"])


def test_prefill_rejects_grids_it_cannot_launch(lib):
    """A sequence's CTAs (256 / G chunk tokens each) are one grid dimension, at most 65535."""
    assert prefill(lib, B=65536) == 2 and "65535" in msg(lib)
    assert prefill(lib, mql=65535 * 64 + 1) == 2 and "max_query_len" in msg(lib)      # G = 4: 64 tokens a CTA
    assert prefill(lib, mql=65535 * 32 + 1, hq=64) == 2 and "32 chunk tokens" in msg(lib)   # G = 8
    assert prefill(lib, mql=-1) == 1
    assert prefill(lib, mql=0, q=None, out=None) == 0                                   # a no-op before the pointers


def prefill_split(lib, **kw):
    a = dict(q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, W=8, cl=FAKE, qs=FAKE, mql=512, B=4, hq=32, hkv=8, d=128, nb=100,
             bs=16, scale=0.088, out=FAKE, S=2, ws=FAKE, wsb=1 << 30, stream=None)
    a.update(kw)
    return lib.pkv_paged_prefill_attention_split(a["q"], a["kc"], a["vc"], a["bt"], a["W"], a["cl"], a["qs"], a["mql"],
                                                 a["B"], a["hq"], a["hkv"], a["d"], a["nb"], a["bs"], a["scale"],
                                                 a["out"], a["S"], a["ws"], a["wsb"], a["stream"])


def test_prefill_workspace_size(lib):
    n = ctypes.c_size_t(0)
    # 3 splits x 4 sequences x 512 rows (a multiple of G = 4's 64 chunk tokens) x 32 q heads x (128 + 2) floats
    assert lib.pkv_prefill_workspace_size(4, 512, 32, 8, 128, 3, ctypes.byref(n)) == 0
    assert n.value == 3 * 4 * 512 * 32 * 130 * 4
    assert lib.pkv_prefill_workspace_size(2, 33, 16, 8, 64, 2, ctypes.byref(n)) == 0   # G = 2: 128-token CTAs
    assert n.value == 2 * 2 * 128 * 16 * 66 * 4
    assert lib.pkv_prefill_workspace_size(4, 512, 32, 8, 128, 1, ctypes.byref(n)) == 0 and n.value == 0
    assert lib.pkv_prefill_workspace_size(4, 512, 32, 8, 128, 33, ctypes.byref(n)) == 1
    assert lib.pkv_prefill_workspace_size(4, 512, 30, 8, 128, 2, ctypes.byref(n)) == 1


def test_prefill_default_splits_checks_arguments_before_the_device(lib):
    n = ctypes.c_int32(0)
    assert lib.pkv_prefill_default_splits(1, 512, 32, 8, None) == 1 and "null" in msg(lib)
    assert lib.pkv_prefill_default_splits(1, 512, 30, 8, ctypes.byref(n)) == 1
    assert lib.pkv_prefill_default_splits(-1, 512, 32, 8, ctypes.byref(n)) == 1


def test_prefill_split_rejects_bad_arguments(lib):
    assert prefill_split(lib, S=0) == 1 and "num_splits" in msg(lib)
    assert prefill_split(lib, S=33) == 1 and "num_splits" in msg(lib)
    assert prefill_split(lib, B=40000, S=2) == 2 and "num_splits" in msg(lib)            # 80000 grid rows
    assert prefill_split(lib, wsb=16) == 1 and "workspace too small" in msg(lib)
    assert prefill_split(lib, ws=None) == 1 and "workspace too small" in msg(lib)
    assert prefill_split(lib, ws=FAKE + 8) == 1 and "aligned" in msg(lib)
    assert prefill_split(lib, mql=0, q=None, out=None, ws=None) == 0                   # a no-op before the pointers


def test_attention_zero_sequences_is_a_noop(lib):
    assert attention(lib, B=0, q=None, out=None) == 0


def test_workspace_size_with_explicit_partitions(lib):
    n = ctypes.c_size_t(0)
    assert lib.pkv_decode_workspace_size(128, 32, 8, 128, 256, 1000, ctypes.byref(n)) == 0
    # Block prefix int32 [B + 1], then the merge's pair records int32 [B * Hkv][2], each 256-byte aligned.
    header = ((128 + 1) * 4 + 255) // 256 * 256 + (128 * 8 * 8 + 255) // 256 * 256
    piece = 4 * 128 + 8                                  # G * D + round_up(2G, 4) floats
    assert n.value == header + 1000 * 2 * piece * 4
    n1 = ctypes.c_size_t(0)
    assert lib.pkv_decode_workspace_size(4, 2, 1, 64, 3, 12, ctypes.byref(n1)) == 0
    assert n1.value == 256 + 256 + 12 * 2 * (2 * 64 + 4) * 4
    assert lib.pkv_decode_workspace_size(4, 2, 1, 64, 3, -1, ctypes.byref(n1)) == 1


def test_selftest_rejects_limits_outside_range(lib):
    for bad in (0, 999, 1_000_000_001, 2**63):
        assert lib.pkv_selftest_wait_timeout(bad, None) == 1  # PKV_ERR_INVALID_ARGUMENT, before any CUDA call
        assert b"limit_ns" in lib.pkv_last_error_message()


def test_launch_counter_starts_at_zero_without_launches(lib):
    assert lib.pkv_kernel_launch_count() == 0


def test_python_binding_refuses_cpu_tensors():
    import torch
    import paged_kv_cache_275_gb300 as pkv
    q = torch.zeros(1, 2, 64, dtype=torch.bfloat16)
    kc = torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        pkv.paged_decode_attention(q, kc, kc, torch.zeros(1, 1, dtype=torch.int32), torch.ones(1, dtype=torch.int32),
                                   0.1, q.clone())
    with pytest.raises(ValueError, match="CUDA"):
        pkv.kv_append(q[:, :1], q[:, :1], torch.zeros(1, dtype=torch.int64), kc, kc)


def test_missing_library_fails_loudly(tmp_path):
    from paged_kv_cache_275_gb300 import _capi
    with pytest.raises(ImportError, match="no fallback"):
        _capi.load(tmp_path / "libpagedkv.so")
