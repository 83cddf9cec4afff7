"""The allocation-free decode attention entry point, through the C ABI.

pkv_paged_decode_attention_static serves callers that cannot allocate device
memory (a plugin inside a host process that owns every device allocation, or
a serving loop where cudaMalloc would synchronise the device): its scratch is
a fixed array built into the library.  Its output must match the regular
entry point's (caller-provided workspace) within the attention tolerance, on
two calls in a row, since every call reuses the same array.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_275_gb300 as pkv
from gpu_util import MAX_ABS, REL_RMS, errors
from workloads import make_decode_case

pytestmark = pytest.mark.gpu


def _static_call(lib, g, out) -> int:
    return lib.pkv_paged_decode_attention_static(
        g.q.data_ptr(), g.k_cache.data_ptr(), g.v_cache.data_ptr(), g.block_tables.data_ptr(),
        g.block_tables.shape[1], g.context_lens.data_ptr(), g.q.shape[0], g.q.shape[1], g.k_cache.shape[1],
        g.q.shape[2], g.k_cache.shape[0], 16, ctypes.c_float(g.scale), out.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name,num_seqs", [("qwen3_0.6b", None), ("llama3_8b", 64), ("llama3_70b", 64), ("tiny", None)])
def test_static_scratch_entry_matches_workspace_entry(name, num_seqs):
    lib = pkv.load()
    g = make_decode_case(name, seed=21, num_seqs=num_seqs).to("cuda")
    pkv.kv_append(g.new_k, g.new_v, g.slot_mapping, g.k_cache, g.v_cache)
    ref = torch.empty_like(g.q)
    pkv.paged_decode_attention(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale, ref)
    torch.cuda.synchronize()
    ref64 = ref.cpu().to(torch.float64).numpy()
    for call in range(2):
        out = torch.full_like(g.q, float("nan"))
        status = _static_call(lib, g, out)
        assert status == 0, lib.pkv_last_error_message().decode()
        torch.cuda.synchronize()
        got = out.cpu().to(torch.float64).numpy()
        assert np.isfinite(got).all(), f"call {call}: non-finite output"
        max_abs, rel_rms = errors(out, ref64)
        assert max_abs <= MAX_ABS and rel_rms <= REL_RMS, f"call {call}: {max_abs:.3g} {rel_rms:.3g}"
    assert pkv.get_and_clear_device_error() == 0
