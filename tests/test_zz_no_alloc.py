"""The allocation-free decode attention entry point, through the C ABI.

pkv_paged_decode_attention_static serves callers that cannot allocate device
memory: a plugin running inside a host process that owns every device
allocation, or a serving loop where a cudaMalloc would implicitly synchronise
the device and stall its other streams.  Its scratch is a fixed array built
into the library, shared by every call.

It runs the same partition and merge kernels, at the same default partition
count, as the regular entry point (caller-provided workspace), so on two
calls in a row its output must equal that entry point's bit for bit: a
scratch-reuse defect that disturbed even one low bit would show.  Both
outputs are also held to the attention tolerance against the fp64 oracle,
and the second call must leave the device's free memory and torch's reserved
memory unchanged (it allocates nothing).

This file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import paged_kv_cache_275_gb300 as pkv
from gpu_util import assert_close, oracle_step
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
    c = make_decode_case(name, seed=21, num_seqs=num_seqs)
    ref_oracle, _, _ = oracle_step(c)
    g = c.to("cuda")
    pkv.kv_append(g.new_k, g.new_v, g.slot_mapping, g.k_cache, g.v_cache)
    ref = torch.empty_like(g.q)
    pkv.paged_decode_attention(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale, ref)
    torch.cuda.synchronize()
    assert_close(ref, ref_oracle, f"{name}: workspace entry")
    outs = [torch.full_like(g.q, float("nan")) for _ in range(2)]
    for call, out in enumerate(outs):
        torch.cuda.synchronize()
        free0, reserved0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved()
        status = _static_call(lib, g, out)
        assert status == 0, lib.pkv_last_error_message().decode()
        torch.cuda.synchronize()
        if call == 1:  # the first call may still load the library's kernels; the second allocates nothing
            assert torch.cuda.mem_get_info()[0] == free0, f"{name}: device free memory changed"
            assert torch.cuda.memory_reserved() == reserved0, f"{name}: torch reserved memory changed"
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"{name} call {call}: differs from the workspace entry"
        assert_close(out, ref_oracle, f"{name} call {call}: static entry")
    assert pkv.get_and_clear_device_error() == 0
