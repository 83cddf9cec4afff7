"""Fused decode step (RoPE + append + attention in the attention kernels) against the oracle.

The oracle composes its own pieces: RoPE of q and the new k at position L - 1
(fp32 steps, bf16 rounding), append at that position's slot, attention.  The
cache must match bit for bit (the rotated k is a rounding decision both sides
take in the same fp32 steps); the output within the attention tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_275_gb300 as pkv
from gpu_util import assert_close, device_errors
from workloads import DecodeSpec, make_decode_case, rope_cos_sin

pytestmark = pytest.mark.gpu


def _run(c, cos_sin):
    g = c.to("cuda")
    q0 = g.q.clone()
    out = torch.empty_like(g.q)
    pkv.decode_step(g.q, g.new_k, g.new_v, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale, out,
                    None if cos_sin is None else cos_sin.cuda())
    torch.cuda.synchronize()
    assert torch.equal(g.q, q0), "q must not be modified"
    return g, out


def _oracle(c, cos_sin):
    kc, vc = c.k_cache.clone(), c.v_cache.clone()
    ref, st = oracle.decode_step(c.q, c.new_k, c.new_v, kc, vc, c.block_tables, c.context_lens, c.scale, cos_sin)
    assert st == oracle.OK
    return ref, kc, vc


@pytest.mark.parametrize("name,theta", [("tiny", 1e4), ("qwen3_0.6b", 1e6), ("llama3_8b", 5e5)])
def test_fused_step_with_rope(name, theta):
    c = make_decode_case(name, seed=61)
    table = rope_cos_sin(c.spec.max_blocks_per_seq * 16, c.spec.head_dim, theta)
    g, out = _run(c, table)
    ref, kc, vc = _oracle(c, table)
    assert torch.equal(g.k_cache.cpu().view(torch.int16), kc.view(torch.int16))
    assert torch.equal(g.v_cache.cpu().view(torch.int16), vc.view(torch.int16))
    assert_close(out, ref, name)
    assert device_errors() == 0


def test_fused_step_without_rope_equals_separate_calls():
    c = make_decode_case("qwen3_0.6b", seed=62)
    g, out = _run(c, None)
    h = c.to("cuda")
    pkv.kv_append(h.new_k, h.new_v, h.slot_mapping, h.k_cache, h.v_cache)
    ref = torch.empty_like(h.q)
    pkv.paged_decode_attention(h.q, h.k_cache, h.v_cache, h.block_tables, h.context_lens, h.scale, ref)
    assert torch.equal(g.k_cache, h.k_cache) and torch.equal(g.v_cache, h.v_cache)
    assert torch.equal(out, ref)


@pytest.mark.parametrize("head_dim,hq,hkv", [(64, 2, 1), (64, 8, 2), (64, 16, 2), (128, 8, 8), (128, 32, 4)])
def test_fused_step_every_layout_and_length(head_dim, hq, hkv):
    spec = DecodeSpec(name="lens", description="", num_seqs=20, num_q_heads=hq, num_kv_heads=hkv,
                      head_dim=head_dim, max_blocks_per_seq=5, length_kind="fixed",
                      lengths=(0, 1, 2, 15, 16, 17, 31, 32, 33, 47, 48, 49, 64, 65, 70, 79, 80, 3, 9, 40),
                      pool_slack=0.3)
    c = make_decode_case(spec, seed=63)
    table = rope_cos_sin(80, head_dim, 1e4)
    g, out = _run(c, table)
    ref, kc, vc = _oracle(c, table)
    assert torch.equal(g.k_cache.cpu().view(torch.int16), kc.view(torch.int16))
    assert torch.equal(g.v_cache.cpu().view(torch.int16), vc.view(torch.int16))
    assert_close(out, ref, f"D{head_dim} {hq}/{hkv}")
    assert torch.count_nonzero(out[0]) == 0
    assert device_errors() == 0


def test_position_past_the_table_is_flagged():
    c = make_decode_case("tiny", seed=64)
    table = rope_cos_sin(20, 64, 1e4)            # lengths reach 40
    _run(c, table)
    assert device_errors() & pkv.DEVERR_POSITION_OUT_OF_TABLE
