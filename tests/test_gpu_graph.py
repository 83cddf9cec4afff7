"""The calls are stream-ordered and host-sync-free: captured in a CUDA graph (with their workspaces
passed in), replays give bit for bit what eager calls give."""
import pytest
import torch

import paged_kv_cache_275_gb300 as pkv
from gpu_util import device_errors
from workloads import DecodeSpec, make_decode_case, make_prefill_case, rope_cos_sin

# Eight q heads per kv head: the tensor-core path (its K/V tensor maps travel as kernel parameters).
G8 = DecodeSpec(name="g8_graph", description="", num_seqs=24, num_q_heads=32, num_kv_heads=4, head_dim=128,
                max_blocks_per_seq=64, length_kind="uniform", length_range=(1, 1000), pool_slack=0.1)

pytestmark = pytest.mark.gpu


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn(s)  # warm-up on the capture stream (loads the library, sets kernel attributes)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn(s)
    return g


@pytest.mark.parametrize("shape", ["qwen3_0.6b", G8], ids=["G2", "G8"])
def test_decode_step_graph_replay_is_bit_identical(shape):
    c = make_decode_case(shape, seed=90).to("cuda")
    B, hq, d = c.q.shape
    ws = torch.empty(pkv.workspace_size(B, hq, c.k_cache.shape[1], d, c.block_tables.shape[1]), dtype=torch.uint8,
                     device="cuda")
    eager = torch.empty_like(c.q)
    pkv.kv_append(c.new_k, c.new_v, c.slot_mapping, c.k_cache, c.v_cache)
    pkv.paged_decode_attention(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale, eager, workspace=ws)
    torch.cuda.synchronize()
    out = torch.zeros_like(c.q)

    def step(s):
        pkv.kv_append(c.new_k, c.new_v, c.slot_mapping, c.k_cache, c.v_cache, stream=s)
        pkv.paged_decode_attention(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale, out,
                                   workspace=ws, stream=s)

    g = _capture(step)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert device_errors() == 0


@pytest.mark.parametrize("shape", ["tiny", G8], ids=["tiny", "G8"])
def test_fused_step_graph_replay_is_bit_identical(shape):
    c = make_decode_case(shape, seed=91).to("cuda")
    B, hq, d = c.q.shape
    table = rope_cos_sin(c.block_tables.shape[1] * 16, d, 1e4).cuda()
    ws = torch.empty(pkv.workspace_size(B, hq, c.k_cache.shape[1], d, c.block_tables.shape[1]), dtype=torch.uint8,
                     device="cuda")
    k0, v0 = c.k_cache.clone(), c.v_cache.clone()
    eager = torch.empty_like(c.q)
    pkv.decode_step(c.q, c.new_k, c.new_v, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale, eager,
                    table, workspace=ws)
    torch.cuda.synchronize()
    k1, v1 = c.k_cache.clone(), c.v_cache.clone()
    out = torch.zeros_like(c.q)

    def step(s):
        pkv.decode_step(c.q, c.new_k, c.new_v, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale, out,
                        table, workspace=ws, stream=s)

    g = _capture(step)
    for _ in range(2):
        c.k_cache.copy_(k0)
        c.v_cache.copy_(v0)
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager) and torch.equal(c.k_cache, k1) and torch.equal(c.v_cache, v1)
    assert device_errors() == 0


def test_prefill_graph_replay_is_bit_identical():
    c = make_prefill_case("prefill_qwen3_0.6b", seed=92).to("cuda")
    pkv.kv_append(c.new_k, c.new_v, c.slot_mapping, c.k_cache, c.v_cache)
    max_q = int(max(c.spec.chunk_lens))
    eager = torch.empty_like(c.q)
    pkv.paged_prefill_attention(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.query_start, max_q,
                                c.scale, eager)
    torch.cuda.synchronize()
    out = torch.zeros_like(c.q)

    def call(s):
        pkv.paged_prefill_attention(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.query_start, max_q,
                                    c.scale, out, stream=s)

    g = _capture(call)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert device_errors() == 0
