"""Chunked paged prefill on the tensor cores against the fp64 oracle (every output element).

Tolerance as for decode: max |gpu - oracle| <= 1e-2, relative RMS <= 5e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_275_gb300 as pkv
from gpu_util import assert_close, device_errors
from workloads import BLOCK_SIZE, PrefillSpec, make_prefill_case

pytestmark = pytest.mark.gpu


def _run(c):
    g = c.to("cuda")
    pkv.kv_append(g.new_k, g.new_v, g.slot_mapping, g.k_cache, g.v_cache)
    out = torch.full_like(g.q, float("nan"))
    max_q = int(max(c.spec.chunk_lens))
    pkv.paged_prefill_attention(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.query_start, max_q,
                                g.scale, out)
    torch.cuda.synchronize()
    return g, out


def _ref(c):
    kc, vc = c.k_cache.clone(), c.v_cache.clone()
    assert oracle.kv_append(c.new_k, c.new_v, c.slot_mapping, kc, vc) == oracle.OK
    ref, st = oracle.paged_prefill_attention(c.q, kc, vc, c.block_tables, c.context_lens, c.query_start, c.scale)
    assert st == oracle.OK
    return ref


@pytest.mark.parametrize("seed", [0, 1])
def test_prefill_tiny(seed):
    c = make_prefill_case("prefill_tiny", seed=seed)
    _, out = _run(c)
    assert_close(out, _ref(c), f"prefill_tiny seed {seed}")
    assert device_errors() == 0


@pytest.mark.parametrize("head_dim,hq,hkv", [(128, 8, 8), (128, 16, 8), (128, 32, 8), (128, 32, 4), (64, 4, 4),
                                             (64, 16, 4)])
def test_prefill_every_layout_ragged(head_dim, hq, hkv):
    spec = PrefillSpec("ragged", "", hq, hkv, head_dim, (1, 7, 37, 130, 16), (0, 0), 60)
    c = make_prefill_case(spec, seed=5, prefixes=[0, 3, 100, 500, 64])
    _, out = _run(c)
    assert_close(out, _ref(c), f"D{head_dim} {hq}/{hkv}")
    assert device_errors() == 0


def test_prefill_qwen3_chunks():
    c = make_prefill_case("prefill_qwen3_0.6b", seed=0)
    _, out = _run(c)
    assert_close(out, _ref(c), "prefill_qwen3_0.6b")
    assert device_errors() == 0


def test_prefill_llama3_chunks():
    c = make_prefill_case("prefill_llama3_8b", seed=0)
    _, out = _run(c)
    assert_close(out, _ref(c), "prefill_llama3_8b")
    assert device_errors() == 0


def test_prefill_chunks_of_one_match_decode():
    spec = PrefillSpec("ones", "", 32, 8, 128, (1,) * 6, (0, 300), 30)
    c = make_prefill_case(spec, seed=7)
    g, out = _run(c)
    dec = torch.empty_like(g.q)
    pkv.paged_decode_attention(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale, dec)
    ref = _ref(c)
    assert_close(out, ref, "chunks of one")
    assert_close(dec, ref, "decode on the same rows")


@pytest.mark.parametrize("num_seqs", [320, 321])
def test_prefill_many_sequences_either_side_of_the_ranking_limit(num_seqs):
    """Up to 320 sequences each CTA ranks them by length to pick its own; beyond that the grid takes
    them in index order.  Both orders must give the oracle's result."""
    import random
    rng = random.Random(num_seqs)
    chunks = tuple(rng.randint(1, 24) for _ in range(num_seqs))
    spec = PrefillSpec("many", "", 8, 2, 64, chunks, (0, 100), 9)
    c = make_prefill_case(spec, seed=num_seqs)
    _, out = _run(c)
    assert_close(out, _ref(c), f"{num_seqs} sequences")
    assert device_errors() == 0


def test_prefill_long_prefix():
    """A 20000-token prefix: about 160 key steps and 1250 pages, so the block-id window slides ~40 times."""
    spec = PrefillSpec("long", "", 8, 2, 128, (16, 3, 200), (0, 0), 1270)
    c = make_prefill_case(spec, seed=12, prefixes=[20000, 5000, 300])
    _, out = _run(c)
    assert_close(out, _ref(c), "long prefix")
    assert device_errors() == 0


def test_prefill_long_chunk_spans_many_grid_rows():
    """A 2048-token chunk at G = 8 (32 chunk tokens a CTA): 64 CTAs of one sequence and kv head along the
    grid's tile dimension, launched longest first, beside a short chunk whose tiles run out early."""
    spec = PrefillSpec("long_chunk", "", 8, 1, 64, (2048, 45), (0, 0), 140)
    c = make_prefill_case(spec, seed=21, prefixes=[100, 7])
    _, out = _run(c)
    assert_close(out, _ref(c), "long chunk")
    assert device_errors() == 0


@pytest.mark.parametrize("seed", range(8))
def test_prefill_random_shapes(seed):
    """Seeded random layouts: head dim, group size, sequence count, chunk and prefix lengths (chunks from
    one token to several CTAs, prefixes from none to a few thousand tokens)."""
    import random
    rng = random.Random(1000 + seed)
    d = rng.choice([64, 128])
    hkv = rng.choice([1, 2, 4, 8])
    g = rng.choice([1, 2, 4, 8])
    b = rng.randint(1, 12)
    chunks = tuple(rng.choice([1, rng.randint(1, 40), rng.randint(40, 300)]) for _ in range(b))
    prefixes = [rng.choice([0, rng.randint(0, 64), rng.randint(64, 3000)]) for _ in range(b)]
    width = max(-(-(p_ + c_) // BLOCK_SIZE) for p_, c_ in zip(prefixes, chunks)) + rng.randint(0, 3)
    spec = PrefillSpec("random", "", hkv * g, hkv, d, chunks, (0, 0), width)
    c = make_prefill_case(spec, seed=2000 + seed, prefixes=prefixes)
    _, out = _run(c)
    assert_close(out, _ref(c), f"seed {seed}: D{d} {hkv * g}/{hkv} chunks {chunks} prefixes {prefixes}")
    assert device_errors() == 0


def test_prefill_poisoned_unused_slots_do_not_leak():
    c = make_prefill_case("prefill_tiny", seed=8)
    _, clean = _run(c)
    lens = c.context_lens.tolist()
    used = torch.zeros(c.k_cache.shape[0] * BLOCK_SIZE, dtype=torch.bool)
    for b, L in enumerate(lens):
        for t in range(L):
            used[int(c.block_tables[b, t // BLOCK_SIZE]) * BLOCK_SIZE + t % BLOCK_SIZE] = True
    unused = (~used).view(c.k_cache.shape[0], BLOCK_SIZE)
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16)
    c.k_cache.permute(0, 2, 1, 3)[unused] = nan
    c.v_cache.permute(0, 2, 1, 3)[unused] = nan
    _, out = _run(c)
    assert torch.isfinite(out.float()).all()
    assert torch.equal(out, clean)
    assert device_errors() == 0


@pytest.mark.parametrize("num_splits", [1, 2], ids=["unsplit", "split2"])
def test_prefill_device_errors_are_flagged_and_the_gpu_stays_usable(num_splits):
    c = make_prefill_case("prefill_tiny", seed=9)
    g = c.to("cuda")
    pkv.kv_append(g.new_k, g.new_v, g.slot_mapping, g.k_cache, g.v_cache)
    out = torch.empty_like(g.q)
    assert device_errors() == 0
    bt = g.block_tables.clone()
    bt[1, 0] = 10 ** 6
    pkv.paged_prefill_attention(g.q, g.k_cache, g.v_cache, bt, g.context_lens, g.query_start, 40, g.scale, out,
                                num_splits=num_splits)
    assert device_errors() & pkv.DEVERR_BLOCK_ID_OUT_OF_RANGE
    # max_query_len smaller than a chunk: that chunk's rows past the grid are not covered, and it is flagged.
    pkv.paged_prefill_attention(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.query_start, 8,
                                g.scale, out, num_splits=num_splits)
    bits = device_errors()
    assert bits & pkv.DEVERR_CONTEXT_LEN_TOO_LONG and not bits & pkv.DEVERR_SMEM_ALIGNMENT
    # A clean call afterwards is correct.
    pkv.paged_prefill_attention(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.query_start, 40,
                                g.scale, out, num_splits=num_splits)
    assert_close(out, _ref(c), "after errors")
    assert device_errors() == 0


def test_prefill_host_errors_raise_before_launch():
    c = make_prefill_case("prefill_tiny", seed=10).to("cuda")
    before = pkv.kernel_launch_count()
    with pytest.raises(pkv.PagedKVError):
        pkv.paged_prefill_attention(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.query_start, -1,
                                    c.scale, torch.empty_like(c.q))
    with pytest.raises(pkv.PagedKVError):
        pkv.paged_prefill_attention(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.query_start, 40,
                                    float("nan"), torch.empty_like(c.q))
    assert pkv.kernel_launch_count() == before


# ---- Split-K over the key steps (pkv_paged_prefill_attention_split) ----

def _run_split(c, num_splits):
    g = c.to("cuda")
    pkv.kv_append(g.new_k, g.new_v, g.slot_mapping, g.k_cache, g.v_cache)
    out = torch.full_like(g.q, float("nan"))
    max_q = int(max(c.spec.chunk_lens))
    pkv.paged_prefill_attention(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.query_start, max_q,
                                g.scale, out, num_splits=num_splits)
    torch.cuda.synchronize()
    return g, out


@pytest.mark.parametrize("num_splits", [2, 3, 7])
@pytest.mark.parametrize("head_dim,hq,hkv", [(128, 32, 8), (128, 16, 8), (64, 4, 4), (128, 64, 8)])
def test_prefill_split_every_layout_ragged(head_dim, hq, hkv, num_splits):
    """Chunks of 1..130 tokens after 0..500 cached ones: one to five key steps a tile, so with 7 splits most
    CTAs of a short tile have no step and only mark their rows empty."""
    spec = PrefillSpec("ragged", "", hq, hkv, head_dim, (1, 7, 37, 130, 16), (0, 0), 60)
    c = make_prefill_case(spec, seed=6, prefixes=[0, 3, 100, 500, 64])
    _, out = _run_split(c, num_splits)
    assert_close(out, _ref(c), f"split {num_splits} D{head_dim} {hq}/{hkv}")
    assert device_errors() == 0


def test_prefill_split_qwen3_chunks_agree_with_the_unsplit_call():
    c = make_prefill_case("prefill_qwen3_0.6b", seed=3)
    _, whole = _run(c)
    _, split = _run_split(c, 3)
    ref = _ref(c)
    assert_close(split, ref, "prefill_qwen3_0.6b split 3")
    # Same math, fp32 partial states merged in another order: a bf16 step apart at most.
    assert (split.float() - whole.float()).abs().max().item() <= 2 * 2 ** -7 * max(1.0, whole.float().abs().max().item())
    assert device_errors() == 0


def test_prefill_split_long_prefix():
    """A 20 000-token prefix split five ways: each CTA's block-id window starts mid-table."""
    spec = PrefillSpec("long", "", 8, 2, 128, (16, 3, 200), (0, 0), 1270)
    c = make_prefill_case(spec, seed=13, prefixes=[20000, 5000, 300])
    _, out = _run_split(c, 5)
    assert_close(out, _ref(c), "long prefix split 5")
    assert device_errors() == 0


def test_prefill_split_long_chunk():
    spec = PrefillSpec("long_chunk", "", 8, 1, 64, (2048, 45), (0, 0), 140)
    c = make_prefill_case(spec, seed=22, prefixes=[100, 7])
    _, out = _run_split(c, 4)
    assert_close(out, _ref(c), "long chunk split 4")
    assert device_errors() == 0


def test_prefill_split_graph_replay_is_bit_identical():
    c = make_prefill_case("prefill_tiny", seed=4).to("cuda")
    pkv.kv_append(c.new_k, c.new_v, c.slot_mapping, c.k_cache, c.v_cache)
    max_q = int(max(c.spec.chunk_lens))
    B, hq, d = c.context_lens.shape[0], c.q.shape[1], c.q.shape[2]
    ws = torch.empty(pkv.prefill_workspace_size(B, max_q, hq, c.k_cache.shape[1], d, 3), dtype=torch.uint8,
                     device="cuda")
    eager = torch.empty_like(c.q)
    call = lambda o, s=None: pkv.paged_prefill_attention(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens,
                                                         c.query_start, max_q, c.scale, o, stream=s, num_splits=3,
                                                         workspace=ws)
    call(eager)
    torch.cuda.synchronize()
    out = torch.zeros_like(c.q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call(out, s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(out, s)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert device_errors() == 0


def test_prefill_default_splits_fill_one_wave():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # One LLaMA-3 chunk of 512: 8 kv heads x 8 CTAs of 64 tokens.
    assert pkv.prefill_default_splits(1, 512, 32, 8) == max(1, min(32, sms // 64))
    assert pkv.prefill_default_splits(8, 512, 32, 8) == max(1, min(32, sms // 512))   # already fills the GPU
    assert pkv.prefill_default_splits(1, 16, 8, 1) == min(32, sms)                       # a single CTA
