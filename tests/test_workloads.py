"""Host-side checks of the seeded workload generator and block allocator (CPU only)."""
import math

import torch

from workloads import (BLOCK_SIZE, SPECS, TRACE, BlockAllocator, TraceGenerator, TraceSpec, algorithmic_bytes,
                       draw_lengths, make_decode_case, make_generator)


def test_same_seed_same_tensors():
    a = make_decode_case("tiny", seed=0)
    b = make_decode_case("tiny", seed=0)
    for x, y in ((a.q, b.q), (a.k_cache, b.k_cache), (a.block_tables, b.block_tables), (a.new_v, b.new_v)):
        assert torch.equal(x, y)
    c = make_decode_case("tiny", seed=1)
    assert not torch.equal(a.q, c.q)


def test_tiny_workload_shape():
    c = make_decode_case("tiny")
    assert c.context_lens.tolist() == [5, 16, 17, 40]
    assert c.k_cache.shape == (16, 1, BLOCK_SIZE, 64)
    assert c.q.shape == (4, 2, 64)
    used = c.block_tables[c.block_tables >= 0]
    assert used.numel() == 1 + 1 + 2 + 3 and len(set(used.tolist())) == used.numel()
    assert c.scale == 1 / 8


def test_slot_mapping_is_last_position():
    c = make_decode_case("qwen3_0.6b", lengths=[1, 16, 17, 300])
    for b, L in enumerate(c.context_lens.tolist()):
        s = int(c.slot_mapping[b])
        assert s // BLOCK_SIZE == int(c.block_tables[b, (L - 1) // BLOCK_SIZE])
        assert s % BLOCK_SIZE == (L - 1) % BLOCK_SIZE


def test_length_distributions():
    g = make_generator(0)
    lens = draw_lengths(SPECS["llama3_8b"], g)
    assert len(lens) == 128 and min(lens) >= 512 and max(lens) <= 4096
    g = make_generator(0)
    lens = draw_lengths(SPECS["long_skew"], g)
    assert lens[0] == 131072 and all(16 <= L <= 65536 for L in lens[1:])
    # log-uniform: the median sits near the geometric mean of the range.
    med = sorted(lens[1:])[len(lens) // 2]
    assert 200 < med < 5000


def test_llama3_70b_layer_shares_the_8b_lengths():
    """The LLaMA-3-70B layer (eight q heads per kv head) draws the same lengths and pool as the 8B one."""
    a, b = SPECS["llama3_8b"], SPECS["llama3_70b"]
    assert (b.num_q_heads, b.num_kv_heads, b.head_dim) == (64, 8, 128)
    assert (b.num_seqs, b.length_range, b.max_blocks_per_seq) == (a.num_seqs, a.length_range, a.max_blocks_per_seq)
    assert draw_lengths(a, make_generator(0)) == draw_lengths(b, make_generator(0))
    c = make_decode_case("llama3_70b", seed=0, num_seqs=4)
    assert c.q.shape == (4, 64, 128) and c.k_cache.shape[1:] == (8, BLOCK_SIZE, 128)


def test_allocator_takes_block_only_when_full_and_frees_all():
    g = make_generator(3)
    a = BlockAllocator(10, g)
    a.add_sequence(0, 0)
    slots = [a.append_token(0) for _ in range(33)]
    assert len(a.blocks[0]) == 3                 # 33 tokens -> 3 blocks
    assert len(set(slots)) == 33
    assert a.num_free() == 7
    a.free_sequence(0)
    assert a.num_free() == 10
    assert sorted(a.free[a._head:]) == list(range(10))


def test_trace_schedule_invariants():
    spec = TraceSpec(steps=12, max_seqs=32)
    tg = TraceGenerator(spec, seed=0)
    seen_join = seen_finish = False
    for st in tg.steps():
        B = len(st.seq_ids)
        assert 0 < B <= spec.max_seqs
        assert st.slot_mapping.shape == (B,) and st.block_tables.shape == (B, tg.width)
        # Every live block belongs to exactly one sequence.
        live = st.block_tables[st.block_tables >= 0].tolist()
        assert len(live) == len(set(live))
        for r, sid in enumerate(st.seq_ids):
            L = int(st.context_lens[r])
            assert (st.block_tables[r] >= 0).sum().item() == math.ceil(L / BLOCK_SIZE)
            s = int(st.slot_mapping[r])
            assert s // BLOCK_SIZE == int(st.block_tables[r, (L - 1) // BLOCK_SIZE])
        seen_join |= bool(st.joined)
        seen_finish |= bool(st.finished)
    assert seen_join and seen_finish


def test_algorithmic_bytes_formula():
    # One sequence of 17 tokens, 1 kv head, D 64, 2 q heads.
    n = algorithmic_bytes([17], 2, 1, 64)
    assert n == 2 * 17 * 64 * 2 + 4 * 2 + (4 + 2 * 2 * 64 * 2)


def test_default_trace_spec():
    assert TRACE.num_layers == 28 and TRACE.max_seqs == 256 and TRACE.steps == 100
