"""Paged decode attention on the GPU against the fp64 oracle.

Tolerance (bf16 inputs, fp32 accumulation, one bf16 rounding of the output):
max |gpu - oracle| <= 1e-2 and relative RMS <= 5e-3, on every output element.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_275_gb300 as pkv
from gpu_util import assert_close, device_errors, gpu_step, oracle_step
from workloads import BLOCK_SIZE, SPECS, DecodeSpec, make_decode_case, make_generator, randn_bf16

pytestmark = pytest.mark.gpu


# The Qwen3 workload with eight q heads per kv head (64 q / 8 kv): the tensor-core path.
QWEN3_G8 = DecodeSpec(name="qwen3_g8", description="Qwen3 lengths, 64 q / 8 kv heads, D 128", num_seqs=32,
                      num_q_heads=64, num_kv_heads=8, head_dim=128, max_blocks_per_seq=128, length_kind="uniform",
                      length_range=(128, 2048), pool_slack=0.10)
BOTH_PATHS = pytest.mark.parametrize("shape", ["qwen3_0.6b", QWEN3_G8], ids=["G2_cuda_cores", "G8_tensor_cores"])


def _run(c, num_partitions=0):
    g = c.to("cuda")
    out = gpu_step(g, num_partitions)
    torch.cuda.synchronize()
    return g, out


# ---------------------------------------------------------------------------
# Parity on the workloads (every output element)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_every_partition_count(seed):
    """Tiny workload (lens 5, 16, 17, 40; D 64; G 2) under every way of cutting its 7 blocks."""
    c = make_decode_case("tiny", seed=seed)
    ref, _, _ = oracle_step(c)
    for parts in (0, 1, 2, 3, 5, 7, 12):
        _, out = _run(c, parts)
        assert_close(out, ref, f"tiny seed {seed} parts {parts}")
    assert device_errors() == 0


def test_qwen3_layer_full():
    c = make_decode_case("qwen3_0.6b", seed=0)
    ref, _, _ = oracle_step(c)
    for parts in (0, 1, 64, 333):
        _, out = _run(c, parts)
        assert_close(out, ref, f"qwen3_0.6b parts {parts}")
    assert device_errors() == 0


def test_llama3_layer_full():
    """The benchmarked workload at full size, default launch configuration, every output."""
    c = make_decode_case("llama3_8b", seed=0)
    ref, _, _ = oracle_step(c)
    _, out = _run(c, 0)
    assert_close(out, ref, "llama3_8b")
    assert device_errors() == 0


def test_llama3_70b_layer_full():
    """Groups of eight q heads (64 q / 8 kv), which run in two four-head passes per K/V tile."""
    c = make_decode_case("llama3_70b", seed=0)
    ref, _, _ = oracle_step(c)
    for parts in (0, 97):
        _, out = _run(c, parts)
        assert_close(out, ref, f"llama3_70b parts {parts}")
    assert device_errors() == 0


def test_long_context_skew_full():
    """Log-uniform lengths 16..65536 plus one 131072-token sequence (8192 blocks)."""
    c = make_decode_case("long_skew", seed=0)
    ref, _, _ = oracle_step(c)
    _, out = _run(c, 0)
    assert_close(out, ref, "long_skew")
    assert_close(out[0:1], ref[0:1], "long_skew 131072-token sequence")
    assert device_errors() == 0


@pytest.mark.parametrize("head_dim,hq,hkv", [(64, 1, 1), (64, 4, 1), (64, 16, 2), (128, 8, 8), (128, 16, 4),
                                             (128, 32, 4)])
def test_every_head_layout(head_dim, hq, hkv):
    """Every built (head_dim, group) instance, G in {1, 2, 4, 8}, on ragged lengths."""
    spec = DecodeSpec(name="layout", description="", num_seqs=9, num_q_heads=hq, num_kv_heads=hkv,
                      head_dim=head_dim, max_blocks_per_seq=40, length_kind="fixed",
                      lengths=(1, 2, 15, 16, 17, 31, 200, 511, 640), pool_slack=0.2)
    c = make_decode_case(spec, seed=5)
    ref, _, _ = oracle_step(c)
    for parts in (0, 1, 13):
        _, out = _run(c, parts)
        assert_close(out, ref, f"D{head_dim} Hq{hq} Hkv{hkv} parts {parts}")
    assert device_errors() == 0


def test_every_length_through_three_blocks():
    """Lengths 0..48 (every block offset, empty sequences) in one batch."""
    spec = DecodeSpec(name="lens", description="", num_seqs=49, num_q_heads=16, num_kv_heads=8, head_dim=128,
                      max_blocks_per_seq=3, length_kind="fixed", lengths=tuple(range(49)), pool_slack=0.1)
    c = make_decode_case(spec, seed=6)
    # Length-0 sequences have no token: give their append a padding slot.
    c.slot_mapping[c.context_lens == 0] = -1
    ref, _, _ = oracle_step(c)
    for parts in (0, 1, 5, 97):
        _, out = _run(c, parts)
        assert_close(out, ref, f"lengths 0..48 parts {parts}")
        assert torch.count_nonzero(out[0]) == 0
    assert device_errors() == 0


@pytest.mark.parametrize("seed", range(8))
def test_random_shapes(seed):
    """Seeded random layouts, batch sizes, length mixes (empty to a few thousand tokens) and
    partition counts (the default, one, and a random count that may exceed the work)."""
    import random
    rng = random.Random(3000 + seed)
    d = rng.choice([64, 128])
    hkv = rng.choice([1, 2, 4, 8])
    g = rng.choice([1, 2, 4, 8])
    b = rng.randint(1, 40)
    lens = tuple(rng.choice([0, rng.randint(1, 48), rng.randint(48, 3000)]) for _ in range(b))
    width = max(1, max(-(-L // BLOCK_SIZE) for L in lens)) + rng.randint(0, 3)
    spec = DecodeSpec(name="random", description="", num_seqs=b, num_q_heads=hkv * g, num_kv_heads=hkv,
                      head_dim=d, max_blocks_per_seq=width, length_kind="fixed", lengths=lens,
                      pool_slack=rng.choice([0.0, 0.3]))
    c = make_decode_case(spec, seed=4000 + seed)
    c.slot_mapping[c.context_lens == 0] = -1
    ref, _, _ = oracle_step(c)
    for parts in (0, 1, rng.randint(2, 3000)):
        _, out = _run(c, parts)
        assert_close(out, ref, f"seed {seed}: D{d} {hkv * g}/{hkv} B{b} parts {parts}")
    assert device_errors() == 0


# ---------------------------------------------------------------------------
# Invariants and special cases
# ---------------------------------------------------------------------------
@BOTH_PATHS
def test_single_token_returns_its_value_exactly(shape):
    c = make_decode_case(shape, seed=7, lengths=[1] * 8)
    g, out = _run(c, 0)
    # The one cached token is the appended one.
    expect = c.new_v.repeat_interleave(c.q.shape[1] // c.k_cache.shape[1], dim=1)
    assert torch.equal(out.cpu(), expect)


@BOTH_PATHS
def test_block_relabelling_is_bit_identical(shape):
    c = make_decode_case(shape, seed=8)
    _, out1 = _run(c, 0)
    perm = torch.randperm(c.num_blocks, generator=make_generator(3))
    kc2 = torch.empty_like(c.k_cache)
    vc2 = torch.empty_like(c.v_cache)
    kc2[perm] = c.k_cache
    vc2[perm] = c.v_cache
    c.k_cache, c.v_cache = kc2, vc2
    c.block_tables = torch.where(c.block_tables >= 0, perm[c.block_tables.clamp(min=0).long()].to(torch.int32),
                                 c.block_tables)
    c.slot_mapping = perm[c.slot_mapping // BLOCK_SIZE] * BLOCK_SIZE + c.slot_mapping % BLOCK_SIZE
    _, out2 = _run(c, 0)
    assert torch.equal(out1, out2)


@pytest.mark.parametrize("shape", ["llama3_8b", "llama3_70b"])
def test_repeated_runs_are_bit_identical(shape):
    c = make_decode_case(shape, seed=9, num_seqs=48)
    g = c.to("cuda")
    pkv.kv_append(g.new_k, g.new_v, g.slot_mapping, g.k_cache, g.v_cache)
    outs = []
    for _ in range(3):
        o = torch.empty_like(g.q)
        pkv.paged_decode_attention(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale, o)
        outs.append(o)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


@BOTH_PATHS
def test_poisoned_unused_slots_do_not_leak(shape):
    """NaN in every slot no sequence owns and garbage past each table row: output unchanged."""
    c = make_decode_case(shape, seed=10)
    _, clean = _run(c, 0)
    used = torch.zeros(c.num_blocks * BLOCK_SIZE, dtype=torch.bool)
    for sid in range(c.spec.num_seqs):
        for p in range(c.allocator.length[sid]):
            used[c.allocator.slot(sid, p)] = True
    unused = (~used).view(c.num_blocks, BLOCK_SIZE)
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16)
    c.k_cache.permute(0, 2, 1, 3)[unused] = nan
    c.v_cache.permute(0, 2, 1, 3)[unused] = nan
    c.block_tables[c.block_tables < 0] = 10 ** 8
    for parts in (0, 1, 77):
        _, out = _run(c, parts)
        assert torch.isfinite(out.float()).all()
        if parts == 0:
            assert torch.equal(out, clean)
    assert device_errors() == 0


@BOTH_PATHS
def test_partition_counts_agree(shape):
    """Cutting the block stream differently changes only rounding: the fp32 sums' order, and on the
    tensor-core path also the running maxima the bf16 weights are rounded against."""
    c = make_decode_case(shape, seed=11)
    _, base = _run(c, 1)
    share = []
    for parts in (2, 7, 100, 1000, 0):
        _, out = _run(c, parts)
        d = (out.float() - base.float()).abs()
        assert d.max().item() <= 2 * 2 ** -8 * max(1.0, base.float().abs().max().item())
        share.append((d > 0).float().mean().item())
    print(f"{c.spec.name}: share of outputs that differ from one piece per pair: {share}")
    assert max(share) < 0.05


@BOTH_PATHS
def test_huge_scale_selects_argmax(shape):
    c = make_decode_case(shape, seed=12, lengths=[5, 40, 300])
    g = c.to("cuda")
    pkv.kv_append(g.new_k, g.new_v, g.slot_mapping, g.k_cache, g.v_cache)
    out = torch.empty_like(g.q)
    pkv.paged_decode_attention(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, 50.0, out)
    _, kc, vc = oracle_step(c)
    ref, st = oracle.paged_decode_attention(c.q, kc, vc, c.block_tables, c.context_lens, 50.0)
    assert st == 0
    assert_close(out, ref, "scale 50")


def test_phases_split_equals_single_call():
    c = make_decode_case("qwen3_0.6b", seed=13)
    g = c.to("cuda")
    pkv.kv_append(g.new_k, g.new_v, g.slot_mapping, g.k_cache, g.v_cache)
    a = torch.empty_like(g.q)
    b = torch.empty_like(g.q)
    pkv.paged_decode_attention(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale, a)
    pkv.paged_decode_attention(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale, b,
                               phases=pkv.PHASE_PARTITION)
    pkv.paged_decode_attention(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale, b,
                               phases=pkv.PHASE_MERGE)
    assert torch.equal(a, b)


# ---------------------------------------------------------------------------
# Device-side errors: flagged, skipped, never a fault
# ---------------------------------------------------------------------------
def test_bad_block_id_and_lengths_are_flagged():
    c = make_decode_case("tiny", seed=14)
    g = c.to("cuda")
    out = torch.empty_like(g.q)
    assert device_errors() == 0
    bt = g.block_tables.clone()
    bt[3, 1] = 1000
    pkv.paged_decode_attention(g.q, g.k_cache, g.v_cache, bt, g.context_lens, g.scale, out)
    assert device_errors() & pkv.DEVERR_BLOCK_ID_OUT_OF_RANGE
    cl = g.context_lens.clone()
    cl[0] = -4
    cl[1] = 3 * BLOCK_SIZE + 1
    pkv.paged_decode_attention(g.q, g.k_cache, g.v_cache, g.block_tables, cl, g.scale, out)
    bits = device_errors()
    assert bits & pkv.DEVERR_CONTEXT_LEN_NEGATIVE and bits & pkv.DEVERR_CONTEXT_LEN_TOO_LONG
    assert torch.count_nonzero(out[0]) == 0   # a negative length reads as empty
    # The GPU stays usable: a clean call succeeds and raises nothing.
    ref, _ = oracle.paged_decode_attention(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale)
    pkv.paged_decode_attention(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale, out)
    assert_close(out, ref, "after errors")
    assert device_errors() == 0


@pytest.mark.parametrize("head_dim,hq,hkv", [(64, 8, 2), (128, 16, 2)])
def test_largest_batch(head_dim, hq, hkv):
    """num_seqs = PKV_MAX_SEQS (4096) short sequences, empty ones among them: every CTA ranks and
    prefixes the whole batch in shared memory (at D = 128 with eight q heads per kv head, next to the
    largest ring of swizzled tensor-copy stages)."""
    import random
    rng = random.Random(77)
    lens = tuple(rng.choice([0, rng.randint(1, 40)]) for _ in range(pkv.MAX_SEQS))
    spec = DecodeSpec(name="max_batch", description="", num_seqs=pkv.MAX_SEQS, num_q_heads=hq, num_kv_heads=hkv,
                      head_dim=head_dim, max_blocks_per_seq=3, length_kind="fixed", lengths=lens, pool_slack=0.1)
    c = make_decode_case(spec, seed=78)
    c.slot_mapping[c.context_lens == 0] = -1
    ref, _, _ = oracle_step(c)
    for parts in (0, 1000):
        _, out = _run(c, parts)
        assert_close(out, ref, f"4096 sequences parts {parts}")
    assert device_errors() == 0


def test_batch_larger_than_one_launch():
    """5000 sequences (more than PKV_MAX_SEQS = 4096 per launch pair): the call runs as a slice of 4096
    and one of 904 on the same workspace.  Its output equals, bit for bit, two calls made on those
    slices, and matches the oracle; the fused decode step too.  (Lengths of 16 to 40 tokens, or
    empty: a one- or two-token sequence can give outputs above 4, where one bf16 rounding step alone
    exceeds the 1e-2 absolute tolerance.)"""
    import random
    rng = random.Random(79)
    n = pkv.MAX_SEQS + 904
    lens = tuple(rng.choice([0, rng.randint(16, 40)]) for _ in range(n))
    spec = DecodeSpec(name="over_max_batch", description="", num_seqs=n, num_q_heads=16, num_kv_heads=2,
                      head_dim=128, max_blocks_per_seq=3, length_kind="fixed", lengths=lens, pool_slack=0.1)
    c = make_decode_case(spec, seed=80)
    c.slot_mapping[c.context_lens == 0] = -1
    ref, _, _ = oracle_step(c)
    before = pkv.kernel_launch_count()
    g, out = _run(c, 0)
    assert pkv.kernel_launch_count() - before == 1 + 2 * 2   # append, then two partition + merge pairs
    assert_close(out, ref, "5000 sequences")
    parts = torch.empty_like(g.q)
    for lo, hi in ((0, pkv.MAX_SEQS), (pkv.MAX_SEQS, n)):
        pkv.paged_decode_attention(g.q[lo:hi], g.k_cache, g.v_cache, g.block_tables[lo:hi].contiguous(),
                                   g.context_lens[lo:hi].contiguous(), g.scale, parts[lo:hi])
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), parts.view(torch.int16))
    g2 = c.to("cuda")
    step_out = torch.empty_like(g2.q)
    pkv.decode_step(g2.q, g2.new_k, g2.new_v, g2.k_cache, g2.v_cache, g2.block_tables, g2.context_lens, g2.scale,
                    step_out)
    torch.cuda.synchronize()
    assert_close(step_out, ref, "5000 sequences, fused step")
    assert device_errors() == 0


def test_host_errors_raise_before_launch():
    c = make_decode_case("tiny", seed=15).to("cuda")
    before = pkv.kernel_launch_count()
    with pytest.raises(ValueError, match="workspace"):
        pkv.paged_decode_attention(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale,
                                   torch.empty_like(c.q), workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert pkv.kernel_launch_count() == before
