"""Pins for the CPU oracle: each test ties it to something other than itself.

The pages print no worked numerical example, so the pins are closed forms,
invariants of the definition, special cases that reduce to a library routine
(torch's float64 scaled-dot-product attention on un-paged tensors, numpy
indexing), and brute force on tiny inputs.  Each test names the mistake it
would catch.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from workloads import BLOCK_SIZE, BlockAllocator, make_decode_case, make_generator, randn_bf16

pytestmark = pytest.mark.usefixtures("oracle_lib")


def f64(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.float64)


def contiguous_kv(case_k, case_v, block_tables, context_lens, b):
    """Un-paged K/V of sequence b, [Hkv, L, D] float64, via torch advanced indexing on a slot view."""
    L = int(context_lens[b])
    nb, hkv, bs, d = case_k.shape
    pos = torch.arange(L)
    slots = block_tables[b, pos // bs].to(torch.int64) * bs + pos % bs
    kflat = case_k.permute(0, 2, 1, 3).reshape(nb * bs, hkv, d)
    vflat = case_v.permute(0, 2, 1, 3).reshape(nb * bs, hkv, d)
    return f64(kflat[slots]).permute(1, 0, 2), f64(vflat[slots]).permute(1, 0, 2)


def sdpa_reference(q, k_cache, v_cache, block_tables, context_lens, scale):
    """torch float64 SDPA per sequence on the un-paged K/V, GQA by repeat_interleave."""
    B, hq, d = q.shape
    hkv = k_cache.shape[1]
    out = torch.zeros(B, hq, d, dtype=torch.float64)
    for b in range(B):
        if int(context_lens[b]) == 0:
            continue
        K, V = contiguous_kv(k_cache, v_cache, block_tables, context_lens, b)
        K = K.repeat_interleave(hq // hkv, dim=0)
        V = V.repeat_interleave(hq // hkv, dim=0)
        o = F.scaled_dot_product_attention(f64(q[b]).unsqueeze(1), K, V, scale=scale)
        out[b] = o.squeeze(1)
    return out.numpy()


def run_oracle(q, kc, vc, bt, cl, scale):
    out, st = oracle.paged_decode_attention(q, kc, vc, bt, cl, scale)
    assert st == oracle.OK
    return out


def bf16(x) -> torch.Tensor:
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("scale,kscale", [(1.0, 1.0), (0.5, 2.0), (0.125, 8.0)])
def test_closed_form_softmax_weights(scale, kscale):
    """s_t = t with one-hot V_t: out[d] = e^d / sum_u e^u.  Catches a missing exp, a
    wrong normalisation, a sign error in the softmax and a misapplied scale."""
    D, L = 64, 20                        # 20 tokens: crosses a block edge
    nb = 4
    kc = torch.zeros(nb, 1, BLOCK_SIZE, D, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    table = torch.tensor([[2, 0]], dtype=torch.int32)  # logical block 0 -> physical 2, 1 -> 0
    weights_exp = []
    for t in range(L):
        s = t % 5                         # scores 0..4 repeating
        phys, off = int(table[0, t // BLOCK_SIZE]), t % BLOCK_SIZE
        kc[phys, 0, off, 0] = bf16(s * kscale)
        vc[phys, 0, off, t] = bf16(1.0)  # one-hot value at dim t
        weights_exp.append(math.exp(s))
    q = torch.zeros(1, 1, D, dtype=torch.bfloat16)
    q[0, 0, 0] = 1.0
    out = run_oracle(q, kc, vc, table, torch.tensor([L], dtype=torch.int32), scale)
    total = sum(weights_exp)
    expect = np.zeros(D)
    expect[:L] = [w / total for w in weights_exp]
    np.testing.assert_allclose(out[0, 0], expect, rtol=0, atol=1e-15)


def test_single_token_returns_its_value_exactly():
    """L = 1: the only weight is 1, so out = V_0 exactly.  Catches off-by-one token ranges."""
    case = make_decode_case("tiny", seed=3, lengths=[1, 1, 1, 1])
    out = run_oracle(case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens, case.scale)
    for b in range(4):
        phys = int(case.block_tables[b, 0])
        v0 = f64(case.v_cache[phys, 0, 0]).numpy()
        for h in range(2):
            assert np.array_equal(out[b, h], v0)


def test_zero_query_gives_mean_of_values():
    """q = 0 makes every score equal: out = mean_t V_t (numpy mean).  Catches weights that
    do not sum to one and tokens read twice or skipped."""
    case = make_decode_case("tiny", seed=4)
    q = torch.zeros_like(case.q)
    out = run_oracle(q, case.k_cache, case.v_cache, case.block_tables, case.context_lens, case.scale)
    for b in range(4):
        _, V = contiguous_kv(case.k_cache, case.v_cache, case.block_tables, case.context_lens, b)
        np.testing.assert_allclose(out[b, 0], V[0].numpy().mean(axis=0), rtol=0, atol=1e-14)


def test_huge_scale_selects_argmax_value():
    """As scale grows the softmax tends to a one-hot on the largest score.  Catches a
    reversed softmax (that would pick the smallest score)."""
    case = make_decode_case("tiny", seed=5)
    out = run_oracle(case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens, 1e4)
    for b in range(4):
        K, V = contiguous_kv(case.k_cache, case.v_cache, case.block_tables, case.context_lens, b)
        for h in range(2):
            s = K[0].numpy() @ f64(case.q[b, h]).numpy()
            top2 = np.sort(s)[-2:]
            assert (top2[1] - top2[0]) * 1e4 > 60  # the second-best weight is below e^-60
            np.testing.assert_allclose(out[b, h], V[0, int(np.argmax(s))].numpy(), rtol=0, atol=1e-20)


def test_gqa_head_mapping_contiguous_groups():
    """V constant c_j on kv head j gives out = c_j for every q head of group j, whatever
    the weights.  With Hq = 8, Hkv = 4 this separates h // G from h % Hkv."""
    g = make_generator(11)
    hq, hkv, D, nb = 8, 4, 64, 6
    kc = randn_bf16((nb, hkv, BLOCK_SIZE, D), g)
    vc = torch.zeros_like(kc)
    for j in range(hkv):
        vc[:, j] = bf16(j + 1.0)
    q = randn_bf16((2, hq, D), g)
    table = torch.tensor([[5, 1, 3], [0, 2, -1]], dtype=torch.int32)
    out = run_oracle(q, kc, vc, table, torch.tensor([40, 17], dtype=torch.int32), 0.125)
    for h in range(hq):
        np.testing.assert_allclose(out[:, h], np.full((2, D), h // (hq // hkv) + 1.0), rtol=0, atol=1e-13)


def test_context_len_zero_gives_zeros():
    case = make_decode_case("tiny", seed=6, lengths=[0, 5, 0, 16])
    out = run_oracle(case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens, case.scale)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    assert np.any(out[1] != 0) and np.any(out[3] != 0)


# ---------------------------------------------------------------------------
# Library routine on un-paged tensors; brute force on tiny inputs
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", [0, 1])
def test_tiny_workload_matches_torch_sdpa(seed):
    """The tiny workload (lens 5, 16, 17, 40 over a permuted 16-block pool) against
    torch float64 SDPA on the un-paged K/V.  Catches index, GQA, transposition and
    block-table mistakes."""
    c = make_decode_case("tiny", seed=seed)
    out = run_oracle(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale)
    ref = sdpa_reference(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_qwen_shape_sample_matches_torch_sdpa():
    """Qwen3-0.6B head layout (16 q / 8 kv, D 128) on a few lengths around block edges."""
    lens = [1, 15, 16, 17, 33, 130, 511]
    c = make_decode_case("qwen3_0.6b", seed=7, lengths=lens)
    out = run_oracle(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale)
    ref = sdpa_reference(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_brute_force_every_length_up_to_three_blocks():
    """Every length 0..48 (every offset in three blocks), GQA 2, D 64, vs SDPA."""
    lens = list(range(0, 49))
    spec = make_decode_case("tiny", seed=8, lengths=[1]).spec
    from workloads import DecodeSpec
    spec = DecodeSpec(**{**spec.__dict__, "pool_blocks": None, "pool_slack": 0.3})
    c = make_decode_case(spec, seed=8, lengths=lens)
    out = run_oracle(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, 0.3)
    ref = sdpa_reference(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, 0.3)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Invariants
# ---------------------------------------------------------------------------
def test_physical_block_relabelling_is_invisible():
    """Paging changes where K/V live, not what is computed: relabel every physical block
    by a permutation (cache and tables together) and the output is bit-identical.
    Catches any use of a physical id where a logical position belongs."""
    c = make_decode_case("tiny", seed=9)
    base = run_oracle(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale)
    g = make_generator(99)
    perm = torch.randperm(c.num_blocks, generator=g)
    kc2 = torch.empty_like(c.k_cache)
    vc2 = torch.empty_like(c.v_cache)
    kc2[perm] = c.k_cache
    vc2[perm] = c.v_cache
    bt2 = torch.where(c.block_tables >= 0, perm[c.block_tables.clamp(min=0).long()].to(torch.int32),
                      c.block_tables)
    out2 = run_oracle(c.q, kc2, vc2, bt2, c.context_lens, c.scale)
    assert np.array_equal(base, out2)


def test_unused_slots_and_table_entries_are_never_read():
    """NaN in every slot no sequence owns (block tails and free blocks) and garbage in the
    table past each sequence's blocks change nothing."""
    c = make_decode_case("tiny", seed=10)
    base = run_oracle(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale)
    kc, vc = c.k_cache.clone(), c.v_cache.clone()
    used = torch.zeros(c.num_blocks * BLOCK_SIZE, dtype=torch.bool)
    for sid in range(4):
        for p in range(c.allocator.length[sid]):
            used[c.allocator.slot(sid, p)] = True
    unused = (~used).view(c.num_blocks, BLOCK_SIZE)
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16)
    kc.permute(0, 2, 1, 3)[unused] = nan
    vc.permute(0, 2, 1, 3)[unused] = nan
    bt = c.block_tables.clone()
    bt[bt < 0] = 123456
    out = run_oracle(c.q, kc, vc, bt, c.context_lens, c.scale)
    assert np.isfinite(out).all()
    assert np.array_equal(base, out)


def test_identical_queries_in_a_group_give_identical_outputs():
    c = make_decode_case("qwen3_0.6b", seed=12, lengths=[3, 40, 77])
    q = c.q.clone()
    q[:, 1] = q[:, 0]                    # heads 0 and 1 share kv head 0
    out = run_oracle(q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale)
    assert np.array_equal(out[:, 0], out[:, 1])
    assert not np.array_equal(out[:, 0], out[:, 2])


def test_sampled_equals_full():
    c = make_decode_case("qwen3_0.6b", seed=13, lengths=[5, 300, 64])
    full = run_oracle(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale)
    si = np.array([2, 0, 1, 1], dtype=np.int32)
    hi = np.array([15, 3, 0, 9], dtype=np.int32)
    samp, st = oracle.paged_decode_sampled(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens,
                                           c.scale, si, hi)
    assert st == oracle.OK
    assert np.array_equal(samp, full[si, hi])


def test_bad_block_id_and_length_are_reported():
    c = make_decode_case("tiny", seed=14)
    bt = c.block_tables.clone()
    bt[1, 0] = 99
    _, st = oracle.paged_decode_attention(c.q, c.k_cache, c.v_cache, bt, c.context_lens, c.scale)
    assert st & oracle.BLOCK_ID_OUT_OF_RANGE
    cl = c.context_lens.clone()
    cl[0] = 3 * BLOCK_SIZE + 1
    _, st = oracle.paged_decode_attention(c.q, c.k_cache, c.v_cache, c.block_tables, cl, c.scale)
    assert st & oracle.CONTEXT_LEN_OUT_OF_RANGE


# ---------------------------------------------------------------------------
# Append
# ---------------------------------------------------------------------------
def test_append_writes_exact_bits_at_the_slot_and_nothing_else():
    """Append into a sentinel-filled pool, read back with numpy multi-dimensional indexing
    cache[s // 16, h, s % 16, :].  Catches a swapped block / offset, a wrong head stride
    and stray writes."""
    g = make_generator(21)
    nb, hkv, D, N = 7, 2, 64, 40
    sentinel = torch.tensor(-7.25, dtype=torch.bfloat16)
    kc = torch.full((nb, hkv, BLOCK_SIZE, D), float(sentinel), dtype=torch.bfloat16)
    vc = kc.clone()
    slots = torch.randperm(nb * BLOCK_SIZE, generator=g)[:N].to(torch.int64)
    slots[3] = -1                       # padding: skipped
    k = randn_bf16((N, hkv, D), g)
    v = randn_bf16((N, hkv, D), g)
    assert oracle.kv_append(k, v, slots, kc, vc) == oracle.OK
    kb = kc.view(torch.int16).numpy()
    vb = vc.view(torch.int16).numpy()
    written = np.zeros((nb, BLOCK_SIZE), dtype=bool)
    for i, s in enumerate(slots.tolist()):
        if s < 0:
            continue
        blk, off = divmod(s, BLOCK_SIZE)
        written[blk, off] = True
        assert np.array_equal(kb[blk, :, off, :], k[i].view(torch.int16).numpy())
        assert np.array_equal(vb[blk, :, off, :], v[i].view(torch.int16).numpy())
    sbits = int(sentinel.view(torch.int16))
    assert np.all(kb.transpose(0, 2, 1, 3)[~written] == sbits)
    assert np.all(vb.transpose(0, 2, 1, 3)[~written] == sbits)


def test_append_rejects_out_of_range_and_duplicate_slots():
    g = make_generator(22)
    nb, hkv, D = 2, 1, 64
    kc = torch.zeros(nb, hkv, BLOCK_SIZE, D, dtype=torch.bfloat16)
    vc = kc.clone()
    k = randn_bf16((2, hkv, D), g)
    st = oracle.kv_append(k, k, torch.tensor([5, nb * BLOCK_SIZE], dtype=torch.int64), kc, vc)
    assert st & oracle.SLOT_OUT_OF_RANGE
    assert torch.equal(kc[0, 0, 5], k[0, 0])
    st = oracle.kv_append(k, k, torch.tensor([9, 9], dtype=torch.int64), kc, vc)
    assert st & oracle.DUPLICATE_SLOT


# ---------------------------------------------------------------------------
# Block copy (copy-on-write of shared blocks)
# ---------------------------------------------------------------------------
def test_copy_blocks_equals_numpy_block_assignment_in_pair_order():
    """The copy half of copy-on-write ("v0版本介绍", section 为什么需要推理框架: requests share
    prompt blocks, so a shared block is copied before one of its users appends into it),
    restated as numpy block assignment cache[dst] = cache[src] for K and V, pair by pair in
    order, on a pool whose every element holds a distinct bit pattern.  The pairs include a
    chain (a -> b, then b -> c: c must end up with a's contents, which fixes the order of
    application) and an out-of-range pair (flagged, skipped, nothing written).  Catches a
    per-block stride without the kv heads, V left uncopied or copied from K, pairs applied
    out of order, and swapped source and destination."""
    nb, hkv, D = 10, 3, 8
    n_el = nb * hkv * BLOCK_SIZE * D
    # Distinct finite bf16 bit patterns (exponent field kept away from 0xff: no NaN or inf).
    bits = (np.arange(n_el, dtype=np.int64) % 0x3f00 + 0x0100).astype(np.int16)
    kc = torch.from_numpy(bits.reshape(nb, hkv, BLOCK_SIZE, D).copy()).view(torch.bfloat16)
    vc = torch.from_numpy((-bits).reshape(nb, hkv, BLOCK_SIZE, D).copy()).view(torch.bfloat16)
    assert len(np.unique(kc.view(torch.int16).numpy())) == n_el
    pairs = np.array([[1, 4], [4, 7], [2, 9], [0, nb], [8, 3]], dtype=np.int64)

    k_ref = kc.view(torch.int16).numpy().copy()
    v_ref = vc.view(torch.int16).numpy().copy()
    for src, dst in pairs.tolist():
        if 0 <= src < nb and 0 <= dst < nb:
            k_ref[dst] = k_ref[src]
            v_ref[dst] = v_ref[src]
    assert np.array_equal(k_ref[7], kc.view(torch.int16).numpy()[1])  # the chain carried block 1 to block 7

    st = oracle.copy_blocks(kc, vc, torch.from_numpy(pairs))
    assert st == oracle.BLOCK_ID_OUT_OF_RANGE
    assert np.array_equal(kc.view(torch.int16).numpy(), k_ref)
    assert np.array_equal(vc.view(torch.int16).numpy(), v_ref)


def test_copy_blocks_with_no_valid_pair_changes_nothing():
    nb, hkv, D = 3, 2, 8
    g = make_generator(24)
    kc = randn_bf16((nb, hkv, BLOCK_SIZE, D), g)
    vc = randn_bf16((nb, hkv, BLOCK_SIZE, D), g)
    k0, v0 = kc.clone(), vc.clone()
    st = oracle.copy_blocks(kc, vc, torch.tensor([[-1, 0], [1, 3]], dtype=torch.int64))
    assert st == oracle.BLOCK_ID_OUT_OF_RANGE
    assert torch.equal(kc.view(torch.int16), k0.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), v0.view(torch.int16))
    assert oracle.copy_blocks(kc, vc, torch.zeros((0, 2), dtype=torch.int64)) == oracle.OK


def test_append_then_attend_equals_contiguous_attention():
    """Write each sequence token by token through the allocator's slots, then attend:
    equals SDPA over the tokens as written.  Ties the append layout to the gather."""
    g = make_generator(23)
    hq, hkv, D, nb = 4, 2, 128, 24
    lens = [1, 16, 17, 50]
    alloc = BlockAllocator(nb, g)
    kc = torch.zeros(nb, hkv, BLOCK_SIZE, D, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    tok_k = [randn_bf16((L, hkv, D), g) for L in lens]
    tok_v = [randn_bf16((L, hkv, D), g) for L in lens]
    for sid, L in enumerate(lens):
        alloc.add_sequence(sid, 0)
        for p in range(L):
            s = alloc.append_token(sid)
            assert oracle.kv_append(tok_k[sid][p:p + 1], tok_v[sid][p:p + 1],
                                    torch.tensor([s], dtype=torch.int64), kc, vc) == oracle.OK
    bt = alloc.block_table(list(range(len(lens))), 4)
    q = randn_bf16((len(lens), hq, D), g)
    out = run_oracle(q, kc, vc, bt, torch.tensor(lens, dtype=torch.int32), 0.09)
    for b, L in enumerate(lens):
        K = f64(tok_k[b]).permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)
        V = f64(tok_v[b]).permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)
        ref = F.scaled_dot_product_attention(f64(q[b]).unsqueeze(1), K, V, scale=0.09).squeeze(1)
        np.testing.assert_allclose(out[b], ref.numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# RoPE and bf16 rounding (decode step)
# ---------------------------------------------------------------------------
def test_bf16_rounding_matches_torch_including_ties():
    """Round-to-nearest-even written from the definition equals torch's fp32 -> bf16 cast."""
    g = make_generator(51)
    x = torch.randn(200000, generator=g, dtype=torch.float32) * torch.exp(torch.randn(200000, generator=g) * 4)
    ties = (torch.arange(0, 4096, dtype=torch.int32) << 16 | 0x8000).view(torch.float32)  # exact halfway
    odd = ((torch.arange(0, 4096, dtype=torch.int32) << 16) | 0x18000).view(torch.float32)
    x = torch.cat([x, ties, odd, torch.tensor([0.0, -0.0, float("inf"), -float("inf"), 3.4e38, 1e-40])])
    got = oracle.float_to_bf16(x)
    want = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_rope_position_zero_is_identity():
    from workloads import rope_cos_sin
    g = make_generator(52)
    x = randn_bf16((5, 3, 128), g)
    y = x.clone()
    assert oracle.rope(y, np.zeros(5, np.int64), rope_cos_sin(8, 128)) == oracle.OK
    assert torch.equal(x, y)


@pytest.mark.parametrize("d,theta", [(128, 1e6), (64, 1e4)])
def test_rope_matches_float64_rotate_half(d, theta):
    """Against an independent float64 rotate_half on the same table, rounded once to bf16:
    equal, or one bf16 ulp apart where the fp32 steps round across a boundary (rare)."""
    from workloads import rope_cos_sin
    g = make_generator(53)
    n, heads = 64, 4
    table = rope_cos_sin(5000, d, theta)
    pos = torch.randint(0, 5000, (n,), generator=g)
    x = randn_bf16((n, heads, d), g)
    y = x.clone()
    assert oracle.rope(y, pos.numpy(), table) == oracle.OK
    xf = x.to(torch.float64)
    c = table[pos, : d // 2].to(torch.float64)[:, None, :]
    s = table[pos, d // 2:].to(torch.float64)[:, None, :]
    x1, x2 = xf[..., : d // 2], xf[..., d // 2:]
    ref = torch.cat([x1 * c - x2 * s, x2 * c + x1 * s], dim=-1).to(torch.float32).to(torch.bfloat16)
    a = y.view(torch.int16).to(torch.int32)
    b = ref.view(torch.int16).to(torch.int32)
    assert (a - b).abs().max().item() <= 1
    assert (a != b).float().mean().item() < 0.01


def test_decode_step_without_rope_is_append_then_attend():
    c = make_decode_case("qwen3_0.6b", seed=54, lengths=[1, 17, 40, 300])
    kc, vc = c.k_cache.clone(), c.v_cache.clone()
    out, st = oracle.decode_step(c.q, c.new_k, c.new_v, kc, vc, c.block_tables, c.context_lens, c.scale)
    assert st == oracle.OK
    kc2, vc2 = c.k_cache.clone(), c.v_cache.clone()
    assert oracle.kv_append(c.new_k, c.new_v, c.slot_mapping, kc2, vc2) == oracle.OK
    ref = run_oracle(c.q, kc2, vc2, c.block_tables, c.context_lens, c.scale)
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2)
    assert np.array_equal(out, ref)


# ---------------------------------------------------------------------------
# Chunked prefill
# ---------------------------------------------------------------------------
def _prefill_ref_sdpa(c):
    """torch float64 SDPA per sequence on un-paged K/V with the causal mask offset by the prefix."""
    T, hq, d = c.q.shape
    hkv = c.k_cache.shape[1]
    out = torch.zeros(T, hq, d, dtype=torch.float64)
    qs = c.query_start.tolist()
    for b, L in enumerate(c.context_lens.tolist()):
        C = qs[b + 1] - qs[b]
        P = L - C
        K, V = contiguous_kv(c.k_cache, c.v_cache, c.block_tables, c.context_lens, b)
        K = K.repeat_interleave(hq // hkv, dim=0)
        V = V.repeat_interleave(hq // hkv, dim=0)
        qb = f64(c.q[qs[b]:qs[b + 1]]).permute(1, 0, 2)               # [hq, C, d]
        mask = torch.arange(L)[None, :] <= (P + torch.arange(C))[:, None]
        o = F.scaled_dot_product_attention(qb, K, V, attn_mask=mask, scale=c.scale)
        out[qs[b]:qs[b + 1]] = o.permute(1, 0, 2)
    return out.numpy()


def _appended(c):
    kc, vc = c.k_cache.clone(), c.v_cache.clone()
    assert oracle.kv_append(c.new_k, c.new_v, c.slot_mapping, kc, vc) == oracle.OK
    return kc, vc


@pytest.mark.parametrize("seed", [0, 1])
def test_prefill_matches_causal_sdpa(seed):
    from workloads import make_prefill_case
    c = make_prefill_case("prefill_tiny", seed=seed)
    c.k_cache, c.v_cache = _appended(c)
    out, st = oracle.paged_prefill_attention(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens,
                                             c.query_start, c.scale)
    assert st == oracle.OK
    np.testing.assert_allclose(out, _prefill_ref_sdpa(c), rtol=0, atol=1e-12)


def test_prefill_with_chunks_of_one_is_decode():
    from workloads import PrefillSpec, make_prefill_case
    spec = PrefillSpec("ones", "", 8, 2, 128, (1, 1, 1), (0, 60), 5)
    c = make_prefill_case(spec, seed=2)
    out, st = oracle.paged_prefill_attention(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens,
                                             c.query_start, c.scale)
    dec, st2 = oracle.paged_decode_attention(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale)
    assert st == st2 == oracle.OK and np.array_equal(out, dec)


def test_prefill_last_chunk_row_is_decode_and_first_row_with_no_prefix_is_its_value():
    from workloads import make_prefill_case
    c = make_prefill_case("prefill_tiny", seed=3, prefixes=[0, 21])
    out, _ = oracle.paged_prefill_attention(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens,
                                            c.query_start, c.scale)
    qs = c.query_start.tolist()
    last = torch.tensor([qs[1] - 1, qs[2] - 1])
    dec, _ = oracle.paged_decode_attention(c.q[last].contiguous(), c.k_cache, c.v_cache, c.block_tables,
                                           c.context_lens, c.scale)
    assert np.array_equal(out[last.numpy()], dec)
    # Sequence 0 has no prefix: its first query row sees one token, so out = V_0.
    v0 = f64(c.v_cache[int(c.block_tables[0, 0]), :, 0]).numpy()       # [hkv, d]
    assert np.array_equal(out[0], np.repeat(v0, 2, axis=0))
