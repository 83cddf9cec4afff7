"""Shared prompt blocks on the GPU: block copy, fork + copy-on-write + append + decode.

The block manager hands out slots and copy-on-write pairs; the GPU runs
copy_blocks, kv_append and decode attention; the oracle replays the same
copies and appends on its own CPU copy of the pool (built only from the
generated inputs) and computes attention from it.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_275_gb300 as pkv
from gpu_util import assert_close, device_errors
from workloads import make_generator, randn_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("hkv,d", [(8, 128), (1, 64), (2, 128)])
def test_copy_blocks_bit_exact(hkv, d):
    g = make_generator(41)
    nb = 300
    kc = randn_bf16((nb, hkv, 16, d), g)
    vc = randn_bf16((nb, hkv, 16, d), g)
    perm = torch.randperm(nb, generator=g)
    pairs = torch.stack([perm[:100], perm[100:200]], dim=1).to(torch.int64)   # distinct, disjoint
    kg, vg = kc.cuda(), vc.cuda()
    pkv.copy_blocks(kg, vg, pairs.cuda())
    assert oracle.copy_blocks(kc, vc, pairs) == oracle.OK
    assert torch.equal(kg.cpu().view(torch.int16), kc.view(torch.int16))
    assert torch.equal(vg.cpu().view(torch.int16), vc.view(torch.int16))
    assert device_errors() == 0


def test_copy_blocks_out_of_range_is_flagged():
    kc = torch.zeros(4, 2, 16, 128, dtype=torch.bfloat16, device="cuda")
    pairs = torch.tensor([[0, 1], [2, 9]], dtype=torch.int64, device="cuda")
    kc[0] = 1.0
    pkv.copy_blocks(kc, kc.clone(), pairs)
    assert device_errors() & pkv.DEVERR_COPY_OUT_OF_RANGE
    assert torch.equal(kc[1], kc[0])


@pytest.mark.parametrize("prompt", [37, 48])
def test_parallel_sampling_fork_copy_on_write_decode(prompt):
    """One prompt, forked into 4 samples that decode 24 tokens each: the shared partial
    block is copied on first write, every sample attends to the common prompt plus its own
    tokens, and the pool matches the oracle's bit for bit."""
    g = make_generator(43)
    hq, hkv, d, nb, width = 16, 8, 128, 64, 8
    scale = d ** -0.5
    order = torch.randperm(nb, generator=g).tolist()
    bm = pkv.BlockManager(nb, order)
    k_pool = randn_bf16((nb, hkv, 16, d), g)
    v_pool = randn_bf16((nb, hkv, 16, d), g)
    mk, mv = k_pool.clone(), v_pool.clone()          # the oracle's pool
    kg, vg = k_pool.cuda(), v_pool.cuda()
    # Prompt of sequence 0, written by one multi-token append.
    slots = torch.from_numpy(bm.add_sequence(0, prompt).copy())
    pk, pv = randn_bf16((prompt, hkv, d), g), randn_bf16((prompt, hkv, d), g)
    pkv.kv_append(pk.cuda(), pv.cuda(), slots.cuda(), kg, vg)
    assert oracle.kv_append(pk, pv, slots, mk, mv) == oracle.OK
    seqs = [0, 1, 2, 3]
    for child in seqs[1:]:
        bm.fork(0, child)
    total_copies = 0
    for step in range(24):
        new_slots, copies = bm.append_slots(seqs)
        total_copies += len(copies)
        if len(copies):
            cp = torch.from_numpy(copies.copy())
            pkv.copy_blocks(kg, vg, cp.cuda())
            assert oracle.copy_blocks(mk, mv, cp) == oracle.OK
        nk, nv = randn_bf16((4, hkv, d), g), randn_bf16((4, hkv, d), g)
        s = torch.from_numpy(new_slots.copy())
        pkv.kv_append(nk.cuda(), nv.cuda(), s.cuda(), kg, vg)
        assert oracle.kv_append(nk, nv, s, mk, mv) == oracle.OK
        tables, lens = bm.block_tables(seqs, width)
        bt, cl = torch.from_numpy(tables.copy()), torch.from_numpy(lens.copy())
        q = randn_bf16((4, hq, d), g)
        out = torch.empty(4, hq, d, dtype=torch.bfloat16, device="cuda")
        pkv.paged_decode_attention(q.cuda(), kg, vg, bt.cuda(), cl.cuda(), scale, out)
        ref, st = oracle.paged_decode_attention(q, mk, mv, bt, cl, scale)
        assert st == oracle.OK
        assert_close(out, ref, f"prompt {prompt} step {step}")
    # A partial shared block is copied once per sample that writes it while shared (3 of 4);
    # a full one never.
    assert total_copies == (3 if prompt % 16 else 0)
    assert torch.equal(kg.cpu().view(torch.int16), mk.view(torch.int16))
    assert torch.equal(vg.cpu().view(torch.int16), mv.view(torch.int16))
    # The prompt's full blocks are still shared by all four samples.
    tables, _ = bm.block_tables(seqs, width)
    for j in range(prompt // 16):
        assert len(set(tables[:, j].tolist())) == 1 and bm.ref_count(int(tables[0, j])) == 4
    assert device_errors() == 0
    bm.close()
