"""Continuous-batching trace on the GPU (Qwen3-0.6B shape, 28 layers, 256 sequences, 100 decode steps).

Each step: sequences finish and join by seeded Poisson draws, freed blocks go
back to a fragmenting free list, a joining sequence's prompt K/V is written
with one multi-token kv_append per layer, then every layer appends one token
per running sequence and attends.

The oracle keeps its own CPU copy of two layers' pools: it starts from the
pools as generated (copied before any kernel runs) and replays every append
from the generated inputs, so none of its inputs comes from the GPU path.
At sampled steps the GPU pools must equal the oracle's bit for bit and the
attention outputs must meet the tolerance.
"""
import pytest
import torch

import oracle
import paged_kv_cache_275_gb300 as pkv
from gpu_util import assert_close, device_errors
from workloads import TRACE, TraceGenerator, make_generator, randn_bf16

pytestmark = pytest.mark.gpu

MIRRORED_LAYERS = (0, TRACE.num_layers - 1)
CHECK_STEPS = (0, 50, TRACE.steps - 1)


def test_continuous_batching_trace():
    spec = TRACE
    tg = TraceGenerator(spec, seed=0)
    H, Hkv, D, L = spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.num_layers
    scale = D ** -0.5
    gen = make_generator(1, "cuda")
    k_pools, v_pools, mirror = [], [], {}
    for layer in range(L):
        kp = randn_bf16((tg.num_blocks, Hkv, 16, D), gen, "cuda")
        vp = randn_bf16((tg.num_blocks, Hkv, 16, D), gen, "cuda")
        k_pools.append(kp)
        v_pools.append(vp)
        if layer in MIRRORED_LAYERS:
            mirror[layer] = (kp.cpu(), vp.cpu())
    torch.cuda.synchronize()
    assert device_errors() == 0

    checks = 0
    seen_join = seen_finish = False
    for st in tg.steps():
        B = len(st.seq_ids)
        seen_join |= bool(st.joined)
        seen_finish |= bool(st.finished)
        bt = st.block_tables.cuda()
        cl = st.context_lens.cuda()
        slots = st.slot_mapping.cuda()
        join_slots = torch.cat([st.join_slots[s] for s in st.joined]) if st.joined else None
        check = st.step in CHECK_STEPS
        for layer in range(L):
            q = randn_bf16((B, H, D), gen, "cuda")
            nk = randn_bf16((B, Hkv, D), gen, "cuda")
            nv = randn_bf16((B, Hkv, D), gen, "cuda")
            if join_slots is not None:
                pk = randn_bf16((join_slots.numel(), Hkv, D), gen, "cuda")
                pv = randn_bf16((join_slots.numel(), Hkv, D), gen, "cuda")
                pkv.kv_append(pk, pv, join_slots.cuda(), k_pools[layer], v_pools[layer])
            pkv.kv_append(nk, nv, slots, k_pools[layer], v_pools[layer])
            out = torch.empty_like(q)
            pkv.paged_decode_attention(q, k_pools[layer], v_pools[layer], bt, cl, scale, out)
            if layer in mirror:
                mk, mv = mirror[layer]
                if join_slots is not None:
                    assert oracle.kv_append(pk.cpu(), pv.cpu(), join_slots, mk, mv) == oracle.OK
                assert oracle.kv_append(nk.cpu(), nv.cpu(), st.slot_mapping, mk, mv) == oracle.OK
                if check:
                    assert torch.equal(k_pools[layer].cpu().view(torch.int16), mk.view(torch.int16))
                    assert torch.equal(v_pools[layer].cpu().view(torch.int16), mv.view(torch.int16))
                    ref, status = oracle.paged_decode_attention(q.cpu(), mk, mv, st.block_tables, st.context_lens,
                                                                scale)
                    assert status == oracle.OK
                    assert_close(out, ref, f"step {st.step} layer {layer}")
                    checks += 1
            elif check:
                assert torch.isfinite(out.float()).all()
        assert device_errors() == 0, f"device error at step {st.step}"
    assert checks == len(CHECK_STEPS) * len(MIRRORED_LAYERS)
    assert seen_join and seen_finish
