"""kv_append on the GPU against the oracle: bit-exact on the whole cache."""
import pytest
import torch

import oracle
import paged_kv_cache_275_gb300 as pkv
from gpu_util import device_errors
from workloads import make_decode_case, make_generator, randn_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "qwen3_0.6b", "llama3_8b"])
def test_decode_append_bit_exact(name):
    c = make_decode_case(name, seed=0)
    g = c.to("cuda")
    pkv.kv_append(g.new_k, g.new_v, g.slot_mapping, g.k_cache, g.v_cache)
    torch.cuda.synchronize()
    kc, vc = c.k_cache.clone(), c.v_cache.clone()
    assert oracle.kv_append(c.new_k, c.new_v, c.slot_mapping, kc, vc) == oracle.OK
    assert torch.equal(g.k_cache.cpu().view(torch.int16), kc.view(torch.int16))
    assert torch.equal(g.v_cache.cpu().view(torch.int16), vc.view(torch.int16))
    assert device_errors() == 0


@pytest.mark.parametrize("head_dim,hkv", [(64, 1), (64, 4), (128, 8), (128, 2)])
def test_prompt_append_with_padding_and_sentinels(head_dim, hkv):
    """A multi-token append (a prompt) with padding slots (-1) into a sentinel-filled pool:
    written slots carry the input bits, every other slot keeps the sentinel."""
    gen = make_generator(31)
    nb, n = 97, 700
    kc = torch.full((nb, hkv, 16, head_dim), -3.5, dtype=torch.bfloat16)
    vc = torch.full_like(kc, 2.25)
    slots = torch.randperm(nb * 16, generator=gen)[:n].to(torch.int64)
    slots[::7] = -1
    k = randn_bf16((n, hkv, head_dim), gen)
    v = randn_bf16((n, hkv, head_dim), gen)
    kg, vg = kc.cuda(), vc.cuda()
    pkv.kv_append(k.cuda(), v.cuda(), slots.cuda(), kg, vg)
    assert oracle.kv_append(k, v, slots, kc, vc) == oracle.OK
    assert torch.equal(kg.cpu().view(torch.int16), kc.view(torch.int16))
    assert torch.equal(vg.cpu().view(torch.int16), vc.view(torch.int16))
    assert device_errors() == 0


def test_out_of_range_slot_is_flagged_and_skipped():
    gen = make_generator(32)
    nb, hkv, d = 4, 2, 128
    kc = torch.zeros(nb, hkv, 16, d, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    k = randn_bf16((3, hkv, d), gen).cuda()
    slots = torch.tensor([5, nb * 16, 63], dtype=torch.int64, device="cuda")
    assert device_errors() == 0
    pkv.kv_append(k, k, slots, kc, vc)
    assert device_errors() & pkv.DEVERR_SLOT_OUT_OF_RANGE
    assert torch.equal(kc[0, :, 5], k[0]) and torch.equal(kc[3, :, 15], k[2])
    # The context stays usable and the word was cleared.
    pkv.kv_append(k[:1], k[:1], slots[:1], kc, vc)
    assert device_errors() == 0


def test_zero_tokens_is_a_noop():
    kc = torch.zeros(2, 1, 16, 64, dtype=torch.bfloat16, device="cuda")
    e = torch.empty(0, 1, 64, dtype=torch.bfloat16, device="cuda")
    before = pkv.kernel_launch_count()
    pkv.kv_append(e, e, torch.empty(0, dtype=torch.int64, device="cuda"), kc, kc.clone())
    assert pkv.kernel_launch_count() == before
