"""Split-K consistency before rounding: the fp32 partial states the partition phase parks.

The decode pass cuts the batch's block stream into pieces; a piece that covers part of a
(sequence, kv head) pair parks that pair's partial softmax state (acc[G][D], m[G] in base-2
units, l[G]) in the workspace, and the merge combines a pair's states.  This test runs the
partition phase alone with partition counts that cut every pair, reads the parked fp32 states
back, combines each pair's states on the host in fp64 (M = max m_p; out = sum 2^(m_p - M) acc_p /
sum 2^(m_p - M) l_p), and checks, before any rounding to bf16:
  - two different ways of cutting the stream give the same result to 1e-5 relative;
  - each equals the fp64 oracle (unrounded) to 1e-5 relative.
Relative means normwise over all cut rows: ||x - y||_2 / ||y||_2.  The states' slots are found
with the integer arithmetic restated in test_split_k_bookkeeping.py, and the pair records the merge
kernel reads are checked against that model's walk.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_275_gb300 as pkv
from gpu_util import device_errors, oracle_step
from test_gpu_decode import QWEN3_G8
from test_split_k_bookkeeping import merge_view, walk
from workloads import make_decode_case

pytestmark = pytest.mark.gpu

REL = 1e-5


def parked_combination(ws: torch.Tensor, lens_blocks, hkv: int, G: int, D: int, P: int):
    """{(b, kvh): fp64 [G, D]} for every pair the partition phase left as partial states."""
    B = len(lens_blocks)
    raw = ws.cpu()
    prefix = raw[:4 * (B + 1)].view(torch.int32).numpy()
    assert list(prefix) == list(np.concatenate([[0], np.cumsum(lens_blocks)]))
    # Workspace: block prefix int32 [B + 1], then the pair records int32 [B * Hkv][2], each 256-byte aligned.
    rec_at = ((B + 1) * 4 + 255) & ~255
    header = rec_at + ((B * hkv * 8 + 255) & ~255)
    recs = raw[rec_at:rec_at + B * hkv * 8].view(torch.int32).numpy().reshape(B, hkv, 2)
    model: dict = {}
    walk(list(lens_blocks), hkv, P, model)
    for (b, k), (rec_a, rec_b) in model.items():   # the records the merge reads are the modelled walk's
        assert (int(recs[b, k, 0]), int(recs[b, k, 1])) == (rec_a, rec_b), (b, k)
    pf = G * D + ((2 * G + 3) // 4) * 4
    pieces = raw[header:header + P * 2 * pf * 4].view(torch.float32).numpy().astype(np.float64).reshape(P, 2, pf)
    N = hkv * int(prefix[-1])
    out = {}
    for b, nb in enumerate(lens_blocks):
        for k in range(hkv):
            if nb == 0:
                continue
            view = merge_view(list(lens_blocks), hkv, P, N, b, k)
            if view is None:
                continue
            st = np.stack([pieces[w, slot] for w, slot in view])   # [n, pf]
            acc = st[:, :G * D].reshape(-1, G, D)
            m = st[:, G * D:G * D + G]
            l = st[:, G * D + G:G * D + 2 * G]
            assert np.isfinite(m).all() and (l > 0).all()
            M = m.max(axis=0)
            w = np.exp2(m - M)
            out[(b, k)] = (w[:, :, None] * acc).sum(axis=0) / (w * l).sum(axis=0)[:, None]
    return out


def rel_err(x: np.ndarray, y: np.ndarray) -> float:
    return float(np.linalg.norm(x - y) / np.linalg.norm(y))


@pytest.mark.parametrize("shape", ["qwen3_0.6b", "llama3_8b", QWEN3_G8],
                         ids=["G2_cuda_cores", "G4_cuda_cores", "G8_tensor_cores"])
def test_parked_states_agree_across_cuts_and_with_the_oracle(shape):
    c = make_decode_case(shape, seed=31, num_seqs=24)
    ref, _, _ = oracle_step(c)                       # fp64, unrounded
    s = c.spec
    B, hq, hkv, D = s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_dim
    G = hq // hkv
    lens_blocks = [(int(L) + 15) // 16 for L in c.context_lens]
    assert min(lens_blocks) >= 2                      # every pair can be cut
    N = hkv * sum(lens_blocks)
    g = c.to("cuda")
    pkv.kv_append(g.new_k, g.new_v, g.slot_mapping, g.k_cache, g.v_cache)
    combos = {}
    for P in (N, (N + 4) // 5):                       # one block per piece; about five per piece
        ws = torch.empty(pkv.workspace_size(B, hq, hkv, D, s.max_blocks_per_seq, P), dtype=torch.uint8,
                         device="cuda")
        out = torch.empty_like(g.q)
        pkv.paged_decode_attention(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale, out,
                                   num_partitions=P, phases=pkv.PHASE_PARTITION, workspace=ws)
        torch.cuda.synchronize()
        combos[P] = parked_combination(ws, lens_blocks, hkv, G, D, P)
    assert device_errors() == 0
    a, b = combos[N], combos[(N + 4) // 5]
    assert len(a) == B * hkv                          # one block per piece cuts every pair
    both = sorted(set(a) & set(b))
    assert len(both) >= B * hkv // 2
    xa = np.stack([a[p] for p in both])
    xb = np.stack([b[p] for p in both])
    refs = {p: ref[p[0], p[1] * G:(p[1] + 1) * G] for p in a}
    e_cut = rel_err(xa, xb)
    e_a = rel_err(np.stack([a[p] for p in sorted(a)]), np.stack([refs[p] for p in sorted(a)]))
    e_b = rel_err(xb, np.stack([refs[p] for p in both]))
    print(f"{s.name}: cut vs cut {e_cut:.3g}, one block per piece vs oracle {e_a:.3g}, "
          f"five per piece vs oracle {e_b:.3g} ({len(both)} pairs in both)")
    assert e_cut <= REL and e_a <= REL and e_b <= REL
