"""Cross-machine regression of the oracle against the committed fixture."""
import importlib.util
import json
from pathlib import Path

import numpy as np

import oracle

GOLDEN = Path(__file__).parent / "golden"


def _maker():
    spec = importlib.util.spec_from_file_location("make_oracle_golden", GOLDEN / "make_oracle_golden.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_oracle_reproduces_committed_fixture(oracle_lib):
    doc = json.loads((GOLDEN / "oracle_regression.json").read_text())
    m = _maker()
    s = doc["shape"]
    B, hq, hkv, D, bs, nb = (s[k] for k in ("num_seqs", "num_q_heads", "num_kv_heads", "head_dim", "block_size",
                                            "num_blocks"))
    q = np.array(m.lcg_bf16(B * hq * D, doc["q_bits_lcg_seed"]), np.uint16).reshape(B, hq, D)
    kc = np.array(m.lcg_bf16(nb * hkv * bs * D, doc["k_cache_bits_lcg_seed"]), np.uint16).reshape(nb, hkv, bs, D)
    vc = np.array(m.lcg_bf16(nb * hkv * bs * D, doc["v_cache_bits_lcg_seed"]), np.uint16).reshape(nb, hkv, bs, D)
    out, st = oracle.paged_decode_attention(q, kc, vc, np.array(doc["block_tables"], np.int32),
                                            np.array(doc["context_lens"], np.int32), doc["scale"])
    assert st == oracle.OK
    expect = np.array([[[float.fromhex(x) for x in row] for row in head] for head in doc["out"]])
    np.testing.assert_allclose(out, expect, rtol=0, atol=1e-13)
