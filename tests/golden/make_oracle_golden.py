"""Write ``oracle_regression.json``: a small decode problem and the oracle's fp64 answer.

This script calls only ``oracle/``.  The file pins the oracle against itself
across CPU architectures (an x86 and an Arm build must give the same fp64
values to 1e-13); it is not a correctness pin -- the pages print no
worked numerical example, so correctness is pinned by closed forms,
invariants and brute force in ``tests/test_oracle_pins.py``.

Inputs are explicit bf16 bit patterns from a fixed linear congruential
sequence, so the fixture does not depend on any library's random generator.

Run:  python tests/golden/make_oracle_golden.py
"""
import json
import sys
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parents[2]
sys.path.insert(0, str(ROOT))
import oracle  # noqa: E402

OUT = Path(__file__).with_name("oracle_regression.json")


def lcg_bf16(n: int, state: int) -> list[int]:
    """n bf16 bit patterns of moderate magnitude (|x| < 4), from a 32-bit LCG."""
    out = []
    for _ in range(n):
        state = (1664525 * state + 1013904223) % (1 << 32)
        sign = (state >> 31) & 1
        exponent = 125 + ((state >> 24) % 4)        # 2^-2 .. 2^1
        mantissa = (state >> 8) & 0x7F
        out.append((sign << 15) | (exponent << 7) | mantissa)
    return out


def main():
    B, hq, hkv, D, bs, nb, W = 3, 4, 2, 64, 16, 6, 3
    lens = [1, 17, 40]
    tables = [[4, -1, -1], [0, 5, -1], [3, 1, 2]]
    scale = 0.125
    q = np.array(lcg_bf16(B * hq * D, 1), dtype=np.uint16).reshape(B, hq, D)
    kc = np.array(lcg_bf16(nb * hkv * bs * D, 2), dtype=np.uint16).reshape(nb, hkv, bs, D)
    vc = np.array(lcg_bf16(nb * hkv * bs * D, 3), dtype=np.uint16).reshape(nb, hkv, bs, D)
    out, st = oracle.paged_decode_attention(q, kc, vc, np.array(tables, np.int32), np.array(lens, np.int32),
                                            scale, num_threads=1)
    assert st == oracle.OK
    doc = {
        "what": "oracle regression fixture (cross-machine); not a correctness pin",
        "shape": {"num_seqs": B, "num_q_heads": hq, "num_kv_heads": hkv, "head_dim": D, "block_size": bs,
                  "num_blocks": nb, "max_blocks_per_seq": W},
        "context_lens": lens, "block_tables": tables, "scale": scale,
        "q_bits_lcg_seed": 1, "k_cache_bits_lcg_seed": 2, "v_cache_bits_lcg_seed": 3,
        "out": [[[float(x).hex() for x in row] for row in head] for head in out],
    }
    OUT.write_text(json.dumps(doc, indent=0) + "\n")
    print("wrote", OUT)


if __name__ == "__main__":
    main()
