"""The split-K bookkeeping of paged decode attention, modelled on the CPU.

The batch's (sequence, kv head, block) items form one sequence-major stream of N items, cut into P
pieces, piece w holding items [floor(w N / P), floor((w + 1) N / P)).  Walking its piece, a warp
writes a pair's output itself when it saw the whole pair, and otherwise parks a partial state in
slot 0 (the first pair it finishes) or slot 1 (a later one).  The walk also records, for every pair,
the piece holding its first block with the slot its state takes there, and the piece holding its
last block; the merge reads those records.  The same pieces follow from the integer arithmetic alone:
wa = floor(((s + 1) P - 1) / N) holds the pair's first item s, wb = floor((e P - 1) / N) its last item
e - 1, and piece wa's state is in slot 1 exactly when the piece began before s.

This test restates that integer arithmetic in Python and checks the scheme on random length mixes
and partition counts, with empty pieces (P > N) and empty sequences:
- every pair is finished exactly once;
- a cut pair's states are exactly the non-empty pieces wa..wb, in the slots the merge reads, and the
  records the walk leaves find the same states;
- no piece parks more than two states.
The CUDA kernels' own use of it is checked on the GPU (every partition count against the oracle).
"""
import random

import pytest


def walk(lens_blocks: list[int], hkv: int, P: int, records: dict | None = None):
    """Simulate the partition kernel's walk: (states, outputs) keyed by pair (b, kvh).  `records`, if
    given, receives what the walk writes for the merge: pair -> [first piece * 2 + slot, last piece]."""
    items = [(b, k, j) for b, nb in enumerate(lens_blocks) for k in range(hkv) for j in range(nb)]
    N = len(items)
    states: dict[tuple[int, int], list[tuple[int, int]]] = {}
    outputs: dict[tuple[int, int], int] = {}
    parked = [0] * P
    for w in range(P):
        st, en = w * N // P, (w + 1) * N // P
        first_pair = True
        from_start = False
        for i in range(st, en):
            b, k, j = items[i]
            if i == st or j == 0:
                from_start = j == 0
                if from_start and records is not None:
                    records.setdefault((b, k), [None, None])[0] = 2 * w + (0 if first_pair else 1)
            nb = lens_blocks[b]
            last_of_pair = j == nb - 1
            if last_of_pair and records is not None:
                records.setdefault((b, k), [None, None])[1] = w
            if last_of_pair or i == en - 1:
                if from_start and last_of_pair:
                    assert (b, k) not in outputs
                    outputs[(b, k)] = w
                else:
                    states.setdefault((b, k), []).append((w, 0 if first_pair else 1))
                    parked[w] += 1
                first_pair = False
    return N, states, outputs, parked


def record_view(records: dict, lens_blocks: list[int], hkv: int, P: int, N: int, b: int, kvh: int):
    """What the merge kernel computes from the walk's records: None if one piece finished the pair,
    else its (piece, slot) states.  Piece bounds are used only to skip empty pieces (P > N)."""
    rec_a, wb = records[(b, kvh)]
    wa = rec_a // 2
    if wa == wb:
        return None
    got = []
    for w in range(wa, wb + 1):
        if P > N and w * N // P == (w + 1) * N // P:
            continue
        got.append((w, rec_a % 2 if w == wa else 0))
    return got


def merge_view(lens_blocks: list[int], hkv: int, P: int, N: int, b: int, kvh: int):
    """What the merge kernel computes for pair (b, kvh): None if one piece finished it, else its states."""
    prefix = [0]
    for nb in lens_blocks:
        prefix.append(prefix[-1] + nb)
    nblk = lens_blocks[b]
    s = hkv * prefix[b] + kvh * nblk
    e = s + nblk
    wa = ((s + 1) * P - 1) // N
    wb = (e * P - 1) // N
    if wa == wb:
        return None
    got = []
    for w in range(wa, wb + 1):
        st, en = w * N // P, (w + 1) * N // P
        if st == en:
            continue
        got.append((w, 1 if (w == wa and st < s) else 0))
    return got


@pytest.mark.parametrize("seed", range(40))
def test_every_pair_is_finished_once_and_the_merge_finds_its_states(seed):
    rng = random.Random(seed)
    B = rng.randint(1, 12)
    hkv = rng.choice([1, 2, 8])
    lens_blocks = [rng.choice([0, 1, 2, rng.randint(1, 40)]) for _ in range(B)]
    if sum(lens_blocks) == 0:
        lens_blocks[0] = 3
    n_items = hkv * sum(lens_blocks)
    for P in sorted({1, 2, 3, rng.randint(1, 50), n_items, n_items + 7, 3 * n_items}):
        records: dict = {}
        N, states, outputs, parked = walk(lens_blocks, hkv, P, records)
        assert N == n_items
        assert max(parked) <= 2
        for b, nb in enumerate(lens_blocks):
            for k in range(hkv):
                if nb == 0:
                    assert (b, k) not in outputs and (b, k) not in states  # zeros come from the merge kernel
                    continue
                view = merge_view(lens_blocks, hkv, P, N, b, k)
                assert record_view(records, lens_blocks, hkv, P, N, b, k) == view  # the records find the same states
                if view is None:
                    assert (b, k) in outputs and (b, k) not in states
                else:
                    assert (b, k) not in outputs
                    assert sorted(states[(b, k)]) == sorted(view)
                    assert len(view) >= 2


def test_a_long_sequence_spreads_over_many_pieces():
    lens_blocks = [8192] + [3] * 63           # one 131072-token sequence among short ones
    hkv, P = 8, 1216
    N, states, outputs, parked = walk(lens_blocks, hkv, P)
    pieces = [len(merge_view(lens_blocks, hkv, P, N, 0, k) or []) for k in range(hkv)]
    assert min(pieces) >= 100                 # each of its kv heads spans more than a hundred pieces
    assert max(parked) <= 2
