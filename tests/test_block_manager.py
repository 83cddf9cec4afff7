"""The C-ABI block manager (pkv_bm_*) against a plain reference model, on the CPU.

The model (oracle/block_manager.py) is pinned first: hand-worked scenarios,
structural invariants, and the property copy-on-write exists for -- writes
through one sequence's slots are never visible through another sequence,
while a fork sees everything its parent wrote before the fork.  Then the C++
manager must return exactly what the model returns, call by call, on seeded
random operation sequences.
"""
import random

import numpy as np
import pytest

from oracle.block_manager import BLOCK, ModelBlockManager, NoFreeBlocks


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_275_gb300 import build
    build.build(quiet=True)
    import paged_kv_cache_275_gb300 as pkv
    return pkv


# ---------------------------------------------------------------------------
# Pins of the model
# ---------------------------------------------------------------------------
def test_model_fork_then_copy_on_write_by_hand():
    m = ModelBlockManager(4)
    assert m.add_sequence(0, 20) == list(range(20))          # blocks 0, 1; 4 tokens in block 1
    m.fork(0, 1)
    assert m.refs == [2, 2, 0, 0]
    slots, copies = m.append_slots([1])
    assert copies == [(1, 2)] and slots == [2 * BLOCK + 4]   # seq 1 moves onto a copy of block 1
    assert m.refs == [2, 1, 1, 0]
    slots, copies = m.append_slots([0])
    assert copies == [] and slots == [1 * BLOCK + 4]         # block 1 is now seq 0's alone
    assert m.block_tables([0, 1], 3) == ([[0, 1, -1], [0, 2, -1]], [21, 21])


def test_model_full_shared_block_needs_no_copy():
    m = ModelBlockManager(6)
    m.add_sequence(0, 32)                                     # two full blocks
    m.fork(0, 1)
    slots, copies = m.append_slots([0, 1])
    assert copies == [] and slots == [2 * BLOCK, 3 * BLOCK]  # each takes a fresh block
    assert m.refs[:4] == [2, 2, 1, 1]


def test_model_free_list_is_fifo_in_table_order():
    m = ModelBlockManager(5, initial_free_order=[4, 3, 2, 1, 0])
    m.add_sequence(7, 40)                                     # blocks 4, 3, 2
    m.free_sequence(7)
    assert m.free == [1, 0, 4, 3, 2]
    assert m.add_sequence(8, 1) == [1 * BLOCK]


def test_model_failed_call_changes_nothing():
    m = ModelBlockManager(3)
    m.add_sequence(0, 16)
    m.add_sequence(1, 16)
    m.fork(0, 2)
    before = (list(m.free), list(m.refs), {k: list(v) for k, v in m.blocks.items()}, dict(m.length))
    with pytest.raises(NoFreeBlocks):
        m.append_slots([0, 1])                                # both full: needs 2 blocks, 1 free
    assert (list(m.free), list(m.refs), {k: list(v) for k, v in m.blocks.items()}, dict(m.length)) == before


def _random_ops(seed, model, n_ops=400):
    """Seeded manager calls (add / append / fork / free) drawn from the model's live sequences.

    Yields each op before the caller applies it to the model; a failed add is simply not live.
    """
    rng = random.Random(seed)
    next_id = 0
    for _ in range(n_ops):
        live = sorted(model.blocks)
        r = rng.random()
        if r < 0.2 or not live:
            yield ("add", next_id, rng.randint(0, 70))
            next_id += 1
        elif r < 0.35:
            yield ("fork", rng.choice(live), next_id)
            next_id += 1
        elif r < 0.5:
            yield ("free", rng.choice(live))
        else:
            yield ("append", rng.sample(live, rng.randint(1, len(live))))


def _apply(mgr, op):
    kind = op[0]
    if kind == "add":
        return list(mgr.add_sequence(op[1], op[2]))
    if kind == "fork":
        return mgr.fork(op[1], op[2])
    if kind == "free":
        return mgr.free_sequence(op[1])
    slots, copies = mgr.append_slots(op[1])
    return [int(x) for x in slots], [tuple(int(v) for v in c) for c in copies]


@pytest.mark.parametrize("seed", range(6))
def test_model_invariants_and_isolation(seed):
    """Every block is either free or referenced by exactly the sequences whose table holds it;
    a sequence never reads another's writes; a fork reads its parent's earlier writes."""
    m = ModelBlockManager(64)
    memory = {}                       # slot -> (sequence, position) written there
    expect = {}                       # sequence -> list of (writer, position) for its positions
    for op in _random_ops(seed, m):
        try:
            out = _apply(m, op)
        except NoFreeBlocks:
            continue
        kind = op[0]
        if kind == "add":
            expect[op[1]] = []
            for p, s in enumerate(out):
                memory[s] = (op[1], p)
                expect[op[1]].append((op[1], p))
        elif kind == "fork":
            expect[op[2]] = list(expect[op[1]])
        elif kind == "free":
            del expect[op[1]]
        else:
            slots, copies = out
            for src, dst in copies:   # the caller's block copy
                for o in range(BLOCK):
                    if src * BLOCK + o in memory:
                        memory[dst * BLOCK + o] = memory[src * BLOCK + o]
            for s, slot in zip(op[1], slots):
                memory[slot] = (s, len(expect[s]))
                expect[s].append((s, len(expect[s])))
        # structural invariants
        held = [0] * m.num_blocks
        for bl in m.blocks.values():
            for b in bl:
                held[b] += 1
        assert held == m.refs
        assert sorted(m.free) == [b for b in range(m.num_blocks) if m.refs[b] == 0]
        for s, bl in m.blocks.items():
            L = m.length[s]
            assert len(bl) == -(-L // BLOCK)
            # isolation: reading each position through the table gives what this sequence saw written
            got = [memory.get(bl[p // BLOCK] * BLOCK + p % BLOCK) for p in range(L)]
            assert got == expect[s], f"sequence {s} reads foreign data"


# ---------------------------------------------------------------------------
# The C++ manager against the model
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(6))
def test_capi_manager_matches_model(pkv, seed):
    order = list(range(64))
    random.Random(100 + seed).shuffle(order)
    m = ModelBlockManager(64, order)
    c = pkv.BlockManager(64, order)
    for op in _random_ops(seed, m):
        try:
            want = _apply(m, op)
            want_err = None
        except NoFreeBlocks:
            want_err = "no free"
        if want_err:
            with pytest.raises(pkv.PagedKVError) as e:
                _apply(c, op)
            assert e.value.status == 4
        else:
            assert _apply(c, op) == want, op
        assert c.num_free() == m.num_free()
        live = sorted(m.blocks)
        if live:
            width = max(1, max(len(m.blocks[s]) for s in live))
            tables, lens = c.block_tables(live, width)
            mt, ml = m.block_tables(live, width)
            assert tables.tolist() == mt and lens.tolist() == ml
        assert [c.ref_count(b) for b in range(64)] == m.refs
    c.close()


def test_capi_manager_rejects_bad_calls(pkv):
    c = pkv.BlockManager(8)
    c.add_sequence(1, 5)
    for bad in (lambda: c.add_sequence(1, 3), lambda: c.add_sequence(-1, 3), lambda: c.fork(9, 2),
                lambda: c.fork(1, 1), lambda: c.free_sequence(42), lambda: c.append_slots([1, 1]),
                lambda: c.append_slots([5]), lambda: c.block_tables([1], 0), lambda: c.ref_count(8)):
        with pytest.raises(pkv.PagedKVError) as e:
            bad()
        assert e.value.status == 1
    with pytest.raises(pkv.PagedKVError) as e:
        c.add_sequence(2, 16 * 8)
    assert e.value.status == 4 and c.num_free() == 7
    with pytest.raises(pkv.PagedKVError):
        pkv.BlockManager(4, [0, 1, 1, 3])
    c.close()


def test_isolation_pin_catches_missing_copy_on_write():
    """Plant the mistake in a copy of the model (append into a shared block in place): the
    isolation test must fail."""
    import oracle.block_manager as bmod
    src = open(bmod.__file__).read()
    anchor = "elif self.refs[self.blocks[s][-1]] > 1:\n                old"
    assert src.count(anchor) == 1
    ns = {}
    exec(compile(src.replace(anchor, "elif False:\n                old"), "planted", "exec"), ns)
    global ModelBlockManager
    saved = ModelBlockManager
    ModelBlockManager = ns["ModelBlockManager"]
    try:
        caught = 0
        for seed in range(3):
            try:
                test_model_invariants_and_isolation(seed)
            except AssertionError:
                caught += 1
        assert caught == 3
    finally:
        ModelBlockManager = saved
