"""Seeded synthetic workloads for the paged KV-cache hot path.

This module is shared by the tests, the smoke check and the benchmark.  It
holds none of the method's arithmetic: no append, no gather through a block
table, no attention.  It only draws random tensors and emulates the block
allocator that the pages describe (a pool of fixed 16-token blocks, a free
list, a block table per sequence, a new block taken only when the current
one is full, all blocks returned when a sequence finishes):

  "跟着 Claude Code，我用 Python 实现了一个轻量级的 vLLM", section
  "核心机制一：分页 KV Cache"; "从零实现一个 mini vLLM--开篇", section 5
  (phase 4, block tables) and section 7 (blocks released at the end of a
  request); "v0版本介绍", section "为什么需要推理框架" (a block is taken only
  when the current one fills).

The allocator's only index bookkeeping is the slot number it hands out for a
token position: ``blocks[pos // 16] * 16 + pos % 16`` (a block id and the
offset inside it, packed into one integer, as the cache library documents).

All values are bf16 drawn from N(0, 1) (fp32 draws rounded to bf16), block
ids come from a seeded random permutation of the pool, and the same seed
always gives the same tensors.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BLOCK_SIZE = 16


# ----------------------------------------------------------------------------
# Workload shapes (head layouts of the models the pages name; synthetic data).
# ----------------------------------------------------------------------------
@dataclass(frozen=True)
class DecodeSpec:
    name: str
    description: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    max_blocks_per_seq: int
    length_kind: str            # "fixed" | "uniform" | "loguniform"
    lengths: tuple = ()         # "fixed": the lengths
    length_range: tuple = ()    # "uniform": inclusive (lo, hi); "loguniform": (lo, hi)
    first_len: int | None = None  # "loguniform": the first sequence's fixed length
    pool_blocks: int | None = None  # fixed pool size; else needed * (1 + slack)
    pool_slack: float = 0.0


SPECS = {
    "tiny": DecodeSpec(
        name="tiny", description="4 seqs, lens {5,16,17,40}, 2 q / 1 kv heads, D 64, 16-block pool",
        num_seqs=4, num_q_heads=2, num_kv_heads=1, head_dim=64, max_blocks_per_seq=3,
        length_kind="fixed", lengths=(5, 16, 17, 40), pool_blocks=16),
    "qwen3_0.6b": DecodeSpec(
        name="qwen3_0.6b", description="Qwen3-0.6B layer: 16 q / 8 kv heads, D 128, B 32, L~U{128..2048}",
        num_seqs=32, num_q_heads=16, num_kv_heads=8, head_dim=128, max_blocks_per_seq=128,
        length_kind="uniform", length_range=(128, 2048), pool_slack=0.10),
    "llama3_8b": DecodeSpec(
        name="llama3_8b", description="LLaMA-3-8B layer: 32 q / 8 kv heads, D 128, B 128, L~U{512..4096}",
        num_seqs=128, num_q_heads=32, num_kv_heads=8, head_dim=128, max_blocks_per_seq=256,
        length_kind="uniform", length_range=(512, 4096)),
    "llama3_70b": DecodeSpec(
        name="llama3_70b", description="LLaMA-3-70B layer: 64 q / 8 kv heads, D 128, B 128, L~U{512..4096}",
        num_seqs=128, num_q_heads=64, num_kv_heads=8, head_dim=128, max_blocks_per_seq=256,
        length_kind="uniform", length_range=(512, 4096)),
    "long_skew": DecodeSpec(
        name="long_skew",
        description="long-context skew: 32 q / 8 kv heads, D 128, B 64, L log-uniform 16..65536, one seq 131072",
        num_seqs=64, num_q_heads=32, num_kv_heads=8, head_dim=128, max_blocks_per_seq=8192,
        length_kind="loguniform", length_range=(16, 65536), first_len=131072),
}


@dataclass(frozen=True)
class TraceSpec:
    name: str = "qwen3_0.6b_trace"
    num_layers: int = 28
    max_seqs: int = 256
    steps: int = 100
    num_q_heads: int = 16
    num_kv_heads: int = 8
    head_dim: int = 128
    init_len_range: tuple = (128, 2048)
    join_rate: float = 4.0
    finish_rate: float = 4.0
    pool_slack: float = 0.25


TRACE = TraceSpec()


def draw_lengths(spec: DecodeSpec, g: torch.Generator) -> list[int]:
    if spec.length_kind == "fixed":
        return [int(x) for x in spec.lengths]
    if spec.length_kind == "uniform":
        lo, hi = spec.length_range
        return [int(x) for x in torch.randint(lo, hi + 1, (spec.num_seqs,), generator=g)]
    if spec.length_kind == "loguniform":
        lo, hi = spec.length_range
        u = torch.rand(spec.num_seqs, generator=g, dtype=torch.float64)
        lens = [int(round(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo))))) for x in u]
        if spec.first_len is not None:
            lens[0] = spec.first_len
        return lens
    raise ValueError(spec.length_kind)


# ----------------------------------------------------------------------------
# Block allocator (free list + per-sequence block lists).
# ----------------------------------------------------------------------------
class BlockAllocator:
    """A pool of ``num_blocks`` 16-token blocks with a free list.

    The free list starts as a seeded random permutation of the pool; blocks
    are popped from its front and returned (shuffled) to its back, so a long
    run fragments it.
    """

    def __init__(self, num_blocks: int, g: torch.Generator):
        self.num_blocks = int(num_blocks)
        self.g = g
        self.free = [int(x) for x in torch.randperm(self.num_blocks, generator=g)]
        self._head = 0
        self.blocks: dict[int, list[int]] = {}
        self.length: dict[int, int] = {}

    def num_free(self) -> int:
        return len(self.free) - self._head

    def _pop(self) -> int:
        if self._head >= len(self.free):
            raise MemoryError("KV block pool exhausted")
        b = self.free[self._head]
        self._head += 1
        if self._head > 4096 and self._head * 2 > len(self.free):
            self.free = self.free[self._head:]
            self._head = 0
        return b

    def add_sequence(self, seq_id: int, length: int) -> list[int]:
        """Register a sequence holding ``length`` tokens; returns their slots."""
        if seq_id in self.blocks:
            raise KeyError(seq_id)
        self.blocks[seq_id] = [self._pop() for _ in range(-(-length // BLOCK_SIZE))]
        self.length[seq_id] = length
        return [self.slot(seq_id, p) for p in range(length)]

    def append_token(self, seq_id: int) -> int:
        """Grow a sequence by one token (taking a block only when the last is full); returns its slot."""
        pos = self.length[seq_id]
        if pos % BLOCK_SIZE == 0:
            self.blocks[seq_id].append(self._pop())
        self.length[seq_id] = pos + 1
        return self.slot(seq_id, pos)

    def slot(self, seq_id: int, pos: int) -> int:
        return self.blocks[seq_id][pos // BLOCK_SIZE] * BLOCK_SIZE + pos % BLOCK_SIZE

    def free_sequence(self, seq_id: int) -> None:
        blocks = self.blocks.pop(seq_id)
        self.length.pop(seq_id)
        order = torch.randperm(len(blocks), generator=self.g)
        self.free.extend(blocks[int(i)] for i in order)

    def block_table(self, seq_ids: list[int], width: int, pad: int = -1) -> torch.Tensor:
        t = torch.full((len(seq_ids), width), pad, dtype=torch.int32)
        for r, s in enumerate(seq_ids):
            bl = self.blocks[s]
            if len(bl) > width:
                raise ValueError("block table too narrow")
            if bl:
                t[r, :len(bl)] = torch.tensor(bl, dtype=torch.int32)
        return t


def randn_bf16(shape, g: torch.Generator, device="cpu", chunk: int = 1 << 26) -> torch.Tensor:
    """bf16 tensor of N(0,1) draws (fp32 draws rounded to nearest bf16), generated in chunks."""
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        out[lo:hi] = torch.randn(hi - lo, generator=g, dtype=torch.float32, device=device).to(torch.bfloat16)
    return out.view(*shape)


def make_generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


# ----------------------------------------------------------------------------
# One decode step of a batch.
# ----------------------------------------------------------------------------
@dataclass
class DecodeCase:
    spec: DecodeSpec
    q: torch.Tensor              # [B, Hq, D] bf16
    k_cache: torch.Tensor        # [NB, Hkv, 16, D] bf16
    v_cache: torch.Tensor
    block_tables: torch.Tensor   # [B, W] int32, -1 past each sequence's blocks
    context_lens: torch.Tensor   # [B] int32 (includes this step's token)
    new_k: torch.Tensor          # [B, Hkv, D] bf16: this step's token, at position L-1
    new_v: torch.Tensor
    slot_mapping: torch.Tensor   # [B] int64: slot of position L-1
    scale: float
    allocator: BlockAllocator = field(repr=False)

    @property
    def num_blocks(self) -> int:
        return self.k_cache.shape[0]

    def to(self, device) -> "DecodeCase":
        return DecodeCase(self.spec, *(t.to(device) for t in (
            self.q, self.k_cache, self.v_cache, self.block_tables, self.context_lens, self.new_k, self.new_v,
            self.slot_mapping)), self.scale, self.allocator)


def make_decode_case(name: str | DecodeSpec, seed: int = 0, device="cpu", lengths=None,
                     num_seqs: int | None = None) -> DecodeCase:
    """Build one decode step of the named workload.

    ``lengths`` / ``num_seqs`` override the spec (used for bounded samples of
    a workload and for edge cases).  The generator runs on ``device``.
    """
    spec = SPECS[name] if isinstance(name, str) else name
    if num_seqs is not None:
        spec = DecodeSpec(**{**spec.__dict__, "num_seqs": int(num_seqs)})
    g_cpu = make_generator(seed)
    lens = [int(x) for x in lengths] if lengths is not None else draw_lengths(spec, g_cpu)
    if lengths is not None:
        spec = DecodeSpec(**{**spec.__dict__, "num_seqs": len(lens)})
    if any(L < 0 or L > spec.max_blocks_per_seq * BLOCK_SIZE for L in lens):
        raise ValueError("context length outside the block table")
    needed = sum(-(-L // BLOCK_SIZE) for L in lens)
    num_blocks = spec.pool_blocks if spec.pool_blocks is not None else max(1, int(math.ceil(needed * (1 + spec.pool_slack))))
    if num_blocks < needed:
        raise ValueError("pool too small")
    alloc = BlockAllocator(num_blocks, g_cpu)
    slots = []
    for b, L in enumerate(lens):
        s = alloc.add_sequence(b, L)
        slots.append(s[-1] if L > 0 else -1)
    block_tables = alloc.block_table(list(range(len(lens))), spec.max_blocks_per_seq)

    g = make_generator(seed + 1, device) if str(device) != "cpu" else g_cpu
    B, Hq, Hkv, D = len(lens), spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    q = randn_bf16((B, Hq, D), g, device)
    k_cache = randn_bf16((num_blocks, Hkv, BLOCK_SIZE, D), g, device)
    v_cache = randn_bf16((num_blocks, Hkv, BLOCK_SIZE, D), g, device)
    new_k = randn_bf16((B, Hkv, D), g, device)
    new_v = randn_bf16((B, Hkv, D), g, device)
    return DecodeCase(spec, q, k_cache, v_cache, block_tables.to(device),
                      torch.tensor(lens, dtype=torch.int32, device=device), new_k, new_v,
                      torch.tensor(slots, dtype=torch.int64, device=device), 1.0 / math.sqrt(D), alloc)


def algorithmic_bytes(context_lens, num_q_heads: int, num_kv_heads: int, head_dim: int) -> int:
    """Bytes a decode-attention call must move at minimum (bf16 K/V/q/out, int32 tables and lengths).

    K and V of every cached token of every kv head, one block-table entry per
    used block, each sequence's length, q and the output.
    """
    lens = [int(x) for x in (context_lens.tolist() if hasattr(context_lens, "tolist") else context_lens)]
    kv = sum(2 * L * num_kv_heads * head_dim * 2 for L in lens)
    tables = sum(4 * (-(-L // BLOCK_SIZE)) for L in lens)
    per_seq = len(lens) * (4 + 2 * num_q_heads * head_dim * 2)
    return kv + tables + per_seq


def append_bytes(num_tokens: int, num_kv_heads: int, head_dim: int) -> int:
    """Bytes of one append: read k and v, write them into the cache, read the int64 slots."""
    return num_tokens * (4 * num_kv_heads * head_dim * 2 + 8)


# ----------------------------------------------------------------------------
# Continuous-batching trace (Qwen3-0.6B shape, 28 layers).
# ----------------------------------------------------------------------------
@dataclass
class TraceStep:
    step: int
    finished: list[int]          # seq ids released before this step
    joined: list[int]            # seq ids admitted before this step (prompt written this step)
    join_slots: dict             # seq id -> int64 tensor of its prompt slots
    seq_ids: list[int]           # running batch after admission, in batch order
    slot_mapping: torch.Tensor   # [B] int64: slot of each sequence's new token
    block_tables: torch.Tensor   # [B, W] int32
    context_lens: torch.Tensor   # [B] int32 (after this step's token)


class TraceGenerator:
    """Seeded continuous-batching schedule: sequences join and finish by Poisson draws,
    blocks are freed to and re-taken from a fragmenting free list.

    Only the schedule (ids, slots, block tables, lengths) is produced here; the
    K/V/q values are drawn by the caller from ``value_generator``.
    """

    def __init__(self, spec: TraceSpec = TRACE, seed: int = 0):
        self.spec = spec
        self.g = make_generator(seed)
        lo, hi = spec.init_len_range
        init = [int(x) for x in torch.randint(lo, hi + 1, (spec.max_seqs,), generator=self.g)]
        # Room for the initial batch plus the joins of every step (growth + slack).
        expected = sum(-(-L // BLOCK_SIZE) for L in init)
        growth = spec.max_seqs * (-(-spec.steps // BLOCK_SIZE) + 1)
        self.num_blocks = int((expected + growth) * (1 + spec.pool_slack))
        self.max_len = hi + spec.steps + 1
        self.width = -(-self.max_len // BLOCK_SIZE)
        self.alloc = BlockAllocator(self.num_blocks, self.g)
        self.running: list[int] = []
        self.next_id = 0
        self.initial_slots: dict[int, list[int]] = {}
        for L in init:
            sid = self._new_id()
            self.initial_slots[sid] = self.alloc.add_sequence(sid, L)
            self.running.append(sid)

    def _new_id(self) -> int:
        sid = self.next_id
        self.next_id += 1
        return sid

    def steps(self):
        spec = self.spec
        lo, hi = spec.init_len_range
        for step in range(spec.steps):
            finished, joined, join_slots = [], [], {}
            if step > 0:
                n_fin = int(torch.poisson(torch.tensor([spec.finish_rate]), generator=self.g).item())
                n_fin = min(n_fin, len(self.running))
                if n_fin:
                    pick = torch.randperm(len(self.running), generator=self.g)[:n_fin].tolist()
                    for idx in sorted(pick, reverse=True):
                        sid = self.running.pop(idx)
                        self.alloc.free_sequence(sid)
                        finished.append(sid)
                n_join = int(torch.poisson(torch.tensor([spec.join_rate]), generator=self.g).item())
                n_join = min(n_join, spec.max_seqs - len(self.running))
                for _ in range(n_join):
                    L = int(torch.randint(lo, hi + 1, (1,), generator=self.g))
                    sid = self._new_id()
                    join_slots[sid] = torch.tensor(self.alloc.add_sequence(sid, L), dtype=torch.int64)
                    self.running.append(sid)
                    joined.append(sid)
            slots = [self.alloc.append_token(sid) for sid in self.running]
            yield TraceStep(
                step=step, finished=finished, joined=joined, join_slots=join_slots,
                seq_ids=list(self.running),
                slot_mapping=torch.tensor(slots, dtype=torch.int64),
                block_tables=self.alloc.block_table(self.running, self.width),
                context_lens=torch.tensor([self.alloc.length[s] for s in self.running], dtype=torch.int32))


def rope_cos_sin(max_position: int, head_dim: int, theta: float = 10000.0) -> torch.Tensor:
    """The rotary table the decode step reads: [max_position, head_dim] fp32 with cos in the first half
    and sin in the second, angle(pos, i) = pos * theta^(-2i / head_dim), computed in fp64, rounded once.
    (An input table like a weight: Qwen3 uses theta 1e6, LLaMA-3 5e5.)"""
    half = head_dim // 2
    inv = theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / head_dim)
    ang = torch.arange(max_position, dtype=torch.float64)[:, None] * inv[None, :]
    return torch.cat([torch.cos(ang), torch.sin(ang)], dim=1).to(torch.float32).contiguous()


# ----------------------------------------------------------------------------
# Chunked prefill: C new tokens per sequence after P cached ones.
# ----------------------------------------------------------------------------
@dataclass(frozen=True)
class PrefillSpec:
    name: str
    description: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    chunk_lens: tuple          # C_b
    prefix_range: tuple        # P_b ~ U{lo..hi}
    max_blocks_per_seq: int


PREFILL_SPECS = {
    "prefill_tiny": PrefillSpec("prefill_tiny", "2 seqs, chunks 5 and 33, 4 q / 2 kv, D 64", 4, 2, 64, (5, 33),
                                (0, 40), 6),
    "prefill_qwen3_0.6b": PrefillSpec("prefill_qwen3_0.6b", "Qwen3-0.6B layer: 4 chunks of 512 after 0..2048 cached",
                                      16, 8, 128, (512, 512, 512, 512), (0, 2048), 160),
    "prefill_llama3_8b_one": PrefillSpec("prefill_llama3_8b_one",
                                         "LLaMA-3-8B layer: one chunk of 512 after 2048..3584 cached (32 q / 8 kv)",
                                         32, 8, 128, (512,), (2048, 3584), 256),
    "prefill_llama3_8b": PrefillSpec("prefill_llama3_8b",
                                     "LLaMA-3-8B layer: 8 chunks of 512 after 0..3584 cached (32 q / 8 kv)",
                                     32, 8, 128, (512,) * 8, (0, 3584), 256),
}


@dataclass
class PrefillCase:
    spec: PrefillSpec
    q: torch.Tensor              # [T, Hq, D] bf16
    k_cache: torch.Tensor        # [NB, Hkv, 16, D]
    v_cache: torch.Tensor
    block_tables: torch.Tensor   # [B, W] int32
    context_lens: torch.Tensor   # [B] int32 = prefix + chunk
    query_start: torch.Tensor    # [B + 1] int32
    new_k: torch.Tensor          # [T, Hkv, D]: the chunks' K/V, to append before attending
    new_v: torch.Tensor
    slot_mapping: torch.Tensor   # [T] int64
    scale: float

    def to(self, device) -> "PrefillCase":
        return PrefillCase(self.spec, *(t.to(device) for t in (
            self.q, self.k_cache, self.v_cache, self.block_tables, self.context_lens, self.query_start, self.new_k,
            self.new_v, self.slot_mapping)), self.scale)


def make_prefill_case(name: str | PrefillSpec, seed: int = 0, prefixes=None, device="cpu") -> PrefillCase:
    spec = PREFILL_SPECS[name] if isinstance(name, str) else name
    g = make_generator(seed)
    B = len(spec.chunk_lens)
    lo, hi = spec.prefix_range
    pre = [int(x) for x in (prefixes if prefixes is not None else torch.randint(lo, hi + 1, (B,), generator=g))]
    lens = [p + c for p, c in zip(pre, spec.chunk_lens)]
    if max(lens) > spec.max_blocks_per_seq * BLOCK_SIZE:
        raise ValueError("sequence longer than the block table")
    num_blocks = sum(-(-L // BLOCK_SIZE) for L in lens) + 4
    alloc = BlockAllocator(num_blocks, g)
    chunk_slots = []
    for b, (p, L) in enumerate(zip(pre, lens)):
        s = alloc.add_sequence(b, L)
        chunk_slots += s[p:]
    tables = alloc.block_table(list(range(B)), spec.max_blocks_per_seq)
    T = sum(spec.chunk_lens)
    qs = [0]
    for c in spec.chunk_lens:
        qs.append(qs[-1] + c)
    Hq, Hkv, D = spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    return PrefillCase(spec, randn_bf16((T, Hq, D), g), randn_bf16((num_blocks, Hkv, BLOCK_SIZE, D), g),
                       randn_bf16((num_blocks, Hkv, BLOCK_SIZE, D), g), tables,
                       torch.tensor(lens, dtype=torch.int32), torch.tensor(qs, dtype=torch.int32),
                       randn_bf16((T, Hkv, D), g), randn_bf16((T, Hkv, D), g),
                       torch.tensor(chunk_slots, dtype=torch.int64), 1.0 / math.sqrt(D)).to(device)


def prefill_flops(context_lens, query_start, num_q_heads: int, head_dim: int) -> int:
    """Causal attention flops of a prefill call: 4 * D per (query row, visible key, q head)."""
    lens = [int(x) for x in context_lens]
    qs = [int(x) for x in query_start]
    total = 0
    for b, L in enumerate(lens):
        C = qs[b + 1] - qs[b]
        P = L - C
        total += C * P + C * (C + 1) // 2
    return 4 * head_dim * num_q_heads * total
