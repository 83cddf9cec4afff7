"""ctypes binding of libpagedkv.so (include/pagedkv.h).

Argument marshalling only: shapes are read from the tensors, pointers and the
current CUDA stream are passed through, and every step of the computation
runs in the library's kernels.  There is no CPU or PyTorch fallback: if the
library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import threading
from pathlib import Path

import torch

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libpagedkv.so"

OK = 0
ERR_INVALID_ARGUMENT = 1
ERR_UNSUPPORTED = 2
ERR_CUDA = 3
ERR_NO_FREE_BLOCKS = 4
STATUS_NAMES = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARGUMENT", 2: "PKV_ERR_UNSUPPORTED", 3: "PKV_ERR_CUDA",
                4: "PKV_ERR_NO_FREE_BLOCKS"}

DEVERR_SLOT_OUT_OF_RANGE = 0x1
DEVERR_BLOCK_ID_OUT_OF_RANGE = 0x2
DEVERR_CONTEXT_LEN_NEGATIVE = 0x4
DEVERR_CONTEXT_LEN_TOO_LONG = 0x8
DEVERR_PIPELINE_TIMEOUT = 0x10
DEVERR_COPY_OUT_OF_RANGE = 0x20
DEVERR_POSITION_OUT_OF_TABLE = 0x40
DEVERR_SMEM_ALIGNMENT = 0x80

PHASE_PARTITION = 1
PHASE_MERGE = 2
PHASE_ALL = 3

BLOCK_SIZE = 16
MAX_SEQS = 4096

# Every exported symbol of include/pagedkv.h.
EXPORTS = (
    "pkv_kv_append",
    "pkv_decode_workspace_size",
    "pkv_decode_default_partitions",
    "pkv_paged_decode_attention",
    "pkv_paged_decode_attention_split",
    "pkv_paged_decode_attention_static",
    "pkv_copy_blocks",
    "pkv_decode_step",
    "pkv_paged_prefill_attention",
    "pkv_paged_prefill_attention_split",
    "pkv_prefill_workspace_size",
    "pkv_prefill_default_splits",
    "pkv_bm_create",
    "pkv_bm_destroy",
    "pkv_bm_num_free",
    "pkv_bm_add_sequence",
    "pkv_bm_append_slots",
    "pkv_bm_fork",
    "pkv_bm_free_sequence",
    "pkv_bm_block_tables",
    "pkv_bm_ref_count",
    "pkv_get_and_clear_device_error",
    "pkv_selftest_wait_timeout",
    "pkv_last_error_message",
    "pkv_kernel_launch_count",
)


class PagedKVError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None
_lock = threading.Lock()


def load(path: Path | str | None = None) -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = Path(path) if path else LIB_PATH
        if not p.exists():
            raise ImportError(f"{p} is missing: build it with `python -m paged_kv_cache_275_gb300.build` "
                              "(there is no fallback path)")
        lib = ctypes.CDLL(str(p))
        V, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        lib.pkv_kv_append.argtypes = [V, V, V, I64, I32, I32, V, V, I64, I32, V]
        lib.pkv_decode_workspace_size.argtypes = [I32, I32, I32, I32, I32, I32, ctypes.POINTER(SZ)]
        lib.pkv_decode_default_partitions.argtypes = [I32, I32, I32, I32, I32, ctypes.POINTER(I32)]
        lib.pkv_paged_decode_attention.argtypes = [V, V, V, V, I32, V, I32, I32, I32, I32, I64, I32,
                                                   ctypes.c_float, V, V, SZ, V]
        lib.pkv_paged_decode_attention_split.argtypes = [V, V, V, V, I32, V, I32, I32, I32, I32, I64, I32,
                                                         ctypes.c_float, V, V, SZ, I32, I32, V]
        lib.pkv_paged_decode_attention_static.argtypes = [V, V, V, V, I32, V, I32, I32, I32, I32, I64, I32,
                                                          ctypes.c_float, V, V]
        lib.pkv_copy_blocks.argtypes = [V, V, V, I32, I32, I32, I64, V]
        lib.pkv_decode_step.argtypes = [V, V, V, V, I64, V, V, V, I32, V, I32, I32, I32, I32, I64, I32,
                                        ctypes.c_float, V, V, SZ, V]
        lib.pkv_paged_prefill_attention.argtypes = [V, V, V, V, I32, V, V, I32, I32, I32, I32, I32, I64, I32,
                                                    ctypes.c_float, V, V]
        lib.pkv_paged_prefill_attention_split.argtypes = [V, V, V, V, I32, V, V, I32, I32, I32, I32, I32, I64, I32,
                                                          ctypes.c_float, V, I32, V, SZ, V]
        lib.pkv_prefill_workspace_size.argtypes = [I32, I32, I32, I32, I32, I32, ctypes.POINTER(SZ)]
        lib.pkv_prefill_default_splits.argtypes = [I32, I32, I32, I32, ctypes.POINTER(I32)]
        lib.pkv_bm_create.argtypes = [I64, V, ctypes.POINTER(V)]
        lib.pkv_bm_destroy.argtypes = [V]
        lib.pkv_bm_num_free.argtypes = [V, ctypes.POINTER(I64)]
        lib.pkv_bm_add_sequence.argtypes = [V, I64, I64, V]
        lib.pkv_bm_append_slots.argtypes = [V, V, I32, V, V, ctypes.POINTER(I32)]
        lib.pkv_bm_fork.argtypes = [V, I64, I64]
        lib.pkv_bm_free_sequence.argtypes = [V, I64]
        lib.pkv_bm_block_tables.argtypes = [V, V, I32, I32, V, V]
        lib.pkv_bm_ref_count.argtypes = [V, I64, ctypes.POINTER(I32)]
        lib.pkv_get_and_clear_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), V]
        lib.pkv_selftest_wait_timeout.argtypes = [ctypes.c_uint64, V]
        for name in ("pkv_kv_append", "pkv_decode_workspace_size", "pkv_decode_default_partitions",
                     "pkv_paged_decode_attention", "pkv_paged_decode_attention_split",
                     "pkv_paged_decode_attention_static", "pkv_get_and_clear_device_error",
                     "pkv_selftest_wait_timeout", "pkv_copy_blocks", "pkv_decode_step", "pkv_paged_prefill_attention",
                     "pkv_paged_prefill_attention_split", "pkv_prefill_workspace_size", "pkv_prefill_default_splits",
                     "pkv_bm_create", "pkv_bm_destroy", "pkv_bm_num_free", "pkv_bm_add_sequence",
                     "pkv_bm_append_slots", "pkv_bm_fork", "pkv_bm_free_sequence", "pkv_bm_block_tables",
                     "pkv_bm_ref_count"):
            getattr(lib, name).restype = ctypes.c_int
        lib.pkv_last_error_message.argtypes = []
        lib.pkv_last_error_message.restype = ctypes.c_char_p
        lib.pkv_kernel_launch_count.argtypes = []
        lib.pkv_kernel_launch_count.restype = ctypes.c_uint64
        if path is None:
            _lib = lib
        return lib


def _check(status: int) -> None:
    if status != OK:
        msg = load().pkv_last_error_message().decode(errors="replace")
        raise PagedKVError(status, msg)


def _stream_handle(stream: torch.cuda.Stream | None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _require(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int, device: torch.device | None = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def kv_append(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
              v_cache: torch.Tensor, stream: torch.cuda.Stream | None = None) -> None:
    """Scatter k/v [N, Hkv, D] bf16 into k_cache/v_cache [NB, Hkv, 16, D] at slot_mapping [N] int64 (in place)."""
    _require(k_cache, "k_cache", torch.bfloat16, 4)
    dev = k_cache.device
    _require(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _require(k, "k", torch.bfloat16, 3, dev)
    _require(v, "v", torch.bfloat16, 3, dev)
    _require(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    nb, hkv, bs, d = k_cache.shape
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    n = slot_mapping.shape[0]
    if k.shape != (n, hkv, d) or v.shape != (n, hkv, d):
        raise ValueError(f"k/v must be [{n}, {hkv}, {d}], got {tuple(k.shape)} / {tuple(v.shape)}")
    with torch.cuda.device(dev):
        _check(load().pkv_kv_append(k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), n, hkv, d,
                                    k_cache.data_ptr(), v_cache.data_ptr(), nb, bs, _stream_handle(stream)))


def workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int, max_blocks_per_seq: int,
                   num_partitions: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(load().pkv_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                            num_partitions, ctypes.byref(out)))
    return int(out.value)


def default_partitions(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                       max_blocks_per_seq: int) -> int:
    out = ctypes.c_int32(0)
    _check(load().pkv_decode_default_partitions(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                                ctypes.byref(out)))
    return int(out.value)


# One scratch buffer per (device, stream): calls on one stream run in order and may share it.
_workspaces: dict[tuple[int, int], torch.Tensor] = {}


def _workspace(device: torch.device, stream_handle: int, nbytes: int) -> torch.Tensor:
    key = (device.index, stream_handle)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def paged_decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                           out: torch.Tensor, *, num_partitions: int = 0, phases: int = PHASE_ALL,
                           workspace: torch.Tensor | None = None, stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """out[b, h] = softmax(scale * q[b, h] K^T) V over context_lens[b] tokens found through block_tables[b].

    q, out: [B, Hq, D] bf16; k_cache, v_cache: [NB, Hkv, 16, D] bf16; block_tables: [B, W] int32;
    context_lens: [B] int32.  Returns ``out``.
    """
    _require(q, "q", torch.bfloat16, 3)
    dev = q.device
    _require(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _require(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _require(block_tables, "block_tables", torch.int32, 2, dev)
    _require(context_lens, "context_lens", torch.int32, 1, dev)
    _require(out, "out", torch.bfloat16, 3, dev)
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    if v_cache.shape != k_cache.shape or d2 != d:
        raise ValueError("cache shapes do not match q")
    if out.shape != q.shape:
        raise ValueError("out must have the shape of q")
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables / context_lens batch mismatch")
    W = block_tables.shape[1]
    lib = load()
    with torch.cuda.device(dev):
        sh = _stream_handle(stream)
        if B == 0:
            return out
        nbytes = workspace_size(B, hq, hkv, d, W, num_partitions)
        if workspace is None:
            workspace = _workspace(dev, sh, nbytes)
        elif workspace.device != dev or workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError(f"workspace must be a {nbytes}-byte buffer on {dev}")
        wsize = workspace.numel() * workspace.element_size()
        _check(lib.pkv_paged_decode_attention_split(
            q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(), W,
            context_lens.data_ptr(), B, hq, hkv, d, nb, bs, float(scale), out.data_ptr(), workspace.data_ptr(),
            wsize, num_partitions, phases, sh))
    return out


def get_and_clear_device_error(stream: torch.cuda.Stream | None = None) -> int:
    bits = ctypes.c_uint32(0)
    _check(load().pkv_get_and_clear_device_error(ctypes.byref(bits), _stream_handle(stream)))
    return int(bits.value)


def selftest_wait_timeout(limit_ns: int, stream: torch.cuda.Stream | None = None) -> None:
    """Launch one warp that waits, for at most limit_ns, on a shared-memory barrier nothing completes:
    the bounded wait of the attention kernels gives up and sets PKV_DEVERR_PIPELINE_TIMEOUT."""
    _check(load().pkv_selftest_wait_timeout(int(limit_ns), _stream_handle(stream)))


def kernel_launch_count() -> int:
    return int(load().pkv_kernel_launch_count())


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src_dst: torch.Tensor,
                stream: torch.cuda.Stream | None = None) -> None:
    """k_cache[dst] = k_cache[src] and v_cache[dst] = v_cache[src] for every row (src, dst) of src_dst [n, 2] int64."""
    _require(k_cache, "k_cache", torch.bfloat16, 4)
    dev = k_cache.device
    _require(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _require(src_dst, "src_dst", torch.int64, 2, dev)
    if v_cache.shape != k_cache.shape or src_dst.shape[1] != 2:
        raise ValueError("caches must match and src_dst must be [n, 2]")
    nb, hkv, _, d = k_cache.shape
    with torch.cuda.device(dev):
        _check(load().pkv_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(), src_dst.data_ptr(), src_dst.shape[0],
                                      hkv, d, nb, _stream_handle(stream)))


class BlockManager:
    """Host block manager of the C ABI (pkv_bm_*): allocation, append slots, fork, free, copy-on-write."""

    def __init__(self, num_blocks: int, initial_free_order=None):
        import numpy as np
        self._lib = load()
        self._h = ctypes.c_void_p()
        order = None
        if initial_free_order is not None:
            order = np.ascontiguousarray(np.asarray(initial_free_order, dtype=np.int64))
            if order.shape != (num_blocks,):
                raise ValueError("initial_free_order must hold num_blocks entries")
        ptr = order.ctypes.data if order is not None else None
        _check(self._lib.pkv_bm_create(int(num_blocks), ptr, ctypes.byref(self._h)))
        self.num_blocks = int(num_blocks)

    def close(self) -> None:
        if self._h:
            _check(self._lib.pkv_bm_destroy(self._h))
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def num_free(self) -> int:
        n = ctypes.c_int64(0)
        _check(self._lib.pkv_bm_num_free(self._h, ctypes.byref(n)))
        return int(n.value)

    def add_sequence(self, seq_id: int, num_tokens: int):
        import numpy as np
        slots = np.zeros(max(1, num_tokens), dtype=np.int64)
        _check(self._lib.pkv_bm_add_sequence(self._h, int(seq_id), int(num_tokens), slots.ctypes.data))
        return slots[:num_tokens]

    def append_slots(self, seq_ids):
        """Returns (slots [n] int64, copies [k, 2] int64 as (src, dst))."""
        import numpy as np
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        n = ids.shape[0]
        slots = np.zeros(max(1, n), dtype=np.int64)
        copies = np.zeros(max(1, 2 * n), dtype=np.int64)
        k = ctypes.c_int32(0)
        _check(self._lib.pkv_bm_append_slots(self._h, ids.ctypes.data, n, slots.ctypes.data, copies.ctypes.data,
                                             ctypes.byref(k)))
        return slots[:n], copies[:2 * k.value].reshape(-1, 2)

    def fork(self, parent_id: int, child_id: int) -> None:
        _check(self._lib.pkv_bm_fork(self._h, int(parent_id), int(child_id)))

    def free_sequence(self, seq_id: int) -> None:
        _check(self._lib.pkv_bm_free_sequence(self._h, int(seq_id)))

    def block_tables(self, seq_ids, width: int):
        """Returns (tables [n, width] int32 padded with -1, lengths [n] int32)."""
        import numpy as np
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        n = ids.shape[0]
        tables = np.zeros((max(1, n), width), dtype=np.int32)
        lens = np.zeros(max(1, n), dtype=np.int32)
        _check(self._lib.pkv_bm_block_tables(self._h, ids.ctypes.data, n, width, tables.ctypes.data, lens.ctypes.data))
        return tables[:n], lens[:n]

    def ref_count(self, block: int) -> int:
        c = ctypes.c_int32(0)
        _check(self._lib.pkv_bm_ref_count(self._h, int(block), ctypes.byref(c)))
        return int(c.value)


def decode_step(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                v_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                out: torch.Tensor, cos_sin: torch.Tensor | None = None, *, workspace: torch.Tensor | None = None,
                stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Fused decode step: RoPE (if cos_sin [max_pos, D] fp32 is given) of q and k_new at position
    context_len - 1, append of k_new / v_new at that position, attention.  Returns ``out``."""
    _require(q, "q", torch.bfloat16, 3)
    dev = q.device
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        _require(t, name, torch.bfloat16, 3, dev)
    _require(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _require(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _require(block_tables, "block_tables", torch.int32, 2, dev)
    _require(context_lens, "context_lens", torch.int32, 1, dev)
    _require(out, "out", torch.bfloat16, 3, dev)
    B, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    if k_new.shape != (B, hkv, d) or v_new.shape != (B, hkv, d) or out.shape != q.shape:
        raise ValueError("k_new / v_new must be [B, Hkv, D] and out the shape of q")
    cs_ptr, max_pos = None, 0
    if cos_sin is not None:
        _require(cos_sin, "cos_sin", torch.float32, 2, dev)
        if cos_sin.shape[1] != d:
            raise ValueError("cos_sin must be [max_position, head_dim]")
        cs_ptr, max_pos = cos_sin.data_ptr(), cos_sin.shape[0]
    W = block_tables.shape[1]
    with torch.cuda.device(dev):
        sh = _stream_handle(stream)
        if B == 0:
            return out
        nbytes = workspace_size(B, hq, hkv, d, W, 0)
        if workspace is None:
            workspace = _workspace(dev, sh, nbytes)
        wsize = workspace.numel() * workspace.element_size()
        _check(load().pkv_decode_step(q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), cs_ptr, max_pos,
                                      k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(), W,
                                      context_lens.data_ptr(), B, hq, hkv, d, nb, bs, float(scale), out.data_ptr(),
                                      workspace.data_ptr(), wsize, sh))
    return out


def prefill_workspace_size(num_seqs: int, max_query_len: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                           num_splits: int) -> int:
    """Bytes of the workspace of a split prefill call (0 for num_splits = 1)."""
    n = ctypes.c_size_t(0)
    _check(load().pkv_prefill_workspace_size(num_seqs, max_query_len, num_q_heads, num_kv_heads, head_dim, num_splits,
                                             ctypes.byref(n)))
    return n.value


def prefill_default_splits(num_seqs: int, max_query_len: int, num_q_heads: int, num_kv_heads: int) -> int:
    """The split count that keeps the call's CTAs in one wave on the current device (1 when it fills it)."""
    n = ctypes.c_int32(0)
    _check(load().pkv_prefill_default_splits(num_seqs, max_query_len, num_q_heads, num_kv_heads, ctypes.byref(n)))
    return n.value


def paged_prefill_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, context_lens: torch.Tensor, query_start: torch.Tensor,
                            max_query_len: int, scale: float, out: torch.Tensor,
                            stream: torch.cuda.Stream | None = None, num_splits: int = 1,
                            workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Chunked prefill: q / out [T, Hq, D] bf16, query_start [B + 1] int32; causal over each sequence's
    context_lens[b] - (chunk length) cached tokens plus the chunk.  ``num_splits`` > 1 splits each CTA's keys
    over that many CTAs and merges their partial states (a uint8 ``workspace`` of ``prefill_workspace_size``
    bytes, allocated here if not given); ``prefill_default_splits`` gives a count for calls that do not fill
    the GPU.  Returns ``out``."""
    _require(q, "q", torch.bfloat16, 3)
    dev = q.device
    _require(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _require(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _require(block_tables, "block_tables", torch.int32, 2, dev)
    _require(context_lens, "context_lens", torch.int32, 1, dev)
    _require(query_start, "query_start", torch.int32, 1, dev)
    _require(out, "out", torch.bfloat16, 3, dev)
    T, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    B = context_lens.shape[0]
    if out.shape != q.shape or query_start.shape[0] != B + 1 or block_tables.shape[0] != B:
        raise ValueError("shape mismatch")
    with torch.cuda.device(dev):
        if num_splits == 1:
            _check(load().pkv_paged_prefill_attention(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                                      block_tables.data_ptr(), block_tables.shape[1],
                                                      context_lens.data_ptr(), query_start.data_ptr(),
                                                      int(max_query_len), B, hq, hkv, d, nb, bs, float(scale),
                                                      out.data_ptr(), _stream_handle(stream)))
            return out
        if workspace is None:
            workspace = torch.empty(prefill_workspace_size(B, int(max_query_len), hq, hkv, d, int(num_splits)),
                                    dtype=torch.uint8, device=dev)
        _require(workspace, "workspace", torch.uint8, 1, dev)
        _check(load().pkv_paged_prefill_attention_split(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                                        block_tables.data_ptr(), block_tables.shape[1],
                                                        context_lens.data_ptr(), query_start.data_ptr(),
                                                        int(max_query_len), B, hq, hkv, d, nb, bs, float(scale),
                                                        out.data_ptr(), int(num_splits), workspace.data_ptr(),
                                                        workspace.numel(), _stream_handle(stream)))
    return out
