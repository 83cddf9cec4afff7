"""CPU oracle for the paged KV-cache hot path (fp64, plain C, pthreads).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py`` may import this package.
The product path (``paged_kv_cache_275_gb300``) never imports it and has no
CPU fallback; this package never imports the product path either.

The computation lives in ``pkv_oracle.c`` (see its header for the definitions
and the page sections they follow).  This module only builds that file with
gcc and marshals numpy / torch-CPU buffers into it.

Parity pins (tests/test_oracle_pins.py) tie every function here to something
other than itself: closed forms, invariants and brute force against
torch's float64 scaled-dot-product attention on un-paged tensors.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "pkv_oracle.c"
_LIB_PATH = _HERE / "libpkv_oracle.so"

# Return-code bits of the C functions.
OK = 0
BAD_ARGUMENT = 1
SLOT_OUT_OF_RANGE = 2
DUPLICATE_SLOT = 4
BLOCK_ID_OUT_OF_RANGE = 8
CONTEXT_LEN_OUT_OF_RANGE = 16

_lib = None


def build(force: bool = False) -> Path:
    """Compile pkv_oracle.c into libpkv_oracle.so next to it (gcc, no -ffast-math).

    ``-ffp-contract=off`` keeps every multiply and add separately rounded, so the
    x86 and Arm builds round the same way.
    """
    if force or not _LIB_PATH.exists() or _LIB_PATH.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB_PATH.with_suffix(f".so.tmp{os.getpid()}")
        cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
               "-pthread", str(_SRC), "-o", str(tmp), "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(str(_LIB_PATH))
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.pkv_oracle_kv_append.argtypes = [P, P, P, i64, i32, i32, P, P, i64, i32]
        lib.pkv_oracle_kv_append.restype = ctypes.c_int
        lib.pkv_oracle_paged_decode_attention.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i64, i32,
                                                          dbl, P, i32]
        lib.pkv_oracle_paged_decode_attention.restype = ctypes.c_int
        lib.pkv_oracle_paged_decode_sampled.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i64, i32,
                                                        dbl, P, P, i64, P, i32]
        lib.pkv_oracle_paged_decode_sampled.restype = ctypes.c_int
        lib.pkv_oracle_copy_blocks.argtypes = [P, P, P, i64, i32, i32, i64, i32]
        lib.pkv_oracle_copy_blocks.restype = ctypes.c_int
        lib.pkv_oracle_float_to_bf16.argtypes = [P, P, i64]
        lib.pkv_oracle_float_to_bf16.restype = ctypes.c_int
        lib.pkv_oracle_rope.argtypes = [P, i64, i32, i32, P, P, i64]
        lib.pkv_oracle_rope.restype = ctypes.c_int
        lib.pkv_oracle_paged_prefill_attention.argtypes = [P, P, P, P, i32, P, P, i32, i32, i32, i32, i64, i32,
                                                           dbl, P, i32]
        lib.pkv_oracle_paged_prefill_attention.restype = ctypes.c_int
        _lib = lib
    return _lib


def _as_u16(x) -> np.ndarray:
    """bf16 torch tensor or uint16/int16 numpy array -> contiguous uint16 numpy view (shares memory)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            if x.device.type != "cpu":
                raise ValueError("oracle inputs must live on the CPU")
            if x.dtype != torch.bfloat16:
                raise ValueError(f"expected a bf16 tensor, got {x.dtype}")
            if not x.is_contiguous():
                raise ValueError("expected a contiguous tensor")
            return x.view(torch.int16).numpy().view(np.uint16)
    except ImportError:  # pragma: no cover
        pass
    a = np.asarray(x)
    if a.dtype not in (np.uint16, np.int16):
        raise ValueError(f"expected bf16 bits as uint16, got {a.dtype}")
    if not a.flags.c_contiguous:
        raise ValueError("expected a C-contiguous array")
    return a.view(np.uint16)


def _as(x, dtype) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x), dtype=dtype)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def kv_append(k, v, slot_mapping, k_cache, v_cache) -> int:
    """Oracle append, in place on CPU ``k_cache`` / ``v_cache`` ([NB, Hkv, bs, D] bf16).

    ``k``, ``v``: [N, Hkv, D] bf16; ``slot_mapping``: [N] int64.  Returns the C
    status bits (0 = OK).
    """
    kk, vv = _as_u16(k), _as_u16(v)
    kc, vc = _as_u16(k_cache), _as_u16(v_cache)
    slots = _as(slot_mapping, np.int64)
    if kc.ndim != 4 or kc.shape != vc.shape:
        raise ValueError("caches must be [num_blocks, num_kv_heads, block_size, head_dim]")
    num_blocks, hkv, bs, d = kc.shape
    n = slots.shape[0]
    if kk.size != n * hkv * d or vv.size != n * hkv * d:
        raise ValueError("k / v must be [N, num_kv_heads, head_dim]")
    return _load().pkv_oracle_kv_append(_ptr(kk), _ptr(vv), _ptr(slots), n, hkv, d, _ptr(kc), _ptr(vc),
                                        num_blocks, bs)


def _problem(q, k_cache, v_cache, block_tables, context_lens):
    qq = _as_u16(q)
    kc, vc = _as_u16(k_cache), _as_u16(v_cache)
    bt = _as(block_tables, np.int32)
    cl = _as(context_lens, np.int32)
    if qq.ndim != 3:
        raise ValueError("q must be [num_seqs, num_q_heads, head_dim]")
    num_seqs, hq, d = qq.shape
    num_blocks, hkv, bs, d2 = kc.shape
    if d2 != d or vc.shape != kc.shape:
        raise ValueError("cache / q head_dim mismatch")
    if bt.ndim != 2 or bt.shape[0] != num_seqs or cl.shape != (num_seqs,):
        raise ValueError("block_tables must be [num_seqs, W], context_lens [num_seqs]")
    return qq, kc, vc, bt, cl, num_seqs, hq, hkv, d, num_blocks, bs


def paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                           num_threads: int | None = None) -> tuple[np.ndarray, int]:
    """Oracle decode attention for every (seq, q head).  Returns (out [B, Hq, D] float64, status)."""
    qq, kc, vc, bt, cl, B, hq, hkv, d, nb, bs = _problem(q, k_cache, v_cache, block_tables, context_lens)
    out = np.zeros((B, hq, d), dtype=np.float64)
    st = _load().pkv_oracle_paged_decode_attention(
        _ptr(qq), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(cl), B, hq, hkv, d, nb, bs, float(scale),
        _ptr(out), num_threads or default_threads())
    return out, st


def paged_decode_sampled(q, k_cache, v_cache, block_tables, context_lens, scale: float, seq_idx, head_idx,
                         num_threads: int | None = None) -> tuple[np.ndarray, int]:
    """Oracle decode attention on sampled (seq, q head) pairs.  Returns (out [n, D] float64, status)."""
    qq, kc, vc, bt, cl, B, hq, hkv, d, nb, bs = _problem(q, k_cache, v_cache, block_tables, context_lens)
    si = _as(seq_idx, np.int32)
    hi = _as(head_idx, np.int32)
    if si.shape != hi.shape or si.ndim != 1:
        raise ValueError("seq_idx / head_idx must be equal-length 1-D")
    out = np.zeros((si.shape[0], d), dtype=np.float64)
    st = _load().pkv_oracle_paged_decode_sampled(
        _ptr(qq), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(cl), B, hq, hkv, d, nb, bs, float(scale),
        _ptr(si), _ptr(hi), si.shape[0], _ptr(out), num_threads or default_threads())
    return out, st


def copy_blocks(k_cache, v_cache, src_dst) -> int:
    """Oracle block copy, in place on CPU caches ([NB, Hkv, bs, D] bf16); src_dst: [n, 2] int64."""
    kc, vc = _as_u16(k_cache), _as_u16(v_cache)
    pairs = _as(src_dst, np.int64).reshape(-1, 2)
    num_blocks, hkv, bs, d = kc.shape
    return _load().pkv_oracle_copy_blocks(_ptr(kc), _ptr(vc), _ptr(pairs), pairs.shape[0], hkv, d, num_blocks, bs)


def float_to_bf16(x) -> np.ndarray:
    """fp32 values -> bf16 bit patterns (uint16), round to nearest even."""
    a = _as(x, np.float32).ravel()
    out = np.zeros(a.shape, dtype=np.uint16)
    _load().pkv_oracle_float_to_bf16(_ptr(a), _ptr(out), a.size)
    return out


def rope(x, positions, cos_sin) -> int:
    """Oracle rotate-half RoPE, in place on a CPU bf16 tensor x [n, heads, D]; cos_sin [max_pos, D] fp32."""
    xx = _as_u16(x)
    pos = _as(positions, np.int64)
    cs = _as(cos_sin, np.float32)
    n, heads, d = xx.shape
    if pos.shape != (n,) or cs.ndim != 2 or cs.shape[1] != d:
        raise ValueError("positions must be [n] and cos_sin [max_position, head_dim]")
    return _load().pkv_oracle_rope(_ptr(xx), n, heads, d, _ptr(pos), _ptr(cs), cs.shape[0])


def decode_step(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale, cos_sin=None,
                num_threads: int | None = None):
    """One decode step by composition: RoPE of q and the new k at position L - 1, append of the new
    k / v at that position's slot (through the block table), then attention.  Returns
    (out float64 [B, Hq, D], status); k_cache / v_cache are updated in place.
    """
    import torch
    lens = _as(context_lens, np.int64)
    bt = _as(block_tables, np.int64)
    B = lens.shape[0]
    live = lens > 0
    pos = np.where(live, lens - 1, 0)
    q = q.clone()
    k_new = k_new.clone()
    if cos_sin is not None:
        st = rope(q, pos, cos_sin) | rope(k_new, pos, cos_sin)
        if st:
            return None, st
    bs = k_cache.shape[2]
    slots = np.full(B, -1, dtype=np.int64)
    for b in range(B):
        if live[b]:
            p = int(pos[b])
            slots[b] = int(bt[b, p // bs]) * bs + p % bs
    st = kv_append(k_new, v_new.contiguous(), torch.from_numpy(slots), k_cache, v_cache)
    if st:
        return None, st
    return paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale, num_threads)


def paged_prefill_attention(q, k_cache, v_cache, block_tables, context_lens, query_start, scale: float,
                            num_threads: int | None = None) -> tuple[np.ndarray, int]:
    """Oracle chunked prefill: q [T, Hq, D] bf16, query_start [B + 1]; returns (out [T, Hq, D] float64, status)."""
    qq = _as_u16(q)
    kc, vc = _as_u16(k_cache), _as_u16(v_cache)
    bt = _as(block_tables, np.int32)
    cl = _as(context_lens, np.int32)
    qs = _as(query_start, np.int32)
    T, hq, d = qq.shape
    num_blocks, hkv, bs, d2 = kc.shape
    B = cl.shape[0]
    if d2 != d or qs.shape != (B + 1,) or bt.shape[0] != B or int(qs[-1]) != T:
        raise ValueError("shape mismatch")
    out = np.zeros((T, hq, d), dtype=np.float64)
    st = _load().pkv_oracle_paged_prefill_attention(
        _ptr(qq), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(cl), _ptr(qs), B, hq, hkv, d, num_blocks, bs,
        float(scale), _ptr(out), num_threads or default_threads())
    return out, st
