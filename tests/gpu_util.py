"""Shared helpers of the GPU parity tests (not a test module)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_cache_275_gb300 as pkv

# Tolerance for attention against the fp64 oracle (bf16 inputs, fp32 accumulation, bf16 output):
# max |gpu - oracle| <= 1e-2 and ||gpu - oracle||_2 / ||oracle||_2 <= 5e-3.
MAX_ABS = 1e-2
REL_RMS = 5e-3


def errors(gpu_out: torch.Tensor, ref: np.ndarray) -> tuple[float, float]:
    g = gpu_out.detach().to("cpu", torch.float64).numpy().reshape(ref.shape)
    diff = g - ref
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    denom = float(np.sqrt(np.mean(ref * ref))) if ref.size else 1.0
    rel_rms = float(np.sqrt(np.mean(diff * diff)) / denom) if denom > 0 else float(np.sqrt(np.mean(diff * diff)))
    return max_abs, rel_rms


def assert_close(gpu_out: torch.Tensor, ref: np.ndarray, what: str = "") -> tuple[float, float]:
    g = gpu_out.detach().to("cpu", torch.float64).numpy()
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    max_abs, rel_rms = errors(gpu_out, ref)
    assert max_abs <= MAX_ABS and rel_rms <= REL_RMS, f"{what}: max_abs {max_abs:.3g}, rel_rms {rel_rms:.3g}"
    return max_abs, rel_rms


def gpu_step(case_gpu, num_partitions: int = 0, out: torch.Tensor | None = None) -> torch.Tensor:
    """One decode step through the C ABI: append this step's token, then attend."""
    c = case_gpu
    pkv.kv_append(c.new_k, c.new_v, c.slot_mapping, c.k_cache, c.v_cache)
    if out is None:
        out = torch.empty_like(c.q)
    pkv.paged_decode_attention(c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale, out,
                               num_partitions=num_partitions)
    return out


def oracle_step(case_cpu) -> tuple[np.ndarray, torch.Tensor, torch.Tensor]:
    """The same step on the oracle; returns (out, k_cache, v_cache) after the append."""
    c = case_cpu
    kc, vc = c.k_cache.clone(), c.v_cache.clone()
    assert oracle.kv_append(c.new_k, c.new_v, c.slot_mapping, kc, vc) == oracle.OK
    out, st = oracle.paged_decode_attention(c.q, kc, vc, c.block_tables, c.context_lens, c.scale)
    assert st == oracle.OK
    return out, kc, vc


def device_errors() -> int:
    return pkv.get_and_clear_device_error()
