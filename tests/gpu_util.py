"""Helpers shared by the GPU parity tests: run one step through the C ABI and
through the oracle on the same seeded inputs, and compare."""
import numpy as np
import torch

import oracle
from paged_kv_cache_174_gb300 import ops
from paged_kv_cache_174_gb300 import workloads as W

# Attention tolerance (bf16 in, fp32 accumulate, bf16 out) against the fp64
# oracle: maximum absolute error and relative L2 error over all outputs.
MAX_ABS = 1e-2
REL_L2 = 5e-3


def run_gpu_step(b: W.PagedBatch, device="cuda", copy_first=True):
    """copy_blocks (if any), scatter, attention; returns (DeviceBatch, out)."""
    d = W.to_device(b, device)
    if copy_first and b.copy_pairs.size:
        ops.copy_blocks(d.k_cache, d.v_cache, d.copy_pairs)
    ops.reshape_and_cache(d.k_new, d.v_new, d.k_cache, d.v_cache, d.slot_mapping)
    out = torch.full_like(d.q, float("nan"))
    ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens,
                        d.query_start_loc, b.scale, max_q_len=b.max_q_len,
                        max_seq_len=b.max_seq_len, out=out)
    ops.check_device_errors()
    return d, out


def run_oracle_step(b: W.PagedBatch, attention=True):
    kc, vc = b.k_cache.copy(), b.v_cache.copy()
    if b.copy_pairs.size:
        oracle.copy_blocks(kc, vc, b.copy_pairs)
    oracle.reshape_and_cache(b.k_new, b.v_new, kc, vc, b.slot_mapping)
    ref = None
    if attention:
        ref = oracle.paged_attention(b.q, kc, vc, b.block_tables, b.seq_lens,
                                     b.query_start_loc, b.scale)
    return kc, vc, ref


def to_f64(out: torch.Tensor) -> np.ndarray:
    return W.f32_from_bf16(W.bits_of(out)).astype(np.float64)


def attn_errors(got: np.ndarray, ref: np.ndarray):
    diff = got - ref
    return float(np.abs(diff).max()), float(np.linalg.norm(diff) / np.linalg.norm(ref))


def assert_attn_close(got: np.ndarray, ref: np.ndarray, what=""):
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite outputs"
    mx, rel = attn_errors(got, ref)
    assert mx <= MAX_ABS and rel <= REL_L2, f"{what}: max abs {mx:.3e}, rel L2 {rel:.3e}"
    return mx, rel
