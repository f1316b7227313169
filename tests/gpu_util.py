"""Helpers for the GPU parity tests: upload a seeded workload, run it through
the C ABI (via the thin binding), and compare with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import gqa_decode_attention_paged_gb300 as pkv
import oracle

# Tolerances on attention outputs against the fp64 oracle (bf16 and FP8 KV).
MAX_ABS = 1e-2
MEAN_ABS = 1e-3


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def i64_dev(x) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int64)).cuda()


def i32_dev(x) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).cuda()


def make_pool(w, partition_tokens: int | None = None) -> pkv.Pool:
    dt = {"bf16": pkv.BF16, "fp8": pkv.FP8_E4M3, "int4": pkv.INT4}[w.dtype]
    pool = pkv.kv_pool_create(w.num_blocks, w.block_size, w.n_kv, w.d_head, dt)
    if w.dtype == "fp8":
        pool.set_fp8_scales(w.k_scale, w.v_scale)
    if w.dtype == "int4":
        pool.set_int4_key_params(w.k_scale, w.k_zero)
    if partition_tokens:
        pool.set_partition_tokens(partition_tokens)
    return pool


def fill(pool, w, chunk: int = 1 << 20):
    """Prefill every position but the step's token, in chunks of tokens."""
    T = w.fill_slots.shape[0]
    for s in range(0, T, chunk):
        e = min(T, s + chunk)
        pkv.paged_kv_append(pool, bf16_dev(w.fill_k[s:e]), bf16_dev(w.fill_v[s:e]), i64_dev(w.fill_slots[s:e]))


def step_inputs(w) -> dict:
    return {
        "k": bf16_dev(w.step_k), "v": bf16_dev(w.step_v), "slots": i64_dev(w.step_slots),
        "q": bf16_dev(w.q), "tables": i32_dev(w.block_tables), "lens": i32_dev(w.context_lens),
    }


def run_step(pool, w, dev=None):
    """One step on the GPU: append the new token of every sequence, then decode."""
    dev = dev or step_inputs(w)
    pkv.paged_kv_append(pool, dev["k"], dev["v"], dev["slots"])
    return pkv.paged_decode_attention(pool, dev["q"], dev["tables"], dev["lens"], float(w.scale))


def mirror(w) -> oracle.PoolMirror:
    dt = {"bf16": oracle.BF16, "fp8": oracle.E4M3, "int4": oracle.INT4}[w.dtype]
    m = oracle.PoolMirror(w.num_blocks, w.block_size, w.n_kv, w.d_head, dt, w.k_scale, w.v_scale, w.k_zero)
    m.append(w.fill_k, w.fill_v, w.fill_slots)
    m.append(w.step_k, w.step_v, w.step_slots)
    return m


def pool_bytes(pool):
    return pool.k_view().cpu().numpy(), pool.v_view().cpu().numpy()


def mirror_bytes(m):
    return (m.k.view(np.uint8).reshape(m.num_blocks, m.n_kv, m.block_size, -1),
            m.v.view(np.uint8).reshape(m.num_blocks, m.n_kv, m.block_size, -1))


def out_f64(out: torch.Tensor) -> np.ndarray:
    return out.float().cpu().numpy().astype(np.float64)


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    err = np.abs(got - ref)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max abs {mx:.3e}, mean abs {mean:.3e}"
    return mx, mean
