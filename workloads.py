"""Seeded synthetic inputs for paged GQA decode attention.

This module is shared by the tests, ``bench.py`` and ``__graft_entry__``; it
feeds both the CUDA path and the CPU oracle.  It holds none of the attention
arithmetic.  Besides drawing random numbers it plays the host-side block
manager that a serving engine would run: it hands out physical block ids from
a shuffled free list, writes each sequence's block table and gives every
token its slot (physical block x block_size + offset), as described in
"KV cache, PagedAttention and FlashAttention", Problem 4, "The idea"
(blocks are allocated when the previous one fills, anywhere in the pool).

Recipe (every draw is seeded; the same seed gives the same bytes on any host
and any thread count):

* K, V and q values are fp32 draws from N(0, 1) rounded to bf16 (round to
  nearest even, via the torch CPU cast), kept as raw 16-bit patterns.
* Each sequence's ``context_len`` is its length after this step's append: the
  step appends the token at position ``context_len - 1``, and every earlier
  position is filled beforehand (the prefill that populates the cache).
* A shared prefix (``shared_prefix_tokens`` > 0) lives in blocks that every
  block table points to; it is filled once.
* FP8 scales (per KV head, separate for K and V) are the fp32 amax of that
  head's source values over every token of the workload, divided by 448.
* 4-bit key parameters (per KV head and channel) are the channel's min over
  every token of the workload (zero point) and (max - min) / 15 (scale);
  value rows get theirs when appended.
* ``scale`` is fp32(1/sqrt(d_head)).

The named workloads follow the shapes of the pages' examples: a tiny
paged case, the Llama3-8B attention shape ("Memory Management in LLM Serving
Systems", "KV cache sizing"), the 70B long-context shape ("KV cache, PagedAttention
and FlashAttention", Problem 3), an FP8 KV batch with log-normal lengths
(Problem 3's FP8 row; the page's "Practise it" fragmentation exercise uses
log-normal lengths), a shared-prefix batch ("Memory Management in LLM
Serving Systems", "Prefix sharing") and the Llama3-8B shape on a 4-bit KV
pool (Problem 3's 4-bit row).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16
_CHUNK = 1 << 22


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def normal_f32(n: int, key: tuple) -> np.ndarray:
    """``n`` fp32 draws from N(0, 1); chunk i uses the stream seeded by key + (i,)."""
    out = np.empty(n, dtype=np.float32)
    n_chunks = (n + _CHUNK - 1) // _CHUNK

    def work(i):
        s, e = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        np.random.default_rng(list(key) + [i]).standard_normal(e - s, dtype=np.float32, out=out[s:e])

    if n_chunks <= 1:
        for i in range(n_chunks):
            work(i)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(n_chunks)))
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest even) with the torch CPU cast; raw uint16 patterns."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen raw bf16 patterns to fp32 (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16_bits(shape, key: tuple) -> np.ndarray:
    n = int(np.prod(shape))
    return f32_to_bf16_bits(normal_f32(n, key)).reshape(shape)


@dataclass
class Workload:
    """One decode step's worth of seeded inputs plus the prefill that precedes it."""

    name: str
    n_q: int
    n_kv: int
    d_head: int
    block_size: int
    dtype: str  # "bf16", "fp8" or "int4"
    num_blocks: int
    context_lens: np.ndarray  # int32 [B], lengths after the step's append
    block_tables: np.ndarray  # int32 [B, W]; -1 past each sequence's last block
    fill_k: np.ndarray  # uint16 [T_fill, n_kv, D]
    fill_v: np.ndarray
    fill_slots: np.ndarray  # int64 [T_fill]
    step_k: np.ndarray  # uint16 [B, n_kv, D]
    step_v: np.ndarray
    step_slots: np.ndarray  # int64 [B]; -1 for a sequence with no token this step
    q: np.ndarray  # uint16 [B, n_q, D]
    scale: np.float32
    k_scale: np.ndarray | None = None  # float32 [n_kv] (fp8), [n_kv, d_head] (int4)
    v_scale: np.ndarray | None = None
    k_zero: np.ndarray | None = None   # float32 [n_kv, d_head] (int4 key zero points)
    shared_prefix_tokens: int = 0
    seed: int = 0
    notes: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 1

    @property
    def kv_bytes_per_token_head(self) -> int:
        """Bytes one cached token stores per KV head: K and V rows (4-bit: two
        codes per byte, plus the value row's fp32 scale and zero point)."""
        if self.dtype == "int4":
            return self.d_head + 8
        return 2 * self.d_head * self.elem_bytes

    def describe(self) -> dict:
        return {
            "workload": self.name,
            "n_q": self.n_q,
            "n_kv": self.n_kv,
            "d_head": self.d_head,
            "block_size": self.block_size,
            "kv_dtype": self.dtype,
            "batch": self.batch,
            "num_blocks": self.num_blocks,
            "max_blocks_per_seq": self.max_blocks_per_seq,
            "context_tokens_total": int(self.context_lens.astype(np.int64).sum()),
            "context_len_min": int(self.context_lens.min()) if self.batch else 0,
            "context_len_max": int(self.context_lens.max()) if self.batch else 0,
            "shared_prefix_tokens": self.shared_prefix_tokens,
            "seed": self.seed,
        }


def build(name: str, n_q: int, n_kv: int, d_head: int, context_lens, *, dtype: str = "bf16",
          block_size: int = BLOCK_SIZE, seed: int = 0, slack: float = 1.25,
          num_blocks: int | None = None, max_blocks_per_seq: int | None = None,
          shared_prefix_tokens: int = 0, scale: float | None = None,
          permute_pool: bool = True) -> Workload:
    """Seeded workload with the given lengths; see the module docstring for the recipe."""
    if n_q % n_kv:
        raise ValueError("n_q must be a multiple of n_kv")
    cl = np.asarray(context_lens, dtype=np.int64)
    B = int(cl.shape[0])
    BS = block_size
    if shared_prefix_tokens % BS:
        raise ValueError("a shared prefix must fill whole blocks")
    n_shared = shared_prefix_tokens // BS
    if shared_prefix_tokens and np.any(cl <= shared_prefix_tokens):
        raise ValueError("every sequence must extend past the shared prefix")

    def blocks_for(c):
        return (int(c) + BS - 1) // BS

    private = [blocks_for(c) - n_shared for c in cl]
    needed = n_shared + int(sum(private))
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(slack * needed)))
    if num_blocks < needed:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {needed}")
    rng = np.random.default_rng([seed, 0])
    free = rng.permutation(num_blocks) if permute_pool else np.arange(num_blocks)
    W = max([blocks_for(c) for c in cl] + [1])
    if max_blocks_per_seq is not None:
        if max_blocks_per_seq < W:
            raise ValueError("max_blocks_per_seq smaller than the longest sequence")
        W = max_blocks_per_seq
    tables = np.full((B, W), -1, dtype=np.int32)
    shared_ids = free[:n_shared]
    cursor = n_shared
    for b in range(B):
        tables[b, :n_shared] = shared_ids
        k = private[b]
        tables[b, n_shared:n_shared + k] = free[cursor:cursor + k]
        cursor += k

    # Slots of every position filled before the step (the block manager's job).
    def slots_for(b, positions):
        positions = np.asarray(positions, dtype=np.int64)
        return tables[b, positions // BS].astype(np.int64) * BS + positions % BS

    fill_parts = []
    if shared_prefix_tokens:
        fill_parts.append(slots_for(0, np.arange(shared_prefix_tokens)))
    for b in range(B):
        start = shared_prefix_tokens
        stop = max(int(cl[b]) - 1, start)
        if stop > start:
            fill_parts.append(slots_for(b, np.arange(start, stop)))
    fill_slots = np.concatenate(fill_parts) if fill_parts else np.zeros(0, dtype=np.int64)
    step_slots = np.array([slots_for(b, [int(cl[b]) - 1])[0] if cl[b] > 0 else -1 for b in range(B)],
                          dtype=np.int64)

    T = int(fill_slots.shape[0])
    fill_k = normal_bf16_bits((T, n_kv, d_head), (seed, 1))
    fill_v = normal_bf16_bits((T, n_kv, d_head), (seed, 2))
    step_k = normal_bf16_bits((B, n_kv, d_head), (seed, 3))
    step_v = normal_bf16_bits((B, n_kv, d_head), (seed, 4))
    q = normal_bf16_bits((B, n_q, d_head), (seed, 5))

    k_scale = v_scale = k_zero = None
    if dtype == "fp8":
        def amax(fill, step):
            a = np.zeros(n_kv, dtype=np.float32)
            for s in range(0, T, 65536):
                a = np.maximum(a, np.abs(bf16_bits_to_f32(fill[s:s + 65536])).max(axis=(0, 2)))
            if B:
                a = np.maximum(a, np.abs(bf16_bits_to_f32(step)).max(axis=(0, 2)))
            a[a == 0] = 1.0
            return (a / np.float32(448.0)).astype(np.float32)

        k_scale = amax(fill_k, step_k)
        v_scale = amax(fill_v, step_v)
    elif dtype == "int4":
        # keys: per (KV head, channel) min and max over the workload's tokens
        lo = np.full((n_kv, d_head), np.inf, dtype=np.float32)
        hi = np.full((n_kv, d_head), -np.inf, dtype=np.float32)
        for part in [fill_k[s:s + 65536] for s in range(0, T, 65536)] + ([step_k] if B else []):
            x = bf16_bits_to_f32(part)
            lo = np.minimum(lo, x.min(axis=0))
            hi = np.maximum(hi, x.max(axis=0))
        lo[~np.isfinite(lo)] = 0.0
        hi[~np.isfinite(hi)] = 0.0
        k_scale = ((hi - lo) / np.float32(15.0)).astype(np.float32)
        k_scale[k_scale == 0] = 1.0
        k_zero = lo.astype(np.float32)
    elif dtype != "bf16":
        raise ValueError("dtype must be bf16, fp8 or int4")

    sc = np.float32(1.0 / math.sqrt(d_head)) if scale is None else np.float32(scale)
    return Workload(name=name, n_q=n_q, n_kv=n_kv, d_head=d_head, block_size=BS, dtype=dtype,
                    num_blocks=int(num_blocks), context_lens=cl.astype(np.int32),
                    block_tables=tables, fill_k=fill_k, fill_v=fill_v, fill_slots=fill_slots,
                    step_k=step_k, step_v=step_v, step_slots=step_slots, q=q, scale=sc,
                    k_scale=k_scale, v_scale=v_scale, k_zero=k_zero, shared_prefix_tokens=shared_prefix_tokens,
                    seed=seed)


# --------------------------------------------------------------------------
# The named workloads
# --------------------------------------------------------------------------

def tiny(seed: int = 1) -> Workload:
    """4 sequences of {1, 17, 100, 256} tokens, n_q=8, n_kv=2, d_head=64, a
    64-block pool whose 26 used ids are the first of a seeded permutation."""
    return build("tiny_paged_decode", 8, 2, 64, [1, 17, 100, 256], seed=seed, num_blocks=64)


def llama3_8b(seed: int = 2, batch: int = 64) -> Workload:
    """Llama3-8B attention shape: n_q=32, n_kv=8, d_head=128, batch 64,
    lengths uniform in [1024, 2048], pool sized 1.25x the blocks in use."""
    rng = np.random.default_rng([seed, 100])
    cl = rng.integers(1024, 2049, size=batch)
    return build("llama3_8b_decode_b64", 32, 8, 128, cl, seed=seed)


def long_context_70b(seed: int = 3, batch: int = 16, context: int = 32768) -> Workload:
    """70B long-context shape: n_q=64, n_kv=8, d_head=128, batch 16, every
    sequence at 32768 tokens (2 GiB of bf16 K+V read per call)."""
    need = batch * (context // BLOCK_SIZE)
    return build(f"llama70b_longctx_b{batch}_{context // 1024}k", 64, 8, 128, [context] * batch, seed=seed,
                 num_blocks=need + 64)


def fp8_lognormal(seed: int = 4, batch: int = 256) -> Workload:
    """FP8 E4M3 KV: n_q=32, n_kv=8, d_head=128, batch 256, lengths
    log-normal with median 1024 and sigma 0.8, clipped to [16, 8192]."""
    rng = np.random.default_rng([seed, 100])
    z = rng.standard_normal(batch)
    cl = np.clip(np.rint(1024.0 * np.exp(0.8 * z)), 16, 8192).astype(np.int64)
    return build("fp8_e4m3_lognormal_b256", 32, 8, 128, cl, dtype="fp8", seed=seed,
                 max_blocks_per_seq=8192 // BLOCK_SIZE)


def shared_prefix(seed: int = 5, batch: int = 128) -> Workload:
    """128 sequences whose tables share the same first 64 blocks (a
    1024-token prefix), each with a private tail of 0..1024 tokens plus the
    token this step appends."""
    rng = np.random.default_rng([seed, 100])
    tails = rng.integers(0, 1025, size=batch)
    cl = 1024 + tails + 1
    return build("shared_prefix_b128", 32, 8, 128, cl, seed=seed, shared_prefix_tokens=1024,
                 max_blocks_per_seq=129)


def shared_prefix_long(seed: int = 7, batch: int = 128) -> Workload:
    """128 sequences sharing an 8192-token prefix (512 blocks, 32 MB of K/V),
    each with a private tail of 0..1024 tokens plus the token this step
    appends: the regime where plain decode re-reads the prefix once per
    sequence (about 4 GB per call, from L2) and the cascade reads it once."""
    rng = np.random.default_rng([seed, 100])
    tails = rng.integers(0, 1025, size=batch)
    cl = 8192 + tails + 1
    return build("shared_prefix_long_b128", 32, 8, 128, cl, seed=seed, shared_prefix_tokens=8192,
                 max_blocks_per_seq=577)


def int4_llama3(seed: int = 6, batch: int = 128) -> Workload:
    """The Llama3-8B decode shape (n_q=32, n_kv=8, d_head=128, lengths
    uniform in [1024, 2048]) on a 4-bit KV pool, batch 128 so that the
    cache (about 210 MB) is larger than L2."""
    rng = np.random.default_rng([seed, 100])
    cl = rng.integers(1024, 2049, size=batch)
    return build("llama3_8b_int4_b128", 32, 8, 128, cl, dtype="int4", seed=seed)


NAMED = {
    "tiny": tiny,
    "llama3_8b": llama3_8b,
    "long_context_70b": long_context_70b,
    # the same kernel on 4 sequences (537 MB of KV): a profiling-sized case
    "long_context_70b_b4": lambda: long_context_70b(batch=4),
    "fp8_lognormal": fp8_lognormal,
    "shared_prefix": shared_prefix,
    "shared_prefix_long": shared_prefix_long,
    "int4_llama3": int4_llama3,
}
