"""Seeded random sweeps of decode, chunked prefill and cascade decode
configurations against the fp64 oracle.

Each case draws the KV type (bf16, FP8 E4M3, 4-bit), the group size, the
head size, the number of KV heads, the batch, lengths that mix random values
with block-boundary edge cases (0, 1, 15, 16, 17, 31, 32, 33, 255, 256, 257),
the pool's partition setting (one equal slice per warp, or fixed slices of 16,
64 or 512 tokens), and the way into the decode kernels: dense block tables
after paged_kv_append, the CSR page list ("Memory Management in LLM Serving
Systems", "Walking the table"), or the fused append + decode step.  Every
case is small enough for the oracle to take about a second; together they
cross shapes that the named workloads leave out.  The prefill sweep draws
chunks around the 128-row tile edge (and empty, single-token and
whole-cache chunks); the cascade sweep draws shared prefixes of 1 to 39
blocks under batches of 1 to 40 (the "Prefix sharing" section of "Memory
Management in LLM Serving Systems"), with the cascade forced on."""
import numpy as np
import pytest
import torch

import gqa_decode_attention_paged_gb300 as pkv
import workloads as wl
from gpu_util import (assert_close, bf16_dev, fill, i32_dev, make_pool, mirror, mirror_bytes, out_f64, pool_bytes,
                      step_inputs)

pytestmark = pytest.mark.gpu

EDGE = np.array([0, 1, 15, 16, 17, 31, 32, 33, 255, 256, 257])


def _pool_matches(pool, m, dtype):
    """The pool after the step holds, byte for byte, what the oracle's
    append wrote (codes, and for 4-bit pools the value parameters too)."""
    gk, gv = pool_bytes(pool)
    if dtype == "int4":
        vp = pool.v_params_view().cpu().numpy()
        return (np.array_equal(gk, m.k) and np.array_equal(gv, m.v)
                and np.array_equal(vp.view(np.uint32), m.v_params.view(np.uint32)))
    mk, mv = mirror_bytes(m)
    return np.array_equal(gk, mk) and np.array_equal(gv, mv)


def _case(i):
    rng = np.random.default_rng([4242, i])
    dtype = ("bf16", "fp8", "int4")[i % 3]
    d_head = (64, 128)[int(rng.integers(2))]
    n_kv = (1, 2, 4, 8)[int(rng.integers(4))]
    G = (1, 2, 4, 8)[int(rng.integers(4))]
    batch = int(rng.integers(1, 41))
    lens = np.where(rng.random(batch) < 0.3, rng.choice(EDGE, batch), rng.integers(1, 3000, batch))
    partition = (0, 0, 16, 64, 512)[int(rng.integers(5))]
    mode = ("dense", "csr", "step")[int(rng.integers(3))]
    return dtype, d_head, n_kv, G, lens.astype(np.int64), partition, mode


@pytest.mark.parametrize("i", range(24))
def test_random_decode_matches_oracle(i):
    dtype, d_head, n_kv, G, lens, partition, mode = _case(i)
    w = wl.build(f"rand{i}", n_kv * G, n_kv, d_head, lens, dtype=dtype, seed=500 + i)
    m = mirror(w)
    ref = m.decode(w.q, w.block_tables, w.context_lens, w.scale)
    with make_pool(w, partition) as pool:
        fill(pool, w)
        d = step_inputs(w)
        if mode == "step":  # the append of each sequence's newest token fused into the decode
            out = pkv.paged_decode_step(pool, d["q"], d["k"], d["v"], d["tables"], d["lens"], float(w.scale))
        else:
            pkv.paged_kv_append(pool, d["k"], d["v"], d["slots"])
            if mode == "dense":
                out = pkv.paged_decode_attention(pool, d["q"], d["tables"], d["lens"], float(w.scale))
            else:  # each sequence's used table entries, concatenated
                nblk = (w.context_lens.astype(np.int64) + 15) // 16
                indptr = np.concatenate([[0], np.cumsum(nblk)]).astype(np.int32)
                indices = np.concatenate([w.block_tables[b, :nblk[b]] for b in range(w.batch)] +
                                         [np.zeros(0, np.int32)]).astype(np.int32)
                out = pkv.paged_decode_attention_csr(pool, d["q"], i32_dev(indptr), i32_dev(indices), d["lens"],
                                                     float(w.scale))
        torch.cuda.synchronize()
        what = f"case {i}: {dtype} d{d_head} n_kv {n_kv} G {G} batch {w.batch} partition {partition} {mode}"
        assert pool.get_error() == 0, what
        assert _pool_matches(pool, m, dtype), what + ": pool bytes"
        got = out_f64(out)
    assert_close(got, ref, what)
    # zero-length sequences give zero rows
    zero = w.context_lens == 0
    assert not np.any(got[zero]), what


def _prefill_case(i):
    rng = np.random.default_rng([4343, i])
    dtype = ("bf16", "fp8")[i % 2]
    d_head = (64, 128)[int(rng.integers(2))]
    n_kv = (1, 2, 4, 8)[int(rng.integers(4))]
    G = (1, 2, 4, 8)[int(rng.integers(4))]
    batch = int(rng.integers(1, 7))
    lens = rng.integers(1, 600, batch)
    # chunk of new tokens per sequence (its last positions): empty, one token, the whole cache, or
    # around the 128-row tile edge
    chunks = np.array([min(int(c), int(x)) for c, x in zip(
        lens, rng.choice([0, 1, 2, 31, 127, 128, 129, 200, 10_000], batch))])
    return dtype, d_head, n_kv, G, lens.astype(np.int64), chunks.astype(np.int64)


@pytest.mark.parametrize("i", range(12))
def test_random_prefill_matches_oracle(i):
    dtype, d_head, n_kv, G, lens, chunks = _prefill_case(i)
    w = wl.build(f"rpf{i}", n_kv * G, n_kv, d_head, lens, dtype=dtype, seed=600 + i)
    rng = np.random.default_rng([4344, i])
    q = wl.f32_to_bf16_bits(rng.normal(size=(int(chunks.sum()), w.n_q, w.d_head)).astype(np.float32))
    indptr = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    ref = mirror(w).prefill(q, indptr, w.block_tables, w.context_lens, w.scale)
    with make_pool(w) as pool:
        fill(pool, w)
        d = step_inputs(w)
        pkv.paged_kv_append(pool, d["k"], d["v"], d["slots"])
        out = pkv.paged_prefill_attention(pool, bf16_dev(q), i32_dev(indptr), d["tables"], d["lens"], float(w.scale))
        torch.cuda.synchronize()
        what = f"prefill case {i}: {dtype} d{d_head} n_kv {n_kv} G {G} lens {list(lens)} chunks {list(chunks)}"
        assert pool.get_error() == 0, what
        got = out_f64(out)
    assert_close(got, ref, what)


def _cascade_case(i):
    rng = np.random.default_rng([4545, i])
    dtype = ("bf16", "fp8")[i % 2]
    d_head = (64, 128)[int(rng.integers(2))]
    n_kv = (1, 2, 4, 8)[int(rng.integers(4))]
    G = (1, 2, 4, 8)[int(rng.integers(4))]
    batch = int(rng.integers(1, 41))
    prefix = 16 * int(rng.integers(1, 40))
    tails = rng.integers(1, 400, batch)  # every sequence extends past the prefix
    return dtype, d_head, n_kv, G, prefix, (prefix + tails).astype(np.int64)


@pytest.mark.parametrize("i", range(10))
def test_random_cascade_matches_oracle(i):
    dtype, d_head, n_kv, G, prefix, lens = _cascade_case(i)
    w = wl.build(f"rcp{i}", n_kv * G, n_kv, d_head, lens, dtype=dtype, seed=700 + i, shared_prefix_tokens=prefix)
    ref = mirror(w).decode(w.q, w.block_tables, w.context_lens, w.scale)
    with make_pool(w) as pool:
        fill(pool, w)
        d = step_inputs(w)
        pkv.paged_kv_append(pool, d["k"], d["v"], d["slots"])
        pool.set_cascade_mode(pkv.CASCADE_ALWAYS)  # the cascade's kernels whatever the prefix length
        out = pkv.paged_decode_attention_prefix(pool, d["q"], i32_dev(w.block_tables[0, :prefix // 16]), d["tables"],
                                                d["lens"], float(w.scale))
        torch.cuda.synchronize()
        what = f"cascade case {i}: {dtype} d{d_head} n_kv {n_kv} G {G} batch {w.batch} prefix {prefix}"
        assert pool.get_error() == 0, what
        got = out_f64(out)
    assert_close(got, ref, what)
