"""Chunked prefill attention over the paged cache against the oracle: each
sequence's chunk of new tokens (the last positions of its cache) attends
causally; shapes span group sizes, head sizes, one-token chunks (decode),
whole-sequence prefills, partial row tiles and empty chunks."""
import numpy as np
import pytest
import torch

import gqa_decode_attention_paged_gb300 as pkv
import workloads as wl
from gpu_util import assert_close, bf16_dev, fill, i32_dev, make_pool, mirror, out_f64, run_step

pytestmark = pytest.mark.gpu


def _chunks(w, chunks, seed):
    rng = np.random.default_rng(seed)
    q = wl.f32_to_bf16_bits(rng.normal(size=(int(sum(chunks)), w.n_q, w.d_head)).astype(np.float32))
    return q, np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)


CASES = [
    (lambda: wl.build("pf_g4", 32, 8, 128, [1, 40, 300, 1000], seed=101), [1, 17, 300, 64]),
    (lambda: wl.build("pf_g8", 64, 8, 128, [200, 33, 700], seed=102), [200, 0, 5]),
    (lambda: wl.build("pf_d64", 8, 2, 64, [90, 5, 257, 16], seed=103), [90, 5, 100, 16]),
    (lambda: wl.build("pf_mha", 4, 4, 64, [100, 31], seed=104), [60, 31]),
    (lambda: wl.build("pf_g2", 16, 8, 128, [64, 512, 3], seed=105), [33, 512, 2]),
    # FP8 E4M3 pools: the oracle dequantises the same E4M3 bytes with the pool's per-head scales
    (lambda: wl.build("pf_fp8_g4", 32, 8, 128, [1, 40, 300, 1000], dtype="fp8", seed=111), [1, 17, 300, 64]),
    (lambda: wl.build("pf_fp8_g8", 64, 8, 128, [200, 33, 700], dtype="fp8", seed=112), [200, 0, 5]),
    (lambda: wl.build("pf_fp8_d64", 8, 2, 64, [90, 5, 257, 16], dtype="fp8", seed=113), [90, 5, 100, 16]),
    (lambda: wl.build("pf_fp8_mha", 4, 4, 64, [100, 31], dtype="fp8", seed=114), [60, 31]),
    (lambda: wl.build("pf_fp8_g2", 16, 8, 128, [64, 512, 3], dtype="fp8", seed=115), [33, 512, 2]),
]


@pytest.mark.parametrize("make,chunks", CASES)
def test_prefill_matches_oracle(make, chunks):
    w = make()
    with make_pool(w) as pool:
        fill(pool, w)
        run_step(pool, w)  # the last position of every sequence
        q, indptr = _chunks(w, chunks, 7)
        out = pkv.paged_prefill_attention(pool, bf16_dev(q), i32_dev(indptr), i32_dev(w.block_tables),
                                          i32_dev(w.context_lens), float(w.scale))
        torch.cuda.synchronize()
        ref = mirror(w).prefill(q, indptr, w.block_tables, w.context_lens, w.scale)
        assert_close(out_f64(out), ref, w.name)
        assert pool.get_error() == 0


def test_prefill_one_token_chunks_are_decode():
    w = CASES[0][0]()
    with make_pool(w) as pool:
        fill(pool, w)
        run_step(pool, w)
        indptr = np.arange(w.batch + 1, dtype=np.int32)
        out = pkv.paged_prefill_attention(pool, bf16_dev(w.q), i32_dev(indptr), i32_dev(w.block_tables),
                                          i32_dev(w.context_lens), float(w.scale))
        torch.cuda.synchronize()
        assert_close(out_f64(out), mirror(w).decode(w.q, w.block_tables, w.context_lens, w.scale), "T = 1")


def test_prefill_flags_a_chunk_longer_than_its_cache():
    w = CASES[2][0]()
    with make_pool(w) as pool:
        fill(pool, w)
        run_step(pool, w)
        q, indptr = _chunks(w, [1, 9, 1, 1], 8)  # sequence 1 holds 5 tokens
        pkv.paged_prefill_attention(pool, bf16_dev(q), i32_dev(indptr), i32_dev(w.block_tables),
                                    i32_dev(w.context_lens), float(w.scale))
        torch.cuda.synchronize()
        assert pool.get_error(clear=True) & pkv.DEVERR_CTX_RANGE


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_prefill_full_size_sampled_rows(dtype):
    """The 64 x 512-token Llama3-8B chunk workload in the launch configuration
    the benchmark times (and the same on an FP8 pool); sampled rows checked
    against the oracle: row i of a chunk is the decode of its query over
    positions 0 .. C - T + i, so each sample is an oracle decode with that
    context length."""
    w = wl.llama3_8b() if dtype == "bf16" else wl.build(
        "llama3_8b_fp8_b64", 32, 8, 128, wl.llama3_8b().context_lens, dtype="fp8", seed=12)
    T = 512
    rng = np.random.default_rng(11)
    q = wl.f32_to_bf16_bits(rng.normal(size=(w.batch * T, w.n_q, w.d_head)).astype(np.float32))
    indptr = np.arange(0, w.batch * T + 1, T, dtype=np.int32)
    with make_pool(w) as pool:
        fill(pool, w)
        run_step(pool, w)
        out = pkv.paged_prefill_attention(pool, bf16_dev(q), i32_dev(indptr), i32_dev(w.block_tables),
                                          i32_dev(w.context_lens), float(w.scale))
        torch.cuda.synchronize()
        assert pool.get_error() == 0
        got = out_f64(out)
    seqs = np.array([0, 1, 17, 31, 32, 46, 62, 63])
    toks = np.array([0, 1, 31, 32, 127, 128, 300, 511])
    sb, si = np.meshgrid(seqs, toks, indexing="ij")
    sb, si = sb.ravel(), si.ravel()
    rows = sb * T + si
    lens = (w.context_lens[sb] - T + si + 1).astype(np.int32)
    ref = mirror(w).decode(q[rows], w.block_tables[sb], lens, w.scale)
    assert_close(got[rows], ref, "full-size sampled rows")


def test_prefill_bad_block_is_flagged_and_other_sequences_exact():
    w = CASES[0][0]()
    q, indptr = _chunks(w, [1, 17, 300, 64], 9)
    tables = w.block_tables.copy()
    tables[2, 3] = w.num_blocks + 5  # sequence 2 reads a block id past the pool
    with make_pool(w) as pool:
        fill(pool, w)
        run_step(pool, w)
        out = pkv.paged_prefill_attention(pool, bf16_dev(q), i32_dev(indptr), i32_dev(tables),
                                          i32_dev(w.context_lens), float(w.scale))
        torch.cuda.synchronize()
        assert pool.get_error(clear=True) & pkv.DEVERR_BLOCK_RANGE
        got = out_f64(out)
    keep = [0, 1, 3]
    sub_rows = np.concatenate([np.arange(indptr[b], indptr[b + 1]) for b in keep])
    sub_indptr = np.concatenate([[0], np.cumsum([indptr[b + 1] - indptr[b] for b in keep])]).astype(np.int32)
    ref = mirror(w).prefill(q[sub_rows], sub_indptr, tables[keep], w.context_lens[keep], w.scale)
    assert_close(got[sub_rows], ref, "sequences beside the bad one")


def test_prefill_rejects_4bit_pools():
    with pkv.kv_pool_create(8, 16, 2, 64, pkv.INT4) as pool:
        pool.set_int4_key_params(np.ones((2, 64)), np.zeros((2, 64)))
        q = torch.zeros(4, 4, 64, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(pkv.PagedKVError) as e:
            pkv.paged_prefill_attention(pool, q, i32_dev([0, 4]), i32_dev(np.zeros((1, 2))), i32_dev([20]), 0.125)
        assert e.value.status == 5
