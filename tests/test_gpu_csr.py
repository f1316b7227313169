"""Decode through the CSR page table (kv_indptr / kv_indices): the pages'
own worked example ("Memory Management in LLM Serving Systems", "Method 3:
PagedAttention" and "Walking the table", fixture tests/golden/page_walk.json)
and random CSR tables, against the oracle (which reads the same blocks
through an equivalent dense table) and against the dense-table decode."""
import json
import os

import numpy as np
import pytest
import torch

import gqa_decode_attention_paged_gb300 as pkv
import oracle
import workloads as wl
from gpu_util import assert_close, bf16_dev, i32_dev, i64_dev, out_f64

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rand_bf16(rng, shape):
    return wl.f32_to_bf16_bits(rng.standard_normal(size=shape).astype(np.float32)).reshape(shape)


def _dense(indptr, indices, batch):
    """The same tables as a -1-padded dense [batch][W] array."""
    W = max(1, max(indptr[b + 1] - indptr[b] for b in range(batch)))
    t = np.full((batch, W), -1, dtype=np.int32)
    for b in range(batch):
        row = indices[indptr[b]:indptr[b + 1]]
        t[b, :len(row)] = row
    return t


def _setup(num_blocks, n_kv, d, seed):
    rng = np.random.default_rng(seed)
    pool = pkv.kv_pool_create(num_blocks, 16, n_kv, d, pkv.BF16)
    m = oracle.PoolMirror(num_blocks, 16, n_kv, d)
    T = num_blocks * 16
    k, v = _rand_bf16(rng, (T, n_kv, d)), _rand_bf16(rng, (T, n_kv, d))
    slots = np.arange(T, dtype=np.int64)
    pkv.paged_kv_append(pool, bf16_dev(k), bf16_dev(v), i64_dev(slots))
    m.append(k, v, slots)
    return rng, pool, m


@pytest.mark.parametrize("lens_kind", ["full", "partial"])
def test_csr_walk_of_the_pages_example(lens_kind):
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "page_walk.json")))
    indptr, indices = np.array(g["kv_indptr"], dtype=np.int32), np.array(g["kv_indices"], dtype=np.int32)
    B = len(indptr) - 1
    pages = np.diff(indptr)
    lens = pages * 16 if lens_kind == "full" else np.maximum(1, pages * 16 - np.array([5, 0, 9, 15]))
    lens = lens.astype(np.int32)
    n_kv, d, n_q = 8, 128, 32
    rng, pool, m = _setup(18, n_kv, d, seed=31)
    q = _rand_bf16(rng, (B, n_q, d))
    scale = float(np.float32(1 / np.sqrt(d)))
    out = pkv.paged_decode_attention_csr(pool, bf16_dev(q), i32_dev(indptr), i32_dev(indices), i32_dev(lens), scale)
    dense = _dense(indptr, indices, B)
    ref = m.decode(q, dense, lens, scale)
    torch.cuda.synchronize()
    assert_close(out_f64(out), ref, "CSR walk")
    # request 2 reads pages 2, 5, 0 (the pages' walk): the dense row says the same
    assert list(dense[2, :3]) == g["request_2_pages"]
    dout = pkv.paged_decode_attention(pool, bf16_dev(q), i32_dev(dense), i32_dev(lens), scale)
    torch.cuda.synchronize()
    assert_close(out_f64(out), out_f64(dout), "CSR against dense tables")
    assert pool.get_error() == 0
    pool.close()


@pytest.mark.parametrize("G", [1, 4, 8])
def test_csr_random_tables_with_empty_rows(G):
    n_kv, d = 4, 64 if G == 1 else 128
    n_q = n_kv * G
    NB = 300
    rng, pool, m = _setup(NB, n_kv, d, seed=40 + G)
    B = 23
    widths = rng.integers(0, 30, size=B)
    widths[[0, 7]] = 0  # empty rows
    indptr = np.concatenate([[0], np.cumsum(widths)]).astype(np.int32)
    indices = rng.integers(0, NB, size=int(indptr[-1])).astype(np.int32)
    lens = np.array([rng.integers(max(1, 16 * (w - 1) + 1), 16 * w + 1) if w else 0 for w in widths], dtype=np.int32)
    q = _rand_bf16(rng, (B, n_q, d))
    scale = float(np.float32(1 / np.sqrt(d)))
    out = pkv.paged_decode_attention_csr(pool, bf16_dev(q), i32_dev(indptr), i32_dev(indices), i32_dev(lens), scale)
    ref = m.decode(q, _dense(indptr, indices, B), lens, scale)
    torch.cuda.synchronize()
    got = out_f64(out)
    assert_close(got, ref, "random CSR")
    assert not got[0].any() and not got[7].any()
    assert pool.get_error() == 0
    pool.close()


def test_csr_bad_rows_are_empty_and_flagged():
    n_kv, d, n_q = 8, 128, 32
    rng, pool, m = _setup(40, n_kv, d, seed=51)
    indptr = np.array([0, 3, 2, 5, 99], dtype=np.int32)  # row 1 runs backwards, row 3 past n_indices
    indices = rng.integers(0, 40, size=6).astype(np.int32)
    lens = np.array([40, 20, 33, 16], dtype=np.int32)
    q = _rand_bf16(rng, (4, n_q, d))
    scale = float(np.float32(1 / np.sqrt(d)))
    out = pkv.paged_decode_attention_csr(pool, bf16_dev(q), i32_dev(indptr), i32_dev(indices), i32_dev(lens), scale)
    torch.cuda.synchronize()
    got = out_f64(out)
    bits = pool.get_error(clear=True)
    assert bits & pkv.DEVERR_BLOCK_RANGE and bits & pkv.DEVERR_CTX_RANGE
    assert not got[1].any() and not got[3].any()
    good = np.array([0, 2])
    dense = np.full((4, 3), -1, dtype=np.int32)
    dense[0] = indices[0:3]
    dense[2, :3] = indices[2:5]
    ref = m.decode(q[good], dense[good], np.array([40, 33], dtype=np.int32), scale)
    assert_close(got[good], ref, "valid rows beside bad ones")
    pool.close()
