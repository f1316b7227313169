"""4-bit KV pools (keys with per-channel scale and zero point, values with
per-token scale and zero point; "KV cache, PagedAttention and
FlashAttention", Problem 3, "Trade-offs"): the append kernel's codes and
value parameters bit-exact against the oracle over the whole pool, and
decode against the oracle's fp64 attention over the dequantised values."""
import numpy as np
import pytest
import torch

import gqa_decode_attention_paged_gb300 as pkv
import workloads as wl
from gpu_util import assert_close, fill, i32_dev, make_pool, mirror, out_f64, pool_bytes, run_step, step_inputs

pytestmark = pytest.mark.gpu

CASES = [
    lambda: wl.build("i4_g4", 32, 8, 128, [1, 15, 16, 17, 300, 1000, 0, 2049], dtype="int4", seed=71),
    lambda: wl.build("i4_g8", 64, 8, 128, [700, 33, 4000], dtype="int4", seed=72),
    lambda: wl.build("i4_d64_g4", 8, 2, 64, [90, 5, 257, 16], dtype="int4", seed=73),
    lambda: wl.build("i4_mha_d64", 4, 4, 64, [100, 31], dtype="int4", seed=74),
    lambda: wl.build("i4_g2", 16, 8, 128, [64, 512, 3], dtype="int4", seed=75),
]


def _check_pool(pool, m):
    gk, gv = pool_bytes(pool)
    assert np.array_equal(gk, m.k) and np.array_equal(gv, m.v), "codes"
    vp = pool.v_params_view().cpu().numpy()
    assert np.array_equal(vp.view(np.uint32), m.v_params.view(np.uint32)), "value scale / zero point"


@pytest.mark.parametrize("make", CASES)
def test_int4_append_and_decode_match_oracle(make):
    w = make()
    with make_pool(w) as pool:
        fill(pool, w)
        out = run_step(pool, w)
        torch.cuda.synchronize()
        m = mirror(w)
        _check_pool(pool, m)
        ref = m.decode(w.q, w.block_tables, w.context_lens, w.scale)
        assert_close(out_f64(out), ref, w.name)
        assert pool.get_error() == 0


def test_int4_full_workload_sampled():
    """The bench's 4-bit workload at full size (Llama3-8B shape, batch 128),
    stepped as the bench steps it (append, then decode): the whole pool's codes
    and value parameters bit-exact, and sampled sequences' outputs against the
    oracle's fp64 attention."""
    w = wl.int4_llama3()
    with make_pool(w) as pool:
        fill(pool, w)
        out = run_step(pool, w)
        torch.cuda.synchronize()
        assert pool.get_error() == 0
        m = mirror(w)
        _check_pool(pool, m)
        rng = np.random.default_rng(7)
        idx = np.sort(rng.choice(w.batch, size=12, replace=False))
        ref = m.decode(w.q[idx], w.block_tables[idx], w.context_lens[idx], w.scale)
        assert_close(out_f64(out)[idx], ref, w.name + " (sampled)")


def test_int4_partitions_csr_and_noalloc_agree():
    w = CASES[1]()
    with make_pool(w, 64) as pool:
        fill(pool, w)
        d = step_inputs(w)
        pkv.paged_kv_append(pool, d["k"], d["v"], d["slots"])
        ref = mirror(w).decode(w.q, w.block_tables, w.context_lens, w.scale)
        out = pkv.paged_decode_attention(pool, d["q"], d["tables"], d["lens"], float(w.scale))
        torch.cuda.synchronize()
        assert_close(out_f64(out), ref, "64-token partitions")
        widths = [int((c + 15) // 16) for c in w.context_lens]
        indptr = np.concatenate([[0], np.cumsum(widths)]).astype(np.int32)
        indices = np.concatenate([w.block_tables[b, :widths[b]] for b in range(w.batch)]).astype(np.int32)
        out = pkv.paged_decode_attention_csr(pool, d["q"], i32_dev(indptr), i32_dev(indices), d["lens"],
                                             float(w.scale))
        torch.cuda.synchronize()
        assert_close(out_f64(out), ref, "CSR tables")
        out = pkv.paged_decode_attention_noalloc(pool, d["q"], d["tables"], d["lens"], float(w.scale))
        torch.cuda.synchronize()
        assert_close(out_f64(out), ref, "no-alloc scratch")
        assert pool.get_error() == 0


def test_int4_needs_key_params():
    w = CASES[2]()
    pool = pkv.kv_pool_create(w.num_blocks, 16, w.n_kv, w.d_head, pkv.INT4)
    d = step_inputs(w)
    with pytest.raises(pkv.PagedKVError):
        pkv.paged_kv_append(pool, d["k"], d["v"], d["slots"])
    with pytest.raises(pkv.PagedKVError):
        pool.set_int4_key_params(np.zeros((w.n_kv, w.d_head), np.float32), w.k_zero)  # scale 0
    pool.set_int4_key_params(w.k_scale, w.k_zero)
    lay = pool.layout()
    assert lay["stride_token"] == w.d_head // 2 and lay["bytes_per_array"] == w.num_blocks * w.n_kv * 16 * w.d_head // 2
    assert lay["v_params_bytes"] == w.num_blocks * w.n_kv * 16 * 8
    # one contiguous (block, KV head) entry: key codes, value codes, value parameters
    entry = 16 * w.d_head + 128
    assert lay["stride_head"] == entry and lay["stride_block"] == w.n_kv * entry
    assert lay["alloc_bytes"] == w.num_blocks * w.n_kv * entry
    assert lay["v"] - lay["k"] == 8 * w.d_head and lay["v_params"] - lay["k"] == 16 * w.d_head
    pool.close()


def test_int4_decode_step_matches_append_then_decode():
    """paged_decode_step on a 4-bit pool (append kernel with table-derived
    slots, then decode) leaves the same pool bytes as paged_kv_append with
    explicit slots and gives the oracle's answer."""
    w = CASES[0]()
    with make_pool(w) as pool:
        fill(pool, w)
        d = step_inputs(w)
        out = pkv.paged_decode_step(pool, d["q"], d["k"], d["v"], d["tables"], d["lens"], float(w.scale))
        torch.cuda.synchronize()
        m = mirror(w)
        _check_pool(pool, m)
        assert_close(out_f64(out), m.decode(w.q, w.block_tables, w.context_lens, w.scale), "int4 step")
        assert pool.get_error() == 0
