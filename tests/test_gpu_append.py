"""Append / scatter on the GPU against the oracle: bit-exact, whole pool."""
import numpy as np
import pytest
import torch

import gqa_decode_attention_paged_gb300 as pkv
import oracle
import workloads as wl
from gpu_util import bf16_dev, fill, i64_dev, make_pool, mirror, mirror_bytes, pool_bytes, run_step

pytestmark = pytest.mark.gpu


def _assert_pool_equal(pool, m):
    gk, gv = pool_bytes(pool)
    mk, mv = mirror_bytes(m)
    assert np.array_equal(gk, mk), f"K pool differs in {int((gk != mk).sum())} bytes"
    assert np.array_equal(gv, mv), f"V pool differs in {int((gv != mv).sum())} bytes"


@pytest.mark.parametrize("make", [
    lambda: wl.tiny(),
    lambda: wl.build("ragged64", 8, 2, 64, [1, 15, 16, 17, 31, 33, 200], seed=8),
    lambda: wl.build("ragged128", 32, 8, 128, [5, 16, 47, 300], seed=9),
    lambda: wl.build("fp8_64", 8, 2, 64, [3, 16, 17, 90], dtype="fp8", seed=10),
    lambda: wl.build("fp8_128", 16, 8, 128, [1, 64, 65, 400], dtype="fp8", seed=11),
])
def test_append_bitexact_small(make):
    w = make()
    with make_pool(w) as pool:
        fill(pool, w)
        run_step(pool, w)
        torch.cuda.synchronize()
        _assert_pool_equal(pool, mirror(w))
        assert pool.get_error() == 0


@pytest.mark.parametrize("name", ["llama3_8b", "fp8_lognormal", "shared_prefix"])
def test_append_bitexact_full_workloads(name):
    w = wl.NAMED[name]()
    with make_pool(w) as pool:
        fill(pool, w)
        run_step(pool, w)
        torch.cuda.synchronize()
        _assert_pool_equal(pool, mirror(w))
        assert pool.get_error() == 0


@pytest.mark.parametrize("scale", [1.0, 0.37, 0.0123, 3.0e-3])
def test_fp8_quantiser_exhaustive_over_bf16(scale):
    """Every finite bf16 pattern, quantised with one scale, equals the
    oracle's brute-force E4M3 encoder (ties, subnormals, saturation, -0)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    exp = (bits >> 7) & 0xFF
    bits = bits[exp != 0xFF]  # drop Inf/NaN
    D = 64
    T = (len(bits) + D - 1) // D
    pad = np.zeros(T * D, dtype=np.uint16)
    pad[:len(bits)] = bits
    kb = pad.reshape(T, 1, D)
    vb = kb[::-1].copy()
    nb = (T + 15) // 16
    s = np.array([scale], dtype=np.float32)
    m = oracle.PoolMirror(nb, 16, 1, D, oracle.E4M3, s, s)
    slots = np.arange(T, dtype=np.int64)
    m.append(kb, vb, slots)
    with pkv.kv_pool_create(nb, 16, 1, D, pkv.FP8_E4M3) as pool:
        pool.set_fp8_scales(s, s)
        pkv.paged_kv_append(pool, bf16_dev(kb), bf16_dev(vb), i64_dev(slots))
        torch.cuda.synchronize()
        _assert_pool_equal(pool, m)


def test_append_skips_padding_and_flags_out_of_range():
    D = 128
    with pkv.kv_pool_create(4, 16, 2, D) as pool:
        kb = wl.normal_bf16_bits((4, 2, D), (77, 1))
        vb = wl.normal_bf16_bits((4, 2, D), (77, 2))
        slots = np.array([-1, 5, 64, 63], dtype=np.int64)  # pad, ok, past the end, ok
        pkv.paged_kv_append(pool, bf16_dev(kb), bf16_dev(vb), i64_dev(slots))
        bits = pool.get_error(clear=True)
        assert bits == pkv.DEVERR_SLOT_RANGE
        assert pool.get_error() == 0
        m = oracle.PoolMirror(4, 16, 2, D)
        assert m.append(kb, vb, slots) == 1
        _assert_pool_equal(pool, m)


def test_append_host_validation():
    with pkv.kv_pool_create(4, 16, 2, 64) as pool:
        k = torch.zeros(3, 2, 64, dtype=torch.bfloat16, device="cuda")
        s = torch.zeros(3, dtype=torch.int64, device="cuda")
        with pytest.raises(ValueError):
            pkv.paged_kv_append(pool, k.float(), k, s)
        with pytest.raises(ValueError):
            pkv.paged_kv_append(pool, k[:, :1], k[:, :1], s)
        lib = pkv.load()
        # misaligned k_new is refused by the library itself
        st = lib.paged_kv_append(pool.handle, k.data_ptr() + 2, k.data_ptr(), s.data_ptr(), 1, None)
        assert st == 1
        assert lib.paged_kv_append(pool.handle, k.data_ptr(), k.data_ptr(), s.data_ptr(), -1, None) == 1
        assert lib.paged_kv_append(pool.handle, None, None, None, 0, None) == 0
    with pkv.kv_pool_create(4, 16, 2, 64, pkv.FP8_E4M3) as pool8:
        with pytest.raises(pkv.PagedKVError):
            pkv.paged_kv_append(pool8, k, k, s)  # scales not set
        with pytest.raises(pkv.PagedKVError):
            pool8.set_fp8_scales(np.array([0.1, 0.0]), np.array([0.1, 0.1]))


def test_layout_is_the_documented_one():
    # one (block, KV head) entry: 16 key rows then 16 value rows (strides in bf16 elements)
    with pkv.kv_pool_create(10, 16, 8, 128) as pool:
        lay = pool.layout()
        assert lay["stride_token"] == 128
        assert lay["stride_head"] == 32 * 128
        assert lay["stride_block"] == 8 * 32 * 128
        assert lay["bytes_per_array"] == 10 * 8 * 16 * 128 * 2
        assert lay["alloc_bytes"] == 2 * lay["bytes_per_array"]
        assert lay["k"] % 256 == 0 and lay["v"] - lay["k"] == 16 * 128 * 2
        k, v = pool_bytes(pool)
        assert not k.any() and not v.any()  # zero-filled at creation
    with pkv.kv_pool_create(10, 16, 8, 64, pkv.FP8_E4M3) as pool:
        lay = pool.layout()
        assert (lay["stride_token"], lay["stride_head"], lay["stride_block"]) == (64, 32 * 64, 8 * 32 * 64)
        assert lay["v"] - lay["k"] == 16 * 64
