"""Decode attention on the GPU against the fp64 oracle.

Tolerance (bf16 and FP8 KV alike, the oracle dequantising the same E4M3
bytes): max abs error <= 1e-2 and mean abs error <= 1e-3 over the outputs."""
import zlib

import numpy as np
import pytest
import torch

import gqa_decode_attention_paged_gb300 as pkv
import oracle
import workloads as wl
from gpu_util import (assert_close, bf16_dev, fill, i32_dev, make_pool, mirror, out_f64, run_step,
                      step_inputs)

pytestmark = pytest.mark.gpu


def _parity(w, partition_tokens=None):
    m = mirror(w)
    ref = m.decode(w.q, w.block_tables, w.context_lens, w.scale)
    with make_pool(w, partition_tokens) as pool:
        fill(pool, w)
        out = run_step(pool, w)
        torch.cuda.synchronize()
        assert pool.get_error() == 0
        got = out_f64(out)
    return assert_close(got, ref, w.name)


def test_tiny_workload():
    _parity(wl.tiny())


CASES = [
    # name, n_q, n_kv, d_head, lens, dtype, partition
    ("g4_d64", 8, 2, 64, [1, 17, 100, 256], "bf16", None),
    ("g1_mha_d64", 4, 4, 64, [3, 16, 33], "bf16", None),
    ("g8_mqa_d128", 8, 1, 128, [1, 2, 700, 1025], "bf16", None),
    ("g2_d128", 16, 8, 128, [15, 16, 17, 513], "bf16", 64),
    ("g8_d128_parts", 64, 8, 128, [64, 65, 511, 512, 513, 2000], "bf16", 64),
    ("g4_d128_parts", 32, 8, 128, [1, 1023, 1024, 1025, 3000], "bf16", 512),
    ("g4_d64_fp8", 8, 2, 64, [1, 17, 100, 700], "fp8", None),
    ("g4_d128_fp8", 32, 8, 128, [16, 300, 1500, 8192], "fp8", None),
    ("g8_d128_fp8", 64, 8, 128, [40, 900], "fp8", 128),
    ("g1_d128_fp8", 8, 8, 128, [5, 77], "fp8", None),
    ("g2_d64_fp8", 4, 2, 64, [1, 31, 250], "fp8", 64),
    ("with_empty", 32, 8, 128, [0, 5, 0, 600, 0], "bf16", 256),
    ("g8_d64_many", 16, 2, 64, list(range(1, 200, 7)), "bf16", 64),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_parity_shapes(case):
    name, nq, nkv, d, lens, dtype, part = case
    w = wl.build(name, nq, nkv, d, lens, dtype=dtype, seed=zlib.crc32(name.encode()) % 1000)
    _parity(w, part)


@pytest.mark.parametrize("name", ["llama3_8b", "long_context_70b", "fp8_lognormal", "shared_prefix"])
def test_parity_full_workloads(name):
    w = wl.NAMED[name]()
    mx, mean = _parity(w)
    print(f"{name}: max abs {mx:.2e} mean abs {mean:.2e}")


def test_single_token_output_is_its_value_exactly():
    w = wl.build("c1", 32, 8, 128, [1, 1, 1], seed=99)
    with make_pool(w) as pool:
        out = run_step(pool, w)
        torch.cuda.synchronize()
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    for b in range(3):
        for h in range(32):
            assert np.array_equal(got[b, h], w.step_v[b, h // 4])


def test_partition_size_does_not_change_the_answer_beyond_rounding():
    w = wl.build("psz", 32, 8, 128, [3000, 100, 4100], seed=5)
    outs = []
    for part in (0, 64, 512, 4096):
        with make_pool(w, part) as pool:
            fill(pool, w)
            outs.append(out_f64(run_step(pool, w)))
    for o in outs[1:]:
        assert np.abs(outs[0] - o).max() < 1e-2


def test_repeat_calls_are_bitwise_deterministic_and_stream_aware():
    w = wl.build("det", 32, 8, 128, [2000, 700, 9], seed=6)
    with make_pool(w) as pool:
        fill(pool, w)
        dev = step_inputs(w)
        a = run_step(pool, w, dev)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            b = pkv.paged_decode_attention(pool, dev["q"], dev["tables"], dev["lens"], float(w.scale), stream=s)
        torch.cuda.synchronize()
        assert torch.equal(a, b)


def test_bad_block_id_is_skipped_and_flagged():
    w = wl.build("bad", 8, 2, 64, [40, 40], seed=12)
    tables = w.block_tables.copy()
    tables[0, 1] = w.num_blocks + 5  # sequence 0's second block points outside the pool
    m = mirror(w)
    ref1 = m.decode(w.q[1:], w.block_tables[1:], w.context_lens[1:], w.scale)
    with make_pool(w) as pool:
        fill(pool, w)
        dev = step_inputs(w)
        pkv.paged_kv_append(pool, dev["k"], dev["v"], dev["slots"])
        out = pkv.paged_decode_attention(pool, dev["q"], i32_dev(tables), dev["lens"], float(w.scale))
        bits = pool.get_error(clear=True)
    assert bits & pkv.DEVERR_BLOCK_RANGE
    assert_close(out_f64(out)[1:], ref1, "healthy sequence")
    assert np.isfinite(out_f64(out)[0]).all()


def test_context_beyond_table_is_clamped_and_flagged():
    w = wl.build("ctx", 8, 2, 64, [32, 20], seed=13)
    lens = w.context_lens.copy()
    lens[0] = 1000  # table holds 2 blocks = 32 tokens
    with make_pool(w) as pool:
        fill(pool, w)
        dev = step_inputs(w)
        pkv.paged_kv_append(pool, dev["k"], dev["v"], dev["slots"])
        out = pkv.paged_decode_attention(pool, dev["q"], dev["tables"], i32_dev(lens), float(w.scale))
        bits = pool.get_error(clear=True)
    assert bits & pkv.DEVERR_CTX_RANGE
    ref = mirror(w).decode(w.q, w.block_tables, w.context_lens, w.scale)
    assert_close(out_f64(out), ref, "clamped")


def test_decode_host_validation_and_batch_zero():
    with pkv.kv_pool_create(8, 16, 2, 64) as pool:
        q = torch.zeros(2, 6, 64, dtype=torch.bfloat16, device="cuda")  # 6 % 2 == 0 but G = 3
        t = torch.zeros(2, 1, dtype=torch.int32, device="cuda")
        c = torch.ones(2, dtype=torch.int32, device="cuda")
        with pytest.raises(pkv.PagedKVError) as e:
            pkv.paged_decode_attention(pool, q, t, c, 0.125)
        assert e.value.status == 5
        q5 = torch.zeros(2, 5, 64, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(pkv.PagedKVError):
            pkv.paged_decode_attention(pool, q5, t, c, 0.125)
        q4 = torch.zeros(0, 4, 64, dtype=torch.bfloat16, device="cuda")
        pkv.paged_decode_attention(pool, q4, t[:0], c[:0], 0.125)
        with pytest.raises(pkv.PagedKVError):
            pkv.paged_decode_attention(pool, torch.zeros(2, 4, 64, dtype=torch.bfloat16, device="cuda"),
                                       t, c, float("nan"))


def test_timing_counts_launches():
    w = wl.build("tm", 32, 8, 128, [3000, 10], seed=14)
    with make_pool(w) as pool:
        fill(pool, w)
        pool.timing_read(reset=True)
        pool.timing_enable(True)
        run_step(pool, w)
        t = pool.timing_read(reset=True)
    # append, decode, and the split-KV merge behind the decode
    assert t["append_launches"] == 1 and t["decode_launches"] == 1 and t["merge_launches"] == 1
    assert t["prefix_launches"] == 0 and t["launches"] == 3
    assert t["timed_decode"] == 1 and t["decode_ms"] > 0 and t["timed_merge"] == 1


def test_workspace_reserve_then_decode():
    w = wl.build("ws", 32, 8, 128, [5000, 17], seed=15)
    with make_pool(w, 64) as pool:
        pool.reserve_workspace(w.batch, w.n_q, w.max_blocks_per_seq)
        fill(pool, w)
        out = run_step(pool, w)
        ref = mirror(w).decode(w.q, w.block_tables, w.context_lens, w.scale)
        assert_close(out_f64(out), ref, "reserved")


def test_bounded_wait_times_out_without_fault_and_context_stays_usable():
    w = wl.build("to", 8, 2, 64, [40, 17], seed=16)
    with make_pool(w) as pool:
        pool.selftest_wait_timeout(2_000_000)  # 2 ms, nothing ever arrives
        bits = pool.get_error(clear=True)
        assert bits == pkv.DEVERR_TIMEOUT
        assert pool.get_error() == 0
        with pytest.raises(pkv.PagedKVError):
            pool.selftest_wait_timeout(10)  # below the 1 us floor
        fill(pool, w)
        out = run_step(pool, w)  # the context still works
        assert_close(out_f64(out), mirror(w).decode(w.q, w.block_tables, w.context_lens, w.scale), "after timeout")

