"""Cascade decode for a shared prefix (read once for the batch) against the
fp64 oracle and against plain paged decode."""
import numpy as np
import pytest
import torch

import gqa_decode_attention_paged_gb300 as pkv
import workloads as wl
from gpu_util import assert_close, fill, i32_dev, make_pool, mirror, out_f64, run_step, step_inputs

pytestmark = pytest.mark.gpu


def _cascade(pool, w, d, n_pre, lens=None, mode=pkv.CASCADE_ALWAYS):
    """paged_decode_attention_prefix; by default with the cascade forced, so
    that its kernels run whatever the prefix length."""
    pool.set_cascade_mode(mode)
    pre = i32_dev(w.block_tables[0, :n_pre])
    return pkv.paged_decode_attention_prefix(pool, d["q"], pre, d["tables"], d["lens"] if lens is None else lens,
                                             float(w.scale))


@pytest.mark.parametrize("make,n_pre", [
    (lambda: wl.shared_prefix(), 64),
    (lambda: wl.build("cp_g8", 64, 8, 128, [321, 400, 257, 1000], seed=61, shared_prefix_tokens=256), 16),
    (lambda: wl.build("cp_d64", 8, 2, 64, [90, 70, 65, 300, 81], seed=62, shared_prefix_tokens=64), 4),
    (lambda: wl.build("cp_ragged", 32, 8, 128, [330, 500, 321], seed=63, shared_prefix_tokens=320), 20),
    (lambda: wl.build("cp_b1", 32, 8, 128, [2000], seed=64, shared_prefix_tokens=1600), 100),
    # FP8 E4M3 pools: both stages read E4M3 bytes with the pool's per-head scales
    (lambda: wl.build("cp_fp8", 32, 8, 128, np.random.default_rng(66).integers(1025, 2050, 48), dtype="fp8",
                      seed=66, shared_prefix_tokens=1024), 64),
    (lambda: wl.build("cp_fp8_g8", 64, 8, 128, [321, 400, 257, 1000], dtype="fp8", seed=67,
                      shared_prefix_tokens=256), 16),
    (lambda: wl.build("cp_fp8_d64", 8, 2, 64, [90, 70, 65, 300, 81], dtype="fp8", seed=68,
                      shared_prefix_tokens=64), 4),
])
def test_cascade_matches_oracle_and_plain_decode(make, n_pre):
    w = make()
    ref = mirror(w).decode(w.q, w.block_tables, w.context_lens, w.scale)
    with make_pool(w) as pool:
        fill(pool, w)
        d = step_inputs(w)
        plain = out_f64(run_step(pool, w, d))  # appends the step token, then decodes
        casc = out_f64(_cascade(pool, w, d, n_pre))
        torch.cuda.synchronize()
        assert pool.get_error() == 0
    assert_close(casc, ref, w.name)
    assert np.abs(casc - plain).max() < 1e-2


def test_cascade_long_prefix_sampled_sequences():
    """The 8192-token shared prefix of the long cascade workload (the prefix
    stage runs many chunks): sampled sequences against the oracle."""
    w = wl.shared_prefix_long()
    n_pre = w.shared_prefix_tokens // 16
    with make_pool(w) as pool:
        fill(pool, w)
        d = step_inputs(w)
        pkv.paged_kv_append(pool, d["k"], d["v"], d["slots"])
        casc = out_f64(_cascade(pool, w, d, n_pre))
        torch.cuda.synchronize()
        assert pool.get_error() == 0
    pick = np.array([0, 1, 37, 64, 100, 127])
    ref = mirror(w).decode(w.q[pick], w.block_tables[pick], w.context_lens[pick], w.scale)
    assert_close(casc[pick], ref, "long shared prefix")


@pytest.mark.parametrize("make,cascade_expected", [
    (lambda: wl.shared_prefix(), False),       # 1024-token prefix, batch 128: plain decode
    (lambda: wl.shared_prefix_long(), True),   # 8192-token prefix, batch 128: the cascade
    (lambda: wl.build("cp_auto_b64", 32, 8, 128, np.random.default_rng(70).integers(1025, 1500, 64), seed=70,
                      shared_prefix_tokens=1024), False),  # 1024 x 64: plain decode
    (lambda: wl.build("cp_auto_b4", 32, 8, 128, [2100, 2500, 2049, 3000], seed=69,
                      shared_prefix_tokens=2048), False),  # long prefix but batch 4: plain decode
    (lambda: wl.build("cp_auto_2k_b64", 32, 8, 128, np.random.default_rng(71).integers(2049, 2600, 64), seed=71,
                      shared_prefix_tokens=2048), True),   # 2048 x 64 = 2^17: the cascade
    (lambda: wl.build("cp_auto_fp8_b128", 32, 8, 128, np.random.default_rng(72).integers(1025, 2050, 128),
                      dtype="fp8", seed=72, shared_prefix_tokens=1024), True),  # FP8, 1024 x 128: the cascade
    (lambda: wl.build("cp_auto_fp8_b32", 32, 8, 128, np.random.default_rng(73).integers(1025, 2050, 32),
                      dtype="fp8", seed=73, shared_prefix_tokens=1024), False),  # FP8, 1024 x 32: plain decode
])
def test_cascade_mode_auto_picks_by_prefix_and_batch(make, cascade_expected):
    w = make()
    n_pre = w.shared_prefix_tokens // 16
    pick = np.arange(0, w.batch, max(1, w.batch // 6))
    ref = mirror(w).decode(w.q[pick], w.block_tables[pick], w.context_lens[pick], w.scale)
    with make_pool(w) as pool:
        fill(pool, w)
        d = step_inputs(w)
        pkv.paged_kv_append(pool, d["k"], d["v"], d["slots"])
        pool.timing_read(reset=True)
        auto = out_f64(_cascade(pool, w, d, n_pre, mode=pkv.CASCADE_AUTO))
        torch.cuda.synchronize()
        ran_prefix_stage = pool.timing_read(reset=True)["prefix_launches"] > 0
        never = out_f64(_cascade(pool, w, d, n_pre, mode=pkv.CASCADE_NEVER))
        torch.cuda.synchronize()
        assert pool.timing_read(reset=True)["prefix_launches"] == 0
        assert pool.get_error() == 0
    assert ran_prefix_stage == cascade_expected
    assert_close(auto[pick], ref, f"{w.name} auto")
    assert_close(never[pick], ref, f"{w.name} never")


def test_cascade_with_prefix_only_sequences():
    w = wl.build("cp_empty", 32, 8, 128, [257, 300, 257], seed=65, shared_prefix_tokens=256)
    lens = w.context_lens.copy()
    lens[0] = lens[2] = 256  # nothing after the prefix
    ref = mirror(w).decode(w.q, w.block_tables, lens, w.scale)
    with make_pool(w) as pool:
        fill(pool, w)
        d = step_inputs(w)
        pkv.paged_kv_append(pool, d["k"], d["v"], d["slots"])
        casc = out_f64(_cascade(pool, w, d, 16, i32_dev(lens)))
        assert pool.get_error() == 0
    assert_close(casc, ref, "prefix-only rows")


def test_cascade_rejects_int4_and_bad_prefix():
    with pkv.kv_pool_create(8, 16, 2, 64, pkv.INT4) as pool:
        pool.set_int4_key_params(np.ones((2, 64)), np.zeros((2, 64)))
        q = torch.zeros(1, 4, 64, dtype=torch.bfloat16, device="cuda")
        t = torch.zeros(1, 2, dtype=torch.int32, device="cuda")
        c = torch.full((1,), 20, dtype=torch.int32, device="cuda")
        with pytest.raises(pkv.PagedKVError) as e:
            pkv.paged_decode_attention_prefix(pool, q, t[0, :1], t, c, 0.125)
        assert e.value.status == 5
    with pkv.kv_pool_create(8, 16, 2, 64) as pool:
        with pytest.raises(pkv.PagedKVError):
            pkv.paged_decode_attention_prefix(pool, q, torch.zeros(3, dtype=torch.int32, device="cuda"), t, c, 0.125)
        with pytest.raises(pkv.PagedKVError) as e:
            pool.set_cascade_mode(3)
        assert e.value.status == 1
