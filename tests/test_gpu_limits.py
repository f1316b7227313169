"""Decode at the documented limits, against the fp64 oracle: the largest
batch a call takes (8192 sequences; one more is refused before any launch),
one very long sequence whose blocks every warp of the grid shares (so each
(sequence, KV head) run is split into hundreds of pieces for the merge), and
the largest number of KV heads a pool holds (256)."""
import numpy as np
import pytest
import torch

import gqa_decode_attention_paged_gb300 as pkv
import workloads as wl
from gpu_util import assert_close, fill, make_pool, mirror, out_f64, run_step, step_inputs

pytestmark = pytest.mark.gpu


def _decode_vs_oracle(w, what):
    ref = mirror(w).decode(w.q, w.block_tables, w.context_lens, w.scale)
    with make_pool(w) as pool:
        fill(pool, w)
        out = run_step(pool, w)
        torch.cuda.synchronize()
        assert pool.get_error() == 0, what
        got = out_f64(out)
    assert_close(got, ref, what)
    return got


def test_largest_batch():
    # 3 to 10 blocks per sequence, some sequences empty.  (Sequences of a few tokens would make
    # outputs of magnitude 2 to 5, where the bf16 output's own rounding reaches 0.8e-2 to 1.6e-2
    # against the fp64 oracle; the 1e-2 bound is meant for outputs below that.)
    rng = np.random.default_rng(801)
    lens = np.where(rng.random(8192) < 0.02, 0, rng.integers(48, 161, 8192))
    w = wl.build("max_batch", 8, 2, 128, lens, seed=801)
    got = _decode_vs_oracle(w, "8192 sequences")
    assert not np.any(got[w.context_lens == 0])


def test_batch_beyond_the_limit_is_refused_before_launch():
    with pkv.kv_pool_create(64, 16, 2, 64) as pool:
        q = torch.zeros(8193, 8, 64, dtype=torch.bfloat16, device="cuda")
        t = torch.zeros(8193, 1, dtype=torch.int32, device="cuda")
        c = torch.ones(8193, dtype=torch.int32, device="cuda")
        with pytest.raises(pkv.PagedKVError) as e:
            pkv.paged_decode_attention(pool, q, t, c, 0.125)
        assert e.value.status == 5  # PKV_EUNSUPPORTED
        assert pool.get_error() == 0


def test_one_long_sequence_split_over_the_whole_grid():
    # 131,072 tokens: 8192 blocks per KV head, about 36 per warp of the grid
    w = wl.build("long_one", 64, 8, 128, [131072], seed=802, slack=1.0)
    _decode_vs_oracle(w, "one 131072-token sequence")


def test_largest_kv_head_count():
    w = wl.build("n_kv_256", 256, 256, 64, [1, 100, 333], seed=803)
    _decode_vs_oracle(w, "256 KV heads")
    with pytest.raises(pkv.PagedKVError):
        pkv.kv_pool_create(16, 16, 257, 64)
