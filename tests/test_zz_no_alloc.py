"""paged_decode_attention_noalloc: the decode call for callers that cannot
allocate device memory while decoding (an engine that reserved nearly all
free HBM for its KV pool at start-up, or a caller that cannot accept the
device-wide synchronisation cudaMalloc/cudaFree may cause).  It keeps its
scratch in a fixed array inside the library, so this file checks it, on two
calls in a row (the array keeps the previous call's contents), against both
the allocating entry point and the fp64 oracle on the same inputs; that a
pool whose only decode call is this one never grows a workspace and that
free device memory does not move across its calls; and that a call needing
more scratch than the array holds is refused before launch.

Collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test.  It also passes on its own in a
fresh process (it builds its own inputs and pools)."""
import numpy as np
import pytest
import torch

import gqa_decode_attention_paged_gb300 as pkv
import workloads as wl
from gpu_util import assert_close, fill, make_pool, mirror, out_f64, step_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("make", [
    lambda: wl.llama3_8b(),
    lambda: wl.build("na_fp8", 32, 8, 128, [16, 300, 1500, 4000, 0, 9], dtype="fp8", seed=41),
    lambda: wl.build("na_g8", 64, 8, 128, [3000, 7000, 1], seed=42),
])
def test_noalloc_matches_allocating_decode_twice(make):
    w = make()
    ref_oracle = mirror(w).decode(w.q, w.block_tables, w.context_lens, w.scale)
    with make_pool(w) as pool:
        fill(pool, w)
        d = step_inputs(w)
        pkv.paged_kv_append(pool, d["k"], d["v"], d["slots"])
        ref = pkv.paged_decode_attention(pool, d["q"], d["tables"], d["lens"], float(w.scale))
        torch.cuda.synchronize()
        ref = out_f64(ref)
        assert_close(ref, ref_oracle, "allocating decode vs oracle")
        for call in range(2):
            out = torch.full_like(d["q"], float("nan"))
            pkv.paged_decode_attention_noalloc(pool, d["q"], d["tables"], d["lens"], float(w.scale), out)
            torch.cuda.synchronize()
            got = out_f64(out)
            assert_close(got, ref, f"noalloc call {call} vs allocating decode")
            assert_close(got, ref_oracle, f"noalloc call {call} vs oracle")
        assert pool.get_error() == 0


def test_noalloc_first_on_a_fresh_pool_allocates_nothing():
    # A pool whose only decode call is the no-allocation one: its workspace
    # stays empty, and after one warm-up call (the first launch of a kernel
    # may load code) free device memory does not move across further calls.
    w = wl.build("na_fresh", 32, 8, 128, [2000, 33, 4096, 700, 1], seed=43)
    ref_oracle = mirror(w).decode(w.q, w.block_tables, w.context_lens, w.scale)
    with make_pool(w) as pool:
        fill(pool, w)
        d = step_inputs(w)
        pkv.paged_kv_append(pool, d["k"], d["v"], d["slots"])
        outs = [torch.full_like(d["q"], float("nan")) for _ in range(4)]
        pkv.paged_decode_attention_noalloc(pool, d["q"], d["tables"], d["lens"], float(w.scale), outs[0])
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        for out in outs[1:]:
            pkv.paged_decode_attention_noalloc(pool, d["q"], d["tables"], d["lens"], float(w.scale), out)
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        assert free1 == free0, f"free device memory moved by {free0 - free1} bytes across no-allocation calls"
        assert pool.timing_read()["workspace_bytes"] == 0
        for i, out in enumerate(outs):
            assert_close(out_f64(out), ref_oracle, f"noalloc call {i} on a fresh pool vs oracle")
        assert pool.get_error() == 0


def test_noalloc_refuses_calls_beyond_its_scratch():
    # 2048 sequences x 8 heads of 16 blocks each in 64-token slices: far more
    # pieces than 16 MiB of scratch can hold.
    with pkv.kv_pool_create(64, 16, 8, 128) as pool:
        pool.set_partition_tokens(64)
        q = torch.zeros(2048, 64, 128, dtype=torch.bfloat16, device="cuda")
        t = torch.zeros(2048, 16, dtype=torch.int32, device="cuda")
        c = torch.full((2048,), 256, dtype=torch.int32, device="cuda")
        with pytest.raises(pkv.PagedKVError) as e:
            pkv.paged_decode_attention_noalloc(pool, q, t, c, 0.088)
        assert e.value.status == 2 and "scratch" in str(e.value)
        assert pool.timing_read()["workspace_bytes"] == 0
