"""The fused step (append + decode in one launch) against the two separate
calls and the oracle: pool bytes and outputs are bit-identical to
paged_kv_append followed by paged_decode_attention."""
import numpy as np
import pytest
import torch

import gqa_decode_attention_paged_gb300 as pkv
import workloads as wl
from gpu_util import (assert_close, fill, make_pool, mirror, mirror_bytes, out_f64, pool_bytes, run_step,
                      step_inputs)

pytestmark = pytest.mark.gpu

CASES = [
    lambda: wl.tiny(),
    lambda: wl.llama3_8b(),
    lambda: wl.fp8_lognormal(),
    lambda: wl.shared_prefix(),
    lambda: wl.build("st_g8", 64, 8, 128, [1, 16, 17, 5000, 0, 33], seed=51),
    lambda: wl.build("st_fp8_d64", 8, 2, 64, [1, 31, 250, 16], dtype="fp8", seed=52),
    lambda: wl.build("st_g1", 8, 8, 128, [40, 7], seed=53),
]


def _step_inputs_by_sequence(w):
    d = step_inputs(w)
    # the fused call takes each sequence's new token by sequence, [B][n_kv][d]
    return d


@pytest.mark.parametrize("make", CASES)
def test_fused_step_equals_append_then_decode(make):
    w = make()
    with make_pool(w) as p1, make_pool(w) as p2:
        fill(p1, w)
        fill(p2, w)
        d = step_inputs(w)
        a = run_step(p1, w, d)  # separate append + decode
        b = pkv.paged_decode_step(p2, d["q"], d["k"], d["v"], d["tables"], d["lens"], float(w.scale))
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        k1, v1 = pool_bytes(p1)
        k2, v2 = pool_bytes(p2)
        assert np.array_equal(k1, k2) and np.array_equal(v1, v2)
        mk, mv = mirror_bytes(mirror(w))
        assert np.array_equal(k2, mk) and np.array_equal(v2, mv)
        assert p2.get_error() == 0


@pytest.mark.parametrize("make", [CASES[1], CASES[2]])
def test_fused_step_against_oracle(make):
    w = make()
    ref = mirror(w).decode(w.q, w.block_tables, w.context_lens, w.scale)
    with make_pool(w) as p:
        fill(p, w)
        d = step_inputs(w)
        out = pkv.paged_decode_step(p, d["q"], d["k"], d["v"], d["tables"], d["lens"], float(w.scale))
        assert_close(out_f64(out), ref, w.name)


def _pinned_offset(t):
    """A copy of t in pinned memory that starts one element past the
    allocation's start (2 bytes for bf16: not 16-byte aligned)."""
    buf = torch.empty(t.numel() + 1, dtype=t.dtype).pin_memory()
    v = buf[1:].view(t.shape)
    v.copy_(t)
    return v


@pytest.mark.parametrize("mode", ["pinned", "pinned_offset", "pageable"])
def test_host_step_equals_device_step(mode):
    """Aligned pinned buffers are read in place by the step's kernels and the
    output written directly; pinned buffers off the 16-byte grid go through
    the gather kernel and a staged output copy; pageable ones one copy per
    array.  All equal the device-pointer step bit for bit."""
    _host_vs_device_step(wl.llama3_8b(), mode)


@pytest.mark.parametrize("make,mode", [
    (lambda: wl.build("hs_fp8", 32, 8, 128, [300, 1, 77, 1000], dtype="fp8", seed=61), "pinned"),
    (lambda: wl.build("hs_int4", 32, 8, 128, [300, 1, 77, 1000], dtype="int4", seed=62), "pinned"),
    (lambda: wl.build("hs_int4_d64", 8, 2, 64, [90, 17, 0, 257], dtype="int4", seed=63), "pinned_offset"),
])
def test_host_step_other_kv_types(make, mode):
    """The host-buffer step on FP8 and 4-bit pools (their own append and
    decode kernels behind the same gather, graph and in-place reads) equals
    the device-pointer step bit for bit."""
    _host_vs_device_step(make(), mode)


def _host_vs_device_step(w, mode):
    with make_pool(w) as p1, make_pool(w) as p2:
        fill(p1, w)
        fill(p2, w)
        d = step_inputs(w)
        a = pkv.paged_decode_step(p1, d["q"], d["k"], d["v"], d["tables"], d["lens"], float(w.scale))
        pin = {"pinned": lambda t: t.pin_memory(), "pinned_offset": _pinned_offset, "pageable": lambda t: t}[mode]
        h = {k: pin(v.cpu()) for k, v in d.items()}
        out = pin(torch.empty(tuple(d["q"].shape), dtype=torch.bfloat16))
        for _ in range(2):  # the staging area is reused on the second call (pinned: a graph replay)
            out.zero_()
            pkv.paged_decode_step_host(p2, h["q"], h["k"], h["v"], h["tables"], h["lens"], float(w.scale), out)
            assert torch.equal(a.cpu().view(torch.int16), out.view(torch.int16))
        # new queries in the same host buffer: the replay reads them
        q2 = torch.flip(d["q"], dims=[0]).contiguous()
        b = pkv.paged_decode_step(p1, q2, d["k"], d["v"], d["tables"], d["lens"], float(w.scale))
        h["q"].copy_(q2.cpu())
        out.zero_()
        pkv.paged_decode_step_host(p2, h["q"], h["k"], h["v"], h["tables"], h["lens"], float(w.scale), out)
        assert torch.equal(b.cpu().view(torch.int16), out.view(torch.int16))
        assert p2.get_error() == 0


def test_host_step_object_equals_call():
    w = wl.llama3_8b()
    with make_pool(w) as p1, make_pool(w) as p2:
        fill(p1, w)
        fill(p2, w)
        d = step_inputs(w)
        h = {k: v.cpu().pin_memory() for k, v in d.items()}
        out1 = torch.empty(tuple(d["q"].shape), dtype=torch.bfloat16).pin_memory()
        out2 = torch.empty_like(out1).pin_memory()
        pkv.paged_decode_step_host(p1, h["q"], h["k"], h["v"], h["tables"], h["lens"], float(w.scale), out1)
        step = pkv.HostStep(p2, h["q"], h["k"], h["v"], h["tables"], h["lens"], float(w.scale), out2)
        for _ in range(3):
            assert step() is out2
            assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
        assert p2.get_error() == 0
