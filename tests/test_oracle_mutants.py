"""Mutation check of the oracle's pins (no GPU).

Each mutant below plants one plausible mistake in a copy of the C oracle (a
dropped term, a wrong sign, index or bound, a transposed layout, a wrong
rounding rule), compiles it with gcc and runs every pin of
``test_oracle.py`` against it in a child process.  At least one pin must fail
for every mutant (or the child must crash); the unmutated copy must pass them
all.  The child process keeps a mutant that reads or writes out of bounds away
from the test process.
"""
import concurrent.futures as cf
import inspect
import json
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "pagedkv_oracle.c")

# (name, text in the oracle, replacement); the text occurs exactly once
MUTANTS = [
    ("sizing drops the factor 2 for K and V",
     "return 2.0 * (double)layers", "return 1.0 * (double)layers"),
    ("slot ignores the block table",
     "return phys * block_size + offset;", "return (logical_block % num_blocks) * block_size + offset;"),
    ("slot accepts the id one past the pool",
     "if (phys < 0 || phys >= num_blocks) return -1;", "if (phys < 0 || phys > num_blocks) return -1;"),
    ("E4M3 exponent bias 8",
     "mag = ldexp(1.0 + (double)m / 8.0, e - 7);", "mag = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("E4M3 subnormal scale 2^-7",
     "mag = ldexp((double)m / 8.0, -6);", "mag = ldexp((double)m / 8.0, -7);"),
    ("E4M3 has no NaN code",
     "if (e == 0xF && m == 0x7) return NAN;", ""),
    ("E4M3 ties go to the larger code",
     "if (dist < best_dist || (dist == best_dist && (c & 1) == 0 && (best & 1) == 1)) {",
     "if (dist <= best_dist) {"),
    ("E4M3 encoder without saturation",
     "if (fabs((double)y) >= 448.0) return (uint8_t)((want_sign << 7) | 0x7E);", ""),
    ("quantiser multiplies by the scale",
     "volatile float y = x / scale;", "volatile float y = x * scale;"),
    ("append: head and token axes transposed",
     "int64_t dst = ((blk * n_kv + g) * block_size + off) * (int64_t)d_head;",
     "int64_t dst = ((blk * block_size + off) * n_kv + g) * (int64_t)d_head;"),
    ("append accepts the slot one past the pool",
     "if (slot >= num_blocks * (int64_t)block_size) {", "if (slot > num_blocks * (int64_t)block_size) {"),
    ("4-bit code rounds half away from zero",
     "float r = rintf(u);", "float r = roundf(u);"),
    ("4-bit value step over 16 levels",
     "volatile float s = range / 15.0f;", "volatile float s = range / 16.0f;"),
    ("4-bit value range drops the minimum",
     "volatile float range = mx - mn;", "volatile float range = mx;"),
    ("4-bit nibbles written high-first",
     "if (c & 1) *b = (uint8_t)((*b & 0x0F) | (code << 4));",
     "if (!(c & 1)) *b = (uint8_t)((*b & 0x0F) | (code << 4));"),
    ("4-bit nibbles read high-first",
     "return (c & 1) ? (uint8_t)(b >> 4) : (uint8_t)(b & 0x0F);",
     "return (c & 1) ? (uint8_t)(b & 0x0F) : (uint8_t)(b >> 4);"),
    # (dropping the key zero point is no mistake: it adds q . z to every score of a query, which the
    # softmax cancels)
    ("4-bit decode takes head 0's key scales for every head",
     "Kc[p * D + d] = orc_get_nibble(krow, d) * (double)job->k_scale[g * D + d] + job->k_zero[g * D + d];",
     "Kc[p * D + d] = orc_get_nibble(krow, d) * (double)job->k_scale[d] + job->k_zero[g * D + d];"),
    ("4-bit decode drops the value zero point",
     "Vc[p * D + d] = orc_get_nibble(vrow, d) * vsc + vz;", "Vc[p * D + d] = orc_get_nibble(vrow, d) * vsc;"),
    ("FP8 values dequantised with the key scale",
     "double vs = job->dtype == ORC_E4M3 ? (double)job->v_scale[g] : 1.0;",
     "double vs = job->dtype == ORC_E4M3 ? (double)job->k_scale[g] : 1.0;"),
    ("decode: head and token axes transposed",
     "int64_t base = ((blk * job->n_kv + g) * BS + off) * (int64_t)D;",
     "int64_t base = ((blk * BS + off) * job->n_kv + g) * (int64_t)D;"),
    ("decode reads sequence 0's table for every sequence",
     "const int32_t *row = job->block_tables + (int64_t)b * job->max_blocks_per_seq;",
     "const int32_t *row = job->block_tables;"),
    ("query heads interleaved over KV heads",
     "int h = g * group + hh;", "int h = hh * job->n_kv + g;"),
    ("new token does not attend to itself",
     "int64_t n_keys = C - (r1 - r) + 1;", "int64_t n_keys = C - (r1 - r);"),
    ("prefill without the causal mask",
     "int64_t n_keys = C - (r1 - r) + 1;", "int64_t n_keys = C;"),
    ("scores scored against V",
     "dot += orc_bf16_to_double(qh[d]) * Kc[p * D + d];", "dot += orc_bf16_to_double(qh[d]) * Vc[p * D + d];"),
    ("score scale dropped",
     "s[p] = job->scale * dot;", "s[p] = dot;"),
    ("softmax in base 2",
     "double w = exp(s[p] - m);", "double w = exp2(s[p] - m);"),
    ("softmax not normalised",
     "for (int d = 0; d < D; ++d) o[d] /= denom;", "(void)denom;"),
]


def _run_pins(src: str, lib: str) -> None:
    """Child process: point the oracle at ``lib`` and print the failing pins."""
    sys.path[:0] = [ROOT, HERE]
    import oracle
    oracle._SRC, oracle._LIB, oracle._lib = src, lib, None
    import test_oracle as t
    failed = []
    for name, fn in inspect.getmembers(t, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        cases = [()]
        for mark in getattr(fn, "pytestmark", []):
            if mark.name == "parametrize":
                cases = [tuple(v) if isinstance(v, (tuple, list)) else (v,) for v in mark.args[1]]
        for c in cases:
            try:
                fn(*c)
            except pytest.skip.Exception:
                pass
            except (Exception, pytest.fail.Exception):  # pytest.raises signals "did not raise" with the latter
                failed.append(name)
    print(json.dumps(sorted(set(failed))))


def _check(tmp: str, idx: int, old: str, new: str):
    with open(SRC) as f:
        text = f.read()
    if old is not None:
        assert text.count(old) == 1, f"mutant {idx}: the text must occur once in the oracle"
        text = text.replace(old, new)
    d = os.path.join(tmp, f"m{idx}")
    os.makedirs(d)
    src, lib = os.path.join(d, "oracle.c"), os.path.join(d, "liboracle.so")
    with open(src, "w") as f:
        f.write(text)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", src, "-o", lib, "-lm", "-lpthread"])
    p = subprocess.run([sys.executable, os.path.abspath(__file__), src, lib], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    if p.returncode != 0:
        return None, p.stderr[-2000:]  # the mutant crashed the child
    return json.loads(p.stdout.strip().splitlines()[-1]), ""


def test_every_planted_mistake_fails_a_pin(tmp_path):
    jobs = [(-1, None, None)] + [(i, old, new) for i, (_, old, new) in enumerate(MUTANTS)]
    with cf.ThreadPoolExecutor(max_workers=max(2, min(8, os.cpu_count() or 2))) as ex:
        res = dict(zip([j[0] for j in jobs], ex.map(lambda j: _check(str(tmp_path), *j), jobs)))
    control, err = res.pop(-1)
    assert control == [], f"the unmutated oracle fails pins {control} {err}"
    # a mutant that writes past a pool (the append bound) may crash the child instead of failing an
    # assertion: that also turns the pins red, so it counts as caught
    survivors = [MUTANTS[i][0] for i, (failed, err) in res.items() if failed == []]
    assert not survivors, f"mutants that pass every pin: {survivors}"


# The oracle's block model (Python): (name, text in oracle/blocks.py, replacement)
BLOCK_MUTANTS = [
    ("copy leaves a 4-bit block's value parameters behind",
     "mirror.v_params[d] = mirror.v_params[s]", "pass"),
    ("copy runs from destination to source",
     "mirror.k[d] = mirror.k[s]", "mirror.k[s] = mirror.k[d]"),
    ("swap entry holds V before K",
     "[mirror.k, mirror.v]", "[mirror.v, mirror.k]"),
    ("swap-in reads every array from the entry's start",
     "off += arr[0].nbytes", "pass"),
    ("swap-in entries without the parameter part",
     "off = n * entry", "off = n * 2 * mirror.k[0].nbytes"),
    ("free blocks handed out highest id first",
     "for i, r in enumerate(self.ref):", "for i, r in reversed(list(enumerate(self.ref))):"),
    ("copy-on-write also copies private blocks",
     "if self.ref[i] > 1:", "if self.ref[i] >= 1:"),
    ("release lets a block go more often than it is referenced",
     "self._check_held(ids, count_repeats=True)", "self._check_held(ids, count_repeats=False)"),
    ("copy-on-write starts without enough free blocks",
     "if self.free_blocks() < need:", "if self.free_blocks() < need - 1:"),
    ("share adds two references",
     "self.ref[i] += 1", "self.ref[i] += 2"),
]


def test_every_planted_mistake_in_the_block_model_fails_a_pin(monkeypatch):
    import types

    sys.path[:0] = [HERE]
    import test_blocks as tb
    with open(os.path.join(ROOT, "oracle", "blocks.py")) as f:
        text = f.read()
    pins = [lambda bm: tb._pin_block_ops(bm)] + [
        (lambda fn: lambda bm: (monkeypatch.setattr(tb, "AllocatorModel", bm.AllocatorModel), fn()))(fn)
        for name, fn in inspect.getmembers(tb, inspect.isfunction) if name.startswith("test_model_")]
    survivors = []
    for name, old, new in [("control", None, None)] + BLOCK_MUTANTS:
        src = text
        if old is not None:
            assert src.count(old) == 1, f"{name}: the text must occur once in the block model"
            src = src.replace(old, new)
        bm = types.ModuleType("mutant_blocks")
        exec(compile(src, f"<{name}>", "exec"), bm.__dict__)
        failed = 0
        for pin in pins:
            try:
                pin(bm)
            except (Exception, pytest.fail.Exception):
                failed += 1
        monkeypatch.undo()
        if old is None:
            assert failed == 0, "the unmutated block model fails its pins"
        elif failed == 0:
            survivors.append(name)
    assert not survivors, f"mutants of the block model that pass every pin: {survivors}"


if __name__ == "__main__":
    _run_pins(sys.argv[1], sys.argv[2])
