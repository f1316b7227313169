"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself: numbers the pages
print, closed forms, textbook special cases computed by an independent
library routine (torch's fp64 CPU attention), the pages' own statement of the
decode step restated in fp64 torch on a contiguous cache, invariants the
pages state, and brute force on tiny inputs.  Each test names what pins it.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Sizing formula: the pages' printed figures
# ---------------------------------------------------------------------------

def test_kv_bytes_per_token_printed_figures():
    g = _golden("kv_bytes_per_token.json")
    for case in g["cases"]:
        L, nkv, d, b = case["args"]
        got = oracle.kv_bytes_per_token(L, nkv, d, b) * case["times"]
        assert got == case["bytes"], case["cite"]
    for case in g["approx"]:
        L, nkv, d, b = case["args"]
        got = oracle.kv_bytes_per_token(L, nkv, d, b) * case["times"] / 1e9
        assert abs(got - case["printed_gb"]) <= case["rel_tol"] * case["printed_gb"], case["cite"]


def test_kv_bytes_gqa_saving_factor():
    # "GQA saves 8x" (Problem 3) and "a 4x reduction ... relative to full MHA"
    # (Memory Management, MHA/MQA/GQA comparison).
    assert oracle.kv_bytes_per_token(80, 64, 128, 2) / oracle.kv_bytes_per_token(80, 8, 128, 2) == 8
    assert oracle.kv_bytes_per_token(32, 32, 128, 2) / oracle.kv_bytes_per_token(32, 8, 128, 2) == 4


# ---------------------------------------------------------------------------
# Address arithmetic: the printed page walk
# ---------------------------------------------------------------------------

def test_page_walk_printed_example():
    g = _golden("page_walk.json")
    indptr, indices = g["kv_indptr"], g["kv_indices"]
    B = g["page_tokens"]
    # Request 2's pages, and every token of it, in the padded block-table form.
    row2 = np.array(indices[indptr[2]:indptr[3]], dtype=np.int32)
    assert row2.tolist() == g["request_2_pages"]
    for lo, hi, page in g["request_2_token_ranges"]:
        for p in range(lo, hi + 1):
            assert oracle.slot_of(row2, p, B, 32) == page * B + (p - lo)
    # Every request: the slot of logical position p names the page that owns p.
    for r in range(len(indptr) - 1):
        row = np.array(indices[indptr[r]:indptr[r + 1]], dtype=np.int32)
        for p in range(len(row) * B):
            assert oracle.slot_of(row, p, B, 32) // B == row[p // B]
            assert oracle.slot_of(row, p, B, 32) % B == p % B


def test_slot_of_rejects_out_of_pool_ids():
    row = np.array([3, 99, -1, 64, 63], dtype=np.int32)
    assert oracle.slot_of(row, 5, 16, 64) == 3 * 16 + 5
    assert oracle.slot_of(row, 16, 16, 64) == -1
    assert oracle.slot_of(row, 40, 16, 64) == -1
    assert oracle.slot_of(row, 48, 16, 64) == -1  # the id one past the pool
    assert oracle.slot_of(row, 79, 16, 64) == 63 * 16 + 15  # the pool's last slot


def test_waste_bound_of_generated_tables():
    # "waste per sequence <= B - 1 tokens (only the last block is partly empty)"
    w = wl.build("waste", 4, 2, 64, [1, 15, 16, 17, 31, 32, 33, 100], seed=7)
    for b, C in enumerate(w.context_lens):
        used = int((w.block_tables[b] >= 0).sum())
        assert used == math.ceil(C / 16)
        assert 0 <= used * 16 - C <= 15


def test_workload_slots_match_oracle_address_function():
    w = wl.build("slots", 4, 2, 64, [3, 20, 47, 64], seed=11)
    pos = {}
    k = 0
    for b, C in enumerate(w.context_lens):
        for p in range(C - 1):
            assert w.fill_slots[k] == oracle.slot_of(w.block_tables[b], p, 16, w.num_blocks)
            k += 1
        assert w.step_slots[b] == oracle.slot_of(w.block_tables[b], C - 1, 16, w.num_blocks)
    assert k == w.fill_slots.shape[0]
    # No two sequences own the same physical block.
    used = w.block_tables[w.block_tables >= 0]
    assert len(np.unique(used)) == len(used)


# ---------------------------------------------------------------------------
# E4M3 codec
# ---------------------------------------------------------------------------

def test_e4m3_decode_all_codes_vs_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got) and (c & 0x7F) == 0x7F
        else:
            assert got == ref[c], hex(c)


def test_e4m3_landmarks():
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6
    assert oracle.e4m3_decode(0x38) == 1.0
    assert oracle.e4m3_encode(1e6) == 0x7E
    assert oracle.e4m3_encode(-1e6) == 0xFE
    assert oracle.e4m3_encode(449.0) == 0x7E
    assert oracle.e4m3_encode(float("inf")) == 0x7E
    assert oracle.e4m3_encode(float("-inf")) == 0xFE
    assert oracle.e4m3_encode(float("nan")) == 0x7F
    assert oracle.e4m3_encode(-1e-30) == 0x80
    for big in (1.16e18, 3.0e38, 2.0 ** 100, 464.0, 500.0):
        assert oracle.e4m3_encode(big) == 0x7E and oracle.e4m3_encode(-big) == 0xFE
    assert oracle.e4m3_encode(0.0) == 0x00
    assert oracle.e4m3_encode(-0.0) == 0x80


def test_e4m3_round_trip_and_ties_to_even():
    finite = [c for c in range(256) if (c & 0x7F) != 0x7F]
    for c in finite:
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c
    # Midpoints between neighbouring positive codes go to the even code.
    for c in range(0, 0x7E):
        lo, hi = oracle.e4m3_decode(c), oracle.e4m3_decode(c + 1)
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2  # exact in fp32
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(float(mid)) == want
        assert oracle.e4m3_encode(-float(mid)) == want | 0x80


def test_e4m3_encode_vs_torch_cast_in_range():
    rng = np.random.default_rng(123)
    x = np.concatenate([
        rng.uniform(-448, 448, 4000),
        rng.standard_normal(4000) * 3,
        rng.standard_normal(2000) * 1e-2,
    ]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_quantise_uses_fp32_division():
    # x / scale is an IEEE single division before encoding.
    bits = wl.f32_to_bf16_bits(np.array([1.5, -3.25, 100.0], dtype=np.float32))
    for b, x in zip(bits, [1.5, -3.25, 100.0]):
        s = np.float32(0.37)
        y = np.float32(np.float32(x) / s)
        assert oracle.quantise_e4m3(int(b), float(s)) == oracle.e4m3_encode(float(y))


# ---------------------------------------------------------------------------
# Append
# ---------------------------------------------------------------------------

def test_append_places_rows_by_documented_layout():
    w = wl.build("app", 4, 2, 64, [5, 33], seed=3)
    m = oracle.PoolMirror(w.num_blocks, 16, 2, 64)
    assert m.append(w.fill_k, w.fill_v, w.fill_slots) == 0
    for t, slot in enumerate(w.fill_slots):
        blk, off = divmod(int(slot), 16)
        assert np.array_equal(m.k[blk, :, off, :], w.fill_k[t])
        assert np.array_equal(m.v[blk, :, off, :], w.fill_v[t])
    # untouched slots stay zero
    mask = np.zeros((w.num_blocks, 16), dtype=bool)
    for slot in w.fill_slots:
        mask[slot // 16, slot % 16] = True
    assert not m.k.transpose(0, 2, 1, 3)[~mask].any()


def test_append_skips_padding_and_counts_out_of_range():
    m = oracle.PoolMirror(2, 16, 1, 64)
    kb = wl.normal_bf16_bits((3, 1, 64), (1, 1))
    assert m.append(kb, kb, np.array([-1, 31, 32], dtype=np.int64)) == 1
    assert np.array_equal(m.k[1, 0, 15], kb[1, 0]) and not m.k[0].any()


def test_append_fp8_matches_elementwise_quantiser():
    w = wl.build("app8", 4, 2, 64, [9, 20], seed=5, dtype="fp8")
    m = oracle.PoolMirror(w.num_blocks, 16, 2, 64, oracle.E4M3, w.k_scale, w.v_scale)
    m.append(w.fill_k, w.fill_v, w.fill_slots)
    for t in [0, 7, len(w.fill_slots) - 1]:
        blk, off = divmod(int(w.fill_slots[t]), 16)
        for g in range(2):
            for d in [0, 13, 63]:
                assert m.k[blk, g, off, d] == oracle.quantise_e4m3(int(w.fill_k[t, g, d]), w.k_scale[g])
                assert m.v[blk, g, off, d] == oracle.quantise_e4m3(int(w.fill_v[t, g, d]), w.v_scale[g])


def test_append_fp8_memoised_path_equals_direct_path():
    # Large appends use a per-head table of the quantiser; small ones call it
    # per element.  Both must give the same bytes.
    T = 4200
    kb = wl.normal_bf16_bits((T, 2, 64), (9, 1))
    vb = wl.normal_bf16_bits((T, 2, 64), (9, 2))
    slots = np.arange(T, dtype=np.int64)
    ks = np.array([0.011, 0.013], dtype=np.float32)
    vs = np.array([0.012, 0.0105], dtype=np.float32)
    big = oracle.PoolMirror(T // 16 + 1, 16, 2, 64, oracle.E4M3, ks, vs)
    big.append(kb, vb, slots)
    small = oracle.PoolMirror(T // 16 + 1, 16, 2, 64, oracle.E4M3, ks, vs)
    for s in range(0, T, 100):
        small.append(kb[s:s + 100], vb[s:s + 100], slots[s:s + 100])
    assert np.array_equal(big.k, small.k) and np.array_equal(big.v, small.v)


# ---------------------------------------------------------------------------
# Decode attention
# ---------------------------------------------------------------------------

def _f64(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


def _mirror_for(w):
    dt = oracle.BF16 if w.dtype == "bf16" else oracle.E4M3
    m = oracle.PoolMirror(w.num_blocks, w.block_size, w.n_kv, w.d_head, dt, w.k_scale, w.v_scale)
    m.append(w.fill_k, w.fill_v, w.fill_slots)
    m.append(w.step_k, w.step_v, w.step_slots)
    return m


def _contiguous_kv(w, b):
    """Sequence b's K and V in position order, fp64, built from the workload's
    own source arrays (not from any pool)."""
    C = int(w.context_lens[b])
    pos_of_slot = {}
    k = np.zeros((C, w.n_kv, w.d_head))
    v = np.zeros((C, w.n_kv, w.d_head))
    slots = [oracle.slot_of(w.block_tables[b], p, 16, w.num_blocks) for p in range(C)]
    for t, s in enumerate(w.fill_slots):
        pos_of_slot[int(s)] = ("fill", t)
    pos_of_slot[int(w.step_slots[b])] = ("step", b)
    for p, s in enumerate(slots):
        kind, t = pos_of_slot[s]
        src_k = w.fill_k if kind == "fill" else w.step_k
        src_v = w.fill_v if kind == "fill" else w.step_v
        k[p], v[p] = _f64(src_k[t]), _f64(src_v[t])
    return k, v


def _pages_decode_step(q, k_cache, v_cache):
    """The pages' decode step ("The KV Cache from First Principles",
    "Implementation"), restated in fp64 torch: expand each KV head to its
    group of query heads with repeat_interleave, score the single query
    against every cached key divided by sqrt(d), softmax over positions,
    weight the values.  q: (n_q, d); k_cache, v_cache: (T, n_kv, d)."""
    qt = torch.from_numpy(q)[None, :, None, :]  # (1, n_q, 1, d)
    kt = torch.from_numpy(k_cache).permute(1, 0, 2)[None]  # (1, n_kv, T, d)
    vt = torch.from_numpy(v_cache).permute(1, 0, 2)[None]
    groups = qt.shape[1] // kt.shape[1]
    kt = kt.repeat_interleave(groups, dim=1)
    vt = vt.repeat_interleave(groups, dim=1)
    scores = (qt @ kt.transpose(-2, -1)) / (qt.shape[-1] ** 0.5)
    return (torch.softmax(scores, dim=-1) @ vt)[0, :, 0, :].numpy()


def test_check_a_paged_equals_contiguous_pages_decode_step():
    # d_head = 64 so that fp32(1/sqrt(64)) = 0.125 exactly and the two sides
    # use the same scale.
    w = wl.build("a", 8, 2, 64, [1, 17, 100, 256], seed=21)
    out = _mirror_for(w).decode(w.q, w.block_tables, w.context_lens, w.scale)
    for b in range(w.batch):
        k, v = _contiguous_kv(w, b)
        ref = _pages_decode_step(_f64(w.q[b]), k, v)
        np.testing.assert_allclose(out[b], ref, rtol=0, atol=1e-13)


def test_check_b_invariant_under_block_id_permutation():
    w = wl.build("b", 8, 2, 64, [40, 77, 160], seed=22, slack=2.0)
    m = _mirror_for(w)
    out = m.decode(w.q, w.block_tables, w.context_lens, w.scale)
    perm = np.random.default_rng(5).permutation(w.num_blocks)
    m2 = oracle.PoolMirror(w.num_blocks, 16, w.n_kv, w.d_head)
    m2.k[perm] = m.k
    m2.v[perm] = m.v
    tables = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    out2 = m2.decode(w.q, tables, w.context_lens, w.scale)
    assert np.array_equal(out, out2)


def _sdpa_per_head(q, k, v, scale):
    """Library attention (torch fp64 CPU) for one query row per head.
    q: (n_q, d); k, v: (n_q, T, d)."""
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[:, None, :], torch.from_numpy(k), torch.from_numpy(v), scale=scale
    )[:, 0, :].numpy()


@pytest.mark.parametrize("n_q,n_kv", [(4, 4), (8, 1)])
def test_check_c_mha_and_mqa_endpoints(n_q, n_kv):
    w = wl.build("c", n_q, n_kv, 64, [23, 70], seed=23)
    out = _mirror_for(w).decode(w.q, w.block_tables, w.context_lens, w.scale)
    for b in range(w.batch):
        k, v = _contiguous_kv(w, b)  # (T, n_kv, d)
        if n_kv == n_q:  # MHA: head h reads its own KV head
            kh, vh = k.transpose(1, 0, 2), v.transpose(1, 0, 2)
        else:  # MQA: every head reads KV head 0
            kh = np.broadcast_to(k[:, 0, :], (n_q,) + k[:, 0, :].shape).copy()
            vh = np.broadcast_to(v[:, 0, :], (n_q,) + v[:, 0, :].shape).copy()
        ref = _sdpa_per_head(_f64(w.q[b]), kh, vh, float(w.scale))
        np.testing.assert_allclose(out[b], ref, rtol=0, atol=1e-12)


def test_check_d_incremental_decode_equals_full_causal_recompute():
    T, n_q, n_kv, D = 40, 4, 2, 64
    Q = wl.normal_bf16_bits((T, n_q, D), (31, 1))
    K = wl.normal_bf16_bits((T, n_kv, D), (31, 2))
    V = wl.normal_bf16_bits((T, n_kv, D), (31, 3))
    # Full causal attention over all T positions, from scratch (library routine).
    q = torch.from_numpy(_f64(Q)).permute(1, 0, 2)  # (n_q, T, D)
    k = torch.from_numpy(_f64(K)).permute(1, 0, 2).repeat_interleave(n_q // n_kv, 0)
    v = torch.from_numpy(_f64(V)).permute(1, 0, 2).repeat_interleave(n_q // n_kv, 0)
    full = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=0.125)
    full = full.permute(1, 0, 2).numpy()  # (T, n_q, D)
    # Incremental: append one token per step into a paged pool, decode the new query.
    m = oracle.PoolMirror(8, 16, n_kv, D)
    table = np.array([[5, 2, 7]], dtype=np.int32)
    for t in range(T):
        slot = oracle.slot_of(table[0], t, 16, 8)
        m.append(K[t:t + 1], V[t:t + 1], np.array([slot], dtype=np.int64))
        out = m.decode(Q[t:t + 1], table, np.array([t + 1], dtype=np.int32), 0.125)
        np.testing.assert_allclose(out[0], full[t], rtol=0, atol=1e-12)


def test_check_e_closed_forms():
    D = 64
    m = oracle.PoolMirror(4, 16, 1, D)
    table = np.array([[2, 0]], dtype=np.int32)
    # C = 1: the only weight is 1, out = v exactly.
    kv = wl.normal_bf16_bits((2, 1, D), (41, 1))
    m.append(kv[:1], kv[1:], np.array([2 * 16], dtype=np.int64))
    q = wl.normal_bf16_bits((1, 2, D), (41, 2))
    out = m.decode(q, table, np.array([1], dtype=np.int32), 0.125)
    assert np.array_equal(out[0, 0], _f64(kv[1, 0])) and np.array_equal(out[0, 1], _f64(kv[1, 0]))
    # Identical keys: uniform weights, out = mean of V.
    C = 20
    k_same = np.repeat(wl.normal_bf16_bits((1, 1, D), (41, 3)), C, axis=0)
    vs = wl.normal_bf16_bits((C, 1, D), (41, 4))
    slots = np.array([oracle.slot_of(table[0], p, 16, 4) for p in range(C)], dtype=np.int64)
    m.append(k_same, vs, slots)
    out = m.decode(q, table, np.array([C], dtype=np.int32), 0.125)
    np.testing.assert_allclose(out[0, 0], _f64(vs)[:, 0, :].mean(axis=0), rtol=0, atol=1e-14)
    # q = 0: also uniform.
    zq = np.zeros((1, 2, D), dtype=np.uint16)
    m.append(wl.normal_bf16_bits((C, 1, D), (41, 5)), vs, slots)
    out = m.decode(zq, table, np.array([C], dtype=np.int32), 0.125)
    np.testing.assert_allclose(out[0, 1], _f64(vs)[:, 0, :].mean(axis=0), rtol=0, atol=1e-14)
    # One key far above the others: out is that key's value.
    kk = np.zeros((C, 1, D), dtype=np.float32)
    kk[13, 0, 0] = 64.0
    qq = np.zeros((1, 2, D), dtype=np.float32)
    qq[0, :, 0] = 64.0
    m.append(wl.f32_to_bf16_bits(kk), vs, slots)
    out = m.decode(wl.f32_to_bf16_bits(qq), table, np.array([C], dtype=np.int32), 0.125)
    np.testing.assert_allclose(out[0, 0], _f64(vs[13, 0]), rtol=0, atol=1e-200)


def test_check_e_two_and_three_tokens_by_hand():
    # D = 2, scale = 1, q = (1, 0): scores are the keys' first components.
    m = oracle.PoolMirror(1, 16, 1, 2)
    k = np.array([[[0.0, 5.0]], [[1.0, -2.0]], [[0.5, 0.0]]], dtype=np.float32)
    v = np.array([[[1.0, 0.0]], [[0.0, 1.0]], [[2.0, 2.0]]], dtype=np.float32)
    m.append(wl.f32_to_bf16_bits(k), wl.f32_to_bf16_bits(v), np.arange(3, dtype=np.int64))
    q = wl.f32_to_bf16_bits(np.array([[[1.0, 0.0]]], dtype=np.float32))
    table = np.array([[0]], dtype=np.int32)
    out2 = m.decode(q, table, np.array([2], dtype=np.int32), 1.0)[0, 0]
    e = math.e
    assert out2[0] == pytest.approx(1 / (1 + e), abs=1e-15)
    assert out2[1] == pytest.approx(e / (1 + e), abs=1e-15)
    out3 = m.decode(q, table, np.array([3], dtype=np.int32), 1.0)[0, 0]
    w = np.array([1.0, e, math.exp(0.5)])
    w /= w.sum()
    assert out3[0] == pytest.approx(w[0] * 1 + w[2] * 2, abs=1e-15)
    assert out3[1] == pytest.approx(w[1] * 1 + w[2] * 2, abs=1e-15)


def test_empty_sequence_gives_zero():
    m = oracle.PoolMirror(2, 16, 1, 64)
    q = wl.normal_bf16_bits((2, 2, 64), (51, 1))
    out = m.decode(q, np.array([[0], [1]], dtype=np.int32), np.array([0, 0], dtype=np.int32), 0.125)
    assert not out.any()


def test_decode_rejects_bad_table_entries():
    m = oracle.PoolMirror(2, 16, 1, 64)
    q = wl.normal_bf16_bits((1, 1, 64), (52, 1))
    with pytest.raises(ValueError):
        m.decode(q, np.array([[7]], dtype=np.int32), np.array([3], dtype=np.int32), 0.125)
    with pytest.raises(ValueError):
        m.decode(q, np.array([[0]], dtype=np.int32), np.array([17], dtype=np.int32), 0.125)


def test_fp8_decode_equals_bf16_decode_on_exact_values():
    # Values exactly representable in both E4M3 and bf16, scale 1: the FP8
    # pool must give the same attention as the bf16 pool, bit for bit.
    rng = np.random.default_rng(61)
    grid = np.array([0, 0.25, 0.5, 1, 1.5, 2, 3, -0.25, -0.75, -1, -2, 0.125], dtype=np.float32)
    T, D = 30, 64
    kf = rng.choice(grid, size=(T, 2, D)).astype(np.float32)
    vf = rng.choice(grid, size=(T, 2, D)).astype(np.float32)
    kb, vb = wl.f32_to_bf16_bits(kf), wl.f32_to_bf16_bits(vf)
    ones = np.ones(2, dtype=np.float32)
    m16 = oracle.PoolMirror(4, 16, 2, D)
    m8 = oracle.PoolMirror(4, 16, 2, D, oracle.E4M3, ones, ones)
    table = np.array([[3, 1]], dtype=np.int32)
    slots = np.array([oracle.slot_of(table[0], p, 16, 4) for p in range(T)], dtype=np.int64)
    m16.append(kb, vb, slots)
    m8.append(kb, vb, slots)
    q = wl.normal_bf16_bits((1, 4, D), (61, 1))
    a = m16.decode(q, table, np.array([T], dtype=np.int32), 0.125)
    b = m8.decode(q, table, np.array([T], dtype=np.int32), 0.125)
    assert np.array_equal(a, b)


def test_fp8_scales_multiply_dequantised_values():
    # Same codes, K scale doubled and V scale tripled: with the attention scale
    # halved the scores are unchanged and every value is 3x, so out is 3x.
    D = 64
    kb = wl.normal_bf16_bits((10, 1, D), (62, 1))
    vb = wl.normal_bf16_bits((10, 1, D), (62, 2))
    s1 = np.array([0.02], dtype=np.float32)
    m1 = oracle.PoolMirror(1, 16, 1, D, oracle.E4M3, s1, s1)
    m1.append(kb, vb, np.arange(10, dtype=np.int64))
    m2 = oracle.PoolMirror(1, 16, 1, D, oracle.E4M3, s1 * 2, s1 * 3)
    m2.k[:], m2.v[:] = m1.k, m1.v
    q = wl.normal_bf16_bits((1, 1, D), (62, 3))
    t = np.array([[0]], dtype=np.int32)
    c = np.array([10], dtype=np.int32)
    o1 = m1.decode(q, t, c, 0.25)
    o2 = m2.decode(q, t, c, 0.125)
    np.testing.assert_allclose(o2, 3 * o1, rtol=1e-14, atol=0)


# ---------------------------------------------------------------------------
# The split-KV recurrence the GPU path relies on, against the oracle
# ---------------------------------------------------------------------------

def test_partitioned_online_softmax_with_lse_merge_equals_oracle():
    """"Write online softmax ... check it matches the naive result" (KV cache,
    PagedAttention and FlashAttention, "Practise it"): the running-max
    recurrence of Problem 5, run per partition, then partitions merged by
    their (max, sum), equals the oracle's plain softmax to fp64 rounding."""
    w = wl.build("split", 8, 2, 64, [300, 1000], seed=71)
    out = _mirror_for(w).decode(w.q, w.block_tables, w.context_lens, w.scale)
    for b in range(w.batch):
        k, v = _contiguous_kv(w, b)
        q = _f64(w.q[b])
        C = k.shape[0]
        for h in range(w.n_q):
            g = h // (w.n_q // w.n_kv)
            s = float(w.scale) * (k[:, g, :] @ q[h])
            parts = []
            for lo in range(0, C, 128):  # partitions of 128 positions
                m, l, o = -np.inf, 0.0, np.zeros(64)
                for t0 in range(lo, min(lo + 128, C), 16):  # tiles of 16
                    sj = s[t0:min(t0 + 16, lo + 128, C)]
                    vj = v[t0:t0 + len(sj), g, :]
                    m_new = max(m, sj.max())
                    l = math.exp(m - m_new) * l + np.exp(sj - m_new).sum()
                    o = math.exp(m - m_new) * o + np.exp(sj - m_new) @ vj
                    m = m_new
                parts.append((m, l, o))
            M = max(p[0] for p in parts)
            L = sum(math.exp(p[0] - M) * p[1] for p in parts)
            O = sum(math.exp(p[0] - M) * p[2] for p in parts) / L
            np.testing.assert_allclose(O, out[b, h], rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# 4-bit KV (the reading of "per-channel keys", KIVI / KVQuant: "KV cache,
# PagedAttention and FlashAttention", Problem 3, "Trade-offs"): asymmetric
# codes c = clamp(rint((x - z) / s), 0, 15) in fp32, keys per (head, channel),
# values per (token, head) from the row's min and max.
# ---------------------------------------------------------------------------

def test_int4_code_against_numpy_fp32_rint():
    rng = np.random.default_rng(11)
    xs = rng.normal(size=3000).astype(np.float32)
    ss = (np.abs(rng.normal(size=3000)) + 0.01).astype(np.float32)
    zs = rng.normal(size=3000).astype(np.float32)
    # exact midpoints (ties must go to the even code) and out-of-range values
    xs[:40] = (np.arange(40) % 15 + np.float32(0.5)) * np.float32(0.5) + np.float32(-1.0)
    ss[:40], zs[:40] = 0.5, -1.0
    xs[40:50], xs[50:60] = -50.0, 50.0
    for x, s, z in zip(xs, ss, zs):
        ref = int(np.clip(np.rint(np.float32(np.float32(x - z) / s)), 0, 15))
        assert oracle.int4_code(x, s, z) == ref, (x, s, z)
    assert oracle.int4_code(0.75, 0.5, -1.0) == 4  # 3.5 -> 4 (even)
    assert oracle.int4_code(1.25, 0.5, -1.0) == 4  # 4.5 -> 4 (even)


def test_int4_row_params_and_error_bound():
    rng = np.random.default_rng(12)
    const = wl.f32_to_bf16_bits(np.full(64, 0.375, np.float32))
    assert oracle.int4_row_params(const) == (1.0, 0.375)  # max == min: s = 1, every code 0
    for _ in range(50):
        row = wl.f32_to_bf16_bits(rng.normal(size=128).astype(np.float32))
        xf = wl.bf16_bits_to_f32(row)
        s, z = oracle.int4_row_params(row)
        assert z == xf.min() and s == np.float32(np.float32(xf.max() - xf.min()) / np.float32(15))
        codes = [oracle.int4_code(x, s, z) for x in xf]
        assert min(codes) == 0 and max(codes) == 15
        err = np.abs(np.array(codes) * np.float64(s) + z - xf)
        assert err.max() <= s / 2 * (1 + 1e-6)  # round to nearest: half a step at most


def test_int4_mirror_layout_and_exact_values():
    """Values exactly on the code grid round-trip: the 4-bit decode then
    equals the bf16 decode of the same values, bit for bit, and the packed
    bytes put the even channel in the low nibble."""
    rng = np.random.default_rng(13)
    n_kv, d, NB = 2, 64, 8
    T = NB * 16  # every slot written (an unwritten 4-bit key reads back as its zero point)
    # per-(head, channel) key scales (powers of two) and zero points, so that a code times its scale plus
    # its zero point is exact in bf16 and a key dequantised with another head's or channel's
    # parameters is a different value
    h, c = np.meshgrid(np.arange(n_kv), np.arange(d), indexing="ij")
    ks = (2.0 ** -(1 + (h + c) % 3)).astype(np.float32)
    kz = (-(1.0 + h) - 0.5 * (c % 4)).astype(np.float32)
    m4 = oracle.PoolMirror(NB, 16, n_kv, d, oracle.INT4, k_scale=ks, k_zero=kz)
    mb = oracle.PoolMirror(NB, 16, n_kv, d)
    kc = rng.integers(0, 16, size=(T, n_kv, d))
    vc = rng.integers(0, 16, size=(T, n_kv, d))
    vc[..., 0], vc[..., 1] = 0, 15  # every value row spans the grid: s = 0.25 exactly
    kb = wl.f32_to_bf16_bits((kc * ks + kz).astype(np.float32))
    assert np.array_equal(wl.bf16_bits_to_f32(kb), kc * ks + kz)  # exact in bf16
    vb = wl.f32_to_bf16_bits((vc * 0.25 - 1.0).astype(np.float32))
    slots = rng.permutation(NB * 16).astype(np.int64)
    m4.append(kb, vb, slots)
    mb.append(kb, vb, slots)
    blk, off = slots[0] // 16, slots[0] % 16
    assert m4.k[blk, 1, off, 0] == kc[0, 1, 0] | (kc[0, 1, 1] << 4)
    assert tuple(m4.v_params[blk, 0, off]) == (0.25, -1.0)
    table = np.full((2, NB), -1, dtype=np.int32)
    table[0] = np.arange(NB)
    table[1, :3] = [5, 0, 2]
    lens = np.array([NB * 16, 40], dtype=np.int32)
    q = wl.f32_to_bf16_bits(rng.normal(size=(2, 4, d)).astype(np.float32))
    assert np.array_equal(m4.decode(q, table, lens, 0.125), mb.decode(q, table, lens, 0.125))


# ---------------------------------------------------------------------------
# Prefill (a chunk of new tokens per sequence, causal over the cache)
# ---------------------------------------------------------------------------

def _chunk_queries(w, chunks, seed):
    rng = np.random.default_rng(seed)
    R = int(sum(chunks))
    q = wl.f32_to_bf16_bits(rng.normal(size=(R, w.n_q, w.d_head)).astype(np.float32))
    indptr = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    return q, indptr


def test_prefill_equals_masked_sdpa_over_the_cached_sequence():
    """Each chunk token at position C-T+i sees keys 0..C-T+i: torch's fp64
    scaled_dot_product_attention with that mask (GQA by repeating KV heads)."""
    w = wl.build("pf_pin", 8, 2, 64, [1, 17, 40, 100], seed=91)
    m = _mirror_for(w)
    chunks = [1, 5, 40, 33]
    q, indptr = _chunk_queries(w, chunks, 92)
    out = m.prefill(q, indptr, w.block_tables, w.context_lens, w.scale)
    G = w.n_q // w.n_kv
    sc = float(np.float32(w.scale))
    for b, T in enumerate(chunks):
        C = int(w.context_lens[b])
        k, v = _contiguous_kv(w, b)
        kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
        vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
        qt = torch.from_numpy(_f64(q[indptr[b]:indptr[b + 1]])).permute(1, 0, 2)[None]
        mask = torch.arange(C)[None, :] <= (C - T + torch.arange(T))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=sc)
        got = out[indptr[b]:indptr[b + 1]]
        assert np.abs(got - ref[0].permute(1, 0, 2).numpy()).max() < 1e-12, b


def test_prefill_one_token_chunks_are_decode_and_chunks_compose():
    w = wl.build("pf_dec", 32, 8, 128, [300, 1, 17, 64], seed=93)
    m = _mirror_for(w)
    B = w.batch
    one = np.arange(B + 1, dtype=np.int32)
    assert np.array_equal(m.prefill(w.q, one, w.block_tables, w.context_lens, w.scale),
                          m.decode(w.q, w.block_tables, w.context_lens, w.scale))
    # a whole-sequence prefill's last rows are the prefill of the last chunk
    full = [int(c) for c in w.context_lens]
    q_full, ip_full = _chunk_queries(w, full, 94)
    tail = [min(7, c) for c in full]
    q_tail = np.concatenate([q_full[ip_full[b + 1] - tail[b]:ip_full[b + 1]] for b in range(B)])
    ip_tail = np.concatenate([[0], np.cumsum(tail)]).astype(np.int32)
    a = m.prefill(q_full, ip_full, w.block_tables, w.context_lens, w.scale)
    t = m.prefill(q_tail, ip_tail, w.block_tables, w.context_lens, w.scale)
    for b in range(B):
        assert np.array_equal(a[ip_full[b + 1] - tail[b]:ip_full[b + 1]], t[ip_tail[b]:ip_tail[b + 1]])
    with pytest.raises(ValueError):  # 3 new tokens for a sequence holding 1: a chunk longer than its cache
        m.prefill(q_full[:3], np.array([0, 0, 3, 3, 3], np.int32), w.block_tables, w.context_lens, w.scale)
