"""Block copy and swap kernels against the oracle's block operations on a
pool mirror, bit-exact over the whole pool; and copy-on-write end to end: a
forked sequence writes into a block it shares, gets a private copy first,
and both sequences then decode to the oracle's answer.

"KV cache, PagedAttention and FlashAttention", Problem 4, "The idea":
sharing by reference count, copy before writing a shared block, swapping a
preempted sequence's blocks to CPU memory."""
import numpy as np
import pytest
import torch

import gqa_decode_attention_paged_gb300 as pkv
import oracle
import workloads as wl
from gpu_util import assert_close, bf16_dev, fill, i32_dev, i64_dev, make_pool, mirror, out_f64, pool_bytes
from gpu_util import mirror_bytes
from oracle.blocks import AllocatorModel, copy_blocks, swap_in, swap_out

pytestmark = pytest.mark.gpu


def _rand_bf16(rng, shape):
    return wl.f32_to_bf16_bits(rng.standard_normal(size=shape).astype(np.float32)).reshape(shape)


def _filled(w):
    pool = make_pool(w)
    fill(pool, w)
    pkv.paged_kv_append(pool, bf16_dev(w.step_k), bf16_dev(w.step_v), i64_dev(w.step_slots))
    return pool, mirror(w)


def _same_pool(pool, m, what):
    gk, gv = pool_bytes(pool)
    mk, mv = mirror_bytes(m)
    assert np.array_equal(gk, mk) and np.array_equal(gv, mv), what
    if m.v_params is not None:  # 4-bit: the value rows' (scale, zero point), bit for bit
        assert np.array_equal(pool.v_params_view().cpu().numpy().view(np.uint32), m.v_params.view(np.uint32)), what


WORKLOADS = [
    lambda: wl.build("bk_bf16", 32, 8, 128, [700, 33, 160, 1000], seed=81),
    lambda: wl.build("bk_fp8_d64", 8, 2, 64, [300, 17, 90], dtype="fp8", seed=82),
    lambda: wl.build("bk_int4", 32, 8, 128, [500, 33, 700], dtype="int4", seed=83),
    lambda: wl.build("bk_int4_d64", 8, 2, 64, [300, 17, 90], dtype="int4", seed=84),
]


@pytest.mark.parametrize("make", WORKLOADS)
def test_block_copy_matches_oracle(make):
    w = make()
    pool, m = _filled(w)
    rng = np.random.default_rng(7)
    ids = rng.permutation(w.num_blocks)
    n = min(37, w.num_blocks // 2)
    src, dst = ids[:n].astype(np.int32), ids[n:2 * n].astype(np.int32)
    pkv.kv_block_copy(pool, i32_dev(src), i32_dev(dst))
    copy_blocks(m, src, dst)
    _same_pool(pool, m, "after copy")
    assert pool.get_error() == 0
    pool.close()


def test_block_copy_skips_out_of_range_pairs():
    w = WORKLOADS[0]()
    pool, m = _filled(w)
    src = np.array([3, w.num_blocks, 5, -1], dtype=np.int32)
    dst = np.array([10, 11, w.num_blocks + 7, 12], dtype=np.int32)
    pkv.kv_block_copy(pool, i32_dev(src), i32_dev(dst))
    copy_blocks(m, [3], [10])  # only the valid pair
    _same_pool(pool, m, "after copy with bad pairs")
    assert pool.get_error(clear=True) == pkv.DEVERR_BLOCK_RANGE
    pool.close()


@pytest.mark.parametrize("make", WORKLOADS)
def test_swap_out_then_in_matches_oracle(make):
    w = make()
    pool, m = _filled(w)
    bb = pkv.kv_block_bytes(pool)
    eb = pkv.kv_swap_entry_bytes(pool)
    if w.dtype == "int4":
        assert bb == w.n_kv * 16 * w.d_head // 2 and eb == 2 * bb + w.n_kv * 16 * 8
    else:
        assert bb == w.n_kv * 16 * w.d_head * w.elem_bytes and eb == 2 * bb
    rng = np.random.default_rng(9)
    out_ids = rng.choice(w.num_blocks, size=min(25, w.num_blocks), replace=False).astype(np.int32)
    host = torch.zeros(len(out_ids) * eb, dtype=torch.uint8).pin_memory()
    pkv.kv_swap_out(pool, i32_dev(out_ids), host)
    torch.cuda.synchronize()
    image = swap_out(m, out_ids)
    assert host.numpy().tobytes() == image
    # swap the same image back in to other blocks
    in_ids = rng.permutation(np.setdiff1d(np.arange(w.num_blocks), out_ids))[:len(out_ids)].astype(np.int32)
    pkv.kv_swap_in(pool, host, i32_dev(in_ids))
    swap_in(m, image, in_ids)
    _same_pool(pool, m, "after swap in")
    # a fresh image from the host side
    rnd = torch.from_numpy(rng.integers(0, 256, size=host.numel(), dtype=np.uint8)).pin_memory()
    pkv.kv_swap_in(pool, rnd, i32_dev(out_ids))
    swap_in(m, rnd.numpy().tobytes(), out_ids)
    _same_pool(pool, m, "after swap in of host bytes")
    assert pool.get_error() == 0
    pool.close()


def test_swap_rejects_pageable_memory_and_bad_ids():
    w = WORKLOADS[0]()
    pool, m = _filled(w)
    bb = pkv.kv_block_bytes(pool)
    ids = i32_dev([1, 2])
    with pytest.raises(TypeError):
        pkv.kv_swap_out(pool, ids, torch.zeros(4 * bb, dtype=torch.uint8))  # not pinned
    lib = pkv.load()
    import ctypes
    pageable = np.zeros(4 * bb, dtype=np.uint8)
    rc = lib.kv_swap_out(pool.handle, ctypes.c_void_p(ids.data_ptr()), 2, pageable.ctypes.data_as(ctypes.c_void_p),
                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 1  # EINVAL before any launch
    host = torch.zeros(2 * 2 * bb, dtype=torch.uint8).pin_memory()
    pkv.kv_swap_out(pool, i32_dev([1, w.num_blocks + 5]), host)
    torch.cuda.synchronize()
    assert host.numpy()[:2 * bb].tobytes() == swap_out(m, [1])
    assert not host.numpy()[2 * bb:].any()  # the bad entry is left untouched
    assert pool.get_error(clear=True) == pkv.DEVERR_BLOCK_RANGE
    pool.close()


def test_copy_on_write_fork_and_decode():
    """A sequence is forked (the fork shares all its blocks); each branch
    appends its own next token into the shared, partly filled last block;
    the allocator hands the branch a private copy first.  Both branches then
    decode, checked against the oracle run through the same operations."""
    n_kv, d, n_q = 8, 128, 32
    C = 16 * 5 + 7  # 5 full blocks and a partial sixth
    rng = np.random.default_rng(21)
    N = 32
    lib_alloc, model = pkv.BlockAllocator(N), AllocatorModel(N)
    table = lib_alloc.take(6)
    assert list(table) == model.take(6)
    pool = pkv.kv_pool_create(N, 16, n_kv, d, pkv.BF16)
    m = oracle.PoolMirror(N, 16, n_kv, d)
    k = _rand_bf16(rng, (C, n_kv, d))
    v = _rand_bf16(rng, (C, n_kv, d))
    slots = np.array([table[p // 16] * 16 + p % 16 for p in range(C)], dtype=np.int64)
    pkv.paged_kv_append(pool, bf16_dev(k), bf16_dev(v), i64_dev(slots))
    m.append(k, v, slots)
    # fork: a second table shares every block
    lib_alloc.share(table)
    model.share([int(x) for x in table])
    tables = [table.copy(), table.copy()]
    new_k = [_rand_bf16(rng, (1, n_kv, d)) for _ in range(2)]
    new_v = [_rand_bf16(rng, (1, n_kv, d)) for _ in range(2)]
    for br in range(2):
        ids, src, dst = lib_alloc.prepare_write([tables[br][5]])
        m_ids, m_copies = model.prepare_write([int(tables[br][5])])
        assert [int(x) for x in ids] == m_ids and list(zip(src.tolist(), dst.tolist())) == m_copies
        if len(src):
            pkv.kv_block_copy(pool, i32_dev(src), i32_dev(dst))
            copy_blocks(m, src, dst)
        tables[br][5] = ids[0]
        slot = np.array([int(tables[br][5]) * 16 + C % 16], dtype=np.int64)
        pkv.paged_kv_append(pool, bf16_dev(new_k[br]), bf16_dev(new_v[br]), i64_dev(slot))
        m.append(new_k[br], new_v[br], slot)
    # branch 0 copied (block shared), branch 1 was then the only owner
    assert tables[0][5] != table[5] and tables[1][5] == table[5]
    _same_pool(pool, m, "pool after copy-on-write")
    q = _rand_bf16(rng, (2, n_q, d))
    bt = np.stack(tables).astype(np.int32)
    lens = np.array([C + 1, C + 1], dtype=np.int32)
    scale = float(np.float32(1.0 / np.sqrt(d)))
    out = pkv.paged_decode_attention(pool, bf16_dev(q), i32_dev(bt), i32_dev(lens), scale)
    torch.cuda.synchronize()
    assert_close(out_f64(out), m.decode(q, bt, lens, scale), "decode after copy-on-write")
    # the two branches differ only through their last token
    assert not np.array_equal(out_f64(out)[0], out_f64(out)[1])
    assert pool.get_error() == 0
    pool.close()
    lib_alloc.close()


def test_int4_blocks_moved_then_decoded():
    """4-bit pool: the shortest sequence's blocks are copied to unused blocks
    and its table pointed at the copies; random host bytes are then swapped
    over the originals.  The pool (codes and value parameters) stays bit-exact
    with the oracle's, and decode reads the copies' codes with their own
    parameters."""
    w = WORKLOADS[2]()
    pool, m = _filled(w)
    b = int(np.argmin(w.context_lens))
    nb0 = -(-int(w.context_lens[b]) // 16)
    used = set(int(x) for x in w.block_tables[w.block_tables >= 0].ravel())
    free = np.array(sorted(set(range(w.num_blocks)) - used), dtype=np.int32)
    assert 0 < nb0 <= len(free)
    src = w.block_tables[b, :nb0].astype(np.int32)
    dst = free[:nb0]
    pkv.kv_block_copy(pool, i32_dev(src), i32_dev(dst))
    copy_blocks(m, src, dst)
    rng = np.random.default_rng(5)
    junk = torch.from_numpy(rng.integers(0, 256, size=nb0 * pkv.kv_swap_entry_bytes(pool), dtype=np.uint8))
    junk = junk.pin_memory()
    pkv.kv_swap_in(pool, junk, i32_dev(src))
    swap_in(m, junk.numpy().tobytes(), src)
    _same_pool(pool, m, "after copy and swap-in")
    bt = w.block_tables.copy()
    bt[b, :nb0] = dst
    out = pkv.paged_decode_attention(pool, bf16_dev(w.q), i32_dev(bt), i32_dev(w.context_lens), float(w.scale))
    torch.cuda.synchronize()
    assert_close(out_f64(out), m.decode(w.q, bt, w.context_lens, w.scale), "4-bit decode after block moves")
    assert pool.get_error() == 0
    pool.close()
