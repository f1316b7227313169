"""Block management without a GPU: the oracle's allocator model pinned to
the pages' description of sharing and copy-on-write, and the library's
host-side allocator (``kv_alloc_*``) checked against the model operation by
operation, bit-exact (ids, reference counts, free counts, which calls fail).

"KV cache, PagedAttention and FlashAttention", Problem 4, "The idea":
parallel samples or beam branches point to the same prompt blocks with a
reference count, and a shared block is copied before it is written."""
import numpy as np
import pytest

import gqa_decode_attention_paged_gb300 as pkv
import oracle
from oracle import blocks as oracle_blocks
from oracle.blocks import AllocatorModel


# ---------------------------------------------------------------- model pins

def test_model_fork_then_write_copies_only_shared_blocks():
    # one prompt of 3 blocks, forked into 3 branches that share them
    m = AllocatorModel(16)
    prompt = m.take(3)
    assert prompt == [0, 1, 2] and m.free_blocks() == 13
    m.share(prompt)
    m.share(prompt)
    assert [m.ref[i] for i in prompt] == [3, 3, 3]
    tables = [list(prompt) for _ in range(3)]
    # branch 0 writes its next token into the partly filled last block: copy first
    new, copies = m.prepare_write([tables[0][2]])
    assert copies == [(2, 3)] and new == [3]
    tables[0][2] = new[0]
    assert m.ref[2] == 2 and m.ref[3] == 1
    # branch 1 likewise
    new, copies = m.prepare_write([tables[1][2]])
    assert copies == [(2, 4)]
    tables[1][2] = new[0]
    # branch 2 is now the only owner of block 2: no copy
    new, copies = m.prepare_write([tables[2][2]])
    assert copies == [] and new == [2] and m.ref[2] == 1
    # the untouched prompt blocks are still shared three ways
    assert m.ref[0] == 3 and m.ref[1] == 3
    # every table entry is one reference
    assert sum(m.ref) == sum(len(t) for t in tables)
    # a finished branch gives back its references; shared blocks survive
    m.release(tables[0])
    assert m.ref[0] == 2 and m.ref[3] == 0 and m.free_blocks() == 16 - 4


def test_model_all_or_nothing():
    m = AllocatorModel(4)
    a = m.take(3)
    before = list(m.ref)
    with pytest.raises(MemoryError):
        m.take(2)
    assert m.ref == before
    with pytest.raises(ValueError):
        m.release([a[0], a[0]])  # one reference, released twice
    assert m.ref == before
    with pytest.raises(ValueError):
        m.share([3])  # free block
    m.share([a[0], a[1]])
    with pytest.raises(MemoryError):  # two copies needed, one block free
        m.prepare_write([a[0], a[1]])
    assert m.ref == [2, 2, 1, 0]


def test_model_duplicate_entries_in_one_write():
    # two table entries of the list point at one block held twice: the first
    # moves to a copy, the second keeps the (now private) original
    m = AllocatorModel(4)
    (b,) = m.take(1)
    m.share([b])
    new, copies = m.prepare_write([b, b])
    assert copies == [(b, 1)] and new == [1, b] and m.ref[:2] == [1, 1]


def _mirror4(nb=5):
    """A 4-bit mirror whose bytes and value parameters differ from block to block and row to row."""
    m = oracle.PoolMirror(nb, 16, 2, 64, oracle.INT4, k_scale=np.ones((2, 64), np.float32),
                          k_zero=np.zeros((2, 64), np.float32))
    m.k[:] = (np.arange(m.k.size) % 251).reshape(m.k.shape)
    m.v[:] = ((np.arange(m.v.size) * 7 + 3) % 253).reshape(m.v.shape)
    m.v_params[:] = np.arange(m.v_params.size, dtype=np.float32).reshape(m.v_params.shape)
    return m


def _pin_block_ops(bm):
    """Copy and swap on a mirror against the documented entry layout: a block's
    K bytes, its V bytes, then (4-bit) its value parameters."""
    m = _mirror4()
    k0, v0, p0 = m.k.copy(), m.v.copy(), m.v_params.copy()
    bm.copy_blocks(m, [1, 3], [4, 0])
    for s_, d_ in ((1, 4), (3, 0)):
        assert (m.k[d_] == k0[s_]).all() and (m.v[d_] == v0[s_]).all() and (m.v_params[d_] == p0[s_]).all()
    for i in (1, 2, 3):
        assert (m.k[i] == k0[i]).all() and (m.v[i] == v0[i]).all() and (m.v_params[i] == p0[i]).all()
    m = _mirror4()
    img = bm.swap_out(m, [2, 0])
    assert img == b"".join(a[i].tobytes() for i in (2, 0) for a in (m.k, m.v, m.v_params))
    m2 = _mirror4()
    m2.k[:], m2.v[:], m2.v_params[:] = 0, 0, 0
    bm.swap_in(m2, img, [3, 1])
    for s_, d_ in ((2, 3), (0, 1)):
        assert (m2.k[d_] == m.k[s_]).all() and (m2.v[d_] == m.v[s_]).all()
        assert (m2.v_params[d_] == m.v_params[s_]).all()
    assert not m2.k[[0, 2, 4]].any() and not m2.v[[0, 2, 4]].any() and not m2.v_params[[0, 2, 4]].any()
    mb = oracle.PoolMirror(3, 16, 1, 64)  # bf16: no parameter part
    mb.k[:] = (np.arange(mb.k.size) % 65000).reshape(mb.k.shape)
    mb.v[:] = 9
    assert bm.swap_out(mb, [1]) == mb.k[1].tobytes() + mb.v[1].tobytes()


def test_model_block_copy_and_swap_layout():
    _pin_block_ops(oracle_blocks)


# ------------------------------------------------- library against the model

def _apply(model, lib, op, arg):
    """Run one operation on both; returns (model result, library result) or
    the exception class each raised."""
    res = []
    for who in (model, lib):
        try:
            if op == "take":
                r = [int(x) for x in who.take(arg)]
            elif op == "share":
                who.share(arg)
                r = None
            elif op == "release":
                who.release(arg)
                r = None
            elif who is lib:
                ids, src, dst = who.prepare_write(arg)
                r = ([int(x) for x in ids], list(zip(src.tolist(), dst.tolist())))
            else:
                ids, copies = who.prepare_write(arg)
                r = (ids, copies)
        except (MemoryError, ValueError, IndexError, pkv.PagedKVError):
            r = "error"
        res.append(r)
    return res


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_library_allocator_matches_model(seed):
    rng = np.random.default_rng(seed)
    N = 40
    model, lib = AllocatorModel(N), pkv.BlockAllocator(N)
    held = []  # table entries the harness holds (with repeats)
    for _ in range(400):
        op = rng.choice(["take", "share", "release", "write", "bad"])
        if op == "take":
            arg = int(rng.integers(0, 8))
            r_model, r_lib = _apply(model, lib, "take", arg)
            if r_model != "error":
                held += r_model
        elif op == "share" and held:
            arg = [int(x) for x in rng.choice(held, size=int(rng.integers(1, 4)))]
            r_model, r_lib = _apply(model, lib, "share", arg)
            if r_model != "error":
                held += arg
        elif op == "release" and held:
            idx = rng.choice(len(held), size=min(len(held), int(rng.integers(1, 5))), replace=False)
            arg = [held[i] for i in idx]
            r_model, r_lib = _apply(model, lib, "release", arg)
            if r_model != "error":
                for i in sorted(idx, reverse=True):
                    held.pop(i)
        elif op == "write" and held:
            idx = rng.choice(len(held), size=min(len(held), int(rng.integers(1, 4))), replace=False)
            arg = [held[i] for i in idx]
            r_model, r_lib = _apply(model, lib, "write", arg)
            if r_model != "error":
                for i, new in zip(idx, r_model[0]):
                    held[i] = new
        else:  # an invalid request: a free or out-of-range block, or a release too many
            bad = int(rng.choice([N + 3, -1] + [i for i in range(N) if model.ref[i] == 0][:1]))
            r_model, r_lib = _apply(model, lib, rng.choice(["share", "release", "write"]), [bad])
            assert r_model == "error"
        assert r_model == r_lib, (op, r_model, r_lib)
        assert model.free_blocks() == lib.free_blocks()
        assert [lib.refcount(i) for i in range(N)] == model.ref
        assert sum(model.ref) == len(held)
    lib.close()


def test_library_allocator_errors():
    with pytest.raises(pkv.PagedKVError):
        pkv.BlockAllocator(0)
    a = pkv.BlockAllocator(3)
    with pytest.raises(pkv.PagedKVError) as e:
        a.take(4)
    assert e.value.status == 3  # ENOMEM
    assert a.free_blocks() == 3
    with pytest.raises(pkv.PagedKVError) as e:
        a.refcount(3)
    assert e.value.status == 2  # ERANGE
    ids = a.take(2)
    with pytest.raises(pkv.PagedKVError):
        a.release([ids[0], ids[0]])
    assert a.refcount(ids[0]) == 1
    a.close()
