"""CPU oracle for paged GQA decode attention (fp64, plain C behind ctypes).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product (``gqa_decode_attention_paged_gb300``) never imports it, and it never
imports the product: the two share no code.

Every function here is a thin numpy marshalling layer over
``pagedkv_oracle.c``, which holds the arithmetic and cites, per function, the
passage of the pages it follows:

* ``kv_bytes_per_token`` -- "KV cache, PagedAttention and FlashAttention",
  Problem 3, "The concepts" (2 x L x n_kv x d_head x bytes).
* ``slot_of`` -- same page, Problem 4, "The idea" (block = p // B,
  offset = p % B, physical block from the block table).
* ``append`` -- "The KV Cache from First Principles", "Deriving the cache".
* ``prefill`` -- a chunk of new tokens per sequence attending causally over
  the cache: "Memory Management in LLM Serving Systems", "FlashAttention";
  "The KV Cache from First Principles", "Deriving the cache".
* ``decode`` -- "The KV Cache from First Principles", "Implementation" and
  "Grouped-query attention: the compromise"; max-subtracted softmax from
  "Memory Management in LLM Serving Systems", "FlashAttention".
* ``e4m3_decode`` / ``e4m3_encode`` -- the E4M3 bit-field definition and a
  brute-force nearest-code encoder (the pages say "FP8"; E4M3 is the reading).

Pool contents mirrored: the keys and the values as two logical arrays
``[num_blocks][n_kv][block_size][d_head]``.  The library's pool places each
(block, KV head)'s key rows and value rows side by side in one entry; the tests
read its keys and values through the strides ``kv_pool_layout`` reports, as
these same logical arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pagedkv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16 = 0
E4M3 = 1
INT4 = 2


def build(force: bool = False) -> str:
    """Compile ``pagedkv_oracle.c`` into ``liboracle.so`` next to it (gcc)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm", "-lpthread"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        c = ctypes
        P = c.c_void_p
        lib.orc_kv_bytes_per_token.argtypes = [c.c_int, c.c_int, c.c_int, c.c_double]
        lib.orc_kv_bytes_per_token.restype = c.c_double
        lib.orc_slot_of.argtypes = [P, c.c_int64, c.c_int, c.c_int64]
        lib.orc_slot_of.restype = c.c_int64
        lib.orc_e4m3_decode.argtypes = [c.c_uint8]
        lib.orc_e4m3_decode.restype = c.c_double
        lib.orc_e4m3_encode.argtypes = [c.c_float]
        lib.orc_e4m3_encode.restype = c.c_uint8
        lib.orc_quantise_e4m3.argtypes = [c.c_uint16, c.c_float]
        lib.orc_quantise_e4m3.restype = c.c_uint8
        lib.orc_append.argtypes = [P, P, c.c_int, c.c_int64, c.c_int, c.c_int, c.c_int,
                                   P, P, P, c.c_int64, P, P]
        lib.orc_append.restype = c.c_int64
        lib.orc_decode.argtypes = [P, P, c.c_int, c.c_int64, c.c_int, c.c_int, c.c_int,
                                   P, c.c_int, c.c_int, P, c.c_int, P, c.c_float, P, P, P, c.c_int]
        lib.orc_decode.restype = c.c_int
        lib.orc_int4_code.argtypes = [c.c_float, c.c_float, c.c_float]
        lib.orc_int4_code.restype = c.c_uint8
        lib.orc_int4_row_params.argtypes = [P, c.c_int, c.POINTER(c.c_float), c.POINTER(c.c_float)]
        lib.orc_append_int4.argtypes = [P, P, P, c.c_int64, c.c_int, c.c_int, c.c_int, P, P, P, c.c_int64, P, P]
        lib.orc_append_int4.restype = c.c_int64
        lib.orc_decode_int4.argtypes = [P, P, P, c.c_int64, c.c_int, c.c_int, c.c_int, P, c.c_int, c.c_int, P,
                                        c.c_int, P, c.c_float, P, P, P, c.c_int]
        lib.orc_decode_int4.restype = c.c_int
        lib.orc_prefill.argtypes = [P, P, c.c_int, c.c_int64, c.c_int, c.c_int, c.c_int, P, P, c.c_int, c.c_int,
                                    P, c.c_int, P, c.c_float, P, P, P, c.c_int]
        lib.orc_prefill.restype = c.c_int
        lib.orc_hardware_threads.argtypes = []
        lib.orc_hardware_threads.restype = c.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def hardware_threads() -> int:
    return int(_load().orc_hardware_threads())


def kv_bytes_per_token(layers: int, n_kv: int, d_head: int, bytes_per_value: float) -> float:
    return float(_load().orc_kv_bytes_per_token(layers, n_kv, d_head, float(bytes_per_value)))


def slot_of(table_row: np.ndarray, pos: int, block_size: int, num_blocks: int) -> int:
    row = np.ascontiguousarray(table_row, dtype=np.int32)
    return int(_load().orc_slot_of(_ptr(row), int(pos), int(block_size), int(num_blocks)))


def e4m3_decode(code: int) -> float:
    return float(_load().orc_e4m3_decode(int(code) & 0xFF))


def e4m3_encode(y: float) -> int:
    return int(_load().orc_e4m3_encode(float(y)))


def quantise_e4m3(bf16_bits: int, scale: float) -> int:
    return int(_load().orc_quantise_e4m3(int(bf16_bits) & 0xFFFF, float(scale)))


def int4_code(x: float, s: float, z: float) -> int:
    """clamp(rint((x - z) / s), 0, 15) in fp32 (the 4-bit reading)."""
    return int(_load().orc_int4_code(float(x), float(s), float(z)))


def int4_row_params(row_bits: np.ndarray) -> tuple[float, float]:
    """A value row's (s, z): z = min, s = (max - min) / 15 (1 if max == min), fp32."""
    r = np.ascontiguousarray(row_bits, dtype=np.uint16)
    sc, ze = ctypes.c_float(), ctypes.c_float()
    _load().orc_int4_row_params(_ptr(r), r.size, ctypes.byref(sc), ctypes.byref(ze))
    return float(sc.value), float(ze.value)


class PoolMirror:
    """Host copy of a K/V block pool's contents, as logical key and value arrays.

    ``k`` and ``v`` are raw element arrays: uint16 bf16 bit patterns or uint8
    E4M3 codes, shaped ``[num_blocks, n_kv, block_size, d_head]`` and
    zero-filled, like a freshly created pool.
    """

    def __init__(self, num_blocks, block_size, n_kv, d_head, dtype=BF16, k_scale=None, v_scale=None,
                 k_zero=None):
        self.num_blocks, self.block_size, self.n_kv, self.d_head = num_blocks, block_size, n_kv, d_head
        self.dtype = dtype
        el = np.uint16 if dtype == BF16 else np.uint8
        cols = d_head // 2 if dtype == INT4 else d_head  # 4-bit: packed codes, two per byte
        shape = (num_blocks, n_kv, block_size, cols)
        self.k = np.zeros(shape, dtype=el)
        self.v = np.zeros(shape, dtype=el)
        # 4-bit pools: per-row value (s, z); k_scale / k_zero are then [n_kv, d_head]
        self.v_params = np.zeros((num_blocks, n_kv, block_size, 2), dtype=np.float32) if dtype == INT4 else None
        self.k_scale = None if k_scale is None else np.ascontiguousarray(k_scale, dtype=np.float32)
        self.v_scale = None if v_scale is None else np.ascontiguousarray(v_scale, dtype=np.float32)
        self.k_zero = None if k_zero is None else np.ascontiguousarray(k_zero, dtype=np.float32)

    def append(self, k_new_bits: np.ndarray, v_new_bits: np.ndarray, slot_mapping: np.ndarray) -> int:
        """Write tokens into their slots; returns how many slots were past the end."""
        kb = np.ascontiguousarray(k_new_bits, dtype=np.uint16)
        vb = np.ascontiguousarray(v_new_bits, dtype=np.uint16)
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        T = sm.shape[0]
        assert kb.shape == (T, self.n_kv, self.d_head) and vb.shape == kb.shape
        if self.dtype == INT4:
            if self.k_scale is None or self.k_zero is None:
                raise ValueError("4-bit pool needs per-channel k_scale and k_zero")
            return int(_load().orc_append_int4(_ptr(self.k), _ptr(self.v), _ptr(self.v_params), self.num_blocks,
                                               self.block_size, self.n_kv, self.d_head, _ptr(kb), _ptr(vb),
                                               _ptr(sm), T, _ptr(self.k_scale), _ptr(self.k_zero)))
        if self.dtype == E4M3 and (self.k_scale is None or self.v_scale is None):
            raise ValueError("E4M3 pool needs k_scale and v_scale")
        return int(_load().orc_append(_ptr(self.k), _ptr(self.v), self.dtype, self.num_blocks,
                                      self.block_size, self.n_kv, self.d_head, _ptr(kb), _ptr(vb),
                                      _ptr(sm), T, _ptr(self.k_scale), _ptr(self.v_scale)))

    def decode(self, q_bits: np.ndarray, block_tables: np.ndarray, context_lens: np.ndarray,
               scale: float, threads: int | None = None) -> np.ndarray:
        """fp64 attention output ``[batch, n_q, d_head]`` for one query per sequence."""
        qb = np.ascontiguousarray(q_bits, dtype=np.uint16)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        B, n_q, D = qb.shape
        assert D == self.d_head and bt.shape[0] == B and cl.shape == (B,)
        out = np.empty((B, n_q, D), dtype=np.float64)
        if self.dtype == INT4:
            rc = _load().orc_decode_int4(_ptr(self.k), _ptr(self.v), _ptr(self.v_params), self.num_blocks,
                                         self.block_size, self.n_kv, self.d_head, _ptr(qb), B, n_q, _ptr(bt),
                                         bt.shape[1], _ptr(cl), float(np.float32(scale)), _ptr(self.k_scale),
                                         _ptr(self.k_zero), _ptr(out), int(threads or hardware_threads()))
            if rc != 0:
                raise ValueError(f"oracle decode failed with code {rc}")
            return out
        rc = _load().orc_decode(_ptr(self.k), _ptr(self.v), self.dtype, self.num_blocks,
                                self.block_size, self.n_kv, self.d_head, _ptr(qb), B, n_q,
                                _ptr(bt), bt.shape[1], _ptr(cl), float(np.float32(scale)),
                                _ptr(self.k_scale), _ptr(self.v_scale), _ptr(out),
                                int(threads or hardware_threads()))
        if rc != 0:
            raise ValueError(f"oracle decode failed with code {rc}")
        return out

    def prefill(self, q_bits: np.ndarray, qo_indptr: np.ndarray, block_tables: np.ndarray,
                context_lens: np.ndarray, scale: float, threads: int | None = None) -> np.ndarray:
        """fp64 causal attention ``[rows, n_q, d_head]`` of each sequence's chunk
        of new tokens (rows qo_indptr[b] .. qo_indptr[b+1], the last positions of
        its cache) over its cache."""
        qb = np.ascontiguousarray(q_bits, dtype=np.uint16)
        ip = np.ascontiguousarray(qo_indptr, dtype=np.int32)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        R, n_q, D = qb.shape
        B = cl.shape[0]
        assert D == self.d_head and ip.shape == (B + 1,) and bt.shape[0] == B and ip[-1] == R
        out = np.empty((R, n_q, D), dtype=np.float64)
        rc = _load().orc_prefill(_ptr(self.k), _ptr(self.v), self.dtype, self.num_blocks, self.block_size,
                                 self.n_kv, self.d_head, _ptr(qb), _ptr(ip), B, n_q, _ptr(bt), bt.shape[1],
                                 _ptr(cl), float(np.float32(scale)), _ptr(self.k_scale), _ptr(self.v_scale),
                                 _ptr(out), int(threads or hardware_threads()))
        if rc != 0:
            raise ValueError(f"oracle prefill failed with code {rc}")
        return out
