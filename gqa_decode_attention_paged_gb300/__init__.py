"""Python binding of libpagedkv.so: paged GQA decode attention for GB300.

Argument marshalling only: every step runs in the library's CUDA kernels
(see ``include/pagedkv.h``).  torch supplies device memory and streams.  The
library must be built (``__graft_entry__.build()`` or
``python -m gqa_decode_attention_paged_gb300._build``); there is no fallback,
and a missing or unloadable library raises.

Names follow the C ABI: ``kv_pool_create``, ``paged_kv_append``,
``paged_decode_attention``, ``kv_bytes_per_token``.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

BF16 = 0
FP8_E4M3 = 1
INT4 = 2

STATUS = {0: "PKV_OK", 1: "PKV_EINVAL", 2: "PKV_ERANGE", 3: "PKV_ENOMEM", 4: "PKV_ECUDA",
          5: "PKV_EUNSUPPORTED", 6: "PKV_EDEVICE"}

CASCADE_AUTO = 0
CASCADE_ALWAYS = 1
CASCADE_NEVER = 2
DEVERR_SLOT_RANGE = 0x1
DEVERR_BLOCK_RANGE = 0x2
DEVERR_CTX_RANGE = 0x4
DEVERR_TIMEOUT = 0x8

_lib = None
_lock = threading.Lock()


class PagedKVError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class _Layout(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("stride_block", ctypes.c_int64),
                ("stride_head", ctypes.c_int64), ("stride_token", ctypes.c_int64),
                ("num_blocks", ctypes.c_int64), ("block_size", ctypes.c_int32),
                ("n_kv", ctypes.c_int32), ("d_head", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("bytes_per_array", ctypes.c_int64), ("v_params", ctypes.c_void_p),
                ("v_params_bytes", ctypes.c_int64), ("alloc_bytes", ctypes.c_int64)]


class _Timing(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int64), ("append_launches", ctypes.c_int64),
                ("decode_launches", ctypes.c_int64), ("merge_launches", ctypes.c_int64),
                ("append_ms", ctypes.c_double), ("decode_ms", ctypes.c_double),
                ("merge_ms", ctypes.c_double), ("timed_append", ctypes.c_int64),
                ("timed_decode", ctypes.c_int64), ("timed_merge", ctypes.c_int64),
                ("prefix_launches", ctypes.c_int64), ("prefix_ms", ctypes.c_double),
                ("timed_prefix", ctypes.c_int64), ("block_launches", ctypes.c_int64),
                ("block_ms", ctypes.c_double), ("timed_block", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_int64)]


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libpagedkv.so (building it first if it is missing and nvcc exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path) and build_if_missing:
            _build.build()
        if not os.path.exists(path):
            raise ImportError(f"libpagedkv.so not found at {path}; run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        c = ctypes
        P = c.c_void_p
        lib.kv_pool_create.argtypes = [c.c_int64, c.c_int32, c.c_int32, c.c_int32, c.c_int32,
                                       c.POINTER(P)]
        lib.kv_pool_destroy.argtypes = [P]
        lib.kv_pool_set_fp8_scales.argtypes = [P, P, P]
        lib.kv_pool_set_int4_key_params.argtypes = [P, P, P]
        lib.kv_pool_layout.argtypes = [P, c.POINTER(_Layout)]
        lib.kv_pool_set_partition_tokens.argtypes = [P, c.c_int32]
        lib.kv_pool_set_cascade_mode.argtypes = [P, c.c_int32]
        lib.kv_pool_reserve_workspace.argtypes = [P, c.c_int32, c.c_int32, c.c_int32]
        lib.paged_kv_append.argtypes = [P, P, P, P, c.c_int64, P]
        lib.paged_decode_attention.argtypes = [P, P, c.c_int32, P, c.c_int32, P, c.c_int32,
                                               c.c_float, P, P]
        lib.paged_decode_attention_noalloc.argtypes = [P, P, c.c_int32, P, c.c_int32, P, c.c_int32,
                                                       c.c_float, P, P]
        lib.paged_decode_attention_prefix.argtypes = [P, P, c.c_int32, P, c.c_int32, P, c.c_int32, P, c.c_int32,
                                                      c.c_float, P, P]
        lib.paged_decode_attention_csr.argtypes = [P, P, c.c_int32, P, P, c.c_int64, P, c.c_int32, c.c_float, P, P]
        lib.paged_prefill_attention.argtypes = [P, P, c.c_int64, c.c_int32, P, P, c.c_int32, P, c.c_int32,
                                                c.c_float, P, P]
        lib.paged_decode_step.argtypes = [P, P, P, P, c.c_int32, P, c.c_int32, P, c.c_int32, c.c_float, P, P]
        lib.paged_decode_step_host.argtypes = [P, P, P, P, c.c_int32, P, c.c_int32, P, c.c_int32, c.c_float,
                                               P, P]
        lib.kv_bytes_per_token.argtypes = [c.c_int32, c.c_int32, c.c_int32, c.c_double]
        lib.kv_bytes_per_token.restype = c.c_double
        lib.pkv_get_error.argtypes = [P, c.c_int32, c.POINTER(c.c_uint32)]
        lib.pkv_timing_enable.argtypes = [P, c.c_int32]
        lib.pkv_selftest_wait_timeout.argtypes = [P, c.c_uint64, P]
        lib.pkv_timing_read.argtypes = [P, c.c_int32, c.POINTER(_Timing)]
        lib.kv_block_bytes.argtypes = [P]
        lib.kv_block_bytes.restype = c.c_int64
        lib.kv_swap_entry_bytes.argtypes = [P]
        lib.kv_swap_entry_bytes.restype = c.c_int64
        lib.kv_block_copy.argtypes = [P, P, P, c.c_int64, P]
        lib.kv_swap_out.argtypes = [P, P, c.c_int64, P, P]
        lib.kv_swap_in.argtypes = [P, P, P, c.c_int64, P]
        I32P = c.POINTER(c.c_int32)
        lib.kv_alloc_create.argtypes = [c.c_int64, c.POINTER(P)]
        lib.kv_alloc_destroy.argtypes = [P]
        lib.kv_alloc_free_blocks.argtypes = [P]
        lib.kv_alloc_free_blocks.restype = c.c_int64
        lib.kv_alloc_refcount.argtypes = [P, c.c_int32, I32P]
        lib.kv_alloc_take.argtypes = [P, c.c_int64, I32P]
        lib.kv_alloc_share.argtypes = [P, I32P, c.c_int64]
        lib.kv_alloc_release.argtypes = [P, I32P, c.c_int64]
        lib.kv_alloc_prepare_write.argtypes = [P, I32P, c.c_int64, I32P, I32P, c.POINTER(c.c_int64)]
        lib.pkv_status_string.argtypes = [c.c_int]
        lib.pkv_status_string.restype = c.c_char_p
        lib.pkv_last_error_message.argtypes = []
        lib.pkv_last_error_message.restype = c.c_char_p
        for name in ("kv_pool_create", "kv_pool_destroy", "kv_pool_set_fp8_scales", "kv_pool_set_int4_key_params",
                     "kv_pool_layout",
                     "kv_pool_set_partition_tokens", "kv_pool_set_cascade_mode", "kv_pool_reserve_workspace",
                     "paged_kv_append",
                     "paged_decode_attention", "paged_decode_attention_noalloc", "paged_decode_step",
                     "paged_decode_attention_csr", "paged_prefill_attention",
                     "paged_decode_step_host", "paged_decode_attention_prefix", "pkv_get_error", "pkv_timing_enable", "pkv_timing_read",
                     "pkv_selftest_wait_timeout", "kv_block_copy", "kv_swap_out", "kv_swap_in", "kv_alloc_create",
                     "kv_alloc_destroy", "kv_alloc_refcount", "kv_alloc_take", "kv_alloc_share", "kv_alloc_release",
                     "kv_alloc_prepare_write"):
            getattr(lib, name).restype = c.c_int
        _lib = lib
        return lib


def _check(status: int, allow=(0,)):
    if status not in allow:
        msg = load().pkv_last_error_message().decode(errors="replace")
        raise PagedKVError(status, msg)
    return status


def _stream_handle(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dev_ptr(t, name, dtype=None, ndim=None, shape=None):
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if shape is not None:
        for i, s in enumerate(shape):
            if s is not None and t.shape[i] != s:
                raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {shape}")
    return ctypes.c_void_p(t.data_ptr())


def kv_bytes_per_token(layers: int, n_kv: int, d_head: int, bytes_per_value: float) -> float:
    """2 x layers x n_kv x d_head x bytes_per_value (host arithmetic in the library)."""
    return float(load().kv_bytes_per_token(layers, n_kv, d_head, float(bytes_per_value)))


class Pool:
    """A K/V block pool owned by the library (one layer).  Use kv_pool_create()."""

    def __init__(self, handle, num_blocks, block_size, n_kv, d_head, dtype):
        self._h = handle
        self.num_blocks, self.block_size, self.n_kv, self.d_head, self.dtype = (
            num_blocks, block_size, n_kv, d_head, dtype)

    @property
    def handle(self):
        if not self._h:
            raise ValueError("pool is closed")
        return self._h

    def close(self):
        if getattr(self, "_h", None):
            load().kv_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def set_fp8_scales(self, k_scale, v_scale):
        import numpy as np

        ks = np.ascontiguousarray(k_scale, dtype=np.float32)
        vs = np.ascontiguousarray(v_scale, dtype=np.float32)
        if ks.shape != (self.n_kv,) or vs.shape != (self.n_kv,):
            raise ValueError(f"scales must have shape ({self.n_kv},)")
        _check(load().kv_pool_set_fp8_scales(self.handle, ks.ctypes.data_as(ctypes.c_void_p),
                                             vs.ctypes.data_as(ctypes.c_void_p)))

    def set_int4_key_params(self, k_scale, k_zero):
        """4-bit pools: per-(KV head, channel) key scale and zero point, [n_kv, d_head] fp32 each."""
        import numpy as np

        ks = np.ascontiguousarray(k_scale, dtype=np.float32)
        kz = np.ascontiguousarray(k_zero, dtype=np.float32)
        if ks.shape != (self.n_kv, self.d_head) or kz.shape != (self.n_kv, self.d_head):
            raise ValueError(f"key parameters must have shape ({self.n_kv}, {self.d_head})")
        _check(load().kv_pool_set_int4_key_params(self.handle, ks.ctypes.data_as(ctypes.c_void_p),
                                                  kz.ctypes.data_as(ctypes.c_void_p)))

    def v_params_view(self):
        """4-bit pools: the value rows' (scale, zero point), float32 [num_blocks, n_kv, block_size, 2]
        (a strided view into the pool's entries)."""
        import torch

        lay = self.layout()
        flat = self._alloc_bytes_view(lay).view(torch.float32)
        off = (lay["v_params"] - lay["k"]) // 4
        return flat.as_strided((self.num_blocks, self.n_kv, self.block_size, 2),
                               (lay["stride_block"] // 4, lay["stride_head"] // 4, 2, 1), off)

    def layout(self) -> dict:
        lay = _Layout()
        _check(load().kv_pool_layout(self.handle, ctypes.byref(lay)))
        return {f: getattr(lay, f) for f, _ in _Layout._fields_}

    def set_partition_tokens(self, tokens: int):
        _check(load().kv_pool_set_partition_tokens(self.handle, int(tokens)))

    def set_cascade_mode(self, mode: int):
        """CASCADE_AUTO, CASCADE_ALWAYS or CASCADE_NEVER for paged_decode_attention_prefix."""
        _check(load().kv_pool_set_cascade_mode(self.handle, int(mode)))

    def reserve_workspace(self, batch: int, n_q: int, max_blocks_per_seq: int):
        _check(load().kv_pool_reserve_workspace(self.handle, batch, n_q, max_blocks_per_seq))

    def get_error(self, clear: bool = False) -> int:
        bits = ctypes.c_uint32(0)
        _check(load().pkv_get_error(self.handle, int(clear), ctypes.byref(bits)), allow=(0, 6))
        return int(bits.value)

    def selftest_wait_timeout(self, limit_ns: int = 1_000_000, stream=None):
        """Run the bounded-wait check: a wait nothing completes gives up after
        limit_ns and sets DEVERR_TIMEOUT (read it with get_error)."""
        _check(load().pkv_selftest_wait_timeout(self.handle, int(limit_ns), _stream_handle(stream)))

    def timing_enable(self, on: bool = True):
        _check(load().pkv_timing_enable(self.handle, int(on)))

    def timing_read(self, reset: bool = False) -> dict:
        t = _Timing()
        _check(load().pkv_timing_read(self.handle, int(reset), ctypes.byref(t)))
        return {f: getattr(t, f) for f, _ in _Timing._fields_}

    def k_view(self):
        """The key rows as a torch uint8 tensor view [num_blocks, n_kv, block_size, row bytes]."""
        return self._view("k")

    def v_view(self):
        return self._view("v")

    @staticmethod
    def _bytes_view(ptr, n):
        import torch

        class _Holder:  # exposes the pool's memory through the CUDA array interface
            __cuda_array_interface__ = {"shape": (n,), "typestr": "|u1", "data": (ptr, False),
                                        "version": 3, "strides": None}

        return torch.as_tensor(_Holder(), device="cuda")

    def _alloc_bytes_view(self, lay):
        """The pool's whole allocation (every (block, KV head) entry), as uint8."""
        return self._bytes_view(lay["k"], lay["alloc_bytes"])

    def _view(self, which):
        """Key or value rows inside the entries, as a strided uint8 view."""
        lay = self.layout()
        elem = 2 if self.dtype == BF16 else 1
        row = self.d_head // 2 if self.dtype == INT4 else self.d_head * elem
        shape = (self.num_blocks, self.n_kv, self.block_size, row)
        strides = (lay["stride_block"] * elem, lay["stride_head"] * elem, lay["stride_token"] * elem, 1)
        return self._alloc_bytes_view(lay).as_strided(shape, strides, lay[which] - lay["k"])


def kv_pool_create(num_blocks: int, block_size: int, n_kv: int, d_head: int, dtype: int = BF16) -> Pool:
    h = ctypes.c_void_p()
    _check(load().kv_pool_create(int(num_blocks), int(block_size), int(n_kv), int(d_head), int(dtype),
                                 ctypes.byref(h)))
    return Pool(h, int(num_blocks), int(block_size), int(n_kv), int(d_head), int(dtype))


def paged_kv_append(pool: Pool, k_new, v_new, slot_mapping, stream=None):
    """k_new, v_new: bf16 [T, n_kv, d_head]; slot_mapping: int64 [T] (all CUDA)."""
    import torch

    T = int(slot_mapping.shape[0]) if slot_mapping is not None else 0
    shape = (T, pool.n_kv, pool.d_head)
    kp = _dev_ptr(k_new, "k_new", torch.bfloat16, 3, shape)
    vp = _dev_ptr(v_new, "v_new", torch.bfloat16, 3, shape)
    sp = _dev_ptr(slot_mapping, "slot_mapping", torch.int64, 1)
    _check(load().paged_kv_append(pool.handle, kp, vp, sp, T, _stream_handle(stream)))


def paged_decode_attention(pool: Pool, q, block_tables, context_lens, scale: float, out=None,
                           stream=None):
    """q: bf16 [B, n_q, d_head]; block_tables: int32 [B, W]; context_lens: int32 [B].
    Returns ``out`` (bf16 [B, n_q, d_head]), allocated if not given."""
    import torch

    qp = _dev_ptr(q, "q", torch.bfloat16, 3, (None, None, pool.d_head))
    B, n_q = int(q.shape[0]), int(q.shape[1])
    tp = _dev_ptr(block_tables, "block_tables", torch.int32, 2, (B, None))
    cp = _dev_ptr(context_lens, "context_lens", torch.int32, 1, (B,))
    if out is None:
        out = torch.empty_like(q)
    op = _dev_ptr(out, "out", torch.bfloat16, 3, tuple(q.shape))
    _check(load().paged_decode_attention(pool.handle, qp, n_q, tp, int(block_tables.shape[1]), cp, B,
                                         float(scale), op, _stream_handle(stream)))
    return out


def paged_decode_attention_csr(pool: Pool, q, kv_indptr, kv_indices, context_lens, scale: float, out=None,
                               stream=None):
    """Decode with the CSR page table: sequence b owns blocks
    kv_indices[kv_indptr[b]:kv_indptr[b+1]] (int32 CUDA tensors)."""
    import torch

    qp = _dev_ptr(q, "q", torch.bfloat16, 3, (None, None, pool.d_head))
    B, n_q = int(q.shape[0]), int(q.shape[1])
    ip = _dev_ptr(kv_indptr, "kv_indptr", torch.int32, 1, (B + 1,))
    xp = _dev_ptr(kv_indices, "kv_indices", torch.int32, 1)
    cp = _dev_ptr(context_lens, "context_lens", torch.int32, 1, (B,))
    if out is None:
        out = torch.empty_like(q)
    op = _dev_ptr(out, "out", torch.bfloat16, 3, tuple(q.shape))
    _check(load().paged_decode_attention_csr(pool.handle, qp, n_q, ip, xp, int(kv_indices.shape[0]), cp, B,
                                             float(scale), op, _stream_handle(stream)))
    return out


def paged_prefill_attention(pool: Pool, q, qo_indptr, block_tables, context_lens, scale: float, out=None,
                            stream=None):
    """Causal attention of each sequence's chunk of new tokens over its cache.
    q: bf16 [rows, n_q, d_head] (the chunks, sequence by sequence);
    qo_indptr: int32 [B + 1] (sequence b owns rows qo_indptr[b]:qo_indptr[b+1]);
    block_tables: int32 [B, W]; context_lens: int32 [B] (including the chunk)."""
    import torch

    qp = _dev_ptr(q, "q", torch.bfloat16, 3, (None, None, pool.d_head))
    rows, n_q = int(q.shape[0]), int(q.shape[1])
    B = int(context_lens.shape[0])
    ip = _dev_ptr(qo_indptr, "qo_indptr", torch.int32, 1, (B + 1,))
    tp = _dev_ptr(block_tables, "block_tables", torch.int32, 2, (B, None))
    cp = _dev_ptr(context_lens, "context_lens", torch.int32, 1, (B,))
    if out is None:
        out = torch.empty_like(q)
    op = _dev_ptr(out, "out", torch.bfloat16, 3, tuple(q.shape))
    _check(load().paged_prefill_attention(pool.handle, qp, rows, n_q, ip, tp, int(block_tables.shape[1]), cp, B,
                                          float(scale), op, _stream_handle(stream)))
    return out


def paged_decode_attention_prefix(pool: Pool, q, prefix_blocks, block_tables, context_lens, scale: float,
                                  out=None, stream=None):
    """Cascade decode: every sequence starts with the shared prefix whose
    physical block ids are ``prefix_blocks`` (int32, CUDA); the prefix is read
    once for the batch.  Same result as paged_decode_attention."""
    import torch

    qp = _dev_ptr(q, "q", torch.bfloat16, 3, (None, None, pool.d_head))
    B, n_q = int(q.shape[0]), int(q.shape[1])
    pp = _dev_ptr(prefix_blocks, "prefix_blocks", torch.int32, 1)
    tp = _dev_ptr(block_tables, "block_tables", torch.int32, 2, (B, None))
    cp = _dev_ptr(context_lens, "context_lens", torch.int32, 1, (B,))
    if out is None:
        out = torch.empty_like(q)
    op = _dev_ptr(out, "out", torch.bfloat16, 3, tuple(q.shape))
    _check(load().paged_decode_attention_prefix(pool.handle, qp, n_q, pp, int(prefix_blocks.shape[0]), tp,
                                                int(block_tables.shape[1]), cp, B, float(scale), op,
                                                _stream_handle(stream)))
    return out


def paged_decode_step(pool: Pool, q, k_new, v_new, block_tables, context_lens, scale: float, out=None,
                      stream=None):
    """Append each sequence's newest token (k_new, v_new: bf16 [B, n_kv, d])
    at position context_lens[b]-1 and decode, in one launch."""
    import torch

    qp = _dev_ptr(q, "q", torch.bfloat16, 3, (None, None, pool.d_head))
    B, n_q = int(q.shape[0]), int(q.shape[1])
    kp = _dev_ptr(k_new, "k_new", torch.bfloat16, 3, (B, pool.n_kv, pool.d_head))
    vp = _dev_ptr(v_new, "v_new", torch.bfloat16, 3, (B, pool.n_kv, pool.d_head))
    tp = _dev_ptr(block_tables, "block_tables", torch.int32, 2, (B, None))
    cp = _dev_ptr(context_lens, "context_lens", torch.int32, 1, (B,))
    if out is None:
        out = torch.empty_like(q)
    op = _dev_ptr(out, "out", torch.bfloat16, 3, tuple(q.shape))
    _check(load().paged_decode_step(pool.handle, qp, kp, vp, n_q, tp, int(block_tables.shape[1]), cp, B,
                                    float(scale), op, _stream_handle(stream)))
    return out


def _host_ptr(t, name, dtype, shape):
    import torch

    if type(t) is not torch.Tensor and not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a CPU torch tensor")
    if t.is_cuda:
        raise TypeError(f"{name} must be a CPU torch tensor")
    if t.dtype is not dtype or t.shape != shape or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)}")
    return t.data_ptr()


def paged_decode_step_host(pool: Pool, q, k_new, v_new, block_tables, context_lens, scale: float, out,
                           stream=None):
    """paged_decode_step from host tensors (pin them for asynchronous copies):
    copies in, steps, copies ``out`` back and synchronises the stream."""
    import torch

    B, n_q, D = q.shape
    W = block_tables.shape[1]
    kv_shape = (B, pool.n_kv, D)
    bf16, i32 = torch.bfloat16, torch.int32
    qp = _host_ptr(q, "q", bf16, q.shape)
    kp = _host_ptr(k_new, "k_new", bf16, kv_shape)
    vp = _host_ptr(v_new, "v_new", bf16, kv_shape)
    tp = _host_ptr(block_tables, "block_tables", i32, (B, W))
    cp = _host_ptr(context_lens, "context_lens", i32, (B,))
    op = _host_ptr(out, "out", bf16, q.shape)
    st = torch.cuda.current_stream().cuda_stream if stream is None else _stream_handle(stream).value
    _check(load().paged_decode_step_host(pool.handle, qp, kp, vp, n_q, tp, W, cp, B, float(scale), op, st))
    return out


class HostStep:
    """paged_decode_step_host on a fixed set of host buffers: the arguments
    are checked once here; each call runs one step on the buffers' current
    contents (refill them in place between calls) and returns ``out``.  With
    pinned buffers the library replays the step's launches from a CUDA graph
    after the first call, so a call is one ctypes call, one graph launch and
    one synchronise."""

    def __init__(self, pool: Pool, q, k_new, v_new, block_tables, context_lens, scale: float, out, stream=None):
        import torch

        B, n_q, D = q.shape
        W = block_tables.shape[1]
        kv_shape = (B, pool.n_kv, D)
        bf16, i32 = torch.bfloat16, torch.int32
        ptrs = (_host_ptr(q, "q", bf16, q.shape), _host_ptr(k_new, "k_new", bf16, kv_shape),
                _host_ptr(v_new, "v_new", bf16, kv_shape))
        tp = _host_ptr(block_tables, "block_tables", i32, (B, W))
        cp = _host_ptr(context_lens, "context_lens", i32, (B,))
        op = _host_ptr(out, "out", bf16, q.shape)
        st = torch.cuda.current_stream().cuda_stream if stream is None else _stream_handle(stream).value
        self.out = out
        self._keep = (pool, q, k_new, v_new, block_tables, context_lens, out)  # the buffers outlive the object
        self._fn = load().paged_decode_step_host
        self._args = (pool.handle, *ptrs, n_q, tp, W, cp, B, float(scale), op, st)

    def __call__(self):
        status = self._fn(*self._args)
        if status:
            _check(status)
        return self.out


def paged_decode_attention_noalloc(pool: Pool, q, block_tables, context_lens, scale: float, out=None,
                                   stream=None):
    """paged_decode_attention with its scratch in the library's fixed 16 MiB
    device array instead of a workspace it allocates: for callers that cannot
    allocate device memory while decoding.  Calls share that array, so calls
    that overlap on the GPU race; see include/pagedkv.h."""
    import torch

    qp = _dev_ptr(q, "q", torch.bfloat16, 3, (None, None, pool.d_head))
    B, n_q = int(q.shape[0]), int(q.shape[1])
    tp = _dev_ptr(block_tables, "block_tables", torch.int32, 2, (B, None))
    cp = _dev_ptr(context_lens, "context_lens", torch.int32, 1, (B,))
    if out is None:
        out = torch.empty_like(q)
    op = _dev_ptr(out, "out", torch.bfloat16, 3, tuple(q.shape))
    _check(load().paged_decode_attention_noalloc(pool.handle, qp, n_q, tp, int(block_tables.shape[1]), cp, B,
                                                 float(scale), op, _stream_handle(stream)))
    return out


def kv_block_bytes(pool: Pool) -> int:
    """Bytes of one block in one array (K or V): n_kv x 16 x d_head x element size."""
    return int(load().kv_block_bytes(pool.handle))


def kv_swap_entry_bytes(pool: Pool) -> int:
    """Bytes of one swapped block: K, V and (4-bit pools) the value rows' (scale, zero point)."""
    return int(load().kv_swap_entry_bytes(pool.handle))


def kv_block_copy(pool: Pool, src_blocks, dst_blocks, stream=None):
    """Copy blocks src_blocks[i] -> dst_blocks[i] (int32 CUDA tensors [n]): K, V and
    (4-bit pools) the value rows' parameters."""
    import torch

    n = int(src_blocks.shape[0])
    sp = _dev_ptr(src_blocks, "src_blocks", torch.int32, 1, (n,))
    dp = _dev_ptr(dst_blocks, "dst_blocks", torch.int32, 1, (n,))
    _check(load().kv_block_copy(pool.handle, sp, dp, n, _stream_handle(stream)))


def _pinned_ptr(t, name, nbytes):
    import torch

    if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_pinned():
        raise TypeError(f"{name} must be a pinned CPU tensor (tensor.pin_memory())")
    if not t.is_contiguous() or t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{name} must be contiguous and hold at least {nbytes} bytes")
    return ctypes.c_void_p(t.data_ptr())


def kv_swap_out(pool: Pool, blocks, host_dst, stream=None):
    """Write blocks[i] (int32 CUDA tensor [n]) into pinned host tensor
    ``host_dst`` as [n][kv_swap_entry_bytes] bytes (K, V, then the value
    rows' parameters of a 4-bit pool)."""
    import torch

    n = int(blocks.shape[0])
    bp = _dev_ptr(blocks, "blocks", torch.int32, 1, (n,))
    hp = _pinned_ptr(host_dst, "host_dst", n * kv_swap_entry_bytes(pool))
    _check(load().kv_swap_out(pool.handle, bp, n, hp, _stream_handle(stream)))
    return host_dst


def kv_swap_in(pool: Pool, host_src, blocks, stream=None):
    """Fill blocks[i] (int32 CUDA tensor [n]) from pinned host tensor ``host_src``
    laid out as kv_swap_out writes it."""
    import torch

    n = int(blocks.shape[0])
    bp = _dev_ptr(blocks, "blocks", torch.int32, 1, (n,))
    hp = _pinned_ptr(host_src, "host_src", n * kv_swap_entry_bytes(pool))
    _check(load().kv_swap_in(pool.handle, hp, bp, n, _stream_handle(stream)))


class BlockAllocator:
    """Refcounted physical-block allocator (host): take, share, release, and
    copy-on-write preparation.  Ids are Python ints / int32 numpy arrays."""

    def __init__(self, num_blocks: int):
        h = ctypes.c_void_p()
        _check(load().kv_alloc_create(int(num_blocks), ctypes.byref(h)))
        self.handle = h
        self.num_blocks = int(num_blocks)

    def close(self):
        if self.handle:
            load().kv_alloc_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @staticmethod
    def _ids(ids):
        import numpy as np

        a = np.ascontiguousarray(np.asarray(ids, dtype=np.int32).reshape(-1))
        return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))

    def free_blocks(self) -> int:
        return int(load().kv_alloc_free_blocks(self.handle))

    def refcount(self, block: int) -> int:
        out = ctypes.c_int32()
        _check(load().kv_alloc_refcount(self.handle, int(block), ctypes.byref(out)))
        return int(out.value)

    def take(self, n: int):
        import numpy as np

        out = np.zeros(int(n), dtype=np.int32)
        _check(load().kv_alloc_take(self.handle, int(n), out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))))
        return out

    def share(self, ids):
        a, p = self._ids(ids)
        _check(load().kv_alloc_share(self.handle, p, a.size))

    def release(self, ids):
        a, p = self._ids(ids)
        _check(load().kv_alloc_release(self.handle, p, a.size))

    def prepare_write(self, ids):
        """Returns (new_ids, copy_src, copy_dst): entries of ``ids`` whose block
        is shared get a private copy target; run kv_block_copy on the pairs."""
        import numpy as np

        a, p = self._ids(ids)
        a = a.copy()
        p = a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        src = np.zeros(max(1, a.size), dtype=np.int32)
        dst = np.zeros(max(1, a.size), dtype=np.int32)
        k = ctypes.c_int64()
        _check(load().kv_alloc_prepare_write(self.handle, p, a.size, src.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                             dst.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), ctypes.byref(k)))
        return a, src[:k.value].copy(), dst[:k.value].copy()


__all__ = ["BF16", "FP8_E4M3", "INT4", "Pool", "PagedKVError", "kv_pool_create", "paged_kv_append",
           "paged_decode_attention", "paged_decode_attention_noalloc", "paged_decode_step",
           "paged_decode_step_host", "paged_decode_attention_prefix", "paged_decode_attention_csr",
           "paged_prefill_attention",
           "kv_bytes_per_token", "kv_block_bytes", "kv_swap_entry_bytes",
           "kv_block_copy", "kv_swap_out", "kv_swap_in", "BlockAllocator", "load", "library_path"]
