"""GB300 paged KV-cache decode attention: Python binding of libpkv.so (include/pkv.h).

Argument marshalling only: every step of the path runs in the library's CUDA kernels and
its C++ host allocator.  If the shared library is missing, importing the kernels raises:
there is no fallback.  Build it with ``python -m paged_kv_cache_159_gb300.build``.

Names follow the C ABI without the ``pkv_`` prefix:

* ``Pool(desc, free_order=None)`` -- pool_create / destroy / alloc / share / free /
  build_block_tables / attach_device / get_device_error.
* ``slot_mapping(tables, seq_lens)`` -- slot of each sequence's newest token (host);
  ``slot_mapping_all`` -- slots of every position (a whole-prompt append).
* ``kv_append(pool, k, v, slot_mapping, key_cache, value_cache)``.
* ``paged_attention_decode(pool, q, key_cache, value_cache, block_tables, seq_lens, scale,
  out, workspace=None, opts=None)``.
* ``decode_step(...)`` -- append each new token at position L-1 and decode, one launch.
* ``kv_append_layers``, ``decode_step_layers`` -- the same over every layer of a pool whose
  caches stack ``num_layers`` layers (``Pool(..., num_layers=L)``), one launch each.
* ``Pool.cow_prepare`` and ``copy_blocks`` -- copy-on-write of shared blocks before an append.
* ``block_hashes``, ``Pool.prefix_lookup / prefix_insert / prefix_evict / prefix_clear`` --
  automatic prefix caching on the host.
* ``slot_mapping_chunks``, ``prefill_plan``, ``paged_prefill`` -- prefill and chunked
  prefill on the tcgen05 tensor cores (plan on the host once per batch, run per layer).
* ``decode_step_host`` -- one decode step from pinned host memory (upload, one-launch step,
  download) in one C call; ``DecodeStepHost`` prepares that call once for a set of reused
  buffers, so each ``run()`` is the C call alone.
* ``decode_workspace_bytes``, ``probe_copy``, ``device_sm_count``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libpkv.so")

OK, ERR_INVALID, ERR_OOM, ERR_DEVICE, ERR_TIMEOUT, ERR_CUDA = range(6)
TEST_EXPIRE_NONE, TEST_EXPIRE_DECODE, TEST_EXPIRE_PREFILL = range(3)
DEVERR_SLOT, DEVERR_BLOCK_ID, DEVERR_SEQ_LEN, DEVERR_TIMEOUT, DEVERR_PLAN = 0x1, 0x2, 0x4, 0x8, 0x10
KV_BF16, KV_FP8E4M3 = 0, 1
BLOCK_SIZE = 16

EXPORTED = (
    "pkv_pool_create", "pkv_pool_destroy", "pkv_pool_get_desc", "pkv_pool_num_free",
    "pkv_pool_refcount", "pkv_pool_alloc", "pkv_pool_share", "pkv_pool_free",
    "pkv_build_block_tables", "pkv_slot_mapping", "pkv_slot_mapping_all",
    "pkv_pool_attach_device", "pkv_kv_append", "pkv_pool_layer_bytes", "pkv_kv_append_layers",
    "pkv_decode_step_layers", "pkv_cow_prepare", "pkv_copy_blocks",
    "pkv_block_hashes", "pkv_prefix_lookup", "pkv_prefix_insert", "pkv_prefix_evict",
    "pkv_prefix_clear", "pkv_prefix_cached_blocks", "pkv_slot_mapping_chunks",
    "pkv_prefill_plan_bytes", "pkv_prefill_plan", "pkv_paged_prefill", "pkv_decode_step_host",
    "pkv_decode_workspace_bytes", "pkv_paged_attention_decode",
    "pkv_paged_attention_decode_ex", "pkv_decode_step", "pkv_paged_attention_decode_noalloc",
    "pkv_get_device_error", "pkv_test_expire_waits", "pkv_probe_copy",
    "pkv_device_sm_count", "pkv_status_string",
)


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (what, status_string(status), status))


class pool_desc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float), ("num_layers", ctypes.c_int32)]


class host_step(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
                ("block_tables", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("contiguous", ctypes.c_int32)]


class device_step(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
                ("block_tables", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p), ("out", ctypes.c_void_p)]


class decode_opts(ctypes.Structure):
    _fields_ = [("grid_ctas", ctypes.c_int32), ("variant", ctypes.c_int32),
                ("warps_per_cta", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("heads_per_copy", ctypes.c_int32), ("shared_prefix_blocks", ctypes.c_int32),
                ("unit_cost", ctypes.c_int32)]


_lib = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32


def lib():
    """The loaded libpkv.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libpkv.so not built (%s); run python -m "
                              "paged_kv_cache_159_gb300.build" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        sig = {
            "pkv_pool_create": (ctypes.c_int, [ctypes.POINTER(pool_desc), _P, ctypes.POINTER(_P)]),
            "pkv_pool_destroy": (ctypes.c_int, [_P]),
            "pkv_pool_get_desc": (ctypes.c_int, [_P, ctypes.POINTER(pool_desc)]),
            "pkv_pool_num_free": (ctypes.c_int, [_P, ctypes.POINTER(_I32)]),
            "pkv_pool_refcount": (ctypes.c_int, [_P, _I32, ctypes.POINTER(_I32)]),
            "pkv_pool_alloc": (ctypes.c_int, [_P, _I32, _P]),
            "pkv_pool_share": (ctypes.c_int, [_P, _P, _I32]),
            "pkv_pool_free": (ctypes.c_int, [_P, _P, _I32]),
            "pkv_build_block_tables": (ctypes.c_int, [_P, _P, _I32, _I32, _P, _I32, _P]),
            "pkv_slot_mapping": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _P]),
            "pkv_slot_mapping_all": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _P]),
            "pkv_pool_attach_device": (ctypes.c_int, [_P, ctypes.c_int]),
            "pkv_kv_append": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _P, _P]),
            "pkv_kv_append_layers": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _P, _P]),
            "pkv_pool_layer_bytes": (ctypes.c_size_t, [_P]),
            "pkv_cow_prepare": (ctypes.c_int, [_P, _P, _P, _I32, _I32, _P, _P, ctypes.POINTER(_I32)]),
            "pkv_copy_blocks": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _P]),
            "pkv_block_hashes": (ctypes.c_int, [_P, _I32, _I32, ctypes.c_uint64, _P]),
            "pkv_prefix_lookup": (ctypes.c_int, [_P, _P, _I32, ctypes.c_uint64, _P, ctypes.POINTER(_I32)]),
            "pkv_prefix_insert": (ctypes.c_int, [_P, _P, _I32, ctypes.c_uint64, _P, _I32,
                                                 ctypes.POINTER(_I32)]),
            "pkv_prefix_evict": (ctypes.c_int, [_P, _I32, _P, ctypes.POINTER(_I32)]),
            "pkv_prefix_clear": (ctypes.c_int, [_P]),
            "pkv_prefix_cached_blocks": (ctypes.c_int, [_P, ctypes.POINTER(_I32)]),
            "pkv_slot_mapping_chunks": (ctypes.c_int, [_P, _P, _P, _I32, _I32, _I32, _P]),
            "pkv_prefill_plan_bytes": (ctypes.c_size_t, [_P, _I32, _I32, _I32]),
            "pkv_prefill_plan": (ctypes.c_int, [_P, _P, _P, _I32, _I32, _I32, _P, ctypes.c_size_t,
                                                ctypes.POINTER(_I32)]),
            "pkv_paged_prefill": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _I32, _I32, _I32,
                                                 ctypes.c_float, _P, _I32, _P, _P]),
            "pkv_decode_step_host": (ctypes.c_int, [_P, ctypes.POINTER(host_step), ctypes.POINTER(device_step),
                                                    _P, _P, _I32, _I32, _I32, ctypes.c_float, _P,
                                                    ctypes.c_size_t, ctypes.POINTER(decode_opts), _P]),
            "pkv_decode_workspace_bytes": (ctypes.c_size_t, [_P, _I32, _I32, _I32, ctypes.POINTER(decode_opts)]),
            "pkv_paged_attention_decode": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I32, _I32, _I32,
                                                          ctypes.c_float, _P, _P, ctypes.c_size_t, _P]),
            "pkv_paged_attention_decode_ex": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I32, _I32, _I32,
                                                             ctypes.c_float, _P, _P, ctypes.c_size_t,
                                                             ctypes.POINTER(decode_opts), _P]),
            "pkv_decode_step": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32,
                                               ctypes.c_float, _P, _P, ctypes.c_size_t,
                                               ctypes.POINTER(decode_opts), _P]),
            "pkv_decode_step_layers": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32,
                                                      ctypes.c_float, _P, _P, ctypes.c_size_t,
                                                      ctypes.POINTER(decode_opts), _P]),
            "pkv_paged_attention_decode_noalloc": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I32, _I32,
                                                                  _I32, ctypes.c_float, _P, _P]),
            "pkv_get_device_error": (ctypes.c_int, [_P, _P, ctypes.POINTER(ctypes.c_uint32)]),
            "pkv_test_expire_waits": (ctypes.c_int, [_I32]),
            "pkv_probe_copy": (ctypes.c_int, [_P, _P, ctypes.c_size_t, _P]),
            "pkv_device_sm_count": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(_I32)]),
            "pkv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().pkv_status_string(int(status)).decode()
    except ImportError:
        return "status %d" % status


def _check(status: int, what: str):
    if status != OK:
        raise PkvError(status, what)


def _np_ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _dev_ptr(t, what: str):
    """Device address of a contiguous CUDA tensor (or None)."""
    if t is None:
        return None
    if not getattr(t, "is_cuda", False):
        raise ValueError("%s must be a CUDA tensor" % what)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % what)
    return ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))


class Pool:
    """A paged K/V pool descriptor with its host block allocator (pkv_pool_*)."""

    def __init__(self, num_blocks, num_kv_heads, head_dim, kv_dtype=KV_BF16, k_scale=1.0,
                 v_scale=1.0, free_order=None, block_size=BLOCK_SIZE, num_layers=1):
        self.desc = pool_desc(int(num_blocks), int(block_size), int(num_kv_heads),
                              int(head_dim), int(kv_dtype), float(k_scale), float(v_scale),
                              int(num_layers))
        h = ctypes.c_void_p()
        order = None
        if free_order is not None:
            order = np.ascontiguousarray(free_order, dtype=np.int32)
            if order.shape != (int(num_blocks),):
                raise ValueError("free_order must have num_blocks entries")
        _check(lib().pkv_pool_create(ctypes.byref(self.desc),
                                     _np_ptr(order) if order is not None else None,
                                     ctypes.byref(h)), "pool_create")
        self._h = h

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            lib().pkv_pool_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def get_desc(self) -> pool_desc:
        out = pool_desc()
        _check(lib().pkv_pool_get_desc(self._h, ctypes.byref(out)), "pool_get_desc")
        return out

    def layer_bytes(self) -> int:
        """Bytes of one layer of one cache tensor (pkv_pool_layer_bytes)."""
        return int(lib().pkv_pool_layer_bytes(self._h))

    def num_free(self) -> int:
        n = _I32()
        _check(lib().pkv_pool_num_free(self._h, ctypes.byref(n)), "pool_num_free")
        return n.value

    def refcount(self, block_id: int) -> int:
        n = _I32()
        _check(lib().pkv_pool_refcount(self._h, int(block_id), ctypes.byref(n)), "pool_refcount")
        return n.value

    def alloc(self, n: int) -> np.ndarray:
        ids = np.empty(int(n), dtype=np.int32)
        _check(lib().pkv_pool_alloc(self._h, int(n), _np_ptr(ids)), "pool_alloc")
        return ids

    def share(self, ids):
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        _check(lib().pkv_pool_share(self._h, _np_ptr(ids), ids.size), "pool_share")

    def free(self, ids):
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        _check(lib().pkv_pool_free(self._h, _np_ptr(ids), ids.size), "pool_free")

    def build_block_tables(self, seq_lens, max_blocks: int, prefix_ids=None) -> np.ndarray:
        seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        prefix = np.ascontiguousarray(prefix_ids if prefix_ids is not None else [], dtype=np.int32)
        out = np.empty((seq_lens.size, int(max_blocks)), dtype=np.int32)
        _check(lib().pkv_build_block_tables(self._h, _np_ptr(seq_lens), seq_lens.size, int(max_blocks),
                                            _np_ptr(prefix) if prefix.size else None, prefix.size,
                                            _np_ptr(out)), "build_block_tables")
        return out

    def cow_prepare(self, tables, seq_lens):
        """Copy-on-write bookkeeping before an append (pkv_cow_prepare): returns (new tables,
        int32 [n, 2] (shared, fresh) pairs); the input tables are not modified."""
        tables = np.array(tables, dtype=np.int32, copy=True, order="C")
        seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        src = np.empty(max(1, seq_lens.size), dtype=np.int32)
        dst = np.empty_like(src)
        n = _I32()
        _check(lib().pkv_cow_prepare(self._h, _np_ptr(tables), _np_ptr(seq_lens), seq_lens.size,
                                     tables.shape[1], _np_ptr(src), _np_ptr(dst), ctypes.byref(n)),
               "cow_prepare")
        return tables, np.stack([src[:n.value], dst[:n.value]], axis=1)

    # ---- automatic prefix caching (host)
    def prefix_lookup(self, tokens, salt: int = 0) -> np.ndarray:
        """Physical blocks of the longest cached prefix of ``tokens`` (pkv_prefix_lookup)."""
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        out = np.empty(max(1, tokens.size // BLOCK_SIZE), dtype=np.int32)
        n = _I32()
        _check(lib().pkv_prefix_lookup(self._h, _np_ptr(tokens), tokens.size, int(salt) & (2**64 - 1),
                                       _np_ptr(out), ctypes.byref(n)), "prefix_lookup")
        return out[:n.value]

    def prefix_insert(self, tokens, salt: int, table_row) -> int:
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        row = np.ascontiguousarray(table_row, dtype=np.int32)
        n = _I32()
        _check(lib().pkv_prefix_insert(self._h, _np_ptr(tokens), tokens.size, int(salt) & (2**64 - 1),
                                       _np_ptr(row), row.size, ctypes.byref(n)), "prefix_insert")
        return n.value

    def prefix_evict(self, max_blocks: int) -> np.ndarray:
        out = np.empty(max(1, int(max_blocks)), dtype=np.int32)
        n = _I32()
        _check(lib().pkv_prefix_evict(self._h, int(max_blocks), _np_ptr(out), ctypes.byref(n)),
               "prefix_evict")
        return out[:n.value]

    def prefix_clear(self):
        _check(lib().pkv_prefix_clear(self._h), "prefix_clear")

    def prefix_cached_blocks(self) -> int:
        n = _I32()
        _check(lib().pkv_prefix_cached_blocks(self._h, ctypes.byref(n)), "prefix_cached_blocks")
        return n.value

    def attach_device(self, device: int = 0):
        _check(lib().pkv_pool_attach_device(self._h, int(device)), "pool_attach_device")

    def get_device_error(self, stream=None):
        """(status, bits): synchronises the stream, reads and clears the error word."""
        bits = ctypes.c_uint32()
        st = lib().pkv_get_device_error(self._h, _stream_ptr(stream), ctypes.byref(bits))
        return st, bits.value


def slot_mapping(tables, seq_lens, block_size: int = BLOCK_SIZE) -> np.ndarray:
    tables = np.ascontiguousarray(tables, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.empty(seq_lens.size, dtype=np.int64)
    _check(lib().pkv_slot_mapping(_np_ptr(tables), _np_ptr(seq_lens), seq_lens.size,
                                  tables.shape[1], int(block_size), _np_ptr(out)), "slot_mapping")
    return out


def slot_mapping_all(tables, seq_lens, block_size: int = BLOCK_SIZE) -> np.ndarray:
    """Slots of every position of every sequence, sequence-major (int64 [sum(seq_lens)])."""
    tables = np.ascontiguousarray(tables, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.empty(int(seq_lens.astype(np.int64).sum()), dtype=np.int64)
    _check(lib().pkv_slot_mapping_all(_np_ptr(tables), _np_ptr(seq_lens), seq_lens.size,
                                      tables.shape[1], int(block_size), _np_ptr(out)),
           "slot_mapping_all")
    return out


def block_hashes(tokens, salt: int = 0, block_size: int = BLOCK_SIZE) -> np.ndarray:
    """Chained 64-bit hash of every full block of ``tokens`` (pkv_block_hashes)."""
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    out = np.empty(max(1, tokens.size // int(block_size)), dtype=np.uint64)
    _check(lib().pkv_block_hashes(_np_ptr(tokens), tokens.size, int(block_size),
                                  int(salt) & (2**64 - 1), _np_ptr(out)), "block_hashes")
    return out[:tokens.size // int(block_size)]


def slot_mapping_chunks(tables, seq_lens, cu_q, block_size: int = BLOCK_SIZE) -> np.ndarray:
    """Slots of every prompt-chunk row: row cu_q[b] + i is position seq_lens[b] - P_b + i."""
    tables = np.ascontiguousarray(tables, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    cu_q = np.ascontiguousarray(cu_q, dtype=np.int32)
    out = np.empty(max(1, int(cu_q[-1])), dtype=np.int64)
    _check(lib().pkv_slot_mapping_chunks(_np_ptr(tables), _np_ptr(seq_lens), _np_ptr(cu_q), seq_lens.size,
                                         tables.shape[1], int(block_size), _np_ptr(out)),
           "slot_mapping_chunks")
    return out[:int(cu_q[-1])]


def prefill_plan(pool: Pool, cu_q, seq_lens, num_q_heads: int, max_blocks: int):
    """Host plan of a prefill batch (pkv_prefill_plan): (uint8 plan bytes, grid).  Copy the
    bytes to the device (e.g. torch.from_numpy(plan).cuda()) for paged_prefill."""
    cu_q = np.ascontiguousarray(cu_q, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    nbytes = int(lib().pkv_prefill_plan_bytes(pool.handle, seq_lens.size, int(num_q_heads), int(cu_q[-1])))
    if nbytes == 0:
        raise PkvError(ERR_INVALID, "prefill_plan_bytes")
    buf = np.zeros(nbytes, dtype=np.uint8)
    grid = _I32()
    _check(lib().pkv_prefill_plan(pool.handle, _np_ptr(cu_q), _np_ptr(seq_lens), seq_lens.size,
                                  int(num_q_heads), int(max_blocks), _np_ptr(buf), nbytes, ctypes.byref(grid)),
           "prefill_plan")
    return buf, grid.value


def paged_prefill(pool: Pool, q, key_cache, value_cache, block_tables, scale: float, plan, grid: int,
                  out, stream=None):
    """q/out: bf16 CUDA [T, Hq, D]; block_tables int32 CUDA [B, MB]; plan: the device copy
    (uint8 CUDA tensor) of prefill_plan's bytes, grid its grid."""
    T, Hq, _ = q.shape
    _check(lib().pkv_paged_prefill(pool.handle, _dev_ptr(q, "q"), _dev_ptr(key_cache, "key_cache"),
                                   _dev_ptr(value_cache, "value_cache"), _dev_ptr(block_tables, "block_tables"),
                                   int(block_tables.shape[0]), int(Hq), int(block_tables.shape[1]), int(T),
                                   float(scale), _dev_ptr(plan, "plan"), int(grid), _dev_ptr(out, "out"),
                                   _stream_ptr(stream)), "paged_prefill")


def kv_append(pool: Pool, k, v, slots, key_cache, value_cache, stream=None):
    """k, v: bf16 CUDA [T, Hkv, D]; slots: int64 CUDA [T]; caches: CUDA pool tensors."""
    _check(lib().pkv_kv_append(pool.handle, _dev_ptr(k, "k"), _dev_ptr(v, "v"),
                               _dev_ptr(slots, "slot_mapping"), int(slots.numel()),
                               _dev_ptr(key_cache, "key_cache"), _dev_ptr(value_cache, "value_cache"),
                               _stream_ptr(stream)), "kv_append")


def kv_append_layers(pool: Pool, k, v, slots, key_cache, value_cache, stream=None):
    """k, v: bf16 CUDA [layers, T, Hkv, D]; slots: int64 CUDA [T] (the same slot in every
    layer); caches: the pool's stacked CUDA tensors [layers, NB, Hkv, 16, D]."""
    _check(lib().pkv_kv_append_layers(pool.handle, _dev_ptr(k, "k"), _dev_ptr(v, "v"),
                                      _dev_ptr(slots, "slot_mapping"), int(slots.numel()),
                                      _dev_ptr(key_cache, "key_cache"),
                                      _dev_ptr(value_cache, "value_cache"), _stream_ptr(stream)),
           "kv_append_layers")


def copy_blocks(pool: Pool, key_cache, value_cache, src, dst, stream=None):
    """Copy blocks src[i] -> dst[i] (int32 CUDA tensors) in every layer, K and V."""
    _check(lib().pkv_copy_blocks(pool.handle, _dev_ptr(key_cache, "key_cache"),
                                 _dev_ptr(value_cache, "value_cache"), _dev_ptr(src, "src"),
                                 _dev_ptr(dst, "dst"), int(src.numel()), _stream_ptr(stream)),
           "copy_blocks")


def _opts(opts):
    if opts is None:
        return None
    if isinstance(opts, decode_opts):
        return opts
    return decode_opts(int(opts.get("grid_ctas", 0)), int(opts.get("variant", 0)),
                       int(opts.get("warps_per_cta", 0)), int(opts.get("stages", 0)),
                       int(opts.get("heads_per_copy", 0)), int(opts.get("shared_prefix_blocks", 0)),
                       int(opts.get("unit_cost", 0)))


def decode_workspace_bytes(pool: Pool, batch: int, num_q_heads: int, max_blocks: int,
                           opts=None) -> int:
    o = _opts(opts)
    return int(lib().pkv_decode_workspace_bytes(pool.handle, int(batch), int(num_q_heads),
                                                int(max_blocks), ctypes.byref(o) if o else None))


def paged_attention_decode(pool: Pool, q, key_cache, value_cache, block_tables, seq_lens,
                           scale: float, out, workspace=None, opts=None, stream=None):
    """q/out: bf16 CUDA [B, Hq, D]; block_tables int32 CUDA [B, MB]; seq_lens int32 CUDA [B];
    workspace: zero-initialised CUDA uint8 tensor of >= decode_workspace_bytes() bytes (calls
    leave it zeroed)."""
    B, Hq, _ = q.shape
    o = _opts(opts)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().pkv_paged_attention_decode_ex(
        pool.handle, _dev_ptr(q, "q"), _dev_ptr(key_cache, "key_cache"),
        _dev_ptr(value_cache, "value_cache"), _dev_ptr(block_tables, "block_tables"),
        _dev_ptr(seq_lens, "seq_lens"), int(B), int(Hq), int(block_tables.shape[1]),
        float(scale), _dev_ptr(out, "out"), _dev_ptr(workspace, "workspace"), int(ws_bytes),
        ctypes.byref(o) if o else None, _stream_ptr(stream)), "paged_attention_decode")


def decode_step(pool: Pool, q, k_new, v_new, key_cache, value_cache, block_tables, seq_lens,
                scale: float, out, workspace, opts=None, stream=None):
    """Append every sequence's new K/V (bf16 CUDA [B, Hkv, D]) at position L-1 and decode,
    in one launch (pkv_decode_step)."""
    B, Hq, _ = q.shape
    o = _opts(opts)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pkv_decode_step(
        pool.handle, _dev_ptr(q, "q"), _dev_ptr(k_new, "k_new"), _dev_ptr(v_new, "v_new"),
        _dev_ptr(key_cache, "key_cache"), _dev_ptr(value_cache, "value_cache"),
        _dev_ptr(block_tables, "block_tables"), _dev_ptr(seq_lens, "seq_lens"), int(B), int(Hq),
        int(block_tables.shape[1]), float(scale), _dev_ptr(out, "out"),
        _dev_ptr(workspace, "workspace"), int(ws_bytes), ctypes.byref(o) if o else None,
        _stream_ptr(stream)), "decode_step")


def decode_step_layers(pool: Pool, q, k_new, v_new, key_cache, value_cache, block_tables,
                       seq_lens, scale: float, out, workspace, opts=None, stream=None):
    """Every layer of a stacked pool in one launch: q/out bf16 CUDA [layers, B, Hq, D];
    k_new/v_new bf16 CUDA [layers, B, Hkv, D], or both None for attention only."""
    _, B, Hq, _ = q.shape
    o = _opts(opts)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pkv_decode_step_layers(
        pool.handle, _dev_ptr(q, "q"), _dev_ptr(k_new, "k_new"), _dev_ptr(v_new, "v_new"),
        _dev_ptr(key_cache, "key_cache"), _dev_ptr(value_cache, "value_cache"),
        _dev_ptr(block_tables, "block_tables"), _dev_ptr(seq_lens, "seq_lens"), int(B), int(Hq),
        int(block_tables.shape[1]), float(scale), _dev_ptr(out, "out"),
        _dev_ptr(workspace, "workspace"), int(ws_bytes), ctypes.byref(o) if o else None,
        _stream_ptr(stream)), "decode_step_layers")


def _host_ptr(t, what: str):
    if t is None:
        return None
    if getattr(t, "is_cuda", False) or not t.is_contiguous():
        raise ValueError("%s must be a contiguous host tensor" % what)
    return t.data_ptr()


def decode_step_host(pool: Pool, host: dict, dev: dict, key_cache, value_cache, scale: float, workspace,
                     opts=None, stream=None):
    """One decode step from host memory in one call (pkv_decode_step_host).  host: dict of
    pinned CPU tensors q, k_new, v_new, block_tables (or None), seq_lens (or None), out, and
    optionally contiguous=True when the inputs are views laid back to back in one host and
    one device buffer; dev: dict of the matching CUDA tensors.  Returns once everything is
    issued."""
    B, Hq, _ = dev["q"].shape
    h = host_step(_host_ptr(host["q"], "q"), _host_ptr(host.get("k_new"), "k_new"), _host_ptr(host.get("v_new"), "v_new"),
                  _host_ptr(host.get("block_tables"), "block_tables"), _host_ptr(host.get("seq_lens"), "seq_lens"),
                  _host_ptr(host["out"], "out"), int(bool(host.get("contiguous", False))))
    d = device_step(*[(_dev_ptr(dev.get(k), k).value if dev.get(k) is not None else None)
                      for k in ("q", "k_new", "v_new", "block_tables", "seq_lens", "out")])
    o = _opts(opts)
    _check(lib().pkv_decode_step_host(pool.handle, ctypes.byref(h), ctypes.byref(d), _dev_ptr(key_cache, "key_cache"),
                                      _dev_ptr(value_cache, "value_cache"), int(B), int(Hq),
                                      int(dev["block_tables"].shape[1]), float(scale), _dev_ptr(workspace, "workspace"),
                                      int(workspace.numel() * workspace.element_size()),
                                      ctypes.byref(o) if o else None, _stream_ptr(stream)), "decode_step_host")


class DecodeStepHost:
    """decode_step_host prepared once for a fixed set of buffers (a serving loop reuses the
    same pinned host and device buffers every step and refills their contents).  The pointer
    structures are built and checked here; each run() is one pkv_decode_step_host call, which
    still copies every input in and the output back.  The tensors must stay alive and in
    place while the object is used."""

    def __init__(self, pool: Pool, host: dict, dev: dict, key_cache, value_cache, scale: float, workspace,
                 opts=None, stream=None):
        B, Hq, _ = dev["q"].shape
        self._keep = (pool, host, dev, key_cache, value_cache, workspace)
        self._h = host_step(_host_ptr(host["q"], "q"), _host_ptr(host.get("k_new"), "k_new"),
                            _host_ptr(host.get("v_new"), "v_new"),
                            _host_ptr(host.get("block_tables"), "block_tables"),
                            _host_ptr(host.get("seq_lens"), "seq_lens"), _host_ptr(host["out"], "out"),
                            int(bool(host.get("contiguous", False))))
        self._d = device_step(*[(_dev_ptr(dev.get(k), k).value if dev.get(k) is not None else None)
                                for k in ("q", "k_new", "v_new", "block_tables", "seq_lens", "out")])
        self._o = _opts(opts)
        self._fn = lib().pkv_decode_step_host
        self._args = (pool.handle, ctypes.byref(self._h), ctypes.byref(self._d), _dev_ptr(key_cache, "key_cache"),
                      _dev_ptr(value_cache, "value_cache"), ctypes.c_int32(int(B)), ctypes.c_int32(int(Hq)),
                      ctypes.c_int32(int(dev["block_tables"].shape[1])), ctypes.c_float(float(scale)),
                      _dev_ptr(workspace, "workspace"),
                      ctypes.c_size_t(int(workspace.numel() * workspace.element_size())),
                      ctypes.byref(self._o) if self._o else None, _stream_ptr(stream))

    def run(self):
        """Issue one step (copies in, the one-launch decode, copy out) on the prepared stream."""
        st = self._fn(*self._args)
        if st:
            _check(st, "decode_step_host")


def paged_attention_decode_noalloc(pool: Pool, q, key_cache, value_cache, block_tables,
                                   seq_lens, scale: float, out, stream=None):
    """Decode without a workspace, for callers that cannot allocate device memory at run
    time: the scratch is a fixed array inside the library (pkv.h documents its limit and
    that overlapping calls race on it)."""
    B, Hq, _ = q.shape
    _check(lib().pkv_paged_attention_decode_noalloc(
        pool.handle, _dev_ptr(q, "q"), _dev_ptr(key_cache, "key_cache"),
        _dev_ptr(value_cache, "value_cache"), _dev_ptr(block_tables, "block_tables"),
        _dev_ptr(seq_lens, "seq_lens"), int(B), int(Hq), int(block_tables.shape[1]),
        float(scale), _dev_ptr(out, "out"), _stream_ptr(stream)), "paged_attention_decode_noalloc")


def test_expire_waits(which: int):
    """Failure-path test hook (pkv_test_expire_waits): while set, every launch of the chosen
    kernel runs one bounded wait out and reports PKV_DEVERR_TIMEOUT."""
    _check(lib().pkv_test_expire_waits(int(which)), "test_expire_waits")


def probe_copy(dst, src, stream=None):
    nbytes = src.numel() * src.element_size()
    _check(lib().pkv_probe_copy(_dev_ptr(dst, "dst"), _dev_ptr(src, "src"), int(nbytes),
                                _stream_ptr(stream)), "probe_copy")


def device_sm_count(device: int = 0) -> int:
    n = _I32()
    _check(lib().pkv_device_sm_count(int(device), ctypes.byref(n)), "device_sm_count")
    return n.value
