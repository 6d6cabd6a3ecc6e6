"""Python binding of the C ABI, same names as include/injectscale.h.

Argument marshalling only: tensors become pointers, dicts become the C
structs, non-OK statuses become ISError.  Every step of the path runs in the
CUDA kernels of libinjectscale.so; nothing here computes.
"""
from __future__ import annotations

import ctypes
from ctypes import byref, c_double, c_int64, c_uint32, c_void_p

import numpy as np

from . import _lib
from ._lib import CacheDesc, RopeParams, StoreConfig, StoreInfo

DTYPE_CODES = {"f32": _lib.IS_F32, "bf16": _lib.IS_BF16, "f16": _lib.IS_F16, "e4m3": _lib.IS_FP8_E4M3}


class ISError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{_lib.STATUS_NAMES.get(status, status)}: {message}")


def _check(status: int) -> None:
    if status != _lib.IS_OK:
        msg = _lib.load().is_last_error_message()
        raise ISError(status, msg.decode() if msg else "")


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else 0
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t) -> int | None:
    if t is None:
        return None
    if hasattr(t, "data_ptr"):
        if not t.is_contiguous():
            raise ValueError("tensor arguments must be contiguous")
        return t.data_ptr()
    return int(t)


class Store:
    """Owning handle of an is_store_t."""

    def __init__(self, handle: int, config: StoreConfig, device: int):
        self.handle = handle
        self.config = config
        self.device = device

    def destroy(self) -> None:
        if self.handle:
            _check(_lib.load().is_store_destroy(c_void_p(self.handle)))
            self.handle = 0

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.destroy()


def make_config(**kw) -> StoreConfig:
    c = StoreConfig()
    for k, v in kw.items():
        if k in ("kv_dtype", "emb_dtype") and isinstance(v, str):
            v = DTYPE_CODES[v]
        elif k == "kv_placement" and isinstance(v, str):
            v = {"device": 0, "host": 1}[v]
        setattr(c, k, int(v))
    return c


def make_rope(theta: float, style: int = 0, scaling: int = 0, factor: float = 1.0,
              low_freq_factor: float = 1.0, high_freq_factor: float = 1.0,
              original_max_pos: int = 0) -> RopeParams:
    return RopeParams(theta, style, scaling, factor, low_freq_factor, high_freq_factor,
                      original_max_pos)


def make_cache_desc(block_size: int, num_blocks: int, dtype, k_scale: float = 1.0,
                    v_scale: float = 1.0) -> CacheDesc:
    """dtype "e4m3" (IS_FP8_E4M3): an FP8 cache holding K / k_scale and V / v_scale."""
    return CacheDesc(block_size, num_blocks, DTYPE_CODES[dtype] if isinstance(dtype, str) else dtype,
                     k_scale, v_scale)


def is_store_create(config: StoreConfig, device: int = 0, stream=None) -> Store:
    h = c_void_p()
    _check(_lib.load().is_store_create(byref(config), device, _stream(stream), byref(h)))
    return Store(h.value, config, device)


def is_store_destroy(store: Store) -> None:
    store.destroy()


def is_store_add_facts(store: Store, user: int, lengths, k_pre_rope, v, emb, stream=None) -> np.ndarray:
    lengths = np.ascontiguousarray(lengths, dtype=np.int32)
    ids = np.empty(len(lengths), dtype=np.int64)
    _check(_lib.load().is_store_add_facts(
        c_void_p(store.handle), int(user), len(lengths),
        lengths.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), _ptr(k_pre_rope), _ptr(v),
        _ptr(emb), ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), _stream(stream)))
    return ids


def is_store_capture_begin(store: Store, user: int, window, lengths, emb, stream=None) -> None:
    """Open a Context-Window Encoding capture of len(lengths) facts of ``user``."""
    window = np.ascontiguousarray(window, dtype=np.int32)
    lengths = np.ascontiguousarray(lengths, dtype=np.int32)
    if window.shape != lengths.shape:
        raise ValueError("window and lengths must have one entry per fact")
    _check(_lib.load().is_store_capture_begin(
        c_void_p(store.handle), int(user), len(lengths),
        window.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
        lengths.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), _ptr(emb), _stream(stream)))


def is_store_capture_layer(store: Store, layer: int, k_pre_rope, v, stream=None) -> None:
    _check(_lib.load().is_store_capture_layer(c_void_p(store.handle), int(layer), _ptr(k_pre_rope), _ptr(v),
                                              _stream(stream)))


def is_store_capture_end(store: Store, n: int, stream=None) -> np.ndarray:
    ids = np.empty(n, dtype=np.int64)
    _check(_lib.load().is_store_capture_end(c_void_p(store.handle),
                                            ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                            _stream(stream)))
    return ids


def is_store_capture_abort(store: Store) -> None:
    _check(_lib.load().is_store_capture_abort(c_void_p(store.handle)))


def is_store_info(store: Store) -> dict:
    info = StoreInfo()
    _check(_lib.load().is_store_info(c_void_p(store.handle), byref(info)))
    return {name: getattr(info, name) for name, _ in StoreInfo._fields_}


def is_retrieve_topk(store: Store, users, q_emb, k: int, ids_out, scores_out, stream=None) -> None:
    _check(_lib.load().is_retrieve_topk(
        c_void_p(store.handle), int(users.shape[0]), _ptr(users), _ptr(q_emb), int(k),
        _ptr(ids_out), _ptr(scores_out), _stream(stream)))


def is_inject(store: Store, fact_ids, n_ids, seg_start, rope: RopeParams, block_table,
              cache: CacheDesc, kv_cache, users=None, seg_len_out=None, slot_mapping_out=None,
              stream=None) -> None:
    R, stride = int(fact_ids.shape[0]), int(fact_ids.shape[1])
    _check(_lib.load().is_inject(
        c_void_p(store.handle), R, _ptr(fact_ids), _ptr(n_ids), stride, _ptr(users),
        _ptr(seg_start), byref(rope), _ptr(block_table), int(block_table.shape[1]), byref(cache),
        _ptr(kv_cache), _ptr(seg_len_out), _ptr(slot_mapping_out), _stream(stream)))


def is_inject_layer(store: Store, layer: int, R: int, seg_start, rope: RopeParams, block_table,
                    cache: CacheDesc, layer_cache, fact_ids=None, n_ids=None, users=None,
                    seg_len_out=None, slot_mapping_out=None, stream=None) -> None:
    """One layer into its own cache tensor; fact_ids=None reuses the last plan."""
    stride = int(fact_ids.shape[1]) if fact_ids is not None else 0
    _check(_lib.load().is_inject_layer(
        c_void_p(store.handle), int(layer), int(R), _ptr(fact_ids), _ptr(n_ids), stride, _ptr(users),
        _ptr(seg_start), byref(rope), _ptr(block_table), int(block_table.shape[1]), byref(cache),
        _ptr(layer_cache), _ptr(seg_len_out), _ptr(slot_mapping_out), _stream(stream)))


def is_inject_layers(store: Store, layer0: int, R: int, seg_start, rope: RopeParams, block_table,
                     cache: CacheDesc, layer_caches, fact_ids=None, n_ids=None, users=None,
                     seg_len_out=None, slot_mapping_out=None, stream=None) -> None:
    """Layers layer0 .. layer0 + len(layer_caches) - 1 in one launch, each into its
    own cache tensor (a list of device tensors); fact_ids=None reuses the last plan."""
    n = len(layer_caches)
    ptrs = (c_void_p * max(n, 1))(*[_ptr(t) for t in layer_caches])
    stride = int(fact_ids.shape[1]) if fact_ids is not None else 0
    _check(_lib.load().is_inject_layers(
        c_void_p(store.handle), int(layer0), n, int(R), _ptr(fact_ids), _ptr(n_ids), stride, _ptr(users),
        _ptr(seg_start), byref(rope), _ptr(block_table), int(block_table.shape[1]), byref(cache),
        ctypes.cast(ptrs, c_void_p), _ptr(seg_len_out), _ptr(slot_mapping_out), _stream(stream)))


def is_retrieve_and_inject(store: Store, users, q_emb, k: int, seg_start, rope: RopeParams,
                           block_table, cache: CacheDesc, kv_cache, ids_out=None, scores_out=None,
                           seg_len_out=None, slot_mapping_out=None, stream=None) -> None:
    _check(_lib.load().is_retrieve_and_inject(
        c_void_p(store.handle), int(users.shape[0]), _ptr(users), _ptr(q_emb), int(k),
        _ptr(seg_start), byref(rope), _ptr(block_table), int(block_table.shape[1]), byref(cache),
        _ptr(kv_cache), _ptr(ids_out), _ptr(scores_out), _ptr(seg_len_out),
        _ptr(slot_mapping_out), _stream(stream)))


def prepare_retrieve_and_inject(store: Store, users, q_emb, k: int, seg_start, rope: RopeParams,
                                block_table, cache: CacheDesc, kv_cache, ids_out=None, scores_out=None,
                                seg_len_out=None, slot_mapping_out=None, stream=None):
    """is_retrieve_and_inject with every argument marshalled once: returns a
    callable that issues the call on the same buffers (whose contents may
    change between calls) and raises ISError on a non-OK status.  For serving
    loops that reuse their buffers."""
    fn = _lib.load().is_retrieve_and_inject
    args = (c_void_p(store.handle), int(users.shape[0]), _ptr(users), _ptr(q_emb), int(k), _ptr(seg_start),
            byref(rope), _ptr(block_table), int(block_table.shape[1]), byref(cache), _ptr(kv_cache),
            _ptr(ids_out), _ptr(scores_out), _ptr(seg_len_out), _ptr(slot_mapping_out), _stream(stream))
    keep = (rope, cache)                      # the structs must outlive the callable

    def call():
        st = fn(*args)
        if st != _lib.IS_OK:
            _check(st)
        return keep is not None
    return call


def _hptr(a) -> int | None:
    """Address of a host array (numpy array or CPU tensor), which must be contiguous."""
    if a is None:
        return None
    if hasattr(a, "data_ptr"):
        if a.is_cuda or not a.is_contiguous():
            raise ValueError("host tensor arguments must be contiguous CPU tensors")
        return a.data_ptr()
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("host array arguments must be C-contiguous")
    return a.ctypes.data


class HostCall:
    """A prepared is_retrieve_and_inject_host (is_host_call_prepare): the
    arguments are bound once, and each call runs the step on the buffers'
    current contents through is_host_call_run, one pointer argument."""

    def __init__(self, handle: int, keep):
        self._lib = _lib.load()
        self._handle = c_void_p(handle)
        self._run = self._lib.is_host_call_run
        self._keep = keep                     # the bound arrays must outlive the handle

    def __call__(self) -> None:
        st = self._run(self._handle)
        if st != _lib.IS_OK:
            _check(st)

    def close(self) -> None:
        if self._handle:
            self._lib.is_host_call_destroy(self._handle)
            self._handle = c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:      # interpreter shutdown
            pass


def prepare_retrieve_and_inject_host(store: Store, users, q_emb, k: int, seg_start, rope: RopeParams,
                                     block_table, cache: CacheDesc, kv_cache, ids_out=None, scores_out=None,
                                     seg_len_out=None, stream=None) -> HostCall:
    """is_retrieve_and_inject_host with every argument bound once
    (is_host_call_prepare): inputs and outputs are host arrays (numpy or CPU
    tensors; contents may change between calls), kv_cache a device tensor.
    Returns a callable; each call is synchronous and raises ISError on a
    non-OK status."""
    out = c_void_p()
    _check(_lib.load().is_host_call_prepare(
        c_void_p(store.handle), int(users.shape[0]), _hptr(users), _hptr(q_emb), int(k), _hptr(seg_start),
        byref(rope), _hptr(block_table), int(block_table.shape[1]), byref(cache), _ptr(kv_cache),
        _hptr(ids_out), _hptr(scores_out), _hptr(seg_len_out), _stream(stream), byref(out)))
    return HostCall(out.value, (store, users, q_emb, seg_start, block_table, ids_out, scores_out, seg_len_out,
                                kv_cache))


def is_retrieve_and_inject_host(store: Store, users, q_emb, k: int, seg_start, rope: RopeParams, block_table,
                                cache: CacheDesc, kv_cache, ids_out=None, scores_out=None, seg_len_out=None,
                                stream=None) -> None:
    """The fused call with host inputs and outputs (see the prepared form)."""
    prepare_retrieve_and_inject_host(store, users, q_emb, k, seg_start, rope, block_table, cache, kv_cache,
                                     ids_out, scores_out, seg_len_out, stream)()


def is_inject_noalloc(kv_arena, arena_tokens: int, fact_tok, fact_len, max_fact_len: int,
                      num_layers: int, num_kv_heads: int, head_dim: int, kv_dtype, fact_ids, n_ids,
                      seg_start, rope: RopeParams, block_table, cache: CacheDesc, kv_cache, status_out,
                      seg_len_out=None, slot_mapping_out=None, stream=None) -> None:
    """Store-free injection from a caller-owned token-major K/V arena of
    ``arena_tokens`` tokens; the library allocates nothing (its plan scratch
    is a static device array)."""
    dt = DTYPE_CODES[kv_dtype] if isinstance(kv_dtype, str) else int(kv_dtype)
    R, stride = int(fact_ids.shape[0]), int(fact_ids.shape[1])
    _check(_lib.load().is_inject_noalloc(
        _ptr(kv_arena), int(arena_tokens), _ptr(fact_tok), _ptr(fact_len), int(fact_len.shape[0]),
        int(max_fact_len), int(num_layers), int(num_kv_heads), int(head_dim), dt, R, _ptr(fact_ids), _ptr(n_ids),
        stride, _ptr(seg_start), byref(rope), _ptr(block_table), int(block_table.shape[1]),
        byref(cache), _ptr(kv_cache), _ptr(seg_len_out), _ptr(slot_mapping_out), _ptr(status_out),
        _stream(stream)))


def is_get_status(store: Store, stream=None) -> int:
    """Device status bits since the last read (cleared).  Raises only on CUDA errors."""
    bits = c_uint32()
    st = _lib.load().is_get_status(c_void_p(store.handle), _stream(stream), byref(bits))
    if st not in (_lib.IS_OK, 6, 7):
        _check(st)
    return int(bits.value)


def is_rope_frequencies(rope: RopeParams, head_dim: int) -> np.ndarray:
    out = np.empty(head_dim // 2, dtype=np.float64)
    _check(_lib.load().is_rope_frequencies(byref(rope), int(head_dim),
                                           out.ctypes.data_as(ctypes.POINTER(ctypes.c_double))))
    return out


def is_set_retrieval_mode(store: Store, mode: int) -> None:
    _check(_lib.load().is_set_retrieval_mode(c_void_p(store.handle), int(mode)))


def is_set_wait_budget(store: Store, budget_ns: int) -> None:
    _check(_lib.load().is_set_wait_budget(c_void_p(store.handle), int(budget_ns)))


def is_set_timing(store: Store, enable: bool) -> None:
    _check(_lib.load().is_set_timing(c_void_p(store.handle), 1 if enable else 0))


def is_get_timing(store: Store, stage: int) -> tuple[float, int]:
    ms, n = c_double(), c_int64()
    _check(_lib.load().is_get_timing(c_void_p(store.handle), int(stage), byref(ms), byref(n)))
    return ms.value, n.value


def is_reset_timing(store: Store) -> None:
    _check(_lib.load().is_reset_timing(c_void_p(store.handle)))
