"""ctypes binding of ``libqa.so`` -- the C ABI of ``include/qa.h``, same names.

Argument marshalling only: tensors are passed as device pointers (torch
tensors or plain integers), host arrays as int32 buffers, streams as
cudaStream_t handles.  Every step of the path runs in the library's kernels.
Importing this module loads the library and raises ImportError if it has not
been built; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

LIB_PATH = _build.LIB

QA_OK = 0
STATUS_NAMES = {0: "QA_OK", 1: "QA_ERR_INVALID_ARG", 2: "QA_ERR_UNSUPPORTED_SHAPE",
                3: "QA_ERR_ALIGNMENT", 4: "QA_ERR_CAPACITY", 5: "QA_ERR_STATE", 6: "QA_ERR_CUDA",
                7: "QA_ERR_DEVICE_TIMEOUT", 8: "QA_ERR_DEVICE_BOUNDS"}
KERNELS = ("norm_rope_append", "prefill_attn", "decode_attn", "reset")


class QaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({qa_status_str(status)})")


class qa_config(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int), ("max_batch", ctypes.c_int),
                ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("capacity", ctypes.c_int),
                ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float)]


_vp = ctypes.c_void_p
_i32p = ctypes.POINTER(ctypes.c_int32)
_u64p = ctypes.POINTER(ctypes.c_uint64)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_i64p = ctypes.POINTER(ctypes.c_int64)

# name -> (restype, argtypes); every entry point declared in include/qa.h
SIGNATURES = {
    "qa_cache_alloc": (ctypes.c_int, [ctypes.POINTER(qa_config), ctypes.POINTER(_vp)]),
    "qa_cache_free": (ctypes.c_int, [_vp]),
    "qa_cache_reset": (ctypes.c_int, [_vp, _vp]),
    "qa_prefill": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.c_int, _i32p, _vp, _vp, _vp, _vp, _vp,
                                  _vp, _vp]),
    "qa_decode_step": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp, _vp, _vp,
                                      _vp, _vp]),
    "qa_decode_step_device_lengths": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp,
                                                     _vp, _vp, _vp, _vp]),
    "qa_cache_sync_lengths": (ctypes.c_int, [_vp, ctypes.c_int, _vp]),
    "qa_cache_set_window": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.c_int]),
    "qa_cache_set_decode_overlap": (ctypes.c_int, [_vp, ctypes.c_int]),
    "qa_cache_view": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                     ctypes.POINTER(_vp), _i64p]),
    "qa_cache_set_lengths": (ctypes.c_int, [_vp, ctypes.c_int, _i32p, _vp]),
    "qa_cache_lengths": (ctypes.c_int, [_vp, ctypes.c_int, _i32p]),
    "qa_prefill_transform": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.c_int, _i32p, _vp, _vp, _vp,
                                            _vp, _vp, _vp, _vp]),
    "qa_get_device_error": (ctypes.c_int, [_vp, _u32p]),
    "qa_stats": (ctypes.c_int, [_vp, _u64p]),
    "qa_memory_info": (ctypes.c_int, [_vp, _u64p, _u64p]),
    "qa_decode_splits": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.c_int]),
    "qa_decode_step_noalloc": (ctypes.c_int, [ctypes.POINTER(qa_config), ctypes.c_int, _i32p, _vp,
                                              _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "qa_noalloc_get_device_error": (ctypes.c_int, [_u32p, _vp]),
    "qa_prefill_attend": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.c_int, _i32p, _vp, _vp, _vp]),
    "qa_debug_arm_wait_timeout": (ctypes.c_int, [ctypes.c_int, ctypes.c_uint32]),
    "qa_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "qa_abi_version": (ctypes.c_int, []),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                          "(the CUDA path has no fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _i32(values):
    arr = (ctypes.c_int32 * max(1, len(values)))(*[int(v) for v in values])
    return arr


def _check(st: int, what: str) -> None:
    if st != QA_OK:
        raise QaError(st, what)


def qa_status_str(status: int) -> str:
    return lib.qa_status_str(status).decode()


def qa_abi_version() -> int:
    return lib.qa_abi_version()


def qa_cache_alloc(num_layers, max_batch, n_q_heads, n_kv_heads, head_dim, capacity,
                   rope_theta=1e6, rms_eps=1e-6) -> int:
    cfg = qa_config(num_layers, max_batch, n_q_heads, n_kv_heads, head_dim, capacity, rope_theta,
                    rms_eps)
    h = _vp()
    _check(lib.qa_cache_alloc(ctypes.byref(cfg), ctypes.byref(h)), "qa_cache_alloc")
    return h.value


def qa_cache_free(cache) -> None:
    _check(lib.qa_cache_free(cache), "qa_cache_free")


def qa_cache_reset(cache, stream=None) -> None:
    _check(lib.qa_cache_reset(cache, _stream(stream)), "qa_cache_reset")


def qa_prefill(cache, layer, prompt_lens, q, k, v, q_norm_w, k_norm_w, out, stream=None) -> None:
    _check(lib.qa_prefill(cache, layer, len(prompt_lens), _i32(prompt_lens), _ptr(q), _ptr(k),
                          _ptr(v), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(out), _stream(stream)),
           "qa_prefill")


def qa_prefill_transform(cache, layer, prompt_lens, q, k, v, q_norm_w, k_norm_w, qprime_out,
                         stream=None) -> None:
    _check(lib.qa_prefill_transform(cache, layer, len(prompt_lens), _i32(prompt_lens), _ptr(q),
                                    _ptr(k), _ptr(v), _ptr(q_norm_w), _ptr(k_norm_w),
                                    _ptr(qprime_out), _stream(stream)),
           "qa_prefill_transform")


def qa_decode_step(cache, layer, batch, q, k, v, q_norm_w, k_norm_w, out, stream=None) -> None:
    _check(lib.qa_decode_step(cache, layer, batch, _ptr(q), _ptr(k), _ptr(v), _ptr(q_norm_w),
                              _ptr(k_norm_w), _ptr(out), _stream(stream)),
           "qa_decode_step")


def qa_decode_step_device_lengths(cache, layer, batch, q, k, v, q_norm_w, k_norm_w, out,
                                  stream=None) -> None:
    _check(lib.qa_decode_step_device_lengths(cache, layer, batch, _ptr(q), _ptr(k), _ptr(v),
                                             _ptr(q_norm_w), _ptr(k_norm_w), _ptr(out),
                                             _stream(stream)),
           "qa_decode_step_device_lengths")


def qa_cache_set_window(cache, layer, window) -> None:
    _check(lib.qa_cache_set_window(cache, layer, window), "qa_cache_set_window")


def qa_cache_set_decode_overlap(cache, launches) -> None:
    _check(lib.qa_cache_set_decode_overlap(cache, launches), "qa_cache_set_decode_overlap")


def qa_cache_sync_lengths(cache, layer, stream=None) -> None:
    _check(lib.qa_cache_sync_lengths(cache, layer, _stream(stream)), "qa_cache_sync_lengths")


def qa_decode_step_noalloc(cfg: qa_config, positions, k_cache, v_cache, q, k, v, q_norm_w,
                           k_norm_w, out, stream=None) -> None:
    """Allocation-free decode step on caller-owned cache memory (see include/qa.h)."""
    _check(lib.qa_decode_step_noalloc(ctypes.byref(cfg), len(positions), _i32(positions),
                                      _ptr(k_cache), _ptr(v_cache), _ptr(q), _ptr(k), _ptr(v),
                                      _ptr(q_norm_w), _ptr(k_norm_w), _ptr(out), _stream(stream)),
           "qa_decode_step_noalloc")


def qa_noalloc_get_device_error(stream=None):
    """(status, raw error word) of the allocation-free step; reading clears the word."""
    w = ctypes.c_uint32()
    st = lib.qa_noalloc_get_device_error(ctypes.byref(w), _stream(stream))
    return st, w.value


def qa_prefill_attend(cache, layer, prompt_lens, qprime, out, stream=None) -> None:
    _check(lib.qa_prefill_attend(cache, layer, len(prompt_lens), _i32(prompt_lens), _ptr(qprime),
                                 _ptr(out), _stream(stream)),
           "qa_prefill_attend")


def qa_debug_arm_wait_timeout(kernel: int, wait_us: int) -> None:
    _check(lib.qa_debug_arm_wait_timeout(kernel, wait_us), "qa_debug_arm_wait_timeout")


def qa_cache_view(cache, layer):
    """(k_ptr, v_ptr, lens_ptr, strides[4]) of one layer."""
    k, v, lens = _vp(), _vp(), _vp()
    strides = (ctypes.c_int64 * 4)()
    _check(lib.qa_cache_view(cache, layer, ctypes.byref(k), ctypes.byref(v), ctypes.byref(lens),
                             strides), "qa_cache_view")
    return k.value, v.value, lens.value, list(strides)


def qa_cache_set_lengths(cache, layer, lens, stream=None) -> None:
    _check(lib.qa_cache_set_lengths(cache, layer, _i32(lens), _stream(stream)),
           "qa_cache_set_lengths")


def qa_cache_lengths(cache, layer, max_batch):
    buf = (ctypes.c_int32 * max_batch)()
    _check(lib.qa_cache_lengths(cache, layer, buf), "qa_cache_lengths")
    return list(buf)


def qa_get_device_error(cache):
    """(status, raw error word); reading clears the word."""
    w = ctypes.c_uint32()
    st = lib.qa_get_device_error(cache, ctypes.byref(w))
    return st, w.value


def qa_stats(cache) -> dict:
    buf = (ctypes.c_uint64 * len(KERNELS))()
    _check(lib.qa_stats(cache, buf), "qa_stats")
    return dict(zip(KERNELS, list(buf)))


def qa_memory_info(cache):
    kv, scr = ctypes.c_uint64(), ctypes.c_uint64()
    _check(lib.qa_memory_info(cache, ctypes.byref(kv), ctypes.byref(scr)), "qa_memory_info")
    return kv.value, scr.value


def qa_decode_splits(cache, layer, batch) -> int:
    return lib.qa_decode_splits(cache, layer, batch)


class _DeviceArray:
    """Zero-copy view of library-owned device memory for torch.as_tensor."""

    def __init__(self, ptr: int, shape, typestr: str, strides_bytes=None):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (ptr, False), "version": 3,
                                         "strides": strides_bytes}


def cache_tensors(cache, layer, max_batch, n_kv_heads, capacity, head_dim):
    """torch views (K, V as bf16 [max_batch, Hkv, cap, D], lens as int32 [max_batch])."""
    import torch
    k, v, lens, _ = qa_cache_view(cache, layer)
    shape = (max_batch, n_kv_heads, capacity, head_dim)
    kt = torch.as_tensor(_DeviceArray(k, shape, "<i2"), device="cuda").view(torch.bfloat16)
    vt = torch.as_tensor(_DeviceArray(v, shape, "<i2"), device="cuda").view(torch.bfloat16)
    lt = torch.as_tensor(_DeviceArray(lens, (max_batch,), "<i4"), device="cuda")
    return kt, vt, lt
