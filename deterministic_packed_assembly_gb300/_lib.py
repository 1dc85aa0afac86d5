"""ctypes binding of ``libnspack.so`` (declared in ``include/nspack.h``).

Argument marshalling only: every step of the packing path runs in the
library's CUDA kernels.  There is no fallback: if the library is missing or
fails to load, importing this module raises.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libnspack.so")

NS_OK = 0
NS_ERR_INVALID_ARG = -1
NS_ERR_CUDA = -2
NS_ERR_OOM = -3
NS_ERR_EXHAUSTED = -4
NS_ERR_HORIZON = -5
NS_ERR_BAD_INPUT = -6
NS_ERR_DEVICE = -7
NS_PACK_DRAIN = 1
NS_PACK_HELDOUT = 2
NS_PACK_SHUFFLE_ROWS = 4
NS_PACK_WRAP = 8
NS_PACK_HOST_CORPUS = 16
NS_PACK_ORDERED_FREE = 32
NS_MAX_T = 1 << 24
NS_MAX_TOKENS = 1 << 47

ns_alloc_fn = C.CFUNCTYPE(C.c_void_p, C.c_size_t, C.c_void_p)
ns_free_fn = C.CFUNCTYPE(None, C.c_void_p, C.c_void_p)


class ns_pack_config(C.Structure):
    _fields_ = [
        ("tokens", C.c_void_p),
        ("n_tokens", C.c_uint64),
        ("doc_offsets", C.c_void_p),
        ("loss_start", C.c_void_p),
        ("n_docs", C.c_uint32),
        ("n_sources", C.c_uint32),
        ("n_streams", C.c_uint32),
        ("T", C.c_uint32),
        ("stream_doc_begin", C.c_void_p),
        ("stream_source", C.c_void_p),
        ("source_weight", C.c_void_p),
        ("stream_weight", C.c_void_p),
        ("source_heldout_bp", C.c_void_p),
        ("seed", C.c_uint64),
        ("hash_key", C.c_uint64),
        ("B", C.c_uint32),
        ("max_steps", C.c_uint32),
        ("flags", C.c_uint32),
        ("pad_id", C.c_int32),
        ("window_segment", C.c_uint32),
        ("n_pieces", C.c_uint32),
        ("piece_begin", C.c_void_p),
        ("piece_B", C.c_void_p),
        ("piece_source_weight", C.c_void_p),
        ("piece_stream_weight", C.c_void_p),
        ("len_bucket", C.c_uint32),
        ("cuda_stream", C.c_void_p),
        ("alloc", ns_alloc_fn),
        ("free", ns_free_fn),
        ("alloc_user", C.c_void_p),
    ]


class ns_pack_out(C.Structure):
    _fields_ = [
        ("tokens", C.c_void_p),
        ("pos", C.c_void_p),
        ("doc", C.c_void_p),
        ("mask", C.c_void_p),
        ("row_fp", C.c_void_p),
        ("row_learned", C.c_void_p),
        ("row_len", C.c_void_p),
    ]


class ns_pack_info_t(C.Structure):
    _fields_ = [
        ("valid_steps", C.c_uint32),
        ("max_steps", C.c_uint32),
        ("n_streams", C.c_uint32),
        ("T", C.c_uint32),
        ("B", C.c_uint32),
        ("levels", C.c_uint32),
        ("order_digest", C.c_uint64),
        ("n_pieces", C.c_uint64),
        ("table_bytes", C.c_uint64),
        ("init_launches", C.c_uint32),
        ("init_passes", C.c_uint32),
        ("host_bytes", C.c_uint64),
        ("hashed_tokens", C.c_uint64),
        ("hashed_docs", C.c_uint64),
        ("hash_ns", C.c_uint64),
    ]


# Every symbol the header declares, for the load check.
SYMBOLS = ("ns_pack_init", "ns_pack_step", "ns_pack_fingerprint", "ns_pack_batch_fp",
           "ns_pack_step_learned", "ns_pack_info", "ns_pack_stream_windows",
           "ns_pack_quota_table", "ns_pack_check", "ns_pack_free", "ns_pack_strerror",
           "ns_pack_quota_noalloc", "ns_pack_probe_hash_terms")


def _load() -> C.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -c \"import __graft_entry__ as g; g.build()\"` "
            "(there is no CPU fallback)")
    L = C.CDLL(LIB_PATH)
    vp, u32, u64, i32 = C.c_void_p, C.c_uint32, C.c_uint64, C.c_int
    L.ns_pack_init.restype = i32
    L.ns_pack_init.argtypes = [C.POINTER(ns_pack_config), C.POINTER(vp)]
    L.ns_pack_step.restype = i32
    L.ns_pack_step.argtypes = [vp, u32, u32, u32, u32, C.POINTER(ns_pack_out), vp]
    L.ns_pack_fingerprint.restype = i32
    L.ns_pack_fingerprint.argtypes = [vp, vp, u32, C.POINTER(C.c_uint64), vp]
    L.ns_pack_batch_fp.restype = i32
    L.ns_pack_batch_fp.argtypes = [vp, vp, u32, u32, vp, vp]
    L.ns_pack_info.restype = i32
    L.ns_pack_info.argtypes = [vp, C.POINTER(ns_pack_info_t)]
    L.ns_pack_step_learned.restype = i32
    L.ns_pack_step_learned.argtypes = [vp, vp, u32, u32, vp, vp]
    L.ns_pack_stream_windows.restype = i32
    L.ns_pack_stream_windows.argtypes = [vp, vp, vp]
    L.ns_pack_quota_table.restype = i32
    L.ns_pack_quota_table.argtypes = [vp, vp, vp]
    L.ns_pack_check.restype = i32
    L.ns_pack_check.argtypes = [vp]
    L.ns_pack_free.restype = None
    L.ns_pack_free.argtypes = [vp]
    L.ns_pack_strerror.restype = C.c_char_p
    L.ns_pack_strerror.argtypes = [i32]
    L.ns_pack_probe_hash_terms.restype = i32
    L.ns_pack_probe_hash_terms.argtypes = [u32, u32, vp, vp]
    L.ns_pack_quota_noalloc.restype = i32
    L.ns_pack_quota_noalloc.argtypes = [vp, u32, vp, vp, u32, u32, u32, vp, vp, vp]
    return L


lib = _load()


class NsPackError(RuntimeError):
    def __init__(self, code: int, what: str):
        msg = lib.ns_pack_strerror(code).decode()
        super().__init__(f"{what}: {msg} ({code})")
        self.code = code


def check(code: int, what: str) -> None:
    if code != NS_OK:
        raise NsPackError(code, what)


# ---- the C ABI under the same names ------------------------------------------
def ns_pack_init(cfg: ns_pack_config) -> C.c_void_p:
    h = C.c_void_p()
    check(lib.ns_pack_init(C.byref(cfg), C.byref(h)), "ns_pack_init")
    return h


def ns_pack_step(ctx, step0: int, n_steps: int, row_begin: int, row_end: int,
                 out: ns_pack_out, stream: int | None = None) -> None:
    check(lib.ns_pack_step(ctx, step0, n_steps, row_begin, row_end, C.byref(out), stream),
          f"ns_pack_step(step0={step0}, n_steps={n_steps}, rows=[{row_begin},{row_end}))")


def ns_pack_fingerprint(ctx, row_fp_ptr: int, n_rows: int, stream: int | None = None) -> int:
    v = C.c_uint64()
    check(lib.ns_pack_fingerprint(ctx, row_fp_ptr, n_rows, C.byref(v), stream),
          "ns_pack_fingerprint")
    return v.value


def ns_pack_batch_fp(ctx, row_fp_ptr: int, n_steps: int, n_rows: int, out_ptr: int,
                     stream: int | None = None) -> None:
    check(lib.ns_pack_batch_fp(ctx, row_fp_ptr, n_steps, n_rows, out_ptr, stream),
          "ns_pack_batch_fp")


def ns_pack_step_learned(ctx, row_learned_ptr: int, n_steps: int, n_rows: int, out_ptr: int,
                         stream: int | None = None) -> None:
    check(lib.ns_pack_step_learned(ctx, row_learned_ptr, n_steps, n_rows, out_ptr, stream),
          "ns_pack_step_learned")


def ns_pack_info(ctx) -> dict:
    info = ns_pack_info_t()
    check(lib.ns_pack_info(ctx, C.byref(info)), "ns_pack_info")
    return {name: getattr(info, name) for name, _ in ns_pack_info_t._fields_}


def ns_pack_stream_windows(ctx, n_streams: int):
    import numpy as np
    w = np.zeros(n_streams, np.uint64)
    c = np.zeros(n_streams, np.uint8)
    check(lib.ns_pack_stream_windows(ctx, w.ctypes.data, c.ctypes.data), "ns_pack_stream_windows")
    return w, c.astype(bool)


def ns_pack_quota_table(ctx, max_steps: int, n_streams: int):
    import numpy as np
    q = np.zeros((max_steps, n_streams), np.int32)
    cum = np.zeros((max_steps + 1, n_streams), np.int32)
    check(lib.ns_pack_quota_table(ctx, q.ctypes.data, cum.ctypes.data), "ns_pack_quota_table")
    return q, cum


def ns_pack_check(ctx) -> None:
    check(lib.ns_pack_check(ctx), "ns_pack_check")


def ns_pack_free(ctx) -> None:
    lib.ns_pack_free(ctx)


def ns_pack_quota_noalloc(source_weight, stream_source, stream_weight, B: int, max_steps: int,
                          quota_ptr: int, cum_ptr: int, stream: int | None = None) -> None:
    """Quota tables of a recipe into caller-owned device buffers, with no
    device allocation (for callers that cannot call cudaMalloc)."""
    import numpy as np
    sw = np.ascontiguousarray(source_weight, dtype=np.uint32)
    ss = np.ascontiguousarray(stream_source, dtype=np.uint32)
    tw = np.ascontiguousarray(stream_weight, dtype=np.uint32)
    check(lib.ns_pack_quota_noalloc(sw.ctypes.data, sw.size, ss.ctypes.data, tw.ctypes.data,
                                    ss.size, B, max_steps, quota_ptr, cum_ptr, stream),
          "ns_pack_quota_noalloc")


def ns_pack_strerror(code: int) -> str:
    return lib.ns_pack_strerror(code).decode()


def ns_pack_probe_hash_terms(blocks: int, terms_per_thread: int, sum_dev: int,
                             stream: int = 0) -> None:
    """Launch the register-only loop of the held-out hash's term (see
    include/nspack_probe.h); adds its sum to the device u64 at sum_dev."""
    check(lib.ns_pack_probe_hash_terms(blocks, terms_per_thread, sum_dev, stream or None),
          "ns_pack_probe_hash_terms")
