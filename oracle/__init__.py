"""CPU oracle of deterministic packed assembly -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg (``bench.py --impl reference`` and its ``cpu_baseline`` figure)
may import this package.  The product path (the CUDA library and its Python
binding) never imports, links or calls it, and the two share no code.

``oracle.c`` is a plain sequential C statement of the method; this module
compiles it with gcc into ``liboracle.so`` beside it and marshals numpy
arrays through ctypes.  Every function here only moves arguments: the
arithmetic is in ``oracle.c``.

Parity status: every function is pinned by tests that do not re-derive it --
published SplitMix64 outputs, a hand-worked packing example and quota
example, brute-force properties on tiny inputs (Feistel bijectivity and its
inverse, greedy maximality, exactly-once coverage, quota bounds and the
exhaustive subset choice), binomial bounds on the held-out rate, the row
fingerprint's keys recovered through the inverse against hand-worked
special cases, and the order digest against the fold of the items rebuilt
from the pinned read-outs.  The pages
print no worked values for this path, so page-level parity of the readings
(what is hashed, the shuffle's construction, the fingerprint) is unpinned.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

OK, INVALID_ARG, OOM, EXHAUSTED, HORIZON, BAD_INPUT = 0, -1, -3, -4, -5, -6
GOLDEN = 0x9E3779B97F4A7C15
M64 = (1 << 64) - 1


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` (plain C11, single-threaded) into ``liboracle.so``."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared",
                               "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


class _Config(C.Structure):
    _fields_ = [
        ("tokens", C.c_void_p), ("n_tokens", C.c_uint64),
        ("doc_offsets", C.c_void_p), ("loss_start", C.c_void_p),
        ("n_docs", C.c_uint32), ("n_sources", C.c_uint32), ("n_streams", C.c_uint32),
        ("T", C.c_uint32),
        ("stream_doc_begin", C.c_void_p), ("stream_source", C.c_void_p),
        ("source_weight", C.c_void_p), ("stream_weight", C.c_void_p),
        ("source_heldout_bp", C.c_void_p),
        ("seed", C.c_uint64), ("hash_key", C.c_uint64),
        ("B", C.c_uint32), ("max_steps", C.c_uint32), ("drain", C.c_uint32),
        ("pad_id", C.c_int32),
        ("heldout_only", C.c_uint32),
        ("window_segment", C.c_uint32),
        ("shuffle_rows", C.c_uint32),
        ("n_pieces", C.c_uint32),
        ("piece_begin", C.c_void_p), ("piece_B", C.c_void_p),
        ("piece_source_weight", C.c_void_p), ("piece_stream_weight", C.c_void_p),
        ("wrap", C.c_uint32), ("len_bucket", C.c_uint32),
    ]


_lib: Optional[C.CDLL] = None


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        L = C.CDLL(build())
        u64, u32, vp, i64 = C.c_uint64, C.c_uint32, C.c_void_p, C.c_int64
        L.or_splitmix64.restype = u64
        L.or_splitmix64.argtypes = [u64]
        L.or_doc_hash.restype = u64
        L.or_doc_hash.argtypes = [vp, u64, u64]
        L.or_is_heldout.restype = C.c_int
        L.or_is_heldout.argtypes = [u64, u32]
        L.or_feistel_bits.restype = u32
        L.or_feistel_bits.argtypes = [u64]
        L.or_feistel_round_key.restype = u64
        L.or_feistel_round_key.argtypes = [u64, u32, u32]
        L.or_feistel_encrypt.restype = u64
        L.or_feistel_encrypt.argtypes = [vp, u32, u64]
        L.or_window_of_rank.restype = u64
        L.or_window_of_rank.argtypes = [u64, u32, u32, u64, u64]
        L.or_row_of_slot.restype = u32
        L.or_row_of_slot.argtypes = [u64, u32, u32, u32]
        L.or_feistel_pi.restype = u64
        L.or_feistel_pi.argtypes = [u64, u32, u64, u64]
        L.or_apportion.restype = C.c_int
        L.or_apportion.argtypes = [u32, vp, vp, i64, i64, vp]
        L.or_build.restype = C.c_int
        L.or_build.argtypes = [C.POINTER(_Config), C.POINTER(vp)]
        L.or_free.restype = None
        L.or_free.argtypes = [vp]
        L.or_rows.restype = C.c_int
        L.or_rows.argtypes = [vp, u32, u32, u32, vp, vp, vp, vp, vp, vp, vp]
        L.or_row_fp.restype = u64
        L.or_row_fp.argtypes = [vp, vp, vp, vp, u32]
        L.or_batch_fp.restype = u64
        L.or_batch_fp.argtypes = [vp, u32]
        L.or_valid_steps.restype = u32
        L.or_valid_steps.argtypes = [vp]
        L.or_digest.restype = u64
        L.or_digest.argtypes = [vp]
        L.or_stream_windows.restype = u64
        L.or_stream_windows.argtypes = [vp, u32]
        L.or_stream_pieces.restype = u64
        L.or_stream_pieces.argtypes = [vp, u32]
        L.or_get_pieces.restype = None
        L.or_get_pieces.argtypes = [vp, u32, vp, vp, vp]
        L.or_get_window_first.restype = None
        L.or_get_window_first.argtypes = [vp, u32, vp]
        L.or_get_heldout.restype = None
        L.or_get_heldout.argtypes = [vp, vp, vp]
        L.or_get_quota.restype = None
        L.or_get_quota.argtypes = [vp, vp, vp, vp]
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]) -> Optional[int]:
    return None if a is None else a.ctypes.data


# ---- single functions -------------------------------------------------------
def splitmix64(x: int) -> int:
    return lib().or_splitmix64(x & M64)


def doc_hash(tokens: np.ndarray, hash_key: int = 0) -> int:
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    return lib().or_doc_hash(_ptr(t) if t.size else None, t.size, hash_key & M64)


def is_heldout(h: int, bp: int) -> bool:
    return bool(lib().or_is_heldout(h & M64, bp))


def feistel_bits(n: int) -> int:
    return lib().or_feistel_bits(n)


def feistel_round_key(seed: int, stream: int, rnd: int) -> int:
    return lib().or_feistel_round_key(seed & M64, stream, rnd)


def feistel_encrypt(keys: list[int], half: int, x: int) -> int:
    k = np.asarray([v & M64 for v in keys], dtype=np.uint64)
    return lib().or_feistel_encrypt(_ptr(k), half, x)


def feistel_pi(seed: int, stream: int, n: int, p: int) -> int:
    return lib().or_feistel_pi(seed & M64, stream, n, p)


def window_of_rank(seed: int, stream: int, G: int, W: int, r: int) -> int:
    return lib().or_window_of_rank(seed & M64, stream, G, W, r)


def row_of_slot(seed: int, step: int, B: int, i: int) -> int:
    return lib().or_row_of_slot(seed & M64, step, B, i)


def apportion(v: list[int], C_before: list[int], n: int, N: int) -> list[int]:
    vv = np.asarray(v, dtype=np.uint64)
    cc = np.asarray(C_before, dtype=np.int64)
    out = np.zeros(len(v), dtype=np.int64)
    rc = lib().or_apportion(len(v), _ptr(vv), _ptr(cc), n, N, _ptr(out))
    if rc != OK:
        raise ValueError(f"or_apportion failed: {rc}")
    return [int(a) for a in out]


def row_fp(tokens, pos, doc, mask) -> int:
    """Fingerprint of one row given its four arrays (length T each)."""
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    p = np.ascontiguousarray(pos, dtype=np.int32)
    d = np.ascontiguousarray(doc, dtype=np.int32)
    m = np.ascontiguousarray(mask, dtype=np.uint8)
    return lib().or_row_fp(_ptr(t), _ptr(p), _ptr(d), _ptr(m), t.size)


def batch_fp(row_fp: np.ndarray) -> int:
    f = np.ascontiguousarray(row_fp, dtype=np.uint64)
    return lib().or_batch_fp(_ptr(f), f.size)


# ---- a whole recipe ---------------------------------------------------------
class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: oracle error {code}")
        self.code = code


class Oracle:
    """Built state of one recipe: held-out flags, packed windows, quotas."""

    def __init__(self, corpus, *, seed: Optional[int] = None, hash_key: Optional[int] = None,
                 max_steps: Optional[int] = None, drain: Optional[bool] = None,
                 T: Optional[int] = None, B: Optional[int] = None,
                 pad_id: Optional[int] = None, heldout_only: bool = False,
                 window_segment: int = 0, shuffle_rows: bool = False,
                 schedule: Optional[list] = None, wrap: bool = False, len_bucket: int = 0):
        c = corpus
        self.corpus = c
        self.T = int(T if T is not None else c.T)
        self.B = int(B if B is not None else c.B)
        self.max_steps = int(max_steps if max_steps is not None else c.max_steps)
        self.n_streams = c.n_streams
        self.n_sources = c.n_sources
        self._keep = [np.ascontiguousarray(c.tokens, dtype=np.int32),
                      np.ascontiguousarray(c.doc_offsets, dtype=np.int64),
                      None if c.loss_start is None else np.ascontiguousarray(c.loss_start, dtype=np.int32),
                      np.ascontiguousarray(c.stream_doc_begin, dtype=np.uint32),
                      np.ascontiguousarray(c.stream_source, dtype=np.uint32),
                      np.ascontiguousarray(c.source_weight, dtype=np.uint32),
                      np.ascontiguousarray(c.stream_weight, dtype=np.uint32),
                      np.ascontiguousarray(c.source_heldout_bp, dtype=np.uint16)]
        tok, off, ls, sdb, ss, sw, tw, bp = self._keep
        cfg = _Config()
        cfg.tokens = _ptr(tok) if tok.size else _ptr(np.zeros(1, np.int32))
        if not tok.size:
            self._keep.append(np.zeros(1, np.int32))
            cfg.tokens = _ptr(self._keep[-1])
        cfg.n_tokens = tok.size
        cfg.doc_offsets = _ptr(off)
        cfg.loss_start = _ptr(ls)
        cfg.n_docs = off.size - 1
        cfg.n_sources = sw.size
        cfg.n_streams = ss.size
        cfg.T = self.T
        cfg.stream_doc_begin = _ptr(sdb)
        cfg.stream_source = _ptr(ss)
        cfg.source_weight = _ptr(sw)
        cfg.stream_weight = _ptr(tw)
        cfg.source_heldout_bp = _ptr(bp)
        cfg.seed = (seed if seed is not None else c.seed) & M64
        cfg.hash_key = (hash_key if hash_key is not None else c.hash_key) & M64
        cfg.B = self.B
        cfg.max_steps = self.max_steps
        cfg.drain = int(bool(drain if drain is not None else c.drain))
        cfg.pad_id = int(pad_id if pad_id is not None else c.pad_id)
        cfg.heldout_only = int(bool(heldout_only))
        cfg.window_segment = int(window_segment)
        cfg.shuffle_rows = int(bool(shuffle_rows))
        cfg.wrap = int(bool(wrap))
        cfg.len_bucket = int(len_bucket)
        self.schedule = schedule
        if schedule:
            pb = np.asarray([int(p["begin"]) for p in schedule], np.uint32)
            pB = np.asarray([int(p["B"]) for p in schedule], np.uint32)
            psw = np.ascontiguousarray([p["source_weight"] for p in schedule], dtype=np.uint32)
            ptw = np.ascontiguousarray([p["stream_weight"] for p in schedule], dtype=np.uint32)
            self._keep += [pb, pB, psw, ptw]
            cfg.n_pieces = pb.size
            cfg.piece_begin, cfg.piece_B = _ptr(pb), _ptr(pB)
            cfg.piece_source_weight, cfg.piece_stream_weight = _ptr(psw), _ptr(ptw)
        self._cfg = cfg
        h = C.c_void_p()
        rc = lib().or_build(C.byref(cfg), C.byref(h))
        if rc != OK:
            raise OracleError(rc, "or_build")
        self._h = h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.or_free(h)
            self._h = None

    @property
    def valid_steps(self) -> int:
        return lib().or_valid_steps(self._h)

    @property
    def digest(self) -> int:
        return lib().or_digest(self._h)

    def n_windows(self, j: int) -> int:
        return lib().or_stream_windows(self._h, j)

    def pieces(self, j: int):
        n = lib().or_stream_pieces(self._h, j)
        doc = np.zeros(n, np.uint32)
        off = np.zeros(n, np.uint32)
        ln = np.zeros(n, np.uint32)
        if n:
            lib().or_get_pieces(self._h, j, _ptr(doc), _ptr(off), _ptr(ln))
        return doc, off, ln

    def window_first(self, j: int) -> np.ndarray:
        w = self.n_windows(j)
        out = np.zeros(w + 1, np.uint64)
        lib().or_get_window_first(self._h, j, _ptr(out))
        return out

    def heldout(self):
        n = self.corpus.n_docs
        flags = np.zeros(max(n, 1), np.uint8)
        hashes = np.zeros(max(n, 1), np.uint64)
        lib().or_get_heldout(self._h, _ptr(flags), _ptr(hashes))
        return flags[:n].astype(bool), hashes[:n]

    def quota(self):
        K, J, S = self.max_steps, self.n_streams, self.n_sources
        q = np.zeros((K, J), np.int64)
        cum = np.zeros((K + 1, J), np.int64)
        sq = np.zeros((K, S), np.int64)
        lib().or_get_quota(self._h, _ptr(q), _ptr(cum), _ptr(sq))
        return q, cum, sq

    def rows_of_step(self, step: int) -> int:
        """Rows of update ``step`` (B, or the schedule's piece's)."""
        if not self.schedule:
            return self.B
        return int([p["B"] for p in self.schedule if p["begin"] <= step][-1])

    def rows(self, step: int, row0: int = 0, row1: Optional[int] = None) -> dict:
        """Rows [row0, row1) of update ``step`` as numpy arrays."""
        if row1 is None:
            row1 = self.rows_of_step(step)
        n = max(row1 - row0, 0)
        T = self.T
        out = dict(tokens=np.zeros((n, T), np.int32), pos=np.zeros((n, T), np.int32),
                   doc=np.zeros((n, T), np.int32), mask=np.zeros((n, T), np.uint8),
                   row_fp=np.zeros(n, np.uint64), row_learned=np.zeros(n, np.int32),
                   row_len=np.zeros(n, np.int32))
        rc = lib().or_rows(self._h, step, row0, row1, _ptr(out["tokens"]), _ptr(out["pos"]),
                           _ptr(out["doc"]), _ptr(out["mask"]), _ptr(out["row_fp"]),
                           _ptr(out["row_learned"]), _ptr(out["row_len"]))
        if rc != OK:
            raise OracleError(rc, f"or_rows(step={step}, rows=[{row0},{row1}))")
        return out
