"""A thin PyTorch-facing wrapper over the C ABI.

PyTorch supplies device memory (its caching allocator, through the
library's allocation callback), the CUDA stream and the output tensors.  All
packing work runs in the library's kernels.
"""
from __future__ import annotations

import ctypes as C
from typing import Optional

import numpy as np
import torch

from . import _lib as L


def _u32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=np.uint32)


def _refuse(what: str) -> None:
    raise L.NsPackError(L.NS_ERR_INVALID_ARG, what)


def _need(t, name: str, dtype: torch.dtype, device=None) -> None:
    """Refuse a tensor the library would misread, or read or write past:
    its pointer is handed over with no shape, stride or type."""
    if not isinstance(t, torch.Tensor):
        _refuse(f"{name}: expected a tensor, got {type(t).__name__}")
    if t.dtype != dtype:
        _refuse(f"{name}: dtype {t.dtype}, expected {dtype}")
    if device is not None and t.device != device:
        _refuse(f"{name}: on {t.device}, expected {device}")
    if not t.is_contiguous():
        _refuse(f"{name}: not contiguous")


class Packer:
    """A packing context over a corpus resident on one CUDA device.

    ``tokens`` (int32), ``doc_offsets`` (int64, n_docs + 1) and ``loss_start``
    (int32 or None) are device tensors that must outlive the packer -- or CPU
    tensors (page-locked for the copies to overlap the hash), which the
    library copies to ``device`` itself while it builds the context.  The
    recipe arrays may be numpy arrays or lists.  ``heldout_only`` packs the
    validation stream (the held-out documents) instead of the training one;
    ``window_segment`` > 0 reads each stream's windows in a shuffled order
    within segments of that many windows; ``shuffle_rows`` shuffles the rows
    of every update; ``schedule`` (a list of ``dict(begin, B, source_weight,
    stream_weight)``) gives pieces of the horizon their own rows per update
    and weights; ``wrap`` cuts each stream's concatenated kept tokens into
    windows of exactly T (across document ends) instead of greedy packing;
    ``len_bucket`` rounds the reported row lengths up to its multiples.
    """

    def __init__(self, tokens: torch.Tensor, doc_offsets: torch.Tensor,
                 loss_start: Optional[torch.Tensor], *, stream_doc_begin, stream_source,
                 source_weight, stream_weight, source_heldout_bp, T: int, B: int,
                 max_steps: int, seed: int = 0, hash_key: int = 0, drain: bool = False,
                 pad_id: int = 0, heldout_only: bool = False, window_segment: int = 0,
                 shuffle_rows: bool = False, schedule: Optional[list] = None,
                 wrap: bool = False, len_bucket: int = 0,
                 stream: Optional[torch.cuda.Stream] = None, device=None):
        _need(tokens, "tokens", torch.int32)
        _need(doc_offsets, "doc_offsets", torch.int64, tokens.device)
        if loss_start is not None:
            _need(loss_start, "loss_start", torch.int32, tokens.device)
        self.host_corpus = not tokens.is_cuda
        if self.host_corpus:
            if tokens.device.type != "cpu":
                raise ValueError("tokens must be a CUDA or a CPU tensor")
            self.device = torch.device(device if device is not None else "cuda")
            if self.device.index is None:
                self.device = torch.device("cuda", torch.cuda.current_device())
        else:
            self.device = tokens.device
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        self.T, self.B, self.max_steps = int(T), int(B), int(max_steps)
        self._corpus = (tokens, doc_offsets, loss_start)
        self._tables = [_u32(stream_doc_begin), _u32(stream_source), _u32(source_weight),
                        _u32(stream_weight),
                        np.ascontiguousarray(np.asarray(source_heldout_bp), dtype=np.uint16)]
        sdb, ssrc, sw, tw, bp = self._tables
        self.n_streams = int(ssrc.size)
        self.n_sources = int(sw.size)
        dev_index = self.device.index if self.device.index is not None else torch.cuda.current_device()
        stream_handle = self.stream.cuda_stream

        def _alloc(nbytes, _user):
            try:
                return torch.cuda.caching_allocator_alloc(int(nbytes), dev_index, self.stream)
            except Exception:  # out of memory: the library reports NS_ERR_OOM
                return None

        def _free(ptr, _user):
            torch.cuda.caching_allocator_delete(ptr)

        self._alloc_cb = L.ns_alloc_fn(_alloc)
        self._free_cb = L.ns_free_fn(_free)
        cfg = L.ns_pack_config()
        cfg.tokens = tokens.data_ptr()
        cfg.n_tokens = tokens.numel()
        cfg.doc_offsets = doc_offsets.data_ptr()
        cfg.loss_start = None if loss_start is None else loss_start.data_ptr()
        cfg.n_docs = doc_offsets.numel() - 1
        cfg.n_sources = self.n_sources
        cfg.n_streams = self.n_streams
        cfg.T = self.T
        cfg.stream_doc_begin = sdb.ctypes.data
        cfg.stream_source = ssrc.ctypes.data
        cfg.source_weight = sw.ctypes.data
        cfg.stream_weight = tw.ctypes.data
        cfg.source_heldout_bp = bp.ctypes.data
        cfg.seed = int(seed) & ((1 << 64) - 1)
        cfg.hash_key = int(hash_key) & ((1 << 64) - 1)
        cfg.B = self.B
        cfg.max_steps = self.max_steps
        cfg.flags = ((L.NS_PACK_DRAIN if drain else 0) | (L.NS_PACK_HELDOUT if heldout_only else 0)
                     | (L.NS_PACK_SHUFFLE_ROWS if shuffle_rows else 0)
                     | (L.NS_PACK_WRAP if wrap else 0)
                     | (L.NS_PACK_HOST_CORPUS if self.host_corpus else 0)
                     # the caching allocator reuses a freed block only on the
                     # stream it was allocated on, after the free
                     | L.NS_PACK_ORDERED_FREE)
        cfg.len_bucket = int(len_bucket)
        cfg.window_segment = int(window_segment)
        self.schedule = schedule
        if schedule:
            pieces = [np.asarray([int(p["begin"]) for p in schedule], np.uint32),
                      np.asarray([int(p["B"]) for p in schedule], np.uint32),
                      np.ascontiguousarray([p["source_weight"] for p in schedule], np.uint32),
                      np.ascontiguousarray([p["stream_weight"] for p in schedule], np.uint32)]
            self._tables += pieces
            cfg.n_pieces = pieces[0].size
            cfg.piece_begin, cfg.piece_B = pieces[0].ctypes.data, pieces[1].ctypes.data
            cfg.piece_source_weight = pieces[2].ctypes.data
            cfg.piece_stream_weight = pieces[3].ctypes.data
        cfg.pad_id = int(pad_id)
        cfg.cuda_stream = stream_handle
        cfg.alloc = self._alloc_cb
        cfg.free = self._free_cb
        cfg.alloc_user = None
        with torch.cuda.device(self.device):
            self._ctx = L.ns_pack_init(cfg)
        info = L.ns_pack_info(self._ctx)
        self.valid_steps = info["valid_steps"]
        self.order_digest = info["order_digest"]
        self.info = info

    @classmethod
    def from_corpus(cls, corpus, device="cuda", **overrides) -> "Packer":
        """Copy a ``corpus.Corpus``-like object's arrays to ``device`` and
        build a packer with its recipe (fields may be overridden)."""
        dev = torch.device(device)
        tok = torch.from_numpy(np.ascontiguousarray(corpus.tokens)).to(dev)
        off = torch.from_numpy(np.ascontiguousarray(corpus.doc_offsets)).to(dev)
        ls = None
        if corpus.loss_start is not None:
            ls = torch.from_numpy(np.ascontiguousarray(corpus.loss_start)).to(dev)
        kw = dict(stream_doc_begin=corpus.stream_doc_begin, stream_source=corpus.stream_source,
                  source_weight=corpus.source_weight, stream_weight=corpus.stream_weight,
                  source_heldout_bp=corpus.source_heldout_bp, T=corpus.T, B=corpus.B,
                  max_steps=corpus.max_steps, seed=corpus.seed, hash_key=corpus.hash_key,
                  drain=corpus.drain, pad_id=corpus.pad_id)
        kw.update(overrides)
        return cls(tok, off, ls, **kw)

    def rows_of_step(self, step: int) -> int:
        """Rows of update ``step`` (B, or the schedule's piece's)."""
        if not self.schedule:
            return self.B
        return int([p["B"] for p in self.schedule if p["begin"] <= step][-1])

    # ---- outputs -----------------------------------------------------------
    def empty_out(self, n_steps: int = 1, n_rows: Optional[int] = None) -> dict:
        n_rows = self.B if n_rows is None else n_rows
        shape = (n_steps, n_rows, self.T)
        d = self.device
        return dict(tokens=torch.empty(shape, dtype=torch.int32, device=d),
                    pos=torch.empty(shape, dtype=torch.int32, device=d),
                    doc=torch.empty(shape, dtype=torch.int32, device=d),
                    mask=torch.empty(shape, dtype=torch.uint8, device=d),
                    row_fp=torch.empty((n_steps, n_rows), dtype=torch.int64, device=d),
                    row_learned=torch.empty((n_steps, n_rows), dtype=torch.int32, device=d),
                    row_len=torch.empty((n_steps, n_rows), dtype=torch.int32, device=d))

    # the output arrays: (name, dtype, one element per position (else per row))
    _OUT = (("tokens", torch.int32, True), ("pos", torch.int32, True),
            ("doc", torch.int32, True), ("mask", torch.uint8, True),
            ("row_fp", torch.int64, False), ("row_learned", torch.int32, False),
            ("row_len", torch.int32, False))

    @staticmethod
    def _out_struct(out: dict) -> L.ns_pack_out:
        dev = out["tokens"].device if isinstance(out.get("tokens"), torch.Tensor) else None
        positions, rows = [], []
        for name, dtype, per_position in Packer._OUT:
            t = out.get(name)
            if t is None and name == "row_len":
                continue
            _need(t, f"out[{name!r}]", dtype, dev)
            (positions if per_position else rows).append(t.numel())
        o = L.ns_pack_out()
        o.tokens = out["tokens"].data_ptr()
        o.pos = out["pos"].data_ptr()
        o.doc = out["doc"].data_ptr()
        o.mask = out["mask"].data_ptr()
        o.row_fp = out["row_fp"].data_ptr()
        o.row_learned = out["row_learned"].data_ptr()
        o.row_len = out["row_len"].data_ptr() if out.get("row_len") is not None else None
        # what the buffers hold, checked against every call that writes them
        o.nspack_device, o.nspack_positions, o.nspack_rows = dev, min(positions), min(rows)
        return o

    @staticmethod
    def prepare(out: dict) -> L.ns_pack_out:
        """The C description of the buffers in ``out``, built once for steps
        that write the same buffers again (``step(..., prepared=...)``)."""
        return Packer._out_struct(out)

    def step(self, step0: int, n_steps: int = 1, rows: Optional[tuple] = None,
             out: Optional[dict] = None, stream: Optional[torch.cuda.Stream] = None,
             prepared: Optional[L.ns_pack_out] = None) -> dict:
        """Assemble rows ``rows = (begin, end)`` of updates [step0, step0 +
        n_steps) into ``out`` (allocated if None); asynchronous.  ``prepared``
        (from ``prepare(out)``) saves describing ``out`` again."""
        r0, r1 = (0, self.rows_of_step(step0)) if rows is None else rows
        if out is None:
            out = self.empty_out(n_steps, r1 - r0)
        o = prepared if prepared is not None else self._out_struct(out)
        if hasattr(o, "nspack_rows"):
            n = max(int(n_steps), 0) * max(int(r1) - int(r0), 0)
            if o.nspack_device != self.device:
                _refuse(f"Packer.step: outputs on {o.nspack_device}, the packer on {self.device}")
            if n > o.nspack_rows or n * self.T > o.nspack_positions:
                _refuse(f"Packer.step: the outputs hold {o.nspack_rows} rows, "
                        f"the call writes {n}")
        st = (stream or self.stream).cuda_stream
        L.ns_pack_step(self._ctx, step0, n_steps, r0, r1, o, st)
        return out

    def batch_fp(self, row_fp: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> int:
        """Fold one batch's row fingerprints (device, row order); synchronises."""
        _need(row_fp, "row_fp", torch.int64, self.device)
        st = (stream or self.stream).cuda_stream
        return L.ns_pack_fingerprint(self._ctx, row_fp.data_ptr(), row_fp.numel(), st)

    def batch_fp_many(self, row_fp: torch.Tensor, out: Optional[torch.Tensor] = None,
                      stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        """Batch fingerprints of [n_steps, n_rows] row fingerprints (async)."""
        _need(row_fp, "row_fp", torch.int64, self.device)
        if row_fp.dim() != 2:
            _refuse(f"row_fp: shape {tuple(row_fp.shape)}, expected [n_steps, n_rows]")
        n_steps, n_rows = row_fp.shape
        if out is None:
            out = torch.empty(n_steps, dtype=torch.int64, device=self.device)
        _need(out, "out", torch.int64, self.device)
        if out.numel() < n_steps:
            _refuse(f"out: {out.numel()} elements, the call writes {n_steps}")
        st = (stream or self.stream).cuda_stream
        L.ns_pack_batch_fp(self._ctx, row_fp.data_ptr(), n_steps, n_rows, out.data_ptr(), st)
        return out

    def step_learned(self, row_learned: torch.Tensor, out: Optional[torch.Tensor] = None,
                     stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        """Learned positions of each update of [n_steps, n_rows] row counts
        (int64, async): what a trainer weighs the update's loss by."""
        _need(row_learned, "row_learned", torch.int32, self.device)
        if row_learned.dim() != 2:
            _refuse(f"row_learned: shape {tuple(row_learned.shape)}, expected [n_steps, n_rows]")
        n_steps, n_rows = row_learned.shape
        if out is None:
            out = torch.empty(n_steps, dtype=torch.int64, device=self.device)
        _need(out, "out", torch.int64, self.device)
        if out.numel() < n_steps:
            _refuse(f"out: {out.numel()} elements, the call writes {n_steps}")
        st = (stream or self.stream).cuda_stream
        L.ns_pack_step_learned(self._ctx, row_learned.data_ptr(), n_steps, n_rows,
                               out.data_ptr(), st)
        return out

    def stream_windows(self):
        return L.ns_pack_stream_windows(self._ctx, self.n_streams)

    def quota_table(self):
        return L.ns_pack_quota_table(self._ctx, self.max_steps, self.n_streams)

    def check(self) -> None:
        L.ns_pack_check(self._ctx)

    def close(self) -> None:
        if getattr(self, "_ctx", None) is not None and self._ctx.value:
            L.ns_pack_free(self._ctx)
            self._ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def as_u64(t: torch.Tensor) -> np.ndarray:
    """Row fingerprints come back as int64 tensors; view them as uint64."""
    return t.detach().cpu().numpy().view(np.uint64)
