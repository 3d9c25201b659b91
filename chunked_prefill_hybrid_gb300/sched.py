"""ctypes binding of include/hb_sched.h: the host decode-maximal scheduler.

Argument marshalling only; the policy runs in libhb.so (csrc/sched.cpp).
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import List

from . import native


class SchedConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("chunk_size", "token_budget", "max_decodes", "tile",
                                             "max_chunks_per_batch", "block_size", "num_blocks",
                                             "max_blocks_per_seq", "request_level")]


class _Batch(ctypes.Structure):
    _fields_ = [("n_chunks", ctypes.c_int), ("chunk_req_ids", ctypes.POINTER(ctypes.c_int32)),
                ("chunk_offsets", ctypes.POINTER(ctypes.c_int32)), ("chunk_lens", ctypes.POINTER(ctypes.c_int32)),
                ("n_decodes", ctypes.c_int), ("decode_req_ids", ctypes.POINTER(ctypes.c_int32)),
                ("decode_ctx_lens", ctypes.POINTER(ctypes.c_int32)), ("n_rows", ctypes.c_int)]


class _Stats(ctypes.Structure):
    _fields_ = [("waiting", ctypes.c_int), ("prefilling", ctypes.c_int), ("decoding", ctypes.c_int),
                ("finished", ctypes.c_int), ("free_blocks", ctypes.c_int), ("iterations", ctypes.c_longlong),
                ("decode_only_iterations", ctypes.c_longlong), ("rows", ctypes.c_longlong)]


@dataclass
class Batch:
    chunks: List[tuple]   # (req_id, offset, length)
    decodes: List[tuple]  # (req_id, ctx)
    n_rows: int


_sigs = False


def _lib():
    global _sigs
    L = native.lib()
    if not _sigs:
        vp, ci, P = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER
        for name, args, res in (
                ("hb_sched_create", [P(SchedConfig), P(vp)], ci),
                ("hb_sched_add", [vp, ci, ci, ci], ci),
                ("hb_sched_next", [vp, P(_Batch)], ci),
                ("hb_sched_complete", [vp], ci),
                ("hb_sched_block_table", [vp, ci, P(P(ctypes.c_int32)), P(ci)], ci),
                ("hb_sched_fill_spec", [vp, P(native.BatchSpec)], ci),
                ("hb_sched_get_stats", [vp, P(_Stats)], ci),
                ("hb_sched_max_batch", [ctypes.c_longlong] * 4, ctypes.c_longlong),
                ("hb_sched_free", [vp], None),
                ("hb_perfect_pd_ratio", [ci, ci], ctypes.c_double),
                ("hb_piggyback_capacity", [ctypes.c_longlong, ctypes.c_longlong, ci, ci], ctypes.c_longlong),
                ("hb_advise_chunk", [ctypes.c_double, ci, ci, ci, ci], ci),
                ("hb_sched_pd_estimate", [vp], ctypes.c_double)):
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _sigs = True
    return L


def max_batch(mem_total: int, mem_params: int, max_len: int, kv_bytes_per_token: int) -> int:
    return int(_lib().hb_sched_max_batch(mem_total, mem_params, max_len, kv_bytes_per_token))


def perfect_pd_ratio(chunk_size: int, batch_size: int) -> float:
    return float(_lib().hb_perfect_pd_ratio(chunk_size, batch_size))


def piggyback_capacity(prompt_len: int, decode_len: int, chunk_size: int, batch_size: int) -> int:
    return int(_lib().hb_piggyback_capacity(prompt_len, decode_len, chunk_size, batch_size))


def advise_chunk(pd_ratio: float, batch_size: int, tile: int = 0, c_min: int = 1, c_max: int = 1 << 30) -> int:
    return int(_lib().hb_advise_chunk(pd_ratio, batch_size, tile, c_min, c_max))


class Scheduler:
    def __init__(self, chunk_size: int, token_budget: int = 0, max_decodes: int = 1 << 20, tile: int = 0,
                 max_chunks_per_batch: int = 1, block_size: int = 16, num_blocks: int = 1 << 16,
                 max_blocks_per_seq: int = 1 << 12, request_level: int = 0):
        self.L = _lib()
        self.cfg = SchedConfig(chunk_size, token_budget, max_decodes, tile, max_chunks_per_batch, block_size,
                               num_blocks, max_blocks_per_seq, int(request_level))
        h = ctypes.c_void_p()
        rc = self.L.hb_sched_create(ctypes.byref(self.cfg), ctypes.byref(h))
        if rc:
            raise native.HbError(rc, "hb_sched_create")
        self.h = h
        self._spec = native.BatchSpec()

    def add(self, req_id: int, prompt_len: int, max_new_tokens: int):
        rc = self.L.hb_sched_add(self.h, req_id, prompt_len, max_new_tokens)
        if rc:
            raise native.HbError(rc, f"hb_sched_add({req_id})")

    def next(self) -> Batch:
        b = _Batch()
        rc = self.L.hb_sched_next(self.h, ctypes.byref(b))
        if rc < 0:
            raise native.HbError(rc, "hb_sched_next")
        chunks = [(b.chunk_req_ids[i], b.chunk_offsets[i], b.chunk_lens[i]) for i in range(b.n_chunks)]
        decodes = [(b.decode_req_ids[i], b.decode_ctx_lens[i]) for i in range(b.n_decodes)]
        return Batch(chunks, decodes, b.n_rows)

    def complete(self) -> int:
        rc = self.L.hb_sched_complete(self.h)
        if rc < 0:
            raise native.HbError(rc, "hb_sched_complete")
        return rc

    def block_table(self, req_id: int):
        p = ctypes.POINTER(ctypes.c_int32)()
        n = ctypes.c_int()
        rc = self.L.hb_sched_block_table(self.h, req_id, ctypes.byref(p), ctypes.byref(n))
        if rc:
            raise native.HbError(rc, "hb_sched_block_table")
        return [p[i] for i in range(n.value)]

    def fill_spec(self) -> native.BatchSpec:
        rc = self.L.hb_sched_fill_spec(self.h, ctypes.byref(self._spec))
        if rc:
            raise native.HbError(rc, "hb_sched_fill_spec")
        return self._spec

    def pd_estimate(self) -> float:
        return float(_lib().hb_sched_pd_estimate(self.h))

    def stats(self) -> dict:
        st = _Stats()
        self.L.hb_sched_get_stats(self.h, ctypes.byref(st))
        return {n: getattr(st, n) for n, _ in _Stats._fields_}

    def free(self):
        if getattr(self, "h", None):
            self.L.hb_sched_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass
