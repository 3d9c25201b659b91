"""ctypes wrapper around oracle.c -- the plain fp64 CPU oracle.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU-baseline leg
of the benchmark may call this; the product path never does.  It imports
nothing from the CUDA library package (it takes plain numpy arrays).

The oracle keeps its own paged KV pool, fp64, laid out [slot][n_kv][d] with
slot = block_table[pos // 16] * 16 + pos % 16 (Sarathi-Serve Guide, production
checklist "Paged KV-Cache Page Sizing").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs = {}

CFLAGS = ["-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-std=c11"]


def lib_path(mutate: int = 0) -> str:
    name = "liboracle.so" if mutate == 0 else f"liboracle_m{mutate}.so"
    return os.path.join(_BUILD, name)


def build(mutate: int = 0, force: bool = False) -> str:
    """Compile oracle.c with gcc (OR_MUTATE plants a mistake for mutation tests)."""
    out = lib_path(mutate)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, f"-DOR_MUTATE={int(mutate)}", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class _Dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("n_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int), ("block_size", ctypes.c_int),
                ("num_blocks", ctypes.c_int), ("rms_eps", ctypes.c_double), ("rope_theta", ctypes.c_double)]


class _Layer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("w_qkv", "w_o", "w_gate_up", "w_down", "norm1", "norm2")]


class _Batch(ctypes.Structure):
    _fields_ = [("chunk_offset", ctypes.c_int), ("chunk_len", ctypes.c_int), ("chunk_bt", ctypes.c_void_p),
                ("chunk_n_blocks", ctypes.c_int), ("n_decodes", ctypes.c_int), ("decode_ctx", ctypes.c_void_p),
                ("decode_bt", ctypes.c_void_p), ("max_blocks_per_seq", ctypes.c_int)]


class _Aux(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "o", "h", "a", "n1", "n2")]


def load(mutate: int = 0) -> ctypes.CDLL:
    with _lock:
        if mutate in _libs:
            return _libs[mutate]
        L = ctypes.CDLL(build(mutate))
        L.or_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.or_bf16_to_f64.restype = ctypes.c_double
        L.or_f64_to_bf16.argtypes = [ctypes.c_double]
        L.or_f64_to_bf16.restype = ctypes.c_uint16
        L.or_matvec.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        L.or_rmsnorm.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_void_p]
        L.or_rope.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_double]
        L.or_silu.argtypes = [ctypes.c_double]
        L.or_silu.restype = ctypes.c_double
        L.or_slot.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.or_slot.restype = ctypes.c_int
        L.or_attention_head.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
        L.or_attention_head.restype = ctypes.c_int
        L.oracle_layer_forward.argtypes = [ctypes.POINTER(_Dims), ctypes.POINTER(_Layer), ctypes.c_int,
                                           ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(_Batch),
                                           ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.POINTER(_Aux)]
        L.oracle_layer_forward.restype = ctypes.c_int
        L.or_max_threads.restype = ctypes.c_int
        L.or_set_threads.argtypes = [ctypes.c_int]
        _libs[mutate] = L
        return L


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- scalar ops

def bf16_round(x, mutate: int = 0) -> np.ndarray:
    """fp64 -> nearest bf16 -> fp64, elementwise (ties to even)."""
    L = load(mutate)
    a = np.asarray(x, np.float64)
    return np.array([L.or_bf16_to_f64(L.or_f64_to_bf16(float(v))) for v in a.ravel()]).reshape(a.shape)


def f64_to_bf16_bits(x, mutate: int = 0) -> np.ndarray:
    L = load(mutate)
    a = np.asarray(x, np.float64)
    return np.array([L.or_f64_to_bf16(float(v)) for v in a.ravel()], np.uint16).reshape(a.shape)


def bf16_bits_to_f64(bits, mutate: int = 0) -> np.ndarray:
    L = load(mutate)
    b = np.asarray(bits, np.uint16)
    return np.array([L.or_bf16_to_f64(int(v)) for v in b.ravel()], np.float64).reshape(b.shape)


def matvec(W_bits: np.ndarray, x: np.ndarray, mutate: int = 0) -> np.ndarray:
    W = _c(W_bits, np.uint16)
    xv = _c(x, np.float64)
    y = np.zeros(W.shape[0], np.float64)
    load(mutate).or_matvec(_p(W), W.shape[0], W.shape[1], _p(xv), _p(y))
    return y


def rmsnorm(x: np.ndarray, gamma_bits: Optional[np.ndarray], eps: float, mutate: int = 0) -> np.ndarray:
    xv = _c(x, np.float64)
    g = None if gamma_bits is None else _c(gamma_bits, np.uint16)
    out = np.zeros_like(xv)
    load(mutate).or_rmsnorm(_p(xv), _p(g), xv.shape[0], eps, _p(out))
    return out


def rope(v: np.ndarray, pos: int, theta: float = 1e4, mutate: int = 0) -> np.ndarray:
    out = _c(v, np.float64).copy()
    load(mutate).or_rope(_p(out), out.shape[0], int(pos), theta)
    return out


def silu(z: float, mutate: int = 0) -> float:
    return load(mutate).or_silu(float(z))


def slot(block_table: np.ndarray, pos: int, num_blocks: int, block_size: int = 16, mutate: int = 0) -> int:
    bt = _c(block_table, np.int32)
    return load(mutate).or_slot(_p(bt), bt.shape[0], block_size, num_blocks, int(pos))


class Pool:
    """The oracle's own fp64 paged KV pool for one layer: [num_blocks*bs][n_kv][d]."""

    def __init__(self, num_blocks: int, n_kv: int, head_dim: int, block_size: int = 16):
        self.num_blocks, self.n_kv, self.head_dim, self.block_size = num_blocks, n_kv, head_dim, block_size
        self.k = np.zeros((num_blocks * block_size, n_kv, head_dim), np.float64)
        self.v = np.zeros_like(self.k)

    def write(self, block_table, start_pos: int, k: np.ndarray, v: np.ndarray, mutate: int = 0):
        """Place k[i], v[i] ([n][n_kv][d]) at position start_pos + i."""
        for i in range(k.shape[0]):
            s = slot(block_table, start_pos + i, self.num_blocks, self.block_size, mutate)
            if s < 0:
                raise IndexError("position outside the block table")
            self.k[s] = k[i]
            self.v[s] = v[i]

    def read(self, block_table, start_pos: int, n: int, mutate: int = 0):
        ks, vs = [], []
        for i in range(n):
            s = slot(block_table, start_pos + i, self.num_blocks, self.block_size, mutate)
            ks.append(self.k[s])
            vs.append(self.v[s])
        return np.array(ks), np.array(vs)

    def copy(self) -> "Pool":
        p = Pool.__new__(Pool)
        p.num_blocks, p.n_kv, p.head_dim, p.block_size = self.num_blocks, self.n_kv, self.head_dim, self.block_size
        p.k, p.v = self.k.copy(), self.v.copy()
        return p


def attention_head(q: np.ndarray, pool: Pool, kv_head: int, block_table, last_pos: int, mutate: int = 0):
    qv = _c(q, np.float64)
    bt = _c(block_table, np.int32)
    out = np.zeros(qv.shape[0], np.float64)
    rc = load(mutate).or_attention_head(_p(qv), qv.shape[0], kv_head, pool.n_kv, _p(pool.k), _p(pool.v),
                                        _p(bt), bt.shape[0], pool.block_size, pool.num_blocks,
                                        int(last_pos), _p(out))
    if rc:
        raise IndexError(f"or_attention_head failed ({rc})")
    return out


# ------------------------------------------------------------ layer forward

class OracleError(RuntimeError):
    pass


def layer_forward(dims, weights: dict, batch, x_in: np.ndarray, pool: Pool, mirror: bool = True,
                  rows: Optional[np.ndarray] = None, aux: bool = False, mutate: int = 0):
    """One decoder layer over a hybrid batch (rows: chunk first, then decodes).

    dims: an object with hidden, n_heads, n_kv_heads, head_dim, ffn, rms_eps,
    rope_theta, block_size.  weights: dict of bf16 bit arrays (see
    oracle.c).  batch: object with .chunk (None or .cached/.block_table),
    .chunk_len and .decodes (each .cached/.block_table).  x_in: [T][hidden]
    fp64.  pool: updated in place with the batch's new K/V.  rows: optional
    boolean mask of rows to compute.  Returns y [T][hidden] (rows not
    selected are NaN) and, if aux, a dict of intermediates.
    """
    more = list(getattr(batch, "more_chunks", None) or [])
    if more:
        return _forward_split(dims, weights, batch, more, x_in, pool, mirror, rows, aux, mutate)
    L = load(mutate)
    T = batch.n_tokens
    H = dims.hidden
    w = {k: _c(v, np.uint16) for k, v in weights.items()}
    dm = _Dims(dims.hidden, dims.n_heads, dims.n_kv_heads, dims.head_dim, dims.ffn, dims.block_size,
               pool.num_blocks, float(dims.rms_eps), float(dims.rope_theta))
    lw = _Layer(*[_p(w[n]) for n in ("w_qkv", "w_o", "w_gate_up", "w_down", "norm1", "norm2")])
    if batch.chunk is not None:
        cbt = _c(batch.chunk.block_table, np.int32)
        coff, clen = batch.chunk.cached, batch.chunk_len
    else:
        cbt, coff, clen = np.zeros(1, np.int32), 0, 0
    D = len(batch.decodes)
    mbs = max([len(s.block_table) for s in batch.decodes] + [1])
    dbt = np.full((max(D, 1), mbs), -1, np.int32)
    dctx = np.zeros(max(D, 1), np.int32)
    for j, s in enumerate(batch.decodes):
        dbt[j, :len(s.block_table)] = s.block_table
        dctx[j] = s.cached
    b = _Batch(coff, clen, _p(cbt), cbt.shape[0], D, _p(dctx), _p(dbt), mbs)
    xv = _c(x_in, np.float64)
    assert xv.shape == (T, H), (xv.shape, T, H)
    y = np.full((T, H), np.nan, np.float64)
    sel = None if rows is None else _c(np.asarray(rows).astype(np.uint8), np.uint8)
    bufs = None
    a = _Aux()
    if aux:
        bufs = {"q": np.full((T, dims.n_heads * dims.head_dim), np.nan),
                "k": np.full((T, dims.n_kv_heads * dims.head_dim), np.nan),
                "v": np.full((T, dims.n_kv_heads * dims.head_dim), np.nan),
                "o": np.full((T, dims.n_heads * dims.head_dim), np.nan),
                "h": np.full((T, H), np.nan),
                "a": np.full((T, dims.ffn), np.nan),
                "n1": np.full((T, H), np.nan),
                "n2": np.full((T, H), np.nan)}
        a = _Aux(*[_p(bufs[n]) for n in ("q", "k", "v", "o", "h", "a", "n1", "n2")])
    rc = L.oracle_layer_forward(ctypes.byref(dm), ctypes.byref(lw), int(bool(mirror)), _p(pool.k), _p(pool.v),
                                ctypes.byref(b), _p(xv), _p(y), _p(sel), ctypes.byref(a))
    if rc:
        raise OracleError(f"oracle_layer_forward returned {rc}")
    return (y, bufs) if aux else y


class _Part:
    """A batch of one chunk (or none) and some decodes."""

    def __init__(self, chunk, chunk_len, decodes):
        self.chunk, self.chunk_len, self.decodes = chunk, chunk_len, decodes
        self.n_tokens = (chunk_len if chunk is not None else 0) + len(decodes)


def _forward_split(dims, weights, batch, more, x_in, pool, mirror, rows, aux, mutate):
    """A batch with several chunks: rows of different requests never meet
    (each attends only its own request's keys), so the first chunk with the
    decodes, and each further chunk on its own, give the batch's rows.  Row
    order: first chunk, further chunks in order, decodes."""
    if aux:
        raise OracleError("aux intermediates are only kept for single-chunk batches")
    T, H = x_in.shape
    c0 = batch.chunk_len if batch.chunk is not None else 0
    starts, at = [], c0
    for _, n in more:
        starts.append(at)
        at += n
    dec = np.arange(at, T)
    y = np.full((T, H), np.nan, np.float64)
    sel = None if rows is None else np.asarray(rows).astype(bool)
    first = np.concatenate([np.arange(c0), dec]).astype(np.int64)
    parts = [(first, _Part(batch.chunk, c0, list(batch.decodes)))]
    for (seq, n), q0 in zip(more, starts):
        parts.append((np.arange(q0, q0 + n), _Part(seq, n, [])))
    for idx, part in parts:
        if part.n_tokens == 0:
            continue
        y[idx] = layer_forward(dims, weights, part, np.ascontiguousarray(x_in[idx]), pool, mirror=mirror,
                               rows=None if sel is None else sel[idx], mutate=mutate)
    return y


def set_threads(n: int, mutate: int = 0):
    load(mutate).or_set_threads(int(n))


def max_threads(mutate: int = 0) -> int:
    return load(mutate).or_max_threads()
