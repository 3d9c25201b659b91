"""Thin ctypes binding of include/hb.h (argument marshalling only).

Every computation runs in libhb.so's CUDA kernels; this module only turns
Python objects into the C structs and pointers of the ABI.  PyTorch tensors
are used as device memory (``tensor.data_ptr()``).  If the library has not
been built, loading it raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

from . import synth

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhb.so")

HB_OK, HB_EINVAL, HB_ERANGE, HB_ENOMEM, HB_ECUDA, HB_EDEVICE, HB_ESTATE = 0, -1, -2, -3, -4, -5, -6
_NAMES = {0: "HB_OK", -1: "HB_EINVAL", -2: "HB_ERANGE", -3: "HB_ENOMEM", -4: "HB_ECUDA", -5: "HB_EDEVICE",
          -6: "HB_ESTATE"}

# Every symbol include/hb.h declares.
ABI_SYMBOLS = ["hb_init", "hb_load_layer", "hb_append_kv", "hb_read_kv", "hb_fill_kv", "hb_forward",
               "hb_forward_layers", "hb_forward_host", "hb_forward_host_async", "hb_sync", "hb_profile", "hb_profile_read",
               "hb_launch_count", "hb_gemm_test", "hb_debug_read", "hb_set_kernels", "hb_test_wait_timeout", "hb_plan",
               "hb_last_error", "hb_free", "hb_decode_attention_noalloc"]


class HbError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_NAMES.get(code, code)}: {msg}")
        self.code = code


class ModelConfig(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("hidden", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float), ("block_size", ctypes.c_int),
                ("num_blocks", ctypes.c_int), ("max_blocks_per_seq", ctypes.c_int), ("max_tokens", ctypes.c_int),
                ("max_decodes", ctypes.c_int), ("max_pos", ctypes.c_int)]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("w_qkv", "w_o", "w_gate_up", "w_down", "norm1", "norm2")]


class BatchSpec(ctypes.Structure):
    _fields_ = [("chunk_req_id", ctypes.c_int), ("chunk_offset", ctypes.c_int), ("chunk_len", ctypes.c_int),
                ("chunk_block_table", ctypes.c_void_p), ("chunk_n_blocks", ctypes.c_int),
                ("n_decodes", ctypes.c_int), ("decode_req_ids", ctypes.c_void_p),
                ("decode_ctx_lens", ctypes.c_void_p), ("decode_block_tables", ctypes.c_void_p),
                ("decode_bt_stride", ctypes.c_int), ("n_more_chunks", ctypes.c_int),
                ("more_chunk_req_ids", ctypes.c_void_p), ("more_chunk_offsets", ctypes.c_void_p),
                ("more_chunk_lens", ctypes.c_void_p), ("more_chunk_block_tables", ctypes.c_void_p),
                ("more_chunk_bt_stride", ctypes.c_int)]

HB_MAX_CHUNKS = 16


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    vp, ci, P = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER
    sig = {
        "hb_init": ([P(ModelConfig), vp, vp, P(vp)], ci),
        "hb_load_layer": ([vp, ci, P(LayerWeights)], ci),
        "hb_append_kv": ([vp, ci, vp, ci, ci, ci, vp, vp], ci),
        "hb_read_kv": ([vp, ci, vp, ci, ci, ci, vp, vp], ci),
        "hb_fill_kv": ([vp, ctypes.c_uint16], ci),
        "hb_forward": ([vp, P(BatchSpec), vp, vp], ci),
        "hb_forward_layers": ([vp, P(BatchSpec), ci, ci, vp, vp], ci),
        "hb_forward_host": ([vp, P(BatchSpec), vp, vp], ci),
        "hb_forward_host_async": ([vp, P(BatchSpec), vp, vp], ci),
        "hb_sync": ([vp], ci),
        "hb_profile": ([vp, ci], ci),
        "hb_profile_read": ([vp, vp, vp, vp, ci], ci),
        "hb_launch_count": ([vp], ctypes.c_longlong),
        "hb_gemm_test": ([vp, vp, vp, vp, ci, ci, ci], ci),
        "hb_debug_read": ([vp, ci, vp, ci], ci),
        "hb_set_kernels": ([vp, ci, ci], ci),
        "hb_test_wait_timeout": ([vp, ctypes.c_longlong], ci),
        "hb_plan": ([P(ModelConfig), P(BatchSpec), vp, vp, ctypes.c_char_p, ci], ci),
        "hb_last_error": ([vp], ctypes.c_char_p),
        "hb_free": ([vp], None),
        "hb_decode_attention_noalloc": ([vp, vp, vp, vp, ci, vp, ci, ci, ci, ci, ci, ci, vp, vp], ci),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    _lib = L
    return L


def model_config(dims: synth.ModelDims, num_blocks: int, max_tokens: int, max_decodes: int, max_pos: int,
                 n_layers: Optional[int] = None) -> ModelConfig:
    mbs = (max_pos + 15) // 16
    return ModelConfig(n_layers if n_layers is not None else dims.n_layers, dims.hidden, dims.n_heads,
                       dims.n_kv_heads, dims.head_dim, dims.ffn, dims.rms_eps, dims.rope_theta, 16, num_blocks,
                       mbs, max_tokens, max_decodes, max_pos)


class Spec:
    """A BatchSpec plus the host arrays it points into (kept alive here)."""

    def __init__(self, batch: synth.HybridBatch, req_ids: Optional[Sequence[int]] = None):
        self.batch = batch
        D = batch.n_decodes
        if batch.chunk is not None:
            self.cbt = np.ascontiguousarray(batch.chunk.block_table, np.int32)
            cid, coff, clen = batch.chunk.req_id, batch.chunk.cached, batch.chunk_len
        else:
            self.cbt = np.zeros(1, np.int32)
            cid, coff, clen = -1, 0, 0
        stride = max([len(s.block_table) for s in batch.decodes] + [1])
        self.dbt = synth.padded_decode_tables(batch, stride)
        self.dids = np.array([s.req_id for s in batch.decodes] or [0], np.int32)
        self.dctx = np.array([s.cached for s in batch.decodes] or [0], np.int32)
        more = list(batch.more_chunks)
        mstride = max([len(sq.block_table) for sq, _ in more] + [1])
        self.mbt = np.full((max(len(more), 1), mstride), -1, np.int32)
        for i, (sq, _) in enumerate(more):
            self.mbt[i, :len(sq.block_table)] = sq.block_table
        self.mids = np.array([sq.req_id for sq, _ in more] or [0], np.int32)
        self.moff = np.array([sq.cached for sq, _ in more] or [0], np.int32)
        self.mlen = np.array([n for _, n in more] or [0], np.int32)
        self.c = BatchSpec(cid, coff, clen, self.cbt.ctypes.data, len(self.cbt) if batch.chunk is not None else 0,
                           D, self.dids.ctypes.data, self.dctx.ctypes.data, self.dbt.ctypes.data, stride,
                           len(more), self.mids.ctypes.data, self.moff.ctypes.data, self.mlen.ctypes.data,
                           self.mbt.ctypes.data, mstride)

    @property
    def T(self) -> int:
        return self.batch.n_tokens


def plan(cfg: ModelConfig, spec: Spec):
    """Host-only validation + (pos, slot) of each row; raises HbError."""
    T = max(spec.T, 1)
    pos = np.zeros(T, np.int32)
    slot = np.zeros(T, np.int32)
    buf = ctypes.create_string_buffer(512)
    rc = lib().hb_plan(ctypes.byref(cfg), ctypes.byref(spec.c), pos.ctypes.data, slot.ctypes.data, buf, 512)
    if rc < 0:
        raise HbError(rc, buf.value.decode())
    return pos[:rc], slot[:rc]


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def decode_attention_noalloc(q, k_pool, v_pool, block_tables, ctx_lens, max_ctx: int, out, stream=None):
    """hb_decode_attention_noalloc on device tensors (no context, no device
    allocation): q, out [n][n_heads][head_dim] bf16 (as int16/uint16/bf16
    storage); k_pool, v_pool [num_blocks][n_kv][16][head_dim]; block_tables
    int32 [n][stride]; ctx_lens int32 [n].  Raises HbError on a bad call."""
    import torch
    n, n_heads, head_dim = q.shape
    num_blocks, n_kv = k_pool.shape[0], k_pool.shape[1]
    for t in (q, k_pool, v_pool, block_tables, ctx_lens, out):
        if not t.is_contiguous():
            raise ValueError("decode_attention_noalloc wants contiguous tensors")
    st = stream if stream is not None else torch.cuda.current_stream()
    rc = lib().hb_decode_attention_noalloc(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                                           int(block_tables.shape[1]), _ptr(ctx_lens), n, n_heads, n_kv, head_dim,
                                           num_blocks, int(max_ctx), _ptr(out), ctypes.c_void_p(st.cuda_stream))
    if rc:
        raise HbError(rc, "hb_decode_attention_noalloc failed")


class Context:
    """An hb_ctx on the current CUDA device."""

    def __init__(self, cfg: ModelConfig, stream=None):
        import torch
        self.cfg = cfg
        self.L = lib()
        self._stream = stream if stream is not None else torch.cuda.current_stream()
        h = ctypes.c_void_p()
        rc = self.L.hb_init(ctypes.byref(cfg), None, ctypes.c_void_p(self._stream.cuda_stream), ctypes.byref(h))
        if rc:
            raise HbError(rc, "hb_init failed")
        self.h = h

    def _check(self, rc):
        if rc:
            raise HbError(rc, self.L.hb_last_error(self.h).decode())
        return rc

    def load_layer(self, layer: int, w: dict):
        lw = LayerWeights(*[_ptr(w[n]) for n in ("w_qkv", "w_o", "w_gate_up", "w_down", "norm1", "norm2")])
        self._check(self.L.hb_load_layer(self.h, layer, ctypes.byref(lw)))

    def append_kv(self, layer: int, table: np.ndarray, start_pos: int, k, v):
        t = np.ascontiguousarray(table, np.int32)
        self._check(self.L.hb_append_kv(self.h, layer, t.ctypes.data, len(t), start_pos, int(k.shape[0]),
                                        _ptr(k), _ptr(v)))

    def read_kv(self, layer: int, table: np.ndarray, start_pos: int, k_out, v_out):
        t = np.ascontiguousarray(table, np.int32)
        self._check(self.L.hb_read_kv(self.h, layer, t.ctypes.data, len(t), start_pos, int(k_out.shape[0]),
                                      _ptr(k_out), _ptr(v_out)))

    def fill_kv(self, bits: int):
        self._check(self.L.hb_fill_kv(self.h, bits))

    def forward(self, spec: Spec, x_in, x_out, layers: Optional[tuple] = None):
        if layers is None:
            self._check(self.L.hb_forward(self.h, ctypes.byref(spec.c), _ptr(x_in), _ptr(x_out)))
        else:
            self._check(self.L.hb_forward_layers(self.h, ctypes.byref(spec.c), layers[0], layers[1], _ptr(x_in),
                                                 _ptr(x_out)))

    def forward_spec(self, spec: "BatchSpec", x_in, x_out):
        """Forward with a raw BatchSpec (e.g. one the scheduler filled)."""
        self._check(self.L.hb_forward(self.h, ctypes.byref(spec), _ptr(x_in), _ptr(x_out)))

    def forward_host(self, spec: Spec, x_in: np.ndarray, x_out: np.ndarray):
        assert x_in.flags.c_contiguous and x_out.flags.c_contiguous
        self._check(self.L.hb_forward_host(self.h, ctypes.byref(spec.c), x_in.ctypes.data, x_out.ctypes.data))

    def forward_host_ptr(self, spec: Spec, x_in_ptr: int, x_out_ptr: int):
        self._check(self.L.hb_forward_host(self.h, ctypes.byref(spec.c), x_in_ptr, x_out_ptr))

    def forward_host_async_ptr(self, spec: Spec, x_in_ptr: int, x_out_ptr: int):
        """hb_forward_host_async: returns once enqueued; read x_out after sync()."""
        self._check(self.L.hb_forward_host_async(self.h, ctypes.byref(spec.c), x_in_ptr, x_out_ptr))

    def sync(self):
        self._check(self.L.hb_sync(self.h))

    def profile(self, enable: bool):
        self._check(self.L.hb_profile(self.h, int(enable)))

    def profile_read(self) -> dict:
        n = 16
        names = (ctypes.c_char_p * n)()
        ms = (ctypes.c_double * n)()
        cnt = (ctypes.c_int * n)()
        k = self.L.hb_profile_read(self.h, ctypes.cast(names, ctypes.c_void_p), ctypes.cast(ms, ctypes.c_void_p),
                                   ctypes.cast(cnt, ctypes.c_void_p), n)
        if k < 0:
            self._check(k)
        return {names[i].decode(): (ms[i], cnt[i]) for i in range(k)}

    @property
    def launch_count(self) -> int:
        return int(self.L.hb_launch_count(self.h))

    def gemm_test(self, X, W, D):
        T, K = X.shape
        N = W.shape[0]
        self._check(self.L.hb_gemm_test(self.h, _ptr(X), _ptr(W), _ptr(D), T, N, K))

    def set_kernels(self, gemm_impl: int, attn_impl: int):
        self._check(self.L.hb_set_kernels(self.h, gemm_impl, attn_impl))

    def test_wait_timeout(self, wait_ns: int):
        """Arm the failure-path test fault in the next tensor-core GEMM launch."""
        self._check(self.L.hb_test_wait_timeout(self.h, int(wait_ns)))

    def debug_read(self, which: int, dst):
        self._check(self.L.hb_debug_read(self.h, which, _ptr(dst), int(dst.shape[0])))

    def free(self):
        if getattr(self, "h", None):
            self.L.hb_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass
