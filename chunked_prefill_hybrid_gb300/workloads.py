"""Synthetic hybrid-batch workloads and their upload into a library context.

A Workload holds host data only (weights, token rows, cached-prefix K/V,
block tables), drawn by ``synth``; ``upload`` copies it into an hb_ctx
through the C ABI (hb_load_layer, hb_append_kv).  Shapes follow the pages'
experiments (SARATHI summary, section 5; Sarathi-Serve Guide):

* tiny:  hidden 256, 4 heads x 64, FFN 688; chunk 64 at offset 64 of a
         128-token prompt + 4 decodes with ctx uniform in [32, 200]
* 13b:   LLaMA-13B layer; chunk 256 at offset 768 of a 1024-token prompt +
         18 decodes at ctx 1024 (T = 274)
* plus decode-only and prefill-only variants used as comparisons.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

from . import synth


@dataclass
class Workload:
    name: str
    dims: synth.ModelDims
    n_layers: int
    seed: int
    batch: synth.HybridBatch
    num_blocks: int
    max_pos: int
    weights: List[dict] = field(default_factory=list)
    x: Optional[np.ndarray] = None          # [T][H] bf16 bits
    prefix: List[tuple] = field(default_factory=list)  # (layer, Seq, k, v): positions 0..cached-1

    @property
    def T(self) -> int:
        return self.batch.n_tokens


def _prefix(seed: int, dims: synth.ModelDims, n_layers: int, batch: synth.HybridBatch):
    out = []
    seqs = ([batch.chunk] if batch.chunk is not None else []) + [s for s, _ in batch.more_chunks]
    seqs += list(batch.decodes)
    for layer in range(n_layers):
        for s in seqs:
            if s.cached > 0:
                k, v = synth.prefix_kv(seed, (1000 + layer, s.req_id), s.cached, dims.n_kv_heads, dims.head_dim)
                out.append((layer, s, k, v))
    return out


def make(name: str, dims: synth.ModelDims, seed: int, chunk_offset: Optional[int], chunk_len: int,
         decode_ctx: Sequence[int], n_layers: int = 1, num_blocks: Optional[int] = None, gamma: str = "ones",
         with_weights: bool = True, with_prefix: bool = True, max_pos: Optional[int] = None) -> Workload:
    lengths = ([chunk_offset + chunk_len] if chunk_offset is not None else []) + [int(c) + 1 for c in decode_ctx]
    need = sum(synth.blocks_needed(n) for n in lengths)
    nb = num_blocks or (need + need // 4 + 8)
    batch = synth.hybrid_batch(seed, (7,), chunk_offset, chunk_len, decode_ctx, nb)
    mp = max_pos or max(lengths + [16])
    w = Workload(name, dims, n_layers, seed, batch, nb, mp)
    if with_weights:
        w.weights = [synth.layer_weights(dims, seed, l, gamma=gamma) for l in range(n_layers)]
    w.x = synth.token_rows(seed, (8,), batch.n_tokens, dims.hidden)
    if with_prefix:
        w.prefix = _prefix(seed, dims, n_layers, batch)
    return w


def tiny(seed: int = 1) -> Workload:
    ctx = synth.uniform_ints(seed, (9,), 4, 32, 200)
    return make("tiny-hybrid-c64-d4", synth.TINY, seed, 64, 64, ctx)


def llama13b_hybrid(seed: int = 2, n_layers: int = 1, **kw) -> Workload:
    return make("llama13b-hybrid-c256@768-d18@1024", synth.LLAMA_13B, seed, 768, 256, [1024] * 18,
                n_layers=n_layers, **kw)


def llama13b_decode_only(seed: int = 2, **kw) -> Workload:
    return make("llama13b-decode-only-d18@1024", synth.LLAMA_13B, seed, None, 0, [1024] * 18, **kw)


def llama13b_prefill_only(T: int, seed: int = 2, **kw) -> Workload:
    return make(f"llama13b-prefill-only-{T}", synth.LLAMA_13B, seed, 0, T, [], **kw)


def llama13b_chunk_alone(seed: int = 2, **kw) -> Workload:
    return make("llama13b-chunk-c256@768", synth.LLAMA_13B, seed, 768, 256, [], **kw)


def config(w: Workload, max_tokens: Optional[int] = None, max_decodes: Optional[int] = None):
    from . import native
    return native.model_config(w.dims, w.num_blocks, max_tokens or max(w.T, 1), max_decodes
                               if max_decodes is not None else max(w.batch.n_decodes, 1), w.max_pos,
                               n_layers=w.n_layers)


def to_device(a: np.ndarray, device="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.to(device)


def upload(w: Workload, ctx, poison: Optional[int] = 0xFFFF):
    """Weights and cached prefix into ctx (an native.Context); returns x on the device."""
    import torch
    if poison is not None:
        ctx.fill_kv(poison)
    for l, lw in enumerate(w.weights):
        dev = {k: to_device(v) for k, v in lw.items()}
        ctx.load_layer(l, dev)
        ctx.sync()
        del dev
    for layer, s, k, v in w.prefix:
        ctx.append_kv(layer, s.block_table, 0, to_device(k), to_device(v))
    ctx.sync()
    return to_device(w.x)
