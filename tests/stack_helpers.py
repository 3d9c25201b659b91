"""Helpers for deep, full-width stacks on the GPU checked on sampled rows.

Rows of a hybrid batch are independent given the cache (SARATHI summary,
section 3.4 "Decode-Maximal Batching", how fusion works), and chunk row i at
offset o reads only the cached prefix and chunk rows 0..i (Figure 6).  So the
oracle computes the first rows of a chunk and any decode row on their own,
from the same seeded inputs, without the rest of the batch.

Inputs at full width: layer l's matrices are one seeded draw with their rows
rotated by l (distinct layers from one draw); gammas 1; a sampled sequence's
cached K/V at layer l is its seeded draw rotated by l along positions; every
other sequence's cache holds the constant bf16 1.0 (finite, not compared).
"""
import numpy as np

from chunked_prefill_hybrid_gb300 import synth, workloads
from harness import f64
from oracle import oracle as orc

ONE = 0x3F80  # bf16 1.0


def kv_bytes_per_token(dims, n_layers):
    return n_layers * 2 * dims.n_kv_heads * dims.head_dim * 2


def need_gpu_bytes(torch, pytest, n_bytes):
    free, _ = torch.cuda.mem_get_info()
    if free < n_bytes:
        pytest.skip(f"needs {n_bytes / 2**30:.0f} GiB of device memory, {free / 2**30:.0f} free")


def layer(base, l):
    return {k: (np.roll(v, l, axis=0) if v.ndim == 2 else v) for k, v in base.items()}


def prefix(dims, seed, s, l):
    k, v = synth.prefix_kv(seed, (1000, s.req_id), s.cached, dims.n_kv_heads, dims.head_dim)
    return np.roll(k, l, axis=0), np.roll(v, l, axis=0)


def upload(torch, ctx, dims, n_layers, base, seed, sampled):
    ctx.fill_kv(ONE)
    dev = {k: workloads.to_device(v) for k, v in base.items()}
    for l in range(n_layers):
        ctx.load_layer(l, {k: (torch.roll(v, l, 0) if v.dim() == 2 else v) for k, v in dev.items()})
        ctx.sync()
    del dev
    for s in sampled:
        if s.cached == 0:
            continue
        k0, v0 = synth.prefix_kv(seed, (1000, s.req_id), s.cached, dims.n_kv_heads, dims.head_dim)
        kd, vd = workloads.to_device(k0), workloads.to_device(v0)
        for l in range(n_layers):
            ctx.append_kv(l, s.block_table, 0, torch.roll(kd, l, 0), torch.roll(vd, l, 0))
        ctx.sync()


def oracle_rows(dims, n_layers, base, seed, x_rows, chunk, n_chunk_rows, decodes, mirror=True):
    """The sampled rows through all layers: a chunk of its first n_chunk_rows
    rows (or none) plus the given decodes, with compact block tables."""
    seqs = ([chunk] if chunk is not None else []) + list(decodes)
    lengths = [chunk.cached + n_chunk_rows] if chunk is not None else []
    lengths += [d.cached + 1 for d in decodes]
    tables, at = [], 0
    for n in lengths:
        nb = synth.blocks_needed(n)
        tables.append(np.arange(at, at + nb, dtype=np.int32))
        at += nb
    small = [synth.Seq(s.req_id, s.cached, t) for s, t in zip(seqs, tables)]
    sub = synth.HybridBatch(small[0] if chunk is not None else None, n_chunk_rows if chunk is not None else 0,
                            small[1:] if chunk is not None else small)
    y = f64(x_rows)
    for l in range(n_layers):
        pool = orc.Pool(at, dims.n_kv_heads, dims.head_dim)
        for s in small:
            if s.cached:
                k, v = prefix(dims, seed, s, l)
                pool.write(s.block_table, 0, f64(k), f64(v))
        y = orc.layer_forward(dims, layer(base, l), sub, y, pool, mirror=mirror)
    return y
