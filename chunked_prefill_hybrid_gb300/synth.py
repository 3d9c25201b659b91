"""Seeded synthetic inputs for hybrid-batch workloads.

This module is the one piece of code that both the CUDA path and the CPU
oracle consume: it draws weights, activations, prefix KV and block tables
from seeded generators and holds none of the layer's arithmetic.  Every array
is returned as host numpy data; bf16 tensors are uint16 bit patterns.

Workload shapes follow the pages' experiments: LLaMA-13B / LLaMA-33B layer
sizes (SARATHI summary, section 5 "Experimental Analysis"), synthetic
parameterised requests rather than a dataset, 16-token paged KV blocks
(Sarathi-Serve Guide, production checklist "Paged KV-Cache Page Sizing") and
a hybrid batch of one prefill chunk at a prefix offset plus D decodes
(SARATHI summary, section 3.4 "Decode-Maximal Batching").

Recipe: numpy ``default_rng(SeedSequence([seed, *key]))``; fp32 standard
normals scaled in fp32 and rounded to bf16 (ties to even).  Linear weights
~N(0, 0.02); RMSNorm gammas 1 (or U[0.5, 1.5] for the gamma-handling case);
token rows and prefix K/V ~N(0, 1); block tables a seeded permutation of the
physical blocks, so that logically adjacent blocks are physically scattered.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import numpy as np

# tensor ids inside a layer's seed key
_T_QKV, _T_O, _T_GU, _T_D, _T_N1, _T_N2 = 1, 2, 3, 4, 5, 6


def bf16_bits(x) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = a.view(np.uint32)
    rounded = ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        rounded = np.where(nan, np.uint16(0x7FC0), rounded)
    return rounded


def bf16_to_f32(bits) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed)] + [int(k) for k in key]))


def normal_bf16(seed: int, key: Sequence[int], shape, std: float = 1.0) -> np.ndarray:
    g = rng(seed, *key)
    n = int(np.prod(shape))
    x = g.standard_normal(n, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return bf16_bits(x).reshape(shape)


@dataclass(frozen=True)
class ModelDims:
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    n_layers: int = 1
    rms_eps: float = 1e-6
    rope_theta: float = 1e4
    block_size: int = 16

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def qkv_dim(self) -> int:
        return self.q_dim + 2 * self.kv_dim

    def params_per_layer(self) -> int:
        return (self.qkv_dim * self.hidden + self.hidden * self.q_dim
                + 2 * self.ffn * self.hidden + self.hidden * self.ffn)

    def kv_bytes_per_token_layer(self) -> int:
        return 2 * self.kv_dim * 2

    def with_layers(self, n: int) -> "ModelDims":
        return dataclasses.replace(self, n_layers=n)


# The tiny layer, LLaMA-13B and LLaMA-33B shapes.
TINY = ModelDims(hidden=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn=688)
LLAMA_13B = ModelDims(hidden=5120, n_heads=40, n_kv_heads=40, head_dim=128, ffn=13824, n_layers=40)
LLAMA_33B = ModelDims(hidden=6656, n_heads=52, n_kv_heads=52, head_dim=128, ffn=17920, n_layers=60)


def layer_weights(dims: ModelDims, seed: int, layer: int, gamma: str = "ones", std: float = 0.02) -> dict:
    """bf16 weights of one layer, row-major [out][in].

    w_qkv: [(n_heads + 2 n_kv) d][hidden] -- q rows, then k rows, then v rows
    w_o: [hidden][n_heads d]; w_gate_up: [2 ffn][hidden] -- gate rows, then up
    rows; w_down: [hidden][ffn]; norm1, norm2: [hidden].
    """
    H = dims.hidden
    w = {
        "w_qkv": normal_bf16(seed, (layer, _T_QKV), (dims.qkv_dim, H), std),
        "w_o": normal_bf16(seed, (layer, _T_O), (H, dims.q_dim), std),
        "w_gate_up": normal_bf16(seed, (layer, _T_GU), (2 * dims.ffn, H), std),
        "w_down": normal_bf16(seed, (layer, _T_D), (H, dims.ffn), std),
    }
    if gamma == "ones":
        w["norm1"] = bf16_bits(np.ones(H, np.float32))
        w["norm2"] = bf16_bits(np.ones(H, np.float32))
    elif gamma == "uniform":
        w["norm1"] = bf16_bits(rng(seed, layer, _T_N1).uniform(0.5, 1.5, H).astype(np.float32))
        w["norm2"] = bf16_bits(rng(seed, layer, _T_N2).uniform(0.5, 1.5, H).astype(np.float32))
    else:
        raise ValueError(gamma)
    return w


def token_rows(seed: int, key: Sequence[int], n_rows: int, hidden: int) -> np.ndarray:
    return normal_bf16(seed, tuple(key), (n_rows, hidden), 1.0)


@dataclass
class Seq:
    """One request's view inside a batch: id, tokens already cached, block table."""
    req_id: int
    cached: int
    block_table: np.ndarray  # int32 physical block ids, logical order


@dataclass
class HybridBatch:
    """One prefill chunk (optional) plus D decodes.

    chunk: Seq with cached = chunk offset; chunk_len tokens are prefilled now.
    decodes: Seqs whose new token sits at position cached.
    """
    chunk: Optional[Seq]
    chunk_len: int
    decodes: List[Seq] = field(default_factory=list)
    # further (Seq, length) chunks of other requests, rows after the first
    # chunk's (Sarathi-Serve batches under a token budget)
    more_chunks: List[Tuple[Seq, int]] = field(default_factory=list)

    @property
    def n_chunk_rows(self) -> int:
        return (self.chunk_len if self.chunk is not None else 0) + sum(n for _, n in self.more_chunks)

    @property
    def n_tokens(self) -> int:
        return self.n_chunk_rows + len(self.decodes)

    @property
    def n_decodes(self) -> int:
        return len(self.decodes)


def blocks_needed(n_tokens: int, block_size: int = 16) -> int:
    return (n_tokens + block_size - 1) // block_size


def allocate_tables(seed: int, key: Sequence[int], lengths: Sequence[int], num_blocks: int,
                    block_size: int = 16) -> List[np.ndarray]:
    """Disjoint block tables covering each length, drawn from a seeded permutation."""
    need = [blocks_needed(n, block_size) for n in lengths]
    if sum(need) > num_blocks:
        raise ValueError(f"need {sum(need)} blocks, pool has {num_blocks}")
    perm = rng(seed, *key).permutation(num_blocks).astype(np.int32)
    out, at = [], 0
    for n in need:
        out.append(perm[at:at + n].copy())
        at += n
    return out


def hybrid_batch(seed: int, key: Sequence[int], chunk_offset: Optional[int], chunk_len: int,
                 decode_ctx: Sequence[int], num_blocks: int, block_size: int = 16,
                 chunk_req_id: int = 0, first_decode_id: int = 1) -> HybridBatch:
    """A batch whose block tables cover every position the batch touches."""
    lengths = []
    if chunk_offset is not None:
        lengths.append(chunk_offset + chunk_len)
    lengths += [int(c) + 1 for c in decode_ctx]
    tables = allocate_tables(seed, key, lengths, num_blocks, block_size)
    chunk = None
    i = 0
    if chunk_offset is not None:
        chunk = Seq(chunk_req_id, int(chunk_offset), tables[0])
        i = 1
    decodes = [Seq(first_decode_id + j, int(c), tables[i + j]) for j, c in enumerate(decode_ctx)]
    return HybridBatch(chunk, chunk_len if chunk is not None else 0, decodes)


def prefix_kv(seed: int, key: Sequence[int], n_tokens: int, n_kv: int, head_dim: int):
    """Cached-prefix K (post-RoPE) and V, ~N(0,1) bf16, [n_tokens][n_kv][d] each."""
    k = normal_bf16(seed, tuple(key) + (1,), (n_tokens, n_kv, head_dim), 1.0)
    v = normal_bf16(seed, tuple(key) + (2,), (n_tokens, n_kv, head_dim), 1.0)
    return k, v


def uniform_ints(seed: int, key: Sequence[int], n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform in [lo, hi] inclusive."""
    return rng(seed, *key).integers(lo, hi + 1, size=n).astype(np.int32)


def log_uniform_ints(seed: int, key: Sequence[int], n: int, lo: int, hi: int) -> np.ndarray:
    g = rng(seed, *key)
    return np.clip(np.round(np.exp(g.uniform(np.log(lo), np.log(hi), size=n))), lo, hi).astype(np.int32)


def max_blocks(batch: HybridBatch) -> int:
    m = 0
    if batch.chunk is not None:
        m = len(batch.chunk.block_table)
    for s in batch.decodes:
        m = max(m, len(s.block_table))
    return m


def padded_decode_tables(batch: HybridBatch, max_blocks_per_seq: int) -> np.ndarray:
    """[n_decodes][max_blocks_per_seq] int32, unused entries -1."""
    out = np.full((max(1, batch.n_decodes), max_blocks_per_seq), -1, np.int32)
    for j, s in enumerate(batch.decodes):
        out[j, :len(s.block_table)] = s.block_table
    return out
