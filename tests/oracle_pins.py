"""Pins that tie the CPU oracle to something other than itself.

Each ``pin_*`` function takes ``mutate`` (0 = the real oracle, n > 0 = a
build with a planted mistake) and raises on disagreement.  The test module
runs every pin on the real oracle and checks that each planted mistake
fails at least one pin.

What pins what:
  * bf16 rounding: PyTorch's fp32->bf16 conversion, a double-rounding case,
    overflow and subnormal values.
  * matvec: numpy's fp64 matmul.
  * RMSNorm: ``torch.nn.functional.rms_norm``, scale invariance, a worked value.
  * RoPE: complex multiplication by e^{i pos theta^(-2j/d)}, identity at
    position 0, relative-position invariance of q.k.
  * SiLU: ``scipy.special.expit(z) * z``.
  * slot: a brute-force walk over the block table's token slots.
  * attention: dense masked softmax (brute force), q = 0 gives the mean of
    the attended values, ctx = 0 gives the decode's own value, constant V.
  * chunked causal mask: the Figure 6 example (tests/golden/fig6_chunked_mask.txt).
  * layer: a textbook fp64 PyTorch layer over the full, unchunked sequence
    (chunked prefill equals full prefill -- SARATHI summary, section 3.4,
    "Chunked-Prefills"), for a prefill, a hybrid batch and a GQA layer.
  * invariants: chunked == monolithic and alone == piggybacked, bit for bit.
  * mirror mode's rounding points: every stored stage equals the bf16 rounding
    (frexp-based round-half-even to 8 significant bits) of a textbook fp64
    recomputation from the previous stored stage.
"""
from __future__ import annotations

import os

import numpy as np
import scipy.special
import torch
import torch.nn.functional as F

from oracle import oracle as orc
from chunked_prefill_hybrid_gb300 import synth
import textbook

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

PIN_DIMS = synth.ModelDims(hidden=64, n_heads=2, n_kv_heads=2, head_dim=32, ffn=96)
GQA_DIMS = synth.ModelDims(hidden=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn=80)
PIN_STD = 0.15  # larger than 0.02 so attention is far from uniform at this width


def _f64(bits):
    return synth.bf16_to_f32(bits).astype(np.float64)


# ------------------------------------------------------------------ scalars

def pin_bf16_vs_torch(mutate=0):
    g = np.random.default_rng(11)
    x = g.standard_normal(4000).astype(np.float32) * np.float32(30.0)
    # exact ties: low 16 bits = 0x8000, both parities of the kept lsb
    u = g.integers(0, 2 ** 31, 200, dtype=np.uint32)
    ties = ((u & np.uint32(0xFFFF0000)) | np.uint32(0x8000)).view(np.float32)
    ties = ties[np.isfinite(ties)]
    vals = np.concatenate([x, ties])
    ours = orc.f64_to_bf16_bits(vals.astype(np.float64), mutate)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref), "bf16 rounding differs from PyTorch"
    back = orc.bf16_bits_to_f64(ref, mutate)
    assert np.array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy())


def pin_bf16_double_rounding(mutate=0):
    # just above a bf16 tie, but the fp32 rounding would land on the tie
    v = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert orc.f64_to_bf16_bits(np.array([v]), mutate)[0] == 0x3F81
    assert orc.f64_to_bf16_bits(np.array([1.0 + 2.0 ** -8]), mutate)[0] == 0x3F80  # tie -> even
    assert orc.f64_to_bf16_bits(np.array([1.0 + 3 * 2.0 ** -8]), mutate)[0] == 0x3F82  # tie -> even


def pin_bf16_specials(mutate=0):
    b = orc.f64_to_bf16_bits(np.array([3.5e38, -3.5e38, 3.3895e38, 2.0 ** -130, -2.0 ** -133, 0.0, -0.0]), mutate)
    assert list(b) == [0x7F80, 0xFF80, 0x7F7F, 0x0008, 0x8001, 0x0000, 0x8000], [hex(t) for t in b]


def pin_matvec_numpy(mutate=0):
    W = synth.normal_bf16(3, (1,), (37, 53), 0.5)
    x = np.random.default_rng(4).standard_normal(53)
    y = orc.matvec(W, x, mutate)
    ref = _f64(W) @ x
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


def pin_rmsnorm_torch(mutate=0):
    g = np.random.default_rng(5)
    x = g.standard_normal(96) * 3.0
    gamma = synth.bf16_bits(g.uniform(0.5, 1.5, 96).astype(np.float32))
    ours = orc.rmsnorm(x, gamma, 1e-6, mutate)
    ref = F.rms_norm(torch.from_numpy(x), (96,), weight=torch.from_numpy(_f64(gamma)), eps=1e-6).numpy()
    assert np.allclose(ours, ref, rtol=1e-13, atol=1e-13)


def pin_rmsnorm_properties(mutate=0):
    x = np.array([3.0, 4.0])
    out = orc.rmsnorm(x, None, 0.0, mutate)
    # mean square 12.5 -> each element divided by sqrt(12.5)
    assert np.allclose(out, [0.848528137423857, 1.131370849898476], rtol=1e-14)
    g = np.random.default_rng(6).standard_normal(64)
    a = orc.rmsnorm(g, None, 0.0, mutate)
    b = orc.rmsnorm(g * 37.5, None, 0.0, mutate)
    assert np.allclose(a, b, rtol=1e-13)
    assert abs(np.sqrt(np.mean(a * a)) - 1.0) < 1e-13


def pin_rope_complex(mutate=0):
    g = np.random.default_rng(7)
    for d in (8, 64, 128):
        v = g.standard_normal(d)
        for pos in (1, 17, 1000):
            ours = orc.rope(v, pos, 1e4, mutate)
            half = d // 2
            z = (v[:half] + 1j * v[half:]) * np.exp(1j * pos * 1e4 ** (-2.0 * np.arange(half) / d))
            ref = np.concatenate([z.real, z.imag])
            assert np.allclose(ours, ref, rtol=1e-12, atol=1e-12), (d, pos)


def pin_rope_properties(mutate=0):
    g = np.random.default_rng(8)
    d = 64
    q, k = g.standard_normal(d), g.standard_normal(d)
    assert np.array_equal(orc.rope(q, 0, 1e4, mutate), q)
    base = orc.rope(q, 9, 1e4, mutate) @ orc.rope(k, 4, 1e4, mutate)
    for s in (1, 50, 777):
        shifted = orc.rope(q, 9 + s, 1e4, mutate) @ orc.rope(k, 4 + s, 1e4, mutate)
        assert abs(shifted - base) < 1e-9 * max(1.0, abs(base))
    r = orc.rope(q, 123, 1e4, mutate)
    assert abs(np.linalg.norm(r) - np.linalg.norm(q)) < 1e-12


def pin_silu_scipy(mutate=0):
    for z in (-30.0, -3.0, -0.5, 0.0, 0.25, 2.0, 40.0):
        ref = z * scipy.special.expit(z)
        assert abs(orc.silu(z, mutate) - ref) <= 1e-15 * max(1.0, abs(ref)), z
    assert orc.silu(0.0, mutate) == 0.0


def pin_slot_walk(mutate=0):
    bt = np.array([7, 2, 9, 0, 5], np.int32)
    walk = [b * 16 + o for b in bt for o in range(16)]
    for pos in range(len(walk)):
        assert orc.slot(bt, pos, 10, 16, mutate) == walk[pos], pos
    assert orc.slot(bt, len(walk), 10, 16, mutate) < 0  # past the table
    assert orc.slot(np.array([10], np.int32), 0, 10, 16, mutate) < 0  # block id out of range


# ---------------------------------------------------------------- attention

def _pool_with(n_tokens, n_kv, d, k, v, seed, num_blocks=None, mutate=0):
    nb = synth.blocks_needed(n_tokens)
    num_blocks = num_blocks or nb + 5
    bt = synth.allocate_tables(seed, (99,), [n_tokens], num_blocks)[0]
    pool = orc.Pool(num_blocks, n_kv, d)
    pool.write(bt, 0, k, v, mutate)
    return pool, bt


def pin_attention_dense(mutate=0):
    g = np.random.default_rng(9)
    n, nkv, d = 45, 2, 16
    k = g.standard_normal((n, nkv, d))
    v = g.standard_normal((n, nkv, d))
    pool, bt = _pool_with(n, nkv, d, k, v, 1, mutate=mutate)
    for last in (0, 15, 16, 31, 44):
        for h in range(nkv):
            q = g.standard_normal(d) * 2.0
            ours = orc.attention_head(q, pool, h, bt, last, mutate)
            # brute force over the whole sequence with an explicit mask
            s = (k[:, h, :] @ q) / np.sqrt(d)
            mask = np.arange(n) <= last
            s = np.where(mask, s, -np.inf)
            p = np.exp(s - s.max())
            p /= p.sum()
            ref = p @ v[:, h, :]
            assert np.allclose(ours, ref, rtol=1e-12, atol=1e-12), (last, h)


def pin_attention_closed_forms(mutate=0):
    g = np.random.default_rng(10)
    n, nkv, d = 40, 1, 8
    k = g.standard_normal((n, nkv, d))
    v = g.standard_normal((n, nkv, d))
    pool, bt = _pool_with(n, nkv, d, k, v, 2, mutate=mutate)
    for last in (0, 7, 39):
        # q = 0: uniform weights -> mean of V over keys 0..last
        o = orc.attention_head(np.zeros(d), pool, 0, bt, last, mutate)
        assert np.allclose(o, v[:last + 1, 0].mean(axis=0), rtol=1e-13, atol=1e-13), last
    # a decode with nothing cached sees only its own key: output is its own v
    o = orc.attention_head(g.standard_normal(d), pool, 0, bt, 0, mutate)
    assert np.allclose(o, v[0, 0], rtol=0, atol=1e-15)
    # constant V
    pool2, bt2 = _pool_with(n, nkv, d, k, np.full((n, nkv, d), 0.75), 3, mutate=mutate)
    o = orc.attention_head(g.standard_normal(d) * 3, pool2, 0, bt2, 39, mutate)
    assert np.allclose(o, 0.75, rtol=0, atol=1e-14)


def load_fig6():
    rows = []
    with open(os.path.join(GOLDEN, "fig6_chunked_mask.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            left, right = line.split(":")
            chunk, qpos = (int(t) for t in left.split())
            rows.append((chunk, qpos, [int(t) for t in right.split()]))
    return rows


def pin_fig6_mask(mutate=0):
    """Which keys each chunk query attends, read off the oracle's layer output.

    A 12-token prompt is run as three 4-token chunks.  With q = 0 (zero
    Q weights) attention weights are uniform over the attended keys, and with
    V = one-hot(position) (V weights picking an input coordinate, inputs
    one-hot) the attention output names those keys.
    """
    n = 12
    dims = synth.ModelDims(hidden=16, n_heads=1, n_kv_heads=1, head_dim=16, ffn=8, rms_eps=0.0)
    one = int(synth.bf16_bits(np.array([1.0], np.float32))[0])
    w_qkv = np.zeros((3 * 16, 16), np.uint16)
    for i in range(16):
        w_qkv[32 + i, i] = one  # v = n1 (identity V projection); q = k = 0
    w_o = np.zeros((16, 16), np.uint16)
    for i in range(16):
        w_o[i, i] = one  # h = x + o
    weights = {"w_qkv": w_qkv, "w_o": w_o,
               "w_gate_up": np.zeros((16, 16), np.uint16), "w_down": np.zeros((16, 8), np.uint16),
               "norm1": np.full(16, one, np.uint16), "norm2": np.full(16, one, np.uint16)}
    x = np.zeros((n, 16))
    x[np.arange(n), np.arange(n)] = 4.0  # rmsnorm of 4*e_i over 16 dims = 4*e_i * 1/sqrt(1) -> e_i*4
    bt = np.arange(1, dtype=np.int32)
    pool = orc.Pool(1, 1, 16)
    attended = {}
    for c in range(3):
        batch = synth.HybridBatch(synth.Seq(0, 4 * c, bt), 4, [])
        y, aux = orc.layer_forward(dims, weights, batch, x[4 * c:4 * c + 4], pool, mirror=False, aux=True,
                                   mutate=mutate)
        for i in range(4):
            o = aux["o"][i]
            attended[4 * c + i] = [j for j in range(16) if o[j] > 1e-9]
    for chunk, qpos, keys in load_fig6():
        assert attended[qpos] == keys, (chunk, qpos, attended[qpos], keys)


# -------------------------------------------------------------------- layer

def _seq_rows(seed, key, n, H):
    return _f64(synth.token_rows(seed, key, n, H))


def _run_prefix(dims, weights, pool, table, rows, mutate):
    """Run rows (positions 0..n-1) as one monolithic chunk."""
    batch = synth.HybridBatch(synth.Seq(0, 0, table), rows.shape[0], [])
    return orc.layer_forward(dims, weights, batch, rows, pool, mirror=False, mutate=mutate)


def pin_layer_textbook_prefill(mutate=0):
    dims = PIN_DIMS
    w = synth.layer_weights(dims, 21, 0, gamma="uniform", std=PIN_STD)
    n = 37
    x = _seq_rows(21, (1,), n, dims.hidden)
    table = synth.allocate_tables(21, (2,), [n], 8)[0]
    pool = orc.Pool(8, dims.n_kv_heads, dims.head_dim)
    y = _run_prefix(dims, w, pool, table, x, mutate)
    ref, _, kref, vref, _ = textbook.layer_full_sequence(dims, w, x)
    assert np.allclose(y, ref, rtol=1e-10, atol=1e-10), np.abs(y - ref).max()
    k, v = pool.read(table, 0, n, mutate)
    assert np.allclose(k.reshape(n, -1), kref, rtol=1e-10, atol=1e-10)
    assert np.allclose(v.reshape(n, -1), vref, rtol=1e-10, atol=1e-10)


def _hybrid_case(dims, seed, mutate, gamma="ones"):
    """Chunk of 16 at offset 24 of a 40-token prompt, plus decodes at ctx 5 and 17."""
    w = synth.layer_weights(dims, seed, 0, gamma=gamma, std=PIN_STD)
    H = dims.hidden
    full = {"A": _seq_rows(seed, (1,), 40, H), "B": _seq_rows(seed, (2,), 6, H), "C": _seq_rows(seed, (3,), 18, H)}
    tables = synth.allocate_tables(seed, (4,), [40, 6, 18], 12)
    tab = dict(zip("ABC", tables))
    pool = orc.Pool(12, dims.n_kv_heads, dims.head_dim)
    _run_prefix(dims, w, pool, tab["A"], full["A"][:24], mutate)
    _run_prefix(dims, w, pool, tab["B"], full["B"][:5], mutate)
    _run_prefix(dims, w, pool, tab["C"], full["C"][:17], mutate)
    batch = synth.HybridBatch(synth.Seq(0, 24, tab["A"]), 16,
                              [synth.Seq(1, 5, tab["B"]), synth.Seq(2, 17, tab["C"])])
    x = np.concatenate([full["A"][24:40], full["B"][5:6], full["C"][17:18]])
    return w, full, tab, pool, batch, x


def pin_layer_textbook_hybrid(mutate=0):
    dims = PIN_DIMS
    w, full, tab, pool, batch, x = _hybrid_case(dims, 22, mutate)
    y = orc.layer_forward(dims, w, batch, x, pool, mirror=False, mutate=mutate)
    refA = textbook.layer_full_sequence(dims, w, full["A"])[0]
    refB = textbook.layer_full_sequence(dims, w, full["B"])[0]
    refC = textbook.layer_full_sequence(dims, w, full["C"])[0]
    ref = np.concatenate([refA[24:40], refB[5:6], refC[17:18]])
    assert np.allclose(y, ref, rtol=1e-10, atol=1e-10), np.abs(y - ref).max()


def pin_layer_textbook_two_chunks(mutate=0):
    """A Sarathi-Serve batch: the leftover chunk of a partially prefilled
    request (16 at offset 24 of 40), the first 10 tokens of a new request,
    and two decodes ("Notes on Sarathi-Serve", "Stall Free Batching",
    illustrated example), against the textbook layer per request."""
    dims = PIN_DIMS
    w, full, tab, pool, batch, x = _hybrid_case(dims, 27, mutate)
    H = dims.hidden
    full["D"] = _seq_rows(27, (5,), 18, H)
    tD = np.arange(12, 14, dtype=np.int32)
    big = orc.Pool(14, dims.n_kv_heads, dims.head_dim)
    big.k[:pool.k.shape[0]] = pool.k
    big.v[:pool.v.shape[0]] = pool.v
    two = synth.HybridBatch(batch.chunk, batch.chunk_len, batch.decodes, [(synth.Seq(3, 0, tD), 10)])
    xx = np.concatenate([x[:16], full["D"][:10], x[16:]])
    y = orc.layer_forward(dims, w, two, xx, big, mirror=False, mutate=mutate)
    ref = np.concatenate([textbook.layer_full_sequence(dims, w, full["A"])[0][24:40],
                          textbook.layer_full_sequence(dims, w, full["D"])[0][0:10],
                          textbook.layer_full_sequence(dims, w, full["B"])[0][5:6],
                          textbook.layer_full_sequence(dims, w, full["C"])[0][17:18]])
    assert np.allclose(y, ref, rtol=1e-10, atol=1e-10), np.abs(y - ref).max()


def pin_layer_textbook_gqa(mutate=0):
    dims = GQA_DIMS
    w, full, tab, pool, batch, x = _hybrid_case(dims, 23, mutate, gamma="uniform")
    y = orc.layer_forward(dims, w, batch, x, pool, mirror=False, mutate=mutate)
    ref = np.concatenate([textbook.layer_full_sequence(dims, w, full["A"])[0][24:40],
                          textbook.layer_full_sequence(dims, w, full["B"])[0][5:6],
                          textbook.layer_full_sequence(dims, w, full["C"])[0][17:18]])
    assert np.allclose(y, ref, rtol=1e-10, atol=1e-10), np.abs(y - ref).max()


def pin_chunking_invariance(mutate=0):
    """Chunks of C in {1, 3, 16, 64} give the monolithic result bit for bit."""
    dims = PIN_DIMS
    w = synth.layer_weights(dims, 24, 0, std=PIN_STD)
    n = 40
    x = _seq_rows(24, (1,), n, dims.hidden)
    table = synth.allocate_tables(24, (2,), [n], 6)[0]
    for mirror in (False, True):
        xin = orc.bf16_round(x) if mirror else x
        mono_pool = orc.Pool(6, dims.n_kv_heads, dims.head_dim)
        mono = orc.layer_forward(dims, w, synth.HybridBatch(synth.Seq(0, 0, table), n, []), xin, mono_pool,
                                 mirror=mirror, mutate=mutate)
        for C in (1, 3, 16, 64):
            pool = orc.Pool(6, dims.n_kv_heads, dims.head_dim)
            out = np.zeros_like(mono)
            for s in range(0, n, C):
                ln = min(C, n - s)
                out[s:s + ln] = orc.layer_forward(dims, w, synth.HybridBatch(synth.Seq(0, s, table), ln, []),
                                                  xin[s:s + ln], pool, mirror=mirror, mutate=mutate)
            assert np.array_equal(out, mono), (mirror, C)
            assert np.array_equal(pool.k, mono_pool.k) and np.array_equal(pool.v, mono_pool.v), (mirror, C)


def pin_piggyback_invariance(mutate=0):
    """A decode's output and K/V are the same alone and piggybacked on a chunk."""
    dims = PIN_DIMS
    w, full, tab, pool, batch, x = _hybrid_case(dims, 25, mutate)
    alone_pool = pool.copy()
    y = orc.layer_forward(dims, w, batch, x, pool, mirror=True, mutate=mutate)
    for j, seq in enumerate(batch.decodes):
        solo = synth.HybridBatch(None, 0, [seq])
        ys = orc.layer_forward(dims, w, solo, x[16 + j:17 + j], alone_pool, mirror=True, mutate=mutate)
        assert np.array_equal(ys[0], y[16 + j]), j
        s = orc.slot(seq.block_table, seq.cached, pool.num_blocks, 16, mutate)
        assert np.array_equal(alone_pool.k[s], pool.k[s]) and np.array_equal(alone_pool.v[s], pool.v[s])


def pin_mirror_close_to_exact(mutate=0):
    dims = PIN_DIMS
    w, full, tab, pool, batch, x = _hybrid_case(dims, 26, mutate)
    p2 = pool.copy()
    ye = orc.layer_forward(dims, w, batch, x, pool, mirror=False, mutate=mutate)
    ym = orc.layer_forward(dims, w, batch, orc.bf16_round(x), p2, mirror=True, mutate=mutate)
    assert np.array_equal(ym, orc.bf16_round(ym)), "mirror output is not bf16"
    assert np.abs(ym - ye).max() < 0.05 and np.abs(ym - ye).mean() < 0.01


def _rb(x):
    """Round fp64 values to the nearest bf16 value (8 significant bits, ties
    to even) through frexp and numpy's round-half-even: a formulation that
    shares nothing with the oracle's bit manipulation."""
    x = np.asarray(x, np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.round(m * 256.0), e - 8)


def _same_after_rounding(stored, exact, what):
    """stored == _rb(exact), except where exact lies within 1e-12 (relative)
    of a rounding boundary, where fp64 summation order may decide."""
    ref = _rb(exact)
    bad = stored != ref
    if bad.any():
        e = exact[bad]
        edge = _rb(e * (1 + 1e-12)) != _rb(e * (1 - 1e-12))
        assert edge.all(), f"{what}: {int((~edge).sum())} of {e.size} stored values are not bf16(recomputation)"


def pin_mirror_rounding_points(mutate=0):
    """Mirror mode stores bf16 at n1, q/k after RoPE, v, o, h, n2, a and y:
    each stored stage is the bf16 rounding of the exact fp64 step applied to
    the previous stored stage (textbook PyTorch ops), over a 37-token prefill."""
    dims = PIN_DIMS
    w = synth.layer_weights(dims, 28, 0, gamma="uniform", std=PIN_STD)
    n, H, nh, nkv, d, Fd = 37, dims.hidden, dims.n_heads, dims.n_kv_heads, dims.head_dim, dims.ffn
    x = orc.bf16_round(_seq_rows(28, (1,), n, H))
    table = synth.allocate_tables(28, (2,), [n], 8)[0]
    pool = orc.Pool(8, nkv, d)
    batch = synth.HybridBatch(synth.Seq(0, 0, table), n, [])
    y, aux = orc.layer_forward(dims, w, batch, x, pool, mirror=True, aux=True, mutate=mutate)
    T = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    W = {k: textbook._w(w[k]) for k in ("w_qkv", "w_o", "w_gate_up", "w_down", "norm1", "norm2")}
    n1 = F.rms_norm(T(x), (H,), weight=W["norm1"], eps=dims.rms_eps)
    _same_after_rounding(aux["n1"], n1.numpy(), "n1")
    qkv = F.linear(T(aux["n1"]), W["w_qkv"])
    pos = torch.arange(n)
    q = textbook.rope_complex(qkv[:, :nh * d].reshape(n, nh, d), pos, dims.rope_theta).reshape(n, -1)
    k = textbook.rope_complex(qkv[:, nh * d:(nh + nkv) * d].reshape(n, nkv, d), pos, dims.rope_theta).reshape(n, -1)
    _same_after_rounding(aux["q"], q.numpy(), "q")
    _same_after_rounding(aux["k"], k.numpy(), "k")
    _same_after_rounding(aux["v"], qkv[:, (nh + nkv) * d:].numpy(), "v")
    qh, kh, vh = (T(aux[t]).reshape(n, -1, d).transpose(0, 1)[None] for t in ("q", "k", "v"))
    o = F.scaled_dot_product_attention(qh, kh, vh, is_causal=True)[0].transpose(0, 1).reshape(n, nh * d)
    _same_after_rounding(aux["o"], o.numpy(), "o")
    _same_after_rounding(aux["h"], (T(x) + F.linear(T(aux["o"]), W["w_o"])).numpy(), "h")
    n2 = F.rms_norm(T(aux["h"]), (H,), weight=W["norm2"], eps=dims.rms_eps)
    _same_after_rounding(aux["n2"], n2.numpy(), "n2")
    gu = F.linear(T(aux["n2"]), W["w_gate_up"])
    _same_after_rounding(aux["a"], (F.silu(gu[:, :Fd]) * gu[:, Fd:]).numpy(), "a")
    _same_after_rounding(y, (T(aux["h"]) + F.linear(T(aux["a"]), W["w_down"])).numpy(), "y")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
