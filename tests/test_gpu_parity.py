"""GPU parity: hb_forward through the C ABI against the CPU oracle.

Every case draws its inputs from the seeded generator, runs them through
libhb.so on cuda:0 and through the oracle (bf16-mirror mode), and compares
element by element (tolerance in harness.py).  KV placement is checked as
well: each written slot must hold the oracle's K/V for that position and
every other slot must still hold the poison pattern.
"""
import numpy as np
import pytest

from chunked_prefill_hybrid_gb300 import native, synth, workloads
import harness
from harness import compare, f64, oracle_run

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _bits(t):
    return t.cpu().numpy().view(np.uint16)


def run_gpu(w, ctx=None, max_tokens=None, max_decodes=None, poison=True, kernels=None):
    own = ctx is None
    if own:
        ctx = native.Context(workloads.config(w, max_tokens, max_decodes))
        if kernels is not None:
            ctx.set_kernels(*kernels)
        x = workloads.upload(w, ctx, poison=harness.POISON if poison else None)
    else:
        x = workloads.to_device(w.x)
    y = torch.empty_like(x)
    ctx.forward(native.Spec(w.batch), x, y)
    ctx.sync()
    return ctx, f64(_bits(y))


def check_kv(ctx, w, pools, layer=0):
    """Written slots hold the oracle's K/V; the rest of the pool is poison."""
    dims = w.dims
    seqs = ([w.batch.chunk] if w.batch.chunk is not None else []) + list(w.batch.decodes)
    nkv, d = dims.n_kv_heads, dims.head_dim
    for s in seqs:
        n = s.cached + (w.batch.chunk_len if s is w.batch.chunk else 1)
        k = torch.empty((n, nkv, d), dtype=torch.int16, device="cuda")
        v = torch.empty_like(k)
        ctx.read_kv(layer, s.block_table, 0, k, v)
        ctx.sync()
        kr, vr = pools[layer].read(s.block_table, 0, n)
        ok_k, st_k = compare(f64(_bits(k)), kr)
        ok_v, st_v = compare(f64(_bits(v)), vr)
        assert ok_k and ok_v, (s.req_id, st_k, st_v)
    # the whole pool: positions never written keep the poison pattern
    if w.num_blocks * 16 <= w.max_pos:
        allb = np.arange(w.num_blocks, dtype=np.int32)
        k = torch.empty((w.num_blocks * 16, nkv, d), dtype=torch.int16, device="cuda")
        v = torch.empty_like(k)
        ctx.read_kv(layer, allb, 0, k, v)
        ctx.sync()
        kb, vb = _bits(k), _bits(v)
        used = set()
        for s in seqs:
            n = s.cached + (w.batch.chunk_len if s is w.batch.chunk else 1)
            for p in range(n):
                used.add(int(s.block_table[p // 16]) * 16 + p % 16)
        unused = np.array(sorted(set(range(w.num_blocks * 16)) - used), np.int64)
        assert (kb[unused] == harness.POISON).all() and (vb[unused] == harness.POISON).all()
        used = np.array(sorted(used), np.int64)
        assert (kb[used] != harness.POISON).all() and (vb[used] != harness.POISON).all()


# head_dim 128 and grouped-query shapes at a size the oracle finishes quickly
D128 = synth.ModelDims(hidden=256, n_heads=2, n_kv_heads=2, head_dim=128, ffn=512)
GQA = synth.ModelDims(hidden=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn=384)
KERNELS = {"tc+hybrid": (1, 1), "tc+simple": (1, 0), "simt+hybrid": (0, 1)}


def _tiny(seed, chunk_offset, chunk_len, ctxs, n_layers=1, gamma="ones", dims=synth.TINY):
    lengths = ([chunk_offset + chunk_len] if chunk_offset is not None else []) + [c + 1 for c in ctxs]
    nb = sum(synth.blocks_needed(n) for n in lengths) + 6
    return workloads.make("tiny", dims, seed, chunk_offset, chunk_len, ctxs, n_layers=n_layers,
                          num_blocks=nb, max_pos=nb * 16, gamma=gamma)


def test_tiny_hybrid_matches_oracle():
    w = workloads.tiny(seed=1)
    w.max_pos = w.num_blocks * 16
    ctx, y = run_gpu(w)
    ref, pools = oracle_run(w)
    ok, st = compare(y, ref, ulp=False)  # |y| < 8 here: the plain 3e-2 bound applies
    assert ok, st
    check_kv(ctx, w, pools)
    ctx.free()


@pytest.mark.parametrize("kern", sorted(KERNELS))
@pytest.mark.parametrize("case", [
    ("decode_only", None, 0, [0, 1, 15, 16, 17, 200]),
    ("prefill_only_offset0", 0, 100, []),
    ("chunk_len_1", 37, 1, [3]),
    ("ragged_chunk", 5, 77, [31, 32, 33]),
    ("many_decodes", 16, 16, list(range(0, 120, 3))),
    ("ctx0_decode_only", None, 0, [0]),
    ("multi_split_decodes", 3, 20, [255, 256, 257, 511, 700]),
    ("long_prefix_chunk", 300, 150, [40]),
])
def test_tiny_edge_cases(case, kern):
    name, off, ln, ctxs = case
    w = _tiny(11, off, ln, ctxs)
    ctx, y = run_gpu(w, kernels=KERNELS[kern])
    ref, pools = oracle_run(w)
    ok, st = compare(y, ref, ulp=False)
    assert ok, (name, st)
    check_kv(ctx, w, pools)
    ctx.free()


@pytest.mark.parametrize("kern", ["tc+hybrid", "simt+hybrid"])
@pytest.mark.parametrize("dims", [D128, GQA], ids=["d128", "gqa"])
@pytest.mark.parametrize("case", [
    ("hybrid", 200, 130, [0, 63, 64, 255, 256, 300, 1000]),
    ("prefill_only", 0, 257, []),
    ("decode_only", None, 0, [5, 511, 512, 513]),
])
def test_head_dim_and_gqa_cases(case, dims, kern):
    name, off, ln, ctxs = case
    w = _tiny(15, off, ln, ctxs, dims=dims)
    ctx, y = run_gpu(w, kernels=KERNELS[kern])
    ref, pools = oracle_run(w)
    ok, st = compare(y, ref)
    assert ok, (name, st)
    check_kv(ctx, w, pools)
    ctx.free()


def test_tiny_gamma_uniform_and_multilayer():
    w = _tiny(12, 40, 50, [10, 70, 130], n_layers=3, gamma="uniform")
    ctx, y = run_gpu(w)
    ref, pools = oracle_run(w)
    ok, st = compare(y, ref)
    assert ok, st
    for l in range(3):
        check_kv(ctx, w, pools, layer=l)
    ctx.free()


def test_chunked_prefill_equals_monolithic_on_gpu():
    """A 120-token prompt as chunks of 1/7/32/120 on the GPU agrees with the oracle's monolithic result."""
    dims = synth.TINY
    n = 120
    mono = _tiny(13, 0, n, [])
    ref, _ = oracle_run(mono)
    for C in (7, 32, 120):
        ctx = native.Context(workloads.config(mono, max_tokens=n))
        workloads.upload(mono, ctx)
        out = np.zeros((n, dims.hidden))
        for s in range(0, n, C):
            ln = min(C, n - s)
            b = synth.HybridBatch(synth.Seq(0, s, mono.batch.chunk.block_table), ln, [])
            x = workloads.to_device(mono.x[s:s + ln])
            y = torch.empty_like(x)
            ctx.forward(native.Spec(b), x, y)
            ctx.sync()
            out[s:s + ln] = f64(_bits(y))
        ok, st = compare(out, ref, ulp=False)
        assert ok, (C, st)
        ctx.free()


def test_piggybacked_decode_matches_alone():
    w = _tiny(14, 32, 48, [20, 90])
    ctx, y = run_gpu(w)
    ctx.free()
    for j, s in enumerate(w.batch.decodes):
        solo = workloads.make("solo", synth.TINY, 14, None, 0, [], num_blocks=w.num_blocks, max_pos=w.max_pos)
        solo.batch = synth.HybridBatch(None, 0, [s])
        solo.weights = w.weights
        solo.prefix = [(l, ss, k, v) for (l, ss, k, v) in w.prefix if ss.req_id == s.req_id]
        solo.x = w.x[w.batch.chunk_len + j:w.batch.chunk_len + j + 1]
        c2, ys = run_gpu(solo, max_decodes=1)
        c2.free()
        ok, st = compare(ys[0], y[w.batch.chunk_len + j], ulp=False)
        assert ok, (j, st)


@pytest.mark.parametrize("impl", [0, 1], ids=["simt", "tcgen05"])
@pytest.mark.parametrize("T,N,K", [(1, 256, 256), (18, 768, 256), (68, 1376, 688), (274, 512, 5120),
                                   (300, 384, 1024), (513, 256, 512), (16, 130, 64), (1100, 640, 192),
                                   (1500, 384, 128), (2048, 256, 64)])
def test_gemm_kernel_against_fp64(impl, T, N, K):
    w = workloads.tiny(seed=1)
    ctx = native.Context(workloads.config(w))
    ctx.set_kernels(impl, 0)
    X = synth.normal_bf16(31, (T, K), (T, K), 1.0)
    W = synth.normal_bf16(32, (N, K), (N, K), 0.05)
    D = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
    ctx.gemm_test(workloads.to_device(X), workloads.to_device(W), D)
    ctx.sync()
    ref = f64(X) @ f64(W).T
    got = D.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all(), "output not fully written"
    err = np.abs(got - ref)
    scale = np.sqrt(K) * 0.05
    assert err.max() <= 2e-6 * scale * np.sqrt(K), (err.max(), scale)
    ctx.free()


def test_llama13b_hybrid_full_layer():
    """LLaMA-13B layer, chunk 256 at offset 768 + 18 decodes at ctx 1024 (T = 274): every row."""
    w = workloads.llama13b_hybrid(seed=2)
    ctx, y = run_gpu(w, poison=True)
    ref, pools = oracle_run(w)
    ok, st = compare(y, ref)
    assert ok, st
    ctx.free()
