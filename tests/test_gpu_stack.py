"""Full-size LLaMA-13B stacks (40 layers) on the GPU against the oracle.

The oracle computes, through all forty layers, the first rows of a chunk and
any decode row on their own (see stack_helpers); the GPU runs the whole batch
in the launch configuration of the benchmark.  The rest of the rows are
checked for finiteness and, at long context, chunked against monolithic
prefill ("Chunked-Prefills": chunking changes nothing in the result).
"""
import numpy as np
import pytest

from chunked_prefill_hybrid_gb300 import native, synth, workloads
from harness import compare, f64
import stack_helpers as sh

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

L = 40
DIMS = synth.LLAMA_13B.with_layers(L)
KV_BYTES_PER_TOKEN = sh.kv_bytes_per_token(DIMS, L)


def _need_gpu_bytes(n_bytes):
    sh.need_gpu_bytes(torch, pytest, n_bytes)


def _upload(ctx, base, seed, sampled):
    sh.upload(torch, ctx, DIMS, L, base, seed, sampled)


def _oracle(base, seed, x_rows, chunk, n_chunk_rows, decodes, mirror=True):
    return sh.oracle_rows(DIMS, L, base, seed, x_rows, chunk, n_chunk_rows, decodes, mirror=mirror)


@pytest.fixture(scope="module")
def base_weights():
    return synth.layer_weights(synth.LLAMA_13B, 31, 0)


@pytest.mark.parametrize("C,D", [(512, 128), (128, 1)])
def test_llama13b_stack_hybrid_sampled_rows(base_weights, C, D):
    """40 layers, chunk C at offset 768 + D decodes with ctx uniform in [128, 2048]: the first two chunk rows and
    three decode rows (the shortest, the longest, the middle one) against the oracle; every row finite."""
    seed = 31
    ctxs = [int(c) for c in synth.uniform_ints(seed, (9, C), D, 128, 2048)]
    lengths = [768 + C] + [c + 1 for c in ctxs]
    nb = sum(synth.blocks_needed(n) for n in lengths) + 8
    _need_gpu_bytes(nb * 16 * KV_BYTES_PER_TOKEN + 30 * 2**30)
    batch = synth.hybrid_batch(seed, (7, C), 768, C, ctxs, nb)
    T = batch.n_tokens
    x = synth.token_rows(seed, (8, C), T, DIMS.hidden)
    order = np.argsort(ctxs, kind="stable")
    picks = sorted({int(order[0]), int(order[-1]), int(order[len(order) // 2])})
    cfg = native.model_config(DIMS, nb, T, D, max(lengths), n_layers=L)
    ctx = native.Context(cfg)
    _upload(ctx, base_weights, seed, [batch.chunk] + [batch.decodes[j] for j in picks])
    xd = workloads.to_device(x)
    yd = torch.empty_like(xd)
    ctx.forward(native.Spec(batch), xd, yd)
    ctx.sync()
    y = f64(yd.cpu().numpy().view(np.uint16))
    ctx.free()
    assert np.isfinite(y).all()
    rows = [0, 1] + [C + j for j in picks]
    ref = _oracle(base_weights, seed, x[rows], batch.chunk, 2, [batch.decodes[j] for j in picks])
    exact = _oracle(base_weights, seed, x[rows], batch.chunk, 2, [batch.decodes[j] for j in picks], mirror=False)
    ok, st = compare(y[rows], ref, exact)
    assert ok, (C, D, st)


def test_llama13b_stack_long_context_chunked_equals_monolithic(base_weights):
    """40 layers, one prompt of log-uniform length in [512, 8192] prefilled in chunks of 255 (the tile-probing
    size) with 64 decodes at log-uniform contexts in [256, 8192] riding on the first chunk, then the same
    prompt as one monolithic prefill in the same context: every prompt row agrees between the two, and the
    first two prompt rows and two decode rows of both runs agree with the oracle."""
    seed, C = 37, 255
    P = int(synth.log_uniform_ints(seed, (1,), 1, 512, 8192)[0])
    ctxs = [int(c) for c in synth.log_uniform_ints(seed, (2,), 64, 256, 8192)]
    lengths = [P] + [c + 1 for c in ctxs]
    nb = sum(synth.blocks_needed(n) for n in lengths) + 8
    _need_gpu_bytes(nb * 16 * KV_BYTES_PER_TOKEN + 30 * 2**30)
    batch = synth.hybrid_batch(seed, (7,), 0, P, ctxs, nb)
    D = len(ctxs)
    x = synth.token_rows(seed, (8,), P + D, DIMS.hidden)
    order = np.argsort(ctxs, kind="stable")
    picks = sorted({int(order[0]), int(order[1])})
    cfg = native.model_config(DIMS, nb, P + D, D, max(lengths), n_layers=L)
    ctx = native.Context(cfg)
    _upload(ctx, base_weights, seed, [batch.decodes[j] for j in picks])
    chunked = np.zeros((P, DIMS.hidden))
    dec = None
    for s0 in range(0, P, C):
        ln = min(C, P - s0)
        decs = batch.decodes if s0 == 0 else []
        b = synth.HybridBatch(synth.Seq(0, s0, batch.chunk.block_table), ln, decs)
        xd = workloads.to_device(np.concatenate([x[s0:s0 + ln]] + ([x[P:]] if decs else [])))
        yd = torch.empty_like(xd)
        ctx.forward(native.Spec(b), xd, yd)
        ctx.sync()
        yy = f64(yd.cpu().numpy().view(np.uint16))
        chunked[s0:s0 + ln] = yy[:ln]
        if decs:
            dec = yy[ln:]
    xd = workloads.to_device(x)
    yd = torch.empty_like(xd)
    ctx.forward(native.Spec(batch), xd, yd)
    ctx.sync()
    mono = f64(yd.cpu().numpy().view(np.uint16))
    ctx.free()
    assert np.isfinite(chunked).all() and np.isfinite(mono).all() and np.isfinite(dec).all()
    print("prompt", P, "rows bit-identical chunked vs monolithic:", int((chunked == mono[:P]).all(axis=1).sum()))
    same = (chunked == mono[:P]).all()
    assert same, ("chunked vs monolithic differ", P, compare(chunked, mono[:P])[1])
    args = (base_weights, seed, np.concatenate([x[:2], x[P + np.array(picks)]]),
            synth.Seq(0, 0, batch.chunk.block_table), 2, [batch.decodes[j] for j in picks])
    ref, exact = _oracle(*args), _oracle(*args, mirror=False)
    for name, got in (("chunked", np.concatenate([chunked[:2], dec[picks]])),
                      ("monolithic", np.concatenate([mono[:2], mono[P + np.array(picks)]]))):
        ok, st = compare(got, ref, exact, what=name)
        assert ok, (name, P, st)
