"""LLaMA-33B width on the GPU against the oracle (hidden 6656, 52 heads x 128,
FFN 17920: SARATHI summary, section 5 "Evaluation Methodology", LLaMA-33B).

At this width the linear ops split differently from the LLaMA-13B layer: the
gate/up product has 140 weight-tile pairs (one data-parallel wave of 76 plus
a stream-K tail of 64), the O and down products 26, and the down product's K
is 17920; attention has 52 heads.  Three layers (one seeded draw, rows rotated
per layer) run on the GPU in the benchmark's launch configuration; the oracle
computes sampled, causally closed rows through all three (stack_helpers), and
the comparison uses the oracle's floor at the same depth (harness).

Two batches:
  * chunk 256 at offset 768 + 256 decodes with contexts uniform in
    [512, 2048]: T = 512, the token budget of the serving configuration;
  * the batch the host decode-maximal scheduler builds for the LLaMA-33B
    serving loop (chunk 256, token budget 512, prompts uniform in
    [512, 2048], P:D = 10) at the first iteration that holds a partly
    prefilled chunk and at least 24 decodes (with one chunk per iteration
    about 25 requests decode at a time in this loop: each prompt takes
    about five iterations and yields about a hundred tokens).
"""
import numpy as np
import pytest

from chunked_prefill_hybrid_gb300 import native, synth, workloads
from chunked_prefill_hybrid_gb300 import sched as hs
from harness import compare, f64
import stack_helpers as sh

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

L = 3
DIMS = synth.LLAMA_33B.with_layers(L)


@pytest.fixture(scope="module")
def base_weights():
    return synth.layer_weights(synth.LLAMA_33B, 43, 0)


def _run(base, seed, batch, nb, max_pos, tag, key):
    T, D = batch.n_tokens, len(batch.decodes)
    C = batch.chunk_len
    sh.need_gpu_bytes(torch, pytest, nb * 16 * sh.kv_bytes_per_token(DIMS, L) + 8 * 2**30)
    x = synth.token_rows(seed, (8, key), T, DIMS.hidden)
    order = np.argsort([s.cached for s in batch.decodes], kind="stable")
    picks = sorted({int(order[0]), int(order[-1]), int(order[len(order) // 2])})
    ctx = native.Context(native.model_config(DIMS, nb, T, D, max_pos, n_layers=L))
    sh.upload(torch, ctx, DIMS, L, base, seed, [batch.chunk] + [batch.decodes[j] for j in picks])
    xd = workloads.to_device(x)
    yd = torch.empty_like(xd)
    ctx.forward(native.Spec(batch), xd, yd)
    ctx.sync()
    y = f64(yd.cpu().numpy().view(np.uint16))
    ctx.free()
    assert np.isfinite(y).all()
    rows = [0, 1] + [C + j for j in picks]
    args = (DIMS, L, base, seed, x[rows], batch.chunk, 2, [batch.decodes[j] for j in picks])
    ref, exact = sh.oracle_rows(*args), sh.oracle_rows(*args, mirror=False)
    ok, st = compare(y[rows], ref, exact, what=tag)
    assert ok, st


def test_llama33b_hybrid_t512_sampled_rows(base_weights):
    seed = 43
    ctxs = [int(c) for c in synth.uniform_ints(seed, (9,), 256, 512, 2048)]
    lengths = [768 + 256] + [c + 1 for c in ctxs]
    nb = sum(synth.blocks_needed(n) for n in lengths) + 8
    batch = synth.hybrid_batch(seed, (7,), 768, 256, ctxs, nb)
    assert batch.n_tokens == 512
    _run(base_weights, seed, batch, nb, max(lengths), "t512", 1)


def test_llama33b_scheduler_iteration_sampled_rows(base_weights):
    seed = 44
    nb, mbs = 20000, 160
    s = hs.Scheduler(256, token_budget=512, num_blocks=nb, max_blocks_per_seq=mbs)
    prompts = synth.uniform_ints(seed, (1,), 512, 512, 2048)
    for i, p in enumerate(prompts):
        s.add(i, int(p), max(1, int(round(int(p) / 10))))
    lengths = {i: int(p) + max(1, int(round(int(p) / 10))) for i, p in enumerate(prompts)}
    for _ in range(5000):
        b = s.next()
        if b.chunks and b.chunks[0][1] > 0 and len(b.decodes) >= 24:
            break
        s.complete()
    else:
        pytest.fail("the scheduler never built a hybrid batch with a partly prefilled chunk and 24 decodes")
    (cid, coff, clen), = b.chunks
    chunk = synth.Seq(cid, coff, np.asarray(s.block_table(cid), np.int32))
    decs = [synth.Seq(r, c, np.asarray(s.block_table(r), np.int32)) for r, c in b.decodes]
    batch = synth.HybridBatch(chunk, clen, decs)
    assert batch.n_tokens == b.n_rows <= 512
    max_pos = max(lengths[r] for r in [cid] + [r for r, _ in b.decodes])
    s.free()
    print("scheduler batch: chunk", (cid, coff, clen), "decodes", len(decs), "rows", batch.n_tokens)
    _run(base_weights, seed, batch, nb, max_pos, "sched", 2)
