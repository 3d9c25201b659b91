"""Batch invariance of the GPU path: a decode's output is bit-identical whether
it runs alone or piggybacked on a hybrid batch (SARATHI summary, section 3.4
"Decode-Maximal Batching": fusing the rows changes nothing per row).

This holds by construction of the default kernels: the GEMMs split their K
loop by the weight shape and the resident CTA-pair count only, never by the
number of rows; each split sums in a fixed order; decode attention splits
by the context length alone; and every normalisation is per row.
"""
import numpy as np
import pytest

from chunked_prefill_hybrid_gb300 import native, synth, workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _forward(w, batch, x_rows, max_tokens, max_decodes, weights_ctx=None):
    cfg = workloads.config(w, max_tokens=max_tokens, max_decodes=max_decodes)
    ctx = native.Context(cfg)
    workloads.upload(w, ctx, poison=None)
    x = workloads.to_device(x_rows)
    y = torch.empty_like(x)
    ctx.forward(native.Spec(batch), x, y)
    ctx.sync()
    out = y.cpu().numpy().view(np.uint16).copy()
    ctx.free()
    return out


def _check(w, picks):
    T = w.T
    hybrid = _forward(w, w.batch, w.x, T, max(w.batch.n_decodes, 1))
    C = w.batch.chunk_len
    for j in picks:
        s = w.batch.decodes[j]
        solo = synth.HybridBatch(None, 0, [s])
        alone = _forward(w, solo, w.x[C + j:C + j + 1], T, max(w.batch.n_decodes, 1))
        assert np.array_equal(alone[0], hybrid[C + j]), (j, int((alone[0] != hybrid[C + j]).sum()))


def test_decode_alone_equals_piggybacked_tiny():
    ctxs = [20, 90, 300]
    lengths = [96 + 1] + [c + 1 for c in ctxs]
    nb = sum(synth.blocks_needed(n) for n in lengths) + 6
    w = workloads.make("inv", synth.TINY, 21, 48, 48, ctxs, num_blocks=nb, max_pos=nb * 16)
    _check(w, [0, 2])


def test_decode_alone_equals_piggybacked_llama13b():
    w = workloads.llama13b_hybrid(seed=5)
    _check(w, [0, 17])
