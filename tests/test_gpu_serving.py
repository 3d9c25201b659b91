"""A decode-maximal serving loop on the GPU, step by step against the oracle.

The library's scheduler builds every batch (checked identical to the
oracle's restatement of the policy), hb_forward runs it through a 2-layer
tiny model, and the oracle replays the same batches in fp64 with its own
paged pools; every iteration's output rows are compared.  Prompt rows are
drawn per request, a decode's input row per (request, position) -- there is
no language-model head, so the "next token" is a fresh seeded row.
"""
import numpy as np
import pytest

from chunked_prefill_hybrid_gb300 import native, sched, synth, workloads
from oracle import oracle as orc
from oracle import sched_oracle
from harness import compare, f64

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.mark.parametrize("mode", ["sarathi", "budget", "multi"])
def test_serving_loop_matches_oracle(mode):
    seed = 41
    dims = synth.TINY.with_layers(2)
    H = dims.hidden
    num_blocks, mbs = 96, 32
    kw = dict(chunk_size=32, num_blocks=num_blocks, max_blocks_per_seq=mbs)
    kw.update({"sarathi": dict(max_decodes=6), "budget": dict(token_budget=40),
               "multi": dict(token_budget=48, max_chunks_per_batch=3)}[mode])
    lib, ref = sched.Scheduler(**kw), sched_oracle.SchedOracle(**kw)
    rng = np.random.default_rng(seed)
    reqs = [(i, int(rng.integers(10, 90)), int(rng.integers(2, 9))) for i in range(7)]
    for rid, p, m in reqs:
        lib.add(rid, p, m)
        ref.add(rid, p, m)
    prompts = {rid: synth.token_rows(seed, (100, rid), p, H) for rid, p, _ in reqs}

    cfg = native.model_config(dims, num_blocks, 64, 64, mbs * 16, n_layers=2)
    ctx = native.Context(cfg)
    weights = [synth.layer_weights(dims, seed, l) for l in range(2)]
    for l, lw in enumerate(weights):
        ctx.load_layer(l, {k: workloads.to_device(v) for k, v in lw.items()})
    ctx.fill_kv(0xFFFF)
    ctx.sync()
    pools = [orc.Pool(num_blocks, dims.n_kv_heads, dims.head_dim) for _ in range(2)]

    steps, most_chunks = 0, 0
    while True:
        b = lib.next()
        chunks, decodes, rows = ref.next()
        assert ([tuple(c) for c in b.chunks], [tuple(d) for d in b.decodes], b.n_rows) == (chunks, decodes, rows)
        if rows == 0:
            break
        xs = []
        for rid, off, ln in b.chunks:
            xs.append(prompts[rid][off:off + ln])
        for rid, c in b.decodes:
            xs.append(synth.token_rows(seed, (200, rid, c), 1, H))
        x = np.concatenate(xs)
        spec = lib.fill_spec()
        xd = workloads.to_device(x)
        yd = torch.empty_like(xd)
        ctx.forward_spec(spec, xd, yd)
        ctx.sync()
        gpu = f64(yd.cpu().numpy().view(np.uint16))
        # the oracle replays the same batch through both layers
        seqs = [(synth.Seq(rid, off, np.array(ref.req[rid]["blocks"], np.int32)), ln) for rid, off, ln in chunks]
        dec = [synth.Seq(rid, c, np.array(ref.req[rid]["blocks"], np.int32)) for rid, c in decodes]
        hb_ = synth.HybridBatch(seqs[0][0] if seqs else None, seqs[0][1] if seqs else 0, dec, seqs[1:])
        most_chunks = max(most_chunks, len(chunks))
        y = f64(x)
        for l in range(2):
            y = orc.layer_forward(dims, weights[l], hb_, y, pools[l], mirror=True)
        ok, st = compare(gpu, y)
        assert ok, (steps, st)
        lib.complete()
        ref.complete()
        steps += 1
    assert steps > 10
    assert most_chunks == 1 if mode != "multi" else most_chunks > 1
    assert lib.stats()["finished"] == len(reqs)
    ctx.free()


@pytest.mark.parametrize("request_level", [0, 1])
def test_serve_loop_latency_bookkeeping(request_level):
    """serve.run on a 2-layer tiny model: every request gets exactly max_new token times, in increasing order,
    the first at its last prompt chunk; decode-maximal batches mix phases, the request-level baseline never does."""
    from chunked_prefill_hybrid_gb300 import serve
    seed = 43
    dims = synth.TINY.with_layers(2)
    num_blocks, mbs = 256, 32
    cfg = native.model_config(dims, num_blocks, 256, 64, mbs * 16, n_layers=2)
    ctx = native.Context(cfg)
    for l in range(2):
        ctx.load_layer(l, {k: workloads.to_device(v) for k, v in synth.layer_weights(dims, seed, l).items()})
    ctx.fill_kv(0x3F80)
    x = workloads.to_device(synth.token_rows(seed, (1,), 256, dims.hidden))
    y = torch.empty_like(x)
    rng = np.random.default_rng(seed)
    reqs = [(i, int(rng.integers(20, 200)), int(rng.integers(1, 12))) for i in range(24)]
    kw = dict(chunk_size=64, token_budget=128, num_blocks=num_blocks, max_blocks_per_seq=mbs)
    if request_level:
        kw.update(chunk_size=1 << 20, token_budget=256, max_chunks_per_batch=16, max_decodes=8, request_level=1)
    s = sched.Scheduler(**kw)
    res = serve.run(ctx, s, reqs, x, y)
    ctx.free()
    for rid, p, m in reqs:
        ts = res.token_times[rid]
        assert len(ts) == m, (rid, len(ts), m)
        assert all(b > a for a, b in zip(ts, ts[1:]))
    mixed = sum(1 for c, d in zip(res.iter_chunks, res.iter_decodes) if c and d)
    assert (mixed == 0) if request_level else (mixed > 0)
    sm = res.summary()
    assert sm["generated_tokens"] == sum(m for _, _, m in reqs)
    assert sm["iterations"] == len(res.iter_ms) and all(t > 0 for t in res.iter_ms)
    assert all(b >= a for a, b in zip(res.iter_end_ms, res.iter_end_ms[1:]))
