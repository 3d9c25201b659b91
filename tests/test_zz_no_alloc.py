"""hb_decode_attention_noalloc -- decode attention with its scratch in a fixed
static device array, for callers that cannot allocate -- against the oracle's
attention on seeded q and K/V, and against the attention output of
hb_forward's decode rows on the same q and K/V.

The file name sorts last so that a full run calls it after every other GPU
test in the same process; it also passes alone.
"""
import numpy as np
import pytest

from chunked_prefill_hybrid_gb300 import native, synth, workloads
from oracle import oracle as orc

torch = pytest.importorskip("torch")

D128 = synth.ModelDims(hidden=256, n_heads=2, n_kv_heads=2, head_dim=128, ffn=512)
GQA = synth.ModelDims(hidden=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn=384)
# decode contexts from one key to five 256-key splits, block edges included
CTX = [0, 15, 16, 255, 256, 257, 700, 1100]
NAN16 = 0x7FC0  # a bf16 NaN: marks output that was never written


def _call_rc(**over):
    a = dict(q=8, k=8, v=8, bt=8, stride=70, ctx=8, n=1, heads=1, kv=1, hd=128, nb=1, max_ctx=1000, out=8)
    a.update(over)
    return native.lib().hb_decode_attention_noalloc(
        a["q"], a["k"], a["v"], a["bt"], a["stride"], a["ctx"], a["n"], a["heads"], a["kv"], a["hd"], a["nb"],
        a["max_ctx"], a["out"], None)


def test_limits_and_arguments_rejected_on_host():
    """Every case here is rejected before any CUDA call, so no pointer is used."""
    assert _call_rc(n=4097) == native.HB_ERANGE                       # decodes x heads > 4096
    assert _call_rc(n=64, heads=64, kv=64, max_ctx=1024) == native.HB_ERANGE  # 4096 x 5 splits > 16384
    assert _call_rc(stride=10) == native.HB_ERANGE                    # table narrower than max_ctx needs
    assert _call_rc(hd=96) == native.HB_EINVAL
    assert _call_rc(heads=3, kv=2) == native.HB_EINVAL
    assert _call_rc(q=None) == native.HB_EINVAL
    assert _call_rc(n=0) == native.HB_EINVAL


def _bf(t):
    return t.view(torch.bfloat16).float()


def _close(a, b):
    # both sides round one fp32 result to bf16; they differ only in the
    # order of fp32 sums, so at most one bf16 step apart
    return torch.all((a - b).abs() <= 1e-3 + 2.0 ** -7 * b.abs()).item()


@pytest.mark.gpu
@pytest.mark.parametrize("dims", [D128, GQA], ids=["d128", "gqa"])
def test_noalloc_matches_forward_attention(dims):
    w = workloads.make("noalloc", dims, 11, 64, 48, CTX)
    ctx = native.Context(workloads.config(w))
    x = workloads.upload(w, ctx)
    y = torch.empty_like(x)
    ctx.forward(native.Spec(w.batch), x, y)
    ctx.sync()
    T, n, nh, nkv, hd = w.T, w.batch.n_decodes, dims.n_heads, dims.n_kv_heads, dims.head_dim
    q_all = torch.empty((T, nh * hd), dtype=torch.int16, device="cuda")
    o_all = torch.empty_like(q_all)
    ctx.debug_read(1, q_all)
    ctx.debug_read(2, o_all)
    ctx.sync()
    q = q_all[T - n:].reshape(n, nh, hd).contiguous()
    ref = _bf(o_all[T - n:].reshape(n, nh, hd))

    # the decodes' keys 0..ctx (the last one written by the forward) in a
    # pool of our own, at the same block-table slots
    kp = torch.zeros((w.num_blocks, nkv, 16, hd), dtype=torch.int16, device="cuda")
    vp = torch.zeros_like(kp)
    for s in w.batch.decodes:
        m = s.cached + 1
        k = torch.empty((m, nkv, hd), dtype=torch.int16, device="cuda")
        v = torch.empty_like(k)
        ctx.read_kv(0, s.block_table, 0, k, v)
        ctx.sync()
        pos = torch.arange(m, device="cuda")
        blk = torch.from_numpy(np.asarray(s.block_table, np.int64)).cuda()[pos // 16]
        kp.permute(0, 2, 1, 3)[blk, pos % 16] = k
        vp.permute(0, 2, 1, 3)[blk, pos % 16] = v
    stride = max(len(s.block_table) for s in w.batch.decodes)
    bt = torch.from_numpy(synth.padded_decode_tables(w.batch, stride)).cuda()
    lens = torch.tensor([s.cached for s in w.batch.decodes], dtype=torch.int32, device="cuda")
    max_ctx = max(CTX)
    ctx.free()

    outs = []
    for _ in range(2):  # two calls in a row: the second finds the counters reset
        out = torch.full_like(q, NAN16)
        native.decode_attention_noalloc(q, kp, vp, bt, lens, max_ctx, out)
        outs.append(out)
    torch.cuda.synchronize()
    for out in outs:
        got = _bf(out)
        assert not torch.isnan(got).any()
        assert _close(got, ref), (got - ref).abs().max().item()
    assert torch.equal(outs[0], outs[1])

    # a context beyond max_ctx flags its row with NaN and leaves the others
    # (and the next call) intact
    bad = lens.clone()
    bad[3] = max_ctx + 1
    out = torch.full_like(q, 0)
    native.decode_attention_noalloc(q, kp, vp, bt, bad, max_ctx, out)
    again = torch.full_like(q, NAN16)
    native.decode_attention_noalloc(q, kp, vp, bt, lens, max_ctx, again)
    torch.cuda.synchronize()
    got = _bf(out)
    assert torch.isnan(got[3]).all()
    keep = [j for j in range(n) if j != 3]
    assert torch.equal(out[keep], outs[0][keep])
    assert torch.equal(again, outs[0])


def _seeded_case(dims, seed, ctxs, num_blocks):
    """q ~ N(0, 4), a whole pool of K/V ~ N(0, 1) in [num_blocks][n_kv][16][d], shuffled block tables."""
    n, nh, nkv, hd = len(ctxs), dims.n_heads, dims.n_kv_heads, dims.head_dim
    q = synth.normal_bf16(seed, (1,), (n, nh, hd), 2.0)
    kp = synth.normal_bf16(seed, (2,), (num_blocks, nkv, 16, hd))
    vp = synth.normal_bf16(seed, (3,), (num_blocks, nkv, 16, hd))
    tables = synth.allocate_tables(seed, (4,), [c + 1 for c in ctxs], num_blocks)
    stride = max(len(t) for t in tables)
    bt = np.full((n, stride), -1, np.int32)
    for j, t in enumerate(tables):
        bt[j, :len(t)] = t
    return q, kp, vp, bt


def _oracle_rows(dims, q, kp, vp, bt, ctxs):
    num_blocks, nkv, _, hd = kp.shape
    pool = orc.Pool(num_blocks, nkv, hd)
    pool.k[:] = synth.bf16_to_f32(kp).astype(np.float64).transpose(0, 2, 1, 3).reshape(-1, nkv, hd)
    pool.v[:] = synth.bf16_to_f32(vp).astype(np.float64).transpose(0, 2, 1, 3).reshape(-1, nkv, hd)
    qf = synth.bf16_to_f32(q).astype(np.float64)
    group = dims.n_heads // nkv
    ref = np.zeros(qf.shape)
    for j, c in enumerate(ctxs):
        for h in range(dims.n_heads):
            ref[j, h] = orc.attention_head(qf[j, h], pool, h // group, bt[j], c)
    return ref


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


@pytest.mark.gpu
@pytest.mark.parametrize("dims", [D128, GQA], ids=["d128", "gqa"])
def test_noalloc_matches_oracle(dims):
    """Against the oracle's fp64 attention: each output is the bf16 rounding of the fp64 answer, give or
    take fp32 error, i.e. |got - ref| <= 2^-8 |ref| + 2e-5 (one bf16 step), and the literal 3e-2 / 3e-3
    bound holds; two calls in a row give the same bytes.  Then one decode's table holds a block id outside
    the pool (num_blocks, and -1) at a 1100-key, five-split context: that row alone is NaN, and the next
    good call matches again."""
    ctxs = CTX
    num_blocks = sum(synth.blocks_needed(c + 1) for c in ctxs) + 5
    q, kp, vp, bt = _seeded_case(dims, 41, ctxs, num_blocks)
    ref = _oracle_rows(dims, q, kp, vp, bt, ctxs)
    qd, kd, vd, btd = _dev(q), _dev(kp), _dev(vp), torch.from_numpy(bt).cuda()
    lens = torch.tensor(ctxs, dtype=torch.int32, device="cuda")
    max_ctx = max(ctxs)
    outs = []
    for _ in range(2):
        out = torch.full_like(qd, NAN16)
        native.decode_attention_noalloc(qd, kd, vd, btd, lens, max_ctx, out)
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
    got = _bf(outs[0]).double().cpu().numpy()
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    assert (err <= 2.0 ** -8 * np.abs(ref) + 2e-5).all(), float((err - 2.0 ** -8 * np.abs(ref)).max())
    assert err.max() <= 3e-2 and err.mean() <= 3e-3, (err.max(), err.mean())

    j = ctxs.index(1100)
    for bad_id in (num_blocks, -1):
        bad = bt.copy()
        bad[j, 40] = bad_id  # keys 640..655: inside the third 256-key split
        out = torch.full_like(qd, 0)
        native.decode_attention_noalloc(qd, kd, vd, torch.from_numpy(bad).cuda(), lens, max_ctx, out)
        again = torch.full_like(qd, NAN16)
        native.decode_attention_noalloc(qd, kd, vd, btd, lens, max_ctx, again)
        torch.cuda.synchronize()
        g = _bf(out)
        assert torch.isnan(g[j]).all(), bad_id
        keep = [i for i in range(len(ctxs)) if i != j]
        assert torch.equal(out[keep], outs[0][keep]), bad_id
        assert torch.equal(again, outs[0]), bad_id
