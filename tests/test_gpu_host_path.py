"""hb_forward_host, the call with HOST buffers: it copies the input rows to the
device, runs the stack and copies the result back, all on the context's
stream.  The same kernels run on the same rows as hb_forward, so the two
outputs are bit-identical; hb_forward itself is checked against the oracle
in the parity tests.  A batch that the host plan rejects after the input
copy has started comes back as an error with the output buffer untouched.
hb_forward_host_async does the same without waiting: a sequence of calls on
different batches, with one hb_sync at the end, gives every batch's
hb_forward result.
"""
import numpy as np
import pytest

from chunked_prefill_hybrid_gb300 import native, synth, workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _setup(n_layers=2, seed=23):
    w = workloads.make("host", synth.TINY, seed, 40, 48, [20, 90, 300], n_layers=n_layers)
    ctx = native.Context(workloads.config(w))
    x = workloads.upload(w, ctx, poison=None)
    return w, ctx, x


def _device_out(ctx, spec, x):
    y = torch.empty_like(x)
    ctx.forward(spec, x, y)
    ctx.sync()
    return y.cpu().numpy().view(np.uint16).copy()


@pytest.mark.parametrize("pinned", [False, True], ids=["pageable", "pinned"])
def test_host_path_equals_device_path(pinned):
    w, ctx, x = _setup()
    spec = native.Spec(w.batch)
    want = _device_out(ctx, spec, x)
    xin = np.ascontiguousarray(w.x).view(np.uint16)
    if pinned:
        xh = torch.from_numpy(xin.view(np.int16).copy()).pin_memory()
        yh = torch.full_like(xh, 0x7FC0).pin_memory()
        for _ in range(3):  # repeated calls: each plans, copies in, runs and copies out
            ctx.forward_host_ptr(spec, xh.data_ptr(), yh.data_ptr())
            assert np.array_equal(yh.numpy().view(np.uint16), want)
    else:
        yout = np.full_like(xin, 0x7FC0)
        ctx.forward_host(spec, xin, yout)
        assert np.array_equal(yout, want)
    ctx.free()


def test_rejected_batch_leaves_output_untouched():
    w, ctx, x = _setup(n_layers=1, seed=29)
    spec = native.Spec(w.batch)
    want = _device_out(ctx, spec, x)
    xin = np.ascontiguousarray(w.x).view(np.uint16)
    yout = np.full_like(xin, 0x7FC0)
    good = spec.dbt[0, 0]
    spec.dbt[0, 0] = w.num_blocks  # a block outside the pool: the row count is fine, the full plan is not
    with pytest.raises(native.HbError) as e:
        ctx.forward_host(spec, xin, yout)
    assert e.value.code == native.HB_ERANGE
    assert np.all(yout == 0x7FC0)
    spec.dbt[0, 0] = good
    ctx.forward_host(spec, xin, yout)  # the context is still usable
    assert np.array_equal(yout, want)
    ctx.free()


def test_async_host_calls_equal_device_path():
    """Five batches of different shapes (chunks, decodes, both), each from its own pinned input into its own
    pinned output, submitted back to back with one sync at the end; the input ring of two device buffers is
    reused three times over."""
    w = workloads.make("host-async", synth.TINY, 31, 40, 48, [20, 90, 300], n_layers=2)
    ctx = native.Context(workloads.config(w))
    workloads.upload(w, ctx, poison=None)
    C, decs, chunk = w.batch.chunk_len, list(w.batch.decodes), w.batch.chunk
    batches = [synth.HybridBatch(chunk, C, decs), synth.HybridBatch(None, 0, decs[:2]),
               synth.HybridBatch(chunk, 16, []), synth.HybridBatch(chunk, 7, decs[1:]),
               synth.HybridBatch(None, 0, decs)]
    rows = []
    xs = np.ascontiguousarray(w.x).view(np.uint16)
    for b in batches:
        idx = list(range(b.chunk_len)) + [C + decs.index(d) for d in b.decodes]
        rows.append(np.ascontiguousarray(xs[idx]))
    want = [_device_out(ctx, native.Spec(b), workloads.to_device(r)) for b, r in zip(batches, rows)]
    specs = [native.Spec(b) for b in batches]
    xh = [torch.from_numpy(r.view(np.int16).copy()).pin_memory() for r in rows]
    yh = [torch.full_like(t, 0x7FC0).pin_memory() for t in xh]
    for sp, a, b in zip(specs, xh, yh):
        ctx.forward_host_async_ptr(sp, a.data_ptr(), b.data_ptr())
    ctx.sync()
    for i, (b, got) in enumerate(zip(want, yh)):
        assert np.array_equal(got.numpy().view(np.uint16), b), i
    # an output buffer the GPU cannot address is refused before anything is enqueued
    with pytest.raises(native.HbError) as e:
        ctx.forward_host_async_ptr(specs[0], xh[0].data_ptr(), np.zeros_like(rows[0]).ctypes.data)
    assert e.value.code == native.HB_EINVAL
    ctx.sync()
    ctx.free()
