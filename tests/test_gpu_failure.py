"""The failure path on the GPU, without faulting the GPU.

Every mbarrier wait in the library's kernels has a wall-clock limit; when one
runs out, the kernel records an error in the device error word, stops
issuing work, drains its own copies and MMAs, frees its tensor memory and
returns, and the host learns of it at the next hb_sync (HB_EDEVICE).  Here a
test hook makes one such wait run out on purpose: in the next tensor-core
GEMM launch every wait gives up after 1 ms, and one CTA withholds one weight
copy (nothing is corrupted, no address changes, no copy is left in flight).
The context must report the error once and then compute the next forward
exactly as before.
"""
import numpy as np
import pytest

from chunked_prefill_hybrid_gb300 import native, workloads
from harness import compare, f64, oracle_run

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _forward(ctx, w, x):
    y = torch.full_like(x, 0x7FC0)
    ctx.forward(native.Spec(w.batch), x, y)
    return y


def test_expired_wait_reports_device_error_then_recovers():
    w = workloads.tiny(seed=5)
    ctx = native.Context(workloads.config(w))
    x = workloads.upload(w, ctx, poison=None)
    y0 = _forward(ctx, w, x)
    ctx.sync()
    before = y0.cpu().numpy().view(np.uint16).copy()

    ctx.test_wait_timeout(1_000_000)  # 1 ms
    _forward(ctx, w, x)
    with pytest.raises(native.HbError) as e:
        ctx.sync()
    assert e.value.code == native.HB_EDEVICE
    assert "device error word = 1" in str(e.value), str(e.value)
    ctx.sync()  # the word was cleared by the report

    y2 = _forward(ctx, w, x)
    ctx.sync()
    after = y2.cpu().numpy().view(np.uint16)
    assert np.array_equal(after, before), "the forward after the fault differs from the one before it"
    ref, _ = oracle_run(w)
    ok, st = compare(f64(after), ref, ulp=False)
    assert ok, st
    ctx.free()


def test_wait_timeout_hook_rejects_bad_limits():
    w = workloads.tiny(seed=5)
    ctx = native.Context(workloads.config(w))
    for bad in (0, 99_999, 2_000_000_001):
        with pytest.raises(native.HbError) as e:
            ctx.test_wait_timeout(bad)
        assert e.value.code == native.HB_EINVAL
    ctx.free()
