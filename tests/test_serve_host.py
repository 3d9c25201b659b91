"""Host-side checks of the serving loop's metrics (no GPU): the pipeline
bubble estimate against closed forms and a hand-worked schedule."""
import pytest

from chunked_prefill_hybrid_gb300 import serve


@pytest.mark.parametrize("S", [1, 2, 4, 8])
@pytest.mark.parametrize("n", [1, 5, 40])
def test_uniform_micro_batches_only_fill_and_drain(S, n):
    r = serve.pipeline_bubble([3.0] * n, S)
    assert r["makespan_ms"] == pytest.approx((n + S - 1) * 3.0 / S)
    assert r["bubble_frac"] == pytest.approx(r["uniform_bubble_frac"])
    assert r["uniform_bubble_frac"] == pytest.approx((S - 1) / (n + S - 1))


def test_alternating_micro_batches_worked_by_hand():
    # two stages; micro-batches of 2, 1, 2, 1 ms spend 1, 0.5, 1, 0.5 ms per stage.
    # stage 0 ends them at 1, 1.5, 2.5, 3; stage 1 runs [1,2] [2,2.5] [2.5,3.5] [3.5,4]:
    # makespan 4, busy 6 of 8 stage-ms -> 25 % idle against 20 % for uniform ones
    r = serve.pipeline_bubble([2.0, 1.0, 2.0, 1.0], 2)
    assert r["makespan_ms"] == pytest.approx(4.0)
    assert r["bubble_frac"] == pytest.approx(0.25)
    assert r["uniform_bubble_frac"] == pytest.approx(0.2)


def test_one_long_micro_batch_stalls_the_ones_after_it():
    # PB1: a long micro-batch between short ones; with S stages, every later micro-batch waits behind it
    short, long_ = 1.0, 9.0
    r = serve.pipeline_bubble([short, long_, short, short], 3)
    u = serve.pipeline_bubble([(3 * short + long_) / 4] * 4, 3)
    assert r["bubble_frac"] > u["bubble_frac"]
    assert r["makespan_ms"] > u["makespan_ms"]


def test_summary_latencies_from_token_times():
    res = serve.ServeResult(iter_ms=[2.0, 1.0, 1.0, 1.0], iter_end_ms=[2.0, 3.0, 4.0, 5.0], iter_rows=[10, 3, 3, 2],
                            iter_chunks=[2, 0, 0, 0], iter_decodes=[0, 2, 2, 2], prompt_tokens=10)
    res.token_times = {0: [2.0, 3.0, 4.0, 5.0], 1: [2.0, 3.0, 4.0]}
    s = res.summary(stages=(2,))
    assert s["generated_tokens"] == 7
    assert s["ttft_ms"]["p50"] == 2.0
    assert s["itl_ms"]["max"] == 1.0
    assert s["tpot_ms"]["mean"] == pytest.approx(1.0)
    assert s["tokens_per_s"] == pytest.approx(17 / 5e-3)
    assert s["iteration_ms"]["cv"] == pytest.approx(0.1875 ** 0.5 / 1.25)  # population sd / mean
