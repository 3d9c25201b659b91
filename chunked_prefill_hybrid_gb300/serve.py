"""Serving loop over the library: the host scheduler (libhb's hb_sched_*)
builds every batch, hb_forward runs it, and the loop records per-iteration
device times and per-request latencies.

Latencies, for a closed set of requests that are all present at t = 0
(Sarathi-Serve Guide, the co-scheduler's loop, which stamps a request's
tokens as iterations finish; "Notes on Sarathi-Serve", TBT/TPOT SLOs):
  * TTFT  -- the end of the iteration that holds a request's last prompt
             chunk (that iteration produces its first token);
  * ITL   -- the gap between two consecutive tokens of one request;
  * TPOT  -- (time of the last token - time of the first) / (tokens - 1).
Times are device time from the start of the first iteration (CUDA events on
the context's stream, read after the loop).

Iteration-time uniformity (SARATHI summary, "Failure 4", pipeline bubbles
PB1-PB3): the coefficient of variation of the per-iteration times, and the
bubbles an in-order pipeline of S equal stages would have with these
iterations as its micro-batches (``pipeline_bubble``).

The model has no vocabulary head, so a token's next input row is not
derived from its output: each iteration reads its T input rows from a
resident device buffer of seeded rows (the rows' values do not change the
work).  Every step of the forward runs in the library's kernels.
"""
from __future__ import annotations

import statistics
import time
from dataclasses import dataclass, field
from typing import Dict, List, Sequence, Tuple

from . import native, sched


def pipeline_bubble(times_ms: Sequence[float], stages: int) -> Dict[str, float]:
    """Run the iterations, in order, as micro-batches through `stages` equal
    pipeline stages: micro-batch i spends t_i / S on every stage, a stage
    takes micro-batches in order, and a micro-batch enters stage k + 1 when
    stage k has finished it.  Returns the makespan, the fraction of stage
    time spent idle, and the idle fraction the same number of uniform
    micro-batches (all of the mean time) would have -- fill and drain only.
    The excess of the first fraction over the second is the bubble that
    non-uniform micro-batches add."""
    n = len(times_ms)
    if n == 0 or stages < 1:
        return {"stages": stages, "makespan_ms": 0.0, "bubble_frac": 0.0, "uniform_bubble_frac": 0.0}
    S = stages
    done = [0.0] * S  # finish time of the last micro-batch on each stage
    for t in times_ms:
        step = t / S
        prev = 0.0
        for k in range(S):
            start = max(prev, done[k])
            done[k] = start + step
            prev = done[k]
    makespan = done[-1]
    busy = sum(times_ms)
    return {"stages": S, "makespan_ms": makespan, "bubble_frac": 1.0 - busy / (S * makespan),
            "uniform_bubble_frac": (S - 1) / (n + S - 1)}


def _pct(v: List[float], q: float) -> float:
    if not v:
        return float("nan")
    s = sorted(v)
    i = min(len(s) - 1, max(0, int(round(q * (len(s) - 1)))))
    return s[i]


@dataclass
class ServeResult:
    iter_ms: List[float] = field(default_factory=list)       # device time of each iteration
    iter_end_ms: List[float] = field(default_factory=list)   # end of each iteration, from the start of the first
    iter_rows: List[int] = field(default_factory=list)
    iter_chunks: List[int] = field(default_factory=list)
    iter_decodes: List[int] = field(default_factory=list)
    token_times: Dict[int, List[float]] = field(default_factory=dict)  # request -> its tokens' times
    prompt_tokens: int = 0
    wall_s: float = 0.0

    def summary(self, stages: Sequence[int] = (2, 4, 8)) -> dict:
        ttft = [ts[0] for ts in self.token_times.values() if ts]
        itl = [b - a for ts in self.token_times.values() for a, b in zip(ts, ts[1:])]
        tpot = [(ts[-1] - ts[0]) / (len(ts) - 1) for ts in self.token_times.values() if len(ts) > 1]
        gen = sum(len(ts) for ts in self.token_times.values())
        total_ms = self.iter_end_ms[-1] if self.iter_end_ms else 0.0
        mean = statistics.fmean(self.iter_ms) if self.iter_ms else 0.0
        cv = statistics.pstdev(self.iter_ms) / mean if len(self.iter_ms) > 1 and mean > 0 else 0.0
        hybrid = [t for t, c, d in zip(self.iter_ms, self.iter_chunks, self.iter_decodes) if c and d]
        return {
            "iterations": len(self.iter_ms), "requests": len(self.token_times),
            "prompt_tokens": self.prompt_tokens, "generated_tokens": gen,
            "device_s": total_ms / 1e3, "wall_s": self.wall_s,
            "tokens_per_s": (self.prompt_tokens + gen) / (total_ms / 1e3) if total_ms else None,
            "decode_tokens_per_s": gen / (total_ms / 1e3) if total_ms else None,
            "ttft_ms": {"p50": _pct(ttft, 0.5), "p99": _pct(ttft, 0.99), "mean": statistics.fmean(ttft) if ttft else None},
            "itl_ms": {"p50": _pct(itl, 0.5), "p99": _pct(itl, 0.99), "max": max(itl) if itl else None},
            "tpot_ms": {"p50": _pct(tpot, 0.5), "p99": _pct(tpot, 0.99), "mean": statistics.fmean(tpot) if tpot else None},
            "iteration_ms": {"mean": mean, "p50": _pct(self.iter_ms, 0.5), "p99": _pct(self.iter_ms, 0.99),
                             "max": max(self.iter_ms) if self.iter_ms else None, "cv": cv},
            "hybrid_iterations": len(hybrid),
            "pipeline_bubbles": [pipeline_bubble(self.iter_ms, s) for s in stages],
        }


def run(ctx: "native.Context", scheduler: "sched.Scheduler", requests: Sequence[Tuple[int, int, int]], x_rows,
        y_rows, max_iters: int = 1 << 30) -> ServeResult:
    """Serve `requests` [(id, prompt_len, max_new_tokens)] to completion (or
    max_iters iterations).  x_rows / y_rows: device bf16 buffers of at least
    the largest batch's rows x hidden (x holds the input rows every
    iteration reads; y receives the outputs)."""
    import torch
    prompt = {}
    for rid, p, m in requests:
        scheduler.add(rid, p, m)
        prompt[rid] = p
    res = ServeResult(prompt_tokens=sum(p for _, p, _ in requests))
    res.token_times = {rid: [] for rid, _, _ in requests}
    stream = torch.cuda.current_stream()
    marks = []   # (start event, end event, chunks, decodes)
    t0 = time.perf_counter()
    it = 0
    while it < max_iters:
        b = scheduler.next()
        if b.n_rows == 0:
            break
        spec = scheduler.fill_spec()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ctx.forward_spec(spec, x_rows, y_rows)
        e1.record(stream)
        marks.append((e0, e1, list(b.chunks), list(b.decodes), b.n_rows))
        scheduler.complete()
        it += 1
    ctx.sync()
    torch.cuda.synchronize()
    res.wall_s = time.perf_counter() - t0
    if not marks:
        return res
    first = marks[0][0]
    for e0, e1, chunks, decodes, rows in marks:
        end = first.elapsed_time(e1)
        res.iter_ms.append(e0.elapsed_time(e1))
        res.iter_end_ms.append(end)
        res.iter_rows.append(rows)
        res.iter_chunks.append(len(chunks))
        res.iter_decodes.append(len(decodes))
        for rid, off, ln in chunks:
            if off + ln == prompt[rid]:
                res.token_times[rid].append(end)
        for rid, _ in decodes:
            res.token_times[rid].append(end)
    return res
