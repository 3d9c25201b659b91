"""Plain-Python restatement of the decode-maximal scheduling policy.

TEST INFRASTRUCTURE ONLY (compared decision by decision with the library's
scheduler; shares no code with it).

Policy, in the pages' terms:
  * chunked prefill -- a prompt of P tokens runs as chunks of at most C
    tokens; the last chunk is the remainder (SARATHI summary, section 3.4,
    "Chunked-Prefills");
  * decode-maximal batching -- one prefill chunk plus as many decodes as
    allowed, decode-only batches when no prefill is pending (section 3.4,
    "Decode-Maximal Batching");
  * KV is reserved for the request's maximum length when it is admitted
    (section 3.4, "The Memory Constraint"), first come first served;
  * stall-free token budget -- decodes first, then chunks of
    min(budget left, prompt left), oldest request first ("Notes on
    Sarathi-Serve", "Stall Free Batching");
  * tile alignment -- with one chunk, shrink it by (rows mod tile) when the
    chunk stays positive (section 3.4, tile quantization: 256 - (B - 1)).
  * request_level -- the pages' baseline ("Evaluation Methodology",
    Baselines (1)): prefill-only and decode-only batches, never mixed; a new
    batch of at most max_decodes requests is admitted only when the last has
    finished; prefill chunks run while any admitted prompt is unfinished.
"""
from __future__ import annotations

import math


class SchedOracle:
    def __init__(self, chunk_size, token_budget=0, max_decodes=1 << 20, tile=0, max_chunks_per_batch=1,
                 block_size=16, num_blocks=1 << 16, max_blocks_per_seq=1 << 12, request_level=0):
        self.C = chunk_size
        self.budget = token_budget if token_budget > 0 else float("inf")
        self.max_decodes = max_decodes
        self.tile = tile
        self.max_chunks = max_chunks_per_batch
        self.bs = block_size
        self.num_blocks = num_blocks
        self.max_bps = max_blocks_per_seq
        self.free = list(range(num_blocks))  # kept sorted
        self.req = {}          # id -> dict
        self.waiting = []      # FCFS
        self.running = []      # admission order
        self.last = None
        self.pd_ewma = None
        self.request_level = bool(request_level)

    def blocks_needed(self, prompt, max_new):
        return math.ceil((prompt + max_new) / self.bs)

    def add(self, rid, prompt, max_new):
        need = self.blocks_needed(prompt, max_new)
        if need > self.num_blocks or need > self.max_bps:
            raise MemoryError(rid)
        self.req[rid] = dict(prompt=prompt, max_new=max_new, processed=0, generated=0, phase="waiting", blocks=[])
        self.waiting.append(rid)

    def _admit(self):
        if self.request_level and self.running:
            return
        while self.waiting:
            if self.request_level and len(self.running) >= max(1, self.max_decodes):
                return
            r = self.req[self.waiting[0]]
            need = self.blocks_needed(r["prompt"], r["max_new"])
            if len(self.free) < need:
                return
            r["blocks"] = self.free[:need]
            self.free = self.free[need:]
            r["phase"] = "prefill"
            self.running.append(self.waiting.pop(0))

    def next(self):
        self._admit()
        rows = 0
        decodes = []
        prefill_left = any(self.req[rid]["phase"] == "prefill" for rid in self.running)
        for rid in self.running:
            if self.request_level and prefill_left:
                break
            r = self.req[rid]
            if r["phase"] != "decode":
                continue
            if len(decodes) >= self.max_decodes or rows + 1 > self.budget:
                break
            decodes.append((rid, r["prompt"] + r["generated"] - 1))
            rows += 1
        chunks = []
        for rid in self.running:
            if len(chunks) >= self.max_chunks or rows >= self.budget:
                break
            r = self.req[rid]
            if r["phase"] != "prefill":
                continue
            n = min(self.C, r["prompt"] - r["processed"], self.budget - rows)
            if n <= 0:
                break
            chunks.append([rid, r["processed"], int(n)])
            rows += int(n)
        if self.tile and len(chunks) == 1:
            rem = rows % self.tile
            if rem and chunks[0][2] > rem:
                chunks[0][2] -= rem
                rows -= rem
        self.last = ([tuple(c) for c in chunks], decodes)
        return self.last[0], self.last[1], rows

    def complete(self):
        chunks, decodes = self.last
        done = 0
        for rid, off, n in chunks:
            r = self.req[rid]
            r["processed"] += n
            if r["processed"] == r["prompt"]:
                r["generated"] = 1
                if r["generated"] >= r["max_new"]:
                    self._finish(rid)
                    done += 1
                else:
                    r["phase"] = "decode"
        for rid, _ in decodes:
            r = self.req[rid]
            r["generated"] += 1
            if r["generated"] >= r["max_new"]:
                self._finish(rid)
                done += 1
        self.last = None
        return done

    def _finish(self, rid):
        r = self.req[rid]
        # online P:D estimate: exponentially weighted, weight 1/8 for the newest
        # finished request (the pages name an EWMA and leave its weight open)
        pd = r["prompt"] / r["generated"]
        self.pd_ewma = pd if self.pd_ewma is None else self.pd_ewma + (pd - self.pd_ewma) / 8
        r["phase"] = "done"
        self.free = sorted(self.free + r["blocks"])
        r["blocks"] = []
        self.running.remove(rid)


def max_batch(mem_total, mem_params, max_len, kv_bytes_per_token):
    """B = floor((M_G - M_S) / (L * m_kv)) (SARATHI summary, "The Memory Constraint")."""
    return (mem_total - mem_params) // (max_len * kv_bytes_per_token)


def perfect_pd_ratio(C, B):
    """P/D at which every decode rides on a prefill chunk: P/D = C / (B - 1)
    (SARATHI summary, "The piggybacking condition")."""
    return C / (B - 1)


def piggyback_capacity(P, D, C, B):
    """Decode tokens of one request that fit on its ceil(P/C) chunks of B - 1
    decode slots each: min(D, (P/C)(B - 1)) with P/C rounded up."""
    return min(D, math.ceil(P / C) * (B - 1))


def advise_chunk(pd, B, tile=0, c_min=1, c_max=1 << 30):
    """The pages' two-step choice ("A two-step chunk selection procedure"):
    C ~ (P/D)(B - 1), then round down so that C + (B - 1) is a multiple of the
    tile (256 - (B - 1) for a chunk of 256 and tile 128)."""
    x = pd * (B - 1)
    r = math.floor(x) + (1 if x - math.floor(x) >= 0.5 else 0)  # nearest, halves up
    c0 = min(max(r, c_min), c_max)
    if tile == 0:
        return c0
    rows = c0 + B - 1
    c = (rows // tile) * tile - (B - 1)
    return c if c >= c_min else c0
