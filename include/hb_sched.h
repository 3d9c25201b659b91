/*
 * hb_sched.h -- C ABI of the host-side decode-maximal batch scheduler (in libhb.so).
 *
 * Policy (host only, no GPU):
 *   "SARATHI ..." (paper-graph-ui summary), section 3.4:
 *     - "Chunked-Prefills": a prompt of P tokens runs as ceil(P / C) chunks of
 *       C tokens, the last one the remainder.
 *     - "Decode-Maximal Batching": every batch holds one prefill chunk plus as
 *       many decodes as memory allows (up to B - 1); decode-only batches when
 *       no prefill is pending.
 *     - "The Memory Constraint": B = floor((M_G - M_S) / (L * m_kv)); KV is
 *       pre-allocated per request for its maximum length.
 *     - tile quantization: the chunk shrinks so that chunk + decodes is a
 *       multiple of the GEMM tile (C' = 256 - (B - 1) for tile 128).
 *   "Notes on Sarathi-Serve" (junupark), "Stall Free Batching": a fixed token
 *   budget per step; decodes first, then the partially-prefilled request,
 *   then new prefills, each chunk = min(remaining budget, remaining prompt);
 *   running decodes are never stalled or preempted.
 *
 * Each iteration: (1) admit waiting requests first-come-first-served while
 * ceil((prompt + max_new) / block_size) free KV blocks exist (reserved until
 * the request finishes; never preempted); (2) take every running decode, in
 * admission order, up to max_decodes and the token budget; (3) take prefill
 * chunks from admitted requests with prompt left, oldest first, each
 * min(chunk_size, budget left, prompt left), at most max_chunks_per_batch;
 * (4) with tile > 0 and a single chunk, shrink it so the row count is a
 * multiple of tile when that leaves a positive chunk.
 * A request whose last prompt chunk ran has produced its first token and
 * decodes next; a decode step produces one token; a request with max_new
 * tokens produced is finished and its blocks are freed.  Free blocks are
 * handed out lowest id first.
 *
 * request_level = 1 is the request-level baseline the SARATHI summary compares
 * against ("Evaluation Methodology", Baselines (1)): prefill-only and
 * decode-only batches, never mixed.  Requests are admitted only when none is
 * running, at most max_decodes of them (the batch size B); while any admitted
 * request has prompt left the batch holds only prefill chunks (steps (3),
 * (4)); otherwise it holds every running decode (step (2)).
 *
 * Return codes are those of hb.h.  Pointers returned by the scheduler stay
 * valid until its next call.  Not thread-safe.
 */
#ifndef HB_SCHED_H
#define HB_SCHED_H

#include <stdint.h>

#include "hb.h"

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

typedef struct {
    int chunk_size;           /* C: prompt tokens of one chunk at most */
    int token_budget;         /* rows per batch at most; <= 0: no budget */
    int max_decodes;          /* decodes per batch at most (B - 1) */
    int tile;                 /* > 0: tile-align a single chunk (see above); 0: off */
    int max_chunks_per_batch; /* 1: SARATHI; > 1: Sarathi-Serve mixed chunks */
    int block_size;           /* tokens per KV block (16) */
    int num_blocks;           /* KV blocks the scheduler may hand out */
    int max_blocks_per_seq;   /* table entries per request at most */
    int request_level;        /* 1: the pages' baseline instead (see below); 0: decode-maximal */
} hb_sched_config;

typedef struct hb_sched hb_sched;

/* One scheduled batch.  Arrays are scheduler-owned. */
typedef struct {
    int n_chunks;
    const int32_t *chunk_req_ids;  /* [n_chunks] */
    const int32_t *chunk_offsets;  /* [n_chunks] prompt tokens already cached */
    const int32_t *chunk_lens;     /* [n_chunks] */
    int n_decodes;
    const int32_t *decode_req_ids;  /* [n_decodes] */
    const int32_t *decode_ctx_lens; /* [n_decodes] tokens already cached */
    int n_rows;                     /* sum of chunk_lens + n_decodes */
} hb_sched_batch;

/* Counters of the scheduler's state. */
typedef struct {
    int waiting, prefilling, decoding, finished;
    int free_blocks;
    long long iterations, decode_only_iterations, rows;
} hb_sched_stats;

int hb_sched_create(const hb_sched_config *cfg, hb_sched **out);

/* Queue a request (ids unique, >= 0).  HB_ENOMEM if it could never fit
 * (more blocks than num_blocks or max_blocks_per_seq); HB_EINVAL on bad
 * arguments (prompt_len >= 1, max_new_tokens >= 1). */
int hb_sched_add(hb_sched *s, int req_id, int prompt_len, int max_new_tokens);

/* Build the next batch.  Returns its row count (0 when nothing is runnable),
 * or a negative error.  Call hb_sched_complete after the batch ran. */
int hb_sched_next(hb_sched *s, hb_sched_batch *out);

/* The batch from the last hb_sched_next has run: advance prompt progress,
 * produce tokens, finish requests, free their blocks.  Returns the number
 * of requests that finished. */
int hb_sched_complete(hb_sched *s);

/* Block table of an admitted request (scheduler-owned). */
int hb_sched_block_table(hb_sched *s, int req_id, const int32_t **table, int *n_blocks);

/* Fill an hb_forward spec for the last batch: its first chunk in the chunk_*
 * fields, further chunks (max_chunks_per_batch > 1) in the more_chunk_*
 * fields, decodes after them (HB_ERANGE beyond HB_MAX_CHUNKS chunks).  Block
 * tables point into scheduler-owned storage, rows of width
 * max_blocks_per_seq, valid until the next hb_sched_* call. */
int hb_sched_fill_spec(hb_sched *s, hb_batch_spec *spec);

int hb_sched_get_stats(hb_sched *s, hb_sched_stats *out);

/* B = floor((mem_total - mem_params) / (max_len * kv_bytes_per_token)),
 * the requests that fit with KV pre-allocated to max_len ("The Memory
 * Constraint").  Returns -1 for non-positive inputs. */
long long hb_sched_max_batch(long long mem_total, long long mem_params, long long max_len,
                             long long kv_bytes_per_token);

void hb_sched_free(hb_sched *s);

/* ---- chunk-size selection ("SARATHI ..." summary, section "The chunk size",
 * "The piggybacking condition" and "A two-step chunk selection procedure").
 * All host-only; no scheduler state unless stated. */

/* P:D ratio at which every decode of a request is piggybacked:
 * C / (B - 1).  Returns -1 for C < 1 or B < 2. */
double hb_perfect_pd_ratio(int chunk_size, int batch_size);

/* Decode tokens of a request (prompt P, D decode tokens) that can ride on its
 * prefill chunks: min(D, ceil(P / C) * (B - 1)).  -1 for bad arguments. */
long long hb_piggyback_capacity(long long prompt_len, long long decode_len, int chunk_size, int batch_size);

/* Two-step chunk size: (1) C0 = round(pd_ratio * (B - 1)) clamped to
 * [c_min, c_max]; (2) if tile > 0, the largest C <= C0 with C + (B - 1) a
 * multiple of tile, provided C >= c_min (else C0).  Returns -1 for bad
 * arguments (pd_ratio <= 0, B < 2, c_min < 1, c_max < c_min, tile < 0). */
int hb_advise_chunk(double pd_ratio, int batch_size, int tile, int c_min, int c_max);

/* Online estimate of the workload's P:D ratio: an exponentially weighted
 * mean (weight 1/8 per observation) of prompt_len / tokens produced over the
 * requests the scheduler has finished; -1 before the first one. */
double hb_sched_pd_estimate(hb_sched *s);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif

#ifdef __cplusplus
}
#endif

#endif /* HB_SCHED_H */
