/*
 * hb.h -- C ABI of the GB300 hybrid-batch forward library (libhb.so).
 *
 * One call runs one decode-maximal hybrid batch -- one prefill chunk of a
 * request at a prefix offset plus D single-token decodes of other requests --
 * through a LLaMA-style decoder-layer stack on one GPU:
 *
 *   "SARATHI: Efficient LLM Inference by Piggybacking Decodes with Chunked
 *   Prefills" (paper-graph-ui summary), section 3.4:
 *     - "Chunked-Prefills" / Figure 6: chunk query i at absolute position
 *       offset+i attends to keys 0..offset+i, the cached prefix plus the
 *       causal triangle; this equals the full prefill.
 *     - "Decode-Maximal Batching", "How fusion works": the chunk's rows come
 *       first, then the decode rows, and every linear op runs once over the
 *       concatenated rows so the weights are fetched once per batch.
 *   "Sarathi-Serve Guide: Chunked-Prefills & LLM Serving" (aifetchly):
 *     - "Deep Dive: Mathematical Formulation and Attention Mechanics": a
 *       decode with S cached tokens attends S+1 keys (cache plus itself);
 *       the block-diagonal hybrid mask isolates requests.
 *     - production checklist, "Paged KV-Cache Page Sizing": 16-token blocks.
 *   The batch description follows the co-scheduler's iteration batch in the
 *   same Guide (chunked request, chunk tokens, chunk prefix length, decode
 *   requests) plus per-request KV block tables.
 *
 * Conventions used by every call:
 *   - Return 0 (HB_OK) or a negative HB_E* code.  On error, nothing was
 *     enqueued (hb_forward_host alone may have started its input copy into
 *     the context's own buffer, and waits for it) and hb_last_error()
 *     describes the cause.  Every argument is validated on the host before
 *     any launch, so an invalid batch never reaches the GPU.
 *   - "device" pointers are CUDA device memory of the context's GPU; "host"
 *     pointers are read only during the call.
 *   - bf16 tensors are raw 16-bit patterns, row-major, densely packed.
 *   - Work is enqueued on the context's stream and the calls return without
 *     waiting (stream-ordered); hb_sync() waits and reports device-side
 *     errors.
 *   - A context is not thread-safe; use one context per host thread.
 */
#ifndef HB_H
#define HB_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

#define HB_OK 0
#define HB_EINVAL (-1)  /* malformed argument or batch */
#define HB_ERANGE (-2)  /* block id, position or size outside its bound */
#define HB_ENOMEM (-3)  /* device or host allocation failed */
#define HB_ECUDA (-4)   /* a CUDA runtime call failed; hb_last_error has its text */
#define HB_EDEVICE (-5) /* a kernel reported an error through the device error word */
#define HB_ESTATE (-6)  /* call not valid in the context's state (e.g. weights missing) */

typedef struct hb_ctx hb_ctx;

/* Model and capacity.  hidden == n_heads * head_dim; n_heads % n_kv_heads == 0;
 * head_dim in {64, 128}; block_size must be 16. */
typedef struct {
    int n_layers;
    int hidden;
    int n_heads;
    int n_kv_heads;
    int head_dim;
    int ffn;
    float rms_eps;      /* RMSNorm epsilon (1e-6 for LLaMA) */
    float rope_theta;   /* RoPE base (1e4 for LLaMA) */
    int block_size;     /* tokens per KV block: 16 */
    int num_blocks;     /* physical KV blocks per layer in the library-owned pool */
    int max_blocks_per_seq;
    int max_tokens;     /* upper bound on rows T = chunk_len + n_decodes of one batch */
    int max_decodes;    /* upper bound on n_decodes */
    int max_pos;        /* every absolute position is < max_pos */
} hb_model_config;

/* One layer's weights, device bf16, row-major [out][in]:
 *   w_qkv     [(n_heads + 2 n_kv_heads) head_dim][hidden]  q rows, k rows, v rows
 *   w_o       [hidden][n_heads head_dim]
 *   w_gate_up [2 ffn][hidden]                              gate rows, then up rows
 *   w_down    [hidden][ffn]
 *   norm1, norm2 [hidden]                                  RMSNorm gammas
 * The library copies and repacks them; the caller may free its buffers once
 * the call's work has completed (hb_sync). */
typedef struct {
    const void *w_qkv, *w_o, *w_gate_up, *w_down;
    const void *norm1, *norm2;
} hb_layer_weights;

/* One hybrid batch.  All arrays are host memory.
 *   chunk_req_id      request id of the prefill chunk, or -1 for no chunk
 *   chunk_offset      tokens of that request already in the KV cache
 *   chunk_len         prompt tokens prefilled now (0 when there is no chunk)
 *   chunk_block_table [chunk_n_blocks] physical block ids, logical order;
 *                     must cover positions 0 .. chunk_offset+chunk_len-1
 *   n_decodes         decode tokens D
 *   decode_req_ids    [n_decodes] distinct, none equal to chunk_req_id
 *   decode_ctx_lens   [n_decodes] tokens already cached; the new token sits
 *                     at position ctx and attends ctx+1 keys
 *   decode_block_tables [n_decodes][decode_bt_stride]; row j covers
 *                     positions 0 .. ctx_j
 *   n_more_chunks     further prefill chunks of other requests in the same
 *                     batch (0 for a SARATHI batch).  Sarathi-Serve's
 *                     stall-free batching ("Notes on Sarathi-Serve",
 *                     "Stall Free Batching" and its illustrated example) fills
 *                     the token budget with several chunks: the partially
 *                     prefilled request first, then the next in FCFS order.
 *                     Needs chunk_req_id >= 0; at most HB_MAX_CHUNKS - 1.
 *   more_chunk_req_ids, more_chunk_offsets, more_chunk_lens [n_more_chunks]:
 *                     as chunk_req_id / chunk_offset / chunk_len (len > 0;
 *                     ids distinct from every other id of the batch)
 *   more_chunk_block_tables [n_more_chunks][more_chunk_bt_stride]; row i
 *                     covers positions 0 .. offset_i + len_i - 1
 * Row order of x_in / x_out: chunk rows 0..chunk_len-1, then the rows of each
 * further chunk in spec order, then decode rows in spec order.  Slot of
 * position p: table[p / 16] * 16 + p % 16.  A chunk of one row computes what
 * a decode at ctx = offset computes. */
typedef struct {
    int chunk_req_id;
    int chunk_offset;
    int chunk_len;
    const int32_t *chunk_block_table;
    int chunk_n_blocks;
    int n_decodes;
    const int32_t *decode_req_ids;
    const int32_t *decode_ctx_lens;
    const int32_t *decode_block_tables;
    int decode_bt_stride;
    int n_more_chunks;
    const int32_t *more_chunk_req_ids;
    const int32_t *more_chunk_offsets;
    const int32_t *more_chunk_lens;
    const int32_t *more_chunk_block_tables;
    int more_chunk_bt_stride;
} hb_batch_spec;

/* Most prefill chunks in one batch (the first plus n_more_chunks). */
#define HB_MAX_CHUNKS 16

/* Create a context on the current CUDA device.
 * cfg: host.  weights: host array of n_layers entries (device pointers
 * inside), or NULL to load layers later with hb_load_layer.  cuda_stream: a
 * cudaStream_t or NULL for the legacy default stream.  *out receives the
 * context.  Allocates the KV pools (n_layers x 2 x num_blocks x 16 tokens),
 * repacked weights and all scratch.  Errors: HB_EINVAL (bad dims),
 * HB_ENOMEM, HB_ECUDA (out is then NULL). */
int hb_init(const hb_model_config *cfg, const hb_layer_weights *weights, void *cuda_stream, hb_ctx **out);

/* Copy and repack layer `layer`'s weights (see hb_layer_weights). */
int hb_load_layer(hb_ctx *ctx, int layer, const hb_layer_weights *w);

/* Write n_tokens tokens of K (post-RoPE) and V for positions start_pos ..
 * start_pos+n_tokens-1 of one request into layer `layer`'s pool.
 * block_table: host [n_blocks].  k, v: device bf16 [n_tokens][n_kv_heads][head_dim].
 * Used to load a cached prefix.  Errors: HB_EINVAL, HB_ERANGE. */
int hb_append_kv(hb_ctx *ctx, int layer, const int32_t *block_table, int n_blocks, int start_pos,
                 int n_tokens, const void *k, const void *v);

/* Read back K and V of positions start_pos .. start_pos+n_tokens-1 (test
 * hook; same layout as hb_append_kv, k and v are device outputs). */
int hb_read_kv(hb_ctx *ctx, int layer, const int32_t *block_table, int n_blocks, int start_pos,
               int n_tokens, void *k, void *v);

/* Fill every K and V element of every layer's pool with the bf16 pattern
 * `bits` (test hook: a poison value proves no write lands outside its slot). */
int hb_fill_kv(hb_ctx *ctx, uint16_t bits);

/* Run the batch through all layers.  x_in, x_out: device bf16 [T][hidden],
 * T = chunk_len + the further chunks' lengths + n_decodes; they may not
 * overlap and must be 16-byte aligned (HB_EINVAL otherwise, before any
 * launch).  Each layer writes the
 * batch's new K/V into its pool at the rows' slots, then attends.  The
 * library does not advance request lengths; the scheduler does. */
int hb_forward(hb_ctx *ctx, const hb_batch_spec *spec, const void *x_in, void *x_out);

/* Same as hb_forward over layers [layer_begin, layer_end) only. */
int hb_forward_layers(hb_ctx *ctx, const hb_batch_spec *spec, int layer_begin, int layer_end,
                      const void *x_in, void *x_out);

/* Like hb_forward, but x_in and x_out are HOST bf16 buffers: the call copies
 * x_in to the device, runs the stack and copies the result back, all on the
 * context's stream, and waits for it.  Use pinned host memory for speed:
 * a page-locked, 16-byte aligned x_out_host that the GPU can address
 * (cudaPointerGetAttributes reports a device pointer for it) is written in
 * place by the last kernel, with no copy after the stack; any other buffer
 * is filled by a device-to-host copy.
 * The input copy starts before the batch is fully validated (it overlaps the
 * host's planning); when the batch is then rejected, the call waits for that
 * copy before it returns the error, so x_in_host is free again on return and
 * x_out_host is untouched. */
int hb_forward_host(hb_ctx *ctx, const hb_batch_spec *spec, const void *x_in_host, void *x_out_host);

/* hb_forward_host that does not wait: it enqueues the input copy, plans the
 * batch and launches the stack, then returns, so that the host can build
 * and submit the next batch while this one runs (a serving loop's natural
 * shape: SARATHI summary, section 3.4, one hybrid batch per iteration).
 *   x_in_host:  host bf16 [T][hidden]; page-locked memory for an asynchronous
 *               copy.  It must stay unchanged until the next hb_sync.
 *   x_out_host: page-locked host memory (HB_EINVAL otherwise) for
 *               [T][hidden] bf16.  Read it after hb_sync.
 * The input is copied into one of two device buffers on a second stream
 * while the previous batch computes; a buffer is refilled only after the
 * batch that read it.  The result goes to one of two device buffers and is
 * copied to x_out_host on a third stream while the next batch computes; a
 * batch reuses an output buffer only after its copy.  Calls are ordered on
 * the context's stream, like hb_forward; hb_sync also waits for the output
 * copies.  A batch rejected by the host checks returns the error with
 * nothing left in flight; device errors show at the next hb_sync.  The first
 * call makes the two input and two output buffers (4 x max_tokens x hidden
 * bf16), two streams and six events. */
int hb_forward_host_async(hb_ctx *ctx, const hb_batch_spec *spec, const void *x_in_host, void *x_out_host);

/* Wait for the context's stream and for the output copies of
 * hb_forward_host_async; returns HB_EDEVICE if a kernel set the
 * device error word since the last hb_sync (and clears it). */
int hb_sync(hb_ctx *ctx);

/* Per-kernel timing of the following forwards (CUDA events on the context's
 * stream around every launch).  enable: 1 starts a fresh window, 0 stops.
 * hb_profile_read: after hb_sync, fills names[i] (static strings), the summed
 * milliseconds and launch counts of up to max_kinds kernel kinds; returns the
 * number of kinds. */
int hb_profile(hb_ctx *ctx, int enable);
int hb_profile_read(hb_ctx *ctx, const char **names, double *total_ms, int *launches, int max_kinds);

/* Number of kernel launches enqueued by this context since it was created. */
long long hb_launch_count(hb_ctx *ctx);

/* Test hook: D[t][n] = sum_k X[t][k] * W[n][k] in fp32, through the same
 * GEMM kernel the forward uses.  X: device bf16 [T][K]; W: device bf16
 * [N][K]; D: device fp32 [T][N].  Requires K % 8 == 0. */
int hb_gemm_test(hb_ctx *ctx, const void *X, const void *W, void *D, int T, int N, int K);

/* Test hook: choose the kernels later calls use.  gemm_impl 0 = reference
 * SIMT GEMM, 2 = tcgen05 GEMM on CTA pairs with the 2-SM MMA, the O and down
 * projections stream-K into partials finished by a reduce pass (default), 3 =
 * the same but O and down split K three ways inside 6-CTA clusters, summed
 * through distributed shared memory with the residual fused (shapes whose
 * clusters do not all fit at once fall back to 2); any other value is
 * HB_EINVAL; attn_impl 0 = one CTA per
 * (row, head), 1 = paged attention with mma.sync chunk tiles (default), 2 =
 * paged attention with tcgen05 chunk tiles.  Every setting computes the same
 * function. */
int hb_set_kernels(hb_ctx *ctx, int gemm_impl, int attn_impl);

/* Test hook for the failure path: arm a fault in the next tensor-core GEMM
 * launch of this context (the first layer's QKV projection of the next
 * forward).  In that launch every mbarrier wait gives up after wait_ns
 * (in [1e5, 2e9] ns) instead of 2 s, and the second CTA of the first CTA pair
 * does not issue its first weight-tile copy, so the first CTA's wait for that
 * pipeline stage runs out.  The kernel then records DERR_MBAR_TIMEOUT in the
 * device error word, stops issuing, drains its own MMAs, frees its tensor
 * memory and returns; no copy is left in flight and no memory is touched out
 * of place.  The forward's output is then undefined and the next hb_sync
 * returns HB_EDEVICE (and clears the word); the forward after that is
 * normal.  HB_EINVAL for a wait_ns out of range or without the tensor-core
 * GEMM.  Nothing on the pages corresponds to this call. */
int hb_test_wait_timeout(hb_ctx *ctx, long long wait_ns);

/* Test hook: copy an intermediate of the LAST layer run by the latest
 * forward into dst (device memory, bf16 rows of the batch):
 *   which = 0: n1 or n2 (the last RMSNorm output)  [T][hidden]
 *           1: q after RoPE                        [T][n_heads head_dim]
 *           2: attention output o                  [T][n_heads head_dim]
 *           3: h = x + o W_o^T                     [T][hidden]
 *           4: a = silu(g) * u                     [T][ffn]
 * Valid after hb_sync.  rows: the batch's T. */
int hb_debug_read(hb_ctx *ctx, int which, void *dst, int rows);

/* Paged decode attention that allocates no device memory.
 *
 * This call has no counterpart on the pages: it is a library convenience
 * for callers that must not allocate -- an engine that has handed nearly
 * all HBM to its own KV-cache arena, or code that may not call
 * cudaMalloc / cudaFree (they can stall every stream on the device) while
 * other work runs.  It needs no hb_ctx.
 *
 * Computes what the batch forward's attention computes for decode rows:
 * query j at position ctx_lens[j] attends keys 0..ctx_lens[j] of its own
 * sequence, found through its block table, softmax(q k^T / sqrt(head_dim)) v,
 * with grouped-query heads (head h reads kv head h / (n_heads / n_kv_heads)).
 *   q, out:       device bf16 [n_decodes][n_heads][head_dim]
 *   k_pool, v_pool: device bf16 [num_blocks][n_kv_heads][16][head_dim]
 *   block_tables: device int32 [n_decodes][bt_stride], bt_stride >=
 *                 max_ctx / 16 + 1
 *   ctx_lens:     device int32 [n_decodes], each in [0, max_ctx]
 *   head_dim 64 or 128; cuda_stream: a cudaStream_t, NULL = legacy default.
 * Split partials and arrival counters live in one fixed static device array
 * inside the library (about 8.5 MB), which bounds the call:
 *   n_decodes * n_heads <= 4096 and
 *   n_decodes * n_heads * ceil((max_ctx + 1) / 256) <= 16384;
 * larger calls return HB_ERANGE and launch nothing.  Other errors:
 * HB_EINVAL (bad argument), HB_ECUDA (a CUDA call failed).  A row whose
 * ctx_lens entry lies outside [0, max_ctx], or whose table holds a block id
 * outside [0, num_blocks), gets NaN.
 * Every call looks up the array's device address with the device current
 * (the array's name in host code is not a device address, and a device
 * reset can move it); the first call on each device, and the first after
 * such a move, also zeroes the counters on cuda_stream: make the first call
 * on each device before any stream capture.  Every call leaves the counters
 * at zero.  Results agree with the decode rows of hb_forward to within one
 * bf16 step, not bit for bit: this call splits at 256 keys, the forward at
 * 1024, so their fp32 sums run in different orders.  All calls on a device share the array, so calls that can overlap
 * on the GPU (different streams without ordering) race and give wrong
 * results: order them.  Asynchronous; errors of the kernel itself show as
 * NaN rows, not as a return code. */
int hb_decode_attention_noalloc(const void *q, const void *k_pool, const void *v_pool, const int32_t *block_tables,
                                int bt_stride, const int32_t *ctx_lens, int n_decodes, int n_heads, int n_kv_heads,
                                int head_dim, int num_blocks, int max_ctx, void *out, void *cuda_stream);

/* Host-only planning of one batch (no GPU, no context needed): validates
 * spec against cfg exactly as hb_forward does and writes each row's
 * absolute position and physical KV slot.  pos, slot: host int32 [T] or
 * NULL; err: host buffer for a message (may be NULL).  Returns T (> 0) or a
 * negative HB_E* code. */
int hb_plan(const hb_model_config *cfg, const hb_batch_spec *spec, int32_t *pos, int32_t *slot,
            char *err, int err_len);

/* Text of the last error on this context (never NULL). */
const char *hb_last_error(hb_ctx *ctx);

/* Release every allocation of the context (synchronizes its stream first). */
void hb_free(hb_ctx *ctx);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif

#ifdef __cplusplus
}
#endif

#endif /* HB_H */
