// runtime.cu -- the C ABI of include/hb.h: context, validation, batch
// metadata, weight repacking and the per-layer launch sequence.
//
// Per layer l of one hybrid batch (rows: chunk first, then decodes -- SARATHI
// summary, section 3.4 "Decode-Maximal Batching", "How fusion works"):
//   n1 = RMSNorm(x)                      -> xn
//   [q|k|v] = n1 W_qkv^T, RoPE, append   -> q scratch, K/V into the paged pool
//   o = hybrid attention(q, pool)        -> o   (chunk causal over its prefix,
//                                               decodes over ctx+1 keys)
//   h = x + o W_o^T                      -> h
//   n2 = RMSNorm(h)                      -> xn
//   a = silu(n2 W_g^T) * (n2 W_u^T)      -> act
//   y = h + a W_d^T                      -> layer output
// All of it is enqueued on one stream with no host synchronisation.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <string>
#include <vector>

#include "hb.h"
#include "gemm_tc.h"
#include "kernels.h"
#include "runtime_internal.h"

using namespace hb;

namespace {

int fail(std::string *err, int code, const char *fmt, ...)
{
    if (err) {
        char buf[512];
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(buf, sizeof buf, fmt, ap);
        va_end(ap);
        *err = buf;
    }
    return code;
}

size_t round_up(size_t x, size_t m) { return (x + m - 1) / m * m; }

}  // namespace

namespace hb {

int validate_config(const hb_model_config &c, std::string *err)
{
    if (c.n_layers <= 0 || c.hidden <= 0 || c.n_heads <= 0 || c.n_kv_heads <= 0 || c.head_dim <= 0 || c.ffn <= 0)
        return fail(err, HB_EINVAL, "model dimensions must be positive");
    if (c.head_dim != 64 && c.head_dim != 128)
        return fail(err, HB_EINVAL, "head_dim must be 64 or 128 (got %d)", c.head_dim);
    if (c.hidden != c.n_heads * c.head_dim)
        return fail(err, HB_EINVAL, "hidden (%d) != n_heads * head_dim (%d)", c.hidden, c.n_heads * c.head_dim);
    if (c.n_heads % c.n_kv_heads)
        return fail(err, HB_EINVAL, "n_heads must be a multiple of n_kv_heads");
    if (c.hidden % 64 || c.ffn % 16)
        return fail(err, HB_EINVAL, "hidden must be a multiple of 64 and ffn of 16");
    if (c.block_size != 16)
        return fail(err, HB_EINVAL, "block_size must be 16 (got %d)", c.block_size);
    if (c.num_blocks <= 0 || c.max_blocks_per_seq <= 0 || c.max_tokens <= 0 || c.max_decodes < 0 || c.max_pos <= 0)
        return fail(err, HB_EINVAL, "capacities must be positive");
    if ((long long)c.max_blocks_per_seq * 16 < c.max_pos)
        return fail(err, HB_EINVAL, "max_blocks_per_seq * 16 must cover max_pos");
    if (!(c.rms_eps >= 0.f) || !(c.rope_theta > 0.f))
        return fail(err, HB_EINVAL, "rms_eps must be >= 0 and rope_theta > 0");
    return HB_OK;
}

// The batch's row count T, with the checks on the spec's counts and lengths
// that fix it (the first part of plan_batch).
static int spec_rows(const hb_model_config &c, const hb_batch_spec *s, int *rows, std::string *err)
{
    if (!s)
        return fail(err, HB_EINVAL, "spec is NULL");
    const bool has_chunk = s->chunk_req_id >= 0;
    if (s->chunk_req_id < -1)
        return fail(err, HB_EINVAL, "chunk_req_id must be -1 or a request id");
    if (has_chunk) {
        if (s->chunk_len <= 0)
            return fail(err, HB_EINVAL, "chunk_len must be > 0 when there is a chunk");
        if (s->chunk_offset < 0)
            return fail(err, HB_EINVAL, "chunk_offset must be >= 0");
        if (!s->chunk_block_table)
            return fail(err, HB_EINVAL, "chunk_block_table is NULL");
    } else if (s->chunk_len != 0) {
        return fail(err, HB_EINVAL, "chunk_len > 0 needs chunk_req_id >= 0");
    }
    if (s->n_decodes < 0)
        return fail(err, HB_EINVAL, "n_decodes < 0");
    if (s->n_decodes > c.max_decodes)
        return fail(err, HB_ERANGE, "n_decodes %d > max_decodes %d", s->n_decodes, c.max_decodes);
    const int n_more = s->n_more_chunks;
    if (n_more < 0)
        return fail(err, HB_EINVAL, "n_more_chunks < 0");
    if (n_more > 0) {
        if (!has_chunk)
            return fail(err, HB_EINVAL, "further chunks need a first chunk (chunk_req_id >= 0)");
        if (n_more > HB_MAX_CHUNKS - 1)
            return fail(err, HB_ERANGE, "%d chunks > HB_MAX_CHUNKS %d", n_more + 1, HB_MAX_CHUNKS);
        if (!s->more_chunk_req_ids || !s->more_chunk_offsets || !s->more_chunk_lens || !s->more_chunk_block_tables)
            return fail(err, HB_EINVAL, "further-chunk arrays are NULL");
        if (s->more_chunk_bt_stride <= 0 || s->more_chunk_bt_stride > c.max_blocks_per_seq)
            return fail(err, HB_ERANGE, "more_chunk_bt_stride %d outside 1..max_blocks_per_seq",
                        s->more_chunk_bt_stride);
        for (int i = 0; i < n_more; ++i) {
            if (s->more_chunk_lens[i] <= 0)
                return fail(err, HB_EINVAL, "further chunk %d: length must be > 0", i);
            if (s->more_chunk_offsets[i] < 0)
                return fail(err, HB_EINVAL, "further chunk %d: offset must be >= 0", i);
        }
    }
    long long chunk_rows = has_chunk ? s->chunk_len : 0;
    for (int i = 0; i < n_more; ++i)
        chunk_rows += s->more_chunk_lens[i];
    if (chunk_rows > c.max_tokens)
        return fail(err, HB_ERANGE, "chunks hold %lld rows > max_tokens %d", chunk_rows, c.max_tokens);
    const int clen = (int)chunk_rows;
    const long long T = (long long)clen + s->n_decodes;
    if (T <= 0)
        return fail(err, HB_EINVAL, "empty batch (no chunk and no decodes)");
    if (T > c.max_tokens)
        return fail(err, HB_ERANGE, "batch has %lld rows > max_tokens %d", T, c.max_tokens);
    *rows = (int)T;
    return HB_OK;
}

// Validation and row metadata of one batch (host only, no GPU).
int plan_batch(const hb_model_config &c, const hb_batch_spec *s, Plan &p, std::string *err)
{
    int T = 0;
    if (const int rc = spec_rows(c, s, &T, err))
        return rc;
    const bool has_chunk = s->chunk_req_id >= 0;
    const int n_more = s->n_more_chunks;
    const int clen = T - s->n_decodes;
    if (s->n_decodes > 0) {
        if (!s->decode_req_ids || !s->decode_ctx_lens || !s->decode_block_tables)
            return fail(err, HB_EINVAL, "decode arrays are NULL");
        if (s->decode_bt_stride <= 0 || s->decode_bt_stride > c.max_blocks_per_seq)
            return fail(err, HB_ERANGE, "decode_bt_stride %d outside 1..max_blocks_per_seq", s->decode_bt_stride);
    }
    // distinct ids
    {
        std::vector<int> ids(s->decode_req_ids, s->decode_req_ids + s->n_decodes);
        for (int id : ids)
            if (id < 0)
                return fail(err, HB_EINVAL, "decode request ids must be >= 0");
        if (has_chunk)
            ids.push_back(s->chunk_req_id);
        for (int i = 0; i < n_more; ++i) {
            if (s->more_chunk_req_ids[i] < 0)
                return fail(err, HB_EINVAL, "further chunk request ids must be >= 0");
            ids.push_back(s->more_chunk_req_ids[i]);
        }
        std::sort(ids.begin(), ids.end());
        if (std::adjacent_find(ids.begin(), ids.end()) != ids.end())
            return fail(err, HB_EINVAL, "duplicate request id in the batch (decode ids and the chunk id must differ)");
    }
    p.T = (int)T;
    p.chunk_len = clen;
    p.n_seq = (has_chunk ? 1 + n_more : 0) + s->n_decodes;
    p.pos.assign(p.T, 0);
    p.slot.assign(p.T, 0);
    p.row_seq.assign(p.T, 0);
    p.seq_q0.clear();
    p.seq_nq.clear();
    p.seq_pos0.clear();
    p.seq_bt.clear();
    p.bt.clear();
    auto add_seq = [&](int q0, int nq, int pos0, const int32_t *bt, int nb_have, const char *what, int idx) -> int {
        const long long last = (long long)pos0 + nq - 1;
        if (last >= c.max_pos)
            return fail(err, HB_ERANGE, "%s %d: position %lld >= max_pos %d", what, idx, last, c.max_pos);
        const int nb = (int)(last / 16) + 1;
        if (nb > nb_have)
            return fail(err, HB_ERANGE, "%s %d: positions up to %lld need %d blocks, table has %d", what, idx, last,
                        nb, nb_have);
        if (nb > c.max_blocks_per_seq)
            return fail(err, HB_ERANGE, "%s %d: needs %d blocks > max_blocks_per_seq %d", what, idx, nb,
                        c.max_blocks_per_seq);
        const int bt0 = (int)p.bt.size();
        for (int b = 0; b < nb; ++b) {
            if (bt[b] < 0 || bt[b] >= c.num_blocks)
                return fail(err, HB_ERANGE, "%s %d: block id %d outside [0, %d)", what, idx, bt[b], c.num_blocks);
            p.bt.push_back(bt[b]);
        }
        const int si = (int)p.seq_q0.size();
        p.seq_q0.push_back(q0);
        p.seq_nq.push_back(nq);
        p.seq_pos0.push_back(pos0);
        p.seq_bt.push_back(bt0);
        for (int i = 0; i < nq; ++i) {
            const int ps = pos0 + i;
            p.pos[q0 + i] = ps;
            p.slot[q0 + i] = bt[ps / 16] * 16 + ps % 16;
            p.row_seq[q0 + i] = si;
        }
        return HB_OK;
    };
    if (has_chunk) {
        if (s->chunk_n_blocks <= 0)
            return fail(err, HB_ERANGE, "chunk_n_blocks must be > 0");
        int rc = add_seq(0, s->chunk_len, s->chunk_offset, s->chunk_block_table, s->chunk_n_blocks, "chunk", 0);
        if (rc)
            return rc;
        int q0 = s->chunk_len;
        for (int i = 0; i < n_more; ++i) {
            rc = add_seq(q0, s->more_chunk_lens[i], s->more_chunk_offsets[i],
                         s->more_chunk_block_tables + (size_t)i * s->more_chunk_bt_stride, s->more_chunk_bt_stride,
                         "further chunk", i);
            if (rc)
                return rc;
            q0 += s->more_chunk_lens[i];
        }
    }
    for (int j = 0; j < s->n_decodes; ++j) {
        const int ctx = s->decode_ctx_lens[j];
        if (ctx < 0)
            return fail(err, HB_EINVAL, "decode %d: ctx %d < 0", j, ctx);
        int rc = add_seq(clen + j, 1, ctx, s->decode_block_tables + (size_t)j * s->decode_bt_stride,
                         s->decode_bt_stride, "decode", j);
        if (rc)
            return rc;
    }
    // no two rows may write the same KV slot
    {
        std::vector<int> sl(p.slot);
        std::sort(sl.begin(), sl.end());
        if (std::adjacent_find(sl.begin(), sl.end()) != sl.end())
            return fail(err, HB_EINVAL, "two rows of the batch map to the same KV slot (block tables overlap)");
    }
    return HB_OK;
}

}  // namespace hb

// ------------------------------------------------------------------ context

#define CK(call)                                                                                     \
    do {                                                                                             \
        cudaError_t e_ = (call);                                                                     \
        if (e_ != cudaSuccess)                                                                       \
            return ctx->set_error(HB_ECUDA, "%s failed: %s", #call, cudaGetErrorString(e_));         \
    } while (0)

int hb_ctx::set_error(int code, const char *fmt, ...)
{
    char buf[768];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    last_error = buf;
    return code;
}

static int ctx_alloc(hb_ctx *ctx, void **p, size_t bytes)
{
    if (bytes == 0)
        bytes = 16;
    cudaError_t e = cudaMalloc(p, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        return ctx->set_error(HB_ENOMEM, "cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
    }
    ctx->allocations.push_back(*p);
    return HB_OK;
}

void hb_ctx::prof_launch_begin(int kind)
{
    n_launches++;
    if (!prof_on)
        return;
    if (prof_used >= prof_events.size()) {
        cudaEvent_t a, b;
        cudaEventCreate(&a);
        cudaEventCreate(&b);
        prof_events.push_back({a, b});
    }
    prof_kinds.push_back(kind);
    cudaEventRecord(prof_events[prof_used].first, stream);
}

void hb_ctx::prof_launch_end()
{
    if (!prof_on)
        return;
    cudaEventRecord(prof_events[prof_used].second, stream);
    prof_used++;
}

extern "C" int hb_plan(const hb_model_config *cfg, const hb_batch_spec *spec, int32_t *pos, int32_t *slot, char *err,
                       int err_len)
{
    std::string e;
    if (!cfg) {
        e = "cfg is NULL";
    } else {
        int rc = validate_config(*cfg, &e);
        if (rc == HB_OK) {
            Plan p;
            rc = plan_batch(*cfg, spec, p, &e);
            if (rc == HB_OK) {
                if (pos)
                    std::copy(p.pos.begin(), p.pos.end(), pos);
                if (slot)
                    std::copy(p.slot.begin(), p.slot.end(), slot);
                return p.T;
            }
        }
        if (err && err_len > 0) {
            snprintf(err, (size_t)err_len, "%s", e.c_str());
        }
        return rc;
    }
    if (err && err_len > 0)
        snprintf(err, (size_t)err_len, "%s", e.c_str());
    return HB_EINVAL;
}

extern "C" int hb_init(const hb_model_config *cfg, const hb_layer_weights *weights, void *cuda_stream,
                       hb_ctx **out)
{
    if (!out)
        return HB_EINVAL;
    *out = nullptr;
    if (!cfg)
        return HB_EINVAL;
    std::string e;
    if (validate_config(*cfg, &e) != HB_OK)
        return HB_EINVAL;
    hb_ctx *ctx = new hb_ctx();
    ctx->cfg = *cfg;
    ctx->stream = (cudaStream_t)cuda_stream;
    const hb_model_config &c = *cfg;
    int rc = HB_OK;
    auto bail = [&](int code) {
        hb_free(ctx);
        return code;
    };
    if (cudaGetDevice(&ctx->device) != cudaSuccess)
        return bail(HB_ECUDA);
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, ctx->device) != cudaSuccess)
        return bail(HB_ECUDA);
    ctx->num_sms = prop.multiProcessorCount;
    ctx->cc_major = prop.major;
    ctx->cc_minor = prop.minor;

    const int d = c.head_dim, H = c.hidden, F = c.ffn;
    const int qd = c.n_heads * d, kvd = c.n_kv_heads * d;
    ctx->n_qkv = qd + 2 * kvd;
    ctx->n_qkv_pad = (int)round_up(ctx->n_qkv, 128);
    ctx->n_gu = 2 * F;
    ctx->n_gu_pad = (int)round_up(ctx->n_gu, 128);

    // KV pools: [layer][K|V][num_blocks][n_kv][16][d]
    ctx->kv_elems_per_pool = (size_t)c.num_blocks * c.n_kv_heads * 16 * d;
    if ((rc = ctx_alloc(ctx, (void **)&ctx->kv, ctx->kv_elems_per_pool * 2 * c.n_layers * sizeof(bf16))))
        return bail(rc);

    ctx->layers.resize(c.n_layers);
    for (int l = 0; l < c.n_layers; ++l) {
        LayerDev &L = ctx->layers[l];
        if ((rc = ctx_alloc(ctx, (void **)&L.w_qkv, tiled_weight_elems(ctx->n_qkv, H) * sizeof(bf16))) ||
            (rc = ctx_alloc(ctx, (void **)&L.w_o, tiled_weight_elems(H, qd) * sizeof(bf16))) ||
            (rc = ctx_alloc(ctx, (void **)&L.w_gu, tiled_weight_elems(ctx->n_gu, H) * sizeof(bf16))) ||
            (rc = ctx_alloc(ctx, (void **)&L.w_d, tiled_weight_elems(H, F) * sizeof(bf16))) ||
            (rc = ctx_alloc(ctx, (void **)&L.g1, (size_t)H * sizeof(float))) ||
            (rc = ctx_alloc(ctx, (void **)&L.g2, (size_t)H * sizeof(float))))
            return bail(rc);
        L.k_pool = ctx->kv + ctx->kv_elems_per_pool * (2 * (size_t)l);
        L.v_pool = ctx->kv + ctx->kv_elems_per_pool * (2 * (size_t)l + 1);
    }

    // RoPE table in fp64 on the host, stored fp32: angle = pos * theta^(-2j/d)
    {
        const int half = d / 2;
        std::vector<float2> tab((size_t)c.max_pos * half);
        for (int p = 0; p < c.max_pos; ++p)
            for (int j = 0; j < half; ++j) {
                const double inv = std::pow((double)c.rope_theta, -2.0 * j / (double)d);
                const double a = (double)p * inv;
                tab[(size_t)p * half + j] = make_float2((float)std::cos(a), (float)std::sin(a));
            }
        if ((rc = ctx_alloc(ctx, (void **)&ctx->rope, tab.size() * sizeof(float2))))
            return bail(rc);
        if (cudaMemcpy(ctx->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess)
            return bail(HB_ECUDA);
    }

    const size_t MT = (size_t)c.max_tokens;
    if ((rc = ctx_alloc(ctx, (void **)&ctx->xn, MT * H * sizeof(bf16))) ||
        (rc = ctx_alloc(ctx, (void **)&ctx->q, MT * qd * sizeof(bf16))) ||
        (rc = ctx_alloc(ctx, (void **)&ctx->attn_o, MT * qd * sizeof(bf16))) ||
        (rc = ctx_alloc(ctx, (void **)&ctx->h, MT * H * sizeof(bf16))) ||
        (rc = ctx_alloc(ctx, (void **)&ctx->act, MT * F * sizeof(bf16))) ||
        (rc = ctx_alloc(ctx, (void **)&ctx->xa, MT * H * sizeof(bf16))) ||
        (rc = ctx_alloc(ctx, (void **)&ctx->xb, MT * H * sizeof(bf16))) ||
        (rc = ctx_alloc(ctx, (void **)&ctx->host_in, MT * H * sizeof(bf16))) ||
        (rc = ctx_alloc(ctx, (void **)&ctx->host_out, MT * H * sizeof(bf16))) ||
        (rc = ctx_alloc(ctx, (void **)&ctx->err_word, sizeof(int))))
        return bail(rc);
    if (cudaMemset(ctx->err_word, 0, sizeof(int)) != cudaSuccess)
        return bail(HB_ECUDA);

    // metadata: 3 T + 4 n_seq + block tables + attention work list
    const size_t max_seq = (size_t)c.max_decodes + HB_MAX_CHUNKS;
    ctx->meta_cap = (3 * MT + 4 * max_seq + max_seq * c.max_blocks_per_seq + kMetaExtraWords(c) + 3) / 4 * 4;
    if ((rc = ctx_alloc(ctx, (void **)&ctx->d_meta, ctx->meta_cap * sizeof(int))))
        return bail(rc);
    if (cudaMallocHost((void **)&ctx->h_err, sizeof(int)) != cudaSuccess) {
        ctx->h_err = nullptr;
        return bail(HB_ENOMEM);
    }
    *ctx->h_err = 0;
    for (int i = 0; i < kMetaRing; ++i) {
        if (cudaHostAlloc((void **)&ctx->h_meta[i], ctx->meta_cap * sizeof(int), cudaHostAllocMapped) != cudaSuccess) {
            ctx->h_meta[i] = nullptr;
            return bail(HB_ENOMEM);
        }
        if (cudaHostGetDevicePointer((void **)&ctx->h_meta_dev[i], ctx->h_meta[i], 0) != cudaSuccess ||
            (uintptr_t)ctx->h_meta_dev[i] % 16 != 0)
            return bail(HB_ECUDA);
        if (cudaEventCreateWithFlags(&ctx->meta_ev[i], cudaEventDisableTiming) != cudaSuccess)
            return bail(HB_ECUDA);
    }
    if ((rc = hb_init_fast_path(ctx)))
        return bail(rc);

    if (weights) {
        for (int l = 0; l < c.n_layers; ++l) {
            if ((rc = hb_load_layer(ctx, l, &weights[l])))
                return bail(rc);
        }
    }
    if (cudaStreamSynchronize(ctx->stream) != cudaSuccess)
        return bail(HB_ECUDA);
    *out = ctx;
    return HB_OK;
}

extern "C" int hb_load_layer(hb_ctx *ctx, int layer, const hb_layer_weights *w)
{
    if (!ctx)
        return HB_EINVAL;
    const hb_model_config &c = ctx->cfg;
    if (layer < 0 || layer >= c.n_layers)
        return ctx->set_error(HB_ERANGE, "layer %d outside [0, %d)", layer, c.n_layers);
    if (!w || !w->w_qkv || !w->w_o || !w->w_gate_up || !w->w_down || !w->norm1 || !w->norm2)
        return ctx->set_error(HB_EINVAL, "layer %d: a weight pointer is NULL", layer);
    LayerDev &L = ctx->layers[layer];
    const int H = c.hidden, qd = c.n_heads * c.head_dim, F = c.ffn;
    cudaStream_t s = ctx->stream;
    ctx->n_launches += 6;
    // tensor-core tiled layout; q/k/v rows paired for RoPE, gate/up rows interleaved
    CK(launch_tile_weights((const bf16 *)w->w_qkv, L.w_qkv, ctx->n_qkv, H, 1, c.head_dim, s));
    CK(launch_tile_weights((const bf16 *)w->w_o, L.w_o, H, qd, 0, 0, s));
    CK(launch_tile_weights((const bf16 *)w->w_gate_up, L.w_gu, ctx->n_gu, H, 2, F, s));
    CK(launch_tile_weights((const bf16 *)w->w_down, L.w_d, H, F, 0, 0, s));
    CK(launch_bf16_to_f32((const bf16 *)w->norm1, L.g1, H, s));
    CK(launch_bf16_to_f32((const bf16 *)w->norm2, L.g2, H, s));
    L.loaded = true;
    return HB_OK;
}

static int kv_io(hb_ctx *ctx, int layer, const int32_t *bt, int n_blocks, int start_pos, int n_tokens, const void *k,
                 const void *v, bool write)
{
    if (!ctx)
        return HB_EINVAL;
    const hb_model_config &c = ctx->cfg;
    if (layer < 0 || layer >= c.n_layers)
        return ctx->set_error(HB_ERANGE, "layer %d outside [0, %d)", layer, c.n_layers);
    if (n_tokens < 0 || start_pos < 0)
        return ctx->set_error(HB_EINVAL, "n_tokens and start_pos must be >= 0");
    if (n_tokens == 0)
        return HB_OK;
    if (!bt || !k || !v)
        return ctx->set_error(HB_EINVAL, "NULL pointer");
    const long long last = (long long)start_pos + n_tokens - 1;
    const int nb = (int)(last / 16) + 1;
    if (nb > n_blocks || nb > c.max_blocks_per_seq)
        return ctx->set_error(HB_ERANGE, "positions up to %lld need %d blocks, table has %d", last, nb, n_blocks);
    for (int b = 0; b < nb; ++b)
        if (bt[b] < 0 || bt[b] >= c.num_blocks)
            return ctx->set_error(HB_ERANGE, "block id %d outside [0, %d)", bt[b], c.num_blocks);
    // stage the table through the metadata ring
    int *hm = ctx->next_meta_host();
    if (!hm)
        return ctx->set_error(HB_ECUDA, "metadata staging wait failed");
    if ((size_t)nb > ctx->meta_cap)
        return ctx->set_error(HB_ERANGE, "table too long");
    std::copy(bt, bt + nb, hm);
    CK(cudaMemcpyAsync(ctx->d_meta, hm, nb * sizeof(int), cudaMemcpyHostToDevice, ctx->stream));
    CK(cudaEventRecord(ctx->meta_ev[ctx->meta_i], ctx->stream));
    LayerDev &L = ctx->layers[layer];
    ctx->prof_launch_begin(K_KVIO);
    cudaError_t e;
    if (write)
        e = launch_kv_write(L.k_pool, L.v_pool, (const bf16 *)k, (const bf16 *)v, ctx->d_meta, start_pos, n_tokens,
                            c.n_kv_heads, c.head_dim, c.num_blocks, ctx->err_word, ctx->stream);
    else
        e = launch_kv_read(L.k_pool, L.v_pool, (bf16 *)k, (bf16 *)v, ctx->d_meta, start_pos, n_tokens, c.n_kv_heads,
                           c.head_dim, c.num_blocks, ctx->err_word, ctx->stream);
    ctx->prof_launch_end();
    if (e != cudaSuccess)
        return ctx->set_error(HB_ECUDA, "kv copy launch: %s", cudaGetErrorString(e));
    return HB_OK;
}

extern "C" int hb_append_kv(hb_ctx *ctx, int layer, const int32_t *block_table, int n_blocks, int start_pos,
                            int n_tokens, const void *k, const void *v)
{
    return kv_io(ctx, layer, block_table, n_blocks, start_pos, n_tokens, k, v, true);
}

extern "C" int hb_read_kv(hb_ctx *ctx, int layer, const int32_t *block_table, int n_blocks, int start_pos,
                          int n_tokens, void *k, void *v)
{
    return kv_io(ctx, layer, block_table, n_blocks, start_pos, n_tokens, k, v, false);
}

extern "C" int hb_fill_kv(hb_ctx *ctx, uint16_t bits)
{
    if (!ctx)
        return HB_EINVAL;
    ctx->n_launches++;
    CK(launch_fill_u16((uint16_t *)ctx->kv, ctx->kv_elems_per_pool * 2 * ctx->cfg.n_layers, bits, ctx->stream));
    return HB_OK;
}

int *hb_ctx::next_meta_host()
{
    meta_i = (meta_i + 1) % kMetaRing;
    if (meta_used[meta_i] && cudaEventSynchronize(meta_ev[meta_i]) != cudaSuccess)
        return nullptr;
    meta_used[meta_i] = true;
    return h_meta[meta_i];
}

// Upload the plan; fills `b` with device pointers into d_meta.
static int upload_plan(hb_ctx *ctx, const Plan &p, BatchDev &b)
{
    int *hm = ctx->next_meta_host();
    if (!hm)
        return ctx->set_error(HB_ECUDA, "metadata staging wait failed");
    size_t at = 0;
    auto put = [&](const std::vector<int> &v) {
        const size_t o = at;
        std::copy(v.begin(), v.end(), hm + at);
        at += v.size();
        return ctx->d_meta + o;
    };
    b.T = p.T;
    b.n_seq = p.n_seq;
    b.chunk_len = p.chunk_len;
    b.pos = put(p.pos);
    b.slot = put(p.slot);
    b.row_seq = put(p.row_seq);
    b.seq_q0 = put(p.seq_q0);
    b.seq_nq = put(p.seq_nq);
    b.seq_pos0 = put(p.seq_pos0);
    b.seq_bt = put(p.seq_bt);
    b.bt = put(p.bt);
    int rc = hb_plan_fast_path(ctx, p, hm, at, b);
    if (rc)
        return rc;
    if (at > ctx->meta_cap)
        return ctx->set_error(HB_ERANGE, "metadata overflow (%zu > %zu words)", at, ctx->meta_cap);
    // the step's first kernel copies the plan to d_meta (no copy breaks the
    // chain of programmatic launches); the staging buffer is reused only
    // after the event that launch_layers records behind the step
    ctx->meta_src = ctx->h_meta_dev[ctx->meta_i];
    ctx->meta_n16 = (int)((at + 3) / 4);
    return HB_OK;
}

// Validates the call, plans the batch into ctx->plan and uploads the plan's
// device metadata (stream-ordered before any later launch).
static int prepare_layers(hb_ctx *ctx, const hb_batch_spec *spec, int l0, int l1, const void *x_in, const void *x_out,
                          BatchDev &b)
{
    if (!ctx)
        return HB_EINVAL;
    const hb_model_config &c = ctx->cfg;
    if (l0 < 0 || l1 > c.n_layers || l0 >= l1)
        return ctx->set_error(HB_ERANGE, "layer range [%d, %d) invalid", l0, l1);
    if (!x_in || !x_out)
        return ctx->set_error(HB_EINVAL, "x_in / x_out is NULL");
    if (((uintptr_t)x_in | (uintptr_t)x_out) % 16 != 0)  // rows are read and written as 16-byte vectors
        return ctx->set_error(HB_EINVAL, "x_in / x_out must be 16-byte aligned");
    for (int l = l0; l < l1; ++l)
        if (!ctx->layers[l].loaded)
            return ctx->set_error(HB_ESTATE, "layer %d has no weights", l);
    Plan &p = ctx->plan;
    std::string e;
    int rc = plan_batch(c, spec, p, &e);
    if (rc)
        return ctx->set_error(rc, "%s", e.c_str());
    const size_t xbytes = (size_t)p.T * c.hidden * sizeof(bf16);
    const char *xi = (const char *)x_in;
    const char *xo = (const char *)x_out;
    if (xi < xo + xbytes && xo < xi + xbytes)
        return ctx->set_error(HB_EINVAL, "x_in and x_out overlap");
    return upload_plan(ctx, p, b);
}

// Launches layers [l0, l1) of the prepared batch.
static int launch_layers(hb_ctx *ctx, const BatchDev &b, int l0, int l1, const void *x_in, void *x_out)
{
    int rc;
    const bf16 *x = (const bf16 *)x_in;
    for (int l = l0; l < l1; ++l) {
        bf16 *y = (l == l1 - 1) ? (bf16 *)x_out : ((l - l0) % 2 == 0 ? ctx->xa : ctx->xb);
        rc = run_layer(ctx, l, l0, l1, b, x, y);
        // behind the plan's copy; recorded on failure too, since the copying
        // kernel may have been launched before a later launch failed
        if (l == l0 && cudaEventRecord(ctx->meta_ev[ctx->meta_i], ctx->stream) != cudaSuccess && !rc)
            rc = ctx->set_error(HB_ECUDA, "cudaEventRecord failed");
        if (rc)
            return rc;
        x = y;
    }
    return HB_OK;
}

static int run_layers(hb_ctx *ctx, const hb_batch_spec *spec, int l0, int l1, const void *x_in, void *x_out)
{
    BatchDev b;
    const int rc = prepare_layers(ctx, spec, l0, l1, x_in, x_out, b);
    return rc ? rc : launch_layers(ctx, b, l0, l1, x_in, x_out);
}

extern "C" int hb_forward(hb_ctx *ctx, const hb_batch_spec *spec, const void *x_in, void *x_out)
{
    if (!ctx)
        return HB_EINVAL;
    return run_layers(ctx, spec, 0, ctx->cfg.n_layers, x_in, x_out);
}

extern "C" int hb_forward_layers(hb_ctx *ctx, const hb_batch_spec *spec, int layer_begin, int layer_end,
                                 const void *x_in, void *x_out)
{
    return run_layers(ctx, spec, layer_begin, layer_end, x_in, x_out);
}

extern "C" int hb_forward_host(hb_ctx *ctx, const hb_batch_spec *spec, const void *x_in_host, void *x_out_host)
{
    if (!ctx)
        return HB_EINVAL;
    if (!x_in_host || !x_out_host)
        return ctx->set_error(HB_EINVAL, "NULL host buffer");
    std::string e;
    int T = 0;
    int rc = spec_rows(ctx->cfg, spec, &T, &e);
    if (rc)
        return ctx->set_error(rc, "%s", e.c_str());
    // the input copy runs while the host plans the batch
    const size_t bytes = (size_t)T * ctx->cfg.hidden * sizeof(bf16);
    CK(cudaMemcpyAsync(ctx->host_in, x_in_host, bytes, cudaMemcpyHostToDevice, ctx->stream));
    // A page-locked output buffer that the GPU can address is written in
    // place by the last kernel's stores (every output store is a plain
    // st.global of 16 bytes, so the buffer must be 16-byte aligned), so no
    // copy follows the stack; any other buffer gets the result by a
    // device-to-host copy.
    void *y_mapped = nullptr;
    cudaPointerAttributes pa{};
    if (cudaPointerGetAttributes(&pa, x_out_host) == cudaSuccess) {
        if (pa.type == cudaMemoryTypeHost && pa.devicePointer && (uintptr_t)pa.devicePointer % 16 == 0)
            y_mapped = pa.devicePointer;
    } else {
        cudaGetLastError();  // not a CUDA-known pointer: clear the error, copy
    }
    void *y = y_mapped ? y_mapped : (void *)ctx->host_out;
    BatchDev b;
    if ((rc = prepare_layers(ctx, spec, 0, ctx->cfg.n_layers, ctx->host_in, y, b)) ||
        (rc = launch_layers(ctx, b, 0, ctx->cfg.n_layers, ctx->host_in, y))) {
        cudaStreamSynchronize(ctx->stream);  // x_in_host is the caller's again once this returns
        return rc;
    }
    if (!y_mapped)
        CK(cudaMemcpyAsync(x_out_host, ctx->host_out, bytes, cudaMemcpyDeviceToHost, ctx->stream));
    return hb_sync(ctx);
}

// The first asynchronous call of a context makes its input ring.
static int async_setup(hb_ctx *ctx)
{
    if (ctx->copy_stream)
        return HB_OK;
    // each piece is made once, so that a setup that failed part-way can be
    // retried by the next call without leaking what it had made
    const size_t bytes = (size_t)ctx->cfg.max_tokens * ctx->cfg.hidden * sizeof(bf16);
    int rc;
    for (bf16 **buf : {&ctx->async_in[0], &ctx->async_in[1], &ctx->async_out[0], &ctx->async_out[1]})
        if (!*buf && (rc = ctx_alloc(ctx, (void **)buf, bytes)))
            return rc;
    for (cudaEvent_t *ev : {&ctx->in_ready[0], &ctx->in_ready[1], &ctx->in_free[0], &ctx->in_free[1],
                            &ctx->out_free[0], &ctx->out_free[1]})
        if (!*ev && cudaEventCreateWithFlags(ev, cudaEventDisableTiming) != cudaSuccess) {
            *ev = nullptr;
            return ctx->set_error(HB_ECUDA, "cudaEventCreate failed");
        }
    // the output stream first: copy_stream marks a finished setup
    if (!ctx->out_stream && cudaStreamCreateWithFlags(&ctx->out_stream, cudaStreamNonBlocking) != cudaSuccess) {
        ctx->out_stream = nullptr;
        return ctx->set_error(HB_ECUDA, "cudaStreamCreate failed");
    }
    if (cudaStreamCreateWithFlags(&ctx->copy_stream, cudaStreamNonBlocking) != cudaSuccess) {
        ctx->copy_stream = nullptr;
        return ctx->set_error(HB_ECUDA, "cudaStreamCreate failed");
    }
    return HB_OK;
}

extern "C" int hb_forward_host_async(hb_ctx *ctx, const hb_batch_spec *spec, const void *x_in_host,
                                     void *x_out_host)
{
    if (!ctx)
        return HB_EINVAL;
    if (!x_in_host || !x_out_host)
        return ctx->set_error(HB_EINVAL, "NULL host buffer");
    std::string e;
    int T = 0;
    int rc = spec_rows(ctx->cfg, spec, &T, &e);
    if (rc)
        return ctx->set_error(rc, "%s", e.c_str());
    if ((rc = async_setup(ctx)))
        return rc;
    // the output must be page-locked, so that its copy is asynchronous
    cudaPointerAttributes pa{};
    if (cudaPointerGetAttributes(&pa, x_out_host) != cudaSuccess) {
        cudaGetLastError();
        return ctx->set_error(HB_EINVAL, "x_out_host is not page-locked host memory");
    }
    if (pa.type != cudaMemoryTypeHost)
        return ctx->set_error(HB_EINVAL, "x_out_host is not page-locked host memory");
    // slot k: the input copy waits for the step that last read input slot k
    // and runs on the copy stream while the previous step computes; the step
    // waits for it and for the copy that last read output slot k; the output
    // copy follows the step on the output stream, beside the next step
    const int k = ctx->in_i ^= 1;
    const size_t bytes = (size_t)T * ctx->cfg.hidden * sizeof(bf16);
    if (ctx->in_used[k])
        CK(cudaStreamWaitEvent(ctx->copy_stream, ctx->in_free[k], 0));
    CK(cudaMemcpyAsync(ctx->async_in[k], x_in_host, bytes, cudaMemcpyHostToDevice, ctx->copy_stream));
    CK(cudaEventRecord(ctx->in_ready[k], ctx->copy_stream));
    CK(cudaStreamWaitEvent(ctx->stream, ctx->in_ready[k], 0));
    if (ctx->in_used[k])
        CK(cudaStreamWaitEvent(ctx->stream, ctx->out_free[k], 0));
    BatchDev b;
    if ((rc = prepare_layers(ctx, spec, 0, ctx->cfg.n_layers, ctx->async_in[k], ctx->async_out[k], b)) ||
        (rc = launch_layers(ctx, b, 0, ctx->cfg.n_layers, ctx->async_in[k], ctx->async_out[k]))) {
        cudaStreamSynchronize(ctx->stream);  // nothing of this call is left in flight
        return rc;
    }
    CK(cudaEventRecord(ctx->in_free[k], ctx->stream));
    CK(cudaStreamWaitEvent(ctx->out_stream, ctx->in_free[k], 0));
    CK(cudaMemcpyAsync(x_out_host, ctx->async_out[k], bytes, cudaMemcpyDeviceToHost, ctx->out_stream));
    CK(cudaEventRecord(ctx->out_free[k], ctx->out_stream));
    ctx->in_used[k] = true;
    return HB_OK;
}

extern "C" int hb_sync(hb_ctx *ctx)
{
    if (!ctx)
        return HB_EINVAL;
    // the error word comes back on the stream, after its work: one wait
    CK(cudaMemcpyAsync(ctx->h_err, ctx->err_word, sizeof(int), cudaMemcpyDeviceToHost, ctx->stream));
    CK(cudaStreamSynchronize(ctx->stream));
    if (ctx->out_stream)
        CK(cudaStreamSynchronize(ctx->out_stream));  // the asynchronous calls' output copies
    const int w = *ctx->h_err;
    if (w) {
        CK(cudaMemset(ctx->err_word, 0, sizeof(int)));
        return ctx->set_error(HB_EDEVICE, "device error word = %d (%s)", w,
                              w == DERR_MBAR_TIMEOUT  ? "mbarrier wait timed out"
                              : w == DERR_BAD_SLOT    ? "slot outside the pool"
                              : w == DERR_TMEM_ALLOC  ? "tensor memory allocation"
                              : w == DERR_BAD_WORK    ? "work item out of bounds"
                                                      : "unknown");
    }
    return HB_OK;
}

extern "C" int hb_profile(hb_ctx *ctx, int enable)
{
    if (!ctx)
        return HB_EINVAL;
    if (enable) {
        ctx->prof_used = 0;
        ctx->prof_kinds.clear();
    }
    ctx->prof_on = enable != 0;
    return HB_OK;
}

extern "C" int hb_profile_read(hb_ctx *ctx, const char **names, double *total_ms, int *launches, int max_kinds)
{
    if (!ctx)
        return HB_EINVAL;
    double tot[K_NUM_KINDS] = {0};
    int cnt[K_NUM_KINDS] = {0};
    for (size_t i = 0; i < ctx->prof_used; ++i) {
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, ctx->prof_events[i].first, ctx->prof_events[i].second) != cudaSuccess)
            return ctx->set_error(HB_ECUDA, "cudaEventElapsedTime failed (call hb_sync first)");
        tot[ctx->prof_kinds[i]] += ms;
        cnt[ctx->prof_kinds[i]]++;
    }
    int n = 0;
    for (int k = 0; k < K_NUM_KINDS && n < max_kinds; ++k) {
        if (!cnt[k])
            continue;
        if (names)
            names[n] = kKindNames[k];
        if (total_ms)
            total_ms[n] = tot[k];
        if (launches)
            launches[n] = cnt[k];
        ++n;
    }
    return n;
}

extern "C" int hb_debug_read(hb_ctx *ctx, int which, void *dst, int rows)
{
    if (!ctx)
        return HB_EINVAL;
    const hb_model_config &c = ctx->cfg;
    if (!dst || rows <= 0 || rows > c.max_tokens)
        return ctx->set_error(HB_EINVAL, "hb_debug_read: bad arguments");
    const void *src = nullptr;
    size_t width = 0;
    switch (which) {
    case 0: src = ctx->xn; width = c.hidden; break;
    case 1: src = ctx->q; width = (size_t)c.n_heads * c.head_dim; break;
    case 2: src = ctx->attn_o; width = (size_t)c.n_heads * c.head_dim; break;
    case 3: src = ctx->h; width = c.hidden; break;
    case 4: src = ctx->act; width = c.ffn; break;
    default: return ctx->set_error(HB_EINVAL, "hb_debug_read: which %d unknown", which);
    }
    CK(cudaMemcpyAsync(dst, src, (size_t)rows * width * sizeof(bf16), cudaMemcpyDeviceToDevice, ctx->stream));
    return HB_OK;
}

extern "C" long long hb_launch_count(hb_ctx *ctx) { return ctx ? ctx->n_launches : -1; }

extern "C" const char *hb_last_error(hb_ctx *ctx) { return ctx ? ctx->last_error.c_str() : "NULL context"; }

extern "C" void hb_free(hb_ctx *ctx)
{
    if (!ctx)
        return;
    cudaStreamSynchronize(ctx->stream);
    if (ctx->copy_stream) {
        cudaStreamSynchronize(ctx->copy_stream);
        cudaStreamDestroy(ctx->copy_stream);
    }
    if (ctx->out_stream) {
        cudaStreamSynchronize(ctx->out_stream);
        cudaStreamDestroy(ctx->out_stream);
    }
    for (int k = 0; k < 2; ++k) {
        if (ctx->in_ready[k])
            cudaEventDestroy(ctx->in_ready[k]);
        if (ctx->in_free[k])
            cudaEventDestroy(ctx->in_free[k]);
        if (ctx->out_free[k])
            cudaEventDestroy(ctx->out_free[k]);
    }
    hb_free_fast_path(ctx);
    for (void *p : ctx->allocations)
        cudaFree(p);
    if (ctx->h_err)
        cudaFreeHost(ctx->h_err);
    for (int i = 0; i < kMetaRing; ++i) {
        if (ctx->h_meta[i])
            cudaFreeHost(ctx->h_meta[i]);
        if (ctx->meta_ev[i])
            cudaEventDestroy(ctx->meta_ev[i]);
    }
    for (auto &pr : ctx->prof_events) {
        cudaEventDestroy(pr.first);
        cudaEventDestroy(pr.second);
    }
    delete ctx;
}
