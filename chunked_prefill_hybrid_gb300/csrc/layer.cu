// layer.cu -- the per-layer launch sequence and kernel selection.
#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "attention.h"
#include "gemm_tc.h"
#include "kernels.h"
#include "runtime_internal.h"

using namespace hb;

namespace hb {

// Tensor maps of a layer's four tiled weights (128-row boxes).
enum WKind { W_QKV = 0, W_O, W_GU, W_D };
struct LayerMaps {
    CUtensorMap m[4];
};

struct FastPath {
    TcRuntime rt;
    std::vector<LayerMaps> maps;
    bf16 *test_w = nullptr;  // tiled copy of the hb_gemm_test operand
    size_t test_w_elems = 0;
    // hybrid attention
    float *attn_part = nullptr;
    int *attn_counters = nullptr;
    std::vector<int> items, part_off;
    const int *d_items = nullptr, *d_part_off = nullptr;
    int n_items = 0, n_chunk_items = 0;
    std::vector<CUtensorMap> kv_maps;  // [layer][K, V] pool maps of the tcgen05 chunk attention
    uint64_t fault_wait_ns = 0;        // armed test fault (hb_test_wait_timeout), 0 = none
    float *ss = nullptr;               // [hidden / 128][max_tokens] partial sums of squares (split-K path)
};

static size_t max_seqs(const hb_model_config &c) { return (size_t)c.max_decodes + HB_MAX_CHUNKS; }
static size_t max_splits_per_seq(const hb_model_config &c) { return (size_t)(c.max_pos + 1) / ATTN_SPLIT + 1; }
static size_t max_items(const hb_model_config &c)
{
    return ((size_t)c.max_tokens + 63) / 64 + HB_MAX_CHUNKS + max_seqs(c) * max_splits_per_seq(c);
}

size_t kMetaExtraWords(const hb_model_config &c) { return 2 * max_items(c) + max_seqs(c); }

}  // namespace hb

int hb_init_fast_path(hb_ctx *ctx)
{
    FastPath *f = new FastPath();
    ctx->fast = f;
    TcRuntime &rt = f->rt;
    if (cudaDeviceGetAttribute(&rt.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, ctx->device) != cudaSuccess)
        return ctx->set_error(HB_ECUDA, "cudaDeviceGetAttribute failed");
    rt.num_sms = ctx->num_sms;
    {
        const hb_model_config &c = ctx->cfg;
        const int Ns[4] = {ctx->n_qkv, c.hidden, ctx->n_gu, c.hidden};
        const int Ks[4] = {c.hidden, c.n_heads * c.head_dim, c.hidden, c.ffn};
        rt.ws_floats = tc_pair_workspace_floats(ctx->num_sms, c.max_tokens, Ns, Ks, 4);
        const size_t floor_floats = (size_t)ctx->num_sms * 2 * 512 * 128;  // room for hb_gemm_test shapes
        if (rt.ws_floats < floor_floats)
            rt.ws_floats = floor_floats;
    }
    rt.n_counters = 8192;
    if (cudaMalloc((void **)&rt.ws, rt.ws_floats * sizeof(float)) != cudaSuccess ||
        cudaMalloc((void **)&rt.counters, rt.n_counters * sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return ctx->set_error(HB_ENOMEM, "GEMM workspace allocation failed");
    }
    if (cudaMemset(rt.counters, 0, rt.n_counters * sizeof(int)) != cudaSuccess)
        return ctx->set_error(HB_ECUDA, "cudaMemset failed");
    const hb_model_config &c = ctx->cfg;
    {
        const size_t parts = max_seqs(c) * max_splits_per_seq(c) * c.n_heads * (2 + (size_t)c.head_dim);
        const size_t cnts = max_seqs(c) * c.n_heads;
        if (cudaMalloc((void **)&f->attn_part, parts * sizeof(float)) != cudaSuccess ||
            cudaMalloc((void **)&f->attn_counters, cnts * sizeof(int)) != cudaSuccess) {
            cudaGetLastError();
            return ctx->set_error(HB_ENOMEM, "attention workspace allocation failed");
        }
        if (cudaMemset(f->attn_counters, 0, cnts * sizeof(int)) != cudaSuccess)
            return ctx->set_error(HB_ECUDA, "cudaMemset failed");
        const size_t ssn = ((size_t)c.hidden / 128 + 1) * c.max_tokens;
        if (cudaMalloc((void **)&f->ss, ssn * sizeof(float)) != cudaSuccess) {
            cudaGetLastError();
            return ctx->set_error(HB_ENOMEM, "split-K workspace allocation failed");
        }
        f->items.resize(2 * max_items(c));
        f->part_off.resize(max_seqs(c));
    }
    const int H = c.hidden, qd = c.n_heads * c.head_dim;
    f->maps.resize(c.n_layers);
    for (int l = 0; l < c.n_layers; ++l) {
        const LayerDev &L = ctx->layers[l];
        LayerMaps &m = f->maps[l];
        if (!make_tmap_tiled_weights(&m.m[W_QKV], L.w_qkv, ctx->n_qkv, H, 128) ||
            !make_tmap_tiled_weights(&m.m[W_O], L.w_o, H, qd, 128) ||
            !make_tmap_tiled_weights(&m.m[W_GU], L.w_gu, ctx->n_gu, H, 128) ||
            !make_tmap_tiled_weights(&m.m[W_D], L.w_d, H, c.ffn, 128))
            return ctx->set_error(HB_ECUDA, "cuTensorMapEncodeTiled failed (driver entry point unavailable?)");
    }
    f->kv_maps.resize(2 * (size_t)c.n_layers);
    for (int l = 0; l < c.n_layers; ++l)
        if (!make_tmap_kv_pool(&f->kv_maps[2 * l], ctx->layers[l].k_pool, c.num_blocks, c.n_kv_heads, c.head_dim) ||
            !make_tmap_kv_pool(&f->kv_maps[2 * l + 1], ctx->layers[l].v_pool, c.num_blocks, c.n_kv_heads,
                               c.head_dim))
            return ctx->set_error(HB_ECUDA, "cuTensorMapEncodeTiled failed for a KV pool");
    ctx->gemm_impl = 2;
    ctx->attn_impl = 1;
    return HB_OK;
}

void hb_free_fast_path(hb_ctx *ctx)
{
    if (ctx->fast) {
        cudaFree(ctx->fast->rt.ws);
        cudaFree(ctx->fast->rt.counters);
        cudaFree(ctx->fast->test_w);
        cudaFree(ctx->fast->attn_part);
        cudaFree(ctx->fast->attn_counters);
        cudaFree(ctx->fast->ss);
    }
    delete ctx->fast;
    ctx->fast = nullptr;
}

// Attention work list of the batch, appended to the metadata upload.
int hb_plan_fast_path(hb_ctx *ctx, const Plan &p, int *hm, size_t &at, BatchDev &b)
{
    (void)b;
    FastPath *f = ctx->fast;
    int n_chunk = 0;
    const int n = attn_build_items(p.seq_nq.data(), p.seq_pos0.data(), p.n_seq, f->items.data(),
                                   f->part_off.data(), &n_chunk, ctx->attn_impl == 2 ? attn_tc_chunk_rows() : 64);
    if ((size_t)n > max_items(ctx->cfg))
        return ctx->set_error(HB_ERANGE, "attention work list overflow");
    std::copy(f->items.begin(), f->items.begin() + 2 * n, hm + at);
    f->d_items = ctx->d_meta + at;
    at += 2 * (size_t)n;
    std::copy(f->part_off.begin(), f->part_off.begin() + p.n_seq, hm + at);
    f->d_part_off = ctx->d_meta + at;
    at += p.n_seq;
    f->n_items = n;
    f->n_chunk_items = n_chunk;
    return HB_OK;
}

#define LK(kind, call)                                                                                   \
    do {                                                                                                 \
        ctx->prof_launch_begin(kind);                                                                    \
        cudaError_t e_ = (call);                                                                         \
        ctx->prof_launch_end();                                                                          \
        if (e_ != cudaSuccess)                                                                           \
            return ctx->set_error(HB_ECUDA, "launch %s failed: %s", kKindNames[kind], cudaGetErrorString(e_)); \
    } while (0)

// rows per launch of the tensor-core kernel for a batch of T rows: one
// launch takes up to TC_PAIR_MAX_ROWS rows (slabs of up to TC_PAIR_MAX_T
// rows, each with the weights read once from HBM); larger batches run as the
// fewest launches, with their rows balanced
static int launch_rows(int T)
{
    const int mx = TC_PAIR_MAX_ROWS;
    const int n = (T + mx - 1) / mx;
    return n > 1 ? (T + n - 1) / n : mx;
}

// One launch of the tensor-core kernel (a pending test fault goes to the
// first launch after it was armed).
static cudaError_t launch_tc(hb_ctx *ctx, const LayerMaps &M, int kind, const bf16 *W, const bf16 *X, int T,
                             int N, int K, const EpiParams &ep, TcPartition *part = nullptr)
{
    const uint64_t fault = ctx->fast->fault_wait_ns;
    ctx->fast->fault_wait_ns = 0;
    return launch_gemm_pair(M.m[kind], W, X, T, N, K, ep, ctx->fast->rt, ctx->stream, part, true, 0, fault);
}

// The epilogue parameters of rows [t0, t0 + Tn) of a batch.
static EpiParams epi_rows(const EpiParams &ep, int t0, int Tn)
{
    EpiParams e = ep;
    e.T = Tn;
    if (e.pos)
        e.pos += t0;
    if (e.slot)
        e.slot += t0;
    if (e.q_out)
        e.q_out += (size_t)t0 * e.n_heads * e.head_dim;
    if (e.resid)
        e.resid += (size_t)t0 * e.N;
    if (e.out)
        e.out += (size_t)t0 * e.N;
    if (e.act)
        e.act += (size_t)t0 * e.ffn;
    if (e.d32)
        e.d32 += (size_t)t0 * e.N;
    return e;
}

// Attention with the tcgen05 chunk kernel, then the decode kernel as its
// dependent (see attention.h).
static cudaError_t launch_attention_tc(const AttnParams &ap, const CUtensorMap &tmK, const CUtensorMap &tmV,
                                       cudaStream_t s, bool pdl)
{
    cudaError_t e = launch_attention_chunk_tc(ap, tmK, tmV, s, pdl);
    if (e != cudaSuccess)
        return e;
    return launch_attention_hybrid(ap, tmK, tmV, s, pdl, true);
}

// The epilogue parameters of stored output features [n1, N) of a product
// whose first n1 (a multiple of 256) are finished elsewhere.
static EpiParams epi_cols(const EpiParams &ep, int n1)
{
    EpiParams e = ep;
    e.N = ep.N - n1;
    if (e.mode == EPI_SWIGLU)
        e.act += n1 / 2;  // stored rows 2j, 2j + 1 make feature j
    return e;
}

static cudaError_t gemm(hb_ctx *ctx, const LayerMaps &M, int kind, const bf16 *X, const bf16 *W, int T, int N, int K,
                        const EpiParams &ep)
{
    if (ctx->gemm_impl == 0)
        return launch_gemm_simt(X, W, T, N, K, true, ep, ctx->stream);
    const int rows = launch_rows(T);
    // pair kernel on a product of more tile pairs than CTA pairs: one
    // data-parallel wave with the fused epilogue, the rest stream-K into
    // partials that a reduce pass finishes (gate/up only: its epilogue maps
    // stored rows to features by a plain offset, epi_cols); a product that
    // fits the CTA pairs runs data-parallel with the fused epilogue; else
    // every tile stream-K into partials and a reduce pass with the epilogue
    const int dp_tiles = ep.mode == EPI_SWIGLU ? tc_pair_dp_tiles(ctx->fast->rt, N, K) : 0;
    const bool dp = dp_tiles == 0 && tc_pair_data_parallel(ctx->fast->rt, N);
    int launches = 0;
    for (int t0 = 0; t0 < T; t0 += rows) {
        const int Tn = T - t0 < rows ? T - t0 : rows;
        const EpiParams er = epi_rows(ep, t0, Tn);
        cudaError_t e;
        if (dp_tiles > 0) {
            TcPartition part;
            const uint64_t fault = ctx->fast->fault_wait_ns;
            ctx->fast->fault_wait_ns = 0;
            e = launch_gemm_pair(M.m[kind], W, X + (size_t)t0 * K, Tn, N, K, er, ctx->fast->rt, ctx->stream, &part,
                                 true, dp_tiles, fault);
            if (e == cudaSuccess)
                e = launch_reduce_epi(part, epi_cols(er, dp_tiles * 2 * 128), ctx->stream, true);
            launches += 2;
        } else if (dp) {
            e = launch_tc(ctx, M, kind, W, X + (size_t)t0 * K, Tn, N, K, er);
            launches += 1;
        } else {
            EpiParams pp{};
            pp.mode = EPI_PARTIAL;
            pp.T = Tn;
            pp.N = N;
            pp.err = ep.err;
            TcPartition part;
            e = launch_tc(ctx, M, kind, W, X + (size_t)t0 * K, Tn, N, K, pp, &part);
            if (e == cudaSuccess)
                e = launch_reduce_epi(part, er, ctx->stream, true);
            launches += 2;
        }
        if (e != cudaSuccess)
            return e;
    }
    ctx->n_launches += launches - 1;  // one is counted by the caller
    return cudaSuccess;
}

// out = resid + X W^T (+ norm_out = RMSNorm(out) * gamma).  gemm_impl 3:
// the split-K cluster kernel with the residual fused, then the norm pass;
// else (and where the split-K kernel does not fit) the tensor-core GEMM
// leaving stream-K partials, then the fused reduce + residual (+ norm).
static cudaError_t gemm_reduce(hb_ctx *ctx, const LayerMaps &M, int kind, const bf16 *X, const bf16 *W, int T, int N,
                               int K, const bf16 *resid, bf16 *out, const float *gamma, bf16 *norm_out, int *launches)
{
    const hb_model_config &c = ctx->cfg;
    const int rows = launch_rows(T);
    if (ctx->gemm_impl == 3) {
        // whether the split-K kernel runs depends on the weight shape only
        // (its first launch answers for all): a row's result does not depend
        // on the batch it rides in
        FastPath *f = ctx->fast;
        cudaError_t e = cudaSuccess;
        for (int t0 = 0; t0 < T && e == cudaSuccess; t0 += rows) {
            const int Tn = T - t0 < rows ? T - t0 : rows;
            e = launch_gemm_ksplit(M.m[kind], W, X + (size_t)t0 * K, Tn, N, K, resid + (size_t)t0 * N,
                                   out + (size_t)t0 * N, gamma ? f->ss : nullptr, c.max_tokens, ctx->err_word, f->rt,
                                   ctx->stream, true);
            if (e == cudaErrorNotSupported && t0 == 0)
                break;
            *launches += 1;
            if (e == cudaSuccess && gamma) {
                e = launch_norm_apply(out + (size_t)t0 * N, f->ss, N / 128, c.max_tokens, gamma, c.rms_eps,
                                      norm_out + (size_t)t0 * N, Tn, N, ctx->stream, true);
                *launches += 1;
            }
        }
        if (e != cudaErrorNotSupported)
            return e;
        cudaGetLastError();
    }
    for (int t0 = 0; t0 < T; t0 += rows) {
        const int Tn = T - t0 < rows ? T - t0 : rows;
        EpiParams pp{};
        pp.mode = EPI_PARTIAL;
        pp.T = Tn;
        pp.N = N;
        TcPartition part;
        cudaError_t e = launch_tc(ctx, M, kind, W, X + (size_t)t0 * K, Tn, N, K, pp, &part);
        if (e != cudaSuccess)
            return e;
        e = launch_reduce_norm(part, Tn, N, resid + (size_t)t0 * N, out + (size_t)t0 * N, gamma,
                               norm_out + (size_t)t0 * N, c.rms_eps, ctx->stream, true);
        if (e != cudaSuccess)
            return e;
        *launches += 2;
    }
    return cudaSuccess;
}

// One decoder layer.  On the tensor-core path the QKV GEMM applies RoPE and
// the KV append in its own epilogue; the gate/up GEMM applies SwiGLU to its
// data-parallel wave and leaves stream-K partials for the rest, which a
// reduce pass finishes with SwiGLU; the O-proj and down-proj GEMMs leave
// stream-K partials that one kernel per token row finishes with the
// residual add and the next RMSNorm.  With the pair kernel a LLaMA-13B layer
// is 10 kernels: [norm-1 for the first layer only], QKV GEMM, chunk and
// decode attention, O GEMM, reduce + residual + norm-2, gate/up GEMM, its
// reduce, down GEMM, reduce + residual (+ norm-1 of the next layer).
int run_layer(hb_ctx *ctx, int l, int l_first, int l_last, const BatchDev &b, const bf16 *x, bf16 *y)
{
    const hb_model_config &c = ctx->cfg;
    const LayerDev &L = ctx->layers[l];
    const LayerMaps &M = ctx->fast->maps[l];
    const int T = b.T, H = c.hidden, d = c.head_dim;
    cudaStream_t s = ctx->stream;
    const bool tc = ctx->gemm_impl >= 2;

    // on the tensor-core path norm-1 of every layer but the first was
    // produced by the previous layer's final reduce
    // the step's first kernel also copies the batch plan to the device
    if (!tc || l == l_first) {
        const bool first = l == l_first;
        LK(K_RMSNORM, launch_rmsnorm(x, L.g1, ctx->xn, T, H, c.rms_eps, s, tc,
                                     first ? ctx->meta_src : nullptr, first ? ctx->d_meta : nullptr,
                                     first ? ctx->meta_n16 : 0));
    }

    EpiParams ep{};
    ep.mode = EPI_QKV;
    ep.T = T;
    ep.N = ctx->n_qkv;
    ep.pos = b.pos;
    ep.slot = b.slot;
    ep.rope = ctx->rope;
    ep.head_dim = d;
    ep.n_heads = c.n_heads;
    ep.n_kv = c.n_kv_heads;
    ep.q_out = ctx->q;
    ep.k_pool = L.k_pool;
    ep.v_pool = L.v_pool;
    ep.num_blocks = c.num_blocks;
    ep.err = ctx->err_word;
    LK(K_GEMM_QKV, gemm(ctx, M, W_QKV, ctx->xn, L.w_qkv, T, ctx->n_qkv, H, ep));

    if (ctx->attn_impl >= 1) {
        const FastPath *f = ctx->fast;
        AttnParams ap;
        ap.b = b;
        ap.q = ctx->q;
        ap.k_pool = L.k_pool;
        ap.v_pool = L.v_pool;
        ap.out = ctx->attn_o;
        ap.n_heads = c.n_heads;
        ap.n_kv = c.n_kv_heads;
        ap.head_dim = d;
        ap.items = f->d_items;
        ap.n_items = f->n_items;
        ap.n_chunk_items = f->n_chunk_items;
        ap.part_off = f->d_part_off;
        ap.part = f->attn_part;
        ap.counters = f->attn_counters;
        ap.err = ctx->err_word;
        const bool pdl = tc;
        if (ctx->attn_impl == 2)
            LK(K_ATTENTION, launch_attention_tc(ap, f->kv_maps[2 * l], f->kv_maps[2 * l + 1], s, pdl));
        else
            LK(K_ATTENTION, launch_attention_hybrid(ap, f->kv_maps[2 * l], f->kv_maps[2 * l + 1], s, pdl));
        // LK counted one: the chunk tiles and the decode splits are separate kernels
        if (f->n_chunk_items > 0 && f->n_items > f->n_chunk_items)
            ctx->n_launches++;
    } else {
        LK(K_ATTENTION,
           launch_attention_simple(ctx->q, L.k_pool, L.v_pool, b, c.n_heads, c.n_kv_heads, d, ctx->attn_o, s));
    }

    EpiParams eg{};
    eg.mode = EPI_SWIGLU;
    eg.T = T;
    eg.N = ctx->n_gu;
    eg.act = ctx->act;
    eg.ffn = c.ffn;

    if (tc) {
        // launch counting: LK counts one launch per call; gemm_reduce reports its own
        int extra = 0;
        LK(K_GEMM_O, gemm_reduce(ctx, M, W_O, ctx->attn_o, L.w_o, T, H, c.n_heads * d, x, ctx->h, L.g2, ctx->xn,
                                 &extra));
        LK(K_GEMM_GATE_UP, gemm(ctx, M, W_GU, ctx->xn, L.w_gu, T, ctx->n_gu, H, eg));
        const float *g_next = (l + 1 < l_last) ? ctx->layers[l + 1].g1 : nullptr;
        LK(K_GEMM_DOWN, gemm_reduce(ctx, M, W_D, ctx->act, L.w_d, T, H, c.ffn, ctx->h, y, g_next, ctx->xn, &extra));
        ctx->n_launches += extra - 2;
        return HB_OK;
    }

    EpiParams eo{};
    eo.mode = EPI_RESID;
    eo.T = T;
    eo.N = H;
    eo.resid = x;
    eo.out = ctx->h;
    LK(K_GEMM_O, gemm(ctx, M, W_O, ctx->attn_o, L.w_o, T, H, c.n_heads * d, eo));

    LK(K_RMSNORM, launch_rmsnorm(ctx->h, L.g2, ctx->xn, T, H, c.rms_eps, s));

    LK(K_GEMM_GATE_UP, gemm(ctx, M, W_GU, ctx->xn, L.w_gu, T, ctx->n_gu, H, eg));

    EpiParams ed{};
    ed.mode = EPI_RESID;
    ed.T = T;
    ed.N = H;
    ed.resid = ctx->h;
    ed.out = y;
    LK(K_GEMM_DOWN, gemm(ctx, M, W_D, ctx->act, L.w_d, T, H, c.ffn, ed));
    return HB_OK;
}

extern "C" int hb_gemm_test(hb_ctx *ctx, const void *X, const void *W, void *D, int T, int N, int K)
{
    if (!ctx)
        return HB_EINVAL;
    if (!X || !W || !D || T <= 0 || N <= 0 || K <= 0 || (K % 8) || (N % 2))
        return ctx->set_error(HB_EINVAL, "hb_gemm_test: bad arguments (K %% 8 == 0 and even N required)");
    EpiParams ep{};
    ep.mode = EPI_F32;
    ep.T = T;
    ep.N = N;
    ep.d32 = (float *)D;
    if (ctx->gemm_impl == 0) {
        LK(K_GEMM_TEST, launch_gemm_simt((const bf16 *)X, (const bf16 *)W, T, N, K, false, ep, ctx->stream));
        return HB_OK;
    }
    // tile the operand into a scratch copy, then run the tensor-core kernel
    FastPath *f = ctx->fast;
    const size_t need = tiled_weight_elems(N, K);
    if (need > f->test_w_elems) {
        cudaFree(f->test_w);
        f->test_w = nullptr;
        f->test_w_elems = 0;
        if (cudaMalloc((void **)&f->test_w, need * sizeof(bf16)) != cudaSuccess) {
            cudaGetLastError();
            return ctx->set_error(HB_ENOMEM, "hb_gemm_test scratch");
        }
        f->test_w_elems = need;
    }
    CUtensorMap tm;
    if (!make_tmap_tiled_weights(&tm, f->test_w, N, K, 128))
        return ctx->set_error(HB_ECUDA, "cuTensorMapEncodeTiled failed");
    ctx->n_launches++;
    if (launch_tile_weights((const bf16 *)W, f->test_w, N, K, 0, 0, ctx->stream) != cudaSuccess)
        return ctx->set_error(HB_ECUDA, "tile launch failed");
    for (int t0 = 0; t0 < T; t0 += TC_PAIR_MAX_ROWS) {
        const int Tn = T - t0 < TC_PAIR_MAX_ROWS ? T - t0 : TC_PAIR_MAX_ROWS;
        EpiParams pp{};
        pp.mode = EPI_PARTIAL;
        pp.T = Tn;
        pp.N = N;
        TcPartition part;
        LK(K_GEMM_TEST, launch_gemm_pair(tm, f->test_w, (const bf16 *)X + (size_t)t0 * K, Tn, N, K, pp, f->rt,
                                         ctx->stream, &part));
        LK(K_GEMM_TEST, launch_reduce_epi(part, epi_rows(ep, t0, Tn), ctx->stream));
    }
    return HB_OK;
}

extern "C" int hb_set_kernels(hb_ctx *ctx, int gemm_impl, int attn_impl)
{
    if (!ctx)
        return HB_EINVAL;
    if ((gemm_impl != 0 && gemm_impl != 2 && gemm_impl != 3) || attn_impl < 0 || attn_impl > 2)
        return ctx->set_error(HB_EINVAL, "hb_set_kernels: gemm_impl must be 0, 2 or 3, attn_impl 0, 1 or 2");
    ctx->gemm_impl = gemm_impl;
    ctx->attn_impl = attn_impl;
    return HB_OK;
}

extern "C" int hb_test_wait_timeout(hb_ctx *ctx, long long wait_ns)
{
    if (!ctx)
        return HB_EINVAL;
    if (wait_ns < 100000 || wait_ns > 2000000000ll)
        return ctx->set_error(HB_EINVAL, "hb_test_wait_timeout: wait_ns must lie in [1e5, 2e9]");
    if (ctx->gemm_impl < 2)
        return ctx->set_error(HB_EINVAL, "hb_test_wait_timeout: needs the tensor-core GEMM (gemm_impl 2 or 3)");
    ctx->fast->fault_wait_ns = (uint64_t)wait_ns;
    return HB_OK;
}
