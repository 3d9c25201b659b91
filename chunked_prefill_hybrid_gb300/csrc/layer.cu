// layer.cu -- the per-layer launch sequence and kernel selection.
#include <cuda_runtime.h>

#include <vector>

#include "gemm_tc.h"
#include "kernels.h"
#include "runtime_internal.h"

using namespace hb;

namespace hb {

struct LayerMaps {
    CUtensorMap qkv, o, gu, d;
};

struct FastPath {
    int max_smem = 0;
    std::vector<LayerMaps> maps;
};

size_t kMetaExtraWords(const hb_model_config &c)
{
    (void)c;
    return 0;
}

}  // namespace hb

int hb_init_fast_path(hb_ctx *ctx)
{
    FastPath *f = new FastPath();
    ctx->fast = f;
    if (cudaDeviceGetAttribute(&f->max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, ctx->device) != cudaSuccess)
        return ctx->set_error(HB_ECUDA, "cudaDeviceGetAttribute failed");
    const hb_model_config &c = ctx->cfg;
    const int H = c.hidden, qd = c.n_heads * c.head_dim;
    f->maps.resize(c.n_layers);
    for (int l = 0; l < c.n_layers; ++l) {
        const LayerDev &L = ctx->layers[l];
        LayerMaps &m = f->maps[l];
        if (!make_tmap_kmajor(&m.qkv, L.w_qkv, ctx->n_qkv_pad, H, 128) ||
            !make_tmap_kmajor(&m.o, L.w_o, H, qd, 128) || !make_tmap_kmajor(&m.gu, L.w_gu, ctx->n_gu_pad, H, 128) ||
            !make_tmap_kmajor(&m.d, L.w_d, H, c.ffn, 128))
            return ctx->set_error(HB_ECUDA, "cuTensorMapEncodeTiled failed (driver entry point unavailable?)");
    }
    ctx->gemm_impl = 1;
    ctx->attn_impl = 0;
    return HB_OK;
}

void hb_free_fast_path(hb_ctx *ctx)
{
    delete ctx->fast;
    ctx->fast = nullptr;
}

int hb_plan_fast_path(hb_ctx *ctx, const Plan &p, int *hm, size_t &at, BatchDev &b)
{
    (void)ctx;
    (void)p;
    (void)hm;
    (void)at;
    (void)b;
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

static cudaError_t gemm(hb_ctx *ctx, const CUtensorMap *tmW, const bf16 *X, const bf16 *W, int T, int N_pad, int N,
                        int K, const EpiParams &ep)
{
    if (ctx->gemm_impl == 1 && tmW)
        return launch_gemm_tc(*tmW, X, T, N_pad, N, K, ep, ctx->stream, ctx->fast->max_smem);
    return launch_gemm_simt(X, W, T, N, K, ep, ctx->stream);
}

int run_layer(hb_ctx *ctx, int l, const BatchDev &b, const bf16 *x, bf16 *y)
{
    const hb_model_config &c = ctx->cfg;
    const LayerDev &L = ctx->layers[l];
    const LayerMaps &M = ctx->fast->maps[l];
    const int T = b.T, H = c.hidden, d = c.head_dim;
    cudaStream_t s = ctx->stream;

    LK(K_RMSNORM, launch_rmsnorm(x, L.g1, ctx->xn, T, H, c.rms_eps, s));

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
    LK(K_GEMM_QKV, gemm(ctx, &M.qkv, ctx->xn, L.w_qkv, T, ctx->n_qkv_pad, ctx->n_qkv, H, ep));

    LK(K_ATTENTION, launch_attention_simple(ctx->q, L.k_pool, L.v_pool, b, c.n_heads, c.n_kv_heads, d, ctx->attn_o, s));

    EpiParams eo{};
    eo.mode = EPI_RESID;
    eo.T = T;
    eo.N = H;
    eo.resid = x;
    eo.out = ctx->h;
    LK(K_GEMM_O, gemm(ctx, &M.o, ctx->attn_o, L.w_o, T, H, H, c.n_heads * d, eo));

    LK(K_RMSNORM, launch_rmsnorm(ctx->h, L.g2, ctx->xn, T, H, c.rms_eps, s));

    EpiParams eg{};
    eg.mode = EPI_SWIGLU;
    eg.T = T;
    eg.N = ctx->n_gu;
    eg.act = ctx->act;
    eg.ffn = c.ffn;
    LK(K_GEMM_GATE_UP, gemm(ctx, &M.gu, ctx->xn, L.w_gu, T, ctx->n_gu_pad, ctx->n_gu, H, eg));

    EpiParams ed{};
    ed.mode = EPI_RESID;
    ed.T = T;
    ed.N = H;
    ed.resid = ctx->h;
    ed.out = y;
    LK(K_GEMM_DOWN, gemm(ctx, &M.d, ctx->act, L.w_d, T, H, H, c.ffn, ed));
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
    CUtensorMap tm;
    const bool have_map = ctx->gemm_impl == 1 && make_tmap_kmajor(&tm, W, N, K, 128);
    if (ctx->gemm_impl == 1 && !have_map)
        return ctx->set_error(HB_ECUDA, "cuTensorMapEncodeTiled failed");
    LK(K_GEMM_TEST, gemm(ctx, have_map ? &tm : nullptr, (const bf16 *)X, (const bf16 *)W, T, (N + 127) / 128 * 128, N,
                         K, ep));
    return HB_OK;
}

extern "C" int hb_set_kernels(hb_ctx *ctx, int gemm_impl, int attn_impl)
{
    if (!ctx)
        return HB_EINVAL;
    if (gemm_impl < 0 || gemm_impl > 1 || attn_impl < 0 || attn_impl > 1)
        return ctx->set_error(HB_EINVAL, "hb_set_kernels: gemm_impl and attn_impl must be 0 or 1");
    ctx->gemm_impl = gemm_impl;
    ctx->attn_impl = attn_impl;
    return HB_OK;
}
