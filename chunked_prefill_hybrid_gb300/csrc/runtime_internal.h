// runtime_internal.h -- the context object behind hb_ctx and the pieces of
// the runtime shared between runtime.cu (ABI, validation, metadata) and
// layer.cu (per-layer launch sequence and kernel selection).
#pragma once

#include <cuda_runtime.h>

#include <string>
#include <utility>
#include <vector>

#include "hb.h"
#include "common.cuh"

namespace hb {

struct LayerDev {
    // weights in the tensor-core tiled layout [N/128][K/64][128][64]
    bf16 *w_qkv = nullptr;  // N = n_qkv, rows permuted within heads (RoPE pairs adjacent)
    bf16 *w_o = nullptr;    // N = H, K = n_heads d
    bf16 *w_gu = nullptr;   // N = 2 ffn, gate/up rows interleaved
    bf16 *w_d = nullptr;    // N = H, K = ffn
    float *g1 = nullptr, *g2 = nullptr;
    bf16 *k_pool = nullptr, *v_pool = nullptr;  // [num_blocks][n_kv][16][d]
    bool loaded = false;
};

// Host-side plan of one batch (rows: chunk first, then decodes).
struct Plan {
    int T = 0, n_seq = 0, chunk_len = 0;
    std::vector<int> pos, slot, row_seq;
    std::vector<int> seq_q0, seq_nq, seq_pos0, seq_bt, bt;
};

// Kernel kinds for per-launch timing.
enum Kind : int {
    K_RMSNORM = 0,
    K_GEMM_QKV,
    K_ATTENTION,
    K_ATTN_COMBINE,
    K_GEMM_O,
    K_GEMM_GATE_UP,
    K_GEMM_DOWN,
    K_KVIO,
    K_GEMM_TEST,
    K_REDUCE_NORM,
    K_REDUCE_QKV,
    K_REDUCE_SWIGLU,
    K_NUM_KINDS
};
static const char *const kKindNames[K_NUM_KINDS] = {"rmsnorm",   "gemm_qkv",  "attention", "attn_combine",
                                                     "gemm_o",    "gemm_gate_up", "gemm_down", "kv_io",
                                                     "gemm_test", "reduce_norm", "reduce_qkv", "reduce_swiglu"};

constexpr int kMetaRing = 4;

struct FastPath;  // tensor-core GEMM and hybrid attention state (layer.cu)

int validate_config(const hb_model_config &c, std::string *err);
int plan_batch(const hb_model_config &c, const hb_batch_spec *s, Plan &p, std::string *err);
size_t kMetaExtraWords(const hb_model_config &c);

}  // namespace hb

struct hb_ctx {
    hb_model_config cfg{};
    cudaStream_t stream = nullptr;
    int device = 0, num_sms = 0, cc_major = 0, cc_minor = 0;
    int n_qkv = 0, n_qkv_pad = 0, n_gu = 0, n_gu_pad = 0;

    std::vector<void *> allocations;
    std::vector<hb::LayerDev> layers;
    hb::bf16 *kv = nullptr;
    size_t kv_elems_per_pool = 0;
    float2 *rope = nullptr;
    hb::bf16 *xn = nullptr, *q = nullptr, *attn_o = nullptr, *h = nullptr, *act = nullptr;
    hb::bf16 *xa = nullptr, *xb = nullptr, *host_in = nullptr, *host_out = nullptr;
    // hb_forward_host_async: a ring of two device input buffers filled on
    // copy_stream (in_ready[k] behind the copy, in_free[k] behind the step
    // that read slot k) and a ring of two device output buffers, slot k
    // copied to the caller's buffer on out_stream once its step is done
    // (out_free[k] behind that copy); made on the first asynchronous call
    hb::bf16 *async_in[2] = {nullptr, nullptr};
    hb::bf16 *async_out[2] = {nullptr, nullptr};
    cudaStream_t copy_stream = nullptr, out_stream = nullptr;
    cudaEvent_t in_ready[2] = {nullptr, nullptr}, in_free[2] = {nullptr, nullptr};
    cudaEvent_t out_free[2] = {nullptr, nullptr};
    bool in_used[2] = {false, false};
    int in_i = 1;
    int *err_word = nullptr;
    int *h_err = nullptr;  // pinned: the error word read back with the stream's work

    // batch metadata: a ring of mapped, page-locked staging buffers + one
    // device buffer.  A forward step's plan is copied from its staging
    // buffer to d_meta by the step's first kernel (meta_src, meta_n16 until
    // that launch); the KV hooks copy theirs with cudaMemcpyAsync.
    int *d_meta = nullptr;
    size_t meta_cap = 0;  // words, a multiple of 4
    int *h_meta[hb::kMetaRing] = {nullptr};
    int *h_meta_dev[hb::kMetaRing] = {nullptr};  // the same buffers as the GPU addresses them
    const int *meta_src = nullptr;
    int meta_n16 = 0;
    cudaEvent_t meta_ev[hb::kMetaRing] = {nullptr};
    bool meta_used[hb::kMetaRing] = {false};
    int meta_i = 0;
    int *next_meta_host();

    hb::Plan plan;
    hb::FastPath *fast = nullptr;
    int gemm_impl = 2;  // 0: SIMT reference, 2: tcgen05 CTA pairs (2-SM MMA), 3: 2 + split-K clusters for O, down
    int attn_impl = 1;  // 0: simple, 1: paged attention (mma.sync chunk tiles), 2: tcgen05 chunk tiles

    // profiling and launch accounting
    long long n_launches = 0;
    bool prof_on = false;
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> prof_events;
    std::vector<int> prof_kinds;
    size_t prof_used = 0;
    void prof_launch_begin(int kind);
    void prof_launch_end();

    std::string last_error;
    int set_error(int code, const char *fmt, ...);
};

// layer.cu
int hb_init_fast_path(hb_ctx *ctx);
void hb_free_fast_path(hb_ctx *ctx);
int hb_plan_fast_path(hb_ctx *ctx, const hb::Plan &p, int *hm, size_t &at, hb::BatchDev &b);
int run_layer(hb_ctx *ctx, int l, int l_first, int l_last, const hb::BatchDev &b, const hb::bf16 *x, hb::bf16 *y);
