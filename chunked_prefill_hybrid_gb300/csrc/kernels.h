// kernels.h -- host-side launchers of the library's CUDA kernels.
#pragma once

#include "common.cuh"

namespace hb {

// RMSNorm: y[t][i] = bf16(x[t][i] * rsqrt(mean_i x[t][i]^2 + eps) * gamma[i]).
// meta_src / meta_dst / meta_n16: when set, the kernel also copies meta_n16
// 16-byte words from meta_src (the batch plan in mapped, page-locked host
// memory) to meta_dst, after its wait for the previous kernel, so that the
// kernels after it find the plan in device memory.
cudaError_t launch_rmsnorm(const bf16 *x, const float *gamma, bf16 *y, int T, int H, float eps,
                           cudaStream_t s, bool pdl = false, const int *meta_src = nullptr, int *meta_dst = nullptr,
                           int meta_n16 = 0);

// Reference SIMT GEMM: acc[t][n] = sum_k X[t][k] W[n][k], then the epilogue.
// tiled: W is in the tensor-core layout [n/128][k/64][128][64], else [N][K].
cudaError_t launch_gemm_simt(const bf16 *X, const bf16 *W, int T, int N, int K, bool tiled, const EpiParams &ep,
                             cudaStream_t s);

// Straightforward attention: one CTA per (row, head), online softmax.
cudaError_t launch_attention_simple(const bf16 *q, const bf16 *k_pool, const bf16 *v_pool, const BatchDev &b,
                                    int n_heads, int n_kv, int head_dim, bf16 *out, cudaStream_t s);

// Scatter / gather of K,V tokens between dense [n][n_kv][d] and the paged pool.
cudaError_t launch_kv_write(bf16 *k_pool, bf16 *v_pool, const bf16 *k, const bf16 *v, const int *bt, int start_pos,
                            int n_tokens, int n_kv, int head_dim, int num_blocks, int *err, cudaStream_t s);
cudaError_t launch_kv_read(const bf16 *k_pool, const bf16 *v_pool, bf16 *k, bf16 *v, const int *bt, int start_pos,
                           int n_tokens, int n_kv, int head_dim, int num_blocks, int *err, cudaStream_t s);
cudaError_t launch_fill_u16(uint16_t *p, size_t n, uint16_t bits, cudaStream_t s);

cudaError_t launch_bf16_to_f32(const bf16 *src, float *dst, int n, cudaStream_t s);

}  // namespace hb
