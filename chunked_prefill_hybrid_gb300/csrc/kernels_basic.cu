// kernels_basic.cu -- RMSNorm, reference SIMT GEMM, straightforward attention,
// KV scatter/gather and weight repacking.
//
// The SIMT GEMM and the simple attention are the bring-up path: plainly
// correct, used by the kernel-selection switch and as a cross-check of the
// tensor-core kernels; the forward's fast path lives in gemm_tc.cu and
// attention_hybrid.cu.
#include "kernels.h"

namespace hb {

// ---------------------------------------------------------------- RMSNorm

template <int THREADS>
__global__ void __launch_bounds__(THREADS) k_rmsnorm(const bf16 *__restrict__ x, const float *__restrict__ gamma,
                                                     bf16 *__restrict__ y, int H, float eps,
                                                     const uint4 *__restrict__ meta_src, uint4 *__restrict__ meta_dst,
                                                     int meta_n16)
{
    pdl_trigger();
    pdl_wait();
    // every earlier kernel has finished: the plan's device copy is free to overwrite
    for (int i = blockIdx.x * THREADS + threadIdx.x; i < meta_n16; i += gridDim.x * THREADS)
        meta_dst[i] = meta_src[i];
    const int t = blockIdx.x;
    const bf16 *xr = x + (size_t)t * H;
    bf16 *yr = y + (size_t)t * H;
    float ss = 0.f;
    // H % 8 == 0: 16-byte vectors
    const uint4 *xv = reinterpret_cast<const uint4 *>(xr);
    for (int i = threadIdx.x; i < H / 8; i += THREADS) {
        uint4 u = xv[i];
        const bf16 *e = reinterpret_cast<const bf16 *>(&u);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float f = bf2f(e[j]);
            ss += f * f;
        }
    }
    __shared__ float red[THREADS / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < THREADS / 32; ++w)
        tot += red[w];
    const float r = rsqrtf(tot / (float)H + eps);
    uint4 *yv = reinterpret_cast<uint4 *>(yr);
    for (int i = threadIdx.x; i < H / 8; i += THREADS) {
        uint4 u = xv[i];
        const bf16 *e = reinterpret_cast<const bf16 *>(&u);
        uint4 o;
        bf16 *oe = reinterpret_cast<bf16 *>(&o);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            oe[j] = f2bf(bf2f(e[j]) * r * gamma[i * 8 + j]);
        yv[i] = o;
    }
}

cudaError_t launch_rmsnorm(const bf16 *x, const float *gamma, bf16 *y, int T, int H, float eps, cudaStream_t s,
                           bool pdl, const int *meta_src, int *meta_dst, int meta_n16)
{
    if (T <= 0)
        return cudaSuccess;
    if (meta_n16 > 0 && (!meta_src || !meta_dst || ((uintptr_t)meta_src | (uintptr_t)meta_dst) % 16 != 0))
        return cudaErrorInvalidValue;
    cudaError_t e = launch_kernel(pdl, k_rmsnorm<256>, dim3(T), dim3(256), 0, s, x, gamma, y, H, eps,
                                  (const uint4 *)meta_src, (uint4 *)meta_dst, meta_n16);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// ------------------------------------------------------- reference GEMM

constexpr int SG_BT = 64, SG_BN = 64, SG_BK = 32;

// W element (n, k): row-major [N][K], or the tensor-core tiled layout
// [n / 128][k / 64][n % 128][k % 64].
__device__ __forceinline__ size_t w_index(int n, int k, int K, bool tiled)
{
    if (!tiled)
        return (size_t)n * K + k;
    const int nkb = (K + 63) / 64;
    return (((size_t)(n >> 7) * nkb + (k >> 6)) * 128 + (n & 127)) * 64 + (k & 63);
}

__global__ void __launch_bounds__(256) k_gemm_simt(const bf16 *__restrict__ X, const bf16 *__restrict__ W, int T,
                                                   int N, int K, bool tiled, EpiParams ep)
{
    __shared__ float Xs[SG_BK][SG_BT + 4];
    __shared__ float Ws[SG_BK][SG_BN + 4];
    const int t0 = blockIdx.y * SG_BT, n0 = blockIdx.x * SG_BN;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            acc[i][j] = 0.f;
    for (int k0 = 0; k0 < K; k0 += SG_BK) {
        for (int e = tid; e < SG_BT * SG_BK; e += 256) {
            const int r = e / SG_BK, c = e % SG_BK, t = t0 + r, k = k0 + c;
            Xs[c][r] = (t < T && k < K) ? bf2f(X[(size_t)t * K + k]) : 0.f;
        }
        for (int e = tid; e < SG_BN * SG_BK; e += 256) {
            const int r = e / SG_BK, c = e % SG_BK, n = n0 + r, k = k0 + c;
            Ws[c][r] = (n < N && k < K) ? bf2f(W[w_index(n, k, K, tiled)]) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < SG_BK; ++kk) {
            float xa[4], wb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xa[i] = Xs[kk][ty * 4 + i];
                wb[i] = Ws[kk][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    acc[i][j] = fmaf(xa[i], wb[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + ty * 4 + i;
        if (t >= T)
            continue;
#pragma unroll
        for (int j = 0; j < 4; j += 2) {
            const int n = n0 + tx * 4 + j;
            if (n < N)
                epi_pair(ep, t, n, acc[i][j], acc[i][j + 1]);
        }
    }
}

cudaError_t launch_gemm_simt(const bf16 *X, const bf16 *W, int T, int N, int K, bool tiled, const EpiParams &ep,
                             cudaStream_t s)
{
    if (T <= 0)
        return cudaSuccess;
    dim3 grid((N + SG_BN - 1) / SG_BN, (T + SG_BT - 1) / SG_BT);
    k_gemm_simt<<<grid, 256, 0, s>>>(X, W, T, N, K, tiled, ep);
    return cudaGetLastError();
}

// ------------------------------------------------------ simple attention

// One CTA of 4 warps per (row, head).  Each lane holds d/32 dims of q and of
// the running output; warps stride over the keys 0..pos and keep their own
// online-softmax state, merged at the end.
template <int D>
__global__ void __launch_bounds__(128) k_attention_simple(const bf16 *__restrict__ q, const bf16 *__restrict__ kp,
                                                          const bf16 *__restrict__ vp, BatchDev b, int n_heads,
                                                          int n_kv, bf16 *__restrict__ out)
{
    constexpr int E = D / 32;
    const int r = blockIdx.x, h = blockIdx.y;
    const int kvh = h / (n_heads / n_kv);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int seq = b.row_seq[r];
    const int pos = b.pos[r];
    const int *bt = b.bt + b.seq_bt[seq];
    const float scale = rsqrtf((float)D);
    float qv[E], acc[E];
    const bf16 *qr = q + ((size_t)r * n_heads + h) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        qv[e] = bf2f(qr[e]) * scale;
        acc[e] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    for (int t = warp; t <= pos; t += 4) {
        const int blk = bt[t >> 4];
        const size_t base = (((size_t)blk * n_kv + kvh) * 16 + (t & 15)) * D + lane * E;
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e)
            dot += qv[e] * bf2f(kp[base + e]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            dot += __shfl_xor_sync(0xffffffffu, dot, o);
        const float mn = fmaxf(m, dot);
        const float corr = __expf(m - mn);
        const float p = __expf(dot - mn);
        l = l * corr + p;
#pragma unroll
        for (int e = 0; e < E; ++e)
            acc[e] = acc[e] * corr + p * bf2f(vp[base + e]);
        m = mn;
    }
    __shared__ float sm[4], sl[4];
    __shared__ float so[4][D];
    if (lane == 0) {
        sm[warp] = m;
        sl[warp] = l;
    }
#pragma unroll
    for (int e = 0; e < E; ++e)
        so[warp][lane * E + e] = acc[e];
    __syncthreads();
    if (warp == 0) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w)
            M = fmaxf(M, sm[w]);
        float L = 0.f, f[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            f[w] = (sl[w] > 0.f) ? __expf(sm[w] - M) : 0.f;
            L += sl[w] * f[w];
        }
        bf16 *orow = out + ((size_t)r * n_heads + h) * D + lane * E;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            float o = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w)
                o += so[w][lane * E + e] * f[w];
            orow[e] = f2bf(o / L);
        }
    }
}

cudaError_t launch_attention_simple(const bf16 *q, const bf16 *k_pool, const bf16 *v_pool, const BatchDev &b,
                                    int n_heads, int n_kv, int head_dim, bf16 *out, cudaStream_t s)
{
    if (b.T <= 0)
        return cudaSuccess;
    dim3 grid(b.T, n_heads);
    if (head_dim == 128)
        k_attention_simple<128><<<grid, 128, 0, s>>>(q, k_pool, v_pool, b, n_heads, n_kv, out);
    else if (head_dim == 64)
        k_attention_simple<64><<<grid, 128, 0, s>>>(q, k_pool, v_pool, b, n_heads, n_kv, out);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

// ------------------------------------------------------ KV scatter/gather

template <bool WRITE>
__global__ void k_kv_copy(bf16 *kp, bf16 *vp, bf16 *k, bf16 *v, const int *__restrict__ bt, int start_pos, int n_kv,
                          int d, int num_blocks, int *err)
{
    const int i = blockIdx.x;  // token
    const int pos = start_pos + i;
    const int blk = bt[pos >> 4];
    if (blk < 0 || blk >= num_blocks) {
        if (threadIdx.x == 0)
            set_dev_err(err, DERR_BAD_SLOT);
        return;
    }
    const int off = pos & 15;
    for (int e = threadIdx.x; e < n_kv * d; e += blockDim.x) {
        const int h = e / d, c = e % d;
        const size_t pidx = (((size_t)blk * n_kv + h) * 16 + off) * d + c;
        const size_t didx = (size_t)i * n_kv * d + e;
        if (WRITE) {
            kp[pidx] = k[didx];
            vp[pidx] = v[didx];
        } else {
            k[didx] = kp[pidx];
            v[didx] = vp[pidx];
        }
    }
}

cudaError_t launch_kv_write(bf16 *k_pool, bf16 *v_pool, const bf16 *k, const bf16 *v, const int *bt, int start_pos,
                            int n_tokens, int n_kv, int head_dim, int num_blocks, int *err, cudaStream_t s)
{
    if (n_tokens <= 0)
        return cudaSuccess;
    k_kv_copy<true><<<n_tokens, 256, 0, s>>>(k_pool, v_pool, const_cast<bf16 *>(k), const_cast<bf16 *>(v), bt,
                                              start_pos, n_kv, head_dim, num_blocks, err);
    return cudaGetLastError();
}

cudaError_t launch_kv_read(const bf16 *k_pool, const bf16 *v_pool, bf16 *k, bf16 *v, const int *bt, int start_pos,
                           int n_tokens, int n_kv, int head_dim, int num_blocks, int *err, cudaStream_t s)
{
    if (n_tokens <= 0)
        return cudaSuccess;
    k_kv_copy<false><<<n_tokens, 256, 0, s>>>(const_cast<bf16 *>(k_pool), const_cast<bf16 *>(v_pool), k, v, bt,
                                               start_pos, n_kv, head_dim, num_blocks, err);
    return cudaGetLastError();
}

__global__ void k_fill_u16(uint16_t *p, size_t n, uint16_t bits)
{
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        p[i] = bits;
}

cudaError_t launch_fill_u16(uint16_t *p, size_t n, uint16_t bits, cudaStream_t s)
{
    if (n == 0)
        return cudaSuccess;
    k_fill_u16<<<1024, 256, 0, s>>>(p, n, bits);
    return cudaGetLastError();
}

// ------------------------------------------------------------- conversion

__global__ void k_bf16_to_f32(const bf16 *src, float *dst, int n)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n)
        dst[i] = bf2f(src[i]);
}

cudaError_t launch_bf16_to_f32(const bf16 *src, float *dst, int n, cudaStream_t s)
{
    k_bf16_to_f32<<<(n + 255) / 256, 256, 0, s>>>(src, dst, n);
    return cudaGetLastError();
}

}  // namespace hb
