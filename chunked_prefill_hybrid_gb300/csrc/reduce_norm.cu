// reduce_norm.cu -- finishes the split-K linear ops whose partial tiles the
// tensor-core GEMM left in its workspace (O-proj and down-proj), fused with
// the residual add and the next RMSNorm:
//   out[t]  = bf16(resid[t] + sum of the partial tiles, in CTA order)
//   norm[t] = bf16(out[t] * rsqrt(mean(out[t]^2) + eps) * gamma)   (optional)
// One CTA per token row; each thread owns groups of 8 consecutive features
// (16-byte bf16 vectors, 32-byte fp32 partial reads).
#include "gemm_tc.h"
#include "kernels.h"

namespace hb {

namespace {

constexpr int RN_THREADS = 256;
constexpr int RN_MAX_GROUPS = 4;  // hidden <= 256 * 8 * 4 = 8192

struct RnArgs {
    TcPartition part;
    int T, N;
    const bf16 *resid;
    bf16 *out;
    const float *gamma;  // null: no norm
    bf16 *norm_out;
    float eps;
};

__device__ __forceinline__ int owner(long long u, const TcPartition &p)
{
    return (int)((u * p.grid + p.grid - 1) / p.units);
}
__device__ __forceinline__ int ubegin(int c, const TcPartition &p) { return (int)((long long)c * p.units / p.grid); }

__global__ void __launch_bounds__(RN_THREADS) k_reduce_norm(RnArgs a)
{
    const int t = blockIdx.x;
    const TcPartition &p = a.part;
    float h[RN_MAX_GROUPS][8];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < RN_MAX_GROUPS; ++i) {
        const int n0 = (threadIdx.x + i * RN_THREADS) * 8;
        if (n0 >= a.N)
            break;
        int mt, r, col;
        tc_part_loc(p, t, n0 >> 7, mt, r, col);
        const long long u0 = (long long)mt * p.nkb;
        const int c_lo = owner(u0, p), c_hi = owner(u0 + p.nkb - 1, p);
        float acc[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            acc[k] = 0.f;
        for (int c = c_lo; c <= c_hi; ++c) {
            const int slot = mt - ubegin(c, p) / p.nkb;
            const float4 *src = reinterpret_cast<const float4 *>(
                p.ws + ((((size_t)c * p.G + r) * p.slots + slot) * p.tg + col) * 128 + (n0 & 127));
            const float4 x0 = __ldcg(src), x1 = __ldcg(src + 1);
            acc[0] += x0.x;
            acc[1] += x0.y;
            acc[2] += x0.z;
            acc[3] += x0.w;
            acc[4] += x1.x;
            acc[5] += x1.y;
            acc[6] += x1.z;
            acc[7] += x1.w;
        }
        const uint4 rv = *reinterpret_cast<const uint4 *>(a.resid + (size_t)t * a.N + n0);
        const bf16 *re = reinterpret_cast<const bf16 *>(&rv);
        float o[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            o[k] = bf2f(f2bf(bf2f(re[k]) + acc[k]));  // the stored bf16 value
            h[i][k] = o[k];
            ss += o[k] * o[k];
        }
        *reinterpret_cast<uint4 *>(a.out + (size_t)t * a.N + n0) = pack8_bf16(o);
    }
    if (!a.gamma)
        return;
    __shared__ float red[RN_THREADS / 32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < RN_THREADS / 32; ++w)
        tot += red[w];
    const float rs = rsqrtf(tot / (float)a.N + a.eps);
#pragma unroll
    for (int i = 0; i < RN_MAX_GROUPS; ++i) {
        const int n0 = (threadIdx.x + i * RN_THREADS) * 8;
        if (n0 >= a.N)
            break;
        float o[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            o[k] = h[i][k] * rs * a.gamma[n0 + k];
        *reinterpret_cast<uint4 *>(a.norm_out + (size_t)t * a.N + n0) = pack8_bf16(o);
    }
}

// Generic finish: every 16-feature group of row t is the sum of its
// contributors' partials, handed to the fused epilogue (RoPE + KV append
// for the QKV projection, SwiGLU for gate/up).
__global__ void __launch_bounds__(128) k_reduce_epi(TcPartition p, EpiParams ep)
{
    const int t = blockIdx.x;
    {
        const int n0 = (blockIdx.y * 128 + threadIdx.x) * 16;
        if (n0 >= ep.N)
            return;
        int mt, r, col;
        tc_part_loc(p, t, n0 >> 7, mt, r, col);
        const long long u0 = (long long)mt * p.nkb;
        const int c_lo = owner(u0, p), c_hi = owner(u0 + p.nkb - 1, p);
        float v[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
            v[k] = 0.f;
        for (int c = c_lo; c <= c_hi; ++c) {
            const int slot = mt - ubegin(c, p) / p.nkb;
            const float4 *src = reinterpret_cast<const float4 *>(
                p.ws + ((((size_t)c * p.G + r) * p.slots + slot) * p.tg + col) * 128 + (n0 & 127));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 f = __ldcg(src + e);
                v[4 * e] += f.x;
                v[4 * e + 1] += f.y;
                v[4 * e + 2] += f.z;
                v[4 * e + 3] += f.w;
            }
        }
        epi_group(ep, t, n0, v);
    }
}

}  // namespace

cudaError_t launch_reduce_epi(const TcPartition &part, const EpiParams &ep, cudaStream_t s)
{
    if (ep.T <= 0)
        return cudaSuccess;
    if (ep.N % 16 != 0 && ep.mode != EPI_F32)  // fp32 output has a scalar tail
        return cudaErrorInvalidValue;
    dim3 grid(ep.T, ((ep.N + 15) / 16 + 127) / 128);
    k_reduce_epi<<<grid, 128, 0, s>>>(part, ep);
    return cudaGetLastError();
}

cudaError_t launch_reduce_norm(const TcPartition &part, int T, int N, const bf16 *resid, bf16 *out, const float *gamma,
                               bf16 *norm_out, float eps, cudaStream_t s)
{
    if (T <= 0)
        return cudaSuccess;
    if (N % 8 != 0 || N > RN_THREADS * 8 * RN_MAX_GROUPS)
        return cudaErrorInvalidValue;
    RnArgs a{part, T, N, resid, out, gamma, norm_out, eps};
    k_reduce_norm<<<T, RN_THREADS, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace hb
