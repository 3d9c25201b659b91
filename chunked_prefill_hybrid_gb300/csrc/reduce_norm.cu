// reduce_norm.cu -- finishes the stream-K linear ops whose partial tiles the
// tensor-core GEMM left in its workspace.  k_reduce_norm (O-proj and
// down-proj) fuses the residual add and the next RMSNorm:
//   out[t]  = bf16(resid[t] + sum of the partial tiles, in CTA order)
//   norm[t] = bf16(out[t] * rsqrt(mean(out[t]^2) + eps) * gamma)   (optional)
// One CTA per token row; each thread owns groups of 8 consecutive features
// (16-byte bf16 vectors, 32-byte fp32 partial reads).
#include "gemm_tc.h"
#include "kernels.h"

namespace hb {

namespace {


struct RnArgs {
    TcPartition part;
    int T, N;
    const bf16 *resid;
    bf16 *out;
    const float *gamma;  // null: no norm
    bf16 *norm_out;
    float eps;
};

constexpr int RD_MAX_GRID = 160;   // CTAs (or CTA pairs) of one GEMM launch
constexpr int RD_MAX_UROWS = 512;  // weight tiles (or tile pairs) of one launch

// Per-CTA tables of a partition, so that the per-element loops need no
// division: first[c] = first unit row of contributor c; clo/chi[u] = the
// contributors of unit row u.
struct RdTab {
    int first[RD_MAX_GRID];
    short clo[RD_MAX_UROWS], chi[RD_MAX_UROWS];
};

// (32-bit arithmetic: the launcher checks units * grid < 2^31)
__device__ __forceinline__ void rd_build(const TcPartition &p, int n_urows, RdTab &tab)
{
    const unsigned g = (unsigned)p.grid, un = (unsigned)p.units, nkb = (unsigned)p.nkb;
    for (int c = threadIdx.x; c < p.grid; c += blockDim.x)
        tab.first[c] = (int)((unsigned)c * un / g / nkb);
    for (int u = threadIdx.x; u < n_urows; u += blockDim.x) {
        const unsigned u0 = (unsigned)u * nkb;
        tab.clo[u] = (short)((u0 * g + g - 1) / un);
        tab.chi[u] = (short)(((u0 + nkb - 1) * g + g - 1) / un);
    }
    __syncthreads();
}

// Sum, in contributor order, the NF (8 or 16) fp32 partials of output
// features n0.. of token t; the loads of up to MAXC contributors are
// issued together.
template <int NF, int MAXC>
__device__ __forceinline__ void rd_sum(const TcPartition &p, const RdTab &tab, int t, int n0, float (&acc)[NF])
{
    int ur, r, col;
    const float *ws;
    tc_part_loc(p, t, n0 >> 7, ur, r, col, ws);
    const int c_lo = tab.clo[ur], c_hi = tab.chi[ur];
#pragma unroll
    for (int k = 0; k < NF; ++k)
        acc[k] = 0.f;
    for (int cb = c_lo; cb <= c_hi; cb += MAXC) {
        float4 v[MAXC][NF / 4];
#pragma unroll
        for (int i = 0; i < MAXC; ++i) {
            const int c = cb + i;
            if (c <= c_hi) {
                const int slot = ur - tab.first[c];
                const float4 *src = reinterpret_cast<const float4 *>(
                    ws + ((((size_t)c * p.G + r) * p.slots + slot) * p.tg + col) * 128 + (n0 & 127));
#pragma unroll
                for (int e = 0; e < NF / 4; ++e)
                    v[i][e] = __ldcg(src + e);
            }
        }
#pragma unroll
        for (int i = 0; i < MAXC; ++i) {
            if (cb + i <= c_hi) {
#pragma unroll
                for (int e = 0; e < NF / 4; ++e) {
                    acc[4 * e] += v[i][e].x;
                    acc[4 * e + 1] += v[i][e].y;
                    acc[4 * e + 2] += v[i][e].z;
                    acc[4 * e + 3] += v[i][e].w;
                }
            }
        }
    }
}

__host__ __device__ inline int rd_urows(const TcPartition &p, int N)
{
    const int mt = (N + 127) / 128;
    return p.pair ? (mt + 1) / 2 : mt;
}

// One thread per 8-feature group of the row (blockDim = groups rounded up
// to whole warps, at most 1024 = hidden 8192).  TWO: rows of at most 5120
// features (640 threads) with registers bounded so that two CTAs share an
// SM, and a pass over T <= 2 x (SM count) rows runs in one wave.
template <bool TWO>
__global__ void __launch_bounds__(TWO ? 640 : 1024, TWO ? 2 : 1) k_reduce_norm(RnArgs a)
{
    __shared__ RdTab tab;
    __shared__ float red[32];
    pdl_trigger();
    const int t = blockIdx.x;
    const TcPartition &p = a.part;
    rd_build(p, rd_urows(p, a.N), tab);
    pdl_wait();
    const int n0 = threadIdx.x * 8;
    float o[8];
    float ss = 0.f;
    if (n0 < a.N) {
        // the residual's load goes out with the partials' first round
        const uint4 rv = *reinterpret_cast<const uint4 *>(a.resid + (size_t)t * a.N + n0);
        float acc[8];
        rd_sum<8, TWO ? 2 : 4>(p, tab, t, n0, acc);
        const bf16 *re = reinterpret_cast<const bf16 *>(&rv);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            o[k] = bf2f(f2bf(bf2f(re[k]) + acc[k]));  // the stored bf16 value
            ss += o[k] * o[k];
        }
        *reinterpret_cast<uint4 *>(a.out + (size_t)t * a.N + n0) = pack8_bf16(o);
    }
    if (!a.gamma)
        return;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w)
        tot += red[w];
    const float rs = rsqrtf(tot / (float)a.N + a.eps);
    if (n0 < a.N) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            o[k] = o[k] * rs * a.gamma[n0 + k];
        *reinterpret_cast<uint4 *>(a.norm_out + (size_t)t * a.N + n0) = pack8_bf16(o);
    }
}

// Generic finish (k_reduce_epi): every 16-feature group of row t is the sum
// of its contributors' partials, handed to the fused epilogue (SwiGLU for
// the stream-K tail of gate/up; RoPE + KV append when a QKV projection runs
// stream-K; plain fp32 for the GEMM test hook).
constexpr int RE_THREADS = 256;

__global__ void __launch_bounds__(RE_THREADS, 4) k_reduce_epi(TcPartition p, EpiParams ep)
{
    __shared__ RdTab tab;
    pdl_trigger();
    const int t = blockIdx.x;
    rd_build(p, rd_urows(p, ep.N), tab);
    pdl_wait();
    // one 16-feature group per thread; blockIdx.y picks the row's slice
    const int n0 = (blockIdx.y * RE_THREADS + threadIdx.x) * 16;
    if (n0 < ep.N) {
        float v[16];
        rd_sum<16, 2>(p, tab, t, n0, v);
        epi_group(ep, t, n0, v);
    }
}

}  // namespace

cudaError_t launch_reduce_epi(const TcPartition &part, const EpiParams &ep, cudaStream_t s, bool pdl)
{
    if (ep.T <= 0)
        return cudaSuccess;
    if (ep.N % 16 != 0 && ep.mode != EPI_F32)  // fp32 output has a scalar tail
        return cudaErrorInvalidValue;
    if (part.grid > RD_MAX_GRID || rd_urows(part, ep.N) > RD_MAX_UROWS ||
        (long long)part.units * part.grid >= (1ll << 31))
        return cudaErrorInvalidValue;
    const int slices = ((ep.N + 15) / 16 + RE_THREADS - 1) / RE_THREADS;
    cudaError_t e = launch_kernel(pdl, k_reduce_epi, dim3(ep.T, slices), dim3(RE_THREADS), 0, s, part, ep);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_reduce_norm(const TcPartition &part, int T, int N, const bf16 *resid, bf16 *out, const float *gamma,
                               bf16 *norm_out, float eps, cudaStream_t s, bool pdl)
{
    if (T <= 0)
        return cudaSuccess;
    if (N % 8 != 0 || N > 8 * 1024)
        return cudaErrorInvalidValue;
    if (part.grid > RD_MAX_GRID || rd_urows(part, N) > RD_MAX_UROWS ||
        (long long)part.units * part.grid >= (1ll << 31))
        return cudaErrorInvalidValue;
    RnArgs a{part, T, N, resid, out, gamma, norm_out, eps};
    const int threads = ((N / 8) + 31) / 32 * 32;
    cudaError_t e = threads <= 640 ? launch_kernel(pdl, k_reduce_norm<true>, dim3(T), dim3(threads), 0, s, a)
                                   : launch_kernel(pdl, k_reduce_norm<false>, dim3(T), dim3(threads), 0, s, a);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace hb
