// decode_noalloc.cu -- paged decode attention for callers that cannot
// allocate device memory.
//
// The batch forward keeps its split-K attention scratch in buffers that
// hb_init allocates.  Some callers cannot use a context that allocates:
// an engine that has already reserved nearly all HBM for its own KV-cache
// arena up front, or code that runs while other work is in flight and must
// not call cudaMalloc / cudaFree (which can synchronise the whole device).
// This entry point computes the same decode attention -- each query at
// position ctx attends to its sequence's keys 0..ctx through its block
// table -- with its scratch (split partials and arrival counters) in a
// fixed, file-scope device array, so it allocates nothing.
//
// Every call asks the runtime (cudaGetSymbolAddress, with the device
// current) where the array lives: the array's name in host code is only a
// host-side stand-in, and the module -- with the array -- may be loaded at
// another address after a device reset.  The first call on a device, and the
// first after the address changed, also zeroes the counters; make the first
// call on each device before any stream capture.  Every call shares the one
// array: calls that overlap on the GPU race and give wrong results.  Each
// call leaves the counters at zero again.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "hb.h"

namespace hb {
namespace {

constexpr int NA_SPLIT = 256;         // keys per split at most: small splits keep the fixed partials array
                                      // small (the batch forward splits at 1024 keys, so its fp32 sums run in
                                      // another order and the two agree to within one bf16 step)
constexpr int NA_MAX_PAIRS = 4096;    // decodes x heads
constexpr int NA_MAX_PARTS = 16384;   // decodes x heads x splits
constexpr int NA_MAX_D = 128;
constexpr size_t NA_COUNTER_BYTES = NA_MAX_PAIRS * sizeof(int);              // 16 KB
constexpr size_t NA_PART_BYTES = (size_t)NA_MAX_PARTS * (2 + NA_MAX_D) * 4;  // 8.5 MB
constexpr size_t NA_SCRATCH_BYTES = NA_COUNTER_BYTES + NA_PART_BYTES;

// counters [NA_MAX_PAIRS] int, then partials [NA_MAX_PARTS][2 + NA_MAX_D] float (m, l, o)
static __device__ __align__(256) unsigned char g_na_scratch[NA_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_na_mu;
unsigned char *g_na_ptr[MAX_DEVICES] = {nullptr};

// Keys [k0, k1) of split `split` of a sequence with nkeys keys.
__device__ __forceinline__ void na_split_range(int nkeys, int split, int &k0, int &k1, int &n_splits)
{
    n_splits = (nkeys + NA_SPLIT - 1) / NA_SPLIT;
    int len = (nkeys + n_splits - 1) / n_splits;
    len = (len + 15) & ~15;
    k0 = split * len;
    k1 = min(nkeys, k0 + len);
}

// One CTA of 4 warps per (decode, head, split); warps stride over the keys
// of the split, each with its own online softmax, merged at the end.
template <int D>
__global__ void __launch_bounds__(128)
    k_decode_noalloc(const bf16 *__restrict__ q, const bf16 *__restrict__ kp, const bf16 *__restrict__ vp,
                     const int *__restrict__ bt, int bt_stride, const int *__restrict__ ctx_lens, int n_heads,
                     int n_kv, int num_blocks, int max_ctx, int max_splits, bf16 *__restrict__ out,
                     unsigned char *scratch)
{
    constexpr int E = D / 32;
    const int pair = blockIdx.x / max_splits, split = blockIdx.x % max_splits;
    const int j = pair / n_heads, h = pair % n_heads;
    const int kvh = h / (n_heads / n_kv);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int *counters = reinterpret_cast<int *>(scratch);
    float *parts = reinterpret_cast<float *>(scratch + NA_COUNTER_BYTES);
    __shared__ float sm[4], sl[4];
    __shared__ float so[4][D];
    __shared__ int last;

    const int ctx = ctx_lens[j];
    bf16 *orow = out + ((size_t)j * n_heads + h) * D;
    if (ctx < 0 || ctx > max_ctx) {
        // outside what the grid was sized for: flag the row with NaN
        if (split == 0 && threadIdx.x < D)
            orow[threadIdx.x] = f2bf(__int_as_float(0x7fc00000));
        return;
    }
    const int nkeys = ctx + 1;
    int k0, k1, n_splits;
    na_split_range(nkeys, split, k0, k1, n_splits);
    if (split >= n_splits)
        return;
    const int *tab = bt + (size_t)j * bt_stride;
    const float scale = rsqrtf((float)D);
    float qv[E], acc[E];
    const bf16 *qr = q + ((size_t)j * n_heads + h) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        qv[e] = bf2f(qr[e]) * scale;
        acc[e] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    bool bad = false;
    for (int t = k0 + warp; t < k1; t += 4) {
        const int blk = tab[t >> 4];
        if (blk < 0 || blk >= num_blocks) {
            bad = true;
            break;
        }
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
        for (int e = 0; e < E; ++e)  // p == 0 adds nothing, not even 0 * NaN
            acc[e] = acc[e] * corr + (p > 0.f ? p * bf2f(vp[base + e]) : 0.f);
        m = mn;
    }
    if (bad)
        m = __int_as_float(0x7fc00000);  // a block id outside the pool poisons the result
    if (lane == 0) {
        sm[warp] = m;
        sl[warp] = l;
    }
#pragma unroll
    for (int e = 0; e < E; ++e)
        so[warp][lane * E + e] = acc[e];
    __syncthreads();
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w)
        M = fmaxf(M, sm[w]);
    float L = 0.f, f[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        f[w] = (sm[w] == -INFINITY) ? 0.f : __expf(sm[w] - M);
        L += sl[w] * f[w];
    }
    float ov = 0.f;
    if (threadIdx.x < D)
#pragma unroll
        for (int w = 0; w < 4; ++w)
            ov += so[w][threadIdx.x] * f[w];
    if (n_splits == 1) {
        if (threadIdx.x < D)
            orow[threadIdx.x] = f2bf(ov / L);
        return;
    }
    float *mine = parts + ((size_t)pair * max_splits + split) * (2 + NA_MAX_D);
    if (threadIdx.x < D)
        mine[2 + threadIdx.x] = ov;
    if (threadIdx.x == 0) {
        mine[0] = M;
        mine[1] = L;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
        last = (atomicAdd(&counters[pair], 1) == n_splits - 1);
    __syncthreads();
    if (!last)
        return;
    __threadfence();
    const float *p0 = parts + (size_t)pair * max_splits * (2 + NA_MAX_D);
    float Mg = -INFINITY;
    for (int s = 0; s < n_splits; ++s)
        Mg = fmaxf(Mg, __ldcg(&p0[s * (2 + NA_MAX_D)]));
    float Lg = 0.f, og = 0.f;
    for (int s = 0; s < n_splits; ++s) {
        const float ms = __ldcg(&p0[s * (2 + NA_MAX_D)]);
        const float fs = (ms == -INFINITY) ? 0.f : __expf(ms - Mg);
        Lg += __ldcg(&p0[s * (2 + NA_MAX_D) + 1]) * fs;
        if (threadIdx.x < D)
            og += __ldcg(&p0[s * (2 + NA_MAX_D) + 2 + threadIdx.x]) * fs;
    }
    if (threadIdx.x < D)
        orow[threadIdx.x] = f2bf(og / Lg);
    if (threadIdx.x == 0)
        counters[pair] = 0;  // ready for the next call
}

}  // namespace
}  // namespace hb

using namespace hb;

extern "C" int hb_decode_attention_noalloc(const void *q, const void *k_pool, const void *v_pool,
                                           const int32_t *block_tables, int bt_stride, const int32_t *ctx_lens,
                                           int n_decodes, int n_heads, int n_kv_heads, int head_dim, int num_blocks,
                                           int max_ctx, void *out, void *cuda_stream)
{
    if (!q || !k_pool || !v_pool || !block_tables || !ctx_lens || !out)
        return HB_EINVAL;
    if (n_decodes < 1 || n_heads < 1 || n_kv_heads < 1 || n_heads % n_kv_heads || num_blocks < 1 || max_ctx < 0)
        return HB_EINVAL;
    if (head_dim != 64 && head_dim != 128)
        return HB_EINVAL;
    if (bt_stride < max_ctx / 16 + 1)
        return HB_ERANGE;
    const long long pairs = (long long)n_decodes * n_heads;
    const int max_splits = (max_ctx + 1 + NA_SPLIT - 1) / NA_SPLIT;
    if (pairs > NA_MAX_PAIRS || pairs * max_splits > NA_MAX_PARTS)
        return HB_ERANGE;  // beyond the fixed scratch: n_decodes * n_heads <= 4096 and
                           // n_decodes * n_heads * ceil((max_ctx + 1) / 256) <= 16384
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES)
        return HB_ECUDA;
    cudaStream_t s = (cudaStream_t)cuda_stream;
    // the device address of the array, looked up on every call (a host-side
    // table lookup once the module is loaded); zero the counters whenever it
    // is new for this device
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_na_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return HB_ECUDA;
    }
    unsigned char *scratch = (unsigned char *)p;
    {
        std::lock_guard<std::mutex> lock(g_na_mu);
        if (g_na_ptr[dev] != scratch) {
            if (cudaMemsetAsync(scratch, 0, NA_COUNTER_BYTES, s) != cudaSuccess)
                return HB_ECUDA;
            g_na_ptr[dev] = scratch;
        }
    }
    const dim3 grid((unsigned)(pairs * max_splits));
    if (head_dim == 128)
        k_decode_noalloc<128><<<grid, 128, 0, s>>>((const bf16 *)q, (const bf16 *)k_pool, (const bf16 *)v_pool,
                                                   block_tables, bt_stride, ctx_lens, n_heads, n_kv_heads,
                                                   num_blocks, max_ctx, max_splits, (bf16 *)out, scratch);
    else
        k_decode_noalloc<64><<<grid, 128, 0, s>>>((const bf16 *)q, (const bf16 *)k_pool, (const bf16 *)v_pool,
                                                  block_tables, bt_stride, ctx_lens, n_heads, n_kv_heads,
                                                  num_blocks, max_ctx, max_splits, (bf16 *)out, scratch);
    return cudaGetLastError() == cudaSuccess ? HB_OK : HB_ECUDA;
}
