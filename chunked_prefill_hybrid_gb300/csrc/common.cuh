// common.cuh -- shared device-side definitions of the hybrid-batch library.
#pragma once

#include <mutex>
#include <unordered_set>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace hb {

typedef __nv_bfloat16 bf16;

// Device error word codes (first error wins, read by hb_sync).
enum DevErr : int {
    DERR_NONE = 0,
    DERR_MBAR_TIMEOUT = 1,   // an mbarrier wait ran past its iteration limit
    DERR_BAD_SLOT = 2,       // a kernel met a slot outside the pool
    DERR_TMEM_ALLOC = 3,     // tensor-memory allocation did not fit
    DERR_BAD_WORK = 4,       // a work item outside its bounds
};

__device__ __forceinline__ void set_dev_err(int *err, int code)
{
    if (err)
        atomicCAS(err, 0, code);
}

__device__ __forceinline__ float bf2f(bf16 x) { return __bfloat162float(x); }
__device__ __forceinline__ bf16 f2bf(float x) { return __float2bfloat16_rn(x); }

// Batch metadata on the device: one contiguous int32 buffer, offsets below.
struct BatchDev {
    int T;                 // rows
    int n_seq;             // sequences (chunk, if any, then decodes)
    int chunk_len;         // rows of the chunk (0 if none)
    const int *pos;        // [T] absolute position of each row
    const int *slot;       // [T] physical slot (block * 16 + offset)
    const int *row_seq;    // [T] sequence index of each row
    const int *seq_q0;     // [n_seq] first row of the sequence
    const int *seq_nq;     // [n_seq] rows of the sequence in this batch
    const int *seq_pos0;   // [n_seq] position of the sequence's first row
    const int *seq_bt;     // [n_seq] offset of its block table in bt
    const int *bt;         // concatenated block tables
};

// Programmatic dependent launch.  A kernel launched with the programmatic
// stream-serialization attribute may start while the previous kernel on
// the stream is still running; pdl_wait() returns once that kernel has
// finished and its writes are visible, so it must precede the first read
// of anything the previous kernel produces.  pdl_trigger() lets the next
// kernel be scheduled as soon as every CTA of this one has started.
// Without the attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Every kernel of the library asks for the largest shared-memory carveout.
// An SM's split between L1 and shared memory is chosen when a CTA lands on
// it while it is idle, from that kernel's preference, and a CTA of another
// kernel can join only within that split: with one preference for all, the
// CTAs of consecutive kernels (the chunk tiles and the decode splits, a
// GEMM and its reduce pass) share SMs whichever kernel arrived first.
inline cudaError_t max_carveout(const void *kernel)
{
    static std::mutex mu;
    static std::unordered_set<const void *> done;
    std::lock_guard<std::mutex> lock(mu);
    if (done.count(kernel))
        return cudaSuccess;
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
        done.insert(kernel);
    return e;
}

// Launch a kernel, with the programmatic stream-serialization attribute
// when pdl is set (the kernel must then call pdl_wait before it reads what
// the previous kernel on the stream writes).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t s, Args... args)
{
    const cudaError_t ce = max_carveout((const void *)kernel);
    if (ce != cudaSuccess)
        return ce;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Epilogue of the fused GEMMs (fp32 accumulators of output pairs).
// EPI_PARTIAL (tensor-core GEMM only): every CTA writes its fp32 partial
// tile(s) to the workspace and a separate kernel reduces them.
enum EpiMode : int { EPI_F32 = 0, EPI_QKV = 1, EPI_RESID = 2, EPI_SWIGLU = 3, EPI_PARTIAL = 4 };

struct EpiParams {
    int mode;
    int T, N;                 // rows, real output features (even)
    // EPI_QKV: rows of W are permuted within each head so that stored rows
    // 2i, 2i+1 hold head features i and i + d/2 (the RoPE rotate-half pair).
    const int *pos, *slot;
    const float2 *rope;       // [max_pos][d/2] (cos, sin)
    int head_dim, n_heads, n_kv;
    bf16 *q_out;              // [T][n_heads d]
    bf16 *k_pool, *v_pool;    // [num_blocks][n_kv][16][d]
    int num_blocks;
    int *err;
    // EPI_RESID: out = resid + acc
    const bf16 *resid;
    bf16 *out;
    // EPI_SWIGLU: stored rows 2j, 2j+1 are gate j and up j; act = silu(g) * u
    bf16 *act;
    int ffn;
    // EPI_F32
    float *d32;
};

__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// One rotate-half RoPE pair (x0 = feature i, x1 = feature i + d/2) turned by
// the angle whose cosine and sine are (c, sn), with each product's rounding
// fixed so every epilogue path gives the same bits.
__device__ __forceinline__ void rope_rot(float &x0, float &x1, float c, float sn)
{
    const float a = __fmaf_rn(x0, c, -__fmul_rn(x1, sn));
    const float b = __fmaf_rn(x1, c, __fmul_rn(x0, sn));
    x0 = a;
    x1 = b;
}

// One output pair (t, n..n+1), n even.
__device__ __forceinline__ void epi_pair(const EpiParams &p, int t, int n, float a0, float a1)
{
    switch (p.mode) {
    case EPI_F32:
        p.d32[(size_t)t * p.N + n] = a0;
        p.d32[(size_t)t * p.N + n + 1] = a1;
        break;
    case EPI_QKV: {
        const int d = p.head_dim, half = d >> 1;
        const int hb = n / d, i = (n % d) >> 1;
        if (hb < p.n_heads + p.n_kv) {
            const float2 cs = p.rope[(size_t)p.pos[t] * half + i];
            rope_rot(a0, a1, cs.x, cs.y);
        }
        if (hb < p.n_heads) {
            bf16 *q = p.q_out + (size_t)t * p.n_heads * d + (size_t)hb * d;
            q[i] = f2bf(a0);
            q[i + half] = f2bf(a1);
        } else {
            const int s = p.slot[t];
            const int blk = s >> 4, off = s & 15;
            if (blk < 0 || blk >= p.num_blocks) {
                set_dev_err(p.err, DERR_BAD_SLOT);
                return;
            }
            const bool is_k = hb < p.n_heads + p.n_kv;
            const int kvh = is_k ? hb - p.n_heads : hb - p.n_heads - p.n_kv;
            bf16 *base = (is_k ? p.k_pool : p.v_pool) + (((size_t)blk * p.n_kv + kvh) * 16 + off) * d;
            base[i] = f2bf(a0);
            base[i + half] = f2bf(a1);
        }
        break;
    }
    case EPI_RESID: {
        const size_t o = (size_t)t * p.N + n;
        p.out[o] = f2bf(bf2f(p.resid[o]) + a0);
        p.out[o + 1] = f2bf(bf2f(p.resid[o + 1]) + a1);
        break;
    }
    case EPI_SWIGLU: {
        const int j = n >> 1;
        if (j < p.ffn)
            p.act[(size_t)t * p.ffn + j] = f2bf(silu_f(a0) * a1);
        break;
    }
    }
}

__device__ __forceinline__ uint4 pack8_bf16(const float (&x)[8])
{
    uint4 u;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k)
        h[k] = __floats2bfloat162_rn(x[2 * k], x[2 * k + 1]);
    return u;
}

// RoPE (cos, sin) of the 8 rotate-half pairs held by the 16 stored QKV
// features n0..n0+15 at position pos (identity outside the q and k heads).
__device__ __forceinline__ void qkv_rope_load(const EpiParams &p, int pos, int n0, float4 (&cs)[4])
{
    const int d = p.head_dim, half = d >> 1;
    const int hb = n0 / d, i0 = (n0 % d) >> 1;
    if (hb < p.n_heads + p.n_kv) {
        const float4 *src = reinterpret_cast<const float4 *>(p.rope + (size_t)pos * half + i0);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            cs[k] = __ldg(src + k);  // (cos, sin) of pairs 2k and 2k+1
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            cs[k] = make_float4(1.f, 0.f, 1.f, 0.f);
    }
}

// The same epilogue as epi_pair over 16 consecutive stored output features
// n0..n0+15 (n0 % 16 == 0) of token t, with 16-byte vector memory accesses.
// For EPI_QKV the 16 stored rows are 8 RoPE pairs: head features i0..i0+7
// and i0+d/2..i0+d/2+7, rotated by cs (from qkv_rope_load at the row's
// position) and written to q or to the row's KV slot; for EPI_SWIGLU they
// are 8 (gate, up) pairs.
__device__ __forceinline__ void epi_group_at(const EpiParams &p, int t, int n0, const float (&v)[16], int slot_t,
                                             const float4 (&cs)[4])
{
    switch (p.mode) {
    case EPI_F32: {
        float *d = p.d32 + (size_t)t * p.N + n0;
        if (n0 + 16 <= p.N && (p.N & 3) == 0) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                reinterpret_cast<float4 *>(d)[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        } else {
#pragma unroll
            for (int k = 0; k < 16; ++k)
                if (n0 + k < p.N)
                    d[k] = v[k];
        }
        break;
    }
    case EPI_QKV: {
        const int d = p.head_dim, half = d >> 1;
        const int hb = n0 / d, i0 = (n0 % d) >> 1;
        float lo[8], hi[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            lo[k] = v[2 * k];
            hi[k] = v[2 * k + 1];
        }
        if (hb < p.n_heads + p.n_kv) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                rope_rot(lo[2 * k], hi[2 * k], cs[k].x, cs[k].y);
                rope_rot(lo[2 * k + 1], hi[2 * k + 1], cs[k].z, cs[k].w);
            }
        }
        bf16 *base;
        if (hb < p.n_heads) {
            base = p.q_out + (size_t)t * p.n_heads * d + (size_t)hb * d;
        } else {
            const int blk = slot_t >> 4, off = slot_t & 15;
            if (blk < 0 || blk >= p.num_blocks) {
                set_dev_err(p.err, DERR_BAD_SLOT);
                return;
            }
            const bool is_k = hb < p.n_heads + p.n_kv;
            const int kvh = is_k ? hb - p.n_heads : hb - p.n_heads - p.n_kv;
            base = (is_k ? p.k_pool : p.v_pool) + (((size_t)blk * p.n_kv + kvh) * 16 + off) * d;
        }
        *reinterpret_cast<uint4 *>(base + i0) = pack8_bf16(lo);
        *reinterpret_cast<uint4 *>(base + i0 + half) = pack8_bf16(hi);
        break;
    }
    case EPI_RESID: {
        const size_t o = (size_t)t * p.N + n0;
        const uint4 r0 = reinterpret_cast<const uint4 *>(p.resid + o)[0];
        const uint4 r1 = reinterpret_cast<const uint4 *>(p.resid + o)[1];
        const bf16 *re0 = reinterpret_cast<const bf16 *>(&r0);
        const bf16 *re1 = reinterpret_cast<const bf16 *>(&r1);
        float a[8], b[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            a[k] = bf2f(re0[k]) + v[k];
            b[k] = bf2f(re1[k]) + v[8 + k];
        }
        reinterpret_cast<uint4 *>(p.out + o)[0] = pack8_bf16(a);
        reinterpret_cast<uint4 *>(p.out + o)[1] = pack8_bf16(b);
        break;
    }
    case EPI_SWIGLU: {
        const int j0 = n0 >> 1;
        if (j0 < p.ffn) {
            float a[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                a[k] = silu_f(v[2 * k]) * v[2 * k + 1];
            *reinterpret_cast<uint4 *>(p.act + (size_t)t * p.ffn + j0) = pack8_bf16(a);
        }
        break;
    }
    }
}

// epi_group_at with the row's position and slot read from p.pos / p.slot.
__device__ __forceinline__ void epi_group(const EpiParams &p, int t, int n0, const float (&v)[16])
{
    float4 cs[4];
    int slot_t = 0;
    if (p.mode == EPI_QKV) {
        qkv_rope_load(p, p.pos[t], n0, cs);
        slot_t = p.slot[t];
    }
    epi_group_at(p, t, n0, v, slot_t, cs);
}

}  // namespace hb
