// common.cuh -- shared device-side definitions of the hybrid-batch library.
#pragma once

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

// Epilogue of the fused GEMMs (fp32 accumulators of output pairs).
enum EpiMode : int { EPI_F32 = 0, EPI_QKV = 1, EPI_RESID = 2, EPI_SWIGLU = 3 };

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

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

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
            const float x0 = a0 * cs.x - a1 * cs.y;
            const float x1 = a1 * cs.x + a0 * cs.y;
            a0 = x0;
            a1 = x1;
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

}  // namespace hb
