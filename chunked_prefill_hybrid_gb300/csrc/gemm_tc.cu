// gemm_tc.cu -- the fused linear ops of the hybrid batch on the sm_103a
// tensor cores: acc[t][n] = sum_k X[t][k] W[n][k] over all T = C + D rows of
// the batch at once, so each weight tile is fetched from HBM once and serves
// the chunk's rows and the piggybacked decode rows together (SARATHI summary,
// section 3.4 "Decode-Maximal Batching", "How fusion works").
//
// Orientation ("swap AB"): the MMA's M is weight rows (output features) and
// its N is the batch's tokens, a multiple of 16 up to 256 per MMA, so a batch
// of T rows is padded to 16 rather than to a 128-row tile -- the
// tile-quantization effect of SARATHI summary section 3.4 / Figure 7 is kept
// small by sizing the token tile to T.
//
// Weights are stored tiled, [n_tile][k_block][128][64], so every TMA box is
// a contiguous 16 KB run of HBM and each CTA streams a contiguous range.
//
// The kernel (k_gemm_pair, further down) runs on CTA pairs with the 2-SM
// MMA, data-parallel, stream-K or one data-parallel wave plus a stream-K
// tail; its own comment describes it.  Stream-K tiles leave fp32 partials
// summed in a fixed contributor order, so results do not depend on timing.
// Every mbarrier wait is bounded (wall clock); on a timeout the kernel
// records an error in the device error word, drains and frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "gemm_tc.h"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace hb {

using namespace tc;

constexpr int TC_BM = 128;
constexpr int TC_BK = 64;
constexpr int TC_THREADS = 192;
constexpr int TC_W_BYTES = TC_BM * TC_BK * 2;
constexpr uint64_t TC_WAIT_NS = 2000000000ull;  // 2 s

struct TcArgs {
    int T, N, K;
    int n_mtiles, nkb;
    int G;            // token groups = CTAs per cluster
    int nsub;         // MMAs per k-block (1 or 2; the second accumulates at TMEM column 256)
    int n_sub;        // tokens per MMA (multiple of 16, <= 256); a CTA holds tg = nsub * n_sub
    int tg;
    int n_sub32;      // n_sub rounded up to 32 (the epilogue's column chunks)
    int nslot;        // pair kernel: TMEM accumulator slots of n_sub columns
    int units, grid;  // units = n_mtiles * nkb over `grid` clusters
    int stages, slots;
    float *ws;        // [grid * G][slots][tg][128]
    int *counters;    // [n_mtiles * G]
    const bf16 *w_tiled;  // the weights, streamed into L2 ahead of the TMA loads
    int rel;              // stages released per commit: 2 when the MMAs are short (N < 224), else 1
    int qkv_smem;         // pair kernel, whole QKV tiles: 1 = stage the RoPE'd bf16 tile in shared memory, store
                          // coalesced; 2 = dump the fp32 accumulator there, then rotate and store with every thread
    int dp_tiles;         // pair kernel: tile pairs 0..dp_tiles-1 go whole to clusters 0..dp_tiles-1 (fused
                          // epilogue); units / grid then cover only the stream-K rest, tile pairs dp_tiles..
    int slabs, slab_rows;  // token slabs of the launch (1: all T rows); slab s is rows s*slab_rows..
    size_t ws_slab;        // workspace floats of one slab group
    uint64_t wait_ns;     // wall-clock limit of every mbarrier wait (2 s; shorter only under a test fault)
    int fault;            // test fault: the odd CTA of pair 0 withholds its first weight-tile copy
};

// A cluster's unit range [u0, u1) is cut at tile boundaries into segments
// (one accumulator each).  They are processed with the split tiles first --
// the range's last segment, then its first -- and the whole tiles after, so
// that the stream-K fixups of split tiles overlap the remaining work.
// Distance (k-blocks of 16 KB) the weight stream is prefetched into L2 ahead
// of its TMA loads; the loads then find their data in L2, so fewer shared-
// memory stages cover the HBM latency.  (Measured on the layer step: 4 beats
// both no prefetch and deeper ones, which only add requests once the weight
// stream is marked evict-first.)
constexpr int TC_PREFETCH = 4;

struct SegIter {
    int u0, u1, nkb, n;
    __device__ SegIter(int u0_, int u1_, int nkb_) : u0(u0_), u1(u1_), nkb(nkb_)
    {
        n = (u1 > u0) ? ((u1 - 1) / nkb - u0 / nkb + 1) : 0;
    }
    // bounds of the segment covering tile index `t` (u0 / nkb <= t)
    __device__ void tile_seg(int t, int &a, int &b) const
    {
        a = max(u0, t * nkb);
        b = min(u1, (t + 1) * nkb);
    }
    // i-th segment in processing order
    __device__ void get(int i, int &a, int &b) const
    {
        const int t0 = u0 / nkb;
        int t;
        if (n == 1)
            t = t0;
        else if (i == 0)
            t = t0 + n - 1;
        else if (i == 1)
            t = t0;
        else
            t = t0 + i - 1;
        tile_seg(t, a, b);
    }
};

// Segments of one pair cluster: with a.dp_tiles > 0, first its whole
// data-parallel tile pair (if it has one), then its stream-K range [u0, u1)
// in SegIter order.  get() returns true for the data-parallel segment.
// (Measured: the other order, which frees the stages for a staged SwiGLU
// epilogue of the data-parallel tile, is slower.)
struct PairSegs {
    SegIter sk;
    int n_dp, dp_u0, n;
    __device__ PairSegs(int clu, const TcArgs &a, int u0, int u1) : sk(u0, u1, a.nkb)
    {
        n_dp = clu < a.dp_tiles ? 1 : 0;
        dp_u0 = clu * a.nkb;
        n = n_dp + sk.n;
    }
    __device__ bool get(int i, int &sa, int &sb) const
    {
        if (i < n_dp) {
            sa = dp_u0;
            sb = dp_u0 + sk.nkb;
            return true;
        }
        sk.get(i - n_dp, sa, sb);
        return false;
    }
};

// Epilogue shared memory: position and KV slot of each of the CTA's token
// columns (at most 2 x 256), read by the fused QKV epilogue, and one
// 32 x 32 transpose tile per epilogue warp (rows padded to 33 floats).
constexpr int TC_MAX_TG = 512;
constexpr int TC_META_BYTES = 2 * TC_MAX_TG * 4;
constexpr int TC_XP_LD = 33;
constexpr int TC_XP_BYTES = 4 * 32 * TC_XP_LD * 4;

__device__ __forceinline__ int unit_owner(long long u, const TcArgs &a)
{
    return (int)((u * a.grid + a.grid - 1) / a.units);
}
__device__ __forceinline__ int unit_begin(int c, const TcArgs &a) { return (int)((long long)c * a.units / a.grid); }

__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Fused epilogue of ncol (<= 32) token columns col0.. of this CTA for the
// warp's 32 features nb..nb+31 (lane = feature); r holds the fp32
// accumulator bits, one token column per register.  Every lane of the warp
// calls this together.
//   EPI_F32: one coalesced 128-byte store per token.
//   bf16 outputs (EPI_QKV, EPI_SWIGLU, EPI_RESID): the warp transposes its
//   32 x 32 block through its own shared-memory tile so that a lane owns
//   (token, 16 consecutive features) items, which epi_group_at writes with
//   16-byte stores; the QKV rotation tables of both items are loaded before
//   either item is stored.
__device__ __forceinline__ void emit_cols(const EpiParams &p, const int *s_pos, const int *s_slot, float *xp,
                                          int t_base, int col0, int ncol, int nb, int lane, const uint32_t (&r)[32])
{
    if (p.mode == EPI_F32) {
        const int n = nb + lane;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int t = t_base + col0 + j;
            if (j < ncol && t < p.T && n < p.N)
                p.d32[(size_t)t * p.N + n] = __uint_as_float(r[j]);
        }
        return;
    }
    if (p.mode == EPI_SWIGLU) {
        // feature-major staging in 16-byte chunks of 4 tokens, chunk c of
        // feature f at c ^ (f & 7): lane f writes its 32 tokens as 8 chunks,
        // then lane (tq, o) reads 4 tokens (chunk tq) of features 8o..8o+7,
        // i.e. 4 (gate, up) pairs, and writes 4 act values per token; both
        // sides cover all 32 banks per quarter-warp
        const uint32_t xs = smem_u32(xp);
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(xs + 128u * (uint32_t)lane +
                                                                           16u * (uint32_t)(c ^ (lane & 7))),
                         "r"(r[4 * c]), "r"(r[4 * c + 1]), "r"(r[4 * c + 2]), "r"(r[4 * c + 3])
                         : "memory");
        __syncwarp();
        const int tq = lane & 7, o = lane >> 3;
        float w[8][4];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(w[k][0]), "=f"(w[k][1]), "=f"(w[k][2]), "=f"(w[k][3])
                         : "r"(xs + 128u * (uint32_t)(8 * o + k) + 16u * (uint32_t)(tq ^ k)));
        __syncwarp();
        const int j0 = (nb + 8 * o) >> 1;  // act feature of this lane's first pair
        if (j0 < p.ffn) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = col0 + 4 * tq + u;
                if (4 * tq + u < ncol && t_base + c < p.T) {
                    float a[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        a[k] = silu_f(w[2 * k][u]) * w[2 * k + 1][u];
                    __nv_bfloat162 h0 = __floats2bfloat162_rn(a[0], a[1]), h1 = __floats2bfloat162_rn(a[2], a[3]);
                    uint2 v;
                    v.x = *reinterpret_cast<uint32_t *>(&h0);
                    v.y = *reinterpret_cast<uint32_t *>(&h1);
                    *reinterpret_cast<uint2 *>(p.act + (size_t)(t_base + c) * p.ffn + j0) = v;
                }
            }
        }
        return;
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 32; ++j)
        xp[j * TC_XP_LD + lane] = __uint_as_float(r[j]);  // row = token, column = feature
    __syncwarp();
    const int g = lane & 1;
    const int n0 = nb + g * 16;
    float v[2][16];
    float4 cs[2][4];
    int c[2];
    bool ok[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int j = (lane >> 1) + 16 * k;
        c[k] = col0 + j;
        ok[k] = j < ncol && t_base + c[k] < p.T && n0 < p.N;
#pragma unroll
        for (int e = 0; e < 16; ++e)
            v[k][e] = xp[j * TC_XP_LD + g * 16 + e];
        if (p.mode == EPI_QKV && ok[k])
            qkv_rope_load(p, s_pos[c[k]], n0, cs[k]);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k)
        if (ok[k])
            epi_group_at(p, t_base + c[k], n0, v[k], p.mode == EPI_QKV ? s_slot[c[k]] : 0, cs[k]);
}

// Stream-K fixup of one tile by its last contributor: the sum of every
// contributor's fp32 partial, added in contributor order so the result does
// not depend on timing, then the fused epilogue.  Warp q covers the
// features nb.. of its quadrant for all the CTA's token columns; each
// contributor's row of 32 features is one coalesced 128-byte load.
__device__ __forceinline__ void fixup_tile(const EpiParams &ep, const TcArgs &a, const int *s_pos, const int *s_slot,
                                           float *xp, int rank, int t_base, int mt, int c_lo, int c_hi, int nb, int f,
                                           int lane)
{
    constexpr int MAXC = 8;  // contributors whose partials are loaded together
    const int ncon = c_hi - c_lo + 1;
    const float *src[MAXC];
#pragma unroll
    for (int k = 0; k < MAXC; ++k) {
        const int c = c_lo + min(k, ncon - 1);
        const int cslot = mt - unit_begin(c, a) / a.nkb;
        src[k] = a.ws + ((size_t)(c * a.G + rank) * a.slots + cslot) * a.tg * TC_BM + f;
    }
    for (int c0 = 0; c0 < a.tg; c0 += 32) {
        const int ncol = min(32, a.tg - c0);
        float acc[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
            acc[j] = 0.f;
        for (int cb = 0; cb < ncon; cb += MAXC) {
            if (ncon > MAXC) {
                // tiles split over more than MAXC clusters: this group's partials
#pragma unroll
                for (int k = 0; k < MAXC; ++k) {
                    const int c = c_lo + min(cb + k, ncon - 1);
                    const int cslot = mt - unit_begin(c, a) / a.nkb;
                    src[k] = a.ws + ((size_t)(c * a.G + rank) * a.slots + cslot) * a.tg * TC_BM + f;
                }
            }
#pragma unroll
            for (int k = 0; k < MAXC; ++k) {
                if (cb + k < ncon) {
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        v[j] = j < ncol ? __ldcg(src[k] + (size_t)(c0 + j) * TC_BM) : 0.f;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        acc[j] += v[j];
                }
            }
        }
        uint32_t r[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
            r[j] = __float_as_uint(acc[j]);
        emit_cols(ep, s_pos, s_slot, xp, t_base, c0, ncol, nb, lane, r);
    }
}

// QKV epilogue of a whole tile staged in shared memory (the pipeline stages
// are idle once the tile's last MMA has completed), so that the stores to q
// and to the KV pool are whole head rows instead of 16-byte pieces of 32
// different rows.  qkv_cols_to_smem is emit_cols for EPI_QKV with the same
// arithmetic, writing token t's rotated features into row t of tile_s
// ([tg][QKV_TS] bf16, rows padded by 16 bytes so the 16-row column writes do
// not share banks); qkv_tile_out then copies row by row, 16 bytes a thread.
constexpr int QKV_TS = TC_BM + 8;  // bf16 per staged token row

__device__ __forceinline__ void sts_v4(uint32_t addr, const uint4 &v)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void qkv_cols_to_smem(const EpiParams &p, const int *s_pos, float *xp, int col0, int ncol,
                                                 int nb, int tile, int lane, const uint32_t (&r)[32], uint32_t tile_s)
{
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 32; ++j)
        xp[j * TC_XP_LD + lane] = __uint_as_float(r[j]);  // row = token, column = feature
    __syncwarp();
    const int g = lane & 1;
    const int n0 = nb + g * 16;
    const int d = p.head_dim, half = d >> 1;
    const int hb = n0 / d, i0 = (n0 % d) >> 1;
    const int lf = (n0 - tile * TC_BM) / d * d + i0;  // feature of the lo half within the tile row
    const bool rot = hb < p.n_heads + p.n_kv;
    int c[2];
    bool ok[2];
    float v[2][16];
    float4 cs[2][4];
    // both groups' (cos, sin) loads are issued before any store, and the next
    // chunk's lines are pulled into L1 meanwhile
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int j = (lane >> 1) + 16 * k;
        c[k] = col0 + j;
        ok[k] = j < ncol && c[k] < p.T && n0 < p.N;
#pragma unroll
        for (int e = 0; e < 16; ++e)
            v[k][e] = xp[j * TC_XP_LD + g * 16 + e];
        if (ok[k])
            qkv_rope_load(p, s_pos[c[k]], n0, cs[k]);
    }
    if (rot) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int cn = c[k] + 32;
            if (cn < p.T)
                asm volatile("prefetch.global.L1 [%0];" ::"l"(p.rope + (size_t)s_pos[cn] * half + i0));
        }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        if (!ok[k])
            continue;
        float lo[8], hi[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            lo[q] = v[k][2 * q];
            hi[q] = v[k][2 * q + 1];
        }
        if (rot) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                rope_rot(lo[2 * q], hi[2 * q], cs[k][q].x, cs[k][q].y);
                rope_rot(lo[2 * q + 1], hi[2 * q + 1], cs[k][q].z, cs[k][q].w);
            }
        }
        const uint32_t row = tile_s + 2u * (uint32_t)(c[k] * QKV_TS);
        sts_v4(row + 2u * (uint32_t)lf, pack8_bf16(lo));
        sts_v4(row + 2u * (uint32_t)(lf + half), pack8_bf16(hi));
    }
}

__device__ __forceinline__ void qkv_tile_out(const EpiParams &p, uint32_t s_slot, uint32_t tile_s, int tile, int et)
{
    const int d = p.head_dim;
    const int lvec = d == 128 ? 4 : 3;  // log2 of the 16-byte vectors per head row (d = 128 or 64)
    const int v16 = et & 15;            // this thread's vector of the tile's 128-feature row
    const int hh = v16 >> lvec, v = v16 & ((1 << lvec) - 1);
    const int hb = tile * TC_BM / d + hh;
    if (hb >= p.n_heads + 2 * p.n_kv)
        return;  // rows past N
    const bool is_q = hb < p.n_heads, is_k = hb < p.n_heads + p.n_kv;
    const int kvh = is_k ? hb - p.n_heads : hb - p.n_heads - p.n_kv;
    bf16 *const qbase = p.q_out + (size_t)hb * d + v * 8;
    bf16 *const pool = (is_k ? p.k_pool : p.v_pool) + (size_t)kvh * 16 * d + v * 8;
    // four tokens per round: their loads are issued before their stores
    for (int t0 = et >> 4; t0 < p.T; t0 += 32) {
        uint4 val[4];
        int sl[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int t = t0 + 8 * u;
            if (t < p.T) {
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(val[u].x), "=r"(val[u].y), "=r"(val[u].z), "=r"(val[u].w)
                             : "r"(tile_s + 2u * (uint32_t)(t * QKV_TS + v16 * 8)));
                sl[u] = 0;
                if (!is_q)
                    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(sl[u]) : "r"(s_slot + 4u * (uint32_t)t));
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int t = t0 + 8 * u;
            if (t >= p.T)
                continue;
            bf16 *dst;
            if (is_q) {
                dst = qbase + (size_t)t * p.n_heads * d;
            } else {
                const int blk = sl[u] >> 4, off = sl[u] & 15;
                if (blk < 0 || blk >= p.num_blocks) {
                    set_dev_err(p.err, DERR_BAD_SLOT);
                    continue;
                }
                dst = pool + ((size_t)blk * p.n_kv * 16 + off) * d;
            }
            asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "r"(val[u].x), "r"(val[u].y),
                         "r"(val[u].z), "r"(val[u].w)
                         : "memory");
        }
    }
}

// QKV epilogue of a whole tile from its fp32 accumulator dumped to shared
// memory, run by every thread of the CTA once the tensor-memory reads are
// done (the producer and MMA warps are idle by then).
//
// The dump is feature-major: row f (one of the tile's 128 stored features,
// RoPE pairs interleaved: even = head feature i, odd = feature i + d/2)
// holds the tile's tokens as 16-byte chunks of 4 tokens, chunk c stored at
// position c ^ ((f >> 4) & 7) (so within c's aligned group of 8: the row's
// 8 * ceil(tg / 32) data chunks are permuted, never overlapped), and a row
// is an odd number of chunks long.
// An epilogue lane holds 32 tokens of one feature, so it writes 8 chunks;
// the 8 lanes of a quarter-warp (8 consecutive features, one XOR) land on
// 8 different bank groups because the row length is odd.  A reader thread
// takes 4 tokens (one chunk) of the 16 features of a group g: the 8
// quarter-warp lanes read the same chunk of the 8 groups, whose XORs differ,
// so they too cover all 32 banks.  The reader then holds 8 RoPE pairs of 4
// tokens; the 8 lanes of a token write its 128-byte lo and hi halves of a
// head row, and read its 512-byte row of the (cos, sin) table.
__host__ __device__ inline int qkv_dump_row_bytes(int tg) { return 16 * (8 * ((tg + 31) / 32) + 1); }

__device__ __forceinline__ void qkv_dump_store(uint32_t dump_s, int row_bytes, int f, int col0, int ncol,
                                               const uint32_t (&r)[32])
{
    const uint32_t row = dump_s + (uint32_t)(f * row_bytes);
    const int x = (f >> 4) & 7, c0 = col0 >> 2;  // c -> c ^ x permutes each aligned group of 8 chunks
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (4 * j < ncol)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + 16u * (uint32_t)((c0 + j) ^ x)),
                         "r"(r[4 * j]), "r"(r[4 * j + 1]), "r"(r[4 * j + 2]), "r"(r[4 * j + 3])
                         : "memory");
}

__device__ __forceinline__ void qkv_dump_out(const EpiParams &p, const int *s_pos, const int *s_slot,
                                             uint32_t dump_s, int row_bytes, int tile, int tid, int nthr)
{
    const int d = p.head_dim, half = d >> 1;
    const int g = tid & 7;  // nthr % 8 == 0: a thread keeps its feature group
    const int n0 = tile * TC_BM + 16 * g;
    const int hb = n0 / d, i0 = (n0 % d) >> 1;
    const int n_rot = p.n_heads + p.n_kv;
    if (hb >= p.n_heads + 2 * p.n_kv)
        return;  // rows past N
    const bool is_q = hb < p.n_heads, rot = hb < n_rot;
    const int kvh = rot ? hb - p.n_heads : hb - n_rot;
    bf16 *const pool = (rot ? p.k_pool : p.v_pool) + (size_t)kvh * 16 * d + i0;
    bf16 *const qcol = p.q_out + (size_t)hb * d + i0;
    const float2 *const rope = p.rope + i0;
    const uint32_t grow = dump_s + (uint32_t)(16 * g * row_bytes);
    for (int tq = tid >> 3; 4 * tq < p.T; tq += nthr >> 3) {
        float w[16][4];
        const uint32_t cpos = 16u * (uint32_t)(tq ^ g);
#pragma unroll
        for (int k = 0; k < 16; ++k)
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(w[k][0]), "=f"(w[k][1]), "=f"(w[k][2]), "=f"(w[k][3])
                         : "r"(grow + (uint32_t)(k * row_bytes) + cpos));
        float4 cs[4][4];
        int sl[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int t = 4 * tq + u;
            sl[u] = 0;
            if (t < p.T) {
                if (!is_q)
                    sl[u] = s_slot[t];
                if (rot) {
                    const float4 *src = reinterpret_cast<const float4 *>(rope + (size_t)s_pos[t] * half);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        cs[u][k] = __ldg(src + k);  // (cos, sin) of pairs 2k and 2k+1
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int t = 4 * tq + u;
            if (t >= p.T)
                continue;
            float lo[8], hi[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                lo[k] = w[2 * k][u];
                hi[k] = w[2 * k + 1][u];
            }
            if (rot) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    rope_rot(lo[2 * k], hi[2 * k], cs[u][k].x, cs[u][k].y);
                    rope_rot(lo[2 * k + 1], hi[2 * k + 1], cs[u][k].z, cs[u][k].w);
                }
            }
            bf16 *dst;
            if (is_q) {
                dst = qcol + (size_t)t * p.n_heads * d;
            } else {
                const int blk = sl[u] >> 4, off = sl[u] & 15;
                if (blk < 0 || blk >= p.num_blocks) {
                    set_dev_err(p.err, DERR_BAD_SLOT);
                    continue;
                }
                dst = pool + ((size_t)blk * p.n_kv * 16 + off) * d;
            }
            *reinterpret_cast<uint4 *>(dst) = pack8_bf16(lo);
            *reinterpret_cast<uint4 *>(dst + half) = pack8_bf16(hi);
        }
    }
}

// ------------------------------------------------------------ pair kernel
// The same linear op on CTA pairs (clusters of two) with the 2-SM MMA: one
// tcgen05.mma.cta_group::2 computes a 256-row x n_sub-token product whose
// rows are two weight tiles, one in each CTA, and whose tokens are split
// between the pair's shared memories (the even CTA holds the first n_sub/2
// of each MMA's tokens, the odd CTA the rest).  Per SM that halves both the
// MMA instructions and the shared-memory fill for a given amount of work
// compared with one CTA per tile, so the weight stream (the HBM bound of
// these small-T products) rather than the issue loop sets the pace.
//
// Work: stream-K over units (weight-tile pair, k-block); a pair's unit range
// is cut into segments at tile-pair boundaries.  CTA r of a pair owns weight
// tile 2p + r of tile pair p for all T tokens (nsub MMAs of n_sub tokens).
// TMEM is a ring of nslot slots of n_sub columns; a segment takes nsub
// consecutive slots, and the epilogue releases each slot as soon as it has
// read it, so the next segment starts before the previous one is drained.
//   warp 0      TMA producer in both CTAs: own weight tile + own token
//               halves, completing on the leader's full barrier
//   warp 1      TMEM allocation (both CTAs); MMA issue (even CTA only)
//   warps 2..5  epilogue in both CTAs on their own TMEM rows
constexpr int TC_MAX_SLOTS = 4;
constexpr int TC_PAIR_CTRL = 512;

__host__ __device__ inline int pair_stage_bytes(int nsub, int n_sub) { return TC_W_BYTES + nsub * (n_sub / 2) * TC_BK * 2; }
__host__ __device__ inline int pair_smem_bytes(int nsub, int n_sub, int stages)
{
    return stages * pair_stage_bytes(nsub, n_sub) + TC_PAIR_CTRL + TC_META_BYTES + TC_XP_BYTES + 1024;
}

// The epilogue parameters of the token rows [t0, t0 + rows) of a launch.
__device__ __forceinline__ EpiParams epi_slab(const EpiParams &e0, int t0, int rows)
{
    EpiParams e = e0;
    e.T = rows;
    if (t0) {
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
    }
    return e;
}

__global__ void __launch_bounds__(TC_THREADS, 1)
    k_gemm_pair(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, TcArgs a,
                EpiParams ep_all)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int S = a.stages;
    const int xhalf = a.n_sub >> 1;  // token rows of one MMA held by this CTA
    const int stage_bytes = pair_stage_bytes(a.nsub, a.n_sub);
    uint64_t *full = (uint64_t *)(smem + (size_t)S * stage_bytes);  // [S] (the leader's count)
    uint64_t *empty = full + S;                                     // [S / rel]
    uint64_t *accf = empty + S;                                     // [4]
    uint64_t *sfree = accf + 4;                                     // [TC_MAX_SLOTS] (leader)
    uint64_t *drain = sfree + TC_MAX_SLOTS;
    uint32_t *tmem_slot = (uint32_t *)(drain + 1);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
    volatile int *last_flag = abort_flag + 1;
    int *s_pos = (int *)(smem + (size_t)S * stage_bytes + TC_PAIR_CTRL);
    int *s_slot = s_pos + TC_MAX_TG;
    float *s_xp = (float *)(s_slot + TC_MAX_TG);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = (int)cluster_ctarank();  // 0: the pair's leader
    // CTA pairs of the slab groups are interleaved (pair c of every group
    // side by side), so they stream the same weight tiles at the same time
    const int pair_id = blockIdx.x >> 1;
    const int slab = pair_id % a.slabs;
    const int clu = pair_id / a.slabs;
    const int cta = clu * 2 + r;
    const int xrow0 = slab * a.slab_rows;
    const EpiParams ep = epi_slab(ep_all, xrow0, min(a.slab_rows, a.T - xrow0));
    const int sk_base = a.dp_tiles * a.nkb;
    const int u0 = sk_base + unit_begin(clu, a), u1 = sk_base + unit_begin(clu + 1, a);
    const int rel_mask = a.rel - 1, rel_shift = a.rel == 2 ? 1 : 0;
    pdl_trigger();

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i)
            mbar_init(&full[i], 1);
        for (int i = 0; i < S / a.rel; ++i)
            mbar_init(&empty[i], 1);  // the leader's commit, multicast to both CTAs
        for (int i = 0; i < 4; ++i)
            mbar_init(&accf[i], 1);
        for (int i = 0; i < TC_MAX_SLOTS; ++i)
            mbar_init(&sfree[i], 8);  // every epilogue warp of both CTAs
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
    }
    if (warp == 1)
        tmem_alloc_pair(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers and TMEM exist before any copy or MMA
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t full_leader = cluster_map(smem_u32(full), 0);
    const uint32_t sfree_leader = cluster_map(smem_u32(sfree), 0);

    if (warp == 0) {
        // ------------------------------------------------------ producer
        const uint32_t bytes = (uint32_t)(2 * stage_bytes);  // both CTAs' copies land on the leader's barrier
        const uint64_t wpol = l2_policy_evict_first();
        const PairSegs seg_it(clu, a, u0, u1);
        int it = 0, s = 0;
        uint32_t ph = 0;
        bool ok = true, waited = false;
        for (int i = 0; i < seg_it.n && ok; ++i) {
            int sa, sb;
            seg_it.get(i, sa, sb);
            const int mp = sa / a.nkb;
            const int tile = 2 * mp + r;
            const bool real = tile < a.n_mtiles;  // an odd tile count pads the last pair
            int kb = sa - mp * a.nkb;
            const bf16 *wbase = a.w_tiled + (size_t)tile * a.nkb * TC_BM * TC_BK;
            if (real)
                for (int k = kb; k < min(kb + (sb - sa), kb + TC_PREFETCH); ++k)
                    bulk_prefetch_l2_hint_elect(wbase + (size_t)k * TC_BM * TC_BK, TC_W_BYTES, wpol);
            for (int u = sa; u < sb; ++u, ++it, ++kb) {
                if (real && u + TC_PREFETCH < sb)
                    bulk_prefetch_l2_hint_elect(wbase + (size_t)(kb + TC_PREFETCH) * TC_BM * TC_BK, TC_W_BYTES, wpol);
                if (it >= S && (s & rel_mask) == 0 &&
                    !__all_sync(0xffffffffu, mbar_wait(&empty[s >> rel_shift], ph ^ 1u, abort_flag, a.wait_ns))) {
                    if (lane == 0) {
                        set_dev_err(ep.err, DERR_MBAR_TIMEOUT);
                        *abort_flag = 1;
                    }
                    ok = false;
                    break;
                }
                uint8_t *sw = smem + (size_t)s * stage_bytes;
                const uint32_t fb = full_leader + (uint32_t)(s * 8);
                if (r == 0)
                    mbar_expect_tx_elect(&full[s], bytes);
                // test fault: withhold one copy, so the leader's wait for this
                // stage runs out (nothing else is changed; no copy is left in flight)
                if (!(a.fault && pair_id == 0 && r == 1 && it == 0))
                    tma_load_2d_pair_hint_elect(sw, &tmW, fb, 0, (tile * a.nkb + kb) * TC_BM, wpol);
                if (!waited) {
                    pdl_wait();  // the activations are the previous kernel's output
                    waited = true;
                }
#pragma unroll
                for (int sub = 0; sub < 2; ++sub)
                    if (sub < a.nsub)
                        tma_load_2d_pair_elect(sw + TC_W_BYTES + sub * xhalf * TC_BK * 2, &tmX, fb, kb * TC_BK,
                                               xrow0 + sub * a.n_sub + r * xhalf);
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        // tail: every stage this CTA filled has been consumed (the leader's
        // commits), so no copy into this CTA is still in flight
        for (int k = (it > S ? it - S : 0); k < it; ++k)
            if (k % S % a.rel == 0)
                mbar_wait(&empty[(k % S) / a.rel], (uint32_t)(k / S) & 1u, ok ? abort_flag : nullptr,
                          ok ? a.wait_ns : a.wait_ns / 4);
    } else if (warp == 1) {
        if (r == 0) {
            // -------------------------------------------------- MMA issuer
            const uint32_t idesc = idesc_bf16_f32(2 * TC_BM, a.n_sub);
            const uint64_t desc0 = sdesc_kmajor_sw128(smem_u32(smem));
            const uint32_t stage16 = (uint32_t)stage_bytes >> 4;
            const uint32_t xsub16 = (uint32_t)(xhalf * TC_BK * 2) >> 4;
            const PairSegs seg_it(clu, a, u0, u1);
            int s = 0, slot_next = 0;
            uint32_t ph = 0, st16 = 0, seen = 0, par = 0;
            bool ok = true;
            for (int seg = 0; seg < seg_it.n && ok; ++seg) {
                int sa, sb;
                seg_it.get(seg, sa, sb);
                uint32_t dcol[2];
#pragma unroll
                for (int sub = 0; sub < 2; ++sub) {
                    if (sub < a.nsub) {
                        const int j = slot_next;
                        slot_next = slot_next + 1 == a.nslot ? 0 : slot_next + 1;
                        dcol[sub] = (uint32_t)(j * a.n_sub);
                        if ((seen >> j) & 1u) {
                            if (!__all_sync(0xffffffffu,
                                            mbar_wait(&sfree[j], (par >> j) & 1u, abort_flag, a.wait_ns))) {
                                if (lane == 0) {
                                    set_dev_err(ep.err, DERR_MBAR_TIMEOUT);
                                    *abort_flag = 1;
                                }
                                ok = false;
                            }
                            par ^= 1u << j;
                        }
                        seen |= 1u << j;
                    }
                }
                if (!ok)
                    break;
                tc_fence_after();
                for (int u = sa; u < sb; ++u) {
                    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], ph, abort_flag, a.wait_ns))) {
                        if (lane == 0) {
                            set_dev_err(ep.err, DERR_MBAR_TIMEOUT);
                            *abort_flag = 1;
                        }
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t dw = desc0 + st16;
                    const uint64_t dx = dw + (TC_W_BYTES >> 4);
#pragma unroll
                    for (int sub = 0; sub < 2; ++sub) {
                        if (sub < a.nsub) {
#pragma unroll
                            for (int k = 0; k < TC_BK / 16; ++k)
                                mma_bf16_pair_elect(tmem + dcol[sub], dw + (uint32_t)(k * 2),
                                                    dx + (uint32_t)(sub * xsub16 + k * 2), idesc,
                                                    (u > sa || k > 0) ? 1u : 0u);
                        }
                    }
                    if ((s & rel_mask) == rel_mask)
                        mma_commit_pair_elect(&empty[s >> rel_shift]);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                        st16 = 0;
                    } else {
                        st16 += stage16;
                    }
                }
                if (!ok)
                    break;
                mma_commit_pair_elect(&accf[seg & 3]);
            }
            if (ok && (s & rel_mask) != 0)
                mma_commit_pair_elect(&empty[(s - 1) >> rel_shift]);
            if (!ok) {
                mma_commit_pair_elect(drain);
                mbar_wait(drain, 0, nullptr, a.wait_ns / 4);
            }
        }
    } else {
        // ------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int et = threadIdx.x - 64;
        const int f = q * 32 + lane;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const bool partial_mode = ep.mode == EPI_PARTIAL;
        float *xp = s_xp + q * 32 * TC_XP_LD;
        if (ep.mode == EPI_QKV) {
            // the rows' positions and slots belong to the batch plan, which the
            // step's first kernel writes: read them after the wait for it
            pdl_wait();
            for (int c = et; c < a.tg; c += 128) {
                s_pos[c] = c < ep.T ? ep.pos[c] : 0;
                s_slot[c] = c < ep.T ? ep.slot[c] : -1;
            }
            epi_bar();
        }
        const PairSegs seg_it(clu, a, u0, u1);
        int slot_next = 0;
        for (int seg = 0; seg < seg_it.n; ++seg) {
            int sa, sb;
            const bool dp_seg = seg_it.get(seg, sa, sb);
            const int mp = sa / a.nkb, kb0 = sa % a.nkb;
            const int kb1 = kb0 + (sb - sa);
            const int tile = 2 * mp + r;
            // hybrid launch: the data-parallel tile is finished here, the
            // stream-K tiles always leave partials for the reduce pass
            const bool seg_partial = partial_mode || (a.dp_tiles > 0 && !dp_seg);
            const bool whole = (kb0 == 0 && kb1 == a.nkb);
            const bool direct = whole && !seg_partial;
            // the CTA's last segment: no copy into the stages is pending once its accumulator is full
            const bool staged = direct && a.qkv_smem && seg == seg_it.n - 1;
            const int nb = tile * TC_BM + q * 32;
            if (direct && ep.mode == EPI_RESID) {
                for (int c = lane; c < a.tg; c += 32)
                    if (c < ep.T && nb < a.N)
                        prefetch_l2(ep.resid + (size_t)c * a.N + nb);
            }
            if (!__all_sync(0xffffffffu,
                            mbar_wait(&accf[seg & 3], (uint32_t)(seg >> 2) & 1u, abort_flag, a.wait_ns * 2))) {
                if (lane == 0 && !*abort_flag) {
                    set_dev_err(ep.err, DERR_MBAR_TIMEOUT);
                    *abort_flag = 1;
                }
                break;
            }
            tc_fence_after();
            if (staged)
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the stages' async-proxy use is over
            const int wslot = dp_seg ? 0 : mp - u0 / a.nkb;
            float *ws_mine = a.ws + (size_t)slab * a.ws_slab + ((size_t)cta * a.slots + wslot) * a.tg * TC_BM;
            for (int sub = 0; sub < a.nsub; ++sub) {
                const int j = slot_next;
                slot_next = slot_next + 1 == a.nslot ? 0 : slot_next + 1;
                const uint32_t d0 = tmem + lane_base + (uint32_t)(j * a.n_sub);
                for (int c0 = 0; c0 < a.n_sub; c0 += 32) {
                    uint32_t rr[32];
                    tmem_ld_32x32b_x16(d0 + (uint32_t)c0, *reinterpret_cast<uint32_t(*)[16]>(rr));
                    tmem_ld_32x32b_x16(d0 + (uint32_t)(c0 + 16), *reinterpret_cast<uint32_t(*)[16]>(rr + 16));
                    tmem_ld_wait();
                    const int col0 = sub * a.n_sub + c0;
                    const int ncol = min(32, a.n_sub - c0);
                    if (staged && a.qkv_smem == 2) {
                        qkv_dump_store(smem_u32(smem), qkv_dump_row_bytes(a.tg), f, col0, ncol, rr);
                    } else if (staged) {
                        qkv_cols_to_smem(ep, s_pos, xp, col0, ncol, nb, tile, lane, rr, smem_u32(smem));
                    } else if (direct) {
                        emit_cols(ep, s_pos, s_slot, xp, 0, col0, ncol, nb, lane, rr);
                    } else {
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj)
                            if (jj < ncol)
                                ws_mine[(size_t)(col0 + jj) * TC_BM + f] = __uint_as_float(rr[jj]);
                    }
                }
                // this slot's columns are read: hand them back to the MMA warp
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_remote_arrive(sfree_leader + (uint32_t)(j * 8));
            }
            if (staged && a.qkv_smem == 1) {
                epi_bar();  // the whole tile is in shared memory
                qkv_tile_out(ep, smem_u32(s_slot), smem_u32(smem), tile, et);
            }
            if (!whole && !seg_partial) {
                __threadfence();
                epi_bar();
                const int c_lo = unit_owner((long long)mp * a.nkb, a);
                const int c_hi = unit_owner((long long)mp * a.nkb + a.nkb - 1, a);
                if (et == 0) {
                    const int old = atomicAdd(&a.counters[tile], 1);
                    *last_flag = (old == c_hi - c_lo);
                }
                epi_bar();
                if (*last_flag) {
                    __threadfence();
                    fixup_tile(ep, a, s_pos, s_slot, xp, r, 0, mp, c_lo, c_hi, nb, f, lane);
                    if (et == 0)
                        a.counters[tile] = 0;
                }
                epi_bar();
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (a.qkv_smem == 2 && !*abort_flag) {
        // the dumped tile (one whole tile pair per CTA pair): every thread
        // rotates and stores; q and the KV pool may still be read by the
        // previous kernel until it has completed
        pdl_wait();
        qkv_dump_out(ep, s_pos, s_slot, smem_u32(smem), qkv_dump_row_bytes(a.tg), 2 * (u0 / a.nkb) + r, threadIdx.x,
                     TC_THREADS);
    }
    cluster_sync();  // the leader's MMAs and both epilogues are done with both CTAs
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

// Rearrange W [N][K] (rows optionally permuted) into [n_tile][k_block][128][64],
// zero outside N x K.  mode 0: identity rows; 1: RoPE pair permutation
// within heads of `a` rows; 2: gate/up interleave with ffn = `a`.
__global__ void k_tile_weights(const bf16 *__restrict__ src, bf16 *__restrict__ dst, int N, int K, int nkb, int mode,
                               int a)
{
    const int r = blockIdx.x;  // destination row in [0, N_pad)
    int sr = r;
    if (r < N) {
        if (mode == 1) {
            const int hb = r / a, w = r % a;
            sr = hb * a + (w >> 1) + (w & 1) * (a >> 1);
        } else if (mode == 2) {
            sr = (r >> 1) + (r & 1) * a;
        }
    }
    const int mt = r / TC_BM, rr = r % TC_BM;
    for (int k = threadIdx.x; k < nkb * TC_BK; k += blockDim.x) {
        const int kb = k / TC_BK, kk = k % TC_BK;
        bf16 v = __float2bfloat16_rn(0.f);
        if (r < N && k < K)
            v = src[(size_t)sr * K + k];
        dst[(((size_t)mt * nkb + kb) * TC_BM + rr) * TC_BK + kk] = v;
    }
}

// ------------------------------------------------------------------- host

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

static bool encode_2d(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                      uint32_t box_inner, uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

size_t tiled_weight_elems(int N, int K)
{
    const size_t npad = (size_t)(N + TC_BM - 1) / TC_BM * TC_BM;
    const size_t nkb = (size_t)(K + TC_BK - 1) / TC_BK;
    return npad * nkb * TC_BK;
}

cudaError_t launch_tile_weights(const bf16 *src, bf16 *dst, int N, int K, int mode, int a, cudaStream_t s)
{
    const int npad = (N + TC_BM - 1) / TC_BM * TC_BM;
    const int nkb = (K + TC_BK - 1) / TC_BK;
    k_tile_weights<<<npad, 256, 0, s>>>(src, dst, N, K, nkb, mode, a);
    return cudaGetLastError();
}

bool make_tmap_tiled_weights(CUtensorMap *m, const void *tiled, int N, int K, int box_rows)
{
    const uint64_t npad = (uint64_t)(N + TC_BM - 1) / TC_BM * TC_BM;
    const uint64_t nkb = (uint64_t)(K + TC_BK - 1) / TC_BK;
    return encode_2d(m, tiled, TC_BK, npad * nkb, TC_BK * 2, TC_BK, (uint32_t)box_rows);
}

bool make_tmap_rows(CUtensorMap *m, const void *X, int K, int T, int box_rows)
{
    return encode_2d(m, X, (uint64_t)K, (uint64_t)T, (uint64_t)K * 2, TC_BK, (uint32_t)box_rows);
}

// The paged K or V pool [num_blocks][n_kv][16][d] as a 2D tensor of
// num_blocks * n_kv * 16 rows of d elements, in boxes of 16 rows x 64
// elements (128-byte swizzle): one box is half (d = 128) or all (d = 64) of
// one head's 16-token block.
bool make_tmap_kv_pool(CUtensorMap *m, const void *pool, int num_blocks, int n_kv, int d)
{
    return encode_2d(m, pool, (uint64_t)d, (uint64_t)num_blocks * n_kv * 16, (uint64_t)d * 2, 64, 16);
}

// Slots (partial tiles) a CTA can hold: the most tiles any cluster's unit range touches.
static int tc_slots(long long units, int grid, int nkb)
{
    const long long per = (units + grid - 1) / grid;
    return (int)((per + nkb - 1) / nkb + 1);
}

static int tc_grid(long long units, int max_clusters)
{
    return (int)(units < max_clusters ? units : max_clusters);
}

// ---------------------------------------------------------- pair launcher
TcShape tc_pair_shape(int T)
{
    TcShape sh;
    sh.G = 2;
    sh.nsub = T <= 256 ? 1 : 2;
    sh.n_sub = ((T + sh.nsub - 1) / sh.nsub + 15) / 16 * 16;
    if (sh.n_sub < 16)
        sh.n_sub = 16;
    sh.tg = sh.nsub * sh.n_sub;
    return sh;
}

static int pair_nslot(int n_sub)
{
    int n = 512 / n_sub;
    if (n > TC_MAX_SLOTS)
        n = TC_MAX_SLOTS;
    while (n > 0 && (n - 1) * n_sub + (n_sub + 31) / 32 * 32 > 512)
        --n;  // the epilogue reads whole 32-column chunks
    return n;
}

size_t tc_pair_workspace_floats(int num_sms, int max_tokens, const int *Ns, const int *Ks, int n_shapes)
{
    size_t need = 0;
    for (int i = 0; i < n_shapes; ++i)
        for (int T = 1; T <= max_tokens && T <= TC_PAIR_MAX_ROWS; ++T) {
            const int slabs = (T + TC_PAIR_MAX_T - 1) / TC_PAIR_MAX_T;
            const int rows = slabs > 1 ? ((T + slabs - 1) / slabs + 15) / 16 * 16 : T;
            const TcShape sh = tc_pair_shape(rows);
            const int n_mpairs = ((Ns[i] + TC_BM - 1) / TC_BM + 1) / 2;
            const int nkb = (Ks[i] + TC_BK - 1) / TC_BK;
            const long long units = (long long)n_mpairs * nkb;
            const int grid = tc_grid(units, num_sms / 2);
            const size_t n = (size_t)slabs * grid * 2 * tc_slots(units, grid, nkb) * sh.tg * TC_BM;
            if (n > need)
                need = n;
        }
    return need;
}

bool tc_pair_data_parallel(const TcRuntime &rt, int N)
{
    const int n_mpairs = ((N + TC_BM - 1) / TC_BM + 1) / 2;
    const int pairs = rt.num_sms / 2;
    return n_mpairs <= pairs && 10 * n_mpairs >= 6 * pairs;
}

int tc_pair_dp_tiles(const TcRuntime &rt, int N, int K)
{
    const int n_mpairs = ((N + TC_BM - 1) / TC_BM + 1) / 2;
    const int pairs = rt.num_sms / 2;
    const long long sk_units = (long long)(n_mpairs - pairs) * ((K + TC_BK - 1) / TC_BK);
    // every cluster must get stream-K units: the reduce pass sums every
    // cluster of a tile's contributor range
    return (n_mpairs > pairs && sk_units >= pairs) ? pairs : 0;
}

cudaError_t launch_gemm_pair(const CUtensorMap &tmW, const bf16 *W_tiled, const bf16 *X, int T, int N, int K,
                             const EpiParams &ep, const TcRuntime &rt, cudaStream_t s, TcPartition *part, bool pdl,
                             int dp_tiles, uint64_t fault_wait_ns)
{
    if (T <= 0)
        return cudaSuccess;
    if (K % 8 != 0 || T > TC_PAIR_MAX_ROWS)
        return cudaErrorInvalidValue;
    // more rows than one CTA pair's TMEM holds: token slabs, each with its
    // own group of CTA pairs (partials only, no data-parallel tiles)
    const int slabs = (T + TC_PAIR_MAX_T - 1) / TC_PAIR_MAX_T;
    const int slab_rows = slabs > 1 ? ((T + slabs - 1) / slabs + 15) / 16 * 16 : T;
    const TcShape sh = tc_pair_shape(slab_rows);
    TcArgs a = {};
    a.T = T;
    a.slabs = slabs;
    a.slab_rows = slab_rows;
    a.N = N;
    a.K = K;
    a.n_mtiles = (N + TC_BM - 1) / TC_BM;
    a.nkb = (K + TC_BK - 1) / TC_BK;
    a.G = 2;
    a.nsub = sh.nsub;
    a.n_sub = sh.n_sub;
    a.tg = sh.tg;
    a.n_sub32 = (sh.n_sub + 31) / 32 * 32;
    a.nslot = pair_nslot(sh.n_sub);
    if (a.nslot < a.nsub || a.tg > TC_MAX_TG)
        return cudaErrorInvalidValue;
    const int n_mpairs = (a.n_mtiles + 1) / 2;
    if (dp_tiles < 0 || dp_tiles >= n_mpairs || (dp_tiles > 0 && (ep.mode == EPI_PARTIAL || !part)) ||
        (dp_tiles > 0 && (long long)(n_mpairs - dp_tiles) * a.nkb < dp_tiles))
        return cudaErrorInvalidValue;
    a.dp_tiles = dp_tiles;
    a.wait_ns = fault_wait_ns ? fault_wait_ns : TC_WAIT_NS;
    a.fault = fault_wait_ns ? 1 : 0;
    const long long units = (long long)(n_mpairs - dp_tiles) * a.nkb;  // the stream-K part
    if (units > (1ll << 30) || (long long)n_mpairs * 2 > rt.n_counters)
        return cudaErrorInvalidValue;
    a.units = (int)units;
    a.rel = (a.tg < 224) ? 2 : 1;  // 1 or 2: the kernel's ring counters assume a power of two <= 2
    int stages = 12;
    while (stages > 2 && pair_smem_bytes(a.nsub, a.n_sub, stages) > rt.max_smem)
        stages -= a.rel;
    if (pair_smem_bytes(a.nsub, a.n_sub, stages) > rt.max_smem || stages % a.rel)
        return cudaErrorInvalidConfiguration;
    a.stages = stages;
    const int smem = pair_smem_bytes(a.nsub, a.n_sub, stages);
    static int configured = 0;
    if (configured < rt.max_smem) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm_pair, cudaFuncAttributeMaxDynamicSharedMemorySize, rt.max_smem);
        if (e == cudaSuccess)
            e = max_carveout((const void *)k_gemm_pair);
        if (e != cudaSuccess)
            return e;
        configured = rt.max_smem;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(TC_THREADS);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static int max_pairs[13] = {};
    int &mc = max_pairs[stages];
    if (!mc) {
        cfg.gridDim = dim3((unsigned)(rt.num_sms / 2 * 2));
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, k_gemm_pair, &cfg) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = rt.num_sms / 2;
        }
        mc = n < rt.num_sms / 2 ? n : rt.num_sms / 2;
    }
    // every slab runs the launch a single slab would (the same grid, so the
    // same split of K: a row's result does not depend on the batch); the
    // slab groups' CTA pairs are interleaved and may take several waves
    a.grid = tc_grid(units, mc);
    if (dp_tiles > 0) {
        // one data-parallel wave (tile pair c whole to cluster c, fused
        // epilogue), then the remaining tile pairs stream-K over all clusters
        if (dp_tiles > mc)
            return cudaErrorInvalidValue;
        a.grid = mc;
    } else if (ep.mode != EPI_PARTIAL) {
        // data-parallel: one whole weight-tile pair per CTA pair, fused
        // epilogue, no partials
        if (n_mpairs > mc)
            return cudaErrorInvalidValue;
        a.grid = n_mpairs;
        const long long stage_total = (long long)stages * pair_stage_bytes(a.nsub, a.n_sub);
        if (ep.mode == EPI_QKV && (ep.head_dim == 128 || ep.head_dim == 64))
            a.qkv_smem = (long long)TC_BM * qkv_dump_row_bytes(a.tg) <= stage_total ? 2
                         : (long long)a.tg * QKV_TS * 2 <= stage_total   ? 1
                                                                          : 0;
    }
    a.slots = tc_slots(units, a.grid, a.nkb);
    a.ws_slab = (size_t)a.grid * 2 * a.slots * a.tg * TC_BM;
    if (a.ws_slab * slabs > rt.ws_floats)
        return cudaErrorInvalidValue;
    if (part) {
        part->ws = rt.ws;
        part->grid = a.grid;
        part->G = 2;
        part->units = a.units;
        part->nkb = a.nkb;
        part->tg = a.tg;
        part->slots = a.slots;
        part->pair = 1;
        part->slabs = slabs;
        part->slab_rows = slab_rows;
        part->ws_slab = a.ws_slab;
    }
    a.ws = rt.ws;
    a.counters = rt.counters;
    a.w_tiled = W_tiled;
    CUtensorMap tmX;
    if (!encode_2d(&tmX, X, (uint64_t)K, (uint64_t)T, (uint64_t)K * 2, TC_BK, (uint32_t)(a.n_sub / 2)))
        return cudaErrorInvalidValue;
    cfg.gridDim = dim3((unsigned)(a.grid * slabs * 2));
    cudaLaunchAttribute attr2[2] = {attr[0], {}};
    if (pdl) {
        attr2[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr2[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr2;
        cfg.numAttrs = 2;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_gemm_pair, tmW, tmX, a, ep);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

}  // namespace hb
