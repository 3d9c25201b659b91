// attention_hybrid.cu -- one launch for the whole hybrid batch's attention.
//
// Semantics (Sarathi-Serve Guide, "Deep Dive: Mathematical Formulation and
// Attention Mechanics"; SARATHI summary, section 3.4 "Chunked-Prefills",
// Figure 6): a query of a request at absolute position p attends to that
// request's keys at positions 0..p -- for the prefill chunk, the cached
// prefix plus the causal triangle inside the chunk; for a decode with S
// cached tokens, S+1 keys.  Keys of other requests are never visible (the
// block-diagonal hybrid mask).  softmax(q.k / sqrt(d)) v in fp32.
//
// Work items, one CTA each, heavy ones first:
//   chunk tile  64 query rows of a multi-row sequence x one head.  Flash-
//               style: Q tile in shared memory, key tiles of 64 gathered from
//               the paged pool with cp.async (double buffered), S = Q K^T and
//               O += P V on the tensor cores (mma.sync m16n8k16, bf16 in, fp32
//               accumulate), online softmax in registers.  P is split into
//               bf16 hi + lo parts for the PV product so the weights keep
//               ~16 significant bits.
//   decode split one head of a single-row sequence over a range of its keys
//               (1024..2047 keys; shorter contexts are one split).  Each
//               16-token block of K and of V is streamed by TMA (16-row x
//               64-dim boxes, 128-byte swizzle) into an 8-stage shared-memory
//               ring (mbarrier pipeline); the 4 warps take the blocks in turn,
//               each with its own online softmax, and compute K q and V^T P
//               on the tensor cores (mma.sync m16n8k16 with the query as the
//               8-column side), merged across the warps at the end.  The
//               number of splits depends on the context length only.
//               Partial (m, l, o) go to a workspace; the last split to finish
//               (per-(sequence, head) arrival counter, no waiting) merges
//               them in split order.
#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "attention.h"
#include "tc_ptx.cuh"

namespace hb {

using namespace tc;

namespace {

constexpr int CQ = 64;            // chunk tile rows
constexpr int CK = 64;            // chunk key tile
constexpr int NSTAGE = 8;         // decode ring depth (16-token blocks)
// The four warps of a decode split take blocks round-robin, and ring slot s
// holds blocks s, s + NSTAGE, s + 2 NSTAGE, ...: with NSTAGE a multiple of
// four, one warp owns every block of a slot, so each slot's mbarrier phases
// are waited for and refilled in order (a warp never waits on a phase two
// ahead, which the parity test cannot tell from a completed one).
static_assert(NSTAGE % 4 == 0, "decode ring depth must be a multiple of the four warps");
constexpr float LOG2E = 1.4426950408889634f;
constexpr uint64_t WAIT_NS = 2000000000ull;

// byte offset of (row, 16-byte chunk) in a [rows][2 D bytes] tile; the
// chunk index is XORed with the row so that 8 consecutive rows of one chunk
// column fall in 8 different bank groups.
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int chunk)
{
    return (uint32_t)(row * (2 * D) + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// ------------------------------------------------------------ chunk tile

template <int D>
__device__ void chunk_tile(const AttnParams &p, int seq, int head, int q0, uint8_t *smem)
{
    constexpr int ROWB = 2 * D, NCH = D / 8, KS = D / 16, NT = D / 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kvh = head / (p.n_heads / p.n_kv);
    const int row0 = p.b.seq_q0[seq], nq = p.b.seq_nq[seq], pos0 = p.b.seq_pos0[seq];
    const int *bt = p.b.bt + p.b.seq_bt[seq];
    const int qrows = min(CQ, nq - q0);
    const int last_key = pos0 + q0 + qrows - 1;  // keys 0..last_key
    const int n_kt = last_key / CK + 1;

    const uint32_t sQ = smem_u32(smem);
    const uint32_t sK[2] = {sQ + CQ * ROWB, sQ + CQ * ROWB + 2 * CK * ROWB};
    const uint32_t sV[2] = {sK[0] + CK * ROWB, sK[1] + CK * ROWB};

    // Q tile (rows past the chunk are zero)
    for (int i = threadIdx.x; i < CQ * NCH; i += blockDim.x) {
        const int r = i / NCH, ch = i % NCH;
        const uint32_t dst = sQ + swz<D>(r, ch);
        if (r < qrows)
            cp_async16(dst, p.q + ((size_t)(row0 + q0 + r) * p.n_heads + head) * D + ch * 8);
        else
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0));
    }
    auto load_kv = [&](int kt, int buf) {
        for (int i = threadIdx.x; i < CK * NCH; i += blockDim.x) {
            const int r = i / NCH, ch = i % NCH;
            const int kp = kt * CK + r;
            const uint32_t dk = sK[buf] + swz<D>(r, ch), dv = sV[buf] + swz<D>(r, ch);
            if (kp <= last_key) {
                const size_t off = (((size_t)bt[kp >> 4] * p.n_kv + kvh) * 16 + (kp & 15)) * D + ch * 8;
                cp_async16(dk, p.k_pool + off);
                cp_async16(dv, p.v_pool + off);
            } else {
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dk), "r"(0));
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dv), "r"(0));
            }
        }
    };
    load_kv(0, 0);
    cp_async_commit();

    const float sl2 = rsqrtf((float)D) * LOG2E;
    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
        o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
    const int wr = warp * 16;                       // this warp's first row in the tile
    const int qpos[2] = {pos0 + q0 + wr + (lane >> 2), pos0 + q0 + wr + (lane >> 2) + 8};
    uint32_t qf[KS][4];

    for (int kt = 0; kt < n_kt; ++kt) {
        const int buf = kt & 1;
        if (kt + 1 < n_kt)
            load_kv(kt + 1, buf ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (kt == 0) {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int r = wr + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int ch = ks * 2 + (lane >> 4);
                ldsm_x4(sQ + swz<D>(r, ch), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
            }
        }
        // S = Q K^T (16 rows x 64 keys per warp)
        float s[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n)
            s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
        for (int np = 0; np < 4; ++np) {      // pairs of 8-key n-tiles
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int r = np * 16 + (lane & 7) + (lane >> 4) * 8;
                const int ch = ks * 2 + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(sK[buf] + swz<D>(r, ch), b0, b1, b2, b3);
                mma16816(s[np * 2], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b0, b1);
                mma16816(s[np * 2 + 1], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b2, b3);
            }
        }
        // mask, online softmax (log2 domain)
        float mnew[2] = {mrow[0], mrow[1]};
#pragma unroll
        for (int n = 0; n < 8; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int kp = kt * CK + n * 8 + (lane & 3) * 2 + (e & 1);
                const int hr = e >> 1;
                float v = s[n][e] * sl2;
                if (kp > qpos[hr])
                    v = -INFINITY;
                s[n][e] = v;
                mnew[hr] = fmaxf(mnew[hr], v);
            }
        }
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            mnew[hr] = fmaxf(mnew[hr], __shfl_xor_sync(0xffffffffu, mnew[hr], 1));
            mnew[hr] = fmaxf(mnew[hr], __shfl_xor_sync(0xffffffffu, mnew[hr], 2));
        }
        float corr[2], rsum[2] = {0.f, 0.f};
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const float mref = (mnew[hr] == -INFINITY) ? 0.f : mnew[hr];
            corr[hr] = exp2f(mrow[hr] - mref);
            mrow[hr] = mnew[hr];
            mnew[hr] = mref;
        }
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float pv = exp2f(s[n][e] - mnew[e >> 1]);
                s[n][e] = pv;
                rsum[e >> 1] += pv;
            }
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            rsum[hr] += __shfl_xor_sync(0xffffffffu, rsum[hr], 1);
            rsum[hr] += __shfl_xor_sync(0xffffffffu, rsum[hr], 2);
            lrow[hr] = lrow[hr] * corr[hr] + rsum[hr];
        }
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            o[n][0] *= corr[0];
            o[n][1] *= corr[0];
            o[n][2] *= corr[1];
            o[n][3] *= corr[1];
        }
        // O += P V with P = hi + lo (both bf16)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {       // 16-key steps
            const float *c0 = s[kk * 2], *c1 = s[kk * 2 + 1];
            uint32_t ah[4], al[4];
            {
                const float x[8] = {c0[0], c0[1], c0[2], c0[3], c1[0], c1[1], c1[2], c1[3]};
                float hi[8], lo[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    hi[i] = __bfloat162float(__float2bfloat16_rn(x[i]));
                    lo[i] = x[i] - hi[i];
                }
                ah[0] = pack_bf16(hi[0], hi[1]);
                ah[1] = pack_bf16(hi[2], hi[3]);
                ah[2] = pack_bf16(hi[4], hi[5]);
                ah[3] = pack_bf16(hi[6], hi[7]);
                al[0] = pack_bf16(lo[0], lo[1]);
                al[1] = pack_bf16(lo[2], lo[3]);
                al[2] = pack_bf16(lo[4], lo[5]);
                al[3] = pack_bf16(lo[6], lo[7]);
            }
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {   // pairs of 8-dim n-tiles
                const int r = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int ch = dp * 2 + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(sV[buf] + swz<D>(r, ch), b0, b1, b2, b3);
                mma16816(o[dp * 2], ah[0], ah[1], ah[2], ah[3], b0, b1);
                mma16816(o[dp * 2 + 1], ah[0], ah[1], ah[2], ah[3], b2, b3);
                mma16816(o[dp * 2], al[0], al[1], al[2], al[3], b0, b1);
                mma16816(o[dp * 2 + 1], al[0], al[1], al[2], al[3], b2, b3);
            }
        }
        __syncthreads();  // buffer `buf` is refilled two iterations later
    }
    // normalise and store
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int r = wr + (lane >> 2) + hr * 8;
        if (r >= qrows)
            continue;
        const float inv = 1.f / lrow[hr];
        bf16 *orow = p.out + ((size_t)(row0 + q0 + r) * p.n_heads + head) * D;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const int c = n * 8 + (lane & 3) * 2;
            *reinterpret_cast<__nv_bfloat162 *>(orow + c) =
                __floats2bfloat162_rn(o[n][hr * 2] * inv, o[n][hr * 2 + 1] * inv);
        }
    }
}

// ----------------------------------------------------------- decode split

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Keys [k0, k1) of split `split` of a sequence with nkeys keys: the splits
// are near-equal, 16-aligned, and depend on nkeys alone.
__device__ __forceinline__ void split_range(int nkeys, int split, int &k0, int &k1, int &n_splits)
{
    n_splits = attn_n_splits(nkeys);
    const int len = attn_split_len(nkeys);
    k0 = split * len;
    k1 = min(nkeys, k0 + len);
}

// One decode split on the tensor cores, transposed so that the single query
// is the 8-column side of each m16n8k16 product (7 of 8 columns padding,
// rather than 15 of 16 rows):
//   S^T[token] = K_block[token][:] . q      A = the block's K (16 tokens x
//                16 dims per k-step), B column 0 = q (lanes 0-3 hold it);
//   O^T[dim]  += V_block^T[dim][:] . P      A = V^T (ldmatrix .trans of the
//                block's V), B column 0 = P (hi + lo bf16 parts, so the
//                weights keep ~16 significant bits).
// Column 0 of every product lands in the lanes with (lane & 3) == 0: lane
// 4g holds tokens g and g + 8 of S^T, and dims 16 mt + g and 16 mt + g + 8
// of O^T.  The ring's blocks arrive by TMA in 16-row x 64-dim boxes with the
// 128-byte swizzle (16-byte chunk c of row r at c ^ (r & 7)), so every
// ldmatrix is free of bank conflicts.  Warp w handles blocks w, w + 4, ...
// with its own online softmax; it owns ring stages w and w + 4 and refills
// them itself, so no cross-warp handshake until the final merge.
// Shared-memory address of (row, 16-byte chunk) of a ring block stored as
// 2048-byte boxes of 16 rows x 128 bytes (64 dims) with the 128-byte swizzle.
__device__ __forceinline__ uint32_t ring_addr(uint32_t block, int row, int chunk)
{
    return block + (uint32_t)((chunk >> 3) * 2048 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

template <int D>
__device__ void decode_split(const AttnParams &p, const CUtensorMap *tmK, const CUtensorMap *tmV, int seq, int head,
                             int split, uint8_t *smem)
{
    constexpr int BLK = 16 * D * 2, STG = 2 * BLK;
    constexpr int KS = D / 16;  // k-steps of S, m-tiles of O
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int kvh = head / (p.n_heads / p.n_kv);
    const int row = p.b.seq_q0[seq];
    const int nkeys = p.b.seq_pos0[seq] + 1;
    const int *bt = p.b.bt + p.b.seq_bt[seq];
    int k0, k1, n_splits;
    split_range(nkeys, split, k0, k1, n_splits);
    const int b0 = k0 >> 4, nb = ((k1 - 1) >> 4) - b0 + 1;

    uint8_t *ring = smem;  // NSTAGE x (K block + V block), 1024-byte aligned
    uint64_t *full = (uint64_t *)(smem + NSTAGE * STG);
    volatile int *flags = (volatile int *)(full + NSTAGE);  // [0] abort, [1] last
    float *red = (float *)(flags + 4);                      // [4][2 + D]

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s)
            mbar_init(&full[s], 1);
        flags[0] = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // a decode's K/V is read once per step: evict-first keeps it from pushing
    // the weights and activations of the neighbouring kernels out of L2
    uint64_t kv_pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(kv_pol));
    auto issue = [&](int i) {
        const int s = i % NSTAGE;
        const int prow = (bt[b0 + i] * p.n_kv + kvh) * 16;  // the block's first row in the pool map
        mbar_expect_tx(&full[s], STG);
#pragma unroll
        for (int bx = 0; bx < D / 64; ++bx) {
            tma_load_2d_hint(ring + s * STG + bx * 2048, tmK, &full[s], bx * 64, prow, kv_pol);
            tma_load_2d_hint(ring + s * STG + BLK + bx * 2048, tmV, &full[s], bx * 64, prow, kv_pol);
        }
    };
    if (lane == 0)
        for (int i = warp; i < min(nb, NSTAGE); i += 4)
            issue(i);

    // q as the B operand's column 0 (lanes 0-3), zero elsewhere
    uint32_t qb[KS][2];
    {
        const unsigned int *qr =
            reinterpret_cast<const unsigned int *>(p.q + ((size_t)row * p.n_heads + head) * D);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            qb[ks][0] = g == 0 ? __ldcg(qr + 8 * ks + t4) : 0u;
            qb[ks][1] = g == 0 ? __ldcg(qr + 8 * ks + 4 + t4) : 0u;
        }
    }
    const float sl2 = rsqrtf((float)D) * LOG2E;
    float o[KS][4];
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
        o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int i = warp; i < nb; i += 4) {
        const int s = i % NSTAGE;
        if (!mbar_wait(&full[s], (uint32_t)(i / NSTAGE) & 1u, &flags[0], WAIT_NS)) {
            if (lane == 0) {
                set_dev_err(p.err, DERR_MBAR_TIMEOUT);
                flags[0] = 1;
            }
            ok = false;
            break;
        }
        const uint32_t kb = smem_u32(ring + s * STG), vb = kb + BLK;
        // tokens of this block outside [k0, k1) (a slot that may never have
        // been written): their V rows become zero, so that a weight of 0
        // never meets a NaN, and their scores -inf
        const int kbase = (b0 + i) * 16;
        const int vlo = max(0, k0 - kbase), vhi = min(16, k1 - kbase);
        if (vlo > 0 || vhi < 16) {
            for (int c = lane; c < 16 * (D / 8); c += 32) {
                const int r = c / (D / 8);
                if (r < vlo || r >= vhi)
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(ring_addr(vb, r, c % (D / 8))),
                                 "r"(0)
                                 : "memory");
            }
            __syncwarp();
        }
        // S^T = K q
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int mi = lane >> 3;
            const int r = (lane & 7) + (mi & 1) * 8, ch = 2 * ks + (mi >> 1);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(ring_addr(kb, r, ch), a0, a1, a2, a3);
            mma16816(sc, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
        }
        // online softmax over the block's 16 tokens (lanes 4g: tokens g, g + 8)
        float s0 = sc[0] * sl2, s1 = sc[2] * sl2;
        if (kbase + g < k0 || kbase + g >= k1)
            s0 = -INFINITY;
        if (kbase + g + 8 < k0 || kbase + g + 8 >= k1)
            s1 = -INFINITY;
        float mx = fmaxf(s0, s1);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mn = fmaxf(m, mx);  // finite in lanes 4g: every block has a key in range
        const float corr = exp2f(m - mn);
        const float p0 = exp2f(s0 - mn), p1 = exp2f(s1 - mn);
        float ps = p0 + p1;
        ps += __shfl_xor_sync(0xffffffffu, ps, 4);
        ps += __shfl_xor_sync(0xffffffffu, ps, 8);
        ps += __shfl_xor_sync(0xffffffffu, ps, 16);
        l = l * corr + ps;
        m = mn;
        if (__any_sync(0xffffffffu, t4 == 0 && corr != 1.f)) {
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                o[mt][0] *= corr;
                o[mt][2] *= corr;
            }
        }
        // P as the B operand's column 0: lane t4 takes tokens 2 t4, 2 t4 + 1
        // (from lanes 8 t4 and 8 t4 + 4) and 8 + 2 t4, 9 + 2 t4
        const float h0 = __bfloat162float(__float2bfloat16_rn(p0)), h1 = __bfloat162float(__float2bfloat16_rn(p1));
        const uint32_t hp = pack_bf16(h0, h1), lp = pack_bf16(p0 - h0, p1 - h1);
        const int src = 8 * t4;
        const uint32_t ha = __shfl_sync(0xffffffffu, hp, src), hb = __shfl_sync(0xffffffffu, hp, src + 4);
        const uint32_t la = __shfl_sync(0xffffffffu, lp, src), lb = __shfl_sync(0xffffffffu, lp, src + 4);
        const uint32_t bh0 = g == 0 ? __byte_perm(ha, hb, 0x5410) : 0u, bh1 = g == 0 ? __byte_perm(ha, hb, 0x7632) : 0u;
        const uint32_t bl0 = g == 0 ? __byte_perm(la, lb, 0x5410) : 0u, bl1 = g == 0 ? __byte_perm(la, lb, 0x7632) : 0u;
        // O^T += V^T P
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            const int mi = lane >> 3;
            const int r = (lane & 7) + (mi >> 1) * 8, ch = 2 * mt + (mi & 1);
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(ring_addr(vb, r, ch), a0, a1, a2, a3);
            mma16816(o[mt], a0, a1, a2, a3, bh0, bh1);
            mma16816(o[mt], a0, a1, a2, a3, bl0, bl1);
        }
        // this warp is the only reader of stage s: refill it
        if (i + NSTAGE < nb) {
            __syncwarp();
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(i + NSTAGE);
            }
        }
    }
    // merge the 4 warps
    if (lane == 0) {
        red[warp * (2 + D) + 0] = m;
        red[warp * (2 + D) + 1] = l;
    }
    if (t4 == 0) {
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            red[warp * (2 + D) + 2 + 16 * mt + g] = o[mt][0];
            red[warp * (2 + D) + 2 + 16 * mt + g + 8] = o[mt][2];
        }
    }
    __syncthreads();
    if (!ok || flags[0]) {
        // let the copies already issued land before the CTA exits
        if (lane == 0)
            for (int i = warp; i < nb; i += 4)
                mbar_wait(&full[i % NSTAGE], (uint32_t)(i / NSTAGE) & 1u, nullptr, WAIT_NS / 8);
        return;
    }
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w)
        M = fmaxf(M, red[w * (2 + D)]);
    float L = 0.f, f[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float mw = red[w * (2 + D)];
        f[w] = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
        L += red[w * (2 + D) + 1] * f[w];
    }
    // thread t < D owns output dim t
    float ov = 0.f;
    if (threadIdx.x < D)
#pragma unroll
        for (int w = 0; w < 4; ++w)
            ov += red[w * (2 + D) + 2 + threadIdx.x] * f[w];
    bf16 *orow = p.out + ((size_t)row * p.n_heads + head) * D;
    if (n_splits == 1) {
        if (threadIdx.x < D)
            orow[threadIdx.x] = f2bf(ov / L);
        return;
    }
    // partial (m, l, o) then the last split merges in split order
    const size_t slot = ((size_t)(p.part_off[seq] + split) * p.n_heads + head) * (2 + D);
    if (threadIdx.x < D)
        p.part[slot + 2 + threadIdx.x] = ov;
    if (threadIdx.x == 0) {
        p.part[slot] = M;
        p.part[slot + 1] = L;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const int old = atomicAdd(&p.counters[seq * p.n_heads + head], 1);
        flags[1] = (old == n_splits - 1);
    }
    __syncthreads();
    if (!flags[1])
        return;
    __threadfence();
    const size_t base = ((size_t)p.part_off[seq] * p.n_heads + head) * (2 + D);
    const size_t stride = (size_t)p.n_heads * (2 + D);
    float Mg = -INFINITY;
    for (int sp = 0; sp < n_splits; ++sp)
        Mg = fmaxf(Mg, __ldcg(&p.part[base + sp * stride]));
    float Lg = 0.f, og = 0.f;
    for (int sp = 0; sp < n_splits; ++sp) {
        const float ms = __ldcg(&p.part[base + sp * stride]);
        const float fs = (ms == -INFINITY) ? 0.f : exp2f(ms - Mg);
        Lg += __ldcg(&p.part[base + sp * stride + 1]) * fs;
        if (threadIdx.x < D)
            og += __ldcg(&p.part[base + sp * stride + 2 + threadIdx.x]) * fs;
    }
    if (threadIdx.x < D)
        orow[threadIdx.x] = f2bf(og / Lg);
    if (threadIdx.x == 0)
        p.counters[seq * p.n_heads + head] = 0;
}

// Chunk tiles and decode splits run as two kernels so that each gets the
// registers and shared memory it needs (the decode splits fit three CTAs on
// an SM beside a chunk tile) and the two overlap: the chunk kernel waits for
// the QKV projection, then lets the decode kernel start; the decode kernel
// reads q and the pool without a wait of its own (through L2 only, never
// L1), and its last CTA waits for the chunk kernel before exiting, so the
// next kernel, which waits for the decode kernel, sees both.
template <int D>
__global__ void __launch_bounds__(128) k_attention_chunk(AttnParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    pdl_wait();  // q and the batch's new K/V come from the previous kernel
    pdl_trigger();
    const int item = blockIdx.x / p.n_heads;
    const int head = blockIdx.x % p.n_heads;
    if (item >= p.n_chunk_items) {
        if (threadIdx.x == 0)
            set_dev_err(p.err, DERR_BAD_WORK);
        return;
    }
    chunk_tile<D>(p, p.items[2 * item], head, p.items[2 * item + 1], smem);
}

template <int D>
__global__ void __launch_bounds__(128) k_attention_decode(const __grid_constant__ CUtensorMap tmK,
                                                          const __grid_constant__ CUtensorMap tmV, AttnParams p,
                                                          int wait_first)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    if (wait_first)
        pdl_wait();  // launched right after the QKV projection
    pdl_trigger();
    const int item = p.n_chunk_items + blockIdx.x / p.n_heads;
    const int head = blockIdx.x % p.n_heads;
    if (item < p.n_items)
        decode_split<D>(p, &tmK, &tmV, p.items[2 * item], head, p.items[2 * item + 1], smem);
    else if (threadIdx.x == 0)
        set_dev_err(p.err, DERR_BAD_WORK);
    if (!wait_first && blockIdx.x == gridDim.x - 1)
        pdl_wait();  // the grid completes only after the chunk kernel
}

}  // namespace

static int chunk_smem_bytes(int D) { return CQ * 2 * D + 4 * CK * 2 * D + 1024; }  // Q + 2 x (K, V)
static int decode_smem_bytes(int D) { return NSTAGE * 64 * D + NSTAGE * 8 + 16 + 4 * (2 + D) * 4 + 1024; }

int attn_smem_bytes(int D)
{
    const int c = chunk_smem_bytes(D), d = decode_smem_bytes(D);
    return c > d ? c : d;
}

// Work list: chunk tiles (64 rows) of every sequence with more than one row,
// then the splits of every single-row sequence.  items: [n_items][2] = (seq,
// q0 or split); part_off: [n_seq] first partial slot of each sequence.
int attn_build_items(const int *seq_nq, const int *seq_pos0, int n_seq, int *items, int *part_off, int *n_chunk_items,
                     int chunk_rows)
{
    int n = 0;
    for (int s = 0; s < n_seq; ++s)
        if (seq_nq[s] > 1)
            for (int q0 = 0; q0 < seq_nq[s]; q0 += chunk_rows) {
                items[2 * n] = s;
                items[2 * n + 1] = q0;
                ++n;
            }
    *n_chunk_items = n;
    int off = 0;
    const int d0 = n;
    for (int s = 0; s < n_seq; ++s) {
        part_off[s] = off;
        if (seq_nq[s] == 1) {
            const int ns = attn_n_splits(seq_pos0[s] + 1);
            for (int sp = 0; sp < ns; ++sp) {
                items[2 * n] = s;
                items[2 * n + 1] = sp;
                ++n;
            }
            off += ns;
        }
    }
    // the decode splits longest first, so that a long split does not start
    // last and stretch the kernel's tail (stable: equal lengths keep their
    // order; a split's result and the merge order do not depend on this)
    auto split_keys = [&](int i) {
        const int nk = seq_pos0[items[2 * i]] + 1;
        const int len = attn_split_len(nk);
        return std::min(nk, (items[2 * i + 1] + 1) * len) - items[2 * i + 1] * len;
    };
    std::vector<int> order(n - d0);
    for (int i = 0; i < n - d0; ++i)
        order[i] = d0 + i;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return split_keys(a) > split_keys(b); });
    std::vector<int> sorted(2 * (n - d0));
    for (int i = 0; i < n - d0; ++i) {
        sorted[2 * i] = items[2 * order[i]];
        sorted[2 * i + 1] = items[2 * order[i] + 1];
    }
    std::copy(sorted.begin(), sorted.end(), items + 2 * d0);
    return n;
}

template <int D>
static cudaError_t launch_attention_d(const AttnParams &p, const CUtensorMap &tmK, const CUtensorMap &tmV,
                                      cudaStream_t s, bool pdl, bool skip_chunk)
{
    static bool configured = false;
    const int cs = chunk_smem_bytes(D), ds = decode_smem_bytes(D);
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k_attention_chunk<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, cs);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_attention_decode<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, ds);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    const int n_dec = p.n_items - p.n_chunk_items;
    if (p.n_chunk_items > 0 && !skip_chunk) {
        cudaError_t e = launch_kernel(pdl, k_attention_chunk<D>, dim3(p.n_chunk_items * p.n_heads), dim3(128),
                                      (size_t)cs, s, p);
        if (e != cudaSuccess)
            return e;
    }
    if (n_dec > 0) {
        // after a chunk kernel the decode kernel starts as its dependent and
        // waits at its end; alone, it waits for the QKV projection first
        const int wait_first = (p.n_chunk_items > 0 && pdl) ? 0 : 1;
        cudaError_t e = launch_kernel(pdl, k_attention_decode<D>, dim3(n_dec * p.n_heads), dim3(128), (size_t)ds, s,
                                      tmK, tmV, p, wait_first);
        if (e != cudaSuccess)
            return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_attention_hybrid(const AttnParams &p, const CUtensorMap &tmK, const CUtensorMap &tmV,
                                    cudaStream_t s, bool pdl, bool skip_chunk)
{
    if (p.n_items <= 0)
        return cudaSuccess;
    if (p.head_dim == 128)
        return launch_attention_d<128>(p, tmK, tmV, s, pdl, skip_chunk);
    if (p.head_dim == 64)
        return launch_attention_d<64>(p, tmK, tmV, s, pdl, skip_chunk);
    return cudaErrorInvalidValue;
}

}  // namespace hb
