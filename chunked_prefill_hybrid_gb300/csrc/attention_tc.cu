// attention_tc.cu -- the prefill chunk's attention on the tcgen05 tensor
// cores (one CTA per 128 query rows x head).
//
// Semantics as in attention_hybrid.cu (Sarathi-Serve Guide, "Deep Dive:
// Mathematical Formulation and Attention Mechanics"; SARATHI summary,
// section 3.4 "Chunked-Prefills", Figure 6): chunk row i, at absolute
// position offset + i, attends to its request's keys 0..offset + i (the
// cached prefix plus the causal triangle), softmax(q.k / sqrt(d)) v.
//
// Two passes over 64-key tiles:
//   pass 1  S = Q K^T into TMEM; one thread per query row keeps the row
//           maximum m (log2 domain).
//   pass 2  S again; P = 2^(s - m), l = sum of P, P written as bf16 hi + lo
//           (P - hi) so the weights keep ~16 significant bits;
//           O += P_hi V + P_lo V in TMEM.  O / l is the output.
// Knowing m before P V avoids rescaling the TMEM accumulator.
//
// Layout: Q, K and V tiles are column blocks of 64 head dimensions
// (128-byte rows, 128-byte swizzle, 8-row atoms).  K and V tiles are
// gathered from the paged pool by TMA, one box per (16-token block, column
// block); the same layout is K-major for S = Q K^T and MN-major for
// O = P V.  Keys past the last valid one are masked by index; V rows past
// it are zeroed before P V so that leftovers in unwritten slots cannot
// reach the output through 0 * NaN.
//
//   warp 0      TMA loader (K tiles in pass 1, K and V tiles in pass 2)
//   warp 1      TMEM owner; one elected lane issues the MMAs and commits
//   warps 2..5  one thread per query row: softmax, P, and the output
// Every wait is bounded; on a timeout the CTA records an error, drains and
// returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include "attention.h"
#include "tc_ptx.cuh"

namespace hb {
namespace {

using namespace tc;

constexpr int AQ = 128;  // query rows per CTA (TMEM lanes)
constexpr int AK = 64;   // keys per tile
#ifndef ATC_STAGES
#define ATC_STAGES 2
#endif
#ifndef ATC_PBUFS
#define ATC_PBUFS 1
#endif
// K/V stages and P buffers: two stages and one P buffer keep the CTA at
// ~130 KB of shared memory, so a decode-attention CTA fits beside it.
constexpr int AST = ATC_STAGES;
constexpr int APB = ATC_PBUFS;
constexpr int AT_THREADS = 192;
constexpr uint64_t AT_WAIT_NS = 2000000000ull;
constexpr float AT_LOG2E = 1.4426950408889634f;

template <int D>
struct At {
    static constexpr int CB = D / 64;                // 64-dim column blocks
    static constexpr int QB = AQ * 128;              // one Q column block (16 KB)
    static constexpr int KB = AK * 128;              // one K or V column block (8 KB)
    static constexpr int Q_BYTES = CB * QB;
    static constexpr int STAGE = 2 * CB * KB;        // K then V
    static constexpr int P_TILE = AQ * AK * 2;       // [128 rows][64 keys] bf16
    static constexpr int SMEM = Q_BYTES + AST * STAGE + APB * 2 * P_TILE + 512 + 1024;
};

// byte offset of (row, 16-byte chunk c) in a 128-byte-swizzled tile
__device__ __forceinline__ int swz(int row, int c) { return (row >> 3) * 1024 + (row & 7) * 128 + ((c ^ (row & 7)) << 4); }

// Descriptor of an MN-major operand with 128-byte swizzle: 64-element column
// blocks `block_stride` bytes apart, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_mnmajor_sw128(uint32_t saddr, uint32_t block_stride)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((block_stride >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

__device__ __forceinline__ void tmem_ld_x16_(uint32_t taddr, uint32_t (&r)[16]) { tmem_ld_32x32b_x16(taddr, r); }

template <int D>
__global__ void __launch_bounds__(AT_THREADS, 1)
    k_attention_chunk_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         AttnParams p)
{
    using C = At<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sQ = smem;
    uint8_t *sKV = sQ + C::Q_BYTES;                   // AST x (K column blocks, V column blocks)
    uint8_t *sP = sKV + AST * C::STAGE;               // [buffer][hi, lo] P tiles
    uint64_t *kv_full = (uint64_t *)(sP + APB * 2 * C::P_TILE);
    uint64_t *kv_empty = kv_full + AST;
    uint64_t *s_full = kv_empty + AST;                // [2]
    uint64_t *s_empty = s_full + 2;                   // [2]
    uint64_t *p_full = s_empty + 2;                   // [2]
    uint64_t *p_empty = p_full + 2;                   // [2]
    uint64_t *o_full = p_empty + 2;
    uint64_t *drain = o_full + 1;
    uint32_t *tmem_slot = (uint32_t *)(drain + 1);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

    pdl_wait();  // q and the batch's new K/V come from the previous kernel
    pdl_trigger();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int item = blockIdx.x / p.n_heads;
    const int head = blockIdx.x % p.n_heads;
    if (item >= p.n_chunk_items) {
        if (threadIdx.x == 0)
            set_dev_err(p.err, DERR_BAD_WORK);
        return;
    }
    const int seq = p.items[2 * item], q0 = p.items[2 * item + 1];
    const int kvh = head / (p.n_heads / p.n_kv);
    const int row0 = p.b.seq_q0[seq], nq = p.b.seq_nq[seq], pos0 = p.b.seq_pos0[seq];
    const int *bt = p.b.bt + p.b.seq_bt[seq];
    const int qrows = min(AQ, nq - q0);
    const int last_key = pos0 + q0 + qrows - 1;  // keys 0..last_key
    const int n_kt = last_key / AK + 1;

    // ---- set-up: barriers, zeroed K/V ring (so skipped blocks hold finite
    // values), Q tile (rows past the chunk are zero), TMEM
    if (threadIdx.x == 0) {
        for (int i = 0; i < AST; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], 4);
            mbar_init(&p_full[i], 4);
            mbar_init(&p_empty[i], 1);
        }
        mbar_init(o_full, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    for (int i = threadIdx.x; i < AST * C::STAGE / 16; i += AT_THREADS)
        reinterpret_cast<uint4 *>(sKV)[i] = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < AQ * (D / 8); i += AT_THREADS) {
        const int r = i / (D / 8), ch = i % (D / 8);
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < qrows)
            v = __ldcg(reinterpret_cast<const uint4 *>(p.q + ((size_t)(row0 + q0 + r) * p.n_heads + head) * D) + ch);
        *reinterpret_cast<uint4 *>(sQ + (ch >> 3) * C::QB + swz(r, ch & 7)) = v;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> async proxy
    if (warp == 1)
        tmem_alloc(tmem_slot, 256);  // S[0] at column 0, S[1] at 64, O at 128
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ loader
        int s = 0;
        uint32_t ph = 0;
        int it = 0;
        bool ok = true;
        for (int pass = 0; pass < 2 && ok; ++pass) {
            for (int t = 0; t < n_kt; ++t, ++it) {
                if (it >= AST &&
                    !__all_sync(0xffffffffu, mbar_wait(&kv_empty[s], ph ^ 1u, abort_flag, AT_WAIT_NS))) {
                    if (lane == 0) {
                        set_dev_err(p.err, DERR_MBAR_TIMEOUT);
                        *abort_flag = 1;
                    }
                    ok = false;
                    break;
                }
                // 16-token blocks of this tile that hold keys <= last_key;
                // lane i issues box i (block, column block, K or V), so one
                // warp instruction covers the whole tile
                const int nblk = min(4, (last_key - t * AK) / 16 + 1);
                const int nbox = nblk * C::CB * (pass + 1);
                mbar_expect_tx_elect(&kv_full[s], (uint32_t)(nbox * 2048));
                __syncwarp();
                if (lane < nbox) {
                    const int j = lane % nblk, rest = lane / nblk;
                    const int cb = rest % C::CB, is_v = rest / C::CB;
                    const int row = (__ldg(bt + t * 4 + j) * p.n_kv + kvh) * 16;
                    uint8_t *dst = sKV + s * C::STAGE + is_v * C::CB * C::KB + cb * C::KB + j * 2048;
                    tma_load_2d(dst, is_v ? &tmV : &tmK, &kv_full[s], cb * 64, row);
                }
                if (++s == AST) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        // no copy may still be landing when the CTA exits
        for (int k = (it > AST ? it - AST : 0); k < it; ++k)
            mbar_wait(&kv_empty[k % AST], (uint32_t)(k / AST) & 1u, ok ? abort_flag : nullptr,
                      ok ? AT_WAIT_NS : AT_WAIT_NS / 4);
        if (!ok)
            for (int k = (it > AST ? it - AST : 0); k < it; ++k)
                mbar_wait(&kv_full[k % AST], (uint32_t)(k / AST) & 1u, nullptr, AT_WAIT_NS / 4);
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        const uint32_t id_s = idesc_bf16_f32(AQ, AK);
        const uint32_t id_o = idesc_bf16_f32(AQ, D) | (1u << 16);  // B (V) MN-major
        const uint32_t q_base = smem_u32(sQ), kv_base = smem_u32(sKV), p_base = smem_u32(sP);
        int s = 0, su = 0;  // K/V stage; S tiles issued so far
        uint32_t ph = 0;
        bool ok = true;
        auto wait_or_fail = [&](uint64_t *bar, uint32_t parity) -> bool {
            if (__all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, AT_WAIT_NS)))
                return true;
            if (lane == 0) {
                set_dev_err(p.err, DERR_MBAR_TIMEOUT);
                *abort_flag = 1;
            }
            ok = false;
            return false;
        };
        // S[su & 1] = Q K^T of the tile in stage s
        auto issue_s = [&](int stage) -> bool {
            const int b = su & 1;
            if (!wait_or_fail(&kv_full[stage], ph))
                return false;
            if (su >= 2 && !wait_or_fail(&s_empty[b], (uint32_t)((su - 2) >> 1) & 1u))
                return false;
            tc_fence_after();
            const uint32_t kst = kv_base + (uint32_t)(stage * C::STAGE);
#pragma unroll
            for (int cb = 0; cb < C::CB; ++cb)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16_elect(tmem + (uint32_t)(b * AK), sdesc_kmajor_sw128(q_base + cb * C::QB + ks * 32),
                                   sdesc_kmajor_sw128(kst + cb * C::KB + ks * 32), id_s, (cb | ks) ? 1u : 0u);
            mma_commit_elect(&s_full[b]);
            ++su;
            return true;
        };
        auto next_stage = [&]() {
            if (++s == AST) {
                s = 0;
                ph ^= 1u;
            }
        };
        // pass 1: S tiles only
        for (int t = 0; t < n_kt && ok; ++t) {
            if (!issue_s(s))
                break;
            mma_commit_elect(&kv_empty[s]);
            next_stage();
        }
        // pass 2: S of tile t+1 overlaps the softmax of tile t; then O += P V
        int s_cur = s;
        uint32_t ph_cur = ph;
        if (ok && issue_s(s))
            next_stage();
        for (int t = 0; t < n_kt && ok; ++t) {
            if (t + 1 < n_kt) {
                if (!issue_s(s))
                    break;
                next_stage();
            }
            const int pb = t % APB;
            if (!wait_or_fail(&p_full[pb], (uint32_t)(t / APB) & 1u))
                break;
            tc_fence_after();
            const uint32_t vst = kv_base + (uint32_t)(s_cur * C::STAGE + C::CB * C::KB);
#pragma unroll
            for (int part = 0; part < 2; ++part) {  // hi, then lo
                const uint32_t pt = p_base + (uint32_t)((pb * 2 + part) * C::P_TILE);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16_elect(tmem + 128u, sdesc_kmajor_sw128(pt + ks * 32),
                                   sdesc_mnmajor_sw128(vst + ks * 2048, C::KB), id_o,
                                   (t > 0 || part > 0 || ks > 0) ? 1u : 0u);
            }
            mma_commit_elect(&p_empty[pb]);
            mma_commit_elect(&kv_empty[s_cur]);
            if (++s_cur == AST) {
                s_cur = 0;
                ph_cur ^= 1u;
            }
        }
        if (ok)
            mma_commit_elect(o_full);
        else {
            mma_commit_elect(drain);
            mbar_wait(drain, 0, nullptr, AT_WAIT_NS / 4);
        }
    } else {
        // ------------------------------------------------------ softmax rows
        const int q = warp & 3;
        const int r = q * 32 + lane;  // query row (TMEM lane)
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const int qpos = min(pos0 + q0 + r, last_key);  // rows past the chunk: any finite row
        const float sl2 = rsqrtf((float)D) * AT_LOG2E;
        float m = -INFINITY, l = 0.f;
        int su = 0;
        bool ok = true;
        auto wait_or_fail = [&](uint64_t *bar, uint32_t parity) -> bool {
            if (__all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, AT_WAIT_NS * 2)))
                return true;
            if (lane == 0 && !*abort_flag) {
                set_dev_err(p.err, DERR_MBAR_TIMEOUT);
                *abort_flag = 1;
            }
            ok = false;
            return false;
        };
        // the 64 scores of this row in tile t, scaled, masked
        auto load_s = [&](int t, float (&sv)[AK]) -> bool {
            const int b = su & 1;
            if (!wait_or_fail(&s_full[b], (uint32_t)(su >> 1) & 1u))
                return false;
            tc_fence_after();
            uint32_t v[4][16];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tmem_ld_x16_(tmem + lane_base + (uint32_t)(b * AK + c * 16), v[c]);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    sv[c * 16 + j] = __uint_as_float(v[c][j]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&s_empty[b]);
            ++su;
#pragma unroll
            for (int j = 0; j < AK; ++j)
                sv[j] = (t * AK + j <= qpos) ? sv[j] * sl2 : -INFINITY;
            return true;
        };
        for (int t = 0; t < n_kt && ok; ++t) {
            float sv[AK];
            if (!load_s(t, sv))
                break;
#pragma unroll
            for (int j = 0; j < AK; ++j)
                m = fmaxf(m, sv[j]);  // finite after tile 0: key 0 is visible to every row
        }
        // pass 2
        int s_kv = n_kt % AST;  // stage of pass 2's first tile
        uint32_t ph_kv = (uint32_t)(n_kt / AST) & 1u;
        for (int t = 0; t < n_kt && ok; ++t) {
            float sv[AK];
            if (!load_s(t, sv))
                break;
            const int pb = t % APB;
            if (t >= APB && !wait_or_fail(&p_empty[pb], (uint32_t)((t - APB) / APB) & 1u))
                break;
            uint8_t *ph_tile = sP + (pb * 2) * C::P_TILE;
            uint8_t *pl_tile = ph_tile + C::P_TILE;
#pragma unroll
            for (int c = 0; c < AK / 8; ++c) {
                float hi[8], lo[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float pv = exp2f(sv[c * 8 + j] - m);
                    l += pv;
                    hi[j] = __bfloat162float(__float2bfloat16_rn(pv));
                    lo[j] = pv - hi[j];
                }
                *reinterpret_cast<uint4 *>(ph_tile + swz(r, c)) = pack8_bf16(hi);
                *reinterpret_cast<uint4 *>(pl_tile + swz(r, c)) = pack8_bf16(lo);
            }
            if (t == n_kt - 1 && (last_key + 1) % AK != 0) {
                // V rows past the last valid key: zero them (the tile's copies
                // have landed once its full barrier completed)
                if (!wait_or_fail(&kv_full[s_kv], ph_kv))
                    break;
                const int first = last_key + 1 - t * AK;
                uint8_t *vst = sKV + s_kv * C::STAGE + C::CB * C::KB;
                for (int i = q * 32 + lane; i < (AK - first) * C::CB * 8; i += 128) {
                    const int row = first + i / (C::CB * 8), rem = i % (C::CB * 8);
                    const int cb = rem / 8, c = rem % 8;
                    *reinterpret_cast<uint4 *>(vst + cb * C::KB + swz(row, c)) = make_uint4(0, 0, 0, 0);
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&p_full[pb]);
            if (++s_kv == AST) {
                s_kv = 0;
                ph_kv ^= 1u;
            }
        }
        // output row: O / l
        if (ok && wait_or_fail(o_full, 0)) {
            tc_fence_after();
            const float inv = 1.f / l;
            bf16 *orow = p.out + ((size_t)(row0 + q0 + r) * p.n_heads + head) * D;
#pragma unroll
            for (int c = 0; c < D; c += 16) {
                uint32_t v[16];
                tmem_ld_x16_(tmem + lane_base + 128u + (uint32_t)c, v);
                tmem_ld_wait();
                if (r < qrows) {
                    float o[8];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            o[j] = __uint_as_float(v[h * 8 + j]) * inv;
                        *reinterpret_cast<uint4 *>(orow + c + h * 8) = pack8_bf16(o);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

}  // namespace

int attn_tc_chunk_rows() { return AQ; }

template <int D>
static cudaError_t launch_chunk_tc_d(const AttnParams &p, const CUtensorMap &tmK, const CUtensorMap &tmV,
                                     cudaStream_t s, bool pdl)
{
    static bool configured = false;
    if (!configured) {
        cudaError_t e =
            cudaFuncSetAttribute(k_attention_chunk_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, At<D>::SMEM);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    return launch_kernel(pdl, k_attention_chunk_tc<D>, dim3(p.n_chunk_items * p.n_heads), dim3(AT_THREADS),
                         (size_t)At<D>::SMEM, s, tmK, tmV, p);
}

cudaError_t launch_attention_chunk_tc(const AttnParams &p, const CUtensorMap &tmK, const CUtensorMap &tmV,
                                      cudaStream_t s, bool pdl)
{
    if (p.n_chunk_items <= 0)
        return cudaSuccess;
    if (p.head_dim == 128)
        return launch_chunk_tc_d<128>(p, tmK, tmV, s, pdl);
    if (p.head_dim == 64)
        return launch_chunk_tc_d<64>(p, tmK, tmV, s, pdl);
    return cudaErrorInvalidValue;
}

}  // namespace hb
