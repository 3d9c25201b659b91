// gemm_ksplit.cu -- split-K linear op with the residual add fused, for the
// O and down projections of the hybrid batch (SARATHI summary, section 5,
// Figure 10: "postproj" and the FFN's second matmul).
//
// out[t][n] = bf16(resid[t][n] + sum_k X[t][k] W[n][k]) over all T = C + D
// rows at once, like the pair GEMM (gemm_tc.cu), but with K split three ways
// inside a thread-block cluster instead of stream-K partials in global
// memory and a separate reduce pass:
//
//   * a cluster of six CTAs -- three CTA pairs -- owns one 256-row weight-
//     tile pair; pair p computes K blocks [p nkb / 3, (p + 1) nkb / 3) with
//     the 2-SM MMA (tcgen05.mma.cta_group::2) into its own TMEM, fed by TMA
//     through a ring of shared-memory stages, exactly as a pair-GEMM segment;
//   * after its last MMA each CTA writes its fp32 accumulator (128 weight
//     rows x the batch's token columns) into its now idle stage memory,
//     token-major;
//   * after a cluster barrier, CTA (p, r) finishes token rows
//     [p T / 3, (p + 1) T / 3) of its 128 features: it reads the three CTAs'
//     accumulators (r's in pairs 0, 1, 2: two of them through distributed
//     shared memory), adds them in pair order -- a fixed order, so a row's
//     result does not depend on the batch -- adds the residual, rounds to
//     bf16, stores, and writes the tile's partial sum of squares of the
//     stored values per token for the RMSNorm that follows;
//   * a second cluster barrier keeps every CTA's shared memory alive until
//     its peers have read it.
//
//   warp 0      TMA producer (own weight tile + own token halves)
//   warp 1      TMEM owner; MMA issue in the pair's even CTA
//   warps 2..5  accumulator dump (TMEM -> shared memory)
//   all warps   the reduction of the CTA's token third
// Every mbarrier wait is bounded; on a timeout the CTA records an error in
// the device error word, drains its MMAs and still reaches both cluster
// barriers, so no CTA waits for one that gave up.
#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_tc.h"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace hb {
namespace {

using namespace tc;

constexpr int KS_PAIRS = 3;          // CTA pairs of a cluster, each one third of K
constexpr int KS_CLUSTER = 2 * KS_PAIRS;
constexpr int KS_THREADS = 192;
constexpr int KS_BM = 128;           // weight rows of one CTA
constexpr int KS_BK = 64;            // K elements of one k-block
constexpr int KS_W_BYTES = KS_BM * KS_BK * 2;
constexpr int KS_CTRL = 256;         // mbarriers and the TMEM address
constexpr uint64_t KS_WAIT_NS = 2000000000ull;  // 2 s

struct KsArgs {
    int T, N, K, nkb;      // T: all rows of the launch
    int slabs, slab_rows;  // token slabs, each with its own clusters (slab s: rows s * slab_rows ..)
    int nsub, n_sub, tg;   // MMAs per k-block, tokens per MMA, token columns (nsub * n_sub)
    int stages, stage_bytes;
    const bf16 *w_tiled;   // streamed into L2 ahead of the TMA loads
    const bf16 *resid;
    bf16 *out;
    float *ss;             // [N / 128][ss_ld] or null
    int ss_ld;
    int *err;
};

__host__ __device__ inline int ks_stage_bytes(int nsub, int n_sub) { return KS_W_BYTES + nsub * (n_sub / 2) * KS_BK * 2; }

__device__ __forceinline__ void ld_cluster_v4(uint32_t addr, float (&v)[4])
{
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
                 : "r"(addr)
                 : "memory");
}

// Arrive on the mbarrier at this offset in the two CTAs of cta_mask once
// every pair MMA issued so far by this thread completes.
__device__ __forceinline__ void mma_commit_mask_elect(uint64_t *bar, uint16_t cta_mask)
{
    asm volatile(
        "{\n"
        ".reg .pred e;\n"
        "elect.sync _|e, 0xffffffff;\n"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n"
        "}\n" ::"r"(smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

__global__ void __launch_bounds__(KS_THREADS, 1)
    k_gemm_ksplit(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, KsArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int S = a.stages;
    uint64_t *full = (uint64_t *)(smem + (size_t)S * a.stage_bytes);  // [S] (the pair's even CTA counts)
    uint64_t *empty = full + S;                                       // [S]
    uint64_t *accf = empty + S;                                       // [1]
    uint64_t *drain = accf + 1;
    uint32_t *tmem_slot = (uint32_t *)(drain + 1);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = (int)cluster_ctarank();
    const int p = rank >> 1, r = rank & 1;     // K third, CTA of the pair
    const int cl = blockIdx.x / KS_CLUSTER;     // clusters of one weight-tile pair (its slabs) are adjacent
    const int mp = cl / a.slabs, slab = cl % a.slabs;
    const int xrow0 = slab * a.slab_rows;       // the slab's first row
    const int Ts = min(a.slab_rows, a.T - xrow0);
    const int tile = 2 * mp + r;                // this CTA's 128 weight rows
    const int kb0 = p * a.nkb / KS_PAIRS, kb1 = (p + 1) * a.nkb / KS_PAIRS;
    const int xhalf = a.n_sub >> 1;
    const uint16_t pair_mask = (uint16_t)(3u << (2 * p));
    pdl_trigger();

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);  // the even CTA's commit, multicast to the pair
        }
        mbar_init(accf, 1);
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
    cluster_sync();  // every CTA's barriers and TMEM exist before any copy or MMA
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t full_even = cluster_map(smem_u32(full), (uint32_t)(2 * p));
    bool failed = false;

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        const uint32_t bytes = (uint32_t)(2 * a.stage_bytes);  // both CTAs' copies land on the even CTA's barrier
        const uint64_t wpol = l2_policy_evict_first();
        const bf16 *wbase = a.w_tiled + (size_t)tile * a.nkb * KS_BM * KS_BK;
        for (int k = kb0; k < kb1 && k < kb0 + 4; ++k)
            bulk_prefetch_l2_hint_elect(wbase + (size_t)k * KS_BM * KS_BK, KS_W_BYTES, wpol);
        int s = 0, issued = 0;
        uint32_t ph = 0;
        bool waited = false;
        for (int k = kb0; k < kb1; ++k) {
            const int it = k - kb0;
            if (k + 4 < kb1)
                bulk_prefetch_l2_hint_elect(wbase + (size_t)(k + 4) * KS_BM * KS_BK, KS_W_BYTES, wpol);
            if (it >= S && !__all_sync(0xffffffffu, mbar_wait(&empty[s], ph ^ 1u, abort_flag, KS_WAIT_NS))) {
                if (lane == 0) {
                    set_dev_err(a.err, DERR_MBAR_TIMEOUT);
                    *abort_flag = 1;
                }
                failed = true;
                break;
            }
            uint8_t *sw = smem + (size_t)s * a.stage_bytes;
            const uint32_t fb = full_even + (uint32_t)(s * 8);
            if (r == 0)
                mbar_expect_tx_elect(&full[s], bytes);
            tma_load_2d_pair_hint_elect(sw, &tmW, fb, 0, (tile * a.nkb + k) * KS_BM, wpol);
            if (!waited) {
                pdl_wait();  // the activations are the previous kernel's output
                waited = true;
            }
            for (int sub = 0; sub < a.nsub; ++sub)
                tma_load_2d_pair_elect(sw + KS_W_BYTES + sub * xhalf * KS_BK * 2, &tmX, fb, k * KS_BK,
                                       xrow0 + sub * a.n_sub + r * xhalf);
            ++issued;
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (!waited)
            pdl_wait();
        // every stage this CTA filled has been consumed (the even CTA's
        // commits), so no copy into this CTA is in flight past this point
        const int n = issued;
        for (int it = (n > S ? n - S : 0); it < n; ++it)
            mbar_wait(&empty[it % S], (uint32_t)(it / S) & 1u, failed ? nullptr : abort_flag,
                      failed ? KS_WAIT_NS / 4 : KS_WAIT_NS);
    } else if (warp == 1) {
        if (r == 0) {
            // ----------------------------------------------------- MMA issue
            const uint32_t idesc = idesc_bf16_f32(2 * KS_BM, a.n_sub);
            const uint64_t desc0 = sdesc_kmajor_sw128(smem_u32(smem));
            const uint32_t stage16 = (uint32_t)a.stage_bytes >> 4;
            const uint32_t xsub16 = (uint32_t)(xhalf * KS_BK * 2) >> 4;
            int s = 0;
            uint32_t ph = 0, st16 = 0;
            bool ok = true;
            for (int k = kb0; k < kb1; ++k) {
                if (!__all_sync(0xffffffffu, mbar_wait(&full[s], ph, abort_flag, KS_WAIT_NS))) {
                    if (lane == 0) {
                        set_dev_err(a.err, DERR_MBAR_TIMEOUT);
                        *abort_flag = 1;
                    }
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t dw = desc0 + st16;
                const uint64_t dx = dw + (KS_W_BYTES >> 4);
                for (int sub = 0; sub < a.nsub; ++sub) {
#pragma unroll
                    for (int kk = 0; kk < KS_BK / 16; ++kk)
                        mma_bf16_pair_elect(tmem + (uint32_t)(sub * a.n_sub), dw + (uint32_t)(kk * 2),
                                            dx + (uint32_t)(sub * xsub16 + kk * 2), idesc,
                                            (k > kb0 || kk > 0) ? 1u : 0u);
                }
                mma_commit_mask_elect(&empty[s], pair_mask);
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                    st16 = 0;
                } else {
                    st16 += stage16;
                }
            }
            if (ok) {
                mma_commit_mask_elect(accf, pair_mask);
            } else {
                failed = true;
                mma_commit_mask_elect(drain, pair_mask);
                mbar_wait(drain, 0, nullptr, KS_WAIT_NS / 4);
            }
        }
    } else {
        // ------------------------------------------- accumulator -> shared memory
        // dump[t][f] fp32 (token-major, 128 features = 512 bytes a token) in
        // the stage memory, which no copy or MMA uses once the accumulator is
        // complete
        const int q = warp & 3;  // TMEM lane quadrant this warp may read
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        if (!__all_sync(0xffffffffu, mbar_wait(accf, 0, abort_flag, KS_WAIT_NS * 2))) {
            if (lane == 0 && !*abort_flag) {
                set_dev_err(a.err, DERR_MBAR_TIMEOUT);
                *abort_flag = 1;
            }
            failed = true;
        } else {
            tc_fence_after();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the stages' async-proxy use is over
            float *dump = (float *)smem;
            const int f = q * 32 + lane;
            for (int sub = 0; sub < a.nsub; ++sub) {
                for (int c0 = 0; c0 < a.n_sub; c0 += 32) {
                    uint32_t rr[32];
                    tmem_ld_32x32b_x16(tmem + lane_base + (uint32_t)(sub * a.n_sub + c0),
                                       *reinterpret_cast<uint32_t(*)[16]>(rr));
                    tmem_ld_32x32b_x16(tmem + lane_base + (uint32_t)(sub * a.n_sub + c0 + 16),
                                       *reinterpret_cast<uint32_t(*)[16]>(rr + 16));
                    tmem_ld_wait();
                    const int col0 = sub * a.n_sub + c0;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c0 + j < a.n_sub)
                            dump[(size_t)(col0 + j) * KS_BM + f] = __uint_as_float(rr[j]);
                }
            }
        }
    }

    // ------------------------------------------------ reduction over the cluster
    tc_fence_before();
    __syncthreads();
    const bool bad = *abort_flag != 0;  // set by every role that gave up: the same for the whole CTA
    cluster_sync();  // every CTA's accumulator is in its shared memory, visible to the cluster
    pdl_wait();      // (the producer waited already; the residual is the earlier kernels' output)
    if (!bad) {
        // CTA (p, r): token rows [t_lo, t_hi) of features tile*128 .. +127.
        // Item (t, g) = 8 features; the 16 items of a token sit in one half
        // warp, which adds up the token's sum of squares by shuffles.
        const int t_lo = p * Ts / KS_PAIRS, t_hi = (p + 1) * Ts / KS_PAIRS;
        const uint32_t own = smem_u32(smem);
        uint32_t src[KS_PAIRS];
#pragma unroll
        for (int pp = 0; pp < KS_PAIRS; ++pp)
            src[pp] = cluster_map(own, (uint32_t)(2 * pp + r));
        const int n_items = (t_hi - t_lo) * 16;
        const int n_loop = (n_items + 31) & ~31;
        for (int i = threadIdx.x; i < n_loop; i += KS_THREADS) {
            const bool live = i < n_items;
            const int t = t_lo + (i >> 4), g = i & 15;
            const int n = tile * KS_BM + g * 8;
            float ssq = 0.f;
            if (live) {
                float acc[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc[e] = 0.f;
#pragma unroll
                for (int pp = 0; pp < KS_PAIRS; ++pp) {
                    const uint32_t at = src[pp] + (uint32_t)((t * KS_BM + g * 8) * 4);
                    float v0[4], v1[4];
                    ld_cluster_v4(at, v0);
                    ld_cluster_v4(at + 16, v1);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc[e] += v0[e];
                        acc[4 + e] += v1[e];
                    }
                }
                const uint4 rv = *reinterpret_cast<const uint4 *>(a.resid + (size_t)(xrow0 + t) * a.N + n);
                const bf16 *re = reinterpret_cast<const bf16 *>(&rv);
                float o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    o[e] = bf2f(f2bf(bf2f(re[e]) + acc[e]));  // the stored bf16 value
                    ssq += o[e] * o[e];
                }
                *reinterpret_cast<uint4 *>(a.out + (size_t)(xrow0 + t) * a.N + n) = pack8_bf16(o);
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1)
                ssq += __shfl_xor_sync(0xffffffffu, ssq, off);
            if (live && g == 0 && a.ss)
                a.ss[(size_t)tile * a.ss_ld + xrow0 + t] = ssq;
        }
    }
    cluster_sync();  // no CTA leaves while a peer may still read its shared memory
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

// One CTA per token row, one thread per 8 features: the row's sum of squares
// is the tiles' partial sums added in tile order.
__global__ void __launch_bounds__(1024) k_norm_apply(const bf16 *__restrict__ h, const float *__restrict__ ss,
                                                     int n_tiles, int ss_ld, const float *__restrict__ gamma,
                                                     float eps, bf16 *__restrict__ out, int N)
{
    __shared__ float s_rs;
    pdl_trigger();
    pdl_wait();
    const int t = blockIdx.x;
    if (threadIdx.x == 0) {
        float tot = 0.f;
        for (int i = 0; i < n_tiles; ++i)
            tot += ss[(size_t)i * ss_ld + t];
        s_rs = rsqrtf(tot / (float)N + eps);
    }
    __syncthreads();
    const int n0 = threadIdx.x * 8;
    if (n0 >= N)
        return;
    const float rs = s_rs;
    const uint4 hv = *reinterpret_cast<const uint4 *>(h + (size_t)t * N + n0);
    const bf16 *he = reinterpret_cast<const bf16 *>(&hv);
    float o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        o[e] = bf2f(he[e]) * rs * gamma[n0 + e];
    *reinterpret_cast<uint4 *>(out + (size_t)t * N + n0) = pack8_bf16(o);
}

}  // namespace

cudaError_t launch_gemm_ksplit(const CUtensorMap &tmW, const bf16 *W_tiled, const bf16 *X, int T, int N, int K,
                               const bf16 *resid, bf16 *out, float *ss, int ss_ld, int *err, const TcRuntime &rt,
                               cudaStream_t s, bool pdl)
{
    if (T <= 0)
        return cudaSuccess;
    if (N % (2 * KS_BM) != 0 || K % KS_BK != 0 || K / KS_BK < KS_PAIRS || !resid || !out || (ss && ss_ld < T))
        return cudaErrorNotSupported;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm_ksplit, cudaFuncAttributeMaxDynamicSharedMemorySize, rt.max_smem);
        if (e == cudaSuccess)
            e = max_carveout((const void *)k_gemm_ksplit);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = KS_CLUSTER;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(KS_THREADS);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // The weight shape alone decides whether this path is taken, so that a
    // row's result never depends on the batch: one slab's clusters must all
    // be resident at once (one CTA per SM at any batch size).
    const int n_mpairs = N / (2 * KS_BM);
    static int max_clusters = 0;
    if (!max_clusters) {
        cfg.gridDim = dim3((unsigned)KS_CLUSTER);
        cfg.dynamicSmemBytes = (size_t)rt.max_smem;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, k_gemm_ksplit, &cfg) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = -1;
        }
        max_clusters = n;
    }
    if (max_clusters < n_mpairs)
        return cudaErrorNotSupported;
    // token slabs: as few as keep each slab's accumulator dump (tg tokens x
    // 512 bytes) within its stages
    KsArgs a = {};
    int slabs = (T + TC_PAIR_MAX_T - 1) / TC_PAIR_MAX_T, stages = 0;
    TcShape sh{};
    for (;; ++slabs) {
        if (slabs > 64)
            return cudaErrorNotSupported;
        const int rows = slabs > 1 ? ((T + slabs - 1) / slabs + 15) / 16 * 16 : T;
        sh = tc_pair_shape(rows);
        const int sb = ks_stage_bytes(sh.nsub, sh.n_sub);
        stages = 12;
        while (stages > 2 && stages * sb + KS_CTRL + 1024 > rt.max_smem)
            --stages;
        if (stages * sb + KS_CTRL + 1024 <= rt.max_smem && (size_t)sh.tg * KS_BM * 4 <= (size_t)stages * sb) {
            a.slab_rows = rows;
            a.stage_bytes = sb;
            break;
        }
    }
    a.T = T;
    a.N = N;
    a.K = K;
    a.nkb = K / KS_BK;
    a.slabs = slabs;
    a.nsub = sh.nsub;
    a.n_sub = sh.n_sub;
    a.tg = sh.tg;
    a.stages = stages;
    a.w_tiled = W_tiled;
    a.resid = resid;
    a.out = out;
    a.ss = ss;
    a.ss_ld = ss_ld;
    a.err = err;
    CUtensorMap tmX;
    if (!make_tmap_rows(&tmX, X, K, T, a.n_sub / 2))
        return cudaErrorInvalidValue;
    cfg.gridDim = dim3((unsigned)(n_mpairs * slabs * KS_CLUSTER));
    cfg.dynamicSmemBytes = (size_t)(stages * a.stage_bytes + KS_CTRL + 1024);
    if (pdl) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_gemm_ksplit, tmW, tmX, a);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_norm_apply(const bf16 *h, const float *ss, int n_tiles, int ss_ld, const float *gamma, float eps,
                              bf16 *norm_out, int T, int N, cudaStream_t s, bool pdl)
{
    if (T <= 0)
        return cudaSuccess;
    if (N % 8 != 0 || N > 8 * 1024)
        return cudaErrorInvalidValue;
    const int threads = ((N / 8) + 31) / 32 * 32;
    cudaError_t e = launch_kernel(pdl, k_norm_apply, dim3(T), dim3(threads), 0, s, h, ss, n_tiles, ss_ld, gamma, eps,
                                  norm_out, N);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace hb
