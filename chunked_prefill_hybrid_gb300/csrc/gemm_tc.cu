// gemm_tc.cu -- the fused linear ops of the hybrid batch on the sm_103a
// tensor cores: acc[t][n] = sum_k X[t][k] W[n][k] for all T = C + D rows of
// the batch at once, so each weight tile is fetched once and serves the
// chunk's rows and the piggybacked decode rows together (SARATHI summary,
// section 3.4 "Decode-Maximal Batching", "How fusion works").
//
// Orientation ("swap AB"): the MMA's M dimension is 128 weight rows (output
// features), its N dimension is a tile of tokens, a multiple of 16 up to 256.
// A hybrid batch of 274 rows then runs as two 144-token tiles (5% padding)
// instead of three 128-row tiles (29% padding): the tile-quantization effect
// the pages measure (SARATHI summary, section 3.4, Figure 7) is kept small by
// sizing the token tile to T.
//
// One CTA computes one 128 x NT output tile over the whole K loop:
//   warp 0      TMA producer: W tile [128][64] and X tile [NT][64] per stage
//   warp 1      TMEM allocation; one thread issues tcgen05.mma (M=128, N=NT,
//               K=16, 4 per stage) and commits stage releases
//   warps 2..5  epilogue: tcgen05.ld of the fp32 accumulator (one TMEM lane =
//               one output feature, columns = tokens), fused epilogue
// Every mbarrier wait is bounded (wall-clock limit); on a timeout the kernel
// records an error in the device error word, drains, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "gemm_tc.h"
#include "tc_ptx.cuh"

namespace hb {

using namespace tc;

constexpr int TC_BM = 128;
constexpr int TC_BK = 64;
constexpr int TC_THREADS = 192;
constexpr uint64_t TC_WAIT_NS = 2000000000ull;  // 2 s

struct TcSmemLayout {
    int stages, nt, a_bytes, b_bytes, stage_bytes, bar_off, total;
};

__host__ __device__ inline TcSmemLayout tc_layout(int nt, int stages)
{
    TcSmemLayout L;
    L.stages = stages;
    L.nt = nt;
    L.a_bytes = TC_BM * TC_BK * 2;
    L.b_bytes = nt * TC_BK * 2;
    L.stage_bytes = L.a_bytes + L.b_bytes;
    L.bar_off = stages * L.stage_bytes;
    L.total = L.bar_off + 256 + 1024;  // barriers + alignment slack
    return L;
}

__global__ void __launch_bounds__(TC_THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, int T, int N, int K,
              int nt, int stages, uint32_t tmem_cols, EpiParams ep)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const TcSmemLayout L = tc_layout(nt, stages);
    uint64_t *full = (uint64_t *)(smem + L.bar_off);
    uint64_t *empty = full + stages;
    uint64_t *accf = empty + stages;
    uint64_t *drain = accf + 1;
    uint32_t *tmem_slot = (uint32_t *)(drain + 1);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * TC_BM, t0 = blockIdx.y * nt;
    const int nk = (K + TC_BK - 1) / TC_BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accf, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
    }
    if (warp == 1)
        tmem_alloc(tmem_slot, tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---------------- producer
        int issued = 0;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % stages;
            const uint32_t use = (uint32_t)(kb / stages);
            if (kb >= stages && !mbar_wait(&empty[s], (use & 1u) ^ 1u, abort_flag, TC_WAIT_NS)) {
                set_dev_err(ep.err, DERR_MBAR_TIMEOUT);
                *abort_flag = 1;
                break;
            }
            uint8_t *sa = smem + (size_t)s * L.stage_bytes;
            mbar_expect_tx(&full[s], (uint32_t)L.stage_bytes);
            tma_load_2d(sa, &tmW, &full[s], kb * TC_BK, m0);
            tma_load_2d(sa + L.a_bytes, &tmX, &full[s], kb * TC_BK, t0);
            issued = kb + 1;
        }
        if (*abort_flag) {
            // let the loads already in flight land before the CTA exits
            for (int kb = (issued > stages ? issued - stages : 0); kb < issued; ++kb)
                mbar_wait(&full[kb % stages], (uint32_t)(kb / stages) & 1u, nullptr, TC_WAIT_NS / 4);
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        const uint32_t idesc = idesc_bf16_f32(TC_BM, nt);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % stages;
            if (!mbar_wait(&full[s], (uint32_t)(kb / stages) & 1u, abort_flag, TC_WAIT_NS)) {
                set_dev_err(ep.err, DERR_MBAR_TIMEOUT);
                *abort_flag = 1;
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t a_base = smem_u32(smem + (size_t)s * L.stage_bytes);
            const uint32_t b_base = a_base + (uint32_t)L.a_bytes;
#pragma unroll
            for (int k = 0; k < TC_BK / 16; ++k) {
                const uint64_t ad = sdesc_kmajor_sw128(a_base + k * 32);
                const uint64_t bd = sdesc_kmajor_sw128(b_base + k * 32);
                mma_bf16(tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
            }
            mma_commit(&empty[s]);
        }
        if (ok) {
            mma_commit(accf);
        } else {
            mma_commit(drain);
            mbar_wait(drain, 0, nullptr, TC_WAIT_NS / 4);
        }
    } else if (warp >= 2) {
        // ---------------- epilogue
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        if (mbar_wait(accf, 0, abort_flag, TC_WAIT_NS * 4)) {
            tc_fence_after();
            const int row = q * 32 + lane;
            const int n = m0 + row;
            const int n_even = n & ~1;
            const bool odd = lane & 1;
            for (int c = 0; c < nt; c += 16) {
                uint32_t r[16];
                tmem_ld_32x32b_x16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float v = __uint_as_float(r[j]);
                    const float pv = __shfl_xor_sync(0xffffffffu, v, 1);
                    const int t = t0 + c + j;
                    // even lanes take even tokens, odd lanes odd tokens
                    if (t < T && (int)odd == (j & 1) && n_even < N) {
                        const float a0 = odd ? pv : v;
                        const float a1 = odd ? v : pv;
                        epi_pair(ep, t, n_even, a0, a1);
                    }
                }
            }
        } else if (!*abort_flag) {
            set_dev_err(ep.err, DERR_MBAR_TIMEOUT);
            *abort_flag = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
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

// 2D bf16 K-major map: rows x K elements, row stride K * 2 bytes, box 64 x box_rows.
bool make_tmap_kmajor(CUtensorMap *m, const void *ptr, int rows, int K, int box_rows)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)TC_BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Token tile: balanced tiles of at most 256 tokens, multiple of 16.
int tc_token_tile(int T)
{
    const int ntiles = (T + 255) / 256;
    int nt = (T + ntiles - 1) / ntiles;
    nt = (nt + 15) / 16 * 16;
    return nt < 16 ? 16 : nt;
}

static uint32_t tmem_cols_for(int nt)
{
    uint32_t c = 32;
    while (c < (uint32_t)nt)
        c <<= 1;
    return c;
}

cudaError_t launch_gemm_tc(const CUtensorMap &tmW, const bf16 *X, int T, int N_pad, int N, int K,
                           const EpiParams &ep, cudaStream_t s, int max_smem)
{
    if (T <= 0)
        return cudaSuccess;
    if (K % 8 != 0 || N_pad % TC_BM != 0)
        return cudaErrorInvalidValue;
    const int nt = tc_token_tile(T);
    CUtensorMap tmX;
    if (!make_tmap_kmajor(&tmX, X, T, K, nt))
        return cudaErrorInvalidValue;
    int stages = 8;
    while (stages > 2 && tc_layout(nt, stages).total > max_smem)
        --stages;
    const TcSmemLayout L = tc_layout(nt, stages);
    if (L.total > max_smem)
        return cudaErrorInvalidConfiguration;
    static int configured = 0;
    if (configured < L.total) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
        if (e != cudaSuccess)
            return e;
        configured = max_smem;
    }
    dim3 grid(N_pad / TC_BM, (T + nt - 1) / nt);
    k_gemm_tc<<<grid, TC_THREADS, L.total, s>>>(tmW, tmX, T, N, K, nt, stages, tmem_cols_for(nt), ep);
    return cudaGetLastError();
}

}  // namespace hb
