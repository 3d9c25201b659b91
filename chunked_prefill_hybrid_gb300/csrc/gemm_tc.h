// gemm_tc.h -- host interface of the tcgen05 stream-K GEMM.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace hb {

// Token tiling of a batch of T rows on a CTA pair (G = 2): tg = nsub * n_sub
// columns, nsub MMAs of N = n_sub (<= 256) per k-block.
struct TcShape {
    int G, nsub, n_sub, tg;
};

// Device resources the GEMM needs (owned by the context).
struct TcRuntime {
    int num_sms = 0, max_smem = 0;
    float *ws = nullptr;      // stream-K partials
    size_t ws_floats = 0;
    int *counters = nullptr;  // per-tile arrival counters, zero between launches
    int n_counters = 0;
};

// Where each CTA of one launch left its fp32 partial tiles.  The batch's
// tokens are cut into `slabs` slabs of slab_rows rows (one slab when T <=
// TC_PAIR_MAX_T); each slab has its own group of `grid` CTA pairs and its own
// workspace region of ws_slab floats.  Units are (weight-tile pair, k-block),
// split evenly over a group's CTA pairs; tile pair p covers units
// [p*nkb, p*nkb+nkb).  CTA r of pair c of slab s holds weight tile 2p + r for
// the slab's tokens (col = token - s * slab_rows) at slot (p - first tile pair
// of c), element [col][feature % 128] of
// ws + s * ws_slab + (((c * G + r) * slots + slot) * tg) * 128, with G = 2.
struct TcPartition {
    const float *ws = nullptr;
    int grid = 0, G = 2, units = 0, nkb = 0, tg = 0, slots = 0;
    int pair = 1;
    int slabs = 1, slab_rows = 1 << 30;
    size_t ws_slab = 0;
};

// Unit row (tile pair), CTA rank and token column holding the partials of
// output (t, feature tile mt) in a partition, and that token's slab region.
__host__ __device__ inline void tc_part_loc(const TcPartition &p, int t, int mt, int &urow, int &r, int &col,
                                            const float *&ws)
{
    const int slab = p.slabs > 1 ? t / p.slab_rows : 0;
    urow = mt >> 1;
    r = mt & 1;
    col = t - slab * p.slab_rows;
    ws = p.ws + (size_t)slab * p.ws_slab;
}

// Weights in the tiled layout [n_tile][k_block][128][64] (zero padded).
size_t tiled_weight_elems(int N, int K);
// mode 0: rows as given; 1: RoPE pair permutation within heads of `a` rows;
// 2: gate/up interleave (gate rows 0..a-1, up rows a..2a-1 of src).
cudaError_t launch_tile_weights(const bf16 *src, bf16 *dst, int N, int K, int mode, int a, cudaStream_t s);
// The paged K or V pool as a TMA map of 16-row x 64-element boxes.
bool make_tmap_kv_pool(CUtensorMap *m, const void *pool, int num_blocks, int n_kv, int d);
// The tiled weights as a TMA map of boxes of box_rows (128) x 64 elements.
bool make_tmap_tiled_weights(CUtensorMap *m, const void *tiled, int N, int K, int box_rows);

// Largest token slab of one CTA pair (its TMEM holds 512 fp32 columns).  A
// launch of more rows, up to TC_PAIR_MAX_SLABS slabs, runs every slab in one
// grid, slab groups interleaved so that the pairs reading the same weight
// tile for different slabs run side by side and the weights leave HBM once.
constexpr int TC_PAIR_MAX_T = 512;
constexpr int TC_PAIR_MAX_SLABS = 4;
constexpr int TC_PAIR_MAX_ROWS = TC_PAIR_MAX_T * TC_PAIR_MAX_SLABS;
TcShape tc_pair_shape(int T);
size_t tc_pair_workspace_floats(int num_sms, int max_tokens, const int *Ns, const int *Ks, int n_shapes);

// The same product on CTA pairs with the 2-SM MMA (T <= TC_PAIR_MAX_ROWS;
// more than TC_PAIR_MAX_T rows only with ep.mode EPI_PARTIAL and no
// data-parallel tiles); tmW must use 128-row boxes.  With ep.mode EPI_PARTIAL the work is split
// stream-K and every CTA leaves fp32 partials (part says where); with a
// fused epilogue the launch is data-parallel (one whole tile pair per CTA
// pair, which tc_pair_data_parallel says is worthwhile and possible).
bool tc_pair_data_parallel(const TcRuntime &rt, int N);
// pdl: launch with programmatic stream serialization (the weight stream
// starts while the previous kernel finishes; activations are read after it).
// dp_tiles > 0 (a fused ep.mode, part given): tile pairs 0..dp_tiles-1 run
// whole on clusters 0..dp_tiles-1 with the fused epilogue, and the remaining
// tile pairs run stream-K over every cluster into partials; *part then
// describes that stream-K part alone (its tile pair 0 is tile pair dp_tiles),
// for launch_reduce_epi with the epilogue of the features from
// dp_tiles * 256 on.
// fault_wait_ns > 0 (test hook only): every wait of this launch gives up
// after fault_wait_ns, and the odd CTA of CTA pair 0 withholds its first
// weight-tile copy, so that the even CTA's wait for that stage runs out; the
// launch then records DERR_MBAR_TIMEOUT, drains, frees TMEM and returns.
cudaError_t launch_gemm_pair(const CUtensorMap &tmW, const bf16 *W_tiled, const bf16 *X, int T, int N, int K,
                             const EpiParams &ep, const TcRuntime &rt, cudaStream_t s, TcPartition *part = nullptr,
                             bool pdl = false, int dp_tiles = 0, uint64_t fault_wait_ns = 0);
// Tile pairs of an N x K product worth running as one data-parallel wave
// ahead of a stream-K rest: one per CTA pair when the product has more tile
// pairs than the GPU has CTA pairs and the rest gives every pair at least one
// k-block; else 0.
int tc_pair_dp_tiles(const TcRuntime &rt, int N, int K);

// The activations X [T][K] bf16 as a TMA map of boxes of box_rows x 64 elements.
bool make_tmap_rows(CUtensorMap *m, const void *X, int K, int T, int box_rows);

// Split-K linear op with the residual add fused (gemm_ksplit.cu), for
// products whose K is long against the GPU's CTA pairs (the O and down
// projections): a cluster of three CTA pairs owns one 256-row weight-tile
// pair, each pair a third of K; the three fp32 accumulators are summed in
// pair order through distributed shared memory and
//   out[t][n] = bf16(resid[t][n] + acc[t][n]),
//   ss[n / 128][t] = sum over the tile's 128 features of out[t][n]^2 (fp32),
// (ss: [N / 128][ss_ld], may be null).  T <= TC_PAIR_MAX_T, N % 256 == 0,
// K % 64 == 0.  Returns cudaErrorNotSupported, launching nothing, when the
// shape or the GPU's cluster occupancy does not fit; the caller then uses
// the stream-K path.
cudaError_t launch_gemm_ksplit(const CUtensorMap &tmW, const bf16 *W_tiled, const bf16 *X, int T, int N, int K,
                               const bf16 *resid, bf16 *out, float *ss, int ss_ld, int *err, const TcRuntime &rt,
                               cudaStream_t s, bool pdl);
// norm_out[t] = bf16(h[t] * rsqrt(sum_i ss[i][t] / N + eps) * gamma), the
// tiles' partial sums of squares added in tile order.
cudaError_t launch_norm_apply(const bf16 *h, const float *ss, int n_tiles, int ss_ld, const float *gamma, float eps,
                              bf16 *norm_out, int T, int N, cudaStream_t s, bool pdl);

// out = bf16(resid + sum of the partial tiles of `part`) for T x N outputs;
// if gamma: norm_out = bf16(out * rsqrt(mean(out^2) + eps) * gamma) per row.
cudaError_t launch_reduce_norm(const TcPartition &part, int T, int N, const bf16 *resid, bf16 *out,
                               const float *gamma, bf16 *norm_out, float eps, cudaStream_t s, bool pdl = false);

// Finish a partial-mode GEMM: sum each (token, 16 stored features) group's
// partials in contributor order and apply ep's fused epilogue (ep.N % 16 == 0
// except for EPI_F32).
cudaError_t launch_reduce_epi(const TcPartition &part, const EpiParams &ep, cudaStream_t s, bool pdl = false);

}  // namespace hb
