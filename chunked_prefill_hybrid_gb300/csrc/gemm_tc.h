// gemm_tc.h -- host interface of the tcgen05 GEMM.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace hb {

// 2D bf16 tensor map of a row-major [rows][K] matrix, box 64 x box_rows,
// 128-byte swizzle.  Returns false if the driver call is unavailable/fails.
bool make_tmap_kmajor(CUtensorMap *m, const void *ptr, int rows, int K, int box_rows);

// Token tile used for a batch of T rows.
int tc_token_tile(int T);

// acc[t][n] = sum_k X[t][k] W[n][k] on the tensor cores, then the epilogue.
// tmW: map of W [N_pad][K] with a 128-row box; X: device [T][K] bf16.
cudaError_t launch_gemm_tc(const CUtensorMap &tmW, const bf16 *X, int T, int N_pad, int N, int K,
                           const EpiParams &ep, cudaStream_t s, int max_smem);

}  // namespace hb
