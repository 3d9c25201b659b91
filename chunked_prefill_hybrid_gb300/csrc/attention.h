// attention.h -- host interface of the hybrid paged-attention kernel.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace hb {

// Decode splits: a decode with n keys runs as max(1, n / ATTN_SPLIT) splits
// of near-equal length (so every split has ATTN_SPLIT..2*ATTN_SPLIT-1 keys).
// The split count depends on the context length only, so a decode's result
// does not depend on the rest of the batch.
constexpr int ATTN_SPLIT = 1024;
// Keys per split (a multiple of 16) and the number of splits; every split
// is non-empty.
__host__ __device__ inline int attn_split_len(int nkeys)
{
    const int n = nkeys / ATTN_SPLIT > 1 ? nkeys / ATTN_SPLIT : 1;
    return ((nkeys + n - 1) / n + 15) & ~15;
}
__host__ __device__ inline int attn_n_splits(int nkeys)
{
    const int len = attn_split_len(nkeys);
    return (nkeys + len - 1) / len;
}

struct AttnParams {
    BatchDev b;
    const bf16 *q;                   // [T][n_heads][d] after RoPE
    const bf16 *k_pool, *v_pool;     // [num_blocks][n_kv][16][d]
    bf16 *out;                       // [T][n_heads][d]
    int n_heads, n_kv, head_dim;
    const int *items;                // [n_items][2]
    int n_items, n_chunk_items;
    const int *part_off;             // [n_seq] first partial slot of a sequence
    float *part;                     // split partials (m, l, o[d])
    int *counters;                   // [n_seq][n_heads], zero between launches
    int *err;
};

int attn_smem_bytes(int head_dim);
// Work list: chunk tiles of chunk_rows rows (64 for the mma.sync kernel,
// attn_tc_chunk_rows() for the tcgen05 one), then the decode splits.
int attn_build_items(const int *seq_nq, const int *seq_pos0, int n_seq, int *items, int *part_off,
                     int *n_chunk_items, int chunk_rows = 64);
// Chunk tiles (mma.sync kernel, unless skip_chunk) then decode splits.
// With skip_chunk the decode kernel follows a chunk kernel launched just
// before it (launch_attention_chunk_tc).  tmK / tmV: make_tmap_kv_pool maps
// of the layer's pools, which the decode splits load from.
cudaError_t launch_attention_hybrid(const AttnParams &p, const CUtensorMap &tmK, const CUtensorMap &tmV,
                                    cudaStream_t s, bool pdl = false, bool skip_chunk = false);

// The chunk's attention on the tcgen05 tensor cores (attention_tc.cu):
// 128-row tiles; tmK / tmV: make_tmap_kv_pool maps of the layer's pools.
int attn_tc_chunk_rows();
cudaError_t launch_attention_chunk_tc(const AttnParams &p, const CUtensorMap &tmK, const CUtensorMap &tmV,
                                      cudaStream_t s, bool pdl);

}  // namespace hb
