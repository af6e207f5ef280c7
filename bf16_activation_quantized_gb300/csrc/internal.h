// internal.h -- host-side launchers shared between the C ABI and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace w4a16 {

struct DecodePlan {
    int mt;               // token octets per warp pass (1: 8 tokens, 2: 16 tokens)
    int token_blocks;     // passes over the tokens (grid.z)
    int n_tiles;          // 128-row tiles (grid.x)
    int split_k;          // K slices (grid.y)
    int groups_per_slice; // 128-wide K groups per slice
};

struct TensorPlan {
    int tile_tokens;      // MMA N: tokens per tile (16..256, multiple of 16)
    int split_k;          // K slices
    int groups_per_slice;
    int n_tiles;          // 128-row feature tiles
    int t_tiles;          // token tiles (per group for the grouped op: an upper bound)
    int ctas;             // persistent CTAs launched
    int stages;           // shared-memory ring depth
    size_t smem_bytes;
};

int device_sm_count(int *sms);  // returns cudaError_t as int

size_t packed_bytes(int N, int K);

cudaError_t launch_pack(const uint8_t *w_canon, uint8_t *w_packed, int N, int K, cudaStream_t s);
cudaError_t launch_dequant(const uint8_t *w_packed, const uint16_t *scales, void *out,
                           bool bf16_out, int N, int K, cudaStream_t s);
cudaError_t launch_decode(const DecodePlan &p, const uint16_t *X, const uint8_t *Wp,
                          const uint16_t *S, uint16_t *Y, float *ws, int M, int N, int K,
                          cudaStream_t s);
cudaError_t launch_reduce(const float *ws, uint16_t *Y, int splits, long long count, bool pdl,
                          cudaStream_t s);

}  // namespace w4a16
