// internal.h -- host-side launchers shared between the C ABI and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace w4a16 {

struct DecodePlan {
    int mt;               // token octets per warp pass (1: 8 tokens, 2: 16 tokens)
    int token_blocks;     // passes over the tokens (grid.z)
    int n_tiles;          // 128-row tiles
    int ctas_per_slice;   // grid.x: CTA c of a slice takes tiles c, c + ctas_per_slice, ...
    int split_k;          // K slices (grid.y)
    int groups_per_slice; // 128-wide K groups per slice (<= kDecodeMaxGps)
    int ring;             // weight-ring stages (decode_ring_stages: from the shared-memory layout)
    int in_flight;        // bulk copies a CTA keeps in the air (<= ring); 0 only in the
                          // test-only stall mode (no copies: every wait runs out)
    int wait_us;          // bounded-wait limit in microseconds (0: the default 2 s)
    int wk_blocks;        // > 0: whole-K kernel, each CTA owns this many 16-row blocks over all
                          // of K (split_k is 1, ctas_per_slice the grid); 0: the slice kernel
    int batch;            // independent products of this shape (batched op; 1 otherwise)
    int sub;              // scale groups per 128-wide block: 1, 2 or 4 (groups of 128, 64, 32
                          // columns); the whole-K kernel takes 1 only
};

struct TensorPlan {
    int tile_tokens;      // MMA N: tokens per tile (16..256, multiple of 16)
    int split_k;          // K slices
    int groups_per_slice;
    int n_tiles;          // 128-row feature tiles
    int t_tiles;          // token tiles (grouped op: the planning estimate; the kernel counts them)
    int ctas;             // persistent CTAs launched
    int x_stages;         // X ring depth (groups of X in shared memory)
    int w_stages;         // W ring depth (groups of packed weights in shared memory)
    int occupancy;        // CTAs per SM the resources are sized for (the planner: always 1)
    bool sep_epilogue;    // two TMEM accumulators drained by dedicated epilogue warps (occupancy 1)
    int sub;              // scale groups per 128-wide block: 1, 2 or 4 (groups of 128, 64, 32)
    size_t smem_bytes;
};

int device_sm_count(int *sms);  // returns cudaError_t as int
int *device_error_word();        // device address of the error word (nullptr on failure)

// Decode arm shared memory: the weight ring, the staged X slice and its
// per-group sums.  kDecodeMaxSmem lets two CTAs share an SM (228 KB, of which
// 1 KB per CTA is reserved).
constexpr int kDecodeMaxGps = 16;
constexpr int kDecodeMaxSmem = 113 * 1024;
int decode_smem_needed(int M, int mt, int groups_per_slice, int sub);
// Ring stages of the sliced kernel for a plan (0: the layout does not fit).
int decode_ring_stages(int M, int mt, int groups_per_slice, int sub);
// Whole-K decode kernel: whether M tokens of K fit its staging, and its launch.
bool decode_wk_fits(int M, int K, int blocks_per_cta);
cudaError_t launch_decode_wk(int blocks_per_cta, int ctas, int batch, const uint16_t *X, const uint8_t *Wp,
                             const uint16_t *S, uint16_t *Y, bool resident, int M, int N, int K,
                             cudaStream_t s);

size_t packed_bytes(int N, int K);

// A tiled TMA descriptor (cuTensorMapEncodeTiled through the runtime's driver
// entry point; element strides 1, L2 promotion 256 B, no OOB fill).
// strides_bytes has rank - 1 entries.
cudaError_t encode_tensor_map(CUtensorMap *map, CUtensorMapDataType type, int rank, const void *base,
                              const cuuint64_t *dims, const cuuint64_t *strides_bytes,
                              const cuuint32_t *box, CUtensorMapSwizzle swizzle);

cudaError_t launch_pack(const uint8_t *w_canon, uint8_t *w_packed, int N, int K, cudaStream_t s);
// G: scale group size (128, 64 or 32 columns); Z: zero points uint8 [N][K/G]
// (nullptr: the symmetric form).
cudaError_t launch_dequant(const uint8_t *w_packed, const uint16_t *scales, void *out,
                           bool bf16_out, int N, int K, int G, cudaStream_t s,
                           const uint8_t *Z = nullptr);
// resident: the weights and scales are not written by the previous kernel on
// the stream, so the weight stream may start before that kernel completes.
// Z: zero points uint8 [N][K/G] (nullptr: the symmetric form, offset 8).
cudaError_t launch_decode(const DecodePlan &p, const uint16_t *X, const uint8_t *Wp,
                          const uint16_t *S, uint16_t *Y, float *ws, bool resident, int M, int N,
                          int K, cudaStream_t s, const uint8_t *Z = nullptr);
// Tensor arm (tensor.cu).
constexpr int kTensorMaxSmem = 227 * 1024;     // per-CTA opt-in maximum
constexpr int kSmemPerSm = 228 * 1024;         // shared memory of one SM
constexpr int kSmemReservedPerCta = 1024;      // the runtime's share of each resident CTA
constexpr int kMaxGroups = 1024;
// Tensor arm: dequantiser teams (four warps each) of the plain and the
// separate-epilogue forms; the W and A rings hold one slot per team at least.
constexpr int kTensorTeamsPlain = 4;
constexpr int kTensorTeamsSep = 2;
// Dynamic shared memory a CTA may use when `occupancy` CTAs share an SM.
inline int tensor_smem_budget(int occupancy) {
    const int b = kSmemPerSm / occupancy - kSmemReservedPerCta;
    return b < kTensorMaxSmem ? b : kTensorMaxSmem;
}
size_t tensor_smem_bytes(int bt, int x_stages, int w_stages, int occupancy, int num_groups, bool sep);
int tensor_a_stages(int bt, int occupancy, bool sep);   // TMEM A ring depth (0: does not fit)
int tensor_tmem_cols(int bt, int occupancy, bool sep);  // TMEM columns a CTA allocates
// m_sizes != nullptr: grouped product; else num_groups > 1 is a batched
// product of num_groups entries of batch_rows rows (M_total = their product).
cudaError_t launch_tensor(const TensorPlan &p, const uint16_t *X, const uint8_t *Wp,
                          const uint16_t *S, uint16_t *Y, float *ws, const int32_t *m_sizes,
                          int *status, int num_groups, int M_total, int N, int K, cudaStream_t s,
                          int batch_rows = 0, const uint8_t *Z = nullptr);   // Z: zero points [groups][N][K/G]

cudaError_t launch_reduce(const float *ws, uint16_t *Y, int splits, long long count, bool pdl,
                          cudaStream_t s);

}  // namespace w4a16
