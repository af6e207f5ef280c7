// pack.cu -- weight layout kernel and the dequantisation probes.
//
// pack: canonical int4 rows (byte j of row n = codes of k = 2j (bits 0-3) and
// k = 2j+1 (bits 4-7), the low-nibble / even-K pairing of "Add Triton
// BF16xINT4 rowwise GEMM for ROCm gfx942/gfx950", "Fused A-operand dot") into
// the tile/chunk/fragment layout described in common.cuh.  One thread writes
// one 32-bit word of the packed buffer, so the writes are fully coalesced; the
// four source bytes it gathers come from two rows (g and g+8).
//
// dequant probes: decode every packed word with the same register trick the
// GEMM arms use and write the dense result, so the trick can be compared bit
// for bit with the CPU reference.
#include "common.cuh"
#include "internal.h"

namespace w4a16 {

namespace {

struct WordCoord {
    int row0;   // row g of the word (row g+8 is row0 + 8)
    int k;      // first of the four columns the word covers
};

// Position of packed word `idx` (0 <= idx < N_pad*K/8) in the weight matrix.
__device__ __forceinline__ WordCoord word_coord(size_t idx, int KC) {
    const int j = int(idx & 3);
    const int lane = int((idx >> 2) & 31);
    const int block = int((idx >> 7) & 7);
    const size_t rest = idx >> 10;              // tile * KC + chunk
    const int chunk = int(rest % size_t(KC));
    const int tile = int(rest / size_t(KC));
    const int g = lane >> 2, t = lane & 3;
    WordCoord c;
    c.row0 = tile * kTileRows + block * 16 + g;
    c.k = chunk * kChunkK + 16 * j + 4 * t;
    return c;
}

__global__ void pack_kernel(const uint8_t *__restrict__ wc, uint32_t *__restrict__ wp, int N,
                            int K, size_t words) {
    const size_t idx = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= words) return;
    const WordCoord c = word_coord(idx, K / kChunkK);
    const size_t row_bytes = size_t(K) / 2;
    const int kb = c.k / 2;  // byte holding columns k, k+1 (k is a multiple of 4)
    uint32_t b0 = 0x88, b1 = 0x88, c0 = 0x88, c1 = 0x88;  // padding rows: code 8
    if (c.row0 < N) {
        b0 = wc[size_t(c.row0) * row_bytes + kb];
        b1 = wc[size_t(c.row0) * row_bytes + kb + 1];
    }
    if (c.row0 + 8 < N) {
        c0 = wc[size_t(c.row0 + 8) * row_bytes + kb];
        c1 = wc[size_t(c.row0 + 8) * row_bytes + kb + 1];
    }
    // b0 = {k: lo, k+1: hi} of row g, b1 = {k+2, k+3}; c0, c1 the same for row g+8.
    const uint32_t w = (b0 & 0xF) | ((c0 & 0xF) << 4) | ((b1 & 0xF) << 8) | ((c1 & 0xF) << 12) |
                       ((b0 >> 4) << 16) | ((c0 >> 4) << 20) | ((b1 >> 4) << 24) |
                       ((c1 >> 4) << 28);
    wp[idx] = w;
}

// Z (zero-point variant, uint8 [N][K/G], low four bits): weight =
// scale * (code - z); nullptr: code - 8.
template <bool kBf16Out>
__global__ void dequant_kernel(const uint32_t *__restrict__ wp, const uint16_t *__restrict__ S,
                               const uint8_t *__restrict__ Z, void *__restrict__ out, int N, int K,
                               int G, size_t words) {
    const size_t idx = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= words) return;
    const WordCoord c = word_coord(idx, K / kChunkK);
    const uint32_t w = wp[idx];
    // A word's four columns c.k .. c.k + 3 share one scale group (G is a
    // multiple of 4).
    const int groups = K / G;
    const int grp = c.k / G;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int row = c.row0 + 8 * half;
        if (row >= N) continue;
        const uint16_t sbits = S[size_t(row) * groups + grp];
        const size_t o = size_t(row) * K + c.k;
        const int z = Z ? int(Z[size_t(row) * groups + grp] & 0xF) : 8;
        if (kBf16Out) {
            const uint32_t s2 = uint32_t(sbits) | (uint32_t(sbits) << 16);
            uint32_t p01, p23;
            if (Z) {
                // 128 + code minus 128 + z, exact in bf16, then one rounding.
                const uint32_t v = w >> (4 * half);
                const uint32_t off = 0xC300C300u | uint32_t(z) | (uint32_t(z) << 16);
                uint32_t d01, d23;
                asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d01) : "r"(magic_pair(v)), "r"(0x3F803F80u), "r"(off));
                asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d23) : "r"(magic_pair(v >> 8)), "r"(0x3F803F80u), "r"(off));
                p01 = bf16x2_mul(d01, s2);
                p23 = bf16x2_mul(d23, s2);
            } else {
                dequant_word_row_scaled(w, half, s2, p01, p23);
            }
            uint16_t *dst = reinterpret_cast<uint16_t *>(out) + o;
            dst[0] = uint16_t(p01 & 0xFFFF);
            dst[1] = uint16_t(p01 >> 16);
            dst[2] = uint16_t(p23 & 0xFFFF);
            dst[3] = uint16_t(p23 >> 16);
        } else {
            uint32_t a[4];
            dequant_word_frag(w, a);
            const float s = bf16_bits_to_f32(sbits);
            const uint32_t q01 = a[half], q23 = a[2 + half];
            // (code - 8) + (8 - z) = code - z, exact in fp32
            const float dz = float(8 - z);
            float *dst = reinterpret_cast<float *>(out) + o;
            dst[0] = s * (bf16_lo_to_f32(q01) + dz);
            dst[1] = s * (bf16_hi_to_f32(q01) + dz);
            dst[2] = s * (bf16_lo_to_f32(q23) + dz);
            dst[3] = s * (bf16_hi_to_f32(q23) + dz);
        }
    }
}

}  // namespace

size_t packed_bytes(int N, int K) {
    const size_t n_pad = (size_t(N) + kTileRows - 1) / kTileRows * kTileRows;
    return n_pad * size_t(K) / 2;
}

cudaError_t launch_pack(const uint8_t *w_canon, uint8_t *w_packed, int N, int K, cudaStream_t s) {
    const size_t words = packed_bytes(N, K) / 4;
    const int threads = 256;
    const size_t blocks = (words + threads - 1) / threads;
    pack_kernel<<<dim3(unsigned(blocks)), threads, 0, s>>>(
        w_canon, reinterpret_cast<uint32_t *>(w_packed), N, K, words);
    return cudaGetLastError();
}

cudaError_t launch_dequant(const uint8_t *w_packed, const uint16_t *scales, void *out,
                           bool bf16_out, int N, int K, int G, cudaStream_t s, const uint8_t *Z) {
    const size_t words = packed_bytes(N, K) / 4;
    const int threads = 256;
    const size_t blocks = (words + threads - 1) / threads;
    const uint32_t *wp = reinterpret_cast<const uint32_t *>(w_packed);
    if (bf16_out)
        dequant_kernel<true><<<dim3(unsigned(blocks)), threads, 0, s>>>(wp, scales, Z, out, N, K, G, words);
    else
        dequant_kernel<false><<<dim3(unsigned(blocks)), threads, 0, s>>>(wp, scales, Z, out, N, K, G, words);
    return cudaGetLastError();
}

}  // namespace w4a16
