// common.cuh -- device helpers shared by the W4A16 kernels (sm_103a).
//
// Packed weight layout (layout version 2), written by pack.cu:
//   W is cut into 128-row tiles (N padded up to a multiple of 128 with code 8)
//   and 64-column K chunks.  One (tile, chunk) is 4096 contiguous bytes: eight
//   16-row blocks of 512 bytes.  Inside a block, lane L = 4*g + t (g = L/4,
//   t = L%4) owns 16 bytes = 4 words; word j covers rows {g, g+8} of the block
//   and columns k0 + 16j + 4t + {0,1,2,3} (k0 = 64 * chunk).  Nibble slots of
//   a word (bit offset: row, column offset):
//       0: g,0   4: g+8,0   8: g,2   12: g+8,2
//      16: g,1  20: g+8,1  24: g,3   28: g+8,3
//   so (w >> s) & 0x000F000F (s = 0, 4, 8, 12) picks a (k, k+1) pair of one
//   row in the two 16-bit halves.  Word j of lane (g, t) is then exactly
//   (a) the 16x256b TMEM fragment of the 16-column slice j of the block
//       ({row g: pairs 2t, 2t+1}, {row g+8: pairs 2t, 2t+1}), which the tensor
//       arm stores as the A operand of one K=16 MMA, and
//   (b) an m16n8k16 mma.sync A fragment whose K slots 2t,2t+1 / 2t+8,2t+9 map
//       to columns 16j + 4t + {0,1} / {2,3}, which the decode arm uses.
//
// Dequantisation trick ("[ROCm][Kernel] W4A16 skinny GEMM: hand-asm kernel
// for gfx1151", section 1 "Magic-constant bf16 dequant"): OR-ing a 4-bit code
// n into the bf16 pattern 0x4300 gives the bf16 value 128 + n; subtracting
// 136 is exact and leaves n - 8.  Here one LOP3 builds two such values (a
// bf16x2 register) and one bf16x2 FMA removes the 136 from both; the scale is
// applied either in fp32 after the per-group MMA sum (decode arm: exact) or by
// one bf16x2 multiply (tensor arm: one rounding of scale * (n - 8)).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace w4a16 {

constexpr int kGroup = 128;          // K elements per scale
constexpr int kTileRows = 128;       // rows per packed tile
constexpr int kChunkK = 64;          // K elements per packed chunk
constexpr int kChunkBytes = 4096;    // bytes per (tile, chunk)
constexpr int kBlockBytes = 512;     // bytes per 16-row block of a chunk
constexpr int kLayoutVersion = 2;

constexpr uint32_t kNibblePairMask = 0x000F000Fu;
constexpr uint32_t kMagic128 = 0x43004300u;      // bf16x2 {128, 128}
constexpr uint32_t kBf16x2One = 0x3F803F80u;     // bf16x2 {1, 1}
constexpr uint32_t kBf16x2Minus136 = 0xC308C308u;  // bf16x2 {-136, -136}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// bf16x2 {128 + n_lo, 128 + n_hi} from the nibbles at bits 0-3 and 16-19 of w.
__device__ __forceinline__ uint32_t magic_pair(uint32_t w) {
    return lop3_and_or(w, kNibblePairMask, kMagic128);
}

// bf16x2 a * 1 - 136, exact for a in [128, 143].
__device__ __forceinline__ uint32_t minus136(uint32_t a) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(kBf16x2One), "r"(kBf16x2Minus136));
    return d;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Exact codes minus 8 of one packed word, as the four A-fragment registers
// {row g: k0,k1}, {row g+8: k0,k1}, {row g: k2,k3}, {row g+8: k2,k3}.
__device__ __forceinline__ void dequant_word_frag(uint32_t w, uint32_t (&a)[4]) {
    a[0] = minus136(magic_pair(w));
    a[1] = minus136(magic_pair(w >> 4));
    a[2] = minus136(magic_pair(w >> 8));
    a[3] = minus136(magic_pair(w >> 12));
}

// One row's four weights of a packed word (half 0: row g, half 1: row g+8),
// scaled and rounded once to bf16: {k0,k1}, {k2,k3}.
__device__ __forceinline__ void dequant_word_row_scaled(uint32_t w, int half, uint32_t scale2,
                                                        uint32_t &p01, uint32_t &p23) {
    const uint32_t v = w >> (4 * half);
    p01 = bf16x2_mul(minus136(magic_pair(v)), scale2);
    p23 = bf16x2_mul(minus136(magic_pair(v >> 8)), scale2);
}

__device__ __forceinline__ float bf16_lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi_to_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t v) { return __uint_as_float(uint32_t(v) << 16); }

// fp32 -> bf16, round to nearest even (NaN kept quiet).
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
    return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// D += A . B for one m16n8k16 bf16 tile with fp32 accumulators.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Streaming 16-byte load that does not allocate in L1 (weights are read once).
// volatile: the load is issued where it is written, so a prefetch ring stays a
// prefetch ring instead of being sunk next to its first use.
__device__ __forceinline__ uint4 ldg_stream16(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// Read-only 16-byte load cached in L1 (activations shared by a CTA's warps).
// d = a * b + c for one m16n8k16 bf16 tile with fp32 accumulation.  Not
// volatile: a pure function of its operands, so the compiler may schedule it
// freely.
__device__ __forceinline__ void mma_16816_c(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                            uint32_t b1, const float (&c)[4]) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
          "f"(c[2]), "f"(c[3]));
}

// Same with fp16 operands.
__device__ __forceinline__ void mma_16816_f16_c(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                                uint32_t b1, const float (&c)[4]) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
          "f"(c[2]), "f"(c[3]));
}

// In place: c += A.B.
__device__ __forceinline__ void mma_16816_f16_acc(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                                  uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ldg_nc16(const void *p) {
    uint4 r;
    asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// Programmatic dependent launch: a dependent kernel waits for its
// predecessor's completion and memory flush; a primary lets dependents be
// scheduled early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace w4a16
