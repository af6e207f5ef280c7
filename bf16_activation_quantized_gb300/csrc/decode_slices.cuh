// decode_slices.cuh -- the sliced decode kernel (memory-bound arm for few tokens).
//
// Decode arm.  A CTA owns one K slice (a run of whole 128-wide blocks of K)
// and a set of 128-row weight tiles (c, c + C, c + 2C, ...).  One producer warp
// streams the 8 KB (tile, group) blocks of those tiles, in order, into a ring
// of up to 16 shared-memory stages with bulk asynchronous copies completed on
// mbarriers; the ring runs across tile boundaries, so HBM never idles between
// tiles (the software pipelining of "[ROCm][Kernel] W4A16 skinny GEMM ...",
// section 2, done with an asynchronous-copy ring).  Each of the 8 consumer
// warps owns one 16-row block of a group: it waits once per group, its lanes
// read 512 consecutive bytes of each of the group's two chunks (consecutive
// lanes, consecutive bytes -- the access pattern the Q4_K decode issue on
// "gfx1151: 61.7% of Qwen3.8-27B's per-token byte budget ..." shows is needed
// to reach the memory ceiling), and it releases the stage as soon as the words
// are in registers.  The CTA's slice of X is staged once in shared memory.
//
// Each 32-bit word becomes, with one LOP3 per register, the A fragment of an
// m16n8k16 fp16 mma.sync holding 1024 + code (the magic-constant trick of that
// page's section 1, moved from bf16 to fp16, two codes per register), and one
// exact fp16x2 subtraction turns it into code - 8.  The B fragment is 8 tokens
// of X (staged as fp16 with a power-of-two shift per token, exact), so the K
// reduction across a quad of lanes happens inside the tensor core instead of a
// shuffle tree; every product is exact in fp32 and the fp32 group scale is
// applied to each group's sum.  With split-K the fp32 partials go to a
// [SPLIT_K][M][N] workspace with plain stores and a separate kernel sums the
// slices in order ("Add Triton BF16xINT4 rowwise GEMM for ROCm gfx942/gfx950",
// "Split-K without atomics"); that kernel is chained with programmatic
// dependent launch so its launch overlaps this one.
#pragma once

#include <atomic>

#include "async.cuh"
#include "common.cuh"
#include "internal.h"

namespace w4a16 {

namespace {

constexpr int kDecodeWarps = 8;                                 // consumer warps
constexpr uint32_t kMagicF16x2_1024 = 0x64006400u;              // fp16x2 {1024, 1024}
constexpr uint32_t kF16x2_1032 = 0x64086408u;                   // fp16x2 {1032, 1032} = 1024 + 8
constexpr uint32_t kF16x2_1152 = 0x64806480u;                   // fp16x2 {1152, 1152} = 1024 + 16 * 8

// fp16x2 a - b.  Exact wherever it is used here: both operands and the
// difference are integers of at most 11 significant bits.
__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
constexpr int kDecodeThreads = (kDecodeWarps + 1) * 32;         // + one producer warp
constexpr int kStageBytes = 2 * kChunkBytes;                    // one 128-wide group of a tile
constexpr int kDecodeMaxStages = 16;
constexpr int kRing = 8;   // whole-K kernel: ring slots of one group (kStageBytes) each

// Sliced kernel: groups per weight-ring stage.  One bulk copy fills a stage;
// measured on GB300, a stream of 16 KB copies with three in flight per CTA
// (two CTAs per SM) reaches 0.94-0.99 of the copy bandwidth where 8 KB
// copies reach 0.74-0.78, so slices of two or more groups copy two groups
// at a time.
__host__ __device__ constexpr int decode_stage_groups(int gps) { return gps >= 2 ? 2 : 1; }
// Ring stages the sliced kernel uses at most, and needs at least.
__host__ __device__ constexpr int decode_ring_max(int gps) { return gps >= 2 ? 6 : 8; }
__host__ __device__ constexpr int decode_ring_min(int gps) { return gps >= 2 ? 4 : 8; }

// Shared memory: the weight ring first (as many stages of
// decode_stage_groups(gps) groups as the budget leaves, at most
// decode_ring_max(gps)), then its barriers, the abort flag, the per-token
// maxima and the staged X rows of the token block.  Host and kernel size it
// from the same row count, min(8 * MT, M).
struct DecodeSmem {
    int x_stride;      // 16-bit elements per staged X row: slice + 32 (row stride = 64 B mod 128 B)
    int stages;        // ring stages
    int stage_bytes;   // bytes per ring stage
    int off_ring, off_bar, off_abort, off_xmax, off_x, total;
};

// sub: scale groups per 128-wide block (1, 2 or 4 for groups of 128, 64, 32).
__host__ __device__ inline DecodeSmem decode_smem_layout(int mt, int rows, int gps, int sub = 1) {
    DecodeSmem L;
    L.x_stride = gps * kGroup + 32;
    L.stage_bytes = decode_stage_groups(gps) * kStageBytes;
    (void)mt;
    (void)sub;
    const int rest = 2 * kDecodeMaxStages * 8 + 16 + 64 + rows * L.x_stride * 2;
    int n = (kDecodeMaxSmem - rest) / L.stage_bytes;
    L.stages = n > decode_ring_max(gps) ? decode_ring_max(gps) : n;
    L.off_ring = 0;
    L.off_bar = L.stages * L.stage_bytes;
    L.off_abort = L.off_bar + 2 * kDecodeMaxStages * 8;
    L.off_xmax = L.off_abort + 16;
    L.off_x = L.off_xmax + 64;
    L.total = L.off_x + rows * L.x_stride * 2;
    return L;
}

// Power-of-two exponent sh for a token's slice of X: x * 2^-sh puts the
// largest |x| in [2^14, 2^15), so every bf16 value down to 2^-31 of it is
// exact in fp16 (fp16 keeps 11 significant bits, bf16 has 8, and fp16
// subnormals still hold 8 bits down to 2^-17).  Clamped so that 2^-sh and
// 2^sh are normal fp32 numbers.
__device__ __forceinline__ int slice_shift(int max_abs_bits) {
    int sh = ((max_abs_bits >> 7) & 0xFF) - 127 - 14;
    return sh < -100 ? -100 : (sh > 114 ? 114 : sh);
}
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_bar_arrive(int id, int count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void consumer_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(kDecodeWarps * 32) : "memory");
}

// Pull the scale rows of weight tile `tile` (128 rows x all groups, one
// contiguous block) into L2, rounded inwards to 16 bytes so nothing outside
// the block is touched.  Every K slice of the tile asks for the whole block;
// only the first request goes to DRAM.
__device__ __forceinline__ void prefetch_tile_scales(const uint16_t *S, int tile, int N, int n_groups) {
    const size_t r0 = size_t(tile) * kTileRows;
    const size_t r1 = min(size_t(N), r0 + kTileRows);
    if (r0 >= r1) return;
    const uintptr_t lo = (reinterpret_cast<uintptr_t>(S + r0 * n_groups) + 15) & ~uintptr_t(15);
    const uintptr_t hi = reinterpret_cast<uintptr_t>(S + r1 * n_groups) & ~uintptr_t(15);
    if (hi > lo) bulk_prefetch_l2(reinterpret_cast<const void *>(lo), uint32_t(hi - lo));
}

// One weight row's GPS scales of a slice, as raw bf16 pairs (group 2i in the
// low half of word i).
template <int GPS>
struct ScaleRow {
    uint32_t w[(GPS + 1) / 2];
};

template <int GPS>
__device__ __forceinline__ ScaleRow<GPS> load_scale_row(const uint16_t *p, bool ok, bool vec) {
    ScaleRow<GPS> r;
#pragma unroll
    for (int i = 0; i < (GPS + 1) / 2; ++i) r.w[i] = 0;
    if (!ok) return r;
    if constexpr (GPS == 16) {
        if (vec) {
            asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]) : "l"(p));
            asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(r.w[4]), "=r"(r.w[5]), "=r"(r.w[6]), "=r"(r.w[7]) : "l"(p + 8));
            return r;
        }
    } else if constexpr (GPS == 8) {
        if (vec) {
            asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]) : "l"(p));
            return r;
        }
    } else if constexpr (GPS == 4) {
        if (vec) {
            asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.w[0]), "=r"(r.w[1]) : "l"(p));
            return r;
        }
    } else if constexpr (GPS == 2) {
        if (vec) {
            asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r.w[0]) : "l"(p));
            return r;
        }
    }
#pragma unroll
    for (int gi = 0; gi < GPS; ++gi) {
        unsigned short v;
        asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p + gi));
        r.w[gi / 2] |= uint32_t(v) << (16 * (gi & 1));
    }
    return r;
}

template <int GPS>
__device__ __forceinline__ float scale_of(const ScaleRow<GPS> &r, int gi) {
    return (gi & 1) ? __uint_as_float(r.w[gi / 2] & 0xFFFF0000u) : __uint_as_float(r.w[gi / 2] << 16);
}

// One weight row's NS zero points of a slice (zero-point variant), one byte
// each, four to a word (byte i % 4 of word i / 4).  vec: the first byte is
// aligned to NS bytes (NS <= 8), so one load fetches them.
template <int NS>
struct ZeroRow {
    uint32_t w[(NS + 3) / 4];
};

template <int NS>
__device__ __forceinline__ ZeroRow<NS> load_zero_row(const uint8_t *p, bool ok, bool vec) {
    ZeroRow<NS> r;
#pragma unroll
    for (int i = 0; i < (NS + 3) / 4; ++i) r.w[i] = 0;
    if (!ok) return r;
    if constexpr (NS == 8) {
        if (vec) {
            asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.w[0]), "=r"(r.w[1]) : "l"(p));
            return r;
        }
    } else if constexpr (NS == 4) {
        if (vec) {
            asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r.w[0]) : "l"(p));
            return r;
        }
    }
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        uint32_t v;
        asm volatile("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(p + i));
        r.w[i / 4] |= v << (8 * (i & 3));
    }
    return r;
}

// The zero point (low four bits) of scale group i of a row.
template <int NS>
__device__ __forceinline__ uint32_t zero_of(const ZeroRow<NS> &r, int i) {
    return (r.w[i / 4] >> (8 * (i & 3))) & 0xFu;
}

// Zero points of the rows of weight tile `tile` into L2 (as prefetch_tile_scales).
__device__ __forceinline__ void prefetch_tile_zeros(const uint8_t *Z, int tile, int N, int n_sg) {
    const size_t r0 = size_t(tile) * kTileRows;
    const size_t r1 = min(size_t(N), r0 + kTileRows);
    if (r0 >= r1) return;
    const uintptr_t lo = (reinterpret_cast<uintptr_t>(Z + r0 * n_sg) + 15) & ~uintptr_t(15);
    const uintptr_t hi = reinterpret_cast<uintptr_t>(Z + r1 * n_sg) & ~uintptr_t(15);
    if (hi > lo) bulk_prefetch_l2(reinterpret_cast<const void *>(lo), uint32_t(hi - lo));
}

// CTA (c, slice, token block): tiles c, c + C, c + 2C, ... of one K slice of
// GPS groups (GPS divides K/128, so every slice is full).  A producer warp
// streams the 8 KB (tile, group) blocks, in order, through a ring that holds
// ring_tiles tiles' worth of groups, so a group's slot is fixed within a tile.
//
// The slice of X is staged once, as fp16 x * 2^-sh per token (exact, see
// slice_shift), so the weights can be fp16 too: in fp16 two of a 16-bit
// half's four nibbles lie inside the 10-bit mantissa, so a 32-bit word gives
// its four A fragments with one shift and four LOP3s -- 1024 + code for rows
// g (nibbles at bits 0-3) and 1024 + 16 code for rows g + 8 (bits 4-7) --
// where bf16's 7-bit mantissa would need three shifts.  One fp16x2
// subtraction per fragment then removes the offset exactly: (1024 + code) -
// 1032 = code - 8 and (1024 + 16 code) - 1152 = 16 (code - 8), small integers
// that fp16 holds exactly, so every product in the MMA is exact and codes of 8
// contribute exact zeros.  Each consumer warp owns one 16-row block of a
// tile.  Per stage it waits, reads its 16 B of each chunk of the stage's
// groups, releases the stage, and per group builds the 32 A fragments and
// runs a chain of 8 MMAs from a zero accumulator, which yields
// sum_k (code_k - 8) x_k, times 16 for rows g + 8; the group's fp32 scale is
// applied to that sum.  The 1/16 and 2^sh are applied when the tile is done;
// the scale loads are issued a tile ahead, off the critical path.
//
// SUB > 1 (scale groups of 128 / SUB columns): a stage's 128-wide block has
// 32-column quarters q that are exactly k16 step q of the chain (both the
// weight words and the staged X are permuted only inside a quarter), so the
// chain is cut into SUB chains of 4 / SUB steps, each scaled by its own
// scale group's scale.
//
// kZp (zero-point variant, Z = uint8 zero points [N][K/G]): the subtracted
// offsets are 1024 + z (rows g) and 1024 + 16 z (rows g + 8), z the row's zero
// point of the chain's scale group, so the chain yields sum_k (code_k - z) x_k
// (times 16), again with exact products.
// decode_kernel and decode_zp_kernel below are the entry points.
template <int MT, int GPS, bool kSplit, int SUB, bool kZp>
__device__ __forceinline__ void
decode_body(const uint16_t *__restrict__ X, const uint8_t *__restrict__ Wp,
            const uint16_t *__restrict__ S, const uint8_t *__restrict__ Z, uint16_t *__restrict__ Y,
            float *__restrict__ ws, int M, int N, int K, int n_tiles, int wait_us, int in_flight,
            int s_vec, int z_vec, int resident, int token_blocks, int *err) {
    extern __shared__ __align__(128) unsigned char smem[];
    // Batched products: grid.z = entries x token blocks; entry b's X, W,
    // scales, Y and partial sums follow each other in memory.
    const int bz = blockIdx.z / token_blocks;
    const int zt = blockIdx.z - bz * token_blocks;
    const int n_entries = gridDim.z / token_blocks;
    X += size_t(bz) * M * K;
    Wp += size_t(bz) * n_tiles * kTileRows * (K / 2);
    S += size_t(bz) * N * (K / kGroup) * SUB;
    if (kZp) Z += size_t(bz) * N * (K / kGroup) * SUB;
    Y += size_t(bz) * M * N;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_groups = K / kGroup;
    const int n_sg = n_groups * SUB;      // scales per weight row
    constexpr int NSC = GPS * SUB;        // scales per weight row of a slice
    const int grp0 = blockIdx.y * GPS;
    const int m0 = zt * 8 * MT;
    const int rows = min(8 * MT, M - m0);
    const int C = gridDim.x;
    const int c0 = blockIdx.x;
    const int n_my = c0 < n_tiles ? (n_tiles - c0 + C - 1) / C : 0;
    const int KC = K / kChunkK;
    const int rows_alloc = min(8 * MT, M);
    const DecodeSmem L = decode_smem_layout(MT, rows_alloc, GPS, SUB);
    constexpr int SG = decode_stage_groups(GPS);     // groups per ring stage
    constexpr int SPT = GPS / SG;                    // stages per tile of the slice
    constexpr int kStage = SG * kStageBytes;         // bytes per stage (one bulk copy)
    const int NS = L.stages;                         // ring stages (the host checks the minimum)
    // A window deeper than the ring would wait on a slot's next phase before
    // issuing it: keep it within the ring.  in_flight == 0 (test only): no
    // copies at all, so every consumer wait runs out after wait_us.
    const int IF = min(in_flight, NS);
    const unsigned long long wait_ns = wait_us > 0 ? 1000ull * unsigned(wait_us) : kWaitLimitNs;
    unsigned char *ring = smem + L.off_ring;
    const uint32_t full0 = smem_u32(smem + L.off_bar);
    const uint32_t empty0 = full0 + 8 * kDecodeMaxStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.off_abort);
    uint16_t *s_x = reinterpret_cast<uint16_t *>(smem + L.off_x);
    int *s_xmax = reinterpret_cast<int *>(smem + L.off_xmax);

    // Let the next kernel in the stream be scheduled while this grid runs.
    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kDecodeWarps);
        }
        *abort_flag = 0;
        for (int r = 0; r < 16; ++r) s_xmax[r] = 0;
        fence_barrier_init();
    }
    if (warp == kDecodeWarps && lane == 0 && n_my > 0) {
        // While the previous grid finishes, pull this CTA's first weight
        // stages into L2 (a prefetch reads nothing into the CTA and writes
        // nothing, so it needs no dependency wait); the copies after the wait
        // then hit L2.  Resident weights are copied straight away instead.
        if (!resident) {
            const uint8_t *src = Wp + (size_t(c0) * KC + size_t(2 * grp0)) * kChunkBytes;
            const size_t tile_step = size_t(C) * KC * kChunkBytes;
            const int first = min(n_my * SPT, NS);
            for (int q = 0; q < first; ++q)
                bulk_prefetch_l2(src + (q / SPT) * tile_step + (q % SPT) * kStage, kStage);
        }
        // The scales of the first tiles (the consumers load a tile's scales
        // two tiles ahead of its use).
        for (int it = 0; it < min(n_my, 3); ++it) {
            prefetch_tile_scales(S, c0 + it * C, N, n_sg);
            if (kZp) prefetch_tile_zeros(Z, c0 + it * C, N, n_sg);
        }
        // This CTA's slice of X (a prefetch only warms L2; where the previous
        // kernel writes X, the loads after the dependency wait see its data).
        for (int r = 0; r < rows; ++r)
            bulk_prefetch_l2(X + size_t(m0 + r) * K + size_t(grp0) * kGroup, uint32_t(GPS * kGroup * 2));
    }
    __syncthreads();

    const int g = lane >> 2, t = lane & 3;
    const bool vec_scales = s_vec != 0;
    ScaleRow<NSC> s_cur[2], s_next[2];
    ZeroRow<NSC> z_cur[2], z_next[2];     // kZp only
    auto load_scales = [&](int tile, ScaleRow<NSC> (&dst)[2], ZeroRow<NSC> (&zdst)[2]) {
        const int f0 = tile * kTileRows + warp * 16 + g;
        const uint16_t *p0 = S + size_t(f0) * n_sg + grp0 * SUB;
        dst[0] = load_scale_row<NSC>(p0, f0 < N, vec_scales);
        dst[1] = load_scale_row<NSC>(p0 + 8 * size_t(n_sg), f0 + 8 < N, vec_scales);
        if constexpr (kZp) {
            const uint8_t *q0 = Z + size_t(f0) * n_sg + grp0 * SUB;
            zdst[0] = load_zero_row<NSC>(q0, f0 < N, z_vec != 0);
            zdst[1] = load_zero_row<NSC>(q0 + 8 * size_t(n_sg), f0 + 8 < N, z_vec != 0);
        }
    };
    // Read nothing that the previous grid in the stream may write before it
    // has completed: X always, and W and the scales unless they are resident
    // (then only the consumers wait, for X, and they load the first tile's
    // scales before waiting).
    if (resident && warp < kDecodeWarps && n_my > 0) load_scales(c0, s_cur, z_cur);
    if (!resident || warp < kDecodeWarps) pdl_wait();

    if (warp == kDecodeWarps) {
        // Producer warp: streams every (tile, group) block of this CTA.
        // Non-resident weights: it starts once the consumers have issued their
        // X and scale loads, so that those small reads are not queued behind
        // the weight stream.  Resident weights: it starts at once and fills
        // the ring while the previous grid finishes.
        if (!resident) named_bar_sync(2, kDecodeThreads);
        // The whole warp runs the loop (warp-uniform values); one elected
        // lane issues the copies and prefetches.
        const size_t tile_step = size_t(C) * KC * kChunkBytes;
        const uint8_t *src = Wp + (size_t(c0) * KC + size_t(2 * grp0)) * kChunkBytes;
        // At most IF copies are in the air at once (the ring may
        // hold more that have landed): a small burst per CTA lets the
        // first stages land early instead of all of them near the end.
        const int total = IF > 0 ? n_my * SPT : 0;     // stages
        int issued = 0, st = 0, gs = 0, lst = 0;
        uint32_t epar = 1;   // parity of the empty phase to wait for (first lap: none)
        uint32_t lpar = 0;   // parity of the full phase of copy q - IF
        for (int q = 0; q < total; ++q) {
            if (q >= NS && !__all_sync(0xffffffffu, mbar_wait(empty0 + 8 * st, epar, abort_flag, err, wait_ns)))
                break;
            if (q >= IF) {
                if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * lst, lpar, abort_flag, err, wait_ns))) break;
                if (++lst == NS) { lst = 0; lpar ^= 1; }
            }
            if (elect_one()) {
                mbar_arrive_expect_tx(full0 + 8 * st, kStage);
                bulk_g2s(smem_u32(ring + st * kStage), src + gs * kStage, kStage, full0 + 8 * st);
            }
            __syncwarp();
            ++issued;
            if (++gs == SPT) {
                gs = 0;
                src += tile_step;
                // Entering tile (q + 1) / SPT: warm L2 with the scales of the
                // tile three ahead, which the consumers load about two tiles later.
                const int ahead = (q + 1) / SPT + 3;
                if (ahead < n_my && elect_one()) {
                    prefetch_tile_scales(S, c0 + ahead * C, N, n_sg);
                    if (kZp) prefetch_tile_zeros(Z, c0 + ahead * C, N, n_sg);
                }
                __syncwarp();
            }
            if (++st == NS) { st = 0; epar ^= 1; }
        }
        if (*abort_flag) {
            for (int q = issued > NS ? issued - NS : 0; q < issued; ++q)
                drain_wait(full0 + 8 * (q % NS), (q / NS) & 1);
        }
        return;
    }


    // Consumers: stage X[m0 .. m0+rows)[slice], permuted so that a lane's B
    // fragments for word pair q of a group are 16 contiguous bytes: natural
    // column cc of a group (chunk h, 16-column slice s, quad t, element e) goes
    // to 32 (2h + s/2) + 8t + 4 (s % 2) + e.  All of a thread's loads are
    // issued before the first store, so their latencies overlap.
    // A vector's two 8-byte halves go to pos and pos + 8; lanes of the second
    // chunk (h = 1) store them in the other order, so each store instruction
    // of a warp covers every bank once per 128 bytes.  The row maximum of |x|
    // is reduced across the lanes of a row before one shared atomic.
    constexpr int vec_per_row = GPS * (kGroup / 8);
    constexpr int lanes_per_row = vec_per_row < 32 ? vec_per_row : 32;
    constexpr int kVecPerThread = (8 * MT * vec_per_row + kDecodeWarps * 32 - 1) / (kDecodeWarps * 32);
    const int n_vec = rows * vec_per_row;
    uint4 xval[kVecPerThread];
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
        const int i = threadIdx.x + k * kDecodeWarps * 32;
        if (i < n_vec) {
            const int r = i / vec_per_row, v = i - r * vec_per_row;
            xval[k] = ldg_nc16(X + size_t(m0 + r) * K + size_t(grp0) * kGroup + v * 8);
        }
    }
    if (!resident) {
        // Scales of rows g and g+8 of this warp's block for the first tile,
        // issued before the weight stream starts.
        if (n_my > 0) load_scales(c0, s_cur, z_cur);
        named_bar_arrive(2, kDecodeThreads);
    }
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
        const int i = threadIdx.x + k * kDecodeWarps * 32;
        const int r = i / vec_per_row, v = i - r * vec_per_row;
        uint32_t mx = 0;
        if (i < n_vec) {
            const uint4 val = xval[k];
            const int gi = v >> 4, u = v & 15;           // 16 vectors per group
            const int h = u >> 3, s16 = (u >> 1) & 3, t0 = (u & 1) * 2;
            const int pos = gi * kGroup + 32 * (2 * h + (s16 >> 1)) + 8 * t0 + 4 * (s16 & 1);
            uint16_t *dst = s_x + r * L.x_stride + pos;
            const uint2 lo = make_uint2(val.x, val.y), hi = make_uint2(val.z, val.w);
            *reinterpret_cast<uint2 *>(dst + (h ? 8 : 0)) = h ? hi : lo;
            *reinterpret_cast<uint2 *>(dst + (h ? 0 : 8)) = h ? lo : hi;
            // bf16 magnitudes order like their bit patterns.
            const uint32_t m01 = max(val.x & 0x7FFFu, (val.x >> 16) & 0x7FFFu);
            const uint32_t m23 = max(val.y & 0x7FFFu, (val.y >> 16) & 0x7FFFu);
            const uint32_t m45 = max(val.z & 0x7FFFu, (val.z >> 16) & 0x7FFFu);
            const uint32_t m67 = max(val.w & 0x7FFFu, (val.w >> 16) & 0x7FFFu);
            mx = max(max(m01, m23), max(m45, m67));
        }
        // Whole warps take part (i < n_vec is uniform per group of lanes_per_row).
#pragma unroll
        for (int off = 1; off < lanes_per_row; off <<= 1)
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if (i < n_vec && (lane & (lanes_per_row - 1)) == 0) atomicMax(s_xmax + r, int(mx));
    }
    if (n_my > 1) load_scales(c0 + C, s_next, z_next);
    consumer_bar();
    {
        // Per (token, group): 8 lanes take 16 values each and convert them in
        // place to fp16 x * 2^-sh.
        const int pairs = rows * GPS;
        const int part = threadIdx.x & 7;
        for (int pi = threadIdx.x >> 3; pi < pairs; pi += kDecodeWarps * 32 / 8) {
            const int r = pi / GPS, gi = pi - r * GPS;
            const float down = pow2f(-slice_shift(s_xmax[r]));
            // Lane `part` takes 8-element pieces part and 8 + part, so each
            // access of 8 lanes covers 128 contiguous bytes.
            uint4 *src = reinterpret_cast<uint4 *>(s_x + r * L.x_stride + gi * kGroup) + part;
#pragma unroll
            for (int h = 0; h < 16; h += 8) {
                const uint4 q = src[h];
                const uint32_t qv[4] = {q.x, q.y, q.z, q.w};
                uint32_t hv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float lo = bf16_lo_to_f32(qv[e]), hi = bf16_hi_to_f32(qv[e]);
                    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(hv[e]) : "f"(hi * down), "f"(lo * down));
                }
                src[h] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
            }
        }
    }
    consumer_bar();

    // Fragment sources: X rows 8o + g (B).  Lanes of rows past the staged ones
    // read the last staged row instead (their tokens' columns are never stored).
    const uint16_t *xs = s_x + t * 8;
    int xrow[MT];
#pragma unroll
    for (int o = 0; o < MT; ++o) xrow[o] = min(8 * o + g, rows_alloc - 1) * L.x_stride;
    // Per-token factors of this lane's C columns (tokens 8o + 2t + e): undo the
    // slice shift, and for rows g + 8 (whose codes carry weight 16) also 1/16.
    float fac[MT][2], fac16[MT][2];
#pragma unroll
    for (int o = 0; o < MT; ++o)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = 8 * o + 2 * t + e;
            fac[o][e] = r < rows ? pow2f(slice_shift(s_xmax[r])) : 0.f;
            fac16[o][e] = 0.0625f * fac[o][e];
        }

    const unsigned char *wlane = ring + warp * kBlockBytes + lane * 16;
    // This warp's outputs of tile `it` (C fragment: {row g: tokens 2t, 2t+1},
    // {row g+8: tokens 2t, 2t+1}) to Y, or to this slice of the workspace.
    auto store_tile = [&](int it, const float (&v)[MT][4]) {
        const int f0 = (c0 + it * C) * kTileRows + warp * 16 + g;
#pragma unroll
        for (int o = 0; o < MT; ++o) {
            const int ma = m0 + 8 * o + 2 * t;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int m = ma + (r & 1);
                const int f = f0 + ((r < 2) ? 0 : 8);
                if (m < M && f < N) {
                    const size_t off = size_t(m) * N + f;
                    if (kSplit)
                        ws[(size_t(blockIdx.y) * n_entries + bz) * size_t(M) * N + off] = v[o][r];
                    else
                        Y[off] = f32_to_bf16_rn(v[o][r]);
                }
            }
        }
    };
    int failed_at = -1;   // first tile this warp could not complete (a wait ran out)
    int slot = 0;         // ring stage of the next wait, and its phase parity
    uint32_t phase = 0;
    for (int it = 0; it < n_my; ++it) {
        float acc[MT][4];
#pragma unroll
        for (int o = 0; o < MT; ++o)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[o][r] = 0.f;
#pragma unroll
        for (int gs = 0; gs < GPS; gs += SG) {
            // Warp-uniform outcome: the MMAs below need every lane.
            if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * slot, phase, abort_flag, err, wait_ns))) {
                failed_at = it;
                break;
            }
            // This lane's 16 B of both chunks of each of the stage's groups.
            const unsigned char *wsrc = wlane + slot * kStage;
            uint32_t wvs[SG][8];
#pragma unroll
            for (int gg = 0; gg < SG; ++gg) {
                const uint4 wa = *reinterpret_cast<const uint4 *>(wsrc + gg * kStageBytes);
                const uint4 wb = *reinterpret_cast<const uint4 *>(wsrc + gg * kStageBytes + kChunkBytes);
                wvs[gg][0] = wa.x; wvs[gg][1] = wa.y; wvs[gg][2] = wa.z; wvs[gg][3] = wa.w;
                wvs[gg][4] = wb.x; wvs[gg][5] = wb.y; wvs[gg][6] = wb.z; wvs[gg][7] = wb.w;
            }
            // The stage's bytes are now in registers: release it.
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * slot);
            if (++slot == NS) {
                slot = 0;
                phase ^= 1u;
            }
#pragma unroll
            for (int gg = 0; gg < SG; ++gg) {
            const int gi = gs + gg;
            const uint32_t (&wv)[8] = wvs[gg];
            // fp16 A fragments: rows g hold 1024 + code (nibble in mantissa
            // bits 0-3), rows g + 8 hold 1024 + 16 code (bits 4-7), so one
            // shift per word serves both halves of the upper byte pair.
            uint32_t af[8][4];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t w8 = wv[j] >> 8;
                af[j][0] = lop3_and_or(wv[j], 0x000F000Fu, kMagicF16x2_1024);
                af[j][1] = lop3_and_or(wv[j], 0x00F000F0u, kMagicF16x2_1024);
                af[j][2] = lop3_and_or(w8, 0x000F000Fu, kMagicF16x2_1024);
                af[j][3] = lop3_and_or(w8, 0x00F000F0u, kMagicF16x2_1024);
            }
#pragma unroll
            for (int j = 0; j < SUB; ++j) {
                // Scales of rows g (C elements 0, 1) and g + 8 (2, 3) for
                // scale group gi * SUB + j, loaded a tile ahead.
                const float s0 = scale_of<NSC>(s_cur[0], gi * SUB + j);
                const float s1 = scale_of<NSC>(s_cur[1], gi * SUB + j);
                // Offsets of rows g and g + 8 as fp16x2 pairs.
                uint32_t off0 = kF16x2_1032, off1 = kF16x2_1152;
                if constexpr (kZp) {
                    off0 = (0x6400u | zero_of<NSC>(z_cur[0], gi * SUB + j)) * 0x10001u;
                    off1 = (0x6400u | (zero_of<NSC>(z_cur[1], gi * SUB + j) << 4)) * 0x10001u;
                }
                // The exact A operands of this chain: code - offset.
#pragma unroll
                for (int w = j * (8 / SUB); w < (j + 1) * (8 / SUB); ++w) {
                    af[w][0] = f16x2_sub(af[w][0], off0);
                    af[w][1] = f16x2_sub(af[w][1], off1);
                    af[w][2] = f16x2_sub(af[w][2], off0);
                    af[w][3] = f16x2_sub(af[w][3], off1);
                }
#pragma unroll
                for (int o = 0; o < MT; ++o) {
                    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int k16 = j * (4 / SUB); k16 < (j + 1) * (4 / SUB); ++k16) {
                        // Lanes of absent tokens read the last staged row (xrow is
                        // clamped): those values reach only absent tokens' output
                        // columns, which are never stored.
                        const uint4 xv = *reinterpret_cast<const uint4 *>(xs + xrow[o] + gi * kGroup + 32 * k16);
                        mma_16816_f16_acc(c, af[2 * k16], xv.x, xv.y);
                        mma_16816_f16_acc(c, af[2 * k16 + 1], xv.z, xv.w);
                    }
                    acc[o][0] = fmaf(s0, c[0], acc[o][0]);
                    acc[o][1] = fmaf(s0, c[1], acc[o][1]);
                    acc[o][2] = fmaf(s1, c[2], acc[o][2]);
                    acc[o][3] = fmaf(s1, c[3], acc[o][3]);
                }
            }
            }   // gg
        }
        if (failed_at >= 0) break;
#pragma unroll
        for (int o = 0; o < MT; ++o) {
            acc[o][0] *= fac[o][0];
            acc[o][1] *= fac[o][1];
            acc[o][2] *= fac16[o][0];
            acc[o][3] *= fac16[o][1];
        }
        store_tile(it, acc);
        s_cur[0] = s_next[0];
        s_cur[1] = s_next[1];
        if (kZp) {
            z_cur[0] = z_next[0];
            z_cur[1] = z_next[1];
        }
        if (it + 2 < n_my) load_scales(c0 + (it + 2) * C, s_next, z_next);
    }
    if (failed_at >= 0) {
        // The CTA is aborting: this warp's remaining outputs become NaN, so
        // the result of an incomplete call is never a plausible number (the
        // error word holds kErrWaitTimeout).
        float nan4[MT][4];
#pragma unroll
        for (int o = 0; o < MT; ++o)
#pragma unroll
            for (int r = 0; r < 4; ++r) nan4[o][r] = __int_as_float(0x7fc00000);
        for (int it = failed_at; it < n_my; ++it) store_tile(it, nan4);
    }
}

template <int MT, int GPS, bool kSplit, int SUB>
__global__ void __launch_bounds__(kDecodeThreads, 2)
decode_kernel(const uint16_t *__restrict__ X, const uint8_t *__restrict__ Wp,
              const uint16_t *__restrict__ S, uint16_t *__restrict__ Y, float *__restrict__ ws,
              int M, int N, int K, int n_tiles, int wait_us, int in_flight, int s_vec,
              int resident, int token_blocks, int *err) {
    decode_body<MT, GPS, kSplit, SUB, false>(X, Wp, S, nullptr, Y, ws, M, N, K, n_tiles, wait_us,
                                             in_flight, s_vec, 0, resident, token_blocks, err);
}

template <int MT, int GPS, bool kSplit, int SUB>
__global__ void __launch_bounds__(kDecodeThreads, 2)
decode_zp_kernel(const uint16_t *__restrict__ X, const uint8_t *__restrict__ Wp,
                 const uint16_t *__restrict__ S, const uint8_t *__restrict__ Z,
                 uint16_t *__restrict__ Y, float *__restrict__ ws, int M, int N, int K, int n_tiles,
                 int wait_us, int in_flight, int s_vec, int z_vec, int resident, int token_blocks,
                 int *err) {
    decode_body<MT, GPS, kSplit, SUB, true>(X, Wp, S, Z, Y, ws, M, N, K, n_tiles, wait_us,
                                            in_flight, s_vec, z_vec, resident, token_blocks, err);
}

// Z != nullptr: the zero-point kernel (instantiated with kZp).
template <int MT, int GPS, bool kSplit, int SUB, bool kZp>
cudaError_t launch_decode_t(const DecodePlan &p, const uint16_t *X, const uint8_t *Wp,
                            const uint16_t *S, const uint8_t *Z, uint16_t *Y, float *ws,
                            bool resident, int M, int N, int K, cudaStream_t s) {
    const int smem = decode_smem_layout(MT, M < 8 * MT ? M : 8 * MT, GPS, SUB).total;
    auto kern = [] {
        if constexpr (kZp) return decode_zp_kernel<MT, GPS, kSplit, SUB>;
        else return decode_kernel<MT, GPS, kSplit, SUB>;
    }();
    if (smem > 48 * 1024) {
        // Opt in to more than 48 KB of shared memory once per device (not a
        // stream operation, so it is also safe while a graph is being captured).
        static std::atomic<unsigned long long> opted{0};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const unsigned long long bit = 1ull << (dev & 63);
        if (!(opted.load(std::memory_order_acquire) & bit)) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecodeMaxSmem);
            if (e != cudaSuccess) return e;
            opted.fetch_or(bit, std::memory_order_acq_rel);
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.ctas_per_slice, p.split_k, p.token_blocks * p.batch);
    cfg.blockDim = dim3(kDecodeThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int *err = device_error_word();
    if (!err) return cudaErrorUnknown;
    // A slice's scales of one row (GPS * SUB of them) start at a multiple of
    // GPS * SUB elements, in every batch entry.
    const int s_vec = (reinterpret_cast<uintptr_t>(S) % (2 * GPS * SUB)) == 0;
    if constexpr (kZp) {
        const int z_vec = (reinterpret_cast<uintptr_t>(Z) % (GPS * SUB)) == 0;
        return cudaLaunchKernelEx(&cfg, kern, X, Wp, S, Z, Y, ws, M, N, K, p.n_tiles, p.wait_us,
                                  p.in_flight, s_vec, z_vec, int(resident), p.token_blocks, err);
    } else {
        return cudaLaunchKernelEx(&cfg, kern, X, Wp, S, Y, ws, M, N, K, p.n_tiles, p.wait_us,
                                  p.in_flight, s_vec, int(resident), p.token_blocks, err);
    }
}

// A slice's scales of one row stay in registers (two rows, this tile's and
// the next one's): at most 16 per row for one token octet, 8 for two; with
// zero points (also in registers) half of that.
template <int MT, int SUB, bool kZp>
constexpr bool decode_gps_ok(int gps) {
    return gps * SUB <= (MT == 1 ? 16 : 8) / (kZp ? 2 : 1);
}

template <int MT, bool kSplit, int SUB, bool kZp>
cudaError_t launch_decode_gps(const DecodePlan &p, const uint16_t *X, const uint8_t *Wp,
                              const uint16_t *S, const uint8_t *Z, uint16_t *Y, float *ws, bool res,
                              int M, int N, int K, cudaStream_t s) {
#define W4A16_DECODE_GPS_CASE(G)                                                                  \
    case G:                                                                                       \
        if constexpr (decode_gps_ok<MT, SUB, kZp>(G))                                             \
            return launch_decode_t<MT, G, kSplit, SUB, kZp>(p, X, Wp, S, Z, Y, ws, res, M, N, K, s); \
        return cudaErrorInvalidValue;
    switch (p.groups_per_slice) {
        W4A16_DECODE_GPS_CASE(1)
        W4A16_DECODE_GPS_CASE(2)
        W4A16_DECODE_GPS_CASE(4)
        W4A16_DECODE_GPS_CASE(8)
        W4A16_DECODE_GPS_CASE(16)
        default: return cudaErrorInvalidValue;
    }
#undef W4A16_DECODE_GPS_CASE
}

template <int SUB, bool kZp = false>
cudaError_t launch_decode_sub(const DecodePlan &p, const uint16_t *X, const uint8_t *Wp,
                              const uint16_t *S, const uint8_t *Z, uint16_t *Y, float *ws, bool res,
                              int M, int N, int K, cudaStream_t s) {
    const bool split = p.split_k > 1;
    if (p.mt == 1)
        return split ? launch_decode_gps<1, true, SUB, kZp>(p, X, Wp, S, Z, Y, ws, res, M, N, K, s)
                     : launch_decode_gps<1, false, SUB, kZp>(p, X, Wp, S, Z, Y, ws, res, M, N, K, s);
    return split ? launch_decode_gps<2, true, SUB, kZp>(p, X, Wp, S, Z, Y, ws, res, M, N, K, s)
                 : launch_decode_gps<2, false, SUB, kZp>(p, X, Wp, S, Z, Y, ws, res, M, N, K, s);
}

}  // namespace

// The instantiations for scale groups of 64 (decode_g64.cu) and 32 columns
// (decode_g32.cu), and the zero-point kernels for every group size
// (decode_zp.cu); the plan has been checked by launch_decode.
cudaError_t launch_decode_sub2(const DecodePlan &p, const uint16_t *X, const uint8_t *Wp,
                               const uint16_t *S, uint16_t *Y, float *ws, bool res, int M, int N,
                               int K, cudaStream_t s);
cudaError_t launch_decode_sub4(const DecodePlan &p, const uint16_t *X, const uint8_t *Wp,
                               const uint16_t *S, uint16_t *Y, float *ws, bool res, int M, int N,
                               int K, cudaStream_t s);
cudaError_t launch_decode_zp(const DecodePlan &p, const uint16_t *X, const uint8_t *Wp,
                             const uint16_t *S, const uint8_t *Z, uint16_t *Y, float *ws, bool res,
                             int M, int N, int K, cudaStream_t s);

}  // namespace w4a16
