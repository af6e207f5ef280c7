// decode.cu -- memory-bound arm for few tokens, and the split-K reduce.
//
// Decode arm.  A CTA owns one K slice (a run of whole 128-wide scale groups)
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
// are in registers.  The CTA's slice of X is staged once
// in shared memory.
//
// Each 32-bit word becomes, with one LOP3 per register, the A fragment of an
// m16n8k16 bf16 mma.sync holding 128 + code (the magic-constant trick of that
// page's section 1, two codes per register).  The B fragment is 8 tokens of X,
// so the K reduction across a quad of lanes happens inside the tensor core
// instead of a shuffle tree.  The constant 128 + 8 = 136 that every weight
// carries is removed once per 128-wide group instead of once per weight:
//     sum_k (code_k - 8) x_k = sum_k (128 + code_k) x_k - 136 * sum_k x_k,
// with the per-group sums of X computed when X is staged; the products are
// exact in fp32, and the fp32 group scale is applied to the corrected partial
// sum.  With split-K the fp32 partials go to a [SPLIT_K][M][N] workspace with
// plain stores and a separate kernel sums the slices in order ("Add Triton
// BF16xINT4 rowwise GEMM for ROCm gfx942/gfx950", "Split-K without atomics");
// that kernel is chained with programmatic dependent launch so its launch
// overlaps this one.
#include <atomic>

#include "async.cuh"
#include "common.cuh"
#include "internal.h"

namespace w4a16 {

namespace {

constexpr int kDecodeWarps = 8;                                 // consumer warps
constexpr uint32_t kMagicF16x2_1024 = 0x64006400u;              // fp16x2 {1024, 1024}
constexpr int kDecodeThreads = (kDecodeWarps + 1) * 32;         // + one producer warp
constexpr int kStageBytes = 2 * kChunkBytes;                    // one 128-wide group of a tile
constexpr int kDecodeMaxStages = 16;
constexpr int kRing = 8;   // weight-ring stages in use (every layout holds at least this many)

// Shared memory: the weight ring first (as many 8 KB stages as the budget
// leaves, at most kDecodeMaxStages), then its barriers, the abort flag, the
// per-token maxima, the staged X rows of the token block and the per-group
// correction table.  Host and kernel size it from the same row count,
// min(8 * MT, M).
struct DecodeSmem {
    int x_stride;      // 16-bit elements per staged X row: slice + 32 (row stride = 64 B mod 128 B)
    int stages;
    int off_ring, off_bar, off_abort, off_xmax, off_x, off_corr, total;
};

__host__ __device__ inline DecodeSmem decode_smem_layout(int mt, int rows, int gps) {
    DecodeSmem L;
    L.x_stride = gps * kGroup + 32;
    const int corr_bytes = gps * mt * 4 * 16;        // one float4 per (group, octet, quad)
    const int rest = 2 * kDecodeMaxStages * 8 + 16 + 64 + rows * L.x_stride * 2 + corr_bytes;
    int n = (kDecodeMaxSmem - rest) / kStageBytes;
    L.stages = n > kDecodeMaxStages ? kDecodeMaxStages : n;
    L.off_ring = 0;
    L.off_bar = L.stages * kStageBytes;
    L.off_abort = L.off_bar + 2 * kDecodeMaxStages * 8;
    L.off_xmax = L.off_abort + 16;
    L.off_x = L.off_xmax + 64;
    L.off_corr = L.off_x + rows * L.x_stride * 2;
    L.total = L.off_corr + corr_bytes;
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

// Wait, ignoring the abort flag, for copies still in flight (used only when
// aborting, so that no copy lands after the CTA has exited).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > 100000000ull) break;
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
// where bf16's 7-bit mantissa would need three shifts.  Each consumer warp
// owns one 16-row block of a tile.  Per group it waits for the stage, reads
// its 16 B of each chunk, builds the 32 A fragments, releases the stage and
// runs a chain of 8 MMAs whose accumulator starts at -1032 S (rows g) or
// -1152 S (rows g + 8), S the group's scaled sum of x, so the chain yields
// sum_k (code_k - 8) x_k, times 16 for rows g + 8.  The group scales, the
// 1/16 and 2^sh are applied when the tile (or, for 16 tokens, a batch of
// groups) is done, so the scale loads -- issued a tile ahead -- are off the
// critical path.
template <int MT, int GPS, bool kSplit>
__global__ void __launch_bounds__(kDecodeThreads, 2)
decode_kernel(const uint16_t *__restrict__ X, const uint8_t *__restrict__ Wp,
              const uint16_t *__restrict__ S, uint16_t *__restrict__ Y, float *__restrict__ ws,
              int M, int N, int K, int n_tiles, int ring_stages, int in_flight, int s_vec,
              int resident, int token_blocks, int *err) {
    extern __shared__ __align__(128) unsigned char smem[];
    // Batched products: grid.z = entries x token blocks; entry b's X, W,
    // scales, Y and partial sums follow each other in memory.
    const int bz = blockIdx.z / token_blocks;
    const int zt = blockIdx.z - bz * token_blocks;
    const int n_entries = gridDim.z / token_blocks;
    X += size_t(bz) * M * K;
    Wp += size_t(bz) * n_tiles * kTileRows * (K / 2);
    S += size_t(bz) * N * (K / kGroup);
    Y += size_t(bz) * M * N;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_groups = K / kGroup;
    const int grp0 = blockIdx.y * GPS;
    const int m0 = zt * 8 * MT;
    const int rows = min(8 * MT, M - m0);
    const int C = gridDim.x;
    const int c0 = blockIdx.x;
    const int n_my = c0 < n_tiles ? (n_tiles - c0 + C - 1) / C : 0;
    const int KC = K / kChunkK;
    const int rows_alloc = min(8 * MT, M);
    const DecodeSmem L = decode_smem_layout(MT, rows_alloc, GPS);
    constexpr int NS = kRing;
    (void)ring_stages;
    // A window deeper than the ring would wait on a slot's next phase before
    // issuing it: keep it within the ring.
    const int IF = min(in_flight, NS);
    unsigned char *ring = smem + L.off_ring;
    const uint32_t full0 = smem_u32(smem + L.off_bar);
    const uint32_t empty0 = full0 + 8 * kDecodeMaxStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.off_abort);
    uint16_t *s_x = reinterpret_cast<uint16_t *>(smem + L.off_x);
    float *s_corr = reinterpret_cast<float *>(smem + L.off_corr);
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
            const int first = min(n_my * GPS, NS);
            for (int q = 0; q < first; ++q)
                bulk_prefetch_l2(src + (q / GPS) * tile_step + (q % GPS) * kStageBytes, kStageBytes);
        }
        // The scales of the first tiles (the consumers load a tile's scales
        // two tiles ahead of its use).
        for (int it = 0; it < min(n_my, 3); ++it) prefetch_tile_scales(S, c0 + it * C, N, n_groups);
        // This CTA's slice of X (a prefetch only warms L2; where the previous
        // kernel writes X, the loads after the dependency wait see its data).
        for (int r = 0; r < rows; ++r)
            bulk_prefetch_l2(X + size_t(m0 + r) * K + size_t(grp0) * kGroup, uint32_t(GPS * kGroup * 2));
    }
    __syncthreads();

    const int g = lane >> 2, t = lane & 3;
    const bool vec_scales = s_vec != 0;
    ScaleRow<GPS> s_cur[2], s_next[2];
    auto load_scales = [&](int tile, ScaleRow<GPS> (&dst)[2]) {
        const int f0 = tile * kTileRows + warp * 16 + g;
        const uint16_t *p0 = S + size_t(f0) * n_groups + grp0;
        dst[0] = load_scale_row<GPS>(p0, f0 < N, vec_scales);
        dst[1] = load_scale_row<GPS>(p0 + 8 * size_t(n_groups), f0 + 8 < N, vec_scales);
    };
    // Read nothing that the previous grid in the stream may write before it
    // has completed: X always, and W and the scales unless they are resident
    // (then only the consumers wait, for X, and they load the first tile's
    // scales before waiting).
    if (resident && warp < kDecodeWarps && n_my > 0) load_scales(c0, s_cur);
    if (!resident || warp < kDecodeWarps) pdl_wait();

    if (warp == kDecodeWarps) {
        // Producer: one lane streams every (tile, group) block of this CTA.
        // Non-resident weights: it starts once the consumers have issued their
        // X and scale loads, so that those small reads are not queued behind
        // the weight stream.  Resident weights: it starts at once and fills
        // the ring while the previous grid finishes.
        if (!resident) named_bar_sync(2, kDecodeThreads);
        if (lane == 0) {
            const size_t tile_step = size_t(C) * KC * kChunkBytes;
            const uint8_t *src = Wp + (size_t(c0) * KC + size_t(2 * grp0)) * kChunkBytes;
            // At most IF copies are in the air at once (the ring may
            // hold more that have landed): a small burst per CTA lets the
            // first stages land early instead of all of them near the end.
            const int total = n_my * GPS;
            int issued = 0, st = 0, gi = 0, lst = 0;
            uint32_t epar = 1;   // parity of the empty phase to wait for (first lap: none)
            uint32_t lpar = 0;   // parity of the full phase of copy q - IF
            for (int q = 0; q < total; ++q) {
                if (q >= NS && !mbar_wait(empty0 + 8 * st, epar, abort_flag, err)) break;
                if (q >= IF) {
                    if (!mbar_wait(full0 + 8 * lst, lpar, abort_flag, err)) break;
                    if (++lst == NS) { lst = 0; lpar ^= 1; }
                }
                mbar_arrive_expect_tx(full0 + 8 * st, kStageBytes);
                bulk_g2s(smem_u32(ring + st * kStageBytes), src + gi * kStageBytes, kStageBytes,
                         full0 + 8 * st);
                ++issued;
                if (++gi == GPS) {
                    gi = 0;
                    src += tile_step;
                    // Entering tile q / GPS: warm L2 with the scales of tile
                    // q / GPS + 3, which the consumers load about two tiles later.
                    const int ahead = (q + 1) / GPS + 3;
                    if (ahead < n_my) prefetch_tile_scales(S, c0 + ahead * C, N, n_groups);
                }
                if (++st == NS) { st = 0; epar ^= 1; }
            }
            if (*abort_flag) {
                for (int q = issued > NS ? issued - NS : 0; q < issued; ++q)
                    drain_wait(full0 + 8 * (q % NS), (q / NS) & 1);
            }
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
        if (n_my > 0) load_scales(c0, s_cur);
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
    if (n_my > 1) load_scales(c0 + C, s_next);
    consumer_bar();
    {
        // Per (token, group): 8 lanes take 16 values each, convert them in
        // place to fp16 x * 2^-sh, and sum them (fp32, then a shuffle
        // reduction) for the correction table: token r, group gi ->
        // s_corr[(gi * MT + r / 8) * 4 + (r % 8) / 2] = {-1032 S(r), -1032 S(r^1),
        // -1152 S(r), -1152 S(r^1)} (pairs of tokens 2t, 2t + 1), S the scaled sum.
        const int pairs = rows * GPS;       // entries of absent tokens stay unwritten
        const int part = threadIdx.x & 7;
        for (int base = 0; base < pairs; base += kDecodeWarps * 32 / 8) {
            const int pi = base + (threadIdx.x >> 3);
            const int r = pi / GPS, gi = pi - r * GPS;
            float a = 0.f;
            if (pi < pairs) {
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
                        a += lo + hi;
                        uint32_t pk;
                        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(pk) : "f"(hi * down), "f"(lo * down));
                        hv[e] = pk;
                    }
                    src[h] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                }
                a *= down;
            }
            a += __shfl_xor_sync(0xffffffffu, a, 1);
            a += __shfl_xor_sync(0xffffffffu, a, 2);
            a += __shfl_xor_sync(0xffffffffu, a, 4);
            if (pi < pairs && part == 0) {
                float *e = s_corr + ((gi * MT + (r >> 3)) * 4 + ((r & 7) >> 1)) * 4 + (r & 1);
                e[0] = -1032.f * a;
                e[2] = -1152.f * a;
            }
        }
    }
    consumer_bar();

    // Fragment sources: X rows 8o + g (B), correction for tokens 8o + 2t, +1 (C).
    // Lanes of rows past the staged ones read the last staged row instead
    // (their tokens' columns are never stored).
    const uint16_t *xs = s_x + t * 8;
    int xrow[MT];
#pragma unroll
    for (int o = 0; o < MT; ++o) xrow[o] = min(8 * o + g, rows_alloc - 1) * L.x_stride;
    const float4 *cs = reinterpret_cast<const float4 *>(s_corr) + t;
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
    for (int it = 0; it < n_my; ++it) {
        float acc[MT][4];
#pragma unroll
        for (int o = 0; o < MT; ++o)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[o][r] = 0.f;
#pragma unroll
        for (int gi = 0; gi < GPS; ++gi) {
            // Stage q of this CTA's stream sits in ring slot q % kRing (a
            // power of two, so with the loop unrolled the slot and its phase
            // parity cost at most a shift and a mask per tile).
            const uint32_t q = uint32_t(it) * GPS + gi;
            const uint32_t slot = q % kRing;
            if (!mbar_wait(full0 + 8 * slot, (q / kRing) & 1u, abort_flag, err)) return;
            const unsigned char *wsrc = wlane + slot * kStageBytes;
            const uint4 wa = *reinterpret_cast<const uint4 *>(wsrc);
            const uint4 wb = *reinterpret_cast<const uint4 *>(wsrc + kChunkBytes);
            const uint32_t wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
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
            // The stage's bytes are now in registers: release it.
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * slot);
            // Group scales of rows g (C elements 0, 1) and g + 8 (2, 3),
            // loaded a tile ahead.
            const float s0 = scale_of<GPS>(s_cur[0], gi);
            const float s1 = scale_of<GPS>(s_cur[1], gi);
#pragma unroll
            for (int o = 0; o < MT; ++o) {
                const float4 cc = cs[(gi * MT + o) * 4];
                float c[4] = {cc.x, cc.y, cc.z, cc.w};
#pragma unroll
                for (int k16 = 0; k16 < 4; ++k16) {
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
#pragma unroll
        for (int o = 0; o < MT; ++o) {
            acc[o][0] *= fac[o][0];
            acc[o][1] *= fac[o][1];
            acc[o][2] *= fac16[o][0];
            acc[o][3] *= fac16[o][1];
        }
        // C fragment: {row g: tokens 2t, 2t+1}, {row g+8: tokens 2t, 2t+1}.
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
                        ws[(size_t(blockIdx.y) * n_entries + bz) * size_t(M) * N + off] = acc[o][r];
                    else
                        Y[off] = f32_to_bf16_rn(acc[o][r]);
                }
            }
        }
        s_cur[0] = s_next[0];
        s_cur[1] = s_next[1];
        if (it + 2 < n_my) load_scales(c0 + (it + 2) * C, s_next);
    }
}

// ---------------------------------------------------------------------------
// Whole-K decode kernel (no split-K).  A CTA owns B consecutive 16-row blocks
// of one 128-row tile over all of K.  Its 8 consumer warps are B blocks x P =
// 8 / B K-parts: warp w takes block w % B and K-part w / B (a contiguous run
// of whole 128-wide groups).  Each K-part has a private sub-ring of B of the
// 8 ring slots (slot kp + P * (j % B) for its j-th stage), so the parts stream
// independently; a stage holds SG groups of the CTA's B blocks (B x 1 KB per
// group: the B blocks' 512-byte pieces of both 64-column chunks lie side by
// side in the packed layout, one bulk copy per chunk).  The whole X row is
// staged once as fp16 with one exponent shift per (token, K-part), and the
// parts' fp32 results are added in shared memory in ascending part order, so
// the kernel writes Y itself: no workspace, no second kernel.
struct WkSmem {
    int x_stride, n_groups;
    int off_ring, off_bar, off_abort, off_xmax, off_x, off_corr, off_scale, off_red, total;
};

// Scale vectors (8 bf16) a consumer thread stages: B * 16 rows x K / 128
// groups <= 8 * 16 * 128 elements for K <= 16384.
constexpr int kWkScaleVecs = 8;

__host__ __device__ inline WkSmem wk_smem_layout(int B, int rows, int K) {
    WkSmem L;
    L.n_groups = K / kGroup;
    L.x_stride = K + 32;                       // fp16 elements per staged row (64 B mod 128 B)
    const int P = kDecodeWarps / B;
    L.off_ring = 0;
    L.off_bar = kRing * kStageBytes;
    L.off_abort = L.off_bar + 2 * kRing * 8;
    L.off_xmax = L.off_abort + 16;             // [8 tokens][P parts] int
    L.off_x = L.off_xmax + 8 * 8 * 4;
    L.off_corr = L.off_x + ((rows * L.x_stride * 2 + 15) & ~15);
    L.off_scale = L.off_corr + L.n_groups * 4 * 16;           // float4 per (group, quad)
    L.off_red = L.off_scale + ((B * 16 * L.n_groups * 2 + 15) & ~15);   // bf16 [B*16 rows][groups]
    L.total = L.off_red + (P - 1) * B * 512;   // float4 per lane per (part > 0, block)
    return L;
}

// K-part kp of P covers groups [wk_part_start(kp), wk_part_start(kp + 1)).
__device__ __forceinline__ int wk_part_start(int kp, int P, int G) { return (kp * G) / P; }

template <int B>
__global__ void __launch_bounds__(kDecodeThreads, 2)
decode_wk_kernel(const uint16_t *__restrict__ X, const uint8_t *__restrict__ Wp,
                 const uint16_t *__restrict__ S, uint16_t *__restrict__ Y, int M, int N, int K,
                 int resident, int s_vec, int *err) {
    constexpr int P = kDecodeWarps / B;
    // Batched products: grid.y = entries; entry b's X, W, scales and Y follow
    // each other in memory.
    {
        const size_t bz = blockIdx.y;
        const size_t n_tiles = (size_t(N) + kTileRows - 1) / kTileRows;
        X += bz * M * K;
        Wp += bz * n_tiles * kTileRows * (K / 2);
        S += bz * N * (K / kGroup);
        Y += bz * M * N;
    }
    constexpr int SG = B == 1 ? 4 : 8 / B;     // groups per stage (B * SG KB <= 8 KB)
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rows = M;                         // tokens (all staged; host checks they fit)
    const WkSmem L = wk_smem_layout(B, rows, K);
    const int G = L.n_groups;
    const int KC = K / kChunkK;
    const int blk0 = blockIdx.x * B;            // first global 16-row block
    const int tile = blk0 / kDecodeWarps, bb0 = blk0 % kDecodeWarps;
    unsigned char *ring = smem + L.off_ring;
    const uint32_t full0 = smem_u32(smem + L.off_bar);
    const uint32_t empty0 = full0 + 8 * kRing;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.off_abort);
    int *s_xmax = reinterpret_cast<int *>(smem + L.off_xmax);
    uint16_t *s_x = reinterpret_cast<uint16_t *>(smem + L.off_x);
    float *s_corr = reinterpret_cast<float *>(smem + L.off_corr);
    uint16_t *s_scale = reinterpret_cast<uint16_t *>(smem + L.off_scale);
    float4 *s_red = reinterpret_cast<float4 *>(smem + L.off_red);

    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRing; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, B);      // the B warps of the slot's K-part
        }
        *abort_flag = 0;
        for (int r = 0; r < 64; ++r) s_xmax[r] = 0;
        fence_barrier_init();
    }
    if (warp == kDecodeWarps && lane == 0) {
        // Warm L2 with X (all rows, contiguous) and the scale rows of the CTA's
        // blocks while the previous grid finishes: a prefetch reads nothing
        // into the CTA, so it needs no dependency wait, and where the previous
        // kernel writes X the L2 copy it leaves is the one the loads see.
        bulk_prefetch_l2(X, uint32_t(size_t(M) * K * 2));
        const size_t r0 = size_t(tile) * kTileRows + bb0 * 16;
        const size_t r1 = min(size_t(N), r0 + 16 * B);
        if (r1 > r0) {
            const uintptr_t lo = (reinterpret_cast<uintptr_t>(S + r0 * G) + 15) & ~uintptr_t(15);
            const uintptr_t hi = reinterpret_cast<uintptr_t>(S + r1 * G) & ~uintptr_t(15);
            if (hi > lo) bulk_prefetch_l2(reinterpret_cast<const void *>(lo), uint32_t(hi - lo));
        }
    }
    __syncthreads();
    if (!resident || warp < kDecodeWarps) pdl_wait();

    if (warp == kDecodeWarps) {
        // Producer: lane kp streams K-part kp through its sub-ring, so a part
        // whose consumers lag never holds back the others' copies.
        if (lane < P) {
            const int kp = lane;
            const uint8_t *wtile = Wp + size_t(tile) * KC * kChunkBytes + size_t(bb0) * kBlockBytes;
            const int ga = wk_part_start(kp, P, G), gb = wk_part_start(kp + 1, P, G);
            const int n_st = (gb - ga + SG - 1) / SG;
            uint32_t used = 0, last_par = 0;    // per slot: issued at least once / parity of the last issue
            // At most IFP of a part's stages in the air (about three stages
            // per CTA, as in decode_kernel): a deeper burst queues the first
            // X and scale loads behind the weight stream.
            constexpr int IFP = P >= 4 ? 1 : (P == 2 ? 2 : 3);
            for (int j = 0; j < n_st; ++j) {
                const int g0 = ga + j * SG;
                const int ng = min(SG, gb - g0);
                const int slot = kp + P * (j % B);
                if (j >= B && !mbar_wait(empty0 + 8 * slot, ((j / B) + 1) & 1, abort_flag, err)) break;
                if (j >= IFP) {
                    const int jl = j - IFP;
                    if (!mbar_wait(full0 + 8 * (kp + P * (jl % B)), (jl / B) & 1, abort_flag, err)) break;
                }
                mbar_arrive_expect_tx(full0 + 8 * slot, uint32_t(ng * 2 * B * kBlockBytes));
                unsigned char *dst = ring + slot * kStageBytes;
                for (int gg = 0; gg < ng; ++gg)
                    for (int h = 0; h < 2; ++h)
                        bulk_g2s(smem_u32(dst + (gg * 2 + h) * B * kBlockBytes),
                                 wtile + size_t(2 * (g0 + gg) + h) * kChunkBytes,
                                 uint32_t(B * kBlockBytes), full0 + 8 * slot);
                used |= 1u << slot;
                last_par = (last_par & ~(1u << slot)) | (uint32_t((j / B) & 1) << slot);
            }
            if (*abort_flag) {
                // Let every copy this lane issued land before the CTA exits.
                for (int s2 = 0; s2 < kRing; ++s2)
                    if (used & (1u << s2)) drain_wait(full0 + 8 * s2, (last_par >> s2) & 1);
            }
        }
        return;
    }

    // ---- consumers (256 threads) ----
    const int g = lane >> 2, t = lane & 3;
    // Scales of the CTA's B * 16 rows (zero past N, one contiguous run of S,
    // 16-byte vectors when aligned) and X rows [0, M) of all K are loaded
    // together (every load before the first store, so their latencies
    // overlap).  Every CTA reads all of X: CTA c starts at a different group
    // (rotation by whole groups), so the CTAs do not all hit the same L2 lines
    // at once.
    const size_t srow0 = size_t(tile) * kTileRows + size_t(bb0) * 16;
    const int E = B * 16 * G;
    const long long rows_in = (long long)N - (long long)srow0;
    const int valid = rows_in <= 0 ? 0 : (rows_in >= 16 * B ? E : int(rows_in) * G);
    const uint16_t *ssrc = S + srow0 * G;
    uint4 sv[kWkScaleVecs];
    if (s_vec) {
#pragma unroll
        for (int k = 0; k < kWkScaleVecs; ++k) {
            const int i = (threadIdx.x + k * kDecodeWarps * 32) * 8;
            sv[k] = make_uint4(0, 0, 0, 0);
            if (i + 8 <= valid) {
                sv[k] = ldg_nc16(ssrc + i);
            } else if (i < valid) {
                uint16_t e[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) e[u] = i + u < valid ? ssrc[i + u] : uint16_t(0);
                sv[k] = make_uint4(e[0] | (uint32_t(e[1]) << 16), e[2] | (uint32_t(e[3]) << 16),
                                   e[4] | (uint32_t(e[5]) << 16), e[6] | (uint32_t(e[7]) << 16));
            }
        }
    }
    const int V = rows * G * 16;                 // 16-byte X vectors (host: V <= 8 * 256)
    const int rot = (int(blockIdx.x) * 16 * 5) % (G * 16);   // whole groups
    uint4 xv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int i = threadIdx.x + k * kDecodeWarps * 32;
        if (i < V) {
            const int r = i / (G * 16);
            int v = i - r * G * 16 + rot;
            if (v >= G * 16) v -= G * 16;
            xv[k] = ldg_nc16(X + size_t(r) * K + size_t(v) * 8);
        }
    }
    if (s_vec) {
#pragma unroll
        for (int k = 0; k < kWkScaleVecs; ++k) {
            const int i = (threadIdx.x + k * kDecodeWarps * 32) * 8;
            if (i < E) *reinterpret_cast<uint4 *>(s_scale + i) = sv[k];
        }
    } else {
        for (int i0 = threadIdx.x; i0 < E; i0 += 8 * kDecodeWarps * 32) {
            uint16_t e[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * kDecodeWarps * 32;
                e[u] = i < valid ? ssrc[i] : uint16_t(0);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * kDecodeWarps * 32;
                if (i < E) s_scale[i] = e[u];
            }
        }
    }
    // X into shared memory, permuted per group as in decode_kernel so that one
    // 16-byte shared load feeds two MMAs; the maximum |x| per (token, K-part)
    // is reduced over the 16 lanes that share a group, then one shared atomic.
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int i = threadIdx.x + k * kDecodeWarps * 32;
        if (k * kDecodeWarps * 32 >= V) break;    // uniform: whole passes only
        uint32_t mx = 0;
        int r = 0, gi = 0;
        if (i < V) {
            r = i / (G * 16);
            int v = i - r * G * 16 + rot;
            if (v >= G * 16) v -= G * 16;
            gi = v >> 4;
            const int u = v & 15;
            const int h = u >> 3, s16 = (u >> 1) & 3, t0 = (u & 1) * 2;
            const int pos = gi * kGroup + 32 * (2 * h + (s16 >> 1)) + 8 * t0 + 4 * (s16 & 1);
            uint16_t *dst = s_x + r * L.x_stride + pos;
            const uint4 val = xv[k];
            const uint2 lo = make_uint2(val.x, val.y), hi = make_uint2(val.z, val.w);
            *reinterpret_cast<uint2 *>(dst + (h ? 8 : 0)) = h ? hi : lo;
            *reinterpret_cast<uint2 *>(dst + (h ? 0 : 8)) = h ? lo : hi;
            const uint32_t m01 = max(val.x & 0x7FFFu, (val.x >> 16) & 0x7FFFu);
            const uint32_t m23 = max(val.y & 0x7FFFu, (val.y >> 16) & 0x7FFFu);
            const uint32_t m45 = max(val.z & 0x7FFFu, (val.z >> 16) & 0x7FFFu);
            const uint32_t m67 = max(val.w & 0x7FFFu, (val.w >> 16) & 0x7FFFu);
            mx = max(max(m01, m23), max(m45, m67));
        }
        // The 16 lanes of a half-warp hold one (row, group): V and the
        // rotation are multiples of 16.
#pragma unroll
        for (int off = 1; off < 16; off <<= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if (i < V && (lane & 15) == 0) {
            int kp = 0;
            while (kp + 1 < P && wk_part_start(kp + 1, P, G) <= gi) ++kp;
            atomicMax(s_xmax + r * 8 + kp, int(mx));
        }
    }
    consumer_bar();
    // Convert X in place to fp16 x * 2^-sh(token, part) and build the
    // per-group correction table (as decode_kernel): 8 lanes per (token, group).
    {
        const int pairs = rows * G;
        const int part = threadIdx.x & 7;
        for (int base = 0; base < pairs; base += kDecodeWarps * 32 / 8) {
            const int pi = base + (threadIdx.x >> 3);
            const int r = pi / G, gi = pi - r * G;
            float a = 0.f;
            if (pi < pairs) {
                int kp = 0;
                while (kp + 1 < P && wk_part_start(kp + 1, P, G) <= gi) ++kp;
                const float down = pow2f(-slice_shift(s_xmax[r * 8 + kp]));
                uint4 *src = reinterpret_cast<uint4 *>(s_x + r * L.x_stride + gi * kGroup) + part;
#pragma unroll
                for (int hh = 0; hh < 16; hh += 8) {
                    const uint4 q = src[hh];
                    const uint32_t qv[4] = {q.x, q.y, q.z, q.w};
                    uint32_t hv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float lo = bf16_lo_to_f32(qv[e]), hi = bf16_hi_to_f32(qv[e]);
                        a += lo + hi;
                        uint32_t pk;
                        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(pk) : "f"(hi * down), "f"(lo * down));
                        hv[e] = pk;
                    }
                    src[hh] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                }
                a *= down;
            }
            a += __shfl_xor_sync(0xffffffffu, a, 1);
            a += __shfl_xor_sync(0xffffffffu, a, 2);
            a += __shfl_xor_sync(0xffffffffu, a, 4);
            if (pi < pairs && part == 0) {
                float *e = s_corr + (gi * 4 + (r >> 1)) * 4 + (r & 1);
                e[0] = -1032.f * a;
                e[2] = -1152.f * a;
            }
        }
    }
    consumer_bar();

    const int b = warp % B, kp = warp / B;
    const int ga = wk_part_start(kp, P, G), gb = wk_part_start(kp + 1, P, G);
    const int n_st = (gb - ga + SG - 1) / SG;
    const uint16_t *xs = s_x + min(g, rows - 1) * L.x_stride + t * 8;
    const float4 *cs = reinterpret_cast<const float4 *>(s_corr) + t;
    const uint16_t *srow = s_scale + (b * 16 + g) * G;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const unsigned char *wlane = ring + b * kBlockBytes + lane * 16;
    bool alive = true;
    for (int j = 0; j < n_st && alive; ++j) {
        const int slot = kp + P * (j % B);
        if (!mbar_wait(full0 + 8 * slot, (j / B) & 1, abort_flag, err)) {
            alive = false;
            break;
        }
        const int g0 = ga + j * SG;
        const int ng = min(SG, gb - g0);
        const unsigned char *wst = wlane + slot * kStageBytes;
        uint32_t wv[SG][8];
#pragma unroll
        for (int gg = 0; gg < SG; ++gg) {
            if (gg < ng) {
                const uint4 wa = *reinterpret_cast<const uint4 *>(wst + (gg * 2) * B * kBlockBytes);
                const uint4 wb = *reinterpret_cast<const uint4 *>(wst + (gg * 2 + 1) * B * kBlockBytes);
                wv[gg][0] = wa.x; wv[gg][1] = wa.y; wv[gg][2] = wa.z; wv[gg][3] = wa.w;
                wv[gg][4] = wb.x; wv[gg][5] = wb.y; wv[gg][6] = wb.z; wv[gg][7] = wb.w;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * slot);
#pragma unroll
        for (int gg = 0; gg < SG; ++gg) {
            if (gg >= ng) break;
            const int gi = g0 + gg;
            uint32_t af[8][4];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const uint32_t w8 = wv[gg][jj] >> 8;
                af[jj][0] = lop3_and_or(wv[gg][jj], 0x000F000Fu, kMagicF16x2_1024);
                af[jj][1] = lop3_and_or(wv[gg][jj], 0x00F000F0u, kMagicF16x2_1024);
                af[jj][2] = lop3_and_or(w8, 0x000F000Fu, kMagicF16x2_1024);
                af[jj][3] = lop3_and_or(w8, 0x00F000F0u, kMagicF16x2_1024);
            }
            const float4 cc = cs[gi * 4];
            float c[4] = {cc.x, cc.y, cc.z, cc.w};
#pragma unroll
            for (int k16 = 0; k16 < 4; ++k16) {
                const uint4 xv = *reinterpret_cast<const uint4 *>(xs + gi * kGroup + 32 * k16);
                mma_16816_f16_acc(c, af[2 * k16], xv.x, xv.y);
                mma_16816_f16_acc(c, af[2 * k16 + 1], xv.z, xv.w);
            }
            const float s0 = __uint_as_float(uint32_t(srow[gi]) << 16);
            const float s1 = __uint_as_float(uint32_t(srow[8 * G + gi]) << 16);
            acc[0] = fmaf(s0, c[0], acc[0]);
            acc[1] = fmaf(s0, c[1], acc[1]);
            acc[2] = fmaf(s1, c[2], acc[2]);
            acc[3] = fmaf(s1, c[3], acc[3]);
        }
    }
    // Undo this part's shift (tokens 2t, 2t + 1; rows g + 8 also carry 16).
    {
        float fac[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = 2 * t + e;
            fac[e] = r < rows ? pow2f(slice_shift(s_xmax[r * 8 + kp])) : 0.f;
        }
        acc[0] *= fac[0];
        acc[1] *= fac[1];
        acc[2] *= 0.0625f * fac[0];
        acc[3] *= 0.0625f * fac[1];
    }
    // Add the K-parts in ascending order; part 0's warps write Y.
    if (kp > 0) s_red[((kp - 1) * B + b) * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    consumer_bar();
    if (kp > 0) return;
#pragma unroll
    for (int q = 1; q < P; ++q) {
        const float4 v = s_red[((q - 1) * B + b) * 32 + lane];
        acc[0] += v.x; acc[1] += v.y; acc[2] += v.z; acc[3] += v.w;
    }
    const int f0 = tile * kTileRows + (bb0 + b) * 16 + g;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int m = 2 * t + (r & 1);
        const int f = f0 + ((r < 2) ? 0 : 8);
        if (m < M && f < N) Y[size_t(m) * N + f] = f32_to_bf16_rn(acc[r]);
    }
}

// Split-K reduce: each thread owns VEC consecutive outputs (one VEC-wide load
// per slice).  VEC shrinks for small outputs so that enough threads run;
// loads are issued a batch of slices at a time so their latencies overlap,
// and the sum runs over the slices in ascending order, so the result does not
// depend on VEC, the batch or the unrolling.
template <int VEC>
struct FloatVec;
template <> struct FloatVec<1> { using T = float; };
template <> struct FloatVec<2> { using T = float2; };
template <> struct FloatVec<4> { using T = float4; };

__device__ __forceinline__ void vadd(float &a, float b) { a += b; }
__device__ __forceinline__ void vadd(float2 &a, float2 b) { a.x += b.x; a.y += b.y; }
__device__ __forceinline__ void vadd(float4 &a, float4 b) { a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w; }
__device__ __forceinline__ void vstore(uint16_t *y, float a) { *y = f32_to_bf16_rn(a); }
__device__ __forceinline__ void vstore(uint16_t *y, float2 a) {
    *reinterpret_cast<uint32_t *>(y) = pack_bf16x2_rn(a.x, a.y);
}
__device__ __forceinline__ void vstore(uint16_t *y, float4 a) {
    *reinterpret_cast<uint2 *>(y) = make_uint2(pack_bf16x2_rn(a.x, a.y), pack_bf16x2_rn(a.z, a.w));
}

// kBatch slices are loaded per round trip: 16, or 64 / VEC for deeper splits
// (a 64-deep batch also costs registers and instructions, which slows the
// short splits down when the kernel is chained between two GEMM launches).
template <int VEC, int kBatch>
__global__ void __launch_bounds__(256)
splitk_reduce_kernel(const float *__restrict__ ws, uint16_t *__restrict__ Y, int splits,
                     long long count) {
    using T = typename FloatVec<VEC>::T;
    pdl_launch_dependents();
    pdl_wait();
    const long long i = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * VEC;
    if (i >= count) return;
    T a;
    const float *q = ws + i;   // slice s of this thread's outputs: q + s * count
    for (int s = 0; s < splits; s += kBatch) {
        const int n = min(kBatch, splits - s);
        T b[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (u < n) b[u] = *reinterpret_cast<const T *>(q);
            q += count;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (u >= n) break;
            if (s + u == 0) a = b[u];
            else vadd(a, b[u]);
        }
    }
    vstore(Y + i, a);
}

template <int MT, int GPS, bool kSplit>
cudaError_t launch_decode_t(const DecodePlan &p, const uint16_t *X, const uint8_t *Wp,
                            const uint16_t *S, uint16_t *Y, float *ws, bool resident, int M, int N,
                            int K, cudaStream_t s) {
    const int smem = decode_smem_layout(MT, M < 8 * MT ? M : 8 * MT, GPS).total;
    auto kern = decode_kernel<MT, GPS, kSplit>;
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
    const int s_vec = (reinterpret_cast<uintptr_t>(S) % (2 * GPS)) == 0;
    return cudaLaunchKernelEx(&cfg, kern, X, Wp, S, Y, ws, M, N, K, p.n_tiles, p.ring, p.in_flight,
                              s_vec, int(resident), p.token_blocks, err);
}

template <int MT, bool kSplit>
cudaError_t launch_decode_gps(const DecodePlan &p, const uint16_t *X, const uint8_t *Wp,
                              const uint16_t *S, uint16_t *Y, float *ws, bool res, int M, int N,
                              int K, cudaStream_t s) {
    switch (p.groups_per_slice) {
        case 1: return launch_decode_t<MT, 1, kSplit>(p, X, Wp, S, Y, ws, res, M, N, K, s);
        case 2: return launch_decode_t<MT, 2, kSplit>(p, X, Wp, S, Y, ws, res, M, N, K, s);
        case 4: return launch_decode_t<MT, 4, kSplit>(p, X, Wp, S, Y, ws, res, M, N, K, s);
        case 8: return launch_decode_t<MT, 8, kSplit>(p, X, Wp, S, Y, ws, res, M, N, K, s);
        case 16:
            if constexpr (MT == 1) return launch_decode_t<MT, 16, kSplit>(p, X, Wp, S, Y, ws, res, M, N, K, s);
            return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

template <int B>
cudaError_t launch_wk_t(int ctas, int batch, const uint16_t *X, const uint8_t *Wp, const uint16_t *S,
                        uint16_t *Y, bool resident, int M, int N, int K, cudaStream_t s) {
    const int smem = wk_smem_layout(B, M, K).total;
    auto kern = decode_wk_kernel<B>;
    if (smem > 48 * 1024) {
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
    cfg.gridDim = dim3(ctas, batch);
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
    // 16-byte scale vectors: every CTA's first scale row (a multiple of 16
    // rows) is 16-byte aligned when S is, and so is every batch entry's block
    // when N * K / 128 * 2 bytes is a multiple of 16.
    const int s_vec = (reinterpret_cast<uintptr_t>(S) % 16) == 0 &&
                      (batch == 1 || (size_t(N) * (K / kGroup) * 2) % 16 == 0);
    return cudaLaunchKernelEx(&cfg, kern, X, Wp, S, Y, M, N, K, int(resident), s_vec, err);
}

}  // namespace

int decode_smem_needed(int M, int mt, int groups_per_slice) {
    return decode_smem_layout(mt, M < 8 * mt ? M : 8 * mt, groups_per_slice).total;
}

cudaError_t launch_decode(const DecodePlan &p, const uint16_t *X, const uint8_t *Wp,
                          const uint16_t *S, uint16_t *Y, float *ws, bool res, int M, int N, int K,
                          cudaStream_t s) {
    if (p.ring != kRing || p.in_flight < 1 || p.in_flight > p.ring) return cudaErrorInvalidValue;
    if (p.batch < 1 || (long long)p.token_blocks * p.batch > 65535) return cudaErrorInvalidValue;
    if (p.groups_per_slice < 1 || p.groups_per_slice > kDecodeMaxGps || p.ctas_per_slice < 1 ||
        decode_smem_needed(M, p.mt, p.groups_per_slice) > kDecodeMaxSmem ||
        decode_smem_layout(p.mt, M < 8 * p.mt ? M : 8 * p.mt, p.groups_per_slice).stages < kRing)
        return cudaErrorInvalidValue;
    if ((K / kGroup) % p.groups_per_slice != 0) return cudaErrorInvalidValue;
    const bool split = p.split_k > 1;
    if (p.mt == 1)
        return split ? launch_decode_gps<1, true>(p, X, Wp, S, Y, ws, res, M, N, K, s)
                     : launch_decode_gps<1, false>(p, X, Wp, S, Y, ws, res, M, N, K, s);
    return split ? launch_decode_gps<2, true>(p, X, Wp, S, Y, ws, res, M, N, K, s)
                 : launch_decode_gps<2, false>(p, X, Wp, S, Y, ws, res, M, N, K, s);
}

bool decode_wk_fits(int M, int K, int B) {
    if (M < 1 || M > 8 || (B != 1 && B != 2 && B != 4 && B != 8)) return false;
    if (M * (K / kGroup) * 16 > 8 * kDecodeWarps * 32) return false;   // X vectors per thread
    if (B * 16 * (K / kGroup) > kWkScaleVecs * 8 * kDecodeWarps * 32) return false;  // scale vectors
    return wk_smem_layout(B, M, K).total <= kDecodeMaxSmem;
}

cudaError_t launch_decode_wk(int B, int ctas, int batch, const uint16_t *X, const uint8_t *Wp,
                             const uint16_t *S, uint16_t *Y, bool resident, int M, int N, int K,
                             cudaStream_t s) {
    if (!decode_wk_fits(M, K, B) || ctas < 1 || batch < 1 || batch > 65535) return cudaErrorInvalidValue;
    switch (B) {
        case 1: return launch_wk_t<1>(ctas, batch, X, Wp, S, Y, resident, M, N, K, s);
        case 2: return launch_wk_t<2>(ctas, batch, X, Wp, S, Y, resident, M, N, K, s);
        case 4: return launch_wk_t<4>(ctas, batch, X, Wp, S, Y, resident, M, N, K, s);
        case 8: return launch_wk_t<8>(ctas, batch, X, Wp, S, Y, resident, M, N, K, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_reduce(const float *ws, uint16_t *Y, int splits, long long count, bool pdl,
                          cudaStream_t s) {
    if (count <= 0) return cudaSuccess;
    // Widest VEC that keeps about two threads per SM slot of 256 busy and
    // that the addresses allow.
    const long long want_threads = 2LL * 152 * 256;
    int vec = 1;
    if (count % 4 == 0 && reinterpret_cast<uintptr_t>(Y) % 8 == 0 &&
        reinterpret_cast<uintptr_t>(ws) % 16 == 0 && count / 4 >= want_threads)
        vec = 4;
    else if (count % 2 == 0 && reinterpret_cast<uintptr_t>(Y) % 4 == 0 &&
             reinterpret_cast<uintptr_t>(ws) % 8 == 0 && count / 2 >= want_threads)
        vec = 2;
    const int threads = 256;
    const long long items = count / vec;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned((items + threads - 1) / threads));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const bool deep = splits > 16;
    if (vec == 4)
        return deep ? cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<4, 16>, ws, Y, splits, count)
                    : cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<4, 16>, ws, Y, splits, count);
    if (vec == 2)
        return deep ? cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<2, 32>, ws, Y, splits, count)
                    : cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<2, 16>, ws, Y, splits, count);
    return deep ? cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<1, 64>, ws, Y, splits, count)
                : cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<1, 16>, ws, Y, splits, count);
}

}  // namespace w4a16
