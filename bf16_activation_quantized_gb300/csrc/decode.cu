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
constexpr int kDecodeThreads = (kDecodeWarps + 1) * 32;         // + one producer warp
constexpr int kStageBytes = 2 * kChunkBytes;                    // one 128-wide group of a tile
constexpr int kDecodeMaxStages = 16;

// Shared memory: the weight ring first (a whole number of tiles' worth of
// groups, as many as the budget allows, at most kDecodeMaxStages stages), then
// its barriers, the abort flag, the staged X slice and the per-group
// correction table.
struct DecodeSmem {
    int x_stride;      // bf16 elements per staged X row: slice + 32 (row stride = 64 B mod 128 B)
    int ring_tiles;    // tiles of the slice held by the ring
    int stages;        // ring_tiles * groups per slice
    int off_ring, off_bar, off_abort, off_x, off_corr, total;
};

__host__ __device__ inline DecodeSmem decode_smem_layout(int mt, int gps) {
    DecodeSmem L;
    const int rows = 8 * mt;
    L.x_stride = gps * kGroup + 32;
    const int rest = 2 * kDecodeMaxStages * 8 + 16 + rows * L.x_stride * 2 + rows * gps * 4;
    int kt = (kDecodeMaxSmem - rest) / (gps * kStageBytes);
    if (kt > kDecodeMaxStages / gps) kt = kDecodeMaxStages / gps;
    L.ring_tiles = kt;
    L.stages = kt * gps;
    L.off_ring = 0;
    L.off_bar = L.stages * kStageBytes;
    L.off_abort = L.off_bar + 2 * kDecodeMaxStages * 8;
    L.off_x = L.off_abort + 16;
    L.off_corr = L.off_x + rows * L.x_stride * 2;
    L.total = L.off_corr + rows * gps * 4;
    return L;
}

__device__ __forceinline__ void consumer_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(kDecodeWarps * 32) : "memory");
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
    if constexpr (GPS == 8) {
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
// Each consumer warp owns one 16-row block of a tile.  Per group it waits for
// the stage, reads its 16 B of each chunk, turns the 8 words into 32 A
// fragments, releases the stage and runs a chain of 8 MMAs whose accumulator
// starts at -136 * sum(x) for the group, so the chain yields
// sum_k (code_k - 8) x_k directly.  The group scales are applied when the tile
// (or, for 16 tokens, a batch of groups) is done, so the scale loads -- issued
// a tile ahead -- are off the critical path.
template <int MT, int GPS, bool kSplit>
__global__ void __launch_bounds__(kDecodeThreads, 2)
decode_kernel(const uint16_t *__restrict__ X, const uint8_t *__restrict__ Wp,
              const uint16_t *__restrict__ S, uint16_t *__restrict__ Y, float *__restrict__ ws,
              int M, int N, int K, int n_tiles, int s_vec, int *err) {
    extern __shared__ __align__(128) unsigned char smem[];
    // Groups between scale applications: the whole slice for 8 tokens, at
    // most 4 groups for 16 (register budget).
    constexpr int D = (MT == 1) ? GPS : (GPS < 4 ? GPS : 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_groups = K / kGroup;
    const int grp0 = blockIdx.y * GPS;
    const int m0 = blockIdx.z * 8 * MT;
    const int rows = min(8 * MT, M - m0);
    const int C = gridDim.x;
    const int c0 = blockIdx.x;
    const int n_my = c0 < n_tiles ? (n_tiles - c0 + C - 1) / C : 0;
    const int KC = K / kChunkK;
    const DecodeSmem L = decode_smem_layout(MT, GPS);
    const int NS = L.stages;
    const int KT = L.ring_tiles;
    unsigned char *ring = smem + L.off_ring;
    const uint32_t full0 = smem_u32(smem + L.off_bar);
    const uint32_t empty0 = full0 + 8 * kDecodeMaxStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.off_abort);
    uint16_t *s_x = reinterpret_cast<uint16_t *>(smem + L.off_x);
    float *s_corr = reinterpret_cast<float *>(smem + L.off_corr);

    // Let the next kernel in the stream be scheduled while this grid runs.
    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kDecodeWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // Touch no global memory before the previous grid in the stream has completed.
    pdl_wait();

    const int g = lane >> 2, t = lane & 3;
    const bool vec_scales = s_vec != 0;
    // Scales of rows g and g+8 of this warp's block for the first tile: issued
    // before anything else so they are not queued behind the weight stream.
    ScaleRow<GPS> s_cur[2], s_next[2];
    auto load_scales = [&](int tile, ScaleRow<GPS> (&dst)[2]) {
        const int f0 = tile * kTileRows + warp * 16 + g;
        const uint16_t *p0 = S + size_t(f0) * n_groups + grp0;
        dst[0] = load_scale_row<GPS>(p0, f0 < N, vec_scales);
        dst[1] = load_scale_row<GPS>(p0 + 8 * size_t(n_groups), f0 + 8 < N, vec_scales);
    };
    if (warp < kDecodeWarps && n_my > 0) load_scales(c0, s_cur);

    if (warp == kDecodeWarps) {
        // Producer: one lane streams every (tile, group) block of this CTA.
        if (lane == 0) {
            const size_t tile_step = size_t(C) * KC * kChunkBytes;
            const uint8_t *src = Wp + (size_t(c0) * KC + size_t(2 * grp0)) * kChunkBytes;
            int issued = 0, ts = 0;
            uint32_t epar = 1;   // parity of the empty phase to wait for (first lap: none)
            bool ok = true;
            for (int it = 0; it < n_my && ok; ++it) {
                const int base = ts * GPS;
#pragma unroll
                for (int gi = 0; gi < GPS; ++gi) {
                    const int slot = base + gi;
                    if (it >= KT && !mbar_wait(empty0 + 8 * slot, epar, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full0 + 8 * slot, kStageBytes);
                    bulk_g2s(smem_u32(ring + slot * kStageBytes), src + gi * kStageBytes,
                             kStageBytes, full0 + 8 * slot);
                    ++issued;
                }
                src += tile_step;
                if (++ts == KT) { ts = 0; epar ^= 1; }
            }
            if (*abort_flag) {
                for (int q = issued > NS ? issued - NS : 0; q < issued; ++q) {
                    const int it = q / GPS, gi = q - it * GPS;
                    drain_wait(full0 + 8 * ((it % KT) * GPS + gi), (it / KT) & 1);
                }
            }
        }
        return;
    }

    // Consumers: stage X[m0 .. m0+rows)[slice], permuted so that a lane's B
    // fragments for word pair q of a group are 16 contiguous bytes: natural
    // column cc of a group (chunk h, 16-column slice s, quad t, element e) goes
    // to 32 (2h + s/2) + 8t + 4 (s % 2) + e.
    constexpr int vec_per_row = GPS * (kGroup / 8);
    for (int i = threadIdx.x; i < rows * vec_per_row; i += kDecodeWarps * 32) {
        const int r = i / vec_per_row, v = i - r * vec_per_row;
        const uint4 val = ldg_nc16(X + size_t(m0 + r) * K + size_t(grp0) * kGroup + v * 8);
        const int gi = v >> 4, u = v & 15;           // 16 vectors per group
        const int h = u >> 3, s16 = (u >> 1) & 3, t0 = (u & 1) * 2;
        const int pos = gi * kGroup + 32 * (2 * h + (s16 >> 1)) + 8 * t0 + 4 * (s16 & 1);
        uint16_t *dst = s_x + r * L.x_stride + pos;
        *reinterpret_cast<uint2 *>(dst) = make_uint2(val.x, val.y);
        *reinterpret_cast<uint2 *>(dst + 8) = make_uint2(val.z, val.w);
    }
    if (n_my > 1) load_scales(c0 + C, s_next);
    consumer_bar();
    {
        // Correction table s_corr[gi][token] = -136 * sum of the group's x:
        // 8 lanes per sum, 16 values each, then a shuffle reduction.
        const int pairs = 8 * MT * GPS;
        const int part = threadIdx.x & 7;
        for (int base = 0; base < pairs; base += kDecodeWarps * 32 / 8) {
            const int pi = base + (threadIdx.x >> 3);
            float a = 0.f;
            if (pi < pairs && pi / GPS < rows) {   // absent tokens: 0 (their rows are never read)
                const int r = pi / GPS, gi = pi - r * GPS;
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    s_x + r * L.x_stride + gi * kGroup + part * 16);
                const uint4 q0 = src[0], q1 = src[1];
                a = ((bf16_lo_to_f32(q0.x) + bf16_hi_to_f32(q0.x)) +
                     (bf16_lo_to_f32(q0.y) + bf16_hi_to_f32(q0.y))) +
                    ((bf16_lo_to_f32(q0.z) + bf16_hi_to_f32(q0.z)) +
                     (bf16_lo_to_f32(q0.w) + bf16_hi_to_f32(q0.w))) +
                    (((bf16_lo_to_f32(q1.x) + bf16_hi_to_f32(q1.x)) +
                      (bf16_lo_to_f32(q1.y) + bf16_hi_to_f32(q1.y))) +
                     ((bf16_lo_to_f32(q1.z) + bf16_hi_to_f32(q1.z)) +
                      (bf16_lo_to_f32(q1.w) + bf16_hi_to_f32(q1.w))));
            }
            a += __shfl_xor_sync(0xffffffffu, a, 1);
            a += __shfl_xor_sync(0xffffffffu, a, 2);
            a += __shfl_xor_sync(0xffffffffu, a, 4);
            if (pi < pairs && part == 0) {
                const int r = pi / GPS, gi = pi - r * GPS;
                s_corr[gi * 8 * MT + r] = -136.f * a;
            }
        }
    }
    consumer_bar();

    // Fragment sources: X rows 8o + g (B), correction for tokens 8o + 2t, +1 (C).
    const bool xok0 = g < rows, xok1 = MT > 1 && 8 + g < rows;
    const uint16_t *xs = s_x + g * L.x_stride + 8 * t;
    const float *cs = s_corr + 2 * t;

    int ts = 0;
    uint32_t fpar = 0;
    const unsigned char *wlane = ring + warp * kBlockBytes + lane * 16;
    for (int it = 0; it < n_my; ++it) {
        const int base = ts * GPS;
        float acc[MT][4];
#pragma unroll
        for (int o = 0; o < MT; ++o)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[o][r] = 0.f;
#pragma unroll
        for (int b0 = 0; b0 < GPS; b0 += D) {
            float p[D][MT][4];
#pragma unroll
            for (int db = 0; db < D; ++db) {
                const int gi = b0 + db;
                const int slot = base + gi;
                if (!mbar_wait(full0 + 8 * slot, fpar, abort_flag, err)) return;
                const unsigned char *wsrc = wlane + slot * kStageBytes;
                const uint4 wa = *reinterpret_cast<const uint4 *>(wsrc);
                const uint4 wb = *reinterpret_cast<const uint4 *>(wsrc + kChunkBytes);
                const uint32_t wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
                uint32_t af[8][4];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    af[j][0] = magic_pair(wv[j]);
                    af[j][1] = magic_pair((wv[j] >> 4));
                    af[j][2] = magic_pair((wv[j] >> 8));
                    af[j][3] = magic_pair((wv[j] >> 12));
                }
                // The stage's bytes are now in registers: release it.
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8 * slot);
#pragma unroll
                for (int o = 0; o < MT; ++o) {
                    const bool xok = o == 0 ? xok0 : xok1;
                    const float2 cc = *reinterpret_cast<const float2 *>(cs + gi * 8 * MT + 8 * o);
                    float c[4] = {cc.x, cc.y, cc.x, cc.y};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 xv = make_uint4(0, 0, 0, 0);
                        if (xok)
                            xv = *reinterpret_cast<const uint4 *>(xs + 8 * o * L.x_stride +
                                                                  gi * kGroup + 32 * q);
                        float d[4];
                        mma_16816_c(d, af[2 * q], xv.x, xv.y, c);
                        mma_16816_c(c, af[2 * q + 1], xv.z, xv.w, d);
                    }
#pragma unroll
                    for (int r = 0; r < 4; ++r) p[db][o][r] = c[r];
                }
            }
            // Scale the batch: rows g (C elements 0, 1) and g+8 (2, 3).
#pragma unroll
            for (int db = 0; db < D; ++db) {
                const float s0 = scale_of<GPS>(s_cur[0], b0 + db);
                const float s1 = scale_of<GPS>(s_cur[1], b0 + db);
#pragma unroll
                for (int o = 0; o < MT; ++o) {
                    acc[o][0] = fmaf(s0, p[db][o][0], acc[o][0]);
                    acc[o][1] = fmaf(s0, p[db][o][1], acc[o][1]);
                    acc[o][2] = fmaf(s1, p[db][o][2], acc[o][2]);
                    acc[o][3] = fmaf(s1, p[db][o][3], acc[o][3]);
                }
            }
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
                        ws[size_t(blockIdx.y) * size_t(M) * N + off] = acc[o][r];
                    else
                        Y[off] = f32_to_bf16_rn(acc[o][r]);
                }
            }
        }
        s_cur[0] = s_next[0];
        s_cur[1] = s_next[1];
        if (it + 2 < n_my) load_scales(c0 + (it + 2) * C, s_next);
        if (++ts == KT) { ts = 0; fpar ^= 1; }
    }
}

// Split-K reduce: each thread owns 4 consecutive outputs (one float4 per
// slice).  Loads are issued 8 slices at a time so their latencies overlap; the
// sum itself runs over the slices in ascending order, so the result is the
// same whatever the unrolling.
template <bool kVec>
__global__ void __launch_bounds__(256)
splitk_reduce_kernel(const float *__restrict__ ws, uint16_t *__restrict__ Y, int splits,
                     long long count) {
    pdl_launch_dependents();
    pdl_wait();
    const long long i = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (i >= count) return;
    if (kVec) {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        int s = 0;
        for (; s + 8 <= splits; s += 8) {
            float4 b[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                b[u] = *reinterpret_cast<const float4 *>(ws + size_t(s + u) * count + i);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (s + u == 0) { a = b[u]; continue; }
                a.x += b[u].x; a.y += b[u].y; a.z += b[u].z; a.w += b[u].w;
            }
        }
        for (; s < splits; ++s) {
            const float4 b = *reinterpret_cast<const float4 *>(ws + size_t(s) * count + i);
            if (s == 0) { a = b; continue; }
            a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
        }
        uint2 o;
        o.x = pack_bf16x2_rn(a.x, a.y);
        o.y = pack_bf16x2_rn(a.z, a.w);
        *reinterpret_cast<uint2 *>(Y + i) = o;
    } else {
        const long long end = i + 4 < count ? i + 4 : count;
        for (long long e = i; e < end; ++e) {
            float a = ws[e];
            for (int s = 1; s < splits; ++s) a += ws[size_t(s) * count + e];
            Y[e] = f32_to_bf16_rn(a);
        }
    }
}

template <int MT, int GPS, bool kSplit>
cudaError_t launch_decode_t(const DecodePlan &p, const uint16_t *X, const uint8_t *Wp,
                            const uint16_t *S, uint16_t *Y, float *ws, int M, int N, int K,
                            cudaStream_t s) {
    const int smem = decode_smem_layout(MT, GPS).total;
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
    cfg.gridDim = dim3(p.ctas_per_slice, p.split_k, p.token_blocks);
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
    return cudaLaunchKernelEx(&cfg, kern, X, Wp, S, Y, ws, M, N, K, p.n_tiles, s_vec, err);
}

template <int MT, bool kSplit>
cudaError_t launch_decode_gps(const DecodePlan &p, const uint16_t *X, const uint8_t *Wp,
                              const uint16_t *S, uint16_t *Y, float *ws, int M, int N, int K,
                              cudaStream_t s) {
    switch (p.groups_per_slice) {
        case 1: return launch_decode_t<MT, 1, kSplit>(p, X, Wp, S, Y, ws, M, N, K, s);
        case 2: return launch_decode_t<MT, 2, kSplit>(p, X, Wp, S, Y, ws, M, N, K, s);
        case 4: return launch_decode_t<MT, 4, kSplit>(p, X, Wp, S, Y, ws, M, N, K, s);
        case 8: return launch_decode_t<MT, 8, kSplit>(p, X, Wp, S, Y, ws, M, N, K, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int decode_smem_needed(int M, int mt, int groups_per_slice) {
    (void)M;
    return decode_smem_layout(mt, groups_per_slice).total;
}

cudaError_t launch_decode(const DecodePlan &p, const uint16_t *X, const uint8_t *Wp,
                          const uint16_t *S, uint16_t *Y, float *ws, int M, int N, int K,
                          cudaStream_t s) {
    if (p.groups_per_slice < 1 || p.groups_per_slice > kDecodeMaxGps || p.ctas_per_slice < 1 ||
        decode_smem_needed(M, p.mt, p.groups_per_slice) > kDecodeMaxSmem)
        return cudaErrorInvalidValue;
    if ((K / kGroup) % p.groups_per_slice != 0) return cudaErrorInvalidValue;
    const bool split = p.split_k > 1;
    if (p.mt == 1)
        return split ? launch_decode_gps<1, true>(p, X, Wp, S, Y, ws, M, N, K, s)
                     : launch_decode_gps<1, false>(p, X, Wp, S, Y, ws, M, N, K, s);
    return split ? launch_decode_gps<2, true>(p, X, Wp, S, Y, ws, M, N, K, s)
                 : launch_decode_gps<2, false>(p, X, Wp, S, Y, ws, M, N, K, s);
}

cudaError_t launch_reduce(const float *ws, uint16_t *Y, int splits, long long count, bool pdl,
                          cudaStream_t s) {
    if (count <= 0) return cudaSuccess;
    const bool vec = (count % 4 == 0) && (reinterpret_cast<uintptr_t>(Y) % 8 == 0) &&
                     (reinterpret_cast<uintptr_t>(ws) % 16 == 0);
    const int threads = 256;
    const long long quads = (count + 3) / 4;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned((quads + threads - 1) / threads));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (vec) return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<true>, ws, Y, splits, count);
    return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<false>, ws, Y, splits, count);
}

}  // namespace w4a16
