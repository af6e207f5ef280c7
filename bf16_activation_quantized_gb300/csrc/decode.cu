// decode.cu -- memory-bound arm for few tokens, and the split-K reduce.
//
// Decode arm.  A CTA owns one K slice (a run of whole 128-wide scale groups)
// and a set of 128-row weight tiles (c, c + C, c + 2C, ...).  One producer warp
// streams the 4 KB (tile, chunk) blocks of those tiles, in order, into a ring
// of kStages shared-memory stages with bulk asynchronous copies completed on
// mbarriers; the ring runs across tile boundaries, so HBM never idles between
// tiles (the software pipelining of "[ROCm][Kernel] W4A16 skinny GEMM ...",
// section 2, done with an asynchronous-copy ring).  Each of the 8 consumer
// warps owns one 16-row block of a chunk: its lanes read 512 consecutive bytes
// (consecutive lanes, consecutive bytes -- the access pattern the Q4_K decode
// issue on "gfx1151: 61.7% of Qwen3.8-27B's per-token byte budget ..." shows
// is needed to reach the memory ceiling).  The CTA's slice of X is staged once
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

constexpr int kConsumerWarps = 8;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;   // + one producer warp
constexpr int kStages = 16;                                  // 4 KB chunks in flight per CTA

struct DecodeSmem {
    int x_stride;     // bf16 elements per staged X row (slice + 16 padding)
    int off_ring, off_full, off_empty, off_abort, off_x, off_xsum, total;
};

__host__ __device__ inline DecodeSmem decode_smem_layout(int rows, int gps) {
    DecodeSmem L;
    L.x_stride = gps * kGroup + 16;                  // +32 bytes: rows start 32 banks-bytes apart
    L.off_ring = 0;
    L.off_full = kStages * kChunkBytes;
    L.off_empty = L.off_full + kStages * 8;
    L.off_abort = L.off_empty + kStages * 8;
    L.off_x = L.off_abort + 16;
    L.off_xsum = L.off_x + rows * L.x_stride * 2;
    L.total = L.off_xsum + rows * gps * 4;
    return L;
}

__device__ __forceinline__ float ldg_scale(const uint16_t *p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return bf16_bits_to_f32(v);
}

__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Wait, ignoring the abort flag, for copies still in flight (used only when
// aborting, so that no copy lands after the CTA has exited).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > 100000000ull) break;
}

template <int MT, bool kSplit>
__device__ __forceinline__ void decode_consumer(
    const uint16_t *__restrict__ S, uint16_t *__restrict__ Y, float *__restrict__ ws,
    int M, int N, int n_groups, int grp0, int ngrp, int nck, int m0, int rows, int n_my, int c0,
    int C, const unsigned char *ring, uint32_t full0, uint32_t empty0, const uint16_t *s_x,
    int x_stride, const float *s_xsum, int gps, volatile int *abort_flag, int *err) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;

    bool xok[MT];
    const uint16_t *xs[MT];
#pragma unroll
    for (int o = 0; o < MT; ++o) {
        xok[o] = 8 * o + g < rows;
        xs[o] = s_x + (xok[o] ? 8 * o + g : 0) * x_stride + 4 * t;
    }
    // Per-lane scales of rows g and g+8 of this warp's block, current and next tile.
    float sc[2][kDecodeMaxGps], sn[2][kDecodeMaxGps];
    auto load_scales = [&](int tile, float (&dst)[2][kDecodeMaxGps]) {
        const int f0 = tile * kTileRows + warp * 16 + g;
#pragma unroll
        for (int gi = 0; gi < kDecodeMaxGps; ++gi) {
            dst[0][gi] = (gi < ngrp && f0 < N) ? ldg_scale(S + size_t(f0) * n_groups + grp0 + gi) : 0.f;
            dst[1][gi] = (gi < ngrp && f0 + 8 < N) ? ldg_scale(S + size_t(f0 + 8) * n_groups + grp0 + gi) : 0.f;
        }
    };
    if (n_my > 0) load_scales(c0, sc);

    for (int it = 0; it < n_my; ++it) {
        const int tile = c0 + it * C;
        if (it + 1 < n_my) load_scales(tile + C, sn);
        float acc[MT][4];
#pragma unroll
        for (int o = 0; o < MT; ++o)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[o][r] = 0.f;
#pragma unroll
        for (int gi = 0; gi < kDecodeMaxGps; ++gi) {
            if (gi < ngrp) {
                // Two independent MMA chains, summed once per group.
                float part[2][MT][4];
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2)
#pragma unroll
                    for (int o = 0; o < MT; ++o)
#pragma unroll
                        for (int r = 0; r < 4; ++r) part[q2][o][r] = 0.f;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int c = 2 * gi + h;
                    const int q = it * nck + c;
                    const int st = q & (kStages - 1);
                    if (!mbar_wait(full0 + 8 * st, (q / kStages) & 1, abort_flag, err)) return;
                    const uint4 w = *reinterpret_cast<const uint4 *>(
                        ring + st * kChunkBytes + warp * kBlockBytes + lane * 16);
                    // B fragments: columns 16j + 4t + {0..3} of this lane's X row.
                    uint32_t xb[MT][8];
#pragma unroll
                    for (int o = 0; o < MT; ++o)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint2 v = make_uint2(0, 0);
                            if (xok[o]) v = *reinterpret_cast<const uint2 *>(xs[o] + c * kChunkK + 16 * j);
                            xb[o][2 * j] = v.x;
                            xb[o][2 * j + 1] = v.y;
                        }
                    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
                    uint32_t a[4][4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        a[j][0] = magic_pair(wv[j]);
                        a[j][1] = magic_pair(wv[j] >> 4);
                        a[j][2] = magic_pair(wv[j] >> 8);
                        a[j][3] = magic_pair(wv[j] >> 12);
                    }
                    // The stage's bytes are now in registers: release it.
                    __syncwarp();
                    if (lane == 0) mbar_arrive(empty0 + 8 * st);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int o = 0; o < MT; ++o)
                            mma_16816(part[j & 1][o], a[j], xb[o][2 * j], xb[o][2 * j + 1]);
                }
                const float s0 = sc[0][gi], s1 = sc[1][gi];
#pragma unroll
                for (int o = 0; o < MT; ++o) {
                    const int tk = 8 * o + 2 * t;     // C-fragment tokens tk, tk+1
                    const float x0 = tk < rows ? s_xsum[tk * gps + gi] : 0.f;
                    const float x1 = tk + 1 < rows ? s_xsum[(tk + 1) * gps + gi] : 0.f;
                    const float p0 = part[0][o][0] + part[1][o][0];
                    const float p1 = part[0][o][1] + part[1][o][1];
                    const float p2 = part[0][o][2] + part[1][o][2];
                    const float p3 = part[0][o][3] + part[1][o][3];
                    acc[o][0] = fmaf(s0, fmaf(-136.f, x0, p0), acc[o][0]);
                    acc[o][1] = fmaf(s0, fmaf(-136.f, x1, p1), acc[o][1]);
                    acc[o][2] = fmaf(s1, fmaf(-136.f, x0, p2), acc[o][2]);
                    acc[o][3] = fmaf(s1, fmaf(-136.f, x1, p3), acc[o][3]);
                }
            }
        }
        // C fragment: {row g: tokens 2t, 2t+1}, {row g+8: tokens 2t, 2t+1}.
        const int f0 = tile * kTileRows + warp * 16 + g;
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
#pragma unroll
        for (int gi = 0; gi < kDecodeMaxGps; ++gi) { sc[0][gi] = sn[0][gi]; sc[1][gi] = sn[1][gi]; }
    }
}

template <int MT, bool kSplit>
__global__ void __launch_bounds__(kDecodeThreads, 2)
decode_kernel(const uint16_t *__restrict__ X, const uint8_t *__restrict__ Wp,
              const uint16_t *__restrict__ S, uint16_t *__restrict__ Y, float *__restrict__ ws,
              int M, int N, int K, int gps, int n_tiles, int *err) {
    extern __shared__ __align__(128) unsigned char smem[];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_groups = K / kGroup;
    const int grp0 = blockIdx.y * gps;
    const int ngrp = min(gps, n_groups - grp0);
    const int nck = 2 * ngrp;               // 64-wide chunks per tile in this slice
    const int m0 = blockIdx.z * 8 * MT;
    const int rows = min(8 * MT, M - m0);
    const int C = gridDim.x;
    const int c0 = blockIdx.x;
    const int n_my = c0 < n_tiles ? (n_tiles - c0 + C - 1) / C : 0;
    const int total = n_my * nck;
    const int KC = K / kChunkK;
    const DecodeSmem L = decode_smem_layout(rows, gps);
    const unsigned char *ring = smem + L.off_ring;
    const uint32_t full0 = smem_u32(smem + L.off_full);
    const uint32_t empty0 = smem_u32(smem + L.off_empty);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.off_abort);
    uint16_t *s_x = reinterpret_cast<uint16_t *>(smem + L.off_x);
    float *s_xsum = reinterpret_cast<float *>(smem + L.off_xsum);

    // Let the next kernel in the stream be scheduled while this grid runs.
    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kConsumerWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // Touch no global memory before the previous grid in the stream has completed.
    pdl_wait();

    if (warp == kConsumerWarps) {
        // Producer: one lane streams every (tile, chunk) of this CTA through the ring.
        if (lane == 0) {
            int issued = 0;
            for (int q = 0; q < total; ++q) {
                const int st = q & (kStages - 1);
                if (q >= kStages && !mbar_wait(empty0 + 8 * st, ((q / kStages) - 1) & 1, abort_flag, err))
                    break;
                const int it = q / nck;
                const int c = q - it * nck;
                const int tile = c0 + it * C;
                const uint8_t *src = Wp + (size_t(tile) * KC + size_t(2 * grp0 + c)) * kChunkBytes;
                mbar_arrive_expect_tx(full0 + 8 * st, kChunkBytes);
                bulk_g2s(smem_u32(ring + st * kChunkBytes), src, kChunkBytes, full0 + 8 * st);
                issued = q + 1;
            }
            if (*abort_flag) {
                for (int q = issued > kStages ? issued - kStages : 0; q < issued; ++q)
                    drain_wait(full0 + 8 * (q & (kStages - 1)), (q / kStages) & 1);
            }
        }
        return;
    }

    // Consumers: stage X[m0 .. m0+rows)[slice] and the per-(token, group) sums.
    const int vec_per_row = ngrp * (kGroup / 8);
    for (int i = threadIdx.x; i < rows * vec_per_row; i += kConsumerWarps * 32) {
        const int r = i / vec_per_row, v = i - r * vec_per_row;
        const uint4 val = ldg_nc16(X + size_t(m0 + r) * K + size_t(grp0) * kGroup + v * 8);
        *reinterpret_cast<uint4 *>(s_x + r * L.x_stride + v * 8) = val;
    }
    consumer_bar();
    {
        // 8 lanes per sum, 16 values each, then a shuffle reduction within the 8 lanes.
        const int pairs = rows * ngrp;
        const int part = threadIdx.x & 7;
        for (int base = 0; base < pairs; base += kConsumerWarps * 32 / 8) {
            const int pi = base + (threadIdx.x >> 3);
            float a = 0.f;
            if (pi < pairs) {
                const int r = pi / ngrp, gi = pi - r * ngrp;
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
                const int r = pi / ngrp, gi = pi - r * ngrp;
                s_xsum[r * gps + gi] = a;
            }
        }
    }
    consumer_bar();

    decode_consumer<MT, kSplit>(S, Y, ws, M, N, n_groups, grp0, ngrp, nck, m0, rows, n_my, c0, C,
                                ring, full0, empty0, s_x, L.x_stride, s_xsum, gps, abort_flag, err);
}

template <bool kVec>
__global__ void __launch_bounds__(256)
splitk_reduce_kernel(const float *__restrict__ ws, uint16_t *__restrict__ Y, int splits,
                     long long count) {
    pdl_launch_dependents();
    pdl_wait();
    const long long i = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (i >= count) return;
    if (kVec) {
        float4 a = *reinterpret_cast<const float4 *>(ws + i);
        for (int s = 1; s < splits; ++s) {
            const float4 b = *reinterpret_cast<const float4 *>(ws + size_t(s) * count + i);
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

template <int MT, bool kSplit>
cudaError_t launch_decode_t(const DecodePlan &p, const uint16_t *X, const uint8_t *Wp,
                            const uint16_t *S, uint16_t *Y, float *ws, int M, int N, int K,
                            cudaStream_t s) {
    const int rows = M < 8 * MT ? M : 8 * MT;
    const int smem = decode_smem_layout(rows, p.groups_per_slice).total;
    auto kern = decode_kernel<MT, kSplit>;
    // Opt in to more than 48 KB of shared memory once per device (not a stream
    // operation, so it is also safe while a graph is being captured).
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
    int *err = device_error_word();
    if (!err) return cudaErrorUnknown;
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
    return cudaLaunchKernelEx(&cfg, kern, X, Wp, S, Y, ws, M, N, K, p.groups_per_slice, p.n_tiles,
                              err);
}

}  // namespace

int decode_smem_needed(int M, int mt, int groups_per_slice) {
    const int rows = M < 8 * mt ? M : 8 * mt;
    return decode_smem_layout(rows, groups_per_slice).total;
}

cudaError_t launch_decode(const DecodePlan &p, const uint16_t *X, const uint8_t *Wp,
                          const uint16_t *S, uint16_t *Y, float *ws, int M, int N, int K,
                          cudaStream_t s) {
    if (p.groups_per_slice < 1 || p.groups_per_slice > kDecodeMaxGps || p.ctas_per_slice < 1 ||
        decode_smem_needed(M, p.mt, p.groups_per_slice) > kDecodeMaxSmem)
        return cudaErrorInvalidValue;
    const bool split = p.split_k > 1;
    if (p.mt == 1)
        return split ? launch_decode_t<1, true>(p, X, Wp, S, Y, ws, M, N, K, s)
                     : launch_decode_t<1, false>(p, X, Wp, S, Y, ws, M, N, K, s);
    return split ? launch_decode_t<2, true>(p, X, Wp, S, Y, ws, M, N, K, s)
                 : launch_decode_t<2, false>(p, X, Wp, S, Y, ws, M, N, K, s);
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
