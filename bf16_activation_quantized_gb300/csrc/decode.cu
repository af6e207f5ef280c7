// decode.cu -- decode-arm launchers, the whole-K decode kernel and the split-K
// reduce.  The sliced decode kernel is in decode_slices.cuh; its instantiations
// for 64- and 32-wide scale groups live in decode_g64.cu and decode_g32.cu, and
// its zero-point instantiations in decode_zp.cu, so that they compile in
// parallel.
#include <atomic>

#include "decode_slices.cuh"

namespace w4a16 {

namespace {

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
    int off_ring, off_bar, off_abort, off_xmax, off_x, off_scale, off_red, total;
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
    L.off_scale = L.off_x + ((rows * L.x_stride * 2 + 15) & ~15);
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
    // Convert X in place to fp16 x * 2^-sh(token, part) (as decode_kernel):
    // 8 lanes per (token, group).
    {
        const int pairs = rows * G;
        const int part = threadIdx.x & 7;
        for (int pi = threadIdx.x >> 3; pi < pairs; pi += kDecodeWarps * 32 / 8) {
            const int r = pi / G, gi = pi - r * G;
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
                    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(hv[e]) : "f"(hi * down), "f"(lo * down));
                }
                src[hh] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
            }
        }
    }
    consumer_bar();

    const int b = warp % B, kp = warp / B;
    const int ga = wk_part_start(kp, P, G), gb = wk_part_start(kp + 1, P, G);
    const int n_st = (gb - ga + SG - 1) / SG;
    const uint16_t *xs = s_x + min(g, rows - 1) * L.x_stride + t * 8;
    const uint16_t *srow = s_scale + (b * 16 + g) * G;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const unsigned char *wlane = ring + b * kBlockBytes + lane * 16;
    bool alive = true;
    for (int j = 0; j < n_st && alive; ++j) {
        const int slot = kp + P * (j % B);
        // Warp-uniform outcome: the MMAs below need every lane.
        if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * slot, (j / B) & 1, abort_flag, err))) {
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
            // Exact A operands code - 8 (rows g) and 16 (code - 8) (rows g + 8),
            // as in decode_kernel.
            uint32_t af[8][4];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const uint32_t w8 = wv[gg][jj] >> 8;
                af[jj][0] = f16x2_sub(lop3_and_or(wv[gg][jj], 0x000F000Fu, kMagicF16x2_1024), kF16x2_1032);
                af[jj][1] = f16x2_sub(lop3_and_or(wv[gg][jj], 0x00F000F0u, kMagicF16x2_1024), kF16x2_1152);
                af[jj][2] = f16x2_sub(lop3_and_or(w8, 0x000F000Fu, kMagicF16x2_1024), kF16x2_1032);
                af[jj][3] = f16x2_sub(lop3_and_or(w8, 0x00F000F0u, kMagicF16x2_1024), kF16x2_1152);
            }
            float c[4] = {0.f, 0.f, 0.f, 0.f};
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
    // A wait of this CTA ran out (every consumer warp has passed the barrier
    // above, so the flag covers them all): the outputs become NaN, never a
    // plausible partial result; the error word holds kErrWaitTimeout.
    if (!alive || *abort_flag) {
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[r] = __int_as_float(0x7fc00000);
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

int decode_smem_needed(int M, int mt, int groups_per_slice, int sub) {
    return decode_smem_layout(mt, M < 8 * mt ? M : 8 * mt, groups_per_slice, sub).total;
}

int decode_ring_stages(int M, int mt, int groups_per_slice, int sub) {
    const int st = decode_smem_layout(mt, M < 8 * mt ? M : 8 * mt, groups_per_slice, sub).stages;
    return st >= decode_ring_min(groups_per_slice) ? st : 0;
}

cudaError_t launch_decode(const DecodePlan &p, const uint16_t *X, const uint8_t *Wp,
                          const uint16_t *S, uint16_t *Y, float *ws, bool res, int M, int N, int K,
                          cudaStream_t s, const uint8_t *Z) {
    if (p.in_flight < 0 || p.in_flight > p.ring || p.wait_us < 0) return cudaErrorInvalidValue;
    // in_flight == 0 (test-only stall) only together with a short wait limit.
    if (p.in_flight == 0 && (p.wait_us == 0 || p.wait_us > 100000)) return cudaErrorInvalidValue;
    if (p.batch < 1 || (long long)p.token_blocks * p.batch > 65535) return cudaErrorInvalidValue;
    if (p.sub != 1 && p.sub != 2 && p.sub != 4) return cudaErrorInvalidValue;
    if (p.groups_per_slice < 1 || p.groups_per_slice > kDecodeMaxGps || p.ctas_per_slice < 1 ||
        p.groups_per_slice * p.sub > (p.mt == 1 ? 16 : 8) / (Z ? 2 : 1) ||
        decode_smem_needed(M, p.mt, p.groups_per_slice, p.sub) > kDecodeMaxSmem ||
        decode_smem_layout(p.mt, M < 8 * p.mt ? M : 8 * p.mt, p.groups_per_slice, p.sub).stages !=
            p.ring ||
        p.ring < decode_ring_min(p.groups_per_slice))
        return cudaErrorInvalidValue;
    if ((K / kGroup) % p.groups_per_slice != 0) return cudaErrorInvalidValue;
    if (Z) return launch_decode_zp(p, X, Wp, S, Z, Y, ws, res, M, N, K, s);
    if (p.sub == 2) return launch_decode_sub2(p, X, Wp, S, Y, ws, res, M, N, K, s);
    if (p.sub == 4) return launch_decode_sub4(p, X, Wp, S, Y, ws, res, M, N, K, s);
    return launch_decode_sub<1>(p, X, Wp, S, nullptr, Y, ws, res, M, N, K, s);
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
