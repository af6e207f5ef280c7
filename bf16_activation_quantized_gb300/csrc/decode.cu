// decode.cu -- memory-bound arm for few tokens, and the split-K reduce.
//
// Decode arm.  A CTA owns one 128-row weight tile and one K slice (a run of
// whole 128-wide scale groups); each of its 8 warps owns a 16-row block.  A
// lane streams its block's K chunks as 16-byte loads, so the 32 lanes of a warp
// read 512 consecutive bytes per chunk (consecutive lanes, consecutive bytes --
// the access pattern the Q4_K decode issue on "gfx1151: 61.7% of
// Qwen3.8-27B's per-token byte budget ..." shows is needed to reach the memory
// ceiling).  The loads run a ring of kRing chunks ahead of the math (the
// software pipelining of "[ROCm][Kernel] W4A16 skinny GEMM ...", section 2,
// done with a register ring instead of a second register set per iteration).
//
// Each 32-bit word becomes, with one LOP3 and one bf16x2 FMA per register, the
// A fragment (exact codes minus 8) of an m16n8k16 bf16 mma.sync whose B
// fragment is 8 tokens of X, so the K reduction across a quad of lanes happens
// inside the tensor core instead of a shuffle tree.  Partial sums of one
// 128-wide group start from zero and are scaled in fp32 once per group
// (acc += scale * partial), which keeps the weights exact.  With split-K the
// fp32 partials go to a [SPLIT_K][M][N] workspace with plain stores and a
// separate kernel sums the slices in order ("Add Triton BF16xINT4 rowwise GEMM
// for ROCm gfx942/gfx950", "Split-K without atomics"); that kernel is chained
// with programmatic dependent launch so its launch overlaps this one.
#include "common.cuh"
#include "internal.h"

namespace w4a16 {

namespace {

constexpr int kDecodeWarps = 8;
constexpr int kRing = 8;              // W chunks in flight per lane
constexpr int kMaxGroupsPerSlice = 64;
constexpr int kScaleStride = kMaxGroupsPerSlice + 1;  // odd stride: rows land in different banks

template <int MT, bool kSplit>
__global__ void __launch_bounds__(kDecodeWarps * 32, 2)
decode_kernel(const uint16_t *__restrict__ X, const uint8_t *__restrict__ Wp,
              const uint16_t *__restrict__ S, uint16_t *__restrict__ Y, float *__restrict__ ws,
              int M, int N, int K, int groups_per_slice) {
    __shared__ float s_scale[kTileRows * kScaleStride];

    if (kSplit) pdl_launch_dependents();

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int tile = blockIdx.x;
    const int n_groups = K / kGroup;
    const int grp0 = blockIdx.y * groups_per_slice;
    const int grp1 = min(grp0 + groups_per_slice, n_groups);
    const int ngrp = grp1 - grp0;
    const int nck = 2 * ngrp;               // 64-wide chunks in this slice
    const int m0 = blockIdx.z * 8 * MT;
    const int KC = K / kChunkK;

    // Scales of this CTA's 128 rows for the slice's groups, as fp32.
    for (int i = threadIdx.x; i < kTileRows * ngrp; i += blockDim.x) {
        const int r = i / ngrp, gi = i - r * ngrp;
        const int row = tile * kTileRows + r;
        s_scale[r * kScaleStride + gi] =
            row < N ? bf16_bits_to_f32(S[size_t(row) * n_groups + grp0 + gi]) : 0.f;
    }

    // This lane's 16 bytes of chunk c: tile-major, chunk, block, lane.
    const uint8_t *wlane = Wp + (size_t(tile) * KC + size_t(2 * grp0)) * kChunkBytes +
                           size_t(warp) * kBlockBytes + size_t(lane) * 16;

    // X rows this lane feeds into the B fragments: token m0 + 8*o + g.
    const uint16_t *xrow[MT];
    bool xok[MT];
#pragma unroll
    for (int o = 0; o < MT; ++o) {
        const int m = m0 + 8 * o + g;
        xok[o] = m < M;
        xrow[o] = X + size_t(xok[o] ? m : 0) * K + size_t(2 * grp0) * kChunkK + 16 * t;
    }

    uint4 wr[kRing];
#pragma unroll
    for (int u = 0; u < kRing; ++u)
        if (u < nck) wr[u] = ldg_stream16(wlane + size_t(u) * kChunkBytes);

    __syncthreads();

    float acc[MT][4], part[MT][4];
#pragma unroll
    for (int o = 0; o < MT; ++o)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[o][r] = 0.f;

    const float *srow0 = s_scale + (warp * 16 + g) * kScaleStride;
    const float *srow1 = srow0 + 8 * kScaleStride;

    for (int base = 0; base < nck; base += kRing) {
#pragma unroll
        for (int u = 0; u < kRing; ++u) {
            const int c = base + u;
            if (c < nck) {
                if ((u & 1) == 0) {
#pragma unroll
                    for (int o = 0; o < MT; ++o)
#pragma unroll
                        for (int r = 0; r < 4; ++r) part[o][r] = 0.f;
                }
                // B fragments: 16 columns of this lane's X row, as 8 bf16 pairs.
                uint32_t xb[MT][8];
#pragma unroll
                for (int o = 0; o < MT; ++o) {
                    uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
                    if (xok[o]) {
                        lo = ldg_nc16(xrow[o] + size_t(c) * kChunkK);
                        hi = ldg_nc16(xrow[o] + size_t(c) * kChunkK + 8);
                    }
                    xb[o][0] = lo.x; xb[o][1] = lo.y; xb[o][2] = lo.z; xb[o][3] = lo.w;
                    xb[o][4] = hi.x; xb[o][5] = hi.y; xb[o][6] = hi.z; xb[o][7] = hi.w;
                }
                const uint32_t wv[4] = {wr[u].x, wr[u].y, wr[u].z, wr[u].w};
                if (c + kRing < nck) wr[u] = ldg_stream16(wlane + size_t(c + kRing) * kChunkBytes);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t a[4];
                    dequant_word_frag(wv[j], a);
#pragma unroll
                    for (int o = 0; o < MT; ++o) mma_16816(part[o], a, xb[o][2 * j], xb[o][2 * j + 1]);
                }
                if (u & 1) {
                    const int gi = c >> 1;
                    const float s0 = srow0[gi], s1 = srow1[gi];
#pragma unroll
                    for (int o = 0; o < MT; ++o) {
                        acc[o][0] = fmaf(s0, part[o][0], acc[o][0]);
                        acc[o][1] = fmaf(s0, part[o][1], acc[o][1]);
                        acc[o][2] = fmaf(s1, part[o][2], acc[o][2]);
                        acc[o][3] = fmaf(s1, part[o][3], acc[o][3]);
                    }
                }
            }
        }
    }

    // C fragment: {row g: tokens 2t, 2t+1}, {row g+8: tokens 2t, 2t+1}.
    const int f0 = tile * kTileRows + warp * 16 + g;
    const int f1 = f0 + 8;
#pragma unroll
    for (int o = 0; o < MT; ++o) {
        const int ma = m0 + 8 * o + 2 * t;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int m = ma + (r & 1);
            const int f = (r < 2) ? f0 : f1;
            if (m < M && f < N) {
                const size_t off = size_t(m) * N + f;
                if (kSplit)
                    ws[size_t(blockIdx.y) * size_t(M) * N + off] = acc[o][r];
                else
                    Y[off] = f32_to_bf16_rn(acc[o][r]);
            }
        }
    }
}

template <bool kVec>
__global__ void __launch_bounds__(256)
splitk_reduce_kernel(const float *__restrict__ ws, uint16_t *__restrict__ Y, int splits,
                     long long count) {
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
    dim3 grid(p.n_tiles, p.split_k, p.token_blocks);
    decode_kernel<MT, kSplit><<<grid, kDecodeWarps * 32, 0, s>>>(X, Wp, S, Y, ws, M, N, K,
                                                                 p.groups_per_slice);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodePlan &p, const uint16_t *X, const uint8_t *Wp,
                          const uint16_t *S, uint16_t *Y, float *ws, int M, int N, int K,
                          cudaStream_t s) {
    if (p.groups_per_slice > kMaxGroupsPerSlice || p.groups_per_slice < 1)
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
