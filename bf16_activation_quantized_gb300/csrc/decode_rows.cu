// decode_rows.cu -- the whole-K decode kernel: no split-K, no reduce kernel.
//
// A CTA owns B consecutive 16-row blocks of one 128-row tile over all of K and
// writes their Y rows itself, so a call is one launch.  Its producer warp
// streams the blocks' packed weights through a ring of 16 KB stages, one 3-D
// TMA box per stage (the blocks' 512-byte pieces of 2 * SG consecutive
// 64-column chunks; SG = 16 / B groups of 128 columns per stage), and puts the
// same SG groups of the M activation rows next to them in the stage (one bulk
// copy per token).  The weights are read before the dependency wait when they
// are resident; X only after it, so the previous kernel on the stream may
// write X.  There is no activation prologue: the first stage's X arrives with
// the stage.
//
// Consumer warp w takes block w % B and, in every stage, groups 2 (w / B) and
// 2 (w / B) + 1 of the stage (P = 8 / B warps share a block, each covering a
// quarter, half ... of K in interleaved pairs of groups), for all M tokens:
// MT = ceil(M / 8) token octets (up to two), each dequantised A fragment
// feeding one m16n8k16 per octet, so the weights are streamed once.  Per
// group it builds the bf16 A fragments 128 + code with one LOP3 per register
// and removes 136 with one exact bf16x2 FMA (the magic-constant trick of
// "[ROCm][Kernel] W4A16 skinny GEMM: hand-asm kernel for gfx1151", section
// 1), so the m16n8k16 chain over the group multiplies exact codes - 8 by the
// bf16 X fragments taken from the stage as they are; the fp32 group scale
// multiplies the chain's sum.  At the end the P warps of a block add their sums in shared
// memory in ascending order and the first writes Y.
#include <atomic>

#include "async.cuh"
#include "common.cuh"
#include "internal.h"

namespace w4a16 {

namespace {

// Consumer warps.  Measured on GB300: 8 warps with two groups of a stage each
// (two independent MMA chains per warp) ran the decode GEMV shapes 10-15 %
// faster than 16 warps with one group each.
constexpr int kRowsWarps = 8;
constexpr int kRowsThreads = (kRowsWarps + 1) * 32;   // + the producer warp
constexpr int kRowsGW = 16 / kRowsWarps;              // groups per warp per stage
constexpr int kRowsStageW = 16384;                    // packed weight bytes per stage
constexpr int kRowsMaxStages = 8;
// Two token octets at most.  Measured on GB300: with four (32 tokens, 128
// rows per CTA, three 33 KB stages) a stage takes ~1.3 us -- the X fragments
// (as many bytes per stage as the weights) hold each stage until its MMAs are
// done, and the ring then keeps too few weight bytes in flight -- slower than
// the tensor arm.
constexpr int kRowsMaxTokens = 16;

// c += A . B for one m16n8k16 bf16 tile, fp32 accumulators in place.
__device__ __forceinline__ void mma_bf16_acc(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Shared memory: the ring (per stage 16 KB of weights, then the M activation
// rows of the stage's groups at x_stride bytes each), the CTA's scales
// transposed (bf16 [G][16 B rows]: the 8 rows a warp reads for one group are
// adjacent, one bank wavefront), the ring's barriers and the abort flag.  The
// K-parts' partial sums are exchanged through ring stage 0 once the ring is
// drained.
struct RowsSmem {
    int sg, parts, stages, x_stride, stage_bytes;
    int off_ring, off_scale, off_bar, off_abort, total;
};

__host__ __device__ inline RowsSmem rows_smem_layout(int B, int M, int G, int budget) {
    RowsSmem L;
    L.sg = 16 / B;
    L.parts = kRowsWarps / B;
    L.x_stride = L.sg * kGroup * 2 + 32;            // 32 B pad: conflict-free 8-byte fragment loads
    L.stage_bytes = (kRowsStageW + M * L.x_stride + 127) & ~127;   // TMA destinations: 128-byte aligned
    const int scale_bytes = (B * 16 * G * 2 + 15) & ~15;
    const int fixed = scale_bytes + 2 * kRowsMaxStages * 8 + 16;
    int n = (budget - fixed - 128) / L.stage_bytes;    // 128: base alignment slack
    L.stages = n > kRowsMaxStages ? kRowsMaxStages : n;
    L.off_ring = 0;
    L.off_scale = L.stages * L.stage_bytes;
    L.off_bar = L.off_scale + scale_bytes;
    L.off_abort = L.off_bar + 2 * kRowsMaxStages * 8;
    L.total = L.off_abort + 16 + 128;
    return L;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tmap, int x, int y, int z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void rows_consumer_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(kRowsWarps * 32) : "memory");
}

// wmap: the packed weights as uint32 [chunk rows][8 blocks][128] with a box of
// {128, B, 2 SG}; wmap_tail: the same with a box of {128, B, 2 (G % SG)} for a
// last stage of fewer groups (unused when SG divides G).  Batch entry b's
// chunk rows follow entry b - 1's.  MT: token octets (M <= 8 MT).
template <int B, int MT>
__global__ void __launch_bounds__(kRowsThreads, 2)
decode_rows_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap wmap_tail,
                   const uint16_t *__restrict__ X, const uint16_t *__restrict__ S,
                   uint16_t *__restrict__ Y, int M, int N, int K, int resident, int s_vec, int *err) {
    constexpr int SG = 16 / B;                 // groups per stage
    constexpr int P = kRowsWarps / B;          // warps per block (K-parts)
    constexpr int GW = kRowsGW;                // groups per warp per stage (SG = P * GW)
    extern __shared__ __align__(128) unsigned char smem_raw[];
    // 128-byte alignment for the TMA destinations (the layout reserves the slack).
    unsigned char *smem = smem_raw + ((128 - (smem_u32(smem_raw) & 127)) & 127);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = K / kGroup;
    const int KC = K / kChunkK;
    const int n_tiles = (N + kTileRows - 1) / kTileRows;
    const int bz = blockIdx.y;                 // batch entry
    X += size_t(bz) * M * K;
    S += size_t(bz) * N * G;
    Y += size_t(bz) * M * N;
    const int blk0 = blockIdx.x * B;           // first 16-row block (B divides 8: one tile)
    const int tile = blk0 / 8, bb = blk0 % 8;
    const int row0 = tile * kTileRows + bb * 16;
    const int n_st = (G + SG - 1) / SG;
    const RowsSmem L = rows_smem_layout(B, M, G, kDecodeMaxSmem);
    const int NS = L.stages;
    unsigned char *ring = smem + L.off_ring;
    uint16_t *s_scale = reinterpret_cast<uint16_t *>(smem + L.off_scale);
    const uint32_t full0 = smem_u32(smem + L.off_bar);
    const uint32_t empty0 = full0 + 8 * kRowsMaxStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.off_abort);

    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kRowsWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kRowsWarps) {
        // Producer warp.  Stage q = groups [q SG, q SG + SG) of the CTA's
        // blocks; its barrier expects the weight box and the M activation
        // rows.  The whole warp runs the loop: one elected lane posts the
        // expected bytes and issues the weight box, then lane m < M issues
        // token m's activation row.
        if (elect_one()) tma_prefetch_desc(&wmap);
        const bool tail = (G % SG) != 0;
        const int zrow0 = (bz * n_tiles + tile) * KC;
        auto groups_of = [&](int q) { return min(SG, G - q * SG); };
        auto bytes_of = [&](int q) {
            const int ng = groups_of(q);
            return uint32_t(2 * ng * B * 512 + M * ng * kGroup * 2);
        };
        auto issue_w = [&](int q, int st) {      // one lane
            const CUtensorMap *m = (tail && q == n_st - 1) ? &wmap_tail : &wmap;
            mbar_arrive_expect_tx(full0 + 8 * st, bytes_of(q));
            tma_load_3d(smem_u32(ring + st * L.stage_bytes), m, 0, bb, zrow0 + 2 * SG * q, full0 + 8 * st);
        };
        auto issue_x = [&](int q, int st) {      // lane m: token m
            if (lane < M) {
                const uint32_t nb = uint32_t(groups_of(q) * kGroup * 2);
                unsigned char *dst = ring + st * L.stage_bytes + kRowsStageW + lane * L.x_stride;
                bulk_g2s(smem_u32(dst), X + size_t(lane) * K + size_t(q) * SG * kGroup, nb, full0 + 8 * st);
            }
        };
        int q0 = 0, issued = 0;
        if (resident) {
            // The weights of the first stages stream in while the previous
            // kernel finishes; X follows once it has completed.
            q0 = min(NS, n_st);
            if (elect_one())
                for (int q = 0; q < q0; ++q) issue_w(q, q);
            __syncwarp();
            pdl_wait();
            for (int q = 0; q < q0; ++q) issue_x(q, q);
            issued = q0;
        } else {
            pdl_wait();
        }
        // Ring slot and the parity of its empty phase, kept as counters
        // (no division by the runtime ring depth in the loop).
        int st = q0 % NS;
        uint32_t epar = uint32_t(q0 / NS + 1) & 1u;
        for (int q = q0; q < n_st; ++q) {
            if (q >= NS && !__all_sync(0xffffffffu, mbar_wait(empty0 + 8 * st, epar, abort_flag, err))) break;
            if (elect_one()) issue_w(q, st);
            __syncwarp();
            issue_x(q, st);
            ++issued;
            if (++st == NS) { st = 0; epar ^= 1u; }
        }
        if (*abort_flag) {
            // Let every copy issued land before the CTA exits.
            for (int q = issued > NS ? issued - NS : 0; q < issued; ++q)
                drain_wait(full0 + 8 * (q % NS), (q / NS) & 1);
        }
        return;
    }

    // ---- consumers (256 threads) ----
    const int g = lane >> 2, t = lane & 3;
    const int b = warp % B, kp = warp / B;
    // Scales of the CTA's 16 B rows (rows past N read as 0), stored
    // transposed.  Consecutive lanes take consecutive rows, each reading 8
    // scales of its row (one 16-byte vector when S allows), so the transposed
    // 2-byte stores of a warp fall in distinct banks.  With resident weights
    // they are loaded while the previous kernel finishes.
    {
        if (!resident) pdl_wait();
        constexpr int R = B * 16;
        const int CH = (G + 7) / 8;
        for (int idx = threadIdx.x; idx < R * CH; idx += kRowsWarps * 32) {
            const int r = idx % R, c = idx / R;
            const bool row_ok = row0 + r < N;
            const uint16_t *src = S + size_t(row0 + r) * G + 8 * c;
            uint16_t e[8];
            if (s_vec && row_ok) {
                const uint4 v = ldg_nc16(src);
                const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    e[2 * u] = uint16_t(vv[u] & 0xFFFFu);
                    e[2 * u + 1] = uint16_t(vv[u] >> 16);
                }
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u) e[u] = (row_ok && 8 * c + u < G) ? src[u] : uint16_t(0);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (8 * c + u < G) s_scale[(8 * c + u) * R + r] = e[u];
        }
        rows_consumer_bar();
    }
    const uint16_t *scol = s_scale + b * 16 + g;               // row g of this warp's block, group 0
    // Octet o's token g; absent tokens read the last row (their sums are dropped).
    int xrow[MT];
#pragma unroll
    for (int o = 0; o < MT; ++o) xrow[o] = min(8 * o + g, M - 1);
    float acc[MT][4];
#pragma unroll
    for (int o = 0; o < MT; ++o)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[o][r] = 0.f;
    bool alive = true;
    int slot = 0;
    uint32_t fpar = 0;       // parity of the slot's full phase
    for (int q = 0; q < n_st; ++q) {
        // Warp-uniform outcome: the MMAs below need every lane.
        if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * slot, fpar, abort_flag, err))) {
            alive = false;
            break;
        }
        const unsigned char *st = ring + slot * L.stage_bytes;
        const int ng = min(SG, G - q * SG);
        // This warp's two groups of the stage: packed words (16 B of each of
        // the group's two 64-column chunks) and, per octet, the X fragments of
        // its 8 k16 steps (token 8 o + g, columns 16 j + 4 t .. + 3: the k
        // slots 2t, 2t+1, 2t+8, 2t+9 of the packed word j).  A group past the
        // last (in a short final stage) is read and multiplied all the same --
        // its bytes lie inside the stage -- and only its sum is dropped, so
        // the loads and MMAs carry no branches and interleave freely.  With
        // one octet the X fragments are loaded up front and the stage is
        // released before the MMAs; with more they are loaded per k16 step
        // (registers) and the stage is released after them.
        uint32_t wv[GW][8];
#pragma unroll
        for (int h = 0; h < GW; ++h) {
            const int gg = GW * kp + h;
            const uint4 wa = *reinterpret_cast<const uint4 *>(st + ((2 * gg) * B + b) * 512 + lane * 16);
            const uint4 wb = *reinterpret_cast<const uint4 *>(st + ((2 * gg + 1) * B + b) * 512 + lane * 16);
            wv[h][0] = wa.x; wv[h][1] = wa.y; wv[h][2] = wa.z; wv[h][3] = wa.w;
            wv[h][4] = wb.x; wv[h][5] = wb.y; wv[h][6] = wb.z; wv[h][7] = wb.w;
        }
        auto xfrag = [&](int o, int h, int j) {
            return *reinterpret_cast<const uint2 *>(st + kRowsStageW + xrow[o] * L.x_stride +
                                                    (GW * kp + h) * kGroup * 2 + 8 * t + 32 * j);
        };
        uint2 xf1[GW][8];             // MT == 1 only
        if constexpr (MT == 1) {
#pragma unroll
            for (int h = 0; h < GW; ++h)
#pragma unroll
                for (int j = 0; j < 8; ++j) xf1[h][j] = xfrag(0, h, j);
            // Operands are in registers: release the stage.
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * slot);
        }
        float c[GW][MT][4];
#pragma unroll
        for (int h = 0; h < GW; ++h)
#pragma unroll
            for (int o = 0; o < MT; ++o)
#pragma unroll
                for (int r = 0; r < 4; ++r) c[h][o][r] = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
#pragma unroll
            for (int h = 0; h < GW; ++h) {
                const uint32_t w = wv[h][j];
                // {row g: cols +0, +1}, {row g+8: +0, +1}, {row g: +2, +3}, {row g+8: +2, +3}
                // minus136: one exact bf16x2 FMA, (128 + code) * 1 - 136.
                const uint32_t a[4] = {minus136(magic_pair(w)), minus136(magic_pair(w >> 4)),
                                       minus136(magic_pair(w >> 8)), minus136(magic_pair(w >> 12))};
#pragma unroll
                for (int o = 0; o < MT; ++o) {
                    const uint2 x = MT == 1 ? xf1[h][j] : xfrag(o, h, j);
                    mma_bf16_acc(c[h][o], a, x.x, x.y);
                }
            }
        }
        if constexpr (MT > 1) {
            // The X fragments have been read: release the stage.
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * slot);
        }
#pragma unroll
        for (int h = 0; h < GW; ++h) {
            const int gi = q * SG + GW * kp + h;
            if (GW * kp + h >= ng) continue;
            const float s0 = bf16_bits_to_f32(scol[gi * 16 * B]);
            const float s1 = bf16_bits_to_f32(scol[gi * 16 * B + 8]);
#pragma unroll
            for (int o = 0; o < MT; ++o) {
                acc[o][0] = fmaf(s0, c[h][o][0], acc[o][0]);
                acc[o][1] = fmaf(s0, c[h][o][1], acc[o][1]);
                acc[o][2] = fmaf(s1, c[h][o][2], acc[o][2]);
                acc[o][3] = fmaf(s1, c[h][o][3], acc[o][3]);
            }
        }
        if (++slot == NS) {
            slot = 0;
            fpar ^= 1u;
        }
    }
    // Add the K-parts in ascending order through ring stage 0 (every stage
    // has been consumed, so the ring is idle; (8 - B) MT x 512 bytes fit in a
    // stage); part 0's warps write Y.
    rows_consumer_bar();
    float4 *red = reinterpret_cast<float4 *>(ring);
    if (kp > 0) {
#pragma unroll
        for (int o = 0; o < MT; ++o)
            red[(((kp - 1) * B + b) * MT + o) * 32 + lane] = make_float4(acc[o][0], acc[o][1], acc[o][2], acc[o][3]);
    }
    rows_consumer_bar();
    if (kp > 0) return;
#pragma unroll
    for (int p = 1; p < P; ++p) {
#pragma unroll
        for (int o = 0; o < MT; ++o) {
            const float4 v = red[(((p - 1) * B + b) * MT + o) * 32 + lane];
            acc[o][0] += v.x; acc[o][1] += v.y; acc[o][2] += v.z; acc[o][3] += v.w;
        }
    }
    // A wait of this CTA ran out (every consumer warp has passed the barriers
    // above, so the flag covers them all): the outputs become NaN, never a
    // plausible partial result; the error word holds kErrWaitTimeout.
    if (!alive || *abort_flag) {
#pragma unroll
        for (int o = 0; o < MT; ++o)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[o][r] = __int_as_float(0x7fc00000);
    }
    // Y may be read by the previous kernel on the stream: write it only after
    // that kernel has completed.
    pdl_wait();
    const int f0 = row0 + b * 16 + g;
#pragma unroll
    for (int o = 0; o < MT; ++o) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int m = 8 * o + 2 * t + (r & 1);
            const int f = f0 + ((r < 2) ? 0 : 8);
            if (m < M && f < N) Y[size_t(m) * N + f] = f32_to_bf16_rn(acc[o][r]);
        }
    }
}

template <int B, int MT>
cudaError_t launch_rows_t(int ctas, int batch, const uint16_t *X, const uint8_t *Wp, const uint16_t *S,
                          uint16_t *Y, bool resident, int M, int N, int K, cudaStream_t s) {
    const int G = K / kGroup;
    const int KC = K / kChunkK;
    const int n_tiles = (N + kTileRows - 1) / kTileRows;
    const RowsSmem L = rows_smem_layout(B, M, G, kDecodeMaxSmem);
    auto kern = decode_rows_kernel<B, MT>;
    {
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
    // The packed weights of all entries as uint32 [chunk rows][8 blocks][128]:
    // one 64-column chunk of a 128-row tile is a chunk row.
    constexpr int SG = 16 / B;
    const cuuint64_t dims[3] = {128, 8, cuuint64_t(batch) * n_tiles * KC};
    const cuuint64_t strides[2] = {512, cuuint64_t(kChunkBytes)};
    CUtensorMap wmap, wmap_tail;
    const cuuint32_t box[3] = {128, cuuint32_t(B), cuuint32_t(2 * SG)};
    cudaError_t e = encode_tensor_map(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, Wp, dims, strides, box,
                                      CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    const int rem = G % SG;
    const cuuint32_t box_tail[3] = {128, cuuint32_t(B), cuuint32_t(2 * (rem ? rem : SG))};
    e = encode_tensor_map(&wmap_tail, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, Wp, dims, strides, box_tail,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas, batch);
    cfg.blockDim = dim3(kRowsThreads);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int *err = device_error_word();
    if (!err) return cudaErrorUnknown;
    // 16-byte scale vectors (8 scales of a row): every row's scales start
    // 16-byte aligned, in every batch entry, when S is and G % 8 == 0.
    const int s_vec = (reinterpret_cast<uintptr_t>(S) % 16) == 0 && G % 8 == 0;
    return cudaLaunchKernelEx(&cfg, kern, wmap, wmap_tail, X, S, Y, M, N, K, int(resident), s_vec, err);
}

}  // namespace

bool decode_wk_fits(int M, int K, int B) {
    if (M < 1 || M > kRowsMaxTokens || (B != 1 && B != 2 && B != 4 && B != 8)) return false;
    const int G = K / kGroup;
    if (B * G > 1024) return false;                    // the CTA's scales in shared memory
    const RowsSmem L = rows_smem_layout(B, M, G, kDecodeMaxSmem);
    return L.stages >= 3;
}

cudaError_t launch_decode_wk(int B, int ctas, int batch, const uint16_t *X, const uint8_t *Wp,
                             const uint16_t *S, uint16_t *Y, bool resident, int M, int N, int K,
                             cudaStream_t s) {
    if (!decode_wk_fits(M, K, B) || ctas < 1 || batch < 1 || batch > 65535) return cudaErrorInvalidValue;
    // Token octets: 1 or 2.
#define W4A16_ROWS_CASE(BB)                                                              \
    case BB:                                                                             \
        return M <= 8 ? launch_rows_t<BB, 1>(ctas, batch, X, Wp, S, Y, resident, M, N, K, s) \
                      : launch_rows_t<BB, 2>(ctas, batch, X, Wp, S, Y, resident, M, N, K, s);
    switch (B) {
        W4A16_ROWS_CASE(1)
        W4A16_ROWS_CASE(2)
        W4A16_ROWS_CASE(4)
        W4A16_ROWS_CASE(8)
        default: return cudaErrorInvalidValue;
    }
#undef W4A16_ROWS_CASE
}

}  // namespace w4a16
