// tensor.cu -- compute arm: TMA-staged activations, register-dequantised weights
// in TMEM, tcgen05.mma with fp32 accumulators in TMEM.  One persistent kernel
// serves the plain product (optionally split along K) and the grouped product.
//
// Roles in a CTA (one per SM; 608 threads in the plain form, 480 with a
// separate epilogue; warp numbers for the plain form):
//   warps 0-15  dequantisers in four teams of four (two teams with a separate
//               epilogue).  Team t takes the CTA's groups q with
//               q % teams == t, in ring order; its warp w converts the 32
//               weight rows that TMEM sub-partition w % 4 holds (two 16-row
//               blocks): one LOP3 per bf16 pair gives 128 + code, one
//               bf16x2 FMA removes 136 exactly, one bf16x2 multiply applies
//               the group scale with a single rounding; two 16x256b
//               tcgen05.st per group, and the A stage goes to the MMA warp as
//               soon as the stores land.  In the plain form the same warps
//               then drain the tile's accumulator.
//   warp 16     X producer: per 128-wide group two TMA 2-D loads of the X
//               tile [tokens x 64] (128-byte swizzle); the X ring is released
//               by the MMA commit.
//   warp 17     W producer: one 8 KB bulk copy of the group's packed weights;
//               the W ring is released by the dequantisers once read, so it
//               runs many groups ahead of the MMA (HBM latency).
//   warp 18     TMEM owner and MMA issuer: eight tcgen05.mma (K = 16) per
//               group, A = weights from TMEM, B = X from shared memory,
//               D = fp32 in TMEM; tcgen05.commit releases the stages.
//   (separate form) four epilogue warps drain one of two accumulators while
//               the next tile runs into the other.
// Producers and the MMA issuer run their loops as whole warps and issue
// from one elected lane.
// The page this follows for the data flow is "[ROCm][Kernel] W4A16 skinny
// GEMM: hand-asm kernel for gfx1151" (magic-constant dequant, section 1;
// loads pipelined ahead of the math, section 2); the tile, the TMEM operand
// and the tensor-core instructions are this library's sm_103a design.
//
// Grouped product ("Add Triton BF16xINT4 rowwise GEMM for ROCm gfx942/gfx950",
// "Native fused grouped kernel"): each CTA reads M_sizes from device memory,
// forms the exclusive prefix sum of the (clamped) sizes and of the groups'
// tile counts in shared memory, and walks the flattened tile list; no host
// synchronisation is needed.
//
// Every mbarrier wait is bounded (async.cuh); a timeout records an error bit
// and the CTA winds down, waits for its own copies and MMAs, frees TMEM and
// exits.
#include <atomic>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "async.cuh"
#include "common.cuh"
#include "internal.h"
#include "tc05.cuh"

namespace w4a16 {

namespace {

// Warp roles (one CTA per SM).  A team is four dequantisers, one per TMEM
// sub-partition, each converting the 32 weight rows (two 16-row blocks) of
// a group that its sub-partition's lanes hold.  Plain form: four teams, team
// t taking the CTA's groups t, t + 4, t + 8, ..., so four groups are in
// flight and one team's waits (weights, TMEM store, A-ring slot) overlap the
// others' arithmetic; then the X producer, the W producer and the MMA warp.
// With a separate epilogue: two teams, the two producers, the MMA warp and 4
// epilogue warps that drain one TMEM accumulator while the dequantisers and
// the MMA go on with the next tile in the other.  (Measured on GB300 against
// two teams of eight warps of one block each: prefill 1322x19456x2560 86.1 ->
// 82.9 us, the grouped 8 x (2048x4096) 59.9 -> 56.3 us, 32x19456x2560 12.5 ->
// 11.6 us.)
constexpr int kTcTeamWarps = 4;
constexpr int kTcEpiWarps = 4;
template <bool kSep>
struct TcRoles {
    static constexpr int kTeams = kSep ? kTensorTeamsSep : kTensorTeamsPlain;
    static constexpr int kDequant = kTcTeamWarps * kTeams;     // warps 0 .. kDequant - 1
    static constexpr int kProducerX = kDequant;                 // the X ring
    static constexpr int kProducerW = kDequant + 1;             // the W ring
    static constexpr int kMma = kDequant + 2;
    static constexpr int kEpi0 = kDequant + 3;                  // kSep only
    static constexpr int kThreads = (kDequant + 3 + (kSep ? kTcEpiWarps : 0)) * 32;
};
constexpr uint32_t kTcDCol = 0;      // accumulator: columns [0, bt); A stage sa: [bt + 32 sa, bt + 32 sa + 32)

// TcArgs::opt_bits.
constexpr int kTcVecStore = 1;   // Y rows are 16-byte aligned: stage the epilogue for 16-byte stores
constexpr int kTcScaleVec = 2;   // scales aligned to 2 * sub bytes: one load per row's sub scales
constexpr int kTcZeroVec = 4;    // zero points aligned to sub bytes: one load per row's sub zeros

struct TcArgs {
    const uint8_t *Wp;
    const uint16_t *S;
    uint16_t *Y;
    float *ws;
    const int32_t *m_sizes;   // nullptr: plain product over M_total rows
    int *status;              // grouped status word (nullptr for the plain product)
    int *err;
    int M_total, N, K, num_groups;
    int bt;                   // tokens per tile = MMA N (multiple of 32, <= 256)
    int n_tiles;              // 128-row weight tiles
    int split_k, gps;         // K slices and 128-wide groups per slice
    int x_stages;             // X ring depth (one 128-column group of X per stage)
    int w_stages;             // W ring depth (8 KB of packed weights per stage)
    int a_stages;             // TMEM A ring depth (one group = 64 columns per stage)
    int tmem_cols;            // TMEM columns allocated (power of two >= dcols + 64 * a_stages)
    int dcols;                // accumulator columns: bt, or 2 bt with a separate epilogue
    int opt_bits;             // kTcVecStore | kTcScaleVec
    unsigned long long w_group_stride;  // bytes between groups' packed weights
    unsigned long long s_group_stride;  // elements between groups' scales
};
// Measured on GB300: growing TcArgs past 128 bytes (the kernel's parameters
// then exceed 256 bytes with the tensor map) slowed the kernel by about 5 %;
// new per-launch facts should be derived from these fields instead.
static_assert(sizeof(TcArgs) == 128, "TcArgs size");

// Shared memory: the X ring (per stage two X boxes, one per 64-column K block,
// 1024-byte aligned, 128-byte swizzle), the W ring (8 KB of packed weights of a
// group per stage), the epilogue staging, the barriers and the group tables.
struct TcSmem {
    int x_stage, off_x, off_w, off_epi, off_bar, off_misc, off_tab, total;
};

constexpr int kGroupBytes = 2 * kChunkBytes;           // packed weights of one 128-column group
constexpr int kEpiBytesPerWarp = 32 * 32 * 2;          // 32 tokens x 32 rows of bf16

// Epilogue staging buffers: one per warp that drains 32-token column blocks
// (the 4 epilogue warps, or in the plain form 4 dequantisers per column
// block, at most all 16).
__host__ __device__ inline int tc_epi_buffers(int bt, bool sep) {
    if (sep) return kTcEpiWarps;
    const int cbs = (bt + 31) / 32;
    return 4 * (cbs < 4 ? cbs : 4);
}

__host__ __device__ inline TcSmem tc_smem_layout(int bt, int x_stages, int w_stages, int a_stages,
                                                 int num_groups, bool sep) {
    TcSmem L;
    L.x_stage = 2 * bt * 128;
    L.off_x = 0;
    L.off_w = L.off_x + x_stages * L.x_stage;
    L.off_epi = L.off_w + w_stages * kGroupBytes;
    L.off_bar = L.off_epi + tc_epi_buffers(bt, sep) * kEpiBytesPerWarp;
    L.off_misc = L.off_bar + (2 * x_stages + 2 * w_stages + 2 * a_stages + 5) * 8;
    L.off_tab = (L.off_misc + 16 + 15) & ~15;           // group tables: 2 x (G + 1) ints
    L.total = L.off_tab + 2 * (num_groups + 1) * 4;
    return L;
}

struct TileInfo {
    int group, ft, tt, slice;
    int x_row0;       // first X/Y row of the tile
    int rows;         // valid rows (<= bt)
};

// Flattened tile order: feature tile fastest, then token tile, then slice
// (plain) or group (grouped), so CTAs running together share X tiles in L2.
// kBatched: a batched product, the plain product of each of num_groups
// entries of M_total / num_groups rows, entry b owning rows [b * rows,
// (b + 1) * rows) of the stacked X and Y and weight / scale block b; order:
// feature tile, token tile, entry, slice.  (A separate instantiation: folding
// it into the plain walk measurably slowed the plain kernel's loops.)
template <bool kBatched>
__device__ __forceinline__ bool tc_tile(const TcArgs &a, const int *tab_tiles, const int *tab_rows,
                                        int id, TileInfo &ti) {
    if constexpr (kBatched) {
        const int rows_b = a.M_total / a.num_groups;
        const int t_tiles = (rows_b + a.bt - 1) / a.bt;
        const int per_entry = t_tiles * a.n_tiles;
        const int per_slice = per_entry * a.num_groups;
        ti.slice = id / per_slice;
        int r = id - ti.slice * per_slice;
        ti.group = r / per_entry;
        r -= ti.group * per_entry;
        ti.tt = r / a.n_tiles;
        ti.ft = r - ti.tt * a.n_tiles;
        ti.x_row0 = ti.group * rows_b + ti.tt * a.bt;
        ti.rows = min(a.bt, rows_b - ti.tt * a.bt);
        return ti.slice < a.split_k;
    }
    if (a.m_sizes == nullptr) {
        const int t_tiles = (a.M_total + a.bt - 1) / a.bt;
        const int per_slice = t_tiles * a.n_tiles;
        ti.group = 0;
        ti.slice = id / per_slice;
        const int r = id - ti.slice * per_slice;
        ti.tt = r / a.n_tiles;
        ti.ft = r - ti.tt * a.n_tiles;
        ti.x_row0 = ti.tt * a.bt;
        ti.rows = min(a.bt, a.M_total - ti.x_row0);
        return ti.slice < a.split_k;
    }
    // binary search: largest g with tab_tiles[g] <= id
    int lo = 0, hi = a.num_groups;
    if (id >= tab_tiles[a.num_groups]) return false;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tab_tiles[mid] <= id) lo = mid; else hi = mid;
    }
    ti.group = lo;
    ti.slice = 0;
    const int r = id - tab_tiles[lo];
    ti.tt = r / a.n_tiles;
    ti.ft = r - ti.tt * a.n_tiles;
    const int g_rows = tab_rows[lo + 1] - tab_rows[lo];
    ti.x_row0 = tab_rows[lo] + ti.tt * a.bt;
    ti.rows = min(a.bt, g_rows - ti.tt * a.bt);
    return true;
}

// A group scale, loaded raw (bits in the low half, 0 past the last row).  The
// bf16x2 pair is formed only where it is used (scale_pair2), so a load issued a
// group ahead is not waited for by an instruction right behind it.
__device__ __forceinline__ uint32_t scale_raw(const uint16_t *S, int row, int N, size_t idx) {
    uint32_t v = 0;
    asm volatile("{\n\t.reg .pred p;\n\tsetp.lt.s32 p, %1, %2;\n\t"
                 "@p ld.global.nc.u16 %0, [%3];\n\t}"
                 : "+r"(v)
                 : "r"(row), "r"(N), "l"(S + idx));
    return v;
}
__device__ __forceinline__ uint32_t scale_pair2(uint32_t raw) { return raw | (raw << 16); }

// The kSub scales of one weight row for one 128-wide block (scale groups of
// 128 / kSub columns), raw, two per 32-bit word (scale i in half i % 2 of word
// i / 2).  kSub == 1 is scale_raw.
template <int kSub>
struct ScaleRaw {
    uint32_t w[(kSub + 1) / 2];
};
// vec: S + idx is aligned to 2 * kSub bytes (a row's kSub scales of one block
// start at a multiple of kSub elements), so one 4- or 8-byte load fetches them.
template <int kSub>
__device__ __forceinline__ ScaleRaw<kSub> scales_raw(const uint16_t *S, int row, int N, size_t idx,
                                                     bool vec) {
    ScaleRaw<kSub> r;
#pragma unroll
    for (int i = 0; i < (kSub + 1) / 2; ++i) r.w[i] = 0;
    if constexpr (kSub == 2) {
        if (vec) {
            asm volatile("{\n\t.reg .pred p;\n\tsetp.lt.s32 p, %1, %2;\n\t"
                         "@p ld.global.nc.u32 %0, [%3];\n\t}"
                         : "+r"(r.w[0])
                         : "r"(row), "r"(N), "l"(S + idx));
            return r;
        }
    } else if constexpr (kSub == 4) {
        if (vec) {
            asm volatile("{\n\t.reg .pred p;\n\tsetp.lt.s32 p, %2, %3;\n\t"
                         "@p ld.global.nc.v2.u32 {%0, %1}, [%4];\n\t}"
                         : "+r"(r.w[0]), "+r"(r.w[1])
                         : "r"(row), "r"(N), "l"(S + idx));
            return r;
        }
    }
#pragma unroll
    for (int i = 0; i < kSub; ++i) r.w[i / 2] |= scale_raw(S, row, N, idx + i) << (16 * (i & 1));
    return r;
}
// The kSub zero points (zero-point variant) of one weight row for one
// 128-wide block, one byte each in a 32-bit word (0 past the last row).
// vec: Z + idx is aligned to kSub bytes.
template <int kSub>
__device__ __forceinline__ uint32_t zeros_raw(const uint8_t *Z, int row, int N, size_t idx, bool vec) {
    uint32_t r = 0;
    if constexpr (kSub == 4) {
        if (vec) {
            asm volatile("{\n\t.reg .pred p;\n\tsetp.lt.s32 p, %1, %2;\n\t"
                         "@p ld.global.nc.u32 %0, [%3];\n\t}"
                         : "+r"(r) : "r"(row), "r"(N), "l"(Z + idx));
            return r;
        }
    } else if constexpr (kSub == 2) {
        if (vec) {
            asm volatile("{\n\t.reg .pred p;\n\tsetp.lt.s32 p, %1, %2;\n\t"
                         "@p ld.global.nc.u16 %0, [%3];\n\t}"
                         : "+r"(r) : "r"(row), "r"(N), "l"(Z + idx));
            return r;
        }
    }
#pragma unroll
    for (int i = 0; i < kSub; ++i) {
        uint32_t v = 0;
        asm volatile("{\n\t.reg .pred p;\n\tsetp.lt.s32 p, %1, %2;\n\t"
                     "@p ld.global.nc.u8 %0, [%3];\n\t}"
                     : "+r"(v) : "r"(row), "r"(N), "l"(Z + idx + i));
        r |= v << (8 * i);
    }
    return r;
}

// bf16x2 pair {-(128 + z), -(128 + z)} of zero point i, from the row's
// zero-point bytes already masked to their low four bits: 128 + z is bf16
// 0x4300 | z exactly, so the pair's bytes are {z, 0xC3, z, 0xC3}, one byte
// permute.
__device__ __forceinline__ uint32_t neg_offset_pair(uint32_t zmasked, int i) {
    return __byte_perm(zmasked, 0xC3C3C3C3u, 0x4040u + 0x0101u * uint32_t(i));
}

// bf16x2 a * 1 + b: with a = 128 + code and b = -(128 + z), code - z exactly.
__device__ __forceinline__ uint32_t bf16x2_add_pair(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(0x3F803F80u), "r"(b));
    return d;
}

// bf16x2 pair {scale i, scale i}.
template <int kSub>
__device__ __forceinline__ uint32_t scale_pair_of(const ScaleRaw<kSub> &r, int i) {
    if constexpr (kSub == 1) return scale_pair2(r.w[0]);
    return __byte_perm(r.w[i / 2], 0, (i & 1) ? 0x3232 : 0x1010);
}

__device__ __forceinline__ void tc_st_16x256b_x8(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x256b.x8.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
        "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
        "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

// One 32-token column block of a warp's 32 accumulator rows (v[i]: row
// fb + lane, token ti.x_row0 + 32 cb + i) to Y (bf16) or to the split-K
// workspace (fp32).  With 16-byte-aligned Y rows the block is transposed
// through shared memory so that each lane writes 16 bytes (8 rows) of four
// tokens.
template <bool kSplit>
__device__ __forceinline__ void tc_store_block(const TcArgs &a, const TileInfo &ti, int fb, int cb,
                                               const uint32_t (&v)[32], unsigned char *epi,
                                               int lane) {
    const int t0 = ti.x_row0 + cb * 32;                // token of v[0]
    const int nt = min(32, ti.rows - cb * 32);         // valid tokens of the block
    if (kSplit || !(a.opt_bits & kTcVecStore)) {
        const int f = fb + lane;
        if (f < a.N) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                if (i < nt) {
                    const size_t off = size_t(t0 + i) * a.N + f;
                    if (kSplit)
                        a.ws[size_t(ti.slice) * a.M_total * a.N + off] = __uint_as_float(v[i]);
                    else
                        a.Y[off] = f32_to_bf16_rn(__uint_as_float(v[i]));
                }
            }
        }
    } else {
        // Transpose through shared memory: [token][32 rows] bf16, then
        // each lane writes 16 bytes (8 rows) of four tokens.
        uint16_t *tile = reinterpret_cast<uint16_t *>(epi);
#pragma unroll
        for (int i = 0; i < 32; ++i) tile[i * 32 + lane] = f32_to_bf16_rn(__uint_as_float(v[i]));
        __syncwarp();
        const int chunk = lane & 3;
        const int f8 = fb + 8 * chunk;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int i = (lane >> 2) + 8 * c;
            if (i < nt && f8 < a.N) {
                const uint4 val = *reinterpret_cast<const uint4 *>(tile + i * 32 + 8 * chunk);
                *reinterpret_cast<uint4 *>(a.Y + size_t(t0 + i) * a.N + f8) = val;
            }
        }
        __syncwarp();
    }
}

// kSub: scale groups per 128-wide block (1, 2, 4: groups of 128, 64, 32
// columns).  Packed word j of a lane covers columns 16 j .. 16 j + 15 of the
// block, so its scale group is j * kSub / 8.
// kZp: zero points Z (uint8 [N][K/G] per group of the product): the
// dequantisers subtract 128 + z, exact in bf16, where the symmetric form
// subtracts 136.  tc_gemm_kernel and tc_gemm_zp_kernel are the entry points.
template <bool kSplit, bool kSep, bool kBatched, int kSub, bool kZp>
__device__ __forceinline__ void tc_gemm_body(const CUtensorMap &tmap_x, const TcArgs &a,
                                             const uint8_t *__restrict__ Z) {
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte alignment for the swizzled X tiles (the host adds the slack).
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    using R = TcRoles<kSep>;
    const TcSmem L = tc_smem_layout(a.bt, a.x_stages, a.w_stages, a.a_stages, a.num_groups, kSep);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int SX = a.x_stages;
    const int SW = a.w_stages;
    const int SA = a.a_stages;
    const uint32_t bar0 = smem_u32(smem + L.off_bar);
    auto xfull_bar = [&](int s) { return bar0 + 8u * s; };
    auto xempty_bar = [&](int s) { return bar0 + 8u * (SX + s); };
    auto wfull_bar = [&](int s) { return bar0 + 8u * (2 * SX + s); };
    auto wempty_bar = [&](int s) { return bar0 + 8u * (2 * SX + SW + s); };
    auto afull_bar = [&](int s) { return bar0 + 8u * (2 * SX + 2 * SW + s); };
    auto aempty_bar = [&](int s) { return bar0 + 8u * (2 * SX + 2 * SW + SA + s); };
    // Accumulator b in {0, 1}: dfull[b] (the MMA commit), dempty[b] (its readers).
    const uint32_t dbar0 = bar0 + 8u * (2 * SX + 2 * SW + 2 * SA);
    auto dfull_bar = [&](int b) { return dbar0 + 8u * b; };
    auto dempty_bar = [&](int b) { return dbar0 + 16u + 8u * b; };
    const uint32_t done_bar = dbar0 + 32;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.off_misc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.off_misc + 4);
    int *tab_tiles = reinterpret_cast<int *>(smem + L.off_tab);
    int *tab_rows = tab_tiles + a.num_groups + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SX; ++s) {
            mbar_init(xfull_bar(s), 1);
            mbar_init(xempty_bar(s), 1);                  // the MMA commit
        }
        for (int s = 0; s < SW; ++s) {
            mbar_init(wfull_bar(s), 1);
            mbar_init(wempty_bar(s), kTcTeamWarps);       // the group's team has read it
        }
        for (int s = 0; s < SA; ++s) {
            mbar_init(afull_bar(s), kTcTeamWarps);
            mbar_init(aempty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(dfull_bar(b), 1);
            mbar_init(dempty_bar(b), kSep ? kTcEpiWarps : R::kDequant);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == R::kMma) {
        tc_alloc(smem_u32(tmem_slot), uint32_t(a.tmem_cols));
        tc_relinquish();
    }
    if (warp == R::kProducerX && lane == 0) tma_prefetch_desc(&tmap_x);
    pdl_launch_dependents();
    pdl_wait();

    // Group tables (grouped product): clamped row starts and tile prefix sums.
    if (a.m_sizes != nullptr && threadIdx.x == 0) {
        int rows = 0, tiles = 0, status = 0;
        for (int g = 0; g < a.num_groups; ++g) {
            int sz = a.m_sizes[g];
            if (sz < 0) { status |= 1; sz = 0; }
            if (rows + sz > a.M_total) { status |= 2; sz = a.M_total - rows; }
            tab_rows[g] = rows;
            tab_tiles[g] = tiles;
            rows += sz;
            tiles += ((sz + a.bt - 1) / a.bt) * a.n_tiles;
        }
        tab_rows[a.num_groups] = rows;
        tab_tiles[a.num_groups] = tiles;
        if (blockIdx.x == 0 && a.status) *a.status = status;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int n_groups = a.K / kGroup;
    const int n_sg = n_groups * kSub;                         // scales per weight row
    const int KC = a.K / kChunkK;
    const uint32_t x_bytes = uint32_t(a.bt) * 128u;          // one X box
    const uint32_t idesc = tc_idesc_bf16(128, a.bt);

    if (warp == R::kProducerX || warp == R::kProducerW) {
        // Two producer warps, one per ring, each walking the CTA's (tile,
        // group) sequence.  The whole warp runs the loop, so its values stay
        // warp-uniform; one elected lane issues the copies.  (Measured on
        // GB300: one thread serving both rings in a divergent loop issued one
        // X and one W copy every ~0.5 us, which paced the whole pipeline at
        // 32 tokens.)  Waits are bounded: a wait that runs out aborts the CTA.
        const bool is_x = warp == R::kProducerX;
        const int S = is_x ? SX : SW;
        // Each time the W producer enters a tile, it pulls the tile's scales
        // (128 rows x all groups, one contiguous block) into L2, so the
        // dequantisers' scale loads, issued one group ahead, hit L2.
        auto prefetch_scales = [&](const TileInfo &ti) {
            const uint16_t *sg = a.S + (unsigned long long)ti.group * a.s_group_stride;
            const size_t r0 = size_t(ti.ft) * kTileRows;
            const size_t r1 = min(size_t(a.N), r0 + kTileRows);
            // Rounded inwards to 16 bytes: never outside the block.
            const uintptr_t lo = (reinterpret_cast<uintptr_t>(sg + r0 * n_sg) + 15) & ~uintptr_t(15);
            const uintptr_t hi = reinterpret_cast<uintptr_t>(sg + r1 * n_sg) & ~uintptr_t(15);
            if (hi > lo) bulk_prefetch_l2(reinterpret_cast<const void *>(lo), uint32_t(hi - lo));
        };
        TileInfo tk;
        int id = blockIdx.x;
        bool more = tc_tile<kBatched>(a, tab_tiles, tab_rows, id, tk);
        int gk = more ? tk.slice * a.gps : 0;
        if (!is_x && more && elect_one()) prefetch_scales(tk);
        __syncwarp();
        int slot = 0, issued = 0;
        uint32_t epar = 1;              // parity of the slot's empty phase (first lap: no wait)
        while (more) {
            const uint32_t empty = is_x ? xempty_bar(slot) : wempty_bar(slot);
            if (issued >= S && !__all_sync(0xffffffffu, mbar_wait(empty, epar, abort_flag, a.err))) break;
            if (elect_one()) {
                if (is_x) {
                    const uint32_t xdst = smem_u32(smem + L.off_x + slot * L.x_stage);
                    mbar_arrive_expect_tx(xfull_bar(slot), 2 * x_bytes);
                    tma_load_2d(xdst, &tmap_x, gk * kGroup, tk.x_row0, xfull_bar(slot));
                    tma_load_2d(xdst + x_bytes, &tmap_x, gk * kGroup + kChunkK, tk.x_row0, xfull_bar(slot));
                } else {
                    const uint8_t *wg = a.Wp + (unsigned long long)tk.group * a.w_group_stride;
                    mbar_arrive_expect_tx(wfull_bar(slot), kGroupBytes);
                    bulk_g2s(smem_u32(smem + L.off_w + slot * kGroupBytes),
                             wg + ((size_t)tk.ft * KC + 2 * gk) * kChunkBytes, kGroupBytes, wfull_bar(slot));
                }
            }
            __syncwarp();
            ++issued;
            if (++slot == S) {
                slot = 0;
                epar ^= 1u;
            }
            if (++gk == min(n_groups, (tk.slice + 1) * a.gps)) {
                id += gridDim.x;
                more = tc_tile<kBatched>(a, tab_tiles, tab_rows, id, tk);
                if (more) {
                    gk = tk.slice * a.gps;
                    if (!is_x && elect_one()) prefetch_scales(tk);
                    __syncwarp();
                }
            }
        }
        if (*abort_flag) {
            // Let every copy issued land before the CTA exits.
            for (int u = issued > S ? issued - S : 0; u < issued; ++u)
                drain_wait(is_x ? xfull_bar(u % S) : wfull_bar(u % S), (u / S) & 1);
        }
    } else if (warp == R::kMma) {
        // The whole warp runs the loop (warp-uniform operands); the elected
        // lane (always the lowest, the warp being converged) issues every MMA
        // and every commit, so the commits track its MMAs.
        int st = 0, sa = 0, tiles = 0;
        uint32_t xph = 0, aph = 0;      // parities of the phases to wait for
        TileInfo ti;
        for (int id = blockIdx.x; tc_tile<kBatched>(a, tab_tiles, tab_rows, id, ti); id += gridDim.x) {
            // Accumulator of this tile and the wait for its previous readers.
            const int db = kSep ? (tiles & 1) : 0;
            const int uses = kSep ? (tiles >> 1) : tiles;     // earlier tiles on this buffer
            if (uses > 0 &&
                !__all_sync(0xffffffffu, mbar_wait(dempty_bar(db), (uses - 1) & 1, abort_flag, a.err)))
                break;
            tc_fence_after();
            const uint32_t dcol = tmem_base + kTcDCol + uint32_t(db * a.bt);
            // A tile of fewer tokens than bt (a group's or the product's last)
            // multiplies only its tokens, rounded up to the MMA's N step of 16;
            // the epilogue stores the valid tokens only.  (Measured on GB300:
            // 1322x19456x2560, whose last 192-token tile holds 170, 83.0 ->
            // 81.8 us; 2858x19456x2560 173.1 -> 170.2 us.)
            const uint32_t idesc_t = ti.rows >= a.bt ? idesc : tc_idesc_bf16(128, (ti.rows + 15) & ~15);
            const int g0 = ti.slice * a.gps;
            const int g1 = min(n_groups, (ti.slice + 1) * a.gps);
            bool ok = true;
            for (int grp = g0; grp < g1; ++grp) {
                if (!__all_sync(0xffffffffu, mbar_wait(xfull_bar(st), xph, abort_flag, a.err) &&
                                                 mbar_wait(afull_bar(sa), aph, abort_flag, a.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t xs = smem_u32(smem + L.off_x + st * L.x_stage);
                const uint32_t acol = tmem_base + uint32_t(a.dcols) + 64u * sa;
                const uint64_t bdesc0 = tc_sdesc_sw128(xs);
                const uint64_t bdesc1 = tc_sdesc_sw128(xs + x_bytes);
                if (elect_one()) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            tc_mma_ts(dcol, acol + 32u * h + 8u * j, (h ? bdesc1 : bdesc0) + 2u * j,
                                      idesc_t, (grp > g0 || h > 0 || j > 0) ? 1u : 0u);
                    }
                    tc_commit(xempty_bar(st));
                    tc_commit(aempty_bar(sa));
                }
                __syncwarp();
                if (++st == SX) { st = 0; xph ^= 1; }
                if (++sa == SA) { sa = 0; aph ^= 1; }
            }
            if (!ok) break;
            if (elect_one()) tc_commit(dfull_bar(db));
            __syncwarp();
            ++tiles;
        }
        // Every MMA issued has completed before TMEM is freed.
        if (elect_one()) tc_commit(done_bar);
        __syncwarp();
        drain_wait(done_bar, 0);
    } else if (warp < R::kDequant) {
        // Dequantisers (and, without a separate epilogue, the epilogue).
        // q counts the CTA's groups in ring order; this warp's team takes
        // those with q % kTeams == team, and its ring slots and phase
        // parities advance kTeams positions per group it takes.  Within a
        // team, warp `sub` converts the 32 weight rows of TMEM sub-partition
        // `sub` (16-row blocks 2 sub and 2 sub + 1): per group it loads both
        // blocks' packed words, hands the W stage back, builds and stores
        // block 2 sub's fragments, waits for its A stage's slot only before
        // that first store, then builds and stores block 2 sub + 1's, and
        // hands the A stage to the MMA warp once both stores have landed.
        const int team = warp / kTcTeamWarps;
        const int sub = warp % kTcTeamWarps;        // TMEM sub-partition of this warp (warp % 4)
        const int g = lane >> 2;
        unsigned char *epi = smem + L.off_epi + warp * kEpiBytesPerWarp;
        int q = 0, tiles = 0;
        int st = team, sa = team;       // ring slots of this warp's next group (kTeams <= SW, SA)
        uint32_t wph = 0;               // parity of the W-ring phase to wait for
        uint32_t eph = 1;               // parity of the A-ring empty phase (first lap: none)
        auto advance = [](int &slot, uint32_t &par, int n) {
            slot += R::kTeams;
            if (slot >= n) {
                slot -= n;
                par ^= 1u;
            }
        };
        // The warp's weight rows are r0 + 8 e (e = 0..3; rows g and g + 8 of
        // its two blocks).  Their scales (and zero points) of the warp's next
        // group are loaded one group ahead.
        ScaleRaw<kSub> ns[4] = {};
        uint32_t nz[4] = {};
        bool have_next = false;
        const bool svec = (a.opt_bits & kTcScaleVec) != 0;
        const bool zvec = (a.opt_bits & kTcZeroVec) != 0;
        TileInfo ti, nx;
        for (int id = blockIdx.x; tc_tile<kBatched>(a, tab_tiles, tab_rows, id, ti); id += gridDim.x) {
            const bool nx_ok = tc_tile<kBatched>(a, tab_tiles, tab_rows, id + gridDim.x, nx);
            const int g0 = ti.slice * a.gps;
            const int g1 = min(n_groups, (ti.slice + 1) * a.gps);
            const int r0 = ti.ft * kTileRows + 32 * sub + g;
            const size_t so = (unsigned long long)ti.group * a.s_group_stride + size_t(r0) * n_sg;
            const size_t rstep = size_t(8) * n_sg;
            const int rn = nx.ft * kTileRows + 32 * sub + g;
            const int gn0 = nx.slice * a.gps;
            const int nx_g1 = nx_ok ? min(n_groups, gn0 + a.gps) : 0;
            const size_t no = nx_ok ? (unsigned long long)nx.group * a.s_group_stride + size_t(rn) * n_sg : 0;
            bool ok = true;
            for (int grp = g0; grp < g1; ++grp, ++q) {
                if (R::kTeams > 1 && q % R::kTeams != team) continue;   // another team's group
                ScaleRaw<kSub> s[4];
                uint32_t z[4] = {0, 0, 0, 0};
                if (have_next) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) { s[e] = ns[e]; z[e] = nz[e]; }
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        s[e] = scales_raw<kSub>(a.S + so + e * rstep, r0 + 8 * e, a.N, size_t(grp) * kSub, svec);
                        if (kZp) z[e] = zeros_raw<kSub>(Z + so + e * rstep, r0 + 8 * e, a.N, size_t(grp) * kSub, zvec);
                    }
                }
                const int gnext = grp + R::kTeams;
                have_next = gnext < g1 || (nx_ok && gn0 + (gnext - g1) < nx_g1);
                if (gnext < g1) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        ns[e] = scales_raw<kSub>(a.S + so + e * rstep, r0 + 8 * e, a.N, size_t(gnext) * kSub, svec);
                        if (kZp) nz[e] = zeros_raw<kSub>(Z + so + e * rstep, r0 + 8 * e, a.N, size_t(gnext) * kSub, zvec);
                    }
                } else if (have_next) {
                    const size_t gi = size_t(gn0 + (gnext - g1)) * kSub;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        ns[e] = scales_raw<kSub>(a.S + no + e * rstep, rn + 8 * e, a.N, gi, svec);
                        if (kZp) nz[e] = zeros_raw<kSub>(Z + no + e * rstep, rn + 8 * e, a.N, gi, zvec);
                    }
                }
                // Warp-uniform outcomes below: tcgen05.st needs every lane.
                if (!__all_sync(0xffffffffu, mbar_wait(wfull_bar(st), wph, abort_flag, a.err))) {
                    ok = false;
                    break;
                }
                const unsigned char *wsrc = smem + L.off_w + st * kGroupBytes + (2 * sub) * kBlockBytes + lane * 16;
                uint32_t wv[2][8];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 wa = *reinterpret_cast<const uint4 *>(wsrc + h * kBlockBytes);
                    const uint4 wb = *reinterpret_cast<const uint4 *>(wsrc + h * kBlockBytes + kChunkBytes);
                    wv[h][0] = wa.x; wv[h][1] = wa.y; wv[h][2] = wa.z; wv[h][3] = wa.w;
                    wv[h][4] = wb.x; wv[h][5] = wb.y; wv[h][6] = wb.z; wv[h][7] = wb.w;
                }
                // The stage's bytes are in registers: hand it back to the producer.
                __syncwarp();
                if (lane == 0) mbar_arrive(wempty_bar(st));
                advance(st, wph, SW);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t p0[kSub], p1[kSub];
#pragma unroll
                    for (int i = 0; i < kSub; ++i) {
                        p0[i] = scale_pair_of<kSub>(s[2 * h], i);
                        p1[i] = scale_pair_of<kSub>(s[2 * h + 1], i);
                    }
                    uint32_t zo0[kSub], zo1[kSub];
                    if constexpr (kZp) {
                        const uint32_t m0 = z[2 * h] & 0x0F0F0F0Fu, m1 = z[2 * h + 1] & 0x0F0F0F0Fu;
#pragma unroll
                        for (int i = 0; i < kSub; ++i) {
                            zo0[i] = neg_offset_pair(m0, i);
                            zo1[i] = neg_offset_pair(m1, i);
                        }
                    }
                    uint32_t frag[32];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t q0 = p0[j * kSub / 8], q1 = p1[j * kSub / 8];
                        const uint32_t w = wv[h][j];
                        if constexpr (kZp) {
                            const uint32_t o0 = zo0[j * kSub / 8];
                            const uint32_t o1 = zo1[j * kSub / 8];
                            frag[4 * j + 0] = bf16x2_mul(bf16x2_add_pair(magic_pair(w), o0), q0);
                            frag[4 * j + 1] = bf16x2_mul(bf16x2_add_pair(magic_pair(w >> 8), o0), q0);
                            frag[4 * j + 2] = bf16x2_mul(bf16x2_add_pair(magic_pair(w >> 4), o1), q1);
                            frag[4 * j + 3] = bf16x2_mul(bf16x2_add_pair(magic_pair(w >> 12), o1), q1);
                            continue;
                        }
                        frag[4 * j + 0] = bf16x2_mul(minus136(magic_pair(w)), q0);
                        frag[4 * j + 1] = bf16x2_mul(minus136(magic_pair(w >> 8)), q0);
                        frag[4 * j + 2] = bf16x2_mul(minus136(magic_pair(w >> 4)), q1);
                        frag[4 * j + 3] = bf16x2_mul(minus136(magic_pair(w >> 12)), q1);
                    }
                    if (h == 0) {
                        if (q >= SA && !__all_sync(0xffffffffu, mbar_wait(aempty_bar(sa), eph, abort_flag, a.err))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    tc_st_16x256b_x8(tmem_base + (uint32_t(32 * sub + 16 * h) << 16) + uint32_t(a.dcols) + 64u * sa, frag);
                }
                if (!ok) break;
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(afull_bar(sa));
                advance(sa, eph, SA);
            }
            if (!ok) break;
            if (kSep) continue;
            // Epilogue: warp w reads lanes 32 (w % 4) .. + 31 (its weight rows)
            // for the 32-token column blocks w / 4, w / 4 + kDequant / 4, ...
            if (!__all_sync(0xffffffffu, mbar_wait(dfull_bar(0), tiles & 1, abort_flag, a.err))) break;
            tc_fence_after();
            const int fb = ti.ft * kTileRows + 32 * sub;           // first weight row of the warp
            for (int cb = warp >> 2; cb * 32 < a.bt; cb += R::kDequant / 4) {
                uint32_t v[32];
                tc_ld_32x32b_x32(tmem_base + (uint32_t(32 * sub) << 16) + kTcDCol + 32u * cb, v);
                tc_wait_ld();
                tc_store_block<kSplit>(a, ti, fb, cb, v, epi, lane);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dempty_bar(0));
            ++tiles;
        }
    } else if (kSep) {
        // Separate epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 (its
        // 32 weight rows) for every 32-token column block of the tile's
        // accumulator, alternating between the two accumulators.
        const int sub = warp & 3;
        unsigned char *epi = smem + L.off_epi + (warp - R::kEpi0) * kEpiBytesPerWarp;
        int tiles = 0;
        TileInfo ti;
        for (int id = blockIdx.x; tc_tile<kBatched>(a, tab_tiles, tab_rows, id, ti); id += gridDim.x) {
            const int db = tiles & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(dfull_bar(db), (tiles >> 1) & 1, abort_flag, a.err))) break;
            tc_fence_after();
            const int fb = ti.ft * kTileRows + 32 * sub;
            for (int cb = 0; cb * 32 < a.bt; ++cb) {
                uint32_t v[32];
                tc_ld_32x32b_x32(tmem_base + (uint32_t(32 * sub) << 16) + kTcDCol +
                                     uint32_t(db * a.bt) + 32u * cb,
                                 v);
                tc_wait_ld();
                tc_store_block<kSplit>(a, ti, fb, cb, v, epi, lane);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dempty_bar(db));
            ++tiles;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == R::kMma) tc_dealloc(tmem_base, uint32_t(a.tmem_cols));
    if (*abort_flag && warp < R::kDequant) {
        // A wait ran out (the error word holds kErrWaitTimeout): every output
        // of this CTA's tiles becomes NaN, so an incomplete result is never a
        // plausible number.
        TileInfo ti;
        for (int id = blockIdx.x; tc_tile<kBatched>(a, tab_tiles, tab_rows, id, ti); id += gridDim.x) {
            for (int e = threadIdx.x; e < ti.rows * kTileRows; e += R::kDequant * 32) {
                const int m = ti.x_row0 + e / kTileRows;
                const int f = ti.ft * kTileRows + e % kTileRows;
                if (f >= a.N) continue;
                const size_t off = size_t(m) * a.N + f;
                if (kSplit) a.ws[size_t(ti.slice) * a.M_total * a.N + off] = __int_as_float(0x7fc00000);
                else a.Y[off] = uint16_t(0x7fc0);
            }
        }
    }
}

template <bool kSplit, bool kSep, bool kBatched, int kSub>
__global__ void __launch_bounds__(TcRoles<kSep>::kThreads, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const TcArgs a) {
    tc_gemm_body<kSplit, kSep, kBatched, kSub, false>(tmap_x, a, nullptr);
}

template <bool kSplit, bool kSep, bool kBatched, int kSub>
__global__ void __launch_bounds__(TcRoles<kSep>::kThreads, 1)
tc_gemm_zp_kernel(const __grid_constant__ CUtensorMap tmap_x, const TcArgs a,
                  const uint8_t *__restrict__ Z) {
    tc_gemm_body<kSplit, kSep, kBatched, kSub, true>(tmap_x, a, Z);
}

}  // namespace

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiledFn encode_tiled() {
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load(std::memory_order_acquire);
    if (!f) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !p) {
            cudaGetLastError();
            return nullptr;
        }
        f = reinterpret_cast<EncodeTiledFn>(p);
        fn.store(f, std::memory_order_release);
    }
    return f;
}

cudaError_t encode_tensor_map(CUtensorMap *map, CUtensorMapDataType type, int rank, const void *base,
                              const cuuint64_t *dims, const cuuint64_t *strides_bytes,
                              const cuuint32_t *box, CUtensorMapSwizzle swizzle) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return cudaErrorNotSupported;
    cuuint32_t estride[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(map, type, cuuint32_t(rank), const_cast<void *>(base), dims, strides_bytes, box,
                     estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// A ring depth: as many 64-column group stages (at most four) as fit next to
// the bt accumulator columns in the CTA's share of the SM's 512 TMEM columns
// (all of them with one CTA per SM, half with two); 0 if none fits.
// A ring depth: as many 64-column group stages (at most four) as fit next to
// the accumulator columns (bt, or 2 bt with a separate epilogue) in the CTA's
// share of the SM's 512 TMEM columns (all of them with one CTA per SM, half
// with two); 0 if none fits.
int tensor_a_stages(int bt, int occupancy, bool sep) {
    const int share = 512 / occupancy;
    const int dcols = sep ? 2 * bt : bt;
    int sa = (share - dcols) / 64;
    return sa > 4 ? 4 : (sa < 0 ? 0 : sa);
}

int tensor_tmem_cols(int bt, int occupancy, bool sep) {
    const int need = (sep ? 2 * bt : bt) + 64 * tensor_a_stages(bt, occupancy, sep);
    int cols = 32;
    while (cols < need) cols <<= 1;
    return cols;
}

size_t tensor_smem_bytes(int bt, int x_stages, int w_stages, int occupancy, int num_groups, bool sep) {
    return size_t(tc_smem_layout(bt, x_stages, w_stages, tensor_a_stages(bt, occupancy, sep),
                                 num_groups, sep)
                      .total) +
           1024;  // + alignment slack
}

namespace {

// One of the kernel's eight (split, separate epilogue, batched) forms for
// kSub scale groups per 128-wide block.
// Z != nullptr: the zero-point kernel (plain products only).
template <int kSub>
cudaError_t launch_tc_sub(const TensorPlan &p, const CUtensorMap &tmap, const TcArgs &a, bool batched,
                          size_t smem, cudaStream_t s, const uint8_t *Z) {
    const bool split = p.split_k > 1;
    const bool sep = p.sep_epilogue;
    auto kern = batched ? (split ? (sep ? tc_gemm_kernel<true, true, true, kSub> : tc_gemm_kernel<true, false, true, kSub>)
                                 : (sep ? tc_gemm_kernel<false, true, true, kSub> : tc_gemm_kernel<false, false, true, kSub>))
                        : (split ? (sep ? tc_gemm_kernel<true, true, false, kSub> : tc_gemm_kernel<true, false, false, kSub>)
                                 : (sep ? tc_gemm_kernel<false, true, false, kSub> : tc_gemm_kernel<false, false, false, kSub>));
    auto kern_zp = batched
        ? (split ? (sep ? tc_gemm_zp_kernel<true, true, true, kSub> : tc_gemm_zp_kernel<true, false, true, kSub>)
                 : (sep ? tc_gemm_zp_kernel<false, true, true, kSub> : tc_gemm_zp_kernel<false, false, true, kSub>))
        : (split ? (sep ? tc_gemm_zp_kernel<true, true, false, kSub> : tc_gemm_zp_kernel<true, false, false, kSub>)
                 : (sep ? tc_gemm_zp_kernel<false, true, false, kSub> : tc_gemm_zp_kernel<false, false, false, kSub>));
    static std::atomic<unsigned long long> opted[16];
    const int ki = (Z ? 8 : 0) + (batched ? 4 : 0) + (split ? 2 : 0) + (sep ? 1 : 0);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(opted[ki].load(std::memory_order_acquire) & bit)) {
        e = Z ? cudaFuncSetAttribute(kern_zp, cudaFuncAttributeMaxDynamicSharedMemorySize, kTensorMaxSmem)
              : cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kTensorMaxSmem);
        if (e != cudaSuccess) return e;
        opted[ki].fetch_or(bit, std::memory_order_acq_rel);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.ctas);
    cfg.blockDim = dim3(sep ? TcRoles<true>::kThreads : TcRoles<false>::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (Z) return cudaLaunchKernelEx(&cfg, kern_zp, tmap, a, Z);
    return cudaLaunchKernelEx(&cfg, kern, tmap, a);
}

}  // namespace

cudaError_t launch_tensor(const TensorPlan &p, const uint16_t *X, const uint8_t *Wp,
                          const uint16_t *S, uint16_t *Y, float *ws, const int32_t *m_sizes,
                          int *status, int num_groups, int M_total, int N, int K, cudaStream_t s,
                          int batch_rows, const uint8_t *Z) {
    if (p.tile_tokens < 32 || p.tile_tokens > 256 || p.tile_tokens % 32 || p.x_stages < 2 ||
        p.w_stages < (p.sep_epilogue ? TcRoles<true>::kTeams : TcRoles<false>::kTeams) ||
        p.ctas < 1 || num_groups < 1 || num_groups > kMaxGroups || p.occupancy != 1 ||
        (p.sub != 1 && p.sub != 2 && p.sub != 4) ||
        // one W and one A ring slot per dequantiser team at least
        tensor_a_stages(p.tile_tokens, p.occupancy, p.sep_epilogue) <
            (p.sep_epilogue ? TcRoles<true>::kTeams : TcRoles<false>::kTeams))
        return cudaErrorInvalidValue;
    CUtensorMap tmap;
    const cuuint64_t gdim[2] = {cuuint64_t(K), cuuint64_t(M_total)};
    const cuuint64_t gstride[1] = {cuuint64_t(K) * 2};
    const cuuint32_t box[2] = {64u, cuuint32_t(p.tile_tokens)};
    cudaError_t er = encode_tensor_map(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, X, gdim, gstride,
                                       box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (er != cudaSuccess) return er;

    TcArgs a;
    a.Wp = Wp;
    a.S = S;
    a.Y = Y;
    a.ws = ws;
    a.m_sizes = m_sizes;
    a.status = status;
    a.err = device_error_word();
    if (!a.err) return cudaErrorUnknown;
    a.M_total = M_total;
    a.N = N;
    a.K = K;
    a.num_groups = num_groups;
    const bool batched = m_sizes == nullptr && num_groups > 1;
    if (batched && (batch_rows < 1 || (long long)batch_rows * num_groups != M_total))
        return cudaErrorInvalidValue;
    a.bt = p.tile_tokens;
    a.n_tiles = p.n_tiles;
    a.split_k = p.split_k;
    a.gps = p.groups_per_slice;
    a.x_stages = p.x_stages;
    a.w_stages = p.w_stages;
    a.a_stages = tensor_a_stages(p.tile_tokens, p.occupancy, p.sep_epilogue);
    a.tmem_cols = tensor_tmem_cols(p.tile_tokens, p.occupancy, p.sep_epilogue);
    a.dcols = p.sep_epilogue ? 2 * p.tile_tokens : p.tile_tokens;
    a.opt_bits = ((N % 8 == 0) && (reinterpret_cast<uintptr_t>(Y) % 16 == 0) ? kTcVecStore : 0) |
                 (reinterpret_cast<uintptr_t>(S) % (2 * p.sub) == 0 ? kTcScaleVec : 0) |
                 (reinterpret_cast<uintptr_t>(Z) % p.sub == 0 ? kTcZeroVec : 0);
    a.w_group_stride = packed_bytes(N, K);
    a.s_group_stride = (unsigned long long)N * (K / kGroup) * p.sub;

    const size_t smem =
        tensor_smem_bytes(p.tile_tokens, p.x_stages, p.w_stages, p.occupancy, num_groups, p.sep_epilogue);
    if (smem > size_t(tensor_smem_budget(p.occupancy))) return cudaErrorInvalidValue;
    if (p.sub == 2) return launch_tc_sub<2>(p, tmap, a, batched, smem, s, Z);
    if (p.sub == 4) return launch_tc_sub<4>(p, tmap, a, batched, smem, s, Z);
    return launch_tc_sub<1>(p, tmap, a, batched, smem, s, Z);
}

}  // namespace w4a16
