// api.cu -- the C ABI: argument checks, the arm / split-K dispatcher, launches.
//
// Dispatch rule.  Few tokens are HBM-bound and go to the decode arm; the
// pages split their kernels the same way ("Add Triton BF16xINT4 rowwise GEMM
// for ROCm gfx942/gfx950", "Performance": shapes below the ridge point are
// memory-bound, above it compute-bound).  Split-K is chosen only when the
// natural grid is too small to occupy the GPU, and slices always cover whole
// 128-wide scale groups (the occupancy argument of that page's "Split-K
// without atomics" paragraph, here computed from the device's SM count rather
// than autotuned).
#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <cuda_runtime.h>

#include "w4a16.h"
#include "common.cuh"
#include "internal.h"

namespace w4a16 {

int device_sm_count(int *sms) {
    static std::atomic<int> cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return int(e);
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) { *sms = c; return 0; }
    }
    int v = 0;
    e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return int(e);
    if (dev >= 0 && dev < 64) cache[dev].store(v, std::memory_order_relaxed);
    *sms = v;
    return 0;
}

}  // namespace w4a16

using namespace w4a16;

namespace {

constexpr int kDecodeCtasPerSm = 2;           // resident decode CTAs per SM
constexpr int kDecodeInFlight = 3;            // bulk copies (ring stages) in the air per decode CTA
constexpr double kHbmBytesPerS = 6.5e12;      // planning figures, not measurements
constexpr double kCtaBytesPerS = 25e9;        // one CTA's streaming rate (32 KB in flight)
constexpr double kL2BytesPerS = 20e12;
// The tensor arm's fp32 partials (up to tens of MB for a long prefill) are
// charged at HBM speed: measured on GB300, 2048x2560x9728 split 2 (42 MB of
// partials) took 88.4 us against 78.4 us unsplit in 160-token tiles.
constexpr double kTensorPartialBytesPerS = 6.5e12;
// Measured on GB300 with per-CTA %globaltimer timelines of back-to-back
// calls: after the decode kernel's last CTA, the reduce kernel waits about
// 0.7 us for the grid to complete, works about 0.85 us, and the next kernel
// starts about 0.7 us after it (one such boundary every plan has).
constexpr double kReduceSeconds = 1.5e-6;        // reduce kernel and its extra launch boundary
constexpr double kTensorReduceSeconds = 0.5e-6;  // the tensor arm's plans were tuned with this
constexpr double kWholeKSeconds = 0.2e-6;        // whole-K kernel: part sums
// The K-slice kernel stages its slice of X (converted to fp16) before its
// first stage, about 0.5 us longer than the whole-K kernel takes to receive
// the first stage's X with its weights.
constexpr double kSliceStagingSeconds = 0.5e-6;
constexpr double kReducePerSliceSeconds = 0.01e-6;  // reduce latency per extra slice
constexpr int kDecodeMaxM = 16;               // auto dispatch: M <= 16 -> decode arm
constexpr double kClockHz = 1.9e9;            // planning clock
constexpr int kTensorMaxWStages = 8;
constexpr double kTcChainClk = 500.0;         // one CTA's per-K-block dependency chain
constexpr double kTcSmallTileKbClk = 800.0;   // per-SM cycles per K block, tiles <= 128 tokens

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Scale groups of 128, 64 or 32 columns; K stays a multiple of 128 (the
// packed layout's block), so every 128-wide block holds 128 / group_size
// whole scale groups.
w4a16_status check_shape(int M, int N, int K, int group_size) {
    if (group_size != 128 && group_size != 64 && group_size != 32) return W4A16_ERR_UNSUPPORTED;
    if (M < 0 || N < 1 || K < kGroup || K % kGroup) return W4A16_ERR_INVALID_ARG;
    if (N > (1 << 24) || K > (1 << 20) || M > (1 << 24)) return W4A16_ERR_INVALID_ARG;
    return W4A16_OK;
}

struct Plan {
    int arm;
    DecodePlan decode;
    TensorPlan tensor;
    int split_k;
    size_t ws_bytes;
    int ctas;
    int tile_tokens;
};

int ceil_div(long long a, long long b) { return int((a + b - 1) / b); }

// Measured on GB300 across the decode workloads (1 to 16 tokens, N 2560 to
// 19456, K 2560 to 9728, weights resident): at equal modelled time, 8- and
// 4-group slices run fastest (8 first: fewer tile epilogues per CTA), then 2,
// 16 and 1.  The factor breaks near-ties in that order.
double decode_slice_preference(int gps) {
    switch (gps) {
        case 4: return 1.0;
        case 8: return 1.0;
        case 2: return 1.06;
        case 16: return 1.08;
        default: return 1.12;
    }
}

// Decode-arm grid: each CTA keeps one K slice (gps groups) and streams tiles
// c, c + C, ... of it.  Modelled time = max(all weight bytes at HBM speed,
// the busiest CTA's bytes at one CTA's streaming rate) + the split-K
// workspace round trip; at most kDecodeCtasPerSm CTAs per SM are launched so
// that all of them are resident at once.
// Whole-K plans (no split-K) compete with the sliced ones: each CTA owns
// B 16-row blocks over all of K, 8 / B K-parts per CTA; one CTA per B blocks,
// all resident at once.  wk: 0 = either kernel, 1 = whole-K only, 2 = slices only.
// batch > 1: that many independent products of this shape share the GPU
// (each gets its share of the CTA slots; the weight stream is all of theirs).
// sub: scale groups per 128-wide block (1, 2, 4).  Smaller groups keep
// GPS * sub scales of a row in registers (at most 16, 8 for two token
// octets) and have only the slice kernel; their scale bytes (2 per group)
// scale the modelled weight stream relative to 128-wide groups, for which the
// constants were measured.
// zp: the zero-point kernels, which hold half as many scale groups of a row
// per slice (their zero points sit in registers too).
void plan_decode(int M, int N, int K, int sms, int forced_split, int wk, int batch, int sub,
                 bool zp, DecodePlan *d) {
    const int groups = K / kGroup;
    const double sbytes = (0.5 + 2.0 * sub / kGroup) / (0.5 + 2.0 / kGroup);
    d->mt = M <= 8 ? 1 : 2;
    d->token_blocks = ceil_div(M, 8 * d->mt);
    d->n_tiles = ceil_div(N, kTileRows);
    d->batch = batch;
    d->sub = sub;
    long long slots = (long long)kDecodeCtasPerSm * sms / batch;
    if (slots < 1) slots = 1;
    const double w_bytes = double(batch) * d->n_tiles * kTileRows * double(K) / 2.0 * sbytes;
    double best = 1e30;
    d->split_k = groups;
    d->groups_per_slice = 1;
    d->ctas_per_slice = 1;
    d->ring = 0;
    d->in_flight = kDecodeInFlight;
    d->wk_blocks = 0;
    if (wk != 2 && forced_split <= 1 && sub == 1 && !zp) {
        // Whole-K plans: B blocks of 16 rows per CTA, every CTA resident.
        const long long blocks = (N + 15) / 16;
        for (int B : {8, 4, 2, 1}) {
            if (!decode_wk_fits(M, K, B)) continue;
            const long long ctas = (blocks + B - 1) / B;
            if (ctas > slots) continue;   // per entry
            const double cta_bytes = double(B) * 16.0 * double(K) / 2.0;
            double t = w_bytes / kHbmBytesPerS;
            if (cta_bytes / kCtaBytesPerS > t) t = cta_bytes / kCtaBytesPerS;
            t += kWholeKSeconds;
            if (t < best * 0.999) {
                best = t;
                d->wk_blocks = B;
                d->split_k = 1;
                d->groups_per_slice = groups;
                d->ctas_per_slice = int(ctas);
            }
        }
        if (wk == 1) return;
    }
    if (wk == 1) return;   // (smaller groups, zero points: no whole-K kernel)
    // Slices hold 1, 2, 4, 8 or 16 groups and divide K exactly (the kernel
    // unrolls a slice at compile time).  A forced split picks the feasible slice count
    // closest to the request from above.
    // 16-group slices only for one token octet (register budget).
    const int gps_max = (d->mt == 1 ? 16 : 8) / sub / (zp ? 2 : 1);
    int forced_gps = 0;
    if (forced_split > 0) {
        for (int gps : {16, 8, 4, 2, 1})
            if (gps <= gps_max && groups % gps == 0 && groups / gps >= forced_split) {
                forced_gps = gps;
                break;
            }
        if (!forced_gps) forced_gps = 1;
    }
    for (int gps : {16, 8, 4, 2, 1}) {
        if (gps > gps_max || groups % gps) continue;
        if (forced_gps && gps != forced_gps) continue;
        if (decode_ring_stages(M, d->mt, gps, sub) == 0) continue;   // shared memory
        const int sk = groups / gps;
        const long long per_slice = slots / ((long long)sk * d->token_blocks);
        const int cmax = int(per_slice < 1 ? 1 : (per_slice > d->n_tiles ? d->n_tiles : per_slice));
        for (int C = cmax; C >= 1; --C) {
            const int tiles_per = ceil_div(d->n_tiles, C);
            if (C < cmax && ceil_div(d->n_tiles, C + 1) == tiles_per) continue;  // same critical path, fewer CTAs
            const double cta_bytes = double(tiles_per) * 2.0 * gps * kChunkBytes * d->token_blocks * sbytes;
            double t = w_bytes * d->token_blocks / kHbmBytesPerS;
            const double t_cta = cta_bytes / kCtaBytesPerS;
            if (t_cta > t) t = t_cta;
            t += kSliceStagingSeconds;
            if (sk > 1)
                t += 2.0 * double(sk) * M * N * 4.0 / kL2BytesPerS + kReduceSeconds +
                     kReducePerSliceSeconds * sk;
            t *= decode_slice_preference(gps);
            if (t < best * 0.999) {
                best = t;
                d->split_k = sk;
                d->groups_per_slice = gps;
                d->ctas_per_slice = C;
                d->wk_blocks = 0;
                d->ring = decode_ring_stages(M, d->mt, gps, sub);
            }
        }
    }
}

// Tensor-arm tiles: 128 weight rows x bt tokens, K split into sk slices.
// Modelled per-K-block cycles = max(MMA: 2 bt, dequant floor, weight bytes at
// one SM's HBM share + activation bytes at one SM's L2 share); a CTA's time is
// its tile count times (K blocks x that + a fixed per-tile cost), plus the
// split-K round trip.
// Ring depths for the CTA's shared-memory budget: the deepest X ring of 4, 3
// or 2 stages that still leaves at least 4 W stages (one per dequantiser
// team), then as many W stages (8 KB each, up to kTensorMaxWStages) as fit.
// Returns false if even 2 + 4 does not fit.
bool tensor_rings(int bt, int num_groups, int occupancy, bool sep, int *x_stages, int *w_stages) {
    const size_t budget = size_t(tensor_smem_budget(occupancy));
    const size_t fixed = tensor_smem_bytes(bt, 0, 0, occupancy, num_groups, sep);
    if (budget <= fixed) return false;
    const size_t avail = budget - fixed;
    const size_t x_stage = 2 * size_t(bt) * 128 + 16;     // + its two barriers
    const size_t w_stage = size_t(kChunkBytes) * 2 + 16;
    for (int sx = 4; sx >= 2; --sx) {
        if (sx * x_stage > avail) continue;
        size_t sw = (avail - sx * x_stage) / w_stage;
        if (sw > size_t(kTensorMaxWStages)) sw = kTensorMaxWStages;
        if (sw >= size_t(kTensorTeamsPlain)) {
            *x_stages = sx;
            *w_stages = int(sw);
            return true;
        }
    }
    return false;
}

// Tensor-arm tiles: 128 weight rows x bt tokens, K split into sk slices, one
// CTA per SM (608 threads in the plain form, 480 with a separate epilogue).
// Per K block an SM needs at least max(MMA: 2 bt cycles, a dequant floor,
// weight bytes at its HBM share + activation bytes at its L2 share), and a
// CTA cannot go faster than its dependency chain (kTcChainClk per K block).
// batch_rows > 0: a batched product, num_groups entries of batch_rows rows
// (M = their total): the plain product per entry, split-K allowed.
// sub: scale groups per 128-wide block (1, 2, 4); the dequantisers load
// sub scales per row and block, which the model does not charge.
w4a16_status plan_tensor(int M, int N, int K, int sms, int forced_split, int forced_bt,
                         int num_groups, TensorPlan *t, int batch_rows, int sub) {
    const int groups = K / kGroup;
    t->sub = sub;
    const bool grouped = num_groups > 1 && batch_rows == 0;
    t->n_tiles = ceil_div(N, kTileRows);
    double best = 1e30;
    int found = 0;
    for (int bt = 32; bt <= 256; bt += 32) {
        if (forced_bt > 0 && bt != forced_bt) continue;
        // a batched entry's tile wider than the entry is all padding
        if (forced_bt == 0 && batch_rows > 0 && bt >= batch_rows + 32) continue;
        for (int variant = 0; variant < 2; ++variant) {
            // the plain form; a separate epilogue
            const int occ = 1;
            const bool sep = variant == 1;
            // TMEM share too small for one A stage per dequantiser team
            if (tensor_a_stages(bt, occ, sep) < (sep ? kTensorTeamsSep : kTensorTeamsPlain)) continue;
            int sx = 0, sw = 0;
            if (!tensor_rings(bt, num_groups, occ, sep, &sx, &sw)) continue;
            const int max_sk = grouped ? 1 : (groups < 16 ? groups : 16);
            for (int sk_req = 1; sk_req <= max_sk; ++sk_req) {
                int sk = sk_req;
                if (forced_split > 0) sk = forced_split > groups ? groups : forced_split;
                if (grouped) sk = 1;
                const int gps = ceil_div(groups, sk);
                sk = ceil_div(groups, gps);
                // Grouped: the sizes live on the device; plan with the average
                // size and, per group, half a tile more for its ragged last
                // tile (the remainder of a size that varies is about uniform).
                // Measured on GB300 (8 groups of about 512 rows, N=2048,
                // K=4096): 128-token tiles 63 us, 256-token tiles 87 us.
                const double rows_per_unit = double(M) / num_groups;
                const long long t_tiles =
                    !grouped ? (long long)num_groups * ceil_div((long long)M / num_groups, bt)
                             : (long long)std::ceil(num_groups * (rows_per_unit / bt + 0.5));
                const long long tiles = (long long)t->n_tiles * t_tiles * sk;
                const long long slots = (long long)occ * sms;
                const long long ctas = tiles < slots ? tiles : slots;
                const int conc = int(ceil_div(ctas, sms));
                const double kb_tp = std::max(std::max(2.0 * bt, 150.0),
                                              kChunkBytes / 22.0 + bt * 128.0 / 64.0);
                // A grid that fills the SMs without a split, with tiles of up to
                // 128 tokens or few tokens in all: measured on GB300, an SM then
                // spends about kTcSmallTileKbClk per K block whatever the tile
                // width and whether one or two CTAs share it, so wider tiles
                // buy nothing and splitting K only adds the reduce.  (Wide
                // tiles of many tokens, the prefill case, keep the model above.)
                const bool full = (long long)t->n_tiles * t_tiles >= sms;
                const int rows_entry = batch_rows > 0 ? batch_rows : M;   // tokens of one product
                const double floor_kb = (full && (bt <= 128 || rows_entry <= 256)) ? kTcSmallTileKbClk : 0.0;
                const double kb = std::max(std::max(kb_tp, kTcChainClk / conc), floor_kb);
                const double per_cta_tiles = double(ceil_div(tiles, ctas));
                // Per-tile fixed cost: the epilogue, which a separate epilogue
                // overlaps with the next tile (except the CTA's last one).
                // A split tile drains fp32 partials through the dequant warps
                // while the tensor pipe waits; measured on GB300 that stall
                // grows with the tile width (about (bt / 128)^2 x 1500 cycles
                // per tile before a CTA's last: 512x7168x8192 split 4 took
                // 76.3 us, unsplit 51.9 us; 2048x8192x8192 split 2 288 us,
                // unsplit 199 us).
                const double e_split = 1500.0 * std::max(1.0, (bt / 128.0) * (bt / 128.0));
                // The plain form's in-line drain of a bf16 tile before the
                // CTA's next tile stalls the same way (measured on GB300:
                // 4096x19456x2560 in plain 256-token tiles 312 us, in
                // separate-epilogue 192-token tiles 248 us; 2048x19456x2560
                // 158 vs 125 us).
                const double epi = sep ? 1500.0 : 1500.0 + (per_cta_tiles - 1) * e_split;
                // Plain tiles wider than 192 tokens keep only two 64 KB X
                // stages next to their in-line drain; with several tiles per
                // CTA they measure ~1.6x the per-K-block time of
                // separate-epilogue 192-token tiles where the terms above give
                // ~1.2x (GB300: 1024x19456x2560 79.7 against 68.9 us,
                // 4096x8192x8192 357 against 336 us, 2048x4096x4096 58.0
                // against 54.4 us).  With the penalty the narrower plans
                // chosen measured faster on every shape it moved
                // (2048x4096x4096 at 160 tokens 52.1 us, 1024x7168x8192
                // 96.5 against 103.4 us).
                const double wide = (!sep && bt > 192 && per_cta_tiles > 1) ? 1.25 : 1.0;
                double time = (per_cta_tiles * conc * 2.0 * gps * kb * wide + epi) / kClockHz;
                if (sk > 1) time += 2.0 * sk * double(M) * N * 4.0 / kTensorPartialBytesPerS + kTensorReduceSeconds;
                if (time < best * 0.999) {
                    best = time;
                    t->tile_tokens = bt;
                    t->split_k = sk;
                    t->groups_per_slice = gps;
                    t->t_tiles = int(t_tiles);
                    t->ctas = int(ctas);
                    t->x_stages = sx;
                    t->w_stages = sw;
                    t->occupancy = occ;
                    t->sep_epilogue = sep;
                    t->smem_bytes = tensor_smem_bytes(bt, sx, sw, occ, num_groups, sep);
                    found = 1;
                }
                if (forced_split > 0 || grouped) break;
            }
        }
    }
    return found ? W4A16_OK : W4A16_ERR_UNSUPPORTED;
}

// batch: independent products of this shape in one launch (1: a plain call).
// sub: scale groups per 128-wide block (128 / group_size).  W4A16_FLAG_ZERO_POINTS
// in opts plans the zero-point kernels.
// sms > 0: plan for a device with that many SMs instead of querying the
// current one (host-only planning).
w4a16_status plan_call(int M, int N, int K, const w4a16_options *opts, Plan *p, int batch = 1,
                       int sub = 1, int sms_given = 0) {
    std::memset(p, 0, sizeof *p);
    int arm = opts ? opts->arm : W4A16_ARM_AUTO;
    if (arm != W4A16_ARM_AUTO && arm != W4A16_ARM_DECODE && arm != W4A16_ARM_TENSOR)
        return W4A16_ERR_INVALID_ARG;
    if (opts && opts->split_k < 0) return W4A16_ERR_INVALID_ARG;
    const int flags = opts ? opts->flags : 0;
    if (flags & ~int(W4A16_FLAG_RESIDENT_WEIGHTS | W4A16_FLAG_DECODE_WHOLE_K | W4A16_FLAG_DECODE_K_SLICES |
                     W4A16_FLAG_ZERO_POINTS | W4A16_FLAG_TEST_STALL))
        return W4A16_ERR_INVALID_ARG;
    const bool stall = (flags & W4A16_FLAG_TEST_STALL) != 0;
    const bool zp = (flags & W4A16_FLAG_ZERO_POINTS) != 0;
    if ((flags & W4A16_FLAG_DECODE_WHOLE_K) && (flags & W4A16_FLAG_DECODE_K_SLICES))
        return W4A16_ERR_INVALID_ARG;
    int wk = (flags & W4A16_FLAG_DECODE_WHOLE_K) ? 1 : (flags & W4A16_FLAG_DECODE_K_SLICES) ? 2 : 0;
    if (stall) {
        // Only the K-slice decode kernel has the stall mode.
        if (wk == 1) return W4A16_ERR_UNSUPPORTED;
        wk = 2;
    }
    const int forced_bt = opts ? opts->tile_tokens : 0;
    if (forced_bt != 0 && (forced_bt < 32 || forced_bt > 256 || forced_bt % 32))
        return W4A16_ERR_UNSUPPORTED;
    int sms = sms_given;
    if (sms <= 0 && (device_sm_count(&sms) != 0 || sms < 1)) return W4A16_ERR_CUDA;
    if (arm == W4A16_ARM_AUTO) arm = M <= kDecodeMaxM ? W4A16_ARM_DECODE : W4A16_ARM_TENSOR;
    if (arm == W4A16_ARM_DECODE && forced_bt != 0) return W4A16_ERR_INVALID_ARG;
    if (stall && arm != W4A16_ARM_DECODE) return W4A16_ERR_UNSUPPORTED;
    p->arm = arm;
    if (arm == W4A16_ARM_DECODE) {
        DecodePlan &d = p->decode;
        plan_decode(M, N, K, sms, opts ? opts->split_k : 0, wk, batch, sub, zp, &d);
        if (wk == 1 && d.wk_blocks == 0) return W4A16_ERR_UNSUPPORTED;
        if (stall) {
            // Test only: no weight copies, and waits that give up after 1 ms.
            d.in_flight = 0;
            d.wait_us = 1000;
        }
        p->split_k = d.split_k;
        p->ctas = batch * (d.wk_blocks ? d.ctas_per_slice : d.ctas_per_slice * d.split_k * d.token_blocks);
        p->tile_tokens = 8 * d.mt;
    } else {
        if (wk == 1) return W4A16_ERR_UNSUPPORTED;
        TensorPlan &t = p->tensor;
        w4a16_status st = plan_tensor(batch * M, N, K, sms, opts ? opts->split_k : 0, forced_bt,
                                      batch, &t, batch > 1 ? M : 0, sub);
        if (st != W4A16_OK) return st;
        p->split_k = t.split_k;
        p->ctas = t.ctas;
        p->tile_tokens = t.tile_tokens;
    }
    p->ws_bytes = p->split_k > 1
                      ? size_t(p->split_k) * size_t(batch) * size_t(M) * size_t(N) * sizeof(float)
                      : 0;
    return W4A16_OK;
}

w4a16_status from_cuda(cudaError_t e) { return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA; }

}  // namespace

extern "C" {

const char *w4a16_status_string(int status) {
    switch (status) {
        case W4A16_OK: return "ok";
        case W4A16_ERR_INVALID_ARG: return "invalid argument";
        case W4A16_ERR_UNSUPPORTED: return "unsupported configuration";
        case W4A16_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case W4A16_ERR_CUDA: return "CUDA error";
        default: return "unknown status";
    }
}

int w4a16_layout_version(void) { return kLayoutVersion; }

size_t w4a16_packed_weight_bytes(int N, int K) {
    if (N < 1 || K < kGroup || K % kGroup) return 0;
    return packed_bytes(N, K);
}

w4a16_status w4a16_pack_weights(const uint8_t *w_canon, uint8_t *w_packed, int N, int K,
                                void *stream) {
    if (!w_canon || !w_packed) return W4A16_ERR_INVALID_ARG;
    if (N < 1 || K < kGroup || K % kGroup || N > (1 << 24) || K > (1 << 20))
        return W4A16_ERR_INVALID_ARG;
    if (!aligned(w_packed, 16)) return W4A16_ERR_INVALID_ARG;
    return from_cuda(launch_pack(w_canon, w_packed, N, K, static_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_plan(int M, int N, int K, int group_size, const w4a16_options *opts,
                        w4a16_plan_info *info) {
    w4a16_status st = check_shape(M, N, K, group_size);
    if (st != W4A16_OK) return st;
    Plan p;
    st = plan_call(M, N, K, opts, &p, 1, kGroup / group_size);
    if (st != W4A16_OK) return st;
    if (info) {
        info->arm = p.arm;
        info->split_k = p.split_k;
        info->tile_tokens = p.tile_tokens;
        info->ctas = p.ctas;
        info->workspace_bytes = M == 0 ? 0 : p.ws_bytes;
        info->whole_k = p.arm == W4A16_ARM_DECODE && p.decode.wk_blocks > 0;
    }
    return W4A16_OK;
}

w4a16_status w4a16_workspace_bytes(int M, int N, int K, int group_size, size_t *bytes) {
    if (!bytes) return W4A16_ERR_INVALID_ARG;
    w4a16_plan_info info;
    w4a16_status st = w4a16_plan(M, N, K, group_size, nullptr, &info);
    if (st != W4A16_OK) return st;
    *bytes = info.workspace_bytes;
    return W4A16_OK;
}

// zeros != nullptr: the zero-point variant (opts must then carry
// W4A16_FLAG_ZERO_POINTS, which w4a16_gemm_zp adds).
static w4a16_status gemm_impl(const w4a16_bf16 *X, const uint8_t *W_packed,
                              const w4a16_bf16 *scales, w4a16_bf16 *Y, int M, int N, int K,
                              int group_size, void *workspace, size_t workspace_bytes,
                              const w4a16_options *opts, bool with_reduce, int *split_out,
                              void *stream, int batch = 1, const uint8_t *zeros = nullptr) {
    w4a16_status st = check_shape(M, N, K, group_size);
    if (st != W4A16_OK) return st;
    if (batch < 1 || batch > kMaxGroups || (long long)batch * M > (1 << 24)) return W4A16_ERR_INVALID_ARG;
    if (M == 0) {
        if (split_out) *split_out = 1;
        return W4A16_OK;
    }
    const bool zp_flag = opts && (opts->flags & W4A16_FLAG_ZERO_POINTS);
    if (zp_flag != (zeros != nullptr)) return W4A16_ERR_INVALID_ARG;
    if (!X || !W_packed || !scales || !Y) return W4A16_ERR_INVALID_ARG;
    if (!aligned(X, 16) || !aligned(W_packed, 16) || !aligned(scales, 2) || !aligned(Y, 2))
        return W4A16_ERR_INVALID_ARG;
    Plan p;
    st = plan_call(M, N, K, opts, &p, batch, kGroup / group_size);
    if (st != W4A16_OK) return st;
    if (split_out) *split_out = p.split_k;
    if (p.ws_bytes > 0) {
        if (!workspace || workspace_bytes < p.ws_bytes) return W4A16_ERR_WORKSPACE_TOO_SMALL;
        if (!aligned(workspace, 16)) return W4A16_ERR_INVALID_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float *ws = static_cast<float *>(workspace);
    cudaError_t e;
    const bool resident = opts && (opts->flags & W4A16_FLAG_RESIDENT_WEIGHTS);
    if (p.arm == W4A16_ARM_DECODE && p.decode.wk_blocks > 0)
        e = launch_decode_wk(p.decode.wk_blocks, p.decode.ctas_per_slice, batch, X, W_packed, scales,
                             Y, resident, M, N, K, s);
    else if (p.arm == W4A16_ARM_DECODE)
        e = launch_decode(p.decode, X, W_packed, scales, Y, ws, resident, M, N, K, s, zeros);
    else
        e = launch_tensor(p.tensor, X, W_packed, scales, Y, ws, nullptr, nullptr, batch, batch * M, N,
                          K, s, batch > 1 ? M : 0, zeros);
    if (e != cudaSuccess) return W4A16_ERR_CUDA;
    if (with_reduce && p.split_k > 1) {
        e = launch_reduce(ws, Y, p.split_k, (long long)batch * M * N, true, s);
        if (e != cudaSuccess) return W4A16_ERR_CUDA;
    }
    return W4A16_OK;
}

w4a16_status w4a16_gemm_ex(const w4a16_bf16 *X, const uint8_t *W_packed,
                           const w4a16_bf16 *scales, w4a16_bf16 *Y, int M, int N, int K,
                           int group_size, void *workspace, size_t workspace_bytes,
                           const w4a16_options *opts, void *stream) {
    return gemm_impl(X, W_packed, scales, Y, M, N, K, group_size, workspace, workspace_bytes,
                     opts, true, nullptr, stream);
}

w4a16_status w4a16_gemm_partials(const w4a16_bf16 *X, const uint8_t *W_packed,
                                 const w4a16_bf16 *scales, w4a16_bf16 *Y, int M, int N, int K,
                                 int group_size, void *workspace, size_t workspace_bytes,
                                 const w4a16_options *opts, int *split_k_out, void *stream) {
    return gemm_impl(X, W_packed, scales, Y, M, N, K, group_size, workspace, workspace_bytes,
                     opts, false, split_k_out, stream);
}

w4a16_status w4a16_gemm(const w4a16_bf16 *X, const uint8_t *W_packed, const w4a16_bf16 *scales,
                        w4a16_bf16 *Y, int M, int N, int K, int group_size, void *workspace,
                        size_t workspace_bytes, void *stream) {
    return w4a16_gemm_ex(X, W_packed, scales, Y, M, N, K, group_size, workspace, workspace_bytes,
                         nullptr, stream);
}

w4a16_status w4a16_plan_batched(int batch, int M, int N, int K, int group_size,
                                const w4a16_options *opts, w4a16_plan_info *info) {
    return w4a16_plan_for_sms(0, batch, M, N, K, group_size, opts, info);
}

w4a16_status w4a16_plan_for_sms(int sms, int batch, int M, int N, int K, int group_size,
                                const w4a16_options *opts, w4a16_plan_info *info) {
    w4a16_status st = check_shape(M, N, K, group_size);
    if (st != W4A16_OK) return st;
    if (sms < 0 || sms > 4096) return W4A16_ERR_INVALID_ARG;
    if (batch < 1 || batch > kMaxGroups || (long long)batch * M > (1 << 24)) return W4A16_ERR_INVALID_ARG;
    Plan p;
    st = plan_call(M, N, K, opts, &p, batch, kGroup / group_size, sms);
    if (st != W4A16_OK) return st;
    if (info) {
        info->arm = p.arm;
        info->split_k = p.split_k;
        info->tile_tokens = p.tile_tokens;
        info->ctas = p.ctas;
        info->workspace_bytes = M == 0 ? 0 : p.ws_bytes;
        info->whole_k = p.arm == W4A16_ARM_DECODE && p.decode.wk_blocks > 0;
    }
    return W4A16_OK;
}

w4a16_status w4a16_gemm_batched(const w4a16_bf16 *X, const uint8_t *W_packed,
                                const w4a16_bf16 *scales, w4a16_bf16 *Y, int batch, int M, int N,
                                int K, int group_size, void *workspace, size_t workspace_bytes,
                                const w4a16_options *opts, void *stream) {
    return gemm_impl(X, W_packed, scales, Y, M, N, K, group_size, workspace, workspace_bytes, opts,
                     true, nullptr, stream, batch);
}

w4a16_status w4a16_gemm_zp(const w4a16_bf16 *X, const uint8_t *W_packed, const w4a16_bf16 *scales,
                           const uint8_t *zeros, w4a16_bf16 *Y, int M, int N, int K,
                           int group_size, void *workspace, size_t workspace_bytes,
                           const w4a16_options *opts, void *stream) {
    if (M > 0 && !zeros) return W4A16_ERR_INVALID_ARG;
    w4a16_options o = {};
    if (opts) o = *opts;
    o.flags |= W4A16_FLAG_ZERO_POINTS;
    return gemm_impl(X, W_packed, scales, Y, M, N, K, group_size, workspace, workspace_bytes, &o,
                     true, nullptr, stream, 1, zeros);
}

w4a16_status w4a16_grouped_workspace_bytes(int num_groups, int M_total, int N, int K,
                                           int group_size, size_t *bytes) {
    if (!bytes) return W4A16_ERR_INVALID_ARG;
    w4a16_status st = check_shape(M_total, N, K, group_size);
    if (st != W4A16_OK) return st;
    if (num_groups < 1 || num_groups > kMaxGroups) return W4A16_ERR_INVALID_ARG;
    *bytes = 16;
    return W4A16_OK;
}

static w4a16_status grouped_impl(const w4a16_bf16 *X, const uint8_t *W_packed,
                                 const w4a16_bf16 *scales, const uint8_t *zeros,
                                 const int32_t *M_sizes_dev, w4a16_bf16 *Y, int num_groups,
                                 int M_total, int N, int K, int group_size, void *workspace,
                                 size_t workspace_bytes, void *stream) {
    w4a16_status st = check_shape(M_total, N, K, group_size);
    if (st != W4A16_OK) return st;
    if (num_groups < 1 || num_groups > kMaxGroups) return W4A16_ERR_INVALID_ARG;
    if (!X || !W_packed || !scales || !M_sizes_dev || !Y) return W4A16_ERR_INVALID_ARG;
    if (!aligned(X, 16) || !aligned(W_packed, 16) || !aligned(scales, 2) || !aligned(Y, 2) ||
        !aligned(M_sizes_dev, 4))
        return W4A16_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < 16) return W4A16_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(workspace, 16)) return W4A16_ERR_INVALID_ARG;
    if (M_total == 0) return W4A16_OK;
    int sms = 0;
    if (device_sm_count(&sms) != 0 || sms < 1) return W4A16_ERR_CUDA;
    TensorPlan t;
    st = plan_tensor(M_total, N, K, sms, 1, 0, num_groups, &t, 0, kGroup / group_size);
    if (st != W4A16_OK) return st;
    // Enough CTAs for any split of M_total into the groups: the tile count is
    // at most n_tiles * (ceil(M_total / bt) + num_groups).
    const long long bound = (long long)t.n_tiles * (ceil_div(M_total, t.tile_tokens) + num_groups);
    const long long slots = (long long)t.occupancy * sms;
    t.ctas = int(bound < slots ? bound : slots);
    cudaError_t e = launch_tensor(t, X, W_packed, scales, Y, nullptr, M_sizes_dev,
                                  static_cast<int *>(workspace), num_groups, M_total, N, K,
                                  static_cast<cudaStream_t>(stream), 0, zeros);
    return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}

w4a16_status w4a16_gemm_grouped(const w4a16_bf16 *X, const uint8_t *W_packed,
                                const w4a16_bf16 *scales, const int32_t *M_sizes_dev,
                                w4a16_bf16 *Y, int num_groups, int M_total, int N, int K,
                                int group_size, void *workspace, size_t workspace_bytes,
                                void *stream) {
    return grouped_impl(X, W_packed, scales, nullptr, M_sizes_dev, Y, num_groups, M_total, N, K,
                        group_size, workspace, workspace_bytes, stream);
}

w4a16_status w4a16_gemm_grouped_zp(const w4a16_bf16 *X, const uint8_t *W_packed,
                                   const w4a16_bf16 *scales, const uint8_t *zeros,
                                   const int32_t *M_sizes_dev, w4a16_bf16 *Y, int num_groups,
                                   int M_total, int N, int K, int group_size, void *workspace,
                                   size_t workspace_bytes, void *stream) {
    if (!zeros) return W4A16_ERR_INVALID_ARG;
    return grouped_impl(X, W_packed, scales, zeros, M_sizes_dev, Y, num_groups, M_total, N, K,
                        group_size, workspace, workspace_bytes, stream);
}

w4a16_status w4a16_gemm_batched_zp(const w4a16_bf16 *X, const uint8_t *W_packed,
                                   const w4a16_bf16 *scales, const uint8_t *zeros, w4a16_bf16 *Y,
                                   int batch, int M, int N, int K, int group_size, void *workspace,
                                   size_t workspace_bytes, const w4a16_options *opts,
                                   void *stream) {
    if (M > 0 && !zeros) return W4A16_ERR_INVALID_ARG;
    w4a16_options o = {};
    if (opts) o = *opts;
    o.flags |= W4A16_FLAG_ZERO_POINTS;
    return gemm_impl(X, W_packed, scales, Y, M, N, K, group_size, workspace, workspace_bytes, &o,
                     true, nullptr, stream, batch, zeros);
}

w4a16_status w4a16_dequant_fp32(const uint8_t *W_packed, const w4a16_bf16 *scales, float *out,
                                int N, int K, int group_size, void *stream) {
    w4a16_status st = check_shape(0, N, K, group_size);
    if (st != W4A16_OK) return st;
    if (!W_packed || !scales || !out) return W4A16_ERR_INVALID_ARG;
    if (!aligned(W_packed, 16) || !aligned(scales, 2) || !aligned(out, 4))
        return W4A16_ERR_INVALID_ARG;
    return from_cuda(launch_dequant(W_packed, scales, out, false, N, K, group_size,
                                    static_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_dequant_bf16(const uint8_t *W_packed, const w4a16_bf16 *scales,
                                w4a16_bf16 *out, int N, int K, int group_size, void *stream) {
    w4a16_status st = check_shape(0, N, K, group_size);
    if (st != W4A16_OK) return st;
    if (!W_packed || !scales || !out) return W4A16_ERR_INVALID_ARG;
    if (!aligned(W_packed, 16) || !aligned(scales, 2) || !aligned(out, 2))
        return W4A16_ERR_INVALID_ARG;
    return from_cuda(launch_dequant(W_packed, scales, out, true, N, K, group_size,
                                    static_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_dequant_zp_fp32(const uint8_t *W_packed, const w4a16_bf16 *scales,
                                   const uint8_t *zeros, float *out, int N, int K, int group_size,
                                   void *stream) {
    w4a16_status st = check_shape(0, N, K, group_size);
    if (st != W4A16_OK) return st;
    if (!W_packed || !scales || !zeros || !out) return W4A16_ERR_INVALID_ARG;
    if (!aligned(W_packed, 16) || !aligned(scales, 2) || !aligned(out, 4)) return W4A16_ERR_INVALID_ARG;
    return from_cuda(launch_dequant(W_packed, scales, out, false, N, K, group_size,
                                    static_cast<cudaStream_t>(stream), zeros));
}

w4a16_status w4a16_dequant_zp_bf16(const uint8_t *W_packed, const w4a16_bf16 *scales,
                                   const uint8_t *zeros, w4a16_bf16 *out, int N, int K,
                                   int group_size, void *stream) {
    w4a16_status st = check_shape(0, N, K, group_size);
    if (st != W4A16_OK) return st;
    if (!W_packed || !scales || !zeros || !out) return W4A16_ERR_INVALID_ARG;
    if (!aligned(W_packed, 16) || !aligned(scales, 2) || !aligned(out, 2)) return W4A16_ERR_INVALID_ARG;
    return from_cuda(launch_dequant(W_packed, scales, out, true, N, K, group_size,
                                    static_cast<cudaStream_t>(stream), zeros));
}

w4a16_status w4a16_splitk_reduce(const float *ws, w4a16_bf16 *Y, int splits, int M, int N,
                                 void *stream) {
    if (splits < 1 || splits > 4096 || M < 0 || N < 1) return W4A16_ERR_INVALID_ARG;
    if (M == 0) return W4A16_OK;
    if (!ws || !Y || !aligned(ws, 16) || !aligned(Y, 2)) return W4A16_ERR_INVALID_ARG;
    return from_cuda(launch_reduce(ws, Y, splits, (long long)M * N, false,
                                   static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
