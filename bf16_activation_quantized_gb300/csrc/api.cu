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
#include <atomic>
#include <cstdint>
#include <cstring>
#include <cuda_runtime.h>

#include "../../include/w4a16.h"
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

constexpr int kDecodeMaxM = 16;
constexpr int kMaxSplit = 32;
constexpr int kMaxDecodeGroupsPerSlice = 64;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

w4a16_status check_shape(int M, int N, int K, int group_size) {
    if (group_size != kGroup) return W4A16_ERR_UNSUPPORTED;
    if (M < 0 || N < 1 || K < kGroup || K % kGroup) return W4A16_ERR_INVALID_ARG;
    if (N > (1 << 24) || K > (1 << 20) || M > (1 << 24)) return W4A16_ERR_INVALID_ARG;
    return W4A16_OK;
}

struct Plan {
    int arm;
    DecodePlan decode;
    int split_k;
    size_t ws_bytes;
    int ctas;
    int tile_tokens;
};

int ceil_div(long long a, long long b) { return int((a + b - 1) / b); }

// Slices of whole groups: at most `want` slices, each at most `max_gps` groups.
void make_slices(int groups, int want, int max_gps, int *split, int *gps) {
    if (want < 1) want = 1;
    if (want > groups) want = groups;
    int per = ceil_div(groups, want);
    if (per > max_gps) per = max_gps;
    *gps = per;
    *split = ceil_div(groups, per);
}

w4a16_status plan_call(int M, int N, int K, const w4a16_options *opts, Plan *p) {
    std::memset(p, 0, sizeof *p);
    int sms = 0;
    if (device_sm_count(&sms) != 0 || sms < 1) return W4A16_ERR_CUDA;
    const int arm_req = opts ? opts->arm : W4A16_ARM_AUTO;
    if (arm_req == W4A16_ARM_TENSOR) return W4A16_ERR_UNSUPPORTED;
    if (arm_req != W4A16_ARM_AUTO && arm_req != W4A16_ARM_DECODE) return W4A16_ERR_INVALID_ARG;
    if (opts && (opts->split_k < 0 || opts->tile_tokens != 0)) return W4A16_ERR_INVALID_ARG;

    const int groups = K / kGroup;
    DecodePlan &d = p->decode;
    d.mt = M <= 8 ? 1 : 2;
    d.token_blocks = ceil_div(M, 8 * d.mt);
    d.n_tiles = ceil_div(N, kTileRows);
    int want;
    if (opts && opts->split_k > 0) {
        want = opts->split_k;
    } else {
        // Aim for two resident CTAs per SM; one slice when the grid already fills it.
        const long long base = (long long)d.n_tiles * d.token_blocks;
        want = ceil_div(2LL * sms, base);
        if (want > kMaxSplit) want = kMaxSplit;
        if (M > kDecodeMaxM) want = 1;
    }
    make_slices(groups, want, kMaxDecodeGroupsPerSlice, &d.split_k, &d.groups_per_slice);
    p->arm = W4A16_ARM_DECODE;
    p->split_k = d.split_k;
    p->ws_bytes = d.split_k > 1 ? size_t(d.split_k) * size_t(M) * size_t(N) * sizeof(float) : 0;
    p->ctas = d.n_tiles * d.split_k * d.token_blocks;
    p->tile_tokens = 8 * d.mt;
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
    st = plan_call(M, N, K, opts, &p);
    if (st != W4A16_OK) return st;
    if (info) {
        info->arm = p.arm;
        info->split_k = p.split_k;
        info->tile_tokens = p.tile_tokens;
        info->ctas = p.ctas;
        info->workspace_bytes = M == 0 ? 0 : p.ws_bytes;
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

static w4a16_status gemm_impl(const w4a16_bf16 *X, const uint8_t *W_packed,
                              const w4a16_bf16 *scales, w4a16_bf16 *Y, int M, int N, int K,
                              int group_size, void *workspace, size_t workspace_bytes,
                              const w4a16_options *opts, bool with_reduce, int *split_out,
                              void *stream) {
    w4a16_status st = check_shape(M, N, K, group_size);
    if (st != W4A16_OK) return st;
    if (M == 0) {
        if (split_out) *split_out = 1;
        return W4A16_OK;
    }
    if (!X || !W_packed || !scales || !Y) return W4A16_ERR_INVALID_ARG;
    if (!aligned(X, 16) || !aligned(W_packed, 16) || !aligned(scales, 2) || !aligned(Y, 2))
        return W4A16_ERR_INVALID_ARG;
    Plan p;
    st = plan_call(M, N, K, opts, &p);
    if (st != W4A16_OK) return st;
    if (split_out) *split_out = p.split_k;
    if (p.ws_bytes > 0) {
        if (!workspace || workspace_bytes < p.ws_bytes) return W4A16_ERR_WORKSPACE_TOO_SMALL;
        if (!aligned(workspace, 16)) return W4A16_ERR_INVALID_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float *ws = static_cast<float *>(workspace);
    cudaError_t e = launch_decode(p.decode, X, W_packed, scales, Y, ws, M, N, K, s);
    if (e != cudaSuccess) return W4A16_ERR_CUDA;
    if (with_reduce && p.split_k > 1) {
        e = launch_reduce(ws, Y, p.split_k, (long long)M * N, true, s);
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

w4a16_status w4a16_grouped_workspace_bytes(int num_groups, int M_total, int N, int K,
                                           int group_size, size_t *bytes) {
    if (!bytes) return W4A16_ERR_INVALID_ARG;
    w4a16_status st = check_shape(M_total, N, K, group_size);
    if (st != W4A16_OK) return st;
    if (num_groups < 1 || num_groups > 4096) return W4A16_ERR_INVALID_ARG;
    *bytes = 16;
    return W4A16_OK;
}

w4a16_status w4a16_gemm_grouped(const w4a16_bf16 *X, const uint8_t *W_packed,
                                const w4a16_bf16 *scales, const int32_t *M_sizes_dev,
                                w4a16_bf16 *Y, int num_groups, int M_total, int N, int K,
                                int group_size, void *workspace, size_t workspace_bytes,
                                void *stream) {
    w4a16_status st = check_shape(M_total, N, K, group_size);
    if (st != W4A16_OK) return st;
    if (num_groups < 1 || num_groups > 4096) return W4A16_ERR_INVALID_ARG;
    if (!X || !W_packed || !scales || !M_sizes_dev || !Y) return W4A16_ERR_INVALID_ARG;
    if (!aligned(X, 16) || !aligned(W_packed, 16) || !aligned(scales, 2) || !aligned(Y, 2) ||
        !aligned(M_sizes_dev, 4))
        return W4A16_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < 16) return W4A16_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(workspace, 16)) return W4A16_ERR_INVALID_ARG;
    (void)stream;
    return W4A16_ERR_UNSUPPORTED;
}

w4a16_status w4a16_dequant_fp32(const uint8_t *W_packed, const w4a16_bf16 *scales, float *out,
                                int N, int K, int group_size, void *stream) {
    w4a16_status st = check_shape(0, N, K, group_size);
    if (st != W4A16_OK) return st;
    if (!W_packed || !scales || !out) return W4A16_ERR_INVALID_ARG;
    if (!aligned(W_packed, 16) || !aligned(scales, 2) || !aligned(out, 4))
        return W4A16_ERR_INVALID_ARG;
    return from_cuda(launch_dequant(W_packed, scales, out, false, N, K,
                                    static_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_dequant_bf16(const uint8_t *W_packed, const w4a16_bf16 *scales,
                                w4a16_bf16 *out, int N, int K, int group_size, void *stream) {
    w4a16_status st = check_shape(0, N, K, group_size);
    if (st != W4A16_OK) return st;
    if (!W_packed || !scales || !out) return W4A16_ERR_INVALID_ARG;
    if (!aligned(W_packed, 16) || !aligned(scales, 2) || !aligned(out, 2))
        return W4A16_ERR_INVALID_ARG;
    return from_cuda(launch_dequant(W_packed, scales, out, true, N, K,
                                    static_cast<cudaStream_t>(stream)));
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
