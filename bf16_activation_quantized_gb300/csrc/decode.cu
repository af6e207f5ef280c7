// decode.cu -- decode-arm launchers and the split-K reduce.  The sliced decode
// kernel is in decode_slices.cuh; its instantiations for 64- and 32-wide scale
// groups live in decode_g64.cu and decode_g32.cu, and its zero-point
// instantiations in decode_zp.cu, so that they compile in parallel.  The
// whole-K decode kernel is in decode_rows.cu.
#include <atomic>

#include "decode_slices.cuh"

namespace w4a16 {

namespace {

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
