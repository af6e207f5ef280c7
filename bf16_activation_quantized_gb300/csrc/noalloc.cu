// noalloc.cu -- a GEMM entry point for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc on the path that runs the GEMM: a
// framework plugin that is handed only its inputs and outputs while the host
// framework owns the rest of device memory as its own arena, or code that is
// being captured into a CUDA graph, where cudaMalloc is not allowed.  For them
// w4a16_gemm_noalloc keeps the split-K partial sums in a scratch array that is
// part of the library image itself: a file-scope __device__ array of
// kNoAllocScratchBytes bytes, which every GPU that loads the library holds
// until the process exits.
//
// The array's name is only a host-side stand-in in host code, never a device
// address: the device address is fetched once per device with
// cudaGetSymbolAddress, with that device current, and passed to the kernels.
#include <atomic>
#include <cuda_runtime.h>

#include "w4a16.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::atomic<void *> g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device (set-up on the
// first call per device).
w4a16_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return W4A16_ERR_CUDA;
    void *p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return W4A16_ERR_CUDA;
        }
        g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return W4A16_OK;
}

}  // namespace

extern "C" w4a16_status w4a16_gemm_noalloc(const w4a16_bf16 *X, const uint8_t *W_packed,
                                           const w4a16_bf16 *scales, w4a16_bf16 *Y, int M,
                                           int N, int K, int group_size, void *stream) {
    size_t need = 0;
    w4a16_status st = w4a16_workspace_bytes(M, N, K, group_size, &need);
    if (st != W4A16_OK) return st;
    if (need > kNoAllocScratchBytes) return W4A16_ERR_WORKSPACE_TOO_SMALL;
    void *scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != W4A16_OK) return st;
    // The split-K workspace needs no zeroing: every slice element is written
    // before the reduce reads it.
    return w4a16_gemm(X, W_packed, scales, Y, M, N, K, group_size, scratch, kNoAllocScratchBytes,
                      stream);
}
