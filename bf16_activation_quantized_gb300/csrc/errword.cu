// errword.cu -- the library's device-side error word.
//
// Kernels that can detect a broken pipeline (a bounded wait that timed out)
// record it by OR-ing bits into one int in device memory instead of trapping.
// The word is a file-scope __device__ variable; its device address is looked
// up once per device with cudaGetSymbolAddress and passed to the kernels, and
// w4a16_read_error_word copies it back to the host.
#include <atomic>
#include <cuda_runtime.h>

#include "w4a16.h"
#include "internal.h"

namespace w4a16 {

namespace {
__device__ int g_error_word;
std::atomic<int *> g_error_ptr[64];
}  // namespace

int *device_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    int *p = g_error_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        void *q = nullptr;
        if (cudaGetSymbolAddress(&q, g_error_word) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        p = static_cast<int *>(q);
        g_error_ptr[dev].store(p, std::memory_order_release);
    }
    return p;
}

}  // namespace w4a16

extern "C" w4a16_status w4a16_read_error_word(int *out, int clear) {
    if (!out) return W4A16_ERR_INVALID_ARG;
    // Every kernel that may still set a bit has finished once the device is
    // idle; the copies below are synchronous.
    if (cudaDeviceSynchronize() != cudaSuccess) return W4A16_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, w4a16::g_error_word, sizeof v) != cudaSuccess) return W4A16_ERR_CUDA;
    if (clear) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(w4a16::g_error_word, &zero, sizeof zero) != cudaSuccess)
            return W4A16_ERR_CUDA;
    }
    *out = v;
    return W4A16_OK;
}
