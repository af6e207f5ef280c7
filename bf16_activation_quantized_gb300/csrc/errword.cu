// errword.cu -- the library's device-side error word.
//
// Kernels that can detect a broken pipeline (a bounded wait that timed out)
// record it by OR-ing bits into one int in device memory instead of trapping.
// The word is a file-scope __device__ variable; its device address is looked
// up once per device with cudaGetSymbolAddress and passed to the kernels.
#include <atomic>
#include <cuda_runtime.h>

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
