// decode_g64.cu -- the sliced decode kernel for scale groups of 64 columns
// (2 scale groups per 128-wide block), compiled apart so that the
// instantiations build in parallel with the rest.
#include "decode_slices.cuh"

namespace w4a16 {

cudaError_t launch_decode_sub2(const DecodePlan &p, const uint16_t *X, const uint8_t *Wp,
                               const uint16_t *S, uint16_t *Y, float *ws, bool res, int M, int N,
                               int K, cudaStream_t s) {
    return launch_decode_sub<2>(p, X, Wp, S, nullptr, Y, ws, res, M, N, K, s);
}

}  // namespace w4a16
