// decode_zp.cu -- the sliced decode kernel with zero points (weight =
// scale * (code - z)), for scale groups of 128, 64 and 32 columns, compiled
// apart so that the instantiations build in parallel with the rest.
#include "decode_slices.cuh"

namespace w4a16 {

cudaError_t launch_decode_zp(const DecodePlan &p, const uint16_t *X, const uint8_t *Wp,
                             const uint16_t *S, const uint8_t *Z, uint16_t *Y, float *ws, bool res,
                             int M, int N, int K, cudaStream_t s) {
    switch (p.sub) {
        case 1: return launch_decode_sub<1, true>(p, X, Wp, S, Z, Y, ws, res, M, N, K, s);
        case 2: return launch_decode_sub<2, true>(p, X, Wp, S, Z, Y, ws, res, M, N, K, s);
        case 4: return launch_decode_sub<4, true>(p, X, Wp, S, Z, Y, ws, res, M, N, K, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace w4a16
