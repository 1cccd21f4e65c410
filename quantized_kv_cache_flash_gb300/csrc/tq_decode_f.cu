// Decode kernel variants: fp16 K (turbo4-asym, turbo3-asym).
#include "tq_decode_kernel.cuh"

namespace tq {

int decode_variant_f(bool launch, int kb, int vb, int rows, bool table, bool res, const DecodeParams& p,
                     const CUtensorMap* kmap, cudaStream_t stream, cudaEvent_t ev0, cudaEvent_t ev1) {
    TQ_DECODE_VARIANT(0, 4, 8, false, false)
    TQ_DECODE_VARIANT(0, 4, 16, false, false)
    TQ_DECODE_VARIANT(0, 3, 8, false, false)
    TQ_DECODE_VARIANT(0, 3, 16, false, false)
    return launch ? static_cast<int>(cudaErrorInvalidValue) : 0;
}

}  // namespace tq
