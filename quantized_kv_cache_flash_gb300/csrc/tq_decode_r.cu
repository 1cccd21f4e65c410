// Decode kernel variants: quantized K with a codebook that is not all fp16 values (the fp8 centroid residual product).
#include "tq_decode_kernel.cuh"

namespace tq {

int decode_variant_r(bool launch, int kb, int vb, int rows, bool table, bool res, const DecodeParams& p,
                     const CUtensorMap* kmap, cudaStream_t stream, cudaEvent_t ev0, cudaEvent_t ev1) {
    TQ_DECODE_VARIANT(3, 3, 4, false, true)
    TQ_DECODE_VARIANT(3, 3, 8, false, true)
    TQ_DECODE_VARIANT(3, 3, 16, false, true)
    TQ_DECODE_VARIANT(4, 4, 4, false, true)
    TQ_DECODE_VARIANT(4, 4, 8, false, true)
    TQ_DECODE_VARIANT(4, 4, 16, false, true)
    TQ_DECODE_VARIANT(4, 3, 4, false, true)
    TQ_DECODE_VARIANT(4, 3, 8, false, true)
    TQ_DECODE_VARIANT(4, 3, 16, false, true)
    return launch ? static_cast<int>(cudaErrorInvalidValue) : 0;
}

}  // namespace tq
