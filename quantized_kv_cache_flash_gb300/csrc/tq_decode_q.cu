// Decode kernel variants: quantized K, fp16 codebook (no residual product), and the table records.
#include "tq_decode_kernel.cuh"

namespace tq {

int decode_variant_q(bool launch, int kb, int vb, int rows, bool table, bool res, const DecodeParams& p,
                     const CUtensorMap* kmap, cudaStream_t stream, cudaEvent_t ev0, cudaEvent_t ev1) {
    TQ_DECODE_VARIANT(3, 3, 4, false, false)
    TQ_DECODE_VARIANT(3, 3, 8, false, false)
    TQ_DECODE_VARIANT(3, 3, 16, false, false)
    TQ_DECODE_VARIANT(4, 4, 4, false, false)
    TQ_DECODE_VARIANT(4, 4, 8, false, false)
    TQ_DECODE_VARIANT(4, 4, 16, false, false)
    TQ_DECODE_VARIANT(4, 3, 4, false, false)
    TQ_DECODE_VARIANT(4, 3, 8, false, false)
    TQ_DECODE_VARIANT(4, 3, 16, false, false)
    TQ_DECODE_VARIANT(3, 3, 4, true, false)
    TQ_DECODE_VARIANT(3, 3, 8, true, false)
    TQ_DECODE_VARIANT(3, 3, 16, true, false)
    return launch ? static_cast<int>(cudaErrorInvalidValue) : 0;
}

}  // namespace tq
