// hl_rows_fp32.cu -- row-kernel instantiations for fp32 logits (one per feature set).
#include "hl_rows_kernel.cuh"

namespace hl {

#define HL_CASE(F) \
    case F: return reinterpret_cast<const void*>(&rows_kernel<float, F>);

const void* rows_kernel_fp32(int feat) {
    switch (feat) {
        HL_CASE(0)
        HL_CASE(F_ENT)
        HL_CASE(F_TEACH)
        HL_CASE(F_TEACH | F_ENT)
        HL_CASE(F_TEACH | F_RKL)
        HL_CASE(F_TEACH | F_RKL | F_ENT)
        HL_CASE(F_SOFTCAP)
        HL_CASE(F_SOFTCAP | F_ENT)
        HL_CASE(F_SOFTCAP | F_TEACH)
        HL_CASE(F_SOFTCAP | F_TEACH | F_ENT)
        HL_CASE(F_SOFTCAP | F_TEACH | F_RKL)
        HL_CASE(F_SOFTCAP | F_TEACH | F_RKL | F_ENT)
        HL_CASE(F_DF)
        HL_CASE(F_DF | F_ENT)
        default: return nullptr;
    }
}

#undef HL_CASE

}  // namespace hl
