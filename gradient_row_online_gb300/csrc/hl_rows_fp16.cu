// hl_rows_fp16.cu -- resident 16-bit row-kernel instantiations for fp16 logits (one per feature set).
#include "hl_rows16.cuh"

namespace hl {

#define HL_CASE(F) \
    case F: return reinterpret_cast<const void*>(&rows_kernel16<__half, F, false>);

const void* rows_kernel_fp16(int feat) {
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
        default: return nullptr;
    }
}

#undef HL_CASE

}  // namespace hl
