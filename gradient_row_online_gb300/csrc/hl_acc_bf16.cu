// hl_acc_bf16.cu -- accumulating instantiations for bf16 logits (the gradient
// is added to grad_out's values): one per base feature set, for the resident
// and the streaming kernel.  The streaming ones carry F_DCE with F_TEACH and
// F_ENTG with F_ENT (each then costs one packed op per element pair when its
// loss or weight is absent, and the results are unchanged).
#include "hl_stream16.cuh"

namespace hl {

#define HL_CASE(F) \
    case F: return reinterpret_cast<const void*>(&rows_kernel16<__nv_bfloat16, F, true>);

const void* rows_kernel_bf16_acc(int feat) {
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

#define HL_CASE(F) \
    case (F) & F_BASE: \
        return reinterpret_cast<const void*>(&stream_kernel16<__nv_bfloat16, F, true>);

const void* stream_kernel_bf16_acc(int feat) {
    switch (feat & F_BASE) {
        HL_CASE(0)
        HL_CASE(F_ENT | F_ENTG)
        HL_CASE(F_TEACH | F_DCE)
        HL_CASE(F_TEACH | F_DCE | F_ENT | F_ENTG)
        HL_CASE(F_TEACH | F_DCE | F_RKL)
        HL_CASE(F_TEACH | F_DCE | F_RKL | F_ENT | F_ENTG)
        HL_CASE(F_SOFTCAP)
        HL_CASE(F_SOFTCAP | F_ENT | F_ENTG)
        HL_CASE(F_SOFTCAP | F_TEACH | F_DCE)
        HL_CASE(F_SOFTCAP | F_TEACH | F_DCE | F_ENT | F_ENTG)
        HL_CASE(F_SOFTCAP | F_TEACH | F_DCE | F_RKL)
        HL_CASE(F_SOFTCAP | F_TEACH | F_DCE | F_RKL | F_ENT | F_ENTG)
        default: return nullptr;
    }
}

#undef HL_CASE

}  // namespace hl
