// hl_stream_bf16.cu -- streaming 16-bit row-kernel instantiations for bf16 logits
// (one per feature set: base x entropy {none, metric, metric + gradient} x
// teacher {none, KL, KL + teacher entropy, with reverse KL, both}).
#include "hl_stream16.cuh"

namespace hl {

#define HL_CASE(F) \
    case F: return reinterpret_cast<const void*>(&stream_kernel16<__nv_bfloat16, F, false>);
#define HL_TEACH_SET(B) \
    HL_CASE(B) HL_CASE(B | F_TEACH) HL_CASE(B | F_TEACH | F_DCE) HL_CASE(B | F_TEACH | F_RKL) \
    HL_CASE(B | F_TEACH | F_RKL | F_DCE)
#define HL_ENT_SET(C) HL_TEACH_SET(C) HL_TEACH_SET(C | F_ENT) HL_TEACH_SET(C | F_ENT | F_ENTG)
// teacher rows without softcap, with L2 cache hints on the copies
#define HL_L2P_SET(B)                                                                 \
    HL_CASE(B | F_TEACH | F_L2P) HL_CASE(B | F_TEACH | F_DCE | F_L2P)                 \
    HL_CASE(B | F_TEACH | F_RKL | F_L2P) HL_CASE(B | F_TEACH | F_RKL | F_DCE | F_L2P)

const void* stream_kernel_bf16(int feat) {
    switch (feat) {
        HL_ENT_SET(0)
        HL_ENT_SET(F_SOFTCAP)
        HL_L2P_SET(0)
        HL_L2P_SET(F_T2)
        HL_L2P_SET(F_ENT)
        HL_L2P_SET(F_ENT | F_ENTG)
        default: return nullptr;
    }
}

#undef HL_L2P_SET
#undef HL_ENT_SET
#undef HL_TEACH_SET
#undef HL_CASE

}  // namespace hl
