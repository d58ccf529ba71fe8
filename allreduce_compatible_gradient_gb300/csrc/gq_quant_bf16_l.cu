// gq_quant_bf16_l.cu -- quantise launchers for bf16 gradients, Global-L (one translation unit
// of the library, compiled in parallel with the others).
#include "gq_quant.cuh"

GQH_DEFINE_QUANT(bf16_l, uint16_t, gq::kLinear)
