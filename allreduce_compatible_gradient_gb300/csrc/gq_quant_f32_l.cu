// gq_quant_f32_l.cu -- quantise launchers for fp32 gradients, Global-L (one translation unit
// of the library, compiled in parallel with the others).
#include "gq_quant.cuh"

GQH_DEFINE_QUANT(f32_l, float, gq::kLinear)
