// gq_quant_f32_e.cu -- quantise launchers for fp32 gradients, Global-E (one translation unit
// of the library, compiled in parallel with the others).
#include "gq_quant.cuh"

GQH_DEFINE_QUANT(f32_e, float, gq::kExp)
