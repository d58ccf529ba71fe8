// gq_quant_bf16_e.cu -- quantise launchers for bf16 gradients, Global-E (one translation unit
// of the library, compiled in parallel with the others).
#include "gq_quant.cuh"

GQH_DEFINE_QUANT(bf16_e, uint16_t, gq::kExp)
