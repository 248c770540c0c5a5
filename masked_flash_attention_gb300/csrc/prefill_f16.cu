// prefill_f16.cu -- the fp16 instantiations of the prefill kernel (the
// kernel source is shared with prefill_sm103.cu; only the element type
// differs: fp16 TMA maps, fp16 MMA operands, fp16 P and output).
#define MFA_PREFILL_F16_UNIT 1
#include "prefill_sm103.cu"
