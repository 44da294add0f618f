// prefill_d64.cu -- the prefill kernel's instantiations for head dimension 64.
#define ATTN_PREFILL_D 64
#include "prefill_kernel.cuh"
