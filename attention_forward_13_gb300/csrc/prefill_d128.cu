// prefill_d128.cu -- the prefill kernel's instantiations for head dimension 128.
#define ATTN_PREFILL_D 128
#include "prefill_kernel.cuh"
