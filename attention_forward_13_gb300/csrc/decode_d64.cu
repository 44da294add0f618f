// decode_d64.cu -- the paged decode kernel's instantiations for head dimension 64.
#define ATTN_DECODE_D 64
#include "decode_kernel.cuh"
