// decode_d128.cu -- the paged decode kernel's instantiations for head dimension 128.
#define ATTN_DECODE_D 128
#include "decode_kernel.cuh"
