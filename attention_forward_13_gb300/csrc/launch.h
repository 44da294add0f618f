// launch.h -- host-side launchers of the kernels (one per translation unit),
// called by the C ABI layer in api.cu after validation.
#pragma once
#include <cstddef>
#include <cuda_runtime.h>
#include "common.cuh"

namespace attn {

// grid = number of CTAs; name receives the kernel's trait string.  xf is a
// ScoreXf value.  Dispatches to launch_prefill_d<64 / 128>.
cudaError_t launch_prefill(const PrefillParams& p, int grid, int d, int dt, bool masked,
                           int xf, cudaStream_t stream, char* name, size_t name_len);
// One per head dimension, each in its own translation unit (prefill_d64.cu,
// prefill_d128.cu) so the two compile in parallel.
// dt: PrefillDt (0 fp16, 1 bf16, 2 e4m3).
template <int D>
cudaError_t launch_prefill_d(const PrefillParams& p, int grid, int dt, bool masked, int xf,
                             cudaStream_t stream);

cudaError_t launch_decode(const DecodeParams& p, int d, bool bf16, bool softcap, int rows,
                          cudaStream_t stream, char* name, size_t name_len);
// feat: 0 none, 1 masks, 2 masks + ALiBi.  One per head dimension
// (decode_d64.cu, decode_d128.cu).
template <int D>
cudaError_t launch_decode_d(const DecodeParams& p, bool bf16, bool softcap, int feat,
                            cudaStream_t stream);

cudaError_t launch_combine(const CombineParams& p, bool bf16, cudaStream_t stream, char* name,
                           size_t name_len);

cudaError_t launch_selftest_timeout(unsigned int* err, unsigned long long timeout_ns,
                                    cudaStream_t stream);

}  // namespace attn
