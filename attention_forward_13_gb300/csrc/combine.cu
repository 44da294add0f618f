// combine.cu -- LSE-weighted merge of split-KV partials.
//
// The pages give the split layout (FlashAttention-3 hopper/epilogue_fwd.hpp:
// O and LSE carry a num_splits dimension; an empty split stores O = 0 and
// LSE = -inf) but not the merge itself; it follows from the definition of
// the log-sum-exp: with M = max_s LSE_s,
//   LSE = M + ln(sum_s e^{LSE_s - M} [+ e^{sink - M}]),
//   O   = sum_s e^{LSE_s - LSE} O_s.
// One warp per output row; each lane owns D/32 consecutive elements of d
// (float4 loads at d = 128), so every partial row is read with coalesced
// 512-byte requests.  The sink of the query head is added here, once.
#include "common.cuh"
#include "launch.h"

#include <cstdio>
#include <type_traits>

namespace attn {

template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_combine_kernel(const CombineParams p) {
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  constexpr int VPL = D / 32;  // values per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rows = static_cast<int64_t>(p.B) * p.Hq * p.Lq;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + warp;  // [b][h][qi]
  if (r >= rows) return;
  const int qi = static_cast<int>(r % p.Lq);
  const int h = static_cast<int>((r / p.Lq) % p.Hq);
  const int b = static_cast<int>(r / (static_cast<int64_t>(p.Lq) * p.Hq));

  // max over the splits' LSE (and the sink)
  float m = -INFINITY;
  for (int s = lane; s < p.num_splits; s += 32) m = fmaxf(m, p.lse_part[s * rows + r]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float sink_l2 = (p.sink != nullptr) ? p.sink[h] * kLog2e : -INFINITY;
  const float m2 = fmaxf(m * kLog2e, sink_l2);  // log2 units

  float acc[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) acc[i] = 0.0f;
  float z = 0.0f;
  if (m2 != -INFINITY) {
    for (int s = 0; s < p.num_splits; ++s) {
      const float ls = p.lse_part[s * rows + r];
      if (ls == -INFINITY) continue;
      const float wgt = exp2f(ls * kLog2e - m2);
      z += wgt;
      const float* src = p.o_part + (s * rows + r) * D + lane * VPL;
      if constexpr (VPL == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        acc[0] += wgt * v.x;
        acc[1] += wgt * v.y;
        acc[2] += wgt * v.z;
        acc[3] += wgt * v.w;
      } else {
#pragma unroll
        for (int i = 0; i < VPL; ++i) acc[i] += wgt * src[i];
      }
    }
    if (p.sink != nullptr) z += exp2f(sink_l2 - m2);
  }
  const float inv = (z > 0.0f) ? 1.0f / z : 0.0f;
  T* dst = reinterpret_cast<T*>(p.o) + ((static_cast<int64_t>(b) * p.Lq + qi) * p.Hq + h) * D +
           lane * VPL;
#pragma unroll
  for (int i = 0; i < VPL; ++i) dst[i] = T(acc[i] * inv);
  if (lane == 0 && p.lse != nullptr) p.lse[r] = (z > 0.0f) ? (m2 + log2f(z)) * kLn2 : -INFINITY;
}

cudaError_t launch_combine(const CombineParams& p, bool bf16, cudaStream_t stream, char* name,
                           size_t name_len) {
  snprintf(name, name_len, "attn_splitkv_combine_d%d_%s_splits%d", p.d, bf16 ? "bf16" : "f16",
           p.num_splits);
  const int64_t rows = static_cast<int64_t>(p.B) * p.Hq * p.Lq;
  const int64_t grid = (rows + 7) / 8;
  if (grid == 0) return cudaSuccess;
  if (p.d == 128 && bf16) attn_combine_kernel<128, true><<<grid, 256, 0, stream>>>(p);
  else if (p.d == 128) attn_combine_kernel<128, false><<<grid, 256, 0, stream>>>(p);
  else if (p.d == 64 && bf16) attn_combine_kernel<64, true><<<grid, 256, 0, stream>>>(p);
  else if (p.d == 64) attn_combine_kernel<64, false><<<grid, 256, 0, stream>>>(p);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace attn
