// paged_noalloc.cu -- attn_fwd_paged_noalloc: the paged split-KV attention
// forward for callers that cannot allocate device memory.
//
// attn_fwd_paged needs split-KV scratch (per-split partial O and LSE) that
// the caller allocates.  Some callers cannot do that at the point of the
// call: a plugin inside a host engine that owns every device allocation and
// gives plugins no allocator, a serving loop that must not call cudaMalloc
// (it can synchronise the device and take milliseconds), or a runtime that
// reserved its whole memory budget up front.  For them this entry point
// takes the scratch from a fixed array in device memory that lives in this
// library: ATTN_NOALLOC_SCRATCH_BYTES (16 MiB) per GPU, reserved when the
// library's module is loaded on that GPU and held until the process exits.
//
// The array is shared by every call in the process on that GPU.  Nothing in
// it has to start at zero: each call's decode kernel writes every partial
// row the combine of the same call reads.  Two calls whose kernels overlap
// on the GPU (for example on two streams without ordering) race on the array
// and may return wrong results; calls in one stream are ordered and safe.
//
// Set-up: the first call on each device looks up the array's device address
// (cudaGetSymbolAddress) with that device current and remembers it; make
// that first call before any stream capture.  No call allocates or frees
// device memory.
#include "../../include/attn_fwd.h"
#include "common.cuh"
#include "launch.h"

#include <cmath>
#include <cstring>
#include <mutex>

namespace {

constexpr size_t kScratchFloats = ATTN_NOALLOC_SCRATCH_BYTES / sizeof(float);
static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

constexpr int kMaxDev = 64;
float* g_scratch_addr[kMaxDev] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once
// per device with that device current).
attn_status scratch_for_current_device(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    float* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) return ATTN_ERR_CUDA;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status attn_fwd_paged_noalloc(const void* q, const void* k_pool,
                                              const void* v_pool, const int32_t* block_table,
                                              const int32_t* seqlens_k, void* o, float* lse,
                                              int B, int Lq, int Hq, int Hkv, int d,
                                              attn_dtype dtype, int page_size, int num_pages,
                                              int max_pages_per_seq, int num_splits,
                                              const attn_opts* opts, void* stream) {
  if (B < 0 || Lq < 0 || Hq <= 0 || num_splits < 0 || num_splits > 64 ||
      max_pages_per_seq <= 0 || Hkv <= 0)
    return ATTN_ERR_INVALID;
  if (B == 0 || Lq == 0) return ATTN_OK;
  // Chunks of more than 16 query rows per kv head run the prefill kernel,
  // which ignores num_splits and uses no scratch: nothing to check or lower.
  if (Hq % Hkv == 0 && static_cast<int64_t>(Lq) * (Hq / Hkv) > 16)
    return attn_fwd_paged(q, k_pool, v_pool, block_table, seqlens_k, o, lse, B, Lq, Hq, Hkv, d,
                          dtype, page_size, num_pages, max_pages_per_seq, 1, nullptr, nullptr,
                          opts, stream);
  // Split count: an explicit count must fit the scratch; the automatic choice
  // is lowered until it fits (one split needs no scratch at all).
  if (num_splits == 0) {
    num_splits = attn_paged_auto_splits(
        B, Hkv, attn_paged_window_pages(Lq, page_size, max_pages_per_seq, opts));
    while (num_splits > 1 &&
           attn_paged_workspace_bytes(B, Lq, Hq, d, num_splits) > ATTN_NOALLOC_SCRATCH_BYTES)
      --num_splits;
  }
  const size_t need = attn_paged_workspace_bytes(B, Lq, Hq, d, num_splits);
  if (need > ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_INVALID;
  float* o_part = nullptr;
  float* lse_part = nullptr;
  if (num_splits > 1) {
    float* base = nullptr;
    const attn_status st = scratch_for_current_device(&base);
    if (st != ATTN_OK) return st;
    const size_t rows = static_cast<size_t>(B) * Hq * Lq;
    o_part = base;
    lse_part = base + static_cast<size_t>(num_splits) * rows * d;
  }
  return attn_fwd_paged(q, k_pool, v_pool, block_table, seqlens_k, o, lse, B, Lq, Hq, Hkv, d,
                        dtype, page_size, num_pages, max_pages_per_seq, num_splits, o_part,
                        lse_part, opts, stream);
}
