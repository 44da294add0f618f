// api.cu -- the C ABI declared in include/attn_fwd.h: argument validation,
// TMA descriptor encoding, split selection and kernel dispatch.  No device
// memory is allocated here; every launch is asynchronous on the caller's
// stream.
#include "../../include/attn_fwd.h"
#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

#include <algorithm>
#include <array>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <vector>

using namespace attn;

namespace {

// Device error word: one per device, set by kernels that give up on a wait.
__device__ unsigned int g_attn_err;

constexpr int kMaxDevices = 64;
unsigned int* g_err_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};
std::mutex g_mu;

thread_local char g_last_name[256] = "";

// Default limit of every in-kernel wait: generous for any legal schedule, and
// still a bounded time if a schedule is ever wrong.
constexpr uint64_t kTimeoutNs = 4ull * 1000000000ull;

bool log_enabled() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("ATTN_LOG");
    v = (e != nullptr && e[0] == '1') ? 1 : 0;
  }
  return v == 1;
}

attn_status device_state(unsigned int** err, int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_err_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_attn_err) != cudaSuccess) return ATTN_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    g_err_ptr[dev] = static_cast<unsigned int*>(ptr);
    g_num_sms[dev] = sms;
  }
  if (err) *err = g_err_ptr[dev];
  if (num_sms) *num_sms = g_num_sms[dev];
  return ATTN_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// Tiled map over a tensor whose innermost dimension is contiguous and whose
// other dimensions have the given extents and byte strides, with the given
// box.  dt: attn_dtype of the elements (e4m3 travels as bytes), or kMapF32.
// Loads of Q/K/V use the 128-byte swizzle (one swizzle atom of 64 16-bit
// elements per box row); the O store the swizzle as wide as its box row (128
// or 64 bytes); LSE none.
constexpr int kMapF32 = -1;
bool make_map(CUtensorMap* m, const void* base, int dt, int rank, const uint64_t* dims,
              const uint64_t* strides_bytes, const uint32_t* box,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  memset(m, 0, sizeof(*m));
  cuuint64_t gd[5];
  cuuint64_t gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) gs[i] = strides_bytes[i];
  const CUtensorMapDataType ty = dt == kMapF32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : dt == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                 : dt == ATTN_F16  ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUresult r = fn(m, ty,
                  rank, const_cast<void*>(base), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// Element strides: positive and a whole number of 16-byte units.
bool stride_ok(int64_t s, int eb = 2) { return s > 0 && (s * eb) % 16 == 0; }

float resolve_scale(const attn_opts* o, int d) {
  return (o != nullptr && o->scale > 0.0f) ? o->scale : 1.0f / sqrtf(static_cast<float>(d));
}

// Effective key bounds (negative = unbounded); causal is a right bound of 0.
void resolve_window(const attn_opts* opts, int* wl, int* wr) {
  *wl = -1;
  *wr = -1;
  if (opts == nullptr) return;
  if (opts->use_window) {
    *wl = opts->window_left < 0 ? -1 : opts->window_left;
    *wr = opts->window_right < 0 ? -1 : opts->window_right;
  }
  if (opts->causal) *wr = 0;  // any window_right >= 0 is looser than causal
}

// PackGQA (FlashAttention-3 epilogue, PackGQA row <-> (head, query) mapping):
// the g = Hq / Hkv query heads of a kv head share each 128-row tile, 128 / g
// queries of each, when g is a power of two from 2 to 16 (the tile then
// holds whole queries of every head of the group, and one TMA box loads it).
#ifndef ATTN_PACK_GQA
#define ATTN_PACK_GQA 1
#endif
int pack_of(int Hq, int Hkv) {
  const int g = Hq / Hkv;
  if (!ATTN_PACK_GQA || Hq % Hkv != 0) return 1;
  return (g == 2 || g == 4 || g == 8 || g == 16) ? g : 1;
}
int log2_int(int x) {
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}

// Query blocks (two 128-row tiles of 128 / pack queries each) of L queries
// (no int overflow for any L >= 0).
int m_blocks(int L, int pack = 1) {
  const int64_t per = 256 / pack;
  return static_cast<int>((static_cast<int64_t>(L) + per - 1) / per);
}

// Packing fields of the launch parameters.
void set_pack(PrefillParams& p, int Hq, int Hkv) {
  p.pack = pack_of(Hq, Hkv);
  p.qpt_log2 = log2_int(128 / p.pack);
  p.units = Hq / p.pack;
}

void fill_common(PrefillParams& p, const attn_opts* opts, int d) {
  const float scale = resolve_scale(opts, d);
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  const float cap = (opts != nullptr && opts->softcap > 0.0f) ? opts->softcap : 0.0f;
  p.softcap = cap;
  p.softcap_inv = cap > 0.0f ? 1.0f / cap : 0.0f;
  p.sink = opts != nullptr ? opts->sink : nullptr;
  resolve_window(opts, &p.win_left, &p.win_right);
  p.top_left = (opts != nullptr && opts->top_left) ? 1 : 0;
  p.inv_scale = 1.0f / scale;
  p.o_scale = ((opts != nullptr && opts->scale_p > 0.0f) ? opts->scale_p : 1.0f) *
              ((opts != nullptr && opts->scale_o > 0.0f) ? opts->scale_o : 1.0f);
  p.alibi = opts != nullptr ? opts->alibi_slopes : nullptr;
  p.alibi_stride = opts != nullptr ? opts->alibi_stride : 0;
  p.timeout_ns = kTimeoutNs;
}

// Options every entry point checks: pointer alignment of the per-head
// vectors, and the combinations the pages leave undefined or that are not
// built (soft-cap with ALiBi or bias: the order is not on the pages; ALiBi
// with a bias: the Composable Kernel bias kind is one or the other).
attn_status check_opts(const attn_opts* opts, int Hq, bool allow_bias) {
  if (opts == nullptr) return ATTN_OK;
  if (opts->sink != nullptr && (reinterpret_cast<uintptr_t>(opts->sink) & 3u))
    return ATTN_ERR_INVALID;
  const bool alibi = opts->alibi_slopes != nullptr, bias = opts->bias != nullptr;
  if (alibi && ((reinterpret_cast<uintptr_t>(opts->alibi_slopes) & 3u) ||
                (opts->alibi_stride != 0 && opts->alibi_stride < Hq)))
    return ATTN_ERR_INVALID;
  if (bias && !allow_bias) return ATTN_ERR_UNSUPPORTED;
  if ((alibi || bias) && opts->softcap > 0.0f) return ATTN_ERR_UNSUPPORTED;
  if (alibi && bias) return ATTN_ERR_UNSUPPORTED;
  if (bias) {
    const attn_strides& b = opts->bias_strides;
    if (!aligned16(opts->bias) || b.row < 0 || b.head < 0 || b.batch < 0 || (b.row % 8) ||
        (b.head % 8) || (b.batch % 8))
      return ATTN_ERR_INVALID;
  }
  return ATTN_OK;
}

int score_xf(const PrefillParams& p) {
  if (p.softcap > 0.0f) return kXfSoftcap;
  if (p.alibi != nullptr) return kXfAlibi;
  if (p.bias != nullptr) return kXfBias;
  return kXfNone;
}

}  // namespace

namespace attn {
cudaError_t launch_decode(const DecodeParams& p, int d, bool bf16, bool softcap, int rows,
                          cudaStream_t stream, char* name, size_t name_len) {
  const int feat = p.alibi != nullptr ? 2 : (p.win_left >= 0 || p.win_right >= 0) ? 1 : 0;
  static const char* const kFeat[3] = {"plain", "masked", "alibi"};
  snprintf(name, name_len, "attn_decode_paged_tcgen05_d%d_%s_%s_%s_rows%d_splits%d", d,
           bf16 ? "bf16" : "f16", softcap ? "softcap" : "nocap", kFeat[feat], rows,
           p.num_splits);
  if (d == 64) return launch_decode_d<64>(p, bf16, softcap, feat, stream);
  if (d == 128) return launch_decode_d<128>(p, bf16, softcap, feat, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_prefill(const PrefillParams& p, int grid, int d, int dt, bool masked,
                           int xf, cudaStream_t stream, char* name, size_t name_len) {
  const char* mask = !masked ? "nomask"
                     : (p.win_left < 0 && p.win_right == 0) ? "causal"
                                                            : "window";
  static const char* const kXfName[4] = {"plain", "softcap", "alibi", "bias"};
  snprintf(name, name_len, "attn_prefill_tcgen05_d%d_%s_%s%s_%s_m256n128_persistent", d,
           dt == kDtE4M3 ? "e4m3" : dt == kDtBF16 ? "bf16" : "f16", mask,
           p.top_left ? "_topleft" : "",
           kXfName[(xf >= 0 && xf < 4) ? xf : 0]);
  if (d == 64) return launch_prefill_d<64>(p, grid, dt, masked, xf, stream);
  if (d == 128) return launch_prefill_d<128>(p, grid, dt, masked, xf, stream);
  return cudaErrorInvalidValue;
}
}  // namespace attn

namespace {

attn_status finish_launch(cudaError_t e) {
  if (e != cudaSuccess) {
    if (log_enabled()) fprintf(stderr, "[attn] launch failed: %s\n", cudaGetErrorString(e));
    return ATTN_ERR_CUDA;
  }
  if (log_enabled()) fprintf(stderr, "[attn] launched %s\n", g_last_name);
  return ATTN_OK;
}

__global__ void attn_selftest_timeout_kernel(unsigned int* err, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const Waiter w{globaltimer_ns() + timeout_ns, &abort_flag, err};
  // Nobody ever arrives on `bar`: the bounded wait must give up and return.
  w.wait(&bar, 0, kErrSelftest);
  __syncthreads();
}

}  // namespace

namespace attn {
cudaError_t launch_selftest_timeout(unsigned int* err, unsigned long long timeout_ns,
                                    cudaStream_t stream) {
  attn_selftest_timeout_kernel<<<1, 32, 0, stream>>>(err, timeout_ns);
  return cudaGetLastError();
}
}  // namespace attn

namespace {

// Static schedule for dense masked prefill.  With a causal or window mask the
// query blocks of one (batch, head) cost different numbers of K/V steps, and
// the snake order over the plain item list leaves some CTAs a block more than
// others at the end.  Here the host packs the items onto the grid once per
// shape: longest processing time first (each item to the least loaded CTA),
// then single moves and pairwise swaps off the most loaded CTA while they
// lower the maximum.  Every CTA runs its own list lightest first: measured
// against heaviest first on causal shapes (B4 H16 L2048 932 -> 959 TFLOP/s,
// B8 H16 L1024 597 -> 643, e4m3 L2048 1013 -> 1031).  The order decides
// only which CTA computes an item, never how.
struct Schedule {
  std::vector<uint16_t> off;   // grid + 1 list bounds
  std::vector<uint16_t> item;  // items, CTA by CTA
};

// K/V steps of query block mb (two 128-row tiles) in a dense problem: the
// union of both tiles' key ranges, as the kernel's item decode computes it.
int dense_block_steps(const PrefillParams& p, int mb) {
  constexpr int BN = 128;
  const int qpt = 1 << p.qpt_log2;  // queries per tile
  const int m0 = mb * 2 * qpt;
  const int diag = p.top_left ? 0 : p.Lk - p.Lq;
  int jb = INT_MAX, je = 0;
  for (int t = 0; t < 2; ++t) {
    const int mt = m0 + t * qpt;
    if (mt >= p.Lq) continue;
    const int last = std::min(mt + qpt - 1, p.Lq - 1);
    int kend = p.Lk, kbeg = 0;
    if (p.win_right >= 0) kend = std::min(p.Lk, last + diag + p.win_right + 1);
    if (p.win_left >= 0) kbeg = std::max(0, mt + diag - p.win_left);
    if (kend > kbeg) {
      jb = std::min(jb, kbeg / BN);
      je = std::max(je, (kend + BN - 1) / BN);
    }
  }
  return je > jb ? je - jb : 0;
}

std::shared_ptr<const Schedule> dense_schedule(const PrefillParams& p, int grid) {
  static std::mutex mu;
  static std::map<std::array<int, 9>, std::shared_ptr<const Schedule>> cache;
  const std::array<int, 9> key = {p.B, p.units, p.Lq, p.Lk, p.win_left, p.win_right, p.top_left,
                                  p.qpt_log2, grid};
  {
    std::lock_guard<std::mutex> lock(mu);
    const auto f = cache.find(key);
    if (f != cache.end()) return f->second;
  }
  const int n = p.num_items, nbh = p.B * p.units;
  // Cost in tenths of a K/V step: the steps plus a fixed per-item share of
  // four steps (the Q load and first S before any PV, the last PV and the
  // epilogue); of the shares 0, 1.6, 4 and 8 steps, 4 gave the shortest
  // measured runs over causal and windowed shapes with L 1024 to 8192.
  std::vector<int> cost(n);
  for (int i = 0; i < n; ++i) {
    const int mb = p.num_m_blocks - 1 - i / nbh;  // the kernel's masked item order
    cost[i] = 10 * dense_block_steps(p, mb) + 40;
  }
  std::vector<int> order(n);
  for (int i = 0; i < n; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return cost[a] > cost[b]; });
  std::vector<std::vector<int>> bins(grid);
  std::vector<long> load(grid, 0);
  for (const int i : order) {
    const int c = static_cast<int>(std::min_element(load.begin(), load.end()) - load.begin());
    bins[c].push_back(i);
    load[c] += cost[i];
  }
  for (int iter = 0; iter < 8 * grid; ++iter) {
    const int hi = static_cast<int>(std::max_element(load.begin(), load.end()) - load.begin());
    const long top = load[hi];
    bool moved = false;
    for (size_t a = 0; a < bins[hi].size() && !moved; ++a) {
      const int ia = bins[hi][a];
      for (int c = 0; c < grid && !moved; ++c) {
        if (c == hi) continue;
        if (load[c] + cost[ia] < top) {  // a move
          bins[c].push_back(ia);
          bins[hi].erase(bins[hi].begin() + a);
          load[c] += cost[ia];
          load[hi] -= cost[ia];
          moved = true;
          break;
        }
        for (size_t b = 0; b < bins[c].size(); ++b) {  // a swap of a heavier for a lighter item
          const int ib = bins[c][b];
          const int dlt = cost[ia] - cost[ib];
          if (dlt > 0 && load[c] + dlt < top) {
            std::swap(bins[hi][a], bins[c][b]);
            load[c] += dlt;
            load[hi] -= dlt;
            moved = true;
            break;
          }
        }
      }
    }
    if (!moved) break;
  }
  auto s = std::make_shared<Schedule>();
  s->off.assign(grid + 1, 0);
  std::vector<int> seen(n, 0);
  for (int c = 0; c < grid; ++c) {
    std::stable_sort(bins[c].begin(), bins[c].end(), [&](int a, int b) {
      return cost[a] != cost[b] ? cost[a] < cost[b] : a < b;
    });
    for (const int i : bins[c]) {
      s->item.push_back(static_cast<uint16_t>(i));
      ++seen[i];
    }
    s->off[c + 1] = static_cast<uint16_t>(s->item.size());
  }
  for (int i = 0; i < n; ++i)
    if (seen[i] != 1) return nullptr;  // never launch a schedule that drops or repeats an item
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() >= 64) cache.clear();
  cache[key] = s;
  return s;
}

// Whether a dense problem runs on the static schedule: a causal or window
// mask, within the bounds the launch parameters carry, and more work items
// than CTAs (else every CTA has at most one item and the order is moot).
bool schedule_applies(const PrefillParams& p, int grid) {
  const bool masked = p.win_left >= 0 || p.win_right >= 0;
  return masked && grid > 0 && grid <= kSchedMaxCtas && p.num_items <= kSchedMaxItems &&
         p.num_items > grid;
}

// Attaches the static schedule to p when it applies; the kernel otherwise
// keeps the snake order (sched_n = 0).
void attach_schedule(PrefillParams& p, int grid) {
  p.sched_n = 0;
  if (!schedule_applies(p, grid)) return;
  const auto s = dense_schedule(p, grid);
  if (s == nullptr) return;
  std::copy(s->off.begin(), s->off.end(), p.sched_off);
  std::copy(s->item.begin(), s->item.end(), p.sched_item);
  p.sched_n = p.num_items;
}

}  // namespace

extern "C" {

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "kernel wait timed out";
  }
  return "unknown status";
}

const char* attn_last_kernel_name(void) { return g_last_name; }

attn_status attn_device_error(unsigned int* bits) {
  unsigned int* err = nullptr;
  attn_status st = device_state(&err, nullptr);
  if (st != ATTN_OK) return st;
  unsigned int h = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
  if (cudaMemcpy(&h, err, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (h != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpy(err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  if (bits) *bits = h;
  return h ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

attn_status attn_selftest_timeout(uint64_t timeout_ns, void* stream) {
  unsigned int* err = nullptr;
  attn_status st = device_state(&err, nullptr);
  if (st != ATTN_OK) return st;
  if (timeout_ns == 0 || timeout_ns > 10ull * 1000000000ull) return ATTN_ERR_INVALID;
  snprintf(g_last_name, sizeof(g_last_name), "attn_selftest_timeout");
  return finish_launch(
      launch_selftest_timeout(err, timeout_ns, static_cast<cudaStream_t>(stream)));
}

attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int Hq, int Hkv, int Lq, int Lk, int d, attn_dtype dtype, attn_strides sq,
                     attn_strides sk, attn_strides sv, attn_strides so, const attn_opts* opts,
                     void* stream) {
  if (B < 0 || Lq < 0 || Lk < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16 && dtype != ATTN_E4M3) return ATTN_ERR_INVALID;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (dtype == ATTN_E4M3 && (d != 128 || (opts != nullptr &&
                                           (opts->softcap > 0.0f || opts->alibi_slopes != nullptr ||
                                            opts->bias != nullptr))))
    return ATTN_ERR_UNSUPPORTED;
  const int eb = dtype == ATTN_E4M3 ? 1 : 2;  // bytes per element
  if (B == 0 || Lq == 0) return ATTN_OK;
  // With Lk = 0 nothing of K/V is read and they may be NULL.
  if (q == nullptr || o == nullptr || (Lk > 0 && (k == nullptr || v == nullptr)))
    return ATTN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return ATTN_ERR_INVALID;
  for (const attn_strides* s : {&sq, &sk, &sv, &so})
    if (!stride_ok(s->row, eb) || !stride_ok(s->head, eb) || !stride_ok(s->batch, eb))
      return ATTN_ERR_INVALID;
  {
    const attn_status so_ = check_opts(opts, Hq, true);
    if (so_ != ATTN_OK) return so_;
  }
  if (static_cast<int64_t>(B) * (Hq / pack_of(Hq, Hkv)) * m_blocks(Lq, pack_of(Hq, Hkv)) >
      0x7fffffffLL)
    return ATTN_ERR_UNSUPPORTED;

  PrefillParams p;
  memset(&p, 0, sizeof(p));
  unsigned int* err = nullptr;
  int num_sms = 0;
  if (device_state(&err, &num_sms) != ATTN_OK) return ATTN_ERR_CUDA;
  const int dt = dtype == ATTN_E4M3 ? kDtE4M3 : dtype == ATTN_BF16 ? kDtBF16 : kDtF16;
  set_pack(p, Hq, Hkv);
  const uint32_t box[4] = {(uint32_t)(128 / eb), 128, 1, 1};
  {
    const uint32_t qbox[4] = {(uint32_t)(128 / eb), (uint32_t)(128 / p.pack), (uint32_t)p.pack, 1};
    const uint64_t dims[4] = {(uint64_t)d, (uint64_t)Lq, (uint64_t)Hq, (uint64_t)B};
    const uint64_t st[3] = {(uint64_t)sq.row * eb, (uint64_t)sq.head * eb, (uint64_t)sq.batch * eb};
    if (!make_map(&p.tm_q, q, dtype, 4, dims, st, qbox)) return ATTN_ERR_INVALID;
  }
  if (Lk > 0) {  // Lk = 0: no key tile is ever loaded, the maps stay unused
    {
      const uint64_t dims[4] = {(uint64_t)d, (uint64_t)Lk, (uint64_t)Hkv, (uint64_t)B};
      const uint64_t st[3] = {(uint64_t)sk.row * eb, (uint64_t)sk.head * eb,
                              (uint64_t)sk.batch * eb};
      if (!make_map(&p.tm_k, k, dtype, 4, dims, st, box)) return ATTN_ERR_INVALID;
    }
    {
      const uint64_t dims[4] = {(uint64_t)d, (uint64_t)Lk, (uint64_t)Hkv, (uint64_t)B};
      const uint64_t st[3] = {(uint64_t)sv.row * eb, (uint64_t)sv.head * eb,
                              (uint64_t)sv.batch * eb};
      if (!make_map(&p.tm_v, v, dtype, 4, dims, st, box)) return ATTN_ERR_INVALID;
    }
  }
  p.o = o;
  p.lse = lse;
  p.o_row = so.row;
  p.o_head = so.head;
  p.o_batch = so.batch;
  p.lse_head = Lq;
  p.lse_batch = static_cast<int64_t>(Hq) * Lq;
  p.cu_q = p.cu_k = nullptr;
  // TMA store of O and LSE (FlashAttention-3 epilogue store, the non-varlen
  // path): each softmax warp owns 32 consecutive queries of one head when at
  // most 4 heads share a tile.  LSE by TMA needs a 16-byte aligned base and
  // rows of a multiple of 4 floats; otherwise each thread stores its own.
  if (p.pack <= 4) {
    const int rb = prefill_o_round_bytes(dt == kDtE4M3, p.pack);  // bytes per row and store
    const uint32_t obox[4] = {(uint32_t)(rb / eb), 32, 1, 1};
    const uint64_t dims[4] = {(uint64_t)d, (uint64_t)Lq, (uint64_t)Hq, (uint64_t)B};
    const uint64_t st[3] = {(uint64_t)so.row * eb, (uint64_t)so.head * eb, (uint64_t)so.batch * eb};
    p.o_tma = make_map(&p.tm_o, o, dtype, 4, dims, st, obox,
                       rb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B) ? rb : 0;
    if (lse != nullptr && aligned16(lse) && Lq % 4 == 0) {
      const uint32_t lbox[3] = {32, 1, 1};
      const uint64_t ldims[3] = {(uint64_t)Lq, (uint64_t)Hq, (uint64_t)B};
      const uint64_t lst[2] = {(uint64_t)Lq * 4, (uint64_t)Hq * Lq * 4};
      p.lse_tma =
          make_map(&p.tm_lse, lse, kMapF32, 3, ldims, lst, lbox, CU_TENSOR_MAP_SWIZZLE_NONE) ? 1 : 0;
    }
  }
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Lq = Lq;
  p.Lk = Lk;
  p.num_m_blocks = m_blocks(Lq, p.pack);
  p.err = err;
  fill_common(p, opts, d);
  if (opts != nullptr && opts->bias != nullptr) {
    p.bias = opts->bias;
    p.bias_row = opts->bias_strides.row;
    p.bias_head = opts->bias_strides.head;
    p.bias_batch = opts->bias_strides.batch;
  }
  const bool masked = p.win_left >= 0 || p.win_right >= 0;
  p.num_items = p.num_m_blocks * B * p.units;
  const int grid = p.num_items < num_sms ? p.num_items : num_sms;  // persistent: one CTA per SM
  attach_schedule(p, grid);
  return finish_launch(launch_prefill(p, grid, d, dt, masked, score_xf(p),
                                      static_cast<cudaStream_t>(stream), g_last_name,
                                      sizeof(g_last_name)));
}

attn_status attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int B,
                            int total_q, int total_k, int max_seqlen_q, int Hq, int Hkv, int d,
                            attn_dtype dtype, attn_strides sq, attn_strides sk, attn_strides sv,
                            attn_strides so, const attn_opts* opts, void* stream) {
  if (B < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || Hq <= 0 || Hkv <= 0 ||
      Hq % Hkv != 0)
    return ATTN_ERR_INVALID;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16 && dtype != ATTN_E4M3) return ATTN_ERR_INVALID;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (dtype == ATTN_E4M3 && (d != 128 || (opts != nullptr &&
                                           (opts->softcap > 0.0f || opts->alibi_slopes != nullptr ||
                                            opts->bias != nullptr))))
    return ATTN_ERR_UNSUPPORTED;
  const int eb = dtype == ATTN_E4M3 ? 1 : 2;  // bytes per element
  if (B == 0 || total_q == 0 || max_seqlen_q == 0) return ATTN_OK;
  if (q == nullptr || o == nullptr || cu_seqlens_q == nullptr || cu_seqlens_k == nullptr ||
      (total_k > 0 && (k == nullptr || v == nullptr)))
    return ATTN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return ATTN_ERR_INVALID;
  for (const attn_strides* s : {&sq, &sk, &sv, &so})
    if (!stride_ok(s->row, eb) || !stride_ok(s->head, eb)) return ATTN_ERR_INVALID;
  if (static_cast<int64_t>(B) * (Hq / pack_of(Hq, Hkv)) *
          m_blocks(max_seqlen_q, pack_of(Hq, Hkv)) > 0x7fffffffLL)
    return ATTN_ERR_UNSUPPORTED;
  {
    const attn_status so_ = check_opts(opts, Hq, false);
    if (so_ != ATTN_OK) return so_;
  }

  PrefillParams p;
  memset(&p, 0, sizeof(p));
  unsigned int* err = nullptr;
  int num_sms = 0;
  if (device_state(&err, &num_sms) != ATTN_OK) return ATTN_ERR_CUDA;
  const int dt = dtype == ATTN_E4M3 ? kDtE4M3 : dtype == ATTN_BF16 ? kDtBF16 : kDtF16;
  set_pack(p, Hq, Hkv);
  const uint32_t box[4] = {(uint32_t)(128 / eb), 128, 1, 1};
  {
    const uint32_t qbox[4] = {(uint32_t)(128 / eb), (uint32_t)(128 / p.pack), (uint32_t)p.pack, 1};
    const uint64_t dims[4] = {(uint64_t)d, (uint64_t)total_q, (uint64_t)Hq, 1};
    const uint64_t st[3] = {(uint64_t)sq.row * eb, (uint64_t)sq.head * eb,
                            (uint64_t)sq.row * eb * (uint64_t)total_q};
    if (!make_map(&p.tm_q, q, dtype, 4, dims, st, qbox)) return ATTN_ERR_INVALID;
  }
  if (total_k > 0) {  // no keys at all: the maps stay unused
    const int tk = total_k;
    {
      const uint64_t dims[4] = {(uint64_t)d, (uint64_t)tk, (uint64_t)Hkv, 1};
      const uint64_t st[3] = {(uint64_t)sk.row * eb, (uint64_t)sk.head * eb,
                              (uint64_t)sk.row * eb * (uint64_t)tk};
      if (!make_map(&p.tm_k, k, dtype, 4, dims, st, box)) return ATTN_ERR_INVALID;
    }
    {
      const uint64_t dims[4] = {(uint64_t)d, (uint64_t)tk, (uint64_t)Hkv, 1};
      const uint64_t st[3] = {(uint64_t)sv.row * eb, (uint64_t)sv.head * eb,
                              (uint64_t)sv.row * eb * (uint64_t)tk};
      if (!make_map(&p.tm_v, v, dtype, 4, dims, st, box)) return ATTN_ERR_INVALID;
    }
  }
  p.o = o;
  p.lse = lse;
  p.o_row = so.row;
  p.o_head = so.head;
  p.o_batch = 0;
  p.lse_head = total_q;
  p.lse_batch = 0;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.total_q = total_q;
  p.total_k = total_k;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Lq = 0;
  p.Lk = 0;
  p.num_m_blocks = m_blocks(max_seqlen_q, p.pack);
  p.err = err;
  fill_common(p, opts, d);
  const bool masked = p.win_left >= 0 || p.win_right >= 0;
  p.num_items = p.num_m_blocks * B * p.units;
  const int grid = p.num_items < num_sms ? p.num_items : num_sms;  // persistent: one CTA per SM
  return finish_launch(launch_prefill(p, grid, d, dt, masked, score_xf(p),
                                      static_cast<cudaStream_t>(stream), g_last_name,
                                      sizeof(g_last_name)));
}

}  // extern "C"

namespace {
// Chunked prefill over a paged KV cache (Lq * g > 16): the prefill kernel with
// its K/V tiles gathered page by page (Composable Kernel paged-KV kernel,
// page block navigator with a query tile per CTA).  q/o [B][Lq][Hq][d],
// lse [B][Hq][Lq]; no split-KV (the query rows give the parallelism).
attn_status paged_prefill(const void* q, const void* k_pool, const void* v_pool,
                          const int32_t* block_table, const int32_t* seqlens_k, void* o,
                          float* lse, int B, int Lq, int Hq, int Hkv, int d, bool bf16,
                          int page_size, int num_pages, int max_pages, const attn_opts* opts,
                          cudaStream_t stream) {
  if (static_cast<int64_t>(B) * (Hq / pack_of(Hq, Hkv)) * m_blocks(Lq, pack_of(Hq, Hkv)) >
      0x7fffffffLL)
    return ATTN_ERR_UNSUPPORTED;
  PrefillParams p;
  memset(&p, 0, sizeof(p));
  unsigned int* err = nullptr;
  int num_sms = 0;
  if (device_state(&err, &num_sms) != ATTN_OK) return ATTN_ERR_CUDA;
  set_pack(p, Hq, Hkv);
  {
    const uint32_t box[4] = {64, (uint32_t)(128 / p.pack), (uint32_t)p.pack, 1};
    const uint64_t dims[4] = {(uint64_t)d, (uint64_t)Lq, (uint64_t)Hq, (uint64_t)B};
    const uint64_t st[3] = {(uint64_t)Hq * d * 2, (uint64_t)d * 2, (uint64_t)Lq * Hq * d * 2};
    if (!make_map(&p.tm_q, q, bf16 ? ATTN_BF16 : ATTN_F16, 4, dims, st, box)) return ATTN_ERR_INVALID;
  }
  {
    const uint32_t boxr[3] = {64, 1, (uint32_t)(page_size < 128 ? page_size : 128)};
    const uint64_t dims[3] = {(uint64_t)d, (uint64_t)Hkv, (uint64_t)num_pages * page_size};
    const uint64_t st[2] = {(uint64_t)d * 2, (uint64_t)Hkv * d * 2};
    if (!make_map(&p.tm_k, k_pool, bf16 ? ATTN_BF16 : ATTN_F16, 3, dims, st, boxr)) return ATTN_ERR_INVALID;
    if (!make_map(&p.tm_v, v_pool, bf16 ? ATTN_BF16 : ATTN_F16, 3, dims, st, boxr)) return ATTN_ERR_INVALID;
  }
  p.o = o;
  p.lse = lse;
  p.o_row = static_cast<int64_t>(Hq) * d;
  p.o_head = d;
  p.o_batch = static_cast<int64_t>(Lq) * Hq * d;
  p.lse_head = Lq;
  p.lse_batch = static_cast<int64_t>(Hq) * Lq;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Lq = Lq;
  p.Lk = max_pages * page_size;
  p.num_m_blocks = m_blocks(Lq, p.pack);
  p.err = err;
  fill_common(p, opts, d);
  p.block_table = block_table;
  p.seqlens_k = seqlens_k;
  p.page_size = page_size;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  const bool masked = p.win_left >= 0 || p.win_right >= 0;
  p.num_items = p.num_m_blocks * B * p.units;
  const int grid = p.num_items < num_sms ? p.num_items : num_sms;
  return finish_launch(launch_prefill(p, grid, d, bf16 ? kDtBF16 : kDtF16, masked, score_xf(p), stream, g_last_name,
                                      sizeof(g_last_name)));
}
}  // namespace

extern "C" {

size_t attn_paged_workspace_bytes(int B, int Lq, int Hq, int d, int num_splits) {
  if (B <= 0 || Lq <= 0 || Hq <= 0 || d <= 0 || num_splits <= 1) return 0;
  const size_t rows = static_cast<size_t>(B) * Hq * Lq;
  return static_cast<size_t>(num_splits) * rows * (static_cast<size_t>(d) + 1) * sizeof(float);
}

attn_status attn_dense_schedule(int B, int Hq, int Hkv, int Lq, int Lk, const attn_opts* opts,
                                int grid, int32_t* off, int32_t* item) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Lq <= 0 || Lk < 0 || grid <= 0 ||
      off == nullptr || item == nullptr)
    return ATTN_ERR_INVALID;
  PrefillParams p;
  memset(&p, 0, sizeof(p));
  set_pack(p, Hq, Hkv);
  const int64_t n = static_cast<int64_t>(m_blocks(Lq, p.pack)) * B * p.units;
  if (n > kSchedMaxItems) return ATTN_ERR_UNSUPPORTED;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Lq = Lq;
  p.Lk = Lk;
  resolve_window(opts, &p.win_left, &p.win_right);
  p.top_left = (opts != nullptr && opts->top_left) ? 1 : 0;
  p.num_m_blocks = m_blocks(Lq, p.pack);
  p.num_items = static_cast<int>(n);
  if (!schedule_applies(p, grid)) return ATTN_ERR_UNSUPPORTED;
  const auto s = dense_schedule(p, grid);
  if (s == nullptr) return ATTN_ERR_INVALID;
  for (int c = 0; c <= grid; ++c) off[c] = s->off[c];
  for (int i = 0; i < p.num_items; ++i) item[i] = s->item[i];
  return ATTN_OK;
}

int attn_paged_window_pages(int Lq, int page_size, int max_pages_per_seq, const attn_opts* opts) {
  int wl = -1, wr = -1;
  resolve_window(opts, &wl, &wr);
  // Top-left bands start at key 0: no saving is claimed for them.
  if (wl < 0 || Lq < 0 || page_size <= 0 || max_pages_per_seq <= 0 ||
      (opts != nullptr && opts->top_left))
    return max_pages_per_seq;
  const int64_t w = (static_cast<int64_t>(Lq) + wl + page_size - 1) / page_size + 1;
  return w < max_pages_per_seq ? static_cast<int>(w) : max_pages_per_seq;
}

int attn_paged_auto_splits(int B, int Hkv, int max_pages_per_seq) {
  int sms = 148;
  device_state(nullptr, &sms);
  if (B <= 0 || Hkv <= 0 || max_pages_per_seq <= 0) return 1;
  // Aim for about two resident CTAs per SM worth of (sequence, kv head, split)
  // work items and at most 32 pages per split (the longest CTA bounds the
  // tail), but never fewer than ~8 pages (512 keys at page 64) per split:
  // every CTA pays a fixed start-up cost (measured on the decode workload:
  // 4 splits best, 12 or more clearly worse).
  const int64_t pairs = static_cast<int64_t>(B) * Hkv;
  int64_t want = (4LL * sms + pairs - 1) / pairs;
  const int64_t by_len = (max_pages_per_seq + 31) / 32;
  if (want < by_len) want = by_len;
  const int64_t max_useful = (max_pages_per_seq + 7) / 8;
  if (want > max_useful) want = max_useful;
  if (want < 1) want = 1;
  if (want > 64) want = 64;
  return static_cast<int>(want);
}

attn_status attn_splitkv_combine(const float* o_partial, const float* lse_partial,
                                 int num_splits, int B, int Hq, int Lq, int d,
                                 const float* sink, void* o, attn_dtype dtype, float* lse,
                                 void* stream) {
  if (num_splits < 1 || num_splits > 64 || B < 0 || Hq <= 0 || Lq < 0) return ATTN_ERR_INVALID;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || Lq == 0) return ATTN_OK;
  if (o_partial == nullptr || lse_partial == nullptr || o == nullptr) return ATTN_ERR_INVALID;
  if (!aligned16(o_partial) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse_partial) & 3u) ||
      (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return ATTN_ERR_INVALID;
  CombineParams c;
  c.o_part = o_partial;
  c.lse_part = lse_partial;
  c.sink = sink;
  c.o = o;
  c.lse = lse;
  c.num_splits = num_splits;
  c.B = B;
  c.Hq = Hq;
  c.Lq = Lq;
  c.d = d;
  return finish_launch(launch_combine(c, dtype == ATTN_BF16, static_cast<cudaStream_t>(stream),
                                      g_last_name, sizeof(g_last_name)));
}

attn_status attn_fwd_paged(const void* q, const void* k_pool, const void* v_pool,
                           const int32_t* block_table, const int32_t* seqlens_k, void* o,
                           float* lse, int B, int Lq, int Hq, int Hkv, int d, attn_dtype dtype,
                           int page_size, int num_pages, int max_pages_per_seq, int num_splits,
                           float* o_partial, float* lse_partial, const attn_opts* opts,
                           void* stream) {
  if (B < 0 || Lq < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || num_pages <= 0 ||
      max_pages_per_seq <= 0 || num_splits < 0 || num_splits > 64)
    return ATTN_ERR_INVALID;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128 &&
      page_size != 256)
    return ATTN_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(num_pages) * page_size > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || Lq == 0) return ATTN_OK;
  if (q == nullptr || k_pool == nullptr || v_pool == nullptr || block_table == nullptr ||
      seqlens_k == nullptr || o == nullptr)
    return ATTN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(o) ||
      (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return ATTN_ERR_INVALID;
  if (B > 65535 || Hkv > 65535) return ATTN_ERR_UNSUPPORTED;
  {
    const attn_status so_ = check_opts(opts, Hq, false);
    if (so_ != ATTN_OK) return so_;
  }
  if (static_cast<int64_t>(Lq) * (Hq / Hkv) > 16)  // a chunk of queries: prefill kernel
    return paged_prefill(q, k_pool, v_pool, block_table, seqlens_k, o, lse, B, Lq, Hq, Hkv, d,
                         dtype == ATTN_BF16, page_size, num_pages, max_pages_per_seq, opts,
                         static_cast<cudaStream_t>(stream));
  const int win_pages = attn_paged_window_pages(Lq, page_size, max_pages_per_seq, opts);
  if (num_splits == 0) num_splits = attn_paged_auto_splits(B, Hkv, win_pages);
  if (num_splits > 1 && (o_partial == nullptr || lse_partial == nullptr ||
                         !aligned16(o_partial) || (reinterpret_cast<uintptr_t>(lse_partial) & 3u)))
    return ATTN_ERR_INVALID;

  DecodeParams p;
  memset(&p, 0, sizeof(p));
  unsigned int* err = nullptr;
  if (device_state(&err, nullptr) != ATTN_OK) return ATTN_ERR_CUDA;
  const bool bf16 = dtype == ATTN_BF16;
  const uint32_t box[3] = {64, (uint32_t)(page_size < 128 ? page_size : 128), 1};
  const uint32_t boxr[3] = {64, 1, box[1]};
  (void)box;
  const uint64_t dims[3] = {(uint64_t)d, (uint64_t)Hkv, (uint64_t)num_pages * page_size};
  const uint64_t st[2] = {(uint64_t)d * 2, (uint64_t)Hkv * d * 2};
  if (!make_map(&p.tm_k, k_pool, bf16 ? ATTN_BF16 : ATTN_F16, 3, dims, st, boxr)) return ATTN_ERR_INVALID;
  if (!make_map(&p.tm_v, v_pool, bf16 ? ATTN_BF16 : ATTN_F16, 3, dims, st, boxr)) return ATTN_ERR_INVALID;
  p.q = q;
  p.block_table = block_table;
  p.seqlens_k = seqlens_k;
  p.o = o;
  p.lse = lse;
  p.o_part = o_partial;
  p.lse_part = o_partial != nullptr && num_splits > 1 ? lse_partial : nullptr;
  p.sink = opts != nullptr ? opts->sink : nullptr;
  p.B = B;
  p.Lq = Lq;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.page_size = page_size;
  p.num_pages = num_pages;
  p.max_pages = max_pages_per_seq;
  p.num_splits = num_splits;
  p.chunk_pages = (win_pages + num_splits - 1) / num_splits;
  const float scale = resolve_scale(opts, d);
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.softcap = (opts != nullptr && opts->softcap > 0.0f) ? opts->softcap : 0.0f;
  p.softcap_inv = p.softcap > 0.0f ? 1.0f / p.softcap : 0.0f;
  resolve_window(opts, &p.win_left, &p.win_right);
  p.top_left = (opts != nullptr && opts->top_left) ? 1 : 0;
  p.alibi = opts != nullptr ? opts->alibi_slopes : nullptr;
  p.alibi_stride = opts != nullptr ? opts->alibi_stride : 0;
  p.err = err;
  p.timeout_ns = kTimeoutNs;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  attn_status st1 = finish_launch(launch_decode(p, d, bf16, p.softcap > 0.0f, Lq * (Hq / Hkv), s,
                                                g_last_name, sizeof(g_last_name)));
  if (st1 != ATTN_OK || num_splits == 1) return st1;
  char decode_name[sizeof(g_last_name)];
  memcpy(decode_name, g_last_name, sizeof(decode_name));
  const attn_status st2 = attn_splitkv_combine(o_partial, p.lse_part, num_splits, B, Hq, Lq, d,
                                               p.sink, o, dtype, lse, stream);
  if (st2 == ATTN_OK) {  // both kernels of the call, in launch order
    char both[sizeof(g_last_name)];
    snprintf(both, sizeof(both), "%s+%s", decode_name, g_last_name);
    memcpy(g_last_name, both, sizeof(both));
  }
  return st2;
}

}  // extern "C"
