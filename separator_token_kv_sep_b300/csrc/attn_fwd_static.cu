// sep_attn_fwd_static: the bf16 Sep-Attention forward for callers that
// cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is off limits. Examples are
// an allocator callback or an out-of-memory handler that must not re-enter
// the allocator, a plug-in whose host framework owns every device
// allocation, and a real-time loop that forbids allocation after start-up.
// sep_attn_fwd asks such a caller for a workspace it cannot provide. This
// entry point instead keeps the forward's one scratch buffer (the gathered
// keep-token K and V rows) in a fixed array inside the library.
//
// The array is a file-scope __device__ variable of SEP_STATIC_SCRATCH_BYTES.
// Every GPU that loads this module holds it until the process exits. Host
// code cannot use the array's name as a device address, so the first call
// on each device looks the address up with cudaGetSymbolAddress (with that
// device current), checks the result and caches it. Make that first call
// before any stream capture.
//
// All calls share the array and it keeps the last call's contents. Nothing
// in it needs clearing: the gather kernel rewrites every row the attention
// kernel will read, zeroing the padding rows past the keep count. Calls
// whose work overlaps on the GPU (different streams, or different host
// threads without ordering) race on the array; the caller must order them.
#include <mutex>

#include "common.cuh"
#include "layout.h"

#define SEP_API extern "C" __attribute__((visibility("default")))

namespace sep {

size_t attn_fwd_tc_workspace(const Geom& geo, int d);
int launch_attn_fwd_tc(IndexPtrs idx, const void* q, const void* k, const void* v, void* o,
                       float* lse, const Geom& geo, int d, float scale, uint64_t full_groups,
                       void* ws, int* status, void* stream);

namespace {

static __device__ __align__(256) uint8_t g_fwd_scratch[SEP_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_fwd_scratch on the current device (null on failure).
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fwd_scratch) != cudaSuccess || !p) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace sep

using namespace sep;

SEP_API sep_status sep_attn_fwd_static(const void* index_buf, const void* q, const void* k,
                                       const void* v, void* o, float* lse, int B, int Hq,
                                       int Hkv, int L, int d, float scale, void* stream) {
  if (!index_buf || !q || !k || !v || !o || !lse) return SEP_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || L < 1 || Hq % Hkv != 0) return SEP_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return SEP_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4) || !aligned(index_buf, 256))
    return SEP_ERR_INVALID_ARG;
  // Checked in double first so that huge shapes cannot wrap size_t.
  if ((double)B * Hkv * L * d * 4.0 > (double)SEP_STATIC_SCRATCH_BYTES) return SEP_ERR_TOO_LARGE;
  const Geom geo = make_geom(B, Hq, Hkv, L, L, 0);
  if (attn_fwd_tc_workspace(geo, d) > SEP_STATIC_SCRATCH_BYTES) return SEP_ERR_TOO_LARGE;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf(static_cast<float>(d));
  void* ws = scratch_address();
  int* st = device_status_ptr();
  if (!ws || !st) return SEP_ERR_CUDA;
  const IndexPtrs idx = index_ptrs(const_cast<void*>(index_buf), index_layout(B, L, SEP_BLOCK_M));
  return launch_attn_fwd_tc(idx, q, k, v, o, lse, geo, d, scale, 0, ws, st, stream) == 0
             ? SEP_OK
             : SEP_ERR_CUDA;
}
