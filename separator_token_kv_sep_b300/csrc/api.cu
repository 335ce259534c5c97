// C ABI of the library (declared in include/sepattn.h): host-side argument
// checks, buffer layouts and kernel launches.  No call here allocates device
// memory.
#include <math.h>
#include <string.h>

#include <atomic>

#include "common.cuh"
#include "layout.h"

#define SEP_API extern "C" __attribute__((visibility("default")))

namespace sep {

// The device status word (one per device context); kernels record the first
// error they meet here.
__device__ int g_device_status;

size_t attn_fwd_tc_workspace(const Geom& geo, int d);
int launch_attn_fwd_tc(IndexPtrs idx, const void* q, const void* k, const void* v, void* o,
                       float* lse, const Geom& geo, int d, float scale, uint64_t full_groups,
                       void* ws, int* status, void* stream);
size_t attn_bwd_tc_workspace(const Geom& geo, int d);
int launch_attn_bwd_tc(IndexPtrs idx, const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dout, void* dq, void* dk, void* dv,
                       const Geom& geo, int d, float scale, uint64_t full_groups, void* ws,
                       int* status, void* stream);

namespace {
thread_local void* t_prof_events[SEP_MAX_PROFILE_EVENTS] = {nullptr};
thread_local int t_prof_n = 0;
}  // namespace

void profile_mark(int i, void* stream) {
  if (i < 0 || i >= t_prof_n || !t_prof_events[i]) return;
  // External records become event nodes when the stream is being captured
  // into a CUDA graph; outside a capture they are ordinary records.
  cudaEventRecordWithFlags(static_cast<cudaEvent_t>(t_prof_events[i]),
                           static_cast<cudaStream_t>(stream), cudaEventRecordExternal);
}

int* device_status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) return nullptr;
  // per-device cache; host threads may race on the first lookup, so the
  // entries are atomic (a lost race repeats the same lookup)
  static std::atomic<int*> cache[64];
  int* p = cache[dev].load(std::memory_order_acquire);
  if (!p) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_device_status) != cudaSuccess || !a) return nullptr;
    p = static_cast<int*>(a);
    cache[dev].store(p, std::memory_order_release);
  }
  return p;
}

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

sep_status from_cuda(int e) { return e == 0 ? SEP_OK : SEP_ERR_CUDA; }

bool fill_sep_ids(const int32_t* sep_ids, int n_sep_ids, SepIdList* out) {
  if (n_sep_ids < 0 || n_sep_ids > SEP_MAX_SEP_IDS) return false;
  if (n_sep_ids > 0 && !sep_ids) return false;
  memset(out, 0, sizeof(*out));
  out->n = n_sep_ids;
  for (int i = 0; i < n_sep_ids; ++i) out->ids[i] = sep_ids[i];
  return true;
}

bool attn_shape_ok(int B, int Hq, int Hkv, int L, int d) {
  if (B < 1 || Hq < 1 || Hkv < 1 || L < 1) return false;
  if (Hq % Hkv != 0) return false;
  if (d != 64 && d != 128) return false;
  // every offset a kernel forms stays below 2^31 elements per plane index
  if ((double)B * Hq * L * d >= 9.0e15) return false;
  return true;
}

// A pack: B sequences of at most max_len rows in `total` packed rows; row and
// tile indices of one head plane stay below 2^31.
bool pack_shape_ok(int B, int total, int max_len, int Hq, int Hkv, int d) {
  if (B < 1 || total < 0 || max_len < 1 || Hq < 1 || Hkv < 1) return false;
  if (Hq % Hkv != 0 || (d != 64 && d != 128)) return false;
  if ((double)total + 128.0 * (B + 1) >= 2.0e9 || (double)B * max_len >= 2.0e9) return false;
  return true;
}

}  // namespace
}  // namespace sep

using namespace sep;

SEP_API size_t sep_index_bytes(int B, int L, int block_m) {
  if (B < 1 || L < 1 || block_m < 1) return 0;
  return index_layout(B, L, block_m).total;
}

SEP_API sep_status sep_build_index(const int32_t* ids, int B, int L, const int32_t* sep_ids,
                                   int n_sep_ids, int a, int n, int block_m, void* index_buf,
                                   size_t index_bytes, void* stream) {
  if (B < 1 || L < 1 || a < 0 || n < 1 || !ids || !index_buf) return SEP_ERR_INVALID_ARG;
  if (!aligned(ids, 4) || !aligned(index_buf, 256)) return SEP_ERR_INVALID_ARG;
  if (block_m != SEP_BLOCK_M) return SEP_ERR_UNSUPPORTED;
  SepIdList sids;
  if (!fill_sep_ids(sep_ids, n_sep_ids, &sids)) return SEP_ERR_INVALID_ARG;
  const IndexLayout lay = index_layout(B, L, block_m);
  if (index_bytes < lay.total) return SEP_ERR_WORKSPACE;
  int* st = device_status_ptr();
  if (!st) return SEP_ERR_CUDA;
  return from_cuda(launch_build_index(ids, nullptr, L, B, L, sids, a, n, block_m, 0,
                                      index_ptrs(index_buf, lay), st, stream));
}

SEP_API sep_status sep_build_index_varlen(const int32_t* ids, const int32_t* cu_seqlens, int B,
                                          int total, int max_len, const int32_t* sep_ids,
                                          int n_sep_ids, int a, int n, int block_m,
                                          void* index_buf, size_t index_bytes, void* stream) {
  if (B < 1 || total < 0 || max_len < 1 || a < 0 || n < 1 || !cu_seqlens || !index_buf ||
      (total > 0 && !ids))
    return SEP_ERR_INVALID_ARG;
  if ((double)B * max_len >= 2.0e9 || (double)total + 128.0 * (B + 1) >= 2.0e9)
    return SEP_ERR_INVALID_ARG;
  if (!aligned(ids, 4) || !aligned(cu_seqlens, 4) || !aligned(index_buf, 256))
    return SEP_ERR_INVALID_ARG;
  if (block_m != SEP_BLOCK_M) return SEP_ERR_UNSUPPORTED;
  SepIdList sids;
  if (!fill_sep_ids(sep_ids, n_sep_ids, &sids)) return SEP_ERR_INVALID_ARG;
  const IndexLayout lay = index_layout(B, max_len, block_m);
  if (index_bytes < lay.total) return SEP_ERR_WORKSPACE;
  int* st = device_status_ptr();
  if (!st) return SEP_ERR_CUDA;
  return from_cuda(launch_build_index(ids, cu_seqlens, total, B, max_len, sids, a, n, block_m, 0,
                                      index_ptrs(index_buf, lay), st, stream));
}

SEP_API sep_status sep_build_index_fixed(int B, int L, int a, int n, int delta, int block_m,
                                         void* index_buf, size_t index_bytes, void* stream) {
  if (B < 1 || L < 1 || a < 0 || n < 1 || delta < 1 || !index_buf) return SEP_ERR_INVALID_ARG;
  if (!aligned(index_buf, 256)) return SEP_ERR_INVALID_ARG;
  if (block_m != SEP_BLOCK_M) return SEP_ERR_UNSUPPORTED;
  const IndexLayout lay = index_layout(B, L, block_m);
  if (index_bytes < lay.total) return SEP_ERR_WORKSPACE;
  int* st = device_status_ptr();
  if (!st) return SEP_ERR_CUDA;
  SepIdList none;
  memset(&none, 0, sizeof(none));
  return from_cuda(launch_build_index(nullptr, nullptr, L, B, L, none, a, n, block_m, delta,
                                      index_ptrs(index_buf, lay), st, stream));
}

SEP_API sep_status sep_index_views(void* index_buf, int B, int L, int block_m,
                                   int32_t** keep_prefix, int32_t** keep_pos,
                                   int32_t** keep_count, int32_t** blocks, uint32_t** keep_bits) {
  if (!index_buf || B < 1 || L < 1 || block_m < 1) return SEP_ERR_INVALID_ARG;
  const IndexPtrs p = index_ptrs(index_buf, index_layout(B, L, block_m));
  if (keep_prefix) *keep_prefix = p.keep_prefix;
  if (keep_pos) *keep_pos = p.keep_pos;
  if (keep_count) *keep_count = p.keep_count;
  if (blocks) *blocks = p.blocks;
  if (keep_bits) *keep_bits = p.keep_bits;
  return SEP_OK;
}

SEP_API size_t sep_attn_workspace_bytes(int B, int Hq, int Hkv, int L, int d, sep_dtype dtype,
                                        int backward) {
  if (!attn_shape_ok(B, Hq, Hkv, L, d)) return 0;
  if (dtype == SEP_F32) return backward ? 0 : 256;
  const Geom geo = make_geom(B, Hq, Hkv, L, L, 0);
  if (backward) return attn_bwd_tc_workspace(geo, d);
  return attn_fwd_tc_workspace(geo, d);
}

SEP_API size_t sep_attn_workspace_bytes_varlen(int B, int total, int max_len, int Hq, int Hkv,
                                               int d, int backward) {
  if (!pack_shape_ok(B, total, max_len, Hq, Hkv, d)) return 0;
  const Geom geo = make_geom(B, Hq, Hkv, max_len, total, 1);
  if (backward) return attn_bwd_tc_workspace(geo, d);
  return attn_fwd_tc_workspace(geo, d);
}

namespace {

// Bits of full_groups at or above Hkv must be clear; with more than 64 kv
// heads no group can be named, so the mask must be 0.
bool groups_ok(uint64_t full_groups, int Hkv) {
  if (Hkv > 64) return full_groups == 0;
  return Hkv == 64 || (full_groups >> Hkv) == 0;
}

sep_status attn_fwd(const void* index_buf, const void* q, const void* k, const void* v, void* o,
                    float* lse, int B, int Hq, int Hkv, int L, int d, sep_dtype dtype,
                    float scale, uint64_t full_groups, void* ws, size_t ws_bytes, void* stream) {
  if (!index_buf || !q || !k || !v || !o || !lse) return SEP_ERR_INVALID_ARG;
  if (!attn_shape_ok(B, Hq, Hkv, L, d)) {
    if (B >= 1 && Hq >= 1 && Hkv >= 1 && L >= 1 && Hq % Hkv == 0) return SEP_ERR_UNSUPPORTED;
    return SEP_ERR_INVALID_ARG;
  }
  if (!groups_ok(full_groups, Hkv)) return SEP_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4) || !aligned(index_buf, 256))
    return SEP_ERR_INVALID_ARG;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf(static_cast<float>(d));
  if (dtype != SEP_F32 && dtype != SEP_BF16) return SEP_ERR_UNSUPPORTED;
  if (dtype == SEP_F32 && full_groups != 0) return SEP_ERR_UNSUPPORTED;
  const Geom geo = make_geom(B, Hq, Hkv, L, L, 0);
  if (dtype == SEP_BF16) {
    const size_t need = attn_fwd_tc_workspace(geo, d);
    if (!ws || ws_bytes < need) return SEP_ERR_WORKSPACE;
    if (!aligned(ws, 256)) return SEP_ERR_INVALID_ARG;
  }
  int* st = device_status_ptr();
  if (!st) return SEP_ERR_CUDA;
  const IndexPtrs idx = index_ptrs(const_cast<void*>(index_buf), index_layout(B, L, SEP_BLOCK_M));
  if (dtype == SEP_F32) {
    return from_cuda(launch_attn_fwd_simt(idx, static_cast<const float*>(q),
                                          static_cast<const float*>(k),
                                          static_cast<const float*>(v), static_cast<float*>(o),
                                          lse, B, Hq, Hkv, L, d, scale, st, stream));
  }
  return from_cuda(launch_attn_fwd_tc(idx, q, k, v, o, lse, geo, d, scale, full_groups, ws, st,
                                      stream));
}

sep_status attn_bwd(const void* index_buf, const void* q, const void* k, const void* v,
                    const void* o, const float* lse, const void* dout, void* dq, void* dk,
                    void* dv, int B, int Hq, int Hkv, int L, int d, sep_dtype dtype, float scale,
                    uint64_t full_groups, void* ws, size_t ws_bytes, void* stream) {
  if (!index_buf || !q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv)
    return SEP_ERR_INVALID_ARG;
  if (!attn_shape_ok(B, Hq, Hkv, L, d)) {
    if (B >= 1 && Hq >= 1 && Hkv >= 1 && L >= 1 && Hq % Hkv == 0) return SEP_ERR_UNSUPPORTED;
    return SEP_ERR_INVALID_ARG;
  }
  if (!groups_ok(full_groups, Hkv)) return SEP_ERR_INVALID_ARG;
  if (dtype != SEP_BF16) return SEP_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(lse, 4) || !aligned(index_buf, 256))
    return SEP_ERR_INVALID_ARG;
  const Geom geo = make_geom(B, Hq, Hkv, L, L, 0);
  const size_t need = attn_bwd_tc_workspace(geo, d);
  if (!ws || ws_bytes < need) return SEP_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return SEP_ERR_INVALID_ARG;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf(static_cast<float>(d));
  int* st = device_status_ptr();
  if (!st) return SEP_ERR_CUDA;
  const IndexPtrs idx = index_ptrs(const_cast<void*>(index_buf), index_layout(B, L, SEP_BLOCK_M));
  return from_cuda(launch_attn_bwd_tc(idx, q, k, v, o, lse, dout, dq, dk, dv, geo, d, scale,
                                      full_groups, ws, st, stream));
}

// Packed batches: the same kernels over the pack's geometry (bf16 only).
sep_status attn_fwd_pack(const void* index_buf, const void* q, const void* k, const void* v,
                         void* o, float* lse, int B, int total, int max_len, int Hq, int Hkv,
                         int d, float scale, void* ws, size_t ws_bytes, void* stream) {
  if (!index_buf || !q || !k || !v || !o || !lse) return SEP_ERR_INVALID_ARG;
  if (!pack_shape_ok(B, total, max_len, Hq, Hkv, d)) {
    if (B >= 1 && total >= 0 && max_len >= 1 && Hq >= 1 && Hkv >= 1 && Hq % Hkv == 0 &&
        d != 64 && d != 128)
      return SEP_ERR_UNSUPPORTED;
    return SEP_ERR_INVALID_ARG;
  }
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4) || !aligned(index_buf, 256))
    return SEP_ERR_INVALID_ARG;
  const Geom geo = make_geom(B, Hq, Hkv, max_len, total, 1);
  if (!ws || ws_bytes < attn_fwd_tc_workspace(geo, d)) return SEP_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return SEP_ERR_INVALID_ARG;
  if (total == 0) return SEP_OK;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf(static_cast<float>(d));
  int* st = device_status_ptr();
  if (!st) return SEP_ERR_CUDA;
  const IndexPtrs idx =
      index_ptrs(const_cast<void*>(index_buf), index_layout(B, max_len, SEP_BLOCK_M));
  return from_cuda(launch_attn_fwd_tc(idx, q, k, v, o, lse, geo, d, scale, 0, ws, st, stream));
}

sep_status attn_bwd_pack(const void* index_buf, const void* q, const void* k, const void* v,
                         const void* o, const float* lse, const void* dout, void* dq, void* dk,
                         void* dv, int B, int total, int max_len, int Hq, int Hkv, int d,
                         float scale, void* ws, size_t ws_bytes, void* stream) {
  if (!index_buf || !q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv)
    return SEP_ERR_INVALID_ARG;
  if (!pack_shape_ok(B, total, max_len, Hq, Hkv, d)) {
    if (B >= 1 && total >= 0 && max_len >= 1 && Hq >= 1 && Hkv >= 1 && Hq % Hkv == 0 &&
        d != 64 && d != 128)
      return SEP_ERR_UNSUPPORTED;
    return SEP_ERR_INVALID_ARG;
  }
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(lse, 4) || !aligned(index_buf, 256))
    return SEP_ERR_INVALID_ARG;
  const Geom geo = make_geom(B, Hq, Hkv, max_len, total, 1);
  if (!ws || ws_bytes < attn_bwd_tc_workspace(geo, d)) return SEP_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return SEP_ERR_INVALID_ARG;
  if (total == 0) return SEP_OK;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf(static_cast<float>(d));
  int* st = device_status_ptr();
  if (!st) return SEP_ERR_CUDA;
  const IndexPtrs idx =
      index_ptrs(const_cast<void*>(index_buf), index_layout(B, max_len, SEP_BLOCK_M));
  return from_cuda(launch_attn_bwd_tc(idx, q, k, v, o, lse, dout, dq, dk, dv, geo, d, scale, 0,
                                      ws, st, stream));
}

}  // namespace

SEP_API sep_status sep_attn_fwd(const void* index_buf, const void* q, const void* k,
                                const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                                int L, int d, sep_dtype dtype, float scale, void* ws,
                                size_t ws_bytes, void* stream) {
  return attn_fwd(index_buf, q, k, v, o, lse, B, Hq, Hkv, L, d, dtype, scale, 0, ws, ws_bytes,
                  stream);
}

SEP_API sep_status sep_attn_fwd_hybrid(const void* index_buf, const void* q, const void* k,
                                       const void* v, void* o, float* lse, int B, int Hq,
                                       int Hkv, int L, int d, unsigned long long full_groups,
                                       float scale, void* ws, size_t ws_bytes, void* stream) {
  return attn_fwd(index_buf, q, k, v, o, lse, B, Hq, Hkv, L, d, SEP_BF16, scale, full_groups, ws,
                  ws_bytes, stream);
}

SEP_API sep_status sep_attn_bwd(const void* index_buf, const void* q, const void* k,
                                const void* v, const void* o, const float* lse,
                                const void* dout, void* dq, void* dk, void* dv, int B, int Hq,
                                int Hkv, int L, int d, sep_dtype dtype, float scale, void* ws,
                                size_t ws_bytes, void* stream) {
  return attn_bwd(index_buf, q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, L, d, dtype, scale, 0,
                  ws, ws_bytes, stream);
}

SEP_API sep_status sep_attn_bwd_hybrid(const void* index_buf, const void* q, const void* k,
                                       const void* v, const void* o, const float* lse,
                                       const void* dout, void* dq, void* dk, void* dv, int B,
                                       int Hq, int Hkv, int L, int d,
                                       unsigned long long full_groups, float scale, void* ws,
                                       size_t ws_bytes, void* stream) {
  return attn_bwd(index_buf, q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, L, d, SEP_BF16, scale,
                  full_groups, ws, ws_bytes, stream);
}

SEP_API sep_status sep_attn_fwd_varlen(const void* index_buf, const void* q, const void* k,
                                       const void* v, void* o, float* lse, int B, int total,
                                       int max_len, int Hq, int Hkv, int d, float scale,
                                       void* ws, size_t ws_bytes, void* stream) {
  return attn_fwd_pack(index_buf, q, k, v, o, lse, B, total, max_len, Hq, Hkv, d, scale, ws,
                       ws_bytes, stream);
}

SEP_API sep_status sep_attn_bwd_varlen(const void* index_buf, const void* q, const void* k,
                                       const void* v, const void* o, const float* lse,
                                       const void* dout, void* dq, void* dk, void* dv, int B,
                                       int total, int max_len, int Hq, int Hkv, int d,
                                       float scale, void* ws, size_t ws_bytes, void* stream) {
  return attn_bwd_pack(index_buf, q, k, v, o, lse, dout, dq, dk, dv, B, total, max_len, Hq, Hkv,
                       d, scale, ws, ws_bytes, stream);
}

SEP_API sep_status sep_profile_events(void* const* events, int n_events) {
  if (n_events < 0 || n_events > SEP_MAX_PROFILE_EVENTS || (n_events > 0 && !events))
    return SEP_ERR_INVALID_ARG;
  for (int i = 0; i < SEP_MAX_PROFILE_EVENTS; ++i)
    t_prof_events[i] = i < n_events ? events[i] : nullptr;
  t_prof_n = n_events;
  return SEP_OK;
}

namespace sep {
namespace {
// One thread waits on an mbarrier that expects an arrival nobody makes.
__global__ void wait_selftest_kernel(uint64_t limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  mbar_init(&bar, 1);
  fence_mbar_init();
  mbar_wait(&bar, 0, status, limit_ns);
}
}  // namespace
}  // namespace sep

SEP_API sep_status sep_selftest_wait_timeout(int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return SEP_ERR_INVALID_ARG;
  int* st = device_status_ptr();
  if (!st) return SEP_ERR_CUDA;
  wait_selftest_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint64_t>(limit_us) * 1000ull, st);
  return from_cuda(static_cast<int>(cudaGetLastError()));
}

SEP_API sep_status sep_get_device_status(void) {
  int* st = device_status_ptr();
  if (!st) return SEP_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return SEP_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, st, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SEP_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(st, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return SEP_ERR_CUDA;
  return static_cast<sep_status>(v);
}

SEP_API const char* sep_status_string(sep_status s) {
  switch (s) {
    case SEP_OK: return "ok";
    case SEP_ERR_INVALID_ARG: return "invalid argument";
    case SEP_ERR_UNSUPPORTED: return "unsupported configuration";
    case SEP_ERR_CAPACITY: return "cache capacities violate a + s + w < c";
    case SEP_ERR_CUDA: return "CUDA runtime error";
    case SEP_ERR_TIMEOUT: return "device wait timed out";
    case SEP_ERR_DEVICE_BOUNDS: return "device index or count out of range";
    case SEP_ERR_WORKSPACE: return "buffer smaller than the size query";
    case SEP_ERR_TOO_LARGE: return "shape exceeds the fixed scratch of sep_attn_fwd_static";
  }
  return "unknown status";
}
