// Keep-token rows of K and V copied into dense tiles, and their gradients
// copied back.
//
// The tokens every query sees before its window (the first a tokens and the
// separators: anthology record lit-748, Key takeaways, "The mask") are read by
// every query tile.  Gathering them once into dense rows -- keep token r of
// sequence b, kv head g at row 128 * tile0_b + r of plane g of K_keep /
// V_keep, zero rows up to the next multiple of 128 -- turns them into full
// 128-row tiles that TMA can load.
//
// Work is cut into units of 16 rows of one (sequence, kv head) pair and one
// warp takes a unit.  Units are numbered chunk-major (unit = chunk * pairs
// + pair), so the units that hold rows come first and the kernels below use
// a grid of a few CTAs per SM that strides over them; a unit past its pair's
// padded keep count costs two cached loads.
#pragma once

#include <atomic>

#include "common.cuh"
#include "layout.h"

namespace sep {

constexpr int kKeepUnitRows = 16;

__host__ __device__ inline int keep_units(int B, int Hkv, int L) {
  return B * Hkv * ((L + kKeepUnitRows - 1) / kKeepUnitRows);
}

// Units below the largest keep count of the batch rounded up to a 128-row
// tile (units run pair-fastest, so the later ones hold neither keep rows nor
// the zero rows that pad a sequence's last gathered tile); computed by each
// calling warp.
__device__ __forceinline__ int live_keep_units(IndexPtrs idx, const Geom& geo, int lane) {
  int mc = 0;
  for (int b = lane; b < geo.B; b += 32) {
    const SeqRec sr = idx.seq[b];
    if (seq_ok(sr, geo)) mc = max(mc, min(max(idx.keep_count[b], 0), sr.len));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mc = max(mc, __shfl_xor_sync(0xffffffffu, mc, off));
  return geo.B * geo.Hkv * ((mc + 127) / 128 * (128 / kKeepUnitRows));
}

// Copies the keep rows of one unit (and, if dk_keep is set, zeroes the rows
// of the fp32 gradient accumulators dk_keep / dv_keep below the keep count,
// the only ones that are added to and read).  A keep position outside its
// sequence is reported as SEP_ERR_DEVICE_BOUNDS and its row left zero.
template <int D>
__device__ __forceinline__ void gather_keep_unit(IndexPtrs idx, const Geom& geo,
                                                 const uint4* __restrict__ k,
                                                 const uint4* __restrict__ v,
                                                 uint4* __restrict__ kk, uint4* __restrict__ vk,
                                                 float4* __restrict__ dk_keep,
                                                 float4* __restrict__ dv_keep, int unit,
                                                 int lane, int* status) {
  constexpr int U = D / 8;                         // 16-byte units of a bf16 row
  constexpr int PER = kKeepUnitRows * U / 32;      // per lane
  const int pairs = geo.B * geo.Hkv;
  const int pair = unit % pairs, row0 = (unit / pairs) * kKeepUnitRows;
  const int b = pair / geo.Hkv, g = pair % geo.Hkv;
  const SeqRec sr = idx.seq[b];
  if (!seq_ok(sr, geo)) return;
  const int count = min(max(idx.keep_count[b], 0), sr.len);
  const int end = (count + 127) / 128 * 128;
  if (row0 >= end) return;
  const int32_t* kpos = idx.keep_pos + (size_t)b * geo.L;
  const size_t src_base = ((size_t)geo.kvplane(b, g) * geo.R + sr.row0) * U;
  const size_t dst_base = ((size_t)g * geo.TT + sr.tile0) * 128 * U;
  uint4 kv[PER], vv[PER];
#pragma unroll
  for (int x = 0; x < PER; ++x) {
    const int e = x * 32 + lane;
    const int row = row0 + e / U, u = e % U;
    const int src = row < count ? kpos[row] : -1;
    kv[x] = make_uint4(0, 0, 0, 0);
    vv[x] = make_uint4(0, 0, 0, 0);
    if (src >= 0 && src < sr.len) {
      kv[x] = k[src_base + (size_t)src * U + u];
      vv[x] = v[src_base + (size_t)src * U + u];
    } else if (row < count) {
      report(status, SEP_ERR_DEVICE_BOUNDS);
    }
  }
#pragma unroll
  for (int x = 0; x < PER; ++x) {
    const int e = x * 32 + lane;
    const int row = row0 + e / U, u = e % U;
    if (row < end) {
      kk[dst_base + (size_t)row * U + u] = kv[x];
      vk[dst_base + (size_t)row * U + u] = vv[x];
    }
  }
  if (dk_keep) {
    constexpr int U4 = D / 4;  // float4 of an fp32 row
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    const size_t base4 = ((size_t)g * geo.TT + sr.tile0) * 128 * U4;
#pragma unroll
    for (int x = 0; x < 2 * PER; ++x) {
      const int e = x * 32 + lane;
      const int row = row0 + e / U4;
      if (row < count) {
        dk_keep[base4 + (size_t)row * U4 + e % U4] = z;
        dv_keep[base4 + (size_t)row * U4 + e % U4] = z;
      }
    }
  }
}

// dK / dV rows of the keep tokens of one unit, from the fp32 accumulators
// (dK times the softmax scale), rounded to bf16 once.  A keep position
// outside its sequence is reported and not written.
template <int D>
__device__ __forceinline__ void scatter_keep_unit(IndexPtrs idx, const Geom& geo,
                                                  const float4* __restrict__ dk_keep,
                                                  const float4* __restrict__ dv_keep,
                                                  __nv_bfloat16* __restrict__ dk,
                                                  __nv_bfloat16* __restrict__ dv, float scale,
                                                  int unit, int lane, int* status) {
  constexpr int U4 = D / 4;
  constexpr int PER = kKeepUnitRows * U4 / 32;
  const int pairs = geo.B * geo.Hkv;
  const int pair = unit % pairs, row0 = (unit / pairs) * kKeepUnitRows;
  const int b = pair / geo.Hkv, g = pair % geo.Hkv;
  const SeqRec sr = idx.seq[b];
  if (!seq_ok(sr, geo)) return;
  const int count = min(max(idx.keep_count[b], 0), sr.len);
  if (row0 >= count) return;
  const int32_t* kpos = idx.keep_pos + (size_t)b * geo.L;
  const size_t base4 = ((size_t)g * geo.TT + sr.tile0) * 128 * U4;
  const size_t out_base = ((size_t)geo.kvplane(b, g) * geo.R + sr.row0) * D;
  float4 a[PER], c[PER];
#pragma unroll
  for (int x = 0; x < PER; ++x) {
    const int e = x * 32 + lane;
    const int row = row0 + e / U4;
    a[x] = make_float4(0.f, 0.f, 0.f, 0.f);
    c[x] = a[x];
    if (row < count) {
      a[x] = dk_keep[base4 + (size_t)row * U4 + e % U4];
      c[x] = dv_keep[base4 + (size_t)row * U4 + e % U4];
    }
  }
#pragma unroll
  for (int x = 0; x < PER; ++x) {
    const int e = x * 32 + lane;
    const int row = row0 + e / U4, u = e % U4;
    if (row >= count) continue;
    const int j = kpos[row];
    if (j < 0 || j >= sr.len) {  // a keep position outside the sequence
      report(status, SEP_ERR_DEVICE_BOUNDS);
      continue;
    }
    uint2 ko, vo;
    ko.x = pack_bf16x2(a[x].x * scale, a[x].y * scale);
    ko.y = pack_bf16x2(a[x].z * scale, a[x].w * scale);
    vo.x = pack_bf16x2(c[x].x, c[x].y);
    vo.y = pack_bf16x2(c[x].z, c[x].w);
    const size_t dst = out_base + (size_t)j * D + 4 * u;
    *reinterpret_cast<uint2*>(dk + dst) = ko;
    *reinterpret_cast<uint2*>(dv + dst) = vo;
  }
}

// Number of SMs of the current device (148 if the query fails).
inline int num_sms() {
  // per-device cache; concurrent first lookups store the same value
  static std::atomic<int> n[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int v = n[dev].load(std::memory_order_relaxed);
  if (!v) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1)
      v = 148;
    n[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

// CTAs of 256 threads for a keep-row pass over `units` units: a few per SM,
// at most one warp per unit.
inline int keep_pass_ctas(long long units, int sms) {
  const long long want = (units + 7) / 8;
  const long long cap = 4LL * sms;
  return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace sep
