// fp32 Sep-Attention forward on CUDA cores (no tensor cores): the path for
// float32 inputs, where the tolerance (1e-4 absolute) leaves no room for
// bf16 operands.
//
// Row i's visible keys are, without overlap, the keep tokens before its
// window start W(i) = max(0, i-n+1) -- keep_pos[0 .. keep_prefix[W(i)]) --
// followed by the whole window [W(i), i] (SepLLM anthology record lit-748,
// Key takeaways, "The mask": first a tokens, preceding separators, n nearest
// tokens).  One warp owns one query row: each lane scores one key of a group
// of 32 against the row's query (held in shared memory), the warp merges the
// group into an online softmax, and each lane accumulates d/32 output
// columns.
#include "common.cuh"
#include "layout.h"

namespace sep {

namespace {

constexpr int kWarps = 8;

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
    attn_fwd_simt_kernel(IndexPtrs idx, const float* __restrict__ q, const float* __restrict__ k,
                         const float* __restrict__ v, float* __restrict__ o,
                         float* __restrict__ lse, int B, int Hq, int Hkv, int L, float scale,
                         int* status) {
  __shared__ float qs[kWarps][D];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int i = blockIdx.x * kWarps + warp;
  const int h = blockIdx.y, b = blockIdx.z;
  const IndexHeader hdr = *idx.header;
  if (hdr.magic != kIndexMagic || hdr.B != B || hdr.L != L || hdr.packed != 0) {
    if (threadIdx.x == 0) report(status, SEP_ERR_DEVICE_BOUNDS);
    return;
  }
  if (i >= L) return;
  const int n = hdr.n;
  const int g = h / (Hq / Hkv);
  const float* qrow = q + (((size_t)b * Hq + h) * L + i) * D;
  const float* kh = k + ((size_t)b * Hkv + g) * (size_t)L * D;
  const float* vh = v + ((size_t)b * Hkv + g) * (size_t)L * D;
  for (int x = lane; x < D; x += 32) qs[warp][x] = qrow[x];
  __syncwarp();

  const int W = max(0, i - n + 1);
  const int n_keep = idx.keep_prefix[(size_t)b * (L + 1) + W];
  const int32_t* kpos = idx.keep_pos + (size_t)b * L;
  const int total = n_keep + (i - W + 1);
  if (n_keep < 0 || n_keep > W) {
    if (lane == 0) report(status, SEP_ERR_DEVICE_BOUNDS);
    return;
  }

  constexpr int PER = D / 32;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float m = -INFINITY, l = 0.f;

  for (int base = 0; base < total; base += 32) {
    const int t = base + lane;
    int j = -1;
    if (t < total) j = (t < n_keep) ? kpos[t] : (W + t - n_keep);
    float s = -INFINITY;
    if (j >= 0 && j < L) {
      const float* kr = kh + (size_t)j * D;
      float dot = 0.f;
#pragma unroll 8
      for (int x = 0; x < D; ++x) dot = fmaf(qs[warp][x], kr[x], dot);
      s = dot * scale;
    } else if (t < total) {
      report(status, SEP_ERR_DEVICE_BOUNDS);
    }
    float gm = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, off));
    const float m_new = fmaxf(m, gm);
    const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
    const float p = (s == -INFINITY) ? 0.f : expf(s - m_new);
    float ps = p;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l = l * alpha + ps;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] *= alpha;
    const int cnt = min(32, total - base);
    for (int u = 0; u < cnt; ++u) {
      const float pu = __shfl_sync(0xffffffffu, p, u);
      const int ju = __shfl_sync(0xffffffffu, j, u);
      if (ju < 0 || ju >= L) continue;
      const float* vr = vh + (size_t)ju * D;
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] = fmaf(pu, vr[lane + 32 * e], acc[e]);
    }
    m = m_new;
  }
  float* orow = o + (((size_t)b * Hq + h) * L + i) * D;
  const float inv = 1.f / l;
#pragma unroll
  for (int e = 0; e < PER; ++e) orow[lane + 32 * e] = acc[e] * inv;
  if (lane == 0) lse[((size_t)b * Hq + h) * L + i] = m + logf(l);
}

}  // namespace

int launch_attn_fwd_simt(IndexPtrs idx, const float* q, const float* k, const float* v, float* o,
                         float* lse, int B, int Hq, int Hkv, int L, int d, float scale,
                         int* status, void* stream) {
  dim3 grid((L + kWarps - 1) / kWarps, Hq, B);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d == 64)
    attn_fwd_simt_kernel<64><<<grid, kWarps * 32, 0, s>>>(idx, q, k, v, o, lse, B, Hq, Hkv, L,
                                                          scale, status);
  else
    attn_fwd_simt_kernel<128><<<grid, kWarps * 32, 0, s>>>(idx, q, k, v, o, lse, B, Hq, Hkv, L,
                                                           scale, status);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace sep
