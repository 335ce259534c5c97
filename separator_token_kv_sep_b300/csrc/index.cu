// Index kernel: separator detection, keep-token prefix scan and compaction,
// and per-query-tile block lists.
//
// keep[j] = (j < a) or ids[j] in the separator set -- the tokens a query
// still sees after they leave its n-token window (SepLLM anthology record
// lit-748, Key takeaways, "The mask"; separator set from the paperhub
// rebuttal, reply A1 to the first reviewer).  The FixLLM control of the
// same record ("What is ablated") replaces the separators by one token per
// interval of fix_delta positions: keep[j] = (j < a) or (j + 1) % fix_delta
// == 0, with no token ids read.
//
// One CTA of 1024 threads per sequence walks the row in chunks of 4096
// tokens, 4 per thread: a warp shuffle scan and a one-warp scan of the 32
// warp totals give every token its exclusive keep count; the running carry
// links the chunks.  Groups of 8 lanes OR their 4-bit keep nibbles into one
// 32-bit word of the keep bitmask.  The block lists are written after the
// scan, from keep_prefix, by the same CTA.
#include "common.cuh"
#include "layout.h"

namespace sep {

namespace {

constexpr int kThreads = 1024;
constexpr int kPerThread = 4;
constexpr int kChunk = kThreads * kPerThread;

__global__ void __launch_bounds__(kThreads)
    build_index_kernel(const int32_t* __restrict__ ids, int B, int L, SepIdList sids, int a, int n,
                       int block_m, int fix_delta, IndexPtrs ptrs, int* status) {
  __shared__ int warp_sums[32];
  __shared__ int chunk_total;
  __shared__ int sep_ids[SEP_MAX_SEP_IDS];
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_sep = sids.n;
  if (tid < n_sep) sep_ids[tid] = sids.ids[tid];
  __syncthreads();

  const int32_t* row = ids + (size_t)b * L;
  int32_t* kp = ptrs.keep_prefix + (size_t)b * (L + 1);
  int32_t* kpos = ptrs.keep_pos + (size_t)b * L;
  const int T = (L + block_m - 1) / block_m;
  const int nwords = (L + 31) / 32;
  uint32_t* bits_out = ptrs.keep_bits + (size_t)b * nwords;
  const bool by_ids = fix_delta <= 0;  // else keep is a function of the position alone
  const bool vec_ok =
      by_ids && ((L & 3) == 0) && ((reinterpret_cast<uintptr_t>(row) & 15) == 0);

  int carry = 0;
  for (int base = 0; base < L; base += kChunk) {
    const int j0 = base + tid * kPerThread;
    int v[kPerThread];
    if (vec_ok && j0 + kPerThread <= L) {
      const int4 x = *reinterpret_cast<const int4*>(row + j0);
      v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    } else {
#pragma unroll
      for (int e = 0; e < kPerThread; ++e) v[e] = (by_ids && j0 + e < L) ? row[j0 + e] : 0;
    }
    uint32_t nib = 0;
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      const int j = j0 + e;
      bool keep = false;
      if (j < L) {
        keep = j < a;
        if (by_ids) {
          for (int s = 0; s < n_sep; ++s) keep |= (v[e] == sep_ids[s]);
        } else {
          keep |= (j + 1) % fix_delta == 0;
        }
      }
      nib |= (keep ? 1u : 0u) << e;
    }
    const int cnt = __popc(nib);
    int incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int w = warp_sums[lane];
      int wi = w;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wi, off);
        if (lane >= off) wi += y;
      }
      warp_sums[lane] = wi - w;
      if (lane == 31) chunk_total = wi;
    }
    __syncthreads();
    int pos = carry + warp_sums[warp] + (incl - cnt);
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      const int j = j0 + e;
      if (j < L) {
        kp[j] = pos;
        if ((nib >> e) & 1u) kpos[pos++] = j;
      }
    }
    // 8 lanes x 4 tokens = one 32-bit word of the keep bitmask
    uint32_t word = nib << (4 * (lane & 7));
    word |= __shfl_xor_sync(0xffffffffu, word, 1);
    word |= __shfl_xor_sync(0xffffffffu, word, 2);
    word |= __shfl_xor_sync(0xffffffffu, word, 4);
    const int widx = j0 >> 5;
    if ((lane & 7) == 0 && widx < nwords) bits_out[widx] = word;
    carry += chunk_total;
    __syncthreads();  // warp_sums / chunk_total are rewritten next chunk
  }

  if (tid == 0) {
    kp[L] = carry;
    ptrs.keep_count[b] = carry;
    if (b == 0) {
      IndexHeader h;
      h.magic = kIndexMagic; h.B = B; h.L = L; h.a = a; h.n = n;
      h.block_m = block_m; h.T = T; h.nwords = nwords;
      *ptrs.header = h;
    }
  }
  for (int j = carry + tid; j < L; j += kThreads) kpos[j] = -1;
  __syncthreads();  // keep_prefix of this row is complete and visible to the CTA

  int32_t* blk = ptrs.blocks + (size_t)b * T * 4;
  for (int t = tid; t < T; t += kThreads) {
    const int i0 = t * block_m;
    const int W = max(0, i0 - n + 1);
    int4 rec;
    rec.x = kp[W];
    rec.y = W;
    rec.z = min(L, i0 + block_m);
    rec.w = (W < a) ? 1 : 0;
    *reinterpret_cast<int4*>(blk + 4 * t) = rec;
  }
}

}  // namespace

int launch_build_index(const int32_t* ids, int B, int L, const SepIdList& sids, int a, int n,
                       int block_m, int fix_delta, IndexPtrs ptrs, int* status, void* stream) {
  build_index_kernel<<<B, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      ids, B, L, sids, a, n, block_m, fix_delta, ptrs, status);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace sep
