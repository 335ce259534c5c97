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
// A pack of variable-length sequences (cu = sequence starts) is indexed the
// same way, sequence by sequence, with positions local to each sequence: its
// first a tokens are its own sinks.  Every per-sequence field is padded to
// the longest length L; tiles and words past a sequence's end hold empty
// records and zero bits.  Each sequence also gets a record {len, row0,
// tile0}: its length, its first packed row and the number of 128-row tiles
// of the sequences before it.
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
    build_index_kernel(const int32_t* __restrict__ ids, const int32_t* __restrict__ cu,
                       int total, int B, int L, SepIdList sids, int a, int n, int block_m,
                       int fix_delta, IndexPtrs ptrs, int* status) {
  __shared__ int warp_sums[32];
  __shared__ int chunk_total;
  __shared__ int tiles_before;
  __shared__ int sep_ids[SEP_MAX_SEP_IDS];
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_sep = sids.n;
  const int T = (L + block_m - 1) / block_m;
  if (tid < n_sep) sep_ids[tid] = sids.ids[tid];
  if (tid == 0) tiles_before = 0;
  __syncthreads();

  // this sequence's extent: a row of L ids, or [cu[b], cu[b+1]) of a pack
  int row0 = 0, len = L, tile0 = b * T;
  if (cu) {
    const int s0 = cu[b], s1 = cu[b + 1];
    const bool ok = cu[0] == 0 && s0 >= 0 && s1 >= s0 && s1 <= total && s1 - s0 <= L;
    int part = 0;  // tiles of the sequences before this one
    for (int x = tid; x < b; x += kThreads) {
      const int lx = cu[x + 1] - cu[x];
      part += lx > 0 ? (lx + block_m - 1) / block_m : 0;
    }
    if (part) atomicAdd(&tiles_before, part);
    __syncthreads();
    if (!ok && tid == 0) report(status, SEP_ERR_DEVICE_BOUNDS);
    row0 = ok ? s0 : 0;
    len = ok ? s1 - s0 : 0;  // a bad extent indexes as an empty sequence
    tile0 = ok ? tiles_before : 0;
  }

  const int32_t* row = ids ? ids + (cu ? (size_t)row0 : (size_t)b * L) : nullptr;
  int32_t* kp = ptrs.keep_prefix + (size_t)b * (L + 1);
  int32_t* kpos = ptrs.keep_pos + (size_t)b * L;
  const int nwords = (L + 31) / 32;
  uint32_t* bits_out = ptrs.keep_bits + (size_t)b * nwords;
  const bool by_ids = fix_delta <= 0;  // else keep is a function of the position alone
  const bool vec_ok = by_ids && ((reinterpret_cast<uintptr_t>(row) & 15) == 0);

  int carry = 0;
  for (int base = 0; base < len; base += kChunk) {
    const int j0 = base + tid * kPerThread;
    int v[kPerThread];
    if (vec_ok && j0 + kPerThread <= len) {
      const int4 x = *reinterpret_cast<const int4*>(row + j0);
      v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    } else {
#pragma unroll
      for (int e = 0; e < kPerThread; ++e) v[e] = (by_ids && j0 + e < len) ? row[j0 + e] : 0;
    }
    uint32_t nib = 0;
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      const int j = j0 + e;
      bool keep = false;
      if (j < len) {
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
      if (j < len) {
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

  // the padding past the sequence's end: prefix held at the count, no keep
  // positions, zero bits
  for (int j = len + tid; j <= L; j += kThreads) kp[j] = carry;
  for (int j = carry + tid; j < L; j += kThreads) kpos[j] = -1;
  for (int w = (len + kChunk - 1) / kChunk * (kChunk / 32) + tid; w < nwords; w += kThreads)
    bits_out[w] = 0u;
  if (tid == 0) {
    ptrs.keep_count[b] = carry;
    SeqRec sr;
    sr.len = len; sr.row0 = row0; sr.tile0 = tile0; sr.pad = 0;
    ptrs.seq[b] = sr;
    if (b == 0) {
      IndexHeader h;
      h.magic = kIndexMagic; h.B = B; h.L = L; h.a = a; h.n = n;
      h.block_m = block_m; h.T = T; h.nwords = nwords;
      h.packed = cu ? 1 : 0;
      h.total = cu ? total : L;
      *ptrs.header = h;
    }
  }
  __syncthreads();  // keep_prefix of this row is complete and visible to the CTA

  int32_t* blk = ptrs.blocks + (size_t)b * T * 4;
  for (int t = tid; t < T; t += kThreads) {
    const int i0 = t * block_m;
    int4 rec = make_int4(0, 0, 0, 0);  // tiles past the sequence's end are empty
    if (i0 < len) {
      const int W = max(0, i0 - n + 1);
      rec.x = kp[W];
      rec.y = W;
      rec.z = min(len, i0 + block_m);
      rec.w = (W < a) ? 1 : 0;
    }
    *reinterpret_cast<int4*>(blk + 4 * t) = rec;
  }
}

}  // namespace

int launch_build_index(const int32_t* ids, const int32_t* cu, int total, int B, int L,
                       const SepIdList& sids, int a, int n, int block_m, int fix_delta,
                       IndexPtrs ptrs, int* status, void* stream) {
  build_index_kernel<<<B, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      ids, cu, total, B, L, sids, a, n, block_m, fix_delta, ptrs, status);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace sep
