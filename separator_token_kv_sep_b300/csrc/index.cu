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
// The row is cut into scan tiles of kScanTile tokens, one CTA each (16
// tokens per thread, loaded as four 16-byte vectors).  A CTA takes its tile from a ticket counter, so the
// tiles of a sequence are claimed in order; it scans its tile (warp
// shuffle scan, then one warp over the warp totals), publishes the tile's
// keep count and looks back over the earlier tiles' published counts for
// its prefix (decoupled look-back: an earlier tile that already knows its
// inclusive prefix ends the walk).  A CTA only ever waits on tiles claimed
// before its own, by CTAs already running, so the walk always ends; it is
// also bounded in time.  Pairs of lanes join their 16 keep bits into one
// 32-bit word of the keep bitmask.  Separator ids are tested through a
// 1024-bit filter first and exactly only when its bit is set.  keep_pos is
// set to -1 by a memset before the launch, so only its valid entries are
// written here.  Each CTA writes the block records of
// the query tiles whose window start falls in its tile; the last tile of a
// sequence writes the count and the padding.  The ticket and the status
// words live in a scratch region of the index buffer that the host zeroes
// before the launch.
#include "common.cuh"
#include "layout.h"

namespace sep {

namespace {

constexpr int kThreads = 512;
static_assert(kThreads * 16 == kScanTile, "16 tokens per thread in a full scan tile");

// status word of a (sequence, scan tile): flag in bits 62-63, count below
constexpr unsigned long long kAggregate = 1ull << 62, kInclusive = 2ull << 62;
constexpr unsigned long long kValueMask = (1ull << 32) - 1;

__device__ __forceinline__ void st_release(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// PER tokens per thread: 16 for rows longer than 2048 tokens (scan tiles of
// kScanTile), 4 for rows of at most 2048 (one tile, four times the active
// threads).
template <int PER>
__global__ void __launch_bounds__(kThreads)
    build_index_kernel(const int32_t* __restrict__ ids, const int32_t* __restrict__ cu,
                       int total, int B, int L, SepIdList sids, int a, int n, int block_m,
                       int fix_delta, IndexPtrs ptrs, int* status) {
  // rows of at most one scan tile need no ticket, no look-back and no
  // scratch: tile (b, 0) is block b
  constexpr int kPerThread = PER;
  static_assert(32 % PER == 0 && PER % 4 == 0, "whole words of keep bits per lane group");
  const bool multi = L > kScanTile;  // (only with PER == 16: the launch guarantees it)
  __shared__ int warp_sums[kThreads / 32];
  __shared__ int tile_total, prefix_sh, tiles_before;
  __shared__ unsigned int ticket;
  __shared__ int sep_ids[SEP_MAX_SEP_IDS];
  // a 1024-bit filter of the separator ids (bit id & 1023): a token whose
  // bit is clear is no separator, one whose bit is set is checked exactly
  __shared__ uint32_t sep_filter[32];
  __shared__ int kposbuf[kScanTile];  // this tile's keep positions, in order
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_sep = sids.n;
  const int T = (L + block_m - 1) / block_m;
  const int ntiles = (L + kScanTile - 1) / kScanTile;
  if (tid < 32) sep_filter[tid] = 0u;
  if (tid == 0) {
    tiles_before = 0;
    ticket = multi ? atomicAdd(ptrs.scan_ticket, 1u) : blockIdx.x;
  }
  __syncthreads();
  if (tid < n_sep) {
    const int id = sids.ids[tid];
    sep_ids[tid] = id;
    atomicOr(&sep_filter[(id >> 5) & 31], 1u << (id & 31));
  }
  __syncthreads();
  const int tau = static_cast<int>(ticket);
  if (tau >= B * ntiles) return;  // cannot happen with a zeroed ticket
  const int b = tau / ntiles, k = tau % ntiles;

  // this sequence's extent: a row of L ids, or [cu[b], cu[b+1]) of a pack
  int row0 = 0, len = L, tile0 = b * T;
  if (cu) {
    const int s0 = cu[b], s1 = cu[b + 1];
    const bool ok = cu[0] == 0 && s0 >= 0 && s1 >= s0 && s1 <= total && s1 - s0 <= L;
    if (k == 0) {
      int part = 0;  // tiles of the sequences before this one
      for (int x = tid; x < b; x += kThreads) {
        const int lx = cu[x + 1] - cu[x];
        part += lx > 0 ? (lx + block_m - 1) / block_m : 0;
      }
      if (part) atomicAdd(&tiles_before, part);
      if (!ok && tid == 0) report(status, SEP_ERR_DEVICE_BOUNDS);
    }
    __syncthreads();
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
  const int base = k * kScanTile;

  // ---- this tile's keep flags and local exclusive scan
  const int j0 = base + tid * kPerThread;
  int v[kPerThread];
  if (by_ids && (reinterpret_cast<uintptr_t>(row + j0) & 15) == 0 && j0 + kPerThread <= len) {
#pragma unroll
    for (int q = 0; q < kPerThread / 4; ++q) {
      const int4 x = *reinterpret_cast<const int4*>(row + j0 + 4 * q);
      v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) v[e] = (by_ids && j0 + e < len) ? row[j0 + e] : 0;
  }
  uint32_t nib = 0;  // keep bits of the thread's 16 tokens
#pragma unroll
  for (int e = 0; e < kPerThread; ++e) {
    const int j = j0 + e;
    bool keep = false;
    if (j < len) {
      keep = j < a;
      if (by_ids) {
        if ((sep_filter[(v[e] >> 5) & 31] >> (v[e] & 31)) & 1u)
          for (int q = 0; q < n_sep; ++q) keep |= (v[e] == sep_ids[q]);
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
    const int w = lane < kThreads / 32 ? warp_sums[lane] : 0;
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += y;
    }
    if (lane < kThreads / 32) warp_sums[lane] = wi - w;
    if (lane == 31) tile_total = wi;
  }
  __syncthreads();
  int lpos = warp_sums[warp] + (incl - cnt);  // keep tokens of the tile before token j0

  // ---- the tile's prefix: publish the count, then look back over the
  // earlier tiles 32 at a time (one status word per lane of warp 0): the sum
  // of the counts down to the nearest tile that knows its inclusive prefix
  if (warp == 0) {
    unsigned long long* st = ptrs.scan_state + (size_t)b * ntiles;
    const unsigned long long mine = static_cast<unsigned long long>(tile_total);
    int prefix = 0;
    if (k == 0) {
      if (lane == 0) st_release(st, kInclusive | mine);
    } else {
      if (lane == 0) st_release(st + k, kAggregate | mine);
      const uint64_t t0 = globaltimer_ns();
      int j_hi = k - 1;
      while (true) {
        const int j = j_hi - lane;
        // before tile 0 reads as an inclusive prefix of 0
        const unsigned long long w = j >= 0 ? ld_acquire(st + j) : kInclusive;
        const unsigned pub = __ballot_sync(0xffffffffu, w != 0ull);
        const unsigned inc = __ballot_sync(0xffffffffu, (w & kInclusive) != 0ull);
        const int f = inc ? __ffs(inc) - 1 : 32;  // nearest inclusive tile
        const unsigned need = f >= 31 ? 0xffffffffu : ((1u << (f + 1)) - 1u);
        if ((pub & need) == need) {  // every tile down to it has published
          int val = (lane <= f && j >= 0) ? static_cast<int>(w & kValueMask) : 0;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) val += __shfl_xor_sync(0xffffffffu, val, off);
          prefix += val;
          if (f < 32) break;
          j_hi -= 32;  // 32 aggregates: go on below them
          continue;
        }
        __nanosleep(64);  // back off while the earlier tiles finish their scans
        bool late = false;
        if (lane == 0) late = globaltimer_ns() - t0 > kWaitLimitNs;
        if (__shfl_sync(0xffffffffu, late, 0)) {
          if (lane == 0) report(status, SEP_ERR_TIMEOUT);
          break;
        }
      }
      if (lane == 0) st_release(st + k, kInclusive | (static_cast<unsigned long long>(prefix) + mine));
    }
    if (lane == 0) prefix_sh = prefix;
  }
  __syncthreads();
  const int prefix = prefix_sh;

  // ---- keep_prefix, keep_pos and the keep bits of the tile.  keep_prefix
  // is written token-major across the warp (lane l writes token 32 m + l of
  // the warp's 512, whose owner thread and bit come by shuffle), so each
  // store covers 128 contiguous bytes; keep positions go through shared
  // memory and leave in order.
  // The block record of query tile t needs keep_prefix at its window start
  // W(t) = max(0, 128 t - n + 1): the lane that computes keep_prefix of a
  // token that is some W(t) writes that record (token 0 those of every tile
  // whose window starts at 0).
  const int Tb = (len + block_m - 1) / block_m;
  int32_t* blk = ptrs.blocks + (size_t)b * T * 4;
  auto record = [&](int t, int W, int kv) {
    int4 rec;
    rec.x = kv;
    rec.y = W;
    rec.z = min(len, t * block_m + block_m);
    rec.w = (W < a) ? 1 : 0;
    *reinterpret_cast<int4*>(blk + 4 * t) = rec;
  };
  {
    const int wbase = base + warp * 32 * kPerThread;  // the warp's first token
#pragma unroll 4
    for (int m = 0; m < kPerThread; ++m) {
      const int owner = (32 * m + lane) / PER, bit = (32 * m + lane) % PER;
      const uint32_t onib = __shfl_sync(0xffffffffu, nib, owner);
      const int olpos = __shfl_sync(0xffffffffu, lpos, owner);
      const int j = wbase + 32 * m + lane;
      if (j < len) {
        const int kv = prefix + olpos + __popc(onib & ((1u << bit) - 1u));
        kp[j] = kv;
        if (j == 0) {
          for (int t = 0; t < Tb && (long long)t * block_m - n + 1 <= 0; ++t) record(t, 0, kv);
        } else if (((long long)j + n - 1) % block_m == 0) {
          const long long t = ((long long)j + n - 1) / block_m;
          if (t < Tb) record(static_cast<int>(t), j, kv);
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < kPerThread; ++e) {
    if ((nib >> e) & 1u) kposbuf[lpos] = j0 + e;
    lpos += (nib >> e) & 1u;
  }
  // 32 / PER lanes x PER tokens = one word of the keep bitmask
  constexpr int LPW = 32 / PER;
  uint32_t word = nib << (PER * (lane % LPW));
#pragma unroll
  for (int off = 1; off < LPW; off <<= 1) word |= __shfl_xor_sync(0xffffffffu, word, off);
  const int widx = j0 >> 5;
  if (lane % LPW == 0 && widx < nwords) bits_out[widx] = word;
  __syncthreads();  // kposbuf is complete
  for (int i = tid; i < tile_total; i += kThreads) kpos[prefix + i] = kposbuf[i];

  // ---- per sequence: the last tile writes the count and the padding; the
  // first one the sequence record (and the header, for sequence 0)
  if (k == ntiles - 1) {
    const int count = prefix + tile_total;
    for (int j = len + tid; j <= L; j += kThreads) kp[j] = count;
    if (!multi)  // (a multi-tile row's keep_pos was set to -1 before the launch)
      for (int j = count + tid; j < L; j += kThreads) kpos[j] = -1;
    for (int t = Tb + tid; t < T; t += kThreads)
      *reinterpret_cast<int4*>(blk + 4 * t) = make_int4(0, 0, 0, 0);
    if (tid == 0) ptrs.keep_count[b] = count;
  }
  if (k == 0 && tid == 0) {
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
}

}  // namespace

int launch_build_index(const int32_t* ids, const int32_t* cu, int total, int B, int L,
                       const SepIdList& sids, int a, int n, int block_m, int fix_delta,
                       IndexPtrs ptrs, int* status, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int ntiles = (L + kScanTile - 1) / kScanTile;
  // the ticket and the status words start at zero; keep_pos starts at -1
  // everywhere (the kernel writes the entries below each count)
  // (rows of one scan tile need neither)
  if (ntiles > 1) {
    cudaError_t e = cudaMemsetAsync(ptrs.scan_ticket, 0,
                                    256 + sizeof(unsigned long long) * (size_t)B * ntiles, s);
    if (e == cudaSuccess)
      e = cudaMemsetAsync(ptrs.keep_pos, 0xff, sizeof(int32_t) * (size_t)B * L, s);
    if (e != cudaSuccess) return static_cast<int>(e);
  }
  if (L <= kThreads * 4)
    build_index_kernel<4><<<B, kThreads, 0, s>>>(ids, cu, total, B, L, sids, a, n, block_m,
                                                 fix_delta, ptrs, status);
  else
    build_index_kernel<16><<<B * ntiles, kThreads, 0, s>>>(ids, cu, total, B, L, sids, a, n,
                                                           block_m, fix_delta, ptrs, status);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace sep
