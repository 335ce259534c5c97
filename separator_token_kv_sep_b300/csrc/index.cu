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
// 32-bit word of the keep bitmask.  Separator ids are looked up in a
// direct-mapped table of 1024 slots (slot = id & 1023): one shared-memory
// load and a compare per token, and a loop over the ids only for a slot
// that two separator ids share.  Only keep_pos entries below the count are
// written.  Each CTA writes the block records of the query tiles whose
// window start falls in its tile (the thread owning that token); the last
// tile of a sequence writes the count and the padding.  The ticket and the
// status words live in a scratch region of the index buffer that the host
// zeroes before the launch.
#include "common.cuh"
#include "layout.h"

namespace sep {

namespace {

constexpr int kThreads = 512;
constexpr int kBM = SEP_BLOCK_M;  // query-tile height of the block records
static_assert(kThreads * 16 == kScanTile, "16 tokens per thread in a full scan tile");
static_assert((kBM & (kBM - 1)) == 0, "block records assume a power-of-two tile height");

// separator table: slot s = id & 1023 holds the separator id of that slot,
// s ^ 1 when no separator id maps there (never equal to an id of slot s) or
// s ^ 2 when several do (then the ids are compared one by one)
constexpr int kSlots = 1024;

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
__global__ void __launch_bounds__(kThreads, 4)
    build_index_kernel(const int32_t* __restrict__ ids, const int32_t* __restrict__ cu,
                       int total, int B, int L, SepIdList sids, int a, int n,
                       int fix_delta, IndexPtrs ptrs, int* status) {
  constexpr int block_m = kBM;
  // rows of at most one scan tile need no ticket, no look-back and no
  // scratch: tile (b, 0) is block b
  constexpr int kPerThread = PER;
  static_assert(32 % PER == 0 && PER % 4 == 0, "whole words of keep bits per lane group");
  const bool multi = L > kScanTile;  // (only with PER == 16: the launch guarantees it)
  __shared__ int warp_sums[kThreads / 32];
  __shared__ int tile_total, prefix_sh, tiles_before;
  __shared__ unsigned int ticket;
  __shared__ int sep_ids[SEP_MAX_SEP_IDS];
  __shared__ int sep_slot[kSlots];
  __shared__ __align__(16) int stage[kThreads * PER];  // keep_prefix values, per warp
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_sep = sids.n;
  const int T = (L + block_m - 1) / block_m;
  const int ntiles = (L + kScanTile - 1) / kScanTile;
  for (int s = tid; s < kSlots; s += kThreads) sep_slot[s] = s ^ 1;
  grid_dep_wait();
  if (tid == 0) {
    tiles_before = 0;
    ticket = multi ? atomicAdd(ptrs.scan_ticket, 1u) : blockIdx.x;
  }
  __syncthreads();
  if (tid < n_sep) {
    const int id = sids.ids[tid], s = id & (kSlots - 1);
    sep_ids[tid] = id;
    const int old = atomicCAS(&sep_slot[s], s ^ 1, id);
    if (old != (s ^ 1) && old != id) sep_slot[s] = s ^ 2;  // shared slot
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
  uint32_t nib = 0;  // keep bits of the thread's tokens
  if (by_ids) {
    uint32_t shared_slot = 0;  // tokens whose slot several separator ids share
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      const int t = sep_slot[v[e] & (kSlots - 1)];
      nib |= (t == v[e] ? 1u : 0u) << e;
      shared_slot |= (((t ^ v[e]) & (kSlots - 1)) == 2 ? 1u : 0u) << e;
    }
    if (__any_sync(0xffffffffu, shared_slot != 0u)) {
#pragma unroll
      for (int e = 0; e < kPerThread; ++e) {
        if (!((shared_slot >> e) & 1u)) continue;
        bool hit = false;
        for (int q = 0; q < n_sep; ++q) hit |= (v[e] == sep_ids[q]);
        nib |= (hit ? 1u : 0u) << e;
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) nib |= ((j0 + e + 1) % fix_delta == 0 ? 1u : 0u) << e;
  }
  if (j0 < a)  // the sinks
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) nib |= (j0 + e < a ? 1u : 0u) << e;
  if (j0 + kPerThread > len)  // past the sequence's end
    nib &= len > j0 ? (1u << (len - j0)) - 1u : 0u;
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

  // ---- block records, keep_prefix, keep_pos and the keep bits of the tile.
  // The block record of query tile t needs keep_prefix at its window start
  // W(t) = max(0, 128 t - n + 1).  A window start above 0 is a token j with
  // j = 1 - n (mod 128); the thread owning it writes the record (at most one
  // per thread).  Tile 0's CTA writes the records of every tile whose window
  // starts at 0.
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
    const int resid = static_cast<int>((1 - static_cast<long long>(n)) & (block_m - 1));
    const int e = (resid - j0) & (block_m - 1);  // the thread's token of that residue
    const int j = j0 + e;
    if (e < kPerThread && j > 0 && j < len) {
      const long long t = ((long long)j + n - 1) / block_m;
      if (t < Tb) record(static_cast<int>(t), j, prefix + lpos + __popc(nib & ((1u << e) - 1u)));
    }
    if (k == 0)  // windows that start at token 0 (keep_prefix[0] = 0)
      for (int t = tid; t < Tb && (long long)t * block_m - n + 1 <= 0; t += kThreads)
        record(t, 0, 0);
  }
  {
    // through the warp's part of the staging buffer: written thread-major,
    // read back token-major, so each global store covers 128 contiguous bytes
    int* wst = stage + warp * 32 * kPerThread;
    int run = prefix + lpos;
#pragma unroll
    for (int q = 0; q < kPerThread / 4; ++q) {
      int4 x;
      x.x = run; run += (nib >> (4 * q)) & 1u;
      x.y = run; run += (nib >> (4 * q + 1)) & 1u;
      x.z = run; run += (nib >> (4 * q + 2)) & 1u;
      x.w = run; run += (nib >> (4 * q + 3)) & 1u;
      *reinterpret_cast<int4*>(wst + lane * kPerThread + 4 * q) = x;
    }
    __syncwarp();
    const int wbase = base + warp * 32 * kPerThread;  // the warp's first token
#pragma unroll
    for (int m = 0; m < kPerThread; ++m) {
      const int j = wbase + 32 * m + lane;
      if (j < len) kp[j] = wst[32 * m + lane];
    }
  }
  // keep positions, in order: a lane's keep tokens go to consecutive
  // entries from its prefix, and a warp's stores stay within its few
  // hundred bytes of keep_pos
  {
    uint32_t rest = nib;
    int* out = kpos + prefix + lpos;
    while (rest) {
      *out++ = j0 + __ffs(rest) - 1;
      rest &= rest - 1u;
    }
  }
  // 32 / PER lanes x PER tokens = one word of the keep bitmask
  constexpr int LPW = 32 / PER;
  uint32_t word = nib << (PER * (lane % LPW));
#pragma unroll
  for (int off = 1; off < LPW; off <<= 1) word |= __shfl_xor_sync(0xffffffffu, word, off);
  const int widx = j0 >> 5;
  if (lane % LPW == 0 && widx < nwords) bits_out[widx] = word;

  // ---- per sequence: the last tile writes the count and the padding; the
  // first one the sequence record (and the header, for sequence 0)
  if (k == ntiles - 1) {
    const int count = prefix + tile_total;
    for (int j = len + tid; j <= L; j += kThreads) kp[j] = count;
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
  if (block_m != kBM) return static_cast<int>(cudaErrorInvalidValue);
  // the ticket and the status words start at zero (rows of one scan tile
  // use neither)
  if (ntiles > 1) {
    const cudaError_t e = cudaMemsetAsync(
        ptrs.scan_ticket, 0, 256 + sizeof(unsigned long long) * (size_t)B * ntiles, s);
    if (e != cudaSuccess) return static_cast<int>(e);
  }
  const cudaError_t e =
      L <= kThreads * 4
          ? launch_dependent(build_index_kernel<4>, dim3(B), dim3(kThreads), 0, s, ids, cu,
                             total, B, L, sids, a, n, fix_delta, ptrs, status)
          : launch_dependent(build_index_kernel<16>, dim3(B * ntiles), dim3(kThreads), 0, s,
                             ids, cu, total, B, L, sids, a, n, fix_delta, ptrs, status);
  return static_cast<int>(e);
}

}  // namespace sep
