// Sep-Attention backward on the tcgen05 tensor cores.
//
// What it computes: the gradients of masked softmax attention under the
// SepLLM mask (first a tokens, preceding separators, n nearest tokens:
// anthology record lit-748, Key takeaways, "The mask"; the pages train with
// this mask, same record, "Training from scratch"), by recomputation from
// the forward's LSE:
//   P = exp(S*scale - LSE), Delta = rowsum(dO o O), dS = P o (dO V^T - Delta),
//   dV = P^T dO, dQ = scale * dS K, dK = scale * dS^T Q.
// With grouped-query heads, dK and dV of a kv head sum over its q heads.
//
// Every visible pair (i, j) belongs to exactly one of the forward's two key
// sources (gathered keep tokens before the query tile's window, or the dense
// band), and the backward keeps that split.  Three launches:
//   bwd_prep_kernel     the keep-token K/V gather, zeroed fp32 keep-token
//                       gradient accumulators, the per-row stats
//                       (-LSE log2 e, -Delta) and, in CTA 0, the dK/dV work
//                       schedule.
//   bwd_kv_persistent   key-major dK/dV, one CTA per SM over the schedule's
//                       items: a 128-key tile (gathered keep tokens, or a
//                       dense key range) against the query tiles that see it,
//                       for every q head of its kv group.  S^T = K Q^T and
//                       dP^T = V dO^T go to TMEM per 64-query half-tile; the
//                       elementwise warpgroups overwrite them with P^T and
//                       dS^T, which the dV += P^T dO and dK += dS^T Q products
//                       read from TMEM.  Keep tokens add into the fp32
//                       accumulators with red.global.add; other keys are
//                       written as bf16 at once.
//   bwd_dq_persistent   query-major dQ, one CTA per SM: the forward's
//                       traversal, S = Q K^T and dP = dO V^T into TMEM, dS to
//                       shared memory, dQ += dS K.  Its elementwise warps
//                       first write the keep tokens' dK / dV rows from the
//                       finished accumulators, while the first item's copies
//                       and products are in flight.
// The MMA issuers run warp-uniform, with one elected lane issuing.
// All waits are bounded; on expiry a kernel records SEP_ERR_TIMEOUT, drains
// its copies and MMAs, frees TMEM and returns.
#include "common.cuh"
#include "keep_rows.cuh"
#include "layout.h"
#include "tma_host.h"

namespace sep {

namespace {

constexpr int kChunk = 128 * 128;  // bytes of a [128 rows x 64 cols] bf16 block
constexpr int kThreads = 320;      // warp 0 TMA, warp 1 MMA, warps 2-9 elementwise
constexpr int kEwThreads = 256;    // two elementwise warpgroups
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kKeepChunk = 8;      // query tiles per keep item of the dK/dV kernel
constexpr int kCtaItems = 128;     // work items a dK/dV CTA keeps in static shared memory

__device__ __forceinline__ uint32_t range_bits(int lo, int hi, int w) {
  // bits c of word w (columns 32w .. 32w+31) with lo <= c < hi
  const int a = max(lo - 32 * w, 0), b = min(hi - 32 * w, 32);
  if (b <= a) return 0u;
  const uint32_t upto_b = b >= 32 ? 0xffffffffu : ((1u << b) - 1u);
  const uint32_t below_a = a >= 32 ? 0xffffffffu : ((1u << a) - 1u);
  return upto_b & ~below_a;
}

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}


// ---------------------------------------------------------------------------
// Work schedule of the key-major pass.  An item is one 128-key tile and a
// range of query tiles [t0, t1), walked for every q head of its kv group:
//   KEEP   keys are gathered keep tokens [row0, row0+128) of K_keep/V_keep;
//          query tile t sees keep token k iff k < n_gather(t).  A keep tile's
//          query tiles are cut into chunks of kKeepChunk tiles.
//   DENSE  keys are positions [row0, row0+128) of K/V; the query tiles are
//          those whose dense band reaches the tile, element mask as in the
//          forward.
// Items are written by CTA 0 of the prep kernel: keep items first
// (they are the longest), then dense items.  Persistent CTAs take items
// round-robin.
// ---------------------------------------------------------------------------
constexpr int kItemKeep = 0, kItemDense = 1;

struct BwdSchedule {  // header of the schedule region; int4 items follow
  int n_items, n_keep, max_count, pad;  // max_count: the largest keep count
};

__host__ __device__ inline size_t bwd_max_items(int B, int Hkv, int T) {
  const size_t chunks = (size_t)(T + kKeepChunk - 1) / kKeepChunk + 1;
  return (size_t)B * Hkv * T * (chunks + 1);
}

// Block-wide exclusive scan of one int per thread (blockDim.x threads,
// a multiple of 32, at most 1024).  Returns the exclusive prefix; *total
// receives the sum.  `sh` holds 33 ints.
__device__ __forceinline__ int block_exclusive_scan(int x, int* sh, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = x;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int v = lane < nw ? sh[lane] : 0;
    int vi = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, vi, off);
      if (lane >= off) vi += y;
    }
    sh[lane] = vi - v;
    if (lane == 31) sh[32] = vi;
  }
  __syncthreads();
  const int r = sh[warp] + incl - x;
  *total = sh[32];
  __syncthreads();
  return r;
}

// The index header sits at offset 0 of any index buffer: every kernel checks
// it against the call's geometry before using the fields whose offsets
// depend on B and L.
__device__ __forceinline__ bool header_matches(const IndexHeader& h, const Geom& geo) {
  return h.magic == kIndexMagic && h.B == geo.B && h.L == geo.L && h.block_m == 128 &&
         h.packed == geo.packed && h.total == geo.R;
}

// Builds the schedule (one CTA).  blocks[b][t] = {n_gather, dense_lo, dense_hi, flags};
// sequence b has T_b = ceil(len_b / 128) query tiles (all T in an
// equal-length batch).  Items of a sequence whose record is unusable are left
// out (the attention kernels report it).
__device__ void build_bwd_schedule(IndexPtrs idx, const Geom& geo, uint64_t full_groups,
                                   BwdSchedule* sched, int4* items) {
  __shared__ int sh[33];
  __shared__ int s_maxc;
  const int B = geo.B, Hkv = geo.Hkv, T = geo.T;
  int total = 0;
  if (threadIdx.x == 0) s_maxc = 0;
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const SeqRec sr = idx.seq[b];
    if (seq_ok(sr, geo)) atomicMax(&s_maxc, min(max(idx.keep_count[b], 0), sr.len));
  }
  // kv groups with full causal attention have no keep items, and every
  // query tile from the key tile on sees their dense key tiles
  int nsep = 0;
  for (int g = 0; g < Hkv; ++g) nsep += group_full(full_groups, g) ? 0 : 1;
  // keep items: (b, keep tile kt) -> chunks of query tiles from t_begin(kt)
  for (int base = 0; base < B * T; base += blockDim.x) {
    const int id = base + threadIdx.x;
    int n = 0, tb = T, Tb = 0;
    if (id < B * T) {
      const int b = id / T, kt = id % T;
      const SeqRec sr = idx.seq[b];
      if (seq_ok(sr, geo)) {
        Tb = (sr.len + 127) >> 7;
        const int count = min(max(idx.keep_count[b], 0), sr.len);
        if (kt * 128 < count) {
          const int32_t* blk = idx.blocks + (size_t)b * T * 4;
          int lo = 0, hi = Tb;  // first t with n_gather(t) > 128 kt
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (blk[4 * mid] > kt * 128) hi = mid; else lo = mid + 1;
          }
          tb = lo;
          n = (Tb - tb + kKeepChunk - 1) / kKeepChunk;
        }
      }
    }
    int sum;
    const int ex = block_exclusive_scan(n, sh, &sum);
    if (n > 0) {
      const int b = id / T, kt = id % T;
      for (int cc = 0; cc < n; ++cc) {
        const int t0 = tb + cc * kKeepChunk, t1 = min(Tb, t0 + kKeepChunk);
        int gi = 0;
        for (int g = 0; g < Hkv; ++g) {
          if (group_full(full_groups, g)) continue;
          items[total + (size_t)(ex + cc) * nsep + gi] =
              make_int4(kItemKeep, b * Hkv + g, kt * 128, (t0 << 16) | t1);
          ++gi;
        }
      }
    }
    total += sum * nsep;
  }
  const int n_keep = total;
  // dense items: (b, key tile jt < T_b) -> query tiles jt .. (last whose band
  // starts before the tile ends)
  for (int base = 0; base < B * T; base += blockDim.x) {
    const int id = base + threadIdx.x;
    int live = 0, Tb = 0;
    if (id < B * T) {
      const SeqRec sr = idx.seq[id / T];
      if (seq_ok(sr, geo)) {
        Tb = (sr.len + 127) >> 7;
        live = (id % T) < Tb ? 1 : 0;
      }
    }
    int sum;
    const int ex = block_exclusive_scan(live, sh, &sum);
    if (live) {
      const int b = id / T, jt = id % T;
      const int32_t* blk = idx.blocks + (size_t)b * T * 4;
      int lo = jt, hi = Tb;  // first t >= jt with dense_lo(t) >= 128 jt + 128
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (blk[4 * mid + 1] < jt * 128 + 128) lo = mid + 1; else hi = mid;
      }
      for (int g = 0; g < Hkv; ++g)
        items[total + (size_t)ex * Hkv + g] =
            make_int4(kItemDense, b * Hkv + g, jt * 128,
                      (jt << 16) | (group_full(full_groups, g) ? Tb : max(lo, jt + 1)));
    }
    total += sum * Hkv;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    sched->n_items = total;
    sched->n_keep = n_keep;
    sched->max_count = s_maxc;
  }
}

// ---------------------------------------------------------------------------
// Prep, one launch before the tensor-core passes:
//   CTA 0      writes the dK/dV work schedule;
//   the rest   stride, one warp per unit, over
//              - the keep-row units: gathered K_keep / V_keep rows and zeroed
//                fp32 keep accumulators dK_keep / dV_keep;
//              - the stats units of kPrepRows rows of the padded
//                [B*Hq][ceil128(L)] row space: (-LSE log2(e), -Delta) with
//                Delta = rowsum(dO o O) in fp32; rows past L get (0, 0).
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 256;
constexpr int kPrepRows = 16;  // rows per stats unit

template <int D>
__device__ __forceinline__ void prep_stats_unit(IndexPtrs idx, const Geom& geo,
                                                const uint4* __restrict__ o,
                                                const uint4* __restrict__ dout,
                                                const float* __restrict__ lse,
                                                float2* __restrict__ stats, size_t unit,
                                                int lane) {
  constexpr int U = D / 8;         // 16-byte units per row
  constexpr int RPI = 32 / U;      // rows per warp instruction
  constexpr int IT = kPrepRows / RPI;
  // unit -> (sequence b, q head h, rows [i0, i0 + kPrepRows) of its T*128)
  const int TP = geo.T * 128;
  const size_t r0 = unit * kPrepRows;
  const int bh = static_cast<int>(r0 / TP), i0 = static_cast<int>(r0 % TP);
  const int b = bh / geo.Hq, h = bh % geo.Hq;
  const SeqRec sr = idx.seq[b];
  if (!seq_ok(sr, geo) || i0 >= (sr.len + 127) / 128 * 128) return;  // no stats rows here
  const size_t src0 = (size_t)geo.qplane(b, h) * geo.R + sr.row0;
  float2* dst = stats + ((size_t)h * geo.TT + sr.tile0) * 128;
  const int sub = lane / U, u = lane % U;
  uint4 xo[IT], xd[IT];
  bool live[IT];
#pragma unroll
  for (int it = 0; it < IT; ++it) {
    const int i = i0 + it * RPI + sub;
    live[it] = i < sr.len;
    xo[it] = live[it] ? o[(src0 + i) * U + u] : make_uint4(0, 0, 0, 0);
    xd[it] = live[it] ? dout[(src0 + i) * U + u] : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int it = 0; it < IT; ++it) {
    const uint32_t xs[4] = {xo[it].x, xo[it].y, xo[it].z, xo[it].w};
    const uint32_t ys[4] = {xd[it].x, xd[it].y, xd[it].z, xd[it].w};
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(__uint_as_float(xs[e] << 16), __uint_as_float(ys[e] << 16), acc);
      acc = fmaf(__uint_as_float(xs[e] & 0xffff0000u), __uint_as_float(ys[e] & 0xffff0000u),
                 acc);
    }
#pragma unroll
    for (int off = U / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    const int i = i0 + it * RPI + sub;
    if (u == 0)
      dst[i] = live[it] ? make_float2(-lse[src0 + i] * kLog2e, -acc) : make_float2(0.f, 0.f);
  }
}

template <int D>
__global__ void __launch_bounds__(kPrepThreads)
    bwd_prep_kernel(IndexPtrs idx, Geom geo, const uint4* __restrict__ k,
                    const uint4* __restrict__ v, uint4* __restrict__ kk, uint4* __restrict__ vk,
                    const uint4* __restrict__ o, const uint4* __restrict__ dout,
                    const float* __restrict__ lse, float2* __restrict__ stats,
                    float4* __restrict__ dk_keep, float4* __restrict__ dv_keep,
                    uint64_t full_groups, BwdSchedule* __restrict__ sched,
                    int4* __restrict__ items, int* status) {
  grid_dep_wait();
  const IndexHeader hdr = *idx.header;
  if (!header_matches(hdr, geo)) return;
  if (blockIdx.x == 0) {
    build_bwd_schedule(idx, geo, full_groups, sched, items);
    return;
  }
  constexpr int WPB = kPrepThreads / 32;
  const int lane = threadIdx.x & 31;
  const size_t w0 = (size_t)(blockIdx.x - 1) * WPB + (threadIdx.x >> 5);
  const size_t nw = (size_t)(gridDim.x - 1) * WPB;
  const size_t gunits = static_cast<size_t>(live_keep_units(idx, geo, lane));
  const size_t sunits = (size_t)geo.B * geo.Hq * geo.T * 128 / kPrepRows;
  for (size_t u = w0; u < gunits + sunits; u += nw) {
    if (u < gunits)
      gather_keep_unit<D>(idx, geo, k, v, kk, vk, dk_keep, dv_keep, static_cast<int>(u), lane,
                          status);
    else
      prep_stats_unit<D>(idx, geo, o, dout, lse, stats, u - gunits, lane);
  }
}

// ---------------------------------------------------------------------------
// Key-major dK / dV, persistent
// ---------------------------------------------------------------------------
template <int D>
struct KvCfg {
  static constexpr int DCH = D / 64;
  static constexpr int TILE = DCH * kChunk;
  static constexpr int KVB = D == 64 ? 2 : 1;   // K/V tile buffers
  static constexpr int NST = D == 64 ? 3 : 2;   // Q/dO ring stages
  static constexpr int ACB = D == 64 ? 2 : 1;   // dK/dV accumulator buffers in TMEM
  // half-tile buffers in TMEM (three with one accumulator buffer at d = 64
  // was measured slower: the epilogue then waits for the item's last MMAs)
  static constexpr int NHB = 2;
  static constexpr int OFF_KV = 0;              // [KVB][K, V]
  static constexpr int OFF_Q = OFF_KV + KVB * 2 * TILE;
  static constexpr int OFF_DO = OFF_Q + NST * TILE;
  static constexpr int OFF_STAT = OFF_DO + NST * TILE;  // [NST][128] (-LSE log2, -Delta)
  static constexpr int SMEM = OFF_STAT + NST * 128 * 8 + 1024;
  // TMEM: half-tile buffers x < NHB at 128x (S^T / P^T, then dP^T / dS^T at
  // +64); accumulator buffer b: dV at TM_ACC + 2bD, dK at TM_ACC + 2bD + D
  static constexpr int TM_ACC = 128 * NHB;
  static constexpr int TM_COLS = 512;
  static_assert(SMEM + 68 * kCtaItems + 256 <= 227 * 1024, "shared memory");
  static_assert(TM_ACC + ACB * 2 * D <= TM_COLS, "tensor memory");
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kv_persistent(const __grid_constant__ CUtensorMap tm_kk,
                      const __grid_constant__ CUtensorMap tm_vk,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_do, IndexPtrs idx,
                      const BwdSchedule* __restrict__ sched, const int4* __restrict__ items,
                      const float2* __restrict__ stats,
                      float* __restrict__ dk_keep, float* __restrict__ dv_keep,
                      __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, Geom geo,
                      float scale, float scale_log2, uint64_t full_groups, int* status) {
  using C = KvCfg<D>;
  constexpr int KVB = C::KVB, NST = C::NST, ACB = C::ACB, NHB = C::NHB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t kv_full[KVB], kv_empty[KVB], qd_full[NST], qd_empty[NST];
  __shared__ __align__(8) uint64_t sd_full[NHB], ps_full[NHB], acc_full[ACB], acc_empty[ACB],
      mma_final;
  __shared__ uint32_t tmem_slot;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = geo.T, Hq = geo.Hq, Hkv = geo.Hkv, L = geo.L;
  const int G = Hq / Hkv;

  if (threadIdx.x == 0) {
    for (int i = 0; i < KVB; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < NST; ++i) {
      mbar_init(&qd_full[i], 1);
      mbar_init(&qd_empty[i], 1);
    }
    for (int i = 0; i < ACB; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEwThreads);
    }
    for (int x = 0; x < NHB; ++x) {
      mbar_init(&sd_full[x], 1);
      mbar_init(&ps_full[x], 128);
    }
    mbar_init(&mma_final, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, C::TM_COLS);
    tmem_relinquish();
  }
  // barriers and tensor memory are set up before waiting for the prep kernel
  grid_dep_wait();
  const IndexHeader hdr = *idx.header;
  const int n_items = sched->n_items;
  if (!header_matches(hdr, geo) || n_items < 0 ||
      (size_t)n_items > bwd_max_items(geo.B, Hkv, T)) {
    if (threadIdx.x == 0) report(status, SEP_ERR_DEVICE_BOUNDS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_slot, C::TM_COLS);
    return;
  }
  const int n_win = hdr.n;
  // this CTA's items (i = snake_item(k, gridDim.x)) and what every role
  // needs of them, read once: the sequence record with its keep count, the
  // block record of the first query tile and, for a dense key tile, its 128
  // keep bits and the keep prefix at its first key.  Items past kCtaItems
  // read the same from global memory when they start.
  __shared__ int4 s_items[kCtaItems];
  __shared__ int4 s_seq[kCtaItems];     // {len, row0, tile0, keep count}
  __shared__ int4 s_blk0[kCtaItems];
  __shared__ uint4 s_kbits[kCtaItems];
  __shared__ int s_kpre[kCtaItems];
  auto item_seq = [&](int4 it) -> int4 {
    const int b = it.y / Hkv;
    const SeqRec sr = idx.seq[b];
    return make_int4(sr.len, sr.row0, sr.tile0, min(max(idx.keep_count[b], 0), sr.len));
  };
  auto item_blk0 = [&](int4 it, int len) -> int4 {
    const int b = it.y / Hkv, g = it.y % Hkv, t0 = it.w >> 16;
    return group_full(full_groups, g)
               ? full_block_record(t0, len)
               : *reinterpret_cast<const int4*>(idx.blocks + ((size_t)b * T + t0) * 4);
  };
  for (int x = threadIdx.x; x < kCtaItems; x += blockDim.x) {
    const int i = snake_item(x, static_cast<int>(gridDim.x));
    if (i < n_items) {
      const int4 it = items[i];
      const int4 sq = item_seq(it);
      s_items[x] = it;
      s_seq[x] = sq;
      s_blk0[x] = item_blk0(it, sq.x);
      uint4 kb = make_uint4(0u, 0u, 0u, 0u);
      int kpre = 0;
      if (it.x == kItemDense) {
        const int b = it.y / Hkv, w0 = it.z >> 5;
        const uint32_t* bw = idx.keep_bits + (size_t)b * hdr.nwords;
        kb.x = w0 < hdr.nwords ? bw[w0] : 0u;
        kb.y = w0 + 1 < hdr.nwords ? bw[w0 + 1] : 0u;
        kb.z = w0 + 2 < hdr.nwords ? bw[w0 + 2] : 0u;
        kb.w = w0 + 3 < hdr.nwords ? bw[w0 + 3] : 0u;
        kpre = idx.keep_prefix[(size_t)b * (L + 1) + it.z];
      }
      s_kbits[x] = kb;
      s_kpre[x] = kpre;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  // item decoding shared by every role; the schedule holds items of usable
  // sequences only, whose records {len, row0, tile0} are read here
  struct Item {
    int kind, b, g, row0, t0, nt;
    int len, srow0, tile0, count;
  };
  auto item_at = [&](int i, int k) -> Item {  // item i, the k-th of this CTA
    const int4 it = k < kCtaItems ? s_items[k] : items[i];
    const int4 sq = k < kCtaItems ? s_seq[k] : item_seq(it);
    Item r;
    r.kind = it.x;
    r.b = it.y / Hkv;
    r.g = it.y % Hkv;
    r.row0 = it.z;
    r.t0 = it.w >> 16;
    r.nt = (it.w & 0xffff) - r.t0;
    r.len = sq.x;
    r.srow0 = sq.y;
    r.tile0 = sq.z;
    r.count = sq.w;
    return r;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int k = 0, ug = 0, kv_issued = 0;
      bool ok = true;
      for (int i = blockIdx.x; ok && i < n_items;
           ++k, i = snake_item(k, static_cast<int>(gridDim.x))) {
        const Item it = item_at(i, k);
        const int kb = k % KVB;
        if (k >= KVB && !mbar_wait(&kv_empty[kb], ((k / KVB) - 1) & 1, status)) {
          ok = false;
          break;
        }
        const bool keep = it.kind == kItemKeep;
        // keep tiles: the sequence's gathered rows in plane g of the
        // workspace; dense tiles: rows of the sequence in its kv plane
        const int plane = keep ? it.g : geo.kvplane(it.b, it.g);
        const int krow = keep ? it.tile0 * 128 + it.row0 : it.srow0 + it.row0;
        uint8_t* sK = smem + C::OFF_KV + kb * 2 * C::TILE;
        uint8_t* sV = sK + C::TILE;
        mbar_arrive_expect_tx(&kv_full[kb], 2 * C::TILE);
        for (int c = 0; c < C::DCH; ++c) {
          tma_load_3d(sK + c * kChunk, keep ? &tm_kk : &tm_k, &kv_full[kb], 64 * c, krow, plane);
          tma_load_3d(sV + c * kChunk, keep ? &tm_vk : &tm_v, &kv_full[kb], 64 * c, krow, plane);
        }
        kv_issued = k + 1;
        const int nU = G * it.nt;
        for (int u = 0; u < nU; ++u) {
          const int st = ug % NST;
          if (ug >= NST && !mbar_wait(&qd_empty[st], ((ug / NST) - 1) & 1, status)) {
            ok = false;
            break;
          }
          ++ug;  // counts issued Q/dO tiles
          const int h = it.g * G + u / it.nt, t = it.t0 + u % it.nt;
          const int plane_q = geo.qplane(it.b, h);
          mbar_arrive_expect_tx(&qd_full[st], 2 * C::TILE + 128 * 8);
          bulk_g2s(smem + C::OFF_STAT + st * 1024,
                   stats + ((size_t)h * geo.TT + it.tile0 + t) * 128, 1024, &qd_full[st]);
          for (int c = 0; c < C::DCH; ++c) {
            tma_load_3d(smem + C::OFF_Q + st * C::TILE + c * kChunk, &tm_q, &qd_full[st],
                        64 * c, it.srow0 + t * 128, plane_q);
            tma_load_3d(smem + C::OFF_DO + st * C::TILE + c * kChunk, &tm_do, &qd_full[st],
                        64 * c, it.srow0 + t * 128, plane_q);
          }
        }
      }
      if (!ok) {
        // after a failed wait, let the copies still in flight land before
        // the CTA's shared memory goes away (on the normal path the MMA
        // thread has consumed every one of them)
        for (int x = max(0, kv_issued - KVB); x < kv_issued; ++x)
          mbar_wait(&kv_full[x % KVB], (x / KVB) & 1, status);
        for (int x = max(0, ug - NST); x < ug; ++x)
          mbar_wait(&qd_full[x % NST], (x / NST) & 1, status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The unit of work is a half-tile: the 64 query columns h of one query
    // tile u against the item's 128 keys, half-tile j = 2u + h of the CTA.
    // It lives in TMEM buffer x = j % NHB: S^T at columns [128x, 128x+64),
    // dP^T at [128x+64, 128x+128); the elementwise warpgroup h overwrites
    // them with P^T and dS^T (packed bf16), which the dV / dK products then
    // read from TMEM.  Order: S/dP of the first NHB half-tiles, then per
    // half-tile j: dV/dK(j), S/dP(j+NHB) -- the two warpgroups' chains
    // interleave on the tensor pipe.
    // The whole warp runs this loop; the elected lane issues.
    {
      const bool leader = elect_one();
      constexpr uint32_t idesc_sd = idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t idesc_acc = idesc_bf16_f32(128, D, false, true);
      const uint32_t q_base = smem_u32(smem + C::OFF_Q), do_base = smem_u32(smem + C::OFF_DO);
      // a cursor over the CTA's half-tiles: item i (k-th of this CTA), query
      // iteration u (global count ug), half h
      struct Cur {
        int i, k, u, ug, h, nU;
        Item it;
      };
      auto cur_load = [&](Cur& c) {
        if (c.i < n_items) {
          c.it = item_at(c.i, c.k);
          c.nU = G * c.it.nt;
        }
      };
      auto cur_next = [&](Cur& c) {
        if (++c.h < 2) return;
        c.h = 0;
        ++c.ug;
        if (++c.u < c.nU) return;
        c.u = 0;
        ++c.k;
        c.i = snake_item(c.k, static_cast<int>(gridDim.x));
        cur_load(c);
      };
      // descriptors of the operand bases, advanced by constant offsets
      const uint64_t dsc_kv = sdesc_sw128(smem_u32(smem + C::OFF_KV), 16, 1024);
      const uint64_t dsc_q = sdesc_sw128(q_base, 16, 1024);
      const uint64_t dsc_do = sdesc_sw128(do_base, 16, 1024);
      const uint64_t dsc_q_mn = sdesc_sw128(q_base, kChunk, 1024);
      const uint64_t dsc_do_mn = sdesc_sw128(do_base, kChunk, 1024);
      auto issue_sd = [&](const Cur& c) -> bool {  // S^T / dP^T of half-tile c
        const int kb = c.k % KVB, st = c.ug % NST;
        if (c.u == 0 && c.h == 0) {
          if (!mbar_wait_warp(&kv_full[kb], (c.k / KVB) & 1, status)) return false;
        }
        if (c.h == 0) {
          if (!mbar_wait_warp(&qd_full[st], (c.ug / NST) & 1, status)) return false;
        }
        tc_fence_after();
        const uint64_t dk = dsc_kv + ((kb * 2 * C::TILE) >> 4), dv = dk + (C::TILE >> 4);
        const uint64_t qo = (st * C::TILE + 8192 * c.h) >> 4;  // query rows 64h .. 64h+63
        const uint64_t dq = dsc_q + qo, ddo = dsc_do + qo;
        const int hb = (2 * c.ug + c.h) % NHB;  // the half-tile's TMEM buffer
        const uint32_t tb = tmem + 128 * hb;
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * kChunk + (kk & 3) * 32) >> 4;
            umma_bf16_ss(tb, dk + off, dq + off, idesc_sd, kk > 0);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * kChunk + (kk & 3) * 32) >> 4;
            umma_bf16_ss(tb + 64, dv + off, ddo + off, idesc_sd, kk > 0);
          }
          umma_commit(&sd_full[hb]);
        }
        __syncwarp();
        return true;
      };
      Cur cs{static_cast<int>(blockIdx.x), 0, 0, 0, 0, 0, Item{}};  // next S/dP to issue
      cur_load(cs);
      Cur ca = cs;  // next dV/dK to issue
      bool ok = true;
      // S/dP run up to NHB half-tiles ahead of dV/dK, but not into an item
      // whose K/V buffer the current item still holds
      int ahead = 0;
      auto top_up = [&]() -> bool {
        while (ahead < NHB && cs.i < n_items && cs.k < ca.k + KVB) {
          if (!issue_sd(cs)) return false;
          cur_next(cs);
          ++ahead;
        }
        return true;
      };
      ok = top_up();
      while (ok && ca.i < n_items) {
        const int ab = ca.k % ACB, st = ca.ug % NST, kb = ca.k % KVB;
        if (ca.u == 0 && ca.h == 0 && ca.k >= ACB) {
          // the epilogue has drained this accumulator buffer
          if (!(ok = mbar_wait_warp(&acc_empty[ab], ((ca.k / ACB) - 1) & 1, status))) break;
        }
        const int ja = 2 * ca.ug + ca.h, hb = ja % NHB;
        if (!(ok = mbar_wait_warp(&ps_full[hb], (ja / NHB) & 1, status))) break;
        tc_fence_after();
        const uint32_t tb = tmem + 128 * hb;
        const uint32_t tm_dv = tmem + C::TM_ACC + ab * 2 * D, tm_dk = tm_dv + D;
        const uint64_t qo = (st * C::TILE + 8192 * ca.h) >> 4;
        const uint64_t ddo = dsc_do_mn + qo, dq = dsc_q_mn + qo;
        const uint32_t first = (ca.u > 0 || ca.h > 0) ? 1u : 0u;
        const bool last_h = ca.h == 1, last_u = ca.u + 1 == ca.nU;
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // 16 queries per step
            const uint32_t acc = kk > 0 ? 1u : first;
            umma_bf16_ts(tm_dv, tb + 8 * kk, ddo + ((kk * 2048) >> 4), idesc_acc, acc);
            umma_bf16_ts(tm_dk, tb + 64 + 8 * kk, dq + ((kk * 2048) >> 4), idesc_acc, acc);
          }
          if (last_h) umma_commit(&qd_empty[st]);  // Q / dO / stats of this tile are done
          if (last_h && last_u) {
            umma_commit(&kv_empty[kb]);  // every MMA reading this item's K and V is issued
            umma_commit(&acc_full[ab]);
          }
        }
        __syncwarp();
        cur_next(ca);
        --ahead;
        if (!(ok = top_up())) break;
      }
      // every MMA issued by the leader completes before TMEM is released
      if (leader) umma_commit(&mma_final);
      __syncwarp();
      mbar_wait_warp(&mma_final, 0, status);
    }
  } else {
    // ---------------------------------------------------------- elementwise
    // Warpgroup `half` owns query columns [64 half, 64 half + 64) of every
    // query tile: warps 2-5 half 0, warps 6-9 half 1 (warp w reads TMEM
    // lanes 32*(w%4)..).  In the epilogue the first writes dV, the second dK.
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quad * 32 + lane;  // key row of the tile
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tl = tmem + lane_base;
    // accumulators of item k -> global memory (half 0 dV, half 1 dK)
    struct Epi {
      int k;
      long long rm;  // 4 * row + mode: mode 1 keep-accumulator row, mode 2 output row
    };
    const float osc = half ? scale : 1.f;
    auto epilogue = [&](const Epi& e) -> bool {
      const int ab = e.k % ACB;
      if (!mbar_wait(&acc_full[ab], (e.k / ACB) & 1, status)) return false;
      tc_fence_after();
      const uint32_t tm_acc = tmem + C::TM_ACC + ab * 2 * D + half * D;
      const int mode = static_cast<int>(e.rm & 3);
      const size_t row = static_cast<size_t>(e.rm >> 2);
      float* accr = (half ? dk_keep : dv_keep) + row * D;
      __nv_bfloat16* outr = (half ? dk : dv) + row * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t vb[32];
        tmem_ld32(tm_acc + lane_base + c0, vb);
        tmem_ld_wait();
        if (mode == 1) {
#pragma unroll
          for (int x = 0; x < 32; x += 4)
            red_add_v4(accr + c0 + x, __uint_as_float(vb[x]), __uint_as_float(vb[x + 1]),
                       __uint_as_float(vb[x + 2]), __uint_as_float(vb[x + 3]));
        } else if (mode == 2) {
#pragma unroll
          for (int x = 0; x < 32; x += 8) {
            uint4 ov;
            ov.x = pack_bf16x2(__uint_as_float(vb[x]) * osc, __uint_as_float(vb[x + 1]) * osc);
            ov.y = pack_bf16x2(__uint_as_float(vb[x + 2]) * osc, __uint_as_float(vb[x + 3]) * osc);
            ov.z = pack_bf16x2(__uint_as_float(vb[x + 4]) * osc, __uint_as_float(vb[x + 5]) * osc);
            ov.w = pack_bf16x2(__uint_as_float(vb[x + 6]) * osc, __uint_as_float(vb[x + 7]) * osc);
            *reinterpret_cast<uint4*>(outr + c0 + x) = ov;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[ab]);
      return true;
    };
    constexpr bool kDeferEpi = ACB >= 2;
    Epi pe{};
    bool pend = false;
    int k = 0, ug = 0;
    bool ok = true;
    for (int i = blockIdx.x; ok && i < n_items;
         ++k, i = snake_item(k, static_cast<int>(gridDim.x))) {
      const Item it = item_at(i, k);
      const bool keep = it.kind == kItemKeep;
      const int len = it.len;
      const int count = it.count;
      const int32_t* blocks = idx.blocks + (size_t)it.b * T * 4;
      const int j = it.row0 + r;  // KEEP: keep index; DENSE: key position
      // a dense row's keep bit and keep prefix (from the staged keep bits of
      // the key tile when the item is staged)
      const bool dense_row = !keep && j < len;
      uint32_t kbw = 0u;
      int kpre = 0;
      if (dense_row) {
        if (k < kCtaItems) {
          const uint32_t* wb = reinterpret_cast<const uint32_t*>(&s_kbits[k]);
          kpre = s_kpre[k];
#pragma unroll
          for (int q = 0; q < 3; ++q)
            if (q < (r >> 5)) kpre += __popc(wb[q]);
          kbw = wb[r >> 5];
          kpre += __popc(kbw & ((1u << (j & 31)) - 1u));
        } else {
          kbw = idx.keep_bits[(size_t)it.b * hdr.nwords + (j >> 5)];
          kpre = idx.keep_prefix[(size_t)it.b * (L + 1) + j];
        }
      }
      const bool keep_j = (kbw >> (j & 31)) & 1u;
      // this item's epilogue: KEEP rows and DENSE keep tokens add into the
      // fp32 keep accumulators (written to dK/dV by the dQ kernel);
      // other DENSE rows are final
      Epi e;
      e.k = k;
      {
        const bool to_acc = keep ? (j < count) : (j < len && keep_j);
        const bool to_out = !keep && j < len && !keep_j;
        const int kidx = keep ? j : (keep_j ? kpre : 0);
        const long long acc_row = ((long long)it.g * geo.TT + it.tile0) * 128 + kidx;
        const long long out_row = (long long)geo.kvplane(it.b, it.g) * geo.R + it.srow0 + j;
        e.rm = to_acc ? ((acc_row << 2) | 1) : to_out ? ((out_row << 2) | 2) : 0;
      }
      const int nU = G * it.nt;
      // a kv group with full causal attention: records for a window n >= len
      const bool full = group_full(full_groups, it.g);
      const int n_w = full ? len : n_win;
      auto record = [&](int t2) {
        return full ? full_block_record(t2, len) : *reinterpret_cast<const int4*>(blocks + 4 * t2);
      };
      int4 blk_next = k < kCtaItems ? s_blk0[k] : record(it.t0);
      for (int u = 0; u < nU; ++u) {
        const int ugl = ug + u;
        const int t = it.t0 + u % it.nt;
        const int i0 = t * 128;
        const int4 blk = blk_next;  // loaded one iteration ahead
        if (u + 1 < nU) blk_next = record(it.t0 + (u + 1) % it.nt);
        // visible query columns of this row among the half's 64, as 2 words
        uint32_t vm[2];
        {
          const int c_end = min(128, len - i0);  // query rows past len are padding
          int c_lo = 0, c_hi = 0;
          if (keep) {
            if (j < blk.x && j < count) c_hi = c_end;  // gathered by this query tile
          } else if (j >= blk.y && j < blk.z && j < len) {
            c_lo = j - i0;
            c_hi = keep_j ? c_end : min(c_end, j + n_w - i0);
          }
          vm[0] = range_bits(c_lo, c_hi, 2 * half);
          vm[1] = range_bits(c_lo, c_hi, 2 * half + 1);
        }
        const int jh = 2 * ugl + half, hb = jh % NHB;  // this half-tile's TMEM buffer
        const uint32_t tb = tl + 128 * hb;
        if (!mbar_wait(&sd_full[hb], (jh / NHB) & 1, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // the query tile's (-LSE log2, -Delta) arrived with its Q / dO tiles
        const int stg = ugl % NST;
        if (!mbar_wait(&qd_full[stg], (ugl / NST) & 1, status)) {
          ok = false;
          break;
        }
        const float4* sst =
            reinterpret_cast<const float4*>(smem + C::OFF_STAT + stg * 1024) + 32 * half;
        // four chunks of 16 columns; the next chunk's S^T and dP^T loads are
        // in flight while this one is computed (a wait covers every load
        // issued before it)
        uint32_t sa[16], da[16], sb[16], db[16];
        tmem_ld16(tb, sa);
        tmem_ld16(tb + 64, da);
        tmem_ld_wait();
        tmem_regs_ready16(sa);
        tmem_regs_ready16(da);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t* sr = (cc & 1) ? sb : sa;
          uint32_t* dr = (cc & 1) ? db : da;
          uint32_t* sn = (cc & 1) ? sa : sb;
          uint32_t* dn = (cc & 1) ? da : db;
          if (cc < 3) {
            tmem_ld16(tb + 16 * (cc + 1), sn);
            tmem_ld16(tb + 64 + 16 * (cc + 1), dn);
          }
          uint32_t pk[8], dk2[8];
          const uint32_t w = (vm[cc >> 1] >> (16 * (cc & 1))) & 0xffffu;
          const bool full = __all_sync(0xffffffffu, w == 0xffffu);
#pragma unroll
          for (int x = 0; x < 16; x += 2) {
            const float4 st2 = sst[8 * cc + x / 2];  // columns (x, x+1): (-lse, -delta)
            float a0, a1, d0, d1;
            ffma2(a0, a1, __uint_as_float(sr[x]), __uint_as_float(sr[x + 1]), scale_log2,
                  scale_log2, st2.x, st2.z);
            float p0 = fast_exp2(a0), p1 = fast_exp2(a1);
            if (!full) {
              p0 = ((w >> x) & 1u) ? p0 : 0.f;
              p1 = ((w >> (x + 1)) & 1u) ? p1 : 0.f;
            }
            ffma2(d0, d1, __uint_as_float(dr[x]), __uint_as_float(dr[x + 1]), 1.f, 1.f, st2.y,
                  st2.w);
            fmul2(d0, d1, p0, p1, d0, d1);
            pk[x / 2] = pack_bf16x2(p0, p1);
            dk2[x / 2] = pack_bf16x2(d0, d1);
          }
          // P^T over S^T, dS^T over dP^T: chunk cc lands on columns
          // [8cc, 8cc+8) of each, which earlier chunks' loads already read
          tmem_st8(tb + 8 * cc, pk);
          tmem_st8(tb + 64 + 8 * cc, dk2);
          if (cc < 3) {
            tmem_ld_wait();
            tmem_regs_ready16(sn);
            tmem_regs_ready16(dn);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&ps_full[hb]);
      }
      if (!ok) break;
      ug += nU;
      // with two accumulator buffers the epilogue of item k runs after the
      // half-tiles of item k + 1, whose S / dP products overlap it
      if (kDeferEpi) {
        if (pend && !(ok = epilogue(pe))) break;
        pe = e;
        pend = true;
      } else if (!(ok = epilogue(e))) {
        break;
      }
    }
    if (kDeferEpi && ok && pend) epilogue(pe);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TM_COLS);
}

// ---------------------------------------------------------------------------
// Query-major dQ, persistent: items are (batch, q head, query tile), longest
// query tiles first, taken round-robin by one CTA per SM.
// ---------------------------------------------------------------------------
template <int D>
struct DqCfg {
  static constexpr int DCH = D / 64;
  static constexpr int TILE = DCH * kChunk;
  static constexpr int QB = D == 64 ? 2 : 1;    // Q/dO tile buffers
  static constexpr int NST = D == 64 ? 3 : 2;   // K/V ring stages
  static constexpr int OFF_QD = 0;              // [QB][Q, dO]
  static constexpr int OFF_K = OFF_QD + QB * 2 * TILE;
  static constexpr int OFF_V = OFF_K + NST * TILE;
  static constexpr int OFF_DS = OFF_V + NST * TILE;
  static constexpr int SMEM = OFF_DS + 2 * kChunk + 1024;
  static constexpr int TM_S = 0, TM_DP = 128, TM_DQ = 256;  // dQ buffer b at +bD
  static constexpr int TM_COLS = 512;
  // block and sequence records of the CTA's first ITEMS items, in static
  // shared memory
  static constexpr int ITEMS = D == 64 ? 128 : 48;
  static_assert(SMEM + 32 * ITEMS + 256 <= 227 * 1024, "shared memory");
  static_assert(TM_DQ + 2 * D <= TM_COLS, "tensor memory");
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_persistent(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_do,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_kk,
                      const __grid_constant__ CUtensorMap tm_vk, IndexPtrs idx,
                      const float2* __restrict__ stats, const BwdSchedule* __restrict__ sched,
                      const float4* __restrict__ dk_keep, const float4* __restrict__ dv_keep,
                      __nv_bfloat16* __restrict__ dq, __nv_bfloat16* __restrict__ dk,
                      __nv_bfloat16* __restrict__ dv, Geom geo, float scale,
                      float scale_log2, uint64_t full_groups, int* status) {
  using C = DqCfg<D>;
  constexpr int QB = C::QB, NST = C::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t qd_full[QB], qd_empty[QB], kv_full[NST], kv_empty[NST];
  __shared__ __align__(8) uint64_t sd_full, sd_free, ds_full, dq_done, acc_full[2], acc_empty[2],
      mma_final;
  __shared__ uint32_t tmem_slot;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = geo.T, B = geo.B, Hq = geo.Hq, Hkv = geo.Hkv;
  const int n_items = B * Hq * T;

  if (threadIdx.x == 0) {
    for (int i = 0; i < QB; ++i) {
      mbar_init(&qd_full[i], 1);
      mbar_init(&qd_empty[i], 1);
    }
    for (int i = 0; i < NST; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEwThreads);
    }
    mbar_init(&sd_full, 1);
    mbar_init(&sd_free, kEwThreads);
    mbar_init(&ds_full, kEwThreads);
    mbar_init(&dq_done, 1);
    mbar_init(&mma_final, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, C::TM_COLS);
    tmem_relinquish();
  }
  // barriers and tensor memory are set up before waiting for the dK/dV kernel
  grid_dep_wait();
  const IndexHeader hdr = *idx.header;
  if (!header_matches(hdr, geo)) {
    if (threadIdx.x == 0) report(status, SEP_ERR_DEVICE_BOUNDS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_slot, C::TM_COLS);
    return;
  }
  const int n_win = hdr.n;
  // block and sequence records of this CTA's items (i = snake_item(x,
  // gridDim.x)), read once; items past C::ITEMS read theirs from global memory
  __shared__ int4 s_blk[C::ITEMS], s_seq[C::ITEMS];
  for (int x = threadIdx.x; x < C::ITEMS; x += blockDim.x) {
    const int i = snake_item(x, static_cast<int>(gridDim.x));
    if (i < n_items) {
      const int bh = i % (B * Hq);
      s_blk[x] = *reinterpret_cast<const int4*>(idx.blocks +
                                                ((size_t)(bh / Hq) * T + (T - 1 - i / (B * Hq))) * 4);
      s_seq[x] = *reinterpret_cast<const int4*>(idx.seq + bh / Hq);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  // Items are (sequence, q head, query tile), longest tiles first.  Tiles
  // past the end of their sequence (a pack's shorter sequences) are empty and
  // skipped by every role; only live items advance the buffer counters.
  struct Item {
    int b, h, g, t, n_gather, lo, hi, nG, nT;
    int len, srow0, tile0;
    bool ok, full, empty;
  };
  auto item_at = [&](int i, int x) -> Item {  // item i, the x-th of this CTA
    Item r;
    r.t = T - 1 - i / (B * Hq);
    const int bh = i % (B * Hq);
    r.b = bh / Hq;
    r.h = bh % Hq;
    r.g = r.h / (Hq / Hkv);
    const int4 sq = x < C::ITEMS ? s_seq[x] : *reinterpret_cast<const int4*>(idx.seq + r.b);
    SeqRec sr;
    sr.len = sq.x; sr.row0 = sq.y; sr.tile0 = sq.z; sr.pad = 0;
    r.len = sr.len;
    r.srow0 = sr.row0;
    r.tile0 = sr.tile0;
    const bool sok = seq_ok(sr, geo);
    r.empty = sok && r.t * 128 >= sr.len;
    r.full = group_full(full_groups, r.g);  // full causal attention: records for n >= len
    const int4 blk = r.full ? full_block_record(r.t, sr.len)
                     : x < C::ITEMS
                         ? s_blk[x]
                         : *reinterpret_cast<const int4*>(idx.blocks + ((size_t)r.b * T + r.t) * 4);
    r.n_gather = blk.x;
    r.lo = blk.y;
    r.hi = blk.z;
    const int q0 = r.t * 128;
    r.ok = sok && !r.empty &&
           !(blk.x < 0 || blk.x > blk.y || blk.y < 0 || blk.y > q0 || blk.z <= q0 ||
             blk.z > sr.len);
    r.nG = r.ok ? (blk.x + 127) >> 7 : 0;
    r.nT = r.ok ? r.nG + ((blk.z - blk.y + 127) >> 7) : 0;
    return r;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int k = 0, ug = 0, qd_issued = 0;  // k: live items so far
      bool ok = true;
      for (int i = blockIdx.x, ix = 0; ok && i < n_items;
           ++ix, i = snake_item(ix, static_cast<int>(gridDim.x))) {
        const Item it = item_at(i, ix);
        if (it.empty) continue;
        if (!it.ok) {
          report(status, SEP_ERR_DEVICE_BOUNDS);
          ok = false;
          break;
        }
        const int qb = k % QB;
        if (k >= QB && !mbar_wait(&qd_empty[qb], ((k / QB) - 1) & 1, status)) {
          ok = false;
          break;
        }
        const int plane_q = geo.qplane(it.b, it.h), plane_kv = geo.kvplane(it.b, it.g);
        const int qrow = it.srow0 + it.t * 128;
        uint8_t* sQ = smem + C::OFF_QD + qb * 2 * C::TILE;
        mbar_arrive_expect_tx(&qd_full[qb], 2 * C::TILE);
        for (int c = 0; c < C::DCH; ++c) {
          tma_load_3d(sQ + c * kChunk, &tm_q, &qd_full[qb], 64 * c, qrow, plane_q);
          tma_load_3d(sQ + C::TILE + c * kChunk, &tm_do, &qd_full[qb], 64 * c, qrow, plane_q);
        }
        qd_issued = k + 1;
        for (int u = 0; u < it.nT; ++u) {
          const int st = ug % NST;
          if (ug >= NST && !mbar_wait(&kv_empty[st], ((ug / NST) - 1) & 1, status)) {
            ok = false;
            break;
          }
          ++ug;  // counts issued K/V tiles
          const bool gat = u < it.nG;
          // gathered tiles: the sequence's keep rows in plane g of the
          // workspace; band tiles: rows of the sequence in its kv plane
          const int row = gat ? 128 * (it.tile0 + u) : it.srow0 + it.lo + 128 * (u - it.nG);
          const int plane = gat ? it.g : plane_kv;
          mbar_arrive_expect_tx(&kv_full[st], 2 * C::TILE);
          for (int c = 0; c < C::DCH; ++c) {
            tma_load_3d(smem + C::OFF_K + st * C::TILE + c * kChunk, gat ? &tm_kk : &tm_k,
                        &kv_full[st], 64 * c, row, plane);
            tma_load_3d(smem + C::OFF_V + st * C::TILE + c * kChunk, gat ? &tm_vk : &tm_v,
                        &kv_full[st], 64 * c, row, plane);
          }
        }
        ++k;
      }
      if (!ok) {
        // after a failed wait, let the copies still in flight land
        for (int x = max(0, qd_issued - QB); x < qd_issued; ++x)
          mbar_wait(&qd_full[x % QB], (x / QB) & 1, status);
        for (int x = max(0, ug - NST); x < ug; ++x)
          mbar_wait(&kv_full[x % NST], (x / NST) & 1, status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop; the elected lane issues.
    {
      const bool leader = elect_one();
      constexpr uint32_t idesc_ss = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_acc = idesc_bf16_f32(128, D, false, true);
      const uint32_t k_base = smem_u32(smem + C::OFF_K), v_base = smem_u32(smem + C::OFF_V),
                     ds_base = smem_u32(smem + C::OFF_DS);
      int k = 0, ug = 0;  // k: live items so far
      bool ok = true;
      for (int i = blockIdx.x, ix = 0; ok && i < n_items;
           ++ix, i = snake_item(ix, static_cast<int>(gridDim.x))) {
        const Item it = item_at(i, ix);
        if (it.empty) continue;
        if (!it.ok) break;
        const int qb = k % QB, ab = k & 1;
        const uint32_t q_base = smem_u32(smem + C::OFF_QD + qb * 2 * C::TILE);
        const uint32_t do_base = q_base + C::TILE;
        const uint32_t tm_dq = tmem + C::TM_DQ + ab * D;
        if (!mbar_wait_warp(&qd_full[qb], (k / QB) & 1, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        auto issue_sdp = [&](int ugl) -> bool {
          const int st = ugl % NST;
          if (!mbar_wait_warp(&kv_full[st], (ugl / NST) & 1, status)) return false;
          tc_fence_after();
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
              umma_bf16_ss(tmem + C::TM_S, sdesc_sw128(q_base + off, 16, 1024),
                           sdesc_sw128(k_base + st * C::TILE + off, 16, 1024), idesc_ss, kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
              umma_bf16_ss(tmem + C::TM_DP, sdesc_sw128(do_base + off, 16, 1024),
                           sdesc_sw128(v_base + st * C::TILE + off, 16, 1024), idesc_ss, kk > 0);
            }
            umma_commit(&sd_full);
          }
          __syncwarp();
          return true;
        };
        if (ug > 0 && !mbar_wait_warp(&sd_free, (ug - 1) & 1, status)) {
          ok = false;
          break;
        }
        if (!issue_sdp(ug)) {
          ok = false;
          break;
        }
        if (k >= 2 && !mbar_wait_warp(&acc_empty[ab], ((k >> 1) - 1) & 1, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int u = 0; ok && u < it.nT; ++u) {
          const int ugl = ug + u;
          if (u + 1 < it.nT) {
            ok = mbar_wait_warp(&sd_free, ugl & 1, status) && issue_sdp(ugl + 1);
            if (!ok) break;
          }
          if (!mbar_wait_warp(&ds_full, ugl & 1, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int st = ugl % NST;
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t aoff = (kk >> 2) * kChunk + (kk & 3) * 32;
              umma_bf16_ss(tm_dq, sdesc_sw128(ds_base + aoff, 16, 1024),
                           sdesc_sw128(k_base + st * C::TILE + kk * 2048, kChunk, 1024),
                           idesc_acc, (u > 0 || kk > 0) ? 1u : 0u);
            }
            umma_commit(&dq_done);
            umma_commit(&kv_empty[st]);
            if (u + 1 == it.nT) umma_commit(&qd_empty[qb]);  // Q / dO of this item are done
          }
          __syncwarp();
        }
        if (!ok) break;
        if (leader) umma_commit(&acc_full[ab]);
        ug += it.nT;
        ++k;
      }
      // every MMA issued by the leader completes before TMEM is released
      if (leader) umma_commit(&mma_final);
      mbar_wait_warp(&mma_final, 0, status);
    }
  } else {
    // ---------------------------------------------------------- elementwise
    // First the keep tokens' dK / dV rows from the fp32 accumulators, which
    // the dK/dV kernel has finished: one warp per 16-row unit over every
    // elementwise warp of the grid, only the units below the largest keep
    // count, while the first item's copies and products are in flight.
    {
      const int max_count = min(max(sched->max_count, 0), geo.L);
      const int units = geo.B * Hkv * ((max_count + kKeepUnitRows - 1) / kKeepUnitRows);
      const int nw = static_cast<int>(gridDim.x) * (kEwThreads / 32);
      for (int u = static_cast<int>(blockIdx.x) * (kEwThreads / 32) + (warp - 2); u < units;
           u += nw)
        scatter_keep_unit<D>(idx, geo, dk_keep, dv_keep, dk, dv, scale, u, lane, status);
    }
    // Two warpgroups share every tile: warps 2-5 take key columns 0-63 and
    // warps 6-9 columns 64-127 of the same 128 query rows; in the epilogue
    // each writes half of the dQ columns.
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t* kb_all = idx.keep_bits;
    const int nwords = hdr.nwords;
    uint8_t* sDS = smem + C::OFF_DS;
    int k = 0, ug = 0;  // k: live items so far
    bool ok = true;
    for (int i = blockIdx.x, ix = 0; ok && i < n_items;
           ++ix, i = snake_item(ix, static_cast<int>(gridDim.x))) {
      const Item it = item_at(i, ix);
      if (it.empty) continue;
      if (!it.ok) break;
      const int ab = k & 1;
      const int i_row = it.t * 128 + r;
      const bool row_live = i_row < it.len;
      // (-LSE log2, -Delta) of this row (zero for padding rows)
      const float2 st2 = stats[((size_t)it.h * geo.TT + it.tile0 + it.t) * 128 + r];
      const uint32_t* kbits = kb_all + (size_t)it.b * nwords;
      for (int u = 0; u < it.nT; ++u) {
        const int ugl = ug + u;
        uint32_t vm[2];
        if (!row_live) {
          vm[0] = vm[1] = 0u;
        } else if (u < it.nG) {
          const int nv = min(128, it.n_gather - 128 * u);
          vm[0] = range_bits(0, nv, 2 * half);
          vm[1] = range_bits(0, nv, 2 * half + 1);
        } else {
          const int jt = it.lo + 128 * (u - it.nG) + 64 * half;  // first key of this half
          const int n_causal = min(64, max(0, i_row - jt + 1));
          const int c_win = i_row - (it.full ? it.len : n_win) + 1 - jt;
          const int wj = jt >> 5, sh = jt & 31;
          uint32_t kw[3];
#pragma unroll
          for (int x = 0; x < 3; ++x) kw[x] = (wj + x < nwords) ? __ldg(kbits + wj + x) : 0u;
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            const uint32_t keepw = sh ? ((kw[w] >> sh) | (kw[w + 1] << (32 - sh))) : kw[w];
            vm[w] = range_bits(0, n_causal, w) & (range_bits(c_win, 64, w) | keepw);
          }
        }
        if (!mbar_wait(&sd_full, ugl & 1, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t dsk[32];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t sr[32], dr[32];
          tmem_ld32(tmem + lane_base + C::TM_S + 64 * half + 32 * cc, sr);
          tmem_ld32(tmem + lane_base + C::TM_DP + 64 * half + 32 * cc, dr);
          tmem_ld_wait();
          const uint32_t w = vm[cc];
          const bool full = __all_sync(0xffffffffu, w == 0xffffffffu);
#pragma unroll
          for (int x = 0; x < 32; x += 2) {
            float a0, a1, d0, d1;
            ffma2(a0, a1, __uint_as_float(sr[x]), __uint_as_float(sr[x + 1]), scale_log2,
                  scale_log2, st2.x, st2.x);
            float p0 = fast_exp2(a0), p1 = fast_exp2(a1);
            if (!full) {
              p0 = ((w >> x) & 1u) ? p0 : 0.f;
              p1 = ((w >> (x + 1)) & 1u) ? p1 : 0.f;
            }
            ffma2(d0, d1, __uint_as_float(dr[x]), __uint_as_float(dr[x + 1]), 1.f, 1.f, st2.y,
                  st2.y);
            fmul2(d0, d1, p0, p1, d0, d1);
            dsk[16 * cc + x / 2] = pack_bf16x2(d0, d1);
          }
        }
        tc_fence_before();
        mbar_arrive(&sd_free);
        if (ugl > 0 && !mbar_wait(&dq_done, (ugl - 1) & 1, status)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int un = 0; un < 8; ++un) {
          const uint32_t off = half * kChunk + sw128_offset(r, un * 8);
          *reinterpret_cast<uint4*>(sDS + off) =
              make_uint4(dsk[4 * un], dsk[4 * un + 1], dsk[4 * un + 2], dsk[4 * un + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&ds_full);
      }
      if (!ok) break;
      ug += it.nT;
      if (!mbar_wait(&acc_full[ab], (k >> 1) & 1, status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tm_dq = tmem + C::TM_DQ + ab * D;
      __nv_bfloat16* qrow =
          dq + ((size_t)geo.qplane(it.b, it.h) * geo.R + it.srow0 + (row_live ? i_row : 0)) * D;
#pragma unroll
      for (int c0 = half * (D / 2); c0 < (half + 1) * (D / 2); c0 += 32) {
        uint32_t qb2[32];
        tmem_ld32(tm_dq + lane_base + c0, qb2);
        tmem_ld_wait();
        if (row_live) {
#pragma unroll
          for (int x = 0; x < 32; x += 8) {
            uint4 pk;
            pk.x = pack_bf16x2(__uint_as_float(qb2[x]) * scale, __uint_as_float(qb2[x + 1]) * scale);
            pk.y = pack_bf16x2(__uint_as_float(qb2[x + 2]) * scale,
                               __uint_as_float(qb2[x + 3]) * scale);
            pk.z = pack_bf16x2(__uint_as_float(qb2[x + 4]) * scale,
                               __uint_as_float(qb2[x + 5]) * scale);
            pk.w = pack_bf16x2(__uint_as_float(qb2[x + 6]) * scale,
                               __uint_as_float(qb2[x + 7]) * scale);
            *reinterpret_cast<uint4*>(qrow + c0 + x) = pk;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[ab]);
      ++k;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TM_COLS);
}

struct BwdWs {
  uint8_t *kk, *vk;
  float *dk_keep, *dv_keep;
  float2* stats;  // [Hq][TT * 128] (-LSE in log2 units, -Delta)
  BwdSchedule* sched;
  int4* items;
  size_t total;
};

BwdWs bwd_ws(void* base, const Geom& geo, int d) {
  BwdWs w;
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  const size_t rows = (size_t)geo.TT * 128;  // rows of one head plane of the tile space
  const size_t kv_bf16 = align_up((size_t)geo.Hkv * rows * d * 2, 256);
  const size_t kv_f32 = align_up((size_t)geo.Hkv * rows * d * 4, 256);
  w.kk = p + off; off += kv_bf16;
  w.vk = p + off; off += kv_bf16;
  w.dk_keep = reinterpret_cast<float*>(p + off); off += kv_f32;
  w.dv_keep = reinterpret_cast<float*>(p + off); off += kv_f32;
  w.stats = reinterpret_cast<float2*>(p + off);
  off += align_up((size_t)geo.Hq * rows * 8, 256);
  w.sched = reinterpret_cast<BwdSchedule*>(p + off); off += 256;
  w.items = reinterpret_cast<int4*>(p + off);
  off += align_up(sizeof(int4) * bwd_max_items(geo.B, geo.Hkv, geo.T), 256);
  w.total = off;
  return w;
}

template <int D>
int launch_bwd_impl(IndexPtrs idx, const void* q, const void* k, const void* v, const void* o,
                    const float* lse, const void* dout, void* dq, void* dk, void* dv,
                    const Geom& geo, float scale, uint64_t full_groups, void* ws, int* status,
                    cudaStream_t s) {
  const BwdWs w = bwd_ws(ws, geo, D);
  const int sms = num_sms();
  profile_mark(0, s);
  {
    // one CTA for the schedule, then a few CTAs per SM for the strided units
    const size_t units = static_cast<size_t>(keep_units(geo.B, geo.Hkv, geo.L)) +
                         (size_t)geo.B * geo.Hq * geo.T * 128 / kPrepRows;
    const size_t want = (units + kPrepThreads / 32 - 1) / (kPrepThreads / 32);
    const int ctas = static_cast<int>(want < (size_t)8 * sms ? want : (size_t)8 * sms);
    const cudaError_t e = launch_dependent(
        bwd_prep_kernel<D>, dim3(ctas + 1), dim3(kPrepThreads), 0, s, idx, geo,
        static_cast<const uint4*>(k), static_cast<const uint4*>(v),
        reinterpret_cast<uint4*>(w.kk), reinterpret_cast<uint4*>(w.vk),
        static_cast<const uint4*>(o), static_cast<const uint4*>(dout), lse, w.stats,
        reinterpret_cast<float4*>(w.dk_keep), reinterpret_cast<float4*>(w.dv_keep), full_groups,
        w.sched, w.items, status);
    if (e != cudaSuccess) return static_cast<int>(e);
  }
  const uint64_t pq = geo.packed ? geo.Hq : (uint64_t)geo.B * geo.Hq;
  const uint64_t pkv = geo.packed ? geo.Hkv : (uint64_t)geo.B * geo.Hkv;
  const uint64_t rk = (uint64_t)geo.TT * 128;
  CUtensorMap mq, mdo, mk, mv, mkk, mvk;
  if (!make_bf16_map(&mq, q, pq, geo.R, D, 128) ||
      !make_bf16_map(&mdo, dout, pq, geo.R, D, 128) ||
      !make_bf16_map(&mk, k, pkv, geo.R, D, 128) || !make_bf16_map(&mv, v, pkv, geo.R, D, 128) ||
      !make_bf16_map(&mkk, w.kk, geo.Hkv, rk, D, 128) ||
      !make_bf16_map(&mvk, w.vk, geo.Hkv, rk, D, 128))
    return static_cast<int>(cudaErrorInvalidValue);
  const float scale_log2 = scale * kLog2e;
  using KC = KvCfg<D>;
  using QC = DqCfg<D>;
  auto kv_k = bwd_kv_persistent<D>;
  auto dq_k = bwd_dq_persistent<D>;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(kv_k, cudaFuncAttributeMaxDynamicSharedMemorySize, KC::SMEM)) ||
      (e = cudaFuncSetAttribute(dq_k, cudaFuncAttributeMaxDynamicSharedMemorySize, QC::SMEM)))
    return static_cast<int>(e);
  __nv_bfloat16* dkb = static_cast<__nv_bfloat16*>(dk);
  __nv_bfloat16* dvb = static_cast<__nv_bfloat16*>(dv);
  profile_mark(1, s);
  e = launch_dependent(kv_k, dim3(sms), dim3(kThreads), KC::SMEM, s, mkk, mvk, mk, mv, mq, mdo,
                       idx, static_cast<const BwdSchedule*>(w.sched),
                       static_cast<const int4*>(w.items), static_cast<const float2*>(w.stats),
                       w.dk_keep, w.dv_keep, dkb, dvb, geo, scale, scale_log2, full_groups,
                       status);
  if (e != cudaSuccess) return static_cast<int>(e);
  profile_mark(2, s);
  // the dQ kernel also writes the keep tokens' dK / dV rows
  const int dq_items = geo.B * geo.Hq * geo.T;
  const cudaError_t err = launch_dependent(
      dq_k, dim3(dq_items < sms ? dq_items : sms), dim3(kThreads), QC::SMEM, s, mq, mdo, mk, mv,
      mkk, mvk, idx, static_cast<const float2*>(w.stats),
      static_cast<const BwdSchedule*>(w.sched), reinterpret_cast<const float4*>(w.dk_keep),
      reinterpret_cast<const float4*>(w.dv_keep), static_cast<__nv_bfloat16*>(dq), dkb, dvb, geo,
      scale, scale_log2, full_groups, status);
  profile_mark(3, s);
  return static_cast<int>(err);
}

}  // namespace

size_t attn_bwd_tc_workspace(const Geom& geo, int d) { return bwd_ws(nullptr, geo, d).total; }

int launch_attn_bwd_tc(IndexPtrs idx, const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dout, void* dq, void* dk, void* dv,
                       const Geom& geo, int d, float scale, uint64_t full_groups, void* ws,
                       int* status, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d == 64)
    return launch_bwd_impl<64>(idx, q, k, v, o, lse, dout, dq, dk, dv, geo, scale, full_groups,
                               ws, status, s);
  return launch_bwd_impl<128>(idx, q, k, v, o, lse, dout, dq, dk, dv, geo, scale, full_groups,
                              ws, status, s);
}

}  // namespace sep
