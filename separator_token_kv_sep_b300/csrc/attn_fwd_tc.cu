// Sep-Attention forward on the tcgen05 tensor cores (bf16 operands, fp32
// accumulation in tensor memory).
//
// What it computes: O = softmax(Q K^T * scale, masked) V and the row LSE
// under the SepLLM mask -- the first a tokens, every preceding separator and
// the n nearest tokens (SepLLM anthology record lit-748, Key takeaways,
// "The mask"; pith.science review, key_machinery).
//
// How: a persistent kernel, one CTA per SM, walks work items of two adjacent
// 128-row query tiles A and B of one (batch, q head).  A tile's keys come
// from two sources, read from the index built by sep_build_index:
//   gathered tiles  the keep tokens before the tile's first window start,
//                   copied densely into K_keep / V_keep by gather_keep_kernel;
//                   the last one is masked by k < n_gather;
//   band tiles      the dense key range [dense_lo, dense_hi), masked per
//                   element by j <= i and (keep[j] or j >= i-n+1).
// A and B walk one K/V stream, the union of their key tiles.
// Warp roles: warp 0 issues TMA loads (each item's two query tiles into one
// of QB buffers, then K and V tiles through an NST-stage ring), warp 1
// issues tcgen05.mma (S_X = Q_X K^T into TMEM, O_X += P_X V with P_X read
// from TMEM), warps 2-5 and 6-9 run the softmax of A and of B, one thread
// per query row: they read S with tcgen05.ld, apply the mask, keep a running
// max (rescaling O in TMEM only when the max grows by more than 2^8, which
// keeps every P <= 256 and the final O / l exact), write P as packed bf16
// over the first half of S, and after the item's last tile normalise O and
// store it with the LSE.  A row's first tile is read twice (its maximum,
// then P); later tiles once, against the running max, with a rescale of the
// part already written when a chunk of the tile exceeds the 2^8 bound.  The next item's query tiles and first S products
// are issued while the current item finishes, so its epilogue overlaps them.
// Every mbarrier wait is bounded; on expiry the kernel records
// SEP_ERR_TIMEOUT, lets its copies and MMAs drain, frees TMEM and returns.
#include "common.cuh"
#include "keep_rows.cuh"
#include "layout.h"
#include "tma_host.h"

namespace sep {

namespace {

constexpr int kChunk = 128 * 128;  // bytes of a [128 rows x 64 cols] bf16 block

// The index header sits at offset 0 of any index buffer: every kernel checks
// it against the call's geometry before using the fields whose offsets
// depend on B and L.
__device__ __forceinline__ bool header_matches(const IndexHeader& h, const Geom& geo) {
  return h.magic == kIndexMagic && h.B == geo.B && h.L == geo.L && h.block_m == 128 &&
         h.packed == geo.packed && h.total == geo.R;
}

template <int D>
__global__ void __launch_bounds__(256)
    gather_keep_kernel(IndexPtrs idx, Geom geo, const uint4* __restrict__ k,
                       const uint4* __restrict__ v, uint4* __restrict__ kk,
                       uint4* __restrict__ vk, int* status) {
  grid_dep_wait();
  const IndexHeader hdr = *idx.header;
  if (!header_matches(hdr, geo)) return;
  const int lane = threadIdx.x & 31;
  const int units = live_keep_units(idx, geo, lane);
  for (int u = blockIdx.x * 8 + (threadIdx.x >> 5); u < units; u += gridDim.x * 8)
    gather_keep_unit<D>(idx, geo, k, v, kk, vk, nullptr, nullptr, u, lane, status);
}

template <int D>
struct FwdCfg {
  static constexpr int DCH = D / 64;
  static constexpr int TILE = DCH * kChunk;  // one [128 x D] bf16 tile
  static constexpr int QB = D == 64 ? 2 : 1;   // query-pair buffers
  static constexpr int NST = D == 64 ? 4 : 2;  // K/V ring stages
  static constexpr int OFF_Q = 0;              // [QB][query tiles A, B]
  static constexpr int OFF_K = OFF_Q + QB * 2 * TILE;
  static constexpr int OFF_V = OFF_K + NST * TILE;
  static constexpr int SMEM = OFF_V + NST * TILE + 1024;
  // tensor memory: per query tile X, S (fp32, 128 columns; P overwrites its
  // first 64 columns as packed bf16) and the O accumulator (D columns)
  static constexpr int TM_S0 = 0, TM_O0 = 128, TM_S1 = 256, TM_O1 = 384;
  static constexpr int TM_COLS = 512;
  static_assert(SMEM + 32 * 64 + 256 <= 227 * 1024, "shared memory (with the item records)");
};

constexpr int kThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-5 softmax A, 6-9 softmax B
constexpr float kRescaleLog2 = 8.0f;
constexpr float kRescaleBound = 256.0f;  // 2^kRescaleLog2

// One work item: query tiles A = 2p and B = 2p + 1 of one (batch, q head).
// Items are numbered longest first (pair index descending, then batch and
// head), and CTA c of a grid of G takes one item per round of G in snake
// order (snake_item): c, 2G - 1 - c, 2G + c, ...
//
// The key tiles an item visits, in order: the gathered keep tiles of the
// longer gathered list, then the dense band from A's window start to B's
// last row.  Tile u is active for X when it holds keys X can see: gathered
// tile u when 128u < n_gather(X); a band tile for A below A's last row, for
// B when it reaches past B's window start.
struct PairPlan {
  int nA, loA, hiA, nB, loB, hiB;  // block records of A and B
  int b, h, tA;
  int len, row0, tile0;  // the sequence: length, first row in its planes, first tile
  bool hasB, valid, empty;
  int nG, nT;  // gathered tiles, total tiles
  __device__ bool active(int u, int x) const {
    if (x == 1 && !hasB) return false;
    if (u < nG) return 128 * u < (x == 0 ? nA : nB);
    const int jt = loA + 128 * (u - nG);
    return x == 0 ? jt < hiA : (jt + 128 > loB && jt < hiB);
  }
  __device__ bool any(int u) const { return active(u, 0) || active(u, 1); }
  // first active tile after u (nT if none)
  __device__ int next(int u) const {
    ++u;
    while (u < nT && !any(u)) ++u;
    return u;
  }
};

constexpr int kCtaItems = 64;  // items whose records a CTA keeps in shared memory

// Records of one item: block records of tiles A and B, and the sequence's.
__device__ __forceinline__ void read_item_records(IndexPtrs idx, const Geom& geo, int item,
                                                  int4& ba, int4& bb, int4& sq) {
  const int P = (geo.T + 1) >> 1, BH = geo.B * geo.Hq;
  const int b = (item % BH) / geo.Hq, tA = 2 * (P - 1 - item / BH);
  ba = *reinterpret_cast<const int4*>(idx.blocks + ((size_t)b * geo.T + tA) * 4);
  bb = tA + 1 < geo.T
           ? *reinterpret_cast<const int4*>(idx.blocks + ((size_t)b * geo.T + tA + 1) * 4)
           : ba;
  sq = *reinterpret_cast<const int4*>(idx.seq + b);
}

// Records of the CTA's k-th item, from shared memory for the first
// kCtaItems items.
__device__ __forceinline__ void item_records(IndexPtrs idx, const int4* s_rec, int item,
                                             const Geom& geo, int4& ba, int4& bb, int4& sq) {
  const int k = item / static_cast<int>(gridDim.x);  // the round, = the CTA's k-th item
  if (k < kCtaItems) {
    ba = s_rec[3 * k];
    bb = s_rec[3 * k + 1];
    sq = s_rec[3 * k + 2];
    return;
  }
  read_item_records(idx, geo, item, ba, bb, sq);
}

// The plan of one item.  Items whose pair of tiles starts past the end of
// their sequence are empty (a pack's shorter sequences) and are skipped by
// every role; items with inconsistent records are invalid (reported by the
// TMA producer, skipped by every role).
__device__ __forceinline__ PairPlan load_plan(IndexPtrs idx, const int4* s_rec, int item,
                                              int n_items, const Geom& geo,
                                              uint64_t full_groups, int grp) {
  PairPlan pl;
  pl.valid = false;
  pl.empty = true;
  pl.nT = 0;
  if (item >= n_items) return pl;
  const int P = (geo.T + 1) >> 1, BH = geo.B * geo.Hq;
  const int pair = P - 1 - item / BH, bh = item % BH;
  pl.b = bh / geo.Hq;
  pl.h = bh % geo.Hq;
  pl.tA = 2 * pair;
  int4 ba, bb, sq;
  item_records(idx, s_rec, item, geo, ba, bb, sq);
  SeqRec sr;
  sr.len = sq.x; sr.row0 = sq.y; sr.tile0 = sq.z; sr.pad = 0;
  pl.len = sr.len; pl.row0 = sr.row0; pl.tile0 = sr.tile0;
  if (!seq_ok(sr, geo)) {
    pl.empty = false;  // invalid, not empty: reported
    return pl;
  }
  if (pl.tA * 128 >= pl.len) return pl;  // empty
  pl.empty = false;
  const int len = pl.len;
  pl.hasB = pl.tA * 128 + 128 < len;
  if (group_full(full_groups, pl.h / grp)) {
    ba = full_block_record(pl.tA, len);
    bb = full_block_record(pl.tA + 1, len);
  }
  pl.nA = ba.x; pl.loA = ba.y; pl.hiA = ba.z;
  pl.nB = bb.x; pl.loB = bb.y; pl.hiB = bb.z;
  auto bad = [&](int4 r, int q0) {
    return r.x < 0 || r.x > r.y || r.y < 0 || r.y > q0 || r.z <= q0 || r.z > len;
  };
  pl.valid = !(bad(ba, pl.tA * 128) ||
               (pl.hasB && (bad(bb, pl.tA * 128 + 128) || bb.x < ba.x || bb.y < ba.y)));
  if (pl.valid) {
    pl.nG = ((pl.hasB ? pl.nB : pl.nA) + 127) >> 7;
    pl.nT = pl.nG + (((pl.hasB ? pl.hiB : pl.hiA) - pl.loA + 127) >> 7);
  }
  return pl;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_kk,
                       const __grid_constant__ CUtensorMap tm_vk, IndexPtrs idx,
                       __nv_bfloat16* __restrict__ o, float* __restrict__ lse, Geom geo,
                       float scale_log2, uint64_t full_groups, int* status) {
  using C = FwdCfg<D>;
  constexpr int QB = C::QB, NST = C::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t q_full[QB], q_empty[QB], kv_full[NST], kv_empty[NST],
      s_full[2], p_full[2], o_done[2], mma_final;
  __shared__ uint32_t tmem_slot;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = geo.T;
  const int Hq = geo.Hq;
  const int n_items = geo.B * Hq * ((T + 1) >> 1);
  const int G = gridDim.x;
  const int grp = Hq / geo.Hkv;

  if (threadIdx.x == 0) {
    for (int s = 0; s < QB; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < NST; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 128);
      mbar_init(&o_done[x], 1);
    }
    mbar_init(&mma_final, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, C::TM_COLS);
    tmem_relinquish();
  }
  // barriers and tensor memory are set up before waiting for the keep gather
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
  // records of this CTA's items (item = snake_item(k, G)), read once
  __shared__ int4 s_rec[3 * kCtaItems];
  for (int x = threadIdx.x; x < kCtaItems; x += blockDim.x) {
    const int item = snake_item(x, G);
    if (item < n_items) read_item_records(idx, geo, item, s_rec[3 * x], s_rec[3 * x + 1],
                                          s_rec[3 * x + 2]);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_kk);
      tma_prefetch_desc(&tm_vk);
      int n = 0, kq = 0;  // K/V stages and query pairs loaded
      bool ok = true;
      for (int it = blockIdx.x; ok && it < n_items; it = snake_item(it / G + 1, G)) {
        const PairPlan pl = load_plan(idx, s_rec, it, n_items, geo, full_groups, grp);
        if (!pl.valid) {
          if (!pl.empty) report(status, SEP_ERR_DEVICE_BOUNDS);
          continue;
        }
        const int qs = kq % QB;
        if (kq >= QB && !mbar_wait(&q_empty[qs], ((kq / QB) - 1) & 1, status)) {
          ok = false;
          break;
        }
        const int g = pl.h / grp;
        const int plane_q = geo.qplane(pl.b, pl.h), plane_kv = geo.kvplane(pl.b, g);
        mbar_arrive_expect_tx(&q_full[qs], (pl.hasB ? 2 : 1) * C::TILE);
        for (int x = 0; x < (pl.hasB ? 2 : 1); ++x)
          for (int c = 0; c < C::DCH; ++c)
            tma_load_3d(smem + C::OFF_Q + (qs * 2 + x) * C::TILE + c * kChunk, &tm_q, &q_full[qs],
                        64 * c, pl.row0 + (pl.tA + x) * 128, plane_q);
        ++kq;
        for (int u = 0; u < pl.nT; ++u) {
          if (!pl.any(u)) continue;
          const int st = n % NST;
          if (n >= NST && !mbar_wait(&kv_empty[st], ((n / NST) - 1) & 1, status)) {
            ok = false;
            break;
          }
          const bool gat = u < pl.nG;
          const CUtensorMap* mk = gat ? &tm_kk : &tm_k;
          const CUtensorMap* mv = gat ? &tm_vk : &tm_v;
          // gathered tiles: the sequence's keep rows in plane g of the
          // workspace; band tiles: rows of the sequence in its kv plane
          const int row = gat ? 128 * (pl.tile0 + u) : pl.row0 + pl.loA + 128 * (u - pl.nG);
          const int plane = gat ? g : plane_kv;
          mbar_arrive_expect_tx(&kv_full[st], 2 * C::TILE);
          for (int c = 0; c < C::DCH; ++c) {
            tma_load_3d(smem + C::OFF_K + st * C::TILE + c * kChunk, mk, &kv_full[st], 64 * c,
                        row, plane);
            tma_load_3d(smem + C::OFF_V + st * C::TILE + c * kChunk, mv, &kv_full[st], 64 * c,
                        row, plane);
          }
          ++n;
        }
      }
      if (!ok) {
        // let the copies still in flight land before the CTA's smem goes away
        for (int x = n - NST; x < n; ++x)
          if (x >= 0) mbar_wait(&kv_full[x % NST], (x / NST) & 1, status);
        for (int x = kq - QB; x < kq; ++x)
          if (x >= 0) mbar_wait(&q_full[x % QB], (x / QB) & 1, status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The issuer walks one flat stream of (item, key tile) steps.  Per step
    // it issues P.V of tile A, S of A's next step, P.V of B, then S of B's
    // next step, so one tile's softmax runs while the other's products do;
    // the next step may belong to the next item, whose S products then
    // overlap this item's last P.V and the epilogue.  The whole warp runs
    // this loop; the elected lane issues.
    {
      const bool leader = elect_one();
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, false, true);
      const uint32_t k_base = smem_u32(smem + C::OFF_K), v_base = smem_u32(smem + C::OFF_V);
      int cnt0 = 0, cnt1 = 0;  // P.V products issued per query tile (p_full parity)
      int ci0 = 0, ci1 = 0;    // ... within the current item (accumulate flag)
      auto issue_qk = [&](int x, int qs, int st) {
        const uint32_t q_base = smem_u32(smem + C::OFF_Q + (qs * 2 + x) * C::TILE);
        const uint32_t d_s = tmem + (x ? C::TM_S1 : C::TM_S0);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
            umma_bf16_ss(d_s, sdesc_sw128(q_base + off, 16, 1024),
                         sdesc_sw128(k_base + st * C::TILE + off, 16, 1024), idesc_qk, kk > 0);
          }
          umma_commit(&s_full[x]);
        }
        __syncwarp();
      };
      auto issue_pv = [&](int x, int st) -> bool {  // O_x (+)= P_x V, P_x from TMEM
        int& cx = x ? cnt1 : cnt0;
        int& cix = x ? ci1 : ci0;
        if (!mbar_wait_warp(&p_full[x], cx & 1, status)) return false;
        tc_fence_after();
        const uint32_t a_p = tmem + (x ? C::TM_S1 : C::TM_S0);
        const uint32_t d_o = tmem + (x ? C::TM_O1 : C::TM_O0);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_bf16_ts(d_o, a_p + 8 * kk,
                         sdesc_sw128(v_base + st * C::TILE + kk * 2048, kChunk, 1024), idesc_pv,
                         (cix > 0 || kk > 0) ? 1u : 0u);
        }
        __syncwarp();
        ++cx;
        ++cix;
        return true;
      };
      bool ok = true;
      int it = blockIdx.x;
      PairPlan pc = load_plan(idx, s_rec, it, n_items, geo, full_groups, grp);
      while (it < n_items && !pc.valid) {
        it = snake_item(it / G + 1, G);
        pc = load_plan(idx, s_rec, it, n_items, geo, full_groups, grp);
      }
      if (it < n_items) {
        int kq = 0, qs = 0, n = 0;  // current item's index and Q buffer; K/V stage count
        int u = pc.next(-1);
        int itn = snake_item(it / G + 1, G);
        PairPlan pn = load_plan(idx, s_rec, itn, n_items, geo, full_groups, grp);  // prefetched
        ok = mbar_wait_warp(&q_full[0], 0, status) && mbar_wait_warp(&kv_full[0], 0, status);
        tc_fence_after();
        if (ok) {
          if (pc.active(u, 0)) issue_qk(0, 0, 0);
          if (pc.active(u, 1)) issue_qk(1, 0, 0);
          if (leader && pc.next(u) >= pc.nT) umma_commit(&q_empty[0]);  // every S of the item issued
        }
        while (ok) {
          const int st = n % NST, stn = (n + 1) % NST;
          int un = pc.next(u);
          const bool same = un < pc.nT;
          if (!same) {
            while (itn < n_items && !pn.valid) {
              itn = snake_item(itn / G + 1, G);
              pn = load_plan(idx, s_rec, itn, n_items, geo, full_groups, grp);
            }
            if (itn < n_items) un = pn.next(-1);
          }
          const bool has_next = same || itn < n_items;
          const int qsn = same ? qs : (kq + 1) % QB;
          const PairPlan px = same ? pc : pn;
          if (pc.active(u, 0) && !(ok = issue_pv(0, st))) break;
          if (leader && !same) umma_commit(&o_done[0]);
          if (has_next) {
            if (!same && !(ok = mbar_wait_warp(&q_full[qsn], ((kq + 1) / QB) & 1, status))) break;
            if (!(ok = mbar_wait_warp(&kv_full[stn], ((n + 1) / NST) & 1, status))) break;
            tc_fence_after();
            if (px.active(un, 0)) issue_qk(0, qsn, stn);
          }
          if (pc.active(u, 1) && !(ok = issue_pv(1, st))) break;
          if (leader) umma_commit(&kv_empty[st]);  // every MMA reading this K/V stage is issued
          if (leader && !same && pc.hasB) umma_commit(&o_done[1]);
          if (has_next) {
            if (px.active(un, 1)) issue_qk(1, qsn, stn);
            if (leader && px.next(un) >= px.nT) umma_commit(&q_empty[qsn]);
          }
          ++n;
          if (!has_next) break;
          if (!same) {
            pc = pn;
            it = itn;
            ++kq;
            qs = qsn;
            ci0 = ci1 = 0;
            itn = snake_item(it / G + 1, G);
            pn = load_plan(idx, s_rec, itn, n_items, geo, full_groups, grp);
          }
          u = un;
        }
      }
      // every MMA issued by the leader completes before TMEM is released
      if (leader) umma_commit(&mma_final);
      mbar_wait_warp(&mma_final, 0, status);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int x = (warp - 2) >> 2;  // query tile: 0 = A, 1 = B
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_base + (x ? C::TM_S1 : C::TM_S0);
    const uint32_t tO = tmem + lane_base + (x ? C::TM_O1 : C::TM_O0);
    const int nwords = hdr.nwords;
    int cnt = 0, ko = 0;  // S tiles and items finished by this query tile
    bool ok = true;
    PairPlan pn = load_plan(idx, s_rec, blockIdx.x, n_items, geo, full_groups, grp);
    for (int it = blockIdx.x; ok && it < n_items; it = snake_item(it / G + 1, G)) {
      const PairPlan pl = pn;
      pn = load_plan(idx, s_rec, snake_item(it / G + 1, G), n_items, geo, full_groups,
                     grp);  // prefetch the next item
      if (!pl.valid || (x == 1 && !pl.hasB)) continue;
      const int b = pl.b, h = pl.h;
      const int i = (pl.tA + x) * 128 + r;
      const uint32_t* kbits = idx.keep_bits + (size_t)b * nwords;
      const int n_gath = x ? pl.nB : pl.nA;
      const int lo_x = x ? pl.loB : pl.loA;
      const int n_w = group_full(full_groups, h / grp) ? pl.len : n_win;  // full groups: no window
      const int len = pl.len;
      const size_t orow0 = (size_t)geo.qplane(b, h) * geo.R + pl.row0;  // row 0 of the sequence
      float m_used = -INFINITY, l = 0.f;
      int ci = 0;
      for (int u = 0; u < pl.nT; ++u) {
        if (!pl.active(u, x)) continue;
        // visibility of the 128 columns as 4 words
        uint32_t vm[4];
        if (u < pl.nG) {
          const int nv = min(128, n_gath - 128 * u);
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int c = nv - 32 * w;
            vm[w] = c >= 32 ? 0xffffffffu : (c <= 0 ? 0u : ((1u << c) - 1u));
          }
        } else {
          const int jt = pl.loA + 128 * (u - pl.nG);
          const int n_causal = min(128, max(0, i - jt + 1));  // columns c with jt+c <= i
          const int c_win = i - n_w + 1 - jt;                 // columns c >= c_win: window
          const int c_lo = lo_x - jt;                         // columns below it: gathered
          const int wj = jt >> 5, sh = jt & 31;
          uint32_t kw[5];
#pragma unroll
          for (int q = 0; q < 5; ++q) kw[q] = (wj + q < nwords) ? __ldg(kbits + wj + q) : 0u;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const uint32_t keepw = sh ? ((kw[w] >> sh) | (kw[w + 1] << (32 - sh))) : kw[w];
            const int cc = n_causal - 32 * w;
            const uint32_t causal = cc >= 32 ? 0xffffffffu : (cc <= 0 ? 0u : ((1u << cc) - 1u));
            const int cw = c_win - 32 * w;
            const uint32_t win = cw <= 0 ? 0xffffffffu : (cw >= 32 ? 0u : ~((1u << cw) - 1u));
            const int cl = c_lo - 32 * w;
            const uint32_t above = cl <= 0 ? 0xffffffffu : (cl >= 32 ? 0u : ~((1u << cl) - 1u));
            vm[w] = causal & above & (win | keepw);
          }
        }
        if (!mbar_wait(&s_full[x], cnt & 1, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // A tile takes one pass against the running maximum m_used (for a
        // row's first tile, the maximum of its first 32 columns; a row that
        // has seen no visible column yet takes two passes: the row maximum,
        // then P): the lazy rescale keeps every P within 2^kRescaleLog2 while
        // m_used stands.
        // A chunk holding a larger P (a score more than kRescaleLog2 above
        // m_used) ends that pass before it is written; the maximum of the
        // chunks not yet written then sets the new m_used (the written
        // chunks stayed below the bound, so they cannot hold it), and the
        // written P, the row sum and O are rescaled.
        float rs = 0.f, alpha = 1.f;
        int c0 = 0;  // first chunk of 32 columns whose P is not yet written
        bool need_max;
        if (ci == 0) {
          // a row's first tile: the maximum of its first 32 columns stands
          // in for the running max (O holds nothing yet), unless a row of the
          // warp sees none of them
          uint32_t sr[32];
          tmem_ld32(tS, sr);
          tmem_ld_wait();
          float mt0 = -INFINITY;
#pragma unroll
          for (int q = 0; q < 32; ++q)
            if ((vm[0] >> q) & 1u) mt0 = fmaxf(mt0, __uint_as_float(sr[q]));
          need_max = __any_sync(0xffffffffu, mt0 == -INFINITY);
          if (!need_max) m_used = mt0 * scale_log2;
        } else {
          need_max = __any_sync(0xffffffffu, m_used == -INFINITY);
        }
        float msub = m_used;
        if (!need_max) {
#pragma unroll 1
          for (; c0 < 4; ++c0) {
            uint32_t sr[32], pk[16];
            tmem_ld32(tS + 32 * c0, sr);
            tmem_ld_wait();
            const uint32_t w = c0 == 0 ? vm[0] : c0 == 1 ? vm[1] : c0 == 2 ? vm[2] : vm[3];
            const float rs0 = rs;
            float pm = 0.f;
#pragma unroll
            for (int q = 0; q < 32; q += 2) {
              float a0, a1;
              ffma2(a0, a1, __uint_as_float(sr[q]), __uint_as_float(sr[q + 1]), scale_log2,
                    scale_log2, -msub, -msub);
              float p0 = fast_exp2(a0), p1 = fast_exp2(a1);
              p0 = ((w >> q) & 1u) ? p0 : 0.f;
              p1 = ((w >> (q + 1)) & 1u) ? p1 : 0.f;
              rs += p0 + p1;
              pm = fmaxf(pm, fmaxf(p0, p1));
              pk[q >> 1] = pack_bf16x2(p0, p1);
            }
            if (__any_sync(0xffffffffu, !(pm <= kRescaleBound))) {
              rs = rs0;
              need_max = true;
              break;
            }
            tmem_st16(tS + 16 * c0, pk);
          }
        }
        if (need_max) {
          // the row maximum over the visible columns of chunks c0 .. 3
          float mt = -INFINITY;
#pragma unroll 1
          for (int c = c0; c < 4; ++c) {
            uint32_t sr[32];
            tmem_ld32(tS + 32 * c, sr);
            tmem_ld_wait();
            const uint32_t w = c == 0 ? vm[0] : c == 1 ? vm[1] : c == 2 ? vm[2] : vm[3];
#pragma unroll
            for (int q = 0; q < 32; ++q)
              if ((w >> q) & 1u) mt = fmaxf(mt, __uint_as_float(sr[q]));
          }
          mt *= scale_log2;  // scale_log2 > 0 keeps the maximum where it is
          const float m_new = fmaxf(m_used, mt);
          const bool rescale = m_new > m_used + kRescaleLog2;
          if (rescale) {
            alpha = fast_exp2(m_used - m_new);
            m_used = m_new;
          }
          msub = (m_used == -INFINITY) ? 0.f : m_used;
          if (__any_sync(0xffffffffu, rescale)) {
            // the P already written (chunks before c0) and the row sum
#pragma unroll 1
            for (int c = 0; c < c0; ++c) {
              uint32_t pw[16];
              tmem_ld16(tS + 16 * c, pw);
              tmem_ld_wait();
#pragma unroll
              for (int q = 0; q < 16; ++q)
                pw[q] = pack_bf16x2(__uint_as_float(pw[q] << 16) * alpha,
                                    __uint_as_float(pw[q] & 0xffff0000u) * alpha);
              tmem_st16(tS + 16 * c, pw);
            }
            rs *= alpha;
            // O: S of this tile being ready means the previous P.V of this
            // query tile has completed (the tensor pipe runs in order)
            if (ci > 0) {
              uint32_t ob[32];
#pragma unroll
              for (int o0 = 0; o0 < D; o0 += 32) {
                tmem_ld32(tO + o0, ob);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 32; ++q)
                  ob[q] = __float_as_uint(__uint_as_float(ob[q]) * alpha);
                tmem_st32(tO + o0, ob);
              }
            }
          }
          // P = exp2(S * scale - m) as packed bf16 for chunks c0 .. 3, written
          // over the first 64 columns of S (chunk c's P lands on S columns
          // [16c, 16c+16), all of which have been read by then)
#pragma unroll 1
          for (int c = c0; c < 4; ++c) {
            uint32_t sr[32], pk[16];
            tmem_ld32(tS + 32 * c, sr);
            tmem_ld_wait();
            const uint32_t w = c == 0 ? vm[0] : c == 1 ? vm[1] : c == 2 ? vm[2] : vm[3];
#pragma unroll
            for (int q = 0; q < 32; q += 2) {
              float a0, a1;
              ffma2(a0, a1, __uint_as_float(sr[q]), __uint_as_float(sr[q + 1]), scale_log2,
                    scale_log2, -msub, -msub);
              float p0 = fast_exp2(a0), p1 = fast_exp2(a1);
              p0 = ((w >> q) & 1u) ? p0 : 0.f;
              p1 = ((w >> (q + 1)) & 1u) ? p1 : 0.f;
              rs += p0 + p1;
              pk[q >> 1] = pack_bf16x2(p0, p1);
            }
            tmem_st16(tS + 16 * c, pk);
          }
        }
        l = l * alpha + rs;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[x]);
        ++cnt;
        ++ci;
      }
      if (!ok || !mbar_wait(&o_done[x], ko & 1, status)) {
        ok = false;
        break;
      }
      ++ko;
      tc_fence_after();
      const float inv_l = 1.f / l;
      uint32_t ob[32];
      __nv_bfloat16* orow = o + (orow0 + i) * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        tmem_ld32(tO + c0, ob);
        tmem_ld_wait();
        if (i < len) {
#pragma unroll
          for (int q = 0; q < 32; q += 8) {
            uint4 pk;
            pk.x = pack_bf16x2(__uint_as_float(ob[q]) * inv_l, __uint_as_float(ob[q + 1]) * inv_l);
            pk.y = pack_bf16x2(__uint_as_float(ob[q + 2]) * inv_l,
                               __uint_as_float(ob[q + 3]) * inv_l);
            pk.z = pack_bf16x2(__uint_as_float(ob[q + 4]) * inv_l,
                               __uint_as_float(ob[q + 5]) * inv_l);
            pk.w = pack_bf16x2(__uint_as_float(ob[q + 6]) * inv_l,
                               __uint_as_float(ob[q + 7]) * inv_l);
            *reinterpret_cast<uint4*>(orow + c0 + q) = pk;
          }
        }
      }
      if (i < len) lse[orow0 + i] = (m_used + __log2f(l)) * 0.69314718055994531f;
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TM_COLS);
}

template <int D>
int launch_fwd_impl(IndexPtrs idx, const void* q, const void* k, const void* v, void* o, float* lse,
                    const Geom& geo, float scale, uint64_t full_groups, void* ws, int* status,
                    cudaStream_t s) {
  using C = FwdCfg<D>;
  uint8_t* kk = static_cast<uint8_t*>(ws);
  uint8_t* vk = kk + align_up((size_t)geo.Hkv * geo.TT * 128 * D * 2, 256);
  const int sms = num_sms();
  profile_mark(0, s);
  cudaError_t e = launch_dependent(
      gather_keep_kernel<D>, dim3(keep_pass_ctas(keep_units(geo.B, geo.Hkv, geo.L), sms)),
      dim3(256), 0, s, idx, geo, static_cast<const uint4*>(k), static_cast<const uint4*>(v),
      reinterpret_cast<uint4*>(kk), reinterpret_cast<uint4*>(vk), status);
  if (e != cudaSuccess) return static_cast<int>(e);
  // head planes of q / k / v: (sequence, head) planes of L rows, or one plane
  // per head of a pack; the gathered keep rows: one plane per kv head over
  // the tile space
  const uint64_t pq = geo.packed ? geo.Hq : (uint64_t)geo.B * geo.Hq;
  const uint64_t pkv = geo.packed ? geo.Hkv : (uint64_t)geo.B * geo.Hkv;
  const uint64_t rk = (uint64_t)geo.TT * 128;
  CUtensorMap mq, mk, mv, mkk, mvk;
  if (!make_bf16_map(&mq, q, pq, geo.R, D, 128) || !make_bf16_map(&mk, k, pkv, geo.R, D, 128) ||
      !make_bf16_map(&mv, v, pkv, geo.R, D, 128) ||
      !make_bf16_map(&mkk, kk, geo.Hkv, rk, D, 128) ||
      !make_bf16_map(&mvk, vk, geo.Hkv, rk, D, 128))
    return static_cast<int>(cudaErrorInvalidValue);
  auto kern = attn_fwd_tc_kernel<D>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return static_cast<int>(e);
  const float scale_log2 = scale * 1.4426950408889634f;
  const long long items = (long long)geo.B * geo.Hq * ((geo.T + 1) / 2);
  const int grid = static_cast<int>(items < sms ? items : sms);  // persistent: one CTA per SM
  profile_mark(1, s);
  const cudaError_t err =
      launch_dependent(kern, dim3(grid), dim3(kThreads), C::SMEM, s, mq, mk, mv, mkk, mvk, idx,
                       static_cast<__nv_bfloat16*>(o), lse, geo, scale_log2, full_groups, status);
  profile_mark(2, s);
  return static_cast<int>(err);
}

}  // namespace

size_t attn_fwd_tc_workspace(const Geom& geo, int d) {
  return 2 * align_up((size_t)geo.Hkv * geo.TT * 128 * d * 2, 256);
}

int launch_attn_fwd_tc(IndexPtrs idx, const void* q, const void* k, const void* v, void* o,
                       float* lse, const Geom& geo, int d, float scale, uint64_t full_groups,
                       void* ws, int* status, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d == 64)
    return launch_fwd_impl<64>(idx, q, k, v, o, lse, geo, scale, full_groups, ws, status, s);
  return launch_fwd_impl<128>(idx, q, k, v, o, lse, geo, scale, full_groups, ws, status, s);
}

}  // namespace sep
