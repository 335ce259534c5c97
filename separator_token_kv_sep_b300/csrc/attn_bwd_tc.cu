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
// band), and the backward keeps that split:
//   bwd_dq_kernel    query-major, the forward's traversal: S = Q K^T and
//                    dP = dO V^T into TMEM, dS to shared memory, dQ += dS K.
//   bwd_kv_kernel<KEEP>   key-major over the gathered keep tiles: each CTA
//                    owns 128 keep tokens and one q head and walks the query
//                    tiles that gather them; its fp32 dK/dV sums are added
//                    into a per-keep-token accumulator with red.global.add.
//   bwd_kv_kernel<DENSE>  key-major over aligned 128-key tiles and the query
//                    tiles whose dense band covers them (all q heads of the
//                    kv group); its epilogue adds the keep accumulator of
//                    keep tokens and rounds each gradient to bf16 once.
// In the key-major kernels S^T = K Q^T and dP^T = V dO^T go to TMEM; the
// elementwise warps (one thread per key) turn them into P^T and dS^T in
// shared memory and release TMEM first, so (with two Q/dO stages) the next
// query tile's S^T / dP^T overlap this tile's dV += P^T dO and dK += dS^T Q
// on the tensor pipe.
// All waits are bounded; on expiry a kernel records SEP_ERR_TIMEOUT, drains
// its copies and MMAs, frees TMEM and returns.
#include "common.cuh"
#include "layout.h"
#include "tma_host.h"

namespace sep {

namespace {

constexpr int kChunk = 128 * 128;  // bytes of a [128 rows x 64 cols] bf16 block
constexpr int kThreads = 192;      // warp 0 TMA, warp 1 MMA, warps 2-5 elementwise
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kKeepChunk = 4;      // query tiles per CTA of the keep-tile dK/dV kernel

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

// Named barrier among the 128 elementwise threads (warps 2-5).
__device__ __forceinline__ void ew_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Prep: Delta = rowsum(dO o O) in fp32, and zeroed keep-token accumulators.
// The first kPrepDeltaBlocks(..) CTAs compute Delta: U = D/8 lanes share a
// row (16 bytes each, so a warp reads 32/U whole rows per instruction) and
// each warp covers kPrepRows rows.  The remaining CTAs zero, per (batch, kv
// head), the contiguous accumulator rows [0, ceil128(keep_count)).
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 256;
constexpr int kPrepRows = 16;  // rows per warp in the Delta part

template <int D>
__host__ __device__ constexpr int prep_rows_per_block() {
  return (kPrepThreads / 32) * kPrepRows;
}

template <int D>
__global__ void __launch_bounds__(kPrepThreads)
    bwd_prep_kernel(IndexPtrs idx, const uint4* __restrict__ o, const uint4* __restrict__ dout,
                    float* __restrict__ delta, float4* __restrict__ dk_keep,
                    float4* __restrict__ dv_keep, int B, int Hq, int Hkv, int L,
                    int delta_blocks) {
  constexpr int U = D / 8;         // 16-byte units per row
  constexpr int RPI = 32 / U;      // rows per warp instruction
  constexpr int IT = kPrepRows / RPI;
  const IndexHeader hdr = *idx.header;
  if (hdr.magic != kIndexMagic || hdr.B != B || hdr.L != L) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (static_cast<int>(blockIdx.x) < delta_blocks) {
    const size_t R = (size_t)B * Hq * L;
    const size_t row0 = ((size_t)blockIdx.x * (kPrepThreads / 32) + warp) * kPrepRows;
    const int sub = lane / U, u = lane % U;
    uint4 xo[IT], xd[IT];
#pragma unroll
    for (int it = 0; it < IT; ++it) {
      const size_t row = row0 + it * RPI + sub;
      xo[it] = row < R ? o[row * U + u] : make_uint4(0, 0, 0, 0);
      xd[it] = row < R ? dout[row * U + u] : make_uint4(0, 0, 0, 0);
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
      const size_t row = row0 + it * RPI + sub;
      if (u == 0 && row < R) delta[row] = acc;
    }
    return;
  }
  // zero the keep accumulators: per_plane consecutive blocks cover one plane
  const int zb = static_cast<int>(blockIdx.x) - delta_blocks;
  const int per_plane = (L * (D / 4) + kPrepThreads * 4 - 1) / (kPrepThreads * 4);
  const int plane = zb / per_plane, part = zb % per_plane;
  if (plane >= B * Hkv) return;
  const int b = plane / Hkv;
  const int count = min(max(idx.keep_count[b], 0), L);
  const int end = min(L, (count + 127) / 128 * 128) * (D / 4);  // float4s in use
  const size_t base = (size_t)plane * L * (D / 4);
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int e = (part * 4 + r) * kPrepThreads + threadIdx.x;
    if (e < end) {
      dk_keep[base + e] = z;
      dv_keep[base + e] = z;
    }
  }
}

// Gathered keep-token K/V rows, zero-filled up to the next multiple of 128.
template <int D>
__global__ void __launch_bounds__(256)
    bwd_gather_kernel(IndexPtrs idx, const uint4* __restrict__ k, const uint4* __restrict__ v,
                      uint4* __restrict__ kk, uint4* __restrict__ vk, int Hkv, int L) {
  constexpr int U = D / 8;
  constexpr int ROWS = 64;
  const int g = blockIdx.y, b = blockIdx.z;
  // the header sits at offset 0 of any index buffer: check it before using
  // the fields whose offsets depend on B and L
  const IndexHeader hdr = *idx.header;
  if (hdr.magic != kIndexMagic || hdr.B != static_cast<int>(gridDim.z) || hdr.L != L) return;
  const int count = idx.keep_count[b];
  if (count < 0 || count > L) return;
  const int end = min(L, (count + 127) / 128 * 128);
  const int r0 = blockIdx.x * ROWS;
  if (r0 >= end) return;
  const int32_t* kpos = idx.keep_pos + (size_t)b * L;
  const size_t plane = ((size_t)b * Hkv + g) * (size_t)L * U;
  for (int e = threadIdx.x; e < ROWS * U; e += blockDim.x) {
    const int row = r0 + e / U, u = e % U;
    if (row >= end) break;
    const int src = row < count ? kpos[row] : -1;
    uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
    if (src >= 0 && src < L) {
      kv = k[plane + (size_t)src * U + u];
      vv = v[plane + (size_t)src * U + u];
    }
    kk[plane + (size_t)row * U + u] = kv;
    vk[plane + (size_t)row * U + u] = vv;
  }
}

// ---------------------------------------------------------------------------
// Key-major dK / dV
// ---------------------------------------------------------------------------
template <int D, int NST>
struct KvCfg {
  static constexpr int DCH = D / 64;
  static constexpr int TILE = DCH * kChunk;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = TILE;
  static constexpr int OFF_Q = 2 * TILE;
  static constexpr int OFF_DO = OFF_Q + NST * TILE;
  static constexpr int OFF_P = OFF_DO + NST * TILE;
  static constexpr int OFF_DS = OFF_P + 2 * kChunk;
  static constexpr int OFF_STAT = OFF_DS + 2 * kChunk;  // [2][2][128] floats
  static constexpr int SMEM = OFF_STAT + 2 * 2 * 128 * 4 + 1024;
  static constexpr int TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 256 + D;
  static constexpr int TM_COLS = 512;
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

template <int D, bool KEEP, int NST>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kv_kernel(const __grid_constant__ CUtensorMap tm_kx,
                  const __grid_constant__ CUtensorMap tm_vx,
                  const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_do, IndexPtrs idx,
                  const float* __restrict__ lse, const float* __restrict__ delta,
                  float* __restrict__ dk_keep, float* __restrict__ dv_keep,
                  __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, int B, int Hq,
                  int Hkv, int L, float scale, float scale_log2, int* status) {
  using C = KvCfg<D, NST>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t kv_full, sd_full, sd_free, ps_full, pd_done, mma_final;
  __shared__ __align__(8) uint64_t qd_full[NST], qd_empty[NST];
  __shared__ uint32_t tmem_slot;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = (L + 127) >> 7;
  const int G = Hq / Hkv;
  // DENSE: one key tile per CTA (longest first).  KEEP: one keep tile and one
  // chunk of kKeepChunk query tiles per CTA, so a keep tile's many query
  // tiles spread over several CTAs (their partial sums meet in the fp32 keep
  // accumulators).
  const int n_qc = (T + kKeepChunk - 1) / kKeepChunk;
  const int tile = KEEP ? static_cast<int>(blockIdx.x) / n_qc
                        : T - 1 - static_cast<int>(blockIdx.x);
  const int qc = KEEP ? static_cast<int>(blockIdx.x) % n_qc : 0;
  const int b = blockIdx.z;
  // KEEP: blockIdx.y is the q head; DENSE: the kv head
  const int g = KEEP ? static_cast<int>(blockIdx.y) / G : static_cast<int>(blockIdx.y);
  const int h_fixed = KEEP ? static_cast<int>(blockIdx.y) : -1;

  const IndexHeader hdr = *idx.header;
  if (hdr.magic != kIndexMagic || hdr.B != B || hdr.L != L || hdr.block_m != 128) {
    if (threadIdx.x == 0) report(status, SEP_ERR_DEVICE_BOUNDS);
    return;
  }
  const int32_t* blocks = idx.blocks + (size_t)b * T * 4;
  const int count = idx.keep_count[b];
  if (count < 0 || count > L) {
    if (threadIdx.x == 0) report(status, SEP_ERR_DEVICE_BOUNDS);
    return;
  }
  const int j0 = tile * 128;  // first key (KEEP: first keep index) of the tile
  int t_begin, n_t;
  if (KEEP) {
    if (j0 >= count) return;
    // first query tile whose gathered list reaches past j0 (n_gather is
    // non-decreasing in t)
    int lo_t = 0, hi_t = T;
    while (lo_t < hi_t) {
      const int mid = (lo_t + hi_t) >> 1;
      if (blocks[4 * mid] > j0) hi_t = mid; else lo_t = mid + 1;
    }
    t_begin = max(lo_t, qc * kKeepChunk);
    n_t = min(T, (qc + 1) * kKeepChunk) - t_begin;
    if (n_t <= 0) return;
  } else {
    // query tiles t >= tile whose dense band starts before this key tile ends
    t_begin = tile;
    int lo_t = tile, hi_t = T;
    while (lo_t < hi_t) {
      const int mid = (lo_t + hi_t) >> 1;
      if (blocks[4 * mid + 1] < j0 + 128) lo_t = mid + 1; else hi_t = mid;
    }
    n_t = lo_t - tile;
    if (n_t <= 0) return;  // unreachable: tile t = `tile` always covers its own keys
  }
  const int nU = KEEP ? n_t : G * n_t;
  const int n_win = hdr.n;

  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sDO = smem + C::OFF_DO;
  uint8_t* sP = smem + C::OFF_P;
  uint8_t* sDS = smem + C::OFF_DS;
  float* sStat = reinterpret_cast<float*>(smem + C::OFF_STAT);

  if (threadIdx.x == 0) {
    mbar_init(&kv_full, 1);
    mbar_init(&sd_full, 1);
    mbar_init(&sd_free, 128);
    mbar_init(&ps_full, 128);
    mbar_init(&pd_done, 1);
    mbar_init(&mma_final, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&qd_full[s], 1);
      mbar_init(&qd_empty[s], 1);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  auto head_of = [&](int u) { return KEEP ? h_fixed : g * G + u / n_t; };
  auto qtile_of = [&](int u) { return t_begin + (KEEP ? u : u % n_t); };

  if (warp == 0) {
    if (lane == 0) {
      const int plane_kv = b * Hkv + g;
      mbar_arrive_expect_tx(&kv_full, 2 * C::TILE);
      for (int c = 0; c < C::DCH; ++c) {
        tma_load_3d(sK + c * kChunk, &tm_kx, &kv_full, 64 * c, j0, plane_kv);
        tma_load_3d(sV + c * kChunk, &tm_vx, &kv_full, 64 * c, j0, plane_kv);
      }
      int issued = 0;
      bool ok = true;
      for (int u = 0; u < nU; ++u) {
        const int st = u % NST;
        if (u >= NST && !mbar_wait(&qd_empty[st], ((u / NST) - 1) & 1, status)) {
          ok = false;
          break;
        }
        const int plane_q = b * Hq + head_of(u), row = qtile_of(u) * 128;
        mbar_arrive_expect_tx(&qd_full[st], 2 * C::TILE);
        for (int c = 0; c < C::DCH; ++c) {
          tma_load_3d(sQ + st * C::TILE + c * kChunk, &tm_q, &qd_full[st], 64 * c, row, plane_q);
          tma_load_3d(sDO + st * C::TILE + c * kChunk, &tm_do, &qd_full[st], 64 * c, row,
                      plane_q);
        }
        issued = u + 1;
      }
      if (!ok) {
        for (int u = issued - NST; u < issued; ++u)
          if (u >= 0) mbar_wait(&qd_full[u % NST], (u / NST) & 1, status);
        mbar_wait(&kv_full, 0, status);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_ss = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_acc = idesc_bf16_f32(128, D, false, true);
      const uint32_t k_base = smem_u32(sK), v_base = smem_u32(sV), q_base = smem_u32(sQ),
                     do_base = smem_u32(sDO), p_base = smem_u32(sP), ds_base = smem_u32(sDS);
      auto issue_sdp = [&](int u) -> bool {
        const int st = u % NST;
        if (!mbar_wait(&qd_full[st], (u / NST) & 1, status)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
          umma_bf16_ss(tmem + C::TM_S, sdesc_sw128(k_base + off, 16, 1024),
                       sdesc_sw128(q_base + st * C::TILE + off, 16, 1024), idesc_ss, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
          umma_bf16_ss(tmem + C::TM_DP, sdesc_sw128(v_base + off, 16, 1024),
                       sdesc_sw128(do_base + st * C::TILE + off, 16, 1024), idesc_ss, kk > 0);
        }
        umma_commit(&sd_full);
        return true;
      };
      auto issue_acc = [&](int u) -> bool {
        const int st = u % NST;
        if (!mbar_wait(&ps_full, u & 1, status)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t aoff = (kk >> 2) * kChunk + (kk & 3) * 32;
          const uint32_t boff = st * C::TILE + kk * 2048;
          const uint32_t acc = (u > 0 || kk > 0) ? 1u : 0u;
          umma_bf16_ss(tmem + C::TM_DV, sdesc_sw128(p_base + aoff, 16, 1024),
                       sdesc_sw128(do_base + boff, kChunk, 1024), idesc_acc, acc);
          umma_bf16_ss(tmem + C::TM_DK, sdesc_sw128(ds_base + aoff, 16, 1024),
                       sdesc_sw128(q_base + boff, kChunk, 1024), idesc_acc, acc);
        }
        umma_commit(&pd_done);
        umma_commit(&qd_empty[st]);
        return true;
      };
      auto next_sdp = [&](int u) -> bool {  // S^T / dP^T of tile u+1
        if (u + 1 >= nU) return true;
        if (!mbar_wait(&sd_free, u & 1, status)) return false;
        return issue_sdp(u + 1);
      };
      bool ok = mbar_wait(&kv_full, 0, status);
      tc_fence_after();
      if (ok) ok = issue_sdp(0);
      for (int u = 0; ok && u < nU; ++u) {
        // With one Q/dO stage, tile u+1 cannot be loaded before dV/dK of tile
        // u release the stage, so the order flips.
        if (NST > 1) ok = next_sdp(u);
        if (ok) ok = issue_acc(u);
        if (ok && NST == 1) ok = next_sdp(u);
      }
      umma_commit(&mma_final);
      mbar_wait(&mma_final, 0, status);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- elementwise
    const int quad = warp & 3;
    const int r = quad * 32 + lane;   // key row of the tile
    const int ew = threadIdx.x - 64;  // 0..127
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const int j = j0 + r;  // KEEP: keep index; DENSE: key position
    bool keep_j = false;
    if (!KEEP && j < L)
      keep_j = (idx.keep_bits[(size_t)b * hdr.nwords + (j >> 5)] >> (j & 31)) & 1u;
    bool ok = true;
    for (int u = 0; u < nU; ++u) {
      const int h = head_of(u), t = qtile_of(u);
      const int i0 = t * 128;
      // stage this query tile's LSE (log2 units) and Delta for all 128 columns
      {
        float* st = sStat + (u & 1) * 256;
        const int i = i0 + ew;
        const size_t ri = ((size_t)b * Hq + h) * L + i;
        st[ew] = i < L ? lse[ri] * kLog2e : 0.f;
        st[128 + ew] = i < L ? delta[ri] : 0.f;
      }
      ew_sync();
      const float* sl = sStat + (u & 1) * 256;
      const float* sd = sl + 128;
      // visible columns of this row as 4 words
      uint32_t vm[4];
      const int4 blk = *reinterpret_cast<const int4*>(blocks + 4 * t);
      const int c_end = min(128, L - i0);  // query rows past L are padding
      if (KEEP) {
        const bool row_ok = j < blk.x;  // gathered by this query tile
#pragma unroll
        for (int w = 0; w < 4; ++w) vm[w] = row_ok ? range_bits(0, c_end, w) : 0u;
      } else {
        const bool in_band = j >= blk.y && j < blk.z && j < L;
        // columns i with i >= j, and i <= j + n - 1 unless j is a keep token
        const int c_lo = j - i0;
        const int c_hi = keep_j ? c_end : min(c_end, j + n_win - i0);
#pragma unroll
        for (int w = 0; w < 4; ++w) vm[w] = in_band ? range_bits(c_lo, c_hi, w) : 0u;
      }
      if (!mbar_wait(&sd_full, u & 1, status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t pk[64], dk2[64];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t sr[32], dr[32];
        tmem_ld32(tmem + lane_base + C::TM_S + 32 * cc, sr);
        tmem_ld32(tmem + lane_base + C::TM_DP + 32 * cc, dr);
        tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < 32; x += 2) {
          const int c = 32 * cc + x;
          const bool v0 = (vm[cc] >> x) & 1u, v1 = (vm[cc] >> (x + 1)) & 1u;
          const float p0 = v0 ? fast_exp2(__uint_as_float(sr[x]) * scale_log2 - sl[c]) : 0.f;
          const float p1 =
              v1 ? fast_exp2(__uint_as_float(sr[x + 1]) * scale_log2 - sl[c + 1]) : 0.f;
          const float d0 = p0 * (__uint_as_float(dr[x]) - sd[c]);
          const float d1 = p1 * (__uint_as_float(dr[x + 1]) - sd[c + 1]);
          pk[c >> 1] = pack_bf16x2(p0, p1);
          dk2[c >> 1] = pack_bf16x2(d0, d1);
        }
      }
      tc_fence_before();
      mbar_arrive(&sd_free);
      if (u > 0 && !mbar_wait(&pd_done, (u - 1) & 1, status)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int un = 0; un < 16; ++un) {
        const uint32_t off = (un >> 3) * kChunk + sw128_offset(r, (un & 7) * 8);
        *reinterpret_cast<uint4*>(sP + off) =
            make_uint4(pk[4 * un], pk[4 * un + 1], pk[4 * un + 2], pk[4 * un + 3]);
        *reinterpret_cast<uint4*>(sDS + off) =
            make_uint4(dk2[4 * un], dk2[4 * un + 1], dk2[4 * un + 2], dk2[4 * un + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&ps_full);
    }
    if (ok && mbar_wait(&pd_done, (nU - 1) & 1, status)) {
      tc_fence_after();
      uint32_t vb[32], kb[32];
      if (KEEP) {
        const bool live = j < count;
        float* dkr = dk_keep + (((size_t)b * Hkv + g) * L + j) * D;
        float* dvr = dv_keep + (((size_t)b * Hkv + g) * L + j) * D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          tmem_ld32(tmem + lane_base + C::TM_DV + c0, vb);
          tmem_ld32(tmem + lane_base + C::TM_DK + c0, kb);
          tmem_ld_wait();
          if (live) {
#pragma unroll
            for (int x = 0; x < 32; x += 4) {
              red_add_v4(dvr + c0 + x, __uint_as_float(vb[x]), __uint_as_float(vb[x + 1]),
                         __uint_as_float(vb[x + 2]), __uint_as_float(vb[x + 3]));
              red_add_v4(dkr + c0 + x, __uint_as_float(kb[x]), __uint_as_float(kb[x + 1]),
                         __uint_as_float(kb[x + 2]), __uint_as_float(kb[x + 3]));
            }
          }
        }
      } else {
        const bool live = j < L;
        const int kidx = keep_j ? idx.keep_prefix[(size_t)b * (L + 1) + j] : 0;
        const float* dkr = dk_keep + (((size_t)b * Hkv + g) * L + kidx) * D;
        const float* dvr = dv_keep + (((size_t)b * Hkv + g) * L + kidx) * D;
        __nv_bfloat16* dko = dk + (((size_t)b * Hkv + g) * L + j) * D;
        __nv_bfloat16* dvo = dv + (((size_t)b * Hkv + g) * L + j) * D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          tmem_ld32(tmem + lane_base + C::TM_DV + c0, vb);
          tmem_ld32(tmem + lane_base + C::TM_DK + c0, kb);
          tmem_ld_wait();
          if (live) {
#pragma unroll
            for (int x = 0; x < 32; x += 8) {
              float fv[8], fk[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                fv[e] = __uint_as_float(vb[x + e]);
                fk[e] = __uint_as_float(kb[x + e]);
              }
              if (keep_j) {
                const float4 a0 = *reinterpret_cast<const float4*>(dvr + c0 + x);
                const float4 a1 = *reinterpret_cast<const float4*>(dvr + c0 + x + 4);
                const float4 b0 = *reinterpret_cast<const float4*>(dkr + c0 + x);
                const float4 b1 = *reinterpret_cast<const float4*>(dkr + c0 + x + 4);
                fv[0] += a0.x; fv[1] += a0.y; fv[2] += a0.z; fv[3] += a0.w;
                fv[4] += a1.x; fv[5] += a1.y; fv[6] += a1.z; fv[7] += a1.w;
                fk[0] += b0.x; fk[1] += b0.y; fk[2] += b0.z; fk[3] += b0.w;
                fk[4] += b1.x; fk[5] += b1.y; fk[6] += b1.z; fk[7] += b1.w;
              }
              uint4 ov, ok4;
              ov.x = pack_bf16x2(fv[0], fv[1]); ov.y = pack_bf16x2(fv[2], fv[3]);
              ov.z = pack_bf16x2(fv[4], fv[5]); ov.w = pack_bf16x2(fv[6], fv[7]);
              ok4.x = pack_bf16x2(fk[0] * scale, fk[1] * scale);
              ok4.y = pack_bf16x2(fk[2] * scale, fk[3] * scale);
              ok4.z = pack_bf16x2(fk[4] * scale, fk[5] * scale);
              ok4.w = pack_bf16x2(fk[6] * scale, fk[7] * scale);
              *reinterpret_cast<uint4*>(dvo + c0 + x) = ov;
              *reinterpret_cast<uint4*>(dko + c0 + x) = ok4;
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TM_COLS);
}

// ---------------------------------------------------------------------------
// Query-major dQ
// ---------------------------------------------------------------------------
template <int D, int NST>
struct DqCfg {
  static constexpr int DCH = D / 64;
  static constexpr int TILE = DCH * kChunk;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = TILE;
  static constexpr int OFF_K = 2 * TILE;
  static constexpr int OFF_V = OFF_K + NST * TILE;
  static constexpr int OFF_DS = OFF_V + NST * TILE;
  static constexpr int SMEM = OFF_DS + 2 * kChunk + 1024;
  static constexpr int TM_S = 0, TM_DP = 128, TM_DQ = 256;
  static constexpr int TM_COLS = 512;
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(NST >= 2, "the next tile's S/dP is issued before this tile's dQ");
};

template <int D, int NST>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_kk,
                  const __grid_constant__ CUtensorMap tm_vk, IndexPtrs idx,
                  const float* __restrict__ lse, const float* __restrict__ delta,
                  __nv_bfloat16* __restrict__ dq, int B, int Hq, int Hkv, int L, float scale,
                  float scale_log2, int* status) {
  using C = DqCfg<D, NST>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t qd_full, sd_full, sd_free, ds_full, dq_done, mma_final;
  __shared__ __align__(8) uint64_t kv_full[NST], kv_empty[NST];
  __shared__ uint32_t tmem_slot;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = (L + 127) >> 7;
  const int t = T - 1 - static_cast<int>(blockIdx.x);
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = h / (Hq / Hkv);
  const int q0 = t * 128;

  const IndexHeader hdr = *idx.header;
  if (hdr.magic != kIndexMagic || hdr.B != B || hdr.L != L || hdr.block_m != 128) {
    if (threadIdx.x == 0) report(status, SEP_ERR_DEVICE_BOUNDS);
    return;
  }
  const int4 blk = *reinterpret_cast<const int4*>(idx.blocks + ((size_t)b * T + t) * 4);
  const int n_gather = blk.x, lo = blk.y, hi = blk.z;
  if (n_gather < 0 || n_gather > lo || lo < 0 || lo > q0 || hi <= q0 || hi > L) {
    if (threadIdx.x == 0) report(status, SEP_ERR_DEVICE_BOUNDS);
    return;
  }
  const int nG = (n_gather + 127) >> 7;
  const int nT = nG + ((hi - lo + 127) >> 7);
  const int n_win = hdr.n;

  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sDO = smem + C::OFF_DO;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sDS = smem + C::OFF_DS;

  if (threadIdx.x == 0) {
    mbar_init(&qd_full, 1);
    mbar_init(&sd_full, 1);
    mbar_init(&sd_free, 128);
    mbar_init(&ds_full, 128);
    mbar_init(&dq_done, 1);
    mbar_init(&mma_final, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      const int plane_q = b * Hq + h, plane_kv = b * Hkv + g;
      mbar_arrive_expect_tx(&qd_full, 2 * C::TILE);
      for (int c = 0; c < C::DCH; ++c) {
        tma_load_3d(sQ + c * kChunk, &tm_q, &qd_full, 64 * c, q0, plane_q);
        tma_load_3d(sDO + c * kChunk, &tm_do, &qd_full, 64 * c, q0, plane_q);
      }
      int issued = 0;
      bool ok = true;
      for (int u = 0; u < nT; ++u) {
        const int st = u % NST;
        if (u >= NST && !mbar_wait(&kv_empty[st], ((u / NST) - 1) & 1, status)) {
          ok = false;
          break;
        }
        const bool gat = u < nG;
        const CUtensorMap* mk = gat ? &tm_kk : &tm_k;
        const CUtensorMap* mv = gat ? &tm_vk : &tm_v;
        const int row = gat ? 128 * u : lo + 128 * (u - nG);
        mbar_arrive_expect_tx(&kv_full[st], 2 * C::TILE);
        for (int c = 0; c < C::DCH; ++c) {
          tma_load_3d(sK + st * C::TILE + c * kChunk, mk, &kv_full[st], 64 * c, row, plane_kv);
          tma_load_3d(sV + st * C::TILE + c * kChunk, mv, &kv_full[st], 64 * c, row, plane_kv);
        }
        issued = u + 1;
      }
      if (!ok) {
        for (int u = issued - NST; u < issued; ++u)
          if (u >= 0) mbar_wait(&kv_full[u % NST], (u / NST) & 1, status);
        mbar_wait(&qd_full, 0, status);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_ss = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_acc = idesc_bf16_f32(128, D, false, true);
      const uint32_t q_base = smem_u32(sQ), do_base = smem_u32(sDO), k_base = smem_u32(sK),
                     v_base = smem_u32(sV), ds_base = smem_u32(sDS);
      auto issue_sdp = [&](int u) -> bool {
        const int st = u % NST;
        if (!mbar_wait(&kv_full[st], (u / NST) & 1, status)) return false;
        tc_fence_after();
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
        return true;
      };
      auto issue_dq = [&](int u) -> bool {
        const int st = u % NST;
        if (!mbar_wait(&ds_full, u & 1, status)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t aoff = (kk >> 2) * kChunk + (kk & 3) * 32;
          umma_bf16_ss(tmem + C::TM_DQ, sdesc_sw128(ds_base + aoff, 16, 1024),
                       sdesc_sw128(k_base + st * C::TILE + kk * 2048, kChunk, 1024), idesc_acc,
                       (u > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&dq_done);
        umma_commit(&kv_empty[st]);
        return true;
      };
      bool ok = mbar_wait(&qd_full, 0, status);
      tc_fence_after();
      if (ok) ok = issue_sdp(0);
      for (int u = 0; ok && u < nT; ++u) {
        if (u + 1 < nT) {
          ok = mbar_wait(&sd_free, u & 1, status);
          if (ok) ok = issue_sdp(u + 1);
        }
        if (ok) ok = issue_dq(u);
      }
      umma_commit(&mma_final);
      mbar_wait(&mma_final, 0, status);
    }
    __syncwarp();
  } else {
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int i = q0 + r;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t* kbits = idx.keep_bits + (size_t)b * hdr.nwords;
    const int nwords = hdr.nwords;
    const bool row_live = i < L;
    const size_t ri = ((size_t)b * Hq + h) * L + (row_live ? i : 0);
    const float lse2 = row_live ? lse[ri] * kLog2e : 0.f;
    const float dlt = row_live ? delta[ri] : 0.f;
    bool ok = true;
    for (int u = 0; u < nT; ++u) {
      uint32_t vm[4];
      if (!row_live) {
        vm[0] = vm[1] = vm[2] = vm[3] = 0u;
      } else if (u < nG) {
        const int nv = min(128, n_gather - 128 * u);
#pragma unroll
        for (int w = 0; w < 4; ++w) vm[w] = range_bits(0, nv, w);
      } else {
        const int jt = lo + 128 * (u - nG);
        const int n_causal = min(128, max(0, i - jt + 1));
        const int c_win = i - n_win + 1 - jt;
        const int wj = jt >> 5, sh = jt & 31;
        uint32_t kw[5];
#pragma unroll
        for (int x = 0; x < 5; ++x) kw[x] = (wj + x < nwords) ? __ldg(kbits + wj + x) : 0u;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t keepw = sh ? ((kw[w] >> sh) | (kw[w + 1] << (32 - sh))) : kw[w];
          vm[w] = range_bits(0, n_causal, w) & (range_bits(c_win, 128, w) | keepw);
        }
      }
      if (!mbar_wait(&sd_full, u & 1, status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t dsk[64];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t sr[32], dr[32];
        tmem_ld32(tmem + lane_base + C::TM_S + 32 * cc, sr);
        tmem_ld32(tmem + lane_base + C::TM_DP + 32 * cc, dr);
        tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < 32; x += 2) {
          const bool v0 = (vm[cc] >> x) & 1u, v1 = (vm[cc] >> (x + 1)) & 1u;
          const float p0 = v0 ? fast_exp2(__uint_as_float(sr[x]) * scale_log2 - lse2) : 0.f;
          const float p1 = v1 ? fast_exp2(__uint_as_float(sr[x + 1]) * scale_log2 - lse2) : 0.f;
          dsk[(32 * cc + x) >> 1] = pack_bf16x2(p0 * (__uint_as_float(dr[x]) - dlt),
                                                p1 * (__uint_as_float(dr[x + 1]) - dlt));
        }
      }
      tc_fence_before();
      mbar_arrive(&sd_free);
      if (u > 0 && !mbar_wait(&dq_done, (u - 1) & 1, status)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int un = 0; un < 16; ++un) {
        const uint32_t off = (un >> 3) * kChunk + sw128_offset(r, (un & 7) * 8);
        *reinterpret_cast<uint4*>(sDS + off) =
            make_uint4(dsk[4 * un], dsk[4 * un + 1], dsk[4 * un + 2], dsk[4 * un + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&ds_full);
    }
    if (ok && mbar_wait(&dq_done, (nT - 1) & 1, status)) {
      tc_fence_after();
      uint32_t qb[32];
      __nv_bfloat16* qrow = dq + (((size_t)b * Hq + h) * L + i) * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        tmem_ld32(tmem + lane_base + C::TM_DQ + c0, qb);
        tmem_ld_wait();
        if (row_live) {
#pragma unroll
          for (int x = 0; x < 32; x += 8) {
            uint4 pk;
            pk.x = pack_bf16x2(__uint_as_float(qb[x]) * scale, __uint_as_float(qb[x + 1]) * scale);
            pk.y = pack_bf16x2(__uint_as_float(qb[x + 2]) * scale,
                               __uint_as_float(qb[x + 3]) * scale);
            pk.z = pack_bf16x2(__uint_as_float(qb[x + 4]) * scale,
                               __uint_as_float(qb[x + 5]) * scale);
            pk.w = pack_bf16x2(__uint_as_float(qb[x + 6]) * scale,
                               __uint_as_float(qb[x + 7]) * scale);
            *reinterpret_cast<uint4*>(qrow + c0 + x) = pk;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TM_COLS);
}

struct BwdWs {
  uint8_t *kk, *vk;
  float *dk_keep, *dv_keep, *delta;
  size_t total;
};

BwdWs bwd_ws(void* base, int B, int Hq, int Hkv, int L, int d) {
  BwdWs w;
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  const size_t kv_bf16 = align_up((size_t)B * Hkv * L * d * 2, 256);
  const size_t kv_f32 = align_up((size_t)B * Hkv * L * d * 4, 256);
  w.kk = p + off; off += kv_bf16;
  w.vk = p + off; off += kv_bf16;
  w.dk_keep = reinterpret_cast<float*>(p + off); off += kv_f32;
  w.dv_keep = reinterpret_cast<float*>(p + off); off += kv_f32;
  w.delta = reinterpret_cast<float*>(p + off); off += align_up((size_t)B * Hq * L * 4, 256);
  w.total = off;
  return w;
}

template <int D, int NST_KV, int NST_DQ>
int launch_bwd_impl(IndexPtrs idx, const void* q, const void* k, const void* v, const void* o,
                    const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                    int Hq, int Hkv, int L, float scale, void* ws, int* status,
                    cudaStream_t s) {
  const BwdWs w = bwd_ws(ws, B, Hq, Hkv, L, D);
  const int T = (L + 127) / 128;
  profile_mark(0, s);
  bwd_gather_kernel<D><<<dim3((L + 63) / 64, Hkv, B), 256, 0, s>>>(
      idx, static_cast<const uint4*>(k), static_cast<const uint4*>(v),
      reinterpret_cast<uint4*>(w.kk), reinterpret_cast<uint4*>(w.vk), Hkv, L);
  profile_mark(1, s);
  {
    const size_t rows = (size_t)B * Hq * L;
    const int delta_blocks =
        static_cast<int>((rows + prep_rows_per_block<D>() - 1) / prep_rows_per_block<D>());
    const int per_plane = (L * (D / 4) + kPrepThreads * 4 - 1) / (kPrepThreads * 4);
    bwd_prep_kernel<D><<<delta_blocks + B * Hkv * per_plane, kPrepThreads, 0, s>>>(
        idx, static_cast<const uint4*>(o), static_cast<const uint4*>(dout), w.delta,
        reinterpret_cast<float4*>(w.dk_keep), reinterpret_cast<float4*>(w.dv_keep), B, Hq, Hkv,
        L, delta_blocks);
  }
  CUtensorMap mq, mdo, mk, mv, mkk, mvk;
  if (!make_bf16_map(&mq, q, (uint64_t)B * Hq, L, D, 128) ||
      !make_bf16_map(&mdo, dout, (uint64_t)B * Hq, L, D, 128) ||
      !make_bf16_map(&mk, k, (uint64_t)B * Hkv, L, D, 128) ||
      !make_bf16_map(&mv, v, (uint64_t)B * Hkv, L, D, 128) ||
      !make_bf16_map(&mkk, w.kk, (uint64_t)B * Hkv, L, D, 128) ||
      !make_bf16_map(&mvk, w.vk, (uint64_t)B * Hkv, L, D, 128))
    return static_cast<int>(cudaErrorInvalidValue);
  const float scale_log2 = scale * kLog2e;
  using KC = KvCfg<D, NST_KV>;
  using QC = DqCfg<D, NST_DQ>;
  auto keep_k = bwd_kv_kernel<D, true, NST_KV>;
  auto dense_k = bwd_kv_kernel<D, false, NST_KV>;
  auto dq_k = bwd_dq_kernel<D, NST_DQ>;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(keep_k, cudaFuncAttributeMaxDynamicSharedMemorySize, KC::SMEM)) ||
      (e = cudaFuncSetAttribute(dense_k, cudaFuncAttributeMaxDynamicSharedMemorySize, KC::SMEM)) ||
      (e = cudaFuncSetAttribute(dq_k, cudaFuncAttributeMaxDynamicSharedMemorySize, QC::SMEM)))
    return static_cast<int>(e);
  __nv_bfloat16* dkb = static_cast<__nv_bfloat16*>(dk);
  __nv_bfloat16* dvb = static_cast<__nv_bfloat16*>(dv);
  profile_mark(2, s);
  keep_k<<<dim3(T * ((T + kKeepChunk - 1) / kKeepChunk), Hq, B), kThreads, KC::SMEM, s>>>(mkk, mvk, mq, mdo, idx, lse, w.delta,
                                                      w.dk_keep, w.dv_keep, dkb, dvb, B, Hq, Hkv,
                                                      L, scale, scale_log2, status);
  profile_mark(3, s);
  dense_k<<<dim3(T, Hkv, B), kThreads, KC::SMEM, s>>>(mk, mv, mq, mdo, idx, lse, w.delta,
                                                        w.dk_keep, w.dv_keep, dkb, dvb, B, Hq,
                                                        Hkv, L, scale, scale_log2, status);
  profile_mark(4, s);
  dq_k<<<dim3(T, Hq, B), kThreads, QC::SMEM, s>>>(mq, mdo, mk, mv, mkk, mvk, idx, lse, w.delta,
                                                    static_cast<__nv_bfloat16*>(dq), B, Hq, Hkv,
                                                    L, scale, scale_log2, status);
  const cudaError_t err = cudaGetLastError();
  profile_mark(5, s);
  return static_cast<int>(err);
}

}  // namespace

size_t attn_bwd_tc_workspace(int B, int Hq, int Hkv, int L, int d) {
  return bwd_ws(nullptr, B, Hq, Hkv, L, d).total;
}

int launch_attn_bwd_tc(IndexPtrs idx, const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                       int Hq, int Hkv, int L, int d, float scale, void* ws, int* status,
                       void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d == 64)
    return launch_bwd_impl<64, 2, 3>(idx, q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, L,
                                     scale, ws, status, s);
  return launch_bwd_impl<128, 1, 2>(idx, q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, L, scale,
                                    ws, status, s);
}

}  // namespace sep
