// Sep-Attention forward on the tcgen05 tensor cores (bf16 operands, fp32
// accumulation in tensor memory).
//
// What it computes: O = softmax(Q K^T * scale, masked) V and the row LSE
// under the SepLLM mask -- the first a tokens, every preceding separator and
// the n nearest tokens (SepLLM anthology record lit-748, Key takeaways,
// "The mask"; pith.science review, key_machinery).
//
// How: one CTA per (128-row query tile, q head, batch).  The tile's keys come
// from two sources, read from the index built by sep_build_index:
//   gathered tiles  the keep tokens before the tile's first window start,
//                   copied densely into K_keep / V_keep by gather_keep_kernel;
//                   the last one is masked by k < n_gather;
//   band tiles      the dense key range [dense_lo, dense_hi), masked per
//                   element by j <= i and (keep[j] or j >= i-n+1).
// Warp roles: warp 0 issues TMA loads (Q once, then K and V tiles through an
// NST-stage ring), warp 1 issues tcgen05.mma (S = Q K^T into one of NS TMEM
// buffers, O += P V into a TMEM accumulator), warps 2-5 run the softmax, one
// thread per query row: they read S with tcgen05.ld, apply the mask, keep a
// running max (rescaling O in TMEM only when the max grows by more than 2^8,
// which keeps every P <= 256 and the final O / l exact), write P as bf16 into
// shared memory in the 128-byte-swizzle K-major layout the MMA reads, and
// finally normalise O and store it with the LSE.
// Every mbarrier wait is bounded; on expiry the kernel records
// SEP_ERR_TIMEOUT, lets its copies and MMAs drain, frees TMEM and returns.
#include "common.cuh"
#include "layout.h"
#include "tma_host.h"

namespace sep {

namespace {

constexpr int kChunk = 128 * 128;  // bytes of a [128 rows x 64 cols] bf16 block

template <int D, int NS, int NST>
struct FwdCfg {
  static constexpr int DCH = D / 64;
  static constexpr int TILE = DCH * kChunk;  // one [128 x D] bf16 tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + TILE;
  static constexpr int OFF_V = OFF_K + NST * TILE;
  static constexpr int OFF_P = OFF_V + NST * TILE;
  static constexpr int SMEM = OFF_P + 2 * kChunk + 1024;
  static constexpr int TM_O = NS * 128;
  static constexpr int TM_USED = NS * 128 + D;
  static constexpr int TM_COLS = TM_USED <= 256 ? 256 : 512;
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

constexpr int kThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 softmax
constexpr float kRescaleLog2 = 8.0f;

template <int D>
__global__ void __launch_bounds__(256)
    gather_keep_kernel(IndexPtrs idx, const uint4* __restrict__ k, const uint4* __restrict__ v,
                       uint4* __restrict__ kk, uint4* __restrict__ vk, int Hkv, int L) {
  constexpr int U = D / 8;  // 16-byte units per row
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

template <int D, int NS, int NST>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_kk,
                       const __grid_constant__ CUtensorMap tm_vk, IndexPtrs idx,
                       __nv_bfloat16* __restrict__ o, float* __restrict__ lse, int B, int Hq,
                       int Hkv, int L, float scale_log2, int* status) {
  using C = FwdCfg<D, NS, NST>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t q_full, p_full, pv_done, mma_final;
  __shared__ __align__(8) uint64_t k_full[NST], v_full[NST], kv_empty[NST], s_full[NS];
  __shared__ uint32_t tmem_slot;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = (L + 127) >> 7;
  const int t = T - 1 - static_cast<int>(blockIdx.x);  // longest tiles first
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
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sP = smem + C::OFF_P;

  if (threadIdx.x == 0) {
    mbar_init(&q_full, 1);
    mbar_init(&p_full, 128);
    mbar_init(&pv_done, 1);
    mbar_init(&mma_final, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < NS; ++s) mbar_init(&s_full[s], 1);
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
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const int plane_q = b * Hq + h, plane_kv = b * Hkv + g;
      mbar_arrive_expect_tx(&q_full, C::TILE);
      for (int c = 0; c < C::DCH; ++c)
        tma_load_3d(sQ + c * kChunk, &tm_q, &q_full, 64 * c, q0, plane_q);
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
        mbar_arrive_expect_tx(&k_full[st], C::TILE);
        for (int c = 0; c < C::DCH; ++c)
          tma_load_3d(sK + st * C::TILE + c * kChunk, mk, &k_full[st], 64 * c, row, plane_kv);
        mbar_arrive_expect_tx(&v_full[st], C::TILE);
        for (int c = 0; c < C::DCH; ++c)
          tma_load_3d(sV + st * C::TILE + c * kChunk, mv, &v_full[st], 64 * c, row, plane_kv);
        issued = u + 1;
      }
      if (!ok) {
        // drain the copies still in flight before the CTA's smem goes away
        for (int u = issued - NST; u < issued; ++u) {
          if (u < 0) continue;
          mbar_wait(&k_full[u % NST], (u / NST) & 1, status);
          mbar_wait(&v_full[u % NST], (u / NST) & 1, status);
        }
        mbar_wait(&q_full, 0, status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, false, true);
      const uint32_t q_base = smem_u32(sQ), k_base = smem_u32(sK), v_base = smem_u32(sV),
                     p_base = smem_u32(sP);
      bool ok = mbar_wait(&q_full, 0, status);
      tc_fence_after();
      auto issue_qk = [&](int u) -> bool {
        const int st = u % NST;
        if (!mbar_wait(&k_full[st], (u / NST) & 1, status)) return false;
        tc_fence_after();
        const uint32_t d_tm = tmem + 128 * (u % NS);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
          umma_bf16_ss(d_tm, sdesc_sw128(q_base + off, 16, 1024),
                       sdesc_sw128(k_base + st * C::TILE + off, 16, 1024), idesc_qk, kk > 0);
        }
        umma_commit(&s_full[u % NS]);
        return true;
      };
      auto issue_pv = [&](int u) -> bool {
        const int st = u % NST;
        if (!mbar_wait(&p_full, u & 1, status)) return false;
        if (!mbar_wait(&v_full[st], (u / NST) & 1, status)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t aoff = (kk >> 2) * kChunk + (kk & 3) * 32;
          umma_bf16_ss(tmem + C::TM_O, sdesc_sw128(p_base + aoff, 16, 1024),
                       sdesc_sw128(v_base + st * C::TILE + kk * 2048, kChunk, 1024), idesc_pv,
                       (u > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&pv_done);
        umma_commit(&kv_empty[st]);
        return true;
      };
      if (ok) ok = issue_qk(0);
      for (int u = 0; ok && u < nT; ++u) {
        if (NS == 2 && u + 1 < nT) ok = issue_qk(u + 1);
        if (ok) ok = issue_pv(u);
        if (ok && NS == 1 && u + 1 < nT) ok = issue_qk(u + 1);
      }
      // every MMA issued by this thread completes before TMEM is released
      umma_commit(&mma_final);
      mbar_wait(&mma_final, 0, status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int i = q0 + r;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t* kbits = idx.keep_bits + (size_t)b * hdr.nwords;
    const int nwords = hdr.nwords;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    uint32_t sr[128];
    for (int u = 0; u < nT; ++u) {
      const int sb = u % NS;
      if (!mbar_wait(&s_full[sb], (u / NS) & 1, status)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_base + 128 * sb + 32 * c, sr + 32 * c);
      tmem_ld_wait();

      // visibility of the 128 columns as 4 words
      uint32_t vm[4];
      if (u < nG) {
        const int nv = min(128, n_gather - 128 * u);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const int c = nv - 32 * w;
          vm[w] = c >= 32 ? 0xffffffffu : (c <= 0 ? 0u : ((1u << c) - 1u));
        }
      } else {
        const int jt = lo + 128 * (u - nG);
        const int n_causal = min(128, max(0, i - jt + 1));  // columns c with jt+c <= i
        const int c_win = i - n_win + 1 - jt;               // columns c >= c_win are in the window
        const int wj = jt >> 5, sh = jt & 31;
        uint32_t kw[5];
#pragma unroll
        for (int x = 0; x < 5; ++x) kw[x] = (wj + x < nwords) ? __ldg(kbits + wj + x) : 0u;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t keepw = sh ? ((kw[w] >> sh) | (kw[w + 1] << (32 - sh))) : kw[w];
          const int cc = n_causal - 32 * w;
          const uint32_t causal = cc >= 32 ? 0xffffffffu : (cc <= 0 ? 0u : ((1u << cc) - 1u));
          const int cw = c_win - 32 * w;  // bits >= cw
          const uint32_t win = cw <= 0 ? 0xffffffffu : (cw >= 32 ? 0u : ~((1u << cw) - 1u));
          vm[w] = causal & (win | keepw);
        }
      }
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        const float x = ((vm[c >> 5] >> (c & 31)) & 1u) ? __uint_as_float(sr[c]) * scale_log2
                                                         : -INFINITY;
        sr[c] = __float_as_uint(x);
        mt = fmaxf(mt, x);
      }
      const float m_new = fmaxf(m_used, mt);
      const bool rescale = m_new > m_used + kRescaleLog2;
      float alpha = 1.f;
      if (rescale) {
        alpha = fast_exp2(m_used - m_new);
        m_used = m_new;
      }
      const float msub = (m_used == -INFINITY) ? 0.f : m_used;
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < 128; c += 2) {
        const float p0 = fast_exp2(__uint_as_float(sr[c]) - msub);
        const float p1 = fast_exp2(__uint_as_float(sr[c + 1]) - msub);
        rs += p0 + p1;
        sr[c >> 1] = pack_bf16x2(p0, p1);
      }
      l = l * alpha + rs;

      if (u > 0) {
        if (!mbar_wait(&pv_done, (u - 1) & 1, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, rescale)) {
          uint32_t ob[32];
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            tmem_ld32(tmem + lane_base + C::TM_O + c0, ob);
            tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 32; ++x) ob[x] = __float_as_uint(__uint_as_float(ob[x]) * alpha);
            tmem_st32(tmem + lane_base + C::TM_O + c0, ob);
          }
          tmem_st_wait();
        }
      }
      // P row -> shared memory, 128-byte swizzle, two 64-key blocks
#pragma unroll
      for (int un = 0; un < 16; ++un) {
        const uint32_t off = (un >> 3) * kChunk + sw128_offset(r, (un & 7) * 8);
        *reinterpret_cast<uint4*>(sP + off) =
            make_uint4(sr[4 * un], sr[4 * un + 1], sr[4 * un + 2], sr[4 * un + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full);
    }
    if (ok && mbar_wait(&pv_done, (nT - 1) & 1, status)) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      uint32_t ob[32];
      __nv_bfloat16* orow = o + (((size_t)b * Hq + h) * L + i) * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        tmem_ld32(tmem + lane_base + C::TM_O + c0, ob);
        tmem_ld_wait();
        if (i < L) {
#pragma unroll
          for (int x = 0; x < 32; x += 8) {
            uint4 pk;
            pk.x = pack_bf16x2(__uint_as_float(ob[x]) * inv_l, __uint_as_float(ob[x + 1]) * inv_l);
            pk.y = pack_bf16x2(__uint_as_float(ob[x + 2]) * inv_l,
                               __uint_as_float(ob[x + 3]) * inv_l);
            pk.z = pack_bf16x2(__uint_as_float(ob[x + 4]) * inv_l,
                               __uint_as_float(ob[x + 5]) * inv_l);
            pk.w = pack_bf16x2(__uint_as_float(ob[x + 6]) * inv_l,
                               __uint_as_float(ob[x + 7]) * inv_l);
            *reinterpret_cast<uint4*>(orow + c0 + x) = pk;
          }
        }
      }
      if (i < L)
        lse[((size_t)b * Hq + h) * L + i] = (m_used + __log2f(l)) * 0.69314718055994531f;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TM_COLS);
}

template <int D, int NS, int NST>
int launch_fwd_impl(IndexPtrs idx, const void* q, const void* k, const void* v, void* o, float* lse,
                    int B, int Hq, int Hkv, int L, float scale, void* ws, int* status,
                    cudaStream_t s) {
  using C = FwdCfg<D, NS, NST>;
  const size_t plane_elems = (size_t)L * D;
  uint8_t* kk = static_cast<uint8_t*>(ws);
  uint8_t* vk = kk + align_up((size_t)B * Hkv * plane_elems * 2, 256);
  dim3 ggrid((L + 63) / 64, Hkv, B);
  profile_mark(0, s);
  gather_keep_kernel<D><<<ggrid, 256, 0, s>>>(idx, static_cast<const uint4*>(k),
                                               static_cast<const uint4*>(v),
                                               reinterpret_cast<uint4*>(kk),
                                               reinterpret_cast<uint4*>(vk), Hkv, L);
  CUtensorMap mq, mk, mv, mkk, mvk;
  if (!make_bf16_map(&mq, q, (uint64_t)B * Hq, L, D, 128) ||
      !make_bf16_map(&mk, k, (uint64_t)B * Hkv, L, D, 128) ||
      !make_bf16_map(&mv, v, (uint64_t)B * Hkv, L, D, 128) ||
      !make_bf16_map(&mkk, kk, (uint64_t)B * Hkv, L, D, 128) ||
      !make_bf16_map(&mvk, vk, (uint64_t)B * Hkv, L, D, 128))
    return static_cast<int>(cudaErrorInvalidValue);
  auto kern = attn_fwd_tc_kernel<D, NS, NST>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return static_cast<int>(e);
  const float scale_log2 = scale * 1.4426950408889634f;
  dim3 grid((L + 127) / 128, Hq, B);
  profile_mark(1, s);
  kern<<<grid, kThreads, C::SMEM, s>>>(mq, mk, mv, mkk, mvk, idx,
                                       static_cast<__nv_bfloat16*>(o), lse, B, Hq, Hkv, L,
                                       scale_log2, status);
  const cudaError_t err = cudaGetLastError();
  profile_mark(2, s);
  return static_cast<int>(err);
}

}  // namespace

size_t attn_fwd_tc_workspace(int B, int Hkv, int L, int d) {
  return 2 * align_up((size_t)B * Hkv * L * d * 2, 256);
}

int launch_attn_fwd_tc(IndexPtrs idx, const void* q, const void* k, const void* v, void* o,
                       float* lse, int B, int Hq, int Hkv, int L, int d, float scale, void* ws,
                       int* status, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d == 64) return launch_fwd_impl<64, 2, 3>(idx, q, k, v, o, lse, B, Hq, Hkv, L, scale, ws,
                                                status, s);
  return launch_fwd_impl<128, 2, 2>(idx, q, k, v, o, lse, B, Hq, Hkv, L, scale, ws, status, s);
}

}  // namespace sep
