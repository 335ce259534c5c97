// Streaming four-block KV cache (initial, separator, past window, local
// window) and decode attention with position shifting.
//
// What it computes (pith.science review of arXiv 2412.12094, key_machinery;
// paperhub rebuttal, reply A1 to the second reviewer):
//   update  when the cache holds exactly c entries, the past window's
//           separators move, oldest first, into the separator block (whose
//           oldest entries beyond s are dropped) and the rest of the past
//           window is dropped; then the new token enters the initial block
//           while it holds fewer than a entries, else the local window, whose
//           oldest entry spills into the past window once it holds more
//           than w.
//   attend  out = softmax(rope(q, N-1) . rope(K_k, k) * scale) V over the
//           N entries in logical order initial + separator + past + local,
//           entry k at position k (its rank in the cache, not its text
//           position).
//
// Storage: keys are kept un-rotated in bf16, so a position shift never
// rewrites them and the cache contents stay bit-exact; RoPE is applied on
// load.  Each sequence owns a + s + (c - a) slots per kv head: the initial
// block, a ring of s separator slots and a ring of c - a slots holding the
// past and local windows (one contiguous stretch of text).  Logical entry k
// maps to its slot through the ring heads, and attention reduces in logical
// order, so the outputs do not depend on where the rings happen to start.
//
// One step is one launch: a cluster of `split` CTAs per (sequence, kv head).
// Every CTA reads the (sequence, head)'s counters and derives the layout the
// cache will have after this step's update; it then attends over its share
// of the entries in that layout, reading each entry from where it sits
// *before* the update (a separator that moves this step is read from its
// window slot, the new token from the caller's k_new / v_new).  A producer
// warp stages the rows in shared memory with 16-byte asynchronous copies;
// two consumer warps score them and accumulate P.V on the tensor cores
// (mma.sync, bf16 in, fp32 out), rotating keys by RoPE in registers at
// their cache rank.  The partial softmax states
// merge over distributed shared memory, and only after the whole cluster has
// finished reading does CTA 0 write the update (moves, new row, flags,
// counters).  Counters and flags are kept per (sequence, kv head), so no
// cluster ever waits for another.
#include <math.h>
#include <string.h>

#include <vector>

#include "common.cuh"
#include "layout.h"

#define SEP_API extern "C" __attribute__((visibility("default")))

namespace sep {

namespace {

constexpr int kCacheMagic = 0x43504553;  // 'SEPC'
constexpr int kConsumerWarps = 2;        // score / softmax / P.V warps
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one copy producer warp
constexpr int kWarps = kThreads / 32;
constexpr int kMaxC = 1024;              // survivor list is kept in shared memory
constexpr int kMaxHkv = 64;
constexpr int kMaxSplit = 8;             // portable cluster size
constexpr float kLazyRescale = 8.0f;     // log2 growth of the max before a rescale
constexpr int kTargetCtas = 296;         // CTAs per step the split aims at (2 per SM)

struct CacheLayout {
  int S, Hkv, d, a, s, w, c, NSL, rope_rows;
  size_t meta, rope, invf, pos, issep, k, v, total;
};

// Counters of one (sequence, kv head) (int32 x 8 in device memory).  Every
// kv head of a sequence holds the same values; each cluster updates its own
// copy.
struct Meta {
  int n_init, n_sep, sep_head, n_pw, pw_head, t, pad0, pad1;
};

bool params_ok(const sep_cache_params* p) {
  return p && p->S >= 1 && p->Hkv >= 1 && p->d >= 1 && p->a >= 0 && p->s >= 0 && p->w >= 1 &&
         p->c >= 1;
}

CacheLayout cache_layout(const sep_cache_params* p) {
  CacheLayout l;
  l.S = p->S; l.Hkv = p->Hkv; l.d = p->d; l.a = p->a; l.s = p->s; l.w = p->w; l.c = p->c;
  l.NSL = p->a + p->s + (p->c - p->a);
  l.rope_rows = p->c > 64 ? p->c : 64;  // rows 16 and 32 hold the recurrence steps
  size_t off = 0;
  l.meta = off;
  off = align_up(off + sizeof(Meta) * (size_t)l.S * l.Hkv, 256);
  l.rope = off;
  off = align_up(off + sizeof(float2) * (size_t)l.rope_rows * (l.d / 2), 256);
  l.invf = off;  // inv_freq_i = theta^(-2i/d), float32 [d/2]
  off = align_up(off + sizeof(float) * (size_t)(l.d / 2), 256);
  l.pos = off;
  off = align_up(off + sizeof(int32_t) * (size_t)l.S * l.NSL, 256);
  l.issep = off;
  off = align_up(off + (size_t)l.S * l.Hkv * l.NSL, 256);
  l.k = off;
  off = align_up(off + 2 * (size_t)l.S * l.Hkv * l.NSL * l.d, 256);
  l.v = off;
  off = align_up(off + 2 * (size_t)l.S * l.Hkv * l.NSL * l.d, 256);
  l.total = off;
  return l;
}

struct CachePtrs {
  Meta* meta;
  const float2* rope;
  const float* invf;
  int32_t* pos;
  uint8_t* issep;
  uint16_t* k;
  uint16_t* v;
};

CachePtrs cache_ptrs(void* buf, const CacheLayout& l) {
  char* b = static_cast<char*>(buf);
  CachePtrs p;
  p.meta = reinterpret_cast<Meta*>(b + l.meta);
  p.rope = reinterpret_cast<const float2*>(b + l.rope);
  p.invf = reinterpret_cast<const float*>(b + l.invf);
  p.pos = reinterpret_cast<int32_t*>(b + l.pos);
  p.issep = reinterpret_cast<uint8_t*>(b + l.issep);
  p.k = reinterpret_cast<uint16_t*>(b + l.k);
  p.v = reinterpret_cast<uint16_t*>(b + l.v);
  return p;
}

struct StepArgs {
  int S, Hkv, Hq, a, s, w, c, NSL, split;
  float scale_log2;
  SepIdList sids;
};

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ float dsmem_ld(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// The layout after this step's update, expressed through where each entry
// sits before it:
//   [0, I0)                 initial slots 0 .. I0-1
//   [I0, I0+SK)             kept separator-ring entries from ring offset sk0
//   [.., +SV)               separators moving out of the past window now
//                           (window-ring slots in surv_src)
//   [.., +W0)               window-ring entries from ring position pw0
//   N-1                     the new token (caller's k_new / v_new)
struct StepPlan {
  int I0, SK, SV, W0, N;
  int sk0, pw0;
};

// Streaming shape of the decode attention.  A chunk is 16 entries per
// consumer warp; NST chunks of K and V rows are in flight.  The producer
// warp copies them 16 bytes at a time (cp.async) into rows of PU 16-byte
// units (one more than a row holds), unit u of row r at position u ^ ((r >>
// 1) & 7): with that pitch and swizzle the consumers' fragment loads (16-byte
// reads of eight rows at once) touch all 32 banks without conflict.
template <int D>
struct StreamShape {
  static constexpr int HALF = D / 2;
  static constexpr int CPR = D / 8;               // 16-byte units of a K / V row
  static constexpr int CH = kConsumerWarps * 16;  // entries per chunk
  static constexpr int PU = CPR + 1;              // units per staged row
  static constexpr int NST = 3;                   // ring stages
  static constexpr int OFF_V = CH * PU * 16;
  static constexpr int STAGE = 2 * CH * PU * 16;  // bytes: K rows, V rows
  static constexpr int NSLAB = D / 16;            // 16-wide k slabs of a row
  static constexpr int NLO = D / 32;              // slabs of the first half
  static constexpr int LD = D / 8;                // dims of each half a lane holds
  static constexpr int MT = D / 16;               // 16-dim m-tiles of the output
};

// Byte offset of unit u of staged row r.
__device__ __forceinline__ int staged_unit(int r, int u, int pu) {
  return (r * pu + (u ^ ((r >> 1) & 7))) * 16;
}

// 16-byte global -> shared copy (cp.async, L2 only) and the arrive on an
// mbarrier once every cp.async this thread issued so far has landed (the
// arrive counts toward the barrier's expected arrivals).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Dynamic shared memory of the step kernel (byte offsets, 16-byte aligned).
struct StepSmem {
  int ring, q, wstate, part, surv, slots, total;
};

template <int D, int G>
__host__ __device__ inline StepSmem step_smem(int s_cap, int c_cap) {
  using SS = StreamShape<D>;
  auto al = [](int x) { return (x + 15) / 16 * 16; };
  StepSmem m;
  int off = 0;
  m.ring = off;
  off += SS::NST * SS::STAGE;
  // the merge state overlays the ring: it is written only once every chunk
  // has been consumed
  m.wstate = 0;  // per consumer warp: acc[G][D], m[G], l[G]
  m.part = al(kConsumerWarps * G * (D + 2) * 4);  // merged partial: acc[G][D], m[G], l[G]
  m.q = off;
  off += al(G * D * 4);
  m.surv = off;    // surviving separators: window slot, text position
  off += al(2 * (s_cap > 0 ? s_cap : 1) * 4);
  m.slots = off;   // slot of each entry of this CTA's share (-1: the new token)
  off += al(c_cap * 4);
  m.total = off;
  return m;
}

static_assert(kConsumerWarps * 8 * (128 + 2) * 4 + 8 * (128 + 2) * 4 <=
                  StreamShape<64>::NST * StreamShape<64>::STAGE,
              "merge state fits in the ring");


// D (fp32 16x8) += A (bf16 16x16, row) * B (bf16 16x8, col): the warp-level
// tensor-core product.  Fragments (g = lane / 4, t = lane % 4): a0 = A[g][2t,
// 2t+1], a1 = A[g+8][2t, 2t+1], a2 = A[g][2t+8, 2t+9], a3 = A[g+8][2t+8, 2t+9];
// b0 = B[2t, 2t+1][g], b1 = B[2t+8, 2t+9][g]; d0 = D[g][2t], d1 = D[g][2t+1],
// d2 = D[g+8][2t], d3 = D[g+8][2t+1].  Lower index in the low 16 bits.
__device__ __forceinline__ void mma_bf16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 b16 matrix held as one b16x2 per lane (row lane / 4,
// columns 2 (lane % 4), +1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t word_of(const uint4& u, int i) {
  return i == 0 ? u.x : i == 1 ? u.y : i == 2 ? u.z : u.w;
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}
// The consumer warps publish the slot list to the copy warp through named
// barrier 2: they arrive without waiting, the copy warp waits.
__device__ __forceinline__ void slots_published() {
  asm volatile("bar.arrive 2, %0;" ::"n"(kThreads) : "memory");
}
__device__ __forceinline__ void wait_slots_published() {
  asm volatile("bar.sync 2, %0;" ::"n"(kThreads) : "memory");
}

// ---------------------------------------------------------------------------
// The step kernel
// ---------------------------------------------------------------------------
template <int D, int G>
__global__ void __launch_bounds__(kThreads, 4)
    cache_step_kernel(CachePtrs cp, StepArgs args, const uint16_t* __restrict__ q,
                      const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
                      const int32_t* __restrict__ ids_new, uint16_t* __restrict__ out,
                      int* status) {
  using SS = StreamShape<D>;
  constexpr int HALF = SS::HALF, CPR = SS::CPR, CH = SS::CH, NST = SS::NST;
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ int warp_cnt[kWarps];
  __shared__ __align__(8) uint64_t full_bar[NST], empty_bar[NST];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = blockIdx.x, g = blockIdx.y, sq = blockIdx.z;
  const int split = args.split;
  const int a = args.a, s = args.s, w = args.w, c = args.c, NSL = args.NSL;
  const int ring = c - a;
  const bool attend = q != nullptr && out != nullptr;
  const StepSmem L = step_smem<D, G>(s, c);
  float* sQ = reinterpret_cast<float*>(dsm + L.q);
  float* sW = reinterpret_cast<float*>(dsm + L.wstate);
  float* sAcc = reinterpret_cast<float*>(dsm + L.part);
  float* sM = sAcc + G * D;
  float* sL = sM + G;
  int* surv_src = reinterpret_cast<int*>(dsm + L.surv);
  int* surv_pos = surv_src + (s > 0 ? s : 1);

  const size_t mh = (size_t)sq * args.Hkv + g;  // (sequence, kv head)
  // the G query heads' values, loaded by the consumer threads before the
  // plan so that their latency passes while it is made
  constexpr int QPER = (G * HALF + kConsumerWarps * 32 - 1) / (kConsumerWarps * 32);
  float qx1[QPER], qx2[QPER];
#pragma unroll
  for (int j = 0; j < QPER; ++j) {
    const int e = tid + j * kConsumerWarps * 32;
    qx1[j] = qx2[j] = 0.f;
    if (q != nullptr && warp < kConsumerWarps && e < G * HALF) {
      const uint16_t* qr = q + (((size_t)sq * args.Hq) + g * G + e / HALF) * D;
      qx1[j] = __uint_as_float((uint32_t)qr[e % HALF] << 16);
      qx2[j] = __uint_as_float((uint32_t)qr[e % HALF + HALF] << 16);
    }
  }
  // the copy ring's barriers, initialised before any role can touch them
  if (tid == 0) {
    for (int st = 0; st < NST; ++st) {
      mbar_init(&full_bar[st], 32);  // the copy lanes' cp.async arrivals
      mbar_init(&empty_bar[st], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const Meta m = cp.meta[mh];
  const uint8_t* sepr = cp.issep + mh * NSL;
  const bool ok = !(m.n_init < 0 || m.n_init > a || m.n_sep < 0 || m.n_sep > s || m.n_pw < 0 ||
                    m.n_pw > ring || m.sep_head < 0 || (s > 0 && m.sep_head >= s) ||
                    m.pw_head < 0 || m.pw_head >= ring || m.n_init + m.n_sep + m.n_pw > c ||
                    (m.n_init < a && (m.n_sep | m.n_pw) != 0));

  // ---- plan this step's update (identical in every CTA of the cluster)
  Meta nm = m;
  StepPlan pl;
  pl.I0 = m.n_init; pl.SK = m.n_sep; pl.SV = 0; pl.W0 = m.n_pw;
  pl.sk0 = m.sep_head; pl.pw0 = m.pw_head;
  const bool compress = ok && (m.n_init + m.n_sep + m.n_pw == c);
  if (compress) {
    const int n_win = min(w, m.n_pw);
    const int n_past = m.n_pw - n_win;
    // pass 1: separators in the past window
    int ms = 0;
    for (int k0 = 0; k0 < n_past; k0 += kThreads) {
      const int k = k0 + tid;
      const bool is_s = k < n_past && sepr[a + s + (m.pw_head + k) % ring] != 0;
      const uint32_t bal = __ballot_sync(0xffffffffu, is_s);
      if (lane == 0) warp_cnt[warp] = __popc(bal);
      __syncthreads();
      for (int x = 0; x < kWarps; ++x) ms += warp_cnt[x];
      __syncthreads();
    }
    // pass 2: the last min(ms, s) of them survive, oldest first
    const int first = max(0, ms - s);
    int base = 0;
    for (int k0 = 0; k0 < n_past; k0 += kThreads) {
      const int k = k0 + tid;
      const int slot = a + s + (m.pw_head + k) % ring;
      const bool is_s = k < n_past && sepr[slot] != 0;
      const uint32_t bal = __ballot_sync(0xffffffffu, is_s);
      if (lane == 0) warp_cnt[warp] = __popc(bal);
      __syncthreads();
      int before = base, tot = 0;
      for (int x = 0; x < kWarps; ++x) {
        if (x < warp) before += warp_cnt[x];
        tot += warp_cnt[x];
      }
      const int r = before + __popc(bal & ((1u << lane) - 1u));
      if (is_s && r >= first) {
        surv_src[r - first] = slot;
        // text positions are kept once per sequence, by kv head 0's cluster
        surv_pos[r - first] = g == 0 ? cp.pos[(size_t)sq * NSL + slot] : 0;
      }
      base += tot;
      __syncthreads();
    }
    const int n_surv = ms - first;
    const int drop = max(0, m.n_sep + ms - s);
    nm.sep_head = s > 0 ? (m.sep_head + drop) % s : 0;
    nm.n_sep = m.n_sep + ms - drop;
    nm.pw_head = (m.pw_head + n_past) % ring;
    nm.n_pw = n_win;
    pl.SV = n_surv;
    pl.SK = nm.n_sep - n_surv;
    pl.sk0 = nm.sep_head;  // the kept old entries start where the ring now starts
    pl.W0 = n_win;
    pl.pw0 = nm.pw_head;
  }
  int new_slot = 0;
  if (ok) {
    if (nm.n_init < a) {
      new_slot = nm.n_init;
      nm.n_init += 1;
    } else {
      new_slot = a + s + (nm.pw_head + nm.n_pw) % ring;
      nm.n_pw += 1;
    }
    nm.t = m.t + 1;
  }
  pl.N = pl.I0 + pl.SK + pl.SV + pl.W0 + 1;
  // CTA 0 writes the new token's rows at the end: fetch them now
  uint4 nk = make_uint4(0u, 0u, 0u, 0u), nvv = nk;
  int32_t new_id = 0;
  if (rank == 0 && ok && tid < CPR) {
    nk = *reinterpret_cast<const uint4*>(k_new + mh * D + 8 * tid);
    nvv = *reinterpret_cast<const uint4*>(v_new + mh * D + 8 * tid);
    new_id = ids_new[sq];
  }

  // ---- attention over this CTA's share [k0, k1) of the new layout, streamed
  // in chunks of CH entries through an NST-stage ring of asynchronous copies
  bool att_ok = ok && attend;
  const size_t head_off = mh * (size_t)NSL * D;
  if (attend) {
    const int N = pl.N;
    const int k0 = (int)(((long long)N * rank) / split);
    const int k1 = (int)(((long long)N * (rank + 1)) / split);
    const int ne = ok ? k1 - k0 : 0;
    const int n_chunks = (ne + CH - 1) / CH;
    // where each entry of the share sits before the update (-1: the new
    // token, read from the caller's input)
    const int rS = pl.I0, rV = rS + pl.SK, rW = rV + pl.SV, rN = N - 1;
    auto slot_of = [&](int e) -> int {
      if (e == rN) return -1;
      if (e < rS) return e;
      if (e < rV) {
        const int x = pl.sk0 + (e - rS);  // < 2 s
        return a + (x >= s ? x - s : x);
      }
      if (e < rW) return surv_src[e - rV];
      const int x = pl.pw0 + (e - rW);  // < 2 ring
      return a + s + (x >= ring ? x - ring : x);
    };
    int* slots = reinterpret_cast<int*>(dsm + L.slots);
    const uint16_t* kh = cp.k + head_off;
    const uint16_t* vh = cp.v + head_off;
    const size_t new_off = mh * D;  // [S][Hkv][D] inputs
    // The copy warp's copies of chunk ch, entries [c0, c0 + n): each lane
    // copies 16-byte units of their K and V rows, from their slots in
    // `slots`, then arrives on the stage's full barrier.
    auto issue_chunk = [&](int ch) {
      const int st = ch % NST;
      const int c0 = k0 + ch * CH, n = min(k1, c0 + CH) - c0;
      uint8_t* stg = dsm + L.ring + st * SS::STAGE;
      const int* sl_c = slots + (c0 - k0);
      // lane l copies unit l % CPR of rows l / CPR, l / CPR + 32 / CPR, ...
      constexpr int RPI = 32 / CPR;  // rows per pass of the warp
      const int u = lane % CPR, r0 = lane / CPR;
      auto copy_row = [&](int r) {
        const int slot = sl_c[r];
        const uint16_t* bk = slot < 0 ? k_new + new_off : kh + (size_t)slot * D;
        const uint16_t* bv = slot < 0 ? v_new + new_off : vh + (size_t)slot * D;
        const int du = staged_unit(r, u, SS::PU);
        cp_async16(stg + du, bk + 8 * u);
        cp_async16(stg + SS::OFF_V + du, bv + 8 * u);
      };
      if (n == CH) {  // a full chunk: a fixed trip count the compiler unrolls
#pragma unroll
        for (int r = r0; r < CH; r += RPI) copy_row(r);
      } else {
        for (int r = r0; r < n; r += RPI) copy_row(r);
      }
      cp_async_arrive(&full_bar[st]);
    };
    if (warp == kConsumerWarps) {
      // the copy warp starts the first chunk from slots it computes itself,
      // while the consumer warps list the rest
      if (lane < min(ne, CH)) slots[lane] = slot_of(k0 + lane);
      __syncwarp();
      if (ne > 0) issue_chunk(0);
      wait_slots_published();
    } else {
      for (int e = k0 + CH + tid; e < k0 + ne; e += kConsumerWarps * 32)
        slots[e - k0] = slot_of(e);
      slots_published();
      if (ok) {
        // rotated queries of the G heads at position N-1 into sQ[h][D] (fp32)
        const float2* cs_row = cp.rope + (size_t)(N - 1) * HALF;
#pragma unroll
        for (int j = 0; j < QPER; ++j) {
          const int e = tid + j * kConsumerWarps * 32;
          if (e < G * HALF) {
            const int hh = e / HALF, i = e % HALF;
            const float2 cs = cs_row[i];
            const float x1 = qx1[j], x2 = qx2[j];
            sQ[hh * D + i] = x1 * cs.x - x2 * cs.y;
            sQ[hh * D + i + HALF] = x2 * cs.x + x1 * cs.y;
          }
        }
      }
      consumer_sync();
    }

    if (warp == kConsumerWarps) {
      // ------------------------------------------------------------ producer
      // chunk 0 is issued; chunk ch reuses the stage of chunk ch - NST once
      // both consumer warps have released it
      if (ne > 0) {
        for (int ch = 1; ch < n_chunks; ++ch) {
          if (ch >= NST &&
              !mbar_wait_warp(&empty_bar[ch % NST], ((ch / NST) - 1) & 1, status))
            break;
          issue_chunk(ch);
        }
        // nothing this lane copies may land after the CTA is gone
        asm volatile("cp.async.wait_all;" ::: "memory");
      }
    } else {
      // ------------------------------------------------------------ consumers
      // Warp w owns entries [16w, 16w + 16) of every chunk.  Per chunk:
      //   S^T = Krot Q^T on the tensor cores (m = 16 entries, n = 8 heads,
      //   k = d), Krot = K rotated by RoPE at the entry's rank, in registers;
      //   online softmax per head (lazy rescale);
      //   O^T += V^T P^T (m = 16 dims, n = 8 heads, k = 16 entries), P^T by
      //   an in-register transpose of the S^T fragments.
      // Lane (g, t) = (lane / 4, lane % 4).  In the QK product its k columns
      // {2t, 2t+1, 2t+8, 2t+9} of slab s are dims LD t + 4s + {0..3} of the
      // first half (slabs s < NLO) or the same dims + HALF (slabs NLO + s):
      // the pairs RoPE rotates together stay in one lane.  In the PV product
      // its m rows g, g+8 of m-tile mt are dims LD g + mt and LD g + MT + mt.
      constexpr int LD = SS::LD, NLO = SS::NLO, MT = SS::MT;
      const int gq = lane >> 2, tq = lane & 3;
      // Q^T fragments (B operand): b0 = q[gq][dims +0, +1], b1 = q[gq][+2, +3]
      uint32_t qf[SS::NSLAB][2];
#pragma unroll
      for (int sl = 0; sl < SS::NSLAB; ++sl) {
        const int dim = (sl < NLO ? 0 : HALF) + LD * tq + 4 * (sl % NLO);
        if (gq < G) {
          const float* qrow = sQ + gq * D + dim;
          qf[sl][0] = pack_bf16x2(qrow[0], qrow[1]);
          qf[sl][1] = pack_bf16x2(qrow[2], qrow[3]);
        } else {
          qf[sl][0] = qf[sl][1] = 0u;
        }
      }
      const bool hv0 = 2 * tq < G, hv1 = 2 * tq + 1 < G;  // heads 2t, 2t+1 exist
      // inv_freq of the lane's frequencies LD t .. LD t + LD - 1
      float ifr[LD];
#pragma unroll
      for (int j = 0; j < LD; ++j) ifr[j] = cp.invf[LD * tq + j];
      float acc[MT][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
      float mrun0 = -INFINITY, mrun1 = -INFINITY, lrun0 = 0.f, lrun1 = 0.f;
      for (int ch = 0; ch < n_chunks; ++ch) {
        const int st = ch % NST;
        const int c0 = k0 + ch * CH;
        const int nv = min(k1, c0 + CH) - c0;  // live entries of the chunk
        const int e0 = 16 * warp;             // this warp's first chunk row
        const int rg = e0 + gq, rg8 = rg + 8;
        const bool live_g = rg < nv, live_g8 = rg8 < nv;
        if (!mbar_wait(&full_bar[st], (ch / NST) & 1, status)) {
          att_ok = false;
          break;
        }
        const uint8_t* sK = dsm + L.ring + st * SS::STAGE;
        const uint8_t* sV = sK + SS::OFF_V;
        const float pos_g = static_cast<float>(c0 + rg);
        // ---- S^T = Krot Q^T
        // two accumulators (first / second half slabs) halve the MMA chain
        float sacc[4] = {0.f, 0.f, 0.f, 0.f}, sacc2[4] = {0.f, 0.f, 0.f, 0.f};
        {
          // K units of the lane's dims: first half units (LD / 8) t + u,
          // second half HALF / 8 + (LD / 8) t + u (rows of dead entries hold
          // stale values; their scores are masked)
          uint4 klo[2][LD / 8], khi[2][LD / 8];
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            const int r = x ? rg8 : rg;
#pragma unroll
            for (int u = 0; u < LD / 8; ++u) {
              klo[x][u] = *reinterpret_cast<const uint4*>(
                  sK + staged_unit(r, (LD / 8) * tq + u, SS::PU));
              khi[x][u] = *reinterpret_cast<const uint4*>(
                  sK + staged_unit(r, HALF / 8 + (LD / 8) * tq + u, SS::PU));
            }
          }
#pragma unroll
          for (int sl = 0; sl < NLO; ++sl) {
            uint32_t alo[2][2], ahi[2][2];  // [entry g / g+8][dims +0/+1, +2/+3]
            // (cos, sin) of freqs LD t + 4 sl + 0..3 at entry g's rank, and
            // at entry g+8's (8 ranks on: the angle-addition formulas with
            // (cos, sin)(8 theta_i), row 8 of the table)
            float4 cg01, cg23, cq01, cq23;
            __sincosf(pos_g * ifr[4 * sl], &cg01.y, &cg01.x);
            __sincosf(pos_g * ifr[4 * sl + 1], &cg01.w, &cg01.z);
            __sincosf(pos_g * ifr[4 * sl + 2], &cg23.y, &cg23.x);
            __sincosf(pos_g * ifr[4 * sl + 3], &cg23.w, &cg23.z);
            {
              const float4* r8 = reinterpret_cast<const float4*>(cp.rope + 8 * HALF + LD * tq + 4 * sl);
              const float4 e01 = r8[0], e23 = r8[1];  // (cos, sin) of 8 theta, two freqs each
              float t0, t1;
              fmul2(t0, t1, cg01.y, cg01.w, e01.y, e01.w);
              ffma2(cq01.x, cq01.z, cg01.x, cg01.z, e01.x, e01.z, -t0, -t1);
              fmul2(t0, t1, cg01.x, cg01.z, e01.y, e01.w);
              ffma2(cq01.y, cq01.w, cg01.y, cg01.w, e01.x, e01.z, t0, t1);
              fmul2(t0, t1, cg23.y, cg23.w, e23.y, e23.w);
              ffma2(cq23.x, cq23.z, cg23.x, cg23.z, e23.x, e23.z, -t0, -t1);
              fmul2(t0, t1, cg23.x, cg23.z, e23.y, e23.w);
              ffma2(cq23.y, cq23.w, cg23.y, cg23.w, e23.x, e23.z, t0, t1);
            }
#pragma unroll
            for (int x = 0; x < 2; ++x) {
              const float4 c01 = x ? cq01 : cg01, c23 = x ? cq23 : cg23;
              const uint32_t l01 = word_of(klo[x][sl / 2], 2 * (sl % 2));
              const uint32_t l23 = word_of(klo[x][sl / 2], 2 * (sl % 2) + 1);
              const uint32_t h01 = word_of(khi[x][sl / 2], 2 * (sl % 2));
              const uint32_t h23 = word_of(khi[x][sl / 2], 2 * (sl % 2) + 1);
              float rl0, rl1, rl2, rl3, rh0, rh1, rh2, rh3, t0, t1;
              // rl = lo cos - hi sin; rh = hi cos + lo sin
              fmul2(t0, t1, bf_lo(h01), bf_hi(h01), c01.y, c01.w);
              ffma2(rl0, rl1, bf_lo(l01), bf_hi(l01), c01.x, c01.z, -t0, -t1);
              fmul2(t0, t1, bf_lo(l01), bf_hi(l01), c01.y, c01.w);
              ffma2(rh0, rh1, bf_lo(h01), bf_hi(h01), c01.x, c01.z, t0, t1);
              fmul2(t0, t1, bf_lo(h23), bf_hi(h23), c23.y, c23.w);
              ffma2(rl2, rl3, bf_lo(l23), bf_hi(l23), c23.x, c23.z, -t0, -t1);
              fmul2(t0, t1, bf_lo(l23), bf_hi(l23), c23.y, c23.w);
              ffma2(rh2, rh3, bf_lo(h23), bf_hi(h23), c23.x, c23.z, t0, t1);
              alo[x][0] = pack_bf16x2(rl0, rl1);
              alo[x][1] = pack_bf16x2(rl2, rl3);
              ahi[x][0] = pack_bf16x2(rh0, rh1);
              ahi[x][1] = pack_bf16x2(rh2, rh3);
            }
            mma_bf16_16816(sacc, alo[0][0], alo[1][0], alo[0][1], alo[1][1], qf[sl][0],
                           qf[sl][1]);
            mma_bf16_16816(sacc2, ahi[0][0], ahi[1][0], ahi[0][1], ahi[1][1], qf[NLO + sl][0],
                           qf[NLO + sl][1]);
          }
#pragma unroll
          for (int x = 0; x < 4; ++x) sacc[x] += sacc2[x];
        }
        // ---- online softmax per head (heads 2t, 2t+1; entries g, g+8)
        const float sl2 = args.scale_log2;
        const float s00 = (live_g && hv0) ? sacc[0] * sl2 : -INFINITY;
        const float s01 = (live_g && hv1) ? sacc[1] * sl2 : -INFINITY;
        const float s10 = (live_g8 && hv0) ? sacc[2] * sl2 : -INFINITY;
        const float s11 = (live_g8 && hv1) ? sacc[3] * sl2 : -INFINITY;
        float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        // lazy rescale: the running max moves only when a score exceeds it by
        // more than kLazyRescale (uniform over the lanes holding the head)
        float al0 = 1.f, al1 = 1.f;
        if (mx0 > mrun0 + kLazyRescale) {
          al0 = mrun0 == -INFINITY ? 0.f : exp2f(mrun0 - mx0);
          mrun0 = mx0;
        }
        if (mx1 > mrun1 + kLazyRescale) {
          al1 = mrun1 == -INFINITY ? 0.f : exp2f(mrun1 - mx1);
          mrun1 = mx1;
        }
        if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            acc[mt][0] *= al0;
            acc[mt][2] *= al0;
            acc[mt][1] *= al1;
            acc[mt][3] *= al1;
          }
          lrun0 *= al0;
          lrun1 *= al1;
        }
        const float p00 = s00 == -INFINITY ? 0.f : fast_exp2(s00 - mrun0);
        const float p01 = s01 == -INFINITY ? 0.f : fast_exp2(s01 - mrun1);
        const float p10 = s10 == -INFINITY ? 0.f : fast_exp2(s10 - mrun0);
        const float p11 = s11 == -INFINITY ? 0.f : fast_exp2(s11 - mrun1);
        lrun0 += p00 + p10;  // this lane's entries; summed over lanes at the end
        lrun1 += p01 + p11;
        // P^T fragments: rows of P^T(entries x heads) transposed in registers
        const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p00, p01));
        const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p10, p11));
        // ---- O^T += V^T P^T; dead entries' rows read as zero
        {
          constexpr int VW = LD / 2;  // words of a lane's dims in one V row
          uint32_t vr[4][VW];         // entries 2t, 2t+1, 2t+8, 2t+9
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const int r = e0 + 2 * tq + (x & 1) + 8 * (x >> 1);
            const bool live = r < nv;
#pragma unroll
            for (int u = 0; u < VW / 4; ++u) {
              const uint4 w = live ? *reinterpret_cast<const uint4*>(
                                         sV + staged_unit(r, (LD / 8) * gq + u, SS::PU))
                                   : make_uint4(0u, 0u, 0u, 0u);
              vr[x][4 * u] = w.x;
              vr[x][4 * u + 1] = w.y;
              vr[x][4 * u + 2] = w.z;
              vr[x][4 * u + 3] = w.w;
            }
          }
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint32_t sel = (mt & 1) ? 0x7632u : 0x5410u;
            const int wa = mt / 2, wb = (MT + mt) / 2;
            const uint32_t a0 = __byte_perm(vr[0][wa], vr[1][wa], sel);
            const uint32_t a1 = __byte_perm(vr[0][wb], vr[1][wb], sel);
            const uint32_t a2 = __byte_perm(vr[2][wa], vr[3][wa], sel);
            const uint32_t a3 = __byte_perm(vr[2][wb], vr[3][wb], sel);
            mma_bf16_16816(acc[mt], a0, a1, a2, a3, pb0, pb1);
          }
        }
        __syncwarp();  // every lane has read the stage
        if (lane == 0) mbar_arrive(&empty_bar[st]);
      }
      // this warp's state into sW[warp][head]: acc (dims), running max, sum
      // (sW overlays the ring: both warps are past their last chunk first)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        lrun0 += __shfl_xor_sync(0xffffffffu, lrun0, off);
        lrun1 += __shfl_xor_sync(0xffffffffu, lrun1, off);
      }
      consumer_sync();
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int hh = 2 * tq + x;
        if (hh < G) {
          float* ws = sW + (warp * G + hh) * (D + 2);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            ws[LD * gq + mt] = acc[mt][x];
            ws[LD * gq + MT + mt] = acc[mt][2 + x];
          }
          if (gq == 0) {
            ws[D] = x ? mrun1 : mrun0;
            ws[D + 1] = x ? lrun1 : lrun0;
          }
        }
      }
      consumer_sync();
      if (split == 1) {
        // the whole cache is this CTA's: the output is final.  Per thread 8
        // consecutive dims of one head: the warps' weights once, one 16-byte
        // store.
        for (int e8 = tid; e8 < G * D / 8; e8 += kConsumerWarps * 32) {
          const int hh = (8 * e8) / D, x0 = (8 * e8) % D;
          float M = -INFINITY;
#pragma unroll
          for (int r = 0; r < kConsumerWarps; ++r) M = fmaxf(M, sW[(r * G + hh) * (D + 2) + D]);
          float f[kConsumerWarps], den = 0.f;
#pragma unroll
          for (int r = 0; r < kConsumerWarps; ++r) {
            const float* ws = sW + (r * G + hh) * (D + 2);
            f[r] = ws[D] != -INFINITY ? exp2f(ws[D] - M) : 0.f;
            den = fmaf(f[r], ws[D + 1], den);
          }
          const float inv = 1.f / den;
          uint32_t pk[4];
#pragma unroll
          for (int j = 0; j < 8; j += 2) {
            float n0 = 0.f, n1 = 0.f;
#pragma unroll
            for (int r = 0; r < kConsumerWarps; ++r) {
              const float* ws = sW + (r * G + hh) * (D + 2) + x0 + j;
              n0 = fmaf(f[r], ws[0], n0);
              n1 = fmaf(f[r], ws[1], n1);
            }
            pk[j / 2] = pack_bf16x2(n0 * inv, n1 * inv);
          }
          if (att_ok)
            *reinterpret_cast<uint4*>(out + (((size_t)sq * args.Hq) + g * G + hh) * D + x0) =
                make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      } else {
      for (int e = tid; e < G * D; e += kConsumerWarps * 32) {
        const int hh = e / D, x = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int r = 0; r < kConsumerWarps; ++r) M = fmaxf(M, sW[(r * G + hh) * (D + 2) + D]);
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int r = 0; r < kConsumerWarps; ++r) {
          const float* ws = sW + (r * G + hh) * (D + 2);
          if (ws[D] != -INFINITY) {
            const float f = exp2f(ws[D] - M);
            num = fmaf(f, ws[x], num);
            den = fmaf(f, ws[D + 1], den);
          }
        }
        sAcc[e] = num;
        if (x == 0) {
          sM[hh] = M;
          sL[hh] = den;
        }
      }
      }
    }
    att_ok = __syncthreads_and(att_ok || warp == kConsumerWarps);
  }

  // ---- merge the cluster's partial states (each CTA a slice of the outputs),
  // then CTA 0 writes the update once every CTA has finished reading (a
  // cluster of one CTA needs no cluster barrier)
  if (split > 1) {
    cluster_arrive();
    cluster_wait();
  }
  if (attend && att_ok && split > 1) {
    const int per = (G * D + split - 1) / split;
    const int e_lo = rank * per, e_hi = min(G * D, e_lo + per);
    for (int e = e_lo + tid; e < e_hi; e += kThreads) {
      const int hh = e / D;
      float mr[kMaxSplit], ar[kMaxSplit], lr[kMaxSplit];
#pragma unroll
      for (int r = 0; r < kMaxSplit; ++r) {
        if (r < split) {
          mr[r] = dsmem_ld(dsmem_addr(sM + hh, r));
          lr[r] = dsmem_ld(dsmem_addr(sL + hh, r));
          ar[r] = dsmem_ld(dsmem_addr(sAcc + e, r));
        }
      }
      float M = -INFINITY;
#pragma unroll
      for (int r = 0; r < kMaxSplit; ++r)
        if (r < split) M = fmaxf(M, mr[r]);
      float num = 0.f, den = 0.f;
#pragma unroll
      for (int r = 0; r < kMaxSplit; ++r) {
        if (r < split && mr[r] != -INFINITY) {
          const float f = exp2f(mr[r] - M);
          num = fmaf(f, ar[r], num);
          den = fmaf(f, lr[r], den);
        }
      }
      const __nv_bfloat16 bv = __float2bfloat16_rn(num / den);
      out[(((size_t)sq * args.Hq) + g * G + hh) * D + (e % D)] =
          *reinterpret_cast<const uint16_t*>(&bv);
    }
  }
  if (rank == 0) {
    if (!ok) {
      if (tid == 0) report(status, SEP_ERR_DEVICE_BOUNDS);
    } else {
      // the update: surviving separators into the separator ring, then the
      // new token (its slot may be one a survivor was read from)
      uint16_t* kh = cp.k + head_off;
      uint16_t* vh = cp.v + head_off;
      uint8_t* sepw = cp.issep + mh * NSL;
      int32_t* posw = cp.pos + (size_t)sq * NSL;
      const int n_surv = pl.SV;
      for (int e = tid; e < n_surv * CPR; e += kThreads) {
        const int r = e / CPR, u = e % CPR;
        const int dst = a + (pl.sk0 + pl.SK + r) % s;
        const size_t so = (size_t)surv_src[r] * D + 8 * u, dso = (size_t)dst * D + 8 * u;
        const uint4 kx = *reinterpret_cast<const uint4*>(kh + so);
        const uint4 vx = *reinterpret_cast<const uint4*>(vh + so);
        *reinterpret_cast<uint4*>(kh + dso) = kx;
        *reinterpret_cast<uint4*>(vh + dso) = vx;
      }
      for (int r = tid; r < n_surv; r += kThreads) {
        const int dst = a + (pl.sk0 + pl.SK + r) % s;
        sepw[dst] = 1;
        if (g == 0) posw[dst] = surv_pos[r];
      }
      __syncthreads();
      bool new_is_sep = false;  // thread 0 (tid < CPR) holds the id
      for (int x = 0; x < args.sids.n; ++x) new_is_sep |= (new_id == args.sids.ids[x]);
      if (tid < CPR) {
        *reinterpret_cast<uint4*>(kh + (size_t)new_slot * D + 8 * tid) = nk;
        *reinterpret_cast<uint4*>(vh + (size_t)new_slot * D + 8 * tid) = nvv;
      }
      if (tid == 0) {
        sepw[new_slot] = new_is_sep ? 1 : 0;
        if (g == 0) posw[new_slot] = m.t;
        cp.meta[mh] = nm;
      }
    }
  }
  // every CTA has read the partials it needs before any shared memory goes away
  if (split > 1) {
    cluster_arrive();
    cluster_wait();
  }
}

int pick_split(int S, int Hkv, int c) {
  const int pairs = S * Hkv;
  int sp = (kTargetCtas + pairs - 1) / pairs;
  sp = sp < 1 ? 1 : (sp > kMaxSplit ? kMaxSplit : sp);
  const int by_len = c / 16 > 1 ? c / 16 : 1;  // at least ~16 entries per CTA
  return sp < by_len ? sp : by_len;
}

template <int D, int G>
cudaError_t launch_step_t(const CachePtrs& cp, StepArgs args, const void* q, const void* k_new,
                          const void* v_new, const int32_t* ids_new, void* out, int* status,
                          cudaStream_t stream) {
  const size_t smem = step_smem<D, G>(args.s, args.c).total;
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(
        cache_step_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  if (args.split == 1) {  // one CTA per (sequence, kv head): no cluster
    cache_step_kernel<D, G><<<dim3(1, args.Hkv, args.S), kThreads, smem, stream>>>(
        cp, args, static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k_new),
        static_cast<const uint16_t*>(v_new), ids_new, static_cast<uint16_t*>(out), status);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(args.split, args.Hkv, args.S);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = args.split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, cache_step_kernel<D, G>, cp, args,
                            static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k_new),
                            static_cast<const uint16_t*>(v_new), ids_new,
                            static_cast<uint16_t*>(out), status);
}

cudaError_t launch_step(const CachePtrs& cp, const StepArgs& args, int d, int G, const void* q,
                        const void* k_new, const void* v_new, const int32_t* ids_new, void* out,
                        int* status, cudaStream_t stream) {
#define SEP_CASE(DD, GG)                                                                  \
  if (d == DD && G == GG)                                                                 \
    return launch_step_t<DD, GG>(cp, args, q, k_new, v_new, ids_new, out, status, stream);
  SEP_CASE(128, 1) SEP_CASE(128, 2) SEP_CASE(128, 4) SEP_CASE(128, 8)
  SEP_CASE(64, 1) SEP_CASE(64, 2) SEP_CASE(64, 4) SEP_CASE(64, 8)
#undef SEP_CASE
  return cudaErrorNotSupported;
}

// ---------------------------------------------------------------------------
// Bulk prefill: the state T update-only steps leave in an empty cache, in
// one launch.  In text order the cache always holds the first a tokens, the
// newest <= s separators among the tokens the window has left behind
// ([a, cp) for the window start cp), and the window [max(a, cp), T).  Only
// the window start depends on the step-by-step history (it moves when the
// cache is full and the past window is compressed); each CTA replays that
// with a separator prefix count (O(1) per token), then copies its kv head's
// rows into canonical slots (ring heads at 0).  Attention reads the cache
// in logical order, so later steps see exactly what T steps would leave.
// One CTA per (kv head, sequence).
// ---------------------------------------------------------------------------
constexpr int kPrefillThreads = 256;

__global__ void __launch_bounds__(kPrefillThreads)
    cache_prefill_kernel(CachePtrs cp, StepArgs args, int D, const uint16_t* __restrict__ k_in,
                         const uint16_t* __restrict__ v_in, const int32_t* __restrict__ ids,
                         int T, int* __restrict__ sep_prefix_all, int* status) {
  const int g = blockIdx.x, sq = blockIdx.y, tid = threadIdx.x;
  const int S = args.S, Hkv = args.Hkv, a = args.a, s = args.s, w = args.w, c = args.c,
            NSL = args.NSL;
  const int ring = c - a;
  const size_t mh = (size_t)sq * Hkv + g;
  __shared__ int warp_sums[kPrefillThreads / 32];
  __shared__ int carry_sh, bad;
  __shared__ Meta fin;
  __shared__ int cp_fin;
  // separator prefix: sp[t] = #separators among tokens [0, t) (this CTA's
  // own copy in global scratch of T+1 ints per CTA)
  int* sp = sep_prefix_all + mh * (size_t)(T + 1);
  if (tid == 0) {
    const Meta m = cp.meta[mh];
    bad = (m.n_init | m.n_sep | m.n_pw | m.t) != 0;  // only an empty cache is filled
    carry_sh = 0;
  }
  __syncthreads();
  if (bad) {
    if (tid == 0) report(status, SEP_ERR_DEVICE_BOUNDS);
    return;
  }
  for (int base = 0; base < T; base += kPrefillThreads) {
    const int t = base + tid;
    bool is_s = false;
    if (t < T) {
      const int id = ids[(size_t)t * S + sq];
      for (int x = 0; x < args.sids.n; ++x) is_s |= (id == args.sids.ids[x]);
    }
    const uint32_t bal = __ballot_sync(0xffffffffu, is_s);
    const int lane = tid & 31, warp = tid >> 5;
    if (lane == 0) warp_sums[warp] = __popc(bal);
    __syncthreads();
    int before = carry_sh;
    for (int x = 0; x < warp; ++x) before += warp_sums[x];
    before += __popc(bal & ((1u << lane) - 1u));
    if (t < T) sp[t] = before;
    __syncthreads();
    if (tid == 0) {
      int tot = 0;
      for (int x = 0; x < kPrefillThreads / 32; ++x) tot += warp_sums[x];
      carry_sh += tot;
    }
    __syncthreads();
  }
  if (tid == 0) sp[T] = carry_sh;
  __syncthreads();
  // replay the counters (thread 0): the step rule with the window start cp
  if (tid == 0) {
    int n_init = 0, n_sep = 0, n_pw = 0, cpos = a;  // window = [cpos, cpos + n_pw)
    for (int t = 0; t < T; ++t) {
      if (n_init + n_sep + n_pw == c) {
        const int n_win = min(w, n_pw), n_past = n_pw - n_win;
        const int ms = sp[cpos + n_past] - sp[cpos];  // separators leaving the window
        n_sep = min(s, n_sep + ms);
        cpos += n_past;
        n_pw = n_win;
      }
      if (n_init < a) ++n_init; else ++n_pw;
    }
    Meta nm;
    memset(&nm, 0, sizeof(nm));
    nm.n_init = n_init;
    nm.n_sep = n_sep;
    nm.sep_head = 0;
    nm.n_pw = n_pw;
    nm.pw_head = 0;
    nm.t = T;
    fin = nm;
    cp_fin = cpos;
  }
  __syncthreads();
  const Meta nm = fin;
  const int cpos = cp_fin;  // window start (>= a once the initial block is full)
  const int D8 = D / 8;
  uint16_t* kh = cp.k + mh * (size_t)NSL * D;
  uint16_t* vh = cp.v + mh * (size_t)NSL * D;
  uint8_t* sepw = cp.issep + mh * NSL;
  int32_t* posw = cp.pos + (size_t)sq * NSL;
  auto copy_row = [&](int t, int slot, int u) {
    const size_t src = ((size_t)t * S + sq) * Hkv + g;
    reinterpret_cast<uint4*>(kh + (size_t)slot * D)[u] = reinterpret_cast<const uint4*>(k_in + src * D)[u];
    reinterpret_cast<uint4*>(vh + (size_t)slot * D)[u] = reinterpret_cast<const uint4*>(v_in + src * D)[u];
  };
  auto is_sep_at = [&](int t) { return sp[t + 1] != sp[t]; };
  // initial block: tokens [0, n_init) in slots [0, n_init)
  for (int e = tid; e < nm.n_init * D8; e += kPrefillThreads) copy_row(e / D8, e / D8, e % D8);
  for (int t = tid; t < nm.n_init; t += kPrefillThreads) {
    sepw[t] = is_sep_at(t) ? 1 : 0;
    if (g == 0) posw[t] = t;
  }
  // separator block: the newest n_sep separators among [a, cpos), oldest
  // first in slots a .. a + n_sep - 1
  const int first = sp[cpos] - nm.n_sep;  // separator rank of the oldest kept one
  for (int t = a + tid; t < cpos; t += kPrefillThreads) {
    if (!is_sep_at(t) || sp[t] < first) continue;
    const int slot = a + (sp[t] - first);
    for (int u = 0; u < D8; ++u) copy_row(t, slot, u);
    sepw[slot] = 1;
    if (g == 0) posw[slot] = t;
  }
  // window: tokens [cpos, T) in ring slots a + s + 0 ..
  const int w0 = nm.n_init < a ? T : cpos;  // no window until the initial block is full
  for (int e = tid; e < nm.n_pw * D8; e += kPrefillThreads) {
    const int x = e / D8;
    copy_row(w0 + x, a + s + x, e % D8);
  }
  for (int x = tid; x < nm.n_pw; x += kPrefillThreads) {
    sepw[a + s + x] = is_sep_at(w0 + x) ? 1 : 0;
    if (g == 0) posw[a + s + x] = w0 + x;
  }
  (void)ring;
  __syncthreads();
  if (tid == 0) cp.meta[mh] = nm;
}

sep_status shape_check(const sep_cache_params* p) {
  if (!params_ok(p)) return SEP_ERR_INVALID_ARG;
  if (!(p->a + p->s + p->w < p->c)) return SEP_ERR_CAPACITY;
  if (p->Hkv > kMaxHkv || (p->d != 64 && p->d != 128)) return SEP_ERR_UNSUPPORTED;
  if (p->c > kMaxC) return SEP_ERR_UNSUPPORTED;
  return SEP_OK;
}

float theta_of(const sep_cache_params* p) {
  return p->rope_theta > 0.f ? p->rope_theta : 500000.0f;
}

// RoPE table in double precision: inv_freq_i = theta^(-2i/d), entry
// [pos][i] = (cos(pos * inv_freq_i), sin(pos * inv_freq_i)), for positions
// 0 .. rope_rows-1.
std::vector<float2> rope_table(const sep_cache_params* p, int rows) {
  const int half = p->d / 2;
  std::vector<float2> t((size_t)rows * half);
  const double theta = theta_of(p);
  for (int pos = 0; pos < rows; ++pos)
    for (int i = 0; i < half; ++i) {
      const double f = pow(theta, -2.0 * i / p->d);
      t[(size_t)pos * half + i] = make_float2(static_cast<float>(cos(pos * f)),
                                              static_cast<float>(sin(pos * f)));
    }
  return t;
}

// inv_freq_i = theta^(-2i/d) as float32, the per-frequency rate the decode
// kernel turns into (cos, sin) at each entry's rank.
std::vector<float> inv_freqs(const sep_cache_params* p) {
  std::vector<float> f(p->d / 2);
  for (int i = 0; i < p->d / 2; ++i)
    f[i] = static_cast<float>(pow((double)theta_of(p), -2.0 * i / p->d));
  return f;
}


size_t export_bytes(const sep_cache_params* p) {
  return sizeof(int32_t) * 8 + (size_t)p->S * sizeof(int32_t) * 8 +
         (size_t)p->S * p->c * sizeof(int32_t) + (size_t)p->S * p->c +
         2 * (2 * (size_t)p->S * p->c * p->Hkv * p->d);
}

}  // namespace

}  // namespace sep

using namespace sep;

SEP_API size_t sep_cache_bytes(const sep_cache_params* p) {
  if (shape_check(p) != SEP_OK) return 0;
  return cache_layout(p).total;
}

SEP_API sep_status sep_cache_init(const sep_cache_params* p, void* cache_buf, size_t bytes,
                                  void* stream) {
  const sep_status st = shape_check(p);
  if (st != SEP_OK) return st;
  if (!cache_buf || reinterpret_cast<uintptr_t>(cache_buf) % 256) return SEP_ERR_INVALID_ARG;
  const CacheLayout l = cache_layout(p);
  if (bytes < l.total) return SEP_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const std::vector<float2> tab = rope_table(p, l.rope_rows);
  if (cudaMemsetAsync(cache_buf, 0, l.total, s) != cudaSuccess) return SEP_ERR_CUDA;
  const std::vector<float> invf = inv_freqs(p);
  if (cudaMemcpyAsync(static_cast<char*>(cache_buf) + l.rope, tab.data(),
                      tab.size() * sizeof(float2), cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(static_cast<char*>(cache_buf) + l.invf, invf.data(),
                      invf.size() * sizeof(float), cudaMemcpyHostToDevice, s) != cudaSuccess)
    return SEP_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SEP_ERR_CUDA;
  return SEP_OK;
}

SEP_API sep_status sep_cache_step(const sep_cache_params* p, void* cache_buf, const void* q,
                                  const void* k_new, const void* v_new, const int32_t* ids_new,
                                  const int32_t* sep_ids, int n_sep_ids, void* out, int Hq,
                                  float scale, void* stream) {
  const sep_status st = shape_check(p);
  if (st != SEP_OK) return st;
  if (!cache_buf || !k_new || !v_new || !ids_new) return SEP_ERR_INVALID_ARG;
  if ((q == nullptr) != (out == nullptr)) return SEP_ERR_INVALID_ARG;
  if (Hq < 1 || Hq % p->Hkv != 0) return SEP_ERR_INVALID_ARG;
  const int G = Hq / p->Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return SEP_ERR_UNSUPPORTED;
  auto al = [](const void* x, size_t n) { return reinterpret_cast<uintptr_t>(x) % n == 0; };
  if (!al(cache_buf, 256) || !al(k_new, 16) || !al(v_new, 16) || !al(ids_new, 4) ||
      (q && !al(q, 16)) || (out && !al(out, 16)))
    return SEP_ERR_INVALID_ARG;
  StepArgs args;
  memset(&args, 0, sizeof(args));
  if (n_sep_ids < 0 || n_sep_ids > SEP_MAX_SEP_IDS || (n_sep_ids > 0 && !sep_ids))
    return SEP_ERR_INVALID_ARG;
  args.sids.n = n_sep_ids;
  for (int i = 0; i < n_sep_ids; ++i) args.sids.ids[i] = sep_ids[i];
  args.S = p->S; args.Hkv = p->Hkv; args.Hq = Hq; args.a = p->a; args.s = p->s;
  args.w = p->w; args.c = p->c;
  const CacheLayout l = cache_layout(p);
  args.NSL = l.NSL;
  args.split = q ? pick_split(p->S, p->Hkv, p->c) : 1;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf(static_cast<float>(p->d));
  args.scale_log2 = scale * 1.4426950408889634f;
  int* status = device_status_ptr();
  if (!status) return SEP_ERR_CUDA;
  const cudaError_t e = launch_step(cache_ptrs(cache_buf, l), args, p->d, G, q, k_new, v_new,
                                    ids_new, out, status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SEP_OK : SEP_ERR_CUDA;
}

SEP_API size_t sep_cache_prefill_workspace_bytes(const sep_cache_params* p, int T) {
  if (shape_check(p) != SEP_OK || T < 1) return 0;
  return align_up(sizeof(int) * (size_t)p->S * p->Hkv * (T + 1), 256);
}

SEP_API sep_status sep_cache_prefill(const sep_cache_params* p, void* cache_buf,
                                     const void* k_prompt, const void* v_prompt,
                                     const int32_t* ids, int T, const int32_t* sep_ids,
                                     int n_sep_ids, void* ws, size_t ws_bytes, void* stream) {
  const sep_status st = shape_check(p);
  if (st != SEP_OK) return st;
  if (!cache_buf || !k_prompt || !v_prompt || !ids || !ws || T < 1) return SEP_ERR_INVALID_ARG;
  auto al = [](const void* x, size_t n) { return reinterpret_cast<uintptr_t>(x) % n == 0; };
  if (!al(cache_buf, 256) || !al(k_prompt, 16) || !al(v_prompt, 16) || !al(ids, 4) ||
      !al(ws, 256))
    return SEP_ERR_INVALID_ARG;
  if (ws_bytes < sep_cache_prefill_workspace_bytes(p, T)) return SEP_ERR_WORKSPACE;
  if (n_sep_ids < 0 || n_sep_ids > SEP_MAX_SEP_IDS || (n_sep_ids > 0 && !sep_ids))
    return SEP_ERR_INVALID_ARG;
  StepArgs args;
  memset(&args, 0, sizeof(args));
  args.sids.n = n_sep_ids;
  for (int i = 0; i < n_sep_ids; ++i) args.sids.ids[i] = sep_ids[i];
  args.S = p->S; args.Hkv = p->Hkv; args.a = p->a; args.s = p->s; args.w = p->w; args.c = p->c;
  const CacheLayout l = cache_layout(p);
  args.NSL = l.NSL;
  int* status = device_status_ptr();
  if (!status) return SEP_ERR_CUDA;
  cache_prefill_kernel<<<dim3(p->Hkv, p->S), kPrefillThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      cache_ptrs(cache_buf, l), args, p->d, static_cast<const uint16_t*>(k_prompt),
      static_cast<const uint16_t*>(v_prompt), ids, T, static_cast<int*>(ws), status);
  return cudaGetLastError() == cudaSuccess ? SEP_OK : SEP_ERR_CUDA;
}

SEP_API size_t sep_cache_export_bytes(const sep_cache_params* p) {
  if (shape_check(p) != SEP_OK) return 0;
  return export_bytes(p);
}

namespace {

// Host copy of a whole cache buffer plus typed views of its regions.
struct HostCache {
  std::vector<char> raw;
  CacheLayout l;
  Meta* meta() { return reinterpret_cast<Meta*>(raw.data() + l.meta); }
  int32_t* pos() { return reinterpret_cast<int32_t*>(raw.data() + l.pos); }
  uint8_t* issep() { return reinterpret_cast<uint8_t*>(raw.data() + l.issep); }
  uint16_t* k() { return reinterpret_cast<uint16_t*>(raw.data() + l.k); }
  uint16_t* v() { return reinterpret_cast<uint16_t*>(raw.data() + l.v); }
};

struct ImageView {
  int32_t* header;
  int32_t* counts;
  int32_t* pos;
  uint8_t* issep;
  uint16_t* k;
  uint16_t* v;
};

ImageView image_view(void* img, const sep_cache_params* p) {
  char* b = static_cast<char*>(img);
  ImageView v;
  v.header = reinterpret_cast<int32_t*>(b);
  b += sizeof(int32_t) * 8;
  v.counts = reinterpret_cast<int32_t*>(b);
  b += (size_t)p->S * sizeof(int32_t) * 8;
  v.pos = reinterpret_cast<int32_t*>(b);
  b += (size_t)p->S * p->c * sizeof(int32_t);
  v.issep = reinterpret_cast<uint8_t*>(b);
  b += (size_t)p->S * p->c;
  v.k = reinterpret_cast<uint16_t*>(b);
  b += 2 * (size_t)p->S * p->c * p->Hkv * p->d;
  v.v = reinterpret_cast<uint16_t*>(b);
  return v;
}

int host_slot(int k, const Meta& m, int a, int s, int ring) {
  if (k < m.n_init) return k;
  k -= m.n_init;
  if (k < m.n_sep) return a + (m.sep_head + k) % s;
  k -= m.n_sep;
  return a + s + (m.pw_head + k) % ring;
}

}  // namespace

SEP_API sep_status sep_cache_export(const sep_cache_params* p, const void* cache_buf,
                                    void* host_dst, size_t bytes, void* stream) {
  const sep_status st = shape_check(p);
  if (st != SEP_OK) return st;
  if (!cache_buf || !host_dst) return SEP_ERR_INVALID_ARG;
  if (bytes < export_bytes(p)) return SEP_ERR_WORKSPACE;
  HostCache hc;
  hc.l = cache_layout(p);
  hc.raw.resize(hc.l.total);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(hc.raw.data(), cache_buf, hc.l.total, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return SEP_ERR_CUDA;
  memset(host_dst, 0, export_bytes(p));
  ImageView im = image_view(host_dst, p);
  const int hdr[8] = {kCacheMagic, p->S, p->Hkv, p->d, p->a, p->s, p->w, p->c};
  memcpy(im.header, hdr, sizeof(hdr));
  const int ring = p->c - p->a, NSL = hc.l.NSL, HD = p->Hkv * p->d;
  for (int sq = 0; sq < p->S; ++sq) {
    const Meta m = hc.meta()[(size_t)sq * p->Hkv];
    // every kv head keeps its own copy of the counters; they must agree
    for (int g = 1; g < p->Hkv; ++g)
      if (memcmp(&hc.meta()[(size_t)sq * p->Hkv + g], &m, sizeof(Meta)) != 0)
        return SEP_ERR_DEVICE_BOUNDS;
    const int n_win = m.n_pw < p->w ? m.n_pw : p->w;
    const int total = m.n_init + m.n_sep + m.n_pw;
    if (total > p->c || m.n_init > p->a || m.n_sep > p->s || m.n_pw > ring)
      return SEP_ERR_DEVICE_BOUNDS;
    int32_t* cnt = im.counts + 8 * sq;
    cnt[0] = m.n_init; cnt[1] = m.n_sep; cnt[2] = m.n_pw - n_win; cnt[3] = n_win;
    cnt[4] = total; cnt[5] = m.t;
    for (int k = 0; k < p->c; ++k) im.pos[(size_t)sq * p->c + k] = -1;
    for (int k = 0; k < total; ++k) {
      const int slot = host_slot(k, m, p->a, p->s, ring);
      im.pos[(size_t)sq * p->c + k] = hc.pos()[(size_t)sq * NSL + slot];
      im.issep[(size_t)sq * p->c + k] = hc.issep()[(size_t)sq * p->Hkv * NSL + slot];
      for (int g = 0; g < p->Hkv; ++g) {
        const size_t src = (((size_t)sq * p->Hkv + g) * NSL + slot) * p->d;
        const size_t dst = ((size_t)sq * p->c + k) * HD + (size_t)g * p->d;
        memcpy(im.k + dst, hc.k() + src, 2 * p->d);
        memcpy(im.v + dst, hc.v() + src, 2 * p->d);
      }
    }
  }
  return SEP_OK;
}

SEP_API sep_status sep_cache_import(const sep_cache_params* p, void* cache_buf,
                                    const void* host_src, size_t bytes, void* stream) {
  const sep_status st = shape_check(p);
  if (st != SEP_OK) return st;
  if (!cache_buf || !host_src) return SEP_ERR_INVALID_ARG;
  if (bytes < export_bytes(p)) return SEP_ERR_WORKSPACE;
  ImageView im = image_view(const_cast<void*>(host_src), p);
  const int hdr[8] = {kCacheMagic, p->S, p->Hkv, p->d, p->a, p->s, p->w, p->c};
  if (memcmp(im.header, hdr, sizeof(hdr)) != 0) return SEP_ERR_INVALID_ARG;
  HostCache hc;
  hc.l = cache_layout(p);
  hc.raw.assign(hc.l.total, 0);
  const std::vector<float2> tab = rope_table(p, hc.l.rope_rows);
  memcpy(hc.raw.data() + hc.l.rope, tab.data(), tab.size() * sizeof(float2));
  const std::vector<float> invf = inv_freqs(p);
  memcpy(hc.raw.data() + hc.l.invf, invf.data(), invf.size() * sizeof(float));
  const int ring = p->c - p->a, NSL = hc.l.NSL, HD = p->Hkv * p->d;
  for (int sq = 0; sq < p->S; ++sq) {
    const int32_t* cnt = im.counts + 8 * sq;
    Meta m;
    memset(&m, 0, sizeof(m));
    m.n_init = cnt[0];
    m.n_sep = cnt[1];
    m.n_pw = cnt[2] + cnt[3];
    m.t = cnt[5];
    const int total = m.n_init + m.n_sep + m.n_pw;
    if (cnt[0] < 0 || cnt[0] > p->a || cnt[1] < 0 || cnt[1] > p->s || cnt[2] < 0 ||
        cnt[3] < 0 || cnt[3] > p->w || m.n_pw > ring || total != cnt[4] || total > p->c ||
        (cnt[2] > 0 && cnt[3] != p->w) || (m.n_init < p->a && (m.n_sep | m.n_pw) != 0))
      return SEP_ERR_INVALID_ARG;
    for (int g = 0; g < p->Hkv; ++g) hc.meta()[(size_t)sq * p->Hkv + g] = m;
    for (int k = 0; k < total; ++k) {
      const int slot = host_slot(k, m, p->a, p->s, ring);
      hc.pos()[(size_t)sq * NSL + slot] = im.pos[(size_t)sq * p->c + k];
      for (int g = 0; g < p->Hkv; ++g) {
        hc.issep()[((size_t)sq * p->Hkv + g) * NSL + slot] = im.issep[(size_t)sq * p->c + k];
        const size_t dst = (((size_t)sq * p->Hkv + g) * NSL + slot) * p->d;
        const size_t src = ((size_t)sq * p->c + k) * HD + (size_t)g * p->d;
        memcpy(hc.k() + dst, im.k + src, 2 * p->d);
        memcpy(hc.v() + dst, im.v + src, 2 * p->d);
      }
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(cache_buf, hc.raw.data(), hc.l.total, cudaMemcpyHostToDevice, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return SEP_ERR_CUDA;
  return SEP_OK;
}
