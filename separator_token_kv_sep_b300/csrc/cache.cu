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
// load from a cos/sin table of positions 0..c-1.  Each sequence owns
// a + s + (c - a) slots: the initial block, a ring of s separator slots and a
// ring of c - a slots holding the past and local windows (which are one
// contiguous stretch of text).  Logical entry k maps to its slot through the
// ring heads, and attention always reduces in logical order, so the outputs
// do not depend on where the rings happen to start.
//
// One thread-block cluster per sequence, one CTA per kv head: every CTA reads
// the shared counters and separator flags, arrives on the cluster barrier,
// moves and appends its own head's K/V rows, attends for the q heads of its
// group, and CTA 0 alone writes the shared counters and flags after the
// barrier, so no CTA can see half-updated metadata.
#include <math.h>
#include <string.h>

#include <vector>

#include "common.cuh"
#include "layout.h"

#define SEP_API extern "C" __attribute__((visibility("default")))

namespace sep {

namespace {

constexpr int kCacheMagic = 0x43504553;  // 'SEPC'
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxPast = 1024;  // c - a slots of the window ring are scanned in smem

struct CacheLayout {
  int S, Hkv, d, a, s, w, c, NSL;
  size_t meta, rope, pos, issep, k, v, total;
};

// Counters of one sequence (int32 x 8 in device memory).
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
  size_t off = 0;
  l.meta = off;
  off = align_up(off + sizeof(Meta) * (size_t)l.S, 256);
  l.rope = off;
  off = align_up(off + sizeof(float2) * (size_t)l.c * (l.d / 2), 256);
  l.pos = off;
  off = align_up(off + sizeof(int32_t) * (size_t)l.S * l.NSL, 256);
  l.issep = off;
  off = align_up(off + (size_t)l.S * l.NSL, 256);
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
  p.pos = reinterpret_cast<int32_t*>(b + l.pos);
  p.issep = reinterpret_cast<uint8_t*>(b + l.issep);
  p.k = reinterpret_cast<uint16_t*>(b + l.k);
  p.v = reinterpret_cast<uint16_t*>(b + l.v);
  return p;
}

struct StepArgs {
  int S, Hkv, Hq, a, s, w, c, NSL;
  float scale_log2;
  SepIdList sids;
};

__device__ __forceinline__ int slot_of(int k, const Meta& m, int a, int s, int ring) {
  if (k < m.n_init) return k;
  k -= m.n_init;
  if (k < m.n_sep) return a + (m.sep_head + k) % s;
  k -= m.n_sep;
  return a + s + (m.pw_head + k) % ring;
}

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Dynamic shared memory of the step kernel.
template <int D, int G>
struct StepSmem {
  static size_t bytes(int c) {
    return sizeof(float) * ((size_t)G * D + (size_t)G * (c + 32) + (size_t)kWarps * G * D);
  }
};

template <int D, int G>
__global__ void __launch_bounds__(kThreads)
    cache_step_kernel(CachePtrs cp, StepArgs args, const uint16_t* __restrict__ q,
                      const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
                      const int32_t* __restrict__ ids_new, uint16_t* __restrict__ out,
                      int* status) {
  constexpr int LPE = D / 8;     // lanes per cache entry (16 bytes each)
  constexpr int EPW = 32 / LPE;  // entries per warp pass
  constexpr int HALF = D / 2;
  extern __shared__ float dsm[];
  __shared__ int sep_src[kMaxPast];  // window-ring slots of surviving separators
  __shared__ int sep_dst[kMaxPast];  // their separator-ring slots
  __shared__ int src_pos[kMaxPast];
  __shared__ int warp_cnt[kWarps];
  __shared__ int bad;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.x, sq = blockIdx.y;
  const int a = args.a, s = args.s, w = args.w, c = args.c, NSL = args.NSL;
  const int ring = c - a;
  const bool rank0 = cluster_rank() == 0;
  float* qs = dsm;                        // [G][D]
  float* scores = qs + G * D;             // [G][c + 32]
  float* partial = scores + G * (c + 32); // [kWarps][G][D]
  const int SP = c + 32;

  const Meta m = cp.meta[sq];
  const int32_t* posr = cp.pos + (size_t)sq * NSL;
  const uint8_t* sepr = cp.issep + (size_t)sq * NSL;
  if (tid == 0)
    bad = (m.n_init < 0 || m.n_init > a || m.n_sep < 0 || m.n_sep > s || m.n_pw < 0 ||
           m.n_pw > ring || m.sep_head < 0 || (s > 0 && m.sep_head >= s) || m.pw_head < 0 ||
           m.pw_head >= ring || m.n_init + m.n_sep + m.n_pw > c ||
           (m.n_init < a && (m.n_sep | m.n_pw) != 0));
  __syncthreads();
  const bool ok = !bad;

  // ---- new counters (identical in every CTA of the cluster)
  Meta nm = m;
  const bool compress = ok && (m.n_init + m.n_sep + m.n_pw == c);
  int n_surv = 0;
  if (compress) {
    const int n_win = min(w, m.n_pw);
    const int n_past = m.n_pw - n_win;
    // pass 1: number of separators in the past window
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
        sep_src[r - first] = slot;
        sep_dst[r - first] = a + (m.sep_head + m.n_sep + r) % s;
        src_pos[r - first] = posr[slot];
      }
      base += tot;
      __syncthreads();
    }
    n_surv = ms - first;
    const int drop = max(0, m.n_sep + ms - s);
    nm.sep_head = s > 0 ? (m.sep_head + drop) % s : 0;
    nm.n_sep = m.n_sep + ms - drop;
    nm.pw_head = (m.pw_head + n_past) % ring;
    nm.n_pw = n_win;
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
  const int32_t new_id = ids_new[sq];
  bool new_is_sep = false;
  for (int x = 0; x < args.sids.n; ++x) new_is_sep |= (new_id == args.sids.ids[x]);

  cluster_arrive();  // every CTA has read the shared counters and flags

  // ---- move this head's surviving separator rows, then append the new token
  const size_t head_off = ((size_t)sq * args.Hkv + g) * (size_t)NSL * D;
  uint16_t* kh = cp.k + head_off;
  uint16_t* vh = cp.v + head_off;
  for (int e = tid; e < n_surv * (D / 8); e += kThreads) {
    const int r = e / (D / 8), u = e % (D / 8);
    const size_t so = (size_t)sep_src[r] * D + 8 * u, dst = (size_t)sep_dst[r] * D + 8 * u;
    *reinterpret_cast<uint4*>(kh + dst) = *reinterpret_cast<const uint4*>(kh + so);
    *reinterpret_cast<uint4*>(vh + dst) = *reinterpret_cast<const uint4*>(vh + so);
  }
  __syncthreads();  // the new token may land on a slot a survivor was copied from
  if (ok) {
    const size_t src = ((size_t)sq * args.Hkv + g) * D;
    for (int u = tid; u < D / 8; u += kThreads) {
      *reinterpret_cast<uint4*>(kh + (size_t)new_slot * D + 8 * u) =
          *reinterpret_cast<const uint4*>(k_new + src + 8 * u);
      *reinterpret_cast<uint4*>(vh + (size_t)new_slot * D + 8 * u) =
          *reinterpret_cast<const uint4*>(v_new + src + 8 * u);
    }
  }
  __syncthreads();

  // ---- decode attention for the G q heads of kv head g
  if (ok && q != nullptr && out != nullptr) {
    const int N = nm.n_init + nm.n_sep + nm.n_pw;
    const int qpos = N - 1;
    for (int e = tid; e < G * D; e += kThreads) {
      const int hh = e / D, x = e % D;
      const uint16_t* qr = q + (((size_t)sq * args.Hq) + g * G + hh) * D;
      const int i = x % HALF;
      const float2 cs = cp.rope[(size_t)qpos * HALF + i];
      const float x1 = __uint_as_float((uint32_t)qr[i] << 16);
      const float x2 = __uint_as_float((uint32_t)qr[i + HALF] << 16);
      qs[hh * D + x] = x < HALF ? (x1 * cs.x - x2 * cs.y) : (x2 * cs.x + x1 * cs.y);
    }
    __syncthreads();
    const int sub = lane / LPE, l8 = lane % LPE;  // entry within the pass, lane within entry
    const int e0 = 8 * l8;                        // first of this lane's 8 columns
    const bool lo_half = e0 < HALF;
    // scores, rotating each key by its rank in the cache
    for (int k0 = warp * EPW; k0 < N; k0 += kWarps * EPW) {
      const int k = k0 + sub;
      const bool valid = k < N;
      const int slot = valid ? slot_of(k, nm, a, s, ring) : 0;
      float x[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(kh + (size_t)slot * D + e0), x);
      float y[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) y[j] = __shfl_xor_sync(0xffffffffu, x[j], LPE / 2);
      const float4* cs4 =
          reinterpret_cast<const float4*>(cp.rope + (size_t)(valid ? k : 0) * HALF + (e0 % HALF));
      float rk[8];
#pragma unroll
      for (int j2 = 0; j2 < 4; ++j2) {
        const float4 t = cs4[j2];  // (cos, sin) of columns 2*j2 and 2*j2+1
        const int j = 2 * j2;
        rk[j] = lo_half ? (x[j] * t.x - y[j] * t.y) : (x[j] * t.x + y[j] * t.y);
        rk[j + 1] = lo_half ? (x[j + 1] * t.z - y[j + 1] * t.w) : (x[j + 1] * t.z + y[j + 1] * t.w);
      }
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) acc = fmaf(rk[j], qs[hh * D + e0 + j], acc);
#pragma unroll
        for (int off = LPE / 2; off > 0; off >>= 1)
          acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (valid && l8 == 0) scores[hh * SP + k] = acc * args.scale_log2;
      }
    }
    __syncthreads();
    // softmax, one warp per head
    for (int hh = warp; hh < G; hh += kWarps) {
      float* sc = scores + hh * SP;
      float mx = -INFINITY;
      for (int k = lane; k < N; k += 32) mx = fmaxf(mx, sc[k]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      float sum = 0.f;
      for (int k = lane; k < N; k += 32) {
        const float p = exp2f(sc[k] - mx);
        sc[k] = p;
        sum += p;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      const float inv = 1.f / sum;
      for (int k = lane; k < N; k += 32) sc[k] *= inv;
    }
    __syncthreads();
    // P V
    float acc[G][8];
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[hh][j] = 0.f;
    for (int k0 = warp * EPW; k0 < N; k0 += kWarps * EPW) {
      const int k = k0 + sub;
      if (k < N) {
        const int slot = slot_of(k, nm, a, s, ring);
        float x[8];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(vh + (size_t)slot * D + e0), x);
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const float p = scores[hh * SP + k];
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[hh][j] = fmaf(p, x[j], acc[hh][j]);
        }
      }
    }
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int off = LPE; off < 32; off <<= 1)
          acc[hh][j] += __shfl_xor_sync(0xffffffffu, acc[hh][j], off);
      }
    if (sub == 0) {
#pragma unroll
      for (int hh = 0; hh < G; ++hh)
#pragma unroll
        for (int j = 0; j < 8; ++j) partial[(warp * G + hh) * D + e0 + j] = acc[hh][j];
    }
    __syncthreads();
    for (int e = tid; e < G * D; e += kThreads) {
      const int hh = e / D, x = e % D;
      float sacc = 0.f;
#pragma unroll
      for (int r = 0; r < kWarps; ++r) sacc += partial[(r * G + hh) * D + x];
      const __nv_bfloat16 b = __float2bfloat16_rn(sacc);
      out[(((size_t)sq * args.Hq) + g * G + hh) * D + x] = *reinterpret_cast<const uint16_t*>(&b);
    }
  }

  cluster_wait();  // every CTA of the sequence has read the old metadata
  if (rank0) {
    if (!ok) {
      if (tid == 0) report(status, SEP_ERR_DEVICE_BOUNDS);
    } else {
      int32_t* posw = cp.pos + (size_t)sq * NSL;
      uint8_t* sepw = cp.issep + (size_t)sq * NSL;
      for (int r = tid; r < n_surv; r += kThreads) {
        posw[sep_dst[r]] = src_pos[r];
        sepw[sep_dst[r]] = 1;
      }
      __syncthreads();
      if (tid == 0) {
        posw[new_slot] = m.t;
        sepw[new_slot] = new_is_sep ? 1 : 0;
        cp.meta[sq] = nm;
      }
    }
  }
}

template <int D, int G>
cudaError_t launch_step_t(const CachePtrs& cp, const StepArgs& args, const void* q,
                          const void* k_new, const void* v_new, const int32_t* ids_new,
                          void* out, int* status, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(args.Hkv, args.S, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  const size_t smem = StepSmem<D, G>::bytes(args.c);
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(
        cache_step_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = args.Hkv;
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

sep_status shape_check(const sep_cache_params* p) {
  if (!params_ok(p)) return SEP_ERR_INVALID_ARG;
  if (!(p->a + p->s + p->w < p->c)) return SEP_ERR_CAPACITY;
  if (p->Hkv > 8 || (p->d != 64 && p->d != 128)) return SEP_ERR_UNSUPPORTED;
  if (p->c > kMaxPast) return SEP_ERR_UNSUPPORTED;
  return SEP_OK;
}

float theta_of(const sep_cache_params* p) {
  return p->rope_theta > 0.f ? p->rope_theta : 500000.0f;
}

// RoPE table in double precision: inv_freq_i = theta^(-2i/d), entry
// [pos][i] = (cos(pos * inv_freq_i), sin(pos * inv_freq_i)).
std::vector<float2> rope_table(const sep_cache_params* p) {
  const int half = p->d / 2;
  std::vector<float2> t((size_t)p->c * half);
  const double theta = theta_of(p);
  for (int pos = 0; pos < p->c; ++pos)
    for (int i = 0; i < half; ++i) {
      const double f = pow(theta, -2.0 * i / p->d);
      t[(size_t)pos * half + i] = make_float2(static_cast<float>(cos(pos * f)),
                                              static_cast<float>(sin(pos * f)));
    }
  return t;
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
  const std::vector<float2> tab = rope_table(p);
  if (cudaMemsetAsync(cache_buf, 0, l.total, s) != cudaSuccess) return SEP_ERR_CUDA;
  if (cudaMemcpyAsync(static_cast<char*>(cache_buf) + l.rope, tab.data(),
                      tab.size() * sizeof(float2), cudaMemcpyHostToDevice, s) != cudaSuccess)
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
  if (!(scale > 0.f)) scale = 1.0f / sqrtf(static_cast<float>(p->d));
  args.scale_log2 = scale * 1.4426950408889634f;
  int* status = device_status_ptr();
  if (!status) return SEP_ERR_CUDA;
  const cudaError_t e = launch_step(cache_ptrs(cache_buf, l), args, p->d, G, q, k_new, v_new,
                                    ids_new, out, status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SEP_OK : SEP_ERR_CUDA;
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
    const Meta m = hc.meta()[sq];
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
      im.issep[(size_t)sq * p->c + k] = hc.issep()[(size_t)sq * NSL + slot];
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
  const std::vector<float2> tab = rope_table(p);
  memcpy(hc.raw.data() + hc.l.rope, tab.data(), tab.size() * sizeof(float2));
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
    hc.meta()[sq] = m;
    for (int k = 0; k < total; ++k) {
      const int slot = host_slot(k, m, p->a, p->s, ring);
      hc.pos()[(size_t)sq * NSL + slot] = im.pos[(size_t)sq * p->c + k];
      hc.issep()[(size_t)sq * NSL + slot] = im.issep[(size_t)sq * p->c + k];
      for (int g = 0; g < p->Hkv; ++g) {
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
