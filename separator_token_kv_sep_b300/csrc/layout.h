// Internal layouts shared by the host API and the kernels: the index buffer,
// the streaming-cache buffer, and the host launchers of each kernel file.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "../../include/sepattn.h"

namespace sep {

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Separator ids travel by value in the kernel parameters.
struct SepIdList {
  int n;
  int ids[SEP_MAX_SEP_IDS];
};

// ---------------------------------------------------------------------------
// Index buffer: header, keep_prefix [B][L+1], keep_pos [B][L], keep_count [B],
// blocks [B][T][4], keep_bits [B][ceil(L/32)]; every field 256-byte aligned.
// ---------------------------------------------------------------------------
constexpr int kIndexMagic = 0x49504553;  // 'SEPI'

struct IndexHeader {  // first 256 bytes of the buffer
  int magic, B, L, a, n, block_m, T, nwords;
};

struct IndexLayout {
  size_t header, keep_prefix, keep_pos, keep_count, blocks, keep_bits, total;
  int T, nwords;
};

inline IndexLayout index_layout(int B, int L, int block_m) {
  IndexLayout l;
  l.T = (L + block_m - 1) / block_m;
  l.nwords = (L + 31) / 32;
  size_t off = 0;
  l.header = off;
  off += 256;
  l.keep_prefix = off;
  off = align_up(off + sizeof(int32_t) * (size_t)B * (L + 1), 256);
  l.keep_pos = off;
  off = align_up(off + sizeof(int32_t) * (size_t)B * L, 256);
  l.keep_count = off;
  off = align_up(off + sizeof(int32_t) * (size_t)B, 256);
  l.blocks = off;
  off = align_up(off + sizeof(int32_t) * (size_t)B * l.T * 4, 256);
  l.keep_bits = off;
  off = align_up(off + sizeof(uint32_t) * (size_t)B * l.nwords, 256);
  l.total = off;
  return l;
}

struct IndexPtrs {
  IndexHeader* header;
  int32_t* keep_prefix;
  int32_t* keep_pos;
  int32_t* keep_count;
  int32_t* blocks;
  uint32_t* keep_bits;
};

inline IndexPtrs index_ptrs(void* buf, const IndexLayout& l) {
  char* p = static_cast<char*>(buf);
  IndexPtrs r;
  r.header = reinterpret_cast<IndexHeader*>(p + l.header);
  r.keep_prefix = reinterpret_cast<int32_t*>(p + l.keep_prefix);
  r.keep_pos = reinterpret_cast<int32_t*>(p + l.keep_pos);
  r.keep_count = reinterpret_cast<int32_t*>(p + l.keep_count);
  r.blocks = reinterpret_cast<int32_t*>(p + l.blocks);
  r.keep_bits = reinterpret_cast<uint32_t*>(p + l.keep_bits);
  return r;
}

// Records the calling thread's registered profiling event `i` on `stream`
// (no-op when none is registered at that index).  Defined in api.cu.
void profile_mark(int i, void* stream);

// Device address of the library's status word on the current device (null if
// the CUDA runtime is unavailable).  Defined in api.cu.
int* device_status_ptr();

// ---------------------------------------------------------------------------
// Host launchers (each defined in the kernel file named beside it).
// Every launcher enqueues on `stream` and returns the launch's cudaError_t.
// ---------------------------------------------------------------------------
// index.cu
int launch_build_index(const int32_t* ids, int B, int L, const SepIdList& sids, int a, int n,
                       int block_m, int fix_delta, IndexPtrs ptrs, int* status, void* stream);

// attn_simt.cu -- fp32 CUDA-core forward
int launch_attn_fwd_simt(IndexPtrs idx, const float* q, const float* k, const float* v, float* o,
                         float* lse, int B, int Hq, int Hkv, int L, int d, float scale,
                         int* status, void* stream);

}  // namespace sep
