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
// Index buffer: header, seq [B] (int4), keep_prefix [B][L+1], keep_pos [B][L],
// keep_count [B], blocks [B][T][4], keep_bits [B][ceil(L/32)]; every field
// 256-byte aligned.  For a pack of variable-length sequences L is the
// longest length and every per-sequence field is padded to it.
// ---------------------------------------------------------------------------
constexpr int kIndexMagic = 0x49504553;  // 'SEPI'

struct IndexHeader {  // first 256 bytes of the buffer
  int magic, B, L, a, n, block_m, T, nwords;
  int packed;  // 0: B rows of length L; 1: a pack of B sequences (L = longest)
  int total;   // rows of one head plane of q / k / v (B * L or the packed total)
};

// Per-sequence record {len, row0, tile0, 0}: the sequence's length, its first
// row in a head plane of q / k / v (0 in an equal-length batch, where each
// sequence has planes of its own), and its first 128-row tile in the
// workspaces' tile space (the tiles of sequences before it).
struct SeqRec {
  int len, row0, tile0, pad;
};

// Tokens of one scan tile of the index kernel (one CTA per tile).
constexpr int kScanTile = 8192;

struct IndexLayout {
  size_t header, seq, keep_prefix, keep_pos, keep_count, blocks, keep_bits, scan, total;
  int T, nwords, ntiles;
};

inline IndexLayout index_layout(int B, int L, int block_m) {
  IndexLayout l;
  l.T = (L + block_m - 1) / block_m;
  l.nwords = (L + 31) / 32;
  size_t off = 0;
  l.header = off;
  off += 256;
  l.seq = off;
  off = align_up(off + sizeof(SeqRec) * (size_t)B, 256);
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
  // scratch of the index kernel's scan: a tile ticket (first 256 bytes),
  // then one status word per (sequence, scan tile); zeroed before each build
  l.ntiles = (L + kScanTile - 1) / kScanTile;
  l.scan = off;
  off = align_up(off + 256 + sizeof(unsigned long long) * (size_t)B * l.ntiles, 256);
  l.total = off;
  return l;
}

struct IndexPtrs {
  IndexHeader* header;
  SeqRec* seq;
  int32_t* keep_prefix;
  int32_t* keep_pos;
  int32_t* keep_count;
  int32_t* blocks;
  uint32_t* keep_bits;
  unsigned int* scan_ticket;
  unsigned long long* scan_state;
};

inline IndexPtrs index_ptrs(void* buf, const IndexLayout& l) {
  char* p = static_cast<char*>(buf);
  IndexPtrs r;
  r.header = reinterpret_cast<IndexHeader*>(p + l.header);
  r.seq = reinterpret_cast<SeqRec*>(p + l.seq);
  r.keep_prefix = reinterpret_cast<int32_t*>(p + l.keep_prefix);
  r.keep_pos = reinterpret_cast<int32_t*>(p + l.keep_pos);
  r.keep_count = reinterpret_cast<int32_t*>(p + l.keep_count);
  r.blocks = reinterpret_cast<int32_t*>(p + l.blocks);
  r.keep_bits = reinterpret_cast<uint32_t*>(p + l.keep_bits);
  r.scan_ticket = reinterpret_cast<unsigned int*>(p + l.scan);
  r.scan_state = reinterpret_cast<unsigned long long*>(p + l.scan + 256);
  return r;
}

// ---------------------------------------------------------------------------
// Geometry of a batch as the attention kernels see it.  Head planes of q, k,
// v, o and the gradients are [planes][R][d]: an equal-length batch has
// planes (b, h) of R = L rows; a pack has one plane per head holding every
// sequence, R = total rows, sequence b at rows [row0, row0 + len).  The
// workspaces (gathered keep rows, row statistics, keep-row gradients) are
// laid out per head over a tile space of TT tiles of 128 rows, sequence b
// owning tiles [tile0, tile0 + ceil(len / 128)).
// ---------------------------------------------------------------------------
struct Geom {
  int B, Hq, Hkv;
  int L;   // longest sequence (the index's L)
  int T;   // ceil(L / 128)
  int R;   // rows of one head plane of q / k / v / o
  int TT;  // tiles of one head plane of the workspaces
  int packed;
#ifdef __CUDACC__
  __host__ __device__
#endif
  int qplane(int b, int h) const { return packed ? h : b * Hq + h; }
#ifdef __CUDACC__
  __host__ __device__
#endif
  int kvplane(int b, int g) const { return packed ? g : b * Hkv + g; }
};

// A sequence record is usable when the sequence lies inside the head planes
// and its tiles inside the workspaces' tile space (kernels skip, and report,
// any other).
#ifdef __CUDACC__
__host__ __device__
#endif
inline bool seq_ok(const SeqRec& s, const Geom& g) {
  return s.len >= 0 && s.len <= g.L && s.row0 >= 0 && s.row0 <= g.R - s.len && s.tile0 >= 0 &&
         s.tile0 <= g.TT - (s.len + 127) / 128;
}

// Workspace tile space: B * T tiles for an equal-length batch; for a pack of
// `total` rows in B sequences, sum_b ceil(len_b / 128) <= ceil(total / 128) + B.
inline int geom_tiles(int B, int L, int total, int packed) {
  return packed ? (total + 127) / 128 + B : B * ((L + 127) / 128);
}

inline Geom make_geom(int B, int Hq, int Hkv, int L, int total, int packed) {
  Geom g;
  g.B = B; g.Hq = Hq; g.Hkv = Hkv; g.L = L; g.T = (L + 127) / 128;
  g.R = packed ? total : L;
  g.TT = geom_tiles(B, L, total, packed);
  g.packed = packed;
  return g;
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
// cu: device int32 [B + 1] sequence starts of a pack (null: B rows of L ids).
int launch_build_index(const int32_t* ids, const int32_t* cu, int total, int B, int L,
                       const SepIdList& sids, int a, int n, int block_m, int fix_delta,
                       IndexPtrs ptrs, int* status, void* stream);

// attn_simt.cu -- fp32 CUDA-core forward
int launch_attn_fwd_simt(IndexPtrs idx, const float* q, const float* k, const float* v, float* o,
                         float* lse, int B, int Hq, int Hkv, int L, int d, float scale,
                         int* status, void* stream);

}  // namespace sep
