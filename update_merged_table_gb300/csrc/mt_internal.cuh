// Internal declarations of the CUDA path of the merged dynamic embedding table.
//
// A table is a key store and one or more row segments, each in caller-owned
// device memory:
//   key store:    [Header 1 KiB][slots: M x Slot (16 B)][free stack: R x int32]
//   row segment:  [records of rows first .. first + count - 1]
// A row record is [emb: d x row dtype][m: d x fp32][v: d x fp32], each part a
// multiple of 16 bytes, so every part of a row is reached with 16-byte vector
// accesses.  A slot {key, row, meta} maps a merged key to its row and keeps
// the table step at which it was inserted (MTGR section 5, Embedding
// Management: each key leads to its embedding and to bookkeeping data).  The
// key store is separate from the rows, so capacity expansion and compaction
// rebuild it without moving any embedding; new rows arrive as a new segment.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mt.h"

namespace mt {

constexpr unsigned long long kEmpty = MT_KEY_EMPTY;
constexpr unsigned long long kTomb = MT_KEY_TOMBSTONE;
constexpr unsigned long long kIdLimit = 1ull << 56;
constexpr unsigned kFull = 0xFFFFFFFFu;

struct __align__(16) Slot {
  unsigned long long key;
  int32_t row;
  uint32_t meta;  // table step at insertion
};
static_assert(sizeof(Slot) == 16, "slot is 16 bytes");

// Device header at the start of the arena.
struct __align__(256) Header {
  int32_t error;           // first latched device error (0 = none)
  int32_t pad0;
  long long free_top;      // rows on the free stack
  long long step;          // Adam steps taken
  long long export_count;  // scratch for mt_export
  double b1pow, b2pow;     // Adam's beta-power accumulators: b1^t and b2^t, one multiply per step
  long long pad1[2];
  // mt_stats accumulators
  unsigned long long live, tombs, disp;
  unsigned long long hist[MT_HIST_BINS];
};
constexpr size_t kHeaderBytes = 1024;
static_assert(sizeof(Header) <= kHeaderBytes, "header fits");

constexpr int kMaxRowSegments = MT_MAX_ROW_SEGMENTS;

// Everything a kernel needs to reach the table (passed by value).
struct TableDev {
  Header* hdr;
  Slot* slots;
  int32_t* free_stack;
  char* seg_base[kMaxRowSegments];       // row segment s holds rows seg_first[s] .. seg_first[s+1] - 1
  long long seg_first[kMaxRowSegments];  // seg_first[0] = 0
  int nseg;
  unsigned long long mask;       // M - 1
  unsigned long long S;          // odd probe step, reduced mod M
  unsigned long long hash_seed;
  unsigned long long init_seed;
  unsigned long long Sinv;       // S^-1 mod M
  uint32_t log2_slots;
  uint32_t max_probes;
  uint32_t dim;
  uint32_t rec_bytes;            // bytes per row record
  uint32_t emb_bytes;            // d x row element bytes
  uint32_t mv_bytes;             // d x 4
  uint32_t flags;                // mt_config flags (reserved, 0)
  int row_dtype;
  float init_scale;
  long long num_rows;
};

// ---- small device helpers -------------------------------------------------

// splitmix64 output mixer (Steele, Lea, Flood, OOPSLA 2014).
__device__ __forceinline__ unsigned long long mix64(unsigned long long z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Home slot h0 of a key in the table: the top n bits of the mixed key.
__device__ __forceinline__ unsigned long long home_slot(const TableDev& T, unsigned long long key) {
  return mix64(key ^ T.hash_seed) >> (64 - T.log2_slots);
}

__device__ __forceinline__ void latch_error(Header* h, int code) {
  if (atomicCAS(&h->error, 0, code) == 0) { /* first error wins */ }
}

__device__ __forceinline__ unsigned long long load_key_relaxed(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// The record of a row: its segment is found with constant indices only (the
// table view lives in kernel parameter space, which dynamic indexing would
// copy to local memory).
__device__ __forceinline__ char* row_ptr(const TableDev& T, int32_t row) {
  if (T.nseg == 1) return T.seg_base[0] + (size_t)row * T.rec_bytes;  // a table that never grew its rows
  char* base = T.seg_base[0];
  long long first = 0;
#pragma unroll
  for (int s = 1; s < kMaxRowSegments; ++s) {
    if (s < T.nseg && row >= T.seg_first[s]) {
      base = T.seg_base[s];
      first = T.seg_first[s];
    }
  }
  return base + (size_t)(row - first) * T.rec_bytes;
}

// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two
// 64x64->128 multiplies; the key is bumped by the golden-ratio and sqrt(3)-1
// Weyl increments between rounds.
__device__ __forceinline__ void philox4x64_10(unsigned long long c0, unsigned long long c1, unsigned long long c2,
                                              unsigned long long c3, unsigned long long k0, unsigned long long k1,
                                              unsigned long long out[4]) {
  const unsigned long long M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    unsigned long long hi0 = __umul64hi(M0, c0), lo0 = M0 * c0;
    unsigned long long hi1 = __umul64hi(M1, c2), lo1 = M1 * c2;
    unsigned long long n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    k0 += 0x9E3779B97F4A7C15ull;
    k1 += 0xBB67AE8584CAA73Bull;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

// Initial values of columns 8g .. 8g+7 of the row of `key` from one
// Philox4x64-10 block (counter (g, 0, 0, 0), key (merged key, init seed)):
// word k serves columns 8g+2k (its bits 63..40) and 8g+2k+1 (bits 39..16).
// Each 24-bit integer q gives (2q - 2^24) / 2^24 exactly; one fp32 multiply
// by the scale is the only rounding.
__device__ __forceinline__ void init_oct(const TableDev& T, unsigned long long key, uint32_t g, float v[8]) {
  unsigned long long w[4];
  philox4x64_10((unsigned long long)g, 0ull, 0ull, 0ull, key, T.init_seed, w);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int q0 = (int)(w[k] >> 40), q1 = (int)((w[k] >> 16) & 0xFFFFFFull);
    v[2 * k] = __fmul_rn((float)(2 * q0 - (1 << 24)) * (1.0f / 16777216.0f), T.init_scale);
    v[2 * k + 1] = __fmul_rn((float)(2 * q1 - (1 << 24)) * (1.0f / 16777216.0f), T.init_scale);
  }
}

// Write a fresh row: emb = init(key), m = v = 0.  Cooperatively by `nl`
// lanes (lane index `l` in [0, nl)), 16-byte stores.
__device__ __forceinline__ void init_row_coop(const TableDev& T, int32_t row, unsigned long long key, int l, int nl) {
  char* rec = row_ptr(T, row);
  const uint32_t d = T.dim;
  for (uint32_t g = l; g < (d + 7) / 8; g += nl) {
    float v[8];
    init_oct(T, key, g, v);
    if (T.row_dtype == MT_F32) {
      float4* e = reinterpret_cast<float4*>(rec) + 2 * g;
      e[0] = make_float4(v[0], v[1], v[2], v[3]);
      if (8 * g + 4 < d) e[1] = make_float4(v[4], v[5], v[6], v[7]);  // d is a multiple of 4
    } else {
      __nv_bfloat162 p0 = __floats2bfloat162_rn(v[0], v[1]);
      __nv_bfloat162 p1 = __floats2bfloat162_rn(v[2], v[3]);
      __nv_bfloat162 p2 = __floats2bfloat162_rn(v[4], v[5]);
      __nv_bfloat162 p3 = __floats2bfloat162_rn(v[6], v[7]);
      uint4 u;
      u.x = *reinterpret_cast<uint32_t*>(&p0);
      u.y = *reinterpret_cast<uint32_t*>(&p1);
      u.z = *reinterpret_cast<uint32_t*>(&p2);
      u.w = *reinterpret_cast<uint32_t*>(&p3);
      reinterpret_cast<uint4*>(rec)[g] = u;
    }
  }
  float4* mv = reinterpret_cast<float4*>(rec + T.emb_bytes);
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (uint32_t g = l; g < 2 * d / 4; g += nl) mv[g] = z;
}

// Pop `k` rows from the free stack for the lanes in `mask` (warp-aggregated).
// Returns this lane's row, or -1 when the pool ran out.
__device__ __forceinline__ int32_t pop_row_warp(const TableDev& T, unsigned mask) {
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(mask) - 1;
  const int k = __popc(mask);
  const int rank = __popc(mask & ((1u << lane) - 1u));
  long long old = 0;
  if (lane == leader) old = atomicAdd((unsigned long long*)&T.hdr->free_top, (unsigned long long)(-(long long)k));
  old = __shfl_sync(mask, old, leader);
  const long long avail = old < 0 ? 0 : (old < k ? old : k);
  if (lane == leader && avail < k) atomicAdd((unsigned long long*)&T.hdr->free_top, (unsigned long long)(k - avail));
  if (rank < avail) return T.free_stack[old - 1 - rank];
  return -1;
}

// Push rows back onto the free stack (warp-aggregated; lanes in `mask`).
__device__ __forceinline__ void push_row_warp(const TableDev& T, unsigned mask, int32_t row) {
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(mask) - 1;
  const int k = __popc(mask);
  const int rank = __popc(mask & ((1u << lane) - 1u));
  long long old = 0;
  if (lane == leader) old = (long long)atomicAdd((unsigned long long*)&T.hdr->free_top, (unsigned long long)k);
  old = __shfl_sync(mask, old, leader);
  T.free_stack[old + rank] = row;
}

// One probe of find_slot: 1 = the key is in slot s (sv holds it), -1 = an
// EMPTY slot ends the chain, 0 = go on (a tombstone is noted at probe t).
__device__ __forceinline__ int probe_one(unsigned long long key, const ulonglong2& sv, uint32_t t, long long* first_tomb) {
  if (sv.x == key) return 1;
  if (sv.x == kEmpty) return -1;
  if (sv.x == kTomb && *first_tomb < 0) *first_tomb = t;
  return 0;
}

// Find `key` along its probe sequence h_t = (h0 + t*S) mod M (MTGenRec,
// Theorem 1).  Returns the slot index, or -1 when an EMPTY slot or the probe
// limit ends the chain first.  *t_end receives the probe index where the
// search stopped, *t_tomb the first tombstone's probe index (or -1) and
// *row the row of a found key.  Each probe is one 16-byte load from L2;
// with S = 1, the probes after the first come four adjacent slots at a time.
// find_slot_from starts with the home slot s and its contents sv already
// loaded.
__device__ __forceinline__ long long find_slot_from(const TableDev& T, unsigned long long key, unsigned long long s,
                                                    ulonglong2 sv, long long* t_end, long long* t_tomb,
                                                    int32_t* row) {
  long long first_tomb = -1;
  uint32_t t = 0;
  if (T.max_probes > 0) {
    const int r = probe_one(key, sv, 0, &first_tomb);
    if (r != 0) {
      *t_end = 0;
      *t_tomb = first_tomb;
      if (r > 0) *row = (int32_t)(uint32_t)(sv.y & 0xFFFFFFFFull);
      return r > 0 ? (long long)s : -1;
    }
    t = 1;
    s = (s + T.S) & T.mask;
  }
  if (T.S == 1 && T.mask >= 3) {
    // linear probing: the rest of the chain in aligned groups of four adjacent slots (64 bytes of one line),
    // each group's slots loaded together and checked in probe order
    while (t < T.max_probes) {
      const unsigned long long g0 = s & ~3ull;
      const ulonglong2* gp = reinterpret_cast<const ulonglong2*>(&T.slots[g0]);
      const ulonglong2 q0 = __ldcg(gp), q1 = __ldcg(gp + 1), q2 = __ldcg(gp + 2), q3 = __ldcg(gp + 3);
      for (unsigned long long j = s - g0; j < 4 && t < T.max_probes; ++j, ++t) {
        const ulonglong2 q = j == 0 ? q0 : (j == 1 ? q1 : (j == 2 ? q2 : q3));
        const int r = probe_one(key, q, t, &first_tomb);
        if (r != 0) {
          *t_end = t;
          *t_tomb = first_tomb;
          if (r > 0) *row = (int32_t)(uint32_t)(q.y & 0xFFFFFFFFull);
          return r > 0 ? (long long)(g0 + j) : -1;
        }
      }
      s = (g0 + 4) & T.mask;
    }
  } else {
    for (; t < T.max_probes; ++t) {
      sv = __ldcg(reinterpret_cast<const ulonglong2*>(&T.slots[s]));
      const int r = probe_one(key, sv, t, &first_tomb);
      if (r != 0) {
        *t_end = t;
        *t_tomb = first_tomb;
        if (r > 0) *row = (int32_t)(uint32_t)(sv.y & 0xFFFFFFFFull);
        return r > 0 ? (long long)s : -1;
      }
      s = (s + T.S) & T.mask;
    }
  }
  *t_end = T.max_probes;
  *t_tomb = first_tomb;
  return -1;
}

// Find `key` from its home slot (loading it first).
__device__ __forceinline__ long long find_slot(const TableDev& T, unsigned long long key, long long* t_end,
                                               long long* t_tomb, int32_t* row) {
  const unsigned long long s = home_slot(T, key);
  return find_slot_from(T, key, s, __ldcg(reinterpret_cast<const ulonglong2*>(&T.slots[s])), t_end, t_tomb, row);
}

// ---- host-side launchers (defined in the kernel files) --------------------

struct LookupWs;
struct BackwardWs;

// ---- packed fp32 pairs -------------------------------------------------------
// Two adjacent columns travel in one 64-bit register (low half: the even
// column) and are combined by the paired fp32 instructions (add/sub
// .rn.f32x2): each half is rounded to nearest on its own, exactly like the
// scalar __fadd_rn/__fsub_rn, at one instruction per pair.  Only additions
// and subtractions are paired: with no product in the chain nothing can be
// fused, so TwoSum stays exact.
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pk(float lo, float hi) {
  f32x2 d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ float2 upk(f32x2 a) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(a));
  return r;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// Two bf16 in one word (low half: the even column) widened to fp32 (exact).
__device__ __forceinline__ f32x2 bf16x2_to_f32x2(uint32_t w) { return pk(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u)); }

// s + e = a + b exactly, per half (Knuth's TwoSum).
__device__ __forceinline__ void two_sum(f32x2 a, f32x2 b, f32x2& s, f32x2& e) {
  s = add2(a, b);
  const f32x2 bb = sub2(s, a);
  e = add2(sub2(a, sub2(s, bb)), sub2(b, bb));
}


}  // namespace mt
