// Forward path of the merged dynamic embedding table: merged-key encoding,
// ID deduplication in two stages, find/insert with odd-step probing, and the
// embedding gather.
//
// Pages: "MTGenRec" TL;DR and abstract (a dynamic embedding table built on
// hashing, feature tables merged into one, deduplication of IDs in two
// stages to speed up lookups, keys inserted while training runs); Theorem 1 (probe sequence h_t = (h0 + t*S) mod 2^n
// with S odd covers the table); "MTGR" section 5, Embedding Lookup (IDs stay
// unique).
//
// Kernels, in launch order (one CTA per tile of kTile consecutive positions):
//  k_dedup_claim     encode keys; stage 1: dedup inside the tile with a
//                    shared-memory hash (CAS insert, atomicMin of the first
//                    position); stage 2: each tile-local unique claims its
//                    key in a global scratch hash and lowers the key's first
//                    position there (atomicMin); the one thread whose CAS
//                    put the key there finds or inserts it in the table
//                    (odd-step probing, tombstone reuse, warp-aggregated
//                    row pops), publishes the row in the scratch hash and
//                    its block initialises the fresh rows.
//  k_assign_resolve  a tile owns a key when its first position is the key's
//                    global first position; owners take unique indices in
//                    first-occurrence order (tile offsets by a decoupled
//                    look-back over the tiles' owner counts) and publish
//                    them in the scratch hash; key and row come from there.
//  k_expand          per tile-local unique: its unique index and counts;
//                    per position: the inverse index.
//  k_gather          the 16-byte vectorised row gather, grid-stride over
//                    the batch with four independent items per thread.
#include <atomic>

#include "mt_kernels.cuh"

namespace mt {

namespace {

// Home slot in the stage-1 shared hash of kHSA slots (multiply-shift range reduction).
__device__ __forceinline__ uint32_t stage1_hash(unsigned long long key) {
  return (uint32_t)(((mix64(key ^ 0x2545F4914F6CDD1Dull) >> 32) * (unsigned long long)kHSA) >> 32);
}

__device__ __forceinline__ unsigned long long stage2_hash(unsigned long long key) {
  return mix64(key ^ 0x9FB21C651E98DF25ull);
}

// Exclusive scan of one int per thread over a block of NT threads; *total
// receives the block sum.  Contains __syncthreads (all threads must call).
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < NT / 32 ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += y;
    }
    if (lane < NT / 32) s_warp[lane] = w;
  }
  __syncthreads();
  const int r = (warp ? s_warp[warp - 1] : 0) + x - v;
  *total = s_warp[NT / 32 - 1];
  __syncthreads();
  return r;
}

template <int NT>
__device__ __forceinline__ int block_sum(int v, int* s_warp) {
  int t;
  block_exclusive_scan<NT>(v, s_warp, &t);
  return t;
}

constexpr size_t kSmemA = kHSA * 8 + kHSA * 4 + kTile * 4 + kTile * 2 + (MT_MAX_FEATURES + 1) * 8 + MT_MAX_FEATURES;

__global__ void __launch_bounds__(kThreadsA, 3) k_dedup_claim(const LookupParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned long long* s_key = reinterpret_cast<unsigned long long*>(smem);  // [kHSA] stage-1 hash keys
  uint32_t* s_min = reinterpret_cast<uint32_t*>(s_key + kHSA);             // [kHSA] first local position, then local index
  uint32_t* s_item = s_min + kHSA;                                         // [kTile] (hash slot << 16) | first position of local unique l
  uint16_t* s_pslot = reinterpret_cast<uint16_t*>(s_item + kTile);         // [kTile] hash slot of each position
  long long* s_off = reinterpret_cast<long long*>(s_pslot + kTile);        // [F + 1]
  unsigned char* s_tid = reinterpret_cast<unsigned char*>(s_off + MT_MAX_FEATURES + 1);  // [F]
  __shared__ int s_warp[kThreadsA / 32];
  __shared__ int s_frange[2];  // features of the tile's first and last position
  __shared__ int s_nnew;       // fresh rows listed by stage 2

  const int tile = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31;
  const long long base = (long long)tile * kTile;
  const int cnt = (int)min((long long)kTile, p.n - base);

  for (int i = tid; i < kHSA; i += kThreadsA) {
    s_key[i] = kEmpty;
    s_min[i] = 0xFFFFFFFFu;
  }
  for (int i = tid; i <= p.F; i += kThreadsA) s_off[i] = p.feat_off[i];
  for (int i = tid; i < p.F; i += kThreadsA) s_tid[i] = p.table_ids[i];
  if (tid == 0) {
    s_nnew = 0;
    p.tile_status[tile] = 0ull;  // no owner count published yet (read by k_assign_resolve)
    if (tile == 0) *p.ticket = 0;
  }
  __syncthreads();
  if (tid < 2) {  // feature of position base (tid 0) and base + cnt - 1 (tid 1): last f with off[f] <= i
    const long long i = base + (tid == 0 ? 0 : cnt - 1);
    int lo = 0, hi = p.F;  // off[lo] <= i < off[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_off[mid] <= i) lo = mid; else hi = mid;
    }
    s_frange[tid] = lo;
  }
  __syncthreads();
  const int f_first = s_frange[0], f_last = s_frange[1];

  // ---- encode + stage 1 (tile-local dedup) ----
  bool bad = false;
  long long idv[kPPTA];  // every ID load in flight before the shared-memory work
#pragma unroll
  for (int k = 0; k < kPPTA; ++k) {
    const int lp = k * kThreadsA + tid;
    idv[k] = lp < cnt ? __ldg(&p.ids[base + lp]) : 0;
  }
#pragma unroll
  for (int k = 0; k < kPPTA; ++k) {
    const int lp = k * kThreadsA + tid;  // a warp covers 32 consecutive positions
    const bool in = lp < cnt;
    unsigned long long key = kEmpty;
    bool valid = false;
    if (in) {
      const long long i = base + lp;
      const long long id = idv[k];
      int lo = f_first, hi = f_last + 1;  // off[lo] <= i < off[hi]; one step when the tile has one feature
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_off[mid] <= i) lo = mid; else hi = mid;
      }
      valid = id >= 0 && (unsigned long long)id < kIdLimit;
      key = ((unsigned long long)s_tid[lo] << 56) | (unsigned long long)id;
      bad |= !valid;
    }
    if (valid) {
      uint32_t h = stage1_hash(key);
      for (int probe = 0; probe < kHSA; ++probe) {
        const unsigned long long prev = atomicCAS(&s_key[h], kEmpty, key);
        if (prev == kEmpty || prev == key) break;
        h = h + 1 == (uint32_t)kHSA ? 0u : h + 1;
      }
      atomicMin(&s_min[h], (uint32_t)lp);
      s_pslot[lp] = (uint16_t)h;
    } else if (in) {
      s_pslot[lp] = kNoIdx;
    }
  }
  if (bad) latch_error(p.T.hdr, MT_EKEY);
  __syncthreads();

  // ---- local uniques in first-occurrence order (contiguous positions per thread) ----
  uint32_t flags = 0;
  int c = 0;
#pragma unroll
  for (int k = 0; k < kPPTA; ++k) {
    const int lp = tid * kPPTA + k;
    if (lp < cnt) {
      const uint16_t sl = s_pslot[lp];
      if (sl != kNoIdx && s_min[sl] == (uint32_t)lp) {
        flags |= 1u << k;
        ++c;
      }
    }
  }
  int L;
  int l = block_exclusive_scan<kThreadsA>(c, s_warp, &L);  // every s_min read above precedes its barriers
#pragma unroll
  for (int k = 0; k < kPPTA; ++k) {
    if (flags & (1u << k)) {
      const int lp = tid * kPPTA + k;
      const uint16_t sl = s_pslot[lp];
      s_min[sl] = (uint32_t)l;
      s_item[l] = ((uint32_t)sl << 16) | (uint32_t)lp;
      ++l;
    }
  }
  __syncthreads();

  uint16_t* lidx = p.lidx + base;
  for (int lp = tid; lp < cnt; lp += kThreadsA) {
    const uint16_t sl = s_pslot[lp];
    lidx[lp] = sl == kNoIdx ? kNoIdx : (uint16_t)s_min[sl];
  }

  // ---- stage 2: claim every local unique in the global scratch hash; the
  // thread whose CAS puts a key there is the only one in the grid to see it
  // EMPTY, and it resolves the key in the table right away (find, or insert
  // with tombstone reuse and a warp-aggregated row pop) and publishes the
  // row in the scratch hash ----
  __syncthreads();  // s_min and s_pslot are free from here: fresh rows are listed there
  int32_t* s_newrow = reinterpret_cast<int32_t*>(s_min);  // [kHSA >= kTile] rows to initialise
  uint16_t* s_newli = s_pslot;                           // [kTile] their local uniques
  const size_t lb = (size_t)tile * kTile;
  const uint32_t step = (uint32_t)p.T.hdr->step;
  for (int li0 = 0; li0 < L; li0 += kThreadsA) {  // warp-uniform trip count (row pops are warp-wide)
    const int li = li0 + tid;
    const bool act = li < L;
    unsigned long long key = 0, h = 0;
    bool won = false;
    if (act) {
      const uint32_t it = s_item[li];
      key = s_key[it >> 16];
      const uint32_t gpos = (uint32_t)(base + (it & 0xFFFFu));
      h = stage2_hash(key) & p.scratch_mask;
      for (unsigned long long probe = 0; probe <= p.scratch_mask; ++probe) {
        unsigned long long cur = load_key_relaxed(&p.sc_key[h]);
        if (cur == kEmpty) {
          cur = atomicCAS(&p.sc_key[h], kEmpty, key);
          if (cur == kEmpty) {
            won = true;
            cur = key;
          }
        }
        if (cur == key) break;
        h = (h + 1) & p.scratch_mask;
      }
      atomicMin(&p.sc_minpos[h], gpos);
      p.lfirst[lb + li] = gpos;
      p.lsslot[lb + li] = (uint32_t)h;
    }
    int32_t row = -1;
    bool claimed = false;
    unsigned long long cs = 0;
    if (won) {
      long long t_end, t_tomb;
      const long long sidx = find_slot(p.T, key, &t_end, &t_tomb, &row);
      if (sidx < 0 && p.insert_missing) {
        // absent, and no other thread inserts it (it won the scratch hash):
        // take the first tombstone of its chain, else the EMPTY slot that
        // ended the chain, else the next free slot after them
        long long t = t_tomb >= 0 ? t_tomb : t_end;
        unsigned long long slot = (home_slot(p.T, key) + (unsigned long long)t * p.T.S) & p.T.mask;
        for (; t < (long long)p.T.max_probes; ++t) {
          const unsigned long long k = load_key_relaxed(&p.T.slots[slot].key);
          if ((k == kEmpty || k == kTomb) && atomicCAS(&p.T.slots[slot].key, k, key) == k) {
            claimed = true;
            cs = slot;
            break;
          }
          slot = (slot + p.T.S) & p.T.mask;
        }
        if (!claimed) latch_error(p.T.hdr, MT_EFULL);
      }
    }
    const unsigned need = __ballot_sync(kFull, claimed);
    if (claimed) {
      row = pop_row_warp(p.T, need);
      if (row < 0) {
        atomicExch(&p.T.slots[cs].key, kTomb);  // give the slot back; the chain stays intact
        latch_error(p.T.hdr, MT_EFULL);
      } else {
        p.T.slots[cs].row = row;
        p.T.slots[cs].meta = step;
        const int q = atomicAdd(&s_nnew, 1);
        s_newrow[q] = row;
        s_newli[q] = (uint16_t)li;
      }
    }
    if (won) p.sc_row[h] = row;
  }
  if (tid == 0) p.tile_L[tile] = L;
  __syncthreads();

  // initialise fresh rows, one team of lanes per row
  const int nnew = s_nnew;
  const uint32_t vecs = p.T.row_dtype == MT_F32 ? p.T.dim / 4 : p.T.dim / 8;
  int team = 1;
  while (team < 32 && team < (int)vecs) team <<= 1;
  const int nteams = kThreadsA / team, my_team = tid / team, lt = tid % team;
  for (int q = my_team; q < nnew; q += nteams)
    init_row_coop(p.T, s_newrow[q], s_key[s_item[s_newli[q]] >> 16], lt, team);
}

// Tile status words of the owner-count scan: flag in the high half
// (kStatAgg: the tile's own owner count; kStatIncl: owners of this tile and
// all before it), value in the low half.
constexpr unsigned long long kStatAgg = 1ull << 32, kStatIncl = 2ull << 32;
constexpr int kLookbackTries = 1 << 22;

__device__ __forceinline__ void store_status(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long load_status(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Owners take unique indices in first-occurrence order: a tile's owners are
// the tile-local uniques whose first position is the key's global first
// position.  Tiles are taken in start order (a ticket), so every tile
// before a block's tile has started; the block publishes its owner count,
// then its first warp adds up the counts of the tiles before it from their
// status words (a decoupled look-back: a tile that already knows its
// inclusive count ends the walk).  A wait that runs out of polls latches
// MT_ETIMEOUT and leaves every index in bounds.  Key and row of each owner
// come from the scratch hash, where its claimer put them.
__global__ void __launch_bounds__(kThreads, 6) k_assign_resolve(const LookupParams p) {
  __shared__ int s_warp[kThreads / 32];
  __shared__ int s_tile;
  __shared__ long long s_off;

  const int tid = threadIdx.x, lane = tid & 31;
  if (tid == 0) s_tile = atomicAdd(p.ticket, 1);
  __syncthreads();
  const int tile = s_tile;
  const int L = p.tile_L[tile];
  const size_t lb = (size_t)tile * kTile;

  uint32_t sl[kPPT], lf[kPPT], mp[kPPT];  // each round of loads all in flight at once
#pragma unroll
  for (int k = 0; k < kPPT; ++k) {
    const int l = tid * kPPT + k;
    sl[k] = l < L ? __ldg(&p.lsslot[lb + l]) : 0u;
    lf[k] = l < L ? __ldg(&p.lfirst[lb + l]) : 0u;
  }
#pragma unroll
  for (int k = 0; k < kPPT; ++k) mp[k] = tid * kPPT + k < L ? __ldcg(&p.sc_minpos[sl[k]]) : 1u;
  uint32_t flags = 0;
  int c = 0;
#pragma unroll
  for (int k = 0; k < kPPT; ++k) {
    if (mp[k] == lf[k]) {  // this tile holds the key's first position
      flags |= 1u << k;
      ++c;
    }
  }
  int O;
  int j = block_exclusive_scan<kThreads>(c, s_warp, &O);
  unsigned long long* st = p.tile_status;
  if (tid < 32) {
    const bool stall = tile == 0 && (p.T.flags & MT_FLAG_TEST_STALL_SCAN);  // testing only: never publish
    if (lane == 0 && !stall) store_status(st + tile, (tile == 0 ? kStatIncl : kStatAgg) | (unsigned long long)O);
    long long excl = 0;
    bool ok = true;
    for (int q = tile - 1, tries = 0; q >= 0;) {
      const int pq = q - lane;
      const unsigned long long v = pq >= 0 ? load_status(st + pq) : kStatIncl;  // before tile 0: inclusive 0
      const unsigned long long flag = v & ~0xFFFFFFFFull;
      if (__ballot_sync(kFull, flag != 0) != kFull) {  // a tile in this window has not published yet
        if (++tries >= kLookbackTries) {
          ok = false;
          break;
        }
        continue;
      }
      const unsigned incl = __ballot_sync(kFull, flag == kStatIncl);
      const int stop = incl ? __ffs(incl) - 1 : 31;
      long long x = lane <= stop ? (long long)(v & 0xFFFFFFFFull) : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
      excl += x;
      if (incl) break;
      q -= 32;
    }
    if (!ok) excl = 0;  // in bounds (every index stays below this tile's owner count); the call reports the error
    if (lane == 0) {
      if (!ok) latch_error(p.T.hdr, MT_ETIMEOUT);
      if (tile > 0) store_status(st + tile, kStatIncl | (unsigned long long)(excl + O));
      s_off = excl;
    }
  }
  __syncthreads();
  const long long off = s_off;
  if (tid == 0 && tile == p.ntiles - 1) *p.num_unique = off + O;
  unsigned long long key[kPPT];
  int32_t row[kPPT];
#pragma unroll
  for (int k = 0; k < kPPT; ++k) {
    key[k] = (flags >> k) & 1u ? __ldcg(&p.sc_key[sl[k]]) : 0ull;
    row[k] = (flags >> k) & 1u ? __ldcg(&p.sc_row[sl[k]]) : -1;
  }
#pragma unroll
  for (int k = 0; k < kPPT; ++k) {
    if (flags & (1u << k)) {
      const int u = (int)(off + j);
      p.sc_uidx[sl[k]] = u;
      p.unique_keys[u] = key[k];
      p.unique_rows[u] = row[k];
      p.counts[u] = 0;
      ++j;
    }
  }
}

__global__ void __launch_bounds__(kThreads) k_expand(const LookupParams p) {
  __shared__ int32_t s_lcnt[kTile];   // positions of local unique l in this tile, then its rank base
  __shared__ int32_t s_u[kTile];      // unique index of local unique l
  __shared__ uint16_t s_pl[kTile];    // local unique of each position
  __shared__ uint16_t s_lrank[kTile]; // rank of each position among its local unique's positions

  const int tile = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  const long long base = (long long)tile * kTile;
  const int cnt = (int)min((long long)kTile, p.n - base);
  const int L = p.tile_L[tile];
  const size_t lb = (size_t)tile * kTile;

  for (int l = tid; l < L; l += kThreads) s_lcnt[l] = 0;
  __syncthreads();
  uint32_t liv[kPPT];  // every local-index load in flight before the warp-synchronous work
#pragma unroll
  for (int k = 0; k < kPPT; ++k) {
    const int lp = k * kThreads + tid;
    liv[k] = lp < cnt ? __ldg(&p.lidx[base + lp]) : kNoIdx;
  }
#pragma unroll
  for (int k = 0; k < kPPT; ++k) {
    const int lp = k * kThreads + tid;
    const bool in = lp < cnt;
    const uint32_t li = liv[k];
    if (in) s_pl[lp] = (uint16_t)li;
    if (in && li != kNoIdx) s_lrank[lp] = (uint16_t)atomicAdd(&s_lcnt[li], 1);
  }
  __syncthreads();
  // one atomic per (tile, unique): the old count is where this tile's
  // positions start among all positions of the unique
  for (int l0 = tid; l0 < L; l0 += 4 * kThreads) {  // four independent atomics in flight per thread
    int32_t u[4], old[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int l = l0 + k * kThreads;
      u[k] = l < L ? __ldcg(&p.sc_uidx[__ldg(&p.lsslot[lb + l])]) : 0;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int l = l0 + k * kThreads;
      if (l < L) old[k] = atomicAdd(&p.counts[u[k]], s_lcnt[l]);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int l = l0 + k * kThreads;
      if (l < L) {
        s_u[l] = u[k];
        s_lcnt[l] = old[k];
      }
    }
  }
  __syncthreads();
  for (int lp = tid; lp < cnt; lp += kThreads) {
    const uint16_t li = s_pl[lp];
    p.inverse[base + lp] = li == kNoIdx ? -1 : s_u[li];
    if (p.ranks != nullptr) p.ranks[base + lp] = li == kNoIdx ? -1 : s_lcnt[li] + s_lrank[lp];
  }
}

// out[i] = row of unique inverse[i] (zeros for an invalid ID or an absent
// key): 16-byte items (position, vector), consecutive threads on consecutive
// items; each round a block covers kGatherILP * blockDim contiguous items
// (one independent item in flight per thread and step of blockDim), and the
// blocks stride over the whole batch so every SM stays busy to the end.
constexpr int kGatherILP = 2;
__global__ void __launch_bounds__(256) k_gather(const LookupParams p) {
  const int vec16 = (int)(p.T.emb_bytes / 16);
  const int vshift = (vec16 & (vec16 - 1)) == 0 ? __ffs(vec16) - 1 : -1;
  const long long total = p.n * vec16;
  const long long span = (long long)kGatherILP * blockDim.x;  // items a block covers per round, contiguous
  uint4* out = reinterpret_cast<uint4*>(p.out_rows);
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  for (long long b0 = (long long)blockIdx.x * span; b0 < total; b0 += (long long)gridDim.x * span) {
    const long long i0 = b0 + threadIdx.x;
    const long long stride = blockDim.x;
    int32_t row[kGatherILP];
#pragma unroll
    for (int k = 0; k < kGatherILP; ++k) {
      const long long it = i0 + k * stride;
      row[k] = -1;
      if (it < total) {
        const long long i = vshift >= 0 ? (it >> vshift) : it / vec16;
        const int32_t u = __ldg(&p.inverse[i]);
        if (u >= 0) row[k] = __ldg(&p.unique_rows[u]);
      }
    }
    uint4 v[kGatherILP];
#pragma unroll
    for (int k = 0; k < kGatherILP; ++k) {
      const long long it = i0 + k * stride;
      v[k] = zero;
      if (it < total && row[k] >= 0) {
        const long long i = vshift >= 0 ? (it >> vshift) : it / vec16;
        v[k] = __ldg(reinterpret_cast<const uint4*>(row_ptr(p.T, row[k])) + (it - i * vec16));
      }
    }
#pragma unroll
    for (int k = 0; k < kGatherILP; ++k) {
      const long long it = i0 + k * stride;
      if (it < total) __stcs(out + it, v[k]);
    }
  }
}

}  // namespace

LookupWsLayout lookup_ws_layout(long long n) {
  LookupWsLayout L{};
  L.ntiles = (int)((n + kTile - 1) / kTile);
  unsigned long long ss = 1024;
  while (ss < 2ull * (unsigned long long)n) ss <<= 1;
  L.scratch_slots = ss;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const size_t cap = (size_t)L.ntiles * kTile;
  L.sc_key = take(ss * 8);
  L.sc_minpos = take(ss * 4);
  L.sc_uidx = take(ss * 4);
  L.sc_row = take(ss * 4);
  L.tile_L = take((size_t)L.ntiles * 4);
  L.tile_status = take((size_t)L.ntiles * 8);
  L.ticket = take(16);
  L.lfirst = take(cap * 4);
  L.lsslot = take(cap * 4);
  L.lidx = take(cap * 2);
  L.total = off;
  return L;
}

cudaError_t launch_lookup(const LookupParams& p, cudaStream_t s) {
  if (p.n == 0) return cudaMemsetAsync(p.num_unique, 0, sizeof(long long), s);
  static std::atomic<int> gather_grid[kMaxDevices];  // 0: not set up on that device yet
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  if (gather_grid[dev].load(std::memory_order_relaxed) == 0) {
    cudaError_t e = cudaFuncSetAttribute(k_dedup_claim, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemA);
    if (e != cudaSuccess) return e;
    int sms = 0, per = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, k_gather, 256, 0);
    gather_grid[dev].store(sms * (per > 0 ? per : 1), std::memory_order_relaxed);
  }
  // keys EMPTY and first positions "none", in one memset: the layout puts
  // sc_minpos right after sc_key (8-byte keys keep it 256-byte aligned)
  const size_t clear = (size_t)(reinterpret_cast<const char*>(p.sc_minpos) - reinterpret_cast<const char*>(p.sc_key)) +
                       (p.scratch_mask + 1) * 4;
  cudaError_t e = cudaMemsetAsync(p.sc_key, 0xFF, clear, s);
  if (e != cudaSuccess) return e;
  {
    MT_LAUNCH("k_dedup_claim", s);
    k_dedup_claim<<<p.ntiles, kThreadsA, kSmemA, s>>>(p);
  }
  {
    MT_LAUNCH("k_assign_resolve", s);
    k_assign_resolve<<<p.ntiles, kThreads, 0, s>>>(p);
  }
  {
    MT_LAUNCH("k_expand", s);
    k_expand<<<p.ntiles, kThreads, 0, s>>>(p);
  }
  if (p.out_rows != nullptr) {
    MT_LAUNCH("k_gather", s);
    k_gather<<<gather_grid[dev].load(std::memory_order_relaxed), 256, 0, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace mt
