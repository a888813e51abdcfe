// Forward path of the merged dynamic embedding table: merged-key encoding,
// ID deduplication in two stages, find/insert with odd-step probing, and the
// embedding gather.
//
// Pages: "MTGenRec" TL;DR and abstract (a dynamic embedding table built on
// hashing, feature tables merged into one, deduplication of IDs in two
// stages to speed up lookups, keys inserted while training runs); Theorem 1
// (probe sequence h_t = (h0 + t*S) mod 2^n with S odd covers the table);
// "MTGR" section 5, Embedding Lookup (no duplicate IDs on either side of an
// exchange).
//
// The unique keys come out in first-occurrence order.  Kernels, in launch
// order (after one memset that clears the stage-2 scratch hash):
//  k_local    stage 1, per tile of kTile positions: encode keys, dedup inside
//             the tile with a shared-memory hash (first position, count and
//             each position's rank among its key's positions); every
//             tile-local unique becomes one record {key, first position,
//             count}, the tile's records stored together.
//  k_claim    stage 2, one thread per record over the whole GPU: a new key
//             is installed in the global scratch hash by one 128-bit CAS
//             with its record's first position and count; a present key gets
//             one 64-bit atomic that adds the record's count and returns the
//             key's count and first position so far (the count is the rank
//             base of the tile's positions), and an atomicMin only when the
//             record lowers the first position.  The thread that installed a
//             key lists it as a distinct key.
//  k_resolve  one thread per distinct key: find the key in the table
//             (odd-step probing) or insert it (first tombstone or EMPTY slot
//             of its chain, rows popped once per block; fresh rows listed for
//             k_expand); mark the key's first position in a bitmap of the
//             batch's positions.
//  k_prefix   per tile (a warp, a lane per 64-position word): first positions
//             before each word of the tile; the last block to finish turns the
//             tile counts into tile offsets.
//  k_number   one thread per distinct key: its unique index is the number of
//             first positions before its own (tile offset + word offset + a
//             popcount), which is first-occurrence order; it writes the
//             unique key, row and count and leaves the index and the row in
//             the scratch slot.
//  k_expand   per tile: inverse index, rank and table row of every position;
//             then a share of the fresh rows is initialised (Philox-keyed values,
//             m = v = 0) by teams of lanes, filling the issue slots of this
//             latency-bound kernel.
//  k_gather   the 16-byte vectorised row gather over the whole batch.
// No kernel waits on another block.
#include <atomic>

#include "mt_kernels.cuh"

namespace mt {

namespace {

// Home slot in the stage-1 shared hash of kHSA slots (multiply-shift range reduction).
__device__ __forceinline__ uint32_t stage1_hash(unsigned long long key) {
  return (uint32_t)(((mix64(key ^ 0x2545F4914F6CDD1Dull) >> 32) * (unsigned long long)kHSA) >> 32);
}

// Home slot in the stage-2 scratch hash of ss slots (ss < 2^32).
__device__ __forceinline__ unsigned long long stage2_home(unsigned long long key, unsigned long long ss) {
  return ((mix64(key ^ 0x9FB21C651E98DF25ull) >> 32) * ss) >> 32;
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

constexpr size_t kSmemA = kHSA * 8 + kHSA * 4 + kHSA * 4 + kTile * 2 + (MT_MAX_FEATURES + 1) * 8 + MT_MAX_FEATURES;

__global__ void __launch_bounds__(kThreadsA, 4) k_local(const LookupParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned long long* s_key = reinterpret_cast<unsigned long long*>(smem);  // [kHSA] stage-1 hash keys
  uint32_t* s_min = reinterpret_cast<uint32_t*>(s_key + kHSA);             // [kHSA] first local position, then local index
  uint32_t* s_cnt = s_min + kHSA;                                          // [kHSA] positions per key
  uint16_t* s_pslot = reinterpret_cast<uint16_t*>(s_cnt + kHSA);           // [kTile] hash slot of each position
  long long* s_off = reinterpret_cast<long long*>(s_pslot + kTile);        // [F + 1]
  unsigned char* s_tid = reinterpret_cast<unsigned char*>(s_off + MT_MAX_FEATURES + 1);  // [F]
  __shared__ int s_warp[kThreadsA / 32];
  __shared__ int s_frange[2];  // features of the tile's first and last position
  __shared__ int s_rbase;      // where the tile's records start

  const int tile = blockIdx.x;
  const int tid = threadIdx.x;
  const long long base = (long long)tile * kTile;
  const int cnt = (int)min((long long)kTile, p.n - base);

  for (int i = tid; i < kHSA; i += kThreadsA) {
    s_key[i] = kEmpty;
    s_min[i] = 0xFFFFFFFFu;
    s_cnt[i] = 0u;
  }
  for (int i = tid; i <= p.F; i += kThreadsA) s_off[i] = p.feat_off[i];
  for (int i = tid; i < p.F; i += kThreadsA) s_tid[i] = p.table_ids[i];
  if (tid == 0 && tile == 0) *p.done = 0u;
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

  // ---- encode + stage 1 (tile-local dedup: first position, count, rank) ----
  bool bad = false;
  uint32_t rk[kPPTA];    // each position's rank, stored with its local index at the end
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
      if (p.keys_in) {  // a merged key as it is; table id 255 holds the sentinels
        key = (unsigned long long)id;
        valid = (key >> 56) != 0xFFull;
      } else {
        valid = id >= 0 && (unsigned long long)id < kIdLimit;
        key = ((unsigned long long)s_tid[lo] << 56) | (unsigned long long)id;
      }
      bad |= !valid;
    }
    uint16_t rank = 0;
    if (valid) {
      uint32_t h = stage1_hash(key);
      for (int probe = 0; probe < kHSA; ++probe) {
        const unsigned long long prev = atomicCAS(&s_key[h], kEmpty, key);
        if (prev == kEmpty || prev == key) break;
        h = h + 1 == (uint32_t)kHSA ? 0u : h + 1;
      }
      atomicMin(&s_min[h], (uint32_t)lp);
      rank = (uint16_t)atomicAdd(&s_cnt[h], 1u);
      s_pslot[lp] = (uint16_t)h;
    } else if (in) {
      s_pslot[lp] = kNoIdx;
    }
    rk[k] = rank;  // the position's rank among its key's positions in the tile
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
  // the tile's records, stored together (one global atomic per tile)
  if (tid == 0) {
    s_rbase = L ? (int)(atomicAdd(p.rec_n, (uint32_t)L) + 1u) : 0;  // the counter starts at 2^32 - 1
    p.tile_L[tile] = L;
    p.tile_rec[tile] = s_rbase;
  }
  __syncthreads();
  const int rbase = s_rbase;
#pragma unroll
  for (int k = 0; k < kPPTA; ++k) {
    if (flags & (1u << k)) {
      const int lp = tid * kPPTA + k;
      const uint16_t sl = s_pslot[lp];
      s_min[sl] = (uint32_t)l;
      const ulonglong2 r = make_ulonglong2(s_key[sl], (unsigned long long)(uint32_t)(base + lp) |
                                                         ((unsigned long long)s_cnt[sl] << 32));
      __stcg(reinterpret_cast<ulonglong2*>(p.rec) + rbase + l, r);
      ++l;
    }
  }
  __syncthreads();

#pragma unroll
  for (int k = 0; k < kPPTA; ++k) {  // the positions this thread hashed: {local index, rank} in one word
    const int lp = k * kThreadsA + tid;
    if (lp < cnt) {
      const uint16_t sl = s_pslot[lp];
      p.llr[base + lp] = (sl == kNoIdx ? (uint32_t)kNoIdx : s_min[sl]) | (rk[k] << 16);
    }
  }
}

// Stage 2: one thread per record {key, first position in its tile, count in
// its tile}, two records per thread in flight, over the whole GPU.  Each
// record's chain of global round trips is short: a load of the key's home
// slot, then either one 128-bit CAS that installs a new key with its first
// position and count, or one 64-bit atomic that adds to a present key (and an
// atomicMin when the record lowers the key's first position).  Nothing waits
// on a block barrier in between: the block's distinct keys collect in shared
// memory and are listed once at the end (or once per round when the block's
// share of records could overflow that buffer).
constexpr int kClaimILP = 2;     // records per thread per round
constexpr int kWinCap = 4096;    // distinct keys a block holds before listing them

// 128-bit compare-and-swap of a whole scratch slot (sm_90 and later): returns the slot's previous contents.
__device__ __forceinline__ ulonglong2 cas_slot(ScSlot* slot, ulonglong2 expect, ulonglong2 desired) {
  ulonglong2 old;
  asm volatile(
      "{\n\t"
      ".reg .b128 d, e, v;\n\t"
      "mov.b128 e, {%2, %3};\n\t"
      "mov.b128 v, {%4, %5};\n\t"
      "atom.global.cas.b128 d, [%6], e, v;\n\t"
      "mov.b128 {%0, %1}, d;\n\t"
      "}"
      : "=l"(old.x), "=l"(old.y)
      : "l"(expect.x), "l"(expect.y), "l"(desired.x), "l"(desired.y), "l"(slot)
      : "memory");
  return old;
}

// Claims `key` in the scratch hash from slot h whose contents sv were loaded
// already: the first slot holding the key, or an EMPTY one, which a single
// 128-bit CAS fills with the key, the record's first position and its count
// at once.  Returns whether this call put the key there (its record's rank
// base is then 0 and nothing is left to add); otherwise *first_seen is the
// first position the slot held when it was seen with the key.
__device__ __forceinline__ bool claim_from(const LookupParams& p, unsigned long long key, uint32_t gpos,
                                           uint32_t lcount, unsigned long long& h, ulonglong2 sv,
                                           uint32_t* first_seen) {
  // a fresh slot: key EMPTY, first "none", count - 1 = 2^32 - 1 (the memset); {first, count - 1} change
  // only after a key is in the slot
  const ulonglong2 fresh = make_ulonglong2(kEmpty, ~0ull);
  const ulonglong2 mine = make_ulonglong2(key, (unsigned long long)gpos | ((unsigned long long)(lcount - 1u) << 32));
  for (unsigned long long probe = 0; probe < p.ss; ++probe) {
    // a plain load first: the hottest keys have a record from nearly every tile, and a CAS on their
    // slot would queue behind every other tile's at the L2
    if (sv.x == kEmpty) {
      sv = cas_slot(&p.sc[h], fresh, mine);
      if (sv.x == kEmpty) return true;  // the slot was fresh: it now holds this record
    }
    if (sv.x == key) {
      *first_seen = (uint32_t)(sv.y & 0xFFFFFFFFull);
      return false;
    }
    h = h + 1 == p.ss ? 0ull : h + 1;
    sv = __ldcg(reinterpret_cast<const ulonglong2*>(&p.sc[h]));
  }
  *first_seen = 0u;
  return false;  // not reached: the scratch hash has more slots than records
}

// Lists the block's distinct keys held in s_win (call with the whole block).
__device__ __forceinline__ void list_winners(const LookupParams& p, int32_t* s_win, int* s_nwin, int* s_wbase) {
  __syncthreads();
  const int nwin = *s_nwin;
  if (threadIdx.x == 0 && nwin > 0) *s_wbase = (int)(atomicAdd(p.ulist_n, (uint32_t)nwin) + 1u);  // from 2^32 - 1
  __syncthreads();
  for (int i = threadIdx.x; i < nwin; i += kThreadsC) p.ulist[*s_wbase + i] = s_win[i];
  __syncthreads();
  if (threadIdx.x == 0) *s_nwin = 0;
  __syncthreads();
}

__global__ void __launch_bounds__(kThreadsC) k_claim(const LookupParams p) {
  __shared__ int s_nwin, s_wbase;
  __shared__ int32_t s_win[kWinCap];
  const int tid = threadIdx.x;
  const uint32_t R = *p.rec_n + 1u;  // the counter starts at 2^32 - 1
  const uint32_t span = kThreadsC * kClaimILP;
  const uint32_t stride = gridDim.x * span;
  const uint32_t first = blockIdx.x * span;
  const uint32_t rounds = first < R ? (R - first + stride - 1) / stride : 0u;
  const bool list_each_round = (unsigned long long)rounds * span > (unsigned long long)kWinCap;  // block-uniform
  if (tid == 0) s_nwin = 0;
  __syncthreads();
  for (uint32_t b0 = first; b0 < R; b0 += stride) {
    uint32_t r[kClaimILP], gpos[kClaimILP], lcount[kClaimILP];
    unsigned long long key[kClaimILP], h[kClaimILP];
    ulonglong2 sv[kClaimILP];
#pragma unroll
    for (int k = 0; k < kClaimILP; ++k) {
      r[k] = b0 + k * kThreadsC + tid;
      key[k] = kEmpty;
      if (r[k] < R) {
        const ulonglong2 rec = __ldcg(reinterpret_cast<const ulonglong2*>(p.rec) + r[k]);
        key[k] = rec.x;
        gpos[k] = (uint32_t)(rec.y & 0xFFFFFFFFull);
        lcount[k] = (uint32_t)(rec.y >> 32);
      }
    }
#pragma unroll
    for (int k = 0; k < kClaimILP; ++k)
      if (r[k] < R) {
        h[k] = stage2_home(key[k], p.ss);
        sv[k] = __ldcg(reinterpret_cast<const ulonglong2*>(&p.sc[h[k]]));
      }
#pragma unroll
    for (int k = 0; k < kClaimILP; ++k) {
      if (r[k] >= R) continue;
      uint32_t old_first;
      const bool won = claim_from(p, key[k], gpos[k], lcount[k], h[k], sv[k], &old_first);
      int32_t rb = 0;  // the key's first record: no positions before it
      if (won) {
        s_win[atomicAdd(&s_nwin, 1)] = (int32_t)h[k];
      } else {
        if (p.ranks != nullptr) {
          // {first, count - 1} of the slot are one 64-bit word: adding the count to its high half returns
          // both, the count being the rank base of this record's positions
          const unsigned long long old = atomicAdd(reinterpret_cast<unsigned long long*>(&p.sc[h[k]].first),
                                                   (unsigned long long)lcount[k] << 32);
          old_first = (uint32_t)(old & 0xFFFFFFFFull);
          rb = (int32_t)((uint32_t)(old >> 32) + 1u);  // positions of the key added before
        } else {
          atomicAdd(&p.sc[h[k]].cnt, lcount[k]);  // no ranks asked for: the count alone, no value returned
        }
        // lower the key's first position only when this record can (the first position only decreases)
        if (gpos[k] < old_first) atomicMin(&p.sc[h[k]].first, gpos[k]);
      }
      p.rec_sr[r[k]] = make_int2((int32_t)h[k], rb);  // one 8-byte store: the record's slot and rank base
    }
    if (list_each_round) list_winners(p, s_win, &s_nwin, &s_wbase);
  }
  if (!list_each_round) list_winners(p, s_win, &s_nwin, &s_wbase);
}


__global__ void __launch_bounds__(kThreadsR) k_resolve(const LookupParams p) {
  __shared__ int s_need, s_nnew, s_avail;
  __shared__ long long s_rowbase;

  const int tid = threadIdx.x;
  const uint32_t U = *p.ulist_n + 1u;  // the counter starts at 2^32 - 1
  const uint32_t step = (uint32_t)p.T.hdr->step;

  for (uint32_t b0 = blockIdx.x * kThreadsR; b0 < U; b0 += gridDim.x * kThreadsR) {  // block-uniform trip count
    const uint32_t idx = b0 + tid;
    const bool act = idx < U;
    if (tid == 0) {
      s_need = 0;
      s_nnew = 0;
    }
    __syncthreads();
    int32_t slot = 0, row = -1;
    unsigned long long key = 0, cs = 0;
    uint32_t gfirst = 0;
    bool claimed = false;
    if (act) {
      slot = __ldcg(&p.ulist[idx]);
      const ulonglong2 sv = __ldcg(reinterpret_cast<const ulonglong2*>(&p.sc[slot]));
      key = sv.x;
      gfirst = (uint32_t)(sv.y & 0xFFFFFFFFull);
      long long t_end = 0, t_tomb = -1;
      const long long sidx = p.no_table ? -1 : find_slot(p.T, key, &t_end, &t_tomb, &row);
      if (sidx < 0 && p.insert_missing && !p.no_table) {
        // absent, and no other thread inserts it (its key is listed once):
        // take the first tombstone of its chain, else the EMPTY slot that
        // ended the chain, else the next free slot after them
        long long t = t_tomb >= 0 ? t_tomb : t_end;
        unsigned long long s = (home_slot(p.T, key) + (unsigned long long)t * p.T.S) & p.T.mask;
        for (; t < (long long)p.T.max_probes; ++t) {
          const unsigned long long k = load_key_relaxed(&p.T.slots[s].key);
          if ((k == kEmpty || k == kTomb) && atomicCAS(&p.T.slots[s].key, k, key) == k) {
            claimed = true;
            cs = s;
            break;
          }
          s = (s + p.T.S) & p.T.mask;
        }
        if (!claimed) latch_error(p.T.hdr, MT_EFULL);
      }
    }
    const int q = claimed ? atomicAdd(&s_need, 1) : -1;
    __syncthreads();
    if (tid == 0 && s_need > 0) {  // one pop for the block: rows on the stack are free_stack[0 .. free_top)
      const long long k = s_need;
      const long long old = (long long)atomicAdd((unsigned long long*)&p.T.hdr->free_top, (unsigned long long)(-k));
      const long long avail = old < 0 ? 0 : (old < k ? old : k);
      if (avail < k) atomicAdd((unsigned long long*)&p.T.hdr->free_top, (unsigned long long)(k - avail));
      s_rowbase = old;
      s_avail = (int)avail;
    }
    __syncthreads();
    if (claimed) {
      if (q < s_avail) {
        row = p.T.free_stack[s_rowbase - 1 - q];
        p.T.slots[cs].row = row;
        p.T.slots[cs].meta = step;
      } else {
        atomicExch(&p.T.slots[cs].key, kTomb);  // give the slot back; the chain stays intact
        latch_error(p.T.hdr, MT_EFULL);
      }
    }
    if (act) {
      p.urow[idx] = row;  // beside the key's entry of the list: k_number reads both in order
      atomicAnd(&p.owner_nb[gfirst >> 6], ~(1ull << (gfirst & 63)));  // the key's first position
    }
    // the block's fresh rows join the list k_expand initialises (one global atomic per block)
    const bool fresh = claimed && q < s_avail;
    const int w = fresh ? atomicAdd(&s_nnew, 1) : -1;
    __syncthreads();
    if (tid == 0 && s_nnew > 0) s_rowbase = (long long)(atomicAdd(p.fresh_n, (uint32_t)s_nnew) + 1u);  // from 2^32-1
    __syncthreads();
    if (fresh) {
      p.fresh_row[s_rowbase + w] = row;
      p.fresh_key[s_rowbase + w] = key;
    }
    __syncthreads();
  }
}

// First positions per 64-position word and per tile, from the bits k_resolve
// cleared: one warp per tile (a lane per word); the last block to finish turns
// the tile counts into their exclusive prefix.
__global__ void __launch_bounds__(kThreads) k_prefix(const LookupParams p) {
  __shared__ int s_warp[kThreads / 32];
  __shared__ bool s_last;
  const int tid = threadIdx.x, lane = tid & 31;
  static_assert(kTile == 64 * 32, "a warp's lanes cover one tile's words");
  const int tile = blockIdx.x * (kThreads / 32) + (tid >> 5);
  if (tile < p.ntiles) {
    const int w = tile * 32 + lane;
    const int c = __popcll(~__ldcg(&p.owner_nb[w]));
    int x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    p.wpre[w] = (uint16_t)(x - c);
    if (lane == 31) p.tile_pre[tile] = x;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(p.done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  long long carry = 0;
  for (int c0 = 0; c0 < p.ntiles; c0 += kThreads * 4) {
    int v[4], sum = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int t = c0 + tid * 4 + k;
      v[k] = t < p.ntiles ? __ldcg(&p.tile_pre[t]) : 0;
      sum += v[k];
    }
    int tot;
    int run = (int)carry + block_exclusive_scan<kThreads>(sum, s_warp, &tot);  // its barriers order reads first
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int t = c0 + tid * 4 + k;
      if (t < p.ntiles) p.tile_pre[t] = run;
      run += v[k];
    }
    carry += tot;
  }
  if (tid == 0) {
    p.tile_pre[p.ntiles] = (int32_t)carry;
    *p.num_unique = (long long)carry;
  }
}

// One thread per distinct key (the claim-order list): the key's unique index
// is the number of first positions before its own (tile offset + word offset
// + the bits before it in its word), i.e. first-occurrence order.  It writes
// the key's unique entry and leaves the index and the table row in the
// scratch slot for k_expand.
__global__ void __launch_bounds__(kThreadsR) k_number(const LookupParams p) {
  constexpr int ILP = 2;  // keys per thread in flight: every load of both before any store
  const uint32_t U = *p.ulist_n + 1u;  // the counter starts at 2^32 - 1
  for (uint32_t i0 = blockIdx.x * kThreadsR * ILP + threadIdx.x; i0 < U; i0 += gridDim.x * kThreadsR * ILP) {
    int32_t slot[ILP], row[ILP];
    ulonglong2 sv[ILP];
#pragma unroll
    for (int k = 0; k < ILP; ++k) {
      const uint32_t idx = i0 + k * kThreadsR;
      slot[k] = idx < U ? __ldcg(&p.ulist[idx]) : -1;
      row[k] = idx < U ? __ldcg(&p.urow[idx]) : -1;
    }
#pragma unroll
    for (int k = 0; k < ILP; ++k)
      if (slot[k] >= 0) sv[k] = __ldcg(reinterpret_cast<const ulonglong2*>(&p.sc[slot[k]]));
    int u[ILP];
#pragma unroll
    for (int k = 0; k < ILP; ++k)
      if (slot[k] >= 0) {
        const uint32_t g = (uint32_t)(sv[k].y & 0xFFFFFFFFull);
        const unsigned long long below = ~__ldcg(&p.owner_nb[g >> 6]) & ((1ull << (g & 63)) - 1ull);
        u[k] = __ldcg(&p.tile_pre[g / kTile]) + (int)__ldcg(&p.wpre[g >> 6]) + __popcll(below);
      }
#pragma unroll
    for (int k = 0; k < ILP; ++k)
      if (slot[k] >= 0) {
        p.unique_keys[u[k]] = sv[k].x;
        p.unique_rows[u[k]] = row[k];
        p.counts[u[k]] = (int32_t)((uint32_t)(sv[k].y >> 32) + 1u);
        // from here on the slot's {first, count - 1} word holds {unique index, table row}: one load for k_expand
        *reinterpret_cast<unsigned long long*>(&p.sc[slot[k]].first) =
            (unsigned long long)(uint32_t)u[k] | ((unsigned long long)(uint32_t)row[k] << 32);
      }
  }
}

// inverse[i] = unique index of position i (-1 for an invalid ID); ranks[i] =
// the rank base of its tile's record + its rank inside the tile.
__global__ void __launch_bounds__(kThreads, 5) k_expand(const LookupParams p) {
  __shared__ int32_t s_u[kTile];   // unique index of each tile-local unique
  __shared__ int32_t s_rb[kTile];  // rank base of each tile-local unique
  __shared__ int32_t s_row[kTile];  // table row of each tile-local unique (when the lookup gathers)
  const int tile = blockIdx.x, tid = threadIdx.x;
  const long long base = (long long)tile * kTile;
  const int cnt = (int)min((long long)kTile, p.n - base);
  const int L = __ldg(&p.tile_L[tile]);
  const int r0 = __ldg(&p.tile_rec[tile]);
  int32_t sl[kPPT];
#pragma unroll
  for (int k = 0; k < kPPT; ++k) {
    const int l = k * kThreads + tid;
    const int2 sr = l < L ? __ldcg(&p.rec_sr[r0 + l]) : make_int2(-1, 0);
    sl[k] = sr.x;
    if (l < L) s_rb[l] = sr.y;
  }
  const bool gather = p.out_rows != nullptr;
#pragma unroll
  for (int k = 0; k < kPPT; ++k) {
    const int l = k * kThreads + tid;
    if (l < L) {
      const unsigned long long ur = __ldcg(reinterpret_cast<const unsigned long long*>(&p.sc[sl[k]].first));
      s_u[l] = (int32_t)(uint32_t)(ur & 0xFFFFFFFFull);
      s_row[l] = (int32_t)(uint32_t)(ur >> 32);
    }
  }
  __syncthreads();
  uint16_t li[kPPT], lr[kPPT];
#pragma unroll
  for (int k = 0; k < kPPT; ++k) {
    const int lp = k * kThreads + tid;
    const uint32_t w = lp < cnt ? __ldg(&p.llr[base + lp]) : (uint32_t)kNoIdx;
    li[k] = (uint16_t)(w & 0xFFFFu);
    lr[k] = (uint16_t)(w >> 16);
  }
#pragma unroll
  for (int k = 0; k < kPPT; ++k) {
    const int lp = k * kThreads + tid;
    if (lp < cnt) p.inverse[base + lp] = li[k] == kNoIdx ? -1 : s_u[li[k]];
  }
  if (gather) {  // the gather then reads each position's row directly
#pragma unroll
    for (int k = 0; k < kPPT; ++k) {
      const int lp = k * kThreads + tid;
      if (lp < cnt) p.prow[base + lp] = li[k] == kNoIdx ? -1 : s_row[li[k]];
    }
  }
  if (p.ranks != nullptr) {
#pragma unroll
    for (int k = 0; k < kPPT; ++k) {
      const int lp = k * kThreads + tid;
      if (lp < cnt) p.ranks[base + lp] = li[k] == kNoIdx ? -1 : s_rb[li[k]] + (int32_t)lr[k];
    }
  }
  // this block's share of the fresh rows: init(key), m = v = 0, one team of lanes per row (8 columns
  // per lane and Philox block).  The arithmetic fills the issue slots this latency-bound kernel leaves.
  const long long F = (long long)(uint32_t)(*p.fresh_n + 1u);  // the counter starts at 2^32 - 1
  const long long per = (F + gridDim.x - 1) / gridDim.x;
  const long long f0 = (long long)tile * per, f1 = min(f0 + per, F);
  const int oct = (int)((p.T.dim + 7) / 8);
  int team = 1;
  while (team < 32 && team < oct) team <<= 1;
  const int nteams = kThreads / team;
  for (long long f = f0 + tid / team; f < f1; f += nteams)
    init_row_coop(p.T, __ldcg(&p.fresh_row[f]), __ldcg(&p.fresh_key[f]), tid % team, team);
}

// out[i] = row prow[i] of position i (zeros for an invalid ID or an absent
// key): 16-byte items (position, vector), consecutive threads on consecutive
// items; each round a block covers kGatherILP * blockDim contiguous items
// (kGatherILP independent items in flight per thread), and the blocks stride
// over the whole batch so every SM stays busy to the end.
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
        row[k] = __ldg(&p.prow[i]);
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
  // every distinct key needs a slot and every probe chain an EMPTY end: more
  // slots than IDs; a quarter more keeps chains short even if all IDs differ
  L.ss = align_up((size_t)n + (size_t)n / 4 + 1024, 1024);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.sc = take(L.ss * sizeof(ScSlot));
  const size_t cap = (size_t)L.ntiles * kTile;
  L.ulist_n = off;  // right after the slots (with the fresh-row and record counters), then the first-position
  off += 16;        // bits: one memset clears them all
  L.owner_nb = off;
  L.clear_bytes = off + cap / 8;
  take(cap / 8);
  L.ulist = take((size_t)(n > 0 ? n : 1) * 4);
  L.rec = take((size_t)(n > 0 ? n : 1) * 16);
  L.rec_sr = take((size_t)(n > 0 ? n : 1) * 8);
  L.fresh_row = take((size_t)(n > 0 ? n : 1) * 4);
  L.fresh_key = take((size_t)(n > 0 ? n : 1) * 8);
  L.urow = take((size_t)(n > 0 ? n : 1) * 4);
  L.tile_L = take((size_t)L.ntiles * 4);
  L.tile_pre = take((size_t)(L.ntiles + 1) * 4);
  L.done = take(16);
  L.wpre = take(cap / 64 * 2);
  L.prow = take(cap * 4);
  L.tile_rec = take((size_t)L.ntiles * 4);
  L.llr = take(cap * 4);
  L.total = off;
  return L;
}

void bind_lookup_ws(LookupParams& p, char* w, const LookupWsLayout& L) {
  p.sc = reinterpret_cast<ScSlot*>(w + L.sc);
  p.ss = L.ss;
  p.ulist_n = reinterpret_cast<uint32_t*>(w + L.ulist_n);
  p.fresh_n = p.ulist_n + 1;
  p.rec_n = p.ulist_n + 2;
  p.rec = reinterpret_cast<ulonglong2*>(w + L.rec);
  p.rec_sr = reinterpret_cast<int2*>(w + L.rec_sr);
  p.tile_rec = reinterpret_cast<int32_t*>(w + L.tile_rec);
  p.fresh_row = reinterpret_cast<int32_t*>(w + L.fresh_row);
  p.fresh_key = reinterpret_cast<unsigned long long*>(w + L.fresh_key);
  p.ulist = reinterpret_cast<int32_t*>(w + L.ulist);
  p.urow = reinterpret_cast<int32_t*>(w + L.urow);
  p.tile_L = reinterpret_cast<int32_t*>(w + L.tile_L);
  p.owner_nb = reinterpret_cast<unsigned long long*>(w + L.owner_nb);
  p.wpre = reinterpret_cast<uint16_t*>(w + L.wpre);
  p.prow = reinterpret_cast<int32_t*>(w + L.prow);
  p.tile_pre = reinterpret_cast<int32_t*>(w + L.tile_pre);
  p.done = reinterpret_cast<uint32_t*>(w + L.done);
  p.llr = reinterpret_cast<uint32_t*>(w + L.llr);
  p.ntiles = L.ntiles;
  p.clear_bytes = L.clear_bytes;
}

cudaError_t launch_lookup(const LookupParams& p_in, cudaStream_t s) {
  if (p_in.n == 0) return cudaMemsetAsync(p_in.num_unique, 0, sizeof(long long), s);
  static std::atomic<int> gather_grid[kMaxDevices];   // 0: not set up on that device yet
  static std::atomic<int> resolve_slots[kMaxDevices];
  static std::atomic<int> claim_slots[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  if (gather_grid[dev].load(std::memory_order_relaxed) == 0) {
    cudaError_t e = cudaFuncSetAttribute(k_local, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemA);
    if (e != cudaSuccess) return e;
    int sms = 0, per = 0, rper = 0, cper = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, k_gather, 256, 0);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&rper, k_resolve, kThreadsR, 0);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&cper, k_claim, kThreadsC, 0);
    resolve_slots[dev].store(sms * (rper > 0 ? rper : 1), std::memory_order_relaxed);
    claim_slots[dev].store(sms * (cper > 0 ? cper : 1), std::memory_order_relaxed);
    gather_grid[dev].store(sms * (per > 0 ? per : 1), std::memory_order_relaxed);
  }
  LookupParams p = p_in;
  {
    const long long want = (p.n + kThreadsR - 1) / kThreadsR;  // blocks if every ID were distinct
    const int slots = resolve_slots[dev].load(std::memory_order_relaxed);
    p.resolve_grid = (int)(want < slots ? want : slots);
  }
  const long long cwant = (p.n + kThreadsC * kClaimILP - 1) / (kThreadsC * kClaimILP);
  const int cslots = claim_slots[dev].load(std::memory_order_relaxed);
  const int claim_grid = (int)(cwant < cslots ? cwant : cslots);
  // scratch slots (key EMPTY, first "none", count - 1 = 2^32 - 1), the list counters (minus one) and the
  // first-position bits (none set): all ones
  cudaError_t e = cudaMemsetAsync(p.sc, 0xFF, p.clear_bytes, s);
  if (e != cudaSuccess) return e;
  {
    MT_LAUNCH("k_local", s);
    k_local<<<p.ntiles, kThreadsA, kSmemA, s>>>(p);
  }
  {
    MT_LAUNCH("k_claim", s);
    k_claim<<<claim_grid, kThreadsC, 0, s>>>(p);
  }
  {
    MT_LAUNCH("k_resolve", s);
    k_resolve<<<p.resolve_grid, kThreadsR, 0, s>>>(p);
  }
  {
    MT_LAUNCH("k_prefix", s);
    k_prefix<<<(p.ntiles + kThreads / 32 - 1) / (kThreads / 32), kThreads, 0, s>>>(p);
  }
  {
    MT_LAUNCH("k_number", s);
    k_number<<<p.resolve_grid, kThreadsR, 0, s>>>(p);
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
