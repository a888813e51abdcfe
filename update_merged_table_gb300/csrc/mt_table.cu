// Table maintenance kernels: arena initialisation, key deletion with
// tombstones, the occupancy scan, live-key export and row read-back.
//
// Pages: "MTGenRec" abstract (dynamic hash tables whose keys are inserted and deleted while training runs, in
// hash tables) and Theorem 1 (probe sequence h_t = (h0 + t*S) mod 2^n, S odd);
// "MTGR" section 5, Embedding Management (exporting keys by scanning the key store).
#include "mt_kernels.cuh"

namespace mt {

namespace {

__global__ void k_table_init(const TableDev T) {
  const long long R = T.num_rows;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < R; i += (long long)gridDim.x * blockDim.x)
    T.free_stack[i] = (int32_t)(R - 1 - i);  // pops hand out rows 0, 1, 2, ...
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    T.hdr->error = 0;
    T.hdr->free_top = R;
    T.hdr->step = 0;
    T.hdr->b1pow = 1.0;
    T.hdr->b2pow = 1.0;
  }
}

// Pass 1 of an erase: every key is looked up while the store is unchanged,
// so duplicates in the batch all see a live key.
__global__ void k_erase_find(const TableDev T, const unsigned long long* keys, long long n, int32_t* ws_slot) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const unsigned long long key = keys[i];
    long long s = -1;
    if (key != kEmpty && key != kTomb) {
      long long t_end, t_tomb;
      int32_t row;
      s = find_slot(T, key, &t_end, &t_tomb, &row);
    }
    ws_slot[i] = (int32_t)s;
  }
}

// Pass 2: one CAS per found key turns its slot into a tombstone; the winner
// returns the row to the free stack (warp-aggregated push).
__global__ void k_erase_apply(const TableDev T, const unsigned long long* keys, long long n, const int32_t* ws_slot,
                              unsigned char* found) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long n_round = (n + 31) / 32 * 32;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_round; i += stride) {
    const bool in = i < n;
    const int32_t s = in ? ws_slot[i] : -1;
    bool won = false;
    int32_t row = -1;
    if (s >= 0) {
      const unsigned long long key = keys[i];
      row = T.slots[s].row;
      won = atomicCAS(&T.slots[s].key, key, kTomb) == key;
    }
    if (in && found != nullptr) found[i] = s >= 0 ? 1 : 0;
    const unsigned mask = __ballot_sync(kFull, won);
    if (won) push_row_warp(T, mask, row);
  }
}

// Every live key of src's slots, with its row and meta, inserted into `slots`
// (all EMPTY) along its probe sequence in table `dst`: one old slot per
// thread and loop trip, many threads (one CAS each in flight beats several
// per thread here, measured).  Keys are distinct, so a CAS only ever loses to
// another key.  A key that finds no EMPTY slot within dst's probe limit sets
// dst's header flag (and latches MT_EFULL when latch_full).
__device__ __forceinline__ void reinsert_live(const TableDev& src, const TableDev& dst, Slot* slots, bool latch_full) {
  const unsigned long long M = src.mask + 1;
  for (unsigned long long s = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; s < M;
       s += (unsigned long long)gridDim.x * blockDim.x) {
    const Slot old = src.slots[s];
    if (old.key == kEmpty || old.key == kTomb) continue;
    unsigned long long h = home_slot(dst, old.key);
    bool placed = false;
    for (uint32_t t = 0; t < dst.max_probes; ++t) {
      if (atomicCAS(&slots[h].key, kEmpty, old.key) == kEmpty) {
        slots[h].row = old.row;
        slots[h].meta = old.meta;
        placed = true;
        break;
      }
      h = (h + dst.S) & dst.mask;
    }
    if (!placed) {
      atomicExch(&dst.hdr->pad0, 1);
      if (latch_full) latch_error(dst.hdr, MT_EFULL);
    }
  }
}

// Compaction: every live key of the table inserted again into the fresh slot
// array `fresh` along the same probe sequence (a key that does not fit makes
// the call keep the old slots and latch MT_EFULL).
__global__ void __launch_bounds__(256) k_compact_rebuild(const TableDev T, Slot* fresh) {
  reinsert_live(T, T, fresh, true);
}

// Import pass 1: find each key, or insert it like a lookup does (first
// tombstone-or-EMPTY slot of its chain; warp-aggregated row pops); its row
// goes to rows_out[i] (-1 when it could not be placed).
__global__ void k_import_resolve(const TableDev T, const unsigned long long* keys, long long n, int32_t* rows_out) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long n_round = (n + 31) / 32 * 32;
  const uint32_t step = (uint32_t)T.hdr->step;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_round; i += stride) {
    const bool in = i < n;
    const unsigned long long key = in ? keys[i] : kEmpty;
    int32_t row = -1;
    bool claimed = false;
    unsigned long long cs = 0;
    if (in && (key >> 56) == 0xFFull) latch_error(T.hdr, MT_EKEY);  // table id 255 holds the sentinels
    if (in && (key >> 56) != 0xFFull) {
      long long t_end, t_tomb;
      const long long sidx = find_slot(T, key, &t_end, &t_tomb, &row);
      if (sidx < 0) {
        long long t = t_tomb >= 0 ? t_tomb : t_end;
        unsigned long long slot = (home_slot(T, key) + (unsigned long long)t * T.S) & T.mask;
        for (; t < (long long)T.max_probes; ++t) {
          const unsigned long long k = load_key_relaxed(&T.slots[slot].key);
          if ((k == kEmpty || k == kTomb) && atomicCAS(&T.slots[slot].key, k, key) == k) {
            claimed = true;
            cs = slot;
            break;
          }
          slot = (slot + T.S) & T.mask;
        }
        if (!claimed) latch_error(T.hdr, MT_EFULL);
      }
    }
    const unsigned need = __ballot_sync(kFull, claimed);
    if (claimed) {
      row = pop_row_warp(T, need);
      if (row < 0) {
        atomicExch(&T.slots[cs].key, kTomb);  // give the slot back; the chain stays intact
        latch_error(T.hdr, MT_EFULL);
      } else {
        T.slots[cs].row = row;
        T.slots[cs].meta = step;
      }
    }
    if (in) rows_out[i] = row;
  }
}

// Import pass 2: the given embedding and moments into each placed row.
__global__ void k_import_write(const TableDev T, const int32_t* rows, long long n, const float* emb, const float* m,
                               const float* v) {
  const long long d = T.dim;
  const long long total = n * d;
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const long long i = it / d, j = it - i * d;
    const int32_t r = rows[i];
    if (r < 0 || r >= T.num_rows) continue;
    char* rec = row_ptr(T, r);
    if (T.row_dtype == MT_F32) reinterpret_cast<float*>(rec)[j] = emb[it];
    else reinterpret_cast<__nv_bfloat16*>(rec)[j] = __float2bfloat16_rn(emb[it]);
    reinterpret_cast<float*>(rec + T.emb_bytes)[j] = m[it];
    reinterpret_cast<float*>(rec + T.emb_bytes + T.mv_bytes)[j] = v[it];
  }
}

// Capacity expansion, pass 1: the new rows (old R .. new R - 1, the new row
// segment) join the free list above the old free entries, and the free count
// grows with them.
__global__ void k_grow_rows(const TableDev T2, long long old_rows) {
  const long long added = T2.num_rows - old_rows;
  const long long top = T2.hdr->free_top;  // copied from the old header
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < added;
       i += (long long)gridDim.x * blockDim.x)
    T2.free_stack[top + i] = (int32_t)(old_rows + i);
}
__global__ void k_grow_top(const TableDev T2, long long old_rows) {
  T2.hdr->free_top += T2.num_rows - old_rows;
  T2.hdr->pad0 = 0;  // the rebuild's "a key did not fit" flag
}

// Capacity expansion, pass 2: every live key of the old slots is inserted
// into the new (all EMPTY) slots along its probe sequence in the new table.
__global__ void __launch_bounds__(256) k_grow_rebuild(const TableDev T, const TableDev T2) {
  reinsert_live(T, T2, T2.slots, false);
}

// One pass over the slots: live keys, tombstones, total displacement and the
// probe-index histogram.  Nearly every key of a healthy table sits at a small
// probe index, so the first kStatRegBins indices are counted in registers and
// summed per warp (shared-memory atomics on one bin would serialise); longer
// chains go to shared memory.  Four streaming slot loads per thread in flight.
constexpr int kStatRegBins = 8;
constexpr int kStatUnroll = 4;
__global__ void __launch_bounds__(256) k_stats(const TableDev T) {
  __shared__ unsigned long long s_hist[MT_HIST_BINS];
  __shared__ unsigned long long s_live, s_tomb, s_disp;
  for (int i = threadIdx.x; i < MT_HIST_BINS; i += blockDim.x) s_hist[i] = 0;
  if (threadIdx.x == 0) s_live = s_tomb = s_disp = 0;
  __syncthreads();
  unsigned long long live = 0, tomb = 0, disp = 0;
  uint32_t c[kStatRegBins];
#pragma unroll
  for (int j = 0; j < kStatRegBins; ++j) c[j] = 0;
  const unsigned long long M = T.mask + 1;
  const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
  for (unsigned long long s0 = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; s0 < M;
       s0 += stride * kStatUnroll) {
    unsigned long long key[kStatUnroll];
#pragma unroll
    for (int k = 0; k < kStatUnroll; ++k) {
      const unsigned long long s = s0 + k * stride;
      key[k] = s < M ? __ldcs(&T.slots[s].key) : kEmpty;
    }
#pragma unroll
    for (int k = 0; k < kStatUnroll; ++k) {
      if (key[k] == kTomb) {
        ++tomb;
      } else if (key[k] != kEmpty) {
        ++live;
        // slot = h0 + t*S (mod M)  =>  t = (slot - h0) * S^-1 (mod M)
        const unsigned long long s = s0 + k * stride;
        const unsigned long long t = ((s - home_slot(T, key[k])) & T.mask) * T.Sinv & T.mask;
        disp += t;
#pragma unroll
        for (int j = 0; j < kStatRegBins; ++j) c[j] += t == (unsigned long long)j;
        if (t >= (unsigned long long)kStatRegBins) atomicAdd(&s_hist[t < MT_HIST_BINS - 1 ? t : MT_HIST_BINS - 1], 1ull);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kStatRegBins; ++j) {
    const unsigned w = __reduce_add_sync(kFull, c[j]);
    if ((threadIdx.x & 31) == 0 && w) atomicAdd(&s_hist[j], (unsigned long long)w);
  }
  atomicAdd(&s_live, live);
  atomicAdd(&s_tomb, tomb);
  atomicAdd(&s_disp, disp);
  __syncthreads();
  for (int i = threadIdx.x; i < MT_HIST_BINS; i += blockDim.x)
    if (s_hist[i]) atomicAdd(&T.hdr->hist[i], s_hist[i]);
  if (threadIdx.x == 0) {
    atomicAdd(&T.hdr->live, s_live);
    atomicAdd(&T.hdr->tombs, s_tomb);
    atomicAdd(&T.hdr->disp, s_disp);
  }
}

__global__ void k_export(const TableDev T, unsigned long long* keys, int32_t* rows, long long capacity) {
  const unsigned long long M = T.mask + 1;
  const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
  const unsigned long long M_round = (M + 31) / 32 * 32;
  const int lane = threadIdx.x & 31;
  for (unsigned long long s = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; s < M_round; s += stride) {
    bool live = false;
    unsigned long long key = 0;
    int32_t row = -1;
    if (s < M) {
      key = T.slots[s].key;
      live = key != kEmpty && key != kTomb;
      if (live) row = T.slots[s].row;
    }
    const unsigned mask = __ballot_sync(kFull, live);
    if (mask == 0) continue;
    const int leader = __ffs(mask) - 1;
    long long base = 0;
    if (lane == leader) base = (long long)atomicAdd((unsigned long long*)&T.hdr->export_count, (unsigned long long)__popc(mask));
    base = __shfl_sync(kFull, base, leader);
    if (live) {
      const long long idx = base + __popc(mask & ((1u << lane) - 1u));
      if (idx < capacity) {
        keys[idx] = key;
        rows[idx] = row;
      }
    }
  }
}

__global__ void k_read_rows(const TableDev T, const int32_t* rows, long long n, float* emb, float* m, float* v) {
  const long long d = T.dim;
  const long long total = n * d;
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const long long i = it / d, j = it - i * d;
    const int32_t r = rows[i];
    float e = 0.f, a = 0.f, b = 0.f;
    if (r >= 0 && r < T.num_rows) {
      const char* rec = row_ptr(T, r);
      e = T.row_dtype == MT_F32 ? reinterpret_cast<const float*>(rec)[j]
                                : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(rec)[j]);
      a = reinterpret_cast<const float*>(rec + T.emb_bytes)[j];
      b = reinterpret_cast<const float*>(rec + T.emb_bytes + T.mv_bytes)[j];
    }
    if (emb) emb[it] = e;
    if (m) m[it] = a;
    if (v) v[it] = b;
  }
}

}  // namespace

cudaError_t launch_table_init(const TableDev& T, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(T.hdr, 0, kHeaderBytes, s);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(T.slots, 0xFF, (size_t)(T.mask + 1) * sizeof(Slot), s);
  if (e != cudaSuccess) return e;
  {
    MT_LAUNCH("k_table_init", s);
    k_table_init<<<grid_for(T.num_rows, 256, 32), 256, 0, s>>>(T);
  }
  return cudaGetLastError();
}

cudaError_t launch_erase(const TableDev& T, const unsigned long long* keys, long long n, unsigned char* found,
                         int32_t* ws_slot, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  {
    MT_LAUNCH("k_erase_find", s);
    k_erase_find<<<grid_for(n, 256, 32), 256, 0, s>>>(T, keys, n, ws_slot);
  }
  {
    MT_LAUNCH("k_erase_apply", s);
    k_erase_apply<<<grid_for(n, 256, 32), 256, 0, s>>>(T, keys, n, ws_slot, found);
  }
  return cudaGetLastError();
}

cudaError_t launch_compact(const TableDev& T, Slot* fresh, cudaStream_t s) {
  const unsigned long long M = T.mask + 1;
  cudaError_t e = cudaMemsetAsync(fresh, 0xFF, M * sizeof(Slot), s);  // keys EMPTY
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(&T.hdr->pad0, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return e;
  {
    MT_LAUNCH("k_compact_rebuild", s);
    k_compact_rebuild<<<grid_for((long long)M, 256, 32), 256, 0, s>>>(T, fresh);
  }
  return cudaGetLastError();
}

cudaError_t launch_stats(const TableDev& T, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(&T.hdr->live, 0, sizeof(unsigned long long) * (3 + MT_HIST_BINS), s);
  if (e != cudaSuccess) return e;
  {
    MT_LAUNCH("k_stats", s);
    k_stats<<<grid_for((long long)(T.mask + 1) / kStatUnroll, 256, 4), 256, 0, s>>>(T);  // all resident
  }
  return cudaGetLastError();
}

cudaError_t launch_export(const TableDev& T, unsigned long long* keys, int32_t* rows, long long capacity,
                          cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(&T.hdr->export_count, 0, sizeof(long long), s);
  if (e != cudaSuccess) return e;
  {
    MT_LAUNCH("k_export", s);
    k_export<<<grid_for((long long)(T.mask + 1), 256, 32), 256, 0, s>>>(T, keys, rows, capacity);
  }
  return cudaGetLastError();
}

cudaError_t launch_import(const TableDev& T, const unsigned long long* keys, long long n, const float* emb,
                          const float* m, const float* v, int32_t* ws_rows, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  {
    MT_LAUNCH("k_import_resolve", s);
    k_import_resolve<<<grid_for(n, 256, 32), 256, 0, s>>>(T, keys, n, ws_rows);
  }
  {
    MT_LAUNCH("k_import_write", s);
    k_import_write<<<grid_for(n * T.dim, 256, 32), 256, 0, s>>>(T, ws_rows, n, emb, m, v);
  }
  return cudaGetLastError();
}

// The new key store of T2: header and the old free list copied, slots
// cleared, the new row segment's rows pushed, every live key re-inserted.
// No row record is read or written.
cudaError_t launch_grow(const TableDev& T, const TableDev& T2, cudaStream_t s) {
  cudaError_t e = cudaMemcpyAsync(T2.hdr, T.hdr, kHeaderBytes, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(T2.free_stack, T.free_stack, (size_t)T.num_rows * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(T2.slots, 0xFF, (size_t)(T2.mask + 1) * sizeof(Slot), s);  // keys EMPTY
  if (e != cudaSuccess) return e;
  if (T2.num_rows > T.num_rows) {
    MT_LAUNCH("k_grow_rows", s);
    k_grow_rows<<<grid_for(T2.num_rows - T.num_rows, 256, 32), 256, 0, s>>>(T2, T.num_rows);
  }
  {
    MT_LAUNCH("k_grow_top", s);
    k_grow_top<<<1, 1, 0, s>>>(T2, T.num_rows);
  }
  {
    MT_LAUNCH("k_grow_rebuild", s);
    k_grow_rebuild<<<grid_for((long long)(T.mask + 1), 256, 32), 256, 0, s>>>(T, T2);
  }
  return cudaGetLastError();
}

cudaError_t launch_read_rows(const TableDev& T, const int32_t* rows, long long n, float* emb, float* m, float* v,
                             cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  {
    MT_LAUNCH("k_read_rows", s);
    k_read_rows<<<grid_for(n * T.dim, 256, 32), 256, 0, s>>>(T, rows, n, emb, m, v);
  }
  return cudaGetLastError();
}

}  // namespace mt
