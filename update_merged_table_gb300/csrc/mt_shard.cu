// Sharded two-stage deduplication around an exchange, with G logical shards
// on one GPU.
//
// Pages: "MTGenRec" TL;DR (deduplication of IDs in two stages to speed up
// embedding lookups) and "MTGR" section 5, Embedding Lookup (deduplication
// cuts duplicate transfers in the cross-device all-to-all; no duplicate IDs on
// either side of the exchange).  The Meituan TensorFlow article (section 3.6)
// merges Unique with DynamicPartition: the same unique-then-partition shape.
//
// Each logical rank r holds one shard table (the keys whose owner is r) and
// its own batch.  Forward:
//   1. stage 1: rank r deduplicates its batch (first-occurrence unique,
//      inverse, counts, ranks; no table access);
//   2. partition: owner(key) = a second hash of the key, mapped to [0, G);
//      the count of each (rank, owner) pair is exchanged first (read on the
//      host, as the sizes of a variable all-to-all are), then every rank
//      writes its unique keys into the owners' receive buffers (the
//      all-to-all, here a device-local copy) and remembers where each went;
//   3. stage 2: each owner deduplicates what it received (keys that several
//      ranks sent meet here), finds or inserts them in its shard table and
//      gathers one row per received key;
//   4. the rows go back to the ranks (the reverse all-to-all) and each rank
//      expands them to its positions through its inverse.
// Backward: every rank sums its positions' gradients per unique key, sends
// the sums to the owners, and each owner sums what it received per key and
// applies one Adam step to its shard.
#include <cstring>
#include <new>
#include <vector>

#include "mt_kernels.cuh"

struct mt_table;  // defined in mt_api.cu
namespace mt {
const TableDev& table_dev(const mt_table* t);
mt_config table_cfg(const mt_table* t);
void table_count_step(mt_table* t);
int heavy_warp_chunk(long long n, int team_shift);
}  // namespace mt

struct mt_shard_group {
  int G;
  mt_table* shards[MT_MAX_SHARDS];
  // layout of the last lookup, kept for its backward
  bool have_lookup;
  long long n[MT_MAX_SHARDS];          // batch size of each rank
  long long U[MT_MAX_SHARDS];          // unique keys of each rank
  long long N[MT_MAX_SHARDS];          // keys each owner received
  long long recv_base[MT_MAX_SHARDS];  // where owner o's received keys start in the receive space
  long long rank_base[MT_MAX_SHARDS];  // where rank r's per-unique arrays start (prefix of n)
  long long ntot;
  size_t ws_bytes;
};

namespace mt {

namespace {

// Owner of a key: the high 32 bits of a second mix of the key, scaled to [0, G).
__device__ __forceinline__ int owner_of(unsigned long long key, int G) {
  const unsigned hi = (unsigned)(mix64(key ^ 0xD6E8FEB86659FD93ull) >> 32);
  return (int)(((unsigned long long)hi * (unsigned)G) >> 32);
}

struct ShardOffsets {
  long long off[MT_MAX_SHARDS * MT_MAX_SHARDS];  // off[o * G + r]: where rank r's keys for owner o start
};

// counts[r * G + o] += keys of rank r owned by o: per warp and owner one
// ballot, and one atomic by the first lane that holds a key of that owner.
__global__ void __launch_bounds__(256) k_shard_count(const unsigned long long* keys, long long U, int G, int r,
                                                     int32_t* counts) {
  const int lane = threadIdx.x & 31;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long u0 = (long long)blockIdx.x * blockDim.x; u0 < U; u0 += stride) {  // warp-uniform
    const long long u = u0 + threadIdx.x;
    const int o = u < U ? owner_of(keys[u], G) : -1;
    for (int q = 0; q < G; ++q) {
      const unsigned m = __ballot_sync(kFull, o == q);
      if (m != 0 && lane == __ffs(m) - 1) atomicAdd(&counts[r * G + q], __popc(m));
    }
  }
}

// The exchange of keys: rank r writes each unique key into its owner's
// receive buffer (order within a (rank, owner) segment unspecified) and
// records where it went; the lanes of a warp with the same owner take
// consecutive places with one atomic.
__global__ void __launch_bounds__(256) k_shard_send(const unsigned long long* keys, long long U, int G, int r,
                                                    const ShardOffsets off, int32_t* cursor,
                                                    unsigned long long* recv_keys, long long recv_cap, int32_t* perm,
                                                    Header* hdr) {
  const int lane = threadIdx.x & 31;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long u0 = (long long)blockIdx.x * blockDim.x; u0 < U; u0 += stride) {  // warp-uniform
    const long long u = u0 + threadIdx.x;
    const unsigned long long key = u < U ? keys[u] : 0ull;
    const int o = u < U ? owner_of(key, G) : -1;
    long long slot = -1;
    for (int q = 0; q < G; ++q) {
      const unsigned m = __ballot_sync(kFull, o == q);
      if (m == 0) continue;
      const int leader = __ffs(m) - 1;
      int base = 0;
      if (lane == leader) base = atomicAdd(&cursor[r * G + q], __popc(m));
      base = __shfl_sync(kFull, base, leader);
      if (o == q) slot = off.off[q * G + r] + base + __popc(m & ((1u << lane) - 1u));
    }
    if (slot >= recv_cap) {  // counts that disagree with the keys: reported, never written out of range
      latch_error(hdr, MT_EINVAL);
      slot = -1;
    }
    if (u < U) perm[u] = (int32_t)slot;
    if (slot >= 0) recv_keys[slot] = key;
  }
}

// dst[i] = src[idx[i]] for rows of `vec16` 16-byte vectors (idx -1 or absent: zeros).
__global__ void __launch_bounds__(256) k_shard_gather(const uint4* src, long long src_rows, const int32_t* idx,
                                                      long long n, int vec16, uint4* dst) {
  const long long total = n * vec16;
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const long long i = it / vec16;
    const int v = (int)(it - i * vec16);
    const int32_t j = __ldg(&idx[i]);
    dst[it] = (j >= 0 && j < src_rows) ? __ldg(&src[(size_t)j * vec16 + v]) : make_uint4(0u, 0u, 0u, 0u);
  }
}

// dst[idx[i]] = src[i] for rows of `vec16` 16-byte vectors.
__global__ void __launch_bounds__(256) k_shard_scatter(const uint4* src, const int32_t* idx, long long n, int vec16,
                                                       uint4* dst, long long dst_rows) {
  const long long total = n * vec16;
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const long long i = it / vec16;
    const int v = (int)(it - i * vec16);
    const int32_t j = __ldg(&idx[i]);
    if (j >= 0 && j < dst_rows) dst[(size_t)j * vec16 + v] = __ldg(&src[it]);
  }
}

// For the per-rank gradient sums: where each of rank r's unique keys lands
// among its owner's unique keys, as an index into the owners' concatenated
// per-unique sums.
__global__ void __launch_bounds__(256) k_shard_owner_unique(const unsigned long long* keys, const int32_t* perm,
                                                            long long U, int G, const ShardOffsets base,
                                                            const int32_t* inv2, long long cap, int32_t* out) {
  for (long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x; u < U; u += (long long)gridDim.x * blockDim.x) {
    const int o = owner_of(keys[u], G);
    const int32_t slot = perm[u];
    out[u] = (slot >= 0 && slot < cap) ? (int32_t)(base.off[o] + __ldg(&inv2[slot])) : -1;
  }
}

struct ShardLayout {
  size_t perm, counts, cursor, recv_keys, uk2, inv2, cnt2, rows2, rank2, nu2, recv_rows, uniq_rows, gsum, recv_g,
      gsum2, idx, scratch, total;
};

// The scratch holds one lookup (or backward) workspace per rank, or per owner,
// side by side: their batches add up to at most ntot IDs, and splitting a
// batch costs at most one tile's workspace per part (a tile's rounding, the
// scratch hash's rounding, the arrays' alignment).
ShardLayout shard_layout(int G, long long ntot, long long nmax, uint32_t dim, uint32_t rec_emb_bytes) {
  ShardLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const size_t nt = (size_t)(ntot > 0 ? ntot : 1);
  L.perm = take(nt * 4);
  L.counts = take(MT_MAX_SHARDS * MT_MAX_SHARDS * 4);
  L.cursor = take(MT_MAX_SHARDS * MT_MAX_SHARDS * 4);
  L.recv_keys = take(nt * 8);
  L.uk2 = take(nt * 8);
  L.inv2 = take(nt * 4);
  L.cnt2 = take(nt * 4);
  L.rows2 = take(nt * 4);
  L.rank2 = take(nt * 4);
  L.nu2 = take(MT_MAX_SHARDS * 8);
  L.recv_rows = take(nt * rec_emb_bytes);
  L.uniq_rows = take(nt * rec_emb_bytes);
  L.gsum = take(nt * dim * 4);
  L.recv_g = take(nt * dim * 4);
  L.gsum2 = take(nt * dim * 4);
  L.idx = take(nt * 4);
  const long long big = ntot > nmax ? ntot : nmax;
  const size_t lw = lookup_ws_layout(big).total, bw = backward_ws_layout(big, dim).total;
  const size_t lt = lookup_ws_layout(kTile).total, bt = backward_ws_layout(kTile, dim).total;
  L.scratch = take(align_up(lw > bw ? lw : bw, 256) + (size_t)G * align_up(lt > bt ? lt : bt, 256));
  L.total = off;
  return L;
}

int grid_of(long long work) { return grid_for(work, 256, 16); }

}  // namespace

}  // namespace mt

namespace {

using mt::align_up;

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Batch sizes of the ranks and their prefix sums; false when one is out of range.
bool batch_sizes(const mt_shard_group* g, const int64_t* n, long long* base, long long* ntot, long long* nmax) {
  long long t = 0, m = 0;
  for (int r = 0; r < g->G; ++r) {
    if (n[r] < 0 || n[r] > 0x7FFFFFFF) return false;
    base[r] = t;
    t += n[r];
    m = n[r] > m ? n[r] : m;
  }
  if (t > 0x7FFFFFFF) return false;
  *ntot = t;
  *nmax = m;
  return true;
}

// Lookup parameters for one batch against one shard, over the shared scratch.
mt::LookupParams lookup_params(const mt::TableDev& T, const long long* ids, long long n, void* ws) {
  mt::LookupParams p;
  std::memset(&p, 0, sizeof(p));
  p.T = T;
  p.ids = ids;
  p.n = n;
  const mt::LookupWsLayout L = mt::lookup_ws_layout(n);
  char* w = static_cast<char*>(ws);
  if (n > 0) mt::bind_lookup_ws(p, w, L);
  return p;
}

}  // namespace

extern "C" {

int mt_shard_group_create(mt_table* const* shards, int G, mt_shard_group** out) {
  if (out == nullptr) return MT_EINVAL;
  *out = nullptr;
  if (shards == nullptr || G < 1 || G > MT_MAX_SHARDS) return MT_EINVAL;
  for (int r = 0; r < G; ++r) {
    if (shards[r] == nullptr) return MT_EINVAL;
    for (int q = 0; q < r; ++q)
      if (shards[q] == shards[r]) return MT_EINVAL;
    const mt_config a = mt::table_cfg(shards[0]), b = mt::table_cfg(shards[r]);
    if (a.dim != b.dim || a.row_dtype != b.row_dtype || a.init_seed != b.init_seed || a.init_scale != b.init_scale)
      return MT_EINVAL;  // a key's row must not depend on which shard owns it
  }
  mt_shard_group* g = new (std::nothrow) mt_shard_group();
  if (g == nullptr) return MT_ECUDA;
  g->G = G;
  for (int r = 0; r < G; ++r) g->shards[r] = shards[r];
  g->have_lookup = false;
  *out = g;
  return MT_OK;
}

int mt_shard_group_destroy(mt_shard_group* g) {
  if (g == nullptr) return MT_EINVAL;
  delete g;
  return MT_OK;
}

size_t mt_shard_workspace_bytes(const mt_shard_group* g, const int64_t* n) {
  if (g == nullptr || n == nullptr) return 0;
  long long base[MT_MAX_SHARDS], ntot, nmax;
  if (!batch_sizes(g, n, base, &ntot, &nmax)) return 0;
  const mt::TableDev& T = mt::table_dev(g->shards[0]);
  return mt::shard_layout(g->G, ntot, nmax, T.dim, T.emb_bytes).total;
}

int mt_shard_lookup(mt_shard_group* g, const int64_t* const* ids, const int64_t* n, const int64_t* feat_offsets,
                    const uint8_t* table_ids, int F, int insert_missing, void* const* out_rows,
                    const mt_lookup_result* results, void* ws, size_t ws_bytes, mt_stream stream) {
  if (g == nullptr || ids == nullptr || n == nullptr || results == nullptr) return MT_EINVAL;
  const int G = g->G;
  long long base[MT_MAX_SHARDS], ntot, nmax;
  if (!batch_sizes(g, n, base, &ntot, &nmax)) return MT_EINVAL;
  if (feat_offsets == nullptr) F = 1;
  if (F < 1 || F > MT_MAX_FEATURES) return MT_EINVAL;
  const mt::TableDev& T0 = mt::table_dev(g->shards[0]);
  const mt::ShardLayout L = mt::shard_layout(G, ntot, nmax, T0.dim, T0.emb_bytes);
  if (ws == nullptr || ws_bytes < L.total || !aligned(ws, 256)) return MT_ENOSPACE;
  for (int r = 0; r < G; ++r) {
    const mt_lookup_result& R = results[r];
    if (!R.unique_keys || !R.inverse || !R.counts || !R.unique_rows || !R.num_unique) return MT_EINVAL;
    if (n[r] > 0 && (ids[r] == nullptr || !aligned(ids[r], 8))) return MT_EINVAL;
    if (out_rows != nullptr && out_rows[r] != nullptr && !aligned(out_rows[r], 16)) return MT_EINVAL;
  }
  unsigned char tid[MT_MAX_FEATURES];
  for (int f = 0; f < F; ++f) {
    tid[f] = table_ids ? table_ids[f] : 0;
    if (tid[f] == 0xFF) return MT_EINVAL;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  char* scratch = w + L.scratch;
  g->have_lookup = false;

  if (feat_offsets != nullptr) {  // every rank's feature offsets are checked before anything is enqueued
    for (int r = 0; r < G; ++r) {
      const int64_t* fo = feat_offsets + (size_t)r * (F + 1);
      if (fo[0] != 0 || fo[F] != n[r]) return MT_EINVAL;
      for (int f = 1; f <= F; ++f)
        if (fo[f] < fo[f - 1]) return MT_EINVAL;
    }
  }
  const size_t scratch_bytes = L.total - L.scratch;
  // each rank's (or owner's) own slice of the scratch: offsets of lookup workspaces side by side
  auto lookup_slices = [&](const long long* sizes, size_t* off) -> bool {
    size_t o = 0;
    for (int r = 0; r < G; ++r) {
      off[r] = o;
      if (sizes[r] > 0) o = align_up(o + mt::lookup_ws_layout(sizes[r]).total, 256);
    }
    return o <= scratch_bytes;
  };
  size_t soff[MT_MAX_SHARDS];
  long long nn[MT_MAX_SHARDS];
  int active = 0;
  for (int r = 0; r < G; ++r) {
    nn[r] = n[r];
    active += n[r] > 0;
  }
  if (!lookup_slices(nn, soff)) return MT_ENOSPACE;

  // 1. stage 1 on every rank, the ranks side by side: dedup only (first occurrence), no table access
  {
    mt::GroupStreams gs;
    if (gs.begin(s, active) != cudaSuccess) return MT_ECUDA;
    int rc = MT_OK, slot = 0;
    for (int r = 0; r < G && rc == MT_OK; ++r) {
      const cudaStream_t sr = n[r] > 0 ? gs.stream(slot++) : s;
      mt::LookupParams p = lookup_params(mt::table_dev(g->shards[r]), reinterpret_cast<const long long*>(ids[r]),
                                         n[r], scratch + soff[r]);
      p.F = F;
      if (feat_offsets == nullptr) {
        p.feat_off[0] = 0;
        p.feat_off[1] = n[r];
      } else {
        const int64_t* fo = feat_offsets + (size_t)r * (F + 1);
        for (int f = 0; f <= F; ++f) p.feat_off[f] = fo[f];
      }
      for (int f = 0; f < F; ++f) p.table_ids[f] = tid[f];
      p.no_table = 1;
      p.unique_keys = reinterpret_cast<unsigned long long*>(results[r].unique_keys);
      p.inverse = results[r].inverse;
      p.counts = results[r].counts;
      p.unique_rows = results[r].unique_rows;
      p.num_unique = reinterpret_cast<long long*>(results[r].num_unique);
      p.ranks = results[r].ranks;
      if (mt::launch_lookup(p, sr) != cudaSuccess) rc = MT_ECUDA;
    }
    if (gs.end() != cudaSuccess && rc == MT_OK) rc = MT_ECUDA;  // joined also after an error
    if (rc != MT_OK) return rc;
  }
  // 2. the partition counts, read on the host as the sizes of the exchange
  long long U[MT_MAX_SHARDS];
  for (int r = 0; r < G; ++r)
    if (cudaMemcpyAsync(&U[r], results[r].num_unique, sizeof(long long), cudaMemcpyDeviceToHost, s) != cudaSuccess)
      return MT_ECUDA;
  int32_t* counts = reinterpret_cast<int32_t*>(w + L.counts);
  int32_t* cursor = reinterpret_cast<int32_t*>(w + L.cursor);
  if (cudaMemsetAsync(counts, 0, MT_MAX_SHARDS * MT_MAX_SHARDS * 4, s) != cudaSuccess) return MT_ECUDA;
  if (cudaMemsetAsync(cursor, 0, MT_MAX_SHARDS * MT_MAX_SHARDS * 4, s) != cudaSuccess) return MT_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MT_ECUDA;
  for (int r = 0; r < G; ++r) {
    if (U[r] == 0) continue;
    MT_LAUNCH("k_shard_count", s);
    mt::k_shard_count<<<mt::grid_of(U[r]), 256, 0, s>>>(
        reinterpret_cast<const unsigned long long*>(results[r].unique_keys), U[r], G, r, counts);
  }
  int32_t hc[MT_MAX_SHARDS * MT_MAX_SHARDS];
  if (cudaMemcpyAsync(hc, counts, sizeof(int32_t) * G * G, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MT_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MT_ECUDA;
  mt::ShardOffsets off{};
  long long recv_base[MT_MAX_SHARDS], N[MT_MAX_SHARDS], t = 0;
  for (int o = 0; o < G; ++o) {
    recv_base[o] = t;
    for (int r = 0; r < G; ++r) {
      off.off[o * G + r] = t;
      t += hc[r * G + o];
    }
    N[o] = t - recv_base[o];
  }
  // 3. the exchange: every rank writes its keys into the owners' receive buffers
  unsigned long long* recv_keys = reinterpret_cast<unsigned long long*>(w + L.recv_keys);
  int32_t* perm = reinterpret_cast<int32_t*>(w + L.perm);
  for (int r = 0; r < G; ++r) {
    if (U[r] == 0) continue;
    MT_LAUNCH("k_shard_send", s);
    mt::k_shard_send<<<mt::grid_of(U[r]), 256, 0, s>>>(reinterpret_cast<const unsigned long long*>(results[r].unique_keys),
                                                       U[r], G, r, off, cursor, recv_keys, t, perm + base[r],
                                                       mt::table_dev(g->shards[r]).hdr);
  }
  // 4. stage 2 at every owner, the owners side by side: dedup what arrived, find or insert in the shard, gather
  //    one row per received key
  char* recv_rows = w + L.recv_rows;
  const int vec16 = (int)(T0.emb_bytes / 16);
  {
    if (!lookup_slices(N, soff)) return MT_ENOSPACE;
    int owners = 0;
    for (int o = 0; o < G; ++o) owners += N[o] > 0;
    mt::GroupStreams gs;
    if (gs.begin(s, owners) != cudaSuccess) return MT_ECUDA;
    int rc = MT_OK, slot = 0;
    for (int o = 0; o < G && rc == MT_OK; ++o) {
      const cudaStream_t so = N[o] > 0 ? gs.stream(slot++) : s;
      const long long rb = recv_base[o];
      mt::LookupParams p = lookup_params(mt::table_dev(g->shards[o]), reinterpret_cast<const long long*>(recv_keys + rb),
                                         N[o], scratch + soff[o]);
      p.F = 1;
      p.feat_off[0] = 0;
      p.feat_off[1] = N[o];
      p.keys_in = 1;
      p.insert_missing = insert_missing ? 1 : 0;
      p.out_rows = recv_rows + (size_t)rb * T0.emb_bytes;
      p.unique_keys = reinterpret_cast<unsigned long long*>(w + L.uk2) + rb;
      p.inverse = reinterpret_cast<int32_t*>(w + L.inv2) + rb;
      p.counts = reinterpret_cast<int32_t*>(w + L.cnt2) + rb;
      p.unique_rows = reinterpret_cast<int32_t*>(w + L.rows2) + rb;
      p.num_unique = reinterpret_cast<long long*>(w + L.nu2) + o;
      p.ranks = reinterpret_cast<int32_t*>(w + L.rank2) + rb;
      if (mt::launch_lookup(p, so) != cudaSuccess) rc = MT_ECUDA;
    }
    if (gs.end() != cudaSuccess && rc == MT_OK) rc = MT_ECUDA;
    if (rc != MT_OK) return rc;
  }
  // 5. rows back to the ranks, then each rank expands them to its positions
  char* uniq_rows = w + L.uniq_rows;
  for (int r = 0; r < G; ++r) {
    if (U[r] > 0) {
      MT_LAUNCH("k_shard_gather", s);
      mt::k_shard_gather<<<mt::grid_of(U[r] * vec16), 256, 0, s>>>(
          reinterpret_cast<const uint4*>(recv_rows), t, perm + base[r], U[r], vec16,
          reinterpret_cast<uint4*>(uniq_rows + (size_t)base[r] * T0.emb_bytes));
    }
    if (out_rows != nullptr && out_rows[r] != nullptr && n[r] > 0) {
      MT_LAUNCH("k_shard_gather", s);
      mt::k_shard_gather<<<mt::grid_of(n[r] * vec16), 256, 0, s>>>(
          reinterpret_cast<const uint4*>(uniq_rows + (size_t)base[r] * T0.emb_bytes), U[r], results[r].inverse, n[r],
          vec16, static_cast<uint4*>(out_rows[r]));
    }
  }
  if (cudaGetLastError() != cudaSuccess) return MT_ECUDA;
  for (int r = 0; r < G; ++r) {
    g->n[r] = n[r];
    g->U[r] = U[r];
    g->N[r] = N[r];
    g->recv_base[r] = recv_base[r];
    g->rank_base[r] = base[r];
  }
  g->ntot = ntot;
  g->ws_bytes = L.total;
  g->have_lookup = true;
  return MT_OK;
}

int mt_shard_backward_adam(mt_shard_group* g, const mt_lookup_result* results, const void* const* grads,
                           int grad_dtype, const mt_adam* hp, float* const* gsum_out, void* ws, size_t ws_bytes,
                           mt_stream stream) {
  if (g == nullptr || results == nullptr || grads == nullptr || hp == nullptr) return MT_EINVAL;
  if (!g->have_lookup) return MT_EINVAL;
  if (grad_dtype != MT_F32 && grad_dtype != MT_BF16) return MT_EINVAL;
  if (!(hp->lr >= 0.0f) || !(hp->beta1 >= 0.0f && hp->beta1 < 1.0f) || !(hp->beta2 >= 0.0f && hp->beta2 < 1.0f) ||
      !(hp->eps > 0.0f))
    return MT_EINVAL;
  const int G = g->G;
  long long nmax = 0;
  for (int r = 0; r < G; ++r) {
    nmax = g->n[r] > nmax ? g->n[r] : nmax;
    if (g->n[r] > 0 && (grads[r] == nullptr || !aligned(grads[r], 16))) return MT_EINVAL;
    if (gsum_out != nullptr && gsum_out[r] != nullptr && !aligned(gsum_out[r], 16)) return MT_EINVAL;
  }
  const mt::TableDev& T0 = mt::table_dev(g->shards[0]);
  const mt::ShardLayout L = mt::shard_layout(G, g->ntot, nmax, T0.dim, T0.emb_bytes);
  if (ws == nullptr || ws_bytes < L.total || !aligned(ws, 256)) return MT_ENOSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  char* scratch = w + L.scratch;
  const int d = (int)T0.dim;
  const int gvec = d * 4 / 16;
  float* gsum = reinterpret_cast<float*>(w + L.gsum);
  float* recv_g = reinterpret_cast<float*>(w + L.recv_g);
  const int32_t* perm = reinterpret_cast<const int32_t*>(w + L.perm);

  auto run = [&](mt_table* shard, const mt_lookup_result& R, long long n, const void* gr, int gd, float* out,
                 int reduce_only, char* scr, cudaStream_t st) -> int {
    const mt::TableDev& T = mt::table_dev(shard);
    const mt::BackwardWsLayout BL = mt::backward_ws_layout(n, T.dim);
    mt::BackwardParams p;
    std::memset(&p, 0, sizeof(p));
    p.T = T;
    p.n = n;
    p.grad_rows = n;
    p.inverse = R.inverse;
    p.ranks = R.ranks;
    p.counts = R.counts;
    p.unique_rows = R.unique_rows;
    p.num_unique = reinterpret_cast<const long long*>(R.num_unique);
    p.grads = gr;
    p.grad_dtype = gd;
    p.lr = hp->lr;
    p.beta1 = hp->beta1;
    p.beta2 = hp->beta2;
    p.eps = hp->eps;
    p.one_minus_b1 = (float)(1.0 - (double)hp->beta1);
    p.one_minus_b2 = (float)(1.0 - (double)hp->beta2);
    p.gsum_out = out;
    p.reduce_only = reduce_only;
    mt::bind_backward_ws(p, scr, BL);
    p.team_shift = mt::backward_team_shift(T.dim, T.row_dtype);
    p.warp_chunk = mt::heavy_warp_chunk(p.n, p.team_shift);
    return mt::launch_backward(p, st) == cudaSuccess ? MT_OK : MT_ECUDA;
  };
  // each rank's (or owner's) own slice of the scratch: offsets of backward workspaces side by side
  const size_t scratch_bytes = L.total - L.scratch;
  // (an owner that received nothing still runs its backward, which advances its step counter, so every one
  // gets a slice)
  auto backward_slices = [&](const long long* sizes, size_t* off, int* active) -> bool {
    size_t o = 0;
    *active = 0;
    for (int r = 0; r < G; ++r) {
      off[r] = o;
      o = align_up(o + mt::backward_ws_layout(sizes[r], T0.dim).total, 256);
      *active += sizes[r] > 0;
    }
    return o <= scratch_bytes;
  };
  size_t soff[MT_MAX_SHARDS];
  int active = 0;

  // 1. every rank, the ranks side by side: per-unique sums of its positions' gradients (no Adam)
  {
    if (!backward_slices(g->n, soff, &active)) return MT_ENOSPACE;
    mt::GroupStreams gs;
    if (gs.begin(s, active) != cudaSuccess) return MT_ECUDA;
    int rc = MT_OK, slot = 0;
    for (int r = 0; r < G && rc == MT_OK; ++r) {
      if (g->n[r] == 0) continue;
      rc = run(g->shards[r], results[r], g->n[r], grads[r], grad_dtype, gsum + (size_t)g->rank_base[r] * d, 1,
               scratch + soff[r], gs.stream(slot++));
    }
    if (gs.end() != cudaSuccess && rc == MT_OK) rc = MT_ECUDA;  // joined also after an error
    if (rc != MT_OK) return rc;
  }
  // 2. the sums go to the owners (the exchange of the forward, reversed)
  for (int r = 0; r < G; ++r) {
    if (g->U[r] == 0) continue;
    MT_LAUNCH("k_shard_scatter", s);
    mt::k_shard_scatter<<<mt::grid_of(g->U[r] * gvec), 256, 0, s>>>(
        reinterpret_cast<const uint4*>(gsum + (size_t)g->rank_base[r] * d), perm + g->rank_base[r], g->U[r], gvec,
        reinterpret_cast<uint4*>(recv_g), g->ntot);
  }
  // 3. every owner, the owners side by side: sums over the ranks per key, one Adam step on its shard (its step
  //    counter advances once)
  float* gsum2 = reinterpret_cast<float*>(w + L.gsum2);
  {
    if (!backward_slices(g->N, soff, &active)) return MT_ENOSPACE;
    mt::GroupStreams gs;
    if (gs.begin(s, active) != cudaSuccess) return MT_ECUDA;
    int rc = MT_OK, slot = 0;
    for (int o = 0; o < G && rc == MT_OK; ++o) {
      const long long rb = g->recv_base[o];
      mt_lookup_result R2;
      R2.unique_keys = reinterpret_cast<uint64_t*>(w + L.uk2) + rb;
      R2.inverse = reinterpret_cast<int32_t*>(w + L.inv2) + rb;
      R2.counts = reinterpret_cast<int32_t*>(w + L.cnt2) + rb;
      R2.unique_rows = reinterpret_cast<int32_t*>(w + L.rows2) + rb;
      R2.num_unique = reinterpret_cast<int64_t*>(w + L.nu2) + o;
      R2.ranks = reinterpret_cast<int32_t*>(w + L.rank2) + rb;
      const cudaStream_t so = g->N[o] > 0 ? gs.stream(slot++) : s;
      rc = run(g->shards[o], R2, g->N[o], recv_g + (size_t)rb * d, MT_F32, gsum2 + (size_t)rb * d, 0,
               scratch + soff[o], so);
      if (rc == MT_OK) mt::table_count_step(g->shards[o]);
    }
    if (gs.end() != cudaSuccess && rc == MT_OK) rc = MT_ECUDA;
    if (rc != MT_OK) return rc;
  }
  // 4. asked for: each rank's per-unique sums over all ranks, from the owners
  if (gsum_out != nullptr) {
    int32_t* idx = reinterpret_cast<int32_t*>(w + L.idx);
    mt::ShardOffsets ob{};
    for (int o = 0; o < G; ++o) ob.off[o] = g->recv_base[o];
    for (int r = 0; r < G; ++r) {
      if (gsum_out[r] == nullptr || g->U[r] == 0) continue;
      {
        MT_LAUNCH("k_shard_owner_unique", s);
        mt::k_shard_owner_unique<<<mt::grid_of(g->U[r]), 256, 0, s>>>(
            reinterpret_cast<const unsigned long long*>(results[r].unique_keys), perm + g->rank_base[r], g->U[r], G,
            ob, reinterpret_cast<const int32_t*>(w + L.inv2), g->ntot, idx + g->rank_base[r]);
      }
      MT_LAUNCH("k_shard_gather", s);
      mt::k_shard_gather<<<mt::grid_of(g->U[r] * gvec), 256, 0, s>>>(
          reinterpret_cast<const uint4*>(gsum2), g->ntot, idx + g->rank_base[r], g->U[r], gvec,
          reinterpret_cast<uint4*>(gsum_out[r]));
    }
  }
  return cudaGetLastError() == cudaSuccess ? MT_OK : MT_ECUDA;
}

}  // extern "C"
