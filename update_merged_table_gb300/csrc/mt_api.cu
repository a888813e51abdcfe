// The C ABI (include/mt.h): argument validation, arena and workspace
// carving, kernel launches.  No device memory is allocated here.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <new>

#include "mt_kernels.cuh"

namespace mt {
int sm_count() {
  static std::atomic<int> sms[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return 1;
  int v = sms[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) return 1;
    sms[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

// Positions per heavy warp-chunk of a backward over n positions.  A team's
// share stays at most kTeamShare (its positions are staged in shared memory)
// and a warp-chunk at least kTeamShare positions, so that no batch makes more
// warp-chunks than the workspace layout counts (n / kTeamShare + one per
// heavy key).  Within that range the warp-chunk covers n / (6 x SMs)
// positions: long enough to amortise its start and its fp64 partial sums
// (batches of 0.26M and more keep the longest), short enough that a small
// batch's hottest key is not one warp's serial chain (a 4096-ID batch put its
// hottest key's few hundred positions in one 512-position warp-chunk).
int heavy_warp_chunk(long long n, int team_shift) {
  const long long tpw = 32 >> team_shift;  // teams per warp
  const long long parts = (long long)sm_count() * 6;
  long long wc = (n + parts - 1) / parts;
  wc = (wc + tpw - 1) / tpw * tpw;
  return (int)std::max<long long>(kTeamShare, std::min<long long>(wc, kTeamShare * tpw));
}
}  // namespace mt

struct mt_table {
  mt_config cfg;
  mt::TableDev dev;
  char* ks_base;     // the key store in use (header at its start)
  size_t ks_bytes;
  long long step;    // host-side count of backward calls
};

namespace mt {
const TableDev& table_dev(const mt_table* t) { return t->dev; }
mt_config table_cfg(const mt_table* t) { return t->cfg; }
void table_count_step(mt_table* t) { t->step += 1; }
}  // namespace mt

namespace {

using mt::align_up;

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Fill defaults and check a configuration; returns MT_OK or MT_EINVAL.
int normalise(const mt_config* in, mt_config* out) {
  if (in == nullptr) return MT_EINVAL;
  mt_config c = *in;
  if (c.log2_slots < 1 || c.log2_slots > 31) return MT_EINVAL;
  if (c.flags != 0) return MT_EINVAL;
  if (c.row_dtype != MT_F32 && c.row_dtype != MT_BF16) return MT_EINVAL;
  const uint32_t vec = c.row_dtype == MT_F32 ? 4 : 8;
  if (c.dim < 4 || c.dim > MT_MAX_DIM || c.dim % vec != 0) return MT_EINVAL;
  const uint64_t M = 1ull << c.log2_slots;
  c.probe_step &= (M - 1);
  if ((c.probe_step & 1ull) == 0) return MT_EINVAL;  // Theorem 1: only an odd step covers the table
  if (c.max_probes == 0 || c.max_probes > M) c.max_probes = (uint32_t)(M > 0xFFFFFFFFull ? 0xFFFFFFFFull : M);
  if (!(c.init_scale >= 0.0f) || std::isinf(c.init_scale)) return MT_EINVAL;
  if (c.init_scale == 0.0f) c.init_scale = (float)(1.0 / std::sqrt((double)c.dim));
  if (c.num_rows == 0) c.num_rows = (int64_t)M;
  if (c.num_rows < 1 || (uint64_t)c.num_rows > M || c.num_rows > 0x7FFFFFFF) return MT_EINVAL;
  *out = c;
  return MT_OK;
}

// Key store: [header 1 KiB][M slots x 16 B][free list: R x int32], each part 256-byte aligned.
struct KeystoreLayout {
  size_t hdr, slots, stack, total;
  uint32_t rec_bytes, emb_bytes, mv_bytes;
};

KeystoreLayout keystore_layout(const mt_config& c) {
  KeystoreLayout L{};
  const uint64_t M = 1ull << c.log2_slots;
  L.emb_bytes = c.dim * (c.row_dtype == MT_F32 ? 4u : 2u);
  L.mv_bytes = c.dim * 4u;
  L.rec_bytes = L.emb_bytes + 2u * L.mv_bytes;  // each part is a multiple of 16 bytes
  size_t off = 0;
  L.hdr = off;
  off = align_up(off + mt::kHeaderBytes, 256);
  L.slots = off;
  off = align_up(off + (size_t)M * sizeof(mt::Slot), 256);
  L.stack = off;
  off = align_up(off + (size_t)c.num_rows * 4, 256);
  L.total = off;
  return L;
}

size_t rows_bytes_of(const mt_config& c, long long rows) {
  const KeystoreLayout L = keystore_layout(c);
  return align_up((size_t)rows * L.rec_bytes, 256);
}

uint64_t inverse_mod_2_64(uint64_t S);

// The kernels' view of a table whose key store is at `ks` and whose only row segment is `rows`.
mt::TableDev device_view(const mt_config& c, void* ks, void* rows) {
  const KeystoreLayout L = keystore_layout(c);
  mt::TableDev T{};
  char* base = static_cast<char*>(ks);
  T.hdr = reinterpret_cast<mt::Header*>(base + L.hdr);
  T.slots = reinterpret_cast<mt::Slot*>(base + L.slots);
  T.free_stack = reinterpret_cast<int32_t*>(base + L.stack);
  T.seg_base[0] = static_cast<char*>(rows);
  T.seg_first[0] = 0;
  T.nseg = 1;
  const uint64_t M = 1ull << c.log2_slots;
  T.mask = M - 1;
  T.S = c.probe_step;
  T.hash_seed = c.hash_seed;
  T.init_seed = c.init_seed;
  T.Sinv = inverse_mod_2_64(c.probe_step) & (M - 1);
  T.log2_slots = c.log2_slots;
  T.max_probes = c.max_probes;
  T.flags = c.flags;
  T.dim = c.dim;
  T.rec_bytes = L.rec_bytes;
  T.emb_bytes = L.emb_bytes;
  T.mv_bytes = L.mv_bytes;
  T.row_dtype = (int)c.row_dtype;
  T.init_scale = c.init_scale;
  T.num_rows = c.num_rows;
  return T;
}

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

// Does [p, p + n) overlap any memory the table uses (key store, slots, row segments)?
bool overlaps_table(const mt_table* t, const void* p, size_t n) {
  if (overlap(p, n, t->ks_base, t->ks_bytes)) return true;
  if (overlap(p, n, t->dev.slots, (size_t)(t->dev.mask + 1) * sizeof(mt::Slot))) return true;
  for (int s = 0; s < t->dev.nseg; ++s) {
    const long long end = s + 1 < t->dev.nseg ? t->dev.seg_first[s + 1] : t->dev.num_rows;
    if (overlap(p, n, t->dev.seg_base[s], (size_t)(end - t->dev.seg_first[s]) * t->dev.rec_bytes)) return true;
  }
  return false;
}

int create_table(const mt_config& c, void* ks, void* rows, cudaStream_t stream, mt_table** out) {
  mt_table* t = new (std::nothrow) mt_table();
  if (t == nullptr) return MT_ECUDA;
  t->cfg = c;
  t->ks_base = static_cast<char*>(ks);
  t->ks_bytes = keystore_layout(c).total;
  t->step = 0;
  t->dev = device_view(c, ks, rows);
  if (mt::launch_table_init(t->dev, stream) != cudaSuccess) {
    delete t;
    return MT_ECUDA;
  }
  *out = t;
  return MT_OK;
}

// S^-1 mod 2^64 by Newton's iteration x <- x(2 - Sx); exact for odd S.
uint64_t inverse_mod_2_64(uint64_t S) {
  uint64_t x = S;  // correct to 3 bits for odd S
  for (int i = 0; i < 6; ++i) x *= 2 - S * x;
  return x;
}

cudaStream_t as_stream(mt_stream s) { return reinterpret_cast<cudaStream_t>(s); }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MT_OK : MT_ECUDA; }

bool valid_result(const mt_lookup_result* r) {
  return r != nullptr && r->unique_keys && r->inverse && r->counts && r->unique_rows && r->num_unique &&
         aligned(r->unique_keys, 16) && aligned(r->inverse, 16) && aligned(r->counts, 16) &&
         aligned(r->unique_rows, 16) && aligned(r->num_unique, 8) && aligned(r->ranks, 16);
}

int check_backward(const mt_table* t, const mt_lookup_result* res, int grad_dtype, const mt_adam* hp,
                   const float* gsum_out) {
  if (!valid_result(res) || hp == nullptr) return MT_EINVAL;
  if (grad_dtype != MT_F32 && grad_dtype != MT_BF16) return MT_EINVAL;
  if (gsum_out != nullptr && !aligned(gsum_out, 16)) return MT_EINVAL;
  if (!(hp->lr >= 0.0f) || !(hp->beta1 >= 0.0f && hp->beta1 < 1.0f) || !(hp->beta2 >= 0.0f && hp->beta2 < 1.0f) ||
      !(hp->eps > 0.0f))
    return MT_EINVAL;
  return MT_OK;
}

// One backward + Adam step; gradient row r of `grads` feeds every position
// mapped to it (pos_map, or the position itself when pos_map is NULL).
int run_backward(mt_table* t, const mt_lookup_result* res, int64_t n, const void* grads, int grad_dtype,
                 const int32_t* pos_map, int64_t grad_rows, const mt_adam* hp, float* gsum_out, void* ws,
                 const mt::BackwardWsLayout& L, cudaStream_t stream) {
  char* w = static_cast<char*>(ws);
  mt::BackwardParams p;
  std::memset(&p, 0, sizeof(p));
  p.T = t->dev;
  p.n = n;
  p.pos_map = pos_map;
  p.grad_rows = grad_rows;
  p.inverse = res->inverse;
  p.ranks = res->ranks;
  p.counts = res->counts;
  p.unique_rows = res->unique_rows;
  p.num_unique = reinterpret_cast<const long long*>(res->num_unique);
  p.grads = grads;
  p.grad_dtype = grad_dtype;
  p.lr = hp->lr;
  p.beta1 = hp->beta1;
  p.beta2 = hp->beta2;
  p.eps = hp->eps;
  p.one_minus_b1 = (float)(1.0 - (double)hp->beta1);
  p.one_minus_b2 = (float)(1.0 - (double)hp->beta2);
  p.gsum_out = gsum_out;
  mt::bind_backward_ws(p, w, L);
  p.team_shift = mt::backward_team_shift(t->cfg.dim, (int)t->cfg.row_dtype);
  p.warp_chunk = mt::heavy_warp_chunk(n, p.team_shift);
  const int rc = cuda_status(mt::launch_backward(p, stream));
  if (rc == MT_OK) t->step += 1;
  return rc;
}

// Workspace of the pooled backward: the backward's own, the bag of every
// position, and (for the mean) the scaled bag gradients.
struct PooledLayout {
  mt::BackwardWsLayout bw;
  size_t backward, pos_bag, scaled, total;
};

PooledLayout pooled_layout(const mt_table* t, int64_t n, int64_t num_bags) {
  PooledLayout L{};
  L.bw = mt::backward_ws_layout(n, t->cfg.dim);
  L.backward = 0;
  L.pos_bag = align_up(L.bw.total, 256);
  L.scaled = align_up(L.pos_bag + (size_t)(n > 0 ? n : 1) * 4, 256);
  L.total = align_up(L.scaled + (size_t)(num_bags > 0 ? num_bags : 1) * t->cfg.dim * 4, 256);
  return L;
}

}  // namespace

namespace mt {
// The host checks mt_lookup and mt_backward_adam make on a group's own
// arguments before enqueuing anything: the grouped calls run them for every
// group first, so that an error still leaves nothing enqueued.
int lookup_group_status(const mt_lookup_result* res, const void* out_rows) {
  if (!valid_result(res)) return MT_EINVAL;
  if (out_rows != nullptr && !aligned(out_rows, 16)) return MT_EINVAL;
  return MT_OK;
}
int backward_group_status(const mt_table* t, const mt_lookup_result* res, int64_t n, const void* grads,
                          int grad_dtype, const mt_adam* hp, const float* gsum_out) {
  if (t == nullptr || n < 0 || n > 0x7FFFFFFF) return MT_EINVAL;
  if (n > 0 && (grads == nullptr || !aligned(grads, 16))) return MT_EINVAL;
  return check_backward(t, res, grad_dtype, hp, gsum_out);
}
}  // namespace mt

extern "C" {

int mt_abi_version(void) { return MT_ABI_VERSION; }

const char* mt_strerror(int code) {
  switch (code) {
    case MT_OK: return "ok";
    case MT_EINVAL: return "invalid argument";
    case MT_ENOSPACE: return "arena or workspace too small or misaligned";
    case MT_EFULL: return "probe limit reached or row pool exhausted";
    case MT_EKEY: return "ID outside [0, 2^56)";
    case MT_ECUDA: return "CUDA runtime error";
    case MT_ETOOBIG: return "batch larger than the fixed-size workspace allows";
    default: return "unknown status";
  }
}

size_t mt_table_bytes(const mt_config* cfg) {
  mt_config c;
  if (normalise(cfg, &c) != MT_OK) return 0;
  return keystore_layout(c).total + rows_bytes_of(c, c.num_rows);
}

size_t mt_keystore_bytes(const mt_config* cfg) {
  mt_config c;
  if (normalise(cfg, &c) != MT_OK) return 0;
  return keystore_layout(c).total;
}

size_t mt_rows_bytes(const mt_config* cfg, int64_t rows) {
  mt_config c;
  if (normalise(cfg, &c) != MT_OK || rows < 0 || rows > 0x7FFFFFFF) return 0;
  return rows_bytes_of(c, rows);
}

int mt_table_create(const mt_config* cfg, void* dev_mem, size_t bytes, mt_stream stream, mt_table** out) {
  if (out == nullptr) return MT_EINVAL;
  *out = nullptr;
  mt_config c;
  const int rc = normalise(cfg, &c);
  if (rc != MT_OK) return rc;
  const size_t ks = keystore_layout(c).total;
  if (dev_mem == nullptr || bytes < ks + rows_bytes_of(c, c.num_rows) || !aligned(dev_mem, 256)) return MT_ENOSPACE;
  return create_table(c, dev_mem, static_cast<char*>(dev_mem) + ks, as_stream(stream), out);
}

int mt_table_create_split(const mt_config* cfg, void* keystore, size_t keystore_bytes, void* rows,
                          size_t rows_bytes, mt_stream stream, mt_table** out) {
  if (out == nullptr) return MT_EINVAL;
  *out = nullptr;
  mt_config c;
  const int rc = normalise(cfg, &c);
  if (rc != MT_OK) return rc;
  const size_t ks = keystore_layout(c).total, rb = rows_bytes_of(c, c.num_rows);
  if (keystore == nullptr || keystore_bytes < ks || !aligned(keystore, 256)) return MT_ENOSPACE;
  if (rows == nullptr || rows_bytes < rb || !aligned(rows, 256)) return MT_ENOSPACE;
  if (overlap(keystore, ks, rows, rb)) return MT_EINVAL;
  return create_table(c, keystore, rows, as_stream(stream), out);
}

int mt_table_grow(mt_table* t, const mt_config* new_cfg, void* keystore, size_t keystore_bytes, void* rows,
                  size_t rows_bytes, mt_stream stream) {
  if (t == nullptr) return MT_EINVAL;
  mt_config c;
  const int rc = normalise(new_cfg, &c);
  if (rc != MT_OK) return rc;
  const mt_config& o = t->cfg;
  if (c.log2_slots < o.log2_slots || c.num_rows < o.num_rows || c.dim != o.dim || c.row_dtype != o.row_dtype ||
      c.hash_seed != o.hash_seed || c.init_seed != o.init_seed || c.init_scale != o.init_scale ||
      c.flags != o.flags || (c.probe_step & ((1ull << o.log2_slots) - 1)) != o.probe_step)
    return MT_EINVAL;
  const long long added = c.num_rows - o.num_rows;
  if (added > 0 && t->dev.nseg >= mt::kMaxRowSegments) return MT_EINVAL;
  const size_t ks = keystore_layout(c).total, rb = rows_bytes_of(c, added);
  if (keystore == nullptr || keystore_bytes < ks || !aligned(keystore, 256)) return MT_ENOSPACE;
  if (added > 0 && (rows == nullptr || rows_bytes < rb || !aligned(rows, 256))) return MT_ENOSPACE;
  // the rebuild reads the old key store while it writes the new one, and no row may be overwritten
  if (overlaps_table(t, keystore, ks) || (added > 0 && (overlaps_table(t, rows, rb) || overlap(keystore, ks, rows, rb))))
    return MT_EINVAL;
  mt::TableDev T2 = device_view(c, keystore, t->dev.seg_base[0]);
  T2.nseg = t->dev.nseg;
  for (int s = 0; s < t->dev.nseg; ++s) {
    T2.seg_base[s] = t->dev.seg_base[s];
    T2.seg_first[s] = t->dev.seg_first[s];
  }
  if (added > 0) {
    T2.seg_base[T2.nseg] = static_cast<char*>(rows);
    T2.seg_first[T2.nseg] = o.num_rows;
    T2.nseg += 1;
  }
  cudaStream_t s = as_stream(stream);
  if (mt::launch_grow(t->dev, T2, s) != cudaSuccess) return MT_ECUDA;
  int32_t fail = 0;
  if (cudaMemcpyAsync(&fail, &T2.hdr->pad0, sizeof(fail), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MT_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MT_ECUDA;
  if (fail) return MT_EFULL;
  t->cfg = c;
  t->dev = T2;
  t->ks_base = static_cast<char*>(keystore);
  t->ks_bytes = ks;
  return MT_OK;
}

int mt_table_destroy(mt_table* t) {
  if (t == nullptr) return MT_EINVAL;
  delete t;
  return MT_OK;
}

int mt_table_config(const mt_table* t, mt_config* out) {
  if (t == nullptr || out == nullptr) return MT_EINVAL;
  *out = t->cfg;
  return MT_OK;
}

size_t mt_lookup_workspace_bytes(const mt_table* t, int64_t n) {
  if (t == nullptr || n < 0 || n > 0x7FFFFFFF) return 0;
  return mt::lookup_ws_layout(n).total;
}

int mt_lookup(mt_table* t, const int64_t* ids, int64_t n, const int64_t* feat_offsets, const uint8_t* table_ids,
              int F, int insert_missing, void* out_rows, const mt_lookup_result* res, void* ws, size_t ws_bytes,
              mt_stream stream) {
  if (t == nullptr || n < 0 || n > 0x7FFFFFFF || !valid_result(res)) return MT_EINVAL;
  if (n > 0 && (ids == nullptr || !aligned(ids, 8))) return MT_EINVAL;
  if (out_rows != nullptr && !aligned(out_rows, 16)) return MT_EINVAL;
  if (feat_offsets == nullptr) F = 1;
  if (F < 1 || F > MT_MAX_FEATURES) return MT_EINVAL;
  mt::LookupParams p;
  std::memset(&p, 0, sizeof(p));
  p.T = t->dev;
  p.ids = reinterpret_cast<const long long*>(ids);
  p.n = n;
  p.F = F;
  p.insert_missing = insert_missing ? 1 : 0;
  if (feat_offsets == nullptr) {
    p.feat_off[0] = 0;
    p.feat_off[1] = n;
  } else {
    if (feat_offsets[0] != 0 || feat_offsets[F] != n) return MT_EINVAL;
    for (int f = 0; f <= F; ++f) {
      if (f > 0 && feat_offsets[f] < feat_offsets[f - 1]) return MT_EINVAL;
      p.feat_off[f] = feat_offsets[f];
    }
  }
  for (int f = 0; f < F; ++f) {
    const uint8_t tid = table_ids ? table_ids[f] : 0;
    if (tid == 0xFF) return MT_EINVAL;  // table id 255 holds the sentinels
    p.table_ids[f] = tid;
  }
  const mt::LookupWsLayout L = mt::lookup_ws_layout(n);
  if (n > 0 && (ws == nullptr || ws_bytes < L.total || !aligned(ws, 256))) return MT_ENOSPACE;
  char* w = static_cast<char*>(ws);
  p.out_rows = out_rows;
  p.unique_keys = reinterpret_cast<unsigned long long*>(res->unique_keys);
  p.inverse = res->inverse;
  p.counts = res->counts;
  p.unique_rows = res->unique_rows;
  p.num_unique = reinterpret_cast<long long*>(res->num_unique);
  p.ranks = res->ranks;
  if (n > 0) mt::bind_lookup_ws(p, w, L);
  return cuda_status(mt::launch_lookup(p, as_stream(stream)));
}

size_t mt_backward_workspace_bytes(const mt_table* t, int64_t n) {
  if (t == nullptr || n < 0 || n > 0x7FFFFFFF) return 0;
  return mt::backward_ws_layout(n, t->cfg.dim).total;
}

int mt_backward_adam(mt_table* t, const mt_lookup_result* res, int64_t n, const void* grads, int grad_dtype,
                     const mt_adam* hp, float* gsum_out, void* ws, size_t ws_bytes, mt_stream stream) {
  if (t == nullptr || n < 0 || n > 0x7FFFFFFF) return MT_EINVAL;
  if (n > 0 && (grads == nullptr || !aligned(grads, 16))) return MT_EINVAL;
  const int rc = check_backward(t, res, grad_dtype, hp, gsum_out);
  if (rc != MT_OK) return rc;
  const mt::BackwardWsLayout L = mt::backward_ws_layout(n, t->cfg.dim);
  if (ws == nullptr || ws_bytes < L.total || !aligned(ws, 256)) return MT_ENOSPACE;
  return run_backward(t, res, n, grads, grad_dtype, nullptr, n, hp, gsum_out, ws, L, as_stream(stream));
}

size_t mt_pool_workspace_bytes(const mt_table* t, int64_t num_bags) {
  if (t == nullptr || num_bags < 0 || num_bags > 0x7FFFFFFF) return 0;
  return align_up((size_t)(num_bags > 0 ? num_bags : 1) * t->cfg.dim * sizeof(double), 256);
}

int mt_pool_forward(mt_table* t, const mt_lookup_result* res, int64_t n, const int64_t* bag_offsets,
                    int64_t num_bags, int mode, float* out, void* ws, size_t ws_bytes, mt_stream stream) {
  if (t == nullptr || n < 0 || n > 0x7FFFFFFF || num_bags < 0 || num_bags > 0x7FFFFFFF || !valid_result(res))
    return MT_EINVAL;
  if (mode != MT_POOL_SUM && mode != MT_POOL_MEAN) return MT_EINVAL;
  if (num_bags > 0 && (bag_offsets == nullptr || !aligned(bag_offsets, 8) || out == nullptr || !aligned(out, 16)))
    return MT_EINVAL;
  if (num_bags == 0) return MT_OK;
  if (ws == nullptr || ws_bytes < mt_pool_workspace_bytes(t, num_bags) || !aligned(ws, 256)) return MT_ENOSPACE;
  mt::PoolParams p;
  std::memset(&p, 0, sizeof(p));
  p.T = t->dev;
  p.n = n;
  p.inverse = res->inverse;
  p.unique_rows = res->unique_rows;
  p.num_unique = reinterpret_cast<const long long*>(res->num_unique);
  p.bag_offsets = reinterpret_cast<const long long*>(bag_offsets);
  p.num_bags = num_bags;
  p.mode = mode;
  p.team_shift = mt::backward_team_shift(t->cfg.dim, (int)t->cfg.row_dtype);
  p.out = out;
  p.acc = static_cast<double*>(ws);
  return cuda_status(mt::launch_pool(p, as_stream(stream)));
}

size_t mt_backward_pooled_workspace_bytes(const mt_table* t, int64_t n, int64_t num_bags) {
  if (t == nullptr || n < 0 || n > 0x7FFFFFFF || num_bags < 0 || num_bags > 0x7FFFFFFF) return 0;
  return pooled_layout(t, n, num_bags).total;
}

int mt_backward_adam_pooled(mt_table* t, const mt_lookup_result* res, int64_t n, const int64_t* bag_offsets,
                            int64_t num_bags, int mode, const float* dpooled, const mt_adam* hp, float* gsum_out,
                            void* ws, size_t ws_bytes, mt_stream stream) {
  if (t == nullptr || n < 0 || n > 0x7FFFFFFF || num_bags < 0 || num_bags > 0x7FFFFFFF) return MT_EINVAL;
  if (mode != MT_POOL_SUM && mode != MT_POOL_MEAN) return MT_EINVAL;
  if (num_bags > 0 && (bag_offsets == nullptr || !aligned(bag_offsets, 8) || dpooled == nullptr ||
                       !aligned(dpooled, 16)))
    return MT_EINVAL;
  const int rc = check_backward(t, res, MT_F32, hp, gsum_out);
  if (rc != MT_OK) return rc;
  const PooledLayout PL = pooled_layout(t, n, num_bags);
  if (ws == nullptr || ws_bytes < PL.total || !aligned(ws, 256)) return MT_ENOSPACE;
  char* w = static_cast<char*>(ws);
  cudaStream_t s = as_stream(stream);
  int32_t* pos_bag = reinterpret_cast<int32_t*>(w + PL.pos_bag);
  if (mt::launch_pos_bag(reinterpret_cast<const long long*>(bag_offsets), num_bags, n, pos_bag, t->dev.hdr, s) !=
      cudaSuccess)
    return MT_ECUDA;
  const float* g = dpooled;
  if (mode == MT_POOL_MEAN && num_bags > 0) {
    float* scaled = reinterpret_cast<float*>(w + PL.scaled);
    if (mt::launch_pool_scale(reinterpret_cast<const long long*>(bag_offsets), num_bags, (int)t->cfg.dim, dpooled,
                              scaled, s) != cudaSuccess)
      return MT_ECUDA;
    g = scaled;
  }
  return run_backward(t, res, n, g, MT_F32, pos_bag, num_bags, hp, gsum_out, w + PL.backward, PL.bw, s);
}

size_t mt_erase_workspace_bytes(int64_t n) {
  if (n < 0) return 0;
  return align_up((size_t)(n > 0 ? n : 1) * 4, 256);
}

int mt_erase(mt_table* t, const uint64_t* keys, int64_t n, uint8_t* found, void* ws, size_t ws_bytes,
             mt_stream stream) {
  if (t == nullptr || n < 0) return MT_EINVAL;
  if (n > 0 && (keys == nullptr || !aligned(keys, 8))) return MT_EINVAL;
  if (n > 0 && (ws == nullptr || ws_bytes < mt_erase_workspace_bytes(n) || !aligned(ws, 256))) return MT_ENOSPACE;
  return cuda_status(mt::launch_erase(t->dev, reinterpret_cast<const unsigned long long*>(keys), n, found,
                                      static_cast<int32_t*>(ws), as_stream(stream)));
}

size_t mt_compact_workspace_bytes(const mt_table* t) {
  if (t == nullptr) return 0;
  return (size_t)(t->dev.mask + 1) * sizeof(mt::Slot);
}

int mt_compact(mt_table* t, void* ws, size_t ws_bytes, void** released, mt_stream stream) {
  if (t == nullptr || released == nullptr) return MT_EINVAL;
  *released = nullptr;
  const size_t need = mt_compact_workspace_bytes(t);
  if (ws == nullptr || ws_bytes < need || !aligned(ws, 256)) return MT_ENOSPACE;
  if (overlap(ws, need, t->dev.slots, need)) return MT_EINVAL;
  for (int s = 0; s < t->dev.nseg; ++s) {
    const long long end = s + 1 < t->dev.nseg ? t->dev.seg_first[s + 1] : t->dev.num_rows;
    if (overlap(ws, need, t->dev.seg_base[s], (size_t)(end - t->dev.seg_first[s]) * t->dev.rec_bytes)) return MT_EINVAL;
  }
  if (overlap(ws, need, t->dev.hdr, mt::kHeaderBytes) ||
      overlap(ws, need, t->dev.free_stack, (size_t)t->dev.num_rows * 4))
    return MT_EINVAL;
  cudaStream_t s = as_stream(stream);
  mt::Slot* fresh = static_cast<mt::Slot*>(ws);
  if (mt::launch_compact(t->dev, fresh, s) != cudaSuccess) return MT_ECUDA;
  int32_t fail = 0;
  if (cudaMemcpyAsync(&fail, &t->dev.hdr->pad0, sizeof(fail), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MT_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MT_ECUDA;
  if (fail) return MT_EFULL;
  *released = t->dev.slots;
  t->dev.slots = fresh;
  return MT_OK;
}

int mt_stats(mt_table* t, mt_stats_out* out, mt_stream stream) {
  if (t == nullptr || out == nullptr) return MT_EINVAL;
  cudaStream_t s = as_stream(stream);
  if (mt::launch_stats(t->dev, s) != cudaSuccess) return MT_ECUDA;
  mt::Header h;
  if (cudaMemcpyAsync(&h, t->dev.hdr, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MT_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MT_ECUDA;
  std::memset(out, 0, sizeof(*out));
  out->live = (int64_t)h.live;
  out->tombstones = (int64_t)h.tombs;
  out->capacity = (int64_t)(t->dev.mask + 1);
  out->num_rows = t->cfg.num_rows;
  out->rows_free = h.free_top;
  out->step = h.step;
  out->total_displacement = (int64_t)h.disp;
  out->load_factor = (double)h.live / (double)(t->dev.mask + 1);
  for (int b = 0; b < MT_HIST_BINS; ++b) out->probe_hist[b] = (int64_t)h.hist[b];
  out->device_error = h.error;
  return MT_OK;
}

int mt_export(mt_table* t, uint64_t* keys, int32_t* rows, int64_t capacity, int64_t* count, mt_stream stream) {
  if (t == nullptr || count == nullptr || capacity < 0) return MT_EINVAL;
  if (capacity > 0 && (keys == nullptr || rows == nullptr)) return MT_EINVAL;
  cudaStream_t s = as_stream(stream);
  if (mt::launch_export(t->dev, reinterpret_cast<unsigned long long*>(keys), rows, capacity, s) != cudaSuccess)
    return MT_ECUDA;
  long long c = 0;
  if (cudaMemcpyAsync(&c, &t->dev.hdr->export_count, sizeof(c), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MT_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MT_ECUDA;
  *count = c;
  return MT_OK;
}

int mt_read_rows(const mt_table* t, const int32_t* rows, int64_t n, float* emb, float* m, float* v,
                 mt_stream stream) {
  if (t == nullptr || n < 0 || (n > 0 && rows == nullptr)) return MT_EINVAL;
  return cuda_status(mt::launch_read_rows(t->dev, rows, n, emb, m, v, as_stream(stream)));
}

size_t mt_import_workspace_bytes(int64_t n) {
  if (n < 0) return 0;
  return align_up((size_t)(n > 0 ? n : 1) * 4, 256);
}

int mt_import(mt_table* t, const uint64_t* keys, int64_t n, const float* emb, const float* m, const float* v,
              void* ws, size_t ws_bytes, mt_stream stream) {
  if (t == nullptr || n < 0) return MT_EINVAL;
  if (n > 0 && (keys == nullptr || emb == nullptr || m == nullptr || v == nullptr || !aligned(keys, 8)))
    return MT_EINVAL;
  if (n > 0 && (ws == nullptr || ws_bytes < mt_import_workspace_bytes(n) || !aligned(ws, 256))) return MT_ENOSPACE;
  return cuda_status(mt::launch_import(t->dev, reinterpret_cast<const unsigned long long*>(keys), n, emb, m, v,
                                       static_cast<int32_t*>(ws), as_stream(stream)));
}

int mt_get_adam_state(mt_table* t, int64_t* step, double* b1pow, double* b2pow, mt_stream stream) {
  if (t == nullptr || step == nullptr || b1pow == nullptr || b2pow == nullptr) return MT_EINVAL;
  cudaStream_t s = as_stream(stream);
  long long st = 0;
  double p[2] = {0.0, 0.0};
  if (cudaMemcpyAsync(&st, &t->dev.hdr->step, sizeof(st), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MT_ECUDA;
  if (cudaMemcpyAsync(p, &t->dev.hdr->b1pow, sizeof(p), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MT_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MT_ECUDA;
  *step = st;
  *b1pow = p[0];
  *b2pow = p[1];
  return MT_OK;
}

int mt_set_adam_state(mt_table* t, int64_t step, double b1pow, double b2pow, mt_stream stream) {
  // The state must be one that backward calls could have produced: before the first step both
  // powers are exactly 1; after it both lie in [0, 1), so every bias correction 1 - b^t is positive.
  if (step < 0) return MT_EINVAL;
  if (step == 0 && !(b1pow == 1.0 && b2pow == 1.0)) return MT_EINVAL;
  if (step > 0 && !(b1pow >= 0.0 && b1pow < 1.0 && b2pow >= 0.0 && b2pow < 1.0)) return MT_EINVAL;
  if (t == nullptr) return MT_EINVAL;
  cudaStream_t s = as_stream(stream);
  const long long st = step;
  const double p[2] = {b1pow, b2pow};
  if (cudaMemcpyAsync(&t->dev.hdr->step, &st, sizeof(st), cudaMemcpyHostToDevice, s) != cudaSuccess) return MT_ECUDA;
  if (cudaMemcpyAsync(&t->dev.hdr->b1pow, p, sizeof(p), cudaMemcpyHostToDevice, s) != cudaSuccess) return MT_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MT_ECUDA;  // the host values above go out of scope
  t->step = step;
  return MT_OK;
}

int mt_get_error(mt_table* t, int32_t* device_error, int clear, mt_stream stream) {
  if (t == nullptr || device_error == nullptr) return MT_EINVAL;
  cudaStream_t s = as_stream(stream);
  int32_t e = 0;
  if (cudaMemcpyAsync(&e, &t->dev.hdr->error, sizeof(e), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MT_ECUDA;
  if (clear && cudaMemsetAsync(&t->dev.hdr->error, 0, sizeof(int32_t), s) != cudaSuccess) return MT_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MT_ECUDA;
  *device_error = e;
  return MT_OK;
}

int64_t mt_step(const mt_table* t) { return t == nullptr ? -1 : t->step; }

}  // extern "C"
