// CPU oracle for the merged dynamic embedding table -- TEST INFRASTRUCTURE ONLY.
//
// Only the tests, the smoke check and the benchmark's CPU-baseline leg may load
// this library.  It shares no code, header or constant table with the CUDA
// path, and it is deliberately plain and single-threaded: a std::unordered_map
// is the table, dedup is a map walk in position order, the gradient sum is a
// double accumulation in position order and Adam is a serial fp32 loop.
//
// What each part follows:
//  * Merged keys -- feature tables merged into one (MTGenRec, TL;DR and abstract):
//    several feature tables share one hash table.  A key is
//    (table_id << 56) | id with table_id in [0, 254]; table_id 255 holds the
//    two sentinels (EMPTY = 2^64-1, TOMBSTONE = 2^64-2).
//  * Unique + inverse -- ID deduplication in two stages (MTGenRec, TL;DR);
//    the IDs a lookup exchanges hold no duplicates on either side of the
//    exchange (MTGR, section 5, Embedding Lookup).  The unique list is in first-occurrence order, the
//    semantics of the Unique operator (Meituan TensorFlow article, section 3.6).
//  * Dynamic table whose keys are inserted and deleted while training runs
//    (MTGenRec, abstract; MTGR section 5, Embedding Management: each key
//    leads to its embedding and to bookkeeping data).
//  * Probe sequence h_t = (h0 + t*S) mod M, M = 2^n, S odd (MTGenRec,
//    Theorem 1) -- used only by the shadow open-addressing simulator that
//    produces occupancy statistics; the table itself is an unordered_map.
//  * Adam -- named in the Meituan TensorFlow article, section 3.2, with
//    beta-power accumulators shared by all parameters: Kingma & Ba's update
//    with bias correction by one step counter per table.
//  * Row initialisation (the pages are silent): Philox4x64-10 (Salmon, Moraes,
//    Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11) keyed by
//    (merged key, init seed).
//
// Build with -ffp-contract=off so every float operation rounds once.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <unordered_map>
#include <utility>
#include <vector>

namespace {

const uint64_t kEmpty = ~0ull;        // never a valid key (table_id 255)
const uint64_t kTomb = ~0ull - 1ull;  // never a valid key (table_id 255)
const uint64_t kIdLimit = 1ull << 56;

enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { ORC_OK = 0, ORC_EINVAL = -1, ORC_EFULL = -3, ORC_EKEY = -4 };

// ---- Philox4x64-10 ----------------------------------------------------------
// One round: the 128-bit products of words 0 and 2 with the two round
// multipliers are split into high and low halves; the new words are
// (hi(x2*M1) ^ x1 ^ k0, lo(x2*M1), hi(x0*M0) ^ x3 ^ k1, lo(x0*M0)).  Between
// rounds the key advances by the two Weyl constants.
void philox4x64(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]) {
  uint64_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint64_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += 0x9E3779B97F4A7C15ull;
      k1 += 0xBB67AE8584CAA73Bull;
    }
    unsigned __int128 p0 = (unsigned __int128)0xD2E7470EE14C6C93ull * x0;
    unsigned __int128 p1 = (unsigned __int128)0xCA5A826395121157ull * x2;
    uint64_t y0 = (uint64_t)(p1 >> 64) ^ x1 ^ k0;
    uint64_t y1 = (uint64_t)p1;
    uint64_t y2 = (uint64_t)(p0 >> 64) ^ x3 ^ k1;
    uint64_t y3 = (uint64_t)p0;
    x0 = y0; x1 = y1; x2 = y2; x3 = y3;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

// fp32 -> bf16 by round-to-nearest-even on the bit pattern.
uint16_t bf16_bits(float x) {
  uint32_t u;
  std::memcpy(&u, &x, 4);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0;  // NaN
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

float bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float x;
  std::memcpy(&x, &u, 4);
  return x;
}

// The value a row element holds in storage of the given dtype.
float store_round(float x, int dtype) { return dtype == ORC_BF16 ? bf16_value(bf16_bits(x)) : x; }

// Initial value of column j of the row of `key`.  Each 64-bit word of
// Philox4x64-10(counter = (j/8, 0, 0, 0), key = (key, seed)) serves two
// columns: word (j/2)%4 gives a 24-bit integer q from its bits 63..40 for an
// even j and from its bits 39..16 for an odd j; (2q - 2^24) / 2^24 is exact
// in fp32 and lies in [-1, 1); one multiply by `scale` is the only rounding.
float init_value(uint64_t key, uint64_t seed, float scale, uint32_t j) {
  uint64_t k[2] = {key, seed};
  uint64_t c[4] = {(uint64_t)(j / 8u), 0, 0, 0};
  uint64_t w[4];
  philox4x64(c, k, w);
  const uint64_t word = w[(j / 2u) % 4u];
  int32_t q = (int32_t)((j % 2u == 0u ? word >> 40 : word >> 16) & 0xFFFFFFu);
  float unit = (float)(2 * q - (1 << 24)) * (1.0f / 16777216.0f);
  return unit * scale;
}

// splitmix64 output mixer (Steele, Lea, Flood, OOPSLA 2014); the top n bits
// of the mixed key are the home slot h0.
uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t home_slot(uint64_t key, uint64_t seed, uint32_t n) {
  if (n == 0) return 0;
  return mix64(key ^ seed) >> (64 - n);
}

// A row of the table.  `touched` is false until the first optimizer step; an
// untouched row still equals init(key) with m = v = 0 and is not stored, so a
// table of tens of millions of keys costs the oracle little memory.
struct Row {
  bool touched = false;
  std::vector<float> emb, m, v;
};

// Serial open-addressing table with the probe sequence of Theorem 1.  It
// records the probe index at which each live key was placed.  Used only for
// occupancy statistics.
struct Simulator {
  uint32_t n;
  uint64_t M, S, seed, max_probes;
  std::vector<uint64_t> slot;
  std::vector<uint32_t> placed_t;

  Simulator(uint32_t n_, uint64_t S_, uint64_t seed_, uint64_t max_probes_)
      : n(n_), M(1ull << n_), S(S_ & ((1ull << n_) - 1)), seed(seed_),
        max_probes(max_probes_ ? max_probes_ : (1ull << n_)), slot(M, kEmpty), placed_t(M, 0) {}

  uint64_t at(uint64_t h0, uint64_t t) const { return (h0 + t * S) % M; }

  // The slot holding key, or -1.  Tombstones are passed over; an EMPTY slot
  // ends the chain.
  int64_t find(uint64_t key) const {
    uint64_t h0 = home_slot(key, seed, n);
    for (uint64_t t = 0; t < max_probes; ++t) {
      uint64_t s = at(h0, t);
      if (slot[s] == key) return (int64_t)s;
      if (slot[s] == kEmpty) return -1;
    }
    return -1;
  }

  // Insert an absent key at the first EMPTY-or-TOMBSTONE slot of its chain.
  int insert(uint64_t key) {
    if (find(key) >= 0) return ORC_OK;
    uint64_t h0 = home_slot(key, seed, n);
    for (uint64_t t = 0; t < max_probes; ++t) {
      uint64_t s = at(h0, t);
      if (slot[s] == kEmpty || slot[s] == kTomb) {
        slot[s] = key;
        placed_t[s] = (uint32_t)t;
        return ORC_OK;
      }
    }
    return ORC_EFULL;
  }

  bool erase(uint64_t key) {
    int64_t s = find(key);
    if (s < 0) return false;
    slot[s] = kTomb;
    return true;
  }
};

struct Table {
  uint32_t n, dim;
  int dtype;
  uint64_t S, hash_seed, init_seed, max_probes;
  float init_scale;
  int64_t num_rows;
  int64_t step = 0;
  double b1pow = 1.0, b2pow = 1.0;  // beta-power accumulators b1^t, b2^t
  int error = 0;
  std::unordered_map<uint64_t, Row> rows;
  Simulator* sim = nullptr;
  // the last lookup, for backward
  std::vector<uint64_t> last_uniq;
  std::vector<int32_t> last_inverse;

  float emb_at(uint64_t key, const Row& r, uint32_t j) const {
    return r.touched ? r.emb[j] : store_round(init_value(key, init_seed, init_scale, j), dtype);
  }
  void touch(uint64_t key, Row& r) const {
    if (r.touched) return;
    r.touched = true;
    r.emb.resize(dim);
    r.m.assign(dim, 0.0f);
    r.v.assign(dim, 0.0f);
    for (uint32_t j = 0; j < dim; ++j) r.emb[j] = store_round(init_value(key, init_seed, init_scale, j), dtype);
  }
};

void latch(Table* t, int code) {
  if (t->error == 0) t->error = code;
}

}  // namespace

extern "C" {

void orc_philox4x64_10(const uint64_t* ctr, const uint64_t* key, uint64_t* out) { philox4x64(ctr, key, out); }

void orc_init_row(uint64_t key, uint64_t seed, float scale, uint32_t dim, int dtype, float* out) {
  for (uint32_t j = 0; j < dim; ++j) out[j] = store_round(init_value(key, seed, scale, j), dtype);
}

uint16_t orc_bf16_bits(float x) { return bf16_bits(x); }

uint64_t orc_home_slot(uint64_t key, uint64_t seed, uint32_t n) { return home_slot(key, seed, n); }

// keys[i] = (table_ids[f] << 56) | ids[i] for feat_offsets[f] <= i < feat_offsets[f+1].
// valid[i] = 0 when ids[i] is negative or >= 2^56, when table_ids[f] is 255,
// or when position i lies in no segment.
void orc_encode(const int64_t* ids, int64_t n, const int64_t* feat_offsets, const uint8_t* table_ids, int F,
                uint64_t* keys, uint8_t* valid) {
  for (int64_t i = 0; i < n; ++i) {
    keys[i] = kEmpty;
    valid[i] = 0;
  }
  for (int f = 0; f < F; ++f) {
    for (int64_t i = std::max<int64_t>(feat_offsets[f], 0); i < feat_offsets[f + 1] && i < n; ++i) {
      if (ids[i] < 0 || (uint64_t)ids[i] >= kIdLimit || table_ids[f] == 255) continue;
      keys[i] = ((uint64_t)table_ids[f] << 56) | (uint64_t)ids[i];
      valid[i] = 1;
    }
  }
}

// First-occurrence unique: walk positions in order; the first time a key is
// seen it is appended to uniq; inverse[i] is the index of key i in uniq and
// counts[u] the number of positions holding uniq[u] (counts nullable).
// Invalid positions get inverse -1.
int64_t orc_unique(const uint64_t* keys, const uint8_t* valid, int64_t n, uint64_t* uniq, int32_t* inverse,
                   int32_t* counts) {
  std::unordered_map<uint64_t, int32_t> seen;
  seen.reserve((size_t)n * 2 + 1);
  int64_t U = 0;
  for (int64_t i = 0; i < n; ++i) {
    if (!valid[i]) {
      inverse[i] = -1;
      continue;
    }
    auto it = seen.find(keys[i]);
    if (it == seen.end()) {
      seen.emplace(keys[i], (int32_t)U);
      uniq[U] = keys[i];
      if (counts) counts[U] = 0;
      inverse[i] = (int32_t)U;
      ++U;
    } else {
      inverse[i] = it->second;
    }
    if (counts) counts[inverse[i]] += 1;
  }
  return U;
}

// The same result by sorting: sort (key, position) pairs, keep the smallest
// position of each key, then order the distinct keys by that position.
int64_t orc_unique_sort(const uint64_t* keys, const uint8_t* valid, int64_t n, uint64_t* uniq, int32_t* inverse) {
  std::vector<std::pair<uint64_t, int64_t>> kp;
  kp.reserve((size_t)n);
  for (int64_t i = 0; i < n; ++i)
    if (valid[i]) kp.emplace_back(keys[i], i);
  std::sort(kp.begin(), kp.end());
  // runs of equal keys: [run_begin, run_end) in kp, first position = kp[run_begin].second
  std::vector<std::pair<int64_t, size_t>> firsts;  // (first position, run begin)
  for (size_t a = 0; a < kp.size();) {
    size_t b = a;
    while (b < kp.size() && kp[b].first == kp[a].first) ++b;
    firsts.emplace_back(kp[a].second, a);
    a = b;
  }
  std::sort(firsts.begin(), firsts.end());
  for (int64_t i = 0; i < n; ++i) inverse[i] = -1;
  for (size_t u = 0; u < firsts.size(); ++u) {
    size_t a = firsts[u].second;
    uniq[u] = kp[a].first;
    for (size_t c = a; c < kp.size() && kp[c].first == kp[a].first; ++c) inverse[kp[c].second] = (int32_t)u;
  }
  return (int64_t)firsts.size();
}

void* orc_table_new(uint32_t log2_slots, uint32_t dim, int row_dtype, uint64_t probe_step, uint64_t hash_seed,
                    uint64_t init_seed, float init_scale, uint64_t max_probes, int64_t num_rows, int simulate) {
  if (log2_slots > 31 || dim == 0 || (row_dtype != ORC_F32 && row_dtype != ORC_BF16)) return nullptr;
  uint64_t M = 1ull << log2_slots;
  if (log2_slots > 0 && (probe_step % M) % 2 == 0) return nullptr;  // Theorem 1: the step must be odd
  Table* t = new Table();
  t->n = log2_slots;
  t->dim = dim;
  t->dtype = row_dtype;
  t->S = probe_step;
  t->hash_seed = hash_seed;
  t->init_seed = init_seed;
  t->init_scale = init_scale;
  t->max_probes = max_probes;
  t->num_rows = num_rows > 0 ? num_rows : (int64_t)M;
  if (simulate) t->sim = new Simulator(log2_slots, probe_step, hash_seed, max_probes);
  return t;
}

void orc_table_free(void* h) {
  Table* t = (Table*)h;
  delete t->sim;
  delete t;
}

// Lookup of one batch: encode, deduplicate (first occurrence), find each
// unique key, insert the absent ones when insert_missing (in first-occurrence
// order; a fresh row holds init(key) with m = v = 0), and gather one row per
// position into out_rows ([n, dim] floats holding the stored values; zeros for
// invalid positions and absent keys; nullable).
// present[u] = 1 when unique key u has a row after the call; counts[u] = its
// number of positions.  Returns U.
int64_t orc_lookup(void* h, const int64_t* ids, int64_t n, const int64_t* feat_offsets, const uint8_t* table_ids,
                   int F, int insert_missing, float* out_rows, uint64_t* uniq, int32_t* inverse, int32_t* counts,
                   uint8_t* present) {
  Table* t = (Table*)h;
  std::vector<uint64_t> keys((size_t)n);
  std::vector<uint8_t> valid((size_t)n);
  orc_encode(ids, n, feat_offsets, table_ids, F, keys.data(), valid.data());
  for (int64_t i = 0; i < n; ++i)
    if (!valid[i]) latch(t, ORC_EKEY);
  int64_t U = orc_unique(keys.data(), valid.data(), n, uniq, inverse, counts);
  std::vector<const Row*> row_of(U, nullptr);
  for (int64_t u = 0; u < U; ++u) {
    auto it = t->rows.find(uniq[u]);
    if (it == t->rows.end() && insert_missing) {
      bool ok = (int64_t)t->rows.size() < t->num_rows;
      if (ok && t->sim) ok = t->sim->insert(uniq[u]) == ORC_OK;
      if (ok) {
        it = t->rows.emplace(uniq[u], Row()).first;
      } else {
        latch(t, ORC_EFULL);
      }
    }
    if (it != t->rows.end()) row_of[u] = &it->second;
    present[u] = row_of[u] != nullptr;
  }
  if (out_rows) {
    for (int64_t i = 0; i < n; ++i) {
      float* o = out_rows + (size_t)i * t->dim;
      const Row* r = inverse[i] >= 0 ? row_of[inverse[i]] : nullptr;
      for (uint32_t j = 0; j < t->dim; ++j) o[j] = r ? t->emb_at(uniq[inverse[i]], *r, j) : 0.0f;
    }
  }
  t->last_uniq.assign(uniq, uniq + U);
  t->last_inverse.assign(inverse, inverse + n);
  return U;
}

// Backward of the last lookup: per-unique gradient sum (double accumulation
// in position order, rounded once to fp32), then one Adam step on every
// present unique row.  The step counter is global to the table and advances
// once per call.  grads: [n, dim], fp32 (dtype 0) or bf16 bit patterns
// (dtype 1).  gsum_out (nullable): [U, dim] fp32.
int orc_backward_adam(void* h, const void* grads, int grad_dtype, float lr, float beta1, float beta2, float eps,
                      float* gsum_out) {
  Table* t = (Table*)h;
  const int64_t U = (int64_t)t->last_uniq.size();
  const int64_t n = (int64_t)t->last_inverse.size();
  const uint32_t d = t->dim;
  std::vector<double> acc((size_t)U * d, 0.0);
  for (int64_t i = 0; i < n; ++i) {
    int32_t u = t->last_inverse[i];
    if (u < 0) continue;
    for (uint32_t j = 0; j < d; ++j) {
      float g = grad_dtype == ORC_BF16 ? bf16_value(((const uint16_t*)grads)[(size_t)i * d + j])
                                       : ((const float*)grads)[(size_t)i * d + j];
      acc[(size_t)u * d + j] += (double)g;
    }
  }
  t->step += 1;
  // Optimizer constants: computed in double, each rounded once to fp32.
  // Kingma & Ba's m_hat / (sqrt(v_hat) + eps) with m_hat = m / (1 - b1^t) and
  // sqrt(v_hat) = sqrt(v) / sqrt(1 - b2^t): the two bias corrections enter as
  // the per-step scalars step_size = lr / (1 - b1^t) and
  // inv_sqrt_bc2 = 1 / sqrt(1 - b2^t).  b1^t and b2^t are the article's
  // beta-power accumulators (section 3.2): one multiply by the step's beta
  // each step, starting from 1.
  const float omb1 = (float)(1.0 - (double)beta1);
  const float omb2 = (float)(1.0 - (double)beta2);
  t->b1pow *= (double)beta1;
  t->b2pow *= (double)beta2;
  const double bc1 = 1.0 - t->b1pow;
  const double bc2 = 1.0 - t->b2pow;
  const float step_size = (float)((double)lr / bc1);
  const float inv_sqrt_bc2 = (float)(1.0 / std::sqrt(bc2));
  for (int64_t u = 0; u < U; ++u) {
    auto it = t->rows.find(t->last_uniq[u]);
    if (it != t->rows.end()) t->touch(t->last_uniq[u], it->second);
    for (uint32_t j = 0; j < d; ++j) {
      float g = (float)acc[(size_t)u * d + j];
      if (gsum_out) gsum_out[(size_t)u * d + j] = g;
      if (it == t->rows.end()) continue;
      Row& r = it->second;
      float m = beta1 * r.m[j] + omb1 * g;
      float v = beta2 * r.v[j] + omb2 * (g * g);
      float den = std::sqrt(v) * inv_sqrt_bc2 + eps;
      float upd = step_size * (m / den);
      r.m[j] = m;
      r.v[j] = v;
      r.emb[j] = store_round(r.emb[j] - upd, t->dtype);
    }
  }
  return ORC_OK;
}

// ---- pooled embeddings of jagged bags ---------------------------------------
// A bag is a run of consecutive positions [bag_offsets[b], bag_offsets[b+1]):
// in the jagged batches of MTGR (section 5, Load Balance: user sequences of
// very different lengths) one bag is one user's tokens of one feature.  The
// bag's pooled embedding is the sum (mode 0) or the mean (mode 1) of the rows
// of its positions.  Positions outside every bag are in no output.

// out[b] = sum over the bag's positions of the (stored) row of the position's
// key after the last lookup, accumulated in double in position order; mode 1
// divides the double sum by the bag's length; each value rounded once to
// fp32.  Invalid positions and absent keys add zero rows.  Empty bags give
// zeros.  Returns ORC_EINVAL (and writes nothing) for offsets that decrease
// or leave [0, n].
int orc_pool_forward(void* h, const int64_t* bag_offsets, int64_t B, int mode, float* out) {
  Table* t = (Table*)h;
  const int64_t n = (int64_t)t->last_inverse.size();
  const uint32_t d = t->dim;
  for (int64_t b = 0; b < B; ++b)
    if (bag_offsets[b] < 0 || bag_offsets[b] > bag_offsets[b + 1] || bag_offsets[b + 1] > n) return ORC_EINVAL;
  std::vector<double> acc(d);
  for (int64_t b = 0; b < B; ++b) {
    std::fill(acc.begin(), acc.end(), 0.0);
    for (int64_t i = bag_offsets[b]; i < bag_offsets[b + 1]; ++i) {
      const int32_t u = t->last_inverse[i];
      if (u < 0) continue;
      auto it = t->rows.find(t->last_uniq[u]);
      if (it == t->rows.end()) continue;
      for (uint32_t j = 0; j < d; ++j) acc[j] += (double)t->emb_at(t->last_uniq[u], it->second, j);
    }
    const int64_t len = bag_offsets[b + 1] - bag_offsets[b];
    for (uint32_t j = 0; j < d; ++j)
      out[(size_t)b * d + j] = (float)(mode == 1 && len > 0 ? acc[j] / (double)len : acc[j]);
  }
  return ORC_OK;
}

// The backward of pooling followed by the table's backward: every position
// of bag b receives the bag's gradient dpooled[b] (mode 0) or, for the mean,
// dpooled[b] * s_b rounded once to fp32, with s_b = 1 / len_b rounded once to
// fp32 (mode 1); positions outside every bag receive zero.  Then exactly
// orc_backward_adam on those per-position gradients.
int orc_backward_adam_pooled(void* h, const int64_t* bag_offsets, int64_t B, int mode, const float* dpooled,
                             float lr, float beta1, float beta2, float eps, float* gsum_out) {
  Table* t = (Table*)h;
  const int64_t n = (int64_t)t->last_inverse.size();
  const uint32_t d = t->dim;
  for (int64_t b = 0; b < B; ++b)
    if (bag_offsets[b] < 0 || bag_offsets[b] > bag_offsets[b + 1] || bag_offsets[b + 1] > n) return ORC_EINVAL;
  std::vector<float> grads((size_t)n * d, 0.0f);
  for (int64_t b = 0; b < B; ++b) {
    const int64_t len = bag_offsets[b + 1] - bag_offsets[b];
    const float s = (float)(1.0 / (double)(len > 0 ? len : 1));
    for (int64_t i = bag_offsets[b]; i < bag_offsets[b + 1]; ++i)
      for (uint32_t j = 0; j < d; ++j) {
        const float g = dpooled[(size_t)b * d + j];
        grads[(size_t)i * d + j] = mode == 1 ? g * s : g;
      }
  }
  return orc_backward_adam(h, grads.data(), ORC_F32, lr, beta1, beta2, eps, gsum_out);
}

// Erase a batch of merged keys.  found[i] = 1 when keys[i] was present before
// the call (every duplicate of a present key reports 1).  A later re-insert
// of an erased key starts again from init(key) with m = v = 0.
void orc_erase(void* h, const uint64_t* keys, int64_t n, uint8_t* found) {
  Table* t = (Table*)h;
  for (int64_t i = 0; i < n; ++i) found[i] = t->rows.count(keys[i]) ? 1 : 0;
  for (int64_t i = 0; i < n; ++i) {
    if (t->rows.erase(keys[i]) && t->sim) t->sim->erase(keys[i]);
  }
}

// Insert keys without a lookup batch (prefill): each absent key gets a fresh
// row.  Returns the number of keys inserted.
int64_t orc_insert_keys(void* h, const uint64_t* keys, int64_t n) {
  Table* t = (Table*)h;
  int64_t added = 0;
  for (int64_t i = 0; i < n; ++i) {
    if (t->rows.count(keys[i])) continue;
    bool ok = (int64_t)t->rows.size() < t->num_rows;
    if (ok && t->sim) ok = t->sim->insert(keys[i]) == ORC_OK;
    if (!ok) {
      latch(t, ORC_EFULL);
      continue;
    }
    t->rows.emplace(keys[i], Row());
    ++added;
  }
  return added;
}

// Copy the stored row of key (emb as floats, m, v; each nullable).  Returns 1
// if the key is present.
int orc_get_row(void* h, uint64_t key, float* emb, float* m, float* v) {
  Table* t = (Table*)h;
  auto it = t->rows.find(key);
  if (it == t->rows.end()) return 0;
  for (uint32_t j = 0; j < t->dim; ++j) {
    if (emb) emb[j] = t->emb_at(key, it->second, j);
    if (m) m[j] = it->second.touched ? it->second.m[j] : 0.0f;
    if (v) v[j] = it->second.touched ? it->second.v[j] : 0.0f;
  }
  return 1;
}

// orc_get_row for n keys: rows [n, dim] each (nullable); present[i] = 1 when
// keys[i] is in the table (absent keys give zero rows).
void orc_get_rows(void* h, const uint64_t* keys, int64_t n, float* emb, float* m, float* v, uint8_t* present) {
  Table* t = (Table*)h;
  const uint32_t d = t->dim;
  for (int64_t i = 0; i < n; ++i) {
    int ok = orc_get_row(h, keys[i], emb ? emb + (size_t)i * d : nullptr, m ? m + (size_t)i * d : nullptr,
                         v ? v + (size_t)i * d : nullptr);
    if (!ok) {
      for (uint32_t j = 0; j < d; ++j) {
        if (emb) emb[(size_t)i * d + j] = 0.0f;
        if (m) m[(size_t)i * d + j] = 0.0f;
        if (v) v[(size_t)i * d + j] = 0.0f;
      }
    }
    if (present) present[i] = (uint8_t)ok;
  }
}

int64_t orc_live_count(void* h) { return (int64_t)((Table*)h)->rows.size(); }

int64_t orc_live_keys(void* h, uint64_t* out, int64_t cap) {
  Table* t = (Table*)h;
  int64_t k = 0;
  for (auto& kv : t->rows) {
    if (k < cap) out[k] = kv.first;
    ++k;
  }
  return k;
}

int64_t orc_step(void* h) { return ((Table*)h)->step; }
int orc_error(void* h) { return ((Table*)h)->error; }

// Occupancy of the shadow simulator: live keys, tombstones, a histogram of
// the probe index t at which each live key sits (bins 0..62; bin 63 holds
// t >= 63) and the total displacement (sum of t).  Returns -1 when the table
// was created without the simulator.
int orc_sim_stats(void* h, int64_t* live, int64_t* tombs, int64_t* hist64, int64_t* total_displacement) {
  Table* t = (Table*)h;
  if (!t->sim) return -1;
  int64_t L = 0, T = 0, D = 0;
  for (int b = 0; b < 64; ++b) hist64[b] = 0;
  for (uint64_t s = 0; s < t->sim->M; ++s) {
    uint64_t k = t->sim->slot[s];
    if (k == kTomb) {
      ++T;
    } else if (k != kEmpty) {
      ++L;
      uint32_t pt = t->sim->placed_t[s];
      D += pt;
      ++hist64[pt < 63 ? pt : 63];
    }
  }
  *live = L;
  *tombs = T;
  *total_displacement = D;
  return 0;
}

// Occupied-slot bitmap of the shadow simulator (1 byte per slot: 0 empty,
// 1 live, 2 tombstone).
int orc_sim_occupancy(void* h, uint8_t* out) {
  Table* t = (Table*)h;
  if (!t->sim) return -1;
  for (uint64_t s = 0; s < t->sim->M; ++s) {
    uint64_t k = t->sim->slot[s];
    out[s] = k == kEmpty ? 0 : (k == kTomb ? 2 : 1);
  }
  return 0;
}

// Raw simulator access for the Theorem 1 and probing tests.
void* orc_sim_new(uint32_t log2_slots, uint64_t probe_step, uint64_t hash_seed, uint64_t max_probes) {
  return new Simulator(log2_slots, probe_step, hash_seed, max_probes);
}
void orc_sim_free(void* s) { delete (Simulator*)s; }
int orc_sim_insert(void* s, uint64_t key) { return ((Simulator*)s)->insert(key); }
int orc_sim_erase(void* s, uint64_t key) { return ((Simulator*)s)->erase(key) ? 1 : 0; }
int64_t orc_sim_find(void* s, uint64_t key) { return ((Simulator*)s)->find(key); }
// The probe index t at which a live key sits, or -1.
int64_t orc_sim_placed(void* s, uint64_t key) {
  Simulator* sim = (Simulator*)s;
  int64_t slot = sim->find(key);
  return slot < 0 ? -1 : (int64_t)sim->placed_t[slot];
}
// The first `count` slots of the probe sequence from home slot h0.
void orc_sim_sequence(void* s, uint64_t h0, uint64_t count, uint64_t* out) {
  Simulator* sim = (Simulator*)s;
  for (uint64_t t = 0; t < count; ++t) out[t] = sim->at(h0, t);
}
// Occupancy of a raw simulator (same coding as orc_sim_occupancy) and its
// total displacement.
int64_t orc_sim_raw_occupancy(void* s, uint8_t* out) {
  Simulator* sim = (Simulator*)s;
  int64_t D = 0;
  for (uint64_t k = 0; k < sim->M; ++k) {
    uint64_t key = sim->slot[k];
    if (out) out[k] = key == kEmpty ? 0 : (key == kTomb ? 2 : 1);
    if (key != kEmpty && key != kTomb) D += sim->placed_t[k];
  }
  return D;
}

}  // extern "C"
