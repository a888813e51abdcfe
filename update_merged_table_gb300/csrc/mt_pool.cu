// Pooled embeddings of jagged bags and the pooled backward.
//
// A bag is a run of consecutive positions [bag_offsets[b], bag_offsets[b+1])
// of a lookup batch: in the jagged sequence batches of "MTGR" section 5 (Load
// Balance: user behaviour sequences of very different lengths) one bag is one
// user's tokens of one feature.  The bag's pooled embedding is the sum (or the
// mean) of the rows of its positions' keys.  The backward hands every
// position its bag's gradient (times 1/len for the mean) and feeds the table's
// per-unique reduction and Adam directly: no per-position gradient rows are
// ever written.
//
// Kernels:
//  k_pool         a warp per chunk of kPoolChunk positions: the chunk's row
//                 indices fetched in one round, its first bag by a warp-wide
//                 multiway search of the offsets; each bag's positions split
//                 over the warp's sub-teams (one 16-byte vector of a row per
//                 lane), rows summed as exact fp32 pairs (TwoSum on the paired
//                 fp32 instructions, two columns each) and the sub-teams'
//                 pairs joined by TwoSums; a bag that lies inside one chunk is
//                 written at once, the pieces of a longer bag meet in an fp64
//                 accumulator.
//  k_pool_finish  bags split over chunks (and empty bags): rounded from the
//                 fp64 accumulator.
//  k_pos_bag      backward: the bag of every position (-1: in no bag).
//  k_pool_scale   backward of the mean: each bag's gradient times
//                 fp32(1/len), rounded once.
#include "mt_kernels.cuh"

namespace mt {

namespace {

constexpr int kPoolChunk = 128;                // positions per chunk (one warp)
constexpr int kPoolRows = kPoolChunk / 32;     // row indices each lane fetches per chunk
constexpr int kPoolUnroll = 4;                 // rows in flight per lane

// Round a bag's sum (or mean) from double to fp32 into out[b, col .. col + VEC).
template <int VEC>
__device__ __forceinline__ void store_pooled(const PoolParams& p, long long b, int col, const double* s, long long len) {
  float o[VEC];
#pragma unroll
  for (int j = 0; j < VEC; ++j) o[j] = (float)(p.mode == MT_POOL_MEAN && len > 0 ? s[j] / (double)len : s[j]);
  float4* dst = reinterpret_cast<float4*>(p.out + (size_t)b * p.T.dim + col);
#pragma unroll
  for (int q = 0; q < VEC / 4; ++q) dst[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
}

// The bag holding position x, searched by a whole team at once: the last b
// with bo[b] <= x (-1 when x lies before every bag; b may be >= B when it lies
// after all of them).  Each round the team's T lanes probe T points that cut
// the open range (lo, hi) into T + 1 parts, so about log_(T+1)(B) rounds.  The
// range shrinks every round and every probe lies in [0, B], also for offsets
// that decrease.
__device__ __forceinline__ long long bag_search(const long long* bo, long long B, long long x, int lt, int team,
                                                unsigned team_mask, int team_base) {
  const unsigned full = team == 32 ? kFull : (1u << team) - 1u;
  long long lo = -1, hi = B + 1;  // bo[lo] <= x < bo[hi] with bo[-1] = -inf, bo[B+1] = +inf
  while (hi - lo > 1) {
    const long long span = hi - lo;
    const long long m = lo + (span * (lt + 1)) / (team + 1);  // lo <= m < hi, non-decreasing in lt
    const bool le = m == lo || __ldg(&bo[m]) <= x;
    const unsigned bits = (__ballot_sync(team_mask, le) >> team_base) & full;
    const int k = bits == full ? team : __ffs(~bits) - 1;  // the first probe above x
    const long long nlo = lo + (span * k) / (team + 1);    // probe k - 1 (lo when k = 0)
    hi = k == team ? hi : lo + (span * (k + 1)) / (team + 1);
    lo = nlo;
  }
  return lo;
}

// A warp per chunk of kPoolChunk positions.  The warp fetches the chunk's
// row indices in one round (kPoolRows positions per lane, inverse and then
// unique_rows, into shared memory) while it searches for the chunk's first
// bag, then walks the bags that meet the chunk with a window of 32 offsets
// held one per lane.  A bag's positions in the chunk are split over the
// warp's S = 32 / team sub-teams (position q goes to sub-team q mod S), each
// lane adding one 16-byte vector of a row per position, kPoolUnroll rows in
// flight, as exact fp32 pairs (TwoSum on the paired instructions).  The
// sub-teams' pairs meet by a butterfly of TwoSums, and sub-team 0 writes the
// bag when the whole bag lies in the chunk, else adds it to the bag's fp64
// accumulator.  A pair's exact sum is rounded to fp32 by one fp32 add
// (correctly rounded); only the mean divides, in double.
template <int RD>
__global__ void __launch_bounds__(256, 4) k_pool(const PoolParams p) {
  constexpr int VEC = RD == MT_F32 ? 4 : 8;  // columns per lane: one 16-byte load of a row
  constexpr int NP = VEC / 2;                // column pairs per lane
  __shared__ int32_t s_row[256 / 32][kPoolChunk];  // per warp: the rows of its chunk (-1: nothing to add)
  const int lane = threadIdx.x & 31;
  const int team_shift = p.team_shift;
  const int team = 1 << team_shift;
  const int lt = lane & (team - 1);
  const int sub = lane >> team_shift;  // sub-team
  const int S = 32 >> team_shift;      // sub-teams per warp
  int32_t* my_row = s_row[threadIdx.x >> 5];
  // positions, bags and unique indices fit in int (the entry point admits n, B < 2^31)
  const int n = (int)p.n;
  const int B = (int)p.num_bags;
  const int U = (int)*p.num_unique;
  const int d = (int)p.T.dim;
  const int nchunks = (n + kPoolChunk - 1) / kPoolChunk;
  const int gw = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int nw = (int)((gridDim.x * blockDim.x) >> 5);
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  // a bag offset relative to the chunk start p0, clamped to [-1, kPoolChunk + 1]: the comparisons with
  // the chunk's positions [0, cnt) stay exact
  auto rel = [](long long x, int p0) -> int {
    const long long r = x - p0;
    return r < 0 ? -1 : (r > kPoolChunk ? kPoolChunk + 1 : (int)r);
  };
  // lane k's entry of the offsets window based at bag w: bo[w + k] relative to p0 (bo[-1] = -inf,
  // bo[i > B] = +inf)
  auto window = [&](int w, int p0) -> int {
    const int i = w + lane;
    return i < 0 ? -1 : (i <= B ? rel(__ldg(&p.bag_offsets[i]), p0) : kPoolChunk + 1);
  };

  for (int c = gw; c < nchunks; c += nw) {  // uniform per warp
    const int p0 = c * kPoolChunk;
    const int cnt = min(kPoolChunk, n - p0);
    int32_t inv[kPoolRows];
#pragma unroll
    for (int k = 0; k < kPoolRows; ++k) {
      const int q = k * 32 + lane;
      inv[k] = q < cnt ? __ldg(&p.inverse[p0 + q]) : -1;
    }
    int b = (int)bag_search(p.bag_offsets, B, p0, lane, 32, kFull, 0);  // the chunk's first bag (-1: none yet)
#pragma unroll
    for (int k = 0; k < kPoolRows; ++k) {
      const int q = k * 32 + lane;
      if (q < cnt) my_row[q] = (inv[k] >= 0 && inv[k] < U) ? __ldg(&p.unique_rows[inv[k]]) : -1;
    }
    int w0 = b;
    int win = window(w0, p0);
    __syncwarp();
    // bag b covers the chunk's positions [qs, qe); b = -1 holds the positions before the first bag
    for (int qs = 0; qs < cnt && b < B; ++b) {
      if (b + 1 - w0 > 31) {  // the window is used up: the next 32 offsets
        w0 = b;
        win = window(w0, p0);
      }
      const int rs = __shfl_sync(kFull, win, b - w0);      // start of bag b, chunk-relative
      const int re = __shfl_sync(kFull, win, b + 1 - w0);  // its end
      const int qe = min(max(re, qs), cnt);
      if (b >= 0 && qe > qs) {
        const bool whole = rs >= 0 && re <= cnt && re > rs;  // the whole bag lies in this chunk
        const double len = (double)(re - rs);
        for (int c0 = 0; c0 < d; c0 += team * VEC) {
          const int col = c0 + lt * VEC;
          const bool active = col < d;
          f32x2 hi[NP], lo[NP];
#pragma unroll
          for (int j = 0; j < NP; ++j) hi[j] = lo[j] = 0ull;
          for (int q0 = qs + sub; q0 < qe; q0 += S * kPoolUnroll) {
            uint4 raw[kPoolUnroll];  // every load of the round issued before the first add
#pragma unroll
            for (int r = 0; r < kPoolUnroll; ++r) {
              const int q = q0 + r * S;
              const int32_t row = q < qe ? my_row[q] : -1;
              raw[r] = active && row >= 0 ? __ldg(reinterpret_cast<const uint4*>(row_ptr(p.T, row) + (size_t)col *
                                                                                  (RD == MT_F32 ? 4 : 2)))
                                          : zero;  // adding zero leaves a pair exactly as it is
            }
#pragma unroll
            for (int r = 0; r < kPoolUnroll; ++r) {
              const uint32_t w[4] = {raw[r].x, raw[r].y, raw[r].z, raw[r].w};
#pragma unroll
              for (int j = 0; j < NP; ++j) {
                const f32x2 x = RD == MT_F32 ? pk(__uint_as_float(w[2 * j]), __uint_as_float(w[2 * j + 1]))
                                             : bf16x2_to_f32x2(w[j]);
                f32x2 s, e;
                two_sum(hi[j], x, s, e);
                hi[j] = s;
                lo[j] = add2(lo[j], e);
              }
            }
          }
          // the sub-teams' pairs meet: lane l and lane l ^ o hold the same columns
          for (int o = team; o < 32; o <<= 1) {
#pragma unroll
            for (int j = 0; j < NP; ++j) {
              const f32x2 oh = __shfl_xor_sync(kFull, hi[j], o), ol = __shfl_xor_sync(kFull, lo[j], o);
              f32x2 s, e;
              two_sum(hi[j], oh, s, e);
              hi[j] = s;
              lo[j] = add2(add2(lo[j], ol), e);
            }
          }
          if (sub == 0 && active) {
#pragma unroll
            for (int j = 0; j < NP; ++j) {
              const float2 h = upk(hi[j]), l = upk(lo[j]);
              if (whole && p.mode != MT_POOL_MEAN) {  // the exact sum h + l, rounded once
                *reinterpret_cast<float2*>(p.out + (size_t)b * d + col + 2 * j) =
                    make_float2(__fadd_rn(h.x, l.x), __fadd_rn(h.y, l.y));
                continue;
              }
              const double s0 = (double)h.x + (double)l.x, s1 = (double)h.y + (double)l.y;
              if (whole) {
                *reinterpret_cast<float2*>(p.out + (size_t)b * d + col + 2 * j) =
                    make_float2((float)(s0 / len), (float)(s1 / len));
              } else {
                double* a = p.acc + (size_t)b * d + col + 2 * j;
                atomicAdd(a, s0);
                atomicAdd(a + 1, s1);
              }
            }
          }
        }
      }
      qs = qe;
    }
    __syncwarp();  // my_row is refilled by the next chunk
  }
}

// Bags that k_pool could not write at once: a bag split over chunks takes
// its fp64 accumulator, an empty bag zeros.  Offsets that decrease or leave
// [0, n] latch MT_EINVAL (the bag is then written as zeros).
__global__ void __launch_bounds__(256) k_pool_finish(const PoolParams p) {
  const int d4 = (int)p.T.dim / 4;  // four columns per item (d is a multiple of 4)
  const long long total = p.num_bags * d4;
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const long long b = it / d4;
    const int j4 = (int)(it - b * d4);
    const long long s = __ldg(&p.bag_offsets[b]), e = __ldg(&p.bag_offsets[b + 1]);
    const bool bad = s < 0 || e < s || e > p.n;
    if (bad && j4 == 0) latch_error(p.T.hdr, MT_EINVAL);
    const bool one_chunk = !bad && e > s && s / kPoolChunk == (e - 1) / kPoolChunk;
    if (one_chunk) continue;  // written by k_pool
    float4 o = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (!bad && e > s) {
      const double2* a = reinterpret_cast<const double2*>(p.acc + (size_t)b * p.T.dim) + 2 * j4;
      const double2 a0 = __ldcg(a), a1 = __ldcg(a + 1);
      const bool mean = p.mode == MT_POOL_MEAN;
      const double len = (double)(e - s);
      o = make_float4((float)(mean ? a0.x / len : a0.x), (float)(mean ? a0.y / len : a0.y),
                      (float)(mean ? a1.x / len : a1.x), (float)(mean ? a1.y / len : a1.y));
    }
    reinterpret_cast<float4*>(p.out + (size_t)b * p.T.dim)[j4] = o;
  }
}

// The bag of every position: a warp per bag writes its positions (the
// positions were set to -1 beforehand).  Offsets that decrease or leave
// [0, n] latch MT_EINVAL; the writes stay inside [0, n).
__global__ void __launch_bounds__(256) k_pos_bag(const long long* bo, long long B, long long n, int32_t* pos_bag,
                                                 Header* hdr) {
  const int lane = threadIdx.x & 31;
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long b = gw; b < B; b += nw) {
    long long s = __ldg(&bo[b]), e = __ldg(&bo[b + 1]);
    if ((s < 0 || e < s || e > n) && lane == 0) latch_error(hdr, MT_EINVAL);
    s = s < 0 ? 0 : (s > n ? n : s);
    e = e < s ? s : (e > n ? n : e);
    for (long long i = s + lane; i < e; i += 32) pos_bag[i] = (int32_t)b;
  }
}

// dscaled[b] = dpooled[b] * fp32(1/len_b), one rounding per product (the
// gradient every position of a mean-pooled bag receives).
__global__ void __launch_bounds__(256) k_pool_scale(const long long* bo, long long B, int d, const float* dpooled,
                                                    float* dscaled) {
  const int d4 = d / 4;  // four columns per item (d is a multiple of 4)
  const long long total = B * d4;
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const long long b = it / d4;
    const long long len = __ldg(&bo[b + 1]) - __ldg(&bo[b]);
    const float s = len > 0 ? __frcp_rn((float)len) : 1.0f;
    const float4 g = __ldg(reinterpret_cast<const float4*>(dpooled) + it);
    reinterpret_cast<float4*>(dscaled)[it] =
        make_float4(__fmul_rn(g.x, s), __fmul_rn(g.y, s), __fmul_rn(g.z, s), __fmul_rn(g.w, s));
  }
}

}  // namespace

cudaError_t launch_pool(const PoolParams& p, cudaStream_t s) {
  if (p.num_bags == 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(p.acc, 0, (size_t)p.num_bags * p.T.dim * sizeof(double), s);
  if (e != cudaSuccess) return e;
  if (p.n > 0) {
    const long long chunks = (p.n + kPoolChunk - 1) / kPoolChunk;
    MT_LAUNCH("k_pool", s);
    const int grid = grid_for(chunks * 32, 256, 16);  // a warp per chunk
    if (p.T.row_dtype == MT_F32) k_pool<MT_F32><<<grid, 256, 0, s>>>(p);
    else k_pool<MT_BF16><<<grid, 256, 0, s>>>(p);
  }
  {
    MT_LAUNCH("k_pool_finish", s);
    k_pool_finish<<<grid_for(p.num_bags * p.T.dim / 4, 256, 16), 256, 0, s>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_pos_bag(const long long* bo, long long B, long long n, int32_t* pos_bag, Header* hdr,
                           cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(pos_bag, 0xFF, (size_t)(n > 0 ? n : 1) * 4, s);
  if (e != cudaSuccess || B == 0) return e;
  MT_LAUNCH("k_pos_bag", s);
  k_pos_bag<<<grid_for(B * 32, 256, 16), 256, 0, s>>>(bo, B, n, pos_bag, hdr);
  return cudaGetLastError();
}

cudaError_t launch_pool_scale(const long long* bo, long long B, int d, const float* dpooled, float* dscaled,
                              cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  MT_LAUNCH("k_pool_scale", s);
  k_pool_scale<<<grid_for(B * d / 4, 256, 16), 256, 0, s>>>(bo, B, d, dpooled, dscaled);
  return cudaGetLastError();
}

}  // namespace mt
