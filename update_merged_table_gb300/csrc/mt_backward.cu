// Backward path of the merged dynamic embedding table: per-unique-ID gradient
// reduction feeding a fused sparse row-wise Adam update.
//
// Pages: Adam is named in the Meituan TensorFlow article (section 3.2, with
// the beta-power accumulators shared by all parameters, i.e. one step
// counter per table); the sparse update of only the rows a batch touched
// follows from the dynamic table of "MTGenRec" (abstract) and "MTGR"
// section 5 (Embedding Management).  The update is Kingma & Ba's Adam with
// bias correction.
//
// Kernels, in launch order:
//  k_bw_blocksum   per block of uniques: sums of counts, of chunks
//                  (ceil(count / kChunk)) and of multi-chunk uniques; block
//                  0 advances the table's step counter.
//  k_scan_small    exclusive offsets of those sums over the blocks.
//  k_bw_offsets    per unique: segment start (cursor), first chunk, index
//                  among multi-chunk uniques; chunk -> unique map; zeroed
//                  cross-chunk accumulators.
//  k_bw_fill       positions grouped by unique (a counting sort): one
//                  shared-memory group per unique per tile, one global
//                  atomic per group to reserve its place in the segment.
//  k_bw_reduce_adam  one team of lanes per chunk of <= kChunk positions sums
//                  its gradient rows in fp32 pair (TwoSum) arithmetic.  A
//                  single-chunk unique applies Adam at once; the chunks of a
//                  larger unique add their partial sums in fp64 in L2 and
//                  the last chunk to finish applies Adam.
#include "mt_kernels.cuh"

namespace mt {

namespace {

template <int NT>
__device__ __forceinline__ void block_scan3(const int v[3], int ex[3], int tot[3], int (*s_warp)[NT / 32]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x[3] = {v[0], v[1], v[2]};
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int c = 0; c < 3; ++c) {
      const int y = __shfl_up_sync(kFull, x[c], o);
      if (lane >= o) x[c] += y;
    }
  }
  if (lane == 31) {
#pragma unroll
    for (int c = 0; c < 3; ++c) s_warp[c][warp] = x[c];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int c = 0; c < 3; ++c) {
      int w = lane < NT / 32 ? s_warp[c][lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, w, o);
        if (lane >= o) w += y;
      }
      if (lane < NT / 32) s_warp[c][lane] = w;
    }
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < 3; ++c) {
    ex[c] = (warp ? s_warp[c][warp - 1] : 0) + x[c] - v[c];
    tot[c] = s_warp[c][NT / 32 - 1];
  }
  __syncthreads();
}

__device__ __forceinline__ int nchunks(int c) { return (c + kChunk - 1) / kChunk; }

__global__ void __launch_bounds__(kScanThreads) k_bw_blocksum(const BackwardParams p) {
  __shared__ int s_warp[3][kScanThreads / 32];
  if (blockIdx.x == 0 && threadIdx.x == 0) p.T.hdr->step += 1;
  const long long U = *p.num_unique;
  const long long u0 = (long long)blockIdx.x * kScanTile;
  int v[3] = {0, 0, 0};
  for (long long u = u0 + threadIdx.x; u < U && u < u0 + kScanTile; u += kScanThreads) {
    const int c = p.counts[u];
    const int nc = nchunks(c);
    v[0] += c;
    v[1] += nc;
    v[2] += nc > 1;
  }
  int ex[3], tot[3];
  block_scan3<kScanThreads>(v, ex, tot, s_warp);
  if (threadIdx.x < 3) p.bsum[(size_t)blockIdx.x * 3 + threadIdx.x] = tot[threadIdx.x];
}

constexpr int kUPT = kScanTile / kScanThreads;  // uniques per thread in k_bw_offsets

// Per unique: segment start (cursor).  Per chunk: a descriptor {start, end,
// row, u or -(heavy index + 1)}, written cooperatively by the block so a hot
// unique with thousands of chunks costs no single thread more than its share.
// Per multi-chunk unique: {u, chunks}, a zero arrival count and zeroed fp64
// accumulators.
__global__ void __launch_bounds__(kScanThreads) k_bw_offsets(const BackwardParams p) {
  __shared__ int s_warp[3][kScanThreads / 32];
  __shared__ int s_chrel[kScanTile + 1];  // first chunk of each local unique, relative to the block
  __shared__ int s_seg[kScanTile];        // segment start, relative to the block
  __shared__ int s_cnt[kScanTile];
  __shared__ int s_row[kScanTile];
  __shared__ int s_hrel[kScanTile];       // multi-chunk index relative to the block, or -1
  const long long U = *p.num_unique;
  const long long ublk = (long long)blockIdx.x * kScanTile;
  if (ublk >= U) return;  // uniform over the block
  const int tid = threadIdx.x;
  const long long u0 = ublk + (long long)tid * kUPT;
  int c[kUPT];
  int v[3] = {0, 0, 0};
#pragma unroll
  for (int k = 0; k < kUPT; ++k) {
    c[k] = u0 + k < U ? p.counts[u0 + k] : 0;
    const int nc = nchunks(c[k]);
    v[0] += c[k];
    v[1] += nc;
    v[2] += nc > 1;
  }
  int ex[3], tot[3];
  block_scan3<kScanThreads>(v, ex, tot, s_warp);
  const int seg_base = p.boff[(size_t)blockIdx.x * 3 + 0];
  const int ch_base = p.boff[(size_t)blockIdx.x * 3 + 1];
  const int hv_base = p.boff[(size_t)blockIdx.x * 3 + 2];
  int seg = ex[0], ch = ex[1], hv = ex[2];
#pragma unroll
  for (int k = 0; k < kUPT; ++k) {
    const int ul = tid * kUPT + k;
    const long long u = u0 + k;
    const int nc = nchunks(c[k]);
    s_chrel[ul] = ch;
    s_seg[ul] = seg;
    s_cnt[ul] = c[k];
    s_hrel[ul] = nc > 1 ? hv : -1;
    s_row[ul] = u < U ? p.unique_rows[u] : -1;
    if (u < U) p.cursor[u] = seg_base + seg;
    ch += nc;
    seg += c[k];
    hv += nc > 1;
  }
  if (tid == 0) s_chrel[kScanTile] = tot[1];
  __syncthreads();
  for (int cc = tid; cc < tot[1]; cc += kScanThreads) {
    int lo = 0, hi = kScanTile;  // s_chrel[lo] <= cc < s_chrel[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_chrel[mid] <= cc) lo = mid; else hi = mid;
    }
    const int k = cc - s_chrel[lo];
    const int start = seg_base + s_seg[lo] + k * kChunk;
    const int end = min(start + kChunk, seg_base + s_seg[lo] + s_cnt[lo]);
    const int w = s_hrel[lo] < 0 ? (int)(ublk + lo) : -(hv_base + s_hrel[lo] + 1);
    p.chunks[ch_base + cc] = make_int4(start, end, s_row[lo], w);
  }
  for (int ul = tid; ul < kScanTile; ul += kScanThreads) {
    if (s_hrel[ul] >= 0) {
      const int h = hv_base + s_hrel[ul];
      p.heavy_info[h] = make_int2((int)(ublk + ul), nchunks(s_cnt[ul]));
      p.arrive[h] = 0;
    }
  }
  const int d2 = (int)p.T.dim / 2;
  double2* acc = reinterpret_cast<double2*>(p.acc64 + (size_t)hv_base * p.T.dim);
  for (int it = tid; it < tot[2] * d2; it += kScanThreads) acc[it] = make_double2(0.0, 0.0);
}

// Positions grouped by unique: each tile groups its positions by unique in
// shared memory, reserves room for each group with one atomic on the
// unique's cursor, then scatters the positions.
__global__ void __launch_bounds__(kThreads) k_bw_fill(const BackwardParams p) {
  __shared__ int32_t s_hkey[kHS];
  __shared__ int32_t s_hcnt[kHS];
  __shared__ uint16_t s_slot[kTile];
  __shared__ uint16_t s_rank[kTile];
  const int tid = threadIdx.x, lane = tid & 31;
  const long long base = (long long)blockIdx.x * kTile;
  const int cnt = (int)min((long long)kTile, p.n - base);
  for (int h = tid; h < kHS; h += kThreads) {
    s_hkey[h] = -1;
    s_hcnt[h] = 0;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kPPT; ++k) {
    const int lp = k * kThreads + tid;
    const int u = lp < cnt ? p.inverse[base + lp] : -1;
    const bool v = u >= 0;
    const unsigned act = __ballot_sync(kFull, v);
    if (v) {
      const unsigned grp = __match_any_sync(act, u);
      const int leader = __ffs(grp) - 1;
      uint32_t slot = 0;
      int old = 0;
      if (lane == leader) {
        uint32_t h = ((uint32_t)u * 2654435761u) >> (32 - 12);
        for (int probe = 0; probe < kHS; ++probe) {
          const int prev = atomicCAS(&s_hkey[h], -1, u);
          if (prev == -1 || prev == u) break;
          h = (h + 1) & (uint32_t)(kHS - 1);
        }
        slot = h;
        old = atomicAdd(&s_hcnt[slot], __popc(grp));
      }
      slot = __shfl_sync(grp, slot, leader);
      old = __shfl_sync(grp, old, leader);
      s_slot[lp] = (uint16_t)slot;
      s_rank[lp] = (uint16_t)(old + __popc(grp & ((1u << lane) - 1u)));
    } else if (lp < cnt) {
      s_slot[lp] = kNoIdx;
    }
  }
  __syncthreads();
  for (int h = tid; h < kHS; h += kThreads) {
    const int u = s_hkey[h];
    if (u >= 0) s_hcnt[h] = atomicAdd(&p.cursor[u], s_hcnt[h]);  // group count -> group base
  }
  __syncthreads();
  for (int lp = tid; lp < cnt; lp += kThreads) {
    const uint16_t sl = s_slot[lp];
    if (sl != kNoIdx) p.pos_sorted[s_hcnt[sl] + s_rank[lp]] = (int32_t)(base + lp);
  }
}

// ---- reduction + Adam -------------------------------------------------------

// a + b = s + e exactly (Knuth's TwoSum); the running pair (hi, lo) carries
// the sum with about twice fp32's precision.
__device__ __forceinline__ void two_sum_add(float& hi, float& lo, float x) {
  const float s = __fadd_rn(hi, x);
  const float bb = __fsub_rn(s, hi);
  const float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(x, bb));
  hi = s;
  lo = __fadd_rn(lo, e);
}

template <int GD, int VEC>
__device__ __forceinline__ void load_grad(const void* grads, long long pos, int d, int col, float g[VEC]) {
  if (GD == MT_F32) {
    const float4* src = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(grads) + (size_t)pos * d + col);
#pragma unroll
    for (int q = 0; q < VEC / 4; ++q) {
      const float4 t = __ldg(src + q);
      g[4 * q + 0] = t.x;
      g[4 * q + 1] = t.y;
      g[4 * q + 2] = t.z;
      g[4 * q + 3] = t.w;
    }
  } else {
    const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(grads) + (size_t)pos * d + col;
    if (VEC == 8) {
      const uint4 t = __ldg(reinterpret_cast<const uint4*>(b));
      const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[q]));
        g[2 * q] = f.x;
        g[2 * q + 1] = f.y;
      }
    } else {
      const uint2 t = __ldg(reinterpret_cast<const uint2*>(b));
      const uint32_t w[2] = {t.x, t.y};
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[q]));
        g[2 * q] = f.x;
        g[2 * q + 1] = f.y;
      }
    }
  }
}

// Adam state of columns [col, col + VEC) of a row: w (as fp32), m, v.
template <int RD, int VEC>
struct RowCols {
  float w[VEC], m[VEC], v[VEC];
};

template <int RD, int VEC>
__device__ __forceinline__ void load_row_cols(const TableDev& T, int32_t row, int col, RowCols<RD, VEC>& r) {
  const char* rec = row_ptr(T, row);
  if (RD == MT_F32) {
    const float4* e = reinterpret_cast<const float4*>(rec) + col / 4;
#pragma unroll
    for (int q = 0; q < VEC / 4; ++q) {
      const float4 t = e[q];
      r.w[4 * q] = t.x; r.w[4 * q + 1] = t.y; r.w[4 * q + 2] = t.z; r.w[4 * q + 3] = t.w;
    }
  } else {
    const uint4 t = *(reinterpret_cast<const uint4*>(rec) + col / 8);
    const uint32_t ww[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ww[q]));
      r.w[2 * q] = f.x;
      r.w[2 * q + 1] = f.y;
    }
  }
  const float4* mp = reinterpret_cast<const float4*>(rec + T.emb_bytes) + col / 4;
  const float4* vp = reinterpret_cast<const float4*>(rec + T.emb_bytes + T.mv_bytes) + col / 4;
#pragma unroll
  for (int q = 0; q < VEC / 4; ++q) {
    const float4 a = mp[q], b = vp[q];
    r.m[4 * q] = a.x; r.m[4 * q + 1] = a.y; r.m[4 * q + 2] = a.z; r.m[4 * q + 3] = a.w;
    r.v[4 * q] = b.x; r.v[4 * q + 1] = b.y; r.v[4 * q + 2] = b.z; r.v[4 * q + 3] = b.w;
  }
}

// One Adam step on the loaded columns, in the operation order of the update
// rule with every operation rounded once, then the store.
template <int RD, int VEC>
__device__ __forceinline__ void adam_apply_store(const BackwardParams& p, int32_t row, int col, const float g[VEC],
                                                 RowCols<RD, VEC>& r, float bc1, float bc2) {
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    r.m[j] = __fadd_rn(__fmul_rn(p.beta1, r.m[j]), __fmul_rn(p.one_minus_b1, g[j]));
    r.v[j] = __fadd_rn(__fmul_rn(p.beta2, r.v[j]), __fmul_rn(p.one_minus_b2, __fmul_rn(g[j], g[j])));
    const float mhat = __fdiv_rn(r.m[j], bc1);
    const float vhat = __fdiv_rn(r.v[j], bc2);
    const float den = __fadd_rn(__fsqrt_rn(vhat), p.eps);
    r.w[j] = __fsub_rn(r.w[j], __fmul_rn(p.lr, __fdiv_rn(mhat, den)));
  }
  char* rec = row_ptr(p.T, row);
  float4* mp = reinterpret_cast<float4*>(rec + p.T.emb_bytes) + col / 4;
  float4* vp = reinterpret_cast<float4*>(rec + p.T.emb_bytes + p.T.mv_bytes) + col / 4;
#pragma unroll
  for (int q = 0; q < VEC / 4; ++q) {
    mp[q] = make_float4(r.m[4 * q], r.m[4 * q + 1], r.m[4 * q + 2], r.m[4 * q + 3]);
    vp[q] = make_float4(r.v[4 * q], r.v[4 * q + 1], r.v[4 * q + 2], r.v[4 * q + 3]);
  }
  if (RD == MT_F32) {
    float4* e = reinterpret_cast<float4*>(rec) + col / 4;
#pragma unroll
    for (int q = 0; q < VEC / 4; ++q) e[q] = make_float4(r.w[4 * q], r.w[4 * q + 1], r.w[4 * q + 2], r.w[4 * q + 3]);
  } else {
    uint32_t ww[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      __nv_bfloat162 b2 = __floats2bfloat162_rn(r.w[2 * q], r.w[2 * q + 1]);
      ww[q] = *reinterpret_cast<uint32_t*>(&b2);
    }
    *(reinterpret_cast<uint4*>(rec) + col / 8) = make_uint4(ww[0], ww[1], ww[2], ww[3]);
  }
}

__device__ __forceinline__ void store_gsum(float* gsum_out, int u, int d, int col, const float* gs, int vec) {
  float4* o = reinterpret_cast<float4*>(gsum_out + (size_t)u * d + col);
  for (int r = 0; r < vec / 4; ++r) o[r] = make_float4(gs[4 * r], gs[4 * r + 1], gs[4 * r + 2], gs[4 * r + 3]);
}

constexpr int kMinTeamShift = 2;                              // teams of at least 4 lanes
constexpr int kMaxTeams = 256 >> kMinTeamShift;               // per block

// One team of 2^team_shift lanes per chunk descriptor.  The team stages the
// chunk's positions in shared memory, prefetches the Adam row of a
// single-chunk unique while the gradient rows load, accumulates in TwoSum
// pairs, and either applies Adam (single-chunk unique) or adds its partial
// sum to the unique's fp64 accumulator in L2, the last chunk applying Adam.
template <int RD, int GD>
__global__ void __launch_bounds__(256) k_bw_reduce_adam(const BackwardParams p, int team_shift) {
  constexpr int VEC = RD == MT_F32 ? 4 : 8;
  constexpr int UNR = VEC == 8 ? 4 : 8;  // gradient rows in flight per lane
  __shared__ float s_bc[2];
  __shared__ int s_pos[kMaxTeams * kChunk];
  if (threadIdx.x == 0) {
    const double t = (double)p.T.hdr->step;
    s_bc[0] = (float)(1.0 - pow((double)p.beta1, t));
    s_bc[1] = (float)(1.0 - pow((double)p.beta2, t));
  }
  __syncthreads();
  const float bc1 = s_bc[0], bc2 = s_bc[1];

  const int team = 1 << team_shift;
  const int lane = threadIdx.x & 31;
  const int lt = lane & (team - 1);
  const unsigned team_mask = team == 32 ? kFull : (((1u << team) - 1u) << (lane & ~(team - 1)));
  int* my_pos = s_pos + (threadIdx.x >> team_shift) * kChunk;
  const long long total_chunks = p.boff[(size_t)p.nblk * 3 + 1];
  const long long gteam = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> team_shift;
  const long long nteam = ((long long)gridDim.x * blockDim.x) >> team_shift;
  const int d = (int)p.T.dim;
  const bool one_pass = d <= team * VEC;

  for (long long c = gteam; c < total_chunks; c += nteam) {
    const int4 dsc = __ldg(&p.chunks[c]);
    const int start = dsc.x, cnt = dsc.y - dsc.x, row = dsc.z;
    const bool heavy = dsc.w < 0;
    for (int q = lt; q < cnt; q += team) my_pos[q] = __ldg(&p.pos_sorted[start + q]);
    RowCols<RD, VEC> rc;
    const int col0 = lt * VEC;
    if (one_pass && !heavy && row >= 0 && col0 < d) load_row_cols<RD, VEC>(p.T, row, col0, rc);
    __syncwarp(team_mask);

    for (int c0 = 0; c0 < d; c0 += team * VEC) {
      const int col = c0 + col0;
      if (col >= d) continue;
      float hi[VEC], lo[VEC];
#pragma unroll
      for (int j = 0; j < VEC; ++j) hi[j] = lo[j] = 0.f;
      for (int q0 = 0; q0 < cnt; q0 += UNR) {
        float g[UNR][VEC];
#pragma unroll
        for (int r = 0; r < UNR; ++r)
          if (q0 + r < cnt) load_grad<GD, VEC>(p.grads, my_pos[q0 + r], d, col, g[r]);
#pragma unroll
        for (int r = 0; r < UNR; ++r)
          if (q0 + r < cnt) {
#pragma unroll
            for (int j = 0; j < VEC; ++j) two_sum_add(hi[j], lo[j], g[r][j]);
          }
      }
      if (!heavy) {
        float gs[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) gs[j] = __fadd_rn(hi[j], lo[j]);
        if (p.gsum_out != nullptr) store_gsum(p.gsum_out, dsc.w, d, col, gs, VEC);
        if (row >= 0) {
          if (!one_pass) load_row_cols<RD, VEC>(p.T, row, col, rc);
          adam_apply_store<RD, VEC>(p, row, col, gs, rc, bc1, bc2);
        }
      } else {
        double* a = p.acc64 + (size_t)(-dsc.w - 1) * d + col;
#pragma unroll
        for (int j = 0; j < VEC; ++j) atomicAdd(a + j, (double)hi[j] + (double)lo[j]);
      }
    }
    if (heavy) {
      const int h = -dsc.w - 1;
      __threadfence();
      __syncwarp(team_mask);
      int old = 0;
      if (lt == 0) old = atomicAdd(&p.arrive[h], 1);
      old = __shfl_sync(team_mask, old, 0, team);
      const int2 hinfo = __ldg(&p.heavy_info[h]);
      if (old == hinfo.y - 1) {  // last chunk of this unique: every partial sum has landed
        __threadfence();
        for (int c0 = 0; c0 < d; c0 += team * VEC) {
          const int col = c0 + col0;
          if (col >= d) continue;
          float gs[VEC];
          const double* a = p.acc64 + (size_t)h * d + col;
#pragma unroll
          for (int j = 0; j < VEC; ++j) gs[j] = (float)__ldcg(a + j);
          if (p.gsum_out != nullptr) store_gsum(p.gsum_out, hinfo.x, d, col, gs, VEC);
          if (row >= 0) {
            load_row_cols<RD, VEC>(p.T, row, col, rc);
            adam_apply_store<RD, VEC>(p, row, col, gs, rc, bc1, bc2);
          }
        }
      }
    }
    __syncwarp(team_mask);  // my_pos is reused by the next chunk
  }
}

int g_reduce_grid[4] = {0, 0, 0, 0};

template <int RD, int GD>
cudaError_t launch_reduce(const BackwardParams& p, int team_shift, cudaStream_t s) {
  int& grid = g_reduce_grid[RD * 2 + GD];
  if (grid == 0) {
    int dev = 0, sms = 0, per = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, k_bw_reduce_adam<RD, GD>, 256, 0);
    grid = sms * (per > 0 ? per : 1);
  }
  MT_LAUNCH("k_bw_reduce_adam", s);
  k_bw_reduce_adam<RD, GD><<<grid, 256, 0, s>>>(p, team_shift);
  return cudaGetLastError();
}

}  // namespace

BackwardWsLayout backward_ws_layout(long long n, uint32_t dim) {
  BackwardWsLayout L{};
  L.nblk = (int)((n + kScanTile - 1) / kScanTile);
  if (L.nblk < 1) L.nblk = 1;
  L.ntiles = (int)((n + kTile - 1) / kTile);
  L.heavy_cap = n / (kChunk + 1) + 1;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const size_t nn = (size_t)(n > 0 ? n : 1);
  L.bsum = take((size_t)L.nblk * 3 * 4);
  L.boff = take(((size_t)L.nblk + 1) * 3 * 4);
  L.cursor = take(nn * 4);
  L.chunks = take(nn * 16);
  L.heavy_info = take((size_t)L.heavy_cap * 8);
  L.pos_sorted = take(nn * 4);
  L.acc64 = take((size_t)L.heavy_cap * dim * 8);
  L.arrive = take((size_t)L.heavy_cap * 4);
  L.total = off;
  return L;
}

cudaError_t launch_backward(const BackwardParams& p, cudaStream_t s) {
  {
    MT_LAUNCH("k_bw_blocksum", s);
    k_bw_blocksum<<<p.nblk, kScanThreads, 0, s>>>(p);
  }
  cudaError_t e = launch_scan_small(p.bsum, p.boff, p.nblk, 3, nullptr, s);
  if (e != cudaSuccess) return e;
  {
    MT_LAUNCH("k_bw_offsets", s);
    k_bw_offsets<<<p.nblk, kScanThreads, 0, s>>>(p);
  }
  if (p.ntiles > 0) {
    MT_LAUNCH("k_bw_fill", s);
    k_bw_fill<<<p.ntiles, kThreads, 0, s>>>(p);
  }
  const int vec = p.T.row_dtype == MT_F32 ? 4 : 8;
  int team = 1 << kMinTeamShift, shift = kMinTeamShift;
  while (team < 32 && team * vec < (int)p.T.dim) {
    team <<= 1;
    ++shift;
  }
  if (p.T.row_dtype == MT_F32) {
    return p.grad_dtype == MT_F32 ? launch_reduce<MT_F32, MT_F32>(p, shift, s) : launch_reduce<MT_F32, MT_BF16>(p, shift, s);
  }
  return p.grad_dtype == MT_F32 ? launch_reduce<MT_BF16, MT_F32>(p, shift, s) : launch_reduce<MT_BF16, MT_BF16>(p, shift, s);
}

}  // namespace mt
