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
//  k_bw_plan         per block of uniques (after a memset of three counters):
//                    each unique's segment {start, count}, a chunk descriptor
//                    per light unique, a record per heavy unique (more than
//                    kChunk positions); each block reserves its ranges with
//                    one atomic per counter.  One extra block advances the
//                    table's step counter and beta powers and computes the
//                    Adam scalars.
//  k_bw_scatter      heavy uniques' warp-chunk descriptors and zeroed fp64
//                    accumulators; positions grouped by unique: segment start + the rank
//                    the lookup recorded (k_bw_fill re-groups them with a
//                    shared-memory hash when the lookup kept no ranks).
//  k_bw_heavy_reduce heavy uniques: a warp per warp-chunk, 16 gradient rows
//                    in flight per lane, TwoSum pairs, shuffle combine; the
//                    last warp-chunk of a unique applies Adam.
//  k_bw_light_reduce light uniques: a team of lanes per unique, software
//                    pipelined across the team's uniques; Adam fused.
#include <atomic>

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

// A unique with more than kChunk positions is "heavy": it is reduced in
// warp-chunks of p.warp_chunk positions, each by one whole warp.
__device__ __forceinline__ int warp_chunks(int c, int wc) { return c > kChunk ? (c + wc - 1) / wc : 0; }

// The grouping plan, one block per kScanTile uniques: each unique gets a
// segment of pos_sorted (its count of positions), and either one team-chunk
// descriptor (light) or a heavy record whose warp-chunks k_bw_scatter writes.
// Segments only need to be disjoint, so each block reserves its ranges with
// one atomic per counter (positions, heavy warp-chunks, heavy uniques) and
// places its uniques by a block scan: no pass over the other blocks' sums.
// Light unique u's descriptor is chunks[light0 + u].  The block after the last one advances the table's step
// counter and beta-power accumulators and computes the step's Adam scalars.
constexpr int kUPT = kScanTile / kScanThreads;  // uniques per thread in k_bw_plan

__global__ void __launch_bounds__(kScanThreads) k_bw_plan(const BackwardParams p) {
  __shared__ int s_warp[3][kScanThreads / 32];
  __shared__ int s_base[3];
  if (blockIdx.x == p.nblk) {  // the extra block: step counter and this step's Adam scalars
    if (threadIdx.x == 0 && p.reduce_only) p.work[0] = 0;
    if (threadIdx.x == 0 && !p.reduce_only) {
      p.T.hdr->step += 1;
      p.work[0] = 0;
      // the beta-power accumulators advance by one multiply each (in
      // double); then, rounded once to fp32, step_size = lr / (1 - b1^t)
      // and inv_sqrt_bc2 = 1 / sqrt(1 - b2^t)
      const double b1t = __dmul_rn(p.T.hdr->b1pow, (double)p.beta1);
      const double b2t = __dmul_rn(p.T.hdr->b2pow, (double)p.beta2);
      p.T.hdr->b1pow = b1t;
      p.T.hdr->b2pow = b2t;
      p.work[2] = __float_as_int((float)__ddiv_rn((double)p.lr, __dsub_rn(1.0, b1t)));
      p.work[3] = __float_as_int((float)__ddiv_rn(1.0, __dsqrt_rn(__dsub_rn(1.0, b2t))));
    }
    return;
  }
  const long long U = *p.num_unique;
  const long long ub = (long long)blockIdx.x * kScanTile;
  if (ub >= U) return;  // the grid is sized for every ID distinct
  const long long u0 = ub + (long long)threadIdx.x * kUPT;
  int c[kUPT], rows[kUPT];
#pragma unroll
  for (int k = 0; k < kUPT; ++k) {
    c[k] = u0 + k < U ? __ldg(&p.counts[u0 + k]) : 0;
    rows[k] = u0 + k < U ? __ldg(&p.unique_rows[u0 + k]) : -1;
  }
  int v[3] = {0, 0, 0};
#pragma unroll
  for (int k = 0; k < kUPT; ++k) {
    v[0] += c[k];
    v[1] += warp_chunks(c[k], p.warp_chunk);
    v[2] += c[k] > kChunk;
  }
  int ex[3], tot[3];
  block_scan3<kScanThreads>(v, ex, tot, s_warp);
  if (threadIdx.x == 0) {
    s_base[0] = atomicAdd(&p.ctr[0], tot[0]);
    s_base[1] = atomicAdd(&p.ctr[1], tot[1]);
    s_base[2] = atomicAdd(&p.ctr[2], tot[2]);
  }
  __syncthreads();
  int seg = ex[0] + s_base[0];
  int hch = ex[1] + s_base[1];
  int hv = ex[2] + s_base[2];
#pragma unroll
  for (int k = 0; k < kUPT; ++k) {
    const long long u = u0 + k;
    if (u >= U) break;
    p.seg[u] = make_int2(seg, c[k]);
    // the team-chunks stay in unique order (the light reduce runs measurably faster so); a heavy unique
    // leaves an empty one there
    p.chunks[p.light0 + u] = c[k] <= kChunk ? make_int4(seg, seg + c[k], rows[k], (int)u) : make_int4(0, 0, -1, -1);
    if (c[k] > kChunk) {
      const int nw = warp_chunks(c[k], p.warp_chunk);
      p.heavy_info[hv] = make_int4((int)u, nw, seg, hch);  // its warp-chunks are written by the grouping kernel
      ++hv;
      hch += nw;
    }
    seg += c[k];
  }
}


// Warp-chunk descriptors of the heavy uniques, a warp per heavy unique over
// the whole grid (the hottest IDs are seen first, so their uniques cluster
// in the first offsets block); a unique with several warp-chunks also gets
// its fp64 accumulator and arrival count cleared.  Called by every thread of
// the grouping kernels before they group.
__device__ __forceinline__ void write_heavy_chunks(const BackwardParams& p) {
  const int H = __ldcg(&p.ctr[2]);
  const int d = (int)p.T.dim;
  const int lane = threadIdx.x & 31;
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nw_grid = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long h = gw; h < H; h += nw_grid) {
    const int4 hi = __ldg(&p.heavy_info[h]);  // {u, warp-chunks, segment start, first warp-chunk}
    const int cnt = __ldg(&p.seg[hi.x]).y, row = __ldg(&p.unique_rows[hi.x]);
    for (int q = lane; q < hi.y; q += 32) {
      const int start = hi.z + q * p.warp_chunk;
      p.chunks[hi.w + q] = make_int4(start, min(start + p.warp_chunk, hi.z + cnt), row, -(int)(h + 1));
    }
    if (hi.y > 1) {
      double2* a = reinterpret_cast<double2*>(p.acc64 + (size_t)h * d);
      for (int q = lane; q < d / 2; q += 32) a[q] = make_double2(0.0, 0.0);
      if (lane == 0) p.arrive[h] = 0;
    }
  }
}

// Positions grouped by unique: each tile groups its positions by unique in
// shared memory, reserves room for each group with one atomic on the
// unique's segment start, then scatters the positions.
__global__ void __launch_bounds__(kThreads) k_bw_fill(const BackwardParams p) {
  __shared__ int32_t s_hkey[kHS];
  __shared__ int32_t s_hcnt[kHS];
  __shared__ uint16_t s_slot[kTile];
  __shared__ uint16_t s_rank[kTile];
  const int tid = threadIdx.x, lane = tid & 31;
  const long long base = (long long)blockIdx.x * kTile;
  const int cnt = (int)min((long long)kTile, p.n - base);
  write_heavy_chunks(p);
  const long long U = *p.num_unique;
  for (int h = tid; h < kHS; h += kThreads) {
    s_hkey[h] = -1;
    s_hcnt[h] = 0;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kPPT; ++k) {
    const int lp = k * kThreads + tid;
    int u = lp < cnt ? p.inverse[base + lp] : -1;
    if (u >= U) {  // not an index of this lookup's uniques: skip it, report it
      latch_error(p.T.hdr, MT_EINVAL);
      u = -1;
    }
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
    if (u >= 0) s_hcnt[h] = atomicAdd(&p.seg[u].x, s_hcnt[h]);  // group count -> group base
  }
  __syncthreads();
  for (int lp = tid; lp < cnt; lp += kThreads) {
    const uint16_t sl = s_slot[lp];
    if (sl != kNoIdx)
      p.pos_sorted[s_hcnt[sl] + s_rank[lp]] = p.pos_map ? __ldg(&p.pos_map[base + lp]) : (int32_t)(base + lp);
  }
}

// ---- reduction + Adam -------------------------------------------------------

// Add x and y (two rows' pairs) to the running pair (hi, lo), which carries
// the sum with about twice fp32's precision: the two rows' TwoSum does not
// depend on the running pair, so the serial chain per column is one TwoSum
// per two rows.
__device__ __forceinline__ void two_sum_add2(f32x2& hi, f32x2& lo, f32x2 x, f32x2 y) {
  f32x2 s, e, s2, e2;
  two_sum(x, y, s, e);
  two_sum(hi, s, s2, e2);
  hi = s2;
  lo = add2(lo, add2(e2, e));
}

// Add one row's pair x to the running pair (hi, lo).
__device__ __forceinline__ void two_sum_add(f32x2& hi, f32x2& lo, f32x2 x) {
  f32x2 s, e;
  two_sum(hi, x, s, e);
  hi = s;
  lo = add2(lo, e);
}

// Raw gradient words of one lane's VEC columns: VEC fp32 words, or VEC/2
// words holding two bf16 each.  Kept raw while in flight (fewer registers)
// and widened to fp32 only when accumulated.
template <int GD, int VEC>
struct GradRaw {
  static constexpr int W = GD == MT_F32 ? VEC : VEC / 2;
  uint32_t w[W];
};

template <int GD, int VEC>
__device__ __forceinline__ void load_grad_raw(const void* grads, long long pos, int d, int col, GradRaw<GD, VEC>& g) {
  constexpr int W = GradRaw<GD, VEC>::W;
  const char* base = reinterpret_cast<const char*>(grads) + ((size_t)pos * d + col) * (GD == MT_F32 ? 4 : 2);
  if (W >= 4) {
#pragma unroll
    for (int q = 0; q < W / 4; ++q) {
      const uint4 t = __ldg(reinterpret_cast<const uint4*>(base) + q);
      g.w[4 * q] = t.x; g.w[4 * q + 1] = t.y; g.w[4 * q + 2] = t.z; g.w[4 * q + 3] = t.w;
    }
  } else {
    const uint2 t = __ldg(reinterpret_cast<const uint2*>(base));
    g.w[0] = t.x;
    g.w[W - 1] = t.y;
  }
}

// Columns 2k and 2k + 1 of a raw gradient share as an fp32 pair.
template <int GD, int VEC>
__device__ __forceinline__ f32x2 grad_pair(const GradRaw<GD, VEC>& g, int k) {
  if (GD == MT_F32) return pk(__uint_as_float(g.w[2 * k]), __uint_as_float(g.w[2 * k + 1]));
  return bf16x2_to_f32x2(g.w[k]);
}

// One Adam step on columns [col, col + VEC) of a row, every operation
// rounded once: m = b1 m + (1-b1) g; v = b2 v + (1-b2) g^2;
// w -= step_size * m / (sqrt(v) * inv_sqrt_bc2 + eps).  Scalar operations
// only: a paired multiply followed by a paired add may be contracted into
// one fused multiply-add by the code generator, which changes the rounding.
// The moments are streamed four columns at a time to keep few registers
// live; the record is written back with evict-first stores (it is not read
// again this step, and it would push prefetched lines out of L2).
template <int RD, int VEC>
__device__ __forceinline__ void adam_cols(const BackwardParams& p, int32_t row, int col, const f32x2 g2[VEC / 2],
                                          float step_size, float inv_sqrt_bc2) {
  char* rec = row_ptr(p.T, row);
  float g[VEC], w[VEC];
#pragma unroll
  for (int j = 0; j < VEC / 2; ++j) {
    const float2 t = upk(g2[j]);
    g[2 * j] = t.x;
    g[2 * j + 1] = t.y;
  }
  if (RD == MT_F32) {
    const float4* e = reinterpret_cast<const float4*>(rec) + col / 4;
#pragma unroll
    for (int q = 0; q < VEC / 4; ++q) {
      const float4 t = e[q];
      w[4 * q] = t.x; w[4 * q + 1] = t.y; w[4 * q + 2] = t.z; w[4 * q + 3] = t.w;
    }
  } else {
    const uint4 t = *(reinterpret_cast<const uint4*>(rec) + col / 8);
    const uint32_t ww[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      w[2 * q] = __uint_as_float(ww[q] << 16);
      w[2 * q + 1] = __uint_as_float(ww[q] & 0xFFFF0000u);
    }
  }
  float4* mp = reinterpret_cast<float4*>(rec + p.T.emb_bytes) + col / 4;
  float4* vp = reinterpret_cast<float4*>(rec + p.T.emb_bytes + p.T.mv_bytes) + col / 4;
#pragma unroll
  for (int q = 0; q < VEC / 4; ++q) {
    const float4 m4 = mp[q], v4 = vp[q];
    float m[4] = {m4.x, m4.y, m4.z, m4.w}, v[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = 4 * q + k;
      m[k] = __fadd_rn(__fmul_rn(p.beta1, m[k]), __fmul_rn(p.one_minus_b1, g[j]));
      v[k] = __fadd_rn(__fmul_rn(p.beta2, v[k]), __fmul_rn(p.one_minus_b2, __fmul_rn(g[j], g[j])));
      const float den = __fadd_rn(__fmul_rn(__fsqrt_rn(v[k]), inv_sqrt_bc2), p.eps);
      w[j] = __fsub_rn(w[j], __fmul_rn(step_size, __fdiv_rn(m[k], den)));
    }
    __stcs(mp + q, make_float4(m[0], m[1], m[2], m[3]));  // written once per step: evict first
    __stcs(vp + q, make_float4(v[0], v[1], v[2], v[3]));
  }
  if (RD == MT_F32) {
    float4* e = reinterpret_cast<float4*>(rec) + col / 4;
#pragma unroll
    for (int q = 0; q < VEC / 4; ++q) __stcs(e + q, make_float4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]));
  } else {
    uint32_t ww[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      __nv_bfloat162 b2 = __floats2bfloat162_rn(w[2 * q], w[2 * q + 1]);
      ww[q] = *reinterpret_cast<uint32_t*>(&b2);
    }
    __stcs(reinterpret_cast<uint4*>(rec) + col / 8, make_uint4(ww[0], ww[1], ww[2], ww[3]));
  }
}

__device__ __forceinline__ void store_gsum(float* gsum_out, int u, int d, int col, const f32x2* gs, int vec) {
  ulonglong2* o = reinterpret_cast<ulonglong2*>(gsum_out + (size_t)u * d + col);
  for (int r = 0; r < vec / 4; ++r) o[r] = make_ulonglong2(gs[2 * r], gs[2 * r + 1]);
}

constexpr int kMinTeamShift = 2;                              // teams of at least 4 lanes
constexpr int kMaxTeams = 256 >> kMinTeamShift;               // per block

// Positions grouped by unique when the lookup recorded ranks: a plain
// scatter, pos_sorted[segment start + rank] = position.  A rank or unique
// index that does not belong to the lookup result (a caller passing some
// other buffer) is skipped and latches MT_EINVAL instead of writing.
constexpr int kScatterILP = 4;  // positions in flight per thread

__global__ void __launch_bounds__(256) k_bw_scatter(const BackwardParams p) {
  write_heavy_chunks(p);
  const long long U = *p.num_unique;
  const long long stride = (long long)gridDim.x * blockDim.x;
  bool bad = false;
  for (long long i0 = (long long)blockIdx.x * blockDim.x + threadIdx.x; i0 < p.n; i0 += kScatterILP * stride) {
    int u[kScatterILP], r[kScatterILP];
    int2 sg[kScatterILP];  // kScatterILP positions' loads in flight
#pragma unroll
    for (int k = 0; k < kScatterILP; ++k) {
      const long long i = i0 + k * stride;
      u[k] = i < p.n ? __ldg(&p.inverse[i]) : -1;
      r[k] = i < p.n ? __ldg(&p.ranks[i]) : -1;
    }
#pragma unroll
    for (int k = 0; k < kScatterILP; ++k) {
      const bool ok = u[k] >= 0 && u[k] < U;
      sg[k] = ok ? __ldg(&p.seg[u[k]]) : make_int2(0, 0);  // {segment start, count}
    }
#pragma unroll
    for (int k = 0; k < kScatterILP; ++k) {
      if (u[k] < 0) continue;
      if (u[k] >= U || r[k] < 0 || r[k] >= sg[k].y) {
        bad = true;
        continue;
      }
      const long long i = i0 + k * stride;
      p.pos_sorted[sg[k].x + r[k]] = p.pos_map ? __ldg(&p.pos_map[i]) : (int32_t)i;
    }
  }
  if (bad) latch_error(p.T.hdr, MT_EINVAL);
}

// A grouped gradient row, or -1 when it lies outside the gradient rows (a
// position in no bag, or inconsistent result buffers the grouping skipped).
__device__ __forceinline__ int valid_pos(const BackwardParams& p, int v) {
  return (unsigned)v < (unsigned long long)p.grad_rows ? v : -1;
}
__device__ __forceinline__ bool pos_ok(const BackwardParams& p, int v) {
  return (unsigned)v < (unsigned long long)p.grad_rows;
}

__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

// Sum of the gradient rows at positions pos[0 .. n) for one lane's VEC
// columns, in TwoSum pairs, UNR rows in flight.
template <int GD, int VEC, int UNR>
__device__ __forceinline__ void accumulate(const BackwardParams& p, const int* pos, int n, int d, int col,
                                           f32x2 hi[VEC / 2], f32x2 lo[VEC / 2]) {
  for (int q0 = 0; q0 < n; q0 += UNR) {
    GradRaw<GD, VEC> g[UNR];
#pragma unroll
    for (int r = 0; r < UNR; ++r)
      if (q0 + r < n && pos[q0 + r] >= 0) load_grad_raw<GD, VEC>(p.grads, pos[q0 + r], d, col, g[r]);
#pragma unroll
    for (int r = 0; r < UNR; ++r)
      if (q0 + r < n && pos[q0 + r] >= 0) {
#pragma unroll
        for (int j = 0; j < VEC / 2; ++j) two_sum_add(hi[j], lo[j], grad_pair<GD, VEC>(g[r], j));
      }
  }
}

// 16-byte asynchronous copy that reads src_bytes (16 or 0) from gmem and
// fills the rest of the 16 bytes with zeros: with 0, nothing is read.
__device__ __forceinline__ void cp_async16_zfill(void* smem, const void* gmem, int src_bytes) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sa), "l"(gmem), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// accumulate() with the gradient rows brought in by asynchronous 16-byte
// copies into a ring of NST stages of HS rows in shared memory (this
// thread's slots only, so no barrier is needed): NST - 1 stages are in
// flight while one is summed, and no register holds a row in flight.  Every
// stage commits one copy group, so waiting until at most NST - 1 groups are
// pending means the stage about to be summed landed.
template <int GD, int VEC, int HS, int NST>
__device__ __forceinline__ void accumulate_async(const BackwardParams& p, const int* pos, int n, int d, int col,
                                                 uint4* ring, f32x2 hi[VEC / 2], f32x2 lo[VEC / 2]) {
  constexpr int W = GradRaw<GD, VEC>::W;
  constexpr int Q = W / 4;  // 16-byte pieces of one lane's share of a row
  const size_t rowb = (size_t)d * (GD == MT_F32 ? 4 : 2);
  const char* cbase = reinterpret_cast<const char*>(p.grads) + (size_t)col * (GD == MT_F32 ? 4 : 2);
  // a row past the end or at an invalid position lands as zeros (nothing is
  // read for it), which the exact pair sum adds without change
  auto issue = [&](int st, int q0) {
#pragma unroll
    for (int r = 0; r < HS; ++r) {
      const int qq = q0 + r;
      const int v = qq < n ? pos[qq] : -1;
      const bool ok = pos_ok(p, v);
      const char* src = ok ? cbase + (size_t)v * rowb : cbase;
#pragma unroll
      for (int q = 0; q < Q; ++q) cp_async16_zfill(ring + ((st * HS + r) * Q + q) * 256, src + 16 * q, ok ? 16 : 0);
    }
    cp_async_commit();
  };
#pragma unroll
  for (int s0 = 0; s0 < NST - 1; ++s0) issue(s0, s0 * HS);
  int st = 0;
  for (int q0 = 0; q0 < n; q0 += HS) {
    issue(st == 0 ? NST - 1 : st - 1, q0 + (NST - 1) * HS);  // the slot summed last round
    cp_async_wait<NST - 1>();
#pragma unroll
    for (int r = 0; r < HS; r += 2) {
      GradRaw<GD, VEC> g0, g1;
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        const uint4 t0 = ring[((st * HS + r) * Q + q) * 256];
        const uint4 t1 = r + 1 < HS ? ring[((st * HS + r + 1) * Q + q) * 256] : make_uint4(0u, 0u, 0u, 0u);
        g0.w[4 * q] = t0.x; g0.w[4 * q + 1] = t0.y; g0.w[4 * q + 2] = t0.z; g0.w[4 * q + 3] = t0.w;
        g1.w[4 * q] = t1.x; g1.w[4 * q + 1] = t1.y; g1.w[4 * q + 2] = t1.z; g1.w[4 * q + 3] = t1.w;
      }
#pragma unroll
      for (int j = 0; j < VEC / 2; ++j) two_sum_add2(hi[j], lo[j], grad_pair<GD, VEC>(g0, j), grad_pair<GD, VEC>(g1, j));
    }
    st = st + 1 == NST ? 0 : st + 1;
  }
  cp_async_wait<0>();  // nothing of this call stays in flight
}

// fp32 gradient matrices up to this size stay in L2 while the heavy kernel
// reads them (a pooled backward's bag rows): read into registers there.
constexpr unsigned long long kL2GradBytes = 16ull << 20;

// Rows per ring stage of the heavy kernel (0: keep rows in registers) and
// stages per ring: 16-byte pieces per lane and row x rows x stages = 16.
constexpr int kHeavyStages = 4;
template <int RD, int GD>
__host__ __device__ constexpr int heavy_stage_rows() {
  return (GradRaw<GD, (RD == MT_F32 ? 4 : 8)>::W % 4) ? 0 : 4 / (GradRaw<GD, (RD == MT_F32 ? 4 : 8)>::W / 4);
}

// Heavy uniques (more than kChunk positions): each warp takes a warp-chunk;
// its teams split the positions, UNR_H gradient rows in flight per lane, and
// the teams' partial sums are combined by shuffles (lanes with the same
// index in their team hold the same columns).  A heavy unique with one
// warp-chunk applies Adam at once; otherwise the warp adds its sum to the
// unique's fp64 accumulator in L2 and the last warp-chunk to arrive applies
// Adam.
template <int RD, int GD>
__global__ void __launch_bounds__(256, 3) k_bw_heavy_reduce(const BackwardParams p) {
  constexpr int VEC = RD == MT_F32 ? 4 : 8;
  constexpr int UNR = 32 / GradRaw<GD, VEC>::W;  // register path: gradient rows in flight per lane
  constexpr int HS = heavy_stage_rows<RD, GD>();
  constexpr int Q = GradRaw<GD, VEC>::W / 4;
  extern __shared__ __align__(16) uint4 dsmem[];  // [kHeavyStages][HS][Q][256] ring, then positions
  uint4* ring = dsmem + threadIdx.x;
  int* s_pos = reinterpret_cast<int*>(dsmem + (HS > 0 ? kHeavyStages * HS * Q * 256 : 0));
  const float step_size = __int_as_float(__ldg(&p.work[2]));  // set by k_bw_plan
  const float inv_sqrt_bc2 = __int_as_float(__ldg(&p.work[3]));

  const int team_shift = p.team_shift;
  const int team = 1 << team_shift;
  const int tpw = 32 >> team_shift;  // teams per warp
  const int lane = threadIdx.x & 31;
  const int lt = lane & (team - 1);
  const int tiw = lane >> team_shift;  // team index in the warp
  const unsigned team_mask = team == 32 ? kFull : (((1u << team) - 1u) << (lane & ~(team - 1)));
  int* my_pos = s_pos + (threadIdx.x >> team_shift) * kTeamShare;
  const int d = (int)p.T.dim;
  const int col0 = lt * VEC;
  const int HWC = __ldcg(&p.ctr[1]);
  const bool l2_rows = (unsigned long long)p.grad_rows * (unsigned long long)d * 4ull <= kL2GradBytes;

  // ---- heavy warp-chunks, handed to warps one at a time (they differ in size) ----
  for (;;) {
    int wc = 0;
    if (lane == 0) wc = atomicAdd(&p.work[0], 1);
    wc = __shfl_sync(kFull, wc, 0);
    if (wc >= HWC) break;
    const int4 dsc = __ldg(&p.chunks[wc]);
    const int h = -dsc.w - 1, row = dsc.z;
    const int4 hinfo = __ldg(&p.heavy_info[h]);  // {u, warp-chunks, ...}
    const int share = (dsc.y - dsc.x + tpw - 1) / tpw;
    const int tb = min(dsc.x + tiw * share, dsc.y), te = min(tb + share, dsc.y);
    for (int c0 = 0; c0 < d; c0 += team * VEC) {
      const int col = c0 + col0;
      const bool active = col < d;
      f32x2 hi[VEC / 2], lo[VEC / 2];
#pragma unroll
      for (int j = 0; j < VEC / 2; ++j) hi[j] = lo[j] = 0ull;
      if (c0 == 0) {  // this team's share of the warp-chunk (at most kTeamShare positions)
        for (int q = lt; q < te - tb; q += team) my_pos[q] = valid_pos(p, __ldg(&p.pos_sorted[tb + q]));
        __syncwarp(team_mask);
      }
      if (active) {
        if constexpr (HS > 0 && GD == MT_F32) {
          // fp32 gradient rows few enough to stay in L2 (a pooled backward's bag rows): read into
          // registers, since the ring's two copies and two shared-memory reads per row and lane would
          // throttle the memory-instruction pipe instead
          if (l2_rows) accumulate<GD, VEC, 2>(p, my_pos, te - tb, d, col, hi, lo);
          else accumulate_async<GD, VEC, HS, kHeavyStages>(p, my_pos, te - tb, d, col, ring, hi, lo);
        } else if constexpr (HS > 0) {
          accumulate_async<GD, VEC, HS, kHeavyStages>(p, my_pos, te - tb, d, col, ring, hi, lo);
        } else {
          accumulate<GD, VEC, UNR>(p, my_pos, te - tb, d, col, hi, lo);
        }
      }
      for (int o = team; o < 32; o <<= 1) {
#pragma unroll
        for (int j = 0; j < VEC / 2; ++j) {
          const f32x2 h2 = __shfl_xor_sync(kFull, hi[j], o);
          const f32x2 l2 = __shfl_xor_sync(kFull, lo[j], o);
          two_sum_add(hi[j], lo[j], h2);
          lo[j] = add2(lo[j], l2);
        }
      }
      if (tiw == 0 && active) {
        if (hinfo.y == 1) {
          f32x2 gs[VEC / 2];
#pragma unroll
          for (int j = 0; j < VEC / 2; ++j) gs[j] = add2(hi[j], lo[j]);
          if (p.gsum_out != nullptr) store_gsum(p.gsum_out, hinfo.x, d, col, gs, VEC);
          if (row >= 0 && !p.reduce_only) adam_cols<RD, VEC>(p, row, col, gs, step_size, inv_sqrt_bc2);
        } else {
          double* a = p.acc64 + (size_t)h * d + col;
#pragma unroll
          for (int j = 0; j < VEC / 2; ++j) {
            const float2 x = upk(hi[j]), y = upk(lo[j]);
            atomicAdd(a + 2 * j, (double)x.x + (double)y.x);
            atomicAdd(a + 2 * j + 1, (double)x.y + (double)y.y);
          }
        }
      }
    }
    __syncwarp();  // my_pos is reused by the next warp-chunk
    if (hinfo.y > 1) {
      __threadfence();
      int old = 0;
      if (lane == 0) old = atomicAdd(&p.arrive[h], 1);
      old = __shfl_sync(kFull, old, 0);
      if (old == hinfo.y - 1 && tiw == 0) {  // last warp-chunk of this unique: every partial sum has landed
        __threadfence();
        for (int c0 = 0; c0 < d; c0 += team * VEC) {
          const int col = c0 + col0;
          if (col >= d) continue;
          f32x2 gs[VEC / 2];
          const double* a = p.acc64 + (size_t)h * d + col;
#pragma unroll
          for (int j = 0; j < VEC / 2; ++j) gs[j] = pk((float)__ldcg(a + 2 * j), (float)__ldcg(a + 2 * j + 1));
          if (p.gsum_out != nullptr) store_gsum(p.gsum_out, hinfo.x, d, col, gs, VEC);
          if (row >= 0 && !p.reduce_only) adam_cols<RD, VEC>(p, row, col, gs, step_size, inv_sqrt_bc2);
        }
      }
    }
  }

}

// Light uniques (at most kChunk positions): one team per unique stages the
// positions in shared memory, starts pulling the Adam row into L2, sums the
// gradient rows (UNR in flight per lane) and applies Adam.  The next
// descriptor loads while a chunk runs.
// fp32 rows with fp32 gradients fit four CTAs per SM without costly spills (measured faster); the bf16
// variants keep three.
template <int RD, int GD>
__global__ void __launch_bounds__(256, (RD == MT_F32 && GD == MT_F32) ? 4 : 3) k_bw_light_reduce(const BackwardParams p) {
  constexpr int VEC = RD == MT_F32 ? 4 : 8;
  constexpr int UNR = 16 / GradRaw<GD, VEC>::W;  // gradient rows in flight per lane (16 raw words)
  __shared__ int s_pos[kMaxTeams * kChunk];
  const float step_size = __int_as_float(__ldg(&p.work[2]));  // set by k_bw_plan
  const float inv_sqrt_bc2 = __int_as_float(__ldg(&p.work[3]));

  const int team_shift = p.team_shift;
  const int team = 1 << team_shift;
  const int lane = threadIdx.x & 31;
  const int lt = lane & (team - 1);
  const unsigned team_mask = team == 32 ? kFull : (((1u << team) - 1u) << (lane & ~(team - 1)));
  int* my_pos = s_pos + (threadIdx.x >> team_shift) * kChunk;
  const int d = (int)p.T.dim;
  const int col0 = lt * VEC;
  const long long light_end = (long long)p.light0 + *p.num_unique;  // heavy uniques' entries are empty

  const long long gteam = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> team_shift;
  const long long nteam = ((long long)gridDim.x * blockDim.x) >> team_shift;
  const bool one_pass = d <= team * VEC;
  const int gbytes = GD == MT_F32 ? 4 : 2;
  // Software pipeline over this team's uniques: while unique c is reduced,
  // the positions of the next one are in flight into registers and its Adam
  // row and gradient rows are being pulled into L2.
  constexpr int kPosRegs = kChunk >> kMinTeamShift;  // positions per lane of one team-chunk
  long long c = p.light0 + gteam;
  int4 dsc = c < light_end ? __ldg(&p.chunks[c]) : make_int4(0, 0, -1, 0);
  if (c < light_end) {
    for (int q = lt; q < dsc.y - dsc.x; q += team) my_pos[q] = valid_pos(p, __ldg(&p.pos_sorted[dsc.x + q]));
    if (one_pass && dsc.z >= 0 && col0 < d) {
      const char* rec = row_ptr(p.T, dsc.z);
      prefetch_l2(rec + (size_t)col0 * (RD == MT_F32 ? 4 : 2));
      prefetch_l2(rec + p.T.emb_bytes + (size_t)col0 * 4);
      prefetch_l2(rec + p.T.emb_bytes + p.T.mv_bytes + (size_t)col0 * 4);
    }
  }
  __syncwarp(team_mask);
  for (; c < light_end; c += nteam) {
    const int cnt = dsc.y - dsc.x, row = dsc.z;
    const bool has_next = c + nteam < light_end;
    const int4 nxt = has_next ? __ldg(&p.chunks[c + nteam]) : make_int4(0, 0, -1, 0);
    int npos[kPosRegs];
#pragma unroll
    for (int k = 0; k < kPosRegs; ++k) {
      const int q = lt + (k << team_shift);
      npos[k] = q < nxt.y - nxt.x ? valid_pos(p, __ldg(&p.pos_sorted[nxt.x + q])) : -1;
    }
    if (one_pass && nxt.z >= 0 && col0 < d) {
      const char* rec = row_ptr(p.T, nxt.z);
      prefetch_l2(rec + (size_t)col0 * (RD == MT_F32 ? 4 : 2));
      prefetch_l2(rec + p.T.emb_bytes + (size_t)col0 * 4);
      prefetch_l2(rec + p.T.emb_bytes + p.T.mv_bytes + (size_t)col0 * 4);
    }
    for (int c0 = 0; c0 < d; c0 += team * VEC) {
      const int col = c0 + col0;
      if (col >= d) continue;
      f32x2 hi[VEC / 2], lo[VEC / 2];
#pragma unroll
      for (int j = 0; j < VEC / 2; ++j) hi[j] = lo[j] = 0ull;
      accumulate<GD, VEC, UNR>(p, my_pos, cnt, d, col, hi, lo);
      if (c0 == 0) {  // the next unique's gradient rows (one 128-byte line per lane-position)
#pragma unroll
        for (int k = 0; k < kPosRegs; ++k)
          if (npos[k] >= 0) prefetch_l2(reinterpret_cast<const char*>(p.grads) + (size_t)npos[k] * d * gbytes);
      }
      f32x2 gs[VEC / 2];
#pragma unroll
      for (int j = 0; j < VEC / 2; ++j) gs[j] = add2(hi[j], lo[j]);
      if (p.gsum_out != nullptr && dsc.w >= 0) store_gsum(p.gsum_out, dsc.w, d, col, gs, VEC);
      if (row >= 0 && !p.reduce_only) adam_cols<RD, VEC>(p, row, col, gs, step_size, inv_sqrt_bc2);
    }
    __syncwarp(team_mask);  // every lane is done with my_pos
#pragma unroll
    for (int k = 0; k < kPosRegs; ++k) {
      const int q = lt + (k << team_shift);
      if (q < nxt.y - nxt.x) my_pos[q] = npos[k];
    }
    __syncwarp(team_mask);
    dsc = nxt;
  }
}

// Per device, per (row dtype, grad dtype) and per team size: grid sizes of
// the two reduce kernels; 0 = not set up yet.  The heavy kernel's
// shared-memory limit is raised once per device to its largest size (the
// smallest team), so any table's launch fits.
constexpr int kTeamShifts = 6 - kMinTeamShift;  // team of 4 .. 32 lanes
std::atomic<int> g_heavy_grid[kMaxDevices][4][kTeamShifts];
std::atomic<int> g_light_grid[kMaxDevices][4][kTeamShifts];

template <int RD, int GD>
size_t heavy_smem_bytes(int team_shift) {
  constexpr int HS = heavy_stage_rows<RD, GD>();
  constexpr int Q = GradRaw<GD, (RD == MT_F32 ? 4 : 8)>::W / 4;
  return (size_t)(HS > 0 ? kHeavyStages * HS * Q * 256 : 0) * 16 + (size_t)(256 >> team_shift) * kTeamShare * 4;
}

template <int RD, int GD>
cudaError_t launch_reduce(const BackwardParams& p, cudaStream_t s) {
  const int idx = RD * 2 + GD;
  const int dev = current_device();
  if (dev < 0 || p.team_shift < kMinTeamShift || p.team_shift > 5) return cudaErrorInvalidValue;
  const int ts = p.team_shift - kMinTeamShift;
  const size_t heavy_smem = heavy_smem_bytes<RD, GD>(p.team_shift);
  if (g_heavy_grid[dev][idx][ts].load(std::memory_order_relaxed) == 0) {
    int sms = 0, per_h = 0, per_l = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaError_t e = cudaFuncSetAttribute(k_bw_heavy_reduce<RD, GD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)heavy_smem_bytes<RD, GD>(kMinTeamShift));
    if (e != cudaSuccess) return e;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_h, k_bw_heavy_reduce<RD, GD>, 256, heavy_smem);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_l, k_bw_light_reduce<RD, GD>, 256, 0);
    g_light_grid[dev][idx][ts].store(sms * (per_l > 0 ? per_l : 1), std::memory_order_relaxed);
    g_heavy_grid[dev][idx][ts].store(sms * (per_h > 0 ? per_h : 1), std::memory_order_relaxed);
  }
  const int heavy_grid = g_heavy_grid[dev][idx][ts].load(std::memory_order_relaxed);
  const int light_grid = g_light_grid[dev][idx][ts].load(std::memory_order_relaxed);
  {
    MT_LAUNCH("k_bw_heavy_reduce", s);
    k_bw_heavy_reduce<RD, GD><<<heavy_grid, 256, heavy_smem, s>>>(p);
  }
  {
    MT_LAUNCH("k_bw_light_reduce", s);
    k_bw_light_reduce<RD, GD><<<light_grid, 256, 0, s>>>(p);
  }
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
  // a heavy unique has more than kChunk positions and at most count / kTeamShare + 1 warp-chunks (a warp-chunk
  // holds kTeamShare positions per team, one team or more), so this bounds the heavy warp-chunks
  L.light0 = (int)(n / kTeamShare + n / (kChunk + 1) + 2);
  L.ctr = take(16);
  L.seg = take(nn * 8);
  L.chunks = take(((size_t)L.light0 + nn) * 16);
  L.heavy_info = take((size_t)L.heavy_cap * 16);
  L.pos_sorted = take(nn * 4);
  L.acc64 = take((size_t)L.heavy_cap * dim * 8);
  L.arrive = take((size_t)L.heavy_cap * 4);
  L.work = take(16);
  L.total = off;
  return L;
}

void bind_backward_ws(BackwardParams& p, char* w, const BackwardWsLayout& L) {
  p.ctr = reinterpret_cast<int32_t*>(w + L.ctr);
  p.seg = reinterpret_cast<int2*>(w + L.seg);
  p.chunks = reinterpret_cast<int4*>(w + L.chunks);
  p.heavy_info = reinterpret_cast<int4*>(w + L.heavy_info);
  p.pos_sorted = reinterpret_cast<int32_t*>(w + L.pos_sorted);
  p.acc64 = reinterpret_cast<double*>(w + L.acc64);
  p.arrive = reinterpret_cast<int32_t*>(w + L.arrive);
  p.work = reinterpret_cast<int32_t*>(w + L.work);
  p.nblk = L.nblk;
  p.light0 = L.light0;
  p.ntiles = L.ntiles;
}

cudaError_t launch_backward(const BackwardParams& p, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(p.ctr, 0, 3 * sizeof(int32_t), s);
  if (e != cudaSuccess) return e;
  {
    MT_LAUNCH("k_bw_plan", s);
    k_bw_plan<<<p.nblk + 1, kScanThreads, 0, s>>>(p);  // + the block that sets up the step
  }
  if (p.ntiles > 0 && p.ranks != nullptr) {
    MT_LAUNCH("k_bw_scatter", s);
    k_bw_scatter<<<grid_for(p.n, 256, 16), 256, 0, s>>>(p);
  } else if (p.ntiles > 0) {
    MT_LAUNCH("k_bw_fill", s);
    k_bw_fill<<<p.ntiles, kThreads, 0, s>>>(p);
  }
  if (p.T.row_dtype == MT_F32) {
    return p.grad_dtype == MT_F32 ? launch_reduce<MT_F32, MT_F32>(p, s) : launch_reduce<MT_F32, MT_BF16>(p, s);
  }
  return p.grad_dtype == MT_F32 ? launch_reduce<MT_BF16, MT_F32>(p, s) : launch_reduce<MT_BF16, MT_BF16>(p, s);
}

// Team size: the smallest power of two (>= 4 lanes, <= 32) whose lanes cover
// the row at VEC columns each.
int backward_team_shift(uint32_t dim, int row_dtype) {
  const int vec = row_dtype == MT_F32 ? 4 : 8;
  int team = 1 << kMinTeamShift, shift = kMinTeamShift;
  while (team < 32 && team * vec < (int)dim) {
    team <<= 1;
    ++shift;
  }
  return shift;
}

}  // namespace mt
