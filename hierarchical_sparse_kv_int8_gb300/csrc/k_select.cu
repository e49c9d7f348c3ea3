// Step 1 of the verification round: indexer scores and per-query top-k.
//
// "Adaptive DHiSparse", section 2.1, eq. (1): the sparse indexer scores every
// historical row s against query t and selects the k best, S_t = Top-k(I_t,:),
// kept as the ordered list the model's top-k returns.  The causal domain of a
// verification query is the committed history (section 3.3, eq. (5)).
#include "dhs_internal.cuh"
#include "ptx_util.cuh"

#include <cooperative_groups.h>

#include <algorithm>
#include <climits>
#include <cstring>

namespace dhs {

// ---------------------------------------------------------------- upload
__global__ void k_upload(int32_t *dst, int n, const __grid_constant__ UploadWords w) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    dst[i] = w.w[i];
}

cudaError_t launch_upload(int32_t *dst, const int32_t *words, int n, cudaStream_t s) {
  UploadWords w;
  for (int i = 0; i < n; ++i) w.w[i] = words[i];
  static bool carve_k_upload = false;
  if (!carve_k_upload) {
    same_carveout(k_upload);
    carve_k_upload = true;
  }
  k_upload<<<(n + 255) / 256, 256, 0, s>>>(dst, n, w);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- scores
// Rows of up to 128 bytes: one thread per key row, read straight from global
// memory with 16-byte loads (each thread consumes whole 32-byte sectors); the
// K_r query chunks are shared-memory broadcasts; dp4a accumulates exact int32
// dot products.  Rows of 192 to 512 bytes in 64-byte multiples take the
// tensor cores (k_index_score_tc), as do 64- and 128-byte rows in launches
// that stream at least 256 MB of keys; other wider rows k_index_score_wide.
constexpr int kScoreThreads = 256;
constexpr int kDirectChunks = 8;  // rows up to 128 bytes use direct loads

template <int NC>
__device__ __forceinline__ void load_direct(const int8_t *__restrict__ krow, int nc_rt,
                                            uint4 (&kv)[kDirectChunks]) {
  const int nc = NC > 0 ? NC : nc_rt;
  const uint4 *p = reinterpret_cast<const uint4 *>(krow);
#pragma unroll
  for (int ch = 0; ch < kDirectChunks; ++ch)
    if (ch < nc) kv[ch] = __ldg(p + ch);
}

template <int NC>
__device__ __forceinline__ void score_direct(const uint4 (&kv)[kDirectChunks], const uint4 *qs,
                                             int Kr, int nc_rt, int (&acc)[kMaxKmax]) {
  const int nc = NC > 0 ? NC : nc_rt;
#pragma unroll
  for (int ch = 0; ch < kDirectChunks; ++ch) {
    if (ch >= nc) break;
#pragma unroll
    for (int j = 0; j < kMaxKmax; ++j) {
      if (j < Kr) {
        const uint4 qv = qs[j * nc + ch];
        acc[j] = __dp4a((int)kv[ch].x, (int)qv.x, acc[j]);
        acc[j] = __dp4a((int)kv[ch].y, (int)qv.y, acc[j]);
        acc[j] = __dp4a((int)kv[ch].z, (int)qv.z, acc[j]);
        acc[j] = __dp4a((int)kv[ch].w, (int)qv.w, acc[j]);
      }
    }
  }
}

// ctl.w holds the round's control words: K_r of every request, then the
// domain of every (request, query); the first CTA of each request publishes
// them for the later launches of the round.
template <int NC>
__global__ void __launch_bounds__(kScoreThreads)
k_index_score(const DevCtx c, const int8_t *__restrict__ q_idx,
              const __grid_constant__ UploadWords ctl) {
  extern __shared__ __align__(16) unsigned char smem[];
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.y;
  const int Kr = ctl.w[r];
  const int *qdom = ctl.w + c.N + r * c.Kmax;
  if (blockIdx.x == 0) {
    if (threadIdx.x == 0) c.Kr[r] = Kr;
    for (int j = threadIdx.x; j < c.Kmax; j += blockDim.x) c.dom[r * c.Kmax + j] = qdom[j];
  }
  if (Kr == 0) return;
  int dom_r = 0;
  for (int j = 0; j < Kr; ++j) dom_r = max(dom_r, qdom[j]);
  const int64_t row0 = (int64_t)blockIdx.x * kScoreThreads;
  if (row0 >= dom_r) return;
  const int RB = c.idx_row, nc = RB >> 4;
  const int rows = (int)(dom_r - row0 < kScoreThreads ? dom_r - row0 : kScoreThreads);
  const int8_t *keys = c.keys[r] + row0 * RB;
  // the row's key chunks are requested first, so their latency overlaps the
  // query copy below
  uint4 kv[kDirectChunks];
  if (threadIdx.x < rows) load_direct<NC>(keys + (size_t)threadIdx.x * RB, nc, kv);
  uint4 *qs = reinterpret_cast<uint4 *>(smem);
  const int8_t *qb = q_idx ? q_idx : reinterpret_cast<const int8_t *>(ctl.w + ctl_qidx_word(c.N, c.Kmax));
  const uint4 *qsrc = reinterpret_cast<const uint4 *>(qb + (size_t)r * c.Kmax * RB);
  for (int u = threadIdx.x; u < Kr * nc; u += blockDim.x) qs[u] = qsrc[u];
  __syncthreads();

  const int t = threadIdx.x;
  int acc[kMaxKmax];
#pragma unroll
  for (int j = 0; j < kMaxKmax; ++j) acc[j] = 0;
  if (t < rows) {
    score_direct<NC>(kv, qs, Kr, nc, acc);
    const int64_t s = row0 + t;
#pragma unroll
    for (int j = 0; j < kMaxKmax; ++j)
      if (j < Kr) c.scores[((size_t)r * c.Kmax + j) * c.Ss + s] = acc[j];
  }
  // range of each query's scores over its domain: one atomic per CTA and query
  __shared__ int smn[kScoreThreads / 32][kMaxKmax], smx[kScoreThreads / 32][kMaxKmax];
  const int lane = t & 31, wid = t >> 5;
#pragma unroll
  for (int j = 0; j < kMaxKmax; ++j) {
    if (j >= Kr) break;
    const bool valid = t < rows && row0 + t < qdom[j];
    int mn = valid ? acc[j] : INT_MAX, mx = valid ? acc[j] : INT_MIN;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (lane == 0) {
      smn[wid][j] = mn;
      smx[wid][j] = mx;
    }
  }
  __syncthreads();
  if (t < Kr) {
    int mn = INT_MAX, mx = INT_MIN;
#pragma unroll
    for (int w = 0; w < kScoreThreads / 32; ++w) {
      mn = min(mn, smn[w][t]);
      mx = max(mx, smx[w][t]);
    }
    if (mn <= mx) {
      atomicMin(&c.minmax[(r * c.Kmax + t) * 2 + 0], mn);
      atomicMax(&c.minmax[(r * c.Kmax + t) * 2 + 1], mx);
    }
  }
}

// Rows wider than 128 bytes: LPR lanes share a row, each holding CPL of its
// 16-byte chunks and the same chunks of every query in registers, so a warp
// reads 32 / LPR whole rows per load instruction, coalesced.  Each lane forms
// dp4a partial sums for the eight (padded) queries; a butterfly
// reduce-scatter over the row's lanes (three halving exchanges, then plain
// sums) leaves query q's score in lane q * LPR / 8 of the row's lanes.
template <int LPR, int CPL>
struct WideScore {
  static constexpr int RPW = 32 / LPR;            // rows per warp load
  static constexpr int BR = CPL == 1 ? 4 : 2;     // loads of rows in flight per lane
  static constexpr int ITERS = 4;
  static constexpr int RPB = (kScoreThreads / 32) * RPW * BR * ITERS;  // rows per CTA
};

template <int LPR, int CPL>
__global__ void __launch_bounds__(kScoreThreads)
k_index_score_wide(const DevCtx c, const int8_t *__restrict__ q_idx,
                   const __grid_constant__ UploadWords ctl) {
  using WS = WideScore<LPR, CPL>;
  constexpr int RPW = WS::RPW, BR = WS::BR;
  static_assert(kMaxKmax == 8, "the reduce-scatter is written for eight queries");
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.y;
  const int Kr = ctl.w[r];
  const int *qdom = ctl.w + c.N + r * c.Kmax;
  if (blockIdx.x == 0) {
    if (threadIdx.x == 0) c.Kr[r] = Kr;
    for (int j = threadIdx.x; j < c.Kmax; j += blockDim.x) c.dom[r * c.Kmax + j] = qdom[j];
  }
  if (Kr == 0) return;
  int dom_r = 0;
  for (int j = 0; j < Kr; ++j) dom_r = max(dom_r, qdom[j]);
  const int64_t b0 = (int64_t)blockIdx.x * WS::RPB;
  if (b0 >= dom_r) return;
  const int64_t b1 = min((int64_t)dom_r, b0 + WS::RPB);
  __shared__ int smn[kMaxKmax], smx[kMaxKmax];
  if (threadIdx.x < kMaxKmax) {
    smn[threadIdx.x] = INT_MAX;
    smx[threadIdx.x] = INT_MIN;
  }
  __syncthreads();

  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int RB = c.idx_row, NC = RB >> 4;
  const int sub = lane % LPR, rsub = lane / LPR;
  // this lane's chunks of every query (zero past K_r and past the row)
  const int8_t *qb = q_idx ? q_idx : reinterpret_cast<const int8_t *>(ctl.w + ctl_qidx_word(c.N, c.Kmax));
  uint4 qv[kMaxKmax][CPL];
#pragma unroll
  for (int j = 0; j < kMaxKmax; ++j)
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int ch = sub + i * LPR;
      qv[j][i] = (j < Kr && ch < NC)
                     ? *reinterpret_cast<const uint4 *>(qb + ((size_t)r * c.Kmax + j) * RB + ch * 16)
                     : make_uint4(0u, 0u, 0u, 0u);
    }
  // after the reduce-scatter this lane holds query qm's score; one lane per
  // (row, query) writes it
  const int qm = ((lane & (LPR / 2)) ? 4 : 0) + ((lane & (LPR / 4)) ? 2 : 0) +
                 ((lane & (LPR / 8)) ? 1 : 0);
  const bool writer = (lane & (LPR / 8 - 1)) == 0 && qm < Kr;
  const int dq = qm < Kr ? qdom[qm] : 0;
  int mn = INT_MAX, mx = INT_MIN;
  const int8_t *keys = c.keys[r];
  int32_t *out = c.scores + ((size_t)r * c.Kmax + min(qm, c.Kmax - 1)) * c.Ss;
  constexpr int kWarps = kScoreThreads / 32;
  for (int64_t g0 = b0 + wid * RPW; g0 < b1; g0 += (int64_t)kWarps * RPW * BR) {
    uint4 kv[BR][CPL];
#pragma unroll
    for (int b = 0; b < BR; ++b) {
      const int64_t s = g0 + (int64_t)b * kWarps * RPW + rsub;
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const int ch = sub + i * LPR;
        kv[b][i] = (s < b1 && ch < NC)
                       ? __ldg(reinterpret_cast<const uint4 *>(keys + s * RB + ch * 16))
                       : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int b = 0; b < BR; ++b) {
      int v[kMaxKmax];
#pragma unroll
      for (int j = 0; j < kMaxKmax; ++j) {
        int a = 0;
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          a = __dp4a((int)kv[b][i].x, (int)qv[j][i].x, a);
          a = __dp4a((int)kv[b][i].y, (int)qv[j][i].y, a);
          a = __dp4a((int)kv[b][i].z, (int)qv[j][i].z, a);
          a = __dp4a((int)kv[b][i].w, (int)qv[j][i].w, a);
        }
        v[j] = a;
      }
      {  // 8 values -> 4 (partner at distance LPR / 2)
        const bool up = lane & (LPR / 2);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int send = up ? v[i] : v[i + 4];
          v[i] = (up ? v[i + 4] : v[i]) + __shfl_xor_sync(0xffffffffu, send, LPR / 2);
        }
      }
      {  // 4 -> 2
        const bool up = lane & (LPR / 4);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int send = up ? v[i] : v[i + 2];
          v[i] = (up ? v[i + 2] : v[i]) + __shfl_xor_sync(0xffffffffu, send, LPR / 4);
        }
      }
      {  // 2 -> 1
        const bool up = lane & (LPR / 8);
        const int send = up ? v[0] : v[1];
        v[0] = (up ? v[1] : v[0]) + __shfl_xor_sync(0xffffffffu, send, LPR / 8);
      }
#pragma unroll
      for (int d = LPR / 16; d >= 1; d >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], d);
      const int64_t s = g0 + (int64_t)b * kWarps * RPW + rsub;
      if (writer && s < b1) {
        out[s] = v[0];
        if (s < dq) {
          mn = min(mn, v[0]);
          mx = max(mx, v[0]);
        }
      }
    }
  }
  // range of each query's scores: shared-memory atomics, then one global
  // atomic per CTA and query
  if (writer && mn <= mx) {
    atomicMin(&smn[qm], mn);
    atomicMax(&smx[qm], mx);
  }
  __syncthreads();
  if (threadIdx.x < Kr && smn[threadIdx.x] <= smx[threadIdx.x]) {
    atomicMin(&c.minmax[(r * c.Kmax + threadIdx.x) * 2 + 0], smn[threadIdx.x]);
    atomicMax(&c.minmax[(r * c.Kmax + threadIdx.x) * 2 + 1], smx[threadIdx.x]);
  }
}

// ---------------------------------------------------------------- top-k
// One thread-block cluster of kTopkCluster CTAs per (request, query); CTA c
// of the cluster owns the c-th contiguous quarter of the query's domain.
//  (1) the score range comes from the scoring kernel;
//  (2) exact radix select on the score minus the minimum, at most 13 bits
//      per pass (one pass when the scores span fewer than 8192 values): each
//      CTA histograms its rows, then every CTA sums the cluster's histograms
//      through distributed shared memory and finds the same threshold;
//  (3) ordered collection: each warp owns a contiguous run of rows, counts
//      those above the threshold and those equal to it; after the counts of
//      all warps and CTAs are known every warp writes its rows, in row order,
//      into the leader CTA's candidate array (the lowest-index rows win the
//      ties at the threshold);
//  (4) the leader sorts the k winners by (score descending, row ascending)
//      with a bitonic network held in registers, two elements per thread,
//      exchanging through shared memory only for strides that cross warps.
constexpr int kTopkThreads = 1024;
constexpr int kTopkCluster = 4;
constexpr int kRadixBits = 13;
constexpr int kBinsPerThread = (1 << kRadixBits) / kTopkThreads;
constexpr int kTopkSpinLimit = 1 << 22;  // bounded wait for the staged scores
static_assert(kMaxTopk <= 2 * kTopkThreads, "the exact placement holds two winners per thread");

__device__ __forceinline__ int block_excl_scan(int v, int *warp_sums, int &total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  total = warp_sums[nw - 1];
  int excl = x - v + (wid > 0 ? warp_sums[wid - 1] : 0);
  __syncthreads();
  return excl;
}

__device__ __forceinline__ unsigned long long topk_key(uint32_t v, int s) {
  return ((unsigned long long)(0xFFFFFFFFu - v) << 32) | (uint32_t)s;
}

// Compare-exchange of a bitonic stage between two registers of one thread.
__device__ __forceinline__ void cmpx(unsigned long long &lo, unsigned long long &hi, bool asc) {
  if ((lo > hi) == asc) {
    const unsigned long long t = lo;
    lo = hi;
    hi = t;
  }
}

// Ascending bitonic sort of kp (a power of two, <= 2 * blockDim.x) keys,
// element e = 2 * thread + h held in x[h]; buf is kp keys of shared memory.
__device__ void bitonic_sort_regs(unsigned long long (&x)[2], unsigned long long *buf, int kp) {
  const int t = threadIdx.x, lane = t & 31;
  const bool active = 2 * t < kp;
  const bool warp_active = (t >> 5) * 64 < kp;  // warps past the data skip register stages
  for (int size = 2; size <= kp; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const int e0 = 2 * t;
      const bool asc = (e0 & size) == 0;
      if (stride == 1) {
        if (active) cmpx(x[0], x[1], asc);
      } else if (stride <= 32) {
        if (!warp_active) continue;
        // partner thread t ^ (stride / 2) holds e ^ stride; both lanes keep
        // the value their position should hold
        const int pm = stride >> 1;
        const bool lower = (t & pm) == 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const unsigned long long o = __shfl_xor_sync(0xffffffffu, x[h], pm);
          const bool keep_min = lower == asc;
          x[h] = keep_min ? (x[h] < o ? x[h] : o) : (x[h] > o ? x[h] : o);
        }
      } else {
        __syncthreads();
        if (active) {
          buf[e0] = x[0];
          buf[e0 + 1] = x[1];
        }
        __syncthreads();
        if (active) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int e = e0 + h;
            const unsigned long long o = buf[e ^ stride];
            const bool lower = (e & stride) == 0;
            const bool keep_min = lower == asc;
            x[h] = keep_min ? (x[h] < o ? x[h] : o) : (x[h] > o ? x[h] : o);
          }
        }
      }
    }
  }
  (void)lane;
}

__global__ void __cluster_dims__(kTopkCluster, 1, 1) __launch_bounds__(kTopkThreads)
k_topk(const DevCtx c, int32_t *__restrict__ topk_out, int stage_cap) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  extern __shared__ __align__(16) unsigned char smem[];
  pdl_wait();
  pdl_trigger();
  const int crank = (int)cl.block_rank();
  const int prob = blockIdx.x / kTopkCluster;
  const int r = prob / c.Kmax, j = prob % c.Kmax;
  // the round's control values, requested together (all are in range
  // whatever K_r is)
  const int Kr = c.Kr[r];
  const int dom = c.dom[r * c.Kmax + j];
  const int lo = c.minmax[(r * c.Kmax + j) * 2 + 0];
  const int hi = c.minmax[(r * c.Kmax + j) * 2 + 1];
  if (j >= Kr) return;  // the whole cluster leaves together
  // (split cluster barrier: every CTA has started before any CTA writes into
  // another's shared memory; the wait follows the staging copy)
  cluster_arrive_relaxed();
  const int k = c.k;
  const int32_t *__restrict__ sc = c.scores + ((size_t)r * c.Kmax + j) * c.Ss;
  int32_t *out = topk_out + ((size_t)r * c.Kmax + j) * k;
  int kp = 1;
  while (kp < k) kp <<= 1;
  unsigned long long *cand = reinterpret_cast<unsigned long long *>(smem);
  uint32_t *hist = reinterpret_cast<uint32_t *>(cand + kp);
  __shared__ int warp_sums[32];
  __shared__ int wgt[32], weq[32];
  __shared__ int sh_bin, sh_above, sh_cta_gt, sh_cta_eq;
  __shared__ int tot_eq[kTopkCluster];  // every CTA's rows equal to T, pushed by that CTA
  __shared__ int ccnt[kTopkThreads];  // per-thread run counts of a radix pass
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int ksel = min(k, dom);
  const int part = (((dom + kTopkCluster - 1) / kTopkCluster) + 31) & ~31;
  const int p0 = min(dom, crank * part), p1 = min(dom, p0 + part);
  // This CTA's part of the scores, read by every pass below: when it fits
  // (stage_cap scores), one bulk asynchronous copy brings it into shared
  // memory first; otherwise the passes read global memory.
  const bool staged = p1 - p0 <= stage_cap && dom > k;
  int32_t *stg = reinterpret_cast<int32_t *>(smem + (((size_t)kp * 8 + 15) & ~(size_t)15) +
                                             ((size_t)2 << kRadixBits) * 4);
  // The first radix pass's histogram size (also computed by the pass loop).
  const uint32_t range = (uint32_t)(hi - lo);
  const int shift0 = range ? 32 - __clz((int)range) : 0;
  const int nbins0 = shift0 > 0 ? 1 << min(kRadixBits, shift0) : 0;
  const bool prezeroed = staged && p1 > p0 && dom > k;
  if (staged && p1 > p0) {
    __shared__ __align__(8) uint64_t sbar;
    if (tid == 0) {
      mbar_init(&sbar, 1);
      fence_proxy_async_smem();
      const uint32_t bytes = (uint32_t)(((p1 - p0) * 4 + 15) & ~15);
      mbar_arrive_expect_tx(&sbar, bytes);
      bulk_g2s(stg, sc + p0, bytes, &sbar);
    }
    // the first pass's histogram is cleared while the copy is in flight
    if (prezeroed)
      for (int i = tid; i < nbins0; i += kTopkThreads) hist[i] = 0;
    // one warp waits for the copy; the block barrier then releases the rest
    if (wid == 0) {
      __syncwarp();
      int spins = 0;
      while (!mbar_try_wait(&sbar, 0u))
        if (++spins > kTopkSpinLimit) {
          record_error(c.err, DC_TIMEOUT, K_TOPK);
          spins = 0;
          while (!mbar_try_wait(&sbar, 0u) && ++spins <= kTopkSpinLimit) {
          }
          break;
        }
    }
    __syncthreads();
  }
  cluster_wait();
  auto val = [&](int s) -> int32_t { return staged ? stg[s - p0] : sc[s]; };
  // the scores of rows s0..s0+3, s0 - p0 a multiple of 4 (16-byte aligned in
  // the stage and in the padded score row; the caller masks rows past its end)
  auto val4 = [&](int s0) -> int4 {
    return staged ? *reinterpret_cast<const int4 *>(stg + (s0 - p0))
                  : __ldg(reinterpret_cast<const int4 *>(sc + s0));
  };
  // Once every CTA of the cluster has read the range (after its first
  // cluster barrier), the leader empties it for the next round's scores.
  auto empty_range = [&]() {
    if (crank == 0 && tid == 0) {
      c.minmax[(r * c.Kmax + j) * 2 + 0] = INT_MAX;
      c.minmax[(r * c.Kmax + j) * 2 + 1] = INT_MIN;
    }
  };

  int nloc = 0;  // candidates this CTA holds
  if (dom <= k) {
    for (int s = p0 + tid; s < p1; s += kTopkThreads)
      cand[s - p0] = topk_key((uint32_t)(val(s) - lo), s);
    nloc = p1 - p0;
  } else {
    int shift = shift0;
    uint32_t prefix = 0;
    int k_rem = k;
    int *rcnt = reinterpret_cast<int *>(hist) + (2 << kRadixBits) - kTopkCluster * kTopkThreads;
    const uint32_t *hr[kTopkCluster];
#pragma unroll
    for (int q = 0; q < kTopkCluster; ++q) hr[q] = cl.map_shared_rank(hist, q);
    int passes = 0, nb_last = 1;
    while (shift > 0) {
      const int width = min(kRadixBits, shift);
      shift -= width;
      const int nbins = 1 << width;
      ++passes;
      nb_last = nbins;
      if (passes > 1) cl.sync();  // every CTA has finished reading the previous histograms
      if (!(passes == 1 && prezeroed))
        for (int i = tid; i < nbins; i += kTopkThreads) hist[i] = 0;
      __syncthreads();
      if (passes == 1 && staged) {
        // the first pass counts every row (v <= range < 2^(shift + width)),
        // four staged scores per load
        const int n = p1 - p0, n4 = n >> 2;
        const int4 *s4 = reinterpret_cast<const int4 *>(stg);
#pragma unroll 2
        for (int i = tid; i < n4; i += kTopkThreads) {
          const int4 x = s4[i];
          atomicAdd(&hist[((uint32_t)(x.x - lo) >> shift) & (nbins - 1)], 1u);
          atomicAdd(&hist[((uint32_t)(x.y - lo) >> shift) & (nbins - 1)], 1u);
          atomicAdd(&hist[((uint32_t)(x.z - lo) >> shift) & (nbins - 1)], 1u);
          atomicAdd(&hist[((uint32_t)(x.w - lo) >> shift) & (nbins - 1)], 1u);
        }
        for (int i = 4 * n4 + tid; i < n; i += kTopkThreads)
          atomicAdd(&hist[((uint32_t)(stg[i] - lo) >> shift) & (nbins - 1)], 1u);
      } else if (passes == 1) {
        // likewise from global memory, four batches of four scores per
        // thread in flight
        const int n = p1 - p0, n4 = n >> 2;
        for (int i0 = tid; i0 < n4; i0 += 4 * kTopkThreads) {
          int4 x[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * kTopkThreads;
            if (i < n4) x[u] = val4(p0 + 4 * i);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (i0 + u * kTopkThreads >= n4) continue;
            atomicAdd(&hist[((uint32_t)(x[u].x - lo) >> shift) & (nbins - 1)], 1u);
            atomicAdd(&hist[((uint32_t)(x[u].y - lo) >> shift) & (nbins - 1)], 1u);
            atomicAdd(&hist[((uint32_t)(x[u].z - lo) >> shift) & (nbins - 1)], 1u);
            atomicAdd(&hist[((uint32_t)(x[u].w - lo) >> shift) & (nbins - 1)], 1u);
          }
        }
        for (int s = p0 + 4 * n4 + tid; s < p1; s += kTopkThreads)
          atomicAdd(&hist[((uint32_t)(val(s) - lo) >> shift) & (nbins - 1)], 1u);
      } else {
#pragma unroll 4
        for (int s = p0 + tid; s < p1; s += kTopkThreads) {
          const uint32_t v = (uint32_t)(val(s) - lo);
          if ((uint32_t)((unsigned long long)v >> (shift + width)) == prefix)
            atomicAdd(&hist[(v >> shift) & (nbins - 1)], 1u);
        }
      }
      // thread t owns a run of bins counted from the top; the runs' counts
      // in this CTA first, so that only runs at or above the threshold need
      // the cluster's bins one by one
      const int per = (nbins + kTopkThreads - 1) / kTopkThreads;
      const int b_hi = nbins - tid * per;
      const int b_lo = max(0, b_hi - per);
      __syncthreads();  // this CTA's histogram is complete
      {
        // (vector reads: a run of 2, 4 or 8 bins starts at a multiple of its
        // length, and the histogram area is 16-byte aligned)
        int lc = 0;
        if (b_hi - b_lo == 8) {
          const uint4 x = *reinterpret_cast<const uint4 *>(hist + b_lo);
          const uint4 y = *reinterpret_cast<const uint4 *>(hist + b_lo + 4);
          lc = (int)(x.x + x.y + x.z + x.w + y.x + y.y + y.z + y.w);
        } else if (b_hi - b_lo == 4) {
          const uint4 x = *reinterpret_cast<const uint4 *>(hist + b_lo);
          lc = (int)(x.x + x.y + x.z + x.w);
        } else if (b_hi - b_lo == 2) {
          const uint2 x = *reinterpret_cast<const uint2 *>(hist + b_lo);
          lc = (int)(x.x + x.y);
        } else {
          for (int b = b_lo; b < b_hi; ++b) lc += (int)hist[b];
        }
        ccnt[tid] = lc;
        // and into every CTA's copy of the cluster's run counts (remote
        // stores, ordered by the barrier below; the copies sit at the top of
        // the base area, which is written only after they are read)
#pragma unroll
        for (int q = 0; q < kTopkCluster; ++q)
          *cl.map_shared_rank(rcnt + crank * kTopkThreads + tid, q) = lc;
      }
      cl.sync();  // all histograms and run counts of the cluster are complete
      int local = 0;  // the run's count in the cluster
#pragma unroll
      for (int q = 0; q < kTopkCluster; ++q) local += rcnt[q * kTopkThreads + tid];
      // an exclusive scan in thread order counts the rows above each run
      int total;
      const int above = block_excl_scan(local, warp_sums, total);
      const bool exact_pass = passes == 1 && shift == 0;
      // The thread whose run holds the threshold finds its bin; in the exact
      // pass every run at or above the threshold in which this CTA has rows
      // also needs base[b] = rows of the domain above offset value b plus
      // rows equal to b in earlier CTAs, which decides the place of each of
      // its winners.  Both need the cluster's count of each bin of the run.
      const bool thr = local > 0 && above < k_rem && k_rem <= above + local;
      const bool need_base = exact_pass && ccnt[tid] > 0 && above < k_rem;
      int *base = reinterpret_cast<int *>(hist + (1 << kRadixBits));
      // The runs at or above the threshold are the first nq threads' (above
      // grows in thread order), so their bins form one window at the top.
      // When it fits in the candidate area (free until the collection) it is
      // gathered once, consecutive threads reading consecutive bins, as the
      // cluster count G and the count in earlier CTAs P of every bin; else
      // each run reads its own bins.
      int *G = reinterpret_cast<int *>(cand), *P = G + kp;
      int b_min = nbins;
      bool win = false;
      if (exact_pass) {
        const int nq = __syncthreads_count(above < k_rem);
        b_min = max(0, nbins - nq * per);
        win = nbins - b_min <= kp;
        if (win) {
          for (int b = b_min + tid; b < nbins; b += kTopkThreads) {
            int hv[kTopkCluster];
#pragma unroll
            for (int q = 0; q < kTopkCluster; ++q) hv[q] = (int)hr[q][b];
            int g = 0, pc = 0;
#pragma unroll
            for (int q = 0; q < kTopkCluster; ++q) {
              g += hv[q];
              if (q < crank) pc += hv[q];
            }
            G[b - b_min] = g;
            P[b - b_min] = pc;
          }
          __syncthreads();
        }
      }
      if (win && (thr || need_base)) {
        // (this thread's run lies in the window: it is one of the first nq)
        if (thr) {
          int acc = above;
          for (int b = b_hi - 1; b >= b_lo; --b) {
            const int g = G[b - b_min];
            if (acc + g >= k_rem) {
              sh_bin = b;
              sh_above = acc;
              break;
            }
            acc += g;
          }
        }
        if (need_base) {
          int acc = above;
          for (int b = b_hi - 1; b >= b_lo; --b) {
            base[b] = acc + P[b - b_min];
            acc += G[b - b_min];
          }
        }
      } else if (thr || need_base) {
        int gsum[kBinsPerThread], psum[kBinsPerThread];  // cluster count; count in earlier CTAs
#pragma unroll
        for (int t = 0; t < kBinsPerThread; ++t) gsum[t] = psum[t] = 0;
        auto add = [&](int t, uint32_t v, int q) {
          gsum[t] += (int)v;
          if (q < crank) psum[t] += (int)v;
        };
        if (b_hi - b_lo == 8) {  // vector reads, as for the run counts
#pragma unroll
          for (int q = 0; q < kTopkCluster; ++q) {
            const uint4 x = *reinterpret_cast<const uint4 *>(hr[q] + b_lo);
            const uint4 y = *reinterpret_cast<const uint4 *>(hr[q] + b_lo + 4);
            add(0, x.x, q); add(1, x.y, q); add(2, x.z, q); add(3, x.w, q);
            add(4, y.x, q); add(5, y.y, q); add(6, y.z, q); add(7, y.w, q);
          }
        } else if (b_hi - b_lo == 4) {
#pragma unroll
          for (int q = 0; q < kTopkCluster; ++q) {
            const uint4 x = *reinterpret_cast<const uint4 *>(hr[q] + b_lo);
            add(0, x.x, q); add(1, x.y, q); add(2, x.z, q); add(3, x.w, q);
          }
        } else {
#pragma unroll
          for (int t = 0; t < kBinsPerThread; ++t) {
            const int b = b_lo + t;
            if (b < b_hi) {
#pragma unroll
              for (int q = 0; q < kTopkCluster; ++q) add(t, hr[q][b], q);
            }
          }
        }
        if (thr) {
          int acc = above;
#pragma unroll
          for (int t = kBinsPerThread - 1; t >= 0; --t) {
            const int b = b_lo + t;
            if (b >= b_hi) continue;
            if (acc + gsum[t] >= k_rem) {
              sh_bin = b;
              sh_above = acc;
              break;
            }
            acc += gsum[t];
          }
        }
        if (need_base) {
          int acc = above;
#pragma unroll
          for (int t = kBinsPerThread - 1; t >= 0; --t) {
            const int b = b_lo + t;
            if (b >= b_hi) continue;
            base[b] = acc + psum[t];
            acc += gsum[t];
          }
        }
      }
      __syncthreads();
      k_rem -= sh_above;
      prefix = (prefix << width) | (uint32_t)sh_bin;
      __syncthreads();
    }
    const uint32_t T = prefix;  // the k-th largest offset score
    const int need = k_rem;     // rows equal to T that are kept
    const int c_gt = k - need;  // rows strictly above T

    // counts of this CTA's warps, then of the cluster's CTAs
    // (runs of a multiple of 128 rows, so that the vector reads below stay
    // inside the warp's own run)
    const int run = ((((p1 - p0) + 31) / 32) + 127) & ~127;
    const int r0 = min(p1, p0 + wid * run), r1 = min(p1, r0 + run);
    const unsigned lt = (1u << lane) - 1u;
    // With staged scores and exact bins, the counting pass also compacts the
    // warp's winners, in row order, into the front of its own run of the
    // stage (a write never lands beyond the rows already read), packed as
    // (above T, value, row - p0); the collection then reads only these lists.
    // Each lane reads four consecutive rows at a time; a group of 128 rows
    // with no row at or above T costs one vote.
    const bool inplace = staged && passes <= 1;
    uint32_t *wl = reinterpret_cast<uint32_t *>(stg) + (r0 - p0);
    int ngt = 0, neq = 0, wcount = 0;
    if (inplace) {
      int gt_lane = 0;
      for (int base = r0; base < r1; base += 128) {
        const int s0 = base + 4 * lane;  // s0 - p0 is a multiple of 4
        int4 x = make_int4(0, 0, 0, 0);
        if (s0 < r1) x = *reinterpret_cast<const int4 *>(stg + (s0 - p0));
        const uint32_t v[4] = {(uint32_t)(x.x - lo), (uint32_t)(x.y - lo), (uint32_t)(x.z - lo),
                               (uint32_t)(x.w - lo)};
        bool cnd[4];
        int nc = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          cnd[i] = s0 + i < r1 && v[i] >= T;
          nc += cnd[i];
        }
        if (!__any_sync(0xffffffffu, nc > 0)) continue;
        // row order: every candidate of the lanes below, then the lane's own
        unsigned bal[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) bal[i] = __ballot_sync(0xffffffffu, cnd[i]);
        int pos = wcount;
#pragma unroll
        for (int i = 0; i < 4; ++i) pos += __popc(bal[i] & lt);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (!cnd[i]) continue;
          const bool gt = v[i] > T;
          gt_lane += gt;
          wl[pos++] = (gt ? 0x80000000u : 0u) | (v[i] << 17) | (uint32_t)(s0 + i - p0);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) wcount += __popc(bal[i]);
      }
      ngt = (int)__reduce_add_sync(0xffffffffu, (unsigned)gt_lane);
      neq = wcount - ngt;
    } else {
      // four rows per lane and load; per-lane counts, summed once
      int gt_lane = 0, eq_lane = 0;
#pragma unroll 2
      for (int base = r0; base < r1; base += 128) {
        const int s0 = base + 4 * lane;
        if (s0 >= r1) continue;
        const int4 x = val4(s0);
        const uint32_t v[4] = {(uint32_t)(x.x - lo), (uint32_t)(x.y - lo), (uint32_t)(x.z - lo),
                               (uint32_t)(x.w - lo)};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const bool ok = s0 + i < r1;
          gt_lane += ok && v[i] > T;
          eq_lane += ok && v[i] == T;
        }
      }
      ngt = (int)__reduce_add_sync(0xffffffffu, (unsigned)gt_lane);
      neq = (int)__reduce_add_sync(0xffffffffu, (unsigned)eq_lane);
    }
    if (lane == 0) {
      wgt[wid] = ngt;
      weq[wid] = neq;
    }
    __syncthreads();
    int gx = wgt[lane], ex = weq[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ga = __shfl_up_sync(0xffffffffu, gx, o), ea = __shfl_up_sync(0xffffffffu, ex, o);
      if (lane >= o) {
        gx += ga;
        ex += ea;
      }
    }
    if (tid == 31) {
      sh_cta_gt = gx;
      sh_cta_eq = ex;
#pragma unroll
      for (int q = 0; q < kTopkCluster; ++q) *cl.map_shared_rank(&tot_eq[crank], q) = ex;
    }
    int gt_off = __shfl_sync(0xffffffffu, gx - wgt[lane], wid);   // within this CTA
    int eq_off = __shfl_sync(0xffffffffu, ex - weq[lane], wid);
    cl.sync();  // every CTA's totals are published
    empty_range();
    int eq_base = 0;  // rows equal to T in earlier CTAs
#pragma unroll
    for (int q = 0; q < kTopkCluster; ++q)
      if (q < crank) eq_base += tot_eq[q];
    cluster_arrive();  // this CTA's distributed reads are done; waited for before it leaves
    const int my_gt = sh_cta_gt, my_eq = sh_cta_eq;
    const int kept_eq = max(0, min(my_eq, need - eq_base));
    nloc = my_gt + kept_eq;
    // Exact bins (one radix pass, or none): every winner's place follows from
    // the histograms (base[], formed in the pass); the rows equal to a value
    // in this CTA follow in row order.  No CTA reads another's histogram after
    // the cluster barrier above, so the histogram area is free for reuse.
    const bool exact = passes <= 1;
    const int *base = reinterpret_cast<const int *>(hist + (1 << kRadixBits));
    const int gt_end = gt_off + ngt, eq_end = eq_off + neq;
    if (inplace) {
      for (int i0 = 0; i0 < wcount; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t e = i < wcount ? wl[i] : 0u;
        const bool gt = i < wcount && (e >> 31), eq = i < wcount && !(e >> 31);
        const unsigned bgt = __ballot_sync(0xffffffffu, gt);
        const unsigned beq = __ballot_sync(0xffffffffu, eq);
        const uint32_t v = (e >> 17) & 0x3FFFu;
        const int s = p0 + (int)(e & 0x1FFFFu);
        if (gt) cand[gt_off + __popc(bgt & lt)] = topk_key(v, s);
        if (eq) {
          const int rr = eq_off + __popc(beq & lt);  // rank among this CTA's ties
          if (rr < kept_eq) out[c_gt + eq_base + rr] = s;
        }
        gt_off += __popc(bgt);
        eq_off += __popc(beq);
      }
    }
    // (four rows per lane and load, in row order: lanes first, then the
    // lane's own rows)
    for (int bs = r0; !inplace && bs < r1 &&
                      (gt_off < gt_end || (eq_off < eq_end && eq_off < kept_eq));
         bs += 128) {
      const int s0 = bs + 4 * lane;
      int4 x = make_int4(0, 0, 0, 0);
      if (s0 < r1) x = val4(s0);
      const uint32_t v[4] = {(uint32_t)(x.x - lo), (uint32_t)(x.y - lo), (uint32_t)(x.z - lo),
                             (uint32_t)(x.w - lo)};
      bool gt[4], eq[4];
      unsigned bg[4], be[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool ok = s0 + i < r1;
        gt[i] = ok && v[i] > T;
        eq[i] = ok && v[i] == T;
        bg[i] = __ballot_sync(0xffffffffu, gt[i]);
        be[i] = __ballot_sync(0xffffffffu, eq[i]);
      }
      int pg = gt_off, pe = eq_off;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        pg += __popc(bg[i] & lt);
        pe += __popc(be[i] & lt);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (gt[i]) cand[pg++] = topk_key(v[i], s0 + i);
        if (eq[i]) {
          const int rr = pe++;  // rank among this CTA's ties
          if (rr < kept_eq) {
            if (exact) out[c_gt + eq_base + rr] = s0 + i;
            else cand[my_gt + rr] = topk_key(v[i], s0 + i);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        gt_off += __popc(bg[i]);
        eq_off += __popc(be[i]);
      }
    }
    if (exact) {
      // This CTA's winners above T, one thread each: a winner of value v takes
      // a slot of v's group [base[v], base[v] + count) with a shared-memory
      // atomic, then its place in the group is the number of the group's rows
      // below its own (row order among equal values).  The candidate area
      // holds the claimed rows meanwhile.
      constexpr int kPer = 2;  // winners per thread: my_gt <= k <= 2 * kTopkThreads
      int *lcnt = reinterpret_cast<int *>(hist);
      for (int i = tid; i < nb_last; i += kTopkThreads) lcnt[i] = 0;
      __syncthreads();  // every warp's winners are in the candidate area
      uint32_t wv[kPer];
      int wrow[kPer];
#pragma unroll
      for (int h = 0; h < kPer; ++h) {
        const int i = tid + h * kTopkThreads;
        const unsigned long long key = i < my_gt ? cand[i] : 0ull;
        wv[h] = 0xFFFFFFFFu - (uint32_t)(key >> 32);
        wrow[h] = i < my_gt ? (int32_t)(uint32_t)(key & 0xFFFFFFFFull) : -1;
      }
      __syncthreads();  // candidates read: the area now holds the claimed rows
      int *claimed = reinterpret_cast<int *>(cand);
#pragma unroll
      for (int h = 0; h < kPer; ++h) {
        if (wrow[h] < 0) continue;
        if (wv[h] >= (uint32_t)nb_last) {
          record_error(c.err, DC_CAPACITY, K_TOPK);
          wrow[h] = -1;
          continue;
        }
        const int pos = base[wv[h]] + atomicAdd(&lcnt[wv[h]], 1);
        if (pos < 0 || pos >= c_gt) {
          record_error(c.err, DC_CAPACITY, K_TOPK);
          wrow[h] = -1;
          continue;
        }
        claimed[pos] = wrow[h];
      }
      __syncthreads();
#pragma unroll
      for (int h = 0; h < kPer; ++h) {
        if (wrow[h] < 0) continue;
        const int b = base[wv[h]], cnt = min(lcnt[wv[h]], c_gt - b);
        int rank = 0;
        for (int t = 0; t < cnt; ++t) rank += claimed[b + t] < wrow[h];
        out[b + rank] = wrow[h];
      }
      if (crank == 0)
        for (int i = ksel + tid; i < k; i += kTopkThreads) out[i] = -1;
      cluster_wait();  // no CTA leaves while another may read its counts
      return;
    }
    cluster_wait();
  }
  // each CTA sorts its own candidates ...
  __shared__ int sh_nloc;
  if (tid == 0) sh_nloc = nloc;
  int kpl = 1;
  while (kpl < nloc) kpl <<= 1;
  __syncthreads();
  unsigned long long x[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int e = 2 * tid + h;
    x[h] = e < nloc ? cand[e] : ~0ull;
  }
  if (nloc > 1) bitonic_sort_regs(x, cand, kpl);
  __syncthreads();
#pragma unroll
  for (int h = 0; h < 2; ++h)
    if (2 * tid + h < nloc) cand[2 * tid + h] = x[h];
  cl.sync();  // every CTA's sorted list is in place
  empty_range();
  // ... copies the other CTAs' lists next to it (one pass of distributed
  // shared-memory reads into the histogram area, free by now) ...
  int lens[kTopkCluster], offs[kTopkCluster];
  int tot = 0;
#pragma unroll
  for (int q = 0; q < kTopkCluster; ++q) {
    lens[q] = *cl.map_shared_rank(&sh_nloc, q);
    offs[q] = tot;
    tot += lens[q];
  }
  unsigned long long *all = reinterpret_cast<unsigned long long *>(hist);
#pragma unroll
  for (int q = 0; q < kTopkCluster; ++q) {
    if (q == crank) continue;
    const unsigned long long *src = cl.map_shared_rank(cand, q);
    for (int i = tid; i < lens[q]; i += kTopkThreads) all[offs[q] + i] = src[i];
  }
  cl.sync();  // copies done: no CTA reads another's memory after this
  // ... and places each key by counting the smaller keys of the other lists
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int e = 2 * tid + h;
    if (e >= nloc) continue;
    const unsigned long long key = x[h];
    int pos = e;
#pragma unroll
    for (int q = 0; q < kTopkCluster; ++q) {
      if (q == crank) continue;
      const unsigned long long *lst = all + offs[q];
      int a = 0, b = lens[q];  // lower bound of key in list q
      while (a < b) {
        const int m = (a + b) >> 1;
        if (lst[m] < key) a = m + 1; else b = m;
      }
      pos += a;
    }
    if (pos < k) out[pos] = (int32_t)(uint32_t)(key & 0xFFFFFFFFull);
  }
  if (crank == 0)
    for (int i = ksel + tid; i < k; i += kTopkThreads) out[i] = -1;
}

// ---------------------------------------------------------------- top-k, one CTA per query
// For rounds with at least as many active queries as SMs: each (request,
// query) is one CTA of kRowThreads threads with a 32 KB histogram and a
// 32 KB candidate area, so several CTAs share an SM and one's passes over
// global memory overlap another's placement.
//  (1) exact radix select on the offset scores (13 bits a pass) over global
//      memory, several 16-byte loads in flight per thread; the pass that
//      resolves the last bits also counts the rows equal to the threshold T;
//  (2) when the rows at or above T fit the candidate area, one more pass
//      collects them.  If one pass resolved every bit (the scores span fewer
//      than 2^13 values), each histogram bin is one score value: the bins at
//      or above T become the first place of their value's group (rows above
//      it), a collected row claims a place in its group, and its final place
//      is the group's start plus the number of the group's rows below its own
//      row -- the ordered list with no sort.  Otherwise the collected rows
//      are sorted by (score descending, row ascending) with a bitonic network;
//  (3) otherwise (many rows equal to T) the rows above T are collected and
//      sorted the same way, and the lowest rows equal to T follow them, placed
//      by an ordered pass in which each warp owns a contiguous run of rows.
// Domains of at least kRowSampleMin rows first try a single read: a
// histogram of a 1/16 systematic sample gives a value t with about
// (k + kRowCap) / 2 rows expected at or above it, one pass stashes those
// rows, and when between k and kRowCap of them were found the stash holds
// every row at or above T, so T, the group starts and the places (or, for
// scores spanning more than 2^13 values, a sort) come from the stash alone.
// A stash outside those bounds (a sample unlike the domain) is counted in
// the statistics and (1)-(3) run.
constexpr int kRowThreads = 512;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kRowCap = 4096;      // candidates: 4096 keys of 8 bytes
constexpr int kRowUnroll = 4;      // 16-byte loads in flight per thread in a pass
constexpr int kRowSampleMin = 32768;  // domains from which the threshold is estimated
constexpr int kRowSampleStride = 16;  // one 128-row chunk in 16 is sampled
constexpr int kRowQueue = 64;         // loads a warp queues in the stash pass
constexpr int kRowAhead = 2;          // pass steps prefetched into L2 ahead of the loads
static_assert(kRowWarps * kRowQueue * 20 <= (4 << kRadixBits), "the queues fit the histogram area");
constexpr size_t kRowSmem = (size_t)kRowCap * 8 + ((size_t)1 << kRadixBits) * 4;
static_assert(kMaxTopk <= kRowCap, "the rows above the threshold always fit the candidates");

// Ascending bitonic sort of kp keys (a power of two) in shared memory.
__device__ __forceinline__ void row_bitonic(unsigned long long *key, int kp) {
  for (int size = 2; size <= kp; size <<= 1) {
    for (int ls = __ffs(size) - 2; ls >= 0; --ls) {  // stride = 2^ls
      const int stride = 1 << ls;
      for (int i = threadIdx.x; i < (kp >> 1); i += kRowThreads) {
        const int a = ((i >> ls) << (ls + 1)) | (i & (stride - 1)), b = a + stride;
        const bool asc = (a & size) == 0;
        const unsigned long long x = key[a], y = key[b];
        if ((x > y) == asc) {
          key[a] = y;
          key[b] = x;
        }
      }
      __syncthreads();
    }
  }
}

__global__ void __launch_bounds__(kRowThreads, 3)
k_topk_row(const DevCtx c, int32_t *__restrict__ topk_out) {
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned long long *cand = reinterpret_cast<unsigned long long *>(smem);
  uint32_t *hist = reinterpret_cast<uint32_t *>(smem + (size_t)kRowCap * 8);
  __shared__ int wcnt[kRowWarps], wsum[kRowWarps];
  __shared__ int sh_bin, sh_above, sh_eq, sh_cnt;
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x / c.Kmax, j = blockIdx.x % c.Kmax;
  if (j >= c.Kr[r]) return;
  const int dom = c.dom[r * c.Kmax + j];
  int32_t *mm = c.minmax + (r * c.Kmax + j) * 2;
  const int lo = mm[0], hi = mm[1];
  const int k = c.k;
  const int32_t *__restrict__ sc = c.scores + ((size_t)r * c.Kmax + j) * c.Ss;
  int32_t *out = topk_out + ((size_t)r * c.Kmax + j) * k;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int ksel = min(k, dom);
  if (tid == 0) sh_cnt = 0;
  __syncthreads();  // every thread has read the range: empty it for the next round
  if (tid == 0) {
    mm[0] = INT_MAX;
    mm[1] = INT_MIN;
  }
  for (int i = ksel + tid; i < k; i += kRowThreads) out[i] = -1;
  if (dom <= 0) return;
  // (a score row is padded to a multiple of 32 entries, so a 16-byte load at
  // any multiple of 4 below dom stays inside it; entries past dom are masked)
  auto load4 = [&](int s) -> int4 { return __ldg(reinterpret_cast<const int4 *>(sc + s)); };
  // Every row whose offset value passes keep(v), claimed in any order into
  // cand[] as (~v << 32 | row); returns nothing, sh_cnt counts them.
  auto collect = [&](auto keep) {
    for (int s0 = wid * 128; s0 < dom; s0 += kRowWarps * 128) {
      const int s = s0 + 4 * lane;
      int4 x = make_int4(0, 0, 0, 0);
      if (s < dom) x = load4(s);
      const int xv[4] = {x.x, x.y, x.z, x.w};
      bool kp4[4];
      int n = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        kp4[e] = s + e < dom && keep((uint32_t)(xv[e] - lo));
        n += kp4[e];
      }
      const unsigned any = __ballot_sync(0xffffffffu, n > 0);
      if (!any) continue;
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int base = 0;
      if (lane == 31) base = atomicAdd(&sh_cnt, incl);
      base = __shfl_sync(0xffffffffu, base, 31);
      int pos = base + incl - n;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (!kp4[e]) continue;
        if (pos < kRowCap)
          cand[pos] = ((unsigned long long)(0xFFFFFFFFu - (uint32_t)(xv[e] - lo)) << 32) |
                      (uint32_t)(s + e);
        else
          record_error(c.err, DC_CAPACITY, K_TOPK);
        ++pos;
      }
    }
  };
  // sort the n collected keys and write the first `m` rows to out[o0..)
  auto sort_out = [&](int n, int o0, int m) {
    int kp = 1;
    while (kp < n) kp <<= 1;
    for (int i = n + tid; i < kp; i += kRowThreads) cand[i] = ~0ull;
    __syncthreads();
    row_bitonic(cand, kp);
    for (int i = tid; i < m; i += kRowThreads)
      out[o0 + i] = (int32_t)(uint32_t)(cand[i] & 0xFFFFFFFFull);
  };
  // Every row whose offset value is at least t, claimed in any order into
  // cand[] as (~v << 32 | row) by one pass over the domain with several
  // 16-byte loads in flight per thread; sh_cnt counts them all, and only the
  // first kRowCap are stored.  A load's four scores are tested at once
  // against lo + t (at most hi: no overflow); the loads holding a row at or
  // above it go to the warp's queue (kRowQueue loads and their first rows, in
  // the histogram area, which the pass does not use), and every 32 queued
  // loads are taken one per lane, so that single rows are looked at by
  // converged lanes (the last load of the domain may hold rows past its end,
  // which are skipped there).
  // One pass step of the CTA covers kRowStep rows; step `it`'s scores are
  // prefetched into L2 kRowAhead steps before the warps load them (the row
  // is padded to a multiple of 32 entries, so the rounded end stays inside).
  constexpr int kRowStep = kRowWarps * 128 * kRowUnroll;
  auto prefetch_step = [&](int it) {
    const int r0 = it * kRowStep;
    if (r0 >= dom) return;
    const int r1 = min((dom + 3) & ~3, r0 + kRowStep);
    bulk_prefetch_l2(sc + r0, (uint32_t)(r1 - r0) * 4u);
  };
  auto stash = [&](uint32_t t) {
    const int thr = lo + (int)t;
    int4 *qx = reinterpret_cast<int4 *>(hist) + wid * kRowQueue;
    int *qs = reinterpret_cast<int *>(hist) + kRowWarps * kRowQueue * 4 + wid * kRowQueue;
    const unsigned lt = (1u << lane) - 1u;
    int qn = 0;  // queued loads (the same in every lane)
    auto drain = [&](int m) {
      __syncwarp();
      int4 y = make_int4(0, 0, 0, 0);
      int sy = dom;
      if (lane < m) {
        y = qx[lane];
        sy = qs[lane];
      }
      const int yv[4] = {y.x, y.y, y.z, y.w};
      bool kp4[4];
      int n = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        kp4[e] = sy + e < dom && yv[e] >= thr;
        n += kp4[e];
      }
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y2 = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y2;
      }
      int base = 0;
      if (lane == 31 && incl > 0) base = atomicAdd(&sh_cnt, incl);
      base = __shfl_sync(0xffffffffu, base, 31);
      int pos = base + incl - n;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (!kp4[e]) continue;
        if (pos < kRowCap)
          cand[pos] = ((unsigned long long)(0xFFFFFFFFu - (uint32_t)(yv[e] - lo)) << 32) |
                      (uint32_t)(sy + e);
        ++pos;
      }
      // the loads queued after the first m move to the front
      const int rest = qn - m;
      int4 z = make_int4(0, 0, 0, 0);
      int sz = 0;
      if (lane < rest) {
        z = qx[m + lane];
        sz = qs[m + lane];
      }
      __syncwarp();
      if (lane < rest) {
        qx[lane] = z;
        qs[lane] = sz;
      }
      qn = rest;
    };
    for (int s0 = wid * 128, it = 0; s0 < dom; s0 += kRowStep, ++it) {
      if (tid == 0) prefetch_step(it + kRowAhead);
      int4 x[kRowUnroll];
#pragma unroll
      for (int u = 0; u < kRowUnroll; ++u) {
        const int s = s0 + u * kRowWarps * 128 + 4 * lane;
        x[u] = s < dom ? load4(s) : make_int4(INT_MIN, INT_MIN, INT_MIN, INT_MIN);
      }
#pragma unroll
      for (int u = 0; u < kRowUnroll; ++u) {
        const bool h = max(max(x[u].x, x[u].y), max(x[u].z, x[u].w)) >= thr;
        const unsigned bal = __ballot_sync(0xffffffffu, h);
        if (!bal) continue;
        if (h) {
          const int p = qn + __popc(bal & lt);
          qx[p] = x[u];
          qs[p] = s0 + u * kRowWarps * 128 + 4 * lane;
        }
        qn += __popc(bal);
        if (qn >= 32) drain(32);
      }
    }
    while (qn > 0) drain(min(qn, 32));
  };
  // hist[0..nbins) = 0 (16-byte stores; the area holds 2^13 bins)
  auto zero_hist = [&](int nbins) {
    uint4 *h4 = reinterpret_cast<uint4 *>(hist);
    for (int i = tid; i < (nbins + 3) >> 2; i += kRowThreads) h4[i] = make_uint4(0u, 0u, 0u, 0u);
  };
  // Warp w owns the w-th run of bins of hist[0..nbins) counted from the top,
  // its lanes reading consecutive bins (lane 0 the highest of each group of
  // 32); the warps' totals give the rows above each run, and the warp whose
  // run holds the kr-th row from the top publishes that bin (sh_bin), the
  // rows above it (sh_above) and its count (sh_eq).  With `starts`, every
  // bin at or above it then holds the rows above it: the first place of its
  // value's group.  Ends with a barrier.
  auto find_bin = [&](int nbins, int kr, bool starts) {
    const int per = (nbins + kRowWarps - 1) / kRowWarps;
    const int b_hi = nbins - wid * per;
    const int b_lo = max(0, b_hi - per);
    int sum = 0;
    for (int b = b_hi - 1 - lane; b >= b_lo; b -= 32) sum += (int)hist[b];
    sum = (int)__reduce_add_sync(0xffffffffu, (unsigned)sum);
    if (lane == 0) wsum[wid] = sum;
    __syncthreads();
    int above = 0;
    for (int w = 0; w < wid; ++w) above += wsum[w];
    // counts of the 32 bins b0 - lane, b0 >= b1, and their inclusive sums in
    // lane order (from the top)
    auto group = [&](int b0, int b1, int &g) {
      const int b = b0 - lane;
      g = b >= b1 ? (int)hist[b] : 0;
      int incl = g;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      return incl;
    };
    if (sum > 0 && above < kr && kr <= above + sum) {
      int acc = above;
      for (int b0 = b_hi - 1; b0 >= b_lo; b0 -= 32) {
        int g;
        const int incl = group(b0, b_lo, g);
        const int tot = __shfl_sync(0xffffffffu, incl, 31);
        if (acc + tot >= kr) {
          const unsigned m = __ballot_sync(0xffffffffu, acc + incl >= kr);
          if (lane == __ffs(m) - 1) {
            sh_bin = b0 - lane;
            sh_above = acc + incl - g;
            sh_eq = g;
          }
          break;
        }
        acc += tot;
      }
    }
    __syncthreads();
    if (starts) {
      const int b1 = max(b_lo, sh_bin);
      int acc = above;
      for (int b0 = b_hi - 1; b0 >= b1; b0 -= 32) {
        int g;
        const int incl = group(b0, b1, g);
        if (b0 - lane >= b1) hist[b0 - lane] = (uint32_t)(acc + incl - g);
        acc += __shfl_sync(0xffffffffu, incl, 31);
      }
      __syncthreads();
    }
  };
  // cand[0..n) holds the rows at or above the threshold, each at a place
  // claimed in its value's group (v << 32 | row); its final place is the
  // group's start plus the number of the group's rows below its own row.
  auto place = [&](int n) {
    for (int p = tid; p < n; p += kRowThreads) {
      const unsigned long long me = cand[p];
      const uint32_t v = (uint32_t)(me >> 32), row = (uint32_t)me;
      int left = 0, below = 0;
      for (int q = p - 1; q >= 0 && (uint32_t)(cand[q] >> 32) == v; --q) {
        ++left;
        below += (uint32_t)cand[q] < row;
      }
      for (int q = p + 1; q < n && (uint32_t)(cand[q] >> 32) == v; ++q)
        below += (uint32_t)cand[q] < row;
      const int fin = p - left + below;
      if (fin < k) out[fin] = (int32_t)row;
    }
  };

  if (dom <= k) {  // every row of the domain is kept, in order
    collect([](uint32_t) { return true; });
    __syncthreads();
    sort_out(dom, 0, dom);
    return;
  }
  const uint32_t range = (uint32_t)(hi - lo);
  int shift = range ? 32 - __clz((int)range) : 0;
  if (dom >= kRowSampleMin && 2 * k <= kRowCap && shift > 0) {
    // Long domains: the threshold is first estimated from a systematic
    // sample (the 128-row chunks whose index is a multiple of
    // kRowSampleStride) as the value with about (k + kRowCap) / 2 rows of
    // the domain at or above it, and one pass stashes those rows.  When the
    // stash holds at least k rows and fits, it holds every row at or above
    // the true threshold, so the list follows from the stash alone and the
    // scores are read once; otherwise the exact passes below run.
    const int sh = max(0, shift - kRadixBits), nb = 1 << min(kRadixBits, shift);
    if (tid == 0)
      for (int it = 0; it < kRowAhead; ++it) prefetch_step(it);
    zero_hist(nb);
    __syncthreads();
    constexpr int kSampleStep = 128 * kRowSampleStride;
    const int nsamp = ((dom + 127) / 128 + kRowSampleStride - 1) / kRowSampleStride;
    for (int i0 = wid; i0 < nsamp; i0 += kRowWarps * kRowUnroll) {
      int4 x[kRowUnroll];
#pragma unroll
      for (int u = 0; u < kRowUnroll; ++u) {
        const int i = i0 + u * kRowWarps, s = i * kSampleStep + 4 * lane;
        x[u] = i < nsamp && s < dom ? load4(s) : make_int4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kRowUnroll; ++u) {
        const int i = i0 + u * kRowWarps, s = i * kSampleStep + 4 * lane;
        if (i >= nsamp) continue;
        const int xv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (s + e < dom) atomicAdd(&hist[((uint32_t)(xv[e] - lo) >> sh) & (nb - 1)], 1u);
      }
    }
    __syncthreads();
    // sampled rows: every sampled chunk but the last is whole
    const int m = (nsamp - 1) * 128 + min(128, dom - (nsamp - 1) * kSampleStep);
    const int target = (k + kRowCap) / 2;
    const int qs = (int)(((long long)target * m + dom - 1) / dom);
    find_bin(nb, qs, false);
    const uint32_t t_est = (uint32_t)sh_bin << sh;
    stash(t_est);
    __syncthreads();
    const int n = sh_cnt;
    if (n >= k && n <= kRowCap) {
      if (sh == 0) {
        // bins are values: count the stash, find T and the group starts,
        // then each stashed row at or above T claims a place in its group
        // (the stash is read into registers first, as the places overwrite it).
        // Every stashed value lies in t_est .. range, so the bins cover only
        // that window (the scans walk a fraction of the 2^13 bins).
        const int nw = (int)(range - t_est) + 1;
        zero_hist(nw);
        __syncthreads();
        for (int p = tid; p < n; p += kRowThreads)
          atomicAdd(&hist[(0xFFFFFFFFu - (uint32_t)(cand[p] >> 32)) - t_est], 1u);
        __syncthreads();
        find_bin(nw, k, true);
        const uint32_t T = t_est + (uint32_t)sh_bin;
        const int ng = sh_above + sh_eq;
        constexpr int kPer = kRowCap / kRowThreads;
        unsigned long long mine[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int p = tid + i * kRowThreads;
          mine[i] = p < n ? cand[p] : 0ull;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          if (tid + i * kRowThreads >= n) continue;
          const uint32_t v = 0xFFFFFFFFu - (uint32_t)(mine[i] >> 32);
          if (v < T) continue;
          const uint32_t p = atomicAdd(&hist[v - t_est], 1u);
          if (p < (uint32_t)kRowCap)
            cand[p] = ((unsigned long long)v << 32) | (uint32_t)mine[i];
          else
            record_error(c.err, DC_CAPACITY, K_TOPK);
        }
        __syncthreads();
        place(ng);
      } else {
        // coarse bins: the stash sorted by (score desc, row asc)
        sort_out(n, 0, k);
      }
      return;
    }
    // the estimate missed (too few rows at or above it, or too many to keep)
    __syncthreads();  // every thread has read the count
    if (tid == 0) {
      sh_cnt = 0;
      atomicAdd(&c.stats[ST_TOPK_RESCAN], 1ull);
    }
  }
  uint32_t prefix = 0;
  int k_rem = k;
  int n_eq = dom;  // rows equal to T (all of them when every score is equal)
  bool first = true;
  int passes = 0;
  while (shift > 0) {
    ++passes;
    const int width = min(kRadixBits, shift);
    shift -= width;
    const int nbins = 1 << width;
    zero_hist(nbins);
    __syncthreads();
    const int hs = shift + width;
    for (int s0 = wid * 128; s0 < dom; s0 += kRowWarps * 128 * kRowUnroll) {
      int4 x[kRowUnroll];
#pragma unroll
      for (int u = 0; u < kRowUnroll; ++u) {
        const int s = s0 + u * kRowWarps * 128 + 4 * lane;
        if (s < dom) x[u] = load4(s);
      }
#pragma unroll
      for (int u = 0; u < kRowUnroll; ++u) {
        const int s = s0 + u * kRowWarps * 128 + 4 * lane;
        const int xv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (s + e >= dom) continue;
          const uint32_t v = (uint32_t)(xv[e] - lo);
          if (first || (uint32_t)((unsigned long long)v >> hs) == prefix)
            atomicAdd(&hist[(v >> shift) & (nbins - 1)], 1u);
        }
      }
    }
    __syncthreads();
    // (with exact bins, bin b >= T becomes the first place of value b's group)
    find_bin(nbins, k_rem, passes == 1 && shift == 0);
    k_rem -= sh_above;
    prefix = (prefix << width) | (uint32_t)sh_bin;
    n_eq = sh_eq;
    first = false;
  }
  const uint32_t T = prefix;  // the k-th largest offset score
  const int need = k_rem;     // rows equal to T that are kept
  const int c_gt = k - need;  // rows strictly above T
  if (c_gt + n_eq <= kRowCap && passes == 1 && shift == 0) {
    // claim a place in the value's group, in any order ...
    for (int s0 = wid * 128; s0 < dom; s0 += kRowWarps * 128) {
      const int s = s0 + 4 * lane;
      if (s >= dom) continue;
      const int4 x = load4(s);
      const int xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t v = (uint32_t)(xv[e] - lo);
        if (s + e < dom && v >= T) {
          const uint32_t p = atomicAdd(&hist[v], 1u);
          if (p < (uint32_t)kRowCap)
            cand[p] = ((unsigned long long)v << 32) | (uint32_t)(s + e);
          else
            record_error(c.err, DC_CAPACITY, K_TOPK);
        }
      }
    }
    __syncthreads();
    // ... then its place: the group's start plus the group's rows below it
    place(c_gt + n_eq);
    return;
  }
  if (c_gt + n_eq <= kRowCap) {
    collect([T](uint32_t v) { return v >= T; });
    __syncthreads();
    if (sh_cnt != c_gt + n_eq) record_error(c.err, DC_CAPACITY, K_TOPK);
    sort_out(min(sh_cnt, kRowCap), 0, k);
    return;
  }
  // many rows equal to T: the rows above it first ...
  collect([T](uint32_t v) { return v > T; });
  __syncthreads();
  if (sh_cnt != c_gt) record_error(c.err, DC_CAPACITY, K_TOPK);
  if (c_gt > 0) sort_out(min(sh_cnt, kRowCap), 0, c_gt);
  // ... then the lowest `need` rows equal to T, in row order: warp w owns
  // rows [w * run, (w + 1) * run); count, scan the warps' counts, place
  const int run = ((dom + kRowWarps - 1) / kRowWarps + 127) & ~127;
  const int r0 = min(dom, wid * run), r1 = min(dom, r0 + run);
  int eq_lane = 0;
  for (int s = r0 + 4 * lane; s < r1; s += 128) {
    const int4 x = load4(s);
    const int xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) eq_lane += s + e < r1 && (uint32_t)(xv[e] - lo) == T;
  }
  const int weq = (int)__reduce_add_sync(0xffffffffu, (unsigned)eq_lane);
  if (lane == 0) wcnt[wid] = weq;
  __syncthreads();
  int wbase = 0;
  for (int w = 0; w < wid; ++w) wbase += wcnt[w];
  if (wbase < need) {
    const unsigned lt = (1u << lane) - 1u;
    for (int s0 = r0; s0 < r1 && wbase < need; s0 += 128) {
      const int s = s0 + 4 * lane;
      int4 x = make_int4(0, 0, 0, 0);
      if (s < r1) x = load4(s);
      const int xv[4] = {x.x, x.y, x.z, x.w};
      bool eq[4];
      unsigned bal[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        eq[e] = s + e < r1 && (uint32_t)(xv[e] - lo) == T;
        bal[e] = __ballot_sync(0xffffffffu, eq[e]);
      }
      // row order: every equal row of the lanes below, then the lane's own
      int pos = wbase;
#pragma unroll
      for (int e = 0; e < 4; ++e) pos += __popc(bal[e] & lt);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (!eq[e]) continue;
        if (pos < need) out[c_gt + pos] = s + e;
        ++pos;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) wbase += __popc(bal[e]);
    }
  }
}

// ---------------------------------------------------------------- scores on tensor cores
// Rows of 64 * NG bytes (NG = 1..8).  The score of eq. (1) is an exact
// integer dot product, and so is this kernel's: every int8 value becomes the
// f16 holding it exactly, the m16n8k16 MMA multiplies 16 key rows by the
// eight (padded) queries with fp32 accumulation, and every partial sum is an
// integer of magnitude at most 512 * 128 * 128 = 2^23 < 2^24, so no rounding
// ever happens and the float result converts back to the exact int32.
//
// Work: tiles of 16 consecutive rows of one request; the tiles of all
// requests form one list, and each warp of the persistent grid owns a
// contiguous run of it.  Every warp streams its tiles through its own ring of
// shared-memory stages, one bulk asynchronous copy per tile (the rows are
// contiguous in global memory and stay dense in the stage), each stage
// tracked by an mbarrier counting the bytes that landed.  For rows of a
// multiple of 128 bytes the fragment loads of rows g and g + 1 meet in the
// same banks (two wavefronts per quarter warp), which the shared-memory
// pipe absorbs at the rate HBM delivers rows.
//
// Fragment layout: the MMA's k index is a permutation of the row's bytes.
// At 64-byte group i, lane (g = lane / 4, t = lane % 4) loads the 16-byte
// chunk 4i + t of rows g and g + 8 of the tile; word w of that chunk holds
// the lane's four k positions (2t, 2t+1, 2t+8, 2t+9) of MMA step 4i + w.  The
// query fragments are built from the same bytes of the query rows, so both
// operands see the same permutation and the dot products are unchanged.
constexpr int kTcWarps = 4;
constexpr int kTcMaxStages = 8;
constexpr int kTcTilesPerWarp = 24;  // tiles of a warp in launches larger than one wave
constexpr int kTcSpinLimit = 1 << 22;
constexpr int kTcMinGroups = 3;                     // always for rows of 192 B and more
constexpr size_t kTcNarrowBytes = (size_t)256 << 20;  // 64/128-B rows: from 256 MB of keys
constexpr int kTcMaxGroups = 8;


// int8 x 4 -> two f16 x 2 with the same values: byte b goes to the f16 whose
// bits are 0x64 | (b ^ 0x80), i.e. 1024 + (b + 128); subtracting 1152 leaves b.
__device__ __forceinline__ void i8x4_to_f16(uint32_t x, uint32_t &lo, uint32_t &hi) {
  const uint32_t u = x ^ 0x80808080u;
  uint32_t l = __byte_perm(u, 0x64646464u, 0x5140);
  uint32_t h = __byte_perm(u, 0x64646464u, 0x7362);
  const uint32_t bias = 0x64806480u;
  asm("sub.f16x2 %0, %1, %2;\n" : "=r"(lo) : "r"(l), "r"(bias));
  asm("sub.f16x2 %0, %1, %2;\n" : "=r"(hi) : "r"(h), "r"(bias));
}

template <int NG>
__global__ void __launch_bounds__(kTcWarps * 32)
k_index_score_tc(const DevCtx c, const int8_t *__restrict__ q_idx,
                 const __grid_constant__ UploadWords ctl, int stages) {
  constexpr int RB = 64 * NG;
  constexpr int STRIDE = RB;
  constexpr int TILE = 16 * STRIDE;
  constexpr int STEPS = 4 * NG;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t mbar[kTcWarps][kTcMaxStages];
  __shared__ int warp_sums[32];
  pdl_wait();
  pdl_trigger();
  const int N = c.N, Kmax = c.Kmax;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (blockIdx.x == 0) {
    for (int i = tid; i < N; i += blockDim.x) c.Kr[i] = ctl.w[i];
    for (int i = tid; i < N * Kmax; i += blockDim.x) c.dom[i] = ctl.w[N + i];
  }
  // tile list: request r owns tiles [tstart[r], tstart[r + 1])
  int *tstart = reinterpret_cast<int *>(smem + (size_t)kTcWarps * stages * TILE);
  {
    int carry = 0;
    for (int base = 0; base < N; base += blockDim.x) {
      const int r = base + tid;
      int cnt = 0;
      if (r < N) {
        const int Kr = ctl.w[r];
        int dm = 0;
        for (int j = 0; j < Kr; ++j) dm = max(dm, ctl.w[N + r * Kmax + j]);
        cnt = (dm + 15) >> 4;
      }
      int tot;
      const int ex = block_excl_scan(cnt, warp_sums, tot);
      if (r < N) tstart[r] = carry + ex;
      carry += tot;
    }
    if (tid == 0) tstart[N] = carry;
    __syncthreads();
  }
  const int T = tstart[N];
  const int64_t W = (int64_t)gridDim.x * kTcWarps, wg = (int64_t)blockIdx.x * kTcWarps + warp;
  const int tb = (int)(wg * T / W), te = (int)((wg + 1) * T / W);
  if (tb >= te) return;  // no block-wide barrier follows
  unsigned char *ring = smem + (size_t)warp * stages * TILE;
  uint64_t *bar = mbar[warp];
  if (lane == 0) {
    for (int s = 0; s < stages; ++s) mbar_init(&bar[s], 1);
    fence_proxy_async_smem();
  }
  __syncwarp();

  auto locate = [&](int tile) {  // the request whose tiles contain `tile`
    int lo = 0, hi = N - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tstart[mid] <= tile) lo = mid;
      else hi = mid - 1;
    }
    return lo;
  };
  auto dom_of = [&](int r) {
    int dm = 0;
    for (int j = 0; j < ctl.w[r]; ++j) dm = max(dm, ctl.w[N + r * Kmax + j]);
    return dm;
  };

  // producer cursor
  int pr = locate(tb), ptile = tb, pdom = dom_of(pr);
  auto issue = [&](int slot) {
    while (ptile >= tstart[pr + 1]) pdom = dom_of(++pr);
    const int64_t row0 = (int64_t)(ptile - tstart[pr]) * 16;
    const int nrows = (int)min((int64_t)16, (int64_t)pdom - row0);
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar[slot], (uint32_t)(nrows * RB));
      bulk_g2s(ring + (size_t)slot * TILE, c.keys[pr] + row0 * RB, (uint32_t)(nrows * RB),
               &bar[slot]);
    }
    ++ptile;
  };
  const int pre = min(stages, te - tb);
  for (int s = 0; s < pre; ++s) issue(s);

  const int g = lane >> 2, t = lane & 3;
  const int q0 = 2 * t, q1 = 2 * t + 1;
  uint32_t bq[STEPS][2];
  int cr = -1, Kr = 0, cdom = 0, dq0 = 0, dq1 = 0;
  int mn0 = INT_MAX, mx0 = INT_MIN, mn1 = INT_MAX, mx1 = INT_MIN;
  auto flush = [&]() {  // the request's score range, one atomic per query and warp
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mn0 = min(mn0, __shfl_xor_sync(0xffffffffu, mn0, o));
      mx0 = max(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mn1 = min(mn1, __shfl_xor_sync(0xffffffffu, mn1, o));
      mx1 = max(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    if (g == 0 && cr >= 0) {
      if (q0 < Kr && mn0 <= mx0) {
        atomicMin(&c.minmax[(cr * Kmax + q0) * 2 + 0], mn0);
        atomicMax(&c.minmax[(cr * Kmax + q0) * 2 + 1], mx0);
      }
      if (q1 < Kr && mn1 <= mx1) {
        atomicMin(&c.minmax[(cr * Kmax + q1) * 2 + 0], mn1);
        atomicMax(&c.minmax[(cr * Kmax + q1) * 2 + 1], mx1);
      }
    }
    mn0 = mn1 = INT_MAX;
    mx0 = mx1 = INT_MIN;
  };

  int it = 0;
  bool bad = false;
  for (int tile = tb; tile < te; ++tile, ++it) {
    if (cr < 0 || tile >= tstart[cr + 1]) {  // next request: its query fragments
      flush();
      cr = cr < 0 ? locate(tile) : cr + 1;
      while (tile >= tstart[cr + 1]) ++cr;
      Kr = ctl.w[cr];
      cdom = dom_of(cr);
      dq0 = q0 < Kr ? ctl.w[N + cr * Kmax + q0] : 0;
      dq1 = q1 < Kr ? ctl.w[N + cr * Kmax + q1] : 0;
      const int8_t *qrow = (q_idx ? q_idx : reinterpret_cast<const int8_t *>(
                                                ctl.w + ctl_qidx_word(N, Kmax))) +
                           ((size_t)cr * Kmax + g) * RB;
#pragma unroll
      for (int i = 0; i < NG; ++i) {
        const uint4 v = g < Kr ? *reinterpret_cast<const uint4 *>(qrow + (4 * i + t) * 16)
                               : make_uint4(0u, 0u, 0u, 0u);
        i8x4_to_f16(v.x, bq[4 * i + 0][0], bq[4 * i + 0][1]);
        i8x4_to_f16(v.y, bq[4 * i + 1][0], bq[4 * i + 1][1]);
        i8x4_to_f16(v.z, bq[4 * i + 2][0], bq[4 * i + 2][1]);
        i8x4_to_f16(v.w, bq[4 * i + 3][0], bq[4 * i + 3][1]);
      }
    }
    const int slot = it % stages;
    {
      const uint32_t parity = (uint32_t)((it / stages) & 1);
      int spins = 0;
      bool late = false;
      while (!mbar_try_wait(&bar[slot], parity))
        if (++spins > kTcSpinLimit) {
          late = true;
          break;
        }
      if (__any_sync(0xffffffffu, late)) {
        if (lane == 0) record_error(c.err, DC_TIMEOUT, K_SCORE);
        bad = true;
        break;
      }
    }
    const unsigned char *st = ring + (size_t)slot * TILE;
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a) acc[a][0] = acc[a][1] = acc[a][2] = acc[a][3] = 0.f;
#pragma unroll
    for (int i = 0; i < NG; ++i) {
      const uint4 lo = *reinterpret_cast<const uint4 *>(st + g * STRIDE + (4 * i + t) * 16);
      const uint4 hi = *reinterpret_cast<const uint4 *>(st + (g + 8) * STRIDE + (4 * i + t) * 16);
      const uint32_t wl[4] = {lo.x, lo.y, lo.z, lo.w}, wh[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t a0, a1, a2, a3;
        i8x4_to_f16(wl[w], a0, a2);
        i8x4_to_f16(wh[w], a1, a3);
        mma_f16_16816(acc[w], a0, a1, a2, a3, bq[4 * i + w][0], bq[4 * i + w][1]);
      }
    }
    __syncwarp();  // every lane has read the stage: it may be refilled
    if (ptile < te) issue(slot);

    const int64_t row0 = (int64_t)(tile - tstart[cr]) * 16;
    const int64_t ra = row0 + g, rb = row0 + g + 8;
    int v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      v[e] = __float2int_rn((acc[0][e] + acc[1][e]) + (acc[2][e] + acc[3][e]));
    if (q0 < Kr) {
      int32_t *o = c.scores + ((size_t)cr * Kmax + q0) * c.Ss;
      if (ra < cdom) o[ra] = v[0];
      if (rb < cdom) o[rb] = v[2];
      if (ra < dq0) { mn0 = min(mn0, v[0]); mx0 = max(mx0, v[0]); }
      if (rb < dq0) { mn0 = min(mn0, v[2]); mx0 = max(mx0, v[2]); }
    }
    if (q1 < Kr) {
      int32_t *o = c.scores + ((size_t)cr * Kmax + q1) * c.Ss;
      if (ra < cdom) o[ra] = v[1];
      if (rb < cdom) o[rb] = v[3];
      if (ra < dq1) { mn1 = min(mn1, v[1]); mx1 = max(mx1, v[1]); }
      if (rb < dq1) { mn1 = min(mn1, v[3]); mx1 = max(mx1, v[3]); }
    }
  }
  if (bad) {
    // copies still in flight land before the warp leaves (each wait bounded)
    for (int k = it; k < ptile - tb; ++k) {
      int spins = 0;
      while (!mbar_try_wait(&bar[k % stages], (uint32_t)((k / stages) & 1)) &&
             ++spins <= kTcSpinLimit) {
      }
    }
    return;
  }
  flush();
}

cudaError_t launch_select(const DevCtx &c, const int8_t *q_idx, const int8_t *q_inline,
                          int32_t *topk_out, int max_dom, const int32_t *ctl_words,
                          int active_queries, int topk_pass, cudaStream_t s, Timer *tm) {
  UploadWords ctl;
  const int nw = c.N + c.N * c.Kmax;
  for (int i = 0; i < nw; ++i) ctl.w[i] = ctl_words[i];
  if (!q_idx)
    std::memcpy(ctl.w + ctl_qidx_word(c.N, c.Kmax), q_inline,
                (size_t)c.N * c.Kmax * c.idx_row);
  // Tensor-core scoring on a persistent grid for rows of 192 to 512 bytes,
  // and for 64- and 128-byte rows once a launch streams at least
  // kTcNarrowBytes of keys: below that the one-thread-per-row kernel, which
  // has no set-up, finishes first (measured: 14.6 against 23 us on 17 MB).
  const size_t key_bytes = (size_t)c.N * (size_t)max(max_dom, 0) * (size_t)c.idx_row;
  const bool tc_width = c.idx_row % 64 == 0 && c.idx_row <= 64 * kTcMaxGroups;
  if (tc_width && (c.idx_row >= 64 * kTcMinGroups || key_bytes >= kTcNarrowBytes)) {
    using TcKern = void (*)(const DevCtx, const int8_t *, const UploadWords, int);
    static const TcKern kerns[kTcMaxGroups] = {
        k_index_score_tc<1>, k_index_score_tc<2>, k_index_score_tc<3>, k_index_score_tc<4>,
        k_index_score_tc<5>, k_index_score_tc<6>, k_index_score_tc<7>, k_index_score_tc<8>};
    static size_t granted[kTcMaxGroups] = {};
    static int grid_of[kTcMaxGroups] = {};
    static size_t grid_smem[kTcMaxGroups] = {};
    const int ng = c.idx_row / 64;
    const size_t stage_set = (size_t)kTcWarps * 16 * c.idx_row;
    // rows of up to 128 bytes: a smaller ring per warp, so that twice as many
    // CTAs (warps to issue the conversions and MMAs) fit on an SM with about
    // the same bytes in flight (measured on 64 histories of 524 288 rows of
    // 128 bytes: 1.08 -> 0.85 ms).  Wider rows: two stages per warp (64 KB
    // a CTA for 512-byte rows, still about twice the bytes in flight HBM
    // needs per SM), which leaves an SM with two indexer CTAs room for a
    // top-k or union/probe CTA of another request group (measured on 128
    // histories of 102 400 rows of 512 bytes: 1.054 -> 1.030 ms alone)
    const size_t ring_budget = ng <= 2 ? (36u << 10) : (70u << 10);
    const int stages = (int)std::min<size_t>(kTcMaxStages, std::max<size_t>(2, ring_budget / stage_set));
    const size_t smem = stage_set * stages + (size_t)(c.N + 1) * 4;
    TcKern kern = kerns[ng - 1];
    cudaError_t e;
    if ((e = ensure_smem(kern, smem, granted[ng - 1])) != cudaSuccess) return e;
    if (grid_smem[ng - 1] != smem) {
      int per_sm = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kTcWarps * 32, smem);
      if (e != cudaSuccess) return e;
      grid_of[ng - 1] = c.sms * std::max(1, per_sm);
      grid_smem[ng - 1] = smem;
    }
    // at least one resident wave; larger launches are cut into CTAs of
    // kTcTilesPerWarp tiles per warp, so that SMs free up while the launch
    // runs and kernels of other streams (request groups) get onto them
    // (measured on 128 histories of 102 400 rows in three groups: 24 and 48
    // tiles alike, 96 and 192 10% slower)
    int64_t tiles = 0;
    for (int r = 0; r < c.N; ++r) {
      int dm = 0;
      for (int j = 0; j < ctl_words[r]; ++j) dm = std::max(dm, ctl_words[c.N + r * c.Kmax + j]);
      tiles += (dm + 15) / 16;
    }
    const int64_t per_cta = (int64_t)kTcWarps * kTcTilesPerWarp;
    const int grid = (int)std::max<int64_t>(grid_of[ng - 1],
                                            std::min<int64_t>((tiles + per_cta - 1) / per_cta, 1 << 30));
    if (tm) tm->begin(K_SCORE, s);
    e = launch_pdl(kern, dim3(grid), dim3(kTcWarps * 32), smem, s, c, q_idx, ctl, stages);
    if (tm) tm->end(K_SCORE, s);
    if (e != cudaSuccess) return e;
  } else {
    // one CTA per request at least, so that the control words are published
    const int nc = c.idx_row >> 4;
    cudaError_t e;
    void (*kern)(const DevCtx, const int8_t *, const UploadWords);
    size_t smem = 0;
    int rpb;
    if (nc <= kDirectChunks) {
      kern = nc == 4 ? k_index_score<4> : nc == 8 ? k_index_score<8> : k_index_score<0>;
      smem = (size_t)c.Kmax * c.idx_row;
      rpb = kScoreThreads;
    } else if (nc <= 16) {
      kern = k_index_score_wide<16, 1>;
      rpb = WideScore<16, 1>::RPB;
    } else if (nc <= 32) {
      kern = k_index_score_wide<32, 1>;
      rpb = WideScore<32, 1>::RPB;
    } else {
      kern = k_index_score_wide<32, 2>;
      rpb = WideScore<32, 2>::RPB;
    }
    static size_t granted[5] = {};
    const int gi = nc == 4 ? 0 : nc == 8 ? 1 : nc <= kDirectChunks ? 2 : nc <= 16 ? 3 : 4;
    if ((e = ensure_smem(kern, smem, granted[gi])) != cudaSuccess) return e;
    dim3 grid(max_dom > 0 ? (max_dom + rpb - 1) / rpb : 1, c.N);
    if (tm) tm->begin(K_SCORE, s);
    e = launch_pdl(kern, grid, dim3(kScoreThreads), smem, s, c, q_idx, ctl);
    if (tm) tm->end(K_SCORE, s);
    if (e != cudaSuccess) return e;
  }
  if (topk_pass == DHS_TOPK_ROW || (topk_pass == DHS_TOPK_AUTO && active_queries >= c.sms)) {
    static size_t granted_row = 0;
    const size_t smem_row = kRowSmem;
    cudaError_t e3 = ensure_smem(k_topk_row, smem_row, granted_row);
    if (e3 != cudaSuccess) return e3;
    if (tm) tm->begin(K_TOPK, s);
    e3 = launch_pdl(k_topk_row, dim3(c.N * c.Kmax), dim3(kRowThreads), smem_row, s, c, topk_out);
    if (tm) tm->end(K_TOPK, s);
    return e3;
  }
  int kp = 1;
  while (kp < c.k) kp <<= 1;
  size_t smem_topk = (size_t)kp * 8 + ((size_t)1 << kRadixBits) * 8;
  // a CTA's part of the widest domain, staged in shared memory when it fits
  const int part = ((max(max_dom, 1) + kTopkCluster - 1) / kTopkCluster + 31) & ~31;
  int stage_cap = 0;
  // (the in-place winner lists pack a row's place in the part into 17 bits)
  // the dynamic shared memory a top-k CTA may take beside its static arrays
  static size_t topk_dyn_max = 0;
  if (!topk_dyn_max) {
    int dev = 0, optin = 0;
    cudaFuncAttributes fa;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, k_topk);
    if (e != cudaSuccess) return e;
    topk_dyn_max = std::min(kMaxDynSmem, (size_t)optin - fa.sharedSizeBytes);
  }
  if (smem_topk + 8 + (size_t)part * 4 <= topk_dyn_max && part <= (1 << 17)) {
    stage_cap = part;
    smem_topk = (((size_t)kp * 8 + 15) & ~(size_t)15) + ((size_t)2 << kRadixBits) * 4 +
                (size_t)part * 4;
  }
  static size_t granted_topk = 0;
  cudaError_t e2 = ensure_smem(k_topk, smem_topk, granted_topk);
  if (e2 != cudaSuccess) return e2;
  if (tm) tm->begin(K_TOPK, s);
  e2 = launch_pdl(k_topk, dim3(c.N * c.Kmax * kTopkCluster), dim3(kTopkThreads), smem_topk, s, c,
                  topk_out, stage_cap);
  if (tm) tm->end(K_TOPK, s);
  return e2;
}

}  // namespace dhs
