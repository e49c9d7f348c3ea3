// Step 1 of the verification round: indexer scores and per-query top-k.
//
// "Adaptive DHiSparse", section 2.1, eq. (1): the sparse indexer scores every
// historical row s against query t and selects the k best, S_t = Top-k(I_t,:),
// kept as the ordered list the model's top-k returns.  The causal domain of a
// verification query is the committed history (section 3.3, eq. (5)).
#include "dhs_internal.cuh"
#include "ptx_util.cuh"

#include <climits>

namespace dhs {

// ---------------------------------------------------------------- upload
__global__ void k_upload(int32_t *dst, int n, const __grid_constant__ UploadWords w) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    dst[i] = w.w[i];
}

cudaError_t launch_upload(int32_t *dst, const int32_t *words, int n, cudaStream_t s) {
  UploadWords w;
  for (int i = 0; i < n; ++i) w.w[i] = words[i];
  k_upload<<<(n + 255) / 256, 256, 0, s>>>(dst, n, w);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- scores
// One CTA scores TILE consecutive key rows of one request against all K_r
// queries: the rows are copied once into shared memory (16-byte cp.async,
// coalesced), each thread then owns one row and accumulates the K_r dot
// products with dp4a, reading each query chunk as a shared-memory broadcast.
// Key chunks are stored rotated by a per-row offset so that the eight rows
// one LDS.128 phase touches fall in distinct bank groups.
constexpr int kScoreTile = 128;

__device__ __forceinline__ int score_rot(int t, int nc) {
  return nc >= 8 ? (t % nc) : ((t * nc) >> 3) % nc;
}

__global__ void __launch_bounds__(kScoreTile)
k_index_score(const DevCtx c, const int8_t *__restrict__ q_idx) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int r = blockIdx.y;
  const int Kr = c.Kr[r];
  if (Kr == 0) return;
  int dom_r = 0;
  for (int j = 0; j < Kr; ++j) dom_r = max(dom_r, c.dom[r * c.Kmax + j]);
  const int64_t row0 = (int64_t)blockIdx.x * kScoreTile;
  if (row0 >= dom_r) return;
  const int RB = c.idx_row, nc = RB >> 4;
  uint4 *tile = reinterpret_cast<uint4 *>(smem);
  uint4 *qs = tile + kScoreTile * nc;
  const int rows = (int)(dom_r - row0 < kScoreTile ? dom_r - row0 : kScoreTile);

  const uint4 *src = reinterpret_cast<const uint4 *>(c.keys[r] + row0 * RB);
  for (int u = threadIdx.x; u < rows * nc; u += blockDim.x) {
    int t = u / nc, ch = u - t * nc;
    int pos = ch + score_rot(t, nc);
    if (pos >= nc) pos -= nc;
    cp_async_16(&tile[t * nc + pos], &src[u]);
  }
  cp_async_commit();
  const uint4 *qsrc = reinterpret_cast<const uint4 *>(q_idx + (size_t)r * c.Kmax * RB);
  for (int u = threadIdx.x; u < Kr * nc; u += blockDim.x) qs[u] = qsrc[u];
  cp_async_wait_all();
  __syncthreads();

  const int t = threadIdx.x;
  int acc[kMaxKmax];
#pragma unroll
  for (int j = 0; j < kMaxKmax; ++j) acc[j] = 0;
  if (t < rows) {
    const int rt = score_rot(t, nc);
    const uint4 *myrow = tile + t * nc;
    int pos = rt;
    for (int ch = 0; ch < nc; ++ch) {
      const uint4 kv = myrow[pos];
      if (++pos == nc) pos = 0;
#pragma unroll
      for (int j = 0; j < kMaxKmax; ++j) {
        if (j < Kr) {
          const uint4 qv = qs[j * nc + ch];
          acc[j] = __dp4a((int)kv.x, (int)qv.x, acc[j]);
          acc[j] = __dp4a((int)kv.y, (int)qv.y, acc[j]);
          acc[j] = __dp4a((int)kv.z, (int)qv.z, acc[j]);
          acc[j] = __dp4a((int)kv.w, (int)qv.w, acc[j]);
        }
      }
    }
  }
  const int64_t s = row0 + t;
  const int lane = t & 31;
#pragma unroll
  for (int j = 0; j < kMaxKmax; ++j) {
    if (j >= Kr) break;
    const int dj = c.dom[r * c.Kmax + j];
    if (t < rows) c.scores[((size_t)r * c.Kmax + j) * c.Sm + s] = acc[j];
    const bool valid = t < rows && s < dj;
    int mn = valid ? acc[j] : INT_MAX, mx = valid ? acc[j] : INT_MIN;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (lane == 0 && mn <= mx) {
      atomicMin(&c.minmax[(r * c.Kmax + j) * 2 + 0], mn);
      atomicMax(&c.minmax[(r * c.Kmax + j) * 2 + 1], mx);
    }
  }
}

__global__ void k_minmax_init(const DevCtx c) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < c.N * c.Kmax) {
    c.minmax[2 * i] = INT_MAX;
    c.minmax[2 * i + 1] = INT_MIN;
  }
}

// ---------------------------------------------------------------- top-k
// One CTA of 1024 threads per (request, query).  Exact radix select on the
// score offset by the query's minimum (so only the bits the scores actually
// span are examined, at most 13 per pass), then one ordered pass that keeps
// every row above the threshold and the lowest-index rows equal to it, then a
// bitonic sort of the k winners by (score descending, row ascending).
constexpr int kTopkThreads = 1024;
constexpr int kRadixBits = 13;

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
    warp_sums[lane] = w;  // inclusive prefix of warp totals
  }
  __syncthreads();
  total = warp_sums[nw - 1];
  int excl = x - v + (wid > 0 ? warp_sums[wid - 1] : 0);
  __syncthreads();
  return excl;
}

__global__ void __launch_bounds__(kTopkThreads)
k_topk(const DevCtx c, int32_t *__restrict__ topk_out) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int r = blockIdx.x / c.Kmax, j = blockIdx.x % c.Kmax;
  if (j >= c.Kr[r]) return;
  const int dom = c.dom[r * c.Kmax + j];
  const int k = c.k;
  const int32_t *__restrict__ sc = c.scores + ((size_t)r * c.Kmax + j) * c.Sm;
  int32_t *out = topk_out + ((size_t)r * c.Kmax + j) * k;

  int kp = 1;
  while (kp < k) kp <<= 1;
  unsigned long long *cand = reinterpret_cast<unsigned long long *>(smem);
  uint32_t *hist = reinterpret_cast<uint32_t *>(cand + kp);
  __shared__ int warp_sums[32];
  __shared__ int sh_bin, sh_above, sh_gt, sh_eqbase;
  const int tid = threadIdx.x;
  const int ksel = min(k, dom);
  const int lo = c.minmax[(r * c.Kmax + j) * 2 + 0];
  const int hi = c.minmax[(r * c.Kmax + j) * 2 + 1];

  if (dom <= k) {
    for (int s = tid; s < dom; s += blockDim.x) {
      uint32_t v = (uint32_t)(sc[s] - lo);
      cand[s] = ((unsigned long long)(0xFFFFFFFFu - v) << 32) | (uint32_t)s;
    }
  } else {
    const uint32_t range = (uint32_t)(hi - lo);
    int shift = range ? 32 - __clz((int)range) : 0;
    uint32_t prefix = 0;
    int k_rem = k;
    while (shift > 0) {
      const int width = min(kRadixBits, shift);
      shift -= width;
      const int nbins = 1 << width;
      for (int i = tid; i < nbins; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      for (int s = tid; s < dom; s += blockDim.x) {
        uint32_t v = (uint32_t)(sc[s] - lo);
        if ((uint32_t)((unsigned long long)v >> (shift + width)) == prefix)
          atomicAdd(&hist[(v >> shift) & (nbins - 1)], 1u);
      }
      __syncthreads();
      // thread t owns a run of bins counted from the top, so an exclusive scan
      // in thread order gives the number of rows above each run
      const int per = (nbins + blockDim.x - 1) / blockDim.x;
      const int b_hi = nbins - tid * per;           // exclusive upper end
      const int b_lo = max(0, b_hi - per);
      int local = 0;
      for (int b = b_lo; b < b_hi; ++b) local += hist[b];
      int total;
      int above = block_excl_scan(b_hi > 0 ? local : 0, warp_sums, total);
      if (b_hi > 0 && above < k_rem && k_rem <= above + local) {
        int acc = above;
        for (int b = b_hi - 1; b >= b_lo; --b) {
          if (acc + (int)hist[b] >= k_rem) {
            sh_bin = b;
            sh_above = acc;
            break;
          }
          acc += hist[b];
        }
      }
      __syncthreads();
      k_rem -= sh_above;
      prefix = (prefix << width) | (uint32_t)sh_bin;
      __syncthreads();
    }
    const uint32_t T = prefix;       // the k-th largest offset score
    const int need = k_rem;          // rows equal to T that are kept
    const int c_gt = k - need;       // rows strictly above T
    if (tid == 0) { sh_gt = 0; sh_eqbase = 0; }
    __syncthreads();
    for (int base = 0; base < dom; base += blockDim.x) {
      const int s = base + tid;
      uint32_t v = s < dom ? (uint32_t)(sc[s] - lo) : 0u;
      const bool gt = s < dom && v > T;
      const bool eq = s < dom && v == T;
      const unsigned long long key = ((unsigned long long)(0xFFFFFFFFu - v) << 32) | (uint32_t)s;
      if (gt) cand[atomicAdd(&sh_gt, 1)] = key;
      int tot;
      const int rank = sh_eqbase + block_excl_scan(eq ? 1 : 0, warp_sums, tot);
      if (eq && rank < need) cand[c_gt + rank] = key;
      __syncthreads();
      if (tid == 0) sh_eqbase += tot;
      __syncthreads();
      const bool done = sh_gt == c_gt && sh_eqbase >= need;
      __syncthreads();  // every thread has read the counters before the next round of atomics
      if (done) break;
    }
  }
  for (int i = ksel + tid; i < kp; i += blockDim.x) cand[i] = ~0ull;
  __syncthreads();
  // bitonic sort ascending on (~score, row)
  for (int size = 2; size <= kp; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < (kp >> 1); i += blockDim.x) {
        const int a = 2 * stride * (i / stride) + (i % stride);
        const int b = a + stride;
        const bool asc = (a & size) == 0;
        unsigned long long x = cand[a], y = cand[b];
        if ((x > y) == asc) { cand[a] = y; cand[b] = x; }
      }
      __syncthreads();
    }
  }
  for (int i = tid; i < k; i += blockDim.x)
    out[i] = i < ksel ? (int32_t)(uint32_t)(cand[i] & 0xFFFFFFFFull) : -1;
}

cudaError_t launch_select(const DevCtx &c, const int8_t *q_idx, int32_t *topk_out, int max_dom,
                          int active, cudaStream_t s, Timer *tm) {
  (void)active;
  k_minmax_init<<<(c.N * c.Kmax + 255) / 256, 256, 0, s>>>(c);
  if (max_dom > 0) {
    const size_t smem = (size_t)(kScoreTile + c.Kmax) * c.idx_row;
    static size_t granted_score = 0;
    cudaError_t e = ensure_smem(k_index_score, smem, granted_score);
    if (e != cudaSuccess) return e;
    dim3 grid((max_dom + kScoreTile - 1) / kScoreTile, c.N);
    if (tm) tm->begin(K_SCORE, s);
    k_index_score<<<grid, kScoreTile, smem, s>>>(c, q_idx);
    if (tm) tm->end(K_SCORE, s);
  }
  int kp = 1;
  while (kp < c.k) kp <<= 1;
  const size_t smem_topk = (size_t)kp * 8 + ((size_t)1 << kRadixBits) * 4;
  static size_t granted_topk = 0;
  cudaError_t e2 = ensure_smem(k_topk, smem_topk, granted_topk);
  if (e2 != cudaSuccess) return e2;
  if (tm) tm->begin(K_TOPK, s);
  k_topk<<<c.N * c.Kmax, kTopkThreads, smem_topk, s>>>(c, topk_out);
  if (tm) tm->end(K_TOPK, s);
  return cudaGetLastError();
}

}  // namespace dhs
