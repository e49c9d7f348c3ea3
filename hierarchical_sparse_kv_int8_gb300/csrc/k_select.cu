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
// One thread per key row.  Rows of up to 128 bytes are read straight from
// global memory with 16-byte loads (each thread consumes whole 32-byte
// sectors); wider rows are first staged in shared memory by coalesced
// cp.async copies, stored rotated by a per-row offset so that the eight rows
// of one LDS.128 phase fall in distinct bank groups.  The K_r query chunks
// are shared-memory broadcasts; dp4a accumulates exact int32 dot products.
constexpr int kScoreThreads = 256;
constexpr int kDirectChunks = 8;  // rows up to 128 bytes use direct loads

template <int NC>
__device__ __forceinline__ void score_direct(const int8_t *__restrict__ krow, const uint4 *qs,
                                             int Kr, int nc_rt, int (&acc)[kMaxKmax]) {
  const int nc = NC > 0 ? NC : nc_rt;
  const uint4 *p = reinterpret_cast<const uint4 *>(krow);
  uint4 kv[kDirectChunks];
#pragma unroll
  for (int ch = 0; ch < kDirectChunks; ++ch)
    if (ch < nc) kv[ch] = __ldg(p + ch);
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

template <int NC>
__global__ void __launch_bounds__(kScoreThreads)
k_index_score(const DevCtx c, const int8_t *__restrict__ q_idx) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int r = blockIdx.y;
  const int Kr = c.Kr[r];
  if (Kr == 0) return;
  int dom_r = 0;
  for (int j = 0; j < Kr; ++j) dom_r = max(dom_r, c.dom[r * c.Kmax + j]);
  const int64_t row0 = (int64_t)blockIdx.x * kScoreThreads;
  if (row0 >= dom_r) return;
  const int RB = c.idx_row, nc = RB >> 4;
  const int rows = (int)(dom_r - row0 < kScoreThreads ? dom_r - row0 : kScoreThreads);
  const int8_t *keys = c.keys[r] + row0 * RB;
  uint4 *qs = reinterpret_cast<uint4 *>(smem);
  uint4 *tile = qs + c.Kmax * nc;
  const bool direct = nc <= kDirectChunks;
  if (!direct) {
    const uint4 *src = reinterpret_cast<const uint4 *>(keys);
    for (int u = threadIdx.x; u < rows * nc; u += blockDim.x) {
      const int t = u / nc, ch = u - t * nc;
      int pos = ch + (t & 7);
      if (pos >= nc) pos -= nc;
      cp_async_16(&tile[t * nc + pos], &src[u]);
    }
    cp_async_commit();
  }
  const uint4 *qsrc = reinterpret_cast<const uint4 *>(q_idx + (size_t)r * c.Kmax * RB);
  for (int u = threadIdx.x; u < Kr * nc; u += blockDim.x) qs[u] = qsrc[u];
  if (!direct) cp_async_wait_all();
  __syncthreads();

  const int t = threadIdx.x;
  int acc[kMaxKmax];
#pragma unroll
  for (int j = 0; j < kMaxKmax; ++j) acc[j] = 0;
  if (t < rows) {
    if (direct) {
      score_direct<NC>(keys + (size_t)t * RB, qs, Kr, nc, acc);
    } else {
      const uint4 *myrow = tile + t * nc;
      int pos = t & 7;
      if (pos >= nc) pos %= nc;
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
#pragma unroll
    for (int j = 0; j < kMaxKmax; ++j)
      if (j < Kr) c.scores[((size_t)r * c.Kmax + j) * c.Sm + s] = acc[j];
  }
}

// ---------------------------------------------------------------- top-k
// One CTA of 1024 threads per (request, query).  (1) min and max of the
// query's scores; (2) exact radix select on the score minus the minimum, at
// most 13 bits per pass (one pass when the scores span fewer than 8192
// values); (3) ordered collection: each warp owns a contiguous run of rows,
// counts the rows above the threshold and those equal to it, and after one
// exchange of the 32 per-warp counts writes its rows in row order, keeping
// the lowest-index rows among those equal to the threshold; (4) bitonic sort
// of the k winners by (score descending, row ascending), with warp-local
// synchronisation for the strides that stay inside one warp's 64 elements.
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
  __shared__ int wmin[32], wmax[32], wgt[32], weq[32];
  __shared__ int sh_bin, sh_above;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int ksel = min(k, dom);

  // (1) range of the scores
  int mn = INT_MAX, mx = INT_MIN;
#pragma unroll 4
  for (int s = tid; s < dom; s += kTopkThreads) {
    const int v = sc[s];
    mn = min(mn, v);
    mx = max(mx, v);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 0) {
    wmin[wid] = mn;
    wmax[wid] = mx;
  }
  __syncthreads();
  mn = wmin[lane];
  mx = wmax[lane];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  const int lo = mn, hi = mx;

  if (dom <= k) {
    for (int s = tid; s < dom; s += kTopkThreads) cand[s] = topk_key((uint32_t)(sc[s] - lo), s);
  } else {
    // (2) radix select of the k-th largest offset score T
    const uint32_t range = (uint32_t)(hi - lo);
    int shift = range ? 32 - __clz((int)range) : 0;
    uint32_t prefix = 0;
    int k_rem = k;
    while (shift > 0) {
      const int width = min(kRadixBits, shift);
      shift -= width;
      const int nbins = 1 << width;
      for (int i = tid; i < nbins; i += kTopkThreads) hist[i] = 0;
      __syncthreads();
#pragma unroll 4
      for (int s = tid; s < dom; s += kTopkThreads) {
        const uint32_t v = (uint32_t)(sc[s] - lo);
        if ((uint32_t)((unsigned long long)v >> (shift + width)) == prefix)
          atomicAdd(&hist[(v >> shift) & (nbins - 1)], 1u);
      }
      __syncthreads();
      // thread t owns a run of bins counted from the top; an exclusive scan in
      // thread order then counts the rows above each run
      const int per = (nbins + kTopkThreads - 1) / kTopkThreads;
      const int b_hi = nbins - tid * per;
      const int b_lo = max(0, b_hi - per);
      int local = 0;
      for (int b = b_lo; b < b_hi; ++b) local += hist[b];
      int total;
      const int above = block_excl_scan(b_hi > 0 ? local : 0, warp_sums, total);
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

    // (3) ordered collection, one contiguous run of rows per warp
    const int run = (((dom + 31) / 32) + 31) & ~31;
    const int r0 = min(dom, wid * run), r1 = min(dom, r0 + run);
    int ngt = 0, neq = 0;
#pragma unroll 8
    for (int base = r0; base < r1; base += 32) {
      const int s = base + lane;
      const bool ok = s < r1;
      const uint32_t v = ok ? (uint32_t)(sc[s] - lo) : 0u;
      ngt += __popc(__ballot_sync(0xffffffffu, ok && v > T));
      neq += __popc(__ballot_sync(0xffffffffu, ok && v == T));
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
    int gt_off = __shfl_sync(0xffffffffu, gx - wgt[lane], wid);
    int eq_off = __shfl_sync(0xffffffffu, ex - weq[lane], wid);
    const unsigned lt = (1u << lane) - 1u;
    const int gt_end = gt_off + ngt, eq_end = eq_off + neq;  // this warp's share
#pragma unroll 4
    for (int base = r0; base < r1 && (gt_off < gt_end || (eq_off < eq_end && eq_off < need));
         base += 32) {
      const int s = base + lane;
      const bool ok = s < r1;
      const uint32_t v = ok ? (uint32_t)(sc[s] - lo) : 0u;
      const unsigned bgt = __ballot_sync(0xffffffffu, ok && v > T);
      const unsigned beq = __ballot_sync(0xffffffffu, ok && v == T);
      if (ok && v > T) cand[gt_off + __popc(bgt & lt)] = topk_key(v, s);
      if (ok && v == T) {
        const int rr = eq_off + __popc(beq & lt);
        if (rr < need) cand[c_gt + rr] = topk_key(v, s);
      }
      gt_off += __popc(bgt);
      eq_off += __popc(beq);
    }
  }

  // (4) bitonic sort ascending on (~score, row); pairs whose elements stay in
  // one warp's block of 64 only need a warp barrier
  for (int i = ksel + tid; i < kp; i += kTopkThreads) cand[i] = ~0ull;
  __syncthreads();
  int prev_stride = 0;
  for (int size = 2; size <= kp; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      // a stage whose pairs cross warp blocks, or that follows one, needs the
      // whole block; two warp-local stages in a row only need the warp
      if (stride > 32 || prev_stride > 32) __syncthreads(); else __syncwarp();
      prev_stride = stride;
      for (int i = tid; i < (kp >> 1); i += kTopkThreads) {
        const int a = 2 * stride * (i / stride) + (i % stride);
        const int b = a + stride;
        const bool asc = (a & size) == 0;
        const unsigned long long x = cand[a], y = cand[b];
        if ((x > y) == asc) {
          cand[a] = y;
          cand[b] = x;
        }
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < k; i += kTopkThreads)
    out[i] = i < ksel ? (int32_t)(uint32_t)(cand[i] & 0xFFFFFFFFull) : -1;
}

cudaError_t launch_select(const DevCtx &c, const int8_t *q_idx, int32_t *topk_out, int max_dom,
                          int active, cudaStream_t s, Timer *tm) {
  (void)active;
  if (max_dom > 0) {
    const int nc = c.idx_row >> 4;
    const size_t smem = (size_t)c.Kmax * c.idx_row +
                        (nc > kDirectChunks ? (size_t)kScoreThreads * c.idx_row : 0);
    dim3 grid((max_dom + kScoreThreads - 1) / kScoreThreads, c.N);
    cudaError_t e;
    if (tm) tm->begin(K_SCORE, s);
    if (nc == 4) {
      static size_t g4 = 0;
      if ((e = ensure_smem(k_index_score<4>, smem, g4)) != cudaSuccess) return e;
      k_index_score<4><<<grid, kScoreThreads, smem, s>>>(c, q_idx);
    } else if (nc == 8) {
      static size_t g8 = 0;
      if ((e = ensure_smem(k_index_score<8>, smem, g8)) != cudaSuccess) return e;
      k_index_score<8><<<grid, kScoreThreads, smem, s>>>(c, q_idx);
    } else {
      static size_t g0 = 0;
      if ((e = ensure_smem(k_index_score<0>, smem, g0)) != cudaSuccess) return e;
      k_index_score<0><<<grid, kScoreThreads, smem, s>>>(c, q_idx);
    }
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
