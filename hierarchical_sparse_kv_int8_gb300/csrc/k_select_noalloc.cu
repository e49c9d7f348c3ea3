// Allocation-free indexer + top-k: dhs_select_noalloc.
//
// Some callers cannot allocate device memory when they need a selection:
// code recording a CUDA graph (cudaMalloc is not allowed while a stream is
// being captured), plug-ins running inside an inference engine that owns and
// accounts for every byte of device memory, and latency-critical decode loops
// where cudaMalloc or cudaFree would synchronise the device.  For them this
// entry point takes only inputs and outputs and keeps its intermediate scores
// in one fixed array that lives in the library's own device image.
//
// The array below is loaded with the library: every GPU that loads libdhs
// holds its kNoallocScoreWords * 4 bytes (8 MiB) until the process exits.
// All calls share it and it keeps the contents of the last call, so calls
// whose work overlaps on the GPU (two streams, or two host threads) race on
// it; callers must order them, for example on one stream.
#include "dhs_internal.cuh"
#include "ptx_util.cuh"

#include <climits>
#include <mutex>

namespace dhs {

// Scores of up to 2^21 (query, row) pairs, followed by the per-query min/max.
constexpr int64_t kNoallocScoreWords = int64_t(1) << 21;
constexpr int kNoallocMinmaxWords = 2 * kMaxKmax;
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoallocScoreWords + kNoallocMinmaxWords];

namespace {

constexpr int kNaTile = 128;
constexpr int kNaThreads = 1024;

__device__ __forceinline__ int na_rot(int t, int nc) {
  return nc >= 8 ? (t % nc) : ((t * nc) >> 3) % nc;
}

// Scores of n_rows key rows against n_q queries; same arithmetic as the
// context's scoring kernel, over one contiguous key array.
__global__ void __launch_bounds__(kNaTile)
k_na_score(const int8_t *__restrict__ q, const int8_t *__restrict__ keys, int n_q, int64_t n_rows,
           int rb, int32_t *__restrict__ scores, int32_t *__restrict__ minmax) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int64_t row0 = (int64_t)blockIdx.x * kNaTile;
  if (row0 >= n_rows) return;
  const int nc = rb >> 4;
  uint4 *tile = reinterpret_cast<uint4 *>(smem);
  uint4 *qs = tile + kNaTile * nc;
  const int rows = (int)(n_rows - row0 < kNaTile ? n_rows - row0 : kNaTile);
  const uint4 *src = reinterpret_cast<const uint4 *>(keys + row0 * rb);
  for (int u = threadIdx.x; u < rows * nc; u += blockDim.x) {
    const int t = u / nc, ch = u - t * nc;
    int pos = ch + na_rot(t, nc);
    if (pos >= nc) pos -= nc;
    cp_async_16(&tile[t * nc + pos], &src[u]);
  }
  cp_async_commit();
  const uint4 *qsrc = reinterpret_cast<const uint4 *>(q);
  for (int u = threadIdx.x; u < n_q * nc; u += blockDim.x) qs[u] = qsrc[u];
  cp_async_wait_all();
  __syncthreads();
  const int t = threadIdx.x;
  int acc[kMaxKmax];
#pragma unroll
  for (int j = 0; j < kMaxKmax; ++j) acc[j] = 0;
  if (t < rows) {
    const uint4 *myrow = tile + t * nc;
    int pos = na_rot(t, nc);
    for (int ch = 0; ch < nc; ++ch) {
      const uint4 kv = myrow[pos];
      if (++pos == nc) pos = 0;
#pragma unroll
      for (int j = 0; j < kMaxKmax; ++j) {
        if (j < n_q) {
          const uint4 qv = qs[j * nc + ch];
          acc[j] = __dp4a((int)kv.x, (int)qv.x, acc[j]);
          acc[j] = __dp4a((int)kv.y, (int)qv.y, acc[j]);
          acc[j] = __dp4a((int)kv.z, (int)qv.z, acc[j]);
          acc[j] = __dp4a((int)kv.w, (int)qv.w, acc[j]);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kMaxKmax; ++j) {
    if (j >= n_q) break;
    if (t < rows) scores[(int64_t)j * n_rows + row0 + t] = acc[j];
    int mn = t < rows ? acc[j] : INT_MAX, mx = t < rows ? acc[j] : INT_MIN;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if ((t & 31) == 0 && mn <= mx) {
      atomicMin(&minmax[2 * j], mn);
      atomicMax(&minmax[2 * j + 1], mx);
    }
  }
}

__global__ void k_na_clear(int32_t *minmax, int n_q) {
  const int j = threadIdx.x;
  if (j < n_q) {
    minmax[2 * j] = INT_MAX;
    minmax[2 * j + 1] = INT_MIN;
  }
}

__device__ __forceinline__ int na_scan(int v, int *warp_sums, int &total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  total = warp_sums[nw - 1];
  const int excl = x - v + (wid > 0 ? warp_sums[wid - 1] : 0);
  __syncthreads();
  return excl;
}

// Ordered top-k of one query's scores: radix select over the offset scores,
// an ordered pass keeping the lowest rows among ties, then a bitonic sort by
// (score descending, row ascending).
__global__ void __launch_bounds__(kNaThreads)
k_na_topk(const int32_t *__restrict__ scores, const int32_t *__restrict__ minmax, int64_t n_rows,
          int k, int32_t *__restrict__ out) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int j = blockIdx.x;
  const int dom = (int)n_rows;
  const int32_t *sc = scores + (int64_t)j * n_rows;
  int32_t *o = out + (int64_t)j * k;
  int kp = 1;
  while (kp < k) kp <<= 1;
  unsigned long long *cand = reinterpret_cast<unsigned long long *>(smem);
  uint32_t *hist = reinterpret_cast<uint32_t *>(cand + kp);
  __shared__ int warp_sums[32];
  __shared__ int sh_bin, sh_above, sh_gt, sh_eqbase;
  const int tid = threadIdx.x;
  const int ksel = min(k, dom);
  const int lo = minmax[2 * j], hi = minmax[2 * j + 1];
  if (dom <= k) {
    for (int s = tid; s < dom; s += blockDim.x) {
      const uint32_t v = (uint32_t)(sc[s] - lo);
      cand[s] = ((unsigned long long)(0xFFFFFFFFu - v) << 32) | (uint32_t)s;
    }
  } else {
    const uint32_t range = (uint32_t)(hi - lo);
    int shift = range ? 32 - __clz((int)range) : 0;
    uint32_t prefix = 0;
    int k_rem = k;
    while (shift > 0) {
      const int width = min(13, shift);
      shift -= width;
      const int nbins = 1 << width;
      for (int i = tid; i < nbins; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      for (int s = tid; s < dom; s += blockDim.x) {
        const uint32_t v = (uint32_t)(sc[s] - lo);
        if ((uint32_t)((unsigned long long)v >> (shift + width)) == prefix)
          atomicAdd(&hist[(v >> shift) & (nbins - 1)], 1u);
      }
      __syncthreads();
      const int per = (nbins + blockDim.x - 1) / blockDim.x;
      const int b_hi = nbins - tid * per;
      const int b_lo = max(0, b_hi - per);
      int local = 0;
      for (int b = b_lo; b < b_hi; ++b) local += hist[b];
      int total;
      const int above = na_scan(b_hi > 0 ? local : 0, warp_sums, total);
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
    const uint32_t T = prefix;
    const int need = k_rem, c_gt = k - need;
    if (tid == 0) {
      sh_gt = 0;
      sh_eqbase = 0;
    }
    __syncthreads();
    for (int base = 0; base < dom; base += blockDim.x) {
      const int s = base + tid;
      const uint32_t v = s < dom ? (uint32_t)(sc[s] - lo) : 0u;
      const bool gt = s < dom && v > T, eq = s < dom && v == T;
      const unsigned long long key = ((unsigned long long)(0xFFFFFFFFu - v) << 32) | (uint32_t)s;
      if (gt) cand[atomicAdd(&sh_gt, 1)] = key;
      int tot;
      const int before = sh_eqbase;
      const int rank = before + na_scan(eq ? 1 : 0, warp_sums, tot);
      if (eq && rank < need) cand[c_gt + rank] = key;
      __syncthreads();
      if (tid == 0) sh_eqbase += tot;
      __syncthreads();
      const bool done = sh_gt == c_gt && sh_eqbase >= need;
      __syncthreads();
      if (done) break;
    }
  }
  for (int i = ksel + tid; i < kp; i += blockDim.x) cand[i] = ~0ull;
  __syncthreads();
  for (int size = 2; size <= kp; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < (kp >> 1); i += blockDim.x) {
        const int a = 2 * stride * (i / stride) + (i % stride), b = a + stride;
        const bool asc = (a & size) == 0;
        const unsigned long long x = cand[a], y = cand[b];
        if ((x > y) == asc) {
          cand[a] = y;
          cand[b] = x;
        }
      }
      __syncthreads();
    }
  }
  for (int i = tid; i < k; i += blockDim.x)
    o[i] = i < ksel ? (int32_t)(uint32_t)(cand[i] & 0xFFFFFFFFull) : -1;
}

// Per-device state, kept under g_noalloc_mu: the device address of
// g_noalloc_scratch (looked up once per device, with that device current) and
// the dynamic shared memory each kernel has been granted on that device
// (cudaFuncSetAttribute applies to the current device only).
constexpr int kNoallocMaxDevices = 64;
struct NoallocDevice {
  int32_t *scratch = nullptr;
  size_t granted_score = 0, granted_topk = 0;
};
std::mutex g_noalloc_mu;
NoallocDevice g_noalloc_dev[kNoallocMaxDevices];

// Scratch address for the current device, after granting the two kernels
// `smem_score` and `smem_topk` bytes of dynamic shared memory on it.
cudaError_t noalloc_setup(size_t smem_score, size_t smem_topk, int32_t **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kNoallocMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoallocDevice &d = g_noalloc_dev[dev];
  if (!d.scratch) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    d.scratch = static_cast<int32_t *>(p);
  }
  e = ensure_smem(k_na_score, smem_score, d.granted_score);
  if (e == cudaSuccess) e = ensure_smem(k_na_topk, smem_topk, d.granted_topk);
  if (e != cudaSuccess) return e;
  *out = d.scratch;
  return cudaSuccess;
}

}  // namespace
}  // namespace dhs

extern "C" int dhs_select_noalloc(const int8_t *q_idx, const int8_t *keys, int32_t n_queries,
                                  int64_t n_rows, int32_t idx_row_bytes, int32_t topk,
                                  int32_t *topk_out, dhs_stream stream) {
  using namespace dhs;
  if (!q_idx || !keys || !topk_out || n_queries < 1 || n_queries > kMaxKmax || n_rows < 1 ||
      idx_row_bytes < 16 || idx_row_bytes > 1024 || idx_row_bytes % 16 || topk < 32 ||
      topk > 4096 || topk % 32 || ((uintptr_t)q_idx & 15u) || ((uintptr_t)keys & 15u))
    return DHS_ERR_INVALID;
  if ((int64_t)n_queries * n_rows > kNoallocScoreWords) return DHS_ERR_CAPACITY;
  const size_t smem_score = (size_t)(kNaTile + kMaxKmax) * idx_row_bytes;
  int kp = 1;
  while (kp < topk) kp <<= 1;
  const size_t smem_topk = (size_t)kp * 8 + ((size_t)1 << 13) * 4;
  int32_t *scratch = nullptr;
  if (noalloc_setup(smem_score, smem_topk, &scratch) != cudaSuccess) {
    cudaGetLastError();
    return DHS_ERR_CUDA;
  }
  int32_t *scores = scratch;
  int32_t *minmax = scratch + kNoallocScoreWords;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  k_na_clear<<<1, 32, 0, s>>>(minmax, n_queries);
  k_na_score<<<(unsigned)((n_rows + kNaTile - 1) / kNaTile), kNaTile, smem_score, s>>>(
      q_idx, keys, n_queries, n_rows, idx_row_bytes, scores, minmax);
  k_na_topk<<<n_queries, kNaThreads, smem_topk, s>>>(scores, minmax, n_rows, topk, topk_out);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DHS_OK : DHS_ERR_CUDA;
}
