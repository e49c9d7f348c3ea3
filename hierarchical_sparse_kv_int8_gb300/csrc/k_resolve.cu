// Steps 2-4 of the verification round: retrieval union, residency-aware
// probe, miss compaction, hot-cache replacement and the shared host gather.
//
// "Adaptive DHiSparse", section 3.2 (residency-aware resolution, Fig. 2) and
// section 3.3 (eq. (6): U_r is the union of the K_r selections, D_r = U_r \ R_r
// the rows to recover from host; each distinct missing row is copied once and
// its location returned to every query that selected it, Fig. 3 callout 2).
//
// GB300 design.  The pages' resolver scans a B-row hot cache per lookup.  Here
// every request keeps two dense row->slot maps in HBM (hot cache and optional
// pool, 4 bytes per history row each), so a probe is one load per union row
// and its cost does not grow with B.  The union is a shared-memory bitmap over
// the history, compacted in ascending row order with popcount prefix sums.
#include "dhs_internal.cuh"
#include "ptx_util.cuh"

#include <climits>

namespace dhs {

constexpr int kUnionThreads = 1024;

__device__ __forceinline__ int ublock_excl_scan(int v, int *warp_sums, int &total) {
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

size_t union_smem_bytes(const DevCtx &c) {
  const size_t nw = (size_t)((c.Sm + 31) / 32);
  const size_t pw = (size_t)((c.B + 31) / 32);
  return nw * 8 + pw * 4 + (size_t)c.B * 8 + (size_t)c.Kmax * c.k * 4;
}

constexpr int32_t kMissMark = -2;
constexpr int kBatch = 8;  // independent global loads in flight per thread

// One CTA per request.  Shared memory holds the union bitmap over the
// history, the per-word prefix counts, the protected-slot bitmap, two B-entry
// slot lists and the location of every union row.
__global__ void __launch_bounds__(kUnionThreads)
k_union_probe(const DevCtx c, const int32_t *__restrict__ topk, int32_t *__restrict__ loc_out,
              int shared, int tick) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int warp_sums[32];
  __shared__ int sh_cnt[4];  // ring, opt, hot hits; selections
  __shared__ int sh_missel, sh_evict;
  const int r = blockIdx.x;
  const int Kr = c.Kr[r];
  if (Kr == 0) return;
  const int tid = threadIdx.x, bs = blockDim.x;
  const int64_t n = c.n[r];
  const int k = c.k, KK = c.Kmax * k, B = c.B;
  const int nw_cap = (int)((c.Sm + 31) / 32);
  const int nw = (int)((n + 31) >> 5);
  const int pw = (B + 31) >> 5;
  uint32_t *bm = reinterpret_cast<uint32_t *>(smem);
  uint32_t *wp = bm + nw_cap;
  uint32_t *prot = wp + nw_cap;
  int32_t *candB = reinterpret_cast<int32_t *>(prot + pw);
  int32_t *tmpB = candB + B;
  int32_t *ul = tmpB + B;  // location of union row q

  const int32_t *tk = topk + (size_t)r * KK;
  int32_t *uni = c.uni + (size_t)r * KK;
  int32_t *miss = c.miss + (size_t)r * KK;
  int32_t *hot_row = c.hot_row + (size_t)r * B;
  int32_t *hot_stamp = c.hot_stamp + (size_t)r * B;
  int32_t *lru = c.lru + (size_t)r * B;
  int32_t *hot_map = c.hot_map + (size_t)r * c.Sm;
  const int32_t *opt_map = c.opt_map + (size_t)r * c.Sm;
  const int64_t ring_lo = max(c.ring_first[r], n - (int64_t)c.W);
  const int nsel = Kr * k;

  // 1. union bitmap over the history rows
  for (int i = tid; i < nw; i += bs) bm[i] = 0;
  for (int i = tid; i < pw; i += bs) prot[i] = 0;
  if (tid < 4) sh_cnt[tid] = 0;
  if (tid == 0) {
    sh_missel = 0;
    sh_evict = 0;
  }
  __syncthreads();
  for (int e0 = tid; e0 < nsel; e0 += kBatch * bs) {
    int32_t sv[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int e = e0 + i * bs;
      sv[i] = e < nsel ? tk[e] : -1;
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int32_t s = sv[i];
      if (s >= 0 && s < n) atomicOr(&bm[s >> 5], 1u << (s & 31));
      else if (s != -1) record_error(c.err, DC_ROW_RANGE, K_UNION_PROBE);
    }
  }
  __syncthreads();

  // 2. ascending compaction; each thread owns a contiguous run of words
  const int per = (nw + bs - 1) / bs;
  const int w0 = min(nw, tid * per), w1 = min(nw, w0 + per);
  int cnt = 0;
  for (int w = w0; w < w1; ++w) cnt += __popc(bm[w]);
  int U;
  const int u_base = ublock_excl_scan(cnt, warp_sums, U);

  // 3. probe each union row: live ring tail, optional map, hot cache, else miss
  int misses_here = 0, ring_h = 0, opt_h = 0, hot_h = 0;
  {
    int q = u_base;
    int w = w0;
    uint32_t bits = 0;
    if (w < w1) {
      wp[w] = q;
      bits = bm[w];
    }
    for (;;) {
      int32_t ub[kBatch];
      int nb = 0;
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        while (bits == 0 && w < w1) {
          if (++w < w1) {
            wp[w] = q + i;
            bits = bm[w];
          }
        }
        if (bits) {
          ub[i] = (w << 5) | (__ffs(bits) - 1);
          bits &= bits - 1;
          nb = i + 1;
        } else {
          ub[i] = -1;
        }
      }
      int32_t hm[kBatch], om[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        hm[i] = ub[i] >= 0 ? hot_map[ub[i]] : -1;
        om[i] = ub[i] >= 0 ? opt_map[ub[i]] : -1;
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int32_t u = ub[i];
        if (u < 0) continue;
        const int32_t hs = hm[i];
        if (hs >= 0) atomicOr(&prot[hs >> 5], 1u << (hs & 31));  // selected rows are protected
        int32_t l;
        if (u >= ring_lo && u < n) {
          l = make_loc(DHS_LOC_RING, (int)(u % c.Rd));
          ++ring_h;
        } else if (om[i] >= 0) {
          l = make_loc(DHS_LOC_OPT, om[i]);
          ++opt_h;
        } else if (hs >= 0) {
          l = make_loc(DHS_LOC_HOT, hs);
          hot_stamp[hs] = tick;
          ++hot_h;
        } else {
          l = kMissMark - u;  // a miss, row kept until its rank is known
          ++misses_here;
        }
        uni[q] = u;
        ul[q] = l;
        ++q;
      }
      if (nb < kBatch) break;
    }
  }
  atomicAdd(&sh_cnt[0], ring_h);
  atomicAdd(&sh_cnt[1], opt_h);
  atomicAdd(&sh_cnt[2], hot_h);
  int M;
  const int m_base = ublock_excl_scan(misses_here, warp_sums, M);
  if (misses_here) {
    int m = m_base;
    for (int q = u_base; q < u_base + cnt; ++q) {
      const int32_t l = ul[q];
      if (l <= kMissMark) {
        miss[m] = kMissMark - l;
        ul[q] = make_loc(DHS_LOC_STAGE, m);
        ++m;
      }
    }
  }
  for (int i = tid; i < M; i += bs) c.first_occ[(size_t)r * KK + i] = INT_MAX;
  __syncthreads();
  const int hits = sh_cnt[2];

  // 4. victims: unprotected slots in LRU order (stamp, slot), empty slots first
  int P = 0;
  const int perB = (B + bs - 1) / bs;
  const int b0 = min(B, tid * perB), b1 = min(B, b0 + perB);
  if (M > 0) {
    int nc = 0;
#pragma unroll 4
    for (int i = b0; i < b1; ++i) {
      const int v = lru[i];
      nc += !((prot[v >> 5] >> (v & 31)) & 1u);
    }
    int ncand;
    int cb = ublock_excl_scan(nc, warp_sums, ncand);
    for (int i = b0; i < b1; ++i) {
      const int v = lru[i];
      if (!((prot[v >> 5] >> (v & 31)) & 1u)) candB[cb++] = v;
    }
    __syncthreads();
    P = min(M, ncand);
    int ev = 0;
    for (int p0 = tid; p0 < P; p0 += kBatch * bs) {
      int vv[kBatch], old[kBatch], uu[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int p = p0 + i * bs;
        vv[i] = p < P ? candB[p] : -1;
        old[i] = vv[i] >= 0 ? hot_row[vv[i]] : -1;
        uu[i] = p < P ? miss[p] : -1;
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int p = p0 + i * bs;
        if (vv[i] < 0) continue;
        if (old[i] >= 0) {
          hot_map[old[i]] = -1;
          ++ev;
        }
        hot_row[vv[i]] = uu[i];
        hot_stamp[vv[i]] = tick;
        hot_map[uu[i]] = vv[i];
        c.promo_dst[(size_t)r * B + p] = vv[i];
        c.promo_src[(size_t)r * B + p] = p;
      }
    }
    if (ev) atomicAdd(&sh_evict, ev);
    __syncthreads();
  }

  // 5. LRU order after this tick: untouched slots keep their order, slots
  //    stamped now follow in ascending slot order
  if (hits + P > 0) {
    int na = 0, nb = 0;
#pragma unroll 4
    for (int i = b0; i < b1; ++i) {
      const int v = lru[i];
      const bool now = hot_stamp[v] == tick;
      na += !now;
      tmpB[i] = now ? -1 : v;  // scratch: this thread's positions only
    }
#pragma unroll 4
    for (int v = b0; v < b1; ++v) nb += hot_stamp[v] == tick;
    int A, Bt;
    int ab = ublock_excl_scan(na, warp_sums, A);
    int bb = ublock_excl_scan(nb, warp_sums, Bt);
    for (int i = b0; i < b1; ++i)
      if (tmpB[i] >= 0) candB[ab++] = tmpB[i];
    for (int v = b0; v < b1; ++v)
      if (hot_stamp[v] == tick) candB[A + bb++] = v;
    __syncthreads();
    for (int i = tid; i < B; i += bs) lru[i] = candB[i];
  }

  // 6. one location per selected entry, in each query's selection order
  int sel_here = 0, missel = 0;
  for (int e0 = tid; e0 < nsel; e0 += kBatch * bs) {
    int32_t sv[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int e = e0 + i * bs;
      sv[i] = e < nsel ? tk[e] : -2;
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int e = e0 + i * bs;
      const int32_t s = sv[i];
      if (s == -2) continue;
      int32_t l = -1;
      if (s >= 0 && s < n) {
        const uint32_t word = bm[s >> 5];
        const int q = wp[s >> 5] + __popc(word & ((1u << (s & 31)) - 1u));
        l = ul[q];
        ++sel_here;
        if (loc_tier(l) == DHS_LOC_STAGE) {
          ++missel;
          if (!shared) {
            atomicMin(&c.first_occ[(size_t)r * KK + loc_index(l)], e);
            l = make_loc(DHS_LOC_STAGE, e);
          }
        }
      }
      loc_out[(size_t)r * KK + e] = l;
    }
  }
  atomicAdd(&sh_cnt[3], sel_here);
  atomicAdd(&sh_missel, missel);
  __syncthreads();
  if (!shared) {
    for (int p = tid; p < P; p += bs)
      c.promo_src[(size_t)r * B + p] = c.first_occ[(size_t)r * KK + p];
  }
  if (tid == 0) {
    c.counts[r * 4 + 0] = U;
    c.counts[r * 4 + 1] = M;
    c.counts[r * 4 + 2] = P;
    c.counts[r * 4 + 3] = hits;
    atomicAdd(&c.stats[ST_SEL], (unsigned long long)sh_cnt[3]);
    atomicAdd(&c.stats[ST_UNION], (unsigned long long)U);
    atomicAdd(&c.stats[ST_RING], (unsigned long long)sh_cnt[0]);
    atomicAdd(&c.stats[ST_OPT], (unsigned long long)sh_cnt[1]);
    atomicAdd(&c.stats[ST_HOT], (unsigned long long)hits);
    atomicAdd(&c.stats[ST_MISS], (unsigned long long)M);
    atomicAdd(&c.stats[ST_MISS_SEL], (unsigned long long)sh_missel);
    atomicAdd(&c.stats[ST_FETCHED], (unsigned long long)(shared ? M : sh_missel));
    atomicAdd(&c.stats[ST_INSTALL], (unsigned long long)P);
    if (sh_evict) atomicAdd(&c.stats[ST_EVICT], (unsigned long long)sh_evict);
    if (M == 0 && hits == 0) atomicAdd(&c.stats[ST_DIRECT], 1ull);
  }
}

// Shared host gather: staging[r][m] <- host[r][D_r[m]], one warp per row,
// 16-byte zero-copy loads from pinned host memory, four rows in flight per
// warp.  In per-query mode every missing selection (j, i) is fetched into
// staging row j*k + i.
constexpr int kGatherWarps = 8;
constexpr int kGatherBatch = 4;
constexpr int kGatherVec = 4;  // up to 4 x 32 x 16 B = 2 KB rows

__global__ void __launch_bounds__(kGatherWarps * 32)
k_gather(const DevCtx c, const int32_t *__restrict__ topk, const int32_t *__restrict__ loc,
         int shared) {
  const int r = blockIdx.y;
  const int Kr = c.Kr[r];
  if (Kr == 0) return;
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kGatherWarps + (threadIdx.x >> 5);
  const int nwt = gridDim.x * kGatherWarps;
  const int KK = c.Kmax * c.k;
  const int nv = (c.row * 2) >> 4;
  const uint16_t *host = c.host[r];
  const int64_t n = c.n[r];
  const int count = shared ? c.counts[r * 4 + 1] : Kr * c.k;
  for (int base = gw; base < count; base += kGatherBatch * nwt) {
    uint4 buf[kGatherBatch][kGatherVec];
    int64_t srow[kGatherBatch];
    int dst[kGatherBatch];
#pragma unroll
    for (int b = 0; b < kGatherBatch; ++b) {
      const int e = base + b * nwt;
      srow[b] = -1;
      dst[b] = e;
      if (e < count) {
        if (shared) {
          srow[b] = c.miss[(size_t)r * KK + e];
        } else {
          const int32_t l = loc[(size_t)r * KK + e];
          if (l >= 0 && loc_tier(l) == DHS_LOC_STAGE) srow[b] = topk[(size_t)r * KK + e];
        }
        if (srow[b] >= n) {
          record_error(c.err, DC_ROW_RANGE, K_GATHER);
          srow[b] = -1;
        }
      }
      if (srow[b] >= 0) {
        const uint4 *src = reinterpret_cast<const uint4 *>(host + srow[b] * c.row);
#pragma unroll
        for (int i = 0; i < kGatherVec; ++i) {
          const int v = lane + 32 * i;
          if (v < nv) buf[b][i] = ld_stream_16(src + v);
        }
      }
    }
#pragma unroll
    for (int b = 0; b < kGatherBatch; ++b) {
      if (srow[b] < 0) continue;
      uint4 *d = reinterpret_cast<uint4 *>(c.stage + ((size_t)r * KK + dst[b]) * c.row);
#pragma unroll
      for (int i = 0; i < kGatherVec; ++i) {
        const int v = lane + 32 * i;
        if (v < nv) d[v] = buf[b][i];
      }
    }
  }
}

cudaError_t launch_resolve(const DevCtx &c, const int32_t *topk, int32_t *loc_out, int shared,
                           int tick, cudaStream_t s, Timer *tm) {
  static size_t granted = 0;
  cudaError_t e = ensure_smem(k_union_probe, union_smem_bytes(c), granted);
  if (e != cudaSuccess) return e;
  if (tm) tm->begin(K_UNION_PROBE, s);
  k_union_probe<<<c.N, kUnionThreads, union_smem_bytes(c), s>>>(c, topk, loc_out, shared, tick);
  if (tm) tm->end(K_UNION_PROBE, s);
  // enough warps in flight to cover the host link's bandwidth-delay product
  int blocks_per_req = (152 * 8 + c.N - 1) / c.N;
  if (blocks_per_req < 1) blocks_per_req = 1;
  dim3 grid(blocks_per_req, c.N);
  if (tm) tm->begin(K_GATHER, s);
  k_gather<<<grid, kGatherWarps * 32, 0, s>>>(c, topk, loc_out, shared);
  if (tm) tm->end(K_GATHER, s);
  return cudaGetLastError();
}

}  // namespace dhs
