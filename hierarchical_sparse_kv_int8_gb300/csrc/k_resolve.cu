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

#include <cooperative_groups.h>

#include <climits>

namespace dhs {

// 512 threads with at most 64 registers each (half an SM's registers) and a
// shared-memory footprint kept under kUnionSmemBudget, so that a probe CTA
// fits on an SM beside two indexer CTAs of another request group.
constexpr int kUnionThreads = 512;
constexpr int kUnionSmemBudget = 96 * 1024;
// Union rows of one slice held in shared memory; a slice with more (a union
// concentrated in one part of the history) keeps its rows, locations and
// query masks in a global scratch area of its own instead.
constexpr int kUnionCap = 4096;

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

// Adds the warp's values to a shared counter with one atomic per warp (all
// lanes call it).
__device__ __forceinline__ void warp_add(int *dst, int v) {
  v = __reduce_add_sync(0xffffffffu, v);
  if ((threadIdx.x & 31) == 0 && v) atomicAdd(dst, v);
}

// The union/probe of one request runs on a cluster of kUnionCluster CTAs.
// CTA c >= 1 owns the (c-1)-th slice of the history rows: its shared memory
// holds the union bitmap of that slice, the prefix count of every word, the
// slice's union rows and their locations, and the protected-slot and
// stamped-now bitmaps of the hot cache marked by its own probes (shared-memory
// atomics).  After the first cluster barrier the leader CTA (rank 0), which
// owns no slice, merges the slices' bitmaps through distributed shared memory
// and chooses the victims while the other CTAs form their locations.
constexpr int kUnionCluster = 8;
constexpr int32_t kMissMark = -2;
constexpr int kBatch = 8;  // independent global loads in flight per thread

// The history is cut into kUnionSlices slices, one per CTA of ranks
// 1..kUnionCluster-1; the leader (rank 0) owns no slice, so its victim choice
// runs while the other CTAs form their locations.
constexpr int kUnionSlices = kUnionCluster - 1;
__host__ __device__ static inline int union_slice(int64_t s_max) {
  return (int)((((s_max + kUnionSlices - 1) / kUnionSlices) + 31) & ~31);
}

// Union rows a slice keeps in shared memory.
__host__ __device__ inline int union_cap(const DevCtx &c) { return min(c.Kmax * c.k, kUnionCap); }
// Shared memory of one CTA without, and with, the slice's hot and optional
// map entries; the entries are kept (fetched while the bitmap is built) when
// they fit the budget.
__host__ __device__ inline size_t union_base_bytes(const DevCtx &c) {
  const int slice = union_slice(c.Sm);
  const size_t sw = (size_t)slice / 32;  // words of one slice
  const size_t pw = (size_t)((c.B + 31) / 32);
  const size_t uc = (size_t)union_cap(c);
  return sw * 8 + pw * 8 + (size_t)c.B * 8 + uc * 8 + (uc + 3) / 4 * 4;
}
__host__ __device__ inline bool union_map_prefetch(const DevCtx &c) {
  return union_base_bytes(c) + (size_t)union_slice(c.Sm) * 8 <= (size_t)kUnionSmemBudget;
}
// Global scratch of a slice whose union outgrows union_cap: rows and
// locations (Kmax * k each) and the query-mask bytes; none when the cap
// covers every selection of a request.
__host__ __device__ inline size_t union_spill_ints(const DevCtx &c) {
  const size_t KK = (size_t)c.Kmax * c.k;
  return KK > (size_t)kUnionCap ? 2 * KK + (KK + 3) / 4 : 0;
}
size_t union_spill_ints_per_request(const DevCtx &c) {
  return union_spill_ints(c) * kUnionSlices;
}
size_t union_smem_bytes(const DevCtx &c) {
  return union_base_bytes(c) + (union_map_prefetch(c) ? (size_t)union_slice(c.Sm) * 8 : 0);
}

__global__ void __cluster_dims__(kUnionCluster, 1, 1) __launch_bounds__(kUnionThreads, 2)
k_union_probe(const DevCtx c, const int32_t *__restrict__ topk, int32_t *__restrict__ loc_out,
              int shared, int tick) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int warp_sums[32];
  __shared__ int sh_cnt[6];  // ring, opt, hot hits, selections, miss selections, mask bits
  __shared__ int sh_p;  // the leader's P
  // every CTA's union rows, misses and hot hits, written by that CTA into
  // each CTA of the cluster before the first cluster barrier
  __shared__ int cl_cnt[kUnionCluster][3];
  const int crank = (int)cl.block_rank();
  const int r = blockIdx.x / kUnionCluster;
  const int Kr = c.Kr[r];  // written two launches back (scoring)
  if (Kr == 0) {
    pdl_wait();
    return;  // the whole cluster leaves together
  }
  // (split cluster barrier: every CTA has started before any CTA writes
  // into another's shared memory; the wait comes just before those writes)
  cluster_arrive_relaxed();
  const int tid = threadIdx.x, bs = blockDim.x;
  const int64_t n = c.n[r];
  const int k = c.k, KK = c.Kmax * k, B = c.B;
  const int slice = union_slice(c.Sm);
  const int sw = slice / 32;
  const int pw = (B + 31) >> 5;
  const int64_t row_lo = crank == 0 ? 0 : (int64_t)(crank - 1) * slice;
  const int64_t row_hi = crank == 0 ? 0 : min(n, row_lo + slice);
  const int nw = row_hi > row_lo ? (int)((row_hi - row_lo + 31) >> 5) : 0;
  uint32_t *bm = reinterpret_cast<uint32_t *>(smem);
  uint32_t *wp = bm + sw;
  uint32_t *prot = wp + sw;  // protected slots (the leader: of the request)
  uint32_t *now = prot + pw;  // slots stamped by this tick (likewise)
  int32_t *candB = reinterpret_cast<int32_t *>(now + pw);
  int32_t *lru_s = candB + B;  // leader: LRU order at the start of the call
  const int ucap = union_cap(c);
  // (these three move to the slice's global scratch when its union outgrows ucap)
  int32_t *ul = lru_s + B;     // location of each union row of this slice
  int32_t *urow = ul + ucap;   // the slice's union rows, by union index
  uint32_t *umw = reinterpret_cast<uint32_t *>(urow + ucap);  // query masks, one byte per union row
  const bool pf = union_map_prefetch(c);
  int32_t *hmap_s = reinterpret_cast<int32_t *>(umw + (ucap + 3) / 4);  // slice's hot-map entries (when pf)
  int32_t *omap_s = hmap_s + slice;

  const int32_t *tk = topk + (size_t)r * KK;
  int32_t *uni = c.uni + (size_t)r * KK;
  int4 *uent = c.uent + (size_t)r * KK;
  int32_t *miss = c.miss + (size_t)r * KK;
  int32_t *hot_stamp = c.hot_stamp + (size_t)r * B;
  int32_t *lru = c.lru + (size_t)r * B;
  int32_t *hot_map = c.hot_map + (size_t)r * c.Sm;
  const int32_t *opt_map = c.opt_map + (size_t)r * c.Sm;
  const int64_t ring_lo = max(c.ring_first[r], n - (int64_t)c.W);
  const int nsel = Kr * k;

  // 0. start fetching what the later phases read: this slice's map entries,
  //    and for the leader the LRU order.  These
  //    are state of earlier rounds, complete before the preceding launch
  //    (top-k) began, so the copies start before that launch has finished.
  const bool any_opt = c.opt_count[r] > 0;
  if (pf) {
    for (int i = tid; i < row_hi - row_lo; i += bs) {
      cp_async_4(&hmap_s[i], &hot_map[row_lo + i]);
      if (any_opt) cp_async_4(&omap_s[i], &opt_map[row_lo + i]);
    }
  }
  if (crank == 0) {
    for (int i = tid; i < B; i += bs) {
      cp_async_4(&lru_s[i], &lru[i]);
    }
  }
  cp_async_commit();
  pdl_wait();  // the selections of the preceding launch are complete
  pdl_trigger();

  // 1. union bitmap of this CTA's slice
  for (int i = tid; i < sw; i += bs) bm[i] = 0;
  for (int i = tid; i < 2 * pw; i += bs) prot[i] = 0;  // prot and now
  if (tid < 6) sh_cnt[tid] = 0;
  __syncthreads();
  for (int e0 = crank == 0 ? nsel : tid; e0 < nsel; e0 += kBatch * bs) {
    int32_t sv[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int e = e0 + i * bs;
      sv[i] = e < nsel ? tk[e] : -1;
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int32_t s = sv[i];
      if (s >= row_lo && s < row_hi) {
        const int rel = (int)(s - row_lo);
        atomicOr(&bm[rel >> 5], 1u << (rel & 31));
      } else if (crank == 1 && s != -1 && (s < 0 || s >= n)) {
        record_error(c.err, DC_ROW_RANGE, K_UNION_PROBE);
      }
    }
  }
  __syncthreads();  // the slice's bitmap is complete

  // 2. ascending compaction of the slice: each thread owns a run of words,
  //    records for every word the union index of its first row, and lists
  //    the run's rows by union index
  const int per = (nw + bs - 1) / bs;
  const int w0 = min(nw, tid * per), w1 = min(nw, w0 + per);
  int cnt = 0;
  for (int w = w0; w < w1; ++w) cnt += __popc(bm[w]);
  int Uc;
  {
    int q = ublock_excl_scan(cnt, warp_sums, Uc);
    if (Uc > ucap) {  // (the same in every thread; only slice CTAs have rows)
      int32_t *sp = c.uspill + ((size_t)r * kUnionSlices + (crank - 1)) * union_spill_ints(c);
      ul = sp;
      urow = sp + KK;
      umw = reinterpret_cast<uint32_t *>(sp + 2 * (size_t)KK);
    }
    for (int i = tid; i < (Uc + 3) / 4; i += bs) umw[i] = 0;
    for (int w = w0; w < w1; ++w) {
      wp[w] = q;
      for (uint32_t bits = bm[w]; bits; bits &= bits - 1)
        urow[q++] = (int32_t)(row_lo + ((w << 5) | (__ffs(bits) - 1)));
    }
  }

  cp_async_wait_all();
  __syncthreads();  // the row list and prefetched map entries are in place

  // 3. probe each union row of the slice: live ring tail, optional map, hot
  //    cache, else miss; the protected and stamped hot slots are marked.
  //    Thread t takes the union indices [t * pr, (t + 1) * pr), in order, so
  //    the misses are ranked by one scan.
  const int pr = (Uc + bs - 1) / bs;
  const int q0 = min(Uc, tid * pr), q1 = min(Uc, q0 + pr);
  int ring_h = 0, opt_h = 0, hot_h = 0, misses_here = 0;
  for (int qb = q0; qb < q1; qb += kBatch) {
    int32_t hsv[kBatch], omv[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {  // map loads of the batch in flight together
      hsv[i] = omv[i] = -1;
      const int q = qb + i;
      if (q < q1) {
        const int32_t u = urow[q];
        const int rel = (int)(u - row_lo);
        hsv[i] = pf ? hmap_s[rel] : hot_map[u];
        if (any_opt) omv[i] = pf ? omap_s[rel] : opt_map[u];
      }
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int q = qb + i;
      if (q >= q1) break;
      const int32_t u = urow[q];
      const int32_t hs = hsv[i], om = omv[i];
      if (hs >= 0) atomicOr(&prot[hs >> 5], 1u << (hs & 31));
      int32_t l;
      if (u >= ring_lo && u < n) {
        l = make_loc(DHS_LOC_RING, (int)(u % c.Rd));
        ++ring_h;
      } else if (om >= 0) {
        l = make_loc(DHS_LOC_OPT, om);
        ++opt_h;
      } else if (hs >= 0) {
        l = make_loc(DHS_LOC_HOT, hs);
        hot_stamp[hs] = tick;
        atomicOr(&now[hs >> 5], 1u << (hs & 31));
        ++hot_h;
      } else {
        l = kMissMark;
        ++misses_here;
      }
      ul[q] = l;
    }
  }
  warp_add(&sh_cnt[0], ring_h);
  warp_add(&sh_cnt[1], opt_h);
  warp_add(&sh_cnt[2], hot_h);
  int Mc;
  const int m_local = ublock_excl_scan(misses_here, warp_sums, Mc);
  cluster_wait();
  if (tid < kUnionCluster) {  // (remote stores: no round trip; S1 orders them)
    int *dst = cl.map_shared_rank(&cl_cnt[crank][0], tid);
    dst[0] = Uc;
    dst[1] = Mc;
    dst[2] = sh_cnt[2];
  }
  cl.sync();  // S1: counts published, protected and stamped slots complete

  int u_base = 0, m_base = 0, U = 0, M = 0, hits = 0;
#pragma unroll
  for (int qr = 0; qr < kUnionCluster; ++qr) {
    const int uq = cl_cnt[qr][0], mq = cl_cnt[qr][1];
    if (qr < crank) {
      u_base += uq;
      m_base += mq;
    }
    U += uq;
    M += mq;
    hits += cl_cnt[qr][2];
  }
  // the leader merges the protected and stamped slots of every slice
  if (crank == 0)
    for (int i = tid; i < pw; i += bs) {
      uint32_t pv = 0, nv = 0;
#pragma unroll
      for (int qr = 0; qr < kUnionCluster; ++qr) {
        pv |= cl.map_shared_rank(prot, qr)[i];
        nv |= cl.map_shared_rank(now, qr)[i];
      }
      prot[i] = pv;
      now[i] = nv;
    }
  // union rows and misses of the slice get their request-wide ranks, each
  // thread over the union indices it probed
  for (int q = q0, m = m_base + m_local; q < q1; ++q) {
    const int32_t u = urow[q];
    uni[u_base + q] = u;
    if (ul[q] == kMissMark) {
      miss[m] = u;
      c.first_occ[(size_t)r * KK + m] = INT_MAX;
      ul[q] = make_loc(DHS_LOC_STAGE, m);
      ++m;
    }
    *reinterpret_cast<int2 *>(&uent[u_base + q]) = make_int2(u, ul[q]);
  }
  __syncthreads();  // the slice's locations and first-selection slots are set

  // 4. one location per selected entry whose row lies in this slice (they
  //    depend on the ranks only; the slice-free leader skips this phase and
  //    picks the victims meanwhile)
  int sel_here = 0, missel = 0;
  for (int e0 = crank == 0 ? nsel : tid; e0 < nsel; e0 += kBatch * bs) {
    int32_t sv[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int e = e0 + i * bs;
      sv[i] = e < nsel ? tk[e] : -1;
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int e = e0 + i * bs;
      if (e >= nsel) continue;
      const int32_t s = sv[i];
      const bool mine = s >= row_lo && s < row_hi;
      if (!mine) {
        if (crank == 1 && (s < 0 || s >= n)) loc_out[(size_t)r * KK + e] = -1;
        continue;
      }
      const int rel = (int)(s - row_lo);
      const uint32_t word = bm[rel >> 5];
      const int q = wp[rel >> 5] + __popc(word & ((1u << (rel & 31)) - 1u));
      int32_t l = ul[q];
      // query e / k, by a multiply with the rounded-up reciprocal of k (exact
      // for e < 8k and k < 2^14)
      const uint32_t qbit = 1u << ((q & 3) * 8 + (int)__umulhi((unsigned)e, c.kinv));
      atomicOr(&umw[q >> 2], qbit);
      ++sel_here;
      if (loc_tier(l) == DHS_LOC_STAGE) {
        ++missel;
        if (!shared) {
          atomicMin(&c.first_occ[(size_t)r * KK + loc_index(l)], e);
          l = make_loc(DHS_LOC_STAGE, e);
          c.inst[(size_t)r * KK + e] = -1;
        }
      }
      loc_out[(size_t)r * KK + e] = l;
    }
  }
  warp_add(&sh_cnt[3], sel_here);
  warp_add(&sh_cnt[4], missel);
  __syncthreads();  // the query masks of the slice are complete
  // 5. second half of each union entry: the queries that selected the row.
  //    A row listed twice by one query sets one bit for two selections, so
  //    the slice's bits fall short of its selections exactly when a query
  //    repeats a row (checked at the end).
  {
    int bits_here = 0;
    for (int q = tid; q < Uc; q += bs) {
      const uint32_t qm = (umw[q >> 2] >> ((q & 3) * 8)) & 0xFFu;
      bits_here += __popc(qm);
      *reinterpret_cast<int2 *>(&uent[u_base + q].z) = make_int2((int)qm, 0);
    }
    warp_add(&sh_cnt[5], bits_here);
  }
  // 6. victims (leader): unprotected slots in LRU order (stamp, slot), empty first
  const int perB = (B + bs - 1) / bs;
  const int b0 = min(B, tid * perB), b1 = min(B, b0 + perB);
  if (crank == 0) {
    int P = 0;
    if (M > 0) {
      int nc = 0;
#pragma unroll 4
      for (int i = b0; i < b1; ++i) {
        const int v = lru_s[i];
        nc += !((prot[v >> 5] >> (v & 31)) & 1u);
      }
      int ncand;
      int cb = ublock_excl_scan(nc, warp_sums, ncand);
      P = min(M, ncand);
      for (int i = b0; i < b1; ++i) {
        const int v = lru_s[i];
        if (!((prot[v >> 5] >> (v & 31)) & 1u)) {
          candB[cb] = v;
          if (cb < P) {
            atomicOr(&now[v >> 5], 1u << (v & 31));  // stamped by this tick
            c.promo_dst[(size_t)r * B + cb] = v;      // the cb-th miss takes slot v
          }
          ++cb;
        }
      }
    }
    if (tid == 0) sh_p = P;
    __syncthreads();  // every stamped-now bit is set
    for (int i = tid; i < pw; i += bs) c.now_bits[(size_t)r * pw + i] = now[i];
  }
  cl.sync();  // S2: every slice's misses are in the miss list and every first
              // selection of a miss is known; no CTA reads the leader's memory
              // after this point
  // The promotions' cache state (slot rows, stamps, maps) and the LRU order
  // after this tick are written by the gather (hot_update below): only the
  // next round and the exported state read them, so they leave this
  // kernel's critical path.
  const int P = crank == 0 ? sh_p : 0;

  // the first selection of each promoted miss also fills its hot slot
  if (!shared && crank == 0)
    for (int p = tid; p < P; p += bs)
      c.inst[(size_t)r * KK + c.first_occ[(size_t)r * KK + p]] = candB[p];
  __syncthreads();
  if (tid == 0) {
    if (sh_cnt[5] != sh_cnt[3]) record_error(c.err, DC_DUPLICATE, K_UNION_PROBE);
    atomicAdd(&c.stats[ST_SEL], (unsigned long long)sh_cnt[3]);
    atomicAdd(&c.stats[ST_RING], (unsigned long long)sh_cnt[0]);
    atomicAdd(&c.stats[ST_OPT], (unsigned long long)sh_cnt[1]);
    atomicAdd(&c.stats[ST_HOT], (unsigned long long)sh_cnt[2]);
    atomicAdd(&c.stats[ST_MISS_SEL], (unsigned long long)sh_cnt[4]);
    if (!shared) atomicAdd(&c.stats[ST_FETCHED], (unsigned long long)sh_cnt[4]);
    if (crank == 0) {
      c.counts[r * 4 + 0] = U;
      c.counts[r * 4 + 1] = M;
      c.counts[r * 4 + 2] = P;
      c.counts[r * 4 + 3] = hits;
      atomicAdd(&c.stats[ST_UNION], (unsigned long long)U);
      atomicAdd(&c.stats[ST_MISS], (unsigned long long)M);
      if (shared) atomicAdd(&c.stats[ST_FETCHED], (unsigned long long)M);
      atomicAdd(&c.stats[ST_INSTALL], (unsigned long long)P);
      if (M == 0 && hits == 0) atomicAdd(&c.stats[ST_DIRECT], 1ull);
    }
  }
}

// Shared host gather: staging[r][m] <- host[r][D_r[m]], one warp per row,
// 16-byte zero-copy loads from pinned host memory, several rows in flight per
// warp.  In per-query mode every missing selection (j, i) is fetched into
// staging row j*k + i.  A promoted row is written to its hot-cache slot from
// the same registers ("Adaptive DHiSparse", section 3.4, installs promoted
// rows after the attention readers; the victim slots are unprotected, so no
// location of this round names them and the install may come first).
// VEC 16-byte vectors per lane cover a row (VEC x 512 B); BATCH rows are in
// flight per warp, so each warp keeps about 4 KB of loads outstanding (deeper
// batches measured no faster: the host link is already saturated).
constexpr int kGatherWarps = 8;
constexpr int kGatherMaxVec = 4;  // rows up to 2 KB

template <int VEC>
struct GatherShape {
  static constexpr int kGatherVec = VEC;
  static constexpr int kGatherBatch = VEC == 1 ? 8 : VEC == 2 ? 4 : 2;
};

// Cache state after this tick for request r, written by one CTA of the
// gather while the others fetch (section 3.2, Fig. 2): each promoted miss p
// takes slot promo_dst[p] (the slot's previous row leaves the hot map), and
// the LRU order becomes the slots not stamped by this tick in their previous
// order, followed by the stamped ones (hits and promotions) in ascending slot
// order.  Only the next round's union/probe and the exported state read
// these; the order is rebuilt in a scratch array and copied back.
__device__ void hot_update(const DevCtx &c, int r, int tick, int *warp_sums) {
  const int B = c.B, pw = (B + 31) >> 5, KK = c.Kmax * c.k;
  const int tid = threadIdx.x, bs = blockDim.x;
  const int P = c.counts[r * 4 + 2], hits = c.counts[r * 4 + 3];
  int32_t *hot_row = c.hot_row + (size_t)r * B;
  int32_t *hot_stamp = c.hot_stamp + (size_t)r * B;
  int32_t *hot_map = c.hot_map + (size_t)r * c.Sm;
  int32_t *lru = c.lru + (size_t)r * B;
  int32_t *nxt = c.lru_next + (size_t)r * B;
  const uint32_t *now = c.now_bits + (size_t)r * pw;
  const int32_t *dst = c.promo_dst + (size_t)r * B;
  const int32_t *miss = c.miss + (size_t)r * KK;
  int ev = 0;
  for (int p = tid; p < P; p += bs) {
    const int v = dst[p];
    const int32_t old = hot_row[v], u = miss[p];
    if (old >= 0) {
      hot_map[old] = -1;
      ++ev;
    }
    hot_row[v] = u;
    hot_stamp[v] = tick;
    hot_map[u] = v;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ev += __shfl_xor_sync(0xffffffffu, ev, o);
  if ((tid & 31) == 0 && ev) atomicAdd(&c.stats[ST_EVICT], (unsigned long long)ev);
  if (hits + P == 0) return;  // nothing stamped: the order stands
  const int per = (B + bs - 1) / bs;
  const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
  auto stamped = [&](int v) { return (now[v >> 5] >> (v & 31)) & 1u; };
  int na = 0, nb = 0;
  for (int i = b0; i < b1; ++i) na += !stamped(lru[i]);
  for (int v = b0; v < b1; ++v) nb += stamped(v);
  int A, Bt;
  int ab = ublock_excl_scan(na, warp_sums, A);
  int bb = ublock_excl_scan(nb, warp_sums, Bt);
  for (int i = b0; i < b1; ++i) {
    const int v = lru[i];
    if (!stamped(v)) nxt[ab++] = v;
  }
  for (int v = b0; v < b1; ++v)
    if (stamped(v)) nxt[A + bb++] = v;
  __syncthreads();  // the new order is complete
  for (int i = tid; i < B; i += bs) lru[i] = nxt[i];
}

template <int VEC>
__global__ void __launch_bounds__(kGatherWarps * 32)
k_gather(const DevCtx c, const int32_t *__restrict__ topk, const int32_t *__restrict__ loc,
         int shared, int tick, int early) {
  constexpr int kGatherVec = GatherShape<VEC>::kGatherVec;
  constexpr int kGatherBatch = GatherShape<VEC>::kGatherBatch;
  __shared__ int warp_sums[32];
  // The per-query attention pass attends the rows already on the GPU
  // before it waits for this gather, so it is released early (`early`); the
  // union passes wait for every gathered row first, and launched early their
  // CTAs would only hold SMs, and their shared memory, that another request
  // group's kernels can use meanwhile.
  pdl_wait();
  if (early) pdl_trigger();
  const int r = blockIdx.y;
  const int Kr = c.Kr[r];
  if (Kr == 0) return;
  // CTA 0 of the request writes the cache state; with more than one CTA per
  // request it leaves the fetching to the others, so no fetch waits for it
  if (blockIdx.x == 0) {
    hot_update(c, r, tick, warp_sums);
    if (gridDim.x > 1) return;
  }
  const int fetchers = gridDim.x > 1 ? gridDim.x - 1 : 1;
  const int lane = threadIdx.x & 31;
  const int gw = (gridDim.x > 1 ? blockIdx.x - 1 : 0) * kGatherWarps + (threadIdx.x >> 5);
  const int nwt = fetchers * kGatherWarps;
  const int KK = c.Kmax * c.k;
  const int nv = (c.row * 2) >> 4;
  const uint16_t *host = c.host[r];
  const int64_t n = c.n[r];
  const int count = shared ? c.counts[r * 4 + 1] : Kr * c.k;
  const int P = c.counts[r * 4 + 2];
  for (int base = gw; base < count; base += kGatherBatch * nwt) {
    uint4 buf[kGatherBatch][kGatherVec];
    int32_t srow[kGatherBatch], slot[kGatherBatch];
#pragma unroll
    for (int b = 0; b < kGatherBatch; ++b) {
      const int e = base + b * nwt;
      srow[b] = -1;
      slot[b] = -1;
      if (e < count) {
        if (shared) {
          srow[b] = c.miss[(size_t)r * KK + e];
          if (e < P) slot[b] = c.promo_dst[(size_t)r * c.B + e];
        } else {
          const int32_t l = loc[(size_t)r * KK + e];
          if (l >= 0 && loc_tier(l) == DHS_LOC_STAGE) {
            srow[b] = topk[(size_t)r * KK + e];
            slot[b] = c.inst[(size_t)r * KK + e];
          }
        }
        if (slot[b] >= c.B) {
          record_error(c.err, DC_CAPACITY, K_GATHER);
          slot[b] = -1;
        }
        if (srow[b] >= n) {
          record_error(c.err, DC_ROW_RANGE, K_GATHER);
          srow[b] = -1;
        }
      }
      if (srow[b] >= 0) {
        const uint4 *src = reinterpret_cast<const uint4 *>(host + (int64_t)srow[b] * c.row);
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
      uint4 *d = reinterpret_cast<uint4 *>(c.stage + ((size_t)r * KK + base + b * nwt) * c.row);
#pragma unroll
      for (int i = 0; i < kGatherVec; ++i) {
        const int v = lane + 32 * i;
        if (v < nv) d[v] = buf[b][i];
      }
      if (slot[b] >= 0) {
        uint4 *h = reinterpret_cast<uint4 *>(c.hot_data + ((size_t)r * c.B + slot[b]) * c.row);
#pragma unroll
        for (int i = 0; i < kGatherVec; ++i) {
          const int v = lane + 32 * i;
          if (v < nv) h[v] = buf[b][i];
        }
      }
    }
  }
}

cudaError_t launch_resolve(const DevCtx &c, const int32_t *topk, int32_t *loc_out, int shared,
                           int gather, int tick, cudaStream_t s, Timer *tm) {
  static size_t granted = 0;
  cudaError_t e = ensure_smem(k_union_probe, union_smem_bytes(c), granted);
  if (e != cudaSuccess) return e;
  if (tm) tm->begin(K_UNION_PROBE, s);
  e = launch_pdl(k_union_probe, dim3(c.N * kUnionCluster), dim3(kUnionThreads),
                 union_smem_bytes(c), s, c, topk, loc_out, shared, tick);
  if (tm) tm->end(K_UNION_PROBE, s);
  if (e != cudaSuccess || !gather) return e;
  return launch_gather(c, topk, loc_out, shared, tick, s, tm, gather == 2);
}

cudaError_t launch_gather(const DevCtx &c, const int32_t *topk, int32_t *loc_out, int shared,
                          int tick, cudaStream_t s, Timer *tm, bool early) {
  cudaError_t e = cudaSuccess;
  const int vec = (c.row * 2 + 511) / 512;
  if (vec > kGatherMaxVec) return cudaErrorInvalidValue;
  void (*kern)(const DevCtx, const int32_t *, const int32_t *, int, int, int) =
      vec == 1 ? k_gather<1> : vec == 2 ? k_gather<2> : vec == 3 ? k_gather<3> : k_gather<4>;
  static bool carved[kGatherMaxVec + 1] = {};
  if (!carved[vec]) {
    same_carveout(kern);
    carved[vec] = true;
  }
  // One CTA per SM, one resident wave over the whole device: 8 warps with
  // 4-8 rows in flight each saturate the host link (far more than its
  // bandwidth-delay product), and with no shared memory and a quarter of the
  // registers a CTA leaves room for other kernels (another request group's
  // indexer) on its SM.
  int blocks_per_req = (c.sms + c.N - 1) / c.N;
  if (blocks_per_req < 1) blocks_per_req = 1;
  dim3 grid(blocks_per_req, c.N);
  if (tm) tm->begin(K_GATHER, s);
  // An ordinary launch: its CTAs are placed once the union/probe has left the
  // SMs, one per SM; placed early they would crowd onto the SMs the
  // union/probe leaves free and keep attention CTAs off them.
  e = launch_prio(kern, grid, dim3(kGatherWarps * 32), 0, s, c, topk, loc_out, shared, tick,
                  early ? 1 : 0);
  if (tm) tm->end(K_GATHER, s);
  return e;
}

}  // namespace dhs
