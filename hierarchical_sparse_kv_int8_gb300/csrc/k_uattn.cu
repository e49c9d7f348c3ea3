// Step 5 for shared retrieval: the attention of all K_r queries of a request
// in one pass over the union of their selections.
//
// "Adaptive DHiSparse", eq. (6) and Fig. 3 callout 2: each distinct row of the
// union U_r is fetched once per round, whichever queries selected it; eq. (1),
// (5): query j attends over its own selection S_{r,j} and the block rows
// n_r .. n_r + j.  Softmax attention is a sum over the attended rows, so
// visiting U_r once with, per row, the set of queries that selected it gives
// each query exactly its own rows -- and each distinct row is read from HBM
// once per round instead of once per query that selected it.
//
// GB300 design.  C thread-block clusters of kUCluster CTAs per (request, kv
// head) walk U_r in ascending row order, followed by the K_r block rows; the
// walk is cut into C x kUCluster contiguous parts.  Rows are copied into
// shared memory with 16-byte cp.async from wherever the union/probe located
// them (hot cache, optional pool, draft ring, staging) or from the caller's
// block buffer; each block row is also written to its draft-ring slot
// (eq. (9)-(10)) from shared memory.
//
// The M side of the bf16 mma.sync m16n8k16 products is every (query, head)
// pair of the kv head's group, K_max x G rows padded to 16; S = Q K^T over 16
// rows at a time, a score is kept only if its query selected the row (a bit of
// the row's query mask; block row i is seen by queries j >= i), online softmax
// in log2 units, O += P V.  The query tile sits in shared memory and is read
// with ldmatrix at every k-step, which keeps the registers of a 128-dim warp
// within the budget of two CTAs per SM.
//   - 128-dim heads: a warp owns one 16-row M-tile.
//   - MLA latent rows (576-dim keys, 512-dim values): four warps share each
//     M-tile, one quarter of the key and value dims each (partial scores
//     summed in shared memory).
// The warps that cover all M-tiles form a group; the CTA's groups walk
// alternate 16-row tiles, each group with its own ring of stages whose copies
// are tracked by mbarriers (every thread of the group ties its cp.async
// operations to the stage's barrier; the wait is bounded and records a device
// error if it runs out).  Groups synchronise only among their own warps
// (named barriers).  Partials are merged in three levels: the groups of a
// CTA in shared memory, the CTAs of a cluster through distributed shared
// memory (each CTA finishing every kUCluster-th (query, head) row), and, with
// C > 1, the clusters of an item through global memory by the cluster that
// takes the item's last ticket.
#include "dhs_internal.cuh"
#include "ptx_util.cuh"

#include <cooperative_groups.h>
#include <math_constants.h>

namespace dhs {

constexpr int kUCluster = 8;
constexpr int kUMaxRowsOwn = 16;  // (query, head) rows one CTA finishes: ceil(128 / 8)
constexpr int kUMaxGroups = 8;
constexpr int kUMaxStages = 32;
constexpr int kUMaxClusters = 8;  // clusters per (request, kv head)
constexpr int kUSpinLimit = 1 << 20;  // bounded wait for a stage's copies
constexpr int kUMinStages = 4;
constexpr size_t kSmemPerSm = 228 * 1024;        // shared memory of one SM
constexpr size_t kSmemReservedPerCta = 1024;     // taken by the system per resident CTA
constexpr size_t kStaticSmemMargin = 512;        // the kernel's static shared memory

template <int DQK, int DV>
struct UShape {
  static constexpr bool kMla = DQK > 256;
  static constexpr int NW = kMla ? 4 : 1;            // warps sharing one M-tile's dims
  static constexpr int KW = DQK / NW;                // key dims per warp
  static constexpr int VW = DV / NW;                 // value dims per warp
  static constexpr int KS = KW / 16;                 // k-steps per warp
  static constexpr int VT = VW / 8;                  // output n-tiles per warp
  static constexpr int RE = kMla ? DQK : DQK + DV;   // staged elements per row
  static constexpr int VOFF = kMla ? 0 : DQK;        // values within a staged row
  static constexpr int NCH = RE * 2 / 16;            // 16-byte chunks per staged row
  static constexpr int KCH = DQK * 2 / 16;           // chunks of the key part
  static constexpr int kWarpsTarget = kMla ? 16 : 4;
  static constexpr int kMaxThreads = kMla ? 512 : 256;  // up to 8 M-tiles of 128-dim heads
  // CTAs per SM aimed at: three for 128-dim heads, one for MLA rows
  static constexpr int kMaxCtasPerSm = kMla ? 1 : 3;
  static constexpr int kMinCtas = kMla ? 1 : 2;  // registers sized for this many per SM
  static_assert(KW % 16 == 0 && VW % 16 == 0, "dims per warp must be multiples of 16");
};

// Launch plan, fixed per context.  A group is the MT x NW warps that share
// one 16-row tile; NG groups walk alternate tiles of the CTA's part, each with
// its own ring of STG stages.
struct UPlan {
  int G, M, MT, NG, GW, warps, STG, C, chunk_max, RO;
  int off_q, off_red, off_mbar, off_meta, off_wt;
  int smem;
};

template <int DQK, int DV>
static UPlan make_uplan(const DevCtx &c) {
  using SH = UShape<DQK, DV>;
  UPlan p{};
  p.G = c.Hq / c.Hkv;
  p.M = c.Kmax * p.G;
  p.MT = (p.M + 15) / 16;
  p.GW = p.MT * SH::NW;
  p.NG = p.GW < SH::kWarpsTarget ? SH::kWarpsTarget / p.GW : 1;
  if (p.NG > kUMaxGroups) p.NG = kUMaxGroups;
  p.warps = p.GW * p.NG;
  // clusters per item: about two CTAs per SM over all items
  const int items = c.N * c.Hkv;
  p.C = (2 * c.sms + kUCluster * items - 1) / (kUCluster * items);
  if (p.C < 1) p.C = 1;
  if (p.C > kUMaxClusters) p.C = kUMaxClusters;
  const int KK = c.Kmax * c.k;
  const int parts = kUCluster * p.C;
  p.chunk_max = ((KK + c.Kmax + parts - 1) / parts + 15) / 16 * 16;
  const int tiles_per_group = (p.chunk_max / 16 + p.NG - 1) / p.NG;
  auto al = [](size_t x) { return (x + 127) / 128 * 128; };
  const size_t stride = (size_t)SH::RE * 2 + 16;
  const size_t qbytes = (size_t)p.MT * 16 * (DQK * 2 + 16);
  const size_t red = SH::kMla ? (size_t)p.NG * 2 * p.MT * SH::NW * 32 * 8 * 4 : 0;
  // receive buffer of the cluster merge: every warp group of every CTA pushes
  // its (O, m, l) for the RO rows each CTA finishes
  p.RO = (p.M + kUCluster - 1) / kUCluster;
  const size_t part = (size_t)kUCluster * p.NG * p.RO * (DV + 2) * 4;
  const size_t wt = ((size_t)kUMaxRowsOwn * kUCluster * kUMaxGroups + 2 * kUMaxRowsOwn) * 4;
  // enough stages for all of a group's tiles, as far as shared memory allows:
  // the most CTAs per SM that still leave each group kUMinStages stages (or
  // all its tiles), then the most stages at that residency
  int stg0 = tiles_per_group + 1;
  if (stg0 > kUMaxStages) stg0 = kUMaxStages;
  if (stg0 < 2) stg0 = 2;
  const int stg_min = stg0 < kUMinStages ? stg0 : kUMinStages;
  auto layout = [&](int stg) {
    p.STG = stg;
    const size_t stages = (size_t)p.NG * p.STG * 16 * stride;
    p.off_q = (int)al(stages);
    p.off_red = (int)al(p.off_q + qbytes);
    const size_t main_end = al(p.off_red + red);
    p.off_mbar = (int)al(main_end > part ? main_end : part);  // the merge reuses the stages
    p.off_meta = (int)al(p.off_mbar + (size_t)p.NG * p.STG * 8);
    p.off_wt = (int)al(p.off_meta + (size_t)p.chunk_max * 16);
    p.smem = (int)(p.off_wt + wt);
    return (size_t)p.smem;
  };
  for (int per_sm = SH::kMaxCtasPerSm; per_sm >= 1; --per_sm) {
    const size_t budget =
        per_sm == 1 ? kMaxDynSmem : kSmemPerSm / per_sm - kSmemReservedPerCta - kStaticSmemMargin;
    if (layout(stg_min) > budget) continue;
    for (int stg = stg0; stg > stg_min; --stg)
      if (layout(stg) <= budget) return p;
    layout(stg_min);
    return p;
  }
  layout(2);
  return p;
}

// Element offset, within a stored row, of 16-byte chunk ch of the staged row
// of kv head kvh (keys of every head first, then values; MLA: one latent).
template <int DQK, int DV>
__device__ __forceinline__ int useg(int ch, int kvh, int Hkv) {
  using SH = UShape<DQK, DV>;
  if constexpr (SH::kMla) {
    return ch * 8;
  } else {
    return ch < SH::KCH ? kvh * DQK + ch * 8 : Hkv * DQK + kvh * DV + (ch - SH::KCH) * 8;
  }
}

template <int DQK, int DV>
__global__ void __cluster_dims__(kUCluster, 1, 1)
    __launch_bounds__(UShape<DQK, DV>::kMaxThreads, UShape<DQK, DV>::kMinCtas)
k_uattn(const DevCtx c, const uint16_t *__restrict__ q, const uint16_t *__restrict__ block,
        uint16_t *__restrict__ out, float *__restrict__ lse, const UPlan pl) {
  using SH = UShape<DQK, DV>;
  constexpr int NW = SH::NW, KS = SH::KS, VT = SH::VT, NCH = SH::NCH;
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  extern __shared__ __align__(128) unsigned char smem[];
  const int crank = (int)cl.block_rank();
  const int item = blockIdx.y / pl.C, cidx = blockIdx.y - item * pl.C;
  const int r = item / c.Hkv, kvh = item - r * c.Hkv;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, nthr = blockDim.x;
  const int GW = pl.GW, GT = GW * 32, STG = pl.STG;
  const int grp = w / GW, wig = w - grp * GW;  // group, warp within the group
  const int mt = wig / NW, wi = wig - mt * NW;  // M-tile, dims quarter (MLA)
  uint64_t *mbar_all = reinterpret_cast<uint64_t *>(smem + pl.off_mbar);
  uint64_t *mbar = mbar_all + grp * STG;
  for (int i = tid; i < pl.NG * STG; i += nthr) mbar_init(&mbar_all[i], (uint32_t)GT);
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  __syncthreads();
  // K_r (scoring), the union entries and U (union/probe) were written two or
  // more launches back: complete once this launch has started.  Rows in the
  // hot cache, optional pool and draft ring are state of earlier rounds (the
  // gather that precedes this launch writes only staging rows and victim hot
  // slots, which no location of this round names).  All of these are read
  // before the wait on the preceding launch; staging rows, queries and block
  // rows after it.
  const int Kr = c.Kr[r];
  if (Kr == 0) {
    pdl_wait();
    return;  // the whole cluster leaves together
  }

  const int g = lane >> 2, t4 = lane & 3;
  const int G = pl.G, M = pl.M, MT16 = pl.MT * 16;
  const int KK = c.Kmax * c.k;
  const int U = c.counts[r * 4 + 0];
  const int T = U + Kr;  // union rows, then block rows
  const int parts = kUCluster * pl.C;
  const int chunk = ((T + parts - 1) / parts + 15) / 16 * 16;
  const int cb = min(T, (cidx * kUCluster + crank) * chunk), ce = min(T, cb + chunk);
  const int stride = SH::RE * 2 + 16;  // 16 bytes of padding: ldmatrix rows in distinct banks
  const int64_t n = c.n[r];
  const uint16_t *brow = block + (size_t)r * c.Kmax * c.row;
  const uint32_t all_q = (1u << Kr) - 1u;
  int4 *meta = reinterpret_cast<int4 *>(smem + pl.off_meta);

  // union entries of this CTA's rows: row, location, query mask
  {
    const int4 *uent = c.uent + (size_t)r * KK;
    const int cu = max(0, min(ce, U) - cb);
    for (int i = tid; i < cu; i += nthr) cp_async_16(&meta[i], &uent[cb + i]);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
  }

  // source of row e of the walk (nullptr: nothing to read); late: the row is
  // written by the preceding launch (staging) or by the caller (block rows)
  auto row_src = [&](int e, bool &late) -> const uint16_t * {
    late = false;
    if (e >= ce) return nullptr;
    if (e >= U) {
      late = true;
      return brow + (size_t)(e - U) * c.row;
    }
    const int32_t l = meta[e - cb].y;
    late = loc_tier(l) == DHS_LOC_STAGE;
    const uint16_t *p = loc_row(c, r, l);
    if (p == nullptr) record_error(c.err, DC_LOC_RANGE, K_ATTN_UNION);
    return p;
  };
  // query mask of row e of the walk
  auto row_mask = [&](int e) -> uint32_t {
    if (e >= ce) return 0u;
    if (e >= U) return all_q & ~((1u << (e - U)) - 1u);
    return (uint32_t)meta[e - cb].z;
  };

  // query tile in shared memory (A operand, read by ldmatrix): row m of the M
  // side is query m / G, head m % G
  const int mrow0 = mt * 16 + g, mrow1 = mrow0 + 8;
  const int j0 = mrow0 / G, j1 = mrow1 / G;
  uint16_t *qs = reinterpret_cast<uint16_t *>(smem + pl.off_q);
  constexpr int QSTR = DQK + 8;  // elements per query row in shared memory
  auto load_q = [&]() {
    for (int idx = tid; idx < MT16 * (DQK / 8); idx += nthr) {
      const int m = idx / (DQK / 8), ch = idx - m * (DQK / 8);
      const int j = m / G;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (m < M && j < Kr)
        v = *reinterpret_cast<const uint4 *>(
            q + (((size_t)r * c.Kmax + j) * c.Hq + (size_t)kvh * G + (m - j * G)) * DQK + ch * 8);
      *reinterpret_cast<uint4 *>(qs + (size_t)m * QSTR + ch * 8) = v;
    }
    __syncthreads();
  };

  // this group's tiles of the CTA's part: grp, grp + NG, ...
  const int nt_all = (ce - cb + 15) / 16;
  const int ntg = nt_all > grp ? (nt_all - grp + pl.NG - 1) / pl.NG : 0;
  unsigned char *gbuf = smem + (size_t)grp * STG * 16 * stride;
  // Copy one tile into its stage: lanes 0..15 of every warp of the group
  // decode the tile's 16 row addresses, each warp then copies its rows chunk
  // by chunk with the address broadcast by shuffle.  The early pass copies the
  // rows that may be read before the wait on the preceding launch, the late
  // pass the others; after the late pass every thread of the group ties its
  // copies to the stage's barrier.
  auto issue_pass = [&](int it, bool late_pass) {
    if (it >= ntg) return;
    const int tile = grp + it * pl.NG;
    unsigned char *sb = gbuf + (size_t)(it % STG) * 16 * stride;
    bool late;
    const uint16_t *mysrc = row_src(cb + tile * 16 + (lane & 15), late);
    const unsigned late_rows = __ballot_sync(0xffffffffu, late) & 0xFFFFu;
    for (int rr = wig; rr < 16; rr += GW) {
      if ((((late_rows >> rr) & 1u) != 0) != late_pass) continue;
      const uint16_t *src = reinterpret_cast<const uint16_t *>(
          __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(mysrc), rr));
      for (int ch = lane; ch < NCH; ch += 32)
        cp_async_16_zfill(sb + (size_t)rr * stride + ch * 16,
                          src ? (const void *)(src + useg<DQK, DV>(ch, kvh, c.Hkv))
                              : (const void *)c.ring,
                          src ? 16 : 0);
    }
    if (late_pass) cp_async_arrive_noinc(&mbar[it % STG]);
  };
  // both passes at once (inside the walk, after the wait): the tile's row
  // addresses are decoded once
  auto issue = [&](int it) {
    if (it >= ntg) return;
    const int tile = grp + it * pl.NG;
    unsigned char *sb = gbuf + (size_t)(it % STG) * 16 * stride;
    bool late;
    const uint16_t *mysrc = row_src(cb + tile * 16 + (lane & 15), late);
    for (int rr = wig; rr < 16; rr += GW) {
      const uint16_t *src = reinterpret_cast<const uint16_t *>(
          __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(mysrc), rr));
      for (int ch = lane; ch < NCH; ch += 32)
        cp_async_16_zfill(sb + (size_t)rr * stride + ch * 16,
                          src ? (const void *)(src + useg<DQK, DV>(ch, kvh, c.Hkv))
                              : (const void *)c.ring,
                          src ? 16 : 0);
    }
    cp_async_arrive_noinc(&mbar[it % STG]);
  };
  auto wait_stage = [&](int it) {
    const int slot = it % STG;
    const uint32_t parity = (uint32_t)((it / STG) & 1);
    int spins = 0;
    while (!mbar_try_wait(&mbar[slot], parity)) {
      if (++spins > kUSpinLimit) {
        record_error(c.err, DC_TIMEOUT, K_ATTN_UNION);
        break;
      }
    }
  };
  // block rows leave through the CTA that reads them: into the draft ring
  auto write_back = [&](int it) {
    const int tile = grp + it * pl.NG;
    const int e0 = cb + tile * 16;
    if (e0 + 16 <= U || e0 >= ce) return;  // no block row in this tile
    const unsigned char *sb = gbuf + (size_t)(it % STG) * 16 * stride;
    for (int rr = wig; rr < 16; rr += GW) {
      const int e = e0 + rr;
      if (e < U || e >= ce) continue;
      uint16_t *d0 = c.ring + ((size_t)r * c.Rd + (n + (e - U)) % c.Rd) * c.row;
      for (int ch = lane; ch < NCH; ch += 32)
        *reinterpret_cast<uint4 *>(d0 + useg<DQK, DV>(ch, kvh, c.Hkv)) =
            *reinterpret_cast<const uint4 *>(sb + (size_t)rr * stride + ch * 16);
    }
  };

  float o[VT][4];
#pragma unroll
  for (int i = 0; i < VT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
  float *red = reinterpret_cast<float *>(smem + pl.off_red) +
               (size_t)grp * 2 * pl.MT * NW * 32 * 8;

  for (int s = 0; s < STG - 1; ++s) issue_pass(s, false);
  pdl_wait();  // the gather's staging rows, and everything the caller wrote
  pdl_trigger();
  for (int s = 0; s < STG - 1; ++s) issue_pass(s, true);
  load_q();
  for (int it = 0; it < ntg; ++it) {
    issue(it + STG - 1);  // into the stage freed at the end of the previous tile
    wait_stage(it);
    write_back(it);
    const int tile = grp + it * pl.NG;
    const unsigned char *sb = gbuf + (size_t)(it % STG) * 16 * stride;
    const int ebase = cb + tile * 16;
    uint32_t cm[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int b = 0; b < 2; ++b) cm[nt][b] = row_mask(ebase + nt * 8 + 2 * t4 + b);

    // S = Q K^T over this warp's key dims: two n-tiles of 8 rows
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int mi = lane >> 3, ri = lane & 7;
      const unsigned char *rowp = sb + (size_t)((mi >> 1) * 8 + ri) * stride;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int col = wi * SH::KW + ks * 16 + (mi & 1) * 8;
        uint32_t a[4];
        ldmatrix_x4(a[0], a[1], a[2], a[3],
                    qs + (size_t)(mt * 16 + (lane & 15)) * QSTR + wi * SH::KW + ks * 16 +
                        (lane >> 4) * 8);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(b0, b1, b2, b3, rowp + col * 2);
        mma_bf16_16816(s[0], a, b0, b1);
        mma_bf16_16816(s[1], a, b2, b3);
      }
    }
    if constexpr (NW > 1) {  // sum the key-dim partials of the M-tile's warps, same order everywhere
      float *my = red + ((size_t)(((it & 1) * pl.MT + mt) * NW + wi) * 32 + lane) * 8;
#pragma unroll
      for (int i = 0; i < 8; ++i) my[i] = s[i >> 2][i & 3];
      named_sync(1 + grp, GT);
#pragma unroll
      for (int i = 0; i < 8; ++i) s[i >> 2][i & 3] = 0.f;
      for (int ww = 0; ww < NW; ++ww) {
        const float *src = red + ((size_t)(((it & 1) * pl.MT + mt) * NW + ww) * 32 + lane) * 8;
#pragma unroll
        for (int i = 0; i < 8; ++i) s[i >> 2][i & 3] += src[i];
      }
    }
    // log2-domain logits; a score counts only if its query selected the row
    float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int jj = i < 2 ? j0 : j1;
        const bool sel = (cm[nt][i & 1] >> jj) & 1u;
        const float x = sel ? s[nt][i] * c.scale_log2 : -CUDART_INF_F;
        s[nt][i] = x;
        if (i < 2) mx0 = fmaxf(mx0, x); else mx1 = fmaxf(mx1, x);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float ref0 = mn0 == -CUDART_INF_F ? 0.f : mn0;
    const float ref1 = mn1 == -CUDART_INF_F ? 0.f : mn1;
    const float al0 = exp2f(m0 - ref0), al1 = exp2f(m1 - ref1);
    m0 = mn0;
    m1 = mn1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      s[nt][0] = exp2f(s[nt][0] - ref0);
      s[nt][1] = exp2f(s[nt][1] - ref0);
      s[nt][2] = exp2f(s[nt][2] - ref1);
      s[nt][3] = exp2f(s[nt][3] - ref1);
      ps0 += s[nt][0] + s[nt][1];
      ps1 += s[nt][2] + s[nt][3];
    }
    l0 = l0 * al0 + ps0;
    l1 = l1 * al1 + ps1;
    if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {  // a running max moved
#pragma unroll
      for (int i = 0; i < VT; ++i) {
        o[i][0] *= al0;
        o[i][1] *= al0;
        o[i][2] *= al1;
        o[i][3] *= al1;
      }
    }
    uint32_t pa[4];
    pa[0] = pack_bf16(s[0][0], s[0][1]);
    pa[1] = pack_bf16(s[0][2], s[0][3]);
    pa[2] = pack_bf16(s[1][0], s[1][1]);
    pa[3] = pack_bf16(s[1][2], s[1][3]);
    {
      const int mi = lane >> 3, ri = lane & 7;
      const unsigned char *rowp = sb + (size_t)((mi & 1) * 8 + ri) * stride;
#pragma unroll
      for (int vt = 0; vt < VT / 2; ++vt) {
        const int dim = SH::VOFF + wi * SH::VW + vt * 16 + (mi >> 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(b0, b1, b2, b3, rowp + dim * 2);
        mma_bf16_16816(o[2 * vt], pa, b0, b1);
        mma_bf16_16816(o[2 * vt + 1], pa, b2, b3);
      }
    }
    named_sync(1 + grp, GT);  // the group's stage is refilled by a later issue
  }
  cp_async_wait_all();
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  // ---- cluster merge.  CTA q finishes the (query, head) rows m = q (mod
  //      kUCluster); every warp group of every CTA pushes its (O, m, l) for a
  //      row into the finishing CTA's receive buffer with distributed
  //      shared-memory stores, which overwrites the stages.
  const int RO = pl.RO, NP = kUCluster * pl.NG;  // partials per row
  float *recv = reinterpret_cast<float *>(smem);           // [NP][RO][DV]
  float *recv_ml = recv + (size_t)NP * RO * DV;            // [NP][RO][2]
  cl.sync();  // (1) every CTA's walk is over
  {
    const int pi = crank * pl.NG + grp;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int mrow = h ? mrow1 : mrow0;
      if (mrow >= M) continue;
      const int owner = mrow % kUCluster, lr = mrow / kUCluster;
      float *dst = cl.map_shared_rank(recv, owner) + ((size_t)pi * RO + lr) * DV;
#pragma unroll
      for (int i = 0; i < VT; ++i) {
        const int dim = wi * SH::VW + i * 8 + 2 * t4;
        *reinterpret_cast<float2 *>(dst + dim) = make_float2(o[i][2 * h], o[i][2 * h + 1]);
      }
      if (wi == 0 && t4 == 0)
        *reinterpret_cast<float2 *>(cl.map_shared_rank(recv_ml, owner) + ((size_t)pi * RO + lr) * 2) =
            make_float2(h ? m1 : m0, h ? l1 : l0);
    }
  }
  cl.sync();  // (2) every push has landed

  // ---- reduce the NP partials of each row this CTA finishes: normalised
  //      outputs when the item has one cluster, else the cluster's
  //      unnormalised partial (O, m, l)
  const int rows_own = crank < M ? (M - crank + kUCluster - 1) / kUCluster : 0;
  float *Wt = reinterpret_cast<float *>(smem + pl.off_wt);  // [rows_own][NP] weights
  float *Rm = Wt + kUMaxRowsOwn * kUCluster * kUMaxGroups;   // [rows_own] max, sum
  float *Rl = Rm + kUMaxRowsOwn;
  const float ln2 = 0.69314718055994531f;
  const bool single = pl.C == 1;
  for (int lr = tid; lr < rows_own; lr += nthr) {
    const int mrow = crank + lr * kUCluster;
    float Mx = -CUDART_INF_F;
    for (int pp = 0; pp < NP; ++pp) Mx = fmaxf(Mx, recv_ml[((size_t)pp * RO + lr) * 2]);
    const float ref = Mx == -CUDART_INF_F ? 0.f : Mx;
    float L = 0.f;
    for (int pp = 0; pp < NP; ++pp) {
      const float wgt = exp2f(recv_ml[((size_t)pp * RO + lr) * 2] - ref);
      Wt[lr * NP + pp] = wgt;
      L += wgt * recv_ml[((size_t)pp * RO + lr) * 2 + 1];
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    if (single)
      for (int pp = 0; pp < NP; ++pp) Wt[lr * NP + pp] *= inv;
    Rm[lr] = Mx;
    Rl[lr] = L;
    const int j = mrow / G;
    if (single && lse && j < Kr)
      lse[((size_t)r * c.Kmax + j) * c.Hq + (size_t)kvh * G + (mrow - j * G)] =
          L > 0.f ? (Mx + log2f(L)) * ln2 : -CUDART_INF_F;
  }
  __syncthreads();
  const size_t nitems = (size_t)c.N * c.Hkv;
  float *cpo = c.u_part + (size_t)(item * pl.C + cidx) * M * DV;                 // [M][DV]
  float *cpml = c.u_part + nitems * pl.C * M * DV + (size_t)(item * pl.C + cidx) * M * 2;
  for (int idx = tid; idx < rows_own * (DV / 2); idx += nthr) {
    const int lr = idx / (DV / 2), d = (idx - lr * (DV / 2)) * 2;
    const int mrow = crank + lr * kUCluster;
    const int j = mrow / G;
    if (j >= Kr) continue;
    float a = 0.f, b = 0.f;
    for (int pp = 0; pp < NP; ++pp) {
      const float wgt = Wt[lr * NP + pp];
      const float2 v = *reinterpret_cast<const float2 *>(recv + ((size_t)pp * RO + lr) * DV + d);
      a += wgt * v.x;
      b += wgt * v.y;
    }
    if (single) {
      *reinterpret_cast<uint32_t *>(
          out + (((size_t)r * c.Kmax + j) * c.Hq + (size_t)kvh * G + (mrow - j * G)) * DV + d) =
          pack_bf16(a, b);
    } else {
      *reinterpret_cast<float2 *>(cpo + (size_t)mrow * DV + d) = make_float2(a, b);
      if (d == 0) *reinterpret_cast<float2 *>(cpml + (size_t)mrow * 2) = make_float2(Rm[lr], Rl[lr]);
    }
  }
  if (single) return;

  // ---- the cluster that finishes an item last merges the item's C partials
  __shared__ int sh_last;
  __threadfence();
  cl.sync();  // every CTA of the cluster has written and fenced its rows
  if (crank == 0 && tid == 0) sh_last = atomicAdd(&c.u_ticket[item], 1) == pl.C - 1;
  cl.sync();
  const int last = *cl.map_shared_rank(&sh_last, 0);
  if (last) {
    __threadfence();
    const float *ipo = c.u_part + (size_t)item * pl.C * M * DV;
    const float *ipml = c.u_part + nitems * pl.C * M * DV + (size_t)item * pl.C * M * 2;
    for (int idx = tid; idx < rows_own * (DV / 2); idx += nthr) {
      const int lr = idx / (DV / 2), d = (idx - lr * (DV / 2)) * 2;
      const int mrow = crank + lr * kUCluster;
      const int j = mrow / G;
      if (j >= Kr) continue;
      float mc[kUMaxClusters], lc[kUMaxClusters];
      float Mx = -CUDART_INF_F;
#pragma unroll
      for (int cc = 0; cc < kUMaxClusters; ++cc) {
        if (cc < pl.C) {
          const float2 ml =
              __ldcg(reinterpret_cast<const float2 *>(ipml + ((size_t)cc * M + mrow) * 2));
          mc[cc] = ml.x;
          lc[cc] = ml.y;
          Mx = fmaxf(Mx, ml.x);
        }
      }
      const float ref = Mx == -CUDART_INF_F ? 0.f : Mx;
      float L = 0.f, a = 0.f, b = 0.f;
#pragma unroll
      for (int cc = 0; cc < kUMaxClusters; ++cc) {
        if (cc < pl.C) {
          const float wgt = exp2f(mc[cc] - ref);
          const float2 v =
              __ldcg(reinterpret_cast<const float2 *>(ipo + ((size_t)cc * M + mrow) * DV + d));
          L += wgt * lc[cc];
          a += wgt * v.x;
          b += wgt * v.y;
        }
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      const size_t o = ((size_t)r * c.Kmax + j) * c.Hq + (size_t)kvh * G + (mrow - j * G);
      *reinterpret_cast<uint32_t *>(out + o * DV + d) = pack_bf16(a * inv, b * inv);
      if (lse && d == 0) lse[o] = L > 0.f ? (Mx + log2f(L)) * ln2 : -CUDART_INF_F;
    }
    if (crank == 0 && tid == 0) c.u_ticket[item] = 0;  // ready for the next launch
  }
  cl.sync();  // rank 0's ticket flag has been read by every CTA
}

template <int DQK, int DV>
static cudaError_t launch_uattn_t(const DevCtx &c, const uint16_t *q, const uint16_t *block,
                                  uint16_t *out, float *lse, cudaStream_t s, Timer *tm) {
  const UPlan pl = make_uplan<DQK, DV>(c);
  static size_t granted = 0;
  cudaError_t e = ensure_smem(k_uattn<DQK, DV>, (size_t)pl.smem, granted);
  if (e != cudaSuccess) return e;
  if (tm) tm->begin(K_ATTN_UNION, s);
  e = launch_pdl(k_uattn<DQK, DV>, dim3(kUCluster, c.N * c.Hkv * pl.C), dim3(pl.warps * 32),
                 (size_t)pl.smem, s, c, q, block, out, lse, pl);
  if (tm) tm->end(K_ATTN_UNION, s);
  return e;
}

size_t uattn_partial_floats(const DevCtx &c) {
  UPlan pl;
  if (c.dqk == 128 && c.dv == 128) pl = make_uplan<128, 128>(c);
  else pl = make_uplan<576, 512>(c);
  return (size_t)c.N * c.Hkv * pl.C * pl.M * (c.dv + 2);
}

bool uattn_supported(const DevCtx &c) {
  UPlan pl;
  int max_threads;
  if (c.dqk == 128 && c.dv == 128 && c.layout == DHS_KV_SPLIT) {
    pl = make_uplan<128, 128>(c);
    max_threads = UShape<128, 128>::kMaxThreads;
  } else if (c.dqk == 576 && c.dv == 512 && c.layout == DHS_KV_LATENT) {
    pl = make_uplan<576, 512>(c);
    max_threads = UShape<576, 512>::kMaxThreads;
  } else {
    return false;
  }
  return pl.warps * 32 <= max_threads && pl.M <= kUMaxRowsOwn * kUCluster &&
         pl.STG >= 2 && (size_t)pl.smem <= kMaxDynSmem;
}

cudaError_t launch_uattn(const DevCtx &c, const uint16_t *q, const uint16_t *block,
                         uint16_t *out, float *lse, cudaStream_t s, Timer *tm) {
  return (c.dqk == 128 && c.dv == 128)
             ? launch_uattn_t<128, 128>(c, q, block, out, lse, s, tm)
             : launch_uattn_t<576, 512>(c, q, block, out, lse, s, tm);
}

}  // namespace dhs
