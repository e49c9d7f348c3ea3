// Step 5 of the verification round: sparse attention over located rows.
//
// "Adaptive DHiSparse", eq. (1) and (5): query j of request r attends over its
// own ordered selection S_{r,j}, read through the locations l_{r,j,i} of
// eq. (11)-(12), and over the block rows n_r .. n_r + j of the tail.
//
// Split-KV flash decoding.  One CTA of four warps handles one split (a range
// of the row list) of one (request, query, kv head) item.  Rows are gathered
// by location into shared memory with 16-byte cp.async, three stages in
// flight, each tracked by an mbarrier (rows of the context's pools arrive by
// bulk asynchronous copies of the TMA engine, the caller's block rows by
// cp.async).  The split's rows of the hot cache,
// optional pool and draft ring, and its block rows, are attended first, while
// the preceding gather may still be running; its staging rows follow once the
// gather has finished.  The query heads that share the kv head (padded to 16) form the M
// side of bf16 mma.sync m16n8k16 tensor-core products with fp32 accumulation:
// S = Q K^T over 16 rows at a time, online softmax in log2 units, O += P V.
//   - GQA rows (128-dim heads): the four warps are independent, each takes
//     every fourth 16-row tile of the split; their (m, l, O) are combined in
//     shared memory at the end.
//   - MLA latent rows (576-dim keys, 512-dim values): the four warps share
//     each tile, each owning a quarter of the key dims (partial S summed in
//     shared memory) and a quarter of the value dims.
// Splits of one item are merged by the CTA that finishes last (a per-item
// ticket taken with one atomic after the partial is written and fenced), so
// no separate merge launch and no device-side waiting are needed.  The first
// split of each (request, query) also writes that query's block row into the
// draft ring (eq. (9)-(10)), so no launch follows attention before commit.
#include "dhs_internal.cuh"
#include "ptx_util.cuh"

#include <cooperative_groups.h>
#include <math_constants.h>

namespace dhs {

constexpr int kAttnStages = 3;
constexpr int kTileRows = 16;
constexpr int kAttnThreads = 128;
constexpr int kAttnSpinLimit = 1 << 20;  // bounded wait for a stage's copies
// An item split exactly kAttnCluster ways (128-dim heads) runs its splits as
// one thread-block cluster and merges them through distributed shared memory.
constexpr int kAttnCluster = 8;

bool attn_shape_supported(int dqk, int dv, int layout) {
  if (layout == DHS_KV_SPLIT) return dqk == 128 && dv == 128;
  return dqk == 576 && dv == 512;
}

template <int DQK, int DV>
struct AttnShape {
  static constexpr int NW = (DQK > 256) ? 4 : 1;  // warps sharing one row tile
  static constexpr int SUB = 4 / NW;              // independent warp groups per CTA
  static constexpr int KW = DQK / NW;             // key dims per warp
  static constexpr int VW = DV / NW;              // value dims per warp
  static constexpr int KS = KW / 16;              // k-steps per warp
  static constexpr int VT = VW / 8;               // output n-tiles per warp
  static_assert(KW % 16 == 0 && VW % 16 == 0, "dims per warp must be multiples of 16");
};

static int attn_rows_per_tile_group(const DevCtx &c) { return c.dqk > 256 ? 16 : 64; }

// Splits per item, fixed at context creation: about two CTAs per SM over all
// items, at least one 16-row tile per warp group.
int attn_splits(const DevCtx &c, int active_queries) {
  (void)active_queries;
  const int rows = c.k + c.Kmax;
  const int gran = attn_rows_per_tile_group(c);
  const int target = c.sms * 2;
  const int items = c.N * c.Kmax * c.Hkv;
  int ns = (target + items - 1) / items;
  const int max_ns = (rows + gran - 1) / gran;
  if (ns > max_ns) ns = max_ns;
  if (ns < 1) ns = 1;
  // near kAttnCluster splits, take exactly that many: the cluster merge
  if (c.dqk == 128 && ns >= 6 && ns <= 12 && kAttnCluster <= max_ns) return kAttnCluster;
  int chunk = (rows + ns - 1) / ns;
  chunk = (chunk + gran - 1) / gran * gran;
  return (rows + chunk - 1) / chunk;
}

static int attn_chunk(const DevCtx &c, int n_split) {
  const int rows = c.k + c.Kmax;
  const int gran = attn_rows_per_tile_group(c);
  int chunk = (rows + n_split - 1) / n_split;
  return (chunk + gran - 1) / gran * gran;
}

size_t attn_partial_floats(const DevCtx &c, int n_split) {
  return (size_t)c.N * c.Kmax * c.Hq * n_split * c.dv;
}

template <int DQK, int DV>
static size_t attn_smem_bytes(int row_elems, int n_split) {
  using SH = AttnShape<DQK, DV>;
  const size_t stride = (size_t)row_elems * 2 + 16;
  const size_t stages = (size_t)SH::SUB * kAttnStages * kTileRows * stride;
  const size_t epilogue = ((size_t)SH::SUB * 16 * DV + 2 * SH::SUB * 16 + 48 * n_split) * 4;
  const size_t body = stages > epilogue ? stages : epilogue;
  return body + (size_t)SH::SUB * kAttnStages * kTileRows * 4 + 2 * SH::NW * 32 * 8 * 4 + 64;
}

// Locations of one split, prefetched once into shared memory, followed by the
// two row lists of the processing order (int16 positions within the split).
static size_t attn_loc_bytes(int chunk) { return ((size_t)chunk * 4 + 127) / 128 * 128; }
static size_t attn_ord_bytes(int chunk) { return ((size_t)chunk * 4 + 127) / 128 * 128; }

template <int DQK, int DV>
__global__ void __launch_bounds__(kAttnThreads)
k_attn(const DevCtx c, const uint16_t *__restrict__ q, const uint16_t *__restrict__ block,
       const int32_t *__restrict__ loc, uint16_t *__restrict__ out, float *__restrict__ lse,
       int n_split, int chunk, size_t body_bytes, size_t loc_off) {
  using SH = AttnShape<DQK, DV>;
  constexpr int NW = SH::NW, SUB = SH::SUB, KS = SH::KS, VT = SH::VT;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int sh_last;
  const int split = blockIdx.x, j = blockIdx.y;
  const int r = blockIdx.z / c.Hkv, kvh = blockIdx.z % c.Hkv;
  if (j >= c.Kr[r]) {
    pdl_wait();
    return;
  }
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int grp = w / NW, wi = w % NW;  // warp group and warp within it
  const int g = lane >> 2, t4 = lane & 3;
  const int G = c.Hq / c.Hkv;
  const int k = c.k;
  const int total = k + j + 1;
  // the split's rows are positions i of the row list e = split + i * n_split
  // (interleaved, so every split gets its share of each tier)
  const int nrows = total > split ? (total - split + n_split - 1) / n_split : 0;
  const int rowb = c.row * 2;
  const int stride = rowb + 16;  // 16 bytes of padding: ldmatrix rows fall in distinct banks
  const int nv = rowb >> 4;
  unsigned char *stage_base = smem + (size_t)grp * kAttnStages * kTileRows * stride;
  int *vflag_all = reinterpret_cast<int *>(smem + body_bytes);
  int *vflag = vflag_all + grp * kAttnStages * kTileRows;
  float *red = reinterpret_cast<float *>(vflag_all + SUB * kAttnStages * kTileRows);
  int32_t *lsm = reinterpret_cast<int32_t *>(smem + body_bytes + loc_off);
  const int koff = (c.layout == DHS_KV_LATENT) ? 0 : kvh * DQK;
  const int voff = (c.layout == DHS_KV_LATENT) ? 0 : c.Hkv * DQK + kvh * DV;
  const int32_t *lrow = loc + ((size_t)r * c.Kmax + j) * k;
  const uint16_t *brow = block + (size_t)r * c.Kmax * c.row;

  // locations of this split's selected rows (written two launches back, by
  // the union/probe), read once, coalesced, before the preceding launch ends
  for (int i = tid; i < nrows; i += kAttnThreads) {
    const int e = split + i * n_split;
    if (e < k) lsm[i] = lrow[e];
  }
  __syncthreads();  // the locations are in shared memory

  // eq. (9)-(10): block row j enters the draft ring at phi(r, n_r + j); the
  // live ring rows this round reads lie in [n_r - W, n_r) and R_d >= W + K,
  // so the write never lands on a row being read, and the preceding launch
  // (the gather) touches no ring row
  if (split == 0 && kvh == 0) {
    const int64_t n = c.n[r];
    const uint4 *src = reinterpret_cast<const uint4 *>(brow + (size_t)j * c.row);
    uint4 *dst = reinterpret_cast<uint4 *>(c.ring + ((size_t)r * c.Rd + (n + j) % c.Rd) * c.row);
    for (int v = tid; v < nv; v += kAttnThreads) dst[v] = src[v];
  }

  // Processing order of the split's rows.  Rows of the hot cache, optional
  // pool and draft ring are state of earlier rounds, and the caller's queries
  // and block rows are complete before the round's first kernel; all of them
  // are attended before the wait on the preceding launch (the gather, which
  // writes only staging rows and victim hot slots, none of them named by a
  // location of this round).  Staging rows follow after the wait.  An empty
  // location adds nothing and is dropped.  Only the order of the softmax sum
  // changes.
  int16_t *ord_e = reinterpret_cast<int16_t *>(reinterpret_cast<unsigned char *>(lsm) +
                                               (((size_t)chunk * 4 + 127) & ~(size_t)127));
  int16_t *ord_l = ord_e + chunk;
  __shared__ int wcnt[2][kAttnThreads / 32];
  int n_early = 0, n_late = 0;
  for (int base = 0; base < nrows; base += kAttnThreads) {
    const int i = base + tid;
    bool early = false, late = false;
    if (i < nrows) {
      if (split + i * n_split >= k) {
        early = true;  // a block row
      } else {
        const int32_t l = lsm[i];
        if (l >= 0) {
          late = loc_tier(l) == DHS_LOC_STAGE;
          early = !late;
        }
      }
    }
    const unsigned be = __ballot_sync(0xffffffffu, early), bl = __ballot_sync(0xffffffffu, late);
    if (lane == 0) {
      wcnt[0][w] = __popc(be);
      wcnt[1][w] = __popc(bl);
    }
    __syncthreads();
    int pe = n_early, pl = n_late;
#pragma unroll
    for (int ww = 0; ww < kAttnThreads / 32; ++ww) {
      if (ww < w) {
        pe += wcnt[0][ww];
        pl += wcnt[1][ww];
      }
      n_early += wcnt[0][ww];
      n_late += wcnt[1][ww];
    }
    const unsigned lt = (1u << lane) - 1u;
    if (early) ord_e[pe + __popc(be & lt)] = (int16_t)i;
    if (late) ord_l[pl + __popc(bl & lt)] = (int16_t)i;
    __syncthreads();
  }

  // tiles of 16 listed rows, early tiles first; this group takes tiles grp,
  // grp + SUB, ...; the first n_pre of them are attended before the wait
  const int nE = (n_early + kTileRows - 1) / kTileRows;
  const int ntiles_all = nE + (n_late + kTileRows - 1) / kTileRows;
  const int ntiles = ntiles_all > grp ? (ntiles_all - grp + SUB - 1) / SUB : 0;
  const int n_pre = nE > grp ? (nE - grp + SUB - 1) / SUB : 0;
  const int gtid = wi * 32 + lane;  // thread index within the group
  __shared__ __align__(8) uint64_t mbar[SUB][kAttnStages];
  if (gtid == 0) {
    for (int s = 0; s < kAttnStages; ++s) mbar_init(&mbar[grp][s], NW * 32);
    fence_proxy_async_smem();  // the bulk copies see the initialised barriers
  }
  __syncthreads();
  // Copy one tile into its stage: lanes 0..15 of every warp decode one row's
  // source address (location tag, bounds check), the group's threads copy the
  // rows chunk by chunk with the address broadcast by shuffle, and then tie
  // their copies to the stage's barrier.
  auto issue = [&](int it) {
    const int tile = grp + it * SUB;
    const bool late_tile = tile >= nE;
    const int16_t *lst = late_tile ? ord_l : ord_e;
    const int i0 = (late_tile ? tile - nE : tile) * kTileRows;
    const int n_in = late_tile ? n_late : n_early;
    unsigned char *st = stage_base + (size_t)(it % kAttnStages) * kTileRows * stride;
    int *vf = vflag + (it % kAttnStages) * kTileRows;
    uint64_t *bar = &mbar[grp][it % kAttnStages];
    const uint16_t *mysrc = nullptr;
    bool pooled = false;  // a row of the context's pools (device memory)
    if (lane < kTileRows) {
      const int i = i0 + lane;
      if (i < n_in) {
        const int pos = lst[i], e = split + pos * n_split;
        if (e < k) {
          mysrc = loc_row(c, r, lsm[pos]);
          pooled = mysrc != nullptr;
          if (mysrc == nullptr && wi == 0) record_error(c.err, DC_LOC_RANGE, K_ATTN);
        } else {
          mysrc = brow + (size_t)(e - k) * c.row;
        }
      }
      if (wi == 0) vf[lane] = mysrc != nullptr;
    }
    // pool rows: one bulk asynchronous copy (TMA engine) per row, issued by
    // the group's first warp and counted in bytes on the stage's barrier
    const unsigned bulk_rows = __ballot_sync(0xffffffffu, pooled);
    if (wi == 0 && bulk_rows) {
      if (lane == 0) mbar_expect_tx(bar, (uint32_t)__popc(bulk_rows) * (uint32_t)rowb);
      __syncwarp();
      if (pooled) bulk_g2s(st + (size_t)lane * stride, mysrc, (uint32_t)rowb, bar);
    }
    // the caller's block rows (which may be page-locked host memory) and
    // empty rows (zero-filled) by 16-byte cp.async
#pragma unroll 4
    for (int rr = 0; rr < kTileRows; ++rr) {
      if ((bulk_rows >> rr) & 1u) continue;
      const uint16_t *src = reinterpret_cast<const uint16_t *>(
          __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(mysrc), rr));
      unsigned char *dst = st + (size_t)rr * stride;
      for (int v = gtid; v < nv; v += NW * 32)
        cp_async_16_zfill(dst + v * 16, src ? (const void *)(src + v * 8) : (const void *)c.ring,
                          src ? 16 : 0);
    }
    cp_async_arrive_noinc(bar);
  };
  auto wait_stage = [&](int it) {
    const uint32_t parity = (uint32_t)((it / kAttnStages) & 1);
    int spins = 0;
    while (!mbar_try_wait(&mbar[grp][it % kAttnStages], parity))
      if (++spins > kAttnSpinLimit) {
        record_error(c.err, DC_TIMEOUT, K_ATTN);
        break;
      }
  };
  int issued = 0;
  for (; issued < min(n_pre, kAttnStages - 1); ++issued) issue(issued);

  // query fragments: rows of the A operand are the query heads of this kv head
  uint32_t qa[KS][4];
  {
    const uint16_t *qb = q + (((size_t)r * c.Kmax + j) * c.Hq + (size_t)kvh * G) * DQK;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int col = wi * SH::KW + ks * 16 + 2 * t4;
      const uint32_t *r0 = reinterpret_cast<const uint32_t *>(qb + (size_t)g * DQK + col);
      const uint32_t *r1 = reinterpret_cast<const uint32_t *>(qb + (size_t)(g + 8) * DQK + col);
      qa[ks][0] = g < G ? r0[0] : 0u;
      qa[ks][1] = g + 8 < G ? r1[0] : 0u;
      qa[ks][2] = g < G ? r0[4] : 0u;
      qa[ks][3] = g + 8 < G ? r1[4] : 0u;
    }
  }

  auto group_sync = [&]() {
    if (NW == 1) __syncwarp(); else __syncthreads();
  };

  float o[VT][4];
#pragma unroll
  for (int i = 0; i < VT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;

  bool waited = false;
  for (int it = 0; it < ntiles; ++it) {
    if (it == n_pre) {  // the staging rows: after the gather
      pdl_wait();
      pdl_trigger();
      waited = true;
    }
    // keep kAttnStages - 1 tiles ahead: early tiles at any time, staging
    // tiles once the wait is over
    for (; issued < min(waited ? ntiles : n_pre, it + kAttnStages); ++issued) issue(issued);
    wait_stage(it);
    group_sync();  // the tile's row flags are visible to the group
    const unsigned char *st = stage_base + (size_t)(it % kAttnStages) * kTileRows * stride;
    const int *vf = vflag + (it % kAttnStages) * kTileRows;

    // S = Q K^T over this warp's key dims: two n-tiles of 8 rows
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int mi = lane >> 3, ri = lane & 7;
      const unsigned char *rowp = st + (size_t)((mi >> 1) * 8 + ri) * stride;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int col = koff + wi * SH::KW + ks * 16 + (mi & 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(b0, b1, b2, b3, rowp + col * 2);
        mma_bf16_16816(s[0], qa[ks], b0, b1);
        mma_bf16_16816(s[1], qa[ks], b2, b3);
      }
    }
    if (NW > 1) {  // sum the key-dim partials of the group's warps, same order everywhere
      float *my = red + ((size_t)((it & 1) * NW + wi) * 32 + lane) * 8;
#pragma unroll
      for (int i = 0; i < 8; ++i) my[i] = s[i >> 2][i & 3];
      __syncthreads();
#pragma unroll
      for (int i = 0; i < 8; ++i) s[i >> 2][i & 3] = 0.f;
      for (int ww = 0; ww < NW; ++ww) {
        const float *src = red + ((size_t)((it & 1) * NW + ww) * 32 + lane) * 8;
#pragma unroll
        for (int i = 0; i < 8; ++i) s[i >> 2][i & 3] += src[i];
      }
    }
    // log2-domain logits, invalid rows masked
    float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int col = nt * 8 + 2 * t4 + (i & 1);
        const float x = vf[col] ? s[nt][i] * c.scale_log2 : -CUDART_INF_F;
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
#pragma unroll
    for (int i = 0; i < VT; ++i) {
      o[i][0] *= al0;
      o[i][1] *= al0;
      o[i][2] *= al1;
      o[i][3] *= al1;
    }
    uint32_t pa[4];
    pa[0] = pack_bf16(s[0][0], s[0][1]);
    pa[1] = pack_bf16(s[0][2], s[0][3]);
    pa[2] = pack_bf16(s[1][0], s[1][1]);
    pa[3] = pack_bf16(s[1][2], s[1][3]);
    {
      const int mi = lane >> 3, ri = lane & 7;
      const unsigned char *rowp = st + (size_t)((mi & 1) * 8 + ri) * stride;
#pragma unroll
      for (int vt = 0; vt < VT / 2; ++vt) {
        const int dim = voff + wi * SH::VW + vt * 16 + (mi >> 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(b0, b1, b2, b3, rowp + dim * 2);
        mma_bf16_16816(o[2 * vt], pa, b0, b1);
        mma_bf16_16816(o[2 * vt + 1], pa, b2, b3);
      }
    }
    group_sync();  // the stage is refilled by a later issue
  }
  cp_async_wait_all();
  if (!waited) {  // a split without staging rows still orders itself after the gather
    pdl_wait();
    pdl_trigger();
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  // ---- combine the warp groups of this CTA (the stage area is reused)
  __syncthreads();
  float *Ob = reinterpret_cast<float *>(smem);  // [SUB][16][DV]
  float *Mb = Ob + SUB * 16 * DV;               // [SUB][16]
  float *Lb = Mb + SUB * 16;                    // [SUB][16]
  float *Wt = Lb + SUB * 16;                    // [16][n_split]
#pragma unroll
  for (int i = 0; i < VT; ++i) {
    const int dim = wi * SH::VW + i * 8 + 2 * t4;
    Ob[(grp * 16 + g) * DV + dim] = o[i][0];
    Ob[(grp * 16 + g) * DV + dim + 1] = o[i][1];
    Ob[(grp * 16 + g + 8) * DV + dim] = o[i][2];
    Ob[(grp * 16 + g + 8) * DV + dim + 1] = o[i][3];
  }
  if (wi == 0 && t4 == 0) {
    Mb[grp * 16 + g] = m0;
    Mb[grp * 16 + g + 8] = m1;
    Lb[grp * 16 + g] = l0;
    Lb[grp * 16 + g + 8] = l1;
  }
  __syncthreads();
  const size_t qbase = ((size_t)r * c.Kmax + j) * c.Hq + (size_t)kvh * G;
  const float ln2 = 0.69314718055994531f;
  // this split's partial (O, max, sum) for the cluster merge, after the
  // in-CTA buffers
  const bool cmerge = DQK == 128 && n_split == kAttnCluster;
  float *Pm = Wt, *Pl = Pm + 16;
  float *Po = reinterpret_cast<float *>(
      (reinterpret_cast<uintptr_t>(Pl + 16) + 15) & ~static_cast<uintptr_t>(15));
  for (int idx = tid; idx < G * DV / 2; idx += kAttnThreads) {
    const int h = (2 * idx) / DV, d = (2 * idx) % DV;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int sg = 0; sg < SUB; ++sg) M = fmaxf(M, Mb[sg * 16 + h]);
    const float ref = M == -CUDART_INF_F ? 0.f : M;
    float L = 0.f, a = 0.f, b = 0.f;
#pragma unroll
    for (int sg = 0; sg < SUB; ++sg) {
      const float wgt = exp2f(Mb[sg * 16 + h] - ref);
      L += wgt * Lb[sg * 16 + h];
      a += wgt * Ob[(sg * 16 + h) * DV + d];
      b += wgt * Ob[(sg * 16 + h) * DV + d + 1];
    }
    if (n_split == 1) {
      const float inv = L > 0.f ? 1.f / L : 0.f;
      *reinterpret_cast<uint32_t *>(out + (qbase + h) * DV + d) = pack_bf16(a * inv, b * inv);
      if (lse && d == 0) lse[qbase + h] = L > 0.f ? (M + log2f(L)) * ln2 : -CUDART_INF_F;
    } else if (cmerge) {
      *reinterpret_cast<float2 *>(Po + (size_t)h * DV + d) = make_float2(a, b);
      if (d == 0) {
        Pm[h] = M;
        Pl[h] = L;
      }
    } else {
      float *po = c.part_o + ((qbase + h) * n_split + split) * DV + d;
      po[0] = a;
      po[1] = b;
      if (d == 0) {
        c.part_ml[((qbase + h) * n_split + split) * 2 + 0] = M;
        c.part_ml[((qbase + h) * n_split + split) * 2 + 1] = L;
      }
    }
  }
  if (n_split == 1) return;

  if (cmerge) {
    // ---- the item's splits form a cluster: split q merges heads h = q
    //      (mod kAttnCluster) from every split's shared memory
    namespace cg = cooperative_groups;
    cg::cluster_group cl = cg::this_cluster();
    cl.sync();  // every split's partial is in its shared memory
    for (int h0 = split; h0 < G; h0 += kAttnCluster) {
      float wgt[kAttnCluster];
      float M = -CUDART_INF_F;
#pragma unroll
      for (int qs = 0; qs < kAttnCluster; ++qs) M = fmaxf(M, cl.map_shared_rank(Pm, qs)[h0]);
      const float ref = M == -CUDART_INF_F ? 0.f : M;
      float L = 0.f;
#pragma unroll
      for (int qs = 0; qs < kAttnCluster; ++qs) {
        wgt[qs] = exp2f(cl.map_shared_rank(Pm, qs)[h0] - ref);
        L += wgt[qs] * cl.map_shared_rank(Pl, qs)[h0];
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      for (int d = 2 * tid; d < DV; d += 2 * kAttnThreads) {
        float a = 0.f, b = 0.f;
#pragma unroll
        for (int qs = 0; qs < kAttnCluster; ++qs) {
          const float2 v = *reinterpret_cast<const float2 *>(cl.map_shared_rank(Po, qs) + (size_t)h0 * DV + d);
          a += wgt[qs] * v.x;
          b += wgt[qs] * v.y;
        }
        *reinterpret_cast<uint32_t *>(out + (qbase + h0) * DV + d) = pack_bf16(a * inv, b * inv);
      }
      if (lse && tid == 0) lse[qbase + h0] = L > 0.f ? (M + log2f(L)) * ln2 : -CUDART_INF_F;
    }
    cl.sync();  // no split leaves while another reads its shared memory
    return;
  }

  // ---- the CTA that finishes an item last merges its splits
  const int item = ((r * c.Kmax + j) * c.Hkv) + kvh;
  __threadfence();
  __syncthreads();
  if (tid == 0) sh_last = atomicAdd(&c.ticket[item], 1) == n_split - 1;
  __syncthreads();
  if (!sh_last) return;
  __threadfence();
  float *Ms = Wt + 16 * n_split;  // [16][n_split] maxima, then sums
  float *Ls = Ms + 16 * n_split;
  // The item's partial outputs are one contiguous block ([G][n_split][DV]
  // floats): when it fits in the free stage area, it is copied into shared
  // memory by one batch of cp.async while the weights are formed ...
  float *Ps = reinterpret_cast<float *>(
      (reinterpret_cast<uintptr_t>(Ls + 16 * n_split) + 15) & ~static_cast<uintptr_t>(15));
  const size_t pbytes = (size_t)G * n_split * DV * 4;
  const bool staged =
      (size_t)(reinterpret_cast<unsigned char *>(Ps) - smem) + pbytes <= body_bytes;
  if (staged) {
    const float4 *src = reinterpret_cast<const float4 *>(c.part_o + qbase * n_split * DV);
    for (int i = tid; i < (int)(pbytes / 16); i += kAttnThreads) cp_async_16(Ps + 4 * i, src + i);
    cp_async_commit();
  }
  // ... every (head, split) pair's max and sum in one parallel load ...
  for (int i = tid; i < G * n_split; i += kAttnThreads) {
    const float2 ml = __ldcg(reinterpret_cast<const float2 *>(c.part_ml + (qbase * n_split + i) * 2));
    Ms[i] = ml.x;
    Ls[i] = ml.y;
  }
  __syncthreads();
  // ... then the weights of each split, from shared memory
  for (int h = tid; h < G; h += kAttnThreads) {
    float M = -CUDART_INF_F;
    for (int sp = 0; sp < n_split; ++sp) M = fmaxf(M, Ms[h * n_split + sp]);
    const float ref = M == -CUDART_INF_F ? 0.f : M;
    float L = 0.f;
    for (int sp = 0; sp < n_split; ++sp) L += Ls[h * n_split + sp] * exp2f(Ms[h * n_split + sp] - ref);
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int sp = 0; sp < n_split; ++sp) Wt[h * n_split + sp] = exp2f(Ms[h * n_split + sp] - ref) * inv;
    if (lse) lse[qbase + h] = L > 0.f ? (M + log2f(L)) * ln2 : -CUDART_INF_F;
  }
  if (staged) {
    cp_async_wait_all();
    __syncthreads();
    for (int idx = tid; idx < G * DV / 2; idx += kAttnThreads) {
      const int h = (2 * idx) / DV, d = (2 * idx) % DV;
      float a = 0.f, b = 0.f;
      for (int sp = 0; sp < n_split; ++sp) {
        const float wgt = Wt[h * n_split + sp];
        const float2 v = *reinterpret_cast<const float2 *>(Ps + ((size_t)h * n_split + sp) * DV + d);
        a += wgt * v.x;
        b += wgt * v.y;
      }
      *reinterpret_cast<uint32_t *>(out + (qbase + h) * DV + d) = pack_bf16(a, b);
    }
    if (tid == 0) c.ticket[item] = 0;  // ready for the next launch
    return;
  }
  __syncthreads();
  constexpr int kMaxUnrolledSplits = 16;  // all partial loads of a thread in flight at once
  for (int idx = tid; idx < G * DV / 2; idx += kAttnThreads) {
    const int h = (2 * idx) / DV, d = (2 * idx) % DV;
    const float *po = c.part_o + (qbase + h) * n_split * DV + d;
    float a = 0.f, b = 0.f;
    for (int sp0 = 0; sp0 < n_split; sp0 += kMaxUnrolledSplits) {
      float2 v[kMaxUnrolledSplits];
#pragma unroll
      for (int u = 0; u < kMaxUnrolledSplits; ++u)
        if (sp0 + u < n_split)
          v[u] = __ldcg(reinterpret_cast<const float2 *>(po + (size_t)(sp0 + u) * DV));
#pragma unroll
      for (int u = 0; u < kMaxUnrolledSplits; ++u) {
        if (sp0 + u < n_split) {
          const float wgt = Wt[h * n_split + sp0 + u];
          a += wgt * v[u].x;
          b += wgt * v[u].y;
        }
      }
    }
    *reinterpret_cast<uint32_t *>(out + (qbase + h) * DV + d) = pack_bf16(a, b);
  }
  if (tid == 0) c.ticket[item] = 0;  // ready for the next launch
}

template <int DQK, int DV>
static cudaError_t launch_attn_t(const DevCtx &c, const uint16_t *q, const uint16_t *block,
                                 const int32_t *loc, uint16_t *out, float *lse, int n_split,
                                 cudaStream_t s, Timer *tm) {
  using SH = AttnShape<DQK, DV>;
  const size_t stride = (size_t)c.row * 2 + 16;
  const size_t stages = (size_t)SH::SUB * kAttnStages * kTileRows * stride;
  const size_t epi = ((size_t)SH::SUB * 16 * DV + 2 * SH::SUB * 16 + 48 * (size_t)n_split) * 4;
  const size_t body = ((stages > epi ? stages : epi) + 127) / 128 * 128;
  const size_t loc_off = ((size_t)SH::SUB * kAttnStages * kTileRows * 4 + 2 * SH::NW * 32 * 8 * 4 +
                          127) / 128 * 128;
  const int chunk = attn_chunk(c, n_split);
  const size_t smem = attn_smem_bytes<DQK, DV>(c.row, n_split) + 128 + loc_off +
                      attn_loc_bytes(chunk) + attn_ord_bytes(chunk);
  static size_t granted = 0;
  cudaError_t e = ensure_smem(k_attn<DQK, DV>, smem, granted);
  if (e != cudaSuccess) return e;
  dim3 grid(n_split, c.Kmax, c.N * c.Hkv);
  if (tm) tm->begin(K_ATTN, s);
  if (DQK == 128 && n_split == kAttnCluster) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = kAttnCluster;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, k_attn<DQK, DV>, c, q, block, loc, out, lse, n_split, chunk, body,
                           loc_off);
  } else {
    e = launch_pdl(k_attn<DQK, DV>, grid, dim3(kAttnThreads), smem, s, c, q, block, loc, out,
                   lse, n_split, chunk, body, loc_off);
  }
  if (tm) tm->end(K_ATTN, s);
  return e;
}

cudaError_t launch_attend(const DevCtx &c, const uint16_t *q, const uint16_t *block,
                          const int32_t *loc, uint16_t *out, float *lse, int n_split,
                          cudaStream_t s, Timer *tm) {
  return (c.dqk == 128 && c.dv == 128)
             ? launch_attn_t<128, 128>(c, q, block, loc, out, lse, n_split, s, tm)
             : launch_attn_t<576, 512>(c, q, block, loc, out, lse, n_split, s, tm);
}

}  // namespace dhs
