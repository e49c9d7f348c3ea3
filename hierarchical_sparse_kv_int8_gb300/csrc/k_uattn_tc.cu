// Step 5 for shared retrieval, 128-dim heads, on the fifth-generation tensor
// cores: the attention of all K_r queries of a request in one pass over the
// union of their selections.
//
// "Adaptive DHiSparse", eq. (6) and Fig. 3 callout 2: each distinct row of the
// union U_r is read once per round, whichever queries selected it; eq. (1),
// (5): query j attends over its own selection S_{r,j} and the block rows
// n_r .. n_r + j.  Visiting U_r once and keeping a row's score only for the
// queries that selected it gives each query exactly its own rows.
//
// One CTA per (request, kv head).  Its M = K_max x G (query, head) pairs are
// the 128 lanes of tensor memory (padded), one lane per pair; the walk (U_r in
// ascending row order, then the K_r block rows) is cut into tiles of kTcN
// rows.  Per tile: S = Q K^T (M = 128, N = kTcN, K = 128) into one of two
// tensor-memory buffers; each softmax thread reads its lane's kTcN scores,
// masks them by the queries that selected each row, keeps a running maximum
// in log2 units (the output is rescaled only when the maximum grows by more
// than kTcRescale, so the exponentials stay below 2^kTcRescale) and writes
// its row of P (bf16) to shared memory; then O += P V (M = 128, N = 128, K =
// kTcN) accumulates in tensor memory.  Warp roles: warps 0-7 are the softmax
// threads in two warpgroups (warps w and w + 4 own lanes 32(w mod 4) ..
// +31, the first group the first half of a tile's columns and of the output,
// the second the second half; they agree on each row's running maximum
// through shared memory), one thread of warp 8 issues every MMA, the
// kTcCopyWarps warps after it copy rows into a ring of kTcStages stages with
// 16-byte cp.async from wherever the union/probe located them (hot cache, optional
// pool, draft ring, staging) or from the caller's block rows, which they also
// write to the draft ring.  The stages, S buffers and P buffers are handed
// between the roles with mbarriers (MMA completion arrives through
// tcgen05.commit); every wait is bounded and, when it runs out, records a
// device error and lets the CTA finish, so tensor memory is always freed.
//
// Launches with few (request, kv head) items split each item's walk into
// nsplit contiguous ranges of tiles, one CTA each (split-KV): a CTA writes its
// unnormalised O, running maximum and sum to a scratch area, and the last of
// the item's CTAs to finish (a device-scope ticket) merges them with the
// usual log-sum-exp weights and writes the output.
#include "dhs_internal.cuh"
#include "ptx_util.cuh"
#include "tc_util.cuh"

#include <math_constants.h>

namespace dhs {
namespace {

constexpr int kTcM = 128;              // (query, head) pairs: tensor-memory lanes
constexpr int kTcD = 128;              // key and value dims
constexpr int kTcN = 64;               // walk rows per tile
constexpr int kTcStages = 4;
constexpr int kTcCopyWarps = 6;        // warps that copy rows (each issues ~64/6 rows a tile)
constexpr int kTcThreads = (9 + kTcCopyWarps) * 32;
constexpr int kTcSoftmax = 256;        // warps 0-7: two warpgroups, one per half tile
constexpr int kTcMmaWarp = 8;
constexpr int kTcLoadWarp0 = 9;        // warps 9 .. 8 + kTcCopyWarps copy
constexpr int kTcLoaders = kTcCopyWarps * 32;
constexpr int kTcHalf = kTcN / 2;      // columns of a tile per softmax warpgroup
constexpr uint32_t kTcCols = 256;      // S: two buffers of kTcN columns; O: 128 columns
constexpr uint32_t kTcColO = 128;
constexpr int kTcSpin = 1 << 20;
constexpr float kTcRescale = 8.f;

// Shared memory (from a 1024-byte boundary).
//   Q: K-major core-matrix layout of tc_util.cuh, cores along K 128 B apart,
//      8-row groups 2048 B apart
//   stage: keys, then values, each in the 128-byte-swizzled layout: two
//          8 KB halves (dims 0-63, 64-127), a walk row's half in 128
//          contiguous bytes at row * 128, its 16-byte chunk c at chunk
//          position c ^ (row mod 8) (keys K-major, values MN-major), so that
//          a warp's copy of a row's 512 bytes fills each 128-byte line once
//   P: K-major core-matrix layout over the tile's rows, cores 128 B apart,
//      8-row groups 1024 B
constexpr int kOffQ = 0;
constexpr int kQBytes = kTcM * kTcD * 2;
constexpr int kOffStage = kOffQ + kQBytes;
constexpr int kKBytes = kTcN * kTcD * 2;
constexpr int kHalfBytes = kKBytes / 2;  // 64 dims of the tile's rows
constexpr int kStageBytes = 2 * kKBytes;
constexpr int kOffP = kOffStage + kTcStages * kStageBytes;
constexpr int kPBytes = kTcM * kTcN * 2;
constexpr int kOffMask = kOffP + 2 * kPBytes;
constexpr int kOffRed = kOffMask + kTcStages * kTcN * 4;  // [2][2][128] partial maxima, [2][128] sums
constexpr int kOffBar = kOffRed + (2 * 2 * kTcM + 2 * kTcM) * 4;
constexpr int kNumBars = kTcStages * 2 + 2 * 4 + 1;
constexpr int kOffTmem = kOffBar + kNumBars * 8;
constexpr int kTcSmem = kOffTmem + 16 + 1024;  // (+ alignment of the swizzled stages)
static_assert(kTcSmem <= (int)kMaxDynSmem, "shared memory of the tensor-core union pass");

constexpr int kTcMaxSplit = 5;  // CTAs per item at most (30 items x 5 fill 150 of 152 SMs)
constexpr int kTcPartFloats = kTcM * kTcD + kTcM * 2;  // O [M][D], then (m, l) [M]
constexpr uint32_t kIdescQK = tc_idesc_bf16(kTcM, kTcN, 0, 0);
constexpr uint32_t kIdescPV = tc_idesc_bf16(kTcM, kTcD, 0, 1);

__device__ __forceinline__ int kmaj(int row, int chunk, int sbo) {
  return (row >> 3) * sbo + chunk * 128 + (row & 7) * 16;
}
// byte offset of 16-byte chunk `chunk` (0-15) of walk row `row` in a
// 128-byte-swizzled 64 x 128 operand
__device__ __forceinline__ int sw128(int row, int chunk) {
  return (chunk >> 3) * kHalfBytes + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

__global__ void __launch_bounds__(kTcThreads, 1)
k_uattn_tc(const DevCtx c, const uint16_t *__restrict__ q, const uint16_t *__restrict__ block,
           uint16_t *__restrict__ out, float *__restrict__ lse, int nsplit) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the swizzle pattern follows shared-memory address bits: start the
  // operands on a 1024-byte boundary
  unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ int abort_flag, sh_last;
  const int item = blockIdx.x / nsplit, sp = blockIdx.x - item * nsplit;
  const int r = item / c.Hkv, kvh = item - r * c.Hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
  uint64_t *full = bars, *empty = bars + kTcStages;
  uint64_t *s_full = bars + 2 * kTcStages, *s_free = s_full + 2, *p_full = s_full + 4,
           *pv_done = s_full + 6, *o_done = s_full + 8;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffTmem);
  volatile int *abort_v = &abort_flag;

  // everything earlier launches wrote (control words, union entries,
  // staging rows) and the caller's queries and block rows
  pdl_wait();
  pdl_trigger();
  const int Kr = c.Kr[r];
  if (Kr == 0) return;

  if (tid == 0) {
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(&full[i], kTcLoaders + kTcN);  // every copy thread's copies, every row's mask
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], kTcSoftmax);
      mbar_init(&p_full[i], kTcSoftmax);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(o_done, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == kTcMmaWarp) tmem_alloc(tmem_slot, kTcCols);

  const int G = c.Hq / c.Hkv, Mq = c.Kmax * G;
  const int KK = c.Kmax * c.k;
  const int U = c.counts[r * 4 + 0];
  const int L = U + Kr;  // union rows, then block rows
  const int T = (L + kTcN - 1) / kTcN;
  // this CTA's tiles: [t0, t1), TL of them (barrier phases count from t0)
  const int t0 = (int)((int64_t)T * sp / nsplit), t1 = (int)((int64_t)T * (sp + 1) / nsplit);
  const int TL = t1 - t0;
  const int64_t n = c.n[r];
  const uint16_t *brow = block + (size_t)r * c.Kmax * c.row;

  // query tile: lane m is query m / G, head m % G of this kv head
  for (int idx = tid; idx < kTcM * (kTcD / 8); idx += kTcThreads) {
    const int m = idx >> 4, ch = idx & 15;
    const int j = m / G;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (m < Mq && j < Kr)
      v = *reinterpret_cast<const uint4 *>(
          q + (((size_t)r * c.Kmax + j) * c.Hq + (size_t)kvh * G + (m - j * G)) * kTcD + ch * 8);
    *reinterpret_cast<uint4 *>(smem + kOffQ + kmaj(m, ch, 2048)) = v;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // (force: keep waiting after another thread gave up -- used for the
  // completion of the MMAs before tensor memory is freed)
  auto wait = [&](uint64_t *bar, uint32_t parity, bool force = false) {
    int spins = 0;
    while (!mbar_try_wait(bar, parity)) {
      if (!force && *abort_v) return;
      if (++spins > kTcSpin) {
        record_error(c.err, DC_TIMEOUT, K_ATTN_UNION);
        *abort_v = 1;
        return;
      }
    }
  };

  if (warp >= kTcLoadWarp0) {
    // ---------------------------------------------------------------- copies
    const int lw = warp - kTcLoadWarp0;
    // the block rows go into their draft-ring slots (this kv head's parts;
    // the item's first CTA writes them)
    for (int i = lw; i < (sp == 0 ? Kr : 0); i += kTcCopyWarps) {
      const int off = lane < 16 ? kvh * kTcD + lane * 8 : c.Hkv * kTcD + kvh * kTcD + (lane - 16) * 8;
      const uint4 v = *reinterpret_cast<const uint4 *>(brow + (size_t)i * c.row + off);
      *reinterpret_cast<uint4 *>(c.ring + ((size_t)r * c.Rd + (n + i) % c.Rd) * c.row + off) = v;
    }
    const int4 *uent = c.uent + (size_t)r * KK;
    const uint32_t all_q = (1u << Kr) - 1u;
    // lane l of copy warp lw holds the union entry of row lw + kTcCopyWarps l of a
    // tile: loaded three tiles ahead, turned into a source address when its
    // tile is issued.  A stage is complete when every copy thread's copies
    // have landed (asynchronous arrivals) and every row's query mask is
    // written (an ordinary arrival by the lane that wrote it).
    const int li = lw + kTcCopyWarps * lane;
    auto fetch = [&](int t) -> int4 {
      const int e = t * kTcN + li;
      return (li < kTcN && e < U && t < t1) ? uent[e] : make_int4(0, 0, 0, 0);
    };
    // entries of tiles t, t + 1, t + 2 (loaded three tiles ahead of their use)
    int4 e0 = fetch(t0), e1 = fetch(t0 + 1), e2 = fetch(t0 + 2);
    const int off = lane < 16 ? kvh * kTcD + lane * 8 : c.Hkv * kTcD + kvh * kTcD + (lane - 16) * 8;
    for (int tl = 0; tl < TL; ++tl) {
      const int t = t0 + tl, s = tl % kTcStages;
      const int4 ent = e0;
      e0 = e1;
      e1 = e2;
      e2 = fetch(t + 3);
      const uint16_t *tsrc = nullptr;
      uint32_t tmask = 0u;
      {
        const int e = t * kTcN + li;
        if (li < kTcN && e < U) {
          tsrc = loc_row(c, r, ent.y);
          if (tsrc == nullptr) record_error(c.err, DC_LOC_RANGE, K_ATTN_UNION);
          tmask = (uint32_t)ent.z;
        } else if (li < kTcN && e < L) {
          tsrc = brow + (size_t)(e - U) * c.row;
          tmask = all_q & ~((1u << (e - U)) - 1u);
        }
      }
      if (tl >= kTcStages) wait(&empty[s], (uint32_t)(((tl / kTcStages) - 1) & 1));
      unsigned char *kst = smem + kOffStage + s * kStageBytes, *vst = kst + kKBytes;
      uint32_t *msk = reinterpret_cast<uint32_t *>(smem + kOffMask) + s * kTcN;
      for (int it = 0; it * kTcCopyWarps + lw < kTcN; ++it) {
        const int i = lw + kTcCopyWarps * it;
        const uint16_t *src = reinterpret_cast<const uint16_t *>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(tsrc), it));
        unsigned char *dst = (lane < 16 ? kst : vst) + sw128(i, lane & 15);
        cp_async_16_zfill(dst, src ? (const void *)(src + off) : (const void *)c.ring, src ? 16 : 0);
      }
      cp_async_arrive_noinc(&full[s]);
      if (li < kTcN) {
        msk[li] = tsrc ? tmask : 0u;
        mbar_arrive(&full[s]);
      }
    }
  } else if (warp == kTcMmaWarp) {
    // ---------------------------------------------------------------- MMAs
    if (lane == 0) {
      const uint32_t sQ = smem_u32(smem + kOffQ);
      auto pv = [&](int u) {
        const int b = u & 1, s = u % kTcStages;
        wait(&p_full[b], (uint32_t)((u >> 1) & 1));
        tc_fence_after();
        const uint32_t sP = smem_u32(smem + kOffP + b * kPBytes);
        const uint32_t sV = smem_u32(smem + kOffStage + s * kStageBytes + kKBytes);
#pragma unroll
        for (int kk = 0; kk < kTcN / 16; ++kk)
          tc_mma(tmem + kTcColO, tc_desc(sP + kk * 256, 128, 1024),
                 tc_desc_sw128(sV + kk * 2048, kHalfBytes, 1024), kIdescPV,
                 (u > 0 || kk > 0) ? 1 : 0);
        tc_commit(&pv_done[b]);
        tc_commit(&empty[s]);
      };
      for (int tl = 0; tl < TL; ++tl) {
        const int s = tl % kTcStages, b = tl & 1;
        wait(&full[s], (uint32_t)((tl / kTcStages) & 1));
        fence_proxy_async_smem();  // the stage's copies, seen by the tensor cores
        if (tl >= 2) wait(&s_free[b], (uint32_t)(((tl - 2) >> 1) & 1));
        tc_fence_after();
        const uint32_t sK = smem_u32(smem + kOffStage + s * kStageBytes);
#pragma unroll
        for (int kk = 0; kk < kTcD / 16; ++kk)
          tc_mma(tmem + (uint32_t)(b * kTcN), tc_desc(sQ + kk * 256, 128, 2048),
                 tc_desc_sw128(sK + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024),
                 kIdescQK, kk > 0 ? 1 : 0);
        tc_commit(&s_full[b]);
        if (tl >= 1) pv(tl - 1);
      }
      if (TL > 0) pv(TL - 1);
      tc_commit(o_done);
      wait(o_done, 0u, true);  // every MMA has completed before tensor memory is freed
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax
    const int hg = warp >> 2;              // warpgroup: half of the tile's columns
    const int m = tid & (kTcM - 1);        // tensor-memory lane: the (query, head) pair
    const int j = m / G;
    const bool valid = m < Mq && j < Kr;
    const uint32_t lrow = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = c.scale_log2;
    float *red = reinterpret_cast<float *>(smem + kOffRed);  // [tile parity][group][lane]
    float *lsum = red + 2 * 2 * kTcM;                        // [group][lane]
    float m_run = -CUDART_INF_F, l = 0.f;
    for (int tl = 0; tl < TL; ++tl) {
      const int b = tl & 1, s = tl % kTcStages;
      wait(&s_full[b], (uint32_t)((tl >> 1) & 1));
      wait(&full[s], (uint32_t)((tl / kTcStages) & 1));  // the tile's masks
      tc_fence_after();
      uint32_t sv[kTcHalf];
      tmem_ld32(tmem + lrow + (uint32_t)(b * kTcN + hg * kTcHalf), sv);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&s_free[b]);
      // this half's query masks: lane l reads row hg * 32 + l; one ballot
      // per query gives the 32-bit word of rows this thread's query selected
      const uint32_t *msk = reinterpret_cast<const uint32_t *>(smem + kOffMask) + s * kTcN;
      const uint32_t ma = msk[hg * kTcHalf + lane];
      uint32_t kw = 0u;
#pragma unroll
      for (int jj = 0; jj < kMaxKmax; ++jj) {
        const uint32_t ba = __ballot_sync(0xffffffffu, (ma >> jj) & 1u);
        if (jj == j) kw = ba;
      }
      if (!valid) kw = 0u;
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int i = 0; i < kTcHalf; ++i) {
        const bool keep = ((kw >> i) & 1u) != 0u;
        const float x = keep ? __uint_as_float(sv[i]) * sl2 : -CUDART_INF_F;
        sv[i] = __float_as_uint(x);
        mx = fmaxf(mx, x);
      }
      // both halves of a row agree on its maximum
      red[(b * 2 + hg) * kTcM + m] = mx;
      named_sync(1, kTcSoftmax);
      mx = fmaxf(mx, red[(b * 2 + (hg ^ 1)) * kTcM + m]);
      const float m_new = fmaxf(m_run, mx);
      const bool need = m_new > m_run + kTcRescale;  // false while nothing is kept
      if (__any_sync(0xffffffffu, need) && tl >= 1) {
        // rescale this lane's half of the output after the previous tile's
        // P V completed
        wait(&pv_done[(tl - 1) & 1], (uint32_t)(((tl - 1) >> 1) & 1));
        tc_fence_after();
        const float f = need ? ex2_approx(m_run - m_new) : 1.f;
#pragma unroll
        for (int cc = 0; cc < kTcD / 2; cc += 32) {
          const uint32_t ta = tmem + lrow + kTcColO + (uint32_t)(hg * (kTcD / 2) + cc);
          uint32_t ov[32];
          tmem_ld32(ta, ov);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f);
          tmem_st32(ta, ov);
        }
        tmem_wait_st();
      }
      if (need) {
        l *= ex2_approx(m_run - m_new);
        m_run = m_new;
      }
      // P_t replaces P_{t-2}: its P V must have completed
      if (tl >= 2) wait(&pv_done[b], (uint32_t)(((tl - 2) >> 1) & 1));
      unsigned char *prow = smem + kOffP + b * kPBytes + (m >> 3) * 1024 + (m & 7) * 16;
      const bool live = m_run != -CUDART_INF_F;
#pragma unroll
      for (int ch = 0; ch < kTcHalf / 8; ++ch) {
        float p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          p[i] = live ? ex2_approx(__uint_as_float(sv[ch * 8 + i]) - m_run) : 0.f;
          l += p[i];
        }
        uint4 w;
        w.x = pack_bf16(p[0], p[1]);
        w.y = pack_bf16(p[2], p[3]);
        w.z = pack_bf16(p[4], p[5]);
        w.w = pack_bf16(p[6], p[7]);
        *reinterpret_cast<uint4 *>(prow + (hg * (kTcHalf / 8) + ch) * 128) = w;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[b]);
    }
    // output: O / l over both halves' sums, and the natural-log sum-exp
    lsum[hg * kTcM + m] = l;
    wait(o_done, 0u);
    named_sync(1, kTcSoftmax);
    l += lsum[(hg ^ 1) * kTcM + m];
    tc_fence_after();
    const int h = kvh * G + (m - j * G);
    uint16_t *orow = valid ? out + (((size_t)r * c.Kmax + j) * c.Hq + h) * kTcD : nullptr;
    if (nsplit > 1) {
      // this CTA's part: O (zero for an empty range), then (m, l) per lane
      float *po = c.tc_part + ((size_t)item * nsplit + sp) * kTcPartFloats;
#pragma unroll
      for (int cc = 0; cc < kTcD / 2; cc += 32) {
        const int col = hg * (kTcD / 2) + cc;
        uint32_t ov[32];
        if (TL > 0) {
          tmem_ld32(tmem + lrow + kTcColO + (uint32_t)col, ov);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = 0u;
        }
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4 *>(po + (size_t)m * kTcD + col + i) =
              make_float4(__uint_as_float(ov[i]), __uint_as_float(ov[i + 1]),
                          __uint_as_float(ov[i + 2]), __uint_as_float(ov[i + 3]));
      }
      if (hg == 0) *reinterpret_cast<float2 *>(po + kTcM * kTcD + 2 * m) = make_float2(m_run, l);
      __threadfence();
      named_sync(1, kTcSoftmax);
      if (tid == 0) sh_last = atomicAdd(&c.u_ticket[item], 1) == nsplit - 1;
      named_sync(1, kTcSoftmax);
      if (sh_last) {
        // the item's last CTA: out = sum_s w_s O_s / sum_s w_s l_s with
        // w_s = 2^(m_s - max_s m_s), for this lane's half of the columns
        __threadfence();
        const float *pi = c.tc_part + (size_t)item * nsplit * kTcPartFloats;
        float mm = -CUDART_INF_F;
        for (int s2 = 0; s2 < nsplit; ++s2)
          mm = fmaxf(mm, pi[(size_t)s2 * kTcPartFloats + kTcM * kTcD + 2 * m]);
        float den = 0.f;
        float wsp[kTcMaxSplit];
#pragma unroll
        for (int s2 = 0; s2 < kTcMaxSplit; ++s2) {
          wsp[s2] = 0.f;
          if (s2 < nsplit) {
            const float2 ml = *reinterpret_cast<const float2 *>(
                pi + (size_t)s2 * kTcPartFloats + kTcM * kTcD + 2 * m);
            wsp[s2] = ml.x == -CUDART_INF_F ? 0.f : ex2_approx(ml.x - mm);
            den += wsp[s2] * ml.y;
          }
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
        if (valid) {
          for (int col = hg * (kTcD / 2); col < (hg + 1) * (kTcD / 2); col += 8) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int s2 = 0; s2 < kTcMaxSplit; ++s2) {
              if (s2 >= nsplit || wsp[s2] == 0.f) continue;
              const float *o = pi + (size_t)s2 * kTcPartFloats + (size_t)m * kTcD + col;
              const float4 a0 = *reinterpret_cast<const float4 *>(o);
              const float4 a1 = *reinterpret_cast<const float4 *>(o + 4);
              acc[0] += wsp[s2] * a0.x; acc[1] += wsp[s2] * a0.y;
              acc[2] += wsp[s2] * a0.z; acc[3] += wsp[s2] * a0.w;
              acc[4] += wsp[s2] * a1.x; acc[5] += wsp[s2] * a1.y;
              acc[6] += wsp[s2] * a1.z; acc[7] += wsp[s2] * a1.w;
            }
            uint4 w;
            w.x = pack_bf16(acc[0] * inv, acc[1] * inv);
            w.y = pack_bf16(acc[2] * inv, acc[3] * inv);
            w.z = pack_bf16(acc[4] * inv, acc[5] * inv);
            w.w = pack_bf16(acc[6] * inv, acc[7] * inv);
            *reinterpret_cast<uint4 *>(orow + col) = w;
          }
          if (lse && hg == 0)
            lse[((size_t)r * c.Kmax + j) * c.Hq + h] =
                den > 0.f ? (mm + log2f(den)) * 0.69314718055994531f : -CUDART_INF_F;
        }
        if (tid == 0) c.u_ticket[item] = 0;  // ready for the next launch
      }
    } else {
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int cc = 0; cc < kTcD / 2; cc += 32) {
      const int col = hg * (kTcD / 2) + cc;
      uint32_t ov[32];
      tmem_ld32(tmem + lrow + kTcColO + (uint32_t)col, ov);
      tmem_wait_ld();
      if (valid) {
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
          uint4 w;
          w.x = pack_bf16(__uint_as_float(ov[i + 0]) * inv, __uint_as_float(ov[i + 1]) * inv);
          w.y = pack_bf16(__uint_as_float(ov[i + 2]) * inv, __uint_as_float(ov[i + 3]) * inv);
          w.z = pack_bf16(__uint_as_float(ov[i + 4]) * inv, __uint_as_float(ov[i + 5]) * inv);
          w.w = pack_bf16(__uint_as_float(ov[i + 6]) * inv, __uint_as_float(ov[i + 7]) * inv);
          *reinterpret_cast<uint4 *>(orow + col + i) = w;
        }
      }
    }
    if (valid && lse && hg == 0)
      lse[((size_t)r * c.Kmax + j) * c.Hq + h] =
          l > 0.f ? (m_run + log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kTcMmaWarp) tmem_dealloc(tmem, kTcCols);
}

}  // namespace

bool uattn_tc_supported(const DevCtx &c) {
  return c.dqk == kTcD && c.dv == kTcD && c.layout == DHS_KV_SPLIT &&
         c.Kmax * (c.Hq / c.Hkv) <= kTcM;
}

size_t uattn_tc_part_floats(const DevCtx &c) {
  return (size_t)c.N * c.Hkv * kTcMaxSplit * kTcPartFloats;
}

cudaError_t launch_uattn_tc(const DevCtx &c, const uint16_t *q, const uint16_t *block,
                            uint16_t *out, float *lse, cudaStream_t s, Timer *tm, int split) {
  static size_t granted = 0;
  cudaError_t e = ensure_smem(k_uattn_tc, (size_t)kTcSmem, granted);
  if (e != cudaSuccess) return e;
  // one CTA per SM (its shared memory): split the items' walks while the
  // launch leaves SMs idle
  const int items = c.N * c.Hkv;
  int nsplit = split > 0 ? split : c.sms / std::max(1, items);
  nsplit = std::max(1, std::min(kTcMaxSplit, nsplit));
  if (!c.tc_part) nsplit = 1;
  if (tm) tm->begin(K_ATTN_UNION, s);
  e = launch_pdl(k_uattn_tc, dim3(items * nsplit), dim3(kTcThreads), (size_t)kTcSmem, s, c, q,
                 block, out, lse, nsplit);
  if (tm) tm->end(K_ATTN_UNION, s);
  return e;
}

}  // namespace dhs
