// Step 5 of the verification round and the state updates around it.
//
// "Adaptive DHiSparse", eq. (1) and (5): query j of request r attends over its
// own ordered selection S_{r,j} (through the locations of eq. (11)-(12)) and
// the block rows n_r .. n_r + j read from the tail.  Section 3.4: promoted rows
// are copied from staging to their stable hot-cache addresses after the
// attention readers.  Eq. (7), (9), (10): block rows live in a draft ring at
// phi(r, t) = r R_d + (t mod R_d); commit keeps the accepted prefix.
//
// Attention is split-KV flash decoding: one CTA per (request, query, kv head,
// split of the row list).  Rows are gathered by location into shared memory
// with 16-byte cp.async (three stages in flight), and the query-head block
// (the query heads sharing one kv head, padded to 16) is multiplied on the
// tensor cores with bf16 mma.sync m16n8k16 and fp32 accumulation: S = Q K^T
// for 16 rows at a time, online softmax in the log2 domain, O += P V.  Splits
// are merged by their log-sum-exp in k_merge.
#include "dhs_internal.cuh"
#include "ptx_util.cuh"

#include <math_constants.h>

namespace dhs {

constexpr int kAttnStages = 3;
constexpr int kTileRows = 16;

bool attn_shape_supported(int dqk, int dv, int layout) {
  if (layout == DHS_KV_SPLIT) return dqk == 128 && dv == 128;
  return dqk == 576 && dv == 512;
}

template <int DQK, int DV>
struct AttnShape {
  static constexpr int NW = (DQK > 256) ? 4 : 1;  // warps per work item
  static constexpr int KW = DQK / NW;             // key dims per warp
  static constexpr int VW = DV / NW;              // value dims per warp
  static constexpr int KS = KW / 16;              // k-steps per warp
  static constexpr int VT = VW / 8;               // n-tiles of the output per warp
  static_assert(KW % 16 == 0 && VW % 16 == 0, "dims per warp must be multiples of 16");
};

int attn_splits(const DevCtx &c, int active_queries) {
  (void)active_queries;
  const int rows = c.k + c.Kmax;
  const bool wide = c.dqk > 256;
  const int target = wide ? 152 * 4 : 152 * 16;
  const int items = c.N * c.Kmax * c.Hkv;
  int ns = (target + items - 1) / items;
  const int max_ns = (rows + 31) / 32;
  if (ns > max_ns) ns = max_ns;
  if (ns < 1) ns = 1;
  int chunk = (rows + ns - 1) / ns;
  chunk = (chunk + kTileRows - 1) / kTileRows * kTileRows;
  return (rows + chunk - 1) / chunk;
}

size_t attn_partial_floats(const DevCtx &c, int n_split) {
  return (size_t)c.N * c.Kmax * c.Hq * n_split * (c.dv + 2);
}

template <int DQK, int DV>
__global__ void __launch_bounds__(AttnShape<DQK, DV>::NW * 32)
k_attn(const DevCtx c, const uint16_t *__restrict__ q, const uint16_t *__restrict__ block,
       const int32_t *__restrict__ loc, uint16_t *__restrict__ out, float *__restrict__ lse,
       int n_split, int chunk) {
  using SH = AttnShape<DQK, DV>;
  constexpr int NW = SH::NW, KS = SH::KS, VT = SH::VT;
  extern __shared__ __align__(128) unsigned char smem[];
  const int split = blockIdx.x, j = blockIdx.y;
  const int r = blockIdx.z / c.Hkv, kvh = blockIdx.z % c.Hkv;
  if (j >= c.Kr[r]) return;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  const int G = c.Hq / c.Hkv;  // query heads per kv head (<= 16)
  const int k = c.k;
  const int total = k + j + 1;
  const int e0 = split * chunk;
  const int e1 = min(e0 + chunk, total);
  const int rowb = c.row * 2;
  const int stride = rowb + 16;  // padded so ldmatrix rows hit distinct banks
  const int nv = rowb >> 4;
  unsigned char *stage_base = smem;
  int *vflag = reinterpret_cast<int *>(smem + (size_t)kAttnStages * kTileRows * stride);
  float *red = reinterpret_cast<float *>(vflag + kAttnStages * kTileRows);  // [2][NW][32][8]
  const int koff = (c.layout == DHS_KV_LATENT) ? 0 : kvh * DQK;
  const int voff = (c.layout == DHS_KV_LATENT) ? 0 : c.Hkv * DQK + kvh * DV;
  const int32_t *lrow = loc + ((size_t)r * c.Kmax + j) * k;
  const uint16_t *brow = block + (size_t)r * c.Kmax * c.row;

  // query fragments (rows = query heads of this kv head, zero padded)
  uint32_t qa[KS][4];
  {
    const uint16_t *qb = q + (((size_t)r * c.Kmax + j) * c.Hq + (size_t)kvh * G) * DQK;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int col = w * SH::KW + ks * 16 + 2 * t4;
      const uint32_t *r0 = reinterpret_cast<const uint32_t *>(qb + (size_t)g * DQK + col);
      const uint32_t *r1 = reinterpret_cast<const uint32_t *>(qb + (size_t)(g + 8) * DQK + col);
      qa[ks][0] = g < G ? r0[0] : 0u;
      qa[ks][1] = g + 8 < G ? r1[0] : 0u;
      qa[ks][2] = g < G ? r0[4] : 0u;
      qa[ks][3] = g + 8 < G ? r1[4] : 0u;
    }
  }

  const int ntiles = e1 > e0 ? (e1 - e0 + kTileRows - 1) / kTileRows : 0;
  auto issue = [&](int it) {
    if (it < ntiles) {
      unsigned char *st = stage_base + (size_t)(it % kAttnStages) * kTileRows * stride;
      int *vf = vflag + (it % kAttnStages) * kTileRows;
      for (int cid = tid; cid < kTileRows * nv; cid += NW * 32) {
        const int rr = cid / nv, v = cid - rr * nv;
        const int e = e0 + it * kTileRows + rr;
        const uint16_t *src = nullptr;
        if (e < e1) {
          if (e < k) {
            const int32_t l = lrow[e];
            if (l >= 0) {
              src = loc_row(c, r, l);
              if (src == nullptr && v == 0) record_error(c.err, DC_LOC_RANGE, K_ATTN);
            }
          } else {
            src = brow + (size_t)(e - k) * c.row;
          }
        }
        cp_async_16_zfill(st + (size_t)rr * stride + v * 16,
                          src ? (const void *)(src + v * 8) : (const void *)brow, src ? 16 : 0);
        if (v == 0) vf[rr] = src != nullptr;
      }
    }
    cp_async_commit();
  };

  float o[VT][4];
#pragma unroll
  for (int i = 0; i < VT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;

#pragma unroll
  for (int s = 0; s < kAttnStages - 1; ++s) issue(s);
  for (int it = 0; it < ntiles; ++it) {
    issue(it + kAttnStages - 1);
    cp_async_wait_group<kAttnStages - 1>();
    __syncthreads();
    const unsigned char *st = stage_base + (size_t)(it % kAttnStages) * kTileRows * stride;
    const int *vf = vflag + (it % kAttnStages) * kTileRows;

    // S = Q K^T over this warp's key dims, two n-tiles of 8 rows
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int mi = lane >> 3, ri = lane & 7;
      const unsigned char *rowp = st + (size_t)((mi >> 1) * 8 + ri) * stride;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int col = koff + w * SH::KW + ks * 16 + (mi & 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(b0, b1, b2, b3, rowp + col * 2);
        mma_bf16_16816(s[0], qa[ks], b0, b1);
        mma_bf16_16816(s[1], qa[ks], b2, b3);
      }
    }
    if (NW > 1) {
      float *my = red + ((size_t)((it & 1) * NW + w) * 32 + lane) * 8;
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
    // scale to log2 units and mask invalid rows
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
      o[i][0] *= al0; o[i][1] *= al0;
      o[i][2] *= al1; o[i][3] *= al1;
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
        const int dim = voff + w * SH::VW + vt * 16 + (mi >> 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(b0, b1, b2, b3, rowp + dim * 2);
        mma_bf16_16816(o[2 * vt], pa, b0, b1);
        mma_bf16_16816(o[2 * vt + 1], pa, b2, b3);
      }
    }
    __syncthreads();  // the stage is refilled by the next issue
  }
  cp_async_wait_all();

  // row sums across the quad
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  const size_t qbase = ((size_t)r * c.Kmax + j) * c.Hq + (size_t)kvh * G;
  if (n_split == 1) {
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
    for (int i = 0; i < VT; ++i) {
      const int dim = w * SH::VW + i * 8 + 2 * t4;
      if (g < G)
        *reinterpret_cast<uint32_t *>(out + (qbase + g) * DV + dim) =
            pack_bf16(o[i][0] * inv0, o[i][1] * inv0);
      if (g + 8 < G)
        *reinterpret_cast<uint32_t *>(out + (qbase + g + 8) * DV + dim) =
            pack_bf16(o[i][2] * inv1, o[i][3] * inv1);
    }
    if (lse && w == 0 && t4 == 0) {
      const float ln2 = 0.69314718055994531f;
      if (g < G) lse[qbase + g] = l0 > 0.f ? (m0 + log2f(l0)) * ln2 : -CUDART_INF_F;
      if (g + 8 < G) lse[qbase + g + 8] = l1 > 0.f ? (m1 + log2f(l1)) * ln2 : -CUDART_INF_F;
    }
  } else {
    // partials: [(r, j, h)][split] -> DV floats of O, then (m, l)
    float *po = c.part_o;
#pragma unroll
    for (int i = 0; i < VT; ++i) {
      const int dim = w * SH::VW + i * 8 + 2 * t4;
      if (g < G) {
        float *d = po + ((qbase + g) * n_split + split) * DV + dim;
        d[0] = o[i][0];
        d[1] = o[i][1];
      }
      if (g + 8 < G) {
        float *d = po + ((qbase + g + 8) * n_split + split) * DV + dim;
        d[0] = o[i][2];
        d[1] = o[i][3];
      }
    }
    if (w == 0 && t4 == 0) {
      if (g < G) {
        c.part_ml[((qbase + g) * n_split + split) * 2 + 0] = m0;
        c.part_ml[((qbase + g) * n_split + split) * 2 + 1] = l0;
      }
      if (g + 8 < G) {
        c.part_ml[((qbase + g + 8) * n_split + split) * 2 + 0] = m1;
        c.part_ml[((qbase + g + 8) * n_split + split) * 2 + 1] = l1;
      }
    }
  }
}

// Log-sum-exp merge of the splits of one (request, query): one CTA.
__global__ void __launch_bounds__(256)
k_merge(const DevCtx c, uint16_t *__restrict__ out, float *__restrict__ lse, int n_split) {
  extern __shared__ float wts[];  // [Hq][n_split]
  __shared__ float sh_lse[16 * 16];
  const int r = blockIdx.x / c.Kmax, j = blockIdx.x % c.Kmax;
  if (j >= c.Kr[r]) return;
  const size_t qbase = ((size_t)r * c.Kmax + j) * c.Hq;
  for (int h = threadIdx.x; h < c.Hq; h += blockDim.x) {
    const float *ml = c.part_ml + (qbase + h) * n_split * 2;
    float M = -CUDART_INF_F;
    for (int s = 0; s < n_split; ++s) M = fmaxf(M, ml[2 * s]);
    const float ref = M == -CUDART_INF_F ? 0.f : M;
    float L = 0.f;
    for (int s = 0; s < n_split; ++s) L += ml[2 * s + 1] * exp2f(ml[2 * s] - ref);
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int s = 0; s < n_split; ++s) wts[h * n_split + s] = exp2f(ml[2 * s] - ref) * inv;
    sh_lse[h] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -CUDART_INF_F;
  }
  __syncthreads();
  const int dv = c.dv;
  for (int idx = threadIdx.x; idx < c.Hq * dv / 2; idx += blockDim.x) {
    const int h = (2 * idx) / dv, dim = (2 * idx) % dv;
    const float *po = c.part_o + (qbase + h) * n_split * dv + dim;
    float a = 0.f, b = 0.f;
    for (int s = 0; s < n_split; ++s) {
      const float wgt = wts[h * n_split + s];
      a += wgt * po[(size_t)s * dv];
      b += wgt * po[(size_t)s * dv + 1];
    }
    *reinterpret_cast<uint32_t *>(out + (qbase + h) * dv + dim) = pack_bf16(a, b);
  }
  if (lse)
    for (int h = threadIdx.x; h < c.Hq; h += blockDim.x) lse[qbase + h] = sh_lse[h];
}

// After attention: block rows into the draft ring at phi(r, n_r + u), and
// promoted rows from staging into their hot-cache slots.  One warp per row.
__global__ void __launch_bounds__(256)
k_post_attend(const DevCtx c, const uint16_t *__restrict__ block) {
  const int r = blockIdx.y;
  const int Kr = c.Kr[r];
  if (Kr == 0) return;
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5), nwt = gridDim.x * 8;
  const int P = c.counts[r * 4 + 2];
  const int64_t n = c.n[r];
  const int nv = (c.row * 2) >> 4;
  const int KK = c.Kmax * c.k;
  for (int job = gw; job < Kr + P; job += nwt) {
    const uint4 *src;
    uint4 *dst;
    if (job < Kr) {
      src = reinterpret_cast<const uint4 *>(block + ((size_t)r * c.Kmax + job) * c.row);
      dst = reinterpret_cast<uint4 *>(c.ring + ((size_t)r * c.Rd + (n + job) % c.Rd) * c.row);
    } else {
      const int p = job - Kr;
      const int sidx = c.promo_src[(size_t)r * c.B + p];
      const int slot = c.promo_dst[(size_t)r * c.B + p];
      if (sidx < 0 || sidx >= KK || slot < 0 || slot >= c.B) {
        if (lane == 0) record_error(c.err, DC_CAPACITY, K_POST_ATTEND);
        continue;
      }
      src = reinterpret_cast<const uint4 *>(c.stage + ((size_t)r * KK + sidx) * c.row);
      dst = reinterpret_cast<uint4 *>(c.hot_data + ((size_t)r * c.B + slot) * c.row);
    }
    for (int v = lane; v < nv; v += 32) dst[v] = src[v];
  }
}

cudaError_t launch_attend(const DevCtx &c, const uint16_t *q, const uint16_t *block,
                          const int32_t *loc, uint16_t *out, float *lse, int n_split,
                          cudaStream_t s, Timer *tm) {
  const int rows = c.k + c.Kmax;
  int chunk = (rows + n_split - 1) / n_split;
  chunk = (chunk + kTileRows - 1) / kTileRows * kTileRows;
  dim3 grid(n_split, c.Kmax, c.N * c.Hkv);
  const int stride = c.row * 2 + 16;
  if (c.dqk == 128 && c.dv == 128) {
    using SH = AttnShape<128, 128>;
    const size_t smem = (size_t)kAttnStages * kTileRows * (stride + 4) + 2 * SH::NW * 32 * 8 * 4;
    static size_t granted = 0;
    cudaError_t e = ensure_smem(k_attn<128, 128>, smem, granted);
    if (e != cudaSuccess) return e;
    if (tm) tm->begin(K_ATTN, s);
    k_attn<128, 128><<<grid, SH::NW * 32, smem, s>>>(c, q, block, loc, out, lse, n_split, chunk);
    if (tm) tm->end(K_ATTN, s);
  } else {
    using SH = AttnShape<576, 512>;
    const size_t smem = (size_t)kAttnStages * kTileRows * (stride + 4) + 2 * SH::NW * 32 * 8 * 4;
    static size_t granted = 0;
    cudaError_t e = ensure_smem(k_attn<576, 512>, smem, granted);
    if (e != cudaSuccess) return e;
    if (tm) tm->begin(K_ATTN, s);
    k_attn<576, 512><<<grid, SH::NW * 32, smem, s>>>(c, q, block, loc, out, lse, n_split, chunk);
    if (tm) tm->end(K_ATTN, s);
  }
  if (n_split > 1) {
    if (tm) tm->begin(K_MERGE, s);
    k_merge<<<c.N * c.Kmax, 256, (size_t)c.Hq * n_split * 4, s>>>(c, out, lse, n_split);
    if (tm) tm->end(K_MERGE, s);
  }
  int bpr = (152 * 4 + c.N - 1) / c.N;
  if (bpr > 64) bpr = 64;
  if (tm) tm->begin(K_POST_ATTEND, s);
  k_post_attend<<<dim3(bpr, c.N), 256, 0, s>>>(c, block);
  if (tm) tm->end(K_POST_ATTEND, s);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- commit
// aux[r*4 + 0] = a_r, aux[r*4 + 1..2] = n_r before the commit (lo, hi words).
__global__ void __launch_bounds__(256) k_commit(const DevCtx c) {
  const int r = blockIdx.y;
  const int a = c.aux[r * 4 + 0];
  const int64_t n_old = (int64_t)(uint32_t)c.aux[r * 4 + 1] | ((int64_t)c.aux[r * 4 + 2] << 32);
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5), nwt = gridDim.x * 8;
  const int nv = (c.row * 2) >> 4;
  uint16_t *host = const_cast<uint16_t *>(c.host[r]);
  for (int u = gw; u < a; u += nwt) {
    const uint4 *src =
        reinterpret_cast<const uint4 *>(c.ring + ((size_t)r * c.Rd + (n_old + u) % c.Rd) * c.row);
    uint4 *dst = reinterpret_cast<uint4 *>(host + (size_t)(n_old + u) * c.row);
    for (int v = lane; v < nv; v += 32) dst[v] = src[v];
  }
  if (blockIdx.x == 0 && threadIdx.x == 0 && c.aux[r * 4 + 3]) {
    c.n[r] = n_old + a;
    c.Kr[r] = 0;
  }
}

cudaError_t launch_commit(const DevCtx &c, cudaStream_t s, Timer *tm) {
  if (tm) tm->begin(K_COMMIT, s);
  k_commit<<<dim3(1, c.N), 256, 0, s>>>(c);
  if (tm) tm->end(K_COMMIT, s);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- residency
__global__ void k_res_clear(const DevCtx c, int slot, int64_t old_count) {
  int32_t *map = c.opt_map + (size_t)slot * c.Sm;
  const int32_t *list = c.opt_list + (size_t)slot * c.opt_max;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < old_count;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t row = list[i];
    if (row >= 0 && row < c.Sm) map[row] = -1;
  }
}

__global__ void __launch_bounds__(256) k_res_fill(const DevCtx c, int slot, int64_t count) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = blockIdx.x * 8 + (threadIdx.x >> 5), nwt = gridDim.x * 8;
  const int nv = (c.row * 2) >> 4;
  const int32_t *list = c.opt_list + (size_t)slot * c.opt_max;
  const uint16_t *host = c.host[slot];
  for (int64_t i = gw; i < count; i += nwt) {
    const int32_t row = list[i];
    if (row < 0 || row >= c.Sm) {
      if (lane == 0) record_error(c.err, DC_ROW_RANGE, K_RESIDENCY_FILL);
      continue;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(host + (size_t)row * c.row);
    uint4 *dst = reinterpret_cast<uint4 *>(c.opt + ((size_t)slot * c.opt_max + i) * c.row);
    for (int v = lane; v < nv; v += 32) dst[v] = ld_stream_16(src + v);
  }
}

__global__ void k_res_publish(const DevCtx c, int slot, int64_t count) {
  int32_t *map = c.opt_map + (size_t)slot * c.Sm;
  const int32_t *list = c.opt_list + (size_t)slot * c.opt_max;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t row = list[i];
    if (row >= 0 && row < c.Sm) map[row] = (int32_t)i;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) c.opt_count[slot] = count;
}

cudaError_t launch_residency(const DevCtx &c, int slot, int64_t old_count, int64_t new_count,
                             cudaStream_t s, Timer *tm) {
  // the clear runs before the caller uploads the new list
  if (old_count >= 0) {
    if (tm) tm->begin(K_RESIDENCY_CLEAR, s);
    k_res_clear<<<256, 256, 0, s>>>(c, slot, old_count);
    if (tm) tm->end(K_RESIDENCY_CLEAR, s);
  }
  if (new_count >= 0) {
    if (tm) tm->begin(K_RESIDENCY_FILL, s);
    k_res_fill<<<512, 256, 0, s>>>(c, slot, new_count);
    if (tm) tm->end(K_RESIDENCY_FILL, s);
    if (tm) tm->begin(K_RESIDENCY_PUBLISH, s);
    k_res_publish<<<256, 256, 0, s>>>(c, slot, new_count);
    if (tm) tm->end(K_RESIDENCY_PUBLISH, s);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------- binding
__global__ void k_bind_reset(const DevCtx c, int slot, int64_t n_committed) {
  const int64_t tid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t nt = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = tid; i < c.Sm; i += nt) {
    c.hot_map[(size_t)slot * c.Sm + i] = -1;
    c.opt_map[(size_t)slot * c.Sm + i] = -1;
  }
  for (int64_t i = tid; i < c.B; i += nt) {
    c.hot_row[(size_t)slot * c.B + i] = -1;
    c.hot_stamp[(size_t)slot * c.B + i] = -1;
    c.lru[(size_t)slot * c.B + i] = (int32_t)i;
  }
  if (tid == 0) {
    c.n[slot] = n_committed;
    c.ring_first[slot] = n_committed;
    c.Kr[slot] = 0;
    c.opt_count[slot] = 0;
  }
}

cudaError_t launch_bind_reset(const DevCtx &c, int slot, int64_t n_committed, cudaStream_t s,
                              Timer *tm) {
  if (tm) tm->begin(K_BIND_RESET, s);
  k_bind_reset<<<512, 256, 0, s>>>(c, slot, n_committed);
  if (tm) tm->end(K_BIND_RESET, s);
  return cudaGetLastError();
}

}  // namespace dhs
