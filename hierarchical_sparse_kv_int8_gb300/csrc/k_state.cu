// State updates around the verification round: commit, residency, binding.
//
// "Adaptive DHiSparse", eq. (7), (9), (10): block rows live in a draft ring at
// phi(r, t) = r R_d + (t mod R_d) (written by the attention launch, k_attn.cu);
// commit keeps the accepted prefix.  This file holds commit and the residency
// and binding updates between rounds.
#include "dhs_internal.cuh"
#include "ptx_util.cuh"

namespace dhs {

// ---------------------------------------------------------------- commit
// aux[r*4 + 0] = a_r, aux[r*4 + 1..2] = n_r before the commit (lo, hi words).
__global__ void __launch_bounds__(256) k_commit(const DevCtx c, const __grid_constant__ UploadWords aux) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.y;
  const int a = aux.w[r * 4 + 0];
  const int64_t n_old = (int64_t)(uint32_t)aux.w[r * 4 + 1] | ((int64_t)aux.w[r * 4 + 2] << 32);
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
  if (blockIdx.x == 0 && threadIdx.x == 0 && aux.w[r * 4 + 3]) {
    c.n[r] = n_old + a;
    c.Kr[r] = 0;
  }
}

cudaError_t launch_commit(const DevCtx &c, const int32_t *aux_words, cudaStream_t s, Timer *tm) {
  UploadWords aux;
  for (int i = 0; i < c.N * 4; ++i) aux.w[i] = aux_words[i];
  static bool carve_k_commit = false;
  if (!carve_k_commit) {
    same_carveout(k_commit);
    carve_k_commit = true;
  }
  if (tm) tm->begin(K_COMMIT, s);
  cudaError_t e = launch_pdl(k_commit, dim3(1, c.N), dim3(256), 0, s, c, aux);
  if (tm) tm->end(K_COMMIT, s);
  return e;
}

// ---------------------------------------------------------------- commit of completed stored rows
// aux[r*4 + 0] = rows completed, aux[r*4 + 1..2] = the first of them (lo, hi
// words), aux[r*4 + 3] = slot active.  Row i of slot r's `rows` (and key row
// i of `keys`, when given) becomes stored row first + i of the host backing
// (and of the bound key buffer); the history then ends after the last of
// them, and the ring holds no history row of the slot.
__global__ void __launch_bounds__(256) k_commit_rows(const DevCtx c, const uint16_t *__restrict__ rows,
                                                     const int8_t *__restrict__ keys, int cmax,
                                                     const __grid_constant__ UploadWords aux) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.y;
  const int cnt = aux.w[r * 4 + 0];
  const int64_t first = (int64_t)(uint32_t)aux.w[r * 4 + 1] | ((int64_t)aux.w[r * 4 + 2] << 32);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nv = (c.row * 2) >> 4, nk = c.idx_row >> 4;
  uint16_t *host = const_cast<uint16_t *>(c.host[r]);
  int8_t *kdst = const_cast<int8_t *>(c.keys[r]);
  for (int i = wid; i < cnt; i += 8) {
    const uint4 *src = reinterpret_cast<const uint4 *>(rows + ((size_t)r * cmax + i) * c.row);
    uint4 *dst = reinterpret_cast<uint4 *>(host + (size_t)(first + i) * c.row);
    for (int v = lane; v < nv; v += 32) dst[v] = src[v];
    if (keys) {
      const uint4 *ks = reinterpret_cast<const uint4 *>(keys + ((size_t)r * cmax + i) * c.idx_row);
      uint4 *kd = reinterpret_cast<uint4 *>(kdst + (size_t)(first + i) * c.idx_row);
      for (int v = lane; v < nk; v += 32) kd[v] = ks[v];
    }
  }
  if (threadIdx.x == 0 && aux.w[r * 4 + 3]) {
    c.n[r] = first + cnt;
    c.ring_first[r] = first + cnt;
    c.Kr[r] = 0;
  }
}

cudaError_t launch_commit_rows(const DevCtx &c, const uint16_t *rows, const int8_t *keys, int cmax,
                               const int32_t *aux_words, cudaStream_t s, Timer *tm) {
  UploadWords aux;
  for (int i = 0; i < c.N * 4; ++i) aux.w[i] = aux_words[i];
  static bool carved = false;
  if (!carved) {
    same_carveout(k_commit_rows);
    carved = true;
  }
  if (tm) tm->begin(K_COMMIT, s);
  cudaError_t e = launch_pdl(k_commit_rows, dim3(1, c.N), dim3(256), 0, s, c, rows, keys, cmax, aux);
  if (tm) tm->end(K_COMMIT, s);
  return e;
}

// ---------------------------------------------------------------- index keys of kept rows
// aux[r*4 + 0] = a_r, aux[r*4 + 1..2] = n_r (lo, hi words): key rows 0..a_r-1
// of slot r's block go to rows n_r .. n_r + a_r - 1 of its bound key buffer
// (16-byte vectors when a key row is a multiple of 16 bytes; both buffers are
// 16-byte aligned).
__global__ void __launch_bounds__(256) k_append_keys(const DevCtx c, const int8_t *__restrict__ block,
                                                     const __grid_constant__ UploadWords aux) {
  const int r = blockIdx.y;
  const int a = aux.w[r * 4 + 0];
  if (a == 0) return;
  const int64_t n = (int64_t)(uint32_t)aux.w[r * 4 + 1] | ((int64_t)aux.w[r * 4 + 2] << 32);
  const size_t bytes = (size_t)a * c.idx_row;
  const int8_t *src = block + (size_t)r * c.Kmax * c.idx_row;
  int8_t *dst = const_cast<int8_t *>(c.keys[r]) + (size_t)n * c.idx_row;
  if ((c.idx_row & 15) == 0) {
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
    for (size_t i = threadIdx.x; i < bytes / 16; i += blockDim.x) d4[i] = s4[i];
  } else {
    for (size_t i = threadIdx.x; i < bytes; i += blockDim.x) dst[i] = src[i];
  }
}

cudaError_t launch_append_keys(const DevCtx &c, const int8_t *block, const int32_t *aux_words,
                               cudaStream_t s) {
  UploadWords aux;
  for (int i = 0; i < c.N * 4; ++i) aux.w[i] = aux_words[i];
  static bool carved = false;
  if (!carved) {
    same_carveout(k_append_keys);
    carved = true;
  }
  return launch_prio(k_append_keys, dim3(1, c.N), dim3(256), 0, s, c, block, aux);
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
