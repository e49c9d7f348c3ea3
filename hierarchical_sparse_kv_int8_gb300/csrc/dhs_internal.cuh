// Internal declarations shared by the translation units of libdhs.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>
#include <vector>

#include "../../include/dhs.h"

namespace dhs {

constexpr int kMaxSlots = 256;
constexpr int kMaxKmax = 8;
constexpr int kMaxTopk = 2048;
constexpr int kUploadWords = 4096;  // int32 words carried by one k_upload launch

// Kernel ids (per-kernel timing and device error sites).
enum KernelId {
  K_UPLOAD = 0,
  K_SCORE,
  K_TOPK,
  K_UNION_PROBE,
  K_GATHER,
  K_ATTN,
  K_ATTN_UNION,
  K_COMMIT,
  K_RESIDENCY_CLEAR,
  K_RESIDENCY_FILL,
  K_RESIDENCY_PUBLISH,
  K_BIND_RESET,
  K_COUNT
};
extern const char *const kKernelNames[K_COUNT];

// Device error codes recorded by kernels (first one wins).
enum DeviceCheck {
  DC_OK = 0,
  DC_ROW_RANGE = 1,   // a selected row outside [0, n_r)
  DC_LOC_RANGE = 2,   // a location tag or index outside its tier
  DC_CAPACITY = 3,    // a staging or pool index beyond capacity
  DC_TIMEOUT = 4,     // a bounded wait on copies in flight ran out
  DC_DUPLICATE = 5,   // a row listed twice in one query's selection
};

// Everything a kernel needs to know about the context, passed by value.
struct DevCtx {
  int N, Kmax, k;
  int64_t Sm;
  int64_t Ss;  // row stride of the score buffer: Sm rounded up to 32
  uint32_t kinv;  // ceil(2^32 / k): e / k = umulhi(e, kinv) for e < 8k
  int idx_row;           // H_idx * d_idx bytes per index-key row
  int Hq, Hkv, dqk, dv, row;  // row = bf16 elements per stored row
  int layout;
  int B;
  int W, p, Rd;
  int64_t opt_max;
  float scale_log2;      // softmax scale * log2(e)
  int sms;               // streaming multiprocessors of the device

  // per-slot binding
  const int8_t *const *keys;     // [N] device index keys
  const uint16_t *const *host;   // [N] device-visible host backing
  int64_t *n;                    // [N] committed frontier
  int64_t *ring_first;           // [N]
  int32_t *Kr;                   // [N] queries this round
  int32_t *dom;                  // [N][Kmax] selectable rows per query

  // payload tiers (one pool, four regions)
  uint16_t *hot_data;            // [N][B][row]
  uint16_t *stage;               // [N][Kmax*k][row]
  uint16_t *ring;                // [N][Rd][row]
  uint16_t *opt;                 // [N][opt_max][row]

  // metadata
  int32_t *hot_row, *hot_stamp, *lru;  // [N][B]
  int32_t *hot_map, *opt_map;          // [N][Sm]
  int32_t *opt_list;                   // [N][opt_max]
  int64_t *opt_count;                  // [N]

  // scratch of one round
  int32_t *scores;      // [N][Kmax][Sm]
  int32_t *minmax;      // [N][Kmax][2]: range of each query's scores
  int32_t *uni;         // [N][Kmax*k]
  int4 *uent;           // [N][Kmax*k] per union row u: row, location, mask of the
                        // queries that selected it, 0
  int32_t *miss;        // [N][Kmax*k]
  int32_t *first_occ;   // [N][Kmax*k]
  int32_t *counts;      // [N][4]
  int32_t *promo_dst;   // [N][B]: hot slot taken by miss p (p < P)
  uint32_t *now_bits;   // [N][ceil(B/32)]: hot slots stamped by this tick
  int32_t *lru_next;    // [N][B]: the LRU order being rebuilt
  int32_t *uspill;      // [N][slices][...] union/probe scratch of slices whose
                        // union outgrows shared memory (or nullptr: never)
  int32_t *inst;        // [N][Kmax*k] per-query mode: hot slot a staged entry
                        // also fills, else -1 (written for staged entries only)
  int32_t *topk_last;   // [N][Kmax][k] selection seen by the last resolve
  float *part_o;        // attention partials [N][Kmax][Hq][n_split][dv]
  float *part_ml;       // [N][Kmax][Hq][n_split][2]: max (log2 units), sum
  int32_t *ticket;      // [N][Kmax][Hkv]: finished splits of each attention item
  float *u_part;        // union attention, per (request, kv head) and cluster:
                        // O [C][M][dv], then (m, l) [C][M][2]
  int32_t *u_ticket;    // [N][Hkv]: clusters (or split CTAs) of an item that have finished
  float *tc_part;       // tensor-core union pass, split-KV parts: per item and
                        // split, O [M][dv] then (m, l) [M] (or nullptr: no split)
  unsigned long long *stats;  // counters, see StatIdx
  int32_t *err;               // [2]: code, site
};

enum StatIdx {
  ST_RESOLVE = 0, ST_SEL, ST_UNION, ST_RING, ST_OPT, ST_HOT, ST_MISS, ST_MISS_SEL,
  ST_FETCHED, ST_INSTALL, ST_EVICT, ST_DIRECT, ST_TOPK_RESCAN, ST_COUNT
};

__device__ __forceinline__ void record_error(int32_t *err, int code, int site) {
  if (atomicCAS(err, 0, code) == 0) err[1] = site;
}

__device__ __forceinline__ int loc_tier(int32_t l) { return (l >> DHS_LOC_TIER_SHIFT) & 3; }
__device__ __forceinline__ int loc_index(int32_t l) { return l & DHS_LOC_INDEX_MASK; }
__device__ __forceinline__ int32_t make_loc(int tier, int idx) {
  return (int32_t)((tier << DHS_LOC_TIER_SHIFT) | idx);
}

// Device address of the payload row a location names, or nullptr when the
// tag or index is out of range (the caller records DC_LOC_RANGE).
__device__ __forceinline__ const uint16_t *loc_row(const DevCtx &c, int r, int32_t l) {
  int tier = loc_tier(l), idx = loc_index(l);
  size_t row = (size_t)c.row;
  switch (tier) {
    case DHS_LOC_RING:
      return idx < c.Rd ? c.ring + ((size_t)r * c.Rd + idx) * row : nullptr;
    case DHS_LOC_OPT:
      return idx < c.opt_max ? c.opt + ((size_t)r * c.opt_max + idx) * row : nullptr;
    case DHS_LOC_HOT:
      return idx < c.B ? c.hot_data + ((size_t)r * c.B + idx) * row : nullptr;
    default:
      return idx < c.Kmax * c.k ? c.stage + ((size_t)r * c.Kmax * c.k + idx) * row : nullptr;
  }
}

// Every kernel of the library asks for the same L1/shared-memory split (all
// shared), so consecutive kernels never make the SMs change their carveout.
template <typename F>
cudaError_t same_carveout(F *func) {
  return cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared);
}

// Raise a kernel's dynamic shared-memory limit to at least `bytes` (cached);
// the first call also sets the common carveout.
template <typename F>
cudaError_t ensure_smem(F *func, size_t bytes, size_t &granted) {
  if (granted == 0) {
    cudaError_t e0 = same_carveout(func);
    if (e0 != cudaSuccess) return e0;
    if (bytes == 0) granted = 1;
  }
  if (bytes <= granted) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) granted = bytes;
  return e;
}
constexpr size_t kMaxDynSmem = 226 * 1024;  // leaves room for static shared memory

// Launch with programmatic stream serialization: the kernel's CTAs may be
// placed while the preceding launch on the stream finishes; the kernel orders
// itself after it with pdl_wait().  Kernels launched this way call
// pdl_trigger() only after pdl_wait(), so when one starts, every launch before
// its immediate predecessor has completed.
template <typename... P, typename... A>
cudaError_t launch_pdl(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       A &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  // the stream's priority travels with the launch (also into captured graphs)
  int prio = 0;
  if (cudaStreamGetPriority(s, &prio) != cudaSuccess) prio = 0;
  at[1].id = cudaLaunchAttributePriority;
  at[1].val.priority = prio;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<A>(args)...);
}
// An ordinary launch (no early start) with the stream's priority.
template <typename... P, typename... A>
cudaError_t launch_prio(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                        A &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  int prio = 0;
  if (cudaStreamGetPriority(s, &prio) != cudaSuccess) prio = 0;
  at[0].id = cudaLaunchAttributePriority;
  at[0].val.priority = prio;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<A>(args)...);
}

// Words uploaded by k_upload (kernel parameter, <= 16 KB).  The indexer
// launch carries its control words here and, when they fit, the queries'
// index rows after them (at a 16-byte aligned word offset).
struct __align__(16) UploadWords {
  int32_t w[kUploadWords];
};
__host__ __device__ inline int ctl_qidx_word(int N, int Kmax) { return (N + N * Kmax + 3) & ~3; }

// ---- launchers (each returns the cudaGetLastError of its launch) -------
cudaError_t launch_upload(int32_t *dst, const int32_t *words, int n, cudaStream_t s);
// q_idx: device index rows, or nullptr with q_inline holding them on the host
// (carried in the launch parameters; ctl_qidx_word + bytes/4 <= kUploadWords).
// active_queries: sum of K_r this round; topk_pass: DHS_TOPK_* of the config.
cudaError_t launch_select(const DevCtx &c, const int8_t *q_idx, const int8_t *q_inline,
                          int32_t *topk_out, int max_dom, const int32_t *ctl_words,
                          int active_queries, int topk_pass, cudaStream_t s, class Timer *tm);
cudaError_t launch_resolve(const DevCtx &c, const int32_t *topk, int32_t *loc_out,
                           int shared, int gather, int tick, cudaStream_t s, class Timer *tm);
// The shared host gather alone (launch_resolve with gather = 1 or 2 issues
// the union/probe and then this; 2 when the per-query attention pass follows,
// which the gather then releases early: `early`).
cudaError_t launch_gather(const DevCtx &c, const int32_t *topk, int32_t *loc_out, int shared,
                          int tick, cudaStream_t s, class Timer *tm, bool early);
// int32 words of union/probe scratch per request slot (0: none needed).
size_t union_spill_ints_per_request(const DevCtx &c);
cudaError_t launch_uattn(const DevCtx &c, const uint16_t *q, const uint16_t *block,
                         uint16_t *out, float *lse, cudaStream_t s, class Timer *tm);
bool uattn_supported(const DevCtx &c);
// The union pass on the fifth-generation tensor cores (128-dim heads, at most
// 128 (query, head) pairs per kv head): one CTA per (request, kv head).
bool uattn_tc_supported(const DevCtx &c);
// split: CTAs per (request, kv head) item (split-KV), 0 = automatic (up to
// the SM count, at most five).
cudaError_t launch_uattn_tc(const DevCtx &c, const uint16_t *q, const uint16_t *block,
                            uint16_t *out, float *lse, cudaStream_t s, class Timer *tm,
                            int split = 0);
// floats of the split-KV scratch of a context (tc_part)
size_t uattn_tc_part_floats(const DevCtx &c);
size_t uattn_partial_floats(const DevCtx &c);
cudaError_t launch_attend(const DevCtx &c, const uint16_t *q, const uint16_t *block,
                          const int32_t *loc, uint16_t *out, float *lse, int n_split,
                          cudaStream_t s, class Timer *tm);
cudaError_t launch_commit(const DevCtx &c, const int32_t *aux_words, cudaStream_t s,
                          class Timer *tm);
// aux: a_r and n_r per slot, as launch_commit's first three words.
// rows/keys: [N][cmax][row] bf16 and [N][cmax][idx_row] int8 (keys may be
// nullptr); aux: completed rows, first row (lo, hi), active, per slot.
cudaError_t launch_commit_rows(const DevCtx &c, const uint16_t *rows, const int8_t *keys, int cmax,
                               const int32_t *aux_words, cudaStream_t s, class Timer *tm);
cudaError_t launch_append_keys(const DevCtx &c, const int8_t *block, const int32_t *aux_words,
                               cudaStream_t s);
cudaError_t launch_residency(const DevCtx &c, int slot, int64_t old_count, int64_t new_count,
                             cudaStream_t s, class Timer *tm);
cudaError_t launch_bind_reset(const DevCtx &c, int slot, int64_t n_committed, cudaStream_t s,
                              class Timer *tm);

// Attention split heuristic and scratch size (floats) for a context.
int attn_splits(const DevCtx &c, int active_queries);
size_t attn_partial_floats(const DevCtx &c, int max_splits);
size_t union_smem_bytes(const DevCtx &c);
bool attn_shape_supported(int dqk, int dv, int layout);

// Per-kernel CUDA-event timing (host side).
class Timer {
 public:
  bool enabled = false;
  void begin(int id, cudaStream_t s);
  void end(int id, cudaStream_t s);
  void collect(int64_t *launches, double *ms);  // synchronises pending events
  void reset();
  // Event pairs recorded while the stream was being captured into a CUDA
  // graph are external event-record nodes; after each launch of that graph,
  // accumulate_graph() adds their durations to the totals.
  void accumulate_graph();
  ~Timer();

 private:
  struct Pending { int id; cudaEvent_t a, b; };
  std::vector<Pending> pending_;
  std::vector<Pending> graph_pairs_;
  bool open_captured_ = false;
  std::vector<cudaEvent_t> pool_;
  int64_t launches_[K_COUNT] = {};
  double ms_[K_COUNT] = {};
  cudaEvent_t take();
  void drain(size_t keep);
  int open_id_ = -1;
  cudaEvent_t open_a_ = nullptr;
};

}  // namespace dhs
