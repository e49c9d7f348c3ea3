// Host side of libdhs: context lifetime, argument checks, host mirrors of the
// per-request round state, and the launch sequence of each C-ABI call.
#include "dhs_internal.cuh"

#include <math.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <vector>

namespace dhs {

const char *const kKernelNames[K_COUNT] = {
    "upload",          "index_score",    "topk",           "union_probe",
    "gather",          "attn",           "attn_union",     "commit",
    "residency_clear", "residency_fill", "residency_publish", "bind_reset"};

// ---------------------------------------------------------------- Timer
cudaEvent_t Timer::take() {
  if (!pool_.empty()) {
    cudaEvent_t e = pool_.back();
    pool_.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}
static bool stream_capturing(cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &st) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return st == cudaStreamCaptureStatusActive;
}
void Timer::begin(int id, cudaStream_t s) {
  if (!enabled) return;
  open_id_ = id;
  open_captured_ = stream_capturing(s);
  if (open_captured_) {
    cudaEventCreate(&open_a_);
    cudaEventRecordWithFlags(open_a_, s, cudaEventRecordExternal);
  } else {
    open_a_ = take();
    cudaEventRecord(open_a_, s);
  }
}
void Timer::end(int id, cudaStream_t s) {
  if (!enabled || open_id_ != id || !open_a_) return;
  cudaEvent_t b = nullptr;
  if (open_captured_) {
    cudaEventCreate(&b);
    cudaEventRecordWithFlags(b, s, cudaEventRecordExternal);
    graph_pairs_.push_back({id, open_a_, b});
  } else {
    b = take();
    cudaEventRecord(b, s);
    pending_.push_back({id, open_a_, b});
  }
  open_a_ = nullptr;
  open_id_ = -1;
  if (pending_.size() > 8192) drain(1024);
}
void Timer::accumulate_graph() {
  for (auto &p : graph_pairs_) {
    cudaEventSynchronize(p.b);
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, p.a, p.b) == cudaSuccess) {
      launches_[p.id] += 1;
      ms_[p.id] += ms;
    } else {
      cudaGetLastError();
    }
  }
}
void Timer::drain(size_t keep) {
  size_t n = pending_.size() > keep ? pending_.size() - keep : 0;
  for (size_t i = 0; i < n; ++i) {
    Pending &p = pending_[i];
    cudaEventSynchronize(p.b);
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, p.a, p.b) == cudaSuccess) {
      launches_[p.id] += 1;
      ms_[p.id] += ms;
    }
    pool_.push_back(p.a);
    pool_.push_back(p.b);
  }
  pending_.erase(pending_.begin(), pending_.begin() + n);
}
void Timer::collect(int64_t *launches, double *ms) {
  drain(0);
  for (int i = 0; i < K_COUNT; ++i) {
    launches[i] = launches_[i];
    ms[i] = ms_[i];
  }
}
void Timer::reset() {
  drain(0);
  for (int i = 0; i < K_COUNT; ++i) {
    launches_[i] = 0;
    ms_[i] = 0.0;
  }
}
Timer::~Timer() {
  for (auto &p : graph_pairs_) {
    cudaEventDestroy(p.a);
    cudaEventDestroy(p.b);
  }
  for (auto &p : pending_) {
    cudaEventDestroy(p.a);
    cudaEventDestroy(p.b);
  }
  for (auto e : pool_) cudaEventDestroy(e);
}

}  // namespace dhs

using namespace dhs;

enum Phase { PH_IDLE = 0, PH_SELECTED, PH_RESOLVED, PH_ATTENDED };

// Verification staging shared by the sources of a layer group.  Arena i is
// taken by one context at a time: its dhs_resolve claims it (after the
// previous user's attention readers, through `released`), its dhs_attend
// calls read it and record `released` after their kernels.
struct dhs_arenas {
  int chi = 0, N = 0, Kmax = 0, k = 0, row = 0;
  uint16_t *base = nullptr;
  std::vector<cudaEvent_t> released;
  std::vector<dhs_ctx *> owner;   // context whose resolve last filled the arena
  std::vector<char> unread;       // that resolve's attention not yet issued
  int users = 0;                  // contexts created on these arenas
};

struct Snapshot {
  std::vector<void *> bufs;
  std::vector<int64_t> n, tok, ring_first, opt_count;
  std::vector<int32_t> K;
  int64_t tick;
  int phase;
};

struct dhs_ctx {
  dhs_config cfg;
  DevCtx d;
  int n_split = 1;
  int device = 0;
  bool fused = false;      // shared retrieval attends with the union pass
  int last_shared = 0;     // mode of the last dhs_resolve
  std::vector<void *> allocs;
  // host mirrors (n: history rows; tok: committed token positions, = n when m = 1)
  int m = 1;
  std::vector<int64_t> n, tok, ring_first, opt_count;
  std::vector<int32_t> K;
  std::vector<char> bound;
  std::vector<const void *> host_ptr;
  std::vector<const int8_t *> key_ptr;
  int64_t tick = 0;
  int phase = PH_IDLE;
  Timer timer;
  std::vector<Snapshot> snaps;
  // device staging for dhs_round_host
  int8_t *rh_qidx = nullptr;
  uint16_t *rh_q = nullptr, *rh_block = nullptr, *rh_out = nullptr;
  float *rh_lse = nullptr;
  int32_t *rh_topk = nullptr, *rh_loc = nullptr;
  // device arrays of per-slot pointers
  const int8_t **d_keys = nullptr;
  const uint16_t **d_host = nullptr;
  const char *last_error = "";
  // layer groups: staging from shared arenas, calls ordered across streams
  dhs_arenas *arenas = nullptr;
  int arena = -1;
  int role = DHS_ROLE_FULL;
  cudaEvent_t last_ev = nullptr;  // recorded after every call's work
  bool last_valid = false;
  // dhs_round: request groups on internal streams
  int groups = 1;
  std::vector<cudaStream_t> gstream;
  std::vector<cudaEvent_t> gevent;  // [0]: fork; [1 + g]: group g done
  std::vector<cudaEvent_t> gsel;    // [g]: group g's selection issued
};

namespace {

template <typename T>
cudaError_t dalloc(dhs_ctx *c, T **p, size_t count) {
  void *q = nullptr;
  size_t bytes = count * sizeof(T);
  if (bytes == 0) bytes = 16;
  cudaError_t e = cudaMalloc(&q, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e;
  }
  c->allocs.push_back(q);
  *p = static_cast<T *>(q);
  return cudaSuccess;
}

void free_all(dhs_ctx *c) {
  for (void *p : c->allocs) cudaFree(p);
  c->allocs.clear();
  for (auto st : c->gstream) cudaStreamDestroy(st);
  c->gstream.clear();
  for (auto ev : c->gevent) cudaEventDestroy(ev);
  c->gevent.clear();
  for (auto ev : c->gsel) cudaEventDestroy(ev);
  c->gsel.clear();
  if (c->last_ev) cudaEventDestroy(c->last_ev);
  c->last_ev = nullptr;
  for (auto &s : c->snaps)
    for (void *p : s.bufs) cudaFree(p);
  c->snaps.clear();
}

// Device address of page-locked, mapped host memory, or nullptr for any other
// pointer (pageable host memory, device memory).
void *mapped_ptr(const void *h) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

struct BufDesc {
  void *ptr;
  size_t bytes;
};

BufDesc buffer_desc(const dhs_ctx *c, int which) {
  const DevCtx &d = c->d;
  const size_t N = d.N, B = d.B, KK = (size_t)d.Kmax * d.k, row2 = (size_t)d.row * 2;
  switch (which) {
    case DHS_BUF_HOT_ROW: return {d.hot_row, N * B * 4};
    case DHS_BUF_HOT_STAMP: return {d.hot_stamp, N * B * 4};
    case DHS_BUF_HOT_DATA: return {d.hot_data, N * B * row2};
    case DHS_BUF_RING: return {d.ring, N * d.Rd * row2};
    case DHS_BUF_STAGE: return {d.stage, N * KK * row2};
    case DHS_BUF_OPT: return {d.opt, N * d.opt_max * row2};
    case DHS_BUF_UNION: return {d.uni, N * KK * 4};
    case DHS_BUF_MISS: return {d.miss, N * KK * 4};
    case DHS_BUF_COUNTS: return {d.counts, N * 16};
    case DHS_BUF_LRU: return {d.lru, N * B * 4};
    case DHS_BUF_FRONTIER: return {d.n, N * 8};
    case DHS_BUF_HOT_MAP: return {d.hot_map, N * d.Sm * 4};
    case DHS_BUF_OPT_MAP: return {d.opt_map, N * d.Sm * 4};
    case DHS_BUF_SCORES: return {d.scores, N * d.Kmax * d.Ss * 4};
    default: return {nullptr, 0};
  }
}

// Buffers that make up the mutable state (snapshot / restore).
const int kStateBufs[] = {DHS_BUF_HOT_ROW, DHS_BUF_HOT_STAMP, DHS_BUF_HOT_DATA, DHS_BUF_RING,
                          DHS_BUF_OPT,     DHS_BUF_LRU,       DHS_BUF_FRONTIER, DHS_BUF_HOT_MAP,
                          DHS_BUF_OPT_MAP};

// Record the CUDA error behind a DHS_ERR_CUDA return.
int cuda_fail(dhs_ctx *c, cudaError_t e) {
  c->last_error = cudaGetErrorString(e);
  cudaGetLastError();
  return DHS_ERR_CUDA;
}

int upload_words(dhs_ctx *c, int32_t *dst, const std::vector<int32_t> &w, cudaStream_t s) {
  for (size_t off = 0; off < w.size(); off += kUploadWords) {
    int n = (int)std::min<size_t>(kUploadWords, w.size() - off);
    cudaError_t e_ = launch_upload(dst + off, w.data() + off, n, s);
    if (e_ != cudaSuccess) return cuda_fail(c, e_);
  }
  return DHS_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// A context on shared arenas may be driven from several streams (its
// gathers on a copy stream, its attention on a compute stream): every call
// first waits for the work of the context's previous call, wherever it ran,
// and records the point its own work ends.
int order_enter(dhs_ctx *c, cudaStream_t s) {
  if (c->arenas && c->last_valid && cudaStreamWaitEvent(s, c->last_ev, 0) != cudaSuccess)
    return cuda_fail(c, cudaGetLastError());
  return DHS_OK;
}
int order_leave(dhs_ctx *c, cudaStream_t s) {
  if (!c->arenas) return DHS_OK;
  if (cudaEventRecord(c->last_ev, s) != cudaSuccess) return cuda_fail(c, cudaGetLastError());
  c->last_valid = true;
  return DHS_OK;
}


}  // namespace

extern "C" {

const char *dhs_last_error(const dhs_ctx *c) { return c ? c->last_error : ""; }

const char *dhs_strerror(int code) {
  switch (code) {
    case DHS_OK: return "ok";
    case DHS_ERR_INVALID: return "invalid argument or call order";
    case DHS_ERR_OOM: return "out of device or pinned memory";
    case DHS_ERR_CAPACITY: return "request exceeds a configured capacity";
    case DHS_ERR_CUDA: return "CUDA runtime error";
    case DHS_ERR_DEVICE_CHECK: return "a kernel found an out-of-range index or a wait ran out";
    case DHS_ERR_TIMEOUT: return "timed out";
    default: return "unknown error";
  }
}

int32_t dhs_kernel_count(void) { return K_COUNT; }
const char *dhs_kernel_name(int32_t id) {
  return (id >= 0 && id < K_COUNT) ? kKernelNames[id] : "?";
}

}  // extern "C"

namespace {
int create_impl(const dhs_config *cfg, dhs_arenas *arenas, int arena, int role, dhs_ctx **out) {
  if (!cfg || !out) return DHS_ERR_INVALID;
  *out = nullptr;
  if (role != DHS_ROLE_FULL && role != DHS_ROLE_FOLLOWER) return DHS_ERR_INVALID;
  const dhs_config &g = *cfg;
  if (g.n_slots < 1 || g.n_slots > kMaxSlots || g.k_max < 1 || g.k_max > kMaxKmax ||
      g.topk < 32 || g.topk > kMaxTopk || g.topk % 32 || g.s_max < 1 || g.s_max > (1 << 27) ||
      g.idx_heads < 1 || g.idx_dim < 1 || (g.idx_heads * g.idx_dim) % 16 ||
      g.idx_heads * g.idx_dim > 1024 || g.q_heads < 1 || g.kv_heads < 1 ||
      g.q_heads % g.kv_heads || g.q_heads / g.kv_heads > 16 || g.q_heads > 128 || g.budget < 1 ||
      g.budget > 65535 || g.ring_window < 1 || g.page_rows < 1 || g.opt_rows_max < 0 ||
      g.opt_rows_max > g.s_max || g.attn_pass < DHS_ATTN_AUTO || g.attn_pass > DHS_ATTN_UNION_MMA ||
      g.topk_pass < DHS_TOPK_AUTO || g.topk_pass > DHS_TOPK_ROW || g.round_groups < 0 ||
      g.round_groups > g.n_slots || g.round_groups > 16 || g.tokens_per_row < 0 ||
      g.tokens_per_row > 64)
    return DHS_ERR_INVALID;
  if (g.kv_layout != DHS_KV_SPLIT && g.kv_layout != DHS_KV_LATENT) return DHS_ERR_INVALID;
  if (g.kv_layout == DHS_KV_LATENT && (g.kv_heads != 1 || g.v_dim > g.qk_dim))
    return DHS_ERR_INVALID;
  if (!attn_shape_supported(g.qk_dim, g.v_dim, g.kv_layout)) return DHS_ERR_INVALID;
  const int row = g.kv_layout == DHS_KV_LATENT ? g.qk_dim : g.kv_heads * (g.qk_dim + g.v_dim);
  if (row * 2 > 2048) return DHS_ERR_INVALID;
  const int64_t Rd = (int64_t)g.page_rows *
                     ((g.ring_window + g.page_rows - 1 + g.k_max + g.page_rows - 1) / g.page_rows);
  if (Rd > DHS_LOC_INDEX_MASK) return DHS_ERR_INVALID;
  if (arenas && (arena < 0 || arena >= arenas->chi || arenas->N != g.n_slots ||
                 arenas->Kmax != g.k_max || arenas->k != g.topk || arenas->row != row))
    return DHS_ERR_INVALID;

  dhs_ctx *c = new (std::nothrow) dhs_ctx();
  if (!c) return DHS_ERR_OOM;
  c->cfg = g;
  c->arenas = arenas;
  c->arena = arenas ? arena : -1;
  c->role = role;
  cudaGetDevice(&c->device);
  DevCtx &d = c->d;
  memset(&d, 0, sizeof(d));
  d.N = g.n_slots;
  d.Kmax = g.k_max;
  d.k = g.topk;
  d.Sm = g.s_max;
  d.Ss = (g.s_max + 31) / 32 * 32;
  d.kinv = 0xFFFFFFFFu / (uint32_t)g.topk + 1u;
  d.idx_row = g.idx_heads * g.idx_dim;
  d.Hq = g.q_heads;
  d.Hkv = g.kv_heads;
  d.dqk = g.qk_dim;
  d.dv = g.v_dim;
  d.row = row;
  d.layout = g.kv_layout;
  d.B = g.budget;
  d.W = g.ring_window;
  d.p = g.page_rows;
  d.Rd = (int)Rd;
  d.opt_max = g.opt_rows_max;
  const float scale = g.softmax_scale > 0.f ? g.softmax_scale : 1.0f / sqrtf((float)g.qk_dim);
  d.scale_log2 = scale * 1.4426950408889634f;
  if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess ||
      d.sms < 1) {
    cudaGetLastError();
    d.sms = 1;
  }
  if (union_smem_bytes(d) > kMaxDynSmem) {
    delete c;
    return DHS_ERR_CAPACITY;
  }
  c->n_split = attn_splits(d, d.N * d.Kmax);
  {
    const bool can = uattn_supported(d);
    const double pq_bytes = (double)d.N * d.Kmax * (d.k + d.Kmax) * row * 2;
    if ((g.attn_pass == DHS_ATTN_UNION || g.attn_pass == DHS_ATTN_UNION_MMA) && !can) {
      delete c;
      return DHS_ERR_INVALID;
    }
    // AUTO: the union pass for 128-dim heads once the per-query pass would
    // stream more than 128 MiB; latent (MLA) rows keep the per-query pass,
    // which measured 3.6x faster on them (0.46 against 1.69 ms at S = 512K)
    c->fused = g.attn_pass == DHS_ATTN_UNION || g.attn_pass == DHS_ATTN_UNION_MMA ||
               (g.attn_pass == DHS_ATTN_AUTO && can && d.dqk == 128 &&
                pq_bytes > 128.0 * 1024 * 1024);
  }

  const size_t N = d.N, KK = (size_t)d.Kmax * d.k, B = d.B, R = row;
  cudaError_t e = cudaSuccess;
#define ALLOC(ptr, count) \
  if (e == cudaSuccess) e = dalloc(c, &(ptr), (count))
  uint16_t *pool = nullptr;
  // (a context on shared arenas stages its misses in its arena instead)
  const size_t own_stage = arenas ? 0 : KK;
  const size_t pool_rows = N * (B + own_stage + (size_t)d.Rd + (size_t)d.opt_max);
  ALLOC(pool, pool_rows * R);
  if (e == cudaSuccess) {
    d.hot_data = pool;
    d.stage = arenas ? arenas->base + (size_t)arena * N * KK * R : d.hot_data + N * B * R;
    d.ring = d.hot_data + N * (B + own_stage) * R;
    d.opt = d.ring + N * d.Rd * R;
  }
  ALLOC(c->d_keys, N);
  ALLOC(c->d_host, N);
  ALLOC(d.n, N);
  ALLOC(d.ring_first, N);
  ALLOC(d.Kr, N);
  ALLOC(d.dom, N * d.Kmax);
  ALLOC(d.hot_row, N * B);
  ALLOC(d.hot_stamp, N * B);
  ALLOC(d.lru, N * B);
  ALLOC(d.hot_map, N * (size_t)d.Sm);
  ALLOC(d.opt_map, N * (size_t)d.Sm);
  ALLOC(d.opt_list, N * (size_t)std::max<int64_t>(1, d.opt_max));
  ALLOC(d.opt_count, N);
  // a follower never scores (its positions come from a producer)
  ALLOC(d.scores, role == DHS_ROLE_FOLLOWER ? 4 : N * d.Kmax * (size_t)d.Ss);
  ALLOC(d.minmax, N * d.Kmax * 2);
  ALLOC(d.uni, N * KK);
  ALLOC(d.uent, N * KK);
  ALLOC(d.miss, N * KK);
  ALLOC(d.first_occ, N * KK);
  ALLOC(d.counts, N * 4);
  ALLOC(d.promo_dst, N * B);
  ALLOC(d.now_bits, N * (size_t)((B + 31) / 32));
  ALLOC(d.lru_next, N * B);
  ALLOC(d.inst, N * KK);
  if (union_spill_ints_per_request(d) > 0) ALLOC(d.uspill, N * union_spill_ints_per_request(d));
  const size_t pf = attn_partial_floats(d, c->n_split);
  ALLOC(d.part_o, c->n_split > 1 ? pf : 1);
  ALLOC(d.part_ml, c->n_split > 1 ? N * d.Kmax * d.Hq * c->n_split * 2 : 1);
  ALLOC(d.ticket, N * d.Kmax * d.Hkv);
  ALLOC(d.u_part, c->fused ? uattn_partial_floats(d) : 1);
  ALLOC(d.u_ticket, N * d.Hkv);
  if (c->fused && uattn_tc_supported(d)) ALLOC(d.tc_part, uattn_tc_part_floats(d));
  ALLOC(d.stats, ST_COUNT);
  ALLOC(d.err, 2);
  ALLOC(c->rh_qidx, N * d.Kmax * d.idx_row);
  ALLOC(c->rh_q, N * d.Kmax * d.Hq * d.dqk);
  ALLOC(c->rh_block, N * d.Kmax * R);
  ALLOC(c->rh_out, N * d.Kmax * d.Hq * d.dv);
  ALLOC(c->rh_lse, N * d.Kmax * d.Hq);
  ALLOC(c->rh_topk, N * KK);
  ALLOC(c->rh_loc, N * KK);
#undef ALLOC
  if (e != cudaSuccess) {
    free_all(c);
    delete c;
    return DHS_ERR_OOM;
  }
  d.keys = c->d_keys;
  d.host = c->d_host;
  e = cudaMemset(c->d_keys, 0, N * sizeof(void *));
  if (e == cudaSuccess) e = cudaMemset(c->d_host, 0, N * sizeof(void *));
  if (e == cudaSuccess) e = cudaMemset(d.Kr, 0, N * 4);
  if (e == cudaSuccess) e = cudaMemset(d.n, 0, N * 8);
  if (e == cudaSuccess) e = cudaMemset(d.stats, 0, ST_COUNT * 8);
  if (e == cudaSuccess) e = cudaMemset(d.err, 0, 8);
  if (e == cudaSuccess) e = cudaMemset(d.counts, 0, N * 16);
  if (e == cudaSuccess) e = cudaMemset(d.ticket, 0, N * d.Kmax * d.Hkv * 4);
  if (e == cudaSuccess) e = cudaMemset(d.u_ticket, 0, N * d.Hkv * 4);
  if (e == cudaSuccess) {
    // score ranges start empty; top-k empties each range again after reading it
    std::vector<int32_t> mm((size_t)N * d.Kmax * 2);
    for (size_t i = 0; i < mm.size(); i += 2) {
      mm[i] = INT32_MAX;
      mm[i + 1] = INT32_MIN;
    }
    e = cudaMemcpy(d.minmax, mm.data(), mm.size() * 4, cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) e = cudaMemset(d.opt_count, 0, N * 8);
  if (e == cudaSuccess) e = cudaMemset(pool, 0, pool_rows * R * 2);
  if (e == cudaSuccess && arenas) e = cudaEventCreateWithFlags(&c->last_ev, cudaEventDisableTiming);
  c->groups = g.round_groups > 1 ? g.round_groups : 1;
  // group g's stream has the g-th highest priority: when SMs free up, the
  // pending kernels of earlier groups (retrieval, attention) are placed
  // before later groups' indexer CTAs
  int prio_least = 0, prio_greatest = 0;
  if (e == cudaSuccess && c->groups > 1)
    e = cudaDeviceGetStreamPriorityRange(&prio_least, &prio_greatest);
  for (int i = 0; e == cudaSuccess && c->groups > 1 && i < c->groups; ++i) {
    cudaStream_t st = nullptr;
    e = cudaStreamCreateWithPriority(&st, cudaStreamNonBlocking,
                                     std::min(prio_least, prio_greatest + i));
    if (e == cudaSuccess) c->gstream.push_back(st);
  }
  for (int i = 0; e == cudaSuccess && c->groups > 1 && i <= c->groups; ++i) {
    cudaEvent_t ev = nullptr;
    e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e == cudaSuccess) c->gevent.push_back(ev);
  }
  for (int i = 0; e == cudaSuccess && c->groups > 1 && i < c->groups; ++i) {
    cudaEvent_t ev = nullptr;
    e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e == cudaSuccess) c->gsel.push_back(ev);
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    free_all(c);
    delete c;
    return DHS_ERR_CUDA;
  }
  if (arenas) arenas->users += 1;
  c->m = g.tokens_per_row > 1 ? g.tokens_per_row : 1;
  c->n.assign(N, 0);
  c->tok.assign(N, 0);
  c->ring_first.assign(N, 0);
  c->opt_count.assign(N, 0);
  c->K.assign(N, 0);
  c->bound.assign(N, 0);
  c->host_ptr.assign(N, nullptr);
  c->key_ptr.assign(N, nullptr);
  *out = c;
  return DHS_OK;
}
}  // namespace

extern "C" {

int dhs_create(const dhs_config *cfg, dhs_ctx **out) {
  return create_impl(cfg, nullptr, -1, DHS_ROLE_FULL, out);
}

int dhs_create_on_arena(const dhs_config *cfg, dhs_arenas *arenas, int32_t arena, int32_t role,
                        dhs_ctx **out) {
  if (!arenas) return DHS_ERR_INVALID;
  return create_impl(cfg, arenas, arena, role, out);
}

int dhs_arenas_create(int32_t chi, int32_t n_slots, int32_t k_max, int32_t topk,
                      int32_t row_elems, dhs_arenas **out) {
  if (!out || chi < 1 || chi > 256 || n_slots < 1 || n_slots > kMaxSlots || k_max < 1 ||
      k_max > kMaxKmax || topk < 32 || topk > kMaxTopk || topk % 32 || row_elems < 8 ||
      row_elems * 2 > 2048 || row_elems % 8)
    return DHS_ERR_INVALID;
  *out = nullptr;
  dhs_arenas *a = new (std::nothrow) dhs_arenas();
  if (!a) return DHS_ERR_OOM;
  a->chi = chi;
  a->N = n_slots;
  a->Kmax = k_max;
  a->k = topk;
  a->row = row_elems;
  const size_t bytes = (size_t)chi * n_slots * k_max * topk * row_elems * 2;
  if (cudaMalloc(&a->base, bytes) != cudaSuccess) {
    cudaGetLastError();
    delete a;
    return DHS_ERR_OOM;
  }
  a->released.assign(chi, nullptr);
  a->owner.assign(chi, nullptr);
  a->unread.assign(chi, 0);
  for (int i = 0; i < chi; ++i) {
    if (cudaEventCreateWithFlags(&a->released[i], cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      for (int j = 0; j < i; ++j) cudaEventDestroy(a->released[j]);
      cudaFree(a->base);
      delete a;
      return DHS_ERR_CUDA;
    }
  }
  if (cudaMemset(a->base, 0, bytes) != cudaSuccess) {
    cudaGetLastError();
    for (auto ev : a->released) cudaEventDestroy(ev);
    cudaFree(a->base);
    delete a;
    return DHS_ERR_CUDA;
  }
  *out = a;
  return DHS_OK;
}

int64_t dhs_arenas_bytes(const dhs_arenas *a) {
  return a ? (int64_t)a->chi * a->N * a->Kmax * a->k * a->row * 2 : 0;
}

int dhs_arenas_destroy(dhs_arenas *a) {
  if (!a) return DHS_OK;
  if (a->users > 0) return DHS_ERR_INVALID;  // a context still stages there
  cudaDeviceSynchronize();
  for (auto ev : a->released) cudaEventDestroy(ev);
  cudaFree(a->base);
  delete a;
  return DHS_OK;
}

void dhs_destroy(dhs_ctx *c) {
  if (!c) return;
  cudaDeviceSynchronize();
  if (c->arenas) {
    dhs_arenas *a = c->arenas;
    if (a->owner[c->arena] == c) {
      a->owner[c->arena] = nullptr;
      a->unread[c->arena] = 0;
    }
    a->users -= 1;
  }
  free_all(c);
  delete c;
}

int64_t dhs_ring_rows(const dhs_ctx *c) { return c ? c->d.Rd : 0; }

int64_t dhs_device_bytes(const dhs_ctx *c) {
  if (!c) return 0;
  int64_t total = 0;
  for (int i = 0; i < DHS_BUF_COUNT_; ++i) total += (int64_t)buffer_desc(c, i).bytes;
  return total;
}

int dhs_bind_request(dhs_ctx *c, int32_t slot, const void *host_kv, const int8_t *idx_keys,
                     int64_t n_committed, dhs_stream stream) {
  if (!c || slot < 0 || slot >= c->d.N || !host_kv || !idx_keys || n_committed < 0 ||
      n_committed / c->m > c->d.Sm || !aligned16(host_kv) || !aligned16(idx_keys))
    return DHS_ERR_INVALID;
  const int64_t rows = n_committed / c->m;  // complete stored rows
  if (c->phase != PH_IDLE) return DHS_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void *dev_host = nullptr;
  if (cudaHostGetDevicePointer(&dev_host, const_cast<void *>(host_kv), 0) != cudaSuccess) {
    cudaGetLastError();
    return DHS_ERR_INVALID;  // not page-locked host memory
  }
  if (int rc = order_enter(c, s)) return rc;
  c->host_ptr[slot] = dev_host;
  c->key_ptr[slot] = idx_keys;
  if (cudaMemcpyAsync(c->d_host, c->host_ptr.data(), c->d.N * sizeof(void *),
                      cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(c->d_keys, c->key_ptr.data(), c->d.N * sizeof(void *),
                      cudaMemcpyHostToDevice, s) != cudaSuccess)
    return DHS_ERR_CUDA;
  // the host arrays above are pageable: the copies are staged before returning
  {
    cudaError_t e_ = launch_bind_reset(c->d, slot, rows, s, &c->timer);
    if (e_ != cudaSuccess) return cuda_fail(c, e_);
  }
  c->n[slot] = rows;
  c->tok[slot] = n_committed;
  c->ring_first[slot] = rows;
  c->opt_count[slot] = 0;
  c->K[slot] = 0;
  c->bound[slot] = 1;
  return order_leave(c, s);
}

}  // extern "C"

namespace {
// dhs_select, with the index rows either in device memory (q_idx) or, when
// q_idx is null, on the host (q_inline), carried in the launch parameters.
// The round's K_r and causal domains as control words (K_r of every
// request, then the domain of every (request, query)), after the checks
// shared by dhs_select and dhs_adopt: a new round starts idle; after a
// round's attention (before its commit) another layer of the same source
// may select again (a Reindex consumer) with the same K_r.
int round_words(dhs_ctx *c, const int32_t *k_per_req, const int64_t *pos,
                std::vector<int32_t> &w, int &max_dom, int &active) {
  const DevCtx &d = c->d;
  if (c->phase != PH_IDLE && c->phase != PH_ATTENDED) return DHS_ERR_INVALID;
  w.assign(d.N + d.N * d.Kmax, 0);
  max_dom = 0;
  active = 0;
  for (int r = 0; r < d.N; ++r) {
    const int kr = k_per_req[r];
    if (kr < 0 || kr > d.Kmax || (kr > 0 && !c->bound[r])) return DHS_ERR_INVALID;
    if (c->phase == PH_ATTENDED && kr != c->K[r]) return DHS_ERR_INVALID;
    active += kr;
  }
  for (int r = 0; r < d.N; ++r) {
    const int kr = k_per_req[r];
    w[r] = kr;
    for (int j = 0; j < kr; ++j) {
      // (stored rows complete up to position p: floor((p + 1) / m), eq. (8))
      const int64_t p = pos ? pos[(size_t)r * d.Kmax + j] : c->tok[r] + j;
      const int64_t dom = std::max<int64_t>(0, std::min<int64_t>(c->n[r], (p + 1) / c->m));
      w[d.N + r * d.Kmax + j] = (int32_t)dom;
      max_dom = std::max<int>(max_dom, (int)dom);
    }
  }
  return DHS_OK;
}

int select_impl(dhs_ctx *c, const int8_t *q_idx, const int8_t *q_inline,
                const int32_t *k_per_req, const int64_t *pos, int32_t *topk_out,
                dhs_stream stream) {
  if (c->role == DHS_ROLE_FOLLOWER) return DHS_ERR_INVALID;
  const DevCtx &d = c->d;
  std::vector<int32_t> w;
  int max_dom = 0, active = 0;
  if (int rc = round_words(c, k_per_req, pos, w, max_dom, active)) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (int rc = order_enter(c, s)) return rc;
  {
    cudaError_t e_ = launch_select(d, q_idx, q_inline, topk_out, max_dom, w.data(), active,
                                   c->cfg.topk_pass, s, &c->timer);
    if (e_ != cudaSuccess) return cuda_fail(c, e_);
  }
  for (int r = 0; r < d.N; ++r) c->K[r] = k_per_req[r];
  c->phase = PH_SELECTED;
  return order_leave(c, s);
}

// The context's slots [a, b) as a context of their own: the same buffers,
// every per-slot pointer advanced to slot a, N = b - a.  The launches of a
// request group take it; stats and the error word stay shared.
DevCtx slot_view(const DevCtx &d, int a, int b, int n_split) {
  DevCtx v = d;
  const size_t A = (size_t)a, KK = (size_t)d.Kmax * d.k, B = d.B, R = d.row;
  v.N = b - a;
  v.keys = d.keys + A;
  v.host = d.host + A;
  v.n = d.n + A;
  v.ring_first = d.ring_first + A;
  v.Kr = d.Kr + A;
  v.dom = d.dom + A * d.Kmax;
  v.hot_data = d.hot_data + A * B * R;
  v.stage = d.stage + A * KK * R;
  v.ring = d.ring + A * d.Rd * R;
  v.opt = d.opt + A * (size_t)d.opt_max * R;
  v.hot_row = d.hot_row + A * B;
  v.hot_stamp = d.hot_stamp + A * B;
  v.lru = d.lru + A * B;
  v.hot_map = d.hot_map + A * d.Sm;
  v.opt_map = d.opt_map + A * d.Sm;
  v.opt_list = d.opt_list + A * (size_t)d.opt_max;
  v.opt_count = d.opt_count + A;
  v.scores = d.scores + (d.Ss ? A * d.Kmax * d.Ss : 0);
  v.minmax = d.minmax + A * d.Kmax * 2;
  v.uni = d.uni + A * KK;
  v.uent = d.uent + A * KK;
  v.miss = d.miss + A * KK;
  v.first_occ = d.first_occ + A * KK;
  v.counts = d.counts + A * 4;
  v.promo_dst = d.promo_dst + A * B;
  v.now_bits = d.now_bits + A * ((B + 31) / 32);
  v.lru_next = d.lru_next + A * B;
  v.inst = d.inst + A * KK;
  if (d.uspill) v.uspill = d.uspill + A * union_spill_ints_per_request(d);
  if (d.topk_last) v.topk_last = d.topk_last + A * d.Kmax * d.k;
  if (n_split > 1) {
    v.part_o = d.part_o + A * d.Kmax * d.Hq * n_split * d.dv;
    v.part_ml = d.part_ml + A * d.Kmax * d.Hq * n_split * 2;
  }
  v.ticket = d.ticket + A * d.Kmax * d.Hkv;
  v.u_ticket = d.u_ticket + A * d.Hkv;
  if (d.tc_part) v.tc_part = d.tc_part + A * (uattn_tc_part_floats(d) / d.N);
  return v;
}
}  // namespace

extern "C" {

// Relative sizes of dhs_round's request groups (all but the last, the last).
constexpr int kGroupWeight = 100, kLastGroupWeight = 60;

int dhs_round(dhs_ctx *c, const int8_t *q_idx, const int32_t *k_per_req, const void *q,
              const void *block_kv, const int32_t *accepted_len, int32_t *topk_out,
              int32_t *loc_out, void *out, float *lse, dhs_stream stream) {
  if (!c || !q_idx || !k_per_req || !q || !block_kv || !accepted_len || !topk_out || !loc_out ||
      !out || !aligned16(q_idx) || !aligned16(block_kv) || ((uintptr_t)q & 3u) ||
      ((uintptr_t)out & 3u))
    return DHS_ERR_INVALID;
  if (c->phase != PH_IDLE || c->role == DHS_ROLE_FOLLOWER || c->arenas || c->m > 1)
    return DHS_ERR_INVALID;
  const DevCtx &d = c->d;
  std::vector<int32_t> w;
  int max_dom = 0, active = 0;
  if (int rc = round_words(c, k_per_req, nullptr, w, max_dom, active)) return rc;
  for (int r = 0; r < d.N; ++r) {
    const int kr = k_per_req[r];
    if (!kr) continue;
    if (accepted_len[r] < 0 || accepted_len[r] > kr) return DHS_ERR_INVALID;
    if (c->n[r] + accepted_len[r] > d.Sm) return DHS_ERR_CAPACITY;
  }
  if (c->tick + 1 > 0x7FFFFFF0) return DHS_ERR_CAPACITY;
  const bool tc = c->cfg.attn_pass != DHS_ATTN_UNION_MMA && uattn_tc_supported(d);
  // Request groups for the tensor-core union pass only: the mma.sync union
  // pass sizes its partials for the whole context, and the per-query pass
  // measured slower in groups (64 histories of 524 288 latent rows: 3.97 ms
  // in one group, 6.1-6.3 ms in two or four; 8 of 32 768 rows: 0.085 against
  // 0.091-0.122 ms).  With per-kernel timing on, the round is issued as one
  // group on the caller's stream, so each kernel's events bracket that kernel
  // alone over the whole batch.
  const int G = (!c->fused || !tc || c->timer.enabled) ? 1 : c->groups;
  const bool fork = G > 1;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int tick = (int)(c->tick + 1);
  if (fork && cudaEventRecord(c->gevent[0], s) != cudaSuccess) return cuda_fail(c, cudaGetLastError());
  const size_t KK = (size_t)d.Kmax * d.k;
  const uint16_t *q16 = static_cast<const uint16_t *>(q);
  const uint16_t *b16 = static_cast<const uint16_t *>(block_kv);
  uint16_t *o16 = static_cast<uint16_t *>(out);
  int prev_sel = -1;  // the last group whose selection was issued
  // a group's attention and commit, issued once the next group's selection is
  struct Tail {
    int a;
    DevCtx v;
    std::vector<int32_t> cw;
    cudaStream_t sg;
    bool pending;
  };
  std::vector<Tail> tails(G);
  auto issue_tail = [&](int g) -> int {
    Tail &T = tails[g];
    T.pending = false;
    const int a = T.a;
    const DevCtx &v = T.v;
    cudaStream_t sg = T.sg;
    const size_t qoff = (size_t)a * d.Kmax * d.Hq;
    cudaError_t e =
        !c->fused ? launch_attend(v, q16 + qoff * d.dqk, b16 + (size_t)a * d.Kmax * d.row,
                                  loc_out + (size_t)a * KK, o16 + qoff * d.dv,
                                  lse ? lse + qoff : nullptr, c->n_split, sg, &c->timer)
        // (split-KV over idle SMs for the last group only: the earlier
        // groups' attention overlaps the next indexer, whose SMs it would
        // take; measured 1.91 -> 1.87 ms against no split on 128
        // histories of 102 400 rows in four groups, 1.94 splitting all)
        : tc ? launch_uattn_tc(v, q16 + qoff * d.dqk, b16 + (size_t)a * d.Kmax * d.row,
                               o16 + qoff * d.dv, lse ? lse + qoff : nullptr, sg, &c->timer,
                               g == G - 1 ? 0 : 1)
             : launch_uattn(v, q16 + qoff * d.dqk, b16 + (size_t)a * d.Kmax * d.row,
                            o16 + qoff * d.dv, lse ? lse + qoff : nullptr, sg, &c->timer);
    if (e == cudaSuccess) e = launch_commit(v, T.cw.data(), sg, &c->timer);
    if (e != cudaSuccess) return cuda_fail(c, e);
    if (fork && (cudaEventRecord(c->gevent[1 + g], sg) != cudaSuccess ||
                 cudaStreamWaitEvent(s, c->gevent[1 + g], 0) != cudaSuccess))
      return cuda_fail(c, cudaGetLastError());
    return DHS_OK;
  };
  // Group g covers slots [edge(g), edge(g + 1)): equal weights, except a
  // lighter last group, whose gather and attention nothing overlaps (they
  // end the round); measured on 128 histories of 102 400 rows in four
  // groups: last weight 1 -> 0.6, 1.876 -> 1.825 ms; 0.4 was slower.
  const int64_t tot_w = (int64_t)kGroupWeight * (G - 1) + kLastGroupWeight;
  auto edge = [&](int x) {
    return x >= G ? d.N : (int)((int64_t)d.N * ((int64_t)kGroupWeight * x) / tot_w);
  };
  for (int g = 0; g < G; ++g) {
    const int a = edge(g), b = edge(g + 1);
    if (a == b) continue;
    cudaStream_t sg = fork ? c->gstream[g] : s;
    if (fork && cudaStreamWaitEvent(sg, c->gevent[0], 0) != cudaSuccess)
      return cuda_fail(c, cudaGetLastError());
    const DevCtx v = slot_view(d, a, b, c->n_split);
    const int n = b - a;
    std::vector<int32_t> wg(n + (size_t)n * d.Kmax), cw((size_t)n * 4);
    int dom_g = 0, act_g = 0;
    for (int r = 0; r < n; ++r) {
      wg[r] = w[a + r];
      act_g += w[a + r];
      for (int j = 0; j < d.Kmax; ++j) {
        wg[n + r * d.Kmax + j] = w[d.N + (a + r) * d.Kmax + j];
        dom_g = std::max(dom_g, w[d.N + (a + r) * d.Kmax + j]);
      }
      const int kr = k_per_req[a + r];
      cw[r * 4 + 0] = kr ? accepted_len[a + r] : 0;
      cw[r * 4 + 1] = (int32_t)(uint32_t)(c->n[a + r] & 0xFFFFFFFF);
      cw[r * 4 + 2] = (int32_t)(c->n[a + r] >> 32);
      cw[r * 4 + 3] = kr ? 1 : 0;
    }
    // The groups' selections run one after another: a group's indexer starts
    // once the previous group's top-k has finished (each indexer alone
    // streams HBM at full rate), and the previous group's union/probe and
    // gather, sized to fit beside two indexer CTAs on an SM, overlap this
    // group's indexer (its attention, below, waits for this group's top-k).
    cudaError_t e = cudaSuccess;
    if (fork && prev_sel >= 0) e = cudaStreamWaitEvent(sg, c->gsel[prev_sel], 0);
    if (e == cudaSuccess)
      e = launch_select(v, q_idx + (size_t)a * d.Kmax * d.idx_row, nullptr,
                        topk_out + (size_t)a * KK, dom_g, wg.data(), act_g, c->cfg.topk_pass, sg,
                        &c->timer);
    if (e == cudaSuccess && fork) e = cudaEventRecord(c->gsel[g], sg);
    if (e != cudaSuccess) return cuda_fail(c, e);
    // the previous group's attention starts after this group's top-k: its
    // CTAs (a whole SM each) would otherwise slow the top-k that the next
    // indexer waits for
    if (prev_sel >= 0 && tails[prev_sel].pending) {
      if (cudaStreamWaitEvent(tails[prev_sel].sg, c->gsel[g], 0) != cudaSuccess)
        return cuda_fail(c, cudaGetLastError());
      if (int rc = issue_tail(prev_sel)) return rc;
    }
    prev_sel = g;
    if (e == cudaSuccess)
      e = launch_resolve(v, topk_out + (size_t)a * KK, loc_out + (size_t)a * KK, 1, 0, tick, sg,
                         &c->timer);
    if (e == cudaSuccess)
      e = launch_gather(v, topk_out + (size_t)a * KK, loc_out + (size_t)a * KK, 1, tick, sg,
                        &c->timer, !c->fused);
    if (e != cudaSuccess) return cuda_fail(c, e);
    tails[g] = Tail{a, v, std::move(cw), sg, true};
    if (!fork || g == G - 1)
      if (int rc = issue_tail(g)) return rc;
  }
  // (a last group left empty by the weights leaves the previous one pending)
  for (int g = 0; g < G; ++g)
    if (tails[g].pending)
      if (int rc = issue_tail(g)) return rc;
  c->tick = tick;
  c->last_shared = 1;
  for (int r = 0; r < d.N; ++r) {
    if (k_per_req[r]) {
      c->n[r] += accepted_len[r];
      c->tok[r] += accepted_len[r];
    }
    c->K[r] = 0;
  }
  c->phase = PH_IDLE;
  return DHS_OK;
}

int dhs_select(dhs_ctx *c, const int8_t *q_idx, const int32_t *k_per_req, const int64_t *pos,
               int32_t *topk_out, dhs_stream stream) {
  if (!c || !q_idx || !k_per_req || !topk_out || !aligned16(q_idx)) return DHS_ERR_INVALID;
  return select_impl(c, q_idx, nullptr, k_per_req, pos, topk_out, stream);
}

int dhs_adopt(dhs_ctx *c, const int32_t *k_per_req, const int64_t *pos, dhs_stream stream) {
  if (!c || !k_per_req) return DHS_ERR_INVALID;
  const DevCtx &d = c->d;
  std::vector<int32_t> w;
  int max_dom = 0, active = 0;
  if (int rc = round_words(c, k_per_req, pos, w, max_dom, active)) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (int rc = order_enter(c, s)) return rc;
  // K_r, then the domains, published by two ordinary launches: both have
  // completed before the resolve's first kernel starts
  {
    cudaError_t e_ = launch_upload(d.Kr, w.data(), d.N, s);
    if (e_ == cudaSuccess) {
      std::vector<int32_t> dw(w.begin() + d.N, w.end());
      if (upload_words(c, d.dom, dw, s)) return DHS_ERR_CUDA;
    } else {
      return cuda_fail(c, e_);
    }
  }
  for (int r = 0; r < d.N; ++r) c->K[r] = k_per_req[r];
  c->phase = PH_SELECTED;
  (void)max_dom;
  (void)active;
  return order_leave(c, s);
}

int dhs_resolve(dhs_ctx *c, const int32_t *topk, int32_t *loc_out, int32_t shared,
                dhs_stream stream) {
  if (!c || !topk || !loc_out || (shared != 0 && shared != 1)) return DHS_ERR_INVALID;
  if (c->phase != PH_SELECTED) return DHS_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  dhs_arenas *ar = c->arenas;
  // the arena's previous user must have issued its attention before its
  // staging rows can be replaced
  if (ar && ar->owner[c->arena] && ar->owner[c->arena] != c && ar->unread[c->arena])
    return DHS_ERR_INVALID;
  if (c->tick + 1 > 0x7FFFFFF0) return DHS_ERR_CAPACITY;
  if (int rc = order_enter(c, s)) return rc;
  if (ar && cudaStreamWaitEvent(s, ar->released[c->arena], 0) != cudaSuccess)
    return cuda_fail(c, cudaGetLastError());
  c->tick += 1;
  {
    // (2: the per-query attention pass follows, which the gather releases early)
    cudaError_t e_ = launch_resolve(c->d, topk, loc_out, shared, (c->fused && shared) ? 1 : 2,
                                    (int)c->tick, s, &c->timer);
    if (e_ != cudaSuccess) return cuda_fail(c, e_);
  }
  if (ar) {
    ar->owner[c->arena] = c;
    ar->unread[c->arena] = 1;
  }
  c->last_shared = shared;
  c->phase = PH_RESOLVED;
  return order_leave(c, s);
}

int dhs_attend(dhs_ctx *c, const void *q, const void *block_kv, const int32_t *loc, void *out,
               float *lse, dhs_stream stream) {
  if (!c || !q || !block_kv || !loc || !out) return DHS_ERR_INVALID;
  if (!aligned16(block_kv) || ((uintptr_t)q & 3u) || ((uintptr_t)out & 3u))
    return DHS_ERR_INVALID;
  // after a resolve, or again after an attend of the same resolve: a Reuse
  // consumer of the same source and location vector
  if (c->phase != PH_RESOLVED && c->phase != PH_ATTENDED) return DHS_ERR_INVALID;
  if (c->arenas && c->arenas->owner[c->arena] != c) return DHS_ERR_INVALID;  // arena taken
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (int rc = order_enter(c, s)) return rc;
  {
    const uint16_t *q16 = static_cast<const uint16_t *>(q);
    const uint16_t *b16 = static_cast<const uint16_t *>(block_kv);
    uint16_t *o16 = static_cast<uint16_t *>(out);
    const bool tc = c->cfg.attn_pass != DHS_ATTN_UNION_MMA && uattn_tc_supported(c->d);
    cudaError_t e_ = !(c->last_shared && c->fused)
                         ? launch_attend(c->d, q16, b16, loc, o16, lse, c->n_split, s, &c->timer)
                     : tc ? launch_uattn_tc(c->d, q16, b16, o16, lse, s, &c->timer)
                          : launch_uattn(c->d, q16, b16, o16, lse, s, &c->timer);
    if (e_ != cudaSuccess) return cuda_fail(c, e_);
  }
  if (c->arenas) {
    if (cudaEventRecord(c->arenas->released[c->arena], s) != cudaSuccess)
      return cuda_fail(c, cudaGetLastError());
    c->arenas->unread[c->arena] = 0;
  }
  c->phase = PH_ATTENDED;
  return order_leave(c, s);
}

int dhs_commit(dhs_ctx *c, const int32_t *accepted_len, dhs_stream stream) {
  if (!c || !accepted_len) return DHS_ERR_INVALID;
  if (c->phase != PH_ATTENDED || c->m > 1) return DHS_ERR_INVALID;
  const DevCtx &d = c->d;
  for (int r = 0; r < d.N; ++r) {
    if (c->K[r] == 0) continue;
    const int a = accepted_len[r];
    if (a < 0 || a > c->K[r]) return DHS_ERR_INVALID;
    if (c->n[r] + a > d.Sm) return DHS_ERR_CAPACITY;
  }
  std::vector<int32_t> w(d.N * 4, 0);
  for (int r = 0; r < d.N; ++r) {
    const int a = c->K[r] ? accepted_len[r] : 0;
    w[r * 4 + 0] = a;
    w[r * 4 + 1] = (int32_t)(uint32_t)(c->n[r] & 0xFFFFFFFF);
    w[r * 4 + 2] = (int32_t)(c->n[r] >> 32);
    w[r * 4 + 3] = c->K[r] ? 1 : 0;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (int rc = order_enter(c, s)) return rc;
  {
    cudaError_t e_ = launch_commit(d, w.data(), s, &c->timer);
    if (e_ != cudaSuccess) return cuda_fail(c, e_);
  }
  for (int r = 0; r < d.N; ++r) {
    if (c->K[r] == 0) continue;
    c->n[r] += accepted_len[r];
    c->tok[r] += accepted_len[r];
    c->K[r] = 0;
  }
  c->phase = PH_IDLE;
  return order_leave(c, s);
}

int dhs_commit_compressed(dhs_ctx *c, const int32_t *accepted_len, const void *rows_kv,
                          const int8_t *rows_idx_keys, dhs_stream stream) {
  if (!c || !accepted_len || !rows_kv || !aligned16(rows_kv) ||
      (rows_idx_keys && !aligned16(rows_idx_keys)))
    return DHS_ERR_INVALID;
  if (c->phase != PH_ATTENDED) return DHS_ERR_INVALID;
  const DevCtx &d = c->d;
  const int m = c->m;
  for (int r = 0; r < d.N; ++r) {
    if (c->K[r] == 0) continue;
    const int a = accepted_len[r];
    if (a < 0 || a > c->K[r]) return DHS_ERR_INVALID;
    if ((c->tok[r] + a) / m > d.Sm) return DHS_ERR_CAPACITY;
  }
  // per slot: completed rows, the first of them (lo, hi words), active
  std::vector<int32_t> w(d.N * 4, 0);
  for (int r = 0; r < d.N; ++r) {
    if (c->K[r] == 0) continue;
    const int64_t lo = c->tok[r] / m, hi = (c->tok[r] + accepted_len[r]) / m;
    w[r * 4 + 0] = (int32_t)(hi - lo);
    w[r * 4 + 1] = (int32_t)(uint32_t)(lo & 0xFFFFFFFF);
    w[r * 4 + 2] = (int32_t)(lo >> 32);
    w[r * 4 + 3] = 1;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (int rc = order_enter(c, s)) return rc;
  {
    cudaError_t e_ = launch_commit_rows(d, static_cast<const uint16_t *>(rows_kv), rows_idx_keys,
                                        (d.Kmax + m - 1) / m, w.data(), s, &c->timer);
    if (e_ != cudaSuccess) return cuda_fail(c, e_);
  }
  for (int r = 0; r < d.N; ++r) {
    if (c->K[r] == 0) continue;
    c->tok[r] += accepted_len[r];
    c->n[r] = c->tok[r] / m;
    c->ring_first[r] = c->n[r];
    c->K[r] = 0;
  }
  c->phase = PH_IDLE;
  return order_leave(c, s);
}

int dhs_append_keys(dhs_ctx *c, const int32_t *accepted_len, const int8_t *block_idx_keys,
                    dhs_stream stream) {
  if (!c || !accepted_len || !block_idx_keys || !aligned16(block_idx_keys)) return DHS_ERR_INVALID;
  if (c->role == DHS_ROLE_FOLLOWER || c->m > 1) return DHS_ERR_INVALID;
  const DevCtx &d = c->d;
  bool any = false;
  for (int r = 0; r < d.N; ++r) {
    const int a = accepted_len[r];
    if (a < 0 || a > d.Kmax || (a > 0 && !c->bound[r])) return DHS_ERR_INVALID;
    if (c->n[r] + a > d.Sm) return DHS_ERR_CAPACITY;
    any = any || a > 0;
  }
  if (!any) return DHS_OK;
  std::vector<int32_t> w(d.N * 4, 0);
  for (int r = 0; r < d.N; ++r) {
    w[r * 4 + 0] = accepted_len[r];
    w[r * 4 + 1] = (int32_t)(uint32_t)(c->n[r] & 0xFFFFFFFF);
    w[r * 4 + 2] = (int32_t)(c->n[r] >> 32);
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (int rc = order_enter(c, s)) return rc;
  {
    cudaError_t e_ = launch_append_keys(d, block_idx_keys, w.data(), s);
    if (e_ != cudaSuccess) return cuda_fail(c, e_);
  }
  return order_leave(c, s);
}

int dhs_set_residency(dhs_ctx *c, int32_t slot, const int32_t *rows, int64_t n_rows,
                      dhs_stream stream) {
  if (!c || slot < 0 || slot >= c->d.N || n_rows < 0 || (n_rows > 0 && !rows))
    return DHS_ERR_INVALID;
  if (!c->bound[slot]) return DHS_ERR_INVALID;
  if (c->phase == PH_RESOLVED) return DHS_ERR_INVALID;
  if (n_rows > c->d.opt_max) return DHS_ERR_CAPACITY;
  {
    std::vector<char> seen((size_t)c->n[slot], 0);
    for (int64_t i = 0; i < n_rows; ++i) {
      const int32_t v = rows[i];
      if (v < 0 || v >= c->n[slot] || seen[v]) return DHS_ERR_INVALID;
      seen[v] = 1;
    }
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (int rc = order_enter(c, s)) return rc;
  {
    cudaError_t e_ = launch_residency(c->d, slot, c->opt_count[slot], -1, s, &c->timer);
    if (e_ != cudaSuccess) return cuda_fail(c, e_);
  }
  if (n_rows > 0 &&
      cudaMemcpyAsync(c->d.opt_list + (size_t)slot * c->d.opt_max, rows, n_rows * 4,
                      cudaMemcpyHostToDevice, s) != cudaSuccess)
    return DHS_ERR_CUDA;
  {
    cudaError_t e_ = launch_residency(c->d, slot, -1, n_rows, s, &c->timer);
    if (e_ != cudaSuccess) return cuda_fail(c, e_);
  }
  c->opt_count[slot] = n_rows;
  return order_leave(c, s);
}

int dhs_get_stats(dhs_ctx *c, dhs_stats *out, dhs_stream stream) {
  if (!c || !out) return DHS_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned long long st[ST_COUNT];
  int32_t err[2];
  if (cudaStreamSynchronize(s) != cudaSuccess) return DHS_ERR_CUDA;
  if (cudaMemcpy(st, c->d.stats, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(err, c->d.err, sizeof(err), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DHS_ERR_CUDA;
  memset(out, 0, sizeof(*out));
  out->resolve_calls = c->tick;
  out->selections = st[ST_SEL];
  out->union_rows = st[ST_UNION];
  out->ring_hits = st[ST_RING];
  out->opt_hits = st[ST_OPT];
  out->hot_hits = st[ST_HOT];
  out->misses = st[ST_MISS];
  out->miss_selections = st[ST_MISS_SEL];
  out->host_rows_fetched = st[ST_FETCHED];
  out->host_bytes = (int64_t)st[ST_FETCHED] * c->d.row * 2;
  out->installs = st[ST_INSTALL];
  out->evictions = st[ST_EVICT];
  out->direct_only = st[ST_DIRECT];
  out->topk_rescans = st[ST_TOPK_RESCAN];
  out->device_error = err[0];
  out->device_error_site = err[1];
  return err[0] ? DHS_ERR_DEVICE_CHECK : DHS_OK;
}

int dhs_reset_stats(dhs_ctx *c, dhs_stream stream) {
  if (!c) return DHS_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(c->d.stats, 0, ST_COUNT * 8, s) != cudaSuccess ||
      cudaMemsetAsync(c->d.err, 0, 8, s) != cudaSuccess)
    return DHS_ERR_CUDA;
  return DHS_OK;
}

int64_t dhs_buffer_bytes(const dhs_ctx *c, int32_t which) {
  if (!c || which < 0 || which >= DHS_BUF_COUNT_) return -1;
  return (int64_t)buffer_desc(c, which).bytes;
}

int dhs_export(dhs_ctx *c, int32_t which, void *dst, int64_t bytes, dhs_stream stream) {
  if (!c || !dst || which < 0 || which >= DHS_BUF_COUNT_) return DHS_ERR_INVALID;
  BufDesc b = buffer_desc(c, which);
  if (bytes < 0 || (size_t)bytes > b.bytes) return DHS_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(dst, b.ptr, bytes, cudaMemcpyDefault, s) != cudaSuccess) return DHS_ERR_CUDA;
  return DHS_OK;
}

int dhs_set_timing(dhs_ctx *c, int32_t enable) {
  if (!c) return DHS_ERR_INVALID;
  c->timer.enabled = enable != 0;
  c->timer.reset();
  return DHS_OK;
}

int dhs_kernel_times(dhs_ctx *c, int32_t max_ids, int64_t *launches, double *total_ms) {
  if (!c || !launches || !total_ms || max_ids < 1) return DHS_ERR_INVALID;
  int64_t l[K_COUNT];
  double ms[K_COUNT];
  c->timer.collect(l, ms);
  for (int i = 0; i < max_ids && i < K_COUNT; ++i) {
    launches[i] = l[i];
    total_ms[i] = ms[i];
  }
  return DHS_OK;
}

int dhs_timing_accumulate_graph(dhs_ctx *c) {
  if (!c) return DHS_ERR_INVALID;
  c->timer.accumulate_graph();
  return DHS_OK;
}

int dhs_snapshot(dhs_ctx *c, int32_t *snapshot_id, dhs_stream stream) {
  if (!c || !snapshot_id) return DHS_ERR_INVALID;
  if (c->phase != PH_IDLE) return DHS_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Snapshot sn;
  for (int which : kStateBufs) {
    BufDesc b = buffer_desc(c, which);
    void *p = nullptr;
    if (cudaMalloc(&p, b.bytes ? b.bytes : 16) != cudaSuccess) {
      cudaGetLastError();
      for (void *q : sn.bufs) cudaFree(q);
      return DHS_ERR_OOM;
    }
    sn.bufs.push_back(p);
    if (b.bytes && cudaMemcpyAsync(p, b.ptr, b.bytes, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return DHS_ERR_CUDA;
  }
  sn.n = c->n;
  sn.tok = c->tok;
  sn.ring_first = c->ring_first;
  sn.opt_count = c->opt_count;
  sn.K = c->K;
  sn.tick = c->tick;
  sn.phase = c->phase;
  c->snaps.push_back(std::move(sn));
  *snapshot_id = (int32_t)c->snaps.size() - 1;
  return DHS_OK;
}

struct dhs_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

int dhs_graph_begin(dhs_stream stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed) == cudaSuccess ? DHS_OK
                                                                                : DHS_ERR_CUDA;
}

int dhs_graph_end(dhs_stream stream, dhs_graph **out) {
  if (!out) return DHS_ERR_INVALID;
  *out = nullptr;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  dhs_graph *g = new (std::nothrow) dhs_graph();
  if (!g) return DHS_ERR_OOM;
  if (cudaStreamEndCapture(s, &g->graph) != cudaSuccess || !g->graph ||
      cudaGraphInstantiateWithFlags(&g->exec, g->graph, cudaGraphInstantiateFlagUseNodePriority) !=
          cudaSuccess) {
    cudaGetLastError();
    if (g->graph) cudaGraphDestroy(g->graph);
    delete g;
    return DHS_ERR_CUDA;
  }
  *out = g;
  return DHS_OK;
}

int dhs_graph_launch(dhs_graph *g, dhs_stream stream) {
  if (!g || !g->exec) return DHS_ERR_INVALID;
  return cudaGraphLaunch(g->exec, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DHS_OK
             : DHS_ERR_CUDA;
}

void dhs_graph_destroy(dhs_graph *g) {
  if (!g) return;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  delete g;
}

int dhs_snapshot_free(dhs_ctx *c, int32_t id) {
  if (!c || id < 0 || id >= (int32_t)c->snaps.size() || c->snaps[id].bufs.empty())
    return DHS_ERR_INVALID;
  // the buffers may still be read by copies in flight on any stream
  if (cudaDeviceSynchronize() != cudaSuccess) return DHS_ERR_CUDA;
  for (void *p : c->snaps[id].bufs) cudaFree(p);
  c->snaps[id].bufs.clear();
  return DHS_OK;
}

int dhs_restore(dhs_ctx *c, int32_t id, dhs_stream stream) {
  if (!c || id < 0 || id >= (int32_t)c->snaps.size() || c->snaps[id].bufs.empty())
    return DHS_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Snapshot &sn = c->snaps[id];
  int i = 0;
  for (int which : kStateBufs) {
    BufDesc b = buffer_desc(c, which);
    if (b.bytes &&
        cudaMemcpyAsync(b.ptr, sn.bufs[i], b.bytes, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return DHS_ERR_CUDA;
    ++i;
  }
  // ring_first, Kr and the optional counts are small: upload from the mirrors
  std::vector<int32_t> w(c->d.N * 2);
  for (int r = 0; r < c->d.N; ++r) {
    w[2 * r] = (int32_t)(uint32_t)(sn.ring_first[r] & 0xFFFFFFFF);
    w[2 * r + 1] = (int32_t)(sn.ring_first[r] >> 32);
  }
  if (upload_words(c, reinterpret_cast<int32_t *>(c->d.ring_first), w, s)) return DHS_ERR_CUDA;
  for (int r = 0; r < c->d.N; ++r) {
    w[2 * r] = (int32_t)(uint32_t)(sn.opt_count[r] & 0xFFFFFFFF);
    w[2 * r + 1] = (int32_t)(sn.opt_count[r] >> 32);
  }
  if (upload_words(c, reinterpret_cast<int32_t *>(c->d.opt_count), w, s)) return DHS_ERR_CUDA;
  std::vector<int32_t> wk(sn.K.begin(), sn.K.end());
  if (upload_words(c, c->d.Kr, wk, s)) return DHS_ERR_CUDA;
  c->n = sn.n;
  c->tok = sn.tok;
  c->ring_first = sn.ring_first;
  c->opt_count = sn.opt_count;
  c->K = sn.K;
  c->tick = sn.tick;
  c->phase = sn.phase;
  return DHS_OK;
}

int dhs_round_host(dhs_ctx *c, const int8_t *q_idx, const int32_t *k_per_req, const void *q,
                   const void *block_kv, const int32_t *accepted_len, void *out, float *lse,
                   dhs_stream stream) {
  if (!c || !q_idx || !k_per_req || !q || !block_kv || !accepted_len || !out)
    return DHS_ERR_INVALID;
  const DevCtx &d = c->d;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t nq = (size_t)d.N * d.Kmax;
  if (c->groups > 1 && !c->arenas && c->role == DHS_ROLE_FULL) {
    // request groups: the whole round through dhs_round on device copies of
    // the index rows (queries, block rows and outputs used in place when
    // page-locked, else through device buffers)
    if (cudaMemcpyAsync(c->rh_qidx, q_idx, nq * d.idx_row, cudaMemcpyHostToDevice, s))
      return DHS_ERR_CUDA;
    const void *q_dev = mapped_ptr(q), *b_dev = mapped_ptr(block_kv);
    void *o_dev = mapped_ptr(out);
    float *l_dev = lse ? static_cast<float *>(mapped_ptr(lse)) : nullptr;
    if (!q_dev) {
      if (cudaMemcpyAsync(c->rh_q, q, nq * d.Hq * d.dqk * 2, cudaMemcpyHostToDevice, s))
        return DHS_ERR_CUDA;
      q_dev = c->rh_q;
    }
    if (!b_dev) {
      if (cudaMemcpyAsync(c->rh_block, block_kv, nq * d.row * 2, cudaMemcpyHostToDevice, s))
        return DHS_ERR_CUDA;
      b_dev = c->rh_block;
    }
    int rc = dhs_round(c, c->rh_qidx, k_per_req, q_dev, b_dev, accepted_len, c->rh_topk,
                       c->rh_loc, o_dev ? o_dev : c->rh_out,
                       lse ? (l_dev ? l_dev : c->rh_lse) : nullptr, stream);
    if (rc) return rc;
    if ((!o_dev &&
         cudaMemcpyAsync(out, c->rh_out, nq * d.Hq * d.dv * 2, cudaMemcpyDeviceToHost, s)) ||
        (lse && !l_dev &&
         cudaMemcpyAsync(lse, c->rh_lse, nq * d.Hq * 4, cudaMemcpyDeviceToHost, s)))
      return DHS_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? DHS_OK : DHS_ERR_CUDA;
  }
  // The indexer is launched first, so the GPU starts while the host prepares
  // the rest.  Small index rows travel in its launch parameters, else
  // through a device buffer.
  const bool inline_q =
      (size_t)ctl_qidx_word(d.N, d.Kmax) * 4 + nq * d.idx_row <= (size_t)kUploadWords * 4;
  if (!inline_q &&
      cudaMemcpyAsync(c->rh_qidx, q_idx, nq * d.idx_row, cudaMemcpyHostToDevice, s))
    return DHS_ERR_CUDA;
  int rc = inline_q ? select_impl(c, nullptr, q_idx, k_per_req, nullptr, c->rh_topk, stream)
                    : dhs_select(c, c->rh_qidx, k_per_req, nullptr, c->rh_topk, stream);
  if (!rc) rc = dhs_resolve(c, c->rh_topk, c->rh_loc, 1, stream);
  if (rc) return rc;
  // Queries, block rows and outputs in page-locked host memory are used in
  // place: the attention kernel reads them and writes its results across the
  // host link (zero copy).  Other host memory goes through device buffers.
  const void *q_dev = mapped_ptr(q), *b_dev = mapped_ptr(block_kv);
  void *o_dev = mapped_ptr(out);
  float *l_dev = lse ? static_cast<float *>(mapped_ptr(lse)) : nullptr;
  if (!q_dev) {
    if (cudaMemcpyAsync(c->rh_q, q, nq * d.Hq * d.dqk * 2, cudaMemcpyHostToDevice, s))
      return DHS_ERR_CUDA;
    q_dev = c->rh_q;
  }
  if (!b_dev) {
    if (cudaMemcpyAsync(c->rh_block, block_kv, nq * d.row * 2, cudaMemcpyHostToDevice, s))
      return DHS_ERR_CUDA;
    b_dev = c->rh_block;
  }
  rc = dhs_attend(c, q_dev, b_dev, c->rh_loc, o_dev ? o_dev : c->rh_out,
                  lse ? (l_dev ? l_dev : c->rh_lse) : nullptr, stream);
  if (!rc) rc = dhs_commit(c, accepted_len, stream);
  if (rc) return rc;
  if ((!o_dev &&
       cudaMemcpyAsync(out, c->rh_out, nq * d.Hq * d.dv * 2, cudaMemcpyDeviceToHost, s)) ||
      (lse && !l_dev &&
       cudaMemcpyAsync(lse, c->rh_lse, nq * d.Hq * 4, cudaMemcpyDeviceToHost, s)))
    return DHS_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DHS_ERR_CUDA;
  return DHS_OK;
}

}  // extern "C"
