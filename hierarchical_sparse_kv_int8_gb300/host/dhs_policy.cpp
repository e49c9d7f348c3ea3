// Residency policy of optional history: host-side page accounting.
//
// "Adaptive DHiSparse", section 3.1: the device pages of a KV pool hold the
// required allocations of the admitted requests (hot cache and tail, never
// lent), their optional history and an admission reserve, within the budget
// of eq. (3): M_req + M_opt + M_res <= M.  An admission that leaves a deficit
// of D pages reclaims whole requests: the admitted requests are walked in the
// reclaim order and the optional pages of the shortest prefix whose pages
// cover D are taken, eq. (4); the others keep theirs.  When pages are free, a
// bounded round-robin scheduler repopulates optional history.  Readings where
// the section leaves a choice open: the reclaim order is the admission order
// (oldest first); an admitted request keeps as much of its imported history
// as the free pages allow (resident-first admission, and after a reclaim the
// new request takes the freed pages); a repopulation attempt serves the
// admitted requests cyclically from where the previous attempt stopped, each
// up to its unmet history, until the attempt's page bound or the free pages
// run out.
//
// Pure host logic, no CUDA call.  The caller carries the decisions out with
// dhs_set_residency (bytes copied first, the rows published ready after the
// copy) and backs up a reclaimed request's rows before its pages are reused.
#include "../../include/dhs.h"

#include <algorithm>
#include <new>
#include <vector>

struct dhs_policy {
  struct Req {
    int32_t id;
    int64_t required, history, optional;
  };
  int64_t total = 0, reserve = 0;
  std::vector<Req> admitted;  // admission order, which is also the reclaim order
  size_t cursor = 0;          // where the next repopulation attempt starts

  int64_t used() const {
    int64_t u = 0;
    for (const Req &q : admitted) u += q.required + q.optional;
    return u;
  }
  int64_t free_pages() const { return total - reserve - used(); }
  int find(int32_t id) const {
    for (size_t i = 0; i < admitted.size(); ++i)
      if (admitted[i].id == id) return (int)i;
    return -1;
  }
};

extern "C" {

int dhs_policy_create(int64_t total_pages, int64_t reserve_pages, dhs_policy **out) {
  if (!out || total_pages < 0 || reserve_pages < 0 || reserve_pages > total_pages)
    return DHS_ERR_INVALID;
  dhs_policy *p = new (std::nothrow) dhs_policy;
  if (!p) return DHS_ERR_OOM;
  p->total = total_pages;
  p->reserve = reserve_pages;
  *out = p;
  return DHS_OK;
}

void dhs_policy_destroy(dhs_policy *p) { delete p; }

int dhs_policy_admit(dhs_policy *p, int32_t request, int64_t required_pages,
                     int64_t history_pages, int32_t *admitted, int64_t *optional_pages,
                     int32_t *reclaimed, int32_t reclaimed_cap, int32_t *n_reclaimed) {
  if (!p || !admitted || !optional_pages || !n_reclaimed || required_pages < 0 ||
      history_pages < 0 || reclaimed_cap < 0 || (reclaimed_cap > 0 && !reclaimed) ||
      p->find(request) >= 0)
    return DHS_ERR_INVALID;
  // Eq. (3) with every other request gone still cannot hold it: no reclaim
  // or completion can ever admit it, so it is refused rather than left waiting.
  if (required_pages > p->total - p->reserve) return DHS_ERR_CAPACITY;
  const int64_t free0 = p->free_pages();
  int64_t freed = 0;
  size_t q = 0;  // the reclaimed prefix of the admission order
  if (required_pages > free0) {
    const int64_t deficit = required_pages - free0;
    while (q < p->admitted.size() && freed < deficit) freed += p->admitted[q++].optional;
    if (freed < deficit) {  // the optional pages cannot cover it: the admission waits
      *admitted = 0;
      *optional_pages = 0;
      *n_reclaimed = 0;
      return DHS_OK;
    }
    int32_t n = 0;
    for (size_t i = 0; i < q; ++i) n += p->admitted[i].optional > 0;
    if (n > reclaimed_cap) return DHS_ERR_CAPACITY;
  }
  int32_t n = 0;
  for (size_t i = 0; i < q; ++i) {
    if (p->admitted[i].optional == 0) continue;
    reclaimed[n++] = p->admitted[i].id;
    p->admitted[i].optional = 0;
  }
  const int64_t opt = std::min(history_pages, free0 + freed - required_pages);
  p->admitted.push_back({request, required_pages, history_pages, opt});
  *admitted = 1;
  *optional_pages = opt;
  *n_reclaimed = n;
  return DHS_OK;
}

int dhs_policy_complete(dhs_policy *p, int32_t request) {
  const int i = p ? p->find(request) : -1;
  if (i < 0) return DHS_ERR_INVALID;
  p->admitted.erase(p->admitted.begin() + i);
  if ((size_t)i < p->cursor) --p->cursor;
  if (p->cursor >= p->admitted.size()) p->cursor = 0;
  return DHS_OK;
}

int dhs_policy_repopulate(dhs_policy *p, int64_t max_pages, int32_t *requests, int64_t *pages,
                          int32_t cap, int32_t *n_out) {
  if (!p || !n_out || max_pages < 0 || cap < 0 || (cap > 0 && (!requests || !pages)))
    return DHS_ERR_INVALID;
  if ((size_t)cap < p->admitted.size()) return DHS_ERR_CAPACITY;
  int64_t budget = std::min(max_pages, p->free_pages());
  const size_t n = p->admitted.size();
  int32_t m = 0;
  size_t next = p->cursor;
  for (size_t k = 0; k < n && budget > 0; ++k) {
    const size_t i = (p->cursor + k) % n;
    dhs_policy::Req &q = p->admitted[i];
    const int64_t give = std::min(q.history - q.optional, budget);
    if (give <= 0) continue;
    q.optional += give;
    budget -= give;
    requests[m] = q.id;
    pages[m] = give;
    ++m;
    next = (i + 1) % n;
  }
  p->cursor = next;
  *n_out = m;
  return DHS_OK;
}

int dhs_policy_query(const dhs_policy *p, int32_t request, int64_t *required_pages,
                     int64_t *optional_pages, int64_t *history_pages) {
  const int i = p ? p->find(request) : -1;
  if (i < 0 || !required_pages || !optional_pages || !history_pages) return DHS_ERR_INVALID;
  *required_pages = p->admitted[i].required;
  *optional_pages = p->admitted[i].optional;
  *history_pages = p->admitted[i].history;
  return DHS_OK;
}

int64_t dhs_policy_free_pages(const dhs_policy *p) { return p ? p->free_pages() : -1; }

}  // extern "C"
