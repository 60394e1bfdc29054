// Continuous-batching scheduler: FIFO admission by credit and on-demand page
// allocation from a shared pool (host only).
//
// Source: samir-vllm article, section "Gestion de la KV cache et strategies de
// batching": continuous batching admits a request as soon as its page budget
// is available; the admission credit is prompt_tokens + allowed_new_tokens - 1
// rounded up to 16-token pages for each layer; a request whose budget exceeds
// the pool is rejected with an explicit error so it cannot deadlock.  The
// free-page list and the -1 initialised block tables follow "2. Weight
// Loading and GPU Buffer Design", section "What else is set up in the
// initialization block".
//
// Rules the article leaves open (kept identical to the FP64 oracle's):
//   FIFO with head-of-line blocking; a request fits when
//   credit <= free - (credit - held summed over running requests); pages come
//   from a LIFO stack initialised [N-1 .. 0]; a finished request pushes its
//   pages back layer by layer in logical order; new requests take the lowest
//   free slot.
#include <deque>
#include <new>
#include <stdint.h>
#include <vector>

#include "pkv.h"

namespace {

struct Request {
  int prompt = 0, allowed_new = 0, credit = 0, held = 0, slot = -1;
  int len = 0;    // KV tokens the request's pages cover (the largest length grown to)
  int state = 0;  // 0 queued, 1 running, 2 done
  std::vector<std::vector<int32_t>> pages;  // [layer][logical page]
};

struct Event {
  int req, layer, logical, page;
};

int ceil_pages(long long tokens) {
  return tokens > 0 ? (int)((tokens + PKV_PAGE_TOKENS - 1) / PKV_PAGE_TOKENS) : 0;
}

}  // namespace

struct pkv_sched {
  int num_pages, num_layers, max_blocks, max_slots;
  std::vector<int32_t> free_stack;
  std::deque<int> queue;
  std::vector<Request> reqs;
  std::vector<int> slot_owner;
  std::vector<Event> events;
  long long reserved = 0;  // sum over running requests of credit - held
  int running = 0;
  std::vector<int> run_list;  // running requests in admission order (= id order)
  int mode = 0;            // 0 continuous, 1 static (admit only when nothing runs)
};

extern "C" int pkv_credit_pages(int prompt_tokens, int allowed_new_tokens, int num_layers) {
  if (prompt_tokens < 0 || allowed_new_tokens < 0 || num_layers < 0) return -1;
  const long long c = (long long)num_layers *
                      ceil_pages((long long)prompt_tokens + allowed_new_tokens - 1);
  return c > 0x7fffffffll ? -1 : (int)c;
}

extern "C" pkv_sched* pkv_sched_create(int num_pages, int num_layers, int max_blocks,
                                       int max_slots) {
  if (num_pages < 1 || num_layers < 1 || max_blocks < 1 || max_slots < 1) return nullptr;
  pkv_sched* s = new (std::nothrow) pkv_sched;
  if (!s) return nullptr;
  try {
    s->num_pages = num_pages;
    s->num_layers = num_layers;
    s->max_blocks = max_blocks;
    s->max_slots = max_slots;
    s->free_stack.reserve(num_pages);
    for (int p = num_pages - 1; p >= 0; --p) s->free_stack.push_back(p);
    s->slot_owner.assign(max_slots, -1);
  } catch (...) {
    delete s;
    return nullptr;
  }
  return s;
}

extern "C" void pkv_sched_destroy(pkv_sched* s) { delete s; }

extern "C" int pkv_sched_set_mode(pkv_sched* s, int mode) {
  if (!s || (mode != 0 && mode != 1)) return PKV_ERR_INVALID_ARGUMENT;
  s->mode = mode;
  return PKV_OK;
}

extern "C" int pkv_sched_submit(pkv_sched* s, int prompt_tokens, int allowed_new_tokens,
                                int* req_id) {
  if (!s || !req_id || prompt_tokens < 1 || allowed_new_tokens < 1)
    return PKV_ERR_INVALID_ARGUMENT;
  *req_id = -1;
  const long long tokens = (long long)prompt_tokens + allowed_new_tokens - 1;
  const long long credit = (long long)s->num_layers * ceil_pages(tokens);
  if (credit > s->num_pages || ceil_pages(tokens) > s->max_blocks) return PKV_ERR_REQUEST_TOO_LARGE;
  Request r;
  r.prompt = prompt_tokens;
  r.allowed_new = allowed_new_tokens;
  r.credit = (int)credit;
  r.pages.assign(s->num_layers, std::vector<int32_t>());
  s->reqs.push_back(std::move(r));
  *req_id = (int)s->reqs.size() - 1;
  s->queue.push_back(*req_id);
  return PKV_OK;
}

extern "C" int pkv_sched_admit(pkv_sched* s, int* admitted, int max_out, int* n_admitted) {
  if (!s || !n_admitted || max_out < 0 || (max_out > 0 && !admitted))
    return PKV_ERR_INVALID_ARGUMENT;
  int n = 0;
  if (s->mode == 1 && s->running > 0) {  // static batching: the group is still running
    *n_admitted = 0;
    return PKV_OK;
  }
  while (!s->queue.empty() && n < max_out) {
    Request& r = s->reqs[s->queue.front()];
    if ((long long)r.credit > (long long)s->free_stack.size() - s->reserved) break;
    int slot = -1;
    for (int i = 0; i < s->max_slots; ++i)
      if (s->slot_owner[i] < 0) {
        slot = i;
        break;
      }
    if (slot < 0) break;
    const int id = s->queue.front();
    s->queue.pop_front();
    s->slot_owner[slot] = id;
    r.slot = slot;
    r.state = 1;
    s->reserved += r.credit - r.held;
    ++s->running;
    s->run_list.push_back(id);
    admitted[n++] = id;
  }
  *n_admitted = n;
  return PKV_OK;
}

// Pages request r still needs in all layers to cover new_len tokens, or -1
// when that is not allowed (beyond max_blocks, its credit or the free pages).
static long long grow_need(const pkv_sched* s, const Request& r, int new_len) {
  const int need = ceil_pages(new_len);
  if (need > s->max_blocks) return -1;
  long long extra = 0;
  for (int l = 0; l < s->num_layers; ++l)
    if ((int)r.pages[l].size() < need) extra += need - (int)r.pages[l].size();
  if (r.held + extra > r.credit || extra > (long long)s->free_stack.size()) return -1;
  return extra;
}

extern "C" int pkv_sched_grow(pkv_sched* s, int req_id, int new_len) {
  if (!s || req_id < 0 || req_id >= (int)s->reqs.size() || new_len < 0)
    return PKV_ERR_INVALID_ARGUMENT;
  Request& r = s->reqs[req_id];
  const int need = ceil_pages(new_len);
  if (r.state != 1 || need > s->max_blocks) return PKV_ERR_INVALID_ARGUMENT;
  if (grow_need(s, r, new_len) < 0) return PKV_ERR_POOL_EXHAUSTED;
  if (new_len > r.len) r.len = new_len;
  for (int l = 0; l < s->num_layers; ++l) {
    while ((int)r.pages[l].size() < need) {
      const int32_t page = s->free_stack.back();
      s->free_stack.pop_back();
      s->events.push_back(Event{req_id, l, (int)r.pages[l].size(), page});
      r.pages[l].push_back(page);
      ++r.held;
      --s->reserved;
    }
  }
  return PKV_OK;
}

extern "C" int pkv_sched_finish(pkv_sched* s, int req_id) {
  if (!s || req_id < 0 || req_id >= (int)s->reqs.size()) return PKV_ERR_INVALID_ARGUMENT;
  Request& r = s->reqs[req_id];
  if (r.state != 1) return PKV_ERR_INVALID_ARGUMENT;
  for (int l = 0; l < s->num_layers; ++l) {
    for (int32_t page : r.pages[l]) s->free_stack.push_back(page);
    r.pages[l].clear();
  }
  s->reserved -= r.credit - r.held;
  r.held = 0;
  s->slot_owner[r.slot] = -1;
  r.slot = -1;
  r.state = 2;
  --s->running;
  for (size_t i = 0; i < s->run_list.size(); ++i)
    if (s->run_list[i] == req_id) {
      s->run_list.erase(s->run_list.begin() + (long)i);
      break;
    }
  return PKV_OK;
}

extern "C" int pkv_sched_begin_step(pkv_sched* s, int32_t* ids, int32_t* lens, int max_out,
                                    int* batch) {
  if (!s || !batch || max_out < 0 || (max_out > 0 && (!ids || !lens))) return PKV_ERR_INVALID_ARGUMENT;
  const int B = (int)s->run_list.size();
  if (B > max_out) return PKV_ERR_INVALID_ARGUMENT;
  // every request must be able to take its token before any grows (all or nothing)
  long long extra = 0;
  for (int id : s->run_list) {
    const Request& r = s->reqs[id];
    const long long e = grow_need(s, r, r.len + 1);
    if (e < 0) return PKV_ERR_POOL_EXHAUSTED;
    extra += e;
  }
  if (extra > (long long)s->free_stack.size()) return PKV_ERR_POOL_EXHAUSTED;
  for (int b = 0; b < B; ++b) {
    const int id = s->run_list[b];
    const int rc = pkv_sched_grow(s, id, s->reqs[id].len + 1);
    if (rc != PKV_OK) return rc;  // cannot happen after the check above
    ids[b] = id;
    lens[b] = s->reqs[id].len;
  }
  *batch = B;
  return PKV_OK;
}

// lens [batch] int32, then (16-byte aligned) tables [L][batch][pages] int32
static size_t step_tables_offset(int batch) { return ((size_t)4 * batch + 15) & ~(size_t)15; }

extern "C" size_t pkv_sched_step_bytes(const pkv_sched* s, int batch, int max_len) {
  if (!s || batch < 0 || max_len < 0) return 0;
  const int pages = ceil_pages(max_len) > 0 ? ceil_pages(max_len) : 1;
  return step_tables_offset(batch) + (size_t)4 * s->num_layers * batch * pages;
}

extern "C" int pkv_sched_pack_step(const pkv_sched* s, const int32_t* ids, int batch, int max_len,
                                   void* block, size_t bytes) {
  if (!s || batch < 0 || max_len < 0 || (batch > 0 && (!ids || !block)))
    return PKV_ERR_INVALID_ARGUMENT;
  if (bytes < pkv_sched_step_bytes(s, batch, max_len)) return PKV_ERR_WORKSPACE_TOO_SMALL;
  const int pages = ceil_pages(max_len) > 0 ? ceil_pages(max_len) : 1;
  int32_t* lens = static_cast<int32_t*>(block);
  int32_t* tab = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(block) + step_tables_offset(batch));
  for (int b = 0; b < batch; ++b) {
    if (ids[b] < 0 || ids[b] >= (int)s->reqs.size() || s->reqs[ids[b]].state != 1)
      return PKV_ERR_INVALID_ARGUMENT;
    if (s->reqs[ids[b]].len > max_len) return PKV_ERR_INVALID_ARGUMENT;
    lens[b] = s->reqs[ids[b]].len;
  }
  for (int l = 0; l < s->num_layers; ++l)
    for (int b = 0; b < batch; ++b) {
      const std::vector<int32_t>& pg = s->reqs[ids[b]].pages[l];
      int32_t* row = tab + ((size_t)l * batch + b) * pages;
      const int have = (int)pg.size() < pages ? (int)pg.size() : pages;
      for (int j = 0; j < have; ++j) row[j] = pg[j];
      for (int j = have; j < pages; ++j) row[j] = -1;
    }
  return PKV_OK;
}

extern "C" int pkv_sched_block_table(const pkv_sched* s, int req_id, int layer, int32_t* row,
                                     int* slot) {
  if (!s || !row || req_id < 0 || req_id >= (int)s->reqs.size() || layer < 0 ||
      layer >= s->num_layers)
    return PKV_ERR_INVALID_ARGUMENT;
  const Request& r = s->reqs[req_id];
  for (int j = 0; j < s->max_blocks; ++j)
    row[j] = j < (int)r.pages[layer].size() ? r.pages[layer][j] : -1;
  if (slot) *slot = r.slot;
  return PKV_OK;
}

extern "C" int pkv_sched_stats(const pkv_sched* s, int* free_pages, int* reserved_pages,
                               int* queued, int* running) {
  if (!s) return PKV_ERR_INVALID_ARGUMENT;
  if (free_pages) *free_pages = (int)s->free_stack.size();
  if (reserved_pages) *reserved_pages = (int)s->reserved;
  if (queued) *queued = (int)s->queue.size();
  if (running) *running = s->running;
  return PKV_OK;
}

extern "C" int pkv_sched_event_count(const pkv_sched* s) {
  return s ? (int)s->events.size() : -1;
}

extern "C" int pkv_sched_event(const pkv_sched* s, int i, int* req_id, int* layer, int* logical,
                               int* page) {
  if (!s || i < 0 || i >= (int)s->events.size()) return PKV_ERR_INVALID_ARGUMENT;
  const Event& e = s->events[i];
  if (req_id) *req_id = e.req;
  if (layer) *layer = e.layer;
  if (logical) *logical = e.logical;
  if (page) *page = e.page;
  return PKV_OK;
}
