// Two-tier prefix index over the page pool (host C++).
//
// ForkKV guide, "DualRadixTree: Two-Tier Hierarchical Cache Indexing" and
// "Two-Tier Lookup Mechanics": tier 1 is one radix tree over prompt token
// prefixes for all requests and adapters; each node owns the physical
// bCache pages of its token span.  Tier 2 hangs adapter leaves (an rCache
// owner: the agent slot holding that adapter's residual rows for the
// prefix) off tier-1 nodes.  A lookup finds the longest cached prefix
// (tier 1) and then the adapter's leaf at that node (tier 2): both present
// is a full hit, base only a partial hit (only the low-rank residual needs
// computing), neither a miss.  "Reference Counting and Eviction": each
// node counts the adapter leaves that depend on it (its own and its
// descendants'); a node nobody depends on stays cached until memory is
// needed and is then evicted least recently used first, leaves first.
//
// Granularity: a page of the pool (page_size tokens).  The KV of a page
// depends on every earlier token, so only whole pages of an exactly equal
// prefix are shared; a trailing partial page is never indexed.
//
// Workflow-aware eviction (KVFlow review, "Agent Step Graph and
// Steps-to-Execution", "Workflow-aware eviction"): an agent's
// steps-to-execution (how many workflow steps until it runs again) follows
// from its predecessors' values, max + 1 behind a barrier (AND), min + 1
// behind a branch (OR).  Each agent marks its fixed-prompt node and every
// ancestor with its value; a node's priority is the smallest value that
// marks it (a shared prefix is kept while any of its agents runs soon).
// Eviction by priority removes the evictable leaf with the largest priority
// first (unmarked nodes, e.g. dynamic suffixes, before all marked ones;
// ties least recently used first) and considers a parent once its last
// child is gone.
//
// The index owns one pool reference per page it holds; the caller takes
// those references when it inserts pages and drops them (fk_pages_release)
// for the ids that eviction returns.  Agents that use the pages hold their
// own references (fk_fork), so evicting a page from the index never frees
// a page an agent still reads.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <map>
#include <memory>
#include <queue>
#include <string>
#include <vector>

#include "forkkv.h"

namespace {

struct Node {
  int64_t id = 0;
  Node* parent = nullptr;
  std::vector<int32_t> tokens;               // span, a whole number of pages
  std::vector<int32_t> pages;                // one physical page per page_size tokens
  std::map<std::vector<int32_t>, std::unique_ptr<Node>> children;   // keyed by first page
  std::map<int32_t, int32_t> adapters;       // tier 2: adapter id -> rCache owner (agent slot)
  int64_t ref = 0;                           // adapter leaves at or below this node
  uint64_t last_use = 0;                     // logical clock of the last lookup through it
  std::map<int32_t, int32_t> steps;          // steps-to-execution -> agents marking this node
};

}  // namespace

struct fk_radix {
  int P = 16;
  std::unique_ptr<Node> root;
  std::map<int64_t, Node*> by_id;            // handle -> node
  int64_t next_id = 1;
  uint64_t clock = 0;
  int64_t n_pages = 0;
};

void fk_internal_set_error(const char* msg);   // the library's last-error text

namespace {

fk_status rfail(fk_status code, const char* msg) {
  fk_internal_set_error(msg);
  return code;
}

std::vector<int32_t> page_key(const int32_t* t, int P) { return std::vector<int32_t>(t, t + P); }

Node* new_node(fk_radix* r, Node* parent) {
  auto n = std::make_unique<Node>();
  n->id = r->next_id++;
  n->parent = parent;
  Node* raw = n.release();   // the caller links it into parent->children
  r->by_id[raw->id] = raw;
  raw->last_use = r->clock;
  return raw;
}

// Pages of `node`'s span that equal tokens[0 ..) page by page (at most `np`).
int common_pages(const Node* node, const int32_t* tok, int np, int P) {
  const int have = (int)node->pages.size();
  int k = 0;
  while (k < have && k < np &&
         std::equal(tok + (size_t)k * P, tok + (size_t)(k + 1) * P, node->tokens.begin() + (size_t)k * P))
    ++k;
  return k;
}

// Split `node` after its first `k` pages (0 < k < pages): a new head node
// takes the first k pages and becomes node's parent.  Node keeps its id,
// adapter leaves and children (handles name the end of a prefix, which
// does not move); the head has the same reference count (every leaf at or
// below node is below the head).
Node* split(fk_radix* r, Node* node, int k) {
  const int P = r->P;
  Node* parent = node->parent;
  const std::vector<int32_t> key = page_key(node->tokens.data(), P);
  Node* head = new_node(r, parent);
  head->tokens.assign(node->tokens.begin(), node->tokens.begin() + (size_t)k * P);
  head->pages.assign(node->pages.begin(), node->pages.begin() + k);
  head->ref = node->ref;
  head->last_use = node->last_use;
  head->steps = node->steps;   // every mark on node passed through its prefix
  std::unique_ptr<Node> own = std::move(parent->children[key]);
  parent->children.erase(key);
  node->tokens.erase(node->tokens.begin(), node->tokens.begin() + (size_t)k * P);
  node->pages.erase(node->pages.begin(), node->pages.begin() + k);
  node->parent = head;
  head->children.emplace(page_key(node->tokens.data(), P), std::move(own));
  parent->children.emplace(key, std::unique_ptr<Node>(head));
  return head;
}

// Walk the longest cached page prefix of tok[0 .. np pages).  Returns the
// deepest node reached and, in *in_node, how many of its pages matched (a
// partial match ends inside that node's span); *matched = pages matched.
Node* walk(fk_radix* r, const int32_t* tok, int np, int* matched, int* in_node, bool touch) {
  const int P = r->P;
  Node* node = r->root.get();
  int m = 0;
  *in_node = 0;
  if (touch) node->last_use = ++r->clock;
  while (m < np) {
    auto it = node->children.find(page_key(tok + (size_t)m * P, P));
    if (it == node->children.end()) break;
    Node* c = it->second.get();
    const int k = common_pages(c, tok + (size_t)m * P, np - m, P);
    if (touch) c->last_use = ++r->clock;
    m += k;
    node = c;
    *in_node = k;
    if (k < (int)c->pages.size()) break;
  }
  *matched = m;
  return node;
}

// Evicts leaves (no children, no adapter leaf at or below) in the order a
// heap with comparator `later` (true: a leaves after b) gives, until
// want_pages page ids are written or nothing is evictable or the next
// node's pages would not fit in cap_pages.  A parent joins the heap once its
// last child is gone.  Keys do not change while it runs, so the order is the
// same as picking the first node of that order among the current leaves
// each time.
template <class Later>
void evict_leaves(fk_radix* r, int want_pages, int32_t* pages_out, int cap_pages, int* n_out,
                  Later later) {
  *n_out = 0;
  std::priority_queue<Node*, std::vector<Node*>, Later> heap(later);
  for (auto& kv : r->by_id) {
    Node* x = kv.second;
    if (x != r->root.get() && x->ref == 0 && x->children.empty()) heap.push(x);
  }
  while (*n_out < want_pages && !heap.empty()) {
    Node* v = heap.top();
    if (*n_out + (int)v->pages.size() > cap_pages) break;
    heap.pop();
    std::copy(v->pages.begin(), v->pages.end(), pages_out + *n_out);
    *n_out += (int)v->pages.size();
    r->n_pages -= (int64_t)v->pages.size();
    Node* parent = v->parent;
    r->by_id.erase(v->id);
    parent->children.erase(page_key(v->tokens.data(), r->P));   // frees v
    if (parent != r->root.get() && parent->ref == 0 && parent->children.empty()) heap.push(parent);
  }
}

}  // namespace

// ================================================================= ABI ==

extern "C" {

fk_status fk_radix_create(int page_size, fk_radix** out) {
  if (!out || page_size < 1) return rfail(FK_ERR_INVALID_ARG, "page_size < 1 or out is NULL");
  auto* r = new fk_radix();
  r->P = page_size;
  r->root = std::make_unique<Node>();
  r->root->id = 0;
  r->by_id[0] = r->root.get();
  *out = r;
  return FK_OK;
}

void fk_radix_destroy(fk_radix* r) { delete r; }

fk_status fk_radix_match(fk_radix* r, const int32_t* tokens, int n_tokens, int32_t* pages,
                         int cap_pages, int* n_matched, int64_t* node) {
  if (!r || (!tokens && n_tokens) || n_tokens < 0 || !n_matched || !node)
    return rfail(FK_ERR_INVALID_ARG, "NULL argument or n_tokens < 0");
  const int np = n_tokens / r->P;
  int m = 0, in_node = 0;
  Node* at = walk(r, tokens, np, &m, &in_node, true);
  if (at != r->root.get() && in_node < (int)at->pages.size()) at = split(r, at, in_node);
  *n_matched = m;
  *node = at->id;
  if (pages) {
    if (cap_pages < m) return rfail(FK_ERR_INVALID_ARG, "cap_pages is below the matched page count");
    int k = m;
    for (Node* x = at; x && x != r->root.get(); x = x->parent) {
      k -= (int)x->pages.size();
      std::copy(x->pages.begin(), x->pages.end(), pages + k);
    }
  }
  return FK_OK;
}

fk_status fk_radix_insert(fk_radix* r, const int32_t* tokens, int n_tokens,
                          const int32_t* new_pages, int n_new, int64_t* node) {
  if (!r || (!tokens && n_tokens) || n_tokens < 0 || (!new_pages && n_new) || n_new < 0 || !node)
    return rfail(FK_ERR_INVALID_ARG, "NULL argument or negative count");
  const int P = r->P, np = n_tokens / P;
  int m = 0, in_node = 0;
  Node* at = walk(r, tokens, np, &m, &in_node, true);
  if (m + n_new != np)
    return rfail(FK_ERR_INVALID_ARG, "new pages must cover exactly the uncached whole pages of the prompt");
  if (at != r->root.get() && in_node < (int)at->pages.size()) at = split(r, at, in_node);
  if (n_new > 0) {
    Node* c = new_node(r, at);
    c->tokens.assign(tokens + (size_t)m * P, tokens + (size_t)np * P);
    c->pages.assign(new_pages, new_pages + n_new);
    c->last_use = ++r->clock;
    at->children.emplace(page_key(c->tokens.data(), P), std::unique_ptr<Node>(c));
    r->n_pages += n_new;
    at = c;
  }
  *node = at->id;
  return FK_OK;
}

fk_status fk_radix_adapter_get(fk_radix* r, int64_t node, int32_t adapter, int32_t* owner) {
  if (!r || !owner) return rfail(FK_ERR_INVALID_ARG, "NULL argument");
  auto it = r->by_id.find(node);
  if (it == r->by_id.end()) return rfail(FK_ERR_INVALID_ARG, "unknown node");
  auto a = it->second->adapters.find(adapter);
  *owner = a == it->second->adapters.end() ? -1 : a->second;
  return FK_OK;
}

fk_status fk_radix_adapter_attach(fk_radix* r, int64_t node, int32_t adapter, int32_t owner) {
  if (!r) return rfail(FK_ERR_INVALID_ARG, "NULL argument");
  auto it = r->by_id.find(node);
  if (it == r->by_id.end() || node == 0) return rfail(FK_ERR_INVALID_ARG, "unknown node or the root");
  Node* x = it->second;
  if (x->adapters.count(adapter)) return rfail(FK_ERR_INVALID_ARG, "adapter already has a leaf here");
  x->adapters[adapter] = owner;
  for (; x; x = x->parent) ++x->ref;
  return FK_OK;
}

fk_status fk_radix_adapter_detach(fk_radix* r, int64_t node, int32_t adapter, int32_t* owner) {
  if (!r) return rfail(FK_ERR_INVALID_ARG, "NULL argument");
  auto it = r->by_id.find(node);
  if (it == r->by_id.end()) return rfail(FK_ERR_INVALID_ARG, "unknown node");
  Node* x = it->second;
  auto a = x->adapters.find(adapter);
  if (a == x->adapters.end()) return rfail(FK_ERR_INVALID_ARG, "adapter has no leaf here");
  if (owner) *owner = a->second;
  x->adapters.erase(a);
  for (; x; x = x->parent) --x->ref;
  return FK_OK;
}

fk_status fk_radix_evict(fk_radix* r, int want_pages, int32_t* pages_out, int cap_pages,
                         int* n_out) {
  if (!r || !n_out || (!pages_out && cap_pages) || cap_pages < 0)
    return rfail(FK_ERR_INVALID_ARG, "NULL argument or negative capacity");
  // least recently used first
  evict_leaves(r, want_pages, pages_out, cap_pages, n_out,
               [](const Node* a, const Node* b) { return a->last_use > b->last_use; });
  return FK_OK;
}

fk_status fk_radix_stats(const fk_radix* r, int64_t* n_nodes, int64_t* n_pages) {
  if (!r || !n_nodes || !n_pages) return rfail(FK_ERR_INVALID_ARG, "NULL argument");
  *n_nodes = (int64_t)r->by_id.size() - 1;
  *n_pages = r->n_pages;
  return FK_OK;
}

fk_status fk_radix_node_ref(const fk_radix* r, int64_t node, int64_t* ref) {
  if (!r || !ref) return rfail(FK_ERR_INVALID_ARG, "NULL argument");
  auto it = r->by_id.find(node);
  if (it == r->by_id.end()) return rfail(FK_ERR_INVALID_ARG, "unknown node");
  *ref = it->second->ref;
  return FK_OK;
}

// ------------------------------------------------- workflow priorities --

fk_status fk_radix_priority_assign(fk_radix* r, int64_t node, int32_t step) {
  if (!r || step < 0) return rfail(FK_ERR_INVALID_ARG, "NULL index or negative step");
  auto it = r->by_id.find(node);
  if (it == r->by_id.end() || node == 0) return rfail(FK_ERR_INVALID_ARG, "unknown node or the root");
  for (Node* x = it->second; x && x != r->root.get(); x = x->parent) ++x->steps[step];
  return FK_OK;
}

fk_status fk_radix_priority_release(fk_radix* r, int64_t node, int32_t step) {
  if (!r) return rfail(FK_ERR_INVALID_ARG, "NULL index");
  auto it = r->by_id.find(node);
  if (it == r->by_id.end() || node == 0) return rfail(FK_ERR_INVALID_ARG, "unknown node or the root");
  for (Node* x = it->second; x && x != r->root.get(); x = x->parent)
    if (!x->steps.count(step)) return rfail(FK_ERR_INVALID_ARG, "no such assignment on this path");
  for (Node* x = it->second; x && x != r->root.get(); x = x->parent)
    if (--x->steps[step] == 0) x->steps.erase(step);
  return FK_OK;
}

fk_status fk_radix_priority_clear(fk_radix* r) {
  if (!r) return rfail(FK_ERR_INVALID_ARG, "NULL index");
  for (auto& kv : r->by_id) kv.second->steps.clear();
  return FK_OK;
}

fk_status fk_radix_node_priority(const fk_radix* r, int64_t node, int32_t* priority) {
  if (!r || !priority) return rfail(FK_ERR_INVALID_ARG, "NULL argument");
  auto it = r->by_id.find(node);
  if (it == r->by_id.end()) return rfail(FK_ERR_INVALID_ARG, "unknown node");
  *priority = it->second->steps.empty() ? -1 : it->second->steps.begin()->first;
  return FK_OK;
}

fk_status fk_radix_evict_workflow(fk_radix* r, int want_pages, int32_t* pages_out, int cap_pages,
                                  int* n_out) {
  if (!r || !n_out || (!pages_out && cap_pages) || cap_pages < 0)
    return rfail(FK_ERR_INVALID_ARG, "NULL argument or negative capacity");
  // larger priority first (unmarked = above every step), then the least
  // recently used
  auto prio = [](const Node* x) -> int64_t {
    return x->steps.empty() ? INT64_MAX : (int64_t)x->steps.begin()->first;
  };
  evict_leaves(r, want_pages, pages_out, cap_pages, n_out, [&](const Node* a, const Node* b) {
    const int64_t pa = prio(a), pb = prio(b);
    if (pa != pb) return pa < pb;
    return a->last_use > b->last_use;
  });
  return FK_OK;
}

fk_status fk_workflow_steps(int n_agents, const int32_t* pred_offsets, const int32_t* preds,
                            const int32_t* join, const int32_t* fixed, int32_t* steps) {
  if (n_agents < 0 || (n_agents > 0 && (!pred_offsets || !join || !fixed || !steps)))
    return rfail(FK_ERR_INVALID_ARG, "NULL argument or negative agent count");
  if (n_agents == 0) return FK_OK;
  if (pred_offsets[0] != 0) return rfail(FK_ERR_INVALID_ARG, "pred_offsets[0] must be 0");
  for (int i = 0; i < n_agents; ++i) {
    if (pred_offsets[i + 1] < pred_offsets[i]) return rfail(FK_ERR_INVALID_ARG, "pred_offsets not monotonic");
    if (join[i] != FK_JOIN_AND && join[i] != FK_JOIN_OR) return rfail(FK_ERR_INVALID_ARG, "bad join type");
    if (fixed[i] < -1) return rfail(FK_ERR_INVALID_ARG, "fixed values are >= 0 or -1");
  }
  if (pred_offsets[n_agents] > 0 && !preds) return rfail(FK_ERR_INVALID_ARG, "preds is NULL");
  for (int e = 0; e < pred_offsets[n_agents]; ++e)
    if (preds[e] < 0 || preds[e] >= n_agents) return rfail(FK_ERR_INVALID_ARG, "predecessor out of range");
  // depth-first over predecessors with an explicit stack; state 0 = not
  // visited, 1 = on the stack, 2 = done (value in out, -1 = never runs)
  std::vector<int32_t> out(n_agents, -1);
  std::vector<uint8_t> state(n_agents, 0);
  for (int i = 0; i < n_agents; ++i)
    if (fixed[i] >= 0) { out[i] = fixed[i]; state[i] = 2; }
  std::vector<std::pair<int, int>> st;   // (agent, next predecessor index)
  for (int s0 = 0; s0 < n_agents; ++s0) {
    if (state[s0] == 2) continue;
    st.push_back({s0, pred_offsets[s0]});
    state[s0] = 1;
    while (!st.empty()) {
      auto& [a, e] = st.back();
      if (e < pred_offsets[a + 1]) {
        const int p = preds[e++];
        if (state[p] == 1) return rfail(FK_ERR_INVALID_ARG, "cycle through agents with no fixed value");
        if (state[p] == 0) {
          state[p] = 1;
          st.push_back({p, pred_offsets[p]});
        }
        continue;
      }
      // every predecessor of a is done
      const int b = pred_offsets[a], eend = pred_offsets[a + 1];
      int32_t v = -1;
      if (eend > b) {
        if (join[a] == FK_JOIN_AND) {
          int32_t m = 0;
          bool ok = true;
          for (int k = b; k < eend; ++k) {
            if (out[preds[k]] < 0) { ok = false; break; }
            m = std::max(m, out[preds[k]]);
          }
          v = ok ? m + 1 : -1;
        } else {
          int32_t m = INT32_MAX;
          for (int k = b; k < eend; ++k)
            if (out[preds[k]] >= 0) m = std::min(m, out[preds[k]]);
          v = m == INT32_MAX ? -1 : m + 1;
        }
      }
      out[a] = v;
      state[a] = 2;
      st.pop_back();
    }
  }
  std::copy(out.begin(), out.end(), steps);
  return FK_OK;
}

}  // extern "C"
