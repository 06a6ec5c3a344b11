// Token-keyed radix index over the block pool ("Dismantling the Memory Wall",
// RadixAttention section: a compressed prefix tree whose nodes hold a token
// sequence and its KV indices, a lock_ref that pins a node and its
// ancestors while in use, and least-recently-used eviction of leaves whose
// lock_ref is zero).
//
// Adapted to the paged pool: the sharing unit is a full 16-token block, so a
// node's key is a whole number of blocks and its value is the physical block
// of each.  The index holds one reference on every block it stores, so a
// cached prefix outlives the branch that produced it.  Recency is a logical
// clock (one tick per match or insert), which makes the index deterministic.

#include <algorithm>
#include <cstring>

#include "internal.h"

using pkv::fail;

namespace {

struct RNode {
  int32_t parent = -1;
  bool live = true;
  std::vector<int32_t> key;     // tokens, 16 per block
  std::vector<int32_t> blocks;  // physical block of each 16-token chunk
  std::vector<int32_t> children;
  int32_t lock_ref = 0;
  int64_t last_access = 0;
};

}  // namespace

struct kv_radix {
  kv_pool* pool = nullptr;
  std::vector<RNode> nodes;  // 0 = root (empty key), never evicted
  int64_t clock = 0;
};

namespace {

constexpr int kB = 16;

void release_block(kv_pool* p, int32_t b) {
  if (--p->ref[b] == 0) p->free_stack.push_back(b);
}

bool first_block_equals(const RNode& n, const int32_t* tok) {
  return std::memcmp(n.key.data(), tok, kB * sizeof(int32_t)) == 0;
}

int32_t find_child(const kv_radix* r, int32_t node, const int32_t* tok) {
  for (int32_t c : r->nodes[node].children)
    if (first_block_equals(r->nodes[c], tok)) return c;
  return -1;
}

// Split node x after its first m blocks: a new node takes the prefix and x's
// place under its parent; x keeps the rest and becomes the new node's child.
int32_t split(kv_radix* r, int32_t x, int32_t m) {
  RNode y;
  {
    RNode& X = r->nodes[x];
    y.parent = X.parent;
    y.key.assign(X.key.begin(), X.key.begin() + m * kB);
    y.blocks.assign(X.blocks.begin(), X.blocks.begin() + m);
    y.lock_ref = X.lock_ref;
    y.last_access = X.last_access;
  }
  const int32_t yid = (int32_t)r->nodes.size();
  y.children.push_back(x);
  r->nodes.push_back(std::move(y));
  RNode& X = r->nodes[x];
  X.key.erase(X.key.begin(), X.key.begin() + m * kB);
  X.blocks.erase(X.blocks.begin(), X.blocks.begin() + m);
  auto& sib = r->nodes[r->nodes[yid].parent].children;
  *std::find(sib.begin(), sib.end(), x) = yid;
  X.parent = yid;
  return yid;
}

// Walk the longest cached prefix of tokens[0 .. 16 * nfull), splitting a node
// where the match ends inside it; every node on the path is touched.
// Returns (deepest matched node, matched blocks).
std::pair<int32_t, int32_t> walk(kv_radix* r, const int32_t* tokens,
                                 int32_t nfull) {
  int32_t cur = 0, pos = 0;
  r->nodes[0].last_access = r->clock;
  while (pos < nfull) {
    const int32_t c = find_child(r, cur, tokens + (int64_t)pos * kB);
    if (c < 0) break;
    const int32_t nb = (int32_t)r->nodes[c].blocks.size();
    int32_t m = 1;
    while (m < nb && pos + m < nfull &&
           std::memcmp(r->nodes[c].key.data() + (int64_t)m * kB,
                       tokens + (int64_t)(pos + m) * kB,
                       kB * sizeof(int32_t)) == 0)
      ++m;
    const int32_t hit = m < nb ? split(r, c, m) : c;
    r->nodes[hit].last_access = r->clock;
    cur = hit;
    pos += m;
  }
  return {cur, pos};
}

kv_status get_node(kv_radix* r, int32_t node) {
  if (!r) return fail(KV_ERR_INVALID_ARG, "null index");
  if (node < 0 || node >= (int32_t)r->nodes.size() || !r->nodes[node].live)
    return fail(KV_ERR_NOT_FOUND, "radix node %d does not exist", node);
  return KV_OK;
}

}  // namespace

extern "C" kv_status kv_radix_create(kv_pool* pool, kv_radix** out) {
  pkv::clear_error();
  if (!pool || !out) return fail(KV_ERR_INVALID_ARG, "null argument");
  if (pool->block_size != kB) return fail(KV_ERR_INVALID_ARG, "block size 16");
  auto* r = new kv_radix;
  r->pool = pool;
  r->nodes.emplace_back();  // root
  *out = r;
  return KV_OK;
}

extern "C" kv_status kv_radix_destroy(kv_radix* r) {
  pkv::clear_error();
  if (!r) return KV_OK;
  for (RNode& n : r->nodes)
    if (n.live)
      for (int32_t b : n.blocks) release_block(r->pool, b);
  delete r;
  return KV_OK;
}

extern "C" kv_status kv_radix_match(kv_radix* r, int32_t n_tokens,
                                    const int32_t* tokens, int32_t* out_node,
                                    int32_t* out_matched_tokens) {
  pkv::clear_error();
  if (!r || n_tokens < 0 || (n_tokens > 0 && !tokens) || !out_node ||
      !out_matched_tokens)
    return fail(KV_ERR_INVALID_ARG, "bad arguments");
  ++r->clock;
  auto [node, blocks] = walk(r, tokens, n_tokens / kB);
  *out_node = node;
  *out_matched_tokens = blocks * kB;
  return KV_OK;
}

extern "C" kv_status kv_radix_insert(kv_radix* r, int32_t branch,
                                     int32_t n_tokens, const int32_t* tokens,
                                     int32_t* out_node) {
  pkv::clear_error();
  if (!r || n_tokens < 0 || (n_tokens > 0 && !tokens) || !out_node)
    return fail(KV_ERR_INVALID_ARG, "bad arguments");
  kv_pool* p = r->pool;
  if (branch < 0 || branch >= (int32_t)p->nodes.size() || !p->nodes[branch].live)
    return fail(KV_ERR_NOT_FOUND, "branch %d does not exist", branch);
  const Node& br = p->nodes[branch];
  if (br.spilled)
    return fail(KV_ERR_INVALID_ARG, "branch %d is spilled: restore it first",
                branch);
  const int32_t nfull = std::min(n_tokens, br.seq_len) / kB;
  ++r->clock;
  auto [cur, pos] = walk(r, tokens, nfull);
  if (pos < nfull) {
    RNode leaf;
    leaf.parent = cur;
    leaf.key.assign(tokens + (int64_t)pos * kB, tokens + (int64_t)nfull * kB);
    leaf.blocks.assign(br.table.begin() + pos, br.table.begin() + nfull);
    for (int32_t b : leaf.blocks) p->ref[b] += 1;
    leaf.last_access = r->clock;
    const int32_t id = (int32_t)r->nodes.size();
    r->nodes.push_back(std::move(leaf));
    r->nodes[cur].children.push_back(id);
    cur = id;
  }
  *out_node = cur;
  return KV_OK;
}

extern "C" kv_status kv_radix_fork(kv_radix* r, int32_t node,
                                   int32_t* out_branch) {
  pkv::clear_error();
  if (kv_status s = get_node(r, node)) return s;
  if (!out_branch) return fail(KV_ERR_INVALID_ARG, "null output");
  std::vector<int32_t> path;
  for (int32_t x = node; x != -1; x = r->nodes[x].parent) path.push_back(x);
  Node br;
  for (auto it = path.rbegin(); it != path.rend(); ++it)
    for (int32_t b : r->nodes[*it].blocks) br.table.push_back(b);
  kv_pool* p = r->pool;
  for (int32_t b : br.table) p->ref[b] += 1;
  br.seq_len = (int32_t)br.table.size() * kB;
  p->nodes.push_back(std::move(br));
  *out_branch = (int32_t)p->nodes.size() - 1;
  return KV_OK;
}

extern "C" kv_status kv_radix_lock(kv_radix* r, int32_t node) {
  pkv::clear_error();
  if (kv_status s = get_node(r, node)) return s;
  for (int32_t x = node; x != -1; x = r->nodes[x].parent) ++r->nodes[x].lock_ref;
  return KV_OK;
}

extern "C" kv_status kv_radix_unlock(kv_radix* r, int32_t node) {
  pkv::clear_error();
  if (kv_status s = get_node(r, node)) return s;
  for (int32_t x = node; x != -1; x = r->nodes[x].parent)
    if (r->nodes[x].lock_ref < 1)
      return fail(KV_ERR_INVALID_ARG, "radix node %d is not locked", node);
  for (int32_t x = node; x != -1; x = r->nodes[x].parent) --r->nodes[x].lock_ref;
  return KV_OK;
}

extern "C" kv_status kv_radix_evict(kv_radix* r, int64_t target_free_blocks,
                                    int32_t* out_n_evicted,
                                    int32_t* out_evicted) {
  pkv::clear_error();
  if (!r) return fail(KV_ERR_INVALID_ARG, "null index");
  kv_pool* p = r->pool;
  int32_t n = 0;
  while ((int64_t)p->free_stack.size() < target_free_blocks) {
    int32_t best = -1;
    for (int32_t i = 1; i < (int32_t)r->nodes.size(); ++i) {
      const RNode& x = r->nodes[i];
      if (!x.live || !x.children.empty() || x.lock_ref != 0) continue;
      if (best < 0 || x.last_access < r->nodes[best].last_access) best = i;
    }
    if (best < 0) break;
    RNode& x = r->nodes[best];
    for (int32_t b : x.blocks) release_block(p, b);
    x.blocks.clear();
    x.key.clear();
    x.live = false;
    auto& sib = r->nodes[x.parent].children;
    sib.erase(std::find(sib.begin(), sib.end(), best));
    if (out_evicted) out_evicted[n] = best;
    ++n;
  }
  if (out_n_evicted) *out_n_evicted = n;
  return KV_OK;
}

extern "C" kv_status kv_radix_node_info(kv_radix* r, int32_t node,
                                        kv_radix_node_t* out) {
  pkv::clear_error();
  if (!r || !out) return fail(KV_ERR_INVALID_ARG, "null argument");
  if (node < 0 || node >= (int32_t)r->nodes.size())
    return fail(KV_ERR_NOT_FOUND, "radix node %d does not exist", node);
  const RNode& x = r->nodes[node];
  out->live = x.live ? 1 : 0;
  out->parent = x.parent;
  out->n_blocks = (int32_t)x.blocks.size();
  out->lock_ref = x.lock_ref;
  out->n_children = (int32_t)x.children.size();
  out->reserved = 0;
  out->last_access = x.last_access;
  return KV_OK;
}

extern "C" kv_status kv_radix_node_blocks(kv_radix* r, int32_t node,
                                          int32_t* out, int32_t cap,
                                          int32_t* out_n) {
  pkv::clear_error();
  if (kv_status s = get_node(r, node)) return s;
  const RNode& x = r->nodes[node];
  if (out_n) *out_n = (int32_t)x.blocks.size();
  if (out) {
    if (cap < (int32_t)x.blocks.size())
      return fail(KV_ERR_INVALID_ARG, "cap too small");
    std::copy(x.blocks.begin(), x.blocks.end(), out);
  }
  return KV_OK;
}

extern "C" kv_status kv_radix_num_nodes(kv_radix* r, int32_t* out) {
  pkv::clear_error();
  if (!r || !out) return fail(KV_ERR_INVALID_ARG, "null argument");
  *out = (int32_t)r->nodes.size();
  return KV_OK;
}
