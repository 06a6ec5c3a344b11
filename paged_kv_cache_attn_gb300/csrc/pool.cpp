// Block pool, branch tree, fork with copy-on-write, free, eviction and the
// decode-batch builder.  Host metadata only; data movement is delegated to
// the kernels in state_kernels.cu.
//
// Rules ("The Reasoning Engine Meltdown", §5 fork rules and §6
// TreePagedKVCacheManager; "Dismantling the Memory Wall", PagedAttention and
// copy-on-write sections; RKSC summary §2.C for the eviction score):
//  * a fork shares the parent's full blocks (+1 reference each) and copies a
//    partial last block into a fresh block of its own;
//  * a block whose reference count reaches 0 is pushed on the free stack;
//  * the free stack is LIFO, seeded by the caller's order (first element
//    handed out first);
//  * every operation is all-or-nothing.

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstring>
#include <numeric>

#include "internal.h"


namespace pkv {

static thread_local std::string g_err;

kv_status fail(kv_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

void clear_error() { g_err.clear(); }

}  // namespace pkv

using pkv::fail;

extern "C" const char* kv_last_error(void) { return pkv::g_err.c_str(); }

extern "C" int64_t kv_bytes_per_token(int32_t num_layers, int32_t num_heads,
                                      int32_t head_dim, int32_t elem_bytes) {
  return 2LL * num_layers * num_heads * head_dim * elem_bytes;
}

static inline int32_t blocks_for(int64_t tokens, int32_t B) {
  return (int32_t)((tokens + B - 1) / B);
}

static kv_status get_live(kv_pool* p, int32_t id, Node** out) {
  if (!p) return fail(KV_ERR_INVALID_ARG, "null pool");
  if (id < 0 || id >= (int32_t)p->nodes.size())
    return fail(KV_ERR_NOT_FOUND, "branch %d does not exist", id);
  if (!p->nodes[id].live)
    return fail(KV_ERR_NOT_FOUND, "branch %d was freed", id);
  *out = &p->nodes[id];
  return KV_OK;
}

extern "C" kv_status kv_pool_create(const kv_pool_desc* d, kv_pool** out) {
  pkv::clear_error();
  if (!d || !out) return fail(KV_ERR_INVALID_ARG, "null argument");
  if (d->num_blocks < 1 || d->num_blocks > (int64_t)INT32_MAX)
    return fail(KV_ERR_INVALID_ARG, "num_blocks %lld out of range",
                (long long)d->num_blocks);
  if (d->block_size != 16)
    return fail(KV_ERR_INVALID_ARG, "block_size must be 16, got %d",
                d->block_size);
  if (d->num_layers < 1 || d->num_kv_heads < 1)
    return fail(KV_ERR_INVALID_ARG, "num_layers and num_kv_heads must be >= 1");
  if (d->head_dim != 64 && d->head_dim != 128)
    return fail(KV_ERR_INVALID_ARG, "head_dim must be 64 or 128, got %d",
                d->head_dim);
  if ((d->k_pool == nullptr) != (d->v_pool == nullptr))
    return fail(KV_ERR_INVALID_ARG, "k_pool and v_pool must both be set or "
                                    "both be NULL");
  if (((uintptr_t)d->k_pool | (uintptr_t)d->v_pool) & 15)
    return fail(KV_ERR_INVALID_ARG, "pools must be 16-byte aligned");
  if (d->kv_dtype != KV_DTYPE_BF16 && d->kv_dtype != KV_DTYPE_E4M3)
    return fail(KV_ERR_INVALID_ARG, "kv_dtype must be KV_DTYPE_BF16 or "
                                    "KV_DTYPE_E4M3, got %d", d->kv_dtype);
  if (d->kv_dtype == KV_DTYPE_E4M3 && d->k_pool != nullptr) {
    if (d->kv_scales == nullptr)
      return fail(KV_ERR_INVALID_ARG, "an e4m3 data pool needs kv_scales");
    if ((uintptr_t)d->kv_scales & 15)
      return fail(KV_ERR_INVALID_ARG, "kv_scales must be 16-byte aligned");
  } else if (d->kv_scales != nullptr) {
    return fail(KV_ERR_INVALID_ARG, "kv_scales is only for e4m3 data pools");
  }
  // Rows of one layer must fit a 2-D TMA coordinate (int32).
  if (d->num_blocks * d->num_kv_heads * d->block_size > (int64_t)INT32_MAX)
    return fail(KV_ERR_INVALID_ARG, "pool too large for one layer's rows");
  auto* p = new kv_pool;
  p->num_blocks = d->num_blocks;
  p->block_size = d->block_size;
  p->num_layers = d->num_layers;
  p->num_kv_heads = d->num_kv_heads;
  p->head_dim = d->head_dim;
  p->k_pool = d->k_pool;
  p->v_pool = d->v_pool;
  p->kv_dtype = d->kv_dtype;
  p->kv_scales = d->kv_scales;
  p->ref.assign(d->num_blocks, 0);
  std::vector<int32_t> order(d->num_blocks);
  if (d->initial_free_order) {
    std::vector<char> seen(d->num_blocks, 0);
    for (int64_t i = 0; i < d->num_blocks; ++i) {
      int32_t b = d->initial_free_order[i];
      if (b < 0 || b >= d->num_blocks || seen[b]) {
        delete p;
        return fail(KV_ERR_INVALID_ARG,
                    "initial_free_order is not a permutation (entry %lld)",
                    (long long)i);
      }
      seen[b] = 1;
      order[i] = b;
    }
  } else {
    std::iota(order.begin(), order.end(), 0);
  }
  p->free_stack.assign(order.rbegin(), order.rend());
  *out = p;
  return KV_OK;
}

extern "C" kv_status kv_pool_destroy(kv_pool* p) {
  pkv::clear_error();
  delete p;
  return KV_OK;
}

extern "C" kv_status kv_branch_create(kv_pool* p, int32_t* out_id) {
  pkv::clear_error();
  if (!p || !out_id) return fail(KV_ERR_INVALID_ARG, "null argument");
  if (p->nodes.size() >= (size_t)INT32_MAX)
    return fail(KV_ERR_INVALID_ARG, "branch id space exhausted");
  p->nodes.emplace_back();
  *out_id = (int32_t)p->nodes.size() - 1;
  return KV_OK;
}

extern "C" kv_status kv_append(kv_pool* p, int32_t id, int32_t n,
                               const void* k_new, const void* v_new,
                               void* stream) {
  pkv::clear_error();
  Node* nd;
  if (kv_status s = get_live(p, id, &nd)) return s;
  if (n < 0) return fail(KV_ERR_INVALID_ARG, "negative token count");
  if (nd->spilled)
    return fail(KV_ERR_INVALID_ARG, "branch %d is spilled: restore it first", id);
  if ((int64_t)nd->seq_len + n > (int64_t)INT32_MAX / 2)
    return fail(KV_ERR_INVALID_ARG, "sequence too long");
  const int32_t B = p->block_size;
  if (p->has_data() && n > 0) {
    if (!k_new || !v_new)
      return fail(KV_ERR_INVALID_ARG, "k_new / v_new required for a data pool");
    if (((uintptr_t)k_new | (uintptr_t)v_new) & 15)
      return fail(KV_ERR_INVALID_ARG, "k_new / v_new must be 16-byte aligned");
  }
  if (!p->has_data() && (k_new || v_new))
    return fail(KV_ERR_INVALID_ARG, "metadata-only pool takes no data");
  if (nd->seq_len % B != 0 && p->ref[nd->table.back()] != 1)
    return fail(KV_ERR_INTERNAL, "partial last block of branch %d is shared",
                id);
  const int32_t need = blocks_for((int64_t)nd->seq_len + n, B) -
                       (int32_t)nd->table.size();
  if ((int64_t)need > (int64_t)p->free_stack.size())
    return fail(KV_ERR_OOM, "append of %d tokens needs %d blocks, %zu free", n,
                need, p->free_stack.size());
  if (n == 0) return KV_OK;
  // The blocks the append will take, in allocation order.
  std::vector<int32_t> fresh(need);
  for (int32_t i = 0; i < need; ++i)
    fresh[i] = p->free_stack[p->free_stack.size() - 1 - i];
  if (p->has_data()) {
    const int32_t first_lb = nd->seq_len / B;
    const int32_t last_lb = (nd->seq_len + n - 1) / B;
    std::vector<int32_t> dst(last_lb - first_lb + 1);
    for (int32_t lb = first_lb; lb <= last_lb; ++lb) {
      dst[lb - first_lb] = lb < (int32_t)nd->table.size()
                               ? nd->table[lb]
                               : fresh[lb - (int32_t)nd->table.size()];
    }
    int err;
    if (p->e4m3()) {
      std::vector<pkv::ScatterRun> runs{{0, n, nd->seq_len, first_lb, dst}};
      err = pkv::launch_append_e4m3(p->k_pool, p->v_pool, p->kv_scales,
                                    p->num_blocks, p->num_layers,
                                    p->num_kv_heads, p->head_dim, k_new, v_new,
                                    n, runs, stream);
    } else {
      err = pkv::launch_append_scatter(
          p->k_pool, p->v_pool, k_new, v_new, p->num_blocks, p->num_layers,
          p->num_kv_heads, p->head_dim, B, n, nd->seq_len, dst.data(),
          (int)dst.size(), stream);
    }
    if (err) return fail(KV_ERR_CUDA, "append copy launch failed (cuda %d)", err);
  }
  for (int32_t b : fresh) {
    p->free_stack.pop_back();
    p->ref[b] = 1;
    nd->table.push_back(b);
  }
  nd->seq_len += n;
  return KV_OK;
}

// Blocks a batch of appends takes, in allocation order, and for each entry
// the logical->physical map of the blocks its tokens land in.  Nothing is
// changed; returns OOM / NOT_FOUND / INVALID_ARG like the single append.
namespace {
struct PlannedAppend {
  int32_t id, n, tok0, first_lb;
  std::vector<int32_t> dst;  // physical block of logical first_lb + i
  int32_t fresh_begin, fresh_count;
};
}  // namespace

static kv_status plan_appends(kv_pool* p, int32_t n, const int32_t* ids,
                              const int32_t* n_tokens,
                              std::vector<PlannedAppend>* out,
                              std::vector<int32_t>* fresh) {
  if (!p) return fail(KV_ERR_INVALID_ARG, "null pool");
  if (n < 0 || (n > 0 && (!ids || !n_tokens)))
    return fail(KV_ERR_INVALID_ARG, "bad batch arrays");
  const int32_t B = p->block_size;
  // Branch lengths and table sizes as the batch proceeds (a branch may
  // appear more than once).
  std::vector<std::pair<int32_t, std::pair<int32_t, int32_t>>> cur;  // id -> (len, nblk)
  auto state = [&](int32_t id) -> std::pair<int32_t, int32_t>& {
    for (auto& c : cur)
      if (c.first == id) return c.second;
    Node& nd = p->nodes[id];
    cur.push_back({id, {nd.seq_len, (int32_t)nd.table.size()}});
    return cur.back().second;
  };
  size_t next_free = 0;  // blocks taken so far from the top of the stack
  for (int32_t i = 0; i < n; ++i) {
    Node* nd;
    if (kv_status s = get_live(p, ids[i], &nd)) return s;
    if (n_tokens[i] < 0) return fail(KV_ERR_INVALID_ARG, "negative token count");
    if (nd->spilled)
      return fail(KV_ERR_INVALID_ARG, "branch %d is spilled: restore it first",
                  ids[i]);
    auto& st = state(ids[i]);
    if ((int64_t)st.first + n_tokens[i] > (int64_t)INT32_MAX / 2)
      return fail(KV_ERR_INVALID_ARG, "sequence too long");
    if (st.first % B != 0 && st.second == (int32_t)nd->table.size() &&
        p->ref[nd->table.back()] != 1)
      return fail(KV_ERR_INTERNAL, "partial last block of branch %d is shared",
                  ids[i]);
    const int32_t need =
        blocks_for((int64_t)st.first + n_tokens[i], B) - st.second;
    if (next_free + (size_t)need > p->free_stack.size())
      return fail(KV_ERR_OOM, "batch append needs more blocks than the %zu free",
                  p->free_stack.size());
    PlannedAppend pa{ids[i], n_tokens[i], st.first, st.first / B, {},
                     (int32_t)next_free, need};
    for (int32_t k = 0; k < need; ++k)
      fresh->push_back(p->free_stack[p->free_stack.size() - 1 - next_free - k]);
    if (n_tokens[i] > 0) {
      const int32_t last_lb = (st.first + n_tokens[i] - 1) / B;
      // Blocks of this branch in logical order: the committed table, then
      // blocks taken earlier in this batch, then this entry's fresh blocks.
      std::vector<int32_t> mine;
      for (auto& q : *out)
        if (q.id == ids[i])
          for (int32_t k = 0; k < q.fresh_count; ++k)
            mine.push_back((*fresh)[q.fresh_begin + k]);
      for (int32_t lb = pa.first_lb; lb <= last_lb; ++lb) {
        const int32_t tsz = (int32_t)nd->table.size();
        int32_t blk;
        if (lb < tsz)
          blk = nd->table[lb];
        else if (lb - tsz < (int32_t)mine.size())
          blk = mine[lb - tsz];
        else
          blk = (*fresh)[next_free + (lb - tsz - (int32_t)mine.size())];
        pa.dst.push_back(blk);
      }
    }
    next_free += need;
    st.first += n_tokens[i];
    st.second += need;
    out->push_back(std::move(pa));
  }
  return KV_OK;
}

static void commit_appends(kv_pool* p, const std::vector<PlannedAppend>& plan,
                           const std::vector<int32_t>& fresh) {
  for (const PlannedAppend& pa : plan) {
    Node& nd = p->nodes[pa.id];
    for (int32_t k = 0; k < pa.fresh_count; ++k) {
      const int32_t b = fresh[pa.fresh_begin + k];
      p->free_stack.pop_back();
      p->ref[b] = 1;
      nd.table.push_back(b);
    }
    nd.seq_len += pa.n;
  }
}

extern "C" kv_status kv_reserve(kv_pool* p, int32_t n, const int32_t* ids,
                                const int32_t* n_tokens) {
  pkv::clear_error();
  std::vector<PlannedAppend> plan;
  std::vector<int32_t> fresh;
  if (kv_status s = plan_appends(p, n, ids, n_tokens, &plan, &fresh)) return s;
  commit_appends(p, plan, fresh);
  return KV_OK;
}

extern "C" kv_status kv_append_batch(kv_pool* p, int32_t n, const int32_t* ids,
                                     const int32_t* n_tokens,
                                     const void* k_new, const void* v_new,
                                     void* stream) {
  pkv::clear_error();
  std::vector<PlannedAppend> plan;
  std::vector<int32_t> fresh;
  if (kv_status s = plan_appends(p, n, ids, n_tokens, &plan, &fresh)) return s;
  int64_t total = 0;
  for (auto& pa : plan) total += pa.n;
  if (total > INT32_MAX / 2) return fail(KV_ERR_INVALID_ARG, "batch too large");
  if (p->has_data() && total > 0) {
    if (!k_new || !v_new)
      return fail(KV_ERR_INVALID_ARG, "k_new / v_new required for a data pool");
    if (((uintptr_t)k_new | (uintptr_t)v_new) & 15)
      return fail(KV_ERR_INVALID_ARG, "k_new / v_new must be 16-byte aligned");
    std::vector<pkv::ScatterRun> runs;
    int32_t row = 0;
    for (auto& pa : plan) {
      if (pa.n > 0)
        runs.push_back({row, pa.n, pa.tok0, pa.first_lb, pa.dst});
      row += pa.n;
    }
    int err =
        p->e4m3()
            ? pkv::launch_append_e4m3(p->k_pool, p->v_pool, p->kv_scales,
                                      p->num_blocks, p->num_layers,
                                      p->num_kv_heads, p->head_dim, k_new,
                                      v_new, (int32_t)total, runs, stream)
            : pkv::launch_append_batch(p->k_pool, p->v_pool, k_new, v_new,
                                       p->num_blocks, p->num_layers,
                                       p->num_kv_heads, p->head_dim,
                                       (int32_t)total, runs, stream);
    if (err) return fail(KV_ERR_CUDA, "batch append launch failed (cuda %d)", err);
  } else if (!p->has_data() && (k_new || v_new)) {
    return fail(KV_ERR_INVALID_ARG, "metadata-only pool takes no data");
  }
  commit_appends(p, plan, fresh);
  return KV_OK;
}

extern "C" kv_status kv_fork_branches(kv_pool* p, int32_t parent, int32_t n,
                                      int32_t* out_children, void* stream) {
  pkv::clear_error();
  Node* pn;
  if (kv_status s = get_live(p, parent, &pn)) return s;
  if (n < 1 || !out_children)
    return fail(KV_ERR_INVALID_ARG, "fork count must be >= 1 with an output");
  if (pn->spilled)
    return fail(KV_ERR_INVALID_ARG, "branch %d is spilled: restore it first",
                parent);
  if (p->nodes.size() + (size_t)n > (size_t)INT32_MAX)
    return fail(KV_ERR_INVALID_ARG, "branch id space exhausted");
  const int32_t B = p->block_size;
  const int32_t full = pn->seq_len / B;
  const bool partial = pn->seq_len % B != 0;
  if (partial && (int64_t)n > (int64_t)p->free_stack.size())
    return fail(KV_ERR_OOM, "fork of %d children needs %d copy-on-write "
                            "blocks, %zu free", n, n, p->free_stack.size());
  std::vector<int32_t> src, dst;
  if (partial) {
    for (int32_t i = 0; i < n; ++i) {
      src.push_back(pn->table[full]);
      dst.push_back(p->free_stack[p->free_stack.size() - 1 - i]);
    }
    if (p->has_data()) {
      const pkv::PoolBufs dev{p->k_pool, p->v_pool, p->kv_scales,
                              p->num_blocks};
      int err = pkv::launch_block_move(dev, dev, p->num_layers,
                                       p->tile_bytes(), p->scale_bytes(),
                                       src.data(), dst.data(), n, stream);
      if (err)
        return fail(KV_ERR_CUDA, "copy-on-write launch failed (cuda %d)", err);
    }
  }
  // Commit.  (pn may move when nodes grows: keep the index.)
  const int32_t depth = pn->depth + 1, seq_len = pn->seq_len;
  std::vector<int32_t> shared(pn->table.begin(), pn->table.begin() + full);
  for (int32_t i = 0; i < n; ++i) {
    Node c;
    c.parent = parent;
    c.depth = depth;
    c.inherited = full;
    c.seq_len = seq_len;
    c.table = shared;
    for (int32_t b : shared) p->ref[b] += 1;
    if (partial) {
      int32_t b = p->free_stack.back();
      p->free_stack.pop_back();
      p->ref[b] = 1;
      c.table.push_back(b);
    }
    p->nodes.push_back(std::move(c));
    const int32_t cid = (int32_t)p->nodes.size() - 1;
    p->nodes[parent].children.push_back(cid);
    out_children[i] = cid;
  }
  return KV_OK;
}

extern "C" kv_status kv_fork_branch(kv_pool* p, int32_t parent,
                                    int32_t* out_child, void* stream) {
  return kv_fork_branches(p, parent, 1, out_child, stream);
}

static void release_node(kv_pool* p, Node& nd) {
  for (int32_t b : nd.table) {
    if (b < 0) {
      p->host_free.push_back(spill_slot(b));   // a spilled block's host slot
      continue;
    }
    if (--p->ref[b] == 0) p->free_stack.push_back(b);
  }
  nd.spilled = 0;
  nd.table.clear();
  nd.table.shrink_to_fit();
  nd.seq_len = 0;
  nd.live = false;
}

extern "C" kv_status kv_free(kv_pool* p, int32_t id) {
  pkv::clear_error();
  Node* nd;
  if (kv_status s = get_live(p, id, &nd)) return s;
  release_node(p, *nd);
  return KV_OK;
}

static void free_subtree_rec(kv_pool* p, int32_t id, std::vector<int32_t>* freed) {
  // Iterative post-order (trees can be deep).
  std::vector<std::pair<int32_t, size_t>> st{{id, 0}};
  while (!st.empty()) {
    auto& [x, i] = st.back();
    if (i < p->nodes[x].children.size()) {
      int32_t c = p->nodes[x].children[i++];
      st.push_back({c, 0});
    } else {
      if (p->nodes[x].live) {
        release_node(p, p->nodes[x]);
        freed->push_back(x);
      }
      st.pop_back();
    }
  }
}

extern "C" kv_status kv_free_subtree(kv_pool* p, int32_t id,
                                     int32_t* out_n_freed,
                                     int32_t* out_freed_ids) {
  pkv::clear_error();
  if (!p) return fail(KV_ERR_INVALID_ARG, "null pool");
  if (id < 0 || id >= (int32_t)p->nodes.size())
    return fail(KV_ERR_NOT_FOUND, "branch %d does not exist", id);
  std::vector<int32_t> freed;
  free_subtree_rec(p, id, &freed);
  if (out_n_freed) *out_n_freed = (int32_t)freed.size();
  if (out_freed_ids) std::copy(freed.begin(), freed.end(), out_freed_ids);
  return KV_OK;
}

static kv_status sorted_by_omega(kv_pool* p, int32_t n, const int32_t* ids,
                                 const double* scores,
                                 std::vector<int32_t>* out) {
  if (!p) return fail(KV_ERR_INVALID_ARG, "null pool");
  if (n < 0 || (n > 0 && (!ids || !scores)))
    return fail(KV_ERR_INVALID_ARG, "bad candidate arrays");
  std::vector<std::pair<double, int32_t>> keyed(n);
  for (int32_t i = 0; i < n; ++i) {
    if (ids[i] < 0 || ids[i] >= (int32_t)p->nodes.size())
      return fail(KV_ERR_NOT_FOUND, "branch %d does not exist", ids[i]);
    if (std::isnan(scores[i]))
      return fail(KV_ERR_INVALID_ARG, "NaN score for branch %d", ids[i]);
    // omega = branch_score / (depth + 1), in binary64.
    keyed[i] = {scores[i] / (double)(p->nodes[ids[i]].depth + 1), ids[i]};
  }
  std::sort(keyed.begin(), keyed.end());
  out->resize(n);
  for (int32_t i = 0; i < n; ++i) (*out)[i] = keyed[i].second;
  return KV_OK;
}

extern "C" kv_status kv_evict_order(kv_pool* p, int32_t n, const int32_t* ids,
                                    const double* scores, int32_t* out_sorted) {
  pkv::clear_error();
  if (n > 0 && !out_sorted) return fail(KV_ERR_INVALID_ARG, "null output");
  std::vector<int32_t> order;
  if (kv_status s = sorted_by_omega(p, n, ids, scores, &order)) return s;
  std::copy(order.begin(), order.end(), out_sorted);
  return KV_OK;
}

extern "C" kv_status kv_evict(kv_pool* p, int32_t n, const int32_t* ids,
                              const double* scores, int32_t stop_kind,
                              int64_t target, int32_t* out_n_evicted,
                              int32_t* out_evicted_ids) {
  pkv::clear_error();
  if (stop_kind != KV_STOP_FREE_BLOCKS && stop_kind != KV_STOP_EVICTED_LEAVES)
    return fail(KV_ERR_INVALID_ARG, "unknown stop rule %d", stop_kind);
  std::vector<int32_t> order;
  if (kv_status s = sorted_by_omega(p, n, ids, scores, &order)) return s;
  int32_t n_ev = 0;
  int64_t leaves = 0;
  std::vector<int32_t> freed;
  for (int32_t id : order) {
    if (stop_kind == KV_STOP_FREE_BLOCKS &&
        (int64_t)p->free_stack.size() >= target)
      break;
    if (stop_kind == KV_STOP_EVICTED_LEAVES && leaves >= target) break;
    freed.clear();
    free_subtree_rec(p, id, &freed);
    if (freed.empty()) continue;
    if (out_evicted_ids) out_evicted_ids[n_ev] = id;
    ++n_ev;
    for (int32_t x : freed)
      if (p->nodes[x].children.empty()) ++leaves;
  }
  if (out_n_evicted) *out_n_evicted = n_ev;
  return KV_OK;
}

extern "C" kv_status kv_branch_info(kv_pool* p, int32_t id,
                                    kv_branch_info_t* out) {
  pkv::clear_error();
  if (!p || !out) return fail(KV_ERR_INVALID_ARG, "null argument");
  if (id < 0 || id >= (int32_t)p->nodes.size())
    return fail(KV_ERR_NOT_FOUND, "branch %d does not exist", id);
  const Node& nd = p->nodes[id];
  out->live = nd.live ? 1 : 0;
  out->parent = nd.parent;
  out->depth = nd.depth;
  out->seq_len = nd.seq_len;
  out->n_blocks = (int32_t)nd.table.size();
  out->n_children = (int32_t)nd.children.size();
  return KV_OK;
}

extern "C" kv_status kv_get_block_table(kv_pool* p, int32_t id, int32_t* out,
                                        int32_t cap, int32_t* out_n,
                                        int32_t* out_seq_len) {
  pkv::clear_error();
  Node* nd;
  if (kv_status s = get_live(p, id, &nd)) return s;
  const int32_t n = (int32_t)nd->table.size();
  if (out_n) *out_n = n;
  if (out_seq_len) *out_seq_len = nd->seq_len;
  if (out) {
    if (cap < n) return fail(KV_ERR_INVALID_ARG, "cap %d < table %d", cap, n);
    std::copy(nd->table.begin(), nd->table.end(), out);
  }
  return KV_OK;
}

extern "C" kv_status kv_get_refcounts(kv_pool* p, int32_t* out) {
  pkv::clear_error();
  if (!p || !out) return fail(KV_ERR_INVALID_ARG, "null argument");
  std::copy(p->ref.begin(), p->ref.end(), out);
  return KV_OK;
}

extern "C" kv_status kv_get_free_stack(kv_pool* p, int32_t* out, int64_t cap,
                                       int64_t* out_n) {
  pkv::clear_error();
  if (!p) return fail(KV_ERR_INVALID_ARG, "null pool");
  const int64_t n = (int64_t)p->free_stack.size();
  if (out_n) *out_n = n;
  if (out) {
    if (cap < n) return fail(KV_ERR_INVALID_ARG, "cap too small");
    std::copy(p->free_stack.rbegin(), p->free_stack.rend(), out);
  }
  return KV_OK;
}

extern "C" kv_status kv_num_branches(kv_pool* p, int32_t* out_n) {
  pkv::clear_error();
  if (!p || !out_n) return fail(KV_ERR_INVALID_ARG, "null argument");
  *out_n = (int32_t)p->nodes.size();
  return KV_OK;
}

extern "C" kv_status kv_batch_max_blocks(kv_pool* p, int32_t nb,
                                         const int32_t* ids,
                                         int32_t* out_max) {
  pkv::clear_error();
  if (!out_max || nb < 0 || (nb > 0 && !ids))
    return fail(KV_ERR_INVALID_ARG, "bad arguments");
  int32_t mx = 0;
  for (int32_t b = 0; b < nb; ++b) {
    Node* nd;
    if (kv_status s = get_live(p, ids[b], &nd)) return s;
    mx = std::max(mx, (int32_t)nd->table.size());
  }
  *out_max = mx;
  return KV_OK;
}

// Segments = nested runs of consecutive rows sharing a prefix of full blocks.
// lcp[i] = shared full blocks of rows i and i + 1.  For rows [lo, hi) whose
// common prefix is known to be >= base: the run's own common prefix l is
// min(lcp[lo .. hi-2]); if l > base the run is a segment over blocks
// [base, l); the run then splits where lcp == l and each part recurses with
// base = l.  Each row's segments tile [0, deepest end) with no gap.
static void emit_segments(const std::vector<int32_t>& lcp, int32_t lo,
                          int32_t hi, int32_t base,
                          std::vector<int32_t>* groups) {
  struct Frame { int32_t lo, hi, base; };
  std::vector<Frame> st{{lo, hi, base}};
  while (!st.empty()) {
    Frame f = st.back();
    st.pop_back();
    if (f.hi - f.lo < 2) continue;
    int32_t l = INT32_MAX;
    for (int32_t i = f.lo; i < f.hi - 1; ++i) l = std::min(l, lcp[i]);
    if (l > f.base) {
      groups->insert(groups->end(), {f.lo, f.hi - f.lo, f.base, l - f.base});
    }
    const int32_t nb = std::max(l, f.base);
    // Children in reverse so they pop in row order.
    std::vector<Frame> kids;
    int32_t s = f.lo;
    for (int32_t i = f.lo; i < f.hi - 1; ++i) {
      if (lcp[i] == l) {
        kids.push_back({s, i + 1, nb});
        s = i + 1;
      }
    }
    kids.push_back({s, f.hi, nb});
    if (kids.size() == 1) continue;  // no split: nothing deeper is common
    for (auto it = kids.rbegin(); it != kids.rend(); ++it) st.push_back(*it);
  }
}

extern "C" kv_status kv_build_batch(kv_pool* p, int32_t nb, const int32_t* ids,
                                    int32_t max_blocks, int32_t* tables,
                                    int32_t* seq_lens, int32_t groups_cap,
                                    int32_t* out_n_groups, int32_t* groups) {
  pkv::clear_error();
  if (!p) return fail(KV_ERR_INVALID_ARG, "null pool");
  if (nb < 1 || !ids || !tables || !seq_lens || !out_n_groups)
    return fail(KV_ERR_INVALID_ARG, "bad arguments");
  std::vector<const Node*> rows(nb);
  for (int32_t b = 0; b < nb; ++b) {
    Node* nd;
    if (kv_status s = get_live(p, ids[b], &nd)) return s;
    if ((int32_t)nd->table.size() > max_blocks)
      return fail(KV_ERR_INVALID_ARG, "branch %d has %zu blocks > max_blocks "
                  "%d", ids[b], nd->table.size(), max_blocks);
    if (nd->seq_len < 1)
      return fail(KV_ERR_INVALID_ARG, "branch %d is empty", ids[b]);
    if (nd->spilled)
      return fail(KV_ERR_INVALID_ARG, "branch %d is spilled: restore it first",
                  ids[b]);
    rows[b] = nd;
  }
  const int32_t B = p->block_size;
  // A lower bound on the common prefix of two branches' tables, in blocks,
  // from fork ancestry: a child shares its parent's full blocks at the fork,
  // and those entries never change while both branches hold them (full
  // blocks are immutable, and a block held twice is never spilled or moved).
  // So two branches agree on the smallest such count along their paths to
  // their lowest common ancestor.  Branches with no common ancestor (e.g.
  // made from the radix index) get 0, and the comparison below does the rest.
  auto ancestry_floor = [&](int32_t a, int32_t c) -> int32_t {
    int32_t fa = INT32_MAX, fc = INT32_MAX;
    while (a != c) {
      if (a < 0 || c < 0) return 0;
      const Node& na = p->nodes[a];
      const Node& nc = p->nodes[c];
      if (na.depth >= nc.depth) {
        fa = std::min(fa, na.inherited);
        a = na.parent;
      } else {
        fc = std::min(fc, nc.inherited);
        c = nc.parent;
      }
    }
    return std::min(fa, fc);
  };
  std::vector<int32_t> lcp(nb > 1 ? nb - 1 : 0);
  for (int32_t i = 0; i + 1 < nb; ++i) {
    const Node* a = rows[i];
    const Node* c = rows[i + 1];
    const int32_t lim = std::min(a->seq_len / B, c->seq_len / B);
    const int32_t* x = a->table.data();
    const int32_t* y = c->table.data();
    int32_t j = std::min(ancestry_floor(ids[i], ids[i + 1]), lim);
    // Whole 64-entry chunks with memcmp, then entry by entry.
    while (j + 64 <= lim && std::memcmp(x + j, y + j, 64 * sizeof(int32_t)) == 0)
      j += 64;
    while (j < lim && x[j] == y[j]) ++j;
    lcp[i] = j;
  }
  std::vector<int32_t> seg;
  if (nb > 1) emit_segments(lcp, 0, nb, 0, &seg);
  const int32_t ng = (int32_t)(seg.size() / 4);
  if (ng > groups_cap || (ng > 0 && !groups))
    return fail(KV_ERR_INVALID_ARG, "groups_cap %d < %d segments", groups_cap,
                ng);
  for (int32_t b = 0; b < nb; ++b) {
    int32_t* row = tables + (int64_t)b * max_blocks;
    const auto& t = rows[b]->table;
    std::copy(t.begin(), t.end(), row);
    std::fill(row + t.size(), row + max_blocks, -1);
    seq_lens[b] = rows[b]->seq_len;
  }
  std::copy(seg.begin(), seg.end(), groups);
  *out_n_groups = ng;
  return KV_OK;
}

// ---- host tier: spill and restore ------------------------------------------
// "Dismantling the Memory Wall", cross-tier offload: blocks leave HBM for
// host memory instead of being dropped, and come back before use.

extern "C" kv_status kv_offload_attach(kv_pool* p, void* host_k, void* host_v,
                                       void* host_scales, int64_t host_slots) {
  pkv::clear_error();
  if (!p) return fail(KV_ERR_INVALID_ARG, "null pool");
  if (host_slots < 1 || host_slots > (int64_t)INT32_MAX / 2)
    return fail(KV_ERR_INVALID_ARG, "host_slots out of range");
  if ((host_k == nullptr) != (host_v == nullptr))
    return fail(KV_ERR_INVALID_ARG, "host_k and host_v both set or both NULL");
  if (p->has_data() != (host_k != nullptr))
    return fail(KV_ERR_INVALID_ARG, "a data pool needs host buffers; a "
                                    "metadata-only pool takes none");
  if (((uintptr_t)host_k | (uintptr_t)host_v | (uintptr_t)host_scales) & 15)
    return fail(KV_ERR_INVALID_ARG, "host buffers must be 16-byte aligned");
  if ((host_scales != nullptr) != (p->has_data() && p->e4m3()))
    return fail(KV_ERR_INVALID_ARG, "host_scales is required for an e4m3 data "
                                    "pool and must be NULL otherwise");
  if (p->host_slots > 0)
    return fail(KV_ERR_INVALID_ARG, "a host tier is already attached");
  p->host_k = host_k;
  p->host_v = host_v;
  p->host_scales = host_scales;
  p->host_slots = host_slots;
  p->host_free.resize(host_slots);
  for (int64_t i = 0; i < host_slots; ++i)
    p->host_free[i] = (int32_t)(host_slots - 1 - i);  // slot 0 handed out first
  return KV_OK;
}

extern "C" kv_status kv_spill(kv_pool* p, int32_t n, const int32_t* ids,
                              void* stream, int32_t* out_n_blocks) {
  pkv::clear_error();
  if (!p) return fail(KV_ERR_INVALID_ARG, "null pool");
  if (p->host_slots < 1) return fail(KV_ERR_INVALID_ARG, "no host tier attached");
  if (n < 0 || (n > 0 && !ids)) return fail(KV_ERR_INVALID_ARG, "bad ids");
  // Blocks owned by one branch alone go to the host; shared ones stay.
  std::vector<int32_t> src, dst;
  std::vector<char> taken(p->num_blocks, 0);
  for (int32_t i = 0; i < n; ++i) {
    Node* nd;
    if (kv_status s = get_live(p, ids[i], &nd)) return s;
    for (int32_t b : nd->table)
      if (b >= 0 && p->ref[b] == 1 && !taken[b]) {
        taken[b] = 1;
        src.push_back(b);
      }
  }
  if (src.size() > p->host_free.size())
    return fail(KV_ERR_OOM, "spill needs %zu host slots, %zu free", src.size(),
                p->host_free.size());
  for (size_t k = 0; k < src.size(); ++k)
    dst.push_back(p->host_free[p->host_free.size() - 1 - k]);
  if (p->has_data() && !src.empty()) {
    const pkv::PoolBufs dev{p->k_pool, p->v_pool, p->kv_scales, p->num_blocks};
    const pkv::PoolBufs host{p->host_k, p->host_v, p->host_scales,
                             p->host_slots};
    int err = pkv::launch_block_move(dev, host, p->num_layers, p->tile_bytes(),
                                     p->scale_bytes(), src.data(), dst.data(),
                                     (int)src.size(), stream);
    if (err) return fail(KV_ERR_CUDA, "spill copy launch failed (cuda %d)", err);
  }
  // Commit in the same order the slots were taken.
  size_t k = 0;
  for (int32_t i = 0; i < n; ++i) {
    Node& nd = p->nodes[ids[i]];
    for (int32_t& b : nd.table) {
      if (b < 0 || k >= src.size() || src[k] != b) continue;
      p->host_free.pop_back();
      p->ref[b] = 0;
      p->free_stack.push_back(b);
      b = spill_code(dst[k]);
      ++nd.spilled;
      ++k;
    }
  }
  if (out_n_blocks) *out_n_blocks = (int32_t)src.size();
  return KV_OK;
}

extern "C" kv_status kv_restore(kv_pool* p, int32_t n, const int32_t* ids,
                                void* stream, int32_t* out_n_blocks) {
  pkv::clear_error();
  if (!p) return fail(KV_ERR_INVALID_ARG, "null pool");
  if (n < 0 || (n > 0 && !ids)) return fail(KV_ERR_INVALID_ARG, "bad ids");
  std::vector<int32_t> src, dst;
  for (int32_t i = 0; i < n; ++i) {
    Node* nd;
    if (kv_status s = get_live(p, ids[i], &nd)) return s;
    for (int32_t j = 0; j < i; ++j)
      if (ids[j] == ids[i])
        return fail(KV_ERR_INVALID_ARG, "branch %d listed twice", ids[i]);
    for (int32_t b : nd->table)
      if (b < 0) src.push_back(spill_slot(b));
  }
  if (src.size() > p->free_stack.size())
    return fail(KV_ERR_OOM, "restore needs %zu blocks, %zu free", src.size(),
                p->free_stack.size());
  for (size_t k = 0; k < src.size(); ++k)
    dst.push_back(p->free_stack[p->free_stack.size() - 1 - k]);
  if (p->has_data() && !src.empty()) {
    const pkv::PoolBufs dev{p->k_pool, p->v_pool, p->kv_scales, p->num_blocks};
    const pkv::PoolBufs host{p->host_k, p->host_v, p->host_scales,
                             p->host_slots};
    int err = pkv::launch_block_move(host, dev, p->num_layers, p->tile_bytes(),
                                     p->scale_bytes(), src.data(), dst.data(),
                                     (int)src.size(), stream);
    if (err)
      return fail(KV_ERR_CUDA, "restore copy launch failed (cuda %d)", err);
  }
  size_t k = 0;
  for (int32_t i = 0; i < n; ++i) {
    Node& nd = p->nodes[ids[i]];
    for (int32_t& b : nd.table) {
      if (b >= 0) continue;
      p->free_stack.pop_back();
      p->ref[dst[k]] = 1;
      p->host_free.push_back(spill_slot(b));
      b = dst[k];
      ++k;
    }
    nd.spilled = 0;
  }
  if (out_n_blocks) *out_n_blocks = (int32_t)src.size();
  return KV_OK;
}

extern "C" kv_status kv_get_host_free(kv_pool* p, int32_t* out, int64_t cap,
                                      int64_t* out_n) {
  pkv::clear_error();
  if (!p) return fail(KV_ERR_INVALID_ARG, "null pool");
  const int64_t n = (int64_t)p->host_free.size();
  if (out_n) *out_n = n;
  if (out) {
    if (cap < n) return fail(KV_ERR_INVALID_ARG, "cap too small");
    std::copy(p->host_free.rbegin(), p->host_free.rend(), out);
  }
  return KV_OK;
}
