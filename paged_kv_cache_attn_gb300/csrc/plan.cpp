// Host half of a decode step: cut the step into work items for the split-KV
// kernel (rows <= 16 per item), the tcgen05 kernel (128-row tiles of large
// shared-prefix segments) and the LSE merge.
//
// Each branch's logical blocks are covered exactly once: by the segments that
// contain its row (which tile [0, shared_end) -- each segment's blocks are
// read once for all of its rows) and by its own suffix [shared_end, n_blocks).
// Every item writes unnormalised partial results (o, m, l) per query row; the
// merge combines a row's partials by their log-sum-exp.  The split sizes do
// not change the result beyond rounding.

#include <algorithm>
#include <cstring>
#include <numeric>

#include "internal.h"

using pkv::fail;

namespace {

struct Unit {
  int32_t branch0, rows, blk_begin, blk_end, masked;
  bool tile;  // tcgen05 tiles
  bool wide;  // ... of 256 rows (two M-tiles per item)
};

int rows_per(const Unit& u) {
  return u.wide ? pkv::kWideRows : u.tile ? pkv::kTileRows : pkv::kRowTile;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int32_t pick_chunk(const std::vector<Unit>& units, bool tile, int Hkv,
                   int num_sms, int32_t start) {
  int32_t chunk = start;
  for (;;) {
    int64_t items = 0;
    for (const Unit& u : units) {
      if (u.tile != tile) continue;
      // A 256-row item counts as two 128-row tiles: it carries their work.
      items += ceil_div(u.blk_end - u.blk_begin, chunk) *
               ceil_div(u.rows, rows_per(u)) * Hkv * (u.wide ? 2 : 1);
    }
    if (chunk <= 8 || items >= 2LL * num_sms) return chunk;
    chunk /= 2;
  }
}

}  // namespace

extern "C" kv_status paged_decode_plan(int32_t nb, int32_t Hq, int32_t Hkv,
                                       int32_t d, int32_t B,
                                       int32_t max_blocks,
                                       const int32_t* seq_lens,
                                       const int32_t* groups, int32_t n_groups,
                                       int32_t num_sms, int32_t flags,
                                       int32_t* plan, int64_t plan_cap,
                                       kv_decode_plan_info* info) {
  pkv::clear_error();
  if (!info || !seq_lens) return fail(KV_ERR_INVALID_ARG, "null argument");
  if (nb < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0)
    return fail(KV_ERR_INVALID_ARG, "bad nb/Hq/Hkv (%d/%d/%d)", nb, Hq, Hkv);
  if (d != 64 && d != 128)
    return fail(KV_ERR_INVALID_ARG, "head_dim must be 64 or 128");
  if (B != 16) return fail(KV_ERR_INVALID_ARG, "block_size must be 16");
  if (max_blocks < 1) return fail(KV_ERR_INVALID_ARG, "max_blocks must be >= 1");
  if (n_groups < 0 || (n_groups > 0 && !groups))
    return fail(KV_ERR_INVALID_ARG, "bad groups");
  if (num_sms <= 0) num_sms = 152;
  const int32_t G = Hq / Hkv;

  std::vector<int32_t> nblk(nb);
  for (int32_t b = 0; b < nb; ++b) {
    if (seq_lens[b] < 1 || (int64_t)seq_lens[b] > (int64_t)max_blocks * B)
      return fail(KV_ERR_INVALID_ARG, "seq_lens[%d] = %d outside [1, %lld]", b,
                  seq_lens[b], (long long)max_blocks * B);
    nblk[b] = (seq_lens[b] + B - 1) / B;
  }

  // Segments: validate and find each row's shared end.
  std::vector<int32_t> shared_end(nb, 0);
  std::vector<Unit> units;
  const bool use_groups = !(flags & KV_PLAN_IGNORE_GROUPS);
  if (flags & ~(KV_PLAN_NO_TENSOR_CORES | KV_PLAN_IGNORE_GROUPS |
                KV_PLAN_KV_E4M3 | KV_PLAN_NARROW_TILES))
    return fail(KV_ERR_INVALID_ARG, "unknown plan flags 0x%x", flags);
  // The tcgen05 tile kernels are built for head_dim 128 (bf16 and e4m3).
  const bool allow_tc = pkv::kTensorCoreKernel && d == 128 &&
                        !(flags & KV_PLAN_NO_TENSOR_CORES);
  // Segments of 129 to 256 rows run as one two-M-tile item per block range
  // (bf16 only), which reads the range once for all of their rows.  Larger
  // segments keep 128-row tiles: with no room in TMEM to double-buffer S
  // for two M-tiles, a two-M-tile item costs more SM time per row.
  const bool allow_wide =
      allow_tc && !(flags & (KV_PLAN_KV_E4M3 | KV_PLAN_NARROW_TILES));
  units.reserve((size_t)(use_groups ? n_groups : 0) + nb);
  if (use_groups && n_groups > 0) {
    // Each row's segment ranges, grouped by row with a counting sort (one
    // flat array instead of a vector per row).
    std::vector<int32_t> first(nb + 1, 0);
    for (int32_t i = 0; i < n_groups; ++i) {
      const int32_t* s = groups + 4 * (int64_t)i;
      const int32_t bb = s[0], bc = s[1], kb = s[2], kc = s[3];
      if (bb < 0 || bc < 1 || (int64_t)bb + bc > nb || kb < 0 || kc < 1)
        return fail(KV_ERR_INVALID_ARG, "segment %d {%d,%d,%d,%d} malformed",
                    i, bb, bc, kb, kc);
      if ((int64_t)bc * G > INT32_MAX / 2)
        return fail(KV_ERR_INVALID_ARG, "segment %d too many rows", i);
      for (int32_t b = bb; b < bb + bc; ++b) {
        if ((int64_t)(kb + kc) * B > seq_lens[b])
          return fail(KV_ERR_INVALID_ARG,
                      "segment %d covers a block not full for row %d", i, b);
        ++first[b + 1];
      }
      const bool tc = allow_tc && bc * G >= pkv::kMinTensorRows;
      units.push_back({bb, bc * G, kb, kb + kc, 0, tc,
                       tc && allow_wide && bc * G > pkv::kTileRows &&
                           bc * G <= pkv::kWideRows});
    }
    for (int32_t b = 0; b < nb; ++b) first[b + 1] += first[b];
    std::vector<std::pair<int32_t, int32_t>> ranges(first[nb]);
    std::vector<int32_t> next(first.begin(), first.end() - 1);
    for (int32_t i = 0; i < n_groups; ++i) {
      const int32_t* s = groups + 4 * (int64_t)i;
      for (int32_t b = s[0]; b < s[0] + s[1]; ++b)
        ranges[next[b]++] = {s[2], s[2] + s[3]};
    }
    for (int32_t b = 0; b < nb; ++b) {
      auto lo_it = ranges.begin() + first[b], hi_it = ranges.begin() + first[b + 1];
      std::sort(lo_it, hi_it);
      int32_t end = 0;
      for (auto it = lo_it; it != hi_it; ++it) {
        if (it->first != end)
          return fail(KV_ERR_INVALID_ARG,
                      "row %d: segments do not tile [0, end) (gap or overlap "
                      "at block %d)", b, it->first);
        end = it->second;
      }
      shared_end[b] = end;
    }
  }
  for (int32_t b = 0; b < nb; ++b) {
    if (shared_end[b] < nblk[b])
      units.push_back({b, G, shared_end[b], nblk[b], 1, false, false});
  }

  // Split-KV items: up to 128 blocks, halved while there are fewer than two
  // items per SM.  A tile item carries several microseconds of fixed cost
  // (TMEM, barriers, Q, the first loads, the epilogue and its 128 partial
  // rows per kv-head) and holds a whole SM, so tile items are made as long
  // as the step allows: up to the step's block work per SM (every item,
  // tile or split, moves its blocks into one SM), with the split-KV pass
  // streaming on the SMs they leave free.  Measured: the fan-out tree with
  // 256 tile items of 32 blocks 0.238 ms, 64 of 128 blocks 0.215 ms; the
  // long-context tree with tile items of 256, 512, 1024 and 2048 blocks
  // 1.037, 1.010, 0.996 and 0.987 ms.  A step with no split-KV item at all
  // halves its tile items until there are two per SM.
  int64_t block_work = 0;
  bool any_rows = false;
  for (const Unit& u : units) {
    any_rows |= !u.tile;
    block_work += (int64_t)(u.blk_end - u.blk_begin) *
                  ceil_div(u.rows, rows_per(u)) * Hkv;
  }
  const int32_t chunk_rows = pick_chunk(units, false, Hkv, num_sms, 128);
  const int32_t chunk_tile =
      any_rows ? (int32_t)std::min<int64_t>(
                     INT32_MAX, std::max<int64_t>(8, block_work / num_sms))
               : pick_chunk(units, true, Hkv, num_sms, 256);

  // Longest units first: their items come first, so the last wave of each
  // kernel is made of the short ones.  (Items of one unit have equal length
  // to within one block.)
  std::stable_sort(units.begin(), units.end(), [](const Unit& x, const Unit& y) {
    return (x.blk_end - x.blk_begin) > (y.blk_end - y.blk_begin);
  });
  std::vector<pkv::WorkItem> row_items, tile_items, wide_items;
  struct Tagged { int32_t branch; pkv::MergeEntry e; };
  std::vector<Tagged> merge_flat;
  {
    // Exact item counts and a bound on the merge entries, so that the loop
    // below never reallocates.
    int64_t n_row = 0, n_tile = 0, n_wide = 0, n_merge = 0;
    for (const Unit& u : units) {
      const int64_t nch =
          ceil_div(u.blk_end - u.blk_begin, u.tile ? chunk_tile : chunk_rows);
      const int64_t tiles = ceil_div(u.rows, rows_per(u));
      (u.wide ? n_wide : u.tile ? n_tile : n_row) += nch * tiles * Hkv;
      n_merge += nch * tiles * (rows_per(u) / G + 2);
    }
    row_items.reserve(n_row);
    tile_items.reserve(n_wide + n_tile);
    wide_items.reserve(n_wide);
    merge_flat.reserve(n_merge);
  }
  int64_t prow = 0;
  for (const Unit& u : units) {
    const int rp = rows_per(u);
    const int32_t chunk = u.tile ? chunk_tile : chunk_rows;
    const int32_t len = u.blk_end - u.blk_begin;
    const int32_t nch = (int32_t)ceil_div(len, chunk);
    for (int32_t c = 0; c < nch; ++c) {
      // Even split of the range into nch pieces.
      const int32_t lo = u.blk_begin + (int32_t)((int64_t)len * c / nch);
      const int32_t hi = u.blk_begin + (int32_t)((int64_t)len * (c + 1) / nch);
      for (int32_t row0 = 0; row0 < u.rows; row0 += rp) {
        const int32_t nrows = std::min(rp, u.rows - row0);
        const int64_t base0 = prow;
        for (int32_t g = 0; g < Hkv; ++g) {
          pkv::WorkItem it{u.branch0, g, row0, nrows, lo, hi,
                           (int32_t)(base0 + (int64_t)g * nrows), u.masked};
          (u.wide ? wide_items : u.tile ? tile_items : row_items).push_back(it);
        }
        prow += (int64_t)nrows * Hkv;
        if (prow > INT32_MAX)
          return fail(KV_ERR_INVALID_ARG, "step too large for one plan");
        // Merge entries for every branch these rows touch.
        const int32_t row1 = row0 + nrows;
        for (int32_t pb = row0 / G; pb * G < row1; ++pb) {
          const int32_t a = std::max(row0, pb * G);
          const int32_t e = std::min(row1, pb * G + G);
          merge_flat.push_back(
              {u.branch0 + pb,
               {(int32_t)(base0 + (a - row0)), nrows, a - pb * G, e - pb * G}});
        }
      }
    }
  }
  // Short split-KV items go last (stable).  When there are more of them
  // than two waves of split-KV CTAs would hold, the bf16 split-KV kernel runs
  // them one per warp, four to a CTA (a warp takes a short item about as
  // long as a CTA takes a long one, but four times as many run at once);
  // fewer of them run one per CTA, which ends the step's last wave sooner.
  // An item's partial rows do not depend on its position, so the merge
  // lists stand.
  const auto first_short = std::stable_partition(
      row_items.begin(), row_items.end(), [](const pkv::WorkItem& it) {
        return it.blk_end - it.blk_begin > pkv::kWarpItemBlocks;
      });
  // Within each part, longest items first (stable: the items of one unit
  // and chunk keep their order).  The hardware hands CTAs out in list order,
  // so this is longest-processing-time-first scheduling: the last items to
  // start are the shortest, and the pass's tail shrinks.  Items of one unit
  // differ by at most a block, so the unit order above only approximates it.
  const auto longer = [](const pkv::WorkItem& x, const pkv::WorkItem& y) {
    return x.blk_end - x.blk_begin > y.blk_end - y.blk_begin;
  };
  std::stable_sort(row_items.begin(), first_short, longer);
  std::stable_sort(first_short, row_items.end(), longer);
  int32_t n_warp_items = (int32_t)(row_items.end() - first_short);
  if (n_warp_items <= 2 * pkv::kSplitCtasPerSm * num_sms) n_warp_items = 0;
  // The 256-row tile items go first in the tile list.
  const int32_t n_wide_items = (int32_t)wide_items.size();
  tile_items.insert(tile_items.begin(), wide_items.begin(), wide_items.end());
  const int64_t n_csr = (int64_t)merge_flat.size();
  const int64_t off_row = pkv::kPlanHeaderInts;
  const int64_t off_tile = off_row + 8 * (int64_t)row_items.size();
  const int64_t off_ptr = off_tile + 8 * (int64_t)tile_items.size();
  const int64_t off_ent = off_ptr + nb + 1;
  const int64_t total = off_ent + 4 * n_csr;
  if (total > INT32_MAX) return fail(KV_ERR_INVALID_ARG, "plan too large");

  info->plan_ints = total;
  info->partial_rows = prow;
  info->workspace_bytes = (int64_t)pkv::ws_total(prow, d);
  info->n_row_items = (int32_t)row_items.size();
  info->n_row_warp_items = n_warp_items;
  info->reserved = 0;
  info->n_tile_items = (int32_t)tile_items.size();
  info->n_merge_rows = nb;
  info->chunk_blocks = chunk_rows;
  info->n_tile_wide_items = n_wide_items;
  info->flags = flags;
  if (!plan) return KV_OK;
  if (plan_cap < total)
    return fail(KV_ERR_INVALID_ARG, "plan_cap %lld < %lld", (long long)plan_cap,
                (long long)total);
  int32_t* h = plan;
  std::fill(h, h + pkv::kPlanHeaderInts, 0);
  h[pkv::H_MAGIC] = pkv::kPlanMagic;
  h[pkv::H_NB] = nb;
  h[pkv::H_HQ] = Hq;
  h[pkv::H_HKV] = Hkv;
  h[pkv::H_D] = d;
  h[pkv::H_N_ROW_ITEMS] = (int32_t)row_items.size();
  h[pkv::H_N_TILE_ITEMS] = (int32_t)tile_items.size();
  h[pkv::H_N_CSR] = (int32_t)n_csr;
  h[pkv::H_OFF_ROW_ITEMS] = (int32_t)off_row;
  h[pkv::H_OFF_TILE_ITEMS] = (int32_t)off_tile;
  h[pkv::H_OFF_CSR_PTR] = (int32_t)off_ptr;
  h[pkv::H_OFF_CSR_ENT] = (int32_t)off_ent;
  h[pkv::H_PARTIAL_ROWS] = (int32_t)prow;
  h[pkv::H_CHUNK] = chunk_rows;
  h[pkv::H_FLAGS] = flags;
  h[pkv::H_TOTAL] = (int32_t)total;
  std::memcpy(h + off_row, row_items.data(), row_items.size() * 32);
  std::memcpy(h + off_tile, tile_items.data(), tile_items.size() * 32);
  // CSR by branch (counting sort, stable).
  int32_t* ptr = h + off_ptr;
  int32_t* ent = h + off_ent;
  std::fill(ptr, ptr + nb + 1, 0);
  for (const Tagged& t : merge_flat) ++ptr[t.branch + 1];
  for (int32_t b = 0; b < nb; ++b) ptr[b + 1] += ptr[b];
  std::vector<int32_t> fill(ptr, ptr + nb);
  for (const Tagged& t : merge_flat) {
    const int32_t k = fill[t.branch]++;
    ent[4 * k + 0] = t.e.base;
    ent[4 * k + 1] = t.e.stride;
    ent[4 * k + 2] = t.e.r_lo;
    ent[4 * k + 3] = t.e.r_hi;
  }
  return KV_OK;
}

extern "C" kv_status paged_decode_attn_workspace_size(
    const kv_decode_plan_info* info, size_t* out_bytes) {
  pkv::clear_error();
  if (!info || !out_bytes) return fail(KV_ERR_INVALID_ARG, "null argument");
  *out_bytes = (size_t)info->workspace_bytes;
  return KV_OK;
}
