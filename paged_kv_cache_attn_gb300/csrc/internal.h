// Internal declarations shared by the library's translation units.
#pragma once

#include <cstdint>
#include <cstdio>
#include <string>
#include <vector>

#include "pagedkv.h"

// ---- pool state (host) -----------------------------------------------------
struct Node {
  int32_t parent = -1;
  int32_t depth = 0;
  int32_t inherited = 0;  // full blocks shared with the parent at the fork
  int32_t seq_len = 0;
  bool live = true;
  int32_t spilled = 0;  // table entries held in the host tier
  // Physical block ids; an entry -(slot + 2) is a block spilled to host slot
  // `slot` (-1 stays free for batch-table padding).
  std::vector<int32_t> table;
  std::vector<int32_t> children;
};

struct kv_pool {
  int64_t num_blocks = 0;
  int32_t block_size = 16, num_layers = 1, num_kv_heads = 1, head_dim = 128;
  void* k_pool = nullptr;
  void* v_pool = nullptr;
  int32_t kv_dtype = KV_DTYPE_BF16;
  void* kv_scales = nullptr;         // e4m3: 16-byte record per (layer, block, head)
  std::vector<int32_t> ref;          // per block
  std::vector<int32_t> free_stack;   // back() is handed out next
  std::vector<Node> nodes;           // index = branch id
  // Host tier (kv_offload_attach): caller-owned pinned host pools with the
  // device pool's layout, `host_slots` blocks each, and a LIFO stack of free
  // slots (back() handed out next).
  void* host_k = nullptr;
  void* host_v = nullptr;
  void* host_scales = nullptr;
  int64_t host_slots = 0;
  std::vector<int32_t> host_free;

  bool has_data() const { return k_pool != nullptr; }
  bool e4m3() const { return kv_dtype == KV_DTYPE_E4M3; }
  // Bytes of one (layer, block) in each of the K and V pools, and in the
  // scale pool (0 for bf16).
  int64_t tile_bytes() const {
    return (int64_t)num_kv_heads * 16 * head_dim * (e4m3() ? 1 : 2);
  }
  int64_t scale_bytes() const { return e4m3() ? (int64_t)num_kv_heads * 16 : 0; }
};

inline int32_t spill_code(int32_t slot) { return -(slot + 2); }
inline int32_t spill_slot(int32_t code) { return -code - 2; }

namespace pkv {

// ---- errors ---------------------------------------------------------------
kv_status fail(kv_status code, const char* fmt, ...);
void clear_error();

// ---- plan format ----------------------------------------------------------
// A plan is an int32 array: a header, the split-KV work items, the tensor-core
// work items, and a CSR list telling the merge pass which partial rows belong
// to each branch.
constexpr int32_t kPlanMagic = 0x31564B50;  // "PKV1"
constexpr int kPlanHeaderInts = 16;
enum PlanHeader {
  H_MAGIC = 0, H_NB, H_HQ, H_HKV, H_D, H_N_ROW_ITEMS, H_N_TILE_ITEMS, H_N_CSR,
  H_OFF_ROW_ITEMS, H_OFF_TILE_ITEMS, H_OFF_CSR_PTR, H_OFF_CSR_ENT,
  H_PARTIAL_ROWS, H_CHUNK, H_FLAGS, H_TOTAL
};

// One work item: query rows [row0, row0 + nrows) of a unit whose first branch
// is `branch0` (row r -> branch branch0 + r / G, q-head g * G + r % G), over
// logical blocks [blk_begin, blk_end) of branch0's table, for kv-head g.
// Partial results go to rows prow_base .. prow_base + nrows - 1.
// masked != 0: the unit is a single branch whose last block may be partial;
// tokens at or past seq_lens[branch0] are excluded.
struct WorkItem {
  int32_t branch0, g, row0, nrows, blk_begin, blk_end, prow_base, masked;
};
static_assert(sizeof(WorkItem) == 32, "WorkItem is 8 int32");

// Merge entry for one branch: q-heads-in-group [r_lo, r_hi) of this branch
// have partial rows base + g * stride + (r - r_lo) for kv-head g.
struct MergeEntry {
  int32_t base, stride, r_lo, r_hi;
};

constexpr bool kTensorCoreKernel = true;  // tcgen05 tile kernel available
constexpr int kTileRows = 128;      // rows of a tcgen05 tile
constexpr int kWideRows = 256;      // rows of a two-M-tile tcgen05 item
constexpr int kRowTile = 16;        // rows of an mma.sync tile
constexpr int kMinTensorRows = 65;  // segments with more rows go to tcgen05
constexpr int kWarpItemBlocks = 16; // split-KV items this short run per warp
constexpr int kSplitCtasPerSm = 3;  // resident bf16 split-KV CTAs per SM

// Workspace layout (bytes): status word block, then (m, l) pairs, then o rows.
constexpr size_t kStatusBytes = 256;
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline size_t ws_ml_offset() { return kStatusBytes; }
inline size_t ws_o_offset(int64_t rows) {
  return align_up(kStatusBytes + (size_t)rows * 8, 256);
}
inline size_t ws_total(int64_t rows, int d) {
  return align_up(ws_o_offset(rows) + (size_t)rows * d * 4, 256);
}

// Device status word (first 16 bytes of the workspace).
struct DeviceStatus {
  uint32_t code;    // 0, KV_ERR_DEVICE or KV_ERR_TIMEOUT (first recorded)
  int32_t detail;   // first bad value (block id, item index, wait site)
  uint32_t count;   // how many events were recorded
  uint32_t pad;
};

// ---- kernel launchers (state_kernels.cu, decode kernels) -------------------
// Copy appended K/V rows into their slots.  dst_blocks[i] = physical block of
// logical block first_lblock + i; rows are tokens [tok0, tok0 + n) of the
// branch (tok0 = its seq_len before the append).
int launch_append_scatter(void* k_pool, void* v_pool, const void* k_new,
                          const void* v_new, int64_t num_blocks, int L,
                          int Hkv, int d, int B, int n, int tok0,
                          const int32_t* dst_blocks, int n_dst,
                          void* stream);
// One branch's run of a batched append: input rows [row, row + n) are the
// branch's tokens tok0 .. tok0 + n - 1, landing in blocks dst[t / 16 -
// first_lblock] (t = branch token index), slot t % 16.
struct ScatterRun {
  int32_t row, n, tok0, first_lblock;
  std::vector<int32_t> dst;
};
// Scatter a batch of runs (input [L][total][Hkv][d]) in as few launches as
// the kernel parameter space allows.
int launch_append_batch(void* k_pool, void* v_pool, const void* k_new,
                        const void* v_new, int64_t num_blocks, int L, int Hkv,
                        int d, int32_t total, const std::vector<ScatterRun>& runs,
                        void* stream);
// One side of a block move: the K, V (and scale, or null) buffers of a pool
// holding `blocks` blocks per layer.  May be pinned host memory reachable
// from the device.
struct PoolBufs {
  const void* k;
  const void* v;
  const void* s;
  int64_t blocks;
};
// Copy whole blocks (every layer; K, V and scale records): block src[i] of
// `from` -> block dst[i] of `to`.  kv_bytes / s_bytes: bytes of one (layer,
// block) in each K/V buffer and in the scale buffer (multiples of 16).
int launch_block_move(const PoolBufs& from, const PoolBufs& to, int L,
                      int64_t kv_bytes, int64_t s_bytes, const int32_t* src,
                      const int32_t* dst, int n, void* stream);
// Quantising append into an e4m3 pool: the runs' rows (input bf16
// [L][total][Hkv][d]) are written block by block under the pool's block
// rule; writes to one block are applied in run order.
int launch_append_e4m3(void* k8, void* v8, void* scales, int64_t num_blocks,
                       int L, int Hkv, int d, const void* k_new,
                       const void* v_new, int32_t total,
                       const std::vector<ScatterRun>& runs, void* stream);
// One layer's newest token of every branch (k_step, v_step bf16
// [nb][Hkv][d]) quantised into slot seq_lens[b] - 1 of its block; bad table
// entries are recorded in `status` and skipped.
int launch_append_step_e4m3(void* k8, void* v8, void* scales,
                            int64_t num_blocks, int Hkv, int d,
                            const int32_t* tables, const int32_t* seq_lens,
                            int nb, int max_blocks, const void* k_step,
                            const void* v_step, DeviceStatus* status,
                            void* stream);

}  // namespace pkv
