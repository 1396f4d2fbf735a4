// Internal declarations shared by the host library and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "augtree.h"

namespace augtree {

enum ItemKind { K_PREFILL_Q = 0, K_REPLAY_Q = 1, K_PROMPT_KV = 2, K_RESP_KV = 3, K_PREFILL_KV = 4, K_TREE_PROMPT_KV = 5 };
constexpr int kNumOps = 5;  // queues per plan: the four calls' ops and the fused backward
constexpr int kMaxSplit = 64;
// Split-KV of the replay forward: KV tiles per split at least, partial states per plan
// at most, and a block's fixed cost (prologue, partial write) in KV tiles for the
// choice of the chunk.
constexpr int kFwdMinChunk = 4;
constexpr int64_t kMaxFwdParts = 4096;
constexpr int kFwdBlockOverhead = 2;
// Limit of a device-side wait on another warp's work: default and largest settable.
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;
constexpr uint64_t kMaxWaitLimitNs = 60000000000ull;
// The plan's error block, 32 bytes of device memory: word 0 error bits, word 1
// reserved, words 2-3 the wait limit (ns), then per forward op (prefill, replay) the two
// work counters of the persistent forward (next item, finished blocks), zero between
// launches.
constexpr int kErrBlockWords = 8;
constexpr int kErrFwdCounter = 4;

// Per-group geometry on the device: first prompt row, prompt length, first response
// row, total response length of the group's branches, and the group's first 128-row
// query tile on the prompt side and on the response side in the tiled backward
// row-statistics buffer (tensor-core family).
struct GroupInfo {
  int32_t p0, lp, r0, lr;
  int32_t tp0, tr0;
};
constexpr int kStatRows = 128;  // rows per tile of the backward row-statistics buffer
constexpr int kTcBwdKvRows = 128;  // query rows per tile of the tensor-core key-side backward (128 or 64)

// Per-group split-K bookkeeping of the replay backward (prompt dK/dV partials).
struct SplitInfo {
  int32_t nsplit;     // 0: group has no prompt-KV items; 1: written in place; >1: partials
  int32_t pad;
  int64_t part_row0;  // first row of the group's partial block in the workspace
};

// Split-KV of the replay forward, per 128-row response query tile (numbered like the
// row statistics, GroupInfo::tr0 + tile): split k of the tile walks its KV tiles
// [k * chunk, min((k + 1) * chunk, a + b)); a tile with nsplit > 1 writes partial states
// (forward: fp32 O / l and lse; query-side backward: fp32 dQ) to slots
// slot0 + head * nsplit + k.
struct FwdSplit {
  int32_t nsplit;
  int32_t chunk;
  int64_t slot0;
};
constexpr int kFwdPartRows = 128;  // rows of one partial slot (the forward query tile)

// Pointers a kernel needs to interpret queue items.
struct Geometry {
  const GroupInfo* groups;    // [n_groups]
  const int32_t* row_bstart;  // [total_resp] first response row of each row's branch
  const SplitInfo* splits;    // [n_groups] (replay backward only)
  const FwdSplit* fsplit;     // [ntiles_r] replay forward split-KV, null if no tile splits
  int32_t hq, hkv, d;
  int32_t total_prompt, total_resp;
  int32_t n_groups;
  float scale;                // softmax scale s
  float scale_log2;           // s * log2(e)
};

// Persistent schedule: a kernel's units placed on lanes (one persistent block each).
struct LaneSet {
  std::vector<int32_t> off, units;  // CSR on the host: lane l runs units[off[l] .. off[l+1])
  int32_t* off_d = nullptr;
  int32_t* units_d = nullptr;
  int32_t n_lanes = 0;
};
}  // namespace augtree

struct augtree_plan {
  augtree_config cfg;
  int device;
  int family;  // AUGTREE_KERNEL_SIMT or AUGTREE_KERNEL_TC
  int32_t n_groups, n_branches, total_prompt, total_resp;
  int32_t bm[augtree::kNumOps], bn[augtree::kNumOps];
  std::vector<augtree::GroupInfo> groups_h;
  std::vector<augtree::SplitInfo> splits_h;
  int64_t part_rows;  // rows of split partials (per dK and per dV), over all groups
  // Replay forward split-KV (tensor-core family): per response query tile its split
  // info; the (group, tile) pairs of the split tiles; the number of partial slots.
  std::vector<augtree::FwdSplit> fsplit_h;
  std::vector<int32_t> fsplit_tiles_h;
  int64_t n_fwd_parts;
  std::vector<int32_t> queue_h[augtree::kNumOps];
  size_t n_items[augtree::kNumOps];
  // device copies
  augtree::GroupInfo* groups_d;
  int32_t* row_bstart_d;
  int32_t* row_bend_d;  // [total_resp] one past the last response row of each row's branch
  augtree::SplitInfo* splits_d;
  augtree::FwdSplit* fsplit_d;      // null when no replay query tile is split
  int32_t* fsplit_tiles_d;
  int32_t* queue_d[augtree::kNumOps];
  int32_t ntiles_p, ntiles_r;  // 128-row query tiles per side (row-statistics buffer)
  uint32_t* err_d;    // error block (kErrBlockWords): error bits, the wait limit (ns), work counters
  // Persistent schedule (cfg.schedule == AUGTREE_SCHED_PERSISTENT, tensor-core family):
  // lanes of the query-side backward (over the forward queues) and of the key-side
  // backward, per op.
  augtree::LaneSet lanes_dq[2], lanes_kv[augtree::kNumOps];
  // Device address of the library's fixed scratch array (augtree_prefill_bwd_static),
  // looked up at plan creation on the plan's device; null if that lookup failed.
  void* static_scratch;
  // Opt-in per-kernel timing: a ring of AUGTREE_TIMING_RING calls per op, each with up
  // to kTimingMarks events (before each kernel, after the last).  Written by the compute
  // calls, which take the plan as const.
  static constexpr int kTimingMarks = 8;
  struct Timing {
    bool on = false;
    bool created = false;
    cudaEvent_t ev[augtree::kNumOps][AUGTREE_TIMING_RING][kTimingMarks];
    int32_t kind[augtree::kNumOps][AUGTREE_TIMING_RING][kTimingMarks];
    int32_t n_marks[augtree::kNumOps][AUGTREE_TIMING_RING] = {};
    uint32_t calls[augtree::kNumOps] = {};
  };
  mutable Timing timing;
};

namespace augtree {

// Persistent schedule: places the units of `queue` (unit_items consecutive items each)
// on min(lanes, U) lanes with augtree_assign_grid.
augtree_status build_lanes(const std::vector<int32_t>& queue, int unit_items, int lanes, LaneSet& out);

// Work-queue build shared by augtree_schedule_build and augtree_plan_create.
// split_fwd: apply the replay forward's split-KV rule (tensor-core family).
augtree_status build_queue(const std::vector<int32_t>& prompt_off, const std::vector<int32_t>& branch_begin,
                           const std::vector<int32_t>& resp_off, int hq, int hkv, int op, int bm, int bn,
                           int num_sms, bool split_fwd, std::vector<int32_t>& out);
// Split counts of the replay query tiles with the given KV-tile costs.
void replay_fwd_splits(const std::vector<int64_t>& costs, int hq, int hkv, int num_sms, std::vector<int64_t>& splits);

// Workspace of the replay forward with split-KV: fp32 O partials [n_parts][128][D],
// then fp32 lse partials [n_parts][128].
struct FwdWorkspace {
  size_t o_off, lse_off, total;
};
FwdWorkspace replay_fwd_ws(const augtree_plan* p);

// Workspace layout of the backward calls.  dqpart: fp32 dQ partials of the split replay
// query tiles [n_fwd_parts][128][D] (tensor-core family).
struct BwdWorkspace {
  size_t delta_off, aug_off, dq_off, dkpart_off, dvpart_off, dqpart_off, slots_off, total;
};
constexpr int kAugTileBytes = 2 * kStatRows * 16;  // {L, D} rows of one query tile
// fp32 flush slots of the tensor-core backward: one per SM id, 128 keys x 256 floats.
constexpr int kFlushSlots = 256;
constexpr size_t kFlushSlotBytes = (size_t)128 * 256 * 4;
BwdWorkspace replay_bwd_ws(const augtree_plan* p);
BwdWorkspace prefill_bwd_ws(const augtree_plan* p);
// Fused backward: the replay layout (with the flush slots), then the prefill layout up
// to its slots, then (SIMT family only) the fp32 prompt-gradient sums.
struct TreeWorkspace {
  BwdWorkspace r, p;
  size_t p_off, sum_off, sum_bytes, total;
};
TreeWorkspace tree_bwd_ws(const augtree_plan* p);

Geometry geometry(const augtree_plan* p);

// Records the timing marks of one compute call (no-op unless the plan's timing is on):
// mark(kind) before each kernel launch, then finish() after the last one.
class CallTimer {
 public:
  CallTimer(const augtree_plan* p, int op, cudaStream_t s);
  void mark(int kind);
  void finish();

 private:
  const augtree_plan* p_;
  int op_, slot_, n_;
  cudaStream_t s_;
};

// 3-D TMA map over a [rows, heads, 128] bf16 tensor (box 64 x 1 x box_rows, 128-byte
// swizzle, zero fill outside the tensor).
bool encode_rows_map(CUtensorMap* map, const void* ptr, int64_t rows, int heads, int box_rows);
// Same over a [rows, heads, 128] fp32 tensor, box 128 x 1 x box_rows, no swizzle.
bool encode_f32_rows_map(CUtensorMap* map, const void* ptr, int64_t rows, int heads, int box_rows);

// ---- launchers (return cudaGetLastError() of their launches) ---------------------
// SIMT family (any dtype).
cudaError_t simt_fwd(const augtree_plan* p, int op, const void* q, const void* kp, const void* vp,
                     const void* kr, const void* vr, void* o, float* lse, cudaStream_t st);
cudaError_t simt_bwd(const augtree_plan* p, int op, const void* q, const void* kp, const void* vp,
                     const void* kr, const void* vr, const float* lse, const void* dO,
                     const float* delta, float* dq_acc, void* dk_out, void* dv_out,
                     float* dk_part, float* dv_part, float* dk_sum, float* dv_sum,
                     const float* dk_add, const float* dv_add, cudaStream_t st);
// Tensor-core family (bf16).
// part_o / part_lse: the replay forward's split-KV partial states (null without split
// tiles); their merge is launch_fwd_split_merge.
cudaError_t tc_fwd(const augtree_plan* p, int op, const void* q, const void* kp, const void* vp,
                   const void* kr, const void* vr, void* o, float* lse, float* part_o, float* part_lse,
                   cudaStream_t st);
// Backward, key side (dK, dV; prompt dK/dV summed over the branches, split-K partials
// reduced afterwards) and query side (dQ, written once per query tile and head).
// Key side of the tensor-core backward.  Primary query rows q / dO / aug: the prompt for
// prefill_bwd, the responses otherwise; secondary rows q2 / dO2 / aug2: the prompt rows
// of the fused backward (nullable elsewhere).  dk2_out / dv2_out: the fused backward's
// bf16 prompt gradient of unsplit groups.
cudaError_t tc_bwd_kv(const augtree_plan* p, int op, const void* q, const void* dO, const void* aug, const void* q2,
                      const void* dO2, const void* aug2, const void* kp, const void* vp, const void* kr, const void* vr,
                      void* dk_out, void* dv_out, void* dk2_out, void* dv2_out, float* dk_part, float* dv_part,
                      float* dk_sum, float* dv_sum, const float* dk_add, const float* dv_add, float* slots,
                      cudaStream_t st);
cudaError_t tc_bwd_dq(const augtree_plan* p, int op, const void* q, const void* kp, const void* vp, const void* kr,
                      const void* vr, const float* stats, const void* dO, void* dq, float* dq_part,
                      cudaStream_t st);

// Fixed scratch array of augtree_prefill_bwd_static (static_scratch.cu): its size, and
// the lookup of its device address on the current device.
constexpr size_t kStaticScratchBytes = 64ull << 20;
cudaError_t static_scratch_address(void** out);

// Memory-bound helpers.
cudaError_t launch_preprocess(const void* o, const void* dO, int dtype, int64_t rows, int hq, int d,
                              float* delta, float* dq_acc, cudaStream_t st);
// Tensor-core backward preprocess: per (128-row query tile, head) writes 1 KB of fp32
// {lse * log2(e) [128], Delta [128]} into stats and 4 KB of bf16 rows {-lse/s, -Delta}
// split three ways into aug (zeros past the group's end).
cudaError_t launch_preprocess_tiled(const augtree_plan* p, bool prompt_side, const void* o, const void* dO,
                                    const float* lse, float* stats, void* aug, cudaStream_t st);
cudaError_t launch_dq_convert(const float* dq_acc, void* dq, int dtype, int64_t n, cudaStream_t st);
cudaError_t launch_split_reduce(const augtree_plan* p, const float* dk_part, const float* dv_part,
                                float* dk_sum, float* dv_sum, cudaStream_t st);
// Fused backward: bf16 prompt dK/dV of the split groups from their partials, in split order.
cudaError_t launch_split_reduce_final(const augtree_plan* p, const float* dk_part, const float* dv_part, void* dkp,
                                      void* dvp, cudaStream_t st);
// Replay forward split-KV: merges each split tile's partial states in split order into
// bf16 O and lse (Sec. 3.3); and sums each split tile's fp32 dQ partials in split order
// into bf16 dQ.
cudaError_t launch_fwd_split_merge(const augtree_plan* p, const float* part_o, const float* part_lse, void* o,
                                   float* lse, cudaStream_t st);
cudaError_t launch_dq_split_reduce(const augtree_plan* p, const float* dq_part, void* dq, cudaStream_t st);
cudaError_t launch_lse_merge(int64_t rows, int h, int d, const float* oa, const float* la,
                             const float* ob, const float* lb, float* o, float* l, cudaStream_t st);
cudaError_t launch_lse_merge_bwd(int64_t rows, int h, int d, const float* oa, const float* la, const float* ob,
                                 const float* lb, const float* dout, const float* dl, float* doa, float* dla,
                                 float* dob, float* dlb, cudaStream_t st);

}  // namespace augtree
