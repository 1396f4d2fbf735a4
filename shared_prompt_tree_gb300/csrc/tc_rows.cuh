// Row geometry of the query-side tensor-core kernels (the forward and the backward's
// query side): where a query row's keys lie in each KV tile of its walk.  Also the
// persistent forward's decoded work items and the source its blocks take them from.
//
// AugTree paper, Sec. 3.2 Eq. 1 (the row's valid keys: the whole prompt of its group,
// then its own branch up to itself; causal over the prompt for prefill rows), Sec. 3.3
// (the prompt-part and own-part states merge associatively; one running state crosses
// both parts) and Sec. 3.4 (replay units taken by lanes: here persistent blocks).
#pragma once

#include "common.cuh"

namespace augtree {
namespace tc {

// Where the row's keys come from in KV tile j: prompt tiles first, then the own-branch
// tiles, and the valid columns [lo, hi] of the row in that tile.
struct FwdRowGeom {
  int64_t row;      // global query row (prompt or response rows)
  bool row_ok;      // row < end of its query tile's group
  bool prefill;
  int64_t bs;       // first response row of the row's branch (replay rows)
  int64_t p0, p_end;  // the group's prompt keys
  int64_t own0;     // first key of the own-branch tiles
  int n_a;          // number of prompt tiles
  int bn;           // keys per tile
  int j0;           // first KV tile of the item (a split item's chunk; 0 otherwise)
};

// Valid columns of the item's j-th KV tile (tile j0 + j of the row's walk), clamped to
// [-1, 128].  Rows and keys are int32 offsets (the descriptors are int32), so every
// difference below fits in 32 bits; 32-bit arithmetic measured 1.4 % faster in the
// forward than 64-bit.
__device__ __forceinline__ void fwd_valid_cols(const FwdRowGeom& g, int j_local, int& lo_i, int& hi_i) {
  const int j = j_local + g.j0;
  const bool own = j >= g.n_a;
  const int key0 = own ? (int)g.own0 + (j - g.n_a) * g.bn : (int)g.p0 + j * g.bn;
  const int row = (int)g.row;
  int lo = 0, hi;
  if (g.prefill) {
    hi = row - key0;
  } else if (!own) {
    hi = (int)g.p_end - 1 - key0;
  } else {
    lo = (int)g.bs - key0;
    hi = row - key0;
  }
  if (!g.row_ok) {
    lo = 1;
    hi = 0;
  }
  lo_i = min(max(lo, -1), 128);
  hi_i = min(max(hi, -1), 128);
}


// A forward work item decoded once by a persistent block's producer for every warp of
// the block.
struct QuerySlot {
  int32_t stop;             // 1: the block has no further item
  int32_t h;                // query head
  int32_t prefill;
  int32_t n_a;              // prompt KV tiles of the rows' walk
  int32_t n_tiles;          // KV tiles this item walks
  int32_t j0;               // first KV tile of the walk (split item), else 0
  int32_t row0, row_end;    // query rows [row0, row_end)
  int32_t own0;             // first key of the own-branch tiles
  int32_t p0, lp;           // the group's prompt keys
  int32_t pad;
  int64_t slot;             // partial-state slot of a split item, else -1
};
static_assert(sizeof(QuerySlot) <= 64, "item slot");

// The slot as read by every lane of a converged warp, each field passed through a warp
// reduction (every lane holds the same value), which tells the compiler that the value
// is the same in every lane (measured 0.5-1.7 % faster forward than the plain read).
__device__ __forceinline__ QuerySlot warp_uniform(const QuerySlot& v) {
  auto u = [](int32_t x) { return (int32_t)__reduce_max_sync(0xffffffffu, (unsigned)x); };
  QuerySlot s;
  s.stop = u(v.stop);
  s.h = u(v.h);
  s.prefill = u(v.prefill);
  s.n_a = u(v.n_a);
  s.n_tiles = u(v.n_tiles);
  s.j0 = u(v.j0);
  s.row0 = u(v.row0);
  s.row_end = u(v.row_end);
  s.own0 = u(v.own0);
  s.p0 = u(v.p0);
  s.lp = u(v.lp);
  s.pad = 0;
  const uint64_t sl = (uint64_t)v.slot;
  s.slot = (int64_t)(((uint64_t)(uint32_t)u((int32_t)(sl >> 32)) << 32) | (uint32_t)u((int32_t)(uint32_t)sl));
  return s;
}

template <bool kSplit>
__device__ __forceinline__ QuerySlot decode_query_item(const int32_t* __restrict__ queue, int idx,
                                                       const Geometry& geo, int bm, int bn, uint32_t* err) {
  QuerySlot s;
  const WorkItem it = load_item(queue, idx);
  // Checked build: the item and its split are valid for the plan's geometry.
  const bool item_ok = !kChecked || (query_item_ok(it, geo, bm, bn) &&
                                     (kSplit ? split_item_ok(it, geo) : it.split == 0));
  if (kChecked && !item_ok) atomicOr(err, kErrCheck);
  const GroupInfo G = geo.groups[item_ok ? it.group : 0];
  s.stop = 0;
  s.h = item_ok ? it.head : 0;
  s.prefill = it.kind == K_PREFILL_Q ? 1 : 0;
  const int base = s.prefill ? G.p0 : G.r0, len = s.prefill ? G.lp : G.lr;
  s.row0 = item_ok ? base + it.tile * bm : 0;
  s.row_end = item_ok ? min(s.row0 + bm, base + len) : 0;
  s.n_a = item_ok ? it.a : 0;
  s.n_tiles = item_ok ? s.n_a + (s.prefill ? 0 : it.b) : 0;
  s.own0 = (s.prefill || !item_ok) ? 0 : geo.row_bstart[s.row0];
  s.p0 = G.p0;
  s.lp = G.lp;
  s.pad = 0;
  s.j0 = 0;
  s.slot = -1;
  if (kSplit && item_ok && !s.prefill) {
    const FwdSplit fs = geo.fsplit[G.tr0 + it.tile];
    if (fs.nsplit > 1) {
      s.j0 = it.split * fs.chunk;
      s.n_tiles = min(fs.chunk, s.n_tiles - s.j0);
      s.slot = fs.slot0 + (int64_t)s.h * fs.nsplit + it.split;
    }
  }
  return s;
}

// Where a persistent block takes its work items: in queue order through two words of
// the plan's device memory (the next item, the blocks that have finished taking items;
// zero between launches), or, with kLanes, from its lane of a static placement.
template <bool kLanes>
struct ItemSource {
  unsigned* ctr;
  const int32_t* units;  // the lane's units (kLanes)
  int n_lane;            // their number
  unsigned n_items;
  int taken;
  __device__ __forceinline__ unsigned next() {
    if constexpr (kLanes) {
      const int k = taken++;
      return k < n_lane ? (unsigned)units[k] : n_items;
    } else {
      return atomicAdd(ctr, 1u);
    }
  }
  // Counter mode: a block that gave up takes the rest of the queue unprocessed, so that
  // the counter always passes the end; the last block to finish zeroes both words for
  // the next launch (launches on one plan are ordered on the GPU).
  __device__ __forceinline__ void finish(unsigned last) {
    if constexpr (!kLanes) {
      while (last < n_items) last = atomicAdd(ctr, 1u);
      __threadfence();
      if (atomicAdd(ctr + 1, 1u) == gridDim.x - 1) {
        atomicExch(ctr, 0u);
        atomicExch(ctr + 1, 0u);
      }
    }
  }
};

template <bool kLanes>
__device__ __forceinline__ ItemSource<kLanes> item_source(unsigned* ctr, const int32_t* lane_off,
                                                          const int32_t* lane_units, unsigned n_items) {
  ItemSource<kLanes> src;
  src.ctr = ctr;
  src.n_items = n_items;
  src.taken = 0;
  src.units = nullptr;
  src.n_lane = 0;
  if (kLanes) {
    src.units = lane_units + lane_off[blockIdx.x];
    src.n_lane = lane_off[blockIdx.x + 1] - lane_off[blockIdx.x];
  }
  return src;
}

}  // namespace tc
}  // namespace augtree
