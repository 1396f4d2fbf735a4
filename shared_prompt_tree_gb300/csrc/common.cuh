// Device helpers shared by the kernel translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace augtree {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Decoded work item (see augtree.h for the encoding).
struct WorkItem {
  int kind, group, tile, head, split, cost, a, b;
};

__device__ __forceinline__ WorkItem load_item(const int32_t* q, int64_t i) {
  const int4* p = reinterpret_cast<const int4*>(q + i * AUGTREE_ITEM_WORDS);
  int4 x = p[0], y = p[1];
  return WorkItem{x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
}

// ---- Checked build (-DAUGTREE_CHECKED=1) ------------------------------------------
// Every kernel validates its work item against the plan's geometry before it uses any
// row or key index the item implies.  A failing item sets kErrCheck in the plan's error
// word (augtree_plan_check then returns AUGTREE_ERR_DEVICE_CHECK) and is skipped: the
// kernel does no work for it and writes nothing, so no access leaves the tensors.  No
// trap is ever raised.  The default build compiles the checks out.
#ifndef AUGTREE_CHECKED
#define AUGTREE_CHECKED 0
#endif
constexpr bool kChecked = AUGTREE_CHECKED != 0;
constexpr uint32_t kErrCheck = 4u;

__device__ __forceinline__ int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// A query-side item (PREFILL_Q or REPLAY_Q; forward and query-side backward): group and
// head in range, its query tile inside its group, its KV tile counts those of the
// encoding, its first row's branch start inside the group and not after the row.
__device__ __forceinline__ bool query_item_ok(const WorkItem& it, const Geometry& geo, int bm, int bn) {
  const bool prefill = it.kind == K_PREFILL_Q;
  if (!prefill && it.kind != K_REPLAY_Q) return false;
  if (it.group < 0 || it.group >= geo.n_groups || it.head < 0 || it.head >= geo.hq) return false;
  const GroupInfo G = geo.groups[it.group];
  const int64_t base = prefill ? G.p0 : G.r0, len = prefill ? G.lp : G.lr;
  const int64_t total = prefill ? geo.total_prompt : geo.total_resp;
  if (G.p0 < 0 || G.lp < 0 || G.r0 < 0 || G.lr < 0 || base + len > total) return false;
  if (it.tile < 0 || (int64_t)it.tile * bm >= len) return false;
  const int64_t row0 = base + (int64_t)it.tile * bm;
  const int64_t row_end = min(row0 + (int64_t)bm, base + len);
  if (prefill) return it.a == ceil_div64(row_end - G.p0, bn) && it.b == 0;
  if (it.a != ceil_div64(G.lp, bn) || (int64_t)G.p0 + G.lp > geo.total_prompt) return false;
  const int64_t own0 = geo.row_bstart[row0];
  if (own0 < G.r0 || own0 > row0) return false;
  return it.b == ceil_div64(row_end - own0, bn);
}

// The split of a query-side item (after query_item_ok): 0 unless the item is a replay
// item of a split-KV tile, then below the tile's split count with a non-empty chunk.
__device__ __forceinline__ bool split_item_ok(const WorkItem& it, const Geometry& geo) {
  if (it.kind != K_REPLAY_Q || geo.fsplit == nullptr) return it.split == 0;
  const FwdSplit fs = geo.fsplit[geo.groups[it.group].tr0 + it.tile];
  if (fs.nsplit <= 1) return it.split == 0;
  return it.split >= 0 && it.split < fs.nsplit && fs.chunk > 0 && (int64_t)it.split * fs.chunk < (int64_t)it.a + it.b &&
         fs.slot0 >= 0;
}

// A key-side item (PROMPT_KV, RESP_KV, PREFILL_KV, TREE_PROMPT_KV): group and KV head in
// range, its KV tile inside its group's keys, its query tiles [a, b) inside the query
// side it walks, its split below the group's split count.
__device__ __forceinline__ bool key_item_ok(const WorkItem& it, const Geometry& geo, int bm, int bn) {
  if (it.kind != K_PROMPT_KV && it.kind != K_RESP_KV && it.kind != K_PREFILL_KV && it.kind != K_TREE_PROMPT_KV)
    return false;
  if (it.group < 0 || it.group >= geo.n_groups || it.head < 0 || it.head >= geo.hkv) return false;
  const GroupInfo G = geo.groups[it.group];
  if (G.p0 < 0 || G.lp < 0 || G.r0 < 0 || G.lr < 0) return false;
  if ((int64_t)G.p0 + G.lp > geo.total_prompt || (int64_t)G.r0 + G.lr > geo.total_resp) return false;
  const bool resp_keys = it.kind == K_RESP_KV;
  if (it.tile < 0 || (int64_t)it.tile * bn >= (resp_keys ? G.lr : G.lp)) return false;
  const int64_t nq = ceil_div64(it.kind == K_PREFILL_KV ? G.lp : G.lr, bm);
  if (it.a < 0 || it.a > it.b || it.b > nq) return false;
  if (it.kind == K_PROMPT_KV || it.kind == K_TREE_PROMPT_KV) {
    const int nsplit = geo.splits ? geo.splits[it.group].nsplit : 1;
    if (it.split < 0 || it.split >= (nsplit > 1 ? nsplit : 1)) return false;
  } else if (it.split != 0) {
    return false;
  }
  return true;
}

}  // namespace augtree
