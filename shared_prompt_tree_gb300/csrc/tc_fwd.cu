// Tensor-core forward of tree attention on sm_103a: persistent blocks, one query head
// per work item, with a double-buffered score tile.
//
// AugTree paper, "Splitting Prompt Prefill from Response Replay ...":
//   Sec. 2.2  attention as Q-KV tile interactions with an online softmax;
//   Sec. 3.2  prefill rows see the prompt causally; a replay row (Eq. 1) sees all prompt
//             keys of its group and its own branch's keys up to itself;
//   Sec. 3.3  partial softmax states merge associatively: here the two halves of every
//             key tile keep separate running states, merged once per row at the end
//             (and, for a split-KV item, its chunk's state goes to the workspace for the
//             merge across chunks);
//   Sec. 3.4  replay units placed on lanes: here a lane is a persistent block.
//
// A work item is one 128-row query tile of one query head.  One block per SM (fewer for
// a short queue) takes items one after the other: in queue order through a counter in
// the plan's device memory (the largest-first, stream-ordered order of the queue, as
// the hardware would hand out one block per item), or from its lane of AssignGrid's
// placement (persistent schedule).  Consecutive items of a block overlap: the next
// item is taken once the current one's query tile and first two K/V tiles are in
// flight, its query tile is warmed in L2 then and loaded once the current item's last S
// product has read Q (its first K/V tile goes out before that wait), its first score
// tiles are computed while the softmax warps finish the current item, and a separate
// warpgroup writes the output.
// Barrier phases, the K/V ring and the score buffers run on across items (counters of
// the block's items and K/V tiles); nothing is re-initialised between items.
//   warp 8       TMA producer: takes and decodes the items (a ring of 4), loads Q and a
//                3-stage ring of K/V tiles (128 keys x 128 dims)
//   warp 9       TMEM allocator and issuer of S(j) = Q K^T into buffer j % 2
//   warp 10      issuer of O_w += P_w(j) V_w(j), w = 0, 1 (V_w: the tile's keys
//                [64w, 64w + 64))
//   warps 0-7    two softmax warpgroups; warpgroup w owns keys [64w, 64w + 64) of every
//                tile and its own running max, sum of rounded weights and accumulator
//                O_w; thread i of each warpgroup owns row i (TMEM lane i)
//   warps 11-14  epilogue: the merge of the two warpgroups' states of a row, O read out
//                of TMEM, the output rows (or a split item's partial state)
// TMEM columns: S0/P0 [0,128), S1/P1 [128,256), O_0 [256,384), O_1 [384,512).
// S(j+1) goes to the other buffer and waits only for the PV products of tile j-1, so
// the softmax of tile j+1 can start as soon as that of tile j ends.  An item's first PV
// products wait until the epilogue warps have read O out for the previous item.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_rows.cuh"
#include "tc_store.cuh"

namespace augtree {
namespace {

using namespace tc;

// 1: the PV issuer issues warpgroup w's product as soon as that warpgroup's P is ready
// (measured 1,469-1,480 against 1,449-1,454 TFLOP/s, prompt-heavy forward); 0: once
// both are.
#ifndef AUGTREE_FWD_PV_EARLY
#define AUGTREE_FWD_PV_EARLY 1
#endif
constexpr bool kFwdPvEarly = AUGTREE_FWD_PV_EARLY != 0;
// Every kFwdFmaPairs-th pair's second exponential of a thread's 32 pairs per tile runs on
// the FMA pipe (exp2_fma): 32 -> one exponential in 64.
#ifndef AUGTREE_FWD_FMA_PAIRS
#define AUGTREE_FWD_FMA_PAIRS 32
#endif
constexpr int kFwdFmaPairs = AUGTREE_FWD_FMA_PAIRS;
static_assert(kFwdFmaPairs >= 1 && 32 % kFwdFmaPairs == 0, "FMA exponential spacing");
// 1: V tiles land on their own barrier, so that S(j) waits only for K(j) (measured
// +1.2 % on the prompt-heavy forward, +0.8 % mixed); 0: one barrier per K/V stage.
#ifndef AUGTREE_FWD_VBAR
#define AUGTREE_FWD_VBAR 1
#endif
constexpr bool kFwdVBar = AUGTREE_FWD_VBAR != 0;
// 1: the epilogue writes each thread's row in 32-byte stores (whole sectors) where the
// destination is 32-byte aligned; 0: 16-byte stores.
#ifndef AUGTREE_FWD_V8_STORE
#define AUGTREE_FWD_V8_STORE 1
#endif
constexpr bool kFwdV8Store = AUGTREE_FWD_V8_STORE != 0;
constexpr int FWD_NST = 3;                     // K/V ring stages
constexpr int FWD_TILE = 128 * 128;            // 128 rows x 64 bf16 columns = 16 KB
constexpr int FWD_Q_OFF = 0;                   // 2 blocks
constexpr int FWD_K_OFF = FWD_Q_OFF + 2 * FWD_TILE;            // [NST][2 blocks]
constexpr int FWD_V_OFF = FWD_K_OFF + FWD_NST * 2 * FWD_TILE;   // [NST][2 blocks]
constexpr int FWD_BAR_OFF = FWD_V_OFF + FWD_NST * 2 * FWD_TILE;

// ---------------------------------------------------------------- kernel
// a0 * s0 + a1 * s1 on a pair of fp32 values (word pairs x0, x1 of two accumulators),
// in the packed two-lane fp32 arithmetic of sm_100 and later: one multiply and one fused
// multiply-add for both lanes, each lane rounded as the scalar operations would be.
__device__ __forceinline__ void f32x2_scale_add(uint32_t a_lo, uint32_t a_hi, uint32_t b_lo, uint32_t b_hi, float s0,
                                                float s1, uint32_t& r_lo, uint32_t& r_hi) {
  asm("{\n .reg .b64 a, b, s, t, r;\n"
      " mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n"
      " mov.b64 s, {%6, %6};\n mov.b64 t, {%7, %7};\n"
      " mul.rn.f32x2 r, a, s;\n fma.rn.f32x2 r, b, t, r;\n"
      " mov.b64 {%0, %1}, r;\n}"
      : "=r"(r_lo), "=r"(r_hi)
      : "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "f"(s0), "f"(s1));
}


constexpr int FWDP_SLOTS = 4;  // ring of decoded items
constexpr int FWDP_THREADS = 480;
constexpr int FWDP_BAR_BYTES = 288;
// Behind the tiles: barriers, the row states handed to the epilogue warps ([2
// warpgroups][128 rows] float2) and the decoded items.
constexpr int FWD_XCH_OFF = FWD_BAR_OFF + FWDP_BAR_BYTES;
constexpr int FWD_SLOT_OFF = FWD_XCH_OFF + 2048;
constexpr int FWDP_END = FWD_SLOT_OFF + 64 * FWDP_SLOTS;
// The block takes the most shared memory a block may have; the tiles start at the first
// 1024-byte boundary of it, and a block whose allocation leaves too little room behind
// that boundary records an error and does nothing.
constexpr int FWDP_SMEM = 232448;
static_assert(FWDP_END <= FWDP_SMEM, "shared memory per block");
constexpr int FWD_CONSUMER_WARPS = 14;  // S and PV issuers, 8 softmax warps, 4 epilogue warps

struct FwdPBars {
  uint64_t q_full, q_empty;
  uint64_t kv_full[FWD_NST];
  uint64_t v_full[FWD_NST];
  uint64_t kv_empty[FWD_NST];
  uint64_t s_full[2];
  uint64_t p_full[2][2];
  uint64_t pv_done[2];
  uint64_t item_full[FWDP_SLOTS];   // a decoded item is in slot i
  uint64_t item_empty[FWDP_SLOTS];  // every consumer warp has read slot i
  uint64_t ml_ready;       // both softmax warpgroups have published (m, l)
  uint64_t ml_free;        // the epilogue warps have read them
  uint64_t o_free;         // the epilogue warps have read O_0 and O_1 out of TMEM
  uint64_t drain[2];
  uint32_t tmem_base;
};
static_assert(sizeof(FwdPBars) <= FWDP_BAR_BYTES, "barrier area");

// kLanes: items from the block's lane (lane_off / lane_units) instead of the counter pair
// ctr.  kSplit: the replay queue holds split-KV items.
template <bool kLanes, bool kSplit>
__global__ void __launch_bounds__(FWDP_THREADS, 1) tc_fwd_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kp,
    const __grid_constant__ CUtensorMap tm_vp, const __grid_constant__ CUtensorMap tm_kr,
    const __grid_constant__ CUtensorMap tm_vr, Geometry geo, const int32_t* __restrict__ queue,
    unsigned n_items, int bm, int bn, __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int64_t lse_rows,
    uint32_t* __restrict__ err, unsigned* __restrict__ ctr, const int32_t* __restrict__ lane_off,
    const int32_t* __restrict__ lane_units, float* __restrict__ part_o, float* __restrict__ part_lse) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if ((smem - smem_raw) + FWDP_END > FWDP_SMEM) {
    if (threadIdx.x == 0) atomicOr(err, kErrLayout);
    return;
  }
  FwdPBars* bars = reinterpret_cast<FwdPBars*>(smem + FWD_BAR_OFF);
  float2* xch = reinterpret_cast<float2*>(smem + FWD_XCH_OFF);
  QuerySlot* slots = reinterpret_cast<QuerySlot*>(smem + FWD_SLOT_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int i = 0; i < FWD_NST; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->p_full[b][0], 128);
      mbar_init(&bars->p_full[b][1], 128);
      mbar_init(&bars->pv_done[b], 1);
      mbar_init(&bars->drain[b], 1);
    }
    for (int i = 0; i < FWDP_SLOTS; ++i) {
      mbar_init(&bars->item_full[i], 1);
      mbar_init(&bars->item_empty[i], FWD_CONSUMER_WARPS);
    }
    mbar_init(&bars->ml_ready, 256);
    mbar_init(&bars->ml_free, 128);
    mbar_init(&bars->o_free, 128);
    fence_mbar_init();
  }
  if (warp == 9) tmem_alloc(&bars->tmem_base, 512);
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_kp);
    prefetch_tmap(&tm_vp);
    prefetch_tmap(&tm_kr);
    prefetch_tmap(&tm_vr);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const int r = geo.hq / geo.hkv;
      bool ok = true;
      int n = 0;         // items of this block so far
      int n_q = 0;       // query tiles loaded
      int jg = 0;        // K/V tiles loaded
      QuerySlot stop_slot{};
      stop_slot.stop = 1;
      ItemSource<kLanes> src = item_source<kLanes>(ctr, lane_off, lane_units, n_items);
      unsigned taken = src.next();
      QuerySlot cur = taken < n_items ? decode_query_item<kSplit>(queue, (int)taken, geo, bm, bn, err) : stop_slot;
      slots[0] = cur;
      mbar_arrive(&bars->item_full[0]);
      if (!cur.stop) {
        tma_prefetch_3d(&tm_q, 0, cur.h, cur.row0);
        tma_prefetch_3d(&tm_q, 64, cur.h, cur.row0);
      }
      while (!cur.stop) {
        const int kvh = cur.h / r;
        // K/V tile j of the current item into the next ring stage, once the PV products
        // of the tile that held that stage are done.
        auto load_kv = [&](int j) {
          const int stage = (int)(jg % FWD_NST);
          const uint32_t use = (uint32_t)(jg / FWD_NST);
          if (!mbar_wait(&bars->kv_empty[stage], (use & 1) ^ 1, err)) return false;
          mbar_expect_tx(&bars->kv_full[stage], (kFwdVBar ? 2 : 4) * FWD_TILE);
          if (kFwdVBar) mbar_expect_tx(&bars->v_full[stage], 2 * FWD_TILE);
          const int jt = cur.j0 + j;  // tile of the rows' walk
          const bool own = jt >= cur.n_a;
          const int krow = own ? cur.own0 + (jt - cur.n_a) * bn : cur.p0 + jt * bn;
          const CUtensorMap* km = own ? &tm_kr : &tm_kp;
          const CUtensorMap* vm = own ? &tm_vr : &tm_vp;
          uint64_t* vbar = kFwdVBar ? &bars->v_full[stage] : &bars->kv_full[stage];
          for (int kb = 0; kb < 2; ++kb)
            tma_load_3d(smem + FWD_K_OFF + (stage * 2 + kb) * FWD_TILE, km, &bars->kv_full[stage], kb * 64, kvh, krow);
          for (int kb = 0; kb < 2; ++kb)
            tma_load_3d(smem + FWD_V_OFF + (stage * 2 + kb) * FWD_TILE, vm, vbar, kb * 64, kvh, krow);
          ++jg;
          return true;
        };
        // The item's first K/V tile goes ahead of its query tile: it needs only a free ring
        // stage, while Q waits for the previous item's last S product, so both have landed
        // when that wait ends and Q arrives.
        int j = 0;
        if (cur.n_tiles > 0) {
          if (!(ok = load_kv(0))) break;
          j = 1;
        }
        // The current item's query tile, once the previous item's S products have read Q.
        if (n >= 1 && !(ok = mbar_wait(&bars->q_empty, (n - 1) & 1, err))) break;
        mbar_expect_tx(&bars->q_full, 2 * FWD_TILE);
        for (int kb = 0; kb < 2; ++kb)
          tma_load_3d(smem + FWD_Q_OFF + kb * FWD_TILE, &tm_q, &bars->q_full, kb * 64, cur.h, cur.row0);
        ++n_q;
        if (j < cur.n_tiles) {
          if (!(ok = load_kv(j))) break;
          ++j;
        }
        // Take the next item and publish it, so that every warp can prepare it, here,
        // with the first two K/V tiles and Q of the current item issued: taking and
        // decoding it is a chain of dependent loads, kept out of the way from the previous
        // item's last S product to this item's query tile.
        taken = src.next();
        const QuerySlot nxt = taken < n_items ? decode_query_item<kSplit>(queue, (int)taken, geo, bm, bn, err) : stop_slot;
        const int u = n + 1, sn = u % FWDP_SLOTS;
        if (u >= FWDP_SLOTS && !(ok = mbar_wait(&bars->item_empty[sn], ((u / FWDP_SLOTS) - 1) & 1, err))) break;
        slots[sn] = nxt;
        mbar_arrive(&bars->item_full[sn]);
        if (!nxt.stop) {
          tma_prefetch_3d(&tm_q, 0, nxt.h, nxt.row0);
          tma_prefetch_3d(&tm_q, 64, nxt.h, nxt.row0);
        }
        for (; j < cur.n_tiles; ++j)
          if (!(ok = load_kv(j))) break;
        if (!ok) break;
        ++n;
        cur = nxt;
      }
      // This thread's copies in flight land before the block frees its memory.
      if (n_q > 0) mbar_wait_drain(&bars->q_full, (n_q - 1) & 1, err);
      for (int t = jg > FWD_NST ? jg - FWD_NST : 0; t < jg; ++t) {
        mbar_wait_drain(&bars->kv_full[t % FWD_NST], (uint32_t)(t / FWD_NST) & 1, err);
        if (kFwdVBar) mbar_wait_drain(&bars->v_full[t % FWD_NST], (uint32_t)(t / FWD_NST) & 1, err);
      }
      src.finish(taken);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer: S
    constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
    const uint64_t dq = smem_desc_sw128(smem_u32(smem + FWD_Q_OFF), 16, 1024);
    const uint64_t dk0 = smem_desc_sw128(smem_u32(smem + FWD_K_OFF), 16, 1024);
    constexpr uint64_t kStage = (2 * FWD_TILE) >> 4;
    auto koff = [](int kk) { return (uint64_t)(((kk >> 2) * FWD_TILE + (kk & 3) * 32) >> 4); };
    bool ok = true;
    int jg = 0;
    for (int n = 0; ok; ++n) {
      const int sn = n % FWDP_SLOTS;
      if (!(ok = mbar_wait_warp_all(&bars->item_full[sn], (n / FWDP_SLOTS) & 1, err))) break;
      const QuerySlot it = warp_uniform(slots[sn]);
      const int stop = it.stop, n_tiles = it.n_tiles;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->item_empty[sn]);
      if (stop) break;
      if (!(ok = mbar_wait_warp_all(&bars->q_full, n & 1, err))) break;
      tc_fence_after();
      for (int j = 0; j < n_tiles; ++j) {
        const int stage = (int)(jg % FWD_NST), b = (int)(jg & 1);
        if (!(ok = mbar_wait_warp_all(&bars->kv_full[stage], (uint32_t)(jg / FWD_NST) & 1, err))) break;
        // S overwrites the P of the tile two before in buffer b (possibly the previous
        // item's): both PV products of that tile must be done.
        if (jg >= 2 && !(ok = mbar_wait_warp_all(&bars->pv_done[b], (uint32_t)((jg >> 1) - 1) & 1, err))) break;
        tc_fence_after();
        const uint64_t dk = dk0 + stage * kStage;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss_w(tmem + b * 128, dq + koff(kk), dk + koff(kk), idesc_qk, kk > 0 ? 1u : 0u);
        mma_commit_w(&bars->s_full[b]);
        ++jg;
      }
      if (!ok) break;
      mma_commit_w(&bars->q_empty);  // Q is free once these products complete
    }
    mma_commit_w(&bars->drain[0]);
    mbar_wait_drain_warp_all(&bars->drain[0], 0, err);
  } else if (warp == 10) {
    // ------------------------------------------------------------ MMA issuer: PV
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 128, false, true);
    const uint64_t dv0 = smem_desc_sw128(smem_u32(smem + FWD_V_OFF), FWD_TILE, 1024);
    constexpr uint64_t kStage = (2 * FWD_TILE) >> 4;
    bool ok = true;
    int jg = 0;
    for (int n = 0; ok; ++n) {
      const int sn = n % FWDP_SLOTS;
      if (!(ok = mbar_wait_warp_all(&bars->item_full[sn], (n / FWDP_SLOTS) & 1, err))) break;
      const QuerySlot it = warp_uniform(slots[sn]);
      const int stop = it.stop, n_tiles = it.n_tiles;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->item_empty[sn]);
      if (stop) break;
      for (int j = 0; j < n_tiles; ++j) {
        const int stage = (int)(jg % FWD_NST), b = (int)(jg & 1);
        const uint32_t par = (uint32_t)(jg >> 1) & 1;
        if (kFwdVBar && !(ok = mbar_wait_warp_all(&bars->v_full[stage], (uint32_t)(jg / FWD_NST) & 1, err))) break;
        // An item's first products overwrite O_0 and O_1, which the epilogue warps read
        // out for the previous item.
        if (j == 0 && n >= 1 && !(ok = mbar_wait_warp_all(&bars->o_free, (n - 1) & 1, err))) break;
        if (!kFwdPvEarly) {
          if (!(ok = mbar_wait_warp_all(&bars->p_full[b][0], par, err))) break;
          if (!(ok = mbar_wait_warp_all(&bars->p_full[b][1], par, err))) break;
          tc_fence_after();
        }
        const uint64_t dv = dv0 + stage * kStage;
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          if (kFwdPvEarly) {
            if (!(ok = mbar_wait_warp_all(&bars->p_full[b][w], par, err))) break;
            tc_fence_after();
          }
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts_w(tmem + 256 + w * 128, tmem + b * 128 + w * 64 + kk * 8, dv + (4 * w + kk) * (2048 >> 4),
                     idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        }
        if (!ok) break;
        mma_commit_w(&bars->pv_done[b]);
        mma_commit_w(&bars->kv_empty[stage]);
        ++jg;
      }
    }
    mma_commit_w(&bars->drain[1]);
    mbar_wait_drain_warp_all(&bars->drain[1], 0, err);
  } else if (warp >= 11) {
    // ------------------------------------------------------------ epilogue warps
    // Warp 11 + i reads TMEM lane quarter (11 + i) % 4; thread r owns row r of the tile,
    // all 128 dims: the merge of the two softmax warpgroups' states (O_0, m_0, l_0) and
    // (O_1, m_1, l_1), O read out of TMEM, the output (or a split item's partial state).
    const int q4 = warp & 3;
    const int r_local = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    // Rows start on 256-byte boundaries of the output (bf16) and 512-byte boundaries of
    // the partial states (fp32), so 32-byte stores need only aligned base pointers.
    const bool v8_out = kFwdV8Store && ((reinterpret_cast<uintptr_t>(out) & 31) == 0);
    const bool v8_part = kFwdV8Store && ((reinterpret_cast<uintptr_t>(part_o) & 31) == 0);
    bool ok = true;
    int jg = 0;
    for (int n = 0; ok; ++n) {
      const int sn = n % FWDP_SLOTS;
      if (!(ok = mbar_wait_warp_all(&bars->item_full[sn], (n / FWDP_SLOTS) & 1, err))) break;
      const QuerySlot cur = warp_uniform(slots[sn]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->item_empty[sn]);
      if (cur.stop) break;
      jg += cur.n_tiles;
      if (!(ok = mbar_wait_warp_all(&bars->ml_ready, n & 1, err))) break;
      const float2 st0 = xch[r_local], st1 = xch[128 + r_local];
      mbar_arrive(&bars->ml_free);
      const int last = jg - 1;
      if (cur.n_tiles > 0 && !(ok = mbar_wait_warp_all(&bars->pv_done[last & 1], (uint32_t)(last >> 1) & 1, err)))
        break;
      tc_fence_after();
      const float m0 = st0.x, l0 = st0.y, m1 = st1.x, l1 = st1.y;
      const float M = fmaxf(m0, m1);
      const float a0 = (m0 == -INFINITY) ? 0.f : fast_exp2(m0 - M);
      const float a1 = (m1 == -INFINITY) ? 0.f : fast_exp2(m1 - M);
      const float L = l0 * a0 + l1 * a1;
      const bool any = L > 0.f && cur.n_tiles > 0;  // a row with no key writes zeros
      const float inv = any ? 1.f / L : 0.f;
      const float s0 = a0 * inv, s1 = a1 * inv;
      // O_0 and O_1 hold the item's products whenever it walked a tile (finite: weights
      // in [0, 1] times finite values), so a row without a key gets 0 * O = 0 from its
      // zero factors; an item without tiles never wrote O and writes zeros.
      const bool live = cur.n_tiles > 0;
      const float lse_v = any ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
      const int row = cur.row0 + r_local;
      const bool row_ok = row < cur.row_end;
      if (kSplit && cur.slot >= 0) {
        // Split-KV item: the chunk's state O / l (fp32) and its lse.
        float* prow = part_o + (cur.slot * kFwdPartRows + r_local) * 128;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o0[32], o1[32];
          tmem_ld32(tmem + lane_off + 256 + 32 * c, o0);
          tmem_ld32(tmem + lane_off + 384 + 32 * c, o1);
          tmem_ld_wait();
          if (c == 3) {
            // O is read out: the next item's first PV products may overwrite it.
            tc_fence_before();
            mbar_arrive(&bars->o_free);
          }
          if (row_ok) {
            uint32_t v[32];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              if (live)
                f32x2_scale_add(o0[2 * i], o0[2 * i + 1], o1[2 * i], o1[2 * i + 1], s0, s1, v[2 * i], v[2 * i + 1]);
              else
                v[2 * i] = v[2 * i + 1] = 0u;
            }
            if (v8_part) {
#pragma unroll
              for (int i = 0; i < 4; ++i) st_global_v8(prow + 32 * c + 8 * i, v + 8 * i);
            } else {
              float4* d4 = reinterpret_cast<float4*>(prow + 32 * c);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                d4[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                    __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
            }
          }
        }
        if (row_ok) part_lse[cur.slot * kFwdPartRows + r_local] = lse_v;
      } else {
        __nv_bfloat16* orow = out + ((int64_t)row * geo.hq + cur.h) * 128;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o0[32], o1[32];
          tmem_ld32(tmem + lane_off + 256 + 32 * c, o0);
          tmem_ld32(tmem + lane_off + 384 + 32 * c, o1);
          tmem_ld_wait();
          if (c == 3) {
            // O is read out: the next item's first PV products may overwrite it.
            tc_fence_before();
            mbar_arrive(&bars->o_free);
          }
          if (row_ok) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              uint32_t v0 = 0u, v1 = 0u;
              if (live) f32x2_scale_add(o0[2 * i], o0[2 * i + 1], o1[2 * i], o1[2 * i + 1], s0, s1, v0, v1);
              pk[i] = pack_bf16x2(__uint_as_float(v0), __uint_as_float(v1));
            }
            if (v8_out) {
              st_global_v8(orow + 32 * c, pk);
              st_global_v8(orow + 32 * c + 16, pk + 8);
            } else {
              uint4* d4 = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
              for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            }
          }
        }
        if (row_ok) lse[(int64_t)cur.h * lse_rows + row] = lse_v;
      }
    }
  } else {
    // ------------------------------------------------------------ softmax (half tiles)
    const int w = warp >> 2;        // keys [64w, 64w + 64) of every tile
    const int q4 = warp & 3;        // TMEM lane quarter
    const int r_local = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const float sl2 = geo.scale_log2;
    const uint32_t tO = tmem + lane_off + 256 + w * 128;
    bool ok = mbar_wait_warp_all(&bars->item_full[0], 0, err);
    QuerySlot cur{};
    cur.stop = 1;
    if (ok) {
      cur = warp_uniform(slots[0]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->item_empty[0]);
    }
    int bs = (!cur.stop && !cur.prefill && cur.row0 + r_local < cur.row_end) ? geo.row_bstart[cur.row0 + r_local] : 0;
    int jg = 0;
    for (int n = 0; ok && !cur.stop; ++n) {
      FwdRowGeom g;
      g.row = cur.row0 + r_local;
      g.row_ok = g.row < cur.row_end;
      g.prefill = cur.prefill != 0;
      g.bs = bs;
      g.p0 = cur.p0;
      g.p_end = (int64_t)cur.p0 + cur.lp;
      g.own0 = cur.own0;
      g.n_a = cur.n_a;
      g.bn = bn;
      g.j0 = cur.j0;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < cur.n_tiles; ++j) {
        const int b = (int)(jg & 1);
        const uint32_t tS = tmem + lane_off + b * 128 + w * 64;
        if (!(ok = mbar_wait_warp_all(&bars->s_full[b], (uint32_t)(jg >> 1) & 1, err))) break;
        tc_fence_after();
        uint32_t raw[2][32];
        tmem_ld32(tS, raw[0]);
        tmem_ld32(tS + 32, raw[1]);
        tmem_ld_wait();
#define FWD_X(c) raw[(c) >> 5][(c) & 31]
        int lo_i, hi_i;
        fwd_valid_cols(g, j, lo_i, hi_i);
        const int lo = lo_i - 64 * w, hi = hi_i - 64 * w;  // valid local columns [lo, hi]
        const bool masked = lo > 0 || hi < 63;
        if (masked) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c < lo || c > hi) FWD_X(c) = 0xFF800000u;  // -inf
        }
        float pm[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          pm[k] = fmax3(__uint_as_float(FWD_X(k)), __uint_as_float(FWD_X(k + 8)), __uint_as_float(FWD_X(k + 16)));
#pragma unroll
        for (int c = 24; c < 56; c += 16)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            pm[k] = fmax3(pm[k], __uint_as_float(FWD_X(c + k)), __uint_as_float(FWD_X(c + 8 + k)));
#pragma unroll
        for (int k = 0; k < 8; ++k) pm[k] = fmaxf(pm[k], __uint_as_float(FWD_X(56 + k)));
        const float tmax = fmaxf(fmax3(pm[0], pm[1], pm[2]), fmax3(fmax3(pm[3], pm[4], pm[5]), pm[6], pm[7]));
        const float mx = tmax * sl2;  // -inf stays -inf
        // Lazy rescaling: the offset moves only when the max grows by more than 2^8
        // (exact: every term of the state shares the offset).
        const bool need = (m != -INFINITY) && (mx > m + 8.0f);
        const float m_new = (m == -INFINITY) ? mx : (need ? mx : m);
        const float alpha = need ? fast_exp2(m - m_new) : 1.f;
        m = m_new;
        const float mu = (m == -INFINITY) ? 0.f : m;
        uint32_t pk[32];
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float a0 = fmaf(__uint_as_float(FWD_X(2 * i)), sl2, -mu);
          const float a1 = fmaf(__uint_as_float(FWD_X(2 * i + 1)), sl2, -mu);
          const float p0 = fast_exp2(a0);
          float p1;
          if (i % kFwdFmaPairs == kFwdFmaPairs - 1) {
            // One exponential in 2 * kFwdFmaPairs on the FMA pipe; a masked column stays
            // exactly zero.
            p1 = exp2_fma(a1);
            if (masked && a1 == -INFINITY) p1 = 0.f;
          } else {
            p1 = fast_exp2(a1);
          }
          pk[i] = pack_bf16x2(p0, p1);
          // The row sum uses the bf16 weights the PV product uses.
          ps[i & 3] = add_bf16x2_f32(ps[i & 3], pk[i]);
        }
#undef FWD_X
        tmem_st32(tS, pk);
        tmem_st_wait();
        l = l * alpha + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
        if (__any_sync(0xffffffffu, need)) {
          // O_w += P(j-1) V must be complete before O_w is rescaled; PV(j) is issued only
          // after this warpgroup signals P(j).
          if (!(ok = mbar_wait_warp_all(&bars->pv_done[(jg - 1) & 1], (uint32_t)((jg - 1) >> 1) & 1, err))) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tO + c * 32, o);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(&bars->p_full[b][w]);
        ++jg;
      }
      // Hand the rows' states to the epilogue warps, once they have read the previous
      // item's.
      if (ok && n >= 1) ok = mbar_wait_warp_all(&bars->ml_free, (n - 1) & 1, err);
      if (ok) xch[w * 128 + r_local] = make_float2(m, l);
      mbar_arrive(&bars->ml_ready);  // also after a failed wait, so that the epilogue's wait ends
      // The next item, published while this one's tiles were loaded: its row's branch
      // start is fetched now.
      QuerySlot nxt{};
      nxt.stop = 1;
      if (ok) {
        const int sn = (n + 1) % FWDP_SLOTS;
        if (mbar_wait_warp_all(&bars->item_full[sn], ((n + 1) / FWDP_SLOTS) & 1, err)) {
          nxt = warp_uniform(slots[sn]);
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->item_empty[sn]);
        }
      }
      const int nrow = nxt.row0 + r_local;
      const int bs_next = (!nxt.stop && !nxt.prefill && nrow < nxt.row_end) ? geo.row_bstart[nrow] : 0;
      cur = nxt;
      bs = bs_next;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

// 3-D map over a [rows, heads, 128] bf16 tensor: box of 64 dims x 1 head x 128 rows,
// 128-byte swizzle; rows outside the tensor read as zero.
bool encode_rows_map(CUtensorMap* map, const void* ptr, int64_t rows, int heads, int box_rows) {
  auto enc = get_encode();
  if (!enc || !ptr || rows <= 0) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {128 * 2, (cuuint64_t)heads * 128 * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over a [rows, heads, 128] fp32 tensor: box of 128 dims x 1 head x box_rows,
// no swizzle (the dQ accumulator, written by bulk reduce-add).
bool encode_f32_rows_map(CUtensorMap* map, const void* ptr, int64_t rows, int heads, int box_rows) {
  auto enc = get_encode();
  if (!enc || !ptr || rows <= 0) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {128 * 4, (cuuint64_t)heads * 128 * 4};
  cuuint32_t box[3] = {128, 1, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t tc_fwd(const augtree_plan* p, int op, const void* q, const void* kp, const void* vp, const void* kr,
                   const void* vr, void* o, float* lse, float* part_o, float* part_lse, cudaStream_t st) {
  const bool prefill = op == AUGTREE_OP_PREFILL_FWD;
  const int64_t q_rows = prefill ? p->total_prompt : p->total_resp;
  CUtensorMap mq, mkp, mvp, mkr, mvr;
  if (!encode_rows_map(&mq, q, q_rows, p->cfg.hq, 128)) return cudaErrorInvalidValue;
  const bool have_p = p->total_prompt > 0 && kp && vp;
  const bool have_r = !prefill && p->total_resp > 0 && kr && vr;
  if (have_p) {
    if (!encode_rows_map(&mkp, kp, p->total_prompt, p->cfg.hkv, 128)) return cudaErrorInvalidValue;
    if (!encode_rows_map(&mvp, vp, p->total_prompt, p->cfg.hkv, 128)) return cudaErrorInvalidValue;
  }
  if (have_r) {
    if (!encode_rows_map(&mkr, kr, p->total_resp, p->cfg.hkv, 128)) return cudaErrorInvalidValue;
    if (!encode_rows_map(&mvr, vr, p->total_resp, p->cfg.hkv, 128)) return cudaErrorInvalidValue;
  }
  // Maps that the queue never uses (no prompt keys, or no response keys) alias a used one.
  if (!have_p) {
    mkp = have_r ? mkr : mq;
    mvp = have_r ? mvr : mq;
  }
  if (!have_r) {
    mkr = mkp;
    mvr = mvp;
  }
  // The split-KV instantiation only where the replay queue has split items.
  const bool split = !prefill && p->n_fwd_parts > 0;
  if (split && (!part_o || !part_lse)) return cudaErrorInvalidValue;
  const unsigned n_items = (unsigned)p->n_items[op];
  // Persistent schedule: one block per lane of AssignGrid's placement; else one block
  // per SM (fewer for a short queue) taking items in queue order.
  const LaneSet& ls = p->lanes_dq[op];
  const bool lanes = ls.off_d != nullptr;
  unsigned grid = (unsigned)ls.n_lanes;
  if (!lanes) {
    int sms = 0;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device);
    if (e != cudaSuccess) return e;
    grid = std::min<unsigned>(n_items, (unsigned)std::max(sms, 1));
  }
  auto kern = lanes ? (split ? tc_fwd_kernel<true, true> : tc_fwd_kernel<true, false>)
                    : (split ? tc_fwd_kernel<false, true> : tc_fwd_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FWDP_SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, FWDP_THREADS, FWDP_SMEM, st>>>(mq, mkp, mvp, mkr, mvr, geometry(p), p->queue_d[op], n_items, p->bm[op],
                                             p->bn[op], (__nv_bfloat16*)o, lse, q_rows, p->err_d,
                                             p->err_d + kErrFwdCounter + 2 * op, lanes ? ls.off_d : nullptr,
                                             lanes ? ls.units_d : nullptr, part_o, part_lse);
  return cudaGetLastError();
}

}  // namespace augtree
