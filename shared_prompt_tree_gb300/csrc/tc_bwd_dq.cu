// Tensor-core backward of tree attention on sm_103a, query side: dQ.
//
// AugTree paper, "Splitting Prompt Prefill from Response Replay ...":
//   Sec. 2.2  attention as Q-KV tile interactions;
//   Sec. 3.2  prefill rows see the prompt causally; a replay row (Eq. 1) sees all prompt
//             keys of its group and its own branch's keys up to itself;
//   Sec. 3.3  the gradient of a response query sums over its prompt part and its own
//             part: here one accumulator walks the prompt tiles, then the own tiles.
//
// One thread block per work item of the forward queue: one query tile of 128 rows for
// one query head.  Q and dO stay in shared memory; K tiles stream through a 3-stage
// ring and V tiles through a 2-stage ring.  Per KV tile j (thread = query row = TMEM
// lane; lse and Delta are per-thread scalars):
//   S    = Q K^T          (TMEM, fp32)  -> P  = exp2(s S log2e - lse)   (registers)
//   dP   = dO V^T         (TMEM, fp32)  -> dS = P (dP - Delta)          (bf16 into TMEM
//                                          over dP, the A operand of the next product)
//   dQ  += dS K           (A = dS from TMEM, B = K read MN-major from the same tile)
// dQ accumulates in TMEM over every KV tile of the row and is written once (bf16, times
// the softmax scale): no atomics, no fp32 accumulator in memory.
// Warps: 0-7 two warpgroups, warpgroup w takes key columns [64w, 64w + 64) of every
//        tile (lanes = rows, as TMEM access requires warp % 4 = lane quarter);
//        8 TMA producer; 9 TMEM allocator + issuer of S and dP; 10 issuer of dQ.
// TMEM columns: S [0,128); dP(j), then dS(j) over it, in region j % 2 ([128,256) or
// [256,384)); dQ [384,512).
// MMA issue order S(j+1), dP(j+1), dQ(j).  S(j+1) waits only for the compute warps to
// have loaded S(j) into registers; dP(j+1) reuses the region dQ(j-1), issued a tile
// earlier, read; dQ(j) waits for dS(j).  No MMA waits on the group issued just before
// it (a tcgen05 group's completion is seen about 280 cycles after its last issue).
#include <cuda.h>

#include <cmath>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_rows.cuh"
#include "tc_store.cuh"

namespace augtree {
namespace {

using namespace tc;

// All exponentials on the MUFU: moving one in eight to the FMA pipe measured 5 % slower
// here, one in 32 or 64 about 1 % slower (unlike the key side, this kernel's compute
// phase is issue-bound).
#ifndef AUGTREE_DQ_EXP_FMA
#define AUGTREE_DQ_EXP_FMA 0
#endif
constexpr int kDqExpFma = AUGTREE_DQ_EXP_FMA;  // 0, or N: one exponential in N via exp2_fma
constexpr int DQ_THREADS = 352;  // 8 compute warps, producer, two MMA issuers
// K tiles are read by S(j) and dQ(j), V tiles only by dP(j), so the two rings are
// separate: a V stage frees as soon as dP(j) is done, and the K ring has one stage more
// so that K(j+2) can be in flight while dQ(j) still reads K(j).
constexpr int KST = 3;                             // K ring stages
constexpr int VST = 2;                             // V ring stages
constexpr int kPrefetchTiles = 4;                  // L2 prefetch distance (KV tiles)
// 1: each block warms L2 with the Q and dO tiles of the item one wave (the SM count)
// ahead in the queue.
#ifndef AUGTREE_DQ_NEXT_WAVE
#define AUGTREE_DQ_NEXT_WAVE 1
#endif
constexpr bool kDqPrefetchNextWave = AUGTREE_DQ_NEXT_WAVE != 0;
constexpr int BLK = 128 * 128;                     // 128 rows x 64 dims bf16 = 16 KB
constexpr int DQ_Q_OFF = 0;                        // 2 blocks
constexpr int DQ_DO_OFF = DQ_Q_OFF + 2 * BLK;      // 2 blocks
constexpr int DQ_K_OFF = DQ_DO_OFF + 2 * BLK;      // [KST][2 blocks]
constexpr int DQ_V_OFF = DQ_K_OFF + KST * 2 * BLK; // [VST][2 blocks]
constexpr int DQ_BAR_OFF = DQ_V_OFF + VST * 2 * BLK;
constexpr int DQ_SMEM = DQ_BAR_OFF + 256 + 1024;

// S [0,128) is reused every tile (free once the compute warps have loaded it); dP and
// then dS of tile j live in region j % 2 at [128,256) / [256,384); dQ [384,512).
constexpr uint32_t T_S = 0, T_DP = 128, T_DQ = 384;

struct DqBars {
  uint64_t q_full;
  uint64_t k_full[KST];
  uint64_t k_empty[KST];
  uint64_t v_full[VST];
  uint64_t v_empty[VST];
  uint64_t s_full;       // S(j) in TMEM
  uint64_t s_free;       // the compute warps have loaded S(j)
  uint64_t dp_full[2];   // per dP/dS region
  uint64_t ds_ready[2];
  uint64_t dq_done[2];
  uint64_t acc_done;
  uint64_t drain;        // every S / dP MMA of the first issuer has completed
  uint32_t tmem_base;
};

static_assert(sizeof(DqBars) <= 256, "barrier area");


// kSplit: the replay queue holds split-KV items, whose dQ over their chunk of KV tiles
// goes to an fp32 partial slot (summed afterwards in split order).
template <bool kPersistent, bool kSplit>
__global__ void __launch_bounds__(DQ_THREADS, 1) tc_bwd_dq_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
    const __grid_constant__ CUtensorMap tm_kp, const __grid_constant__ CUtensorMap tm_vp,
    const __grid_constant__ CUtensorMap tm_kr, const __grid_constant__ CUtensorMap tm_vr, Geometry geo,
    const int32_t* __restrict__ queue, int bm, int bn, const float* __restrict__ stats, int ntiles,
    __nv_bfloat16* __restrict__ dq_out, uint32_t* __restrict__ err,
    const int32_t* __restrict__ sched_off, const int32_t* __restrict__ sched_units, float* __restrict__ dq_part,
    int64_t n_items, int ahead) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DqBars* bars = reinterpret_cast<DqBars*>(smem + DQ_BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // TMEM: allocated once for every unit of the lane (persistent schedule) or, as the
  // block's first step, for its one unit (queue schedule, below).
  if (kPersistent && warp == 9) tmem_alloc(&bars->tmem_base, 512);
  // The queue schedule's instantiation runs exactly one unit (the loop folds away).
  const int n_units = kPersistent ? sched_off[blockIdx.x + 1] - sched_off[blockIdx.x] : 1;
  for (int u_i = 0; u_i < n_units; ++u_i) {
  const int64_t unit = kPersistent ? (int64_t)sched_units[sched_off[blockIdx.x] + u_i] : (int64_t)blockIdx.x;

  const WorkItem it = load_item(queue, unit);
  const bool item_ok = !kChecked || (query_item_ok(it, geo, bm, bn) &&  // checked build only
                                     (kSplit ? split_item_ok(it, geo) : it.split == 0));
  if (kChecked && !item_ok && threadIdx.x == 0) atomicOr(err, kErrCheck);
  const int h = item_ok ? it.head : 0;
  const GroupInfo G = geo.groups[item_ok ? it.group : 0];
  const bool prefill = it.kind == K_PREFILL_Q;
  const int64_t base = prefill ? G.p0 : G.r0;
  const int64_t len = prefill ? G.lp : G.lr;
  const int64_t row0 = item_ok ? base + (int64_t)it.tile * bm : 0;
  const int64_t row_end = item_ok ? min(row0 + (int64_t)bm, base + len) : 0;
  const int n_a = item_ok ? it.a : 0;
  int n_tiles = item_ok ? n_a + (prefill ? 0 : it.b) : 0;
  const int64_t own0 = (prefill || !item_ok) ? 0 : geo.row_bstart[row0];
  const int kvh = h / (geo.hq / geo.hkv);
  // Split-KV item: KV tiles [j0, j0 + n_tiles) of the walk, dQ to partial slot `slot`.
  int j0 = 0;
  int64_t slot = -1;
  if (kSplit && item_ok && !prefill) {
    const FwdSplit fs = geo.fsplit[G.tr0 + it.tile];
    if (fs.nsplit > 1) {
      j0 = it.split * fs.chunk;
      n_tiles = min(fs.chunk, n_tiles - j0);
      slot = fs.slot0 + (int64_t)h * fs.nsplit + it.split;
    }
  }

  // The barriers are set up by the producer thread under the queue schedule, which then
  // starts the item's Q and dO copies at once, ahead of the block-wide barrier (measured:
  // the block's set-up takes about 0.7 us and its first copies about 1.4 us); under the
  // persistent schedule by thread 0, for each unit.
  if (threadIdx.x == (kPersistent ? 0 : 256)) {
    if (kPersistent && u_i > 0) {
      // Every wait, copy and MMA of the previous unit has ended (drains, then the
      // block-wide barrier at its end): its barriers are idle and may be reused.
      for (uint64_t* b = &bars->q_full; b < reinterpret_cast<uint64_t*>(&bars->tmem_base); ++b) mbar_inval(b);
    }
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < KST; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < VST; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 256);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->dp_full[b], 1);
      mbar_init(&bars->ds_ready[b], 256);
      mbar_init(&bars->dq_done[b], 1);
    }
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->drain, 1);
    fence_mbar_init();
    if (!kPersistent) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_do);
      mbar_expect_tx(&bars->q_full, 4 * BLK);
      for (int kb = 0; kb < 2; ++kb) {
        tma_load_3d(smem + DQ_Q_OFF + kb * BLK, &tm_q, &bars->q_full, kb * 64, h, (int)row0);
        tma_load_3d(smem + DQ_DO_OFF + kb * BLK, &tm_do, &bars->q_full, kb * 64, h, (int)row0);
      }
      // The first K/V tile into stage 0 of both rings (free: the barriers are fresh).
      if (n_tiles > 0) {
        const bool own = j0 >= n_a;
        const int krow = own ? (int)(own0 + (int64_t)(j0 - n_a) * bn) : (int)(G.p0 + (int64_t)j0 * bn);
        mbar_expect_tx(&bars->k_full[0], 2 * BLK);
        mbar_expect_tx(&bars->v_full[0], 2 * BLK);
        for (int kb = 0; kb < 2; ++kb) {
          tma_load_3d(smem + DQ_K_OFF + kb * BLK, own ? &tm_kr : &tm_kp, &bars->k_full[0], kb * 64, kvh, krow);
          tma_load_3d(smem + DQ_V_OFF + kb * BLK, own ? &tm_vr : &tm_vp, &bars->v_full[0], kb * 64, kvh, krow);
        }
      }
    }
  }
  if (!kPersistent && warp == 9) tmem_alloc(&bars->tmem_base, 512);
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_do);
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
      if (kPersistent) {
        mbar_expect_tx(&bars->q_full, 4 * BLK);
        for (int kb = 0; kb < 2; ++kb) {
          tma_load_3d(smem + DQ_Q_OFF + kb * BLK, &tm_q, &bars->q_full, kb * 64, h, (int)row0);
          tma_load_3d(smem + DQ_DO_OFF + kb * BLK, &tm_do, &bars->q_full, kb * 64, h, (int)row0);
        }
      }
      // First key row of the item's j-th KV tile (tile j0 + j of the row's walk).
      auto krow_of = [&](int j) {
        const int jt = j0 + j;
        return jt >= n_a ? (int)(own0 + (int64_t)(jt - n_a) * bn) : (int)(G.p0 + (int64_t)jt * bn);
      };
      // Queue schedule: tile 0 went out with Q and dO before the block-wide barrier.
      const int first = (!kPersistent && n_tiles > 0) ? 1 : 0;
      int k_issued = first, v_issued = first;
      if (first && kPrefetchTiles < n_tiles) {
        const CUtensorMap* kmp = j0 + kPrefetchTiles >= n_a ? &tm_kr : &tm_kp;
        const CUtensorMap* vmp = j0 + kPrefetchTiles >= n_a ? &tm_vr : &tm_vp;
        const int rp = krow_of(kPrefetchTiles);
        for (int kb = 0; kb < 2; ++kb) {
          tma_prefetch_3d(kmp, kb * 64, kvh, rp);
          tma_prefetch_3d(vmp, kb * 64, kvh, rp);
        }
      }
      for (int j = first; j < n_tiles; ++j) {
        const bool own = j0 + j >= n_a;
        const int krow = krow_of(j);
        const CUtensorMap* km = own ? &tm_kr : &tm_kp;
        const CUtensorMap* vm = own ? &tm_vr : &tm_vp;
        const int ks = j % KST, vs = j % VST;
        if (!mbar_wait(&bars->k_empty[ks], ((j / KST) & 1) ^ 1, err)) break;
        mbar_expect_tx(&bars->k_full[ks], 2 * BLK);
        for (int kb = 0; kb < 2; ++kb)
          tma_load_3d(smem + DQ_K_OFF + (ks * 2 + kb) * BLK, km, &bars->k_full[ks], kb * 64, kvh, krow);
        k_issued = j + 1;
        if (!mbar_wait(&bars->v_empty[vs], ((j / VST) & 1) ^ 1, err)) break;
        mbar_expect_tx(&bars->v_full[vs], 2 * BLK);
        for (int kb = 0; kb < 2; ++kb)
          tma_load_3d(smem + DQ_V_OFF + (vs * 2 + kb) * BLK, vm, &bars->v_full[vs], kb * 64, kvh, krow);
        v_issued = j + 1;
        // Warm L2 with the K/V tiles a few steps ahead.
        const int jp = j + kPrefetchTiles;
        if (jp < n_tiles) {
          const CUtensorMap* kmp = j0 + jp >= n_a ? &tm_kr : &tm_kp;
          const CUtensorMap* vmp = j0 + jp >= n_a ? &tm_vr : &tm_vp;
          const int rp = krow_of(jp);
          for (int kb = 0; kb < 2; ++kb) {
            tma_prefetch_3d(kmp, kb * 64, kvh, rp);
            tma_prefetch_3d(vmp, kb * 64, kvh, rp);
          }
        }
      }
      // Warm L2 with the Q and dO tiles of the item a wave ahead in the queue (the block
      // that will start on some SM about when this one ends), so that its first copies
      // hit L2.
      if (!kPersistent && ahead > 0 && unit + ahead < n_items) {
        const WorkItem nx = load_item(queue, unit + ahead);
        if (!kChecked || query_item_ok(nx, geo, bm, bn)) {
          const GroupInfo NG = geo.groups[nx.group];
          const int nrow = (nx.kind == K_PREFILL_Q ? NG.p0 : NG.r0) + nx.tile * bm;
          for (int kb = 0; kb < 2; ++kb) {
            tma_prefetch_3d(&tm_q, kb * 64, nx.head, nrow);
            tma_prefetch_3d(&tm_do, kb * 64, nx.head, nrow);
          }
        }
      }
      // Never leave a copy in flight (also after giving up on a wait).
      mbar_wait_drain(&bars->q_full, 0, err);
      for (int j = max(0, k_issued - KST); j < k_issued; ++j)
        mbar_wait_drain(&bars->k_full[j % KST], (j / KST) & 1, err);
      for (int j = max(0, v_issued - VST); j < v_issued; ++j)
        mbar_wait_drain(&bars->v_full[j % VST], (j / VST) & 1, err);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer: S, dP
    if (lane == 0) {
      constexpr uint32_t id_ss = idesc_bf16_f32(128, 128, false, false);  // Q K^T, dO V^T
      const uint64_t dQd = smem_desc_sw128(smem_u32(smem + DQ_Q_OFF), 16, 1024);
      const uint64_t dOd = smem_desc_sw128(smem_u32(smem + DQ_DO_OFF), 16, 1024);
      const uint64_t dK0 = smem_desc_sw128(smem_u32(smem + DQ_K_OFF), 16, 1024);
      const uint64_t dV0 = smem_desc_sw128(smem_u32(smem + DQ_V_OFF), 16, 1024);
      constexpr uint64_t kStage = (2 * BLK) >> 4;
      // K-major k-step kk (16 dims): dim block kk/4, 32 bytes per step in the 128-byte row.
      auto koff = [](int kk) { return (uint64_t)(((kk >> 2) * BLK + (kk & 3) * 32) >> 4); };
      auto issue_s = [&](int j) {
        const uint64_t dk = dK0 + (j % KST) * kStage;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(tmem + T_S, dQd + koff(kk), dk + koff(kk), id_ss, kk > 0 ? 1u : 0u);
        mma_commit(&bars->s_full);
      };
      auto issue_dp = [&](int j) {
        const uint64_t dv = dV0 + (j % VST) * kStage;
        const uint32_t d = tmem + T_DP + (j & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(d, dOd + koff(kk), dv + koff(kk), id_ss, kk > 0 ? 1u : 0u);
        mma_commit(&bars->dp_full[j & 1]);
        mma_commit(&bars->v_empty[j % VST]);  // dP(j) is the only reader of V(j)
      };
      bool ok = mbar_wait(&bars->q_full, 0, err);
      if (ok && n_tiles > 0) ok = mbar_wait(&bars->k_full[0], 0, err) && mbar_wait(&bars->v_full[0], 0, err);
      tc_fence_after();
      if (ok && n_tiles > 0) {
        issue_s(0);
        issue_dp(0);
      }
      for (int j = 0; ok && j + 1 < n_tiles; ++j) {
        // S(j+1) overwrites S(j): the compute warps must have loaded it.
        if (!(ok = mbar_wait(&bars->k_full[(j + 1) % KST], ((j + 1) / KST) & 1, err))) break;
        if (!(ok = mbar_wait(&bars->s_free, j & 1, err))) break;
        tc_fence_after();
        issue_s(j + 1);
        // dP(j+1) goes to the region that held dS(j-1): dQ(j-1), issued a tile earlier by
        // the other issuer, must have read it.
        if (!(ok = mbar_wait(&bars->v_full[(j + 1) % VST], ((j + 1) / VST) & 1, err))) break;
        if (j >= 1 && !(ok = mbar_wait(&bars->dq_done[(j - 1) & 1], ((j - 1) >> 1) & 1, err))) break;
        tc_fence_after();
        issue_dp(j + 1);
      }
      // Never leave an MMA in flight when the block frees TMEM and exits (also after
      // giving up on a wait).
      mma_commit(&bars->drain);
      mbar_wait_drain(&bars->drain, 0, err);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ MMA issuer: dQ
    // A second issuing thread: while one issuer waits on a completion, the other keeps
    // the tensor pipe fed (two issuers measured 72 cycles per N=128 MMA with a wait per
    // group, one issuer 92; 64 is the full rate).
    if (lane == 0) {
      constexpr uint32_t id_dq = idesc_bf16_f32(128, 128, false, true);  // dS K (B MN-major)
      const uint64_t dKm0 = smem_desc_sw128(smem_u32(smem + DQ_K_OFF), BLK, 1024);  // K as [keys x dims], MN-major
      constexpr uint64_t kStage = (2 * BLK) >> 4;
      bool ok = true;
      for (int j = 0; ok && j < n_tiles; ++j) {
        // dQ += dS(j) K(j): 16 keys per step; keys [64w, 64w + 64) were packed by
        // warpgroup w into columns [64w, 64w + 32) of region j % 2.
        if (!(ok = mbar_wait(&bars->ds_ready[j & 1], (j >> 1) & 1, err))) break;
        tc_fence_after();
        const uint32_t a0 = tmem + T_DP + (j & 1) * 128;
        const uint64_t b0 = dKm0 + (j % KST) * kStage;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + T_DQ, a0 + (kk >> 2) * 64 + (kk & 3) * 8, b0 + kk * (2048 >> 4), id_dq,
                 (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars->dq_done[j & 1]);
        // dQ(j) is the last reader of K(j) (S(j) completed before dS(j) existed).
        mma_commit(&bars->k_empty[j % KST]);
      }
      // Every MMA of the item is complete once the last dQ is: the other issuer's S and
      // dP of the last tile completed before its dS was written.  Wait for it here too, so
      // that no MMA of this thread is in flight when the block frees TMEM.
      mma_commit(&bars->acc_done);
      mbar_wait_drain(&bars->acc_done, 0, err);
    }
  } else {
    // ------------------------------------------------------------ P, dS (thread = row)
    const int w = warp >> 2;           // key columns [64w, 64w + 64)
    const int q4 = warp & 3;           // TMEM lane quarter
    const int r_local = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    FwdRowGeom g;
    g.row = row0 + r_local;
    g.row_ok = g.row < row_end;
    g.prefill = prefill;
    g.bs = (!prefill && g.row_ok) ? geo.row_bstart[g.row] : 0;
    g.p0 = G.p0;
    g.p_end = (int64_t)G.p0 + G.lp;
    g.own0 = own0;
    g.n_a = n_a;
    g.bn = bn;
    g.j0 = j0;
    const int tile_base = prefill ? G.tp0 : G.tr0;
    const float* st = stats + (item_ok ? ((int64_t)h * ntiles + tile_base + it.tile) * 2 * kStatRows : 0);
    const float lse2 = st[r_local];
    const float delta = st[kStatRows + r_local];
    const float sl2 = geo.scale_log2;
    const int c0 = 64 * w;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      if (!(ok = mbar_wait_warp_all(&bars->s_full, j & 1, err))) break;
      tc_fence_after();
      const uint32_t ts = tmem + lane_off + T_S + c0;
      const uint32_t tdp = tmem + lane_off + T_DP + (j & 1) * 128 + c0;
      uint32_t sv[2][32];  // S, then P in place (fp32)
      tmem_ld32(ts, sv[0]);
      tmem_ld32(ts + 32, sv[1]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&bars->s_free);
      int lo, hi;
      fwd_valid_cols(g, j, lo, hi);  // valid columns [lo, hi] of the tile, clamped
      const int lo_r = lo - c0;
      const uint32_t span = hi >= lo ? (uint32_t)(hi - lo) : 0xFFFFFFFFu;  // all-invalid if empty
      if (lo_r <= 0 && hi - c0 >= 63 && hi >= lo) {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float x = fmaf(__uint_as_float(sv[c >> 5][c & 31]), sl2, -lse2);
          // One exponential in kDqExpFma on the FMA pipe.
          const bool on_fma = kDqExpFma > 0 && c % (kDqExpFma > 0 ? kDqExpFma : 1) == kDqExpFma - 1;
          sv[c >> 5][c & 31] = __float_as_uint(on_fma ? exp2_fma(x) : fast_exp2(x));
        }
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float e = fast_exp2(fmaf(__uint_as_float(sv[c >> 5][c & 31]), sl2, -lse2));
          const bool v = span != 0xFFFFFFFFu && (uint32_t)(c - lo_r) <= span;
          sv[c >> 5][c & 31] = __float_as_uint(v ? e : 0.f);
        }
      }
      if (!(ok = mbar_wait_warp_all(&bars->dp_full[j & 1], (j >> 1) & 1, err))) break;
      tc_fence_after();
      uint32_t pk[2][16];  // dS as bf16 pairs
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t dp[32];
        tmem_ld32(tdp + half * 32, dp);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float d0 = __uint_as_float(sv[half][2 * i]) * (__uint_as_float(dp[2 * i]) - delta);
          const float d1 = __uint_as_float(sv[half][2 * i + 1]) * (__uint_as_float(dp[2 * i + 1]) - delta);
          pk[half][i] = pack_bf16x2(d0, d1);
        }
      }
      {
        uint32_t all[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          all[i] = pk[0][i];
          all[16 + i] = pk[1][i];
        }
        tmem_st32(tdp, all);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->ds_ready[j & 1]);
    }
    // dQ rows: warpgroup w writes dims [64w, 64w + 64) of its rows.
    if (ok && mbar_wait_warp_all(&bars->acc_done, 0, err)) {
      tc_fence_after();
      // Rows start on 256-byte boundaries of dQ (bf16) and 512-byte boundaries of the
      // partials (fp32): 32-byte stores where the base pointers allow them.
      const bool v8_out = (reinterpret_cast<uintptr_t>(dq_out) & 31) == 0;
      const bool v8_part = (reinterpret_cast<uintptr_t>(dq_part) & 31) == 0;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + T_DQ + c0 + half * 32, v);
        tmem_ld_wait();
        if (kSplit && slot >= 0) {
          // Split-KV item: the fp32 partial (times the scale) of its chunk.
          if (g.row_ok) {
            float* prow = dq_part + (slot * kFwdPartRows + r_local) * 128 + c0 + half * 32;
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * geo.scale);
            if (v8_part) {
#pragma unroll
              for (int i = 0; i < 4; ++i) st_global_v8(prow + 8 * i, v + 8 * i);
            } else {
              float4* d4 = reinterpret_cast<float4*>(prow);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                d4[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                    __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
            }
          }
        } else if (g.row_ok) {
          const bool any = n_tiles > 0;
          uint32_t o[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            o[i] = any ? pack_bf16x2(__uint_as_float(v[2 * i]) * geo.scale, __uint_as_float(v[2 * i + 1]) * geo.scale)
                       : 0u;
          __nv_bfloat16* orow = dq_out + (g.row * geo.hq + h) * 128 + c0 + half * 32;
          if (v8_out) {
            st_global_v8(orow, o);
            st_global_v8(orow + 16, o + 8);
          } else {
            uint4* d4 = reinterpret_cast<uint4*>(orow);
#pragma unroll
            for (int i = 0; i < 4; ++i) d4[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  }  // units of the lane
  if (kPersistent) __syncthreads();  // an empty lane: the address is visible before it is freed
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(bars->tmem_base, 512);
  }
}

}  // namespace

cudaError_t tc_bwd_dq(const augtree_plan* p, int op, const void* q, const void* kp, const void* vp, const void* kr,
                      const void* vr, const float* stats, const void* dO, void* dq, float* dq_part,
                      cudaStream_t st) {
  // The query-side items of the backward are those of the matching forward op.
  const bool prefill = op == AUGTREE_OP_PREFILL_BWD;
  const int fop = prefill ? AUGTREE_OP_PREFILL_FWD : AUGTREE_OP_REPLAY_FWD;
  if (p->n_items[fop] == 0) return cudaSuccess;
  const int64_t q_rows = prefill ? p->total_prompt : p->total_resp;
  CUtensorMap mq, mdo, mkp, mvp, mkr, mvr;
  if (!encode_rows_map(&mq, q, q_rows, p->cfg.hq, 128)) return cudaErrorInvalidValue;
  if (!encode_rows_map(&mdo, dO, q_rows, p->cfg.hq, 128)) return cudaErrorInvalidValue;
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
  if (!have_p) {
    mkp = have_r ? mkr : mq;
    mvp = have_r ? mvr : mq;
  }
  if (!have_r) {
    mkr = mkp;
    mvr = mvp;
  }
  // Persistent schedule: one block per lane, each walking its units.
  const LaneSet& ls = p->lanes_dq[fop];
  const bool persistent = ls.off_d != nullptr;
  // The split-KV instantiation only where the replay queue has split items.
  const bool split = !prefill && p->n_fwd_parts > 0;
  if (split && !dq_part) return cudaErrorInvalidValue;
  auto kern = persistent ? (split ? tc_bwd_dq_kernel<true, true> : tc_bwd_dq_kernel<true, false>)
                         : (split ? tc_bwd_dq_kernel<false, true> : tc_bwd_dq_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DQ_SMEM);
  if (e != cudaSuccess) return e;
  const unsigned grid = persistent ? (unsigned)ls.n_lanes : (unsigned)p->n_items[fop];
  // One block per SM runs at a time: the item a wave ahead is the one an SM's next block
  // is likely to take.
  int sms = 0;
  if (!persistent && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) sms = 0;
  kern<<<grid, DQ_THREADS, DQ_SMEM, st>>>(
      mq, mdo, mkp, mvp, mkr, mvr, geometry(p), p->queue_d[fop], p->bm[fop], p->bn[fop], stats,
      prefill ? p->ntiles_p : p->ntiles_r, (__nv_bfloat16*)dq, p->err_d, persistent ? ls.off_d : nullptr,
      persistent ? ls.units_d : nullptr, dq_part, (int64_t)p->n_items[fop], kDqPrefetchNextWave ? sms : 0);
  return cudaGetLastError();
}

}  // namespace augtree
