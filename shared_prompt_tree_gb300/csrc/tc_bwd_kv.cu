// Tensor-core backward of tree attention on sm_103a, key side: dK and dV
// (KV-stationary).
//
// AugTree paper, "Splitting Prompt Prefill from Response Replay ...":
//   Sec. 3.2, Eq. 2  the prompt K/V gradient is the sum over all G branches of the
//                    branch losses' gradients; it is accumulated and then sent back
//                    through the prompt-prefill graph (prefill backward adds it);
//   Sec. 3.3         MoveQ keeps prompt KV stationary and brings the queries of every
//                    branch to it - on one GPU: a thread block owns one prompt K/V tile
//                    and walks the response query tiles of all branches (split into a
//                    few chunks when the prompt has few tiles; the chunks' partial sums
//                    are reduced in a fixed order afterwards, no atomics).
//
// One thread block per work item: 128 keys of one KV head, query tiles [a, b) of BMQ
// rows for each of the r query heads of that KV head (in the fused backward, split 0
// of a prompt KV tile also walks the prompt's own causal query tiles, so one
// accumulator holds the prompt gradient's replay and prefill parts).  Per query tile
// (keys are the MMA M dimension, one key per TMEM lane):
//   S^T  = K Q^T - lse/s   (TMEM, fp32)  -> P^T  = exp2(s log2e S^T),   bf16 over S^T
//   dP^T = V dO^T - Delta  (TMEM, fp32)  -> dS^T = P^T dP^T,            bf16 over dP^T
//   dV  += P^T dO          (A = P^T from TMEM, B = dO read MN-major)
//   dK  += dS^T Q          (A = dS^T from TMEM, B = Q read MN-major)
// The per-query terms -lse/s and -Delta enter through one extra K=16 MMA step each
// (a ones column block times three-way bf16 splits of the values), so the compute
// warps need no per-query values at all: no shared-memory broadcast loads, which would
// otherwise take about as much shared-memory bandwidth as the MMA operands.
// dQ is computed by the query-side kernel, so nothing here leaves the SM per query
// tile.
// MMA issue order per tile: dV(i), S(i+1), dK(i), dP(i+1).  S(i+1) overwrites the
// columns dV reads and dP(i+1) those dK reads: with 128-row tiles each waits for the
// completion of the group issued just before it (measured at about 280 cycles after
// its last issue); with 64-row tiles S^T and dP^T are double-buffered (64 columns each)
// and the waits target MMAs issued one tile earlier.  128-row tiles measured faster:
// N=64 MMAs issue no faster than about 50 cycles each, and 64-row tiles take twice as
// many round trips between the MMA issuer and the compute warps per unit of work.
// Warps: 0 .. 4 NWG - 1 compute warpgroups, warpgroup w takes query columns
//        [COLS w, COLS (w + 1)) of every tile (thread = key = TMEM lane); then the TMA
//        producer warp, the TMEM allocator + issuer of S^T and dP^T, and the issuer of
//        dV and dK.
// TMEM columns: S^T/P^T [0,128), dP^T/dS^T [128,256) (each 2 x 64 when double-
// buffered), dV [256,384), dK [384,512).
#include <cuda.h>

#include <cmath>

#include "common.cuh"
#include "tc_common.cuh"

namespace augtree {
namespace {

using namespace tc;

constexpr int BMQ = kTcBwdKvRows;                       // query rows per tile (128 or 64)
// With 64-row tiles S^T and dP^T are double-buffered in TMEM (two 64-column halves);
// with 128-row tiles they take 128 columns each and are reused every tile.
constexpr bool DB = BMQ == 64;
// One exponential in kKvExpFma of the P^T phase runs on the FMA pipe (exp2_fma): the
// phase is MUFU-bound (16 exponentials per clock per SM), on the critical chain
// S(i) -> P(i) -> dV(i) -> S(i+1).  Measured on this kernel (prompt-heavy, TFLOP/s):
// none 1,357; one in 4: 1,335; in 6: 1,410; in 8: 1,393; in 12: 1,406; in 16: 1,400.
#ifndef AUGTREE_KV_EXP_FMA
#define AUGTREE_KV_EXP_FMA 12
#endif
constexpr int kKvExpFma = AUGTREE_KV_EXP_FMA;           // 0, or N: one exponential in N via exp2_fma
static_assert(kKvExpFma == 0 || (kKvExpFma >= 2 && kKvExpFma % 2 == 0), "exp2_fma fraction");
constexpr int NWG = 2;                                  // compute warpgroups
constexpr int COLS = BMQ / NWG;                         // query columns per warpgroup
constexpr int PRODUCER_WARP = 4 * NWG, MMA_WARP = 4 * NWG + 1, MMA2_WARP = 4 * NWG + 2;
constexpr int KV_THREADS = (4 * NWG + 3) * 32;
constexpr int NQ = DB ? 4 : 2;                          // Q/dO ring stages
constexpr int kPrefetch = DB ? 6 : 4;                   // L2 prefetch distance (iterations)
constexpr int BLK = 128 * 128;                          // 128 keys x 64 dims bf16 = 16 KB
constexpr int QBLK = BMQ * 128;                         // BMQ rows x 64 dims bf16
constexpr int K_OFF = 0;                                // 2 blocks
constexpr int V_OFF = K_OFF + 2 * BLK;                  // 2 blocks
constexpr int Q_OFF = V_OFF + 2 * BLK;                  // [NQ][2 blocks]
constexpr int DO_OFF = Q_OFF + NQ * 2 * QBLK;           // [NQ][2 blocks]
// Operands of the extra K=16 step that adds -lse/s to S^T and -Delta to dP^T: a constant
// A = [1 1 1 0 ... 0] per key and, per stage, B rows {hi, mid, lo, 0, ...} of -lse/s (L)
// and -Delta (D) per query row.  Unswizzled K-major layout: core matrices of 8 rows x 16
// bytes, 8-row groups 128 bytes apart; the second core matrix along K (columns 8-15) is
// a zero block AUG_LBO bytes further.
constexpr int AUG_ROWS = BMQ * 16;                      // bytes of one L or D block
constexpr int AUG_LBO = 2 * AUG_ROWS;
constexpr int AUGA_OFF = DO_OFF + NQ * 2 * QBLK;        // 2 KB ones rows + 2 KB zeros
constexpr int AUG_OFF = AUGA_OFF + 4096;                // [NQ] x {L, D, zeros x 2}
constexpr int AUG_STAGE = 4 * AUG_ROWS;
constexpr int BAR_OFF = AUG_OFF + NQ * AUG_STAGE;
constexpr int KV_SMEM = BAR_OFF + 512 + 1024;

constexpr uint32_t T_ST = 0, T_DPT = 128, T_DV = 256, T_DK = 384;  // DB: S^T / dP^T buffer b at + 64 b
// TMEM buffer, barrier index and barrier phase of tile i.
__device__ __forceinline__ int kv_buf(int i) { return DB ? (i & 1) : 0; }
__device__ __forceinline__ uint32_t kv_phase(int i) { return DB ? ((i >> 1) & 1) : (i & 1); }

// The tensor cores' fp32 accumulation into TMEM carries a small rounding bias per
// accumulation (measured at about 1e-8 relative), which adds up over the tens of
// thousands of accumulations of a long item.  Every kFlush query tiles the dK/dV
// accumulators are therefore moved into an fp32 slot (round-to-nearest adds) and the
// tensor-core accumulation restarts from zero.
constexpr int kFlush = 32768 / BMQ;  // 2048 accumulation steps (16 query rows each) of dK/dV

struct KvBars {
  uint64_t kv_full;
  uint64_t q_full[NQ];
  uint64_t q_empty[NQ];
  // per TMEM buffer b = tile % 2
  uint64_t s_full[2];
  uint64_t dp_full[2];
  uint64_t p_ready[2];
  uint64_t ds_ready[2];
  uint64_t dv_done[2];
  uint64_t dk_done[2];
  uint64_t acc_done;
  uint64_t flush_ready;  // dK/dV accumulators complete up to a flush point
  uint64_t flushed;      // compute warps have moved them to the slot
  uint64_t drain;        // every S^T / dP^T MMA of the first issuer has completed
  uint32_t tmem_base;
};

static_assert(sizeof(KvBars) <= 512, "barrier area");

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void bulk_prefetch(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}

template <bool kPersistent>
__global__ void __launch_bounds__(KV_THREADS, 1) tc_bwd_kv_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const __grid_constant__ CUtensorMap tm_k2, const __grid_constant__ CUtensorMap tm_v2,
    const __grid_constant__ CUtensorMap tm_q2, const __grid_constant__ CUtensorMap tm_do2, Geometry geo,
    const int32_t* __restrict__ queue, const int32_t* __restrict__ row_bend, int bm, int bn,
    const uint8_t* __restrict__ aug, int ntiles, const uint8_t* __restrict__ aug2, int ntiles2,
    __nv_bfloat16* __restrict__ dk_out, __nv_bfloat16* __restrict__ dv_out, __nv_bfloat16* __restrict__ dk2_out,
    __nv_bfloat16* __restrict__ dv2_out, float* __restrict__ dk_part, float* __restrict__ dv_part,
    float* __restrict__ dk_sum, float* __restrict__ dv_sum, const float* __restrict__ dk_add,
    const float* __restrict__ dv_add, float* __restrict__ slots, int n_slots, uint32_t* __restrict__ err,
    const int32_t* __restrict__ sched_off, const int32_t* __restrict__ sched_units) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  KvBars* bars = reinterpret_cast<KvBars*>(smem + BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // TMEM: allocated once for every unit of the lane (persistent schedule) or, as the
  // block's first step, for its one unit (queue schedule, below).
  if (kPersistent && warp == MMA_WARP) tmem_alloc(&bars->tmem_base, 512);
  // The queue schedule's instantiation runs exactly one unit (the loop folds away).
  const int n_units = kPersistent ? sched_off[blockIdx.x + 1] - sched_off[blockIdx.x] : 1;
  for (int u_i = 0; u_i < n_units; ++u_i) {
  const int64_t unit = kPersistent ? (int64_t)sched_units[sched_off[blockIdx.x] + u_i] : (int64_t)blockIdx.x;

  const WorkItem it = load_item(queue, unit);
  const bool item_ok = !kChecked || key_item_ok(it, geo, bm, bn);  // checked build only
  if (kChecked && !item_ok && threadIdx.x == 0) atomicOr(err, kErrCheck);
  const GroupInfo G = geo.groups[item_ok ? it.group : 0];
  const int r = geo.hq / geo.hkv;
  const int kvh = item_ok ? it.head : 0;
  const bool resp_keys = it.kind == K_RESP_KV;
  const bool prefill = it.kind == K_PREFILL_KV;
  const bool tree_p = it.kind == K_TREE_PROMPT_KV;
  const int64_t kbase = resp_keys ? G.r0 : G.p0;
  const int64_t key0 = kbase + (item_ok ? (int64_t)it.tile * bn : 0);
  const int64_t key_end = min(key0 + (int64_t)bn, kbase + (int64_t)(resp_keys ? G.lr : G.lp));
  // Primary query tiles [a, b): prompt rows for PREFILL_KV, response rows otherwise.
  const int64_t qbase = prefill ? G.p0 : G.r0;
  const int64_t q_end = qbase + (prefill ? G.lp : G.lr);
  const int nqt = it.b - it.a;
  // Secondary query tiles (fused backward, split 0 only): the prompt's own causal query
  // tiles [qa2, qb2) of this prompt KV tile, read through tm_q2 / tm_do2 / aug2.
  const int qb2 = (int)((G.lp + bm - 1) / bm);
  const int qa2 = (int)(((int64_t)it.tile * bn) / bm);
  const int nqt2 = (tree_p && it.split == 0) ? qb2 - qa2 : 0;
  const int nph = nqt + nqt2;  // query tiles per query head
  const int n_iter = item_ok ? nph * r : 0;
  // One block per SM at a time (shared memory and TMEM), so the SM id names a private
  // flush slot.
  uint32_t smid;
  asm("mov.u32 %0, %%smid;" : "=r"(smid));
  const bool flush_on = n_iter > kFlush && (int)smid < n_slots;
  if (n_iter > kFlush && (int)smid >= n_slots && threadIdx.x == 0) atomicOr(err, 2u);
  // Iteration i: query tile l = i / r of the walk, query head kvh*r + i % r (the r heads
  // of one tile back to back); the walk takes the primary tiles b - 1 down to a, then
  // the secondary tiles qb2 - 1 down to qa2.  Every item of a (group, KV head) thus walks
  // the same sequence of Q/dO tiles from the same first tile and only stops at its own
  // last one: blocks of one (group, KV head) that run side by side stay in step and read
  // each tile from L2 once for all of them (the work queue keeps such items together).
  struct QTile {
    int h, qt;
    bool sec;
  };
  auto qtile = [&](int i) {
    QTile t;
    const int l = i / r;
    t.h = kvh * r + i % r;
    t.sec = l >= nqt;
    t.qt = t.sec ? qb2 - 1 - (l - nqt) : it.b - 1 - l;
    return t;
  };

  if (threadIdx.x == 0) {
    if (kPersistent && u_i > 0) {
      // Every wait, copy and MMA of the previous unit has ended (drains, then the
      // block-wide barrier at its end): its barriers are idle and may be reused.
      for (uint64_t* b = &bars->kv_full; b < reinterpret_cast<uint64_t*>(&bars->tmem_base); ++b) mbar_inval(b);
    }
    mbar_init(&bars->kv_full, 1);
    for (int i = 0; i < NQ; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->dp_full[b], 1);
      mbar_init(&bars->p_ready[b], 128 * NWG);
      mbar_init(&bars->ds_ready[b], 128 * NWG);
      mbar_init(&bars->dv_done[b], 1);
      mbar_init(&bars->dk_done[b], 1);
    }
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->flush_ready, 1);
    mbar_init(&bars->flushed, 128 * NWG);
    mbar_init(&bars->drain, 1);
    fence_mbar_init();
  }
  {
    uint4* a = reinterpret_cast<uint4*>(smem + AUGA_OFF);
    for (int r = threadIdx.x; r < 128; r += blockDim.x) a[r] = make_uint4(0x3F803F80u, 0x3F80u, 0u, 0u);  // bf16 1,1,1
    for (int r = threadIdx.x; r < 128; r += blockDim.x) a[128 + r] = make_uint4(0u, 0u, 0u, 0u);
    for (int st = 0; st < NQ; ++st) {
      uint4* z = reinterpret_cast<uint4*>(smem + AUG_OFF + st * AUG_STAGE + 2 * AUG_ROWS);
      for (int r = threadIdx.x; r < 2 * AUG_ROWS / 16; r += blockDim.x) z[r] = make_uint4(0u, 0u, 0u, 0u);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (!kPersistent && warp == MMA_WARP) tmem_alloc(&bars->tmem_base, 512);
  if (warp == PRODUCER_WARP && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_do);
    if (nqt2 > 0) {
      prefetch_tmap(&tm_q2);
      prefetch_tmap(&tm_do2);
    }
    prefetch_tmap(resp_keys ? &tm_k2 : &tm_k);
    prefetch_tmap(resp_keys ? &tm_v2 : &tm_v);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const CUtensorMap* km = resp_keys ? &tm_k2 : &tm_k;
      const CUtensorMap* vm = resp_keys ? &tm_v2 : &tm_v;
      mbar_expect_tx(&bars->kv_full, 4 * BLK);
      for (int kb = 0; kb < 2; ++kb) {
        tma_load_3d(smem + K_OFF + kb * BLK, km, &bars->kv_full, kb * 64, kvh, (int)key0);
        tma_load_3d(smem + V_OFF + kb * BLK, vm, &bars->kv_full, kb * 64, kvh, (int)key0);
      }
      const int tile_base = prefill ? G.tp0 : G.tr0;
      // The {-lse/s, -Delta} rows of query tile qt are those of 128-row statistics tile
      // qt * BMQ / 128 (one half of them for 64-row tiles); secondary tiles are prompt rows.
      auto aug_src = [&](const QTile& t) {
        constexpr int per = kStatRows / BMQ;
        const uint8_t* a = t.sec ? aug2 : aug;
        const int64_t nt = t.sec ? ntiles2 : ntiles, tb = t.sec ? G.tp0 : tile_base;
        return a + ((int64_t)t.h * nt + tb + t.qt / per) * kAugTileBytes + (t.qt % per) * AUG_ROWS;
      };
      auto row_of = [&](const QTile& t) { return (t.sec ? (int64_t)G.p0 : qbase) + (int64_t)t.qt * bm; };
      int issued = 0;
      for (int i = 0; i < n_iter; ++i) {
        const int stage = i % NQ, use = i / NQ;
        if (!mbar_wait(&bars->q_empty[stage], (use & 1) ^ 1, err)) break;
        const QTile t = qtile(i);
        const int64_t row0 = row_of(t);
        const CUtensorMap* qm = t.sec ? &tm_q2 : &tm_q;
        const CUtensorMap* om = t.sec ? &tm_do2 : &tm_do;
        mbar_expect_tx(&bars->q_full[stage], 4 * QBLK + 2 * AUG_ROWS);
        // Q and its -lse/s rows first (S^T needs them first), then dO and its -Delta rows.
        const uint8_t* src = aug_src(t);
        for (int kb = 0; kb < 2; ++kb)
          tma_load_3d(smem + Q_OFF + (stage * 2 + kb) * QBLK, qm, &bars->q_full[stage], kb * 64, t.h, (int)row0);
        bulk_load(smem + AUG_OFF + stage * AUG_STAGE, src, AUG_ROWS, &bars->q_full[stage]);
        for (int kb = 0; kb < 2; ++kb)
          tma_load_3d(smem + DO_OFF + (stage * 2 + kb) * QBLK, om, &bars->q_full[stage], kb * 64, t.h, (int)row0);
        bulk_load(smem + AUG_OFF + stage * AUG_STAGE + AUG_ROWS, src + kStatRows * 16, AUG_ROWS, &bars->q_full[stage]);
        issued = i + 1;
        // Warm L2 with the tiles a few iterations ahead.
        const int ip = i + kPrefetch;
        if (ip < n_iter) {
          const QTile tp = qtile(ip);
          const int rp = (int)row_of(tp);
          for (int kb = 0; kb < 2; ++kb) {
            tma_prefetch_3d(tp.sec ? &tm_q2 : &tm_q, kb * 64, tp.h, rp);
            tma_prefetch_3d(tp.sec ? &tm_do2 : &tm_do, kb * 64, tp.h, rp);
          }
          const uint8_t* ap = aug_src(tp);
          bulk_prefetch(ap, AUG_ROWS);
          bulk_prefetch(ap + kStatRows * 16, AUG_ROWS);
        }
      }
      // Never leave a copy in flight (also after giving up on a wait).
      mbar_wait_drain(&bars->kv_full, 0, err);
      for (int i = max(0, issued - NQ); i < issued; ++i) mbar_wait_drain(&bars->q_full[i % NQ], (i / NQ) & 1, err);
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer: S^T, dP^T
    if (lane == 0) {
      constexpr uint32_t id_ss = idesc_bf16_f32(128, BMQ, false, false);  // K Q^T, V dO^T
      const uint64_t dK = smem_desc_sw128(smem_u32(smem + K_OFF), 16, 1024);
      const uint64_t dV = smem_desc_sw128(smem_u32(smem + V_OFF), 16, 1024);
      const uint64_t dQk0 = smem_desc_sw128(smem_u32(smem + Q_OFF), 16, 1024);
      const uint64_t dOk0 = smem_desc_sw128(smem_u32(smem + DO_OFF), 16, 1024);
      constexpr uint64_t kStage = (2 * QBLK) >> 4;
      const uint64_t dAa = smem_desc_noswz(smem_u32(smem + AUGA_OFF), 2048, 128);
      const uint64_t dL0 = smem_desc_noswz(smem_u32(smem + AUG_OFF), AUG_LBO, 128);
      const uint64_t dD0 = smem_desc_noswz(smem_u32(smem + AUG_OFF + AUG_ROWS), AUG_LBO, 128);
      constexpr uint64_t kAugStage = AUG_STAGE >> 4;
      auto koff = [](int kk) { return (uint64_t)(((kk >> 2) * BLK + (kk & 3) * 32) >> 4); };   // K, V
      auto qoff = [](int kk) { return (uint64_t)(((kk >> 2) * QBLK + (kk & 3) * 32) >> 4); };  // Q, dO
      auto issue_s = [&](int i) {
        const uint64_t b = dQk0 + (i % NQ) * kStage;
        const uint32_t d = tmem + T_ST + kv_buf(i) * 64;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(d, dK + koff(kk), b + qoff(kk), id_ss, kk > 0 ? 1u : 0u);
        mma_ss(d, dAa, dL0 + (i % NQ) * kAugStage, id_ss, 1u);  // - lse/s
        mma_commit(&bars->s_full[kv_buf(i)]);
      };
      auto issue_dp = [&](int i) {
        const uint64_t b = dOk0 + (i % NQ) * kStage;
        const uint32_t d = tmem + T_DPT + kv_buf(i) * 64;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(d, dV + koff(kk), b + qoff(kk), id_ss, kk > 0 ? 1u : 0u);
        mma_ss(d, dAa, dD0 + (i % NQ) * kAugStage, id_ss, 1u);  // - Delta
        mma_commit(&bars->dp_full[kv_buf(i)]);
      };
      bool ok = mbar_wait(&bars->kv_full, 0, err);
      if (ok && n_iter > 0) ok = mbar_wait(&bars->q_full[0], 0, err);
      tc_fence_after();
      if (ok && n_iter > 0) {
        issue_s(0);
        issue_dp(0);
      }
      for (int i = 0; ok && i + 1 < n_iter; ++i) {
        // The tile whose dV/dK last read the buffers that tile i + 1 overwrites: i - 1
        // with double buffering, i itself otherwise (issued by the other issuer).
        const int prev = DB ? i - 1 : i;
        // S(i+1) overwrites P^T(prev): dV(prev) must have read it.
        if (!(ok = mbar_wait(&bars->q_full[(i + 1) % NQ], ((i + 1) / NQ) & 1, err))) break;
        if (prev >= 0 && !(ok = mbar_wait(&bars->dv_done[kv_buf(prev)], kv_phase(prev), err))) break;
        tc_fence_after();
        issue_s(i + 1);
        // dP(i+1) overwrites dS^T(prev): dK(prev) must have read it.
        if (prev >= 0 && !(ok = mbar_wait(&bars->dk_done[kv_buf(prev)], kv_phase(prev), err))) break;
        tc_fence_after();
        issue_dp(i + 1);
      }
      // Never leave an MMA in flight when the block frees TMEM and exits (also after
      // giving up on a wait).
      mma_commit(&bars->drain);
      mbar_wait_drain(&bars->drain, 0, err);
    }
  } else if (warp == MMA2_WARP) {
    // ------------------------------------------------------------ MMA issuer: dV, dK
    // A second issuing thread: while one issuer waits on a completion, the other keeps
    // the tensor pipe fed (two issuers measured 72 cycles per N=128 MMA with a wait per
    // group, one issuer 92; 64 is the full rate).
    if (lane == 0) {
      constexpr uint32_t id_ts = idesc_bf16_f32(128, 128, false, true);  // P^T dO, dS^T Q (B MN-major)
      const uint64_t dQm0 = smem_desc_sw128(smem_u32(smem + Q_OFF), QBLK, 1024);
      const uint64_t dOm0 = smem_desc_sw128(smem_u32(smem + DO_OFF), QBLK, 1024);
      constexpr uint64_t kStage = (2 * QBLK) >> 4;
      // TMEM column of the bf16 A operand for query step kk (16 rows): warpgroup w packed
      // rows [COLS w, COLS (w + 1)) into columns [COLS w, COLS w + COLS / 2) of the buffer.
      auto acol = [](int kk) { return (uint32_t)((kk / (COLS / 16)) * COLS + (kk % (COLS / 16)) * 8); };
      bool ok = true;
      for (int i = 0; ok && i < n_iter; ++i) {
        const int stage = i % NQ;
        const int b = kv_buf(i);
        const bool more = i + 1 < n_iter;
        const bool fresh = flush_on ? (i % kFlush == 0) : (i == 0);
        // dV += P^T dO (from zero at the start and after every flush)
        if (flush_on && i > 0 && i % kFlush == 0 && !(ok = mbar_wait(&bars->flushed, (i / kFlush - 1) & 1, err)))
          break;
        if (!(ok = mbar_wait(&bars->p_ready[b], kv_phase(i), err))) break;
        tc_fence_after();
        {
          const uint64_t b0 = dOm0 + stage * kStage;
          const uint32_t a0 = tmem + T_ST + b * 64;
#pragma unroll
          for (int kk = 0; kk < BMQ / 16; ++kk)
            mma_ts(tmem + T_DV, a0 + acol(kk), b0 + kk * (2048 >> 4), id_ts, (fresh && kk == 0) ? 0u : 1u);
        }
        mma_commit(&bars->dv_done[b]);
        // dK += dS^T Q
        if (!(ok = mbar_wait(&bars->ds_ready[b], kv_phase(i), err))) break;
        tc_fence_after();
        {
          const uint64_t b0 = dQm0 + stage * kStage;
          const uint32_t a0 = tmem + T_DPT + b * 64;
#pragma unroll
          for (int kk = 0; kk < BMQ / 16; ++kk)
            mma_ts(tmem + T_DK, a0 + acol(kk), b0 + kk * (2048 >> 4), id_ts, (fresh && kk == 0) ? 0u : 1u);
        }
        mma_commit(&bars->dk_done[b]);
        // dK(i) is the last reader of Q(i)/dO(i) and of the stage's extra-step rows (S(i)
        // and dP(i) completed before P^T(i) and dS^T(i) existed).
        mma_commit(&bars->q_empty[stage]);
        if (flush_on && i % kFlush == kFlush - 1 && more) mma_commit(&bars->flush_ready);
      }
      // All MMAs of the item are complete once the last dK is.  Wait for that here too,
      // so that no MMA of this thread is in flight when the block frees TMEM (also after
      // giving up on a wait).
      mma_commit(&bars->acc_done);
      mbar_wait_drain(&bars->acc_done, 0, err);
    }
  } else {
    // ------------------------------------------------------------ P^T and dS^T
    const int w = warp >> 2;                 // query columns [COLS w, COLS (w + 1))
    const int q4 = warp & 3;                 // TMEM lane quarter
    const int t = q4 * 32 + lane;            // key row / TMEM lane
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const int c0 = COLS * w;
    const int64_t key = key0 + t;
    const bool key_ok = key < key_end;
    // valid query rows for this key: [q_lo, q_hi)
    int64_t q_lo = qbase, q_hi = q_end;
    if (prefill) q_lo = key;
    if (resp_keys) {
      q_lo = key;
      const int64_t be = key_ok ? (int64_t)row_bend[key] : key;
      q_hi = be < q_end ? be : q_end;
    }
    if (!key_ok) q_hi = q_lo;
    // Secondary (prompt) query tiles of a fused item: causal over the prompt.
    const int64_t q_lo2 = key, q_hi2 = key_ok ? (int64_t)G.p0 + G.lp : key;
    const float sl2 = geo.scale_log2;
    // This warpgroup's share of the key's {dK, dV} row (256 floats): [po, po + 256 / NWG).
    constexpr int SHARE = 256 / NWG;
    const int po = w * SHARE;
    const uint32_t acc_col = (po < 128 ? T_DK : T_DV) + (po & 127);
    bool ok = true;
    // Rows and keys are int32 offsets (the descriptors are int32), so the per-iteration
    // geometry runs in 32-bit arithmetic, and the walk position advances by counters
    // instead of a division by r.
    const int q_lo_i = (int)q_lo, q_hi_i = (int)q_hi, q_lo2_i = (int)q_lo2, q_hi2_i = (int)q_hi2;
    const int qbase_i = (int)qbase;
    int l = 0, lh = 0;  // iteration i = l * r + lh: query tile l of the walk, head lh
    for (int i = 0; i < n_iter; ++i) {
      const bool sec = l >= nqt;
      const int row0 = sec ? G.p0 + (qb2 - 1 - (l - nqt)) * bm : qbase_i + (it.b - 1 - l) * bm;
      const int v_lo = sec ? q_lo2_i : q_lo_i, v_hi = sec ? q_hi2_i : q_hi_i;
      const int b = kv_buf(i);
      const uint32_t ts = tmem + lane_off + T_ST + b * 64 + c0, tdp = tmem + lane_off + T_DPT + b * 64 + c0;
      if (!(ok = mbar_wait_warp_all(&bars->s_full[b], kv_phase(i), err))) break;
      tc_fence_after();
      uint32_t sraw[COLS / 32][32];
#pragma unroll
      for (int k = 0; k < COLS / 32; ++k) tmem_ld32(ts + 32 * k, sraw[k]);
      tmem_ld_wait();
      // this warpgroup's valid columns: [lo, hi) relative to c0
      const int lo = min(max(v_lo - row0 - c0, 0), COLS);
      const int hi = min(max(v_hi - row0 - c0, 0), COLS);
      // P^T as bf16 pairs (A operand of dV and the P factor of dS): the accumulator
      // already holds S^T - lse/s, so P = exp2(s log2e (S^T - lse/s)).
      uint32_t pk[COLS / 2];
      if (lo == 0 && hi == COLS) {
#pragma unroll
        for (int c = 0; c < COLS; c += 2) {
          const float e0 = fast_exp2(__uint_as_float(sraw[c >> 5][c & 31]) * sl2);
          const float x1 = __uint_as_float(sraw[(c + 1) >> 5][(c + 1) & 31]) * sl2;
          // One exponential in kKvExpFma on the FMA pipe: the MUFU sets this phase's pace.
          constexpr int kPairs = kKvExpFma > 0 ? kKvExpFma / 2 : 1;  // FMA exponential every kPairs pairs
          const float e1 = (kKvExpFma > 0 && (c / 2) % kPairs == kPairs - 1) ? exp2_fma(x1) : fast_exp2(x1);
          pk[c >> 1] = pack_bf16x2(e0, e1);
        }
      } else {
        const uint32_t span = (uint32_t)(hi - lo);  // valid iff (c - lo) < span (unsigned)
#pragma unroll
        for (int c = 0; c < COLS; c += 2) {
          float e0 = fast_exp2(__uint_as_float(sraw[c >> 5][c & 31]) * sl2);
          float e1 = fast_exp2(__uint_as_float(sraw[(c + 1) >> 5][(c + 1) & 31]) * sl2);
          e0 = (uint32_t)(c - lo) < span ? e0 : 0.f;
          e1 = (uint32_t)(c + 1 - lo) < span ? e1 : 0.f;
          pk[c >> 1] = pack_bf16x2(e0, e1);
        }
      }
      tmem_st_words<COLS / 2>(ts, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->p_ready[b]);
      // dS^T = P^T (dP^T - Delta), with the same bf16 P the dV product uses
      if (!(ok = mbar_wait_warp_all(&bars->dp_full[b], kv_phase(i), err))) break;
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < COLS / 32; ++k) tmem_ld32(tdp + 32 * k, sraw[k]);
      tmem_ld_wait();
      // the accumulator holds dP^T - Delta
#pragma unroll
      for (int c = 0; c < COLS / 2; ++c) {
        const int e0 = 2 * c, e1 = 2 * c + 1;
        const float p0 = __uint_as_float(pk[c] << 16), p1 = __uint_as_float(pk[c] & 0xFFFF0000u);
        const float d0 = p0 * __uint_as_float(sraw[e0 >> 5][e0 & 31]);
        const float d1 = p1 * __uint_as_float(sraw[e1 >> 5][e1 & 31]);
        pk[c] = pack_bf16x2(d0, d1);
      }
      tmem_st_words<COLS / 2>(tdp, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->ds_ready[b]);
      if (flush_on && i % kFlush == kFlush - 1 && i + 1 < n_iter) {
        // Move this warpgroup's share of dK/dV to this block's slot (the first flush
        // stores, later ones add).
        if (!(ok = mbar_wait_warp_all(&bars->flush_ready, (i / kFlush) & 1, err))) break;
        tc_fence_after();
        float* slot = slots + ((int64_t)smid * 128 + t) * 256 + po;
        const bool first = i == kFlush - 1;
#pragma unroll 1
        for (int c = 0; c < SHARE / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + acc_col + c * 32, v);
          tmem_ld_wait();
          float4* dst = reinterpret_cast<float4*>(slot + c * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float4 x = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                   __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
            if (!first) {
              const float4 y = dst[e];
              x.x += y.x; x.y += y.y; x.z += y.z; x.w += y.w;
            }
            dst[e] = x;
          }
        }
        tc_fence_before();
        mbar_arrive(&bars->flushed);
      }
      if (++lh == r) {
        lh = 0;
        ++l;
      }
    }
    // This warpgroup's share of the key's dK (scaled by s) / dV row
    if (ok && mbar_wait_warp_all(&bars->acc_done, 0, err) && n_iter > 0) {
      tc_fence_after();
      const bool is_dk = po < 128;
      const int col0 = po & 127;
      const int64_t off = (key * geo.hkv + kvh) * 128 + col0;
      float* fdst = nullptr;
      int64_t foff = off;
      __nv_bfloat16* bdst = is_dk ? dk_out : dv_out;
      const float* add = is_dk ? dk_add : dv_add;
      if (it.kind == K_PROMPT_KV || tree_p) {
        // Split groups write fp32 partials (reduced in split order afterwards); an unsplit
        // group writes the replay sum (PROMPT_KV) or, in the fused backward, the final
        // prompt gradient.
        const SplitInfo s = geo.splits[it.group];
        if (s.nsplit > 1) {
          fdst = is_dk ? dk_part : dv_part;
          foff = ((s.part_row0 + (int64_t)it.split * G.lp + (key - G.p0)) * geo.hkv + kvh) * 128 + col0;
        } else if (!tree_p) {
          fdst = is_dk ? dk_sum : dv_sum;
        } else {
          bdst = is_dk ? dk2_out : dv2_out;
          add = nullptr;
        }
      }
      const float mul = is_dk ? geo.scale : 1.f;
      const float* slot = slots + ((int64_t)smid * 128 + t) * 256 + po;
#pragma unroll 1
      for (int c = 0; c < SHARE / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + acc_col + c * 32, v);
        tmem_ld_wait();
        if (!key_ok) continue;
        float a[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) a[e] = __uint_as_float(v[e]);
        if (flush_on) {
#pragma unroll
          for (int e = 0; e < 32; ++e) a[e] += slot[c * 32 + e];
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) a[e] *= mul;
        if (fdst) {
          float4* d4 = reinterpret_cast<float4*>(fdst + foff + c * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e) d4[e] = make_float4(a[4 * e], a[4 * e + 1], a[4 * e + 2], a[4 * e + 3]);
        } else {
          if (add) {
            const float4* a4 = reinterpret_cast<const float4*>(add + off + c * 32);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float4 x = a4[e];
              a[4 * e] += x.x; a[4 * e + 1] += x.y; a[4 * e + 2] += x.z; a[4 * e + 3] += x.w;
            }
          }
          uint4* o4 = reinterpret_cast<uint4*>(bdst + off + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            o4[e] = make_uint4(pack_bf16x2(a[8 * e], a[8 * e + 1]), pack_bf16x2(a[8 * e + 2], a[8 * e + 3]),
                               pack_bf16x2(a[8 * e + 4], a[8 * e + 5]), pack_bf16x2(a[8 * e + 6], a[8 * e + 7]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  }  // units of the lane
  if (kPersistent) __syncthreads();  // an empty lane: the address is visible before it is freed
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(bars->tmem_base, 512);
  }
}

}  // namespace

cudaError_t tc_bwd_kv(const augtree_plan* p, int op, const void* q, const void* dO, const void* aug, const void* q2,
                      const void* dO2, const void* aug2, const void* kp, const void* vp, const void* kr, const void* vr,
                      void* dk_out, void* dv_out, void* dk2_out, void* dv2_out, float* dk_part, float* dv_part,
                      float* dk_sum, float* dv_sum, const float* dk_add, const float* dv_add, float* slots,
                      cudaStream_t st) {
  // Primary query rows: the prompt for prefill_bwd, the responses otherwise; secondary
  // query rows (the fused backward's prompt rows) come through q2 / dO2 / aug2.
  const bool prefill = op == AUGTREE_OP_PREFILL_BWD;
  const bool tree = op == AUGTREE_OP_TREE_BWD;
  if (p->n_items[op] == 0) return cudaSuccess;
  const int64_t q_rows = prefill ? p->total_prompt : p->total_resp;
  CUtensorMap mq, mdo, mq2, mdo2, mk, mv, mk2, mv2;
  if (p->bm[op] != BMQ || p->bn[op] != 128) return cudaErrorInvalidValue;
  const bool have_q = q_rows > 0 && q && dO;
  const bool have_q2 = tree && p->total_prompt > 0 && q2 && dO2;
  if (have_q) {
    if (!encode_rows_map(&mq, q, q_rows, p->cfg.hq, BMQ)) return cudaErrorInvalidValue;
    if (!encode_rows_map(&mdo, dO, q_rows, p->cfg.hq, BMQ)) return cudaErrorInvalidValue;
  }
  if (have_q2) {
    if (!encode_rows_map(&mq2, q2, p->total_prompt, p->cfg.hq, BMQ)) return cudaErrorInvalidValue;
    if (!encode_rows_map(&mdo2, dO2, p->total_prompt, p->cfg.hq, BMQ)) return cudaErrorInvalidValue;
  }
  if (!have_q && !have_q2) return cudaErrorInvalidValue;
  // Maps that the queue never reads alias a used one.
  if (!have_q) {
    mq = mq2;
    mdo = mdo2;
  }
  if (!have_q2) {
    mq2 = mq;
    mdo2 = mdo;
  }
  const bool have_p = p->total_prompt > 0 && kp && vp;
  const bool have_r = !prefill && p->total_resp > 0 && kr && vr;
  if (have_p) {
    if (!encode_rows_map(&mk, kp, p->total_prompt, p->cfg.hkv, 128)) return cudaErrorInvalidValue;
    if (!encode_rows_map(&mv, vp, p->total_prompt, p->cfg.hkv, 128)) return cudaErrorInvalidValue;
  }
  if (have_r) {
    if (!encode_rows_map(&mk2, kr, p->total_resp, p->cfg.hkv, 128)) return cudaErrorInvalidValue;
    if (!encode_rows_map(&mv2, vr, p->total_resp, p->cfg.hkv, 128)) return cudaErrorInvalidValue;
  }
  if (!have_p) {
    mk = have_r ? mk2 : mq;
    mv = have_r ? mv2 : mq;
  }
  if (!have_r) {
    mk2 = mk;
    mv2 = mv;
  }
  // Persistent schedule: one block per lane, each walking its units.
  const LaneSet& ls = p->lanes_kv[op];
  const bool persistent = ls.off_d != nullptr;
  auto kern = persistent ? tc_bwd_kv_kernel<true> : tc_bwd_kv_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, KV_SMEM);
  if (e != cudaSuccess) return e;
  const unsigned grid = persistent ? (unsigned)ls.n_lanes : (unsigned)p->n_items[op];
  kern<<<grid, KV_THREADS, KV_SMEM, st>>>(
      mq, mdo, mk, mv, mk2, mv2, mq2, mdo2, geometry(p), p->queue_d[op], p->row_bend_d, p->bm[op], p->bn[op],
      (const uint8_t*)aug, prefill ? p->ntiles_p : p->ntiles_r, (const uint8_t*)(aug2 ? aug2 : aug), p->ntiles_p,
      (__nv_bfloat16*)dk_out, (__nv_bfloat16*)dv_out, (__nv_bfloat16*)dk2_out, (__nv_bfloat16*)dv2_out, dk_part,
      dv_part, dk_sum, dv_sum, dk_add, dv_add, slots, kFlushSlots, p->err_d, persistent ? ls.off_d : nullptr,
      persistent ? ls.units_d : nullptr);
  return cudaGetLastError();
}

}  // namespace augtree
