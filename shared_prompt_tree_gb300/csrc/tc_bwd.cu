// Tensor-core backward of tree attention on sm_103a (KV-stationary).
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
// One thread block per work item: 128 keys of one KV head, query tiles [a, b) of 64
// rows for each of the r query heads of that KV head.  Per query tile (keys are the
// MMA M dimension, so P^T and dS^T come out with one key per TMEM lane):
//   S^T  = K Q^T            (TMEM, fp32)   -> P^T  = exp2(s S^T log2e - lse)
//   dP^T = V dO^T           (TMEM, fp32)   -> dS^T = P^T (dP^T - Delta)
//   dV  += P^T dO           (A = P^T from TMEM, bf16)
//   dK  += dS^T Q           (A = dS^T from shared memory, K-major)
//   dQ^T = K^T dS^T         (B = the same dS^T tile, MN-major) -> staged in shared
//                            memory as two [32 rows x 128 dims] fp32 halves, each
//                            added to the dQ accumulator with one TMA bulk reduce-add
// dS^T lives in two shared-memory buffers (128-byte swizzle), so dP^T(i+1) can be
// computed as soon as dP^T(i) has been read out of TMEM.
// Warps: 0-3 softmax/dS (thread = key), 4-7 dQ epilogue (thread = head dim),
//        8 TMA producer, 9 TMEM allocator + MMA issuer.
// TMEM columns: S^T x2 [0,128) (P^T over it), dP^T [128,192), dQ^T [192,256),
//               dV [256,384), dK [384,512).
#include <cuda.h>

#include <cmath>

#include "common.cuh"
#include "tc_common.cuh"

namespace augtree {
namespace {

using namespace tc;

constexpr int BWD_THREADS = 320;
constexpr int NQ = 3;                                   // Q/dO ring stages
constexpr int kPrefetch = 5;                            // L2 prefetch distance (iterations)
constexpr int KV_BLK = 128 * 128;                       // 128 rows x 64 dims bf16 = 16 KB
constexpr int Q_BLK = 64 * 128;                         // 64 rows x 64 dims bf16 = 8 KB
constexpr int K_OFF = 0;                                // 2 blocks
constexpr int V_OFF = K_OFF + 2 * KV_BLK;               // 2 blocks
constexpr int Q_OFF = V_OFF + 2 * KV_BLK;               // [NQ][2 blocks]
constexpr int DO_OFF = Q_OFF + NQ * 2 * Q_BLK;          // [NQ][2 blocks]
constexpr int DS_OFF = DO_OFF + NQ * 2 * Q_BLK;         // [2] dS^T [128 keys x 64 q] bf16
constexpr int DQ_OFF = DS_OFF + 2 * KV_BLK;             // dQ half tile [32 q x 128 d] fp32
constexpr int DQ_BYTES = 32 * 128 * 4;
constexpr int ROWS_OFF = DQ_OFF + DQ_BYTES;             // [NQ] x {lse2[64], delta[64]}
constexpr int BAR_OFF = ROWS_OFF + NQ * 2 * 64 * 4;
constexpr int BWD_SMEM = BAR_OFF + 256 + 1024;

constexpr uint32_t T_ST = 0, T_DPT = 128, T_DQT = 192, T_DV = 256, T_DK = 384;

// The tensor cores' fp32 accumulation into TMEM carries a small rounding bias per
// accumulation (measured at about 1e-8 relative), which adds up over the tens of
// thousands of accumulations of a long item.  Every kFlush query tiles the dK/dV
// accumulators are therefore moved into an fp32 slot (round-to-nearest adds) and the
// tensor-core accumulation restarts from zero.
constexpr int kFlush = 512;
constexpr int kSlotFloats = 128 * 256;  // per slot: 128 keys x {dK[128], dV[128]}

struct BwdBars {
  uint64_t kv_full;
  uint64_t q_full[NQ];
  uint64_t q_empty[NQ];
  uint64_t s_full[2];
  uint64_t dp_full;
  uint64_t dp_free;
  // Per-buffer signals: the softmax warps may run one query tile ahead of the MMA
  // issuer, so a single barrier could complete two phases before its waiter looks.
  uint64_t p_ready[2];
  uint64_t ds_ready[2];
  uint64_t ds_free[2];
  uint64_t dv_done;
  uint64_t dq_full;
  uint64_t dq_free;
  uint64_t acc_done;
  uint64_t flush_ready;  // dK/dV accumulators complete up to a flush point
  uint64_t flushed;      // softmax warps have moved them to the slot
  uint32_t tmem_base;
};

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// dQ tile [64 rows x 128 dims] fp32 in shared memory added to the global accumulator.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void bulk_prefetch(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void named_bar(int id, int n) { named_bar_sync(id, n); }

__global__ void __launch_bounds__(BWD_THREADS, 1) tc_bwd_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const __grid_constant__ CUtensorMap tm_k2, const __grid_constant__ CUtensorMap tm_v2,
    const __grid_constant__ CUtensorMap tm_dq, Geometry geo,
    const int32_t* __restrict__ queue, const int32_t* __restrict__ row_bend, int bm, int bn,
    const float* __restrict__ stats, int ntiles,
    __nv_bfloat16* __restrict__ dk_out, __nv_bfloat16* __restrict__ dv_out, float* __restrict__ dk_part,
    float* __restrict__ dv_part, float* __restrict__ dk_sum, float* __restrict__ dv_sum,
    const float* __restrict__ dk_add, const float* __restrict__ dv_add, float* __restrict__ slots, int n_slots,
    uint32_t* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const WorkItem it = load_item(queue, blockIdx.x);
  const GroupInfo G = geo.groups[it.group];
  const int r = geo.hq / geo.hkv;
  const int kvh = it.head;
  const bool resp_keys = it.kind == K_RESP_KV;
  const bool prefill = it.kind == K_PREFILL_KV;
  const int64_t kbase = resp_keys ? G.r0 : G.p0;
  const int64_t key0 = kbase + (int64_t)it.tile * bn;
  const int64_t key_end = min(key0 + (int64_t)bn, kbase + (int64_t)(resp_keys ? G.lr : G.lp));
  const int64_t qbase = prefill ? G.p0 : G.r0;
  const int64_t q_end = qbase + (prefill ? G.lp : G.lr);
  const int64_t q_rows_total = prefill ? geo.total_prompt : geo.total_resp;
  const int nqt = it.b - it.a;
  const int n_iter = nqt * r;
  // One block per SM at a time (shared memory and TMEM), so the SM id names a private
  // flush slot.
  uint32_t smid;
  asm("mov.u32 %0, %%smid;" : "=r"(smid));
  const bool flush_on = n_iter > kFlush && (int)smid < n_slots;
  if (n_iter > kFlush && (int)smid >= n_slots && threadIdx.x == 0) atomicOr(err, 2u);
  // Iteration i: query head kvh*r + i / nqt, query tile b - 1 - i % nqt.  Tiles are
  // walked from the last one down, so blocks that start together (largest first) and
  // share a KV head meet the same query rows at about the same time: their Q/dO reads
  // and dQ reductions then hit the same L2 lines.

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int i = 0; i < NQ; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
    }
    mbar_init(&bars->s_full[0], 1);
    mbar_init(&bars->s_full[1], 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->dp_free, 128);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->p_ready[b], 128);
      mbar_init(&bars->ds_ready[b], 128);
      mbar_init(&bars->ds_free[b], 1);
    }
    mbar_init(&bars->dv_done, 1);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, 128);
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->flush_ready, 1);
    mbar_init(&bars->flushed, 128);
    fence_mbar_init();
  }
  if (warp == 9) tmem_alloc(&bars->tmem_base, 512);
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_do);
    prefetch_tmap(resp_keys ? &tm_k2 : &tm_k);
    prefetch_tmap(resp_keys ? &tm_v2 : &tm_v);
    prefetch_tmap(&tm_dq);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    int issued = 0;
    bool ok = true;
    if (lane == 0) {
      const CUtensorMap* km = resp_keys ? &tm_k2 : &tm_k;
      const CUtensorMap* vm = resp_keys ? &tm_v2 : &tm_v;
      mbar_expect_tx(&bars->kv_full, 4 * KV_BLK);
      for (int kb = 0; kb < 2; ++kb) {
        tma_load_3d(smem + K_OFF + kb * KV_BLK, km, &bars->kv_full, kb * 64, kvh, (int)key0);
        tma_load_3d(smem + V_OFF + kb * KV_BLK, vm, &bars->kv_full, kb * 64, kvh, (int)key0);
      }
    }
    const int tile_base = prefill ? G.tp0 : G.tr0;
    for (int i = 0; i < n_iter && lane == 0; ++i) {
      const int stage = i % NQ, use = i / NQ;
      if (!(ok = mbar_wait(&bars->q_empty[stage], (use & 1) ^ 1, err))) break;
      const int h = kvh * r + i / nqt;
      const int qt = it.b - 1 - i % nqt;
      const int64_t row0 = qbase + (int64_t)qt * bm;
      mbar_expect_tx(&bars->q_full[stage], 4 * Q_BLK + 2 * kStatRows * 4);
      for (int kb = 0; kb < 2; ++kb) {
        tma_load_3d(smem + Q_OFF + (stage * 2 + kb) * Q_BLK, &tm_q, &bars->q_full[stage], kb * 64, h, (int)row0);
        tma_load_3d(smem + DO_OFF + (stage * 2 + kb) * Q_BLK, &tm_do, &bars->q_full[stage], kb * 64, h, (int)row0);
      }
      // {lse * log2(e), Delta} of the tile's 64 rows: one 512-byte bulk copy.
      bulk_load(smem + ROWS_OFF + stage * 2 * kStatRows * 4,
                stats + ((int64_t)h * ntiles + tile_base + qt) * 2 * kStatRows, 2 * kStatRows * 4,
                &bars->q_full[stage]);
      issued = i + 1;
      // Warm L2 with the tiles a few iterations ahead, so that their copies into shared
      // memory, issued once a stage frees up, do not wait on DRAM.
      const int ip = i + kPrefetch;
      if (ip < n_iter) {
        const int hp = kvh * r + ip / nqt;
        const int qp = it.b - 1 - ip % nqt;
        const int rp = (int)(qbase + (int64_t)qp * bm);
        for (int kb = 0; kb < 2; ++kb) {
          tma_prefetch_3d(&tm_q, kb * 64, hp, rp);
          tma_prefetch_3d(&tm_do, kb * 64, hp, rp);
        }
        bulk_prefetch(stats + ((int64_t)hp * ntiles + tile_base + qp) * 2 * kStatRows, 2 * kStatRows * 4);
      }
    }
    if (lane == 0) {
      // Never leave a copy in flight.
      mbar_wait(&bars->kv_full, 0, err);
      for (int i = max(0, issued - NQ); i < issued; ++i) mbar_wait(&bars->q_full[i % NQ], (i / NQ) & 1, err);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(128, 64, false, false);    // K Q^T, V dO^T
      constexpr uint32_t id_acc = idesc_bf16_f32(128, 128, false, true);  // P^T dO, dS^T Q (B MN-major)
      constexpr uint32_t id_dq = idesc_bf16_f32(128, 64, true, true);     // K^T dS^T
      // Descriptors are built once; each MMA step then only adds a compile-time offset
      // (in 16-byte units) to the start-address field.  This keeps the single issuing
      // thread's dependency chain per tcgen05.mma short.
      const uint64_t dK = smem_desc_sw128(smem_u32(smem + K_OFF), 16, 1024);      // K, K-major
      const uint64_t dV = smem_desc_sw128(smem_u32(smem + V_OFF), 16, 1024);      // V, K-major
      const uint64_t dKt = smem_desc_sw128(smem_u32(smem + K_OFF), KV_BLK, 1024);  // K^T, MN-major
      // Stage st of the Q/dO ring sits 2 * Q_BLK bytes after stage st - 1.
      const uint64_t dQk0 = smem_desc_sw128(smem_u32(smem + Q_OFF), 16, 1024);
      const uint64_t dOk0 = smem_desc_sw128(smem_u32(smem + DO_OFF), 16, 1024);
      const uint64_t dQm0 = smem_desc_sw128(smem_u32(smem + Q_OFF), Q_BLK, 1024);
      const uint64_t dOm0 = smem_desc_sw128(smem_u32(smem + DO_OFF), Q_BLK, 1024);
      constexpr uint64_t kStageStep = (2 * Q_BLK) >> 4;
      const uint64_t dSk0 = smem_desc_sw128(smem_u32(smem + DS_OFF), 16, 1024);       // dS^T, K-major
      const uint64_t dSm0 = smem_desc_sw128(smem_u32(smem + DS_OFF), KV_BLK, 1024);   // dS^T, MN-major
      constexpr uint64_t kDsStep = KV_BLK >> 4;  // second dS^T buffer
      // K-major k-step kk: block kk/4, 32 bytes per step inside the 128-byte row.
      auto koff_kv = [](int kk) { return (uint64_t)(((kk >> 2) * KV_BLK + (kk & 3) * 32) >> 4); };
      auto koff_q = [](int kk) { return (uint64_t)(((kk >> 2) * Q_BLK + (kk & 3) * 32) >> 4); };
      bool ok = mbar_wait(&bars->kv_full, 0, err);
      tc_fence_after();
      auto issue_s = [&](int i) {  // S^T(i) -> ST[i % 2]
        const int st = i % NQ;
        const uint32_t d = tmem + T_ST + (i & 1) * 64;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(d, dK + koff_kv(kk), dQk0 + st * kStageStep + koff_q(kk), id_s, kk > 0 ? 1u : 0u);
        mma_commit(&bars->s_full[i & 1]);
      };
      auto issue_dp = [&](int i) {  // dP^T(i) -> DPT
        const int st = i % NQ;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem + T_DPT, dV + koff_kv(kk), dOk0 + st * kStageStep + koff_q(kk), id_s, kk > 0 ? 1u : 0u);
        mma_commit(&bars->dp_full);
      };
      if (ok && n_iter > 0) {
        ok = mbar_wait(&bars->q_full[0], 0, err);
        tc_fence_after();
        if (ok) {
          issue_s(0);
          issue_dp(0);
        }
      }
      for (int i = 0; ok && i < n_iter; ++i) {
        const int stage = i % NQ;
        const bool more = i + 1 < n_iter;
        // S^T(i+1) into the other S buffer, once dV(i-1) has consumed its P^T(i-1).
        if (more) {
          if (!(ok = mbar_wait(&bars->q_full[(i + 1) % NQ], ((i + 1) / NQ) & 1, err))) break;
          if (i >= 1 && !(ok = mbar_wait(&bars->dv_done, (i - 1) & 1, err))) break;
          tc_fence_after();
          issue_s(i + 1);
        }
        // dV += P^T dO (from zero at the start and after every flush)
        const bool fresh = flush_on ? (i % kFlush == 0) : (i == 0);
        if (flush_on && i > 0 && i % kFlush == 0 &&
            !(ok = mbar_wait(&bars->flushed, (i / kFlush - 1) & 1, err)))
          break;
        if (!(ok = mbar_wait(&bars->p_ready[i & 1], (i >> 1) & 1, err))) break;
        tc_fence_after();
        {
          const uint32_t pa = tmem + T_ST + (i & 1) * 64;
          const uint64_t b0 = dOm0 + stage * kStageStep;
          mma_ts(tmem + T_DV, pa, b0, id_acc, fresh ? 0u : 1u);
#pragma unroll
          for (int kk = 1; kk < 4; ++kk) mma_ts(tmem + T_DV, pa + kk * 8, b0 + kk * (2048 >> 4), id_acc, 1u);
        }
        mma_commit(&bars->dv_done);
        // dP^T(i+1) as soon as dP^T(i) has been read out of TMEM
        if (more) {
          if (!(ok = mbar_wait(&bars->dp_free, i & 1, err))) break;
          tc_fence_after();
          issue_dp(i + 1);
        }
        // dK += dS^T Q ; dQ^T = K^T dS^T  (dS^T from shared-memory buffer i % 2)
        if (!(ok = mbar_wait(&bars->ds_ready[i & 1], (i >> 1) & 1, err))) break;
        tc_fence_after();
        {
          const uint64_t a0 = dSk0 + (i & 1) * kDsStep, b0 = dQm0 + stage * kStageStep;
          mma_ss(tmem + T_DK, a0, b0, id_acc, fresh ? 0u : 1u);
#pragma unroll
          for (int kk = 1; kk < 4; ++kk) mma_ss(tmem + T_DK, a0 + kk * (32 >> 4), b0 + kk * (2048 >> 4), id_acc, 1u);
        }
        // dK(i) is the last reader of Q(i)/dO(i): release the stage to the producer.
        mma_commit(&bars->q_empty[stage]);
        if (i >= 1 && !(ok = mbar_wait(&bars->dq_free, (i - 1) & 1, err))) break;
        tc_fence_after();
        {
          const uint64_t b0 = dSm0 + (i & 1) * kDsStep;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + T_DQT, dKt + kk * (2048 >> 4), b0 + kk * (2048 >> 4), id_dq, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->dq_full);
        mma_commit(&bars->ds_free[i & 1]);
        if (flush_on && i % kFlush == kFlush - 1 && more) mma_commit(&bars->flush_ready);
      }
      mma_commit(&bars->acc_done);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ P^T and dS^T
    const int t = warp * 32 + lane;  // key row / TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
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
    const float sl2 = geo.scale_log2;
    bool ok = true;
    for (int i = 0; i < n_iter; ++i) {
      const int stage = i % NQ;
      const int64_t row0 = qbase + (int64_t)(it.b - 1 - i % nqt) * bm;
      const float* rows = reinterpret_cast<const float*>(smem + ROWS_OFF) + stage * 128;
      // rows[] (lse, Delta) of this stage are published by the producer with q_full.
      if (!(ok = mbar_wait(&bars->q_full[stage], (i / NQ) & 1, err))) break;
      if (!(ok = mbar_wait(&bars->s_full[i & 1], (i >> 1) & 1, err))) break;
      tc_fence_after();
      uint32_t sraw[2][32];
      tmem_ld32(tmem + lane_off + T_ST + (i & 1) * 64, sraw[0]);
      tmem_ld32(tmem + lane_off + T_ST + (i & 1) * 64 + 32, sraw[1]);
      tmem_ld_wait();
      const int64_t lo64 = q_lo - row0, hi64 = q_hi - row0;
      const int lo = lo64 < 0 ? 0 : (lo64 > 64 ? 64 : (int)lo64);
      const int hi = hi64 < 0 ? 0 : (hi64 > 64 ? 64 : (int)hi64);  // exclusive
      uint32_t pk[32];  // P^T as bf16 pairs: A operand of dV and the P factor of dS
      const float4* l4 = reinterpret_cast<const float4*>(rows);
      // One exponential in four runs on the FMA pipe (exp2_fma), three on the MUFU.
      if (lo == 0 && hi == 64) {
#pragma unroll
        for (int g = 0; g < 16; ++g) {
          const float4 l = l4[g];
          const int c = 4 * g;
          const float e0 = fast_exp2(fmaf(__uint_as_float(sraw[c >> 5][c & 31]), sl2, -l.x));
          const float e1 = fast_exp2(fmaf(__uint_as_float(sraw[(c + 1) >> 5][(c + 1) & 31]), sl2, -l.y));
          const float e2 = fast_exp2(fmaf(__uint_as_float(sraw[(c + 2) >> 5][(c + 2) & 31]), sl2, -l.z));
          const float e3 = exp2_fma(fmaf(__uint_as_float(sraw[(c + 3) >> 5][(c + 3) & 31]), sl2, -l.w));
          pk[2 * g] = pack_bf16x2(e0, e1);
          pk[2 * g + 1] = pack_bf16x2(e2, e3);
        }
      } else {
#pragma unroll
        for (int g = 0; g < 16; ++g) {
          const float4 l = l4[g];
          const int c = 4 * g;
          float e0 = fast_exp2(fmaf(__uint_as_float(sraw[c >> 5][c & 31]), sl2, -l.x));
          float e1 = fast_exp2(fmaf(__uint_as_float(sraw[(c + 1) >> 5][(c + 1) & 31]), sl2, -l.y));
          float e2 = fast_exp2(fmaf(__uint_as_float(sraw[(c + 2) >> 5][(c + 2) & 31]), sl2, -l.z));
          float e3 = exp2_fma(fmaf(__uint_as_float(sraw[(c + 3) >> 5][(c + 3) & 31]), sl2, -l.w));
          e0 = (c >= lo && c < hi) ? e0 : 0.f;
          e1 = (c + 1 >= lo && c + 1 < hi) ? e1 : 0.f;
          e2 = (c + 2 >= lo && c + 2 < hi) ? e2 : 0.f;
          e3 = (c + 3 >= lo && c + 3 < hi) ? e3 : 0.f;
          pk[2 * g] = pack_bf16x2(e0, e1);
          pk[2 * g + 1] = pack_bf16x2(e2, e3);
        }
      }
      tmem_st32(tmem + lane_off + T_ST + (i & 1) * 64, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->p_ready[i & 1]);
      // dS^T = P^T (dP^T - Delta), with the same bf16 P the dV product uses
      if (!(ok = mbar_wait(&bars->dp_full, i & 1, err))) break;
      tc_fence_after();
      tmem_ld32(tmem + lane_off + T_DPT, sraw[0]);
      tmem_ld32(tmem + lane_off + T_DPT + 32, sraw[1]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&bars->dp_free);
#pragma unroll
      for (int g = 0; g < 16; ++g) {
        const float4 dl = l4[16 + g];  // Delta of columns 4g .. 4g+3
        const float dd[4] = {dl.x, dl.y, dl.z, dl.w};
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int c = 2 * g + h2, c0 = 2 * c, c1 = 2 * c + 1;
          const float p0 = __uint_as_float(pk[c] << 16), p1 = __uint_as_float(pk[c] & 0xFFFF0000u);
          const float d0 = p0 * (__uint_as_float(sraw[c0 >> 5][c0 & 31]) - dd[2 * h2]);
          const float d1 = p1 * (__uint_as_float(sraw[c1 >> 5][c1 & 31]) - dd[2 * h2 + 1]);
          pk[c] = pack_bf16x2(d0, d1);
        }
      }
      // dS^T row into buffer i % 2, once dK(i-2) and dQ^T(i-2) have read that buffer
      if (i >= 2 && !(ok = mbar_wait(&bars->ds_free[i & 1], ((i >> 1) - 1) & 1, err))) break;
      uint8_t* ds_row = smem + DS_OFF + (i & 1) * KV_BLK + t * 128;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const int pos = ch ^ (t & 7);  // 128-byte swizzle: 16-byte chunk index ^ row % 8
        *reinterpret_cast<uint4*>(ds_row + pos * 16) =
            make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->ds_ready[i & 1]);
      if (flush_on && i % kFlush == kFlush - 1 && i + 1 < n_iter) {
        // Move dK/dV to this block's slot (the first flush stores, later ones add).
        if (!(ok = mbar_wait(&bars->flush_ready, (i / kFlush) & 1, err))) break;
        tc_fence_after();
        float* slot = slots + ((int64_t)smid * 128 + t) * 256;
        const bool first = i == kFlush - 1;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + (c < 4 ? T_DK : T_DV) + (c & 3) * 32, v);
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
    }
    // dV, dK rows of this key
    if (ok && mbar_wait(&bars->acc_done, 0, err) && n_iter > 0) {
      tc_fence_after();
      const int64_t off = (key * geo.hkv + kvh) * 128;
      float* fk = nullptr;
      float* fv = nullptr;
      int64_t foff = off;
      if (it.kind == K_PROMPT_KV) {
        const SplitInfo s = geo.splits[it.group];
        fk = dk_sum;
        fv = dv_sum;
        if (s.nsplit > 1) {
          fk = dk_part;
          fv = dv_part;
          foff = ((s.part_row0 + (int64_t)it.split * G.lp + (key - G.p0)) * geo.hkv + kvh) * 128;
        }
      }
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t kv[32], vv[32];
        tmem_ld32(tmem + lane_off + T_DK + c * 32, kv);
        tmem_ld32(tmem + lane_off + T_DV + c * 32, vv);
        tmem_ld_wait();
        if (!key_ok) continue;
        if (flush_on) {
          const float* slot = slots + ((int64_t)smid * 128 + t) * 256;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            kv[i] = __float_as_uint(__uint_as_float(kv[i]) + slot[c * 32 + i]);
            vv[i] = __float_as_uint(__uint_as_float(vv[i]) + slot[128 + c * 32 + i]);
          }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) kv[i] = __float_as_uint(__uint_as_float(kv[i]) * geo.scale);
        if (fk) {
          float4* pk4 = reinterpret_cast<float4*>(fk + foff + c * 32);
          float4* pv4 = reinterpret_cast<float4*>(fv + foff + c * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            pk4[i] = make_float4(__uint_as_float(kv[4 * i]), __uint_as_float(kv[4 * i + 1]),
                                 __uint_as_float(kv[4 * i + 2]), __uint_as_float(kv[4 * i + 3]));
            pv4[i] = make_float4(__uint_as_float(vv[4 * i]), __uint_as_float(vv[4 * i + 1]),
                                 __uint_as_float(vv[4 * i + 2]), __uint_as_float(vv[4 * i + 3]));
          }
        } else {
          uint4* ok4 = reinterpret_cast<uint4*>(dk_out + off + c * 32);
          uint4* ov4 = reinterpret_cast<uint4*>(dv_out + off + c * 32);
          const float4* ak = reinterpret_cast<const float4*>(dk_add + off + c * 32);
          const float4* av = reinterpret_cast<const float4*>(dv_add + off + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float a[8], b[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              a[e] = __uint_as_float(kv[8 * i + e]);
              b[e] = __uint_as_float(vv[8 * i + e]);
            }
            if (dk_add) {
              const float4 x0 = ak[2 * i], x1 = ak[2 * i + 1], y0 = av[2 * i], y1 = av[2 * i + 1];
              a[0] += x0.x; a[1] += x0.y; a[2] += x0.z; a[3] += x0.w;
              a[4] += x1.x; a[5] += x1.y; a[6] += x1.z; a[7] += x1.w;
              b[0] += y0.x; b[1] += y0.y; b[2] += y0.z; b[3] += y0.w;
              b[4] += y1.x; b[5] += y1.y; b[6] += y1.z; b[7] += y1.w;
            }
            ok4[i] = make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                                pack_bf16x2(a[6], a[7]));
            ov4[i] = make_uint4(pack_bf16x2(b[0], b[1]), pack_bf16x2(b[2], b[3]), pack_bf16x2(b[4], b[5]),
                                pack_bf16x2(b[6], b[7]));
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ dQ epilogue
    const int w4 = warp - 4;
    const int dcol = w4 * 32 + lane;  // head-dim index = TMEM lane of dQ^T
    const uint32_t lane_off = (uint32_t)(w4 * 32) << 16;
    float* tile = reinterpret_cast<float*>(smem + DQ_OFF);
    const bool leader = threadIdx.x == 128;
    for (int i = 0; i < n_iter; ++i) {
      if (!mbar_wait(&bars->dq_full, i & 1, err)) break;
      tc_fence_after();
      const int h = kvh * r + i / nqt;
      const int64_t row0 = qbase + (int64_t)(it.b - 1 - i % nqt) * bm;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + T_DQT + half * 32, v);
        tmem_ld_wait();
        if (half == 1) {
          tc_fence_before();
          mbar_arrive(&bars->dq_free);
        }
        // The staging buffer is free once the previous bulk reduce has read it.
        if (leader) bulk_wait_read0();
        named_bar(1, 128);
#pragma unroll
        for (int c = 0; c < 32; ++c) tile[c * 128 + dcol] = __uint_as_float(v[c]) * geo.scale;
        fence_proxy_async_smem();
        named_bar(1, 128);
        if (leader) {
          // Rows past the group's end hold exact zeros (their dS^T columns are zero),
          // and rows past the tensor's end are clipped by the copy.
          tma_reduce_add_3d(&tm_dq, tile, 0, h, (int)(row0 + half * 32));
          bulk_commit();
        }
      }
    }
    if (leader) bulk_wait0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t tc_bwd(const augtree_plan* p, int op, const void* q, const void* kp, const void* vp, const void* kr,
                   const void* vr, const float* stats, const void* dO, float* dq_acc,
                   void* dk_out, void* dv_out, float* dk_part, float* dv_part, float* dk_sum, float* dv_sum,
                   const float* dk_add, const float* dv_add, float* slots, cudaStream_t st) {
  const bool prefill = op == AUGTREE_OP_PREFILL_BWD;
  const int64_t q_rows = prefill ? p->total_prompt : p->total_resp;
  CUtensorMap mq, mdo, mk, mv, mk2, mv2, mdq;
  if (!encode_rows_map(&mq, q, q_rows, p->cfg.hq, 64)) return cudaErrorInvalidValue;
  if (!encode_rows_map(&mdo, dO, q_rows, p->cfg.hq, 64)) return cudaErrorInvalidValue;
  if (!encode_f32_rows_map(&mdq, dq_acc, q_rows, p->cfg.hq, 32)) return cudaErrorInvalidValue;
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
  cudaError_t e = cudaFuncSetAttribute(tc_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, BWD_SMEM);
  if (e != cudaSuccess) return e;
  tc_bwd_kernel<<<(unsigned)p->n_items[op], BWD_THREADS, BWD_SMEM, st>>>(
      mq, mdo, mk, mv, mk2, mv2, mdq, geometry(p), p->queue_d[op], p->row_bend_d, p->bm[op], p->bn[op], stats,
      prefill ? p->ntiles_p : p->ntiles_r, (__nv_bfloat16*)dk_out, (__nv_bfloat16*)dv_out, dk_part, dv_part, dk_sum, dv_sum, dk_add, dv_add,
      slots, kFlushSlots, p->err_d);
  return cudaGetLastError();
}

}  // namespace augtree
