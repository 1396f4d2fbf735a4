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
// One thread block per work item: 128 keys of one KV head, query tiles [a, b) of 128
// rows for each of the r query heads of that KV head.  Per query tile (keys are the
// MMA M dimension, one key per TMEM lane):
//   S^T  = K Q^T     (TMEM, fp32)  -> P^T  = exp2(s S^T log2e - lse), bf16 over S^T
//   dP^T = V dO^T    (TMEM, fp32)  -> dS^T = P^T (dP^T - Delta),     bf16 over dP^T
//   dV  += P^T dO    (A = P^T from TMEM, B = dO read MN-major)
//   dK  += dS^T Q    (A = dS^T from TMEM, B = Q read MN-major)
// dQ is computed by the query-side kernel, so nothing here leaves the SM per query
// tile.  Every operand read from shared memory is a 128-wide tile (N = 128).
// Warps: 0-7 two warpgroups, warpgroup w takes query columns [64w, 64w + 64) of every
//        tile (thread = key = TMEM lane); 8 TMA producer; 9 TMEM allocator + MMA issuer.
// TMEM columns: S^T/P^T [0,128), dP^T/dS^T [128,256), dV [256,384), dK [384,512).
// MMA issue order S(i), dP(i), dV(i), dK(i), S(i+1), dP(i+1), ...: S(i+1) reuses the
// columns dV(i) reads and dP(i+1) those dK(i) reads, and each waits for that reader's
// completion with the next group already queued behind it.
#include <cuda.h>

#include <cmath>

#include "common.cuh"
#include "tc_common.cuh"

namespace augtree {
namespace {

using namespace tc;

constexpr int KV_THREADS = 320;
constexpr int NQ = 2;                                   // Q/dO ring stages
constexpr int kPrefetch = 4;                            // L2 prefetch distance (iterations)
constexpr int BLK = 128 * 128;                          // 128 rows x 64 dims bf16 = 16 KB
constexpr int K_OFF = 0;                                // 2 blocks
constexpr int V_OFF = K_OFF + 2 * BLK;                  // 2 blocks
constexpr int Q_OFF = V_OFF + 2 * BLK;                  // [NQ][2 blocks]
constexpr int DO_OFF = Q_OFF + NQ * 2 * BLK;            // [NQ][2 blocks]
constexpr int ROWS_OFF = DO_OFF + NQ * 2 * BLK;         // [NQ] x {lse2[128], delta[128]}
constexpr int BAR_OFF = ROWS_OFF + NQ * 2 * 128 * 4;
constexpr int KV_SMEM = BAR_OFF + 256 + 1024;

constexpr uint32_t T_ST = 0, T_DPT = 128, T_DV = 256, T_DK = 384;

// The tensor cores' fp32 accumulation into TMEM carries a small rounding bias per
// accumulation (measured at about 1e-8 relative), which adds up over the tens of
// thousands of accumulations of a long item.  Every kFlush query tiles the dK/dV
// accumulators are therefore moved into an fp32 slot (round-to-nearest adds) and the
// tensor-core accumulation restarts from zero.
constexpr int kFlush = 256;

struct KvBars {
  uint64_t kv_full;
  uint64_t q_full[NQ];
  uint64_t q_empty[NQ];
  uint64_t s_full;
  uint64_t dp_full;
  uint64_t p_ready;
  uint64_t ds_ready;
  uint64_t dv_done;
  uint64_t dk_done;
  uint64_t acc_done;
  uint64_t flush_ready;  // dK/dV accumulators complete up to a flush point
  uint64_t flushed;      // compute warps have moved them to the slot
  uint32_t tmem_base;
};

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

__global__ void __launch_bounds__(KV_THREADS, 1) tc_bwd_kv_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const __grid_constant__ CUtensorMap tm_k2, const __grid_constant__ CUtensorMap tm_v2, Geometry geo,
    const int32_t* __restrict__ queue, const int32_t* __restrict__ row_bend, int bm, int bn,
    const float* __restrict__ stats, int ntiles, __nv_bfloat16* __restrict__ dk_out,
    __nv_bfloat16* __restrict__ dv_out, float* __restrict__ dk_part, float* __restrict__ dv_part,
    float* __restrict__ dk_sum, float* __restrict__ dv_sum, const float* __restrict__ dk_add,
    const float* __restrict__ dv_add, float* __restrict__ slots, int n_slots, uint32_t* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  KvBars* bars = reinterpret_cast<KvBars*>(smem + BAR_OFF);
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
  // then hit the same L2 lines.

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int i = 0; i < NQ; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_ready, 256);
    mbar_init(&bars->ds_ready, 256);
    mbar_init(&bars->dv_done, 1);
    mbar_init(&bars->dk_done, 1);
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->flush_ready, 1);
    mbar_init(&bars->flushed, 256);
    fence_mbar_init();
  }
  if (warp == 9) tmem_alloc(&bars->tmem_base, 512);
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_do);
    prefetch_tmap(resp_keys ? &tm_k2 : &tm_k);
    prefetch_tmap(resp_keys ? &tm_v2 : &tm_v);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 8) {
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
      int issued = 0;
      for (int i = 0; i < n_iter; ++i) {
        const int stage = i % NQ, use = i / NQ;
        if (!mbar_wait(&bars->q_empty[stage], (use & 1) ^ 1, err)) break;
        const int h = kvh * r + i / nqt;
        const int qt = it.b - 1 - i % nqt;
        const int64_t row0 = qbase + (int64_t)qt * bm;
        mbar_expect_tx(&bars->q_full[stage], 4 * BLK + 2 * kStatRows * 4);
        for (int kb = 0; kb < 2; ++kb) {
          tma_load_3d(smem + Q_OFF + (stage * 2 + kb) * BLK, &tm_q, &bars->q_full[stage], kb * 64, h, (int)row0);
          tma_load_3d(smem + DO_OFF + (stage * 2 + kb) * BLK, &tm_do, &bars->q_full[stage], kb * 64, h, (int)row0);
        }
        // {lse * log2(e), Delta} of the tile's 128 rows: one 1 KB bulk copy.
        bulk_load(smem + ROWS_OFF + stage * 2 * kStatRows * 4,
                  stats + ((int64_t)h * ntiles + tile_base + qt) * 2 * kStatRows, 2 * kStatRows * 4,
                  &bars->q_full[stage]);
        issued = i + 1;
        // Warm L2 with the tiles a few iterations ahead.
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
      // Never leave a copy in flight.
      mbar_wait(&bars->kv_full, 0, err);
      for (int i = max(0, issued - NQ); i < issued; ++i) mbar_wait(&bars->q_full[i % NQ], (i / NQ) & 1, err);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_ss = idesc_bf16_f32(128, 128, false, false);  // K Q^T, V dO^T
      constexpr uint32_t id_ts = idesc_bf16_f32(128, 128, false, true);   // P^T dO, dS^T Q (B MN-major)
      const uint64_t dK = smem_desc_sw128(smem_u32(smem + K_OFF), 16, 1024);
      const uint64_t dV = smem_desc_sw128(smem_u32(smem + V_OFF), 16, 1024);
      const uint64_t dQk0 = smem_desc_sw128(smem_u32(smem + Q_OFF), 16, 1024);
      const uint64_t dOk0 = smem_desc_sw128(smem_u32(smem + DO_OFF), 16, 1024);
      const uint64_t dQm0 = smem_desc_sw128(smem_u32(smem + Q_OFF), BLK, 1024);
      const uint64_t dOm0 = smem_desc_sw128(smem_u32(smem + DO_OFF), BLK, 1024);
      constexpr uint64_t kStage = (2 * BLK) >> 4;
      auto koff = [](int kk) { return (uint64_t)(((kk >> 2) * BLK + (kk & 3) * 32) >> 4); };
      // TMEM column of the bf16 A operand for query step kk (16 rows): warpgroup w packed
      // rows [64w, 64w + 64) into columns [64w, 64w + 32) of its region.
      auto acol = [](int kk) { return (uint32_t)((kk >> 2) * 64 + (kk & 3) * 8); };
      auto issue_s = [&](int i) {
        const uint64_t b = dQk0 + (i % NQ) * kStage;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(tmem + T_ST, dK + koff(kk), b + koff(kk), id_ss, kk > 0 ? 1u : 0u);
        mma_commit(&bars->s_full);
      };
      auto issue_dp = [&](int i) {
        const uint64_t b = dOk0 + (i % NQ) * kStage;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(tmem + T_DPT, dV + koff(kk), b + koff(kk), id_ss, kk > 0 ? 1u : 0u);
        mma_commit(&bars->dp_full);
      };
      bool ok = mbar_wait(&bars->kv_full, 0, err);
      if (ok && n_iter > 0) ok = mbar_wait(&bars->q_full[0], 0, err);
      tc_fence_after();
      if (ok && n_iter > 0) {
        issue_s(0);
        issue_dp(0);
      }
      for (int i = 0; ok && i < n_iter; ++i) {
        const int stage = i % NQ;
        const bool more = i + 1 < n_iter;
        const bool fresh = flush_on ? (i % kFlush == 0) : (i == 0);
        // dV += P^T dO (from zero at the start and after every flush)
        if (flush_on && i > 0 && i % kFlush == 0 && !(ok = mbar_wait(&bars->flushed, (i / kFlush - 1) & 1, err)))
          break;
        if (!(ok = mbar_wait(&bars->p_ready, i & 1, err))) break;
        tc_fence_after();
        {
          const uint64_t b0 = dOm0 + stage * kStage;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + T_DV, tmem + T_ST + acol(kk), b0 + kk * (2048 >> 4), id_ts, (fresh && kk == 0) ? 0u : 1u);
        }
        mma_commit(&bars->dv_done);
        // dK += dS^T Q
        if (!(ok = mbar_wait(&bars->ds_ready, i & 1, err))) break;
        tc_fence_after();
        {
          const uint64_t b0 = dQm0 + stage * kStage;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + T_DK, tmem + T_DPT + acol(kk), b0 + kk * (2048 >> 4), id_ts, (fresh && kk == 0) ? 0u : 1u);
        }
        mma_commit(&bars->dk_done);
        // dK(i) is the last reader of Q(i)/dO(i) and of the stage's row statistics.
        mma_commit(&bars->q_empty[stage]);
        if (flush_on && i % kFlush == kFlush - 1 && more) mma_commit(&bars->flush_ready);
        if (more) {
          // S(i+1) overwrites P^T(i): dV(i) must have read it (dK(i) is queued behind it).
          if (!(ok = mbar_wait(&bars->q_full[(i + 1) % NQ], ((i + 1) / NQ) & 1, err))) break;
          if (!(ok = mbar_wait(&bars->dv_done, i & 1, err))) break;
          tc_fence_after();
          issue_s(i + 1);
          // dP(i+1) overwrites dS^T(i): dK(i) must have read it (S(i+1) is queued).
          if (!(ok = mbar_wait(&bars->dk_done, i & 1, err))) break;
          tc_fence_after();
          issue_dp(i + 1);
        }
      }
      mma_commit(&bars->acc_done);
    }
  } else {
    // ------------------------------------------------------------ P^T and dS^T
    const int w = warp >> 2;                 // query columns [64w, 64w + 64)
    const int q4 = warp & 3;                 // TMEM lane quarter
    const int t = q4 * 32 + lane;            // key row / TMEM lane
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const int c0 = 64 * w;
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
      const float* rows = reinterpret_cast<const float*>(smem + ROWS_OFF) + stage * 2 * kStatRows;
      // rows[] (lse, Delta) of this stage are published by the producer with q_full.
      if (!(ok = mbar_wait(&bars->q_full[stage], (i / NQ) & 1, err))) break;
      if (!(ok = mbar_wait(&bars->s_full, i & 1, err))) break;
      tc_fence_after();
      uint32_t sraw[2][32];
      tmem_ld32(tmem + lane_off + T_ST + c0, sraw[0]);
      tmem_ld32(tmem + lane_off + T_ST + c0 + 32, sraw[1]);
      tmem_ld_wait();
      // this warpgroup's valid columns: [lo, hi) relative to c0
      const int64_t lo64 = q_lo - row0 - c0, hi64 = q_hi - row0 - c0;
      const int lo = lo64 < 0 ? 0 : (lo64 > 64 ? 64 : (int)lo64);
      const int hi = hi64 < 0 ? 0 : (hi64 > 64 ? 64 : (int)hi64);
      uint32_t pk[32];  // P^T as bf16 pairs: A operand of dV and the P factor of dS
      const float4* l4 = reinterpret_cast<const float4*>(rows + c0);
      if (lo == 0 && hi == 64) {
#pragma unroll
        for (int g = 0; g < 16; ++g) {
          const float4 l = l4[g];
          const int c = 4 * g;
          const float e0 = fast_exp2(fmaf(__uint_as_float(sraw[c >> 5][c & 31]), sl2, -l.x));
          const float e1 = fast_exp2(fmaf(__uint_as_float(sraw[(c + 1) >> 5][(c + 1) & 31]), sl2, -l.y));
          const float e2 = fast_exp2(fmaf(__uint_as_float(sraw[(c + 2) >> 5][(c + 2) & 31]), sl2, -l.z));
          const float e3 = fast_exp2(fmaf(__uint_as_float(sraw[(c + 3) >> 5][(c + 3) & 31]), sl2, -l.w));
          pk[2 * g] = pack_bf16x2(e0, e1);
          pk[2 * g + 1] = pack_bf16x2(e2, e3);
        }
      } else {
        const uint32_t span = (uint32_t)(hi - lo);  // valid iff (c - lo) < span (unsigned)
#pragma unroll
        for (int g = 0; g < 16; ++g) {
          const float4 l = l4[g];
          const int c = 4 * g;
          float e0 = fast_exp2(fmaf(__uint_as_float(sraw[c >> 5][c & 31]), sl2, -l.x));
          float e1 = fast_exp2(fmaf(__uint_as_float(sraw[(c + 1) >> 5][(c + 1) & 31]), sl2, -l.y));
          float e2 = fast_exp2(fmaf(__uint_as_float(sraw[(c + 2) >> 5][(c + 2) & 31]), sl2, -l.z));
          float e3 = fast_exp2(fmaf(__uint_as_float(sraw[(c + 3) >> 5][(c + 3) & 31]), sl2, -l.w));
          e0 = (uint32_t)(c - lo) < span ? e0 : 0.f;
          e1 = (uint32_t)(c + 1 - lo) < span ? e1 : 0.f;
          e2 = (uint32_t)(c + 2 - lo) < span ? e2 : 0.f;
          e3 = (uint32_t)(c + 3 - lo) < span ? e3 : 0.f;
          pk[2 * g] = pack_bf16x2(e0, e1);
          pk[2 * g + 1] = pack_bf16x2(e2, e3);
        }
      }
      tmem_st32(tmem + lane_off + T_ST + c0, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->p_ready);
      // dS^T = P^T (dP^T - Delta), with the same bf16 P the dV product uses
      if (!(ok = mbar_wait(&bars->dp_full, i & 1, err))) break;
      tc_fence_after();
      tmem_ld32(tmem + lane_off + T_DPT + c0, sraw[0]);
      tmem_ld32(tmem + lane_off + T_DPT + c0 + 32, sraw[1]);
      tmem_ld_wait();
      const float4* d4 = reinterpret_cast<const float4*>(rows + kStatRows + c0);
#pragma unroll
      for (int g = 0; g < 16; ++g) {
        const float4 dl = d4[g];  // Delta of columns 4g .. 4g+3
        const float dd[4] = {dl.x, dl.y, dl.z, dl.w};
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int c = 2 * g + h2, e0 = 2 * c, e1 = 2 * c + 1;
          const float p0 = __uint_as_float(pk[c] << 16), p1 = __uint_as_float(pk[c] & 0xFFFF0000u);
          const float d0 = p0 * (__uint_as_float(sraw[e0 >> 5][e0 & 31]) - dd[2 * h2]);
          const float d1 = p1 * (__uint_as_float(sraw[e1 >> 5][e1 & 31]) - dd[2 * h2 + 1]);
          pk[c] = pack_bf16x2(d0, d1);
        }
      }
      tmem_st32(tmem + lane_off + T_DPT + c0, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->ds_ready);
      if (flush_on && i % kFlush == kFlush - 1 && i + 1 < n_iter) {
        // Move dK (warpgroup 0) or dV (warpgroup 1) to this block's slot (the first
        // flush stores, later ones add).
        if (!(ok = mbar_wait(&bars->flush_ready, (i / kFlush) & 1, err))) break;
        tc_fence_after();
        float* slot = slots + ((int64_t)smid * 128 + t) * 256 + w * 128;
        const bool first = i == kFlush - 1;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + (w == 0 ? T_DK : T_DV) + c * 32, v);
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
    // dK (warpgroup 0) or dV (warpgroup 1) row of this key
    if (ok && mbar_wait(&bars->acc_done, 0, err) && n_iter > 0) {
      tc_fence_after();
      const int64_t off = (key * geo.hkv + kvh) * 128;
      float* fdst = nullptr;
      int64_t foff = off;
      if (it.kind == K_PROMPT_KV) {
        const SplitInfo s = geo.splits[it.group];
        fdst = w == 0 ? dk_sum : dv_sum;
        if (s.nsplit > 1) {
          fdst = w == 0 ? dk_part : dv_part;
          foff = ((s.part_row0 + (int64_t)it.split * G.lp + (key - G.p0)) * geo.hkv + kvh) * 128;
        }
      }
      const float mul = w == 0 ? geo.scale : 1.f;
      const float* slot = slots + ((int64_t)smid * 128 + t) * 256 + w * 128;
      __nv_bfloat16* bdst = w == 0 ? dk_out : dv_out;
      const float* add = w == 0 ? dk_add : dv_add;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + (w == 0 ? T_DK : T_DV) + c * 32, v);
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
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t tc_bwd_kv(const augtree_plan* p, int op, const void* q, const void* kp, const void* vp, const void* kr,
                      const void* vr, const float* stats, const void* dO, void* dk_out, void* dv_out, float* dk_part,
                      float* dv_part, float* dk_sum, float* dv_sum, const float* dk_add, const float* dv_add,
                      float* slots, cudaStream_t st) {
  const bool prefill = op == AUGTREE_OP_PREFILL_BWD;
  if (p->n_items[op] == 0) return cudaSuccess;
  const int64_t q_rows = prefill ? p->total_prompt : p->total_resp;
  CUtensorMap mq, mdo, mk, mv, mk2, mv2;
  if (!encode_rows_map(&mq, q, q_rows, p->cfg.hq, 128)) return cudaErrorInvalidValue;
  if (!encode_rows_map(&mdo, dO, q_rows, p->cfg.hq, 128)) return cudaErrorInvalidValue;
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
  cudaError_t e = cudaFuncSetAttribute(tc_bwd_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, KV_SMEM);
  if (e != cudaSuccess) return e;
  tc_bwd_kv_kernel<<<(unsigned)p->n_items[op], KV_THREADS, KV_SMEM, st>>>(
      mq, mdo, mk, mv, mk2, mv2, geometry(p), p->queue_d[op], p->row_bend_d, p->bm[op], p->bn[op], stats,
      prefill ? p->ntiles_p : p->ntiles_r, (__nv_bfloat16*)dk_out, (__nv_bfloat16*)dv_out, dk_part, dv_part, dk_sum,
      dv_sum, dk_add, dv_add, slots, kFlushSlots, p->err_d);
  return cudaGetLastError();
}

}  // namespace augtree
