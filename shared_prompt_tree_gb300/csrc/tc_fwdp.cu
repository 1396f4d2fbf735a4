// Tensor-core forward of tree attention on SM pairs (2-CTA clusters, tcgen05
// cta_group::2): prompt prefill and response replay.
//
// AugTree paper, "Splitting Prompt Prefill from Response Replay ...":
//   Sec. 2.2  attention as Q-KV tile interactions with an online softmax;
//   Sec. 3.2  prefill: causal self-attention of the prompt, computed once; replay,
//             Eq. 1: a response row sees all prompt keys of its group (dense) and its
//             own branch's keys up to itself;
//   Sec. 3.3  the prompt-part and own-branch-part states of a row merge associatively,
//             here as one running online softmax over the prompt tiles and then the
//             own-branch tiles.
//
// A cluster of two CTAs runs one unit: one 128-row query tile for two query heads of
// the same KV head, one head per CTA.  The even CTA issues every MMA for the pair:
//   S = Q K^T    M = 256 (128 rows from each CTA), N = 128 keys, K = 128 dims
//   O += P V     M = 256, N = 128 dims, K = 128 keys (P read from each CTA's TMEM)
// The B operand is split between the two CTAs: each loads half of every K tile (64
// keys, all dims) and half of every V tile (all keys, 64 dims).  Per SM and KV tile the
// shared-memory traffic is then 48 KB of S operands, 16 KB of V and 32 KB of copies,
// against 64 + 32 + 64 KB for one CTA running the same head alone: the single-CTA
// kernels sit at the 128 B/clock shared-memory limit of the tensor pipe's operands.
//
// Per CTA (352 threads):
//   warp 8      TMA producer: this CTA's Q tile, then a 4-stage ring of K/V halves
//   warp 9      TMEM allocator (both CTAs); on the even CTA the issuer of S
//   warp 10     even CTA: the issuer of PV; odd CTA: relays "my K/V half (and Q) landed"
//               to the even CTA's barriers
//   warps 0-7   two softmax warpgroups; warpgroup w owns keys [64w, 64w + 64) of every
//               tile for all 128 rows (thread = row = TMEM lane).  The two exchange
//               their partial row maxima every tile through shared memory, so both use
//               the same running max and write one P that a single K=128 PV product
//               consumes; each warpgroup rescales its half of O's columns.
// TMEM (each CTA, its own 128 rows): S0, S1, S2 [0,384) - three score buffers, so that
// S(j+1) waits only for PV(j-2) - and O [384,512).  P(j) (bf16 pairs) overwrites the
// first 64 columns of its score buffer once both warpgroups have read S(j).
#include <cuda.h>

#include <cmath>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_fwd_softmax.cuh"

namespace augtree {
namespace {

using namespace tc;

constexpr int FP_THREADS = 352;
constexpr int FP_NST = 4;                                  // K/V ring stages
constexpr int FP_NS = 3;                                   // score buffers in TMEM
constexpr int QBLK = 128 * 128;                            // 128 rows x 64 dims bf16 = 16 KB
constexpr int KHBLK = 64 * 128;                            // 64 keys x 64 dims bf16 = 8 KB
constexpr int FP_Q_OFF = 0;                                // [2 dim blocks] x 16 KB
constexpr int FP_K_OFF = FP_Q_OFF + 2 * QBLK;              // [stage][2 dim blocks] x 8 KB (64 keys)
constexpr int FP_V_OFF = FP_K_OFF + FP_NST * 2 * KHBLK;    // [stage] x 16 KB (128 keys x 64 dims)
constexpr int FP_X_OFF = FP_V_OFF + FP_NST * QBLK;         // [2 parities][2 warpgroups][128 rows] fp32 maxima
constexpr int FP_L_OFF = FP_X_OFF + 2 * 2 * 128 * 4;       // [2 warpgroups][128 rows] fp32 row sums
constexpr int FP_BAR_OFF = FP_L_OFF + 2 * 128 * 4;
constexpr int FP_SMEM = FP_BAR_OFF + 512 + 1024;           // + barriers + alignment slack
static_assert(FP_SMEM <= 232448, "shared memory per block");
constexpr uint32_t T_O = 384;                              // O accumulator columns

struct FpBars {
  uint64_t q_full;              // this CTA's Q landed
  uint64_t peer_q;              // even CTA: the odd CTA's Q landed (relayed)
  uint64_t kv_full[FP_NST];     // this CTA's K/V halves of a stage landed
  uint64_t peer_full[FP_NST];   // even CTA: the odd CTA's halves landed (relayed)
  uint64_t kv_empty[FP_NST];    // both: stage free (multicast MMA completion)
  uint64_t s_full[FP_NS];       // both: S(j) in score buffer j % 3 (multicast)
  uint64_t p_full[FP_NS];       // even CTA: P(j) written by the 16 softmax warps of the pair
  uint64_t pv_done[FP_NS];      // both: O += P(j) V done (multicast)
  uint64_t xmx;                 // this CTA: the 8 softmax warps published their tile maxima
  uint64_t xch;                 // this CTA: the 8 softmax warps published their final row sums
  uint64_t drain[2];            // even CTA: all MMAs of issuer 0 / 1 have completed
  uint32_t tmem_base;
};
static_assert(sizeof(FpBars) <= 512, "barrier area");

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Waits whose arrivals may come from the other CTA of the pair take cluster-scope
// acquire semantics.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t* err) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t lim = wait_limit_ns(err);
  const uint64_t t0 = globaltimer();
  while (true) {
    for (int i = 0; i < 4; ++i)
      if (mbar_try_wait_cluster(bar, parity)) return true;
    if (globaltimer() - t0 > lim) {
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
}
__device__ __forceinline__ bool mbar_wait_cluster_warp(uint64_t* bar, uint32_t parity, uint32_t* err) {
  return __all_sync(0xffffffffu, mbar_wait_cluster(bar, parity, err));
}
__device__ __forceinline__ void mma2_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma2_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Completion of this thread's issued MMAs, arriving on the barrier at the same offset in
// both CTAs of the pair.
__device__ __forceinline__ void mma2_commit_both(uint64_t* bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n}\n" ::"r"(
          smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}
// Same, arriving on this CTA's barrier only.
__device__ __forceinline__ void mma2_commit_local(uint64_t* bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(smem_u32(bar))
      : "memory");
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(FP_THREADS, 1) tc_fwdp_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kp,
    const __grid_constant__ CUtensorMap tm_vp, const __grid_constant__ CUtensorMap tm_kr,
    const __grid_constant__ CUtensorMap tm_vr, Geometry geo, const int32_t* __restrict__ queue, int bm, int bn,
    __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int64_t lse_rows, uint32_t* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FpBars* bars = reinterpret_cast<FpBars*>(smem + FP_BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();

  // The pair's unit is queue items 2u (head h) and 2u + 1 (head h + 1) of one query tile;
  // this CTA takes item 2u + rank.
  const WorkItem it = load_item(queue, blockIdx.x);
  const int h = it.head;
  const GroupInfo G = geo.groups[it.group];
  const bool prefill = it.kind == K_PREFILL_Q;
  const int64_t base = prefill ? G.p0 : G.r0;
  const int64_t len = prefill ? G.lp : G.lr;
  const int64_t row0 = base + (int64_t)it.tile * bm;
  const int64_t row_end = min(row0 + (int64_t)bm, base + len);
  const int n_a = it.a;
  const int n_tiles = n_a + (prefill ? 0 : it.b);
  const int64_t own0 = prefill ? 0 : geo.row_bstart[row0];
  const int kvh = h / (geo.hq / geo.hkv);

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->peer_q, 1);
    for (int i = 0; i < FP_NST; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->peer_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
    }
    for (int i = 0; i < FP_NS; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 16);
      mbar_init(&bars->pv_done[i], 1);
    }
    mbar_init(&bars->xmx, 8);
    mbar_init(&bars->xch, 8);
    mbar_init(&bars->drain[0], 1);
    mbar_init(&bars->drain[1], 1);
    fence_mbar_init();
  }
  if (warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&bars->tmem_base)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_kp);
    prefetch_tmap(&tm_vp);
    prefetch_tmap(&tm_kr);
    prefetch_tmap(&tm_vr);
  }
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialized before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer (both)
    if (lane == 0) {
      mbar_expect_tx(&bars->q_full, 2 * QBLK);
      for (int kb = 0; kb < 2; ++kb)
        tma_load_3d(smem + FP_Q_OFF + kb * QBLK, &tm_q, &bars->q_full, kb * 64, h, (int)row0);
      int issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int stage = j % FP_NST, use = j / FP_NST;
        if (!mbar_wait_cluster(&bars->kv_empty[stage], (use & 1) ^ 1, err)) break;
        mbar_expect_tx(&bars->kv_full[stage], 2 * KHBLK + QBLK);
        const bool own = j >= n_a;
        const int krow = own ? (int)(own0 + (int64_t)(j - n_a) * bn) : (int)(G.p0 + (int64_t)j * bn);
        const CUtensorMap* km = own ? &tm_kr : &tm_kp;
        const CUtensorMap* vm = own ? &tm_vr : &tm_vp;
        // K: this CTA's 64 keys of the tile, all dims; V: all 128 keys, this CTA's 64 dims.
        for (int kb = 0; kb < 2; ++kb)
          tma_load_3d(smem + FP_K_OFF + (stage * 2 + kb) * KHBLK, km, &bars->kv_full[stage], kb * 64, kvh,
                      krow + 64 * (int)rank);
        tma_load_3d(smem + FP_V_OFF + stage * QBLK, vm, &bars->kv_full[stage], 64 * (int)rank, kvh, krow);
        issued = j + 1;
      }
      // Never leave a copy in flight (also after giving up on a wait).
      mbar_wait_drain(&bars->q_full, 0, err);
      for (int j = max(0, issued - FP_NST); j < issued; ++j)
        mbar_wait_drain(&bars->kv_full[j % FP_NST], (j / FP_NST) & 1, err);
    }
  } else if (warp == 10 && rank == 1) {
    // ------------------------------------------------------------ relay (odd CTA)
    // The even CTA's issuer may read this CTA's operands only once they have landed.
    if (lane == 0) {
      if (mbar_wait(&bars->q_full, 0, err)) {
        mbar_arrive_cluster(peer_addr(&bars->peer_q, 0));
        for (int j = 0; j < n_tiles; ++j) {
          const int stage = j % FP_NST;
          if (!mbar_wait(&bars->kv_full[stage], (j / FP_NST) & 1, err)) break;
          mbar_arrive_cluster(peer_addr(&bars->peer_full[stage], 0));
        }
      }
    }
  } else if (warp == 9 && rank == 0) {
    // ------------------------------------------------------------ S issuer (even CTA)
    constexpr uint32_t idesc_qk = idesc_bf16_f32(256, 128, false, false);
    const uint64_t dq = smem_desc_sw128(smem_u32(smem + FP_Q_OFF), 16, 1024);
    const uint64_t dk0 = smem_desc_sw128(smem_u32(smem + FP_K_OFF), 16, 1024);
    constexpr uint64_t kKStage = (2 * KHBLK) >> 4;
    // K-major k-step kk (16 dims): dim block kk/4, 32 bytes per step in the 128-byte row.
    auto qoff = [](int kk) { return (uint64_t)(((kk >> 2) * QBLK + (kk & 3) * 32) >> 4); };
    auto koff = [](int kk) { return (uint64_t)(((kk >> 2) * KHBLK + (kk & 3) * 32) >> 4); };
    bool ok = mbar_wait_warp_all(&bars->q_full, 0, err) && mbar_wait_cluster_warp(&bars->peer_q, 0, err);
    tc_fence_after();
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int stage = j % FP_NST, b = j % FP_NS;
      if (!(ok = mbar_wait_warp_all(&bars->kv_full[stage], (j / FP_NST) & 1, err))) break;
      if (!(ok = mbar_wait_cluster_warp(&bars->peer_full[stage], (j / FP_NST) & 1, err))) break;
      // S(j) overwrites P(j-3) in its buffer: PV(j-3) must have completed.
      if (j >= FP_NS && !(ok = mbar_wait_warp_all(&bars->pv_done[b], ((j / FP_NS) - 1) & 1, err))) break;
      tc_fence_after();
      const uint64_t dk = dk0 + stage * kKStage;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) mma2_ss(tmem + b * 128, dq + qoff(kk), dk + koff(kk), idesc_qk, kk > 0 ? 1u : 0u);
      mma2_commit_both(&bars->s_full[b]);
    }
    // Never leave an MMA in flight when the pair frees TMEM (also after giving up).
    mma2_commit_local(&bars->drain[0]);
    mbar_wait_drain_warp_all(&bars->drain[0], 0, err);
  } else if (warp == 10 && rank == 0) {
    // ------------------------------------------------------------ PV issuer (even CTA)
    constexpr uint32_t idesc_pv = idesc_bf16_f32(256, 128, false, true);
    const uint64_t dv0 = smem_desc_sw128(smem_u32(smem + FP_V_OFF), QBLK, 1024);
    constexpr uint64_t kVStage = QBLK >> 4;
    bool ok = true;
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int stage = j % FP_NST, b = j % FP_NS;
      if (!(ok = mbar_wait_cluster_warp(&bars->p_full[b], (j / FP_NS) & 1, err))) break;
      tc_fence_after();
      const uint64_t dv = dv0 + stage * kVStage;
      // 16 keys per step: 16 swizzled 128-byte rows of V = 2048 bytes; P packs two keys
      // per TMEM column.
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma2_ts(tmem + T_O, tmem + b * 128 + kk * 8, dv + kk * (2048 >> 4), idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
      mma2_commit_both(&bars->pv_done[b]);
      mma2_commit_both(&bars->kv_empty[stage]);
    }
    mma2_commit_local(&bars->drain[1]);
    mbar_wait_drain_warp_all(&bars->drain[1], 0, err);
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax (both CTAs)
    // Every wait here is warp-uniform, and warps meet only on mbarriers (bounded waits),
    // never on named barriers: a warp that gives up can then never leave another one
    // waiting without limit.
    const int w = warp >> 2;        // keys [64w, 64w + 64) of every tile
    const int q4 = warp & 3;        // TMEM lane quarter
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
    const float sl2 = geo.scale_log2;
    const uint32_t p_full0 = peer_addr(&bars->p_full[0], 0);  // even CTA's barrier array
    float* sums = reinterpret_cast<float*>(smem + FP_L_OFF);
    float m = -INFINITY, l = 0.f;   // running max (shared by both warpgroups), own half's sum
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int b = j % FP_NS;
      const uint32_t tS = tmem + lane_off + b * 128;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_cluster(&bars->s_full[b], (j / FP_NS) & 1, err)))) break;
      tc_fence_after();
      uint32_t raw[2][32];
      tmem_ld32(tS + 64 * w, raw[0]);
      tmem_ld32(tS + 64 * w + 32, raw[1]);
      tmem_ld_wait();
#define FP_X(c) raw[(c) >> 5][(c) & 31]
      int lo_i, hi_i;
      fwd_valid_cols(g, j, lo_i, hi_i);
      const int lo = lo_i - 64 * w, hi = hi_i - 64 * w;  // valid local columns [lo, hi]
      const bool masked = lo > 0 || hi < 63;
      if (masked) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c < lo || c > hi) FP_X(c) = 0xFF800000u;  // -inf
      }
      float pm[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) pm[k] = __uint_as_float(FP_X(k));
#pragma unroll
      for (int c = 8; c < 64; ++c) pm[c & 7] = fmaxf(pm[c & 7], __uint_as_float(FP_X(c)));
      float tmax =
          fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])), fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
      // Exchange the two halves' maxima (double-buffered by tile parity).  Once the
      // exchange completes, both warpgroups have read S(j) into registers, so P(j) may
      // overwrite the buffer's first 64 columns.
      float* xm = reinterpret_cast<float*>(smem + FP_X_OFF) + (j & 1) * 256;
      xm[w * 128 + r_local] = tmax;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->xmx);
      if (!(ok = mbar_wait_warp_all(&bars->xmx, j & 1, err))) break;
      tmax = fmaxf(tmax, xm[(w ^ 1) * 128 + r_local]);
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
        const float p0 = fast_exp2(fmaf(__uint_as_float(FP_X(2 * i)), sl2, -mu));
        const float p1 = fast_exp2(fmaf(__uint_as_float(FP_X(2 * i + 1)), sl2, -mu));
        pk[i] = pack_bf16x2(p0, p1);
        // The row sum uses the bf16 weights the PV product uses.
        ps[i & 3] += __uint_as_float(pk[i] << 16) + __uint_as_float(pk[i] & 0xFFFF0000u);
      }
#undef FP_X
      // P(j): keys [64w, 64w + 64) as bf16 pairs in columns [32w, 32w + 32).
      tmem_st32(tS + 32 * w, pk);
      l = l * alpha + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
      if (__any_sync(0xffffffffu, need)) {
        // O += P(j-1) V must be complete before O is rescaled; PV(j) is issued only
        // after every softmax warp of the pair signals P(j).  Warpgroup w rescales O's
        // dims [64w, 64w + 64).
        const int jp = j - 1;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait_cluster(&bars->pv_done[jp % FP_NS], (jp / FP_NS) & 1, err))))
          break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + T_O + 64 * w + 32 * c, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tmem + lane_off + T_O + 64 * w + 32 * c, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(p_full0 + b * 8);  // this warp's P(j) (and O rows) are in TMEM
    }
    // Both halves' row sums; then O / l and lse.  Warpgroup w writes dims [64w, 64w + 64).
    const int last = n_tiles - 1;
    if (ok && n_tiles > 0)
      ok = __all_sync(0xffffffffu, mbar_wait_cluster(&bars->pv_done[last % FP_NS], (last / FP_NS) & 1, err));
    tc_fence_after();
    sums[w * 128 + r_local] = l;
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->xch);  // also after a failed wait, so the others' wait ends
    if (ok) ok = mbar_wait_warp_all(&bars->xch, 0, err);
    if (ok) {
      const float L = sums[r_local] + sums[128 + r_local];
      const bool any = L > 0.f && n_tiles > 0;  // a row with no key writes zeros
      const float inv = any ? 1.f / L : 0.f;
      __nv_bfloat16* orow = out + (g.row * geo.hq + h) * 128 + 64 * w;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + T_O + 64 * w + 32 * c, o);
        tmem_ld_wait();
        if (g.row_ok) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = any ? pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv) : 0u;
          uint4* d4 = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
          for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      if (w == 0 && g.row_ok) lse[(int64_t)h * lse_rows + g.row] = any ? (m + log2f(L)) * 0.69314718055994531f : -INFINITY;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the pair's MMAs, copies and TMEM reads are done before TMEM is released
  if (warp == 9) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
  }
}

}  // namespace

cudaError_t tc_fwdp(const augtree_plan* p, int op, const void* q, const void* kp, const void* vp, const void* kr,
                    const void* vr, void* o, float* lse, cudaStream_t st) {
  const bool prefill = op == AUGTREE_OP_PREFILL_FWD;
  const int64_t q_rows = prefill ? p->total_prompt : p->total_resp;
  CUtensorMap mq, mkp, mvp, mkr, mvr;
  if (!encode_rows_map(&mq, q, q_rows, p->cfg.hq, 128)) return cudaErrorInvalidValue;
  const bool have_p = p->total_prompt > 0 && kp && vp;
  const bool have_r = !prefill && p->total_resp > 0 && kr && vr;
  // K halves: boxes of 64 keys; V halves: boxes of 128 keys x 64 dims.
  if (have_p) {
    if (!encode_rows_map(&mkp, kp, p->total_prompt, p->cfg.hkv, 64)) return cudaErrorInvalidValue;
    if (!encode_rows_map(&mvp, vp, p->total_prompt, p->cfg.hkv, 128)) return cudaErrorInvalidValue;
  }
  if (have_r) {
    if (!encode_rows_map(&mkr, kr, p->total_resp, p->cfg.hkv, 64)) return cudaErrorInvalidValue;
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
  cudaError_t e = cudaFuncSetAttribute(tc_fwdp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, FP_SMEM);
  if (e != cudaSuccess) return e;
  tc_fwdp_kernel<<<(unsigned)p->n_items[op], FP_THREADS, FP_SMEM, st>>>(mq, mkp, mvp, mkr, mvr, geometry(p),
                                                                        p->queue_d[op], p->bm[op], p->bn[op],
                                                                        (__nv_bfloat16*)o, lse, q_rows, p->err_d);
  return cudaGetLastError();
}

}  // namespace augtree
