// Tensor-core forward of tree attention on an SM pair (2-CTA cluster, tcgen05
// cta_group::2): prompt prefill and response replay.
//
// AugTree paper, "Splitting Prompt Prefill from Response Replay ...":
//   Sec. 2.2  attention as Q-KV tile interactions with an online softmax;
//   Sec. 3.2  prefill: causal self-attention of the prompt; replay, Eq. 1: a response
//             row sees all prompt keys of its group and its own branch up to itself;
//   Sec. 3.3  prompt-part and own-part states merge in one running online softmax.
//
// A cluster of two CTAs runs one unit: one 128-row query tile for four query heads of
// one KV head (GQA), two heads per CTA.  The even CTA issues every MMA for the pair:
//   S_s  = Q_s K^T   M = 256 (128 rows from each CTA), N = 128 keys, K = 128 dims
//   O_s += P_s V     M = 256, N = 128 dims, K = 128 keys (P read from each CTA's TMEM)
// One M=256 instruction runs at the full tensor rate where a single-CTA M=128 one of
// the same N cannot.  The B operand is split between the CTAs: each loads half of every
// K tile (64 keys, all dims) and half of every V tile (all keys, 64 dims), so each SM
// moves half the K/V bytes of the single-CTA kernel.
// Per CTA: warp 8 TMA producer, warp 9 TMEM allocator (+ MMA issuer on the even CTA),
// warps 0-7 two softmax warpgroups (one per head, thread = query row).
// Hand-offs across the pair: both producers' copies signal the even CTA's barriers
// (cta_group::2 copies); MMA completions are multicast to both CTAs; each softmax
// warpgroup gathers on a named barrier and one thread arrives on the even CTA's
// barrier.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_fwd_softmax.cuh"

namespace augtree {
namespace {

using namespace tc;

constexpr int F2_THREADS = 320;
constexpr int F2_NST = 4;                                 // K/V ring stages
constexpr int QBLK = 128 * 128;                           // 128 rows x 64 dims bf16 = 16 KB
constexpr int KHBLK = 64 * 128;                           // 64 keys x 64 dims = 8 KB
constexpr int F2_Q_OFF = 0;                               // [2 heads][2 dim blocks] x 16 KB
constexpr int F2_K_OFF = F2_Q_OFF + 4 * QBLK;             // [stage][2 dim blocks] x 8 KB (64 keys)
constexpr int F2_V_OFF = F2_K_OFF + F2_NST * 2 * KHBLK;   // [stage] x 16 KB (128 keys x 64 dims)
constexpr int F2_BAR_OFF = F2_V_OFF + F2_NST * QBLK;
constexpr int F2_SMEM = F2_BAR_OFF + 256 + 1024;

struct F2Bars {
  uint64_t q_full;              // even CTA: both CTAs' Q tiles landed
  uint64_t kv_full[F2_NST];     // even CTA: both CTAs' K/V halves of a stage landed
  uint64_t kv_empty[F2_NST];    // both: stage free (multicast MMA completion)
  uint64_t s_full[2];           // both: S_s in TMEM
  uint64_t p_full[2];           // even CTA: P_s written in both CTAs
  uint64_t o_done[2];           // both: O_s += P_s V done
  uint32_t tmem_base;
};

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
__device__ __forceinline__ void mbar_expect_tx_cluster(uint32_t cluster_addr, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(cluster_addr),
               "r"(bytes)
               : "memory");
}
// Bounded wait with cluster-scope acquire (arrivals come from the peer CTA).
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
  const uint64_t t0 = globaltimer();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait_cluster(bar, parity)) return true;
    if (globaltimer() - t0 > kWaitLimitNs) {
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
}
__device__ __forceinline__ bool mbar_wait_cluster_warp(uint64_t* bar, uint32_t parity, uint32_t* err) {
  return __all_sync(0xffffffffu, mbar_wait_cluster(bar, parity, err));
}
// TMA tile load into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (the even CTA's, here).
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster, int c0,
                                                 int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%3, "
      "%4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
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
// Completion of this CTA's issued MMAs, arriving on the barrier at the same offset in
// both CTAs of the pair.
__device__ __forceinline__ void mma2_commit_both(uint64_t* bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n}\n" ::"r"(
          smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(F2_THREADS, 1) tc_fwd2_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kp,
    const __grid_constant__ CUtensorMap tm_vp, const __grid_constant__ CUtensorMap tm_kr,
    const __grid_constant__ CUtensorMap tm_vr, Geometry geo, const int32_t* __restrict__ queue, int bm, int bn,
    __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int64_t lse_rows, uint32_t* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  F2Bars* bars = reinterpret_cast<F2Bars*>(smem + F2_BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();

  // Unit = 4 consecutive queue items: heads 4u'..4u'+3 of one query tile; this CTA
  // takes heads 2*rank and 2*rank+1 of them.
  const int64_t unit = blockIdx.x >> 1;
  const WorkItem it0 = load_item(queue, unit * 4);
  int heads[2];
  heads[0] = it0.head + 2 * (int)rank;
  heads[1] = heads[0] + 1;
  const GroupInfo G = geo.groups[it0.group];
  const bool prefill = it0.kind == K_PREFILL_Q;
  const int64_t base = prefill ? G.p0 : G.r0;
  const int64_t len = prefill ? G.lp : G.lr;
  const int64_t row0 = base + (int64_t)it0.tile * bm;
  const int64_t row_end = min(row0 + (int64_t)bm, base + len);
  const int n_a = it0.a;
  const int n_tiles = n_a + (prefill ? 0 : it0.b);
  const int64_t own0 = prefill ? 0 : geo.row_bstart[row0];
  const int kvh = heads[0] / (geo.hq / geo.hkv);

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 2);
    for (int i = 0; i < F2_NST; ++i) {
      mbar_init(&bars->kv_full[i], 2);
      mbar_init(&bars->kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 2);
      mbar_init(&bars->o_done[i], 1);
    }
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
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint32_t q_full0 = peer_addr(&bars->q_full, 0);
      mbar_expect_tx_cluster(q_full0, 4 * QBLK);
      for (int s = 0; s < 2; ++s)
        for (int kb = 0; kb < 2; ++kb)
          tma_load_3d_pair(smem + F2_Q_OFF + (s * 2 + kb) * QBLK, &tm_q, q_full0, kb * 64, heads[s], (int)row0);
      int issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int stage = j % F2_NST, use = j / F2_NST;
        if (!mbar_wait(&bars->kv_empty[stage], (use & 1) ^ 1, err)) break;
        const uint32_t full0 = peer_addr(&bars->kv_full[stage], 0);
        mbar_expect_tx_cluster(full0, 2 * KHBLK + QBLK);
        const bool own = j >= n_a;
        const int krow = own ? (int)(own0 + (int64_t)(j - n_a) * bn) : (int)(G.p0 + (int64_t)j * bn);
        const CUtensorMap* km = own ? &tm_kr : &tm_kp;
        const CUtensorMap* vm = own ? &tm_vr : &tm_vp;
        // K: this CTA's 64 keys of the tile, all dims; V: all 128 keys, this CTA's 64 dims.
        for (int kb = 0; kb < 2; ++kb)
          tma_load_3d_pair(smem + F2_K_OFF + (stage * 2 + kb) * KHBLK, km, full0, kb * 64, kvh, krow + 64 * (int)rank);
        tma_load_3d_pair(smem + F2_V_OFF + stage * QBLK, vm, full0, 64 * (int)rank, kvh, krow);
        issued = j + 1;
      }
      if (rank == 0) {
        // Never leave a copy in flight: the even CTA's barriers count both CTAs' bytes.
        mbar_wait_cluster(&bars->q_full, 0, err);
        for (int j = max(0, issued - F2_NST); j < issued; ++j)
          mbar_wait_cluster(&bars->kv_full[j % F2_NST], (j / F2_NST) & 1, err);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (rank == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(256, 128, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(256, 128, false, true);
      const uint64_t dq0 = smem_desc_sw128(smem_u32(smem + F2_Q_OFF), 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(smem_u32(smem + F2_K_OFF), 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(smem_u32(smem + F2_V_OFF), QBLK, 1024);
      constexpr uint64_t kQSub = (2 * QBLK) >> 4, kKStage = (2 * KHBLK) >> 4, kVStage = QBLK >> 4;
      // K-major k-step kk (16 dims): dim block kk/4, 32 bytes per step in the 128-byte row.
      auto qoff = [](int kk) { return (uint64_t)(((kk >> 2) * QBLK + (kk & 3) * 32) >> 4); };
      auto koff = [](int kk) { return (uint64_t)(((kk >> 2) * KHBLK + (kk & 3) * 32) >> 4); };
      bool ok = mbar_wait_cluster_warp(&bars->q_full, 0, err);
      tc_fence_after();
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int stage = j % F2_NST, use = j / F2_NST;
        if (!(ok = mbar_wait_cluster_warp(&bars->kv_full[stage], use & 1, err))) break;
        tc_fence_after();
        const uint64_t dk = dk0 + stage * kKStage, dv = dv0 + stage * kVStage;
        for (int s = 0; s < 2; ++s) {
          if (j > 0) {
            // S_s(j) overwrites P_s(j-1): O_s += P_s(j-1) V must have completed.
            if (!(ok = mbar_wait_warp_all(&bars->o_done[s], (j - 1) & 1, err))) break;
            tc_fence_after();
          }
          const uint64_t dq = dq0 + s * kQSub;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma2_ss(tmem + s * 128, dq + qoff(kk), dk + koff(kk), idesc_qk, kk > 0 ? 1u : 0u);
          mma2_commit_both(&bars->s_full[s]);
        }
        if (!ok) break;
        for (int s = 0; s < 2; ++s) {
          if (!(ok = mbar_wait_cluster_warp(&bars->p_full[s], j & 1, err))) break;
          tc_fence_after();
          // 16 keys per step: 16 swizzled 128-byte rows = 2048 bytes.
          const uint32_t pa = tmem + s * 128;
          mma2_ts(tmem + 256 + s * 128, pa, dv, idesc_pv, j > 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 1; kk < 8; ++kk)
            mma2_ts(tmem + 256 + s * 128, pa + kk * 8, dv + kk * (2048 >> 4), idesc_pv, 1u);
          mma2_commit_both(&bars->o_done[s]);
        }
        mma2_commit_both(&bars->kv_empty[stage]);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax (both CTAs)
    const int s = warp >> 2;
    const int q4 = warp & 3;
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
    const int h = heads[s];
    const uint32_t p_full0 = peer_addr(&bars->p_full[s], 0);
    const bool leader_thread = r_local == 0;
    auto signal = [=]() {
      named_bar_sync(1 + s, 128);  // the whole warpgroup has written P_s
      if (leader_thread) mbar_arrive_cluster(p_full0);
    };
    fwd_softmax_row(tmem + s * 128 + lane_off, tmem + 256 + s * 128 + lane_off, g, n_tiles, geo.scale_log2,
                    &bars->s_full[s], &bars->o_done[s], signal, out + (g.row * geo.hq + h) * 128,
                    lse + (int64_t)h * lse_rows + g.row, err);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the pair's MMAs and TMEM reads are done before TMEM is released
  if (warp == 9) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
  }
}

}  // namespace

bool tc_fwd2_supported(const augtree_plan* p, int op) { return p->quad[op] != 0; }

cudaError_t tc_fwd2(const augtree_plan* p, int op, const CUtensorMap& mq, const void* kp, const void* vp,
                    const void* kr, const void* vr, void* o, float* lse, int64_t q_rows, cudaStream_t st) {
  const bool prefill = op == AUGTREE_OP_PREFILL_FWD;
  CUtensorMap mkp, mvp, mkr, mvr;
  const bool have_p = p->total_prompt > 0 && kp && vp;
  const bool have_r = !prefill && p->total_resp > 0 && kr && vr;
  if (have_p) {
    if (!encode_rows_map(&mkp, kp, p->total_prompt, p->cfg.hkv, 64)) return cudaErrorInvalidValue;
    if (!encode_rows_map(&mvp, vp, p->total_prompt, p->cfg.hkv, 128)) return cudaErrorInvalidValue;
  }
  if (have_r) {
    if (!encode_rows_map(&mkr, kr, p->total_resp, p->cfg.hkv, 64)) return cudaErrorInvalidValue;
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
  cudaError_t e = cudaFuncSetAttribute(tc_fwd2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, F2_SMEM);
  if (e != cudaSuccess) return e;
  const size_t units = p->n_items[op] / 4;
  tc_fwd2_kernel<<<(unsigned)(2 * units), F2_THREADS, F2_SMEM, st>>>(mq, mkp, mvp, mkr, mvr, geometry(p), p->queue_d[op],
                                                                    p->bm[op], p->bn[op], (__nv_bfloat16*)o, lse,
                                                                    q_rows, p->err_d);
  return cudaGetLastError();
}

}  // namespace augtree
