// Tensor-core forward of tree attention on sm_103a, one query head per thread block,
// with a double-buffered score tile.
//
// AugTree paper, "Splitting Prompt Prefill from Response Replay ...":
//   Sec. 2.2  attention as Q-KV tile interactions with an online softmax;
//   Sec. 3.2  prefill rows see the prompt causally; a replay row (Eq. 1) sees all prompt
//             keys of its group and its own branch's keys up to itself;
//   Sec. 3.3  partial softmax states merge associatively: here the two halves of every
//             key tile keep separate running states, merged once per row at the end.
//
// One block per work item: one 128-row query tile of one query head.
//   warp 8      TMA producer: Q, then a 3-stage ring of K/V tiles (128 keys x 128 dims)
//   warp 9      TMEM allocator and issuer of S(j) = Q K^T into buffer j % 2
//   warp 10     issuer of O_w += P_w(j) V_w(j), w = 0, 1 (V_w: the tile's keys
//               [64w, 64w + 64))
//   warps 0-7   two softmax warpgroups; warpgroup w owns keys [64w, 64w + 64) of every
//               tile and its own running max, sum of rounded weights and accumulator
//               O_w; thread i of each warpgroup owns row i (TMEM lane i)
// TMEM columns: S0/P0 [0,128), S1/P1 [128,256), O_0 [256,384), O_1 [384,512).
// S(j+1) goes to the other buffer and waits only for the PV products of tile j-1, so
// the softmax of tile j+1 can start as soon as that of tile j ends.
#include <cuda.h>

#include <cmath>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_fwd_softmax.cuh"

namespace augtree {
namespace {

using namespace tc;

constexpr int F1_THREADS = 352;
constexpr int F1_NST = 3;                     // K/V ring stages
constexpr int F1_TILE = 128 * 128;            // 128 rows x 64 bf16 columns = 16 KB
constexpr int F1_Q_OFF = 0;                   // 2 blocks
constexpr int F1_K_OFF = F1_Q_OFF + 2 * F1_TILE;            // [NST][2 blocks]
constexpr int F1_V_OFF = F1_K_OFF + F1_NST * 2 * F1_TILE;   // [NST][2 blocks]
constexpr int F1_BAR_OFF = F1_V_OFF + F1_NST * 2 * F1_TILE;
constexpr int F1_SMEM = F1_BAR_OFF + 256 + 1024;  // + barriers + alignment slack
static_assert(F1_SMEM <= 232448, "shared memory per block");

struct F1Bars {
  uint64_t q_full;
  uint64_t kv_full[F1_NST];
  uint64_t kv_empty[F1_NST];
  uint64_t s_full[2];      // per S buffer
  uint64_t p_full[2][2];   // per S buffer and warpgroup
  uint64_t pv_done[2];     // per S buffer: both PV products of the tile have completed
  uint64_t xch;            // both warpgroups have published their row states
  uint32_t tmem_base;
};
static_assert(sizeof(F1Bars) <= 256, "barrier area");

__global__ void __launch_bounds__(F1_THREADS, 1) tc_fwd1_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kp,
    const __grid_constant__ CUtensorMap tm_vp, const __grid_constant__ CUtensorMap tm_kr,
    const __grid_constant__ CUtensorMap tm_vr, Geometry geo, const int32_t* __restrict__ queue, int bm, int bn,
    __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int64_t lse_rows, uint32_t* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  F1Bars* bars = reinterpret_cast<F1Bars*>(smem + F1_BAR_OFF);
  // Row-state exchange at the end, [2 warpgroups][128 rows][m, l]: it reuses the Q tile,
  // free once the last S product (implied complete by the last PV product) has read it.
  float* xch = reinterpret_cast<float*>(smem + F1_Q_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

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
    for (int i = 0; i < F1_NST; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->p_full[b][0], 128);
      mbar_init(&bars->p_full[b][1], 128);
      mbar_init(&bars->pv_done[b], 1);
    }
    mbar_init(&bars->xch, 256);
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
      mbar_expect_tx(&bars->q_full, 2 * F1_TILE);
      for (int kb = 0; kb < 2; ++kb)
        tma_load_3d(smem + F1_Q_OFF + kb * F1_TILE, &tm_q, &bars->q_full, kb * 64, h, (int)row0);
      int issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int stage = j % F1_NST, use = j / F1_NST;
        if (!mbar_wait(&bars->kv_empty[stage], (use & 1) ^ 1, err)) break;
        mbar_expect_tx(&bars->kv_full[stage], 4 * F1_TILE);
        const bool own = j >= n_a;
        const int krow = own ? (int)(own0 + (int64_t)(j - n_a) * bn) : (int)(G.p0 + (int64_t)j * bn);
        const CUtensorMap* km = own ? &tm_kr : &tm_kp;
        const CUtensorMap* vm = own ? &tm_vr : &tm_vp;
        for (int kb = 0; kb < 2; ++kb) {
          tma_load_3d(smem + F1_K_OFF + (stage * 2 + kb) * F1_TILE, km, &bars->kv_full[stage], kb * 64, kvh, krow);
          tma_load_3d(smem + F1_V_OFF + (stage * 2 + kb) * F1_TILE, vm, &bars->kv_full[stage], kb * 64, kvh, krow);
        }
        issued = j + 1;
      }
      // Never leave a copy in flight: wait for the last fill of every buffer used.
      mbar_wait(&bars->q_full, 0, err);
      for (int j = max(0, issued - F1_NST); j < issued; ++j)
        mbar_wait(&bars->kv_full[j % F1_NST], (j / F1_NST) & 1, err);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer: S
    constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
    const uint64_t dq = smem_desc_sw128(smem_u32(smem + F1_Q_OFF), 16, 1024);
    const uint64_t dk0 = smem_desc_sw128(smem_u32(smem + F1_K_OFF), 16, 1024);
    constexpr uint64_t kStage = (2 * F1_TILE) >> 4;
    auto koff = [](int kk) { return (uint64_t)(((kk >> 2) * F1_TILE + (kk & 3) * 32) >> 4); };
    bool ok = mbar_wait_warp_all(&bars->q_full, 0, err);
    tc_fence_after();
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int stage = j % F1_NST, b = j & 1;
      if (!(ok = mbar_wait_warp_all(&bars->kv_full[stage], (j / F1_NST) & 1, err))) break;
      // S(j) overwrites P(j-2) in buffer b: both PV products of tile j-2 must be done.
      if (j >= 2 && !(ok = mbar_wait_warp_all(&bars->pv_done[b], ((j >> 1) - 1) & 1, err))) break;
      tc_fence_after();
      const uint64_t dk = dk0 + stage * kStage;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss_w(tmem + b * 128, dq + koff(kk), dk + koff(kk), idesc_qk, kk > 0 ? 1u : 0u);
      mma_commit_w(&bars->s_full[b]);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ MMA issuer: PV
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 128, false, true);
    const uint64_t dv0 = smem_desc_sw128(smem_u32(smem + F1_V_OFF), F1_TILE, 1024);
    constexpr uint64_t kStage = (2 * F1_TILE) >> 4;
    bool ok = true;
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int stage = j % F1_NST, b = j & 1;
      const uint32_t par = (j >> 1) & 1;
      if (!(ok = mbar_wait_warp_all(&bars->p_full[b][0], par, err))) break;
      if (!(ok = mbar_wait_warp_all(&bars->p_full[b][1], par, err))) break;
      tc_fence_after();
      const uint64_t dv = dv0 + stage * kStage;
      // 16 keys per step: 16 swizzled 128-byte rows of V = 2048 bytes; P packs two keys
      // per TMEM column.  Warpgroup w's keys [64w, 64w + 64) sit in columns
      // [64w, 64w + 32) of the buffer.
#pragma unroll
      for (int w = 0; w < 2; ++w) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts_w(tmem + 256 + w * 128, tmem + b * 128 + w * 64 + kk * 8, dv + (4 * w + kk) * (2048 >> 4), idesc_pv,
                   (j > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit_w(&bars->pv_done[b]);
      mma_commit_w(&bars->kv_empty[stage]);
    }
  } else {
    // ------------------------------------------------------------ softmax (half tiles)
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
    const uint32_t tO = tmem + lane_off + 256 + w * 128;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int b = j & 1;
      const uint32_t tS = tmem + lane_off + b * 128 + w * 64;
      if (!(ok = mbar_wait(&bars->s_full[b], (j >> 1) & 1, err))) break;
      tc_fence_after();
      uint32_t raw[2][32];
      tmem_ld32(tS, raw[0]);
      tmem_ld32(tS + 32, raw[1]);
      tmem_ld_wait();
#define F1_X(c) raw[(c) >> 5][(c) & 31]
      int lo_i, hi_i;
      fwd_valid_cols(g, j, lo_i, hi_i);
      const int lo = lo_i - 64 * w, hi = hi_i - 64 * w;  // valid local columns [lo, hi]
      const bool masked = lo > 0 || hi < 63;
      if (masked) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c < lo || c > hi) F1_X(c) = 0xFF800000u;  // -inf
      }
      float pm[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) pm[k] = __uint_as_float(F1_X(k));
#pragma unroll
      for (int c = 8; c < 64; ++c) pm[c & 7] = fmaxf(pm[c & 7], __uint_as_float(F1_X(c)));
      const float tmax =
          fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])), fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
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
        const float a0 = fmaf(__uint_as_float(F1_X(2 * i)), sl2, -mu);
        const float a1 = fmaf(__uint_as_float(F1_X(2 * i + 1)), sl2, -mu);
        const float p0 = fast_exp2(a0);
        float p1;
        if (i == 31) {
          // One exponential in 64 on the FMA pipe; a masked column stays exactly zero.
          p1 = exp2_fma(a1);
          if (masked && a1 == -INFINITY) p1 = 0.f;
        } else {
          p1 = fast_exp2(a1);
        }
        pk[i] = pack_bf16x2(p0, p1);
        // The row sum uses the bf16 weights the PV product uses.
        ps[i & 3] += __uint_as_float(pk[i] << 16) + __uint_as_float(pk[i] & 0xFFFF0000u);
      }
#undef F1_X
      tmem_st32(tS, pk);
      tmem_st_wait();
      l = l * alpha + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
      if (__any_sync(0xffffffffu, need)) {
        // O_w += P(j-1) V must be complete before O_w is rescaled; PV(j) is issued only
        // after this warpgroup signals P(j).
        if (!(ok = mbar_wait(&bars->pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, err))) break;
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
    }
    // Merge the two warpgroups' states of each row: (O_0, m_0, l_0) and (O_1, m_1, l_1).
    const int last = n_tiles - 1;
    if (ok && n_tiles > 0) ok = mbar_wait(&bars->pv_done[last & 1], (last >> 1) & 1, err);
    tc_fence_after();
    float* mine = xch + (w * 128 + r_local) * 2;
    mine[0] = m;
    mine[1] = l;
    mbar_arrive(&bars->xch);  // also on a failed wait, so the other warpgroup's wait ends
    if (ok) ok = mbar_wait(&bars->xch, 0, err);
    if (ok) {
      const float m0 = xch[r_local * 2], l0 = xch[r_local * 2 + 1];
      const float m1 = xch[(128 + r_local) * 2], l1 = xch[(128 + r_local) * 2 + 1];
      const float M = fmaxf(m0, m1);
      const float a0 = (m0 == -INFINITY) ? 0.f : fast_exp2(m0 - M);
      const float a1 = (m1 == -INFINITY) ? 0.f : fast_exp2(m1 - M);
      const float L = l0 * a0 + l1 * a1;
      const bool any = L > 0.f && n_tiles > 0;  // a row with no key writes zeros
      const float inv = any ? 1.f / L : 0.f;
      const float s0 = a0 * inv, s1 = a1 * inv;
      // Warpgroup w writes dims [64w, 64w + 64) of its rows.
      __nv_bfloat16* orow = out + (g.row * geo.hq + h) * 128 + 64 * w;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t o0[32], o1[32];
        tmem_ld32(tmem + lane_off + 256 + 64 * w + 32 * c, o0);
        tmem_ld32(tmem + lane_off + 384 + 64 * w + 32 * c, o1);
        tmem_ld_wait();
        if (g.row_ok) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float v0 = any ? __uint_as_float(o0[2 * i]) * s0 + __uint_as_float(o1[2 * i]) * s1 : 0.f;
            const float v1 = any ? __uint_as_float(o0[2 * i + 1]) * s0 + __uint_as_float(o1[2 * i + 1]) * s1 : 0.f;
            pk[i] = pack_bf16x2(v0, v1);
          }
          uint4* d4 = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
          for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      if (w == 0 && g.row_ok) lse[(int64_t)h * lse_rows + g.row] = any ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
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

cudaError_t tc_fwd1(const augtree_plan* p, int op, const CUtensorMap& mq, const CUtensorMap& mkp,
                    const CUtensorMap& mvp, const CUtensorMap& mkr, const CUtensorMap& mvr, void* o, float* lse,
                    int64_t q_rows, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(tc_fwd1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, F1_SMEM);
  if (e != cudaSuccess) return e;
  tc_fwd1_kernel<<<(unsigned)p->n_items[op], F1_THREADS, F1_SMEM, st>>>(
      mq, mkp, mvp, mkr, mvr, geometry(p), p->queue_d[op], p->bm[op], p->bn[op], (__nv_bfloat16*)o, lse, q_rows,
      p->err_d);
  return cudaGetLastError();
}

}  // namespace augtree
