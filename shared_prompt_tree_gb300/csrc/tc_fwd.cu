// Tensor-core forward of tree attention on sm_103a: one query head per thread block,
// with a double-buffered score tile.
//
// AugTree paper, "Splitting Prompt Prefill from Response Replay ...":
//   Sec. 2.2  attention as Q-KV tile interactions with an online softmax;
//   Sec. 3.2  prefill rows see the prompt causally; a replay row (Eq. 1) sees all prompt
//             keys of its group and its own branch's keys up to itself;
//   Sec. 3.3  partial softmax states merge associatively: here the two halves of every
//             key tile keep separate running states, merged once per row at the end
//             (and, for a split-KV item, its chunk's state goes to the workspace for the
//             merge across chunks).
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
// the softmax of tile j+1 can start as soon as that of tile j ends: the per-head chain
// PV(j) -> S(j+1) of a shared score buffer is gone.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_rows.cuh"

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
constexpr int FWD_THREADS = 352;
constexpr int FWD_NST = 3;                     // K/V ring stages
constexpr int FWD_TILE = 128 * 128;            // 128 rows x 64 bf16 columns = 16 KB
constexpr int FWD_Q_OFF = 0;                   // 2 blocks
constexpr int FWD_K_OFF = FWD_Q_OFF + 2 * FWD_TILE;            // [NST][2 blocks]
constexpr int FWD_V_OFF = FWD_K_OFF + FWD_NST * 2 * FWD_TILE;   // [NST][2 blocks]
constexpr int FWD_BAR_OFF = FWD_V_OFF + FWD_NST * 2 * FWD_TILE;
constexpr int FWD_SMEM = FWD_BAR_OFF + 256 + 1024;  // + barriers + alignment slack
static_assert(FWD_SMEM <= 232448, "shared memory per block");

struct FwdBars {
  uint64_t q_full;
  uint64_t kv_full[FWD_NST];   // K landed (and V too unless kFwdVBar)
  uint64_t v_full[FWD_NST];    // V landed (kFwdVBar)
  uint64_t kv_empty[FWD_NST];
  uint64_t s_full[2];      // per S buffer
  uint64_t p_full[2][2];   // per S buffer and warpgroup
  uint64_t pv_done[2];     // per S buffer: both PV products of the tile have completed
  uint64_t xch;            // both warpgroups have published their row states
  uint64_t drain[2];
  uint32_t tmem_base;
};
static_assert(sizeof(FwdBars) <= 256, "barrier area");

// kSplit: the replay queue holds split-KV items (a chunk of a tile's KV walk, partial
// state to the workspace); the instantiation without it is the plain kernel.
template <bool kSplit>
__global__ void __launch_bounds__(FWD_THREADS, 1) tc_fwd_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kp,
    const __grid_constant__ CUtensorMap tm_vp, const __grid_constant__ CUtensorMap tm_kr,
    const __grid_constant__ CUtensorMap tm_vr, Geometry geo, const int32_t* __restrict__ queue, int bm, int bn,
    __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int64_t lse_rows, uint32_t* __restrict__ err,
    float* __restrict__ part_o, float* __restrict__ part_lse) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FwdBars* bars = reinterpret_cast<FwdBars*>(smem + FWD_BAR_OFF);
  // Row-state exchange at the end, [2 warpgroups][128 rows][m, l]: it reuses the Q tile,
  // free once the last S product (implied complete by the last PV product) has read it.
  float* xch = reinterpret_cast<float*>(smem + FWD_Q_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const WorkItem it = load_item(queue, blockIdx.x);
  // Checked build: the item and its split are valid for the plan's geometry.
  const bool item_ok = !kChecked || (query_item_ok(it, geo, bm, bn) &&
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
  // Split-KV item: KV tiles [j0, j0 + n_tiles) of the walk, partial state to `slot`.
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

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
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
    }
    mbar_init(&bars->xch, 256);
    mbar_init(&bars->drain[0], 1);
    mbar_init(&bars->drain[1], 1);
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
      mbar_expect_tx(&bars->q_full, 2 * FWD_TILE);
      for (int kb = 0; kb < 2; ++kb)
        tma_load_3d(smem + FWD_Q_OFF + kb * FWD_TILE, &tm_q, &bars->q_full, kb * 64, h, (int)row0);
      int issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int stage = j % FWD_NST, use = j / FWD_NST;
        if (!mbar_wait(&bars->kv_empty[stage], (use & 1) ^ 1, err)) break;
        mbar_expect_tx(&bars->kv_full[stage], (kFwdVBar ? 2 : 4) * FWD_TILE);
        if (kFwdVBar) mbar_expect_tx(&bars->v_full[stage], 2 * FWD_TILE);
        const int jt = j0 + j;  // tile of the row's walk
        const bool own = jt >= n_a;
        const int krow = own ? (int)(own0 + (int64_t)(jt - n_a) * bn) : (int)(G.p0 + (int64_t)jt * bn);
        const CUtensorMap* km = own ? &tm_kr : &tm_kp;
        const CUtensorMap* vm = own ? &tm_vr : &tm_vp;
        uint64_t* vbar = kFwdVBar ? &bars->v_full[stage] : &bars->kv_full[stage];
        for (int kb = 0; kb < 2; ++kb)
          tma_load_3d(smem + FWD_K_OFF + (stage * 2 + kb) * FWD_TILE, km, &bars->kv_full[stage], kb * 64, kvh, krow);
        for (int kb = 0; kb < 2; ++kb)
          tma_load_3d(smem + FWD_V_OFF + (stage * 2 + kb) * FWD_TILE, vm, vbar, kb * 64, kvh, krow);
        issued = j + 1;
      }
      mbar_wait_drain(&bars->q_full, 0, err);
      for (int j = max(0, issued - FWD_NST); j < issued; ++j) {
        mbar_wait_drain(&bars->kv_full[j % FWD_NST], (j / FWD_NST) & 1, err);
        if (kFwdVBar) mbar_wait_drain(&bars->v_full[j % FWD_NST], (j / FWD_NST) & 1, err);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer: S
    constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
    const uint64_t dq = smem_desc_sw128(smem_u32(smem + FWD_Q_OFF), 16, 1024);
    const uint64_t dk0 = smem_desc_sw128(smem_u32(smem + FWD_K_OFF), 16, 1024);
    constexpr uint64_t kStage = (2 * FWD_TILE) >> 4;
    auto koff = [](int kk) { return (uint64_t)(((kk >> 2) * FWD_TILE + (kk & 3) * 32) >> 4); };
    bool ok = mbar_wait_warp_all(&bars->q_full, 0, err);
    tc_fence_after();
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int stage = j % FWD_NST, b = j & 1;
      if (!(ok = mbar_wait_warp_all(&bars->kv_full[stage], (j / FWD_NST) & 1, err))) break;
      // S(j) overwrites P(j-2) in buffer b: both PV products of tile j-2 must be done.
      if (j >= 2 && !(ok = mbar_wait_warp_all(&bars->pv_done[b], ((j >> 1) - 1) & 1, err))) break;
      tc_fence_after();
      const uint64_t dk = dk0 + stage * kStage;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss_w(tmem + b * 128, dq + koff(kk), dk + koff(kk), idesc_qk, kk > 0 ? 1u : 0u);
      mma_commit_w(&bars->s_full[b]);
    }
    mma_commit_w(&bars->drain[0]);
    mbar_wait_drain_warp_all(&bars->drain[0], 0, err);
  } else if (warp == 10) {
    // ------------------------------------------------------------ MMA issuer: PV
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 128, false, true);
    const uint64_t dv0 = smem_desc_sw128(smem_u32(smem + FWD_V_OFF), FWD_TILE, 1024);
    constexpr uint64_t kStage = (2 * FWD_TILE) >> 4;
    bool ok = true;
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int stage = j % FWD_NST, b = j & 1;
      const uint32_t par = (j >> 1) & 1;
      if (kFwdVBar && !(ok = mbar_wait_warp_all(&bars->v_full[stage], (j / FWD_NST) & 1, err))) break;
      if (!kFwdPvEarly) {
        if (!(ok = mbar_wait_warp_all(&bars->p_full[b][0], par, err))) break;
        if (!(ok = mbar_wait_warp_all(&bars->p_full[b][1], par, err))) break;
        tc_fence_after();
      }
      const uint64_t dv = dv0 + stage * kStage;
      // 16 keys per step: 16 swizzled 128-byte rows of V = 2048 bytes; P packs two keys
      // per TMEM column.  Warpgroup w's keys [64w, 64w + 64) sit in columns
      // [64w, 64w + 32) of the buffer.
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        if (kFwdPvEarly) {
          // O_w's product goes as soon as warpgroup w's P is ready.
          if (!(ok = mbar_wait_warp_all(&bars->p_full[b][w], par, err))) break;
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts_w(tmem + 256 + w * 128, tmem + b * 128 + w * 64 + kk * 8, dv + (4 * w + kk) * (2048 >> 4), idesc_pv,
                   (j > 0 || kk > 0) ? 1u : 0u);
      }
      if (!ok) break;
      mma_commit_w(&bars->pv_done[b]);
      mma_commit_w(&bars->kv_empty[stage]);
    }
    mma_commit_w(&bars->drain[1]);
    mbar_wait_drain_warp_all(&bars->drain[1], 0, err);
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
    g.j0 = j0;
    const float sl2 = geo.scale_log2;
    const uint32_t tO = tmem + lane_off + 256 + w * 128;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int b = j & 1;
      const uint32_t tS = tmem + lane_off + b * 128 + w * 64;
      if (!(ok = mbar_wait_warp_all(&bars->s_full[b], (j >> 1) & 1, err))) break;
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
        for (int k = 0; k < 8; ++k) pm[k] = fmax3(pm[k], __uint_as_float(FWD_X(c + k)), __uint_as_float(FWD_X(c + 8 + k)));
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
        if (!(ok = mbar_wait_warp_all(&bars->pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, err))) break;
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
    if (ok && n_tiles > 0) ok = mbar_wait_warp_all(&bars->pv_done[last & 1], (last >> 1) & 1, err);
    tc_fence_after();
    float* mine = xch + (w * 128 + r_local) * 2;
    mine[0] = m;
    mine[1] = l;
    mbar_arrive(&bars->xch);  // also on a failed wait, so the other warpgroup's wait ends
    if (ok) ok = mbar_wait_warp_all(&bars->xch, 0, err);
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
      if (kSplit && slot >= 0) {
        // Split-KV item: the chunk's state O / l (fp32) and its lse.
        float* prow = part_o + (slot * kFwdPartRows + r_local) * 128 + 64 * w;
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t o0[32], o1[32];
          tmem_ld32(tmem + lane_off + 256 + 64 * w + 32 * c, o0);
          tmem_ld32(tmem + lane_off + 384 + 64 * w + 32 * c, o1);
          tmem_ld_wait();
          if (g.row_ok) {
            float4* d4 = reinterpret_cast<float4*>(prow + 32 * c);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              float v[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                v[e] = any ? __uint_as_float(o0[4 * i + e]) * s0 + __uint_as_float(o1[4 * i + e]) * s1 : 0.f;
              d4[i] = make_float4(v[0], v[1], v[2], v[3]);
            }
          }
        }
        if (w == 0 && g.row_ok)
          part_lse[slot * kFwdPartRows + r_local] = any ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
      } else {
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
  auto kern = split ? tc_fwd_kernel<true> : tc_fwd_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FWD_SMEM);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)p->n_items[op], FWD_THREADS, FWD_SMEM, st>>>(mq, mkp, mvp, mkr, mvr, geometry(p), p->queue_d[op],
                                                                p->bm[op], p->bn[op], (__nv_bfloat16*)o, lse, q_rows,
                                                                p->err_d, part_o, part_lse);
  return cudaGetLastError();
}

}  // namespace augtree
