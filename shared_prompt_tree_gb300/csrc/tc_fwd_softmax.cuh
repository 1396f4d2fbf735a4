// The softmax warpgroup of the tensor-core forward kernels (one and two CTAs per MMA):
// one thread per query row (TMEM lane), shared by the forward kernel and the
// query side of the backward (its row geometry).
//
// AugTree paper, Sec. 2.2 (online softmax over Q-KV tiles), Sec. 3.2 Eq. 1 (the row's
// valid keys: the whole prompt of its group, then its own branch up to itself; causal
// over the prompt for prefill rows) and Sec. 3.3 (the prompt-part and own-part states
// merge associatively; here one running state crosses both parts).
#pragma once

#include <cmath>

#include "common.cuh"
#include "tc_common.cuh"

namespace augtree {
namespace tc {

// In the row's second half, every kFwdFmaStride-th pair's second exponential runs on
// the FMA pipe (exp2_fma): 16 -> one exponential in 64 overall; 0 -> none.  Measured
// with the two heads' exponential phases alternating (prompt-heavy forward, TFLOP/s):
// one in 4: 1,094; in 8: 1,155; in 16: 1,267; in 32: 1,245; in 64: 1,326; none: 1,174.
#ifndef AUGTREE_FWD_FMA_STRIDE
#define AUGTREE_FWD_FMA_STRIDE 16
#endif
constexpr int kFwdFmaStride = AUGTREE_FWD_FMA_STRIDE;
#ifndef AUGTREE_FWD_FMA_OFFSET
#define AUGTREE_FWD_FMA_OFFSET (AUGTREE_FWD_FMA_STRIDE - 1)
#endif
// Which pair of each stride: measured (stride 16) offset 15: 1,293-1,300 TFLOP/s,
// offsets 7 and 0: 1,277; stride 32 offset 31: 1,293 (prompt-heavy forward, one box).
constexpr int kFwdFmaOffset = AUGTREE_FWD_FMA_OFFSET;
// Where the two heads' softmax hand off: 0 = around the exponential loop, 1 = the turn
// passes after the first half of the loop, 2 = the wait also covers the row max.
// Measured (prompt-heavy forward, one box): 1,327 / 1,317 / 1,288 TFLOP/s.
#ifndef AUGTREE_FWD_TURN_POS
#define AUGTREE_FWD_TURN_POS 0
#endif
constexpr int kFwdTurnPos = AUGTREE_FWD_TURN_POS;
// Row max with three-input max instructions and row sum with mixed-precision bf16 adds
// (about 190 instead of about 380 instructions per row and tile); 0: two-input max,
// unpack-and-add.
#ifndef AUGTREE_FWD_MIXED_OPS
#define AUGTREE_FWD_MIXED_OPS 1
#endif
constexpr bool kFwdMixedOps = AUGTREE_FWD_MIXED_OPS != 0;

// Where the row's keys come from in KV tile j: prompt tiles first, then the own-branch
// tiles, and the valid columns [lo, hi] of the row in that tile.
struct FwdRowGeom {
  int64_t row;      // global query row (prompt or response rows)
  bool row_ok;      // row < end of its query tile's group
  bool prefill;
  int64_t bs;       // first response row of the row's branch (replay rows)
  int64_t p0, p_end;  // the group's prompt keys
  int64_t own0;     // first key of the own-branch tiles
  int n_a;          // number of prompt tiles
  int bn;           // keys per tile
  int j0;           // first KV tile of the item (a split item's chunk; 0 otherwise)
};

// Valid columns of the item's j-th KV tile (tile j0 + j of the row's walk).
__device__ __forceinline__ void fwd_valid_cols(const FwdRowGeom& g, int j_local, int& lo_i, int& hi_i) {
  const int j = j_local + g.j0;
  const bool own = j >= g.n_a;
  const int64_t key0 = own ? g.own0 + (int64_t)(j - g.n_a) * g.bn : g.p0 + (int64_t)j * g.bn;
  int64_t lo, hi;
  if (g.prefill) {
    lo = 0;
    hi = g.row - key0;
  } else if (!own) {
    lo = 0;
    hi = g.p_end - 1 - key0;
  } else {
    lo = g.bs - key0;
    hi = g.row - key0;
  }
  if (!g.row_ok) {
    lo = 1;
    hi = 0;
  }
  lo_i = lo < -1 ? -1 : (lo > 128 ? 128 : (int)lo);
  hi_i = hi < -1 ? -1 : (hi > 128 ? 128 : (int)hi);
}

// Exponential-phase hand-off between a block's two softmax warpgroups.  The two heads
// of a block otherwise run their softmax in step, share the MUFU (about twice as slow
// each) and leave the tensor pipe idle meanwhile; alternating them lets one head's
// exponentials overlap the other head's MMAs.  NoTurn: no hand-off.
struct NoTurn {
  __device__ __forceinline__ bool wait(int, uint32_t*) const { return true; }
  __device__ __forceinline__ void pass() const {}
};
// mine / other: mbarriers with an arrival count of 4 (one per warp of the warpgroup
// that passes the turn).  first = 1 for the warpgroup that starts: its tile j waits for
// the other's tile j-1; the other warpgroup's tile j waits for this one's tile j.
struct PingPong {
  uint64_t* mine;
  uint64_t* other;
  int first;
  __device__ __forceinline__ bool wait(int j, uint32_t* err) const {
    const int n = j - first;
    return n < 0 || mbar_wait_warp_all(mine, n & 1, err);
  }
  __device__ __forceinline__ void pass() const {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(other);
  }
};

// Runs the row's online softmax over n_tiles KV tiles of 128 keys.  For each tile:
// waits s_full (S in TMEM), masks, keeps a running max with lazy rescaling of O
// (only when the max grows by more than 2^8; exact, every term shares the offset),
// writes P = exp2(s*log2e*S - m) as bf16 over S (one value in 64 from the FMA-pipe
// exponential), adds the bf16 values to the row sum, and calls signal_p() once its
// warpgroup may hand P to the MMA issuer.  At the end writes O / l (bf16) and lse; or,
// with kMayPart and a non-null part_row (a split-KV item), the partial state O / l as
// fp32 to part_row[128] and its lse to *part_lse (-inf and zeros if no key was valid).
template <bool kMayPart = false, typename SignalP, typename Turn = NoTurn>
__device__ __forceinline__ void fwd_softmax_row(uint32_t tS, uint32_t tO, const FwdRowGeom& g, int n_tiles, float sl2,
                                                uint64_t* s_full, uint64_t* o_done, SignalP signal_p,
                                                __nv_bfloat16* out_row, float* lse_ptr, uint32_t* err,
                                                Turn turn = Turn(), float* part_row = nullptr,
                                                float* part_lse = nullptr) {
  float m = -INFINITY, l = 0.f;
  bool ok = true;
  for (int j = 0; j < n_tiles; ++j) {
    if (!(ok = mbar_wait_warp_all(s_full, j & 1, err))) break;
    tc_fence_after();
    uint32_t raw[4][32];  // S row, reinterpreted as fp32 in place (no second copy)
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, raw[c]);
    tmem_ld_wait();
#define AUGTREE_X(c) raw[(c) >> 5][(c) & 31]
    if (kFwdTurnPos == 2 && !(ok = turn.wait(j, err))) break;
    int lo_i, hi_i;
    fwd_valid_cols(g, j, lo_i, hi_i);
    const bool masked = lo_i > 0 || hi_i < 127;
    if (masked) {
#pragma unroll
      for (int c = 0; c < 128; ++c)
        if (c < lo_i || c > hi_i) AUGTREE_X(c) = 0xFF800000u;  // -inf
    }
    // Row max with 8 independent partial maxima (a single 127-long dependent chain
    // would dominate the latency of the warpgroup's turn).
    float pm[8];
    float tmax;
    if (kFwdMixedOps) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        pm[k] = fmax3(__uint_as_float(AUGTREE_X(k)), __uint_as_float(AUGTREE_X(k + 8)),
                      __uint_as_float(AUGTREE_X(k + 16)));
#pragma unroll
      for (int c = 24; c < 120; c += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          pm[k] = fmax3(pm[k], __uint_as_float(AUGTREE_X(c + k)), __uint_as_float(AUGTREE_X(c + 8 + k)));
#pragma unroll
      for (int k = 0; k < 8; ++k) pm[k] = fmaxf(pm[k], __uint_as_float(AUGTREE_X(120 + k)));
      tmax = fmaxf(fmax3(pm[0], pm[1], pm[2]), fmax3(fmax3(pm[3], pm[4], pm[5]), pm[6], pm[7]));
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) pm[k] = __uint_as_float(AUGTREE_X(k));
#pragma unroll
      for (int c = 8; c < 128; ++c) pm[c & 7] = fmaxf(pm[c & 7], __uint_as_float(AUGTREE_X(c)));
      tmax = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])), fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
    }
    const float mx = tmax * sl2;  // -inf stays -inf
    const bool need = (m != -INFINITY) && (mx > m + 8.0f);
    const float m_new = (m == -INFINITY) ? mx : (need ? mx : m);
    const float alpha = need ? fast_exp2(m - m_new) : 1.f;
    m = m_new;
    const float mu = (m == -INFINITY) ? 0.f : m;
    if (kFwdTurnPos != 2 && !(ok = turn.wait(j, err))) break;
    float ps[4] = {0.f, 0.f, 0.f, 0.f};  // 4 independent partial sums
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int c0 = c * 64 + 2 * i;
        const float a0 = fmaf(__uint_as_float(AUGTREE_X(c0)), sl2, -mu);
        const float a1 = fmaf(__uint_as_float(AUGTREE_X(c0 + 1)), sl2, -mu);
        float p0 = fast_exp2(a0), p1;
        if (kFwdFmaStride > 0 && c == 1 && i % (kFwdFmaStride > 0 ? kFwdFmaStride : 1) == kFwdFmaOffset) {
          // FMA-pipe exponential (second half of the row, where half of S has already
          // been consumed and registers are free); a masked column (-inf) must stay
          // exactly zero.
          p1 = exp2_fma(a1);
          if (masked && a1 == -INFINITY) p1 = 0.f;
        } else {
          p1 = fast_exp2(a1);
        }
        pk[i] = pack_bf16x2(p0, p1);
        // The denominator sums the bf16 values the PV product uses, so numerator and
        // denominator carry the same rounded weights.
        if (kFwdMixedOps)
          ps[i & 3] = add_bf16x2_f32(ps[i & 3], pk[i]);
        else
          ps[i & 3] += __uint_as_float(pk[i] << 16) + __uint_as_float(pk[i] & 0xFFFF0000u);
      }
      tmem_st32(tS + c * 32, pk);
      if (kFwdTurnPos == 1 && c == 0) turn.pass();
    }
#undef AUGTREE_X
    if (kFwdTurnPos != 1) turn.pass();
    tmem_st_wait();
    const float psum = (ps[0] + ps[1]) + (ps[2] + ps[3]);
    l = l * alpha + psum;
    if (__any_sync(0xffffffffu, need)) {
      // O += P(j-1) V must be complete before O is rescaled; PV(j) is issued only
      // after this row's warpgroup signals P(j).
      if (!(ok = mbar_wait_warp_all(o_done, (j - 1) & 1, err))) break;
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
    signal_p();
  }
  if (ok && mbar_wait_warp_all(o_done, (n_tiles - 1) & 1, err)) {
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    if (kMayPart && part_row != nullptr) {
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_ld_wait();
        if (g.row_ok) {
          float4* d4 = reinterpret_cast<float4*>(part_row + c * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            d4[i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
        }
      }
      if (g.row_ok) *part_lse = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
      return;
    }
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      tmem_ld32(tO + c * 32, o);
      tmem_ld_wait();
      if (g.row_ok) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
        uint4* d4 = reinterpret_cast<uint4*>(out_row + c * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
    }
    if (g.row_ok) *lse_ptr = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
  }
}

}  // namespace tc
}  // namespace augtree
