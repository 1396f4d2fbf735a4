// Tensor-core forward of tree attention on sm_103a: prompt prefill and response
// replay in one kernel.
//
// AugTree paper, "Splitting Prompt Prefill from Response Replay ...":
//   Sec. 2.2  attention as Q-KV tile interactions with an online softmax;
//   Sec. 3.2  prefill: causal self-attention of the prompt, computed once; replay,
//             Eq. 1: a response row sees all prompt keys of its group (dense) and its
//             own branch's keys up to itself;
//   Sec. 3.3  the prompt-part and the own-branch-part states of a row are merged
//             associatively - here as one running online softmax over the prompt
//             tiles followed by the own-branch tiles.
//
// One thread block per work unit: one query tile of 128 rows for one or two query
// heads of the same KV head (both heads share every K/V tile, loaded once).
//   warp 8      TMA producer: Q tiles, then a 2-stage ring of K/V tiles (128-byte
//               swizzle, 128 keys x 128 dims each)
//   warp 9      TMEM allocator and MMA issuer: S = Q K^T (bf16 x bf16 -> fp32 TMEM),
//               O += P V with P read from TMEM as the A operand
//   warps 0-7   two softmax warpgroups, one per query head; thread i owns row i
//               (TMEM lane i): masks, running max with lazy rescaling of O (only
//               when the max grows by more than 2^8), P = exp2(...) as bf16 back
//               into TMEM over S, the row sum l of those bf16 values, and the final
//               O / l and lse.
// TMEM columns: S0/P0 [0,128), S1/P1 [128,256), O0 [256,384), O1 [384,512).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "common.cuh"
#include "tc_common.cuh"

namespace augtree {
namespace {

using namespace tc;

constexpr int FWD_THREADS = 320;
constexpr int NST = 2;                  // K/V ring stages
constexpr int TILE_BYTES = 128 * 128;   // one 128-row x 64-column bf16 block = 16 KB
constexpr int Q_OFF = 0;                                  // [2 heads][2 blocks]
constexpr int K_OFF = Q_OFF + 4 * TILE_BYTES;             // [NST][2 blocks]
constexpr int V_OFF = K_OFF + NST * 2 * TILE_BYTES;       // [NST][2 blocks]
constexpr int BAR_OFF = V_OFF + NST * 2 * TILE_BYTES;
constexpr int FWD_SMEM = BAR_OFF + 256 + 1024;            // + barriers + alignment slack

struct FwdBars {
  uint64_t q_full;
  uint64_t kv_full[NST];
  uint64_t kv_empty[NST];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint32_t tmem_base;
};

__global__ void __launch_bounds__(FWD_THREADS, 1) tc_fwd_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kp,
    const __grid_constant__ CUtensorMap tm_vp, const __grid_constant__ CUtensorMap tm_kr,
    const __grid_constant__ CUtensorMap tm_vr, Geometry geo, const int32_t* __restrict__ queue, int paired, int bm,
    int bn, __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int64_t lse_rows, uint32_t* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FwdBars* bars = reinterpret_cast<FwdBars*>(smem + BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int n_sub = paired ? 2 : 1;
  const WorkItem it0 = load_item(queue, (int64_t)blockIdx.x * n_sub);
  int heads[2];
  heads[0] = it0.head;
  heads[1] = paired ? load_item(queue, (int64_t)blockIdx.x * 2 + 1).head : it0.head;
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
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < NST; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 128);
      mbar_init(&bars->o_done[i], 1);
    }
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
      mbar_expect_tx(&bars->q_full, n_sub * 2 * TILE_BYTES);
      for (int s = 0; s < n_sub; ++s)
        for (int kb = 0; kb < 2; ++kb)
          tma_load_3d(smem + Q_OFF + (s * 2 + kb) * TILE_BYTES, &tm_q, &bars->q_full, kb * 64, heads[s], (int)row0);
      int issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int stage = j % NST, use = j / NST;
        if (!mbar_wait(&bars->kv_empty[stage], (use & 1) ^ 1, err)) break;
        mbar_expect_tx(&bars->kv_full[stage], 4 * TILE_BYTES);
        const bool own = j >= n_a;
        const int krow = own ? (int)(own0 + (int64_t)(j - n_a) * bn) : (int)(G.p0 + (int64_t)j * bn);
        const CUtensorMap* km = own ? &tm_kr : &tm_kp;
        const CUtensorMap* vm = own ? &tm_vr : &tm_vp;
        for (int kb = 0; kb < 2; ++kb) {
          tma_load_3d(smem + K_OFF + (stage * 2 + kb) * TILE_BYTES, km, &bars->kv_full[stage], kb * 64, kvh, krow);
          tma_load_3d(smem + V_OFF + (stage * 2 + kb) * TILE_BYTES, vm, &bars->kv_full[stage], kb * 64, kvh, krow);
        }
        issued = j + 1;
      }
      // Never leave a copy in flight: wait for the last fill of every stage used.
      mbar_wait(&bars->q_full, 0, err);
      for (int j = max(0, issued - NST); j < issued; ++j) mbar_wait(&bars->kv_full[j % NST], (j / NST) & 1, err);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 128, false, true);
      bool ok = mbar_wait(&bars->q_full, 0, err);
      tc_fence_after();
      const uint32_t q_addr = smem_u32(smem + Q_OFF);
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int stage = j % NST, use = j / NST;
        if (!(ok = mbar_wait(&bars->kv_full[stage], use & 1, err))) break;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(smem + K_OFF + stage * 2 * TILE_BYTES);
        const uint32_t v_addr = smem_u32(smem + V_OFF + stage * 2 * TILE_BYTES);
        for (int s = 0; s < n_sub; ++s) {
          if (j > 0) {
            // S_s(j) overwrites P_s(j-1): wait until O_s += P_s(j-1) V has completed.
            if (!(ok = mbar_wait(&bars->o_done[s], (j - 1) & 1, err))) break;
            tc_fence_after();
          }
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * TILE_BYTES + (kk & 3) * 32;
            const uint64_t a = smem_desc_sw128(q_addr + s * 2 * TILE_BYTES + off, 16, 1024);
            const uint64_t b = smem_desc_sw128(k_addr + off, 16, 1024);
            mma_ss(tmem + s * 128, a, b, idesc_qk, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bars->s_full[s]);
        }
        if (!ok) break;
        for (int s = 0; s < n_sub; ++s) {
          if (!(ok = mbar_wait(&bars->p_full[s], j & 1, err))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // 16 keys per step: 16 swizzled 128-byte rows = 2048 bytes; the two
            // 64-dim halves of V are 16 KB apart (leading byte offset).
            const uint64_t b = smem_desc_sw128(v_addr + kk * 2048, TILE_BYTES, 1024);
            mma_ts(tmem + 256 + s * 128, tmem + s * 128 + kk * 8, b, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&bars->o_done[s]);
        }
        mma_commit(&bars->kv_empty[stage]);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int s = warp >> 2;
    if (s < n_sub) {
      const int q4 = warp & 3;
      const int r_local = q4 * 32 + lane;
      const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
      const uint32_t tS = tmem + s * 128 + lane_off;
      const uint32_t tO = tmem + 256 + s * 128 + lane_off;
      const int64_t row = row0 + r_local;
      const bool row_ok = row < row_end;
      const int64_t bs = (!prefill && row_ok) ? geo.row_bstart[row] : 0;
      const float sl2 = geo.scale_log2;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < n_tiles; ++j) {
        if (!(ok = mbar_wait(&bars->s_full[s], j & 1, err))) break;
        tc_fence_after();
        uint32_t raw[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, raw[c]);
        tmem_ld_wait();
        float x[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(raw[c >> 5][c & 31]);
        // valid key columns [lo, hi] of this row in tile j
        const bool own = j >= n_a;
        const int64_t key0 = own ? own0 + (int64_t)(j - n_a) * bn : G.p0 + (int64_t)j * bn;
        int64_t lo, hi;
        if (prefill) {
          lo = 0;
          hi = row - key0;
        } else if (!own) {
          lo = 0;
          hi = (int64_t)G.p0 + G.lp - 1 - key0;
        } else {
          lo = bs - key0;
          hi = row - key0;
        }
        if (!row_ok) {
          lo = 1;
          hi = 0;
        }
        if (lo > 0 || hi < 127) {
          const int lo_i = lo < -1 ? -1 : (lo > 128 ? 128 : (int)lo);
          const int hi_i = hi < -1 ? -1 : (hi > 128 ? 128 : (int)hi);
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c < lo_i || c > hi_i) x[c] = -INFINITY;
        }
        float tmax = x[0];
#pragma unroll
        for (int c = 1; c < 128; ++c) tmax = fmaxf(tmax, x[c]);
        const float mx = tmax * sl2;  // -inf stays -inf
        const bool need = (m != -INFINITY) && (mx > m + 8.0f);
        const float m_new = (m == -INFINITY) ? mx : (need ? mx : m);
        const float alpha = need ? fast_exp2(m - m_new) : 1.f;
        m = m_new;
        const float mu = (m == -INFINITY) ? 0.f : m;
        float psum = 0.f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float p0 = fast_exp2(fmaf(x[c * 64 + 2 * i], sl2, -mu));
            const float p1 = fast_exp2(fmaf(x[c * 64 + 2 * i + 1], sl2, -mu));
            pk[i] = pack_bf16x2(p0, p1);
            // The denominator sums the bf16 values the PV product uses, so numerator
            // and denominator carry the same rounded weights.
            psum += __uint_as_float(pk[i] << 16) + __uint_as_float(pk[i] & 0xFFFF0000u);
          }
          tmem_st32(tS + c * 32, pk);
        }
        tmem_st_wait();
        l = l * alpha + psum;
        if (__any_sync(0xffffffffu, need)) {
          // O_s += P_s(j-1) V must be complete before O is rescaled; PV(j) is issued
          // only after p_full(j) below.
          if (!(ok = mbar_wait(&bars->o_done[s], (j - 1) & 1, err))) break;
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
        mbar_arrive(&bars->p_full[s]);
      }
      if (ok && mbar_wait(&bars->o_done[s], (n_tiles - 1) & 1, err)) {
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int h = heads[s];
        __nv_bfloat16* dst = out + (row * geo.hq + h) * 128;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait();
          if (row_ok) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
        if (row_ok) lse[(int64_t)h * lse_rows + row] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
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
                   const void* vr, void* o, float* lse, cudaStream_t st) {
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
  cudaError_t e = cudaFuncSetAttribute(tc_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, FWD_SMEM);
  if (e != cudaSuccess) return e;
  const int paired = p->paired[op];
  const size_t units = paired ? p->n_items[op] / 2 : p->n_items[op];
  tc_fwd_kernel<<<(unsigned)units, FWD_THREADS, FWD_SMEM, st>>>(mq, mkp, mvp, mkr, mvr, geometry(p), p->queue_d[op],
                                                                paired, p->bm[op], p->bn[op], (__nv_bfloat16*)o, lse,
                                                                q_rows, p->err_d);
  return cudaGetLastError();
}

}  // namespace augtree
