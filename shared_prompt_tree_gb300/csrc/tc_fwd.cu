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
//   warps 9-10  MMA issuers, one per query head (warp 9 also allocates TMEM):
//               S = Q K^T (bf16 x bf16 -> fp32 TMEM), O += P V with P read from TMEM as
//               the A operand
//   warps 0-7   two softmax warpgroups, one per query head; thread i owns row i
//               (TMEM lane i): masks, running max with lazy rescaling of O (only
//               when the max grows by more than 2^8), P = exp2(...) as bf16 back
//               into TMEM over S, the row sum l of those bf16 values, and the final
//               O / l and lse.  The two warpgroups' exponential loops alternate (an
//               mbarrier hand-off), so one head's exponentials overlap the other
//               head's MMAs.
// TMEM columns: S0/P0 [0,128), S1/P1 [128,256), O0 [256,384), O1 [384,512).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_fwd_softmax.cuh"

namespace augtree {
namespace {

using namespace tc;

#ifndef AUGTREE_FWD_PINGPONG
#define AUGTREE_FWD_PINGPONG 1
#endif
constexpr bool kFwdPingPong = AUGTREE_FWD_PINGPONG != 0;

constexpr int FWD_THREADS = 352;  // 8 softmax warps, producer, one MMA issuer per head
constexpr int NST = 2;                  // K/V ring stages
// K/V tiles this many ahead of the one being filled are prefetched into L2, so that a
// refill (issued only once the stage frees) waits on L2 rather than DRAM latency.
// Measured neutral on prompt-heavy (1,278 against 1,285 TFLOP/s without): the kernel
// is not bound by load latency; kept off.
#ifndef AUGTREE_FWD_PREFETCH
#define AUGTREE_FWD_PREFETCH 0
#endif
constexpr int kFwdPrefetch = AUGTREE_FWD_PREFETCH;
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
  uint64_t turn[2];  // softmax hand-off: turn[s] completes when head s may run its exponentials
  uint64_t drain[2];  // issuer s: all of its MMAs have completed (before TMEM is freed)
  uint32_t tmem_base;
};

static_assert(sizeof(FwdBars) <= 256, "barrier area");

// kSplit: the replay queue holds split-KV items (a tile's KV walk cut into chunks,
// partial states to the workspace); the instantiation without it is the plain kernel.
template <bool kSplit>
__global__ void __launch_bounds__(FWD_THREADS, 1) tc_fwd_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kp,
    const __grid_constant__ CUtensorMap tm_vp, const __grid_constant__ CUtensorMap tm_kr,
    const __grid_constant__ CUtensorMap tm_vr, Geometry geo, const int32_t* __restrict__ queue, int paired, int bm,
    int bn, __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int64_t lse_rows, uint32_t* __restrict__ err,
    float* __restrict__ part_o, float* __restrict__ part_lse) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FwdBars* bars = reinterpret_cast<FwdBars*>(smem + BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int n_sub = paired ? 2 : 1;
  const WorkItem it0 = load_item(queue, (int64_t)blockIdx.x * n_sub);
  const WorkItem it1 = paired ? load_item(queue, (int64_t)blockIdx.x * 2 + 1) : it0;
  // Checked build: both items valid, and the same query tile and split (heads of one KV
  // head).
  const bool item_ok = !kChecked || (query_item_ok(it0, geo, bm, bn) && query_item_ok(it1, geo, bm, bn) &&
                                     it1.kind == it0.kind && it1.group == it0.group && it1.tile == it0.tile &&
                                     it1.split == it0.split &&
                                     it1.head / (geo.hq / geo.hkv) == it0.head / (geo.hq / geo.hkv) &&
                                     (kSplit ? split_item_ok(it0, geo) : it0.split == 0));
  if (kChecked && !item_ok && threadIdx.x == 0) atomicOr(err, kErrCheck);
  int heads[2];
  heads[0] = item_ok ? it0.head : 0;
  heads[1] = item_ok ? it1.head : 0;
  const GroupInfo G = geo.groups[item_ok ? it0.group : 0];
  const bool prefill = it0.kind == K_PREFILL_Q;
  const int64_t base = prefill ? G.p0 : G.r0;
  const int64_t len = prefill ? G.lp : G.lr;
  const int64_t row0 = item_ok ? base + (int64_t)it0.tile * bm : 0;
  const int64_t row_end = item_ok ? min(row0 + (int64_t)bm, base + len) : 0;
  const int n_a = item_ok ? it0.a : 0;
  int n_tiles = item_ok ? n_a + (prefill ? 0 : it0.b) : 0;
  const int64_t own0 = (prefill || !item_ok) ? 0 : geo.row_bstart[row0];
  const int kvh = heads[0] / (geo.hq / geo.hkv);
  // Split-KV item: KV tiles [j0, j0 + n_tiles) of the walk; partial-state slot of head s
  // = slot0 + heads[s] * nsplit + split.
  int j0 = 0;
  int64_t slot_base = -1, slot_stride = 0;
  if (kSplit && item_ok && !prefill) {
    const FwdSplit fs = geo.fsplit[G.tr0 + it0.tile];
    if (fs.nsplit > 1) {
      j0 = it0.split * fs.chunk;
      n_tiles = min(fs.chunk, n_tiles - j0);
      slot_base = fs.slot0 + it0.split;
      slot_stride = fs.nsplit;
    }
  }

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < NST; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], n_sub);  // one commit per head's issuer
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 128);
      mbar_init(&bars->o_done[i], 1);
      mbar_init(&bars->turn[i], 4);
      mbar_init(&bars->drain[i], 1);
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
        const int jt = j0 + j;  // tile of the row's walk
        const bool own = jt >= n_a;
        const int krow = own ? (int)(own0 + (int64_t)(jt - n_a) * bn) : (int)(G.p0 + (int64_t)jt * bn);
        const CUtensorMap* km = own ? &tm_kr : &tm_kp;
        const CUtensorMap* vm = own ? &tm_vr : &tm_vp;
        for (int kb = 0; kb < 2; ++kb) {
          tma_load_3d(smem + K_OFF + (stage * 2 + kb) * TILE_BYTES, km, &bars->kv_full[stage], kb * 64, kvh, krow);
          tma_load_3d(smem + V_OFF + (stage * 2 + kb) * TILE_BYTES, vm, &bars->kv_full[stage], kb * 64, kvh, krow);
        }
        issued = j + 1;
        if (kFwdPrefetch > 0) {
          // At the start, the first few tiles after the ring's; then one tile per fill.
          const int jp0 = j == 0 ? NST : j + kFwdPrefetch;
          for (int jp = jp0; jp <= j + kFwdPrefetch && jp < n_tiles; ++jp) {
            const int jpt = j0 + jp;
            const bool own_p = jpt >= n_a;
            const int rp = own_p ? (int)(own0 + (int64_t)(jpt - n_a) * bn) : (int)(G.p0 + (int64_t)jpt * bn);
            for (int kb = 0; kb < 2; ++kb) {
              tma_prefetch_3d(own_p ? &tm_kr : &tm_kp, kb * 64, kvh, rp);
              tma_prefetch_3d(own_p ? &tm_vr : &tm_vp, kb * 64, kvh, rp);
            }
          }
        }
      }
      // Never leave a copy in flight (also after giving up on a wait): wait for the last
      // fill of every stage used.
      mbar_wait_drain(&bars->q_full, 0, err);
      for (int j = max(0, issued - NST); j < issued; ++j)
        mbar_wait_drain(&bars->kv_full[j % NST], (j / NST) & 1, err);
    }
  } else if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 9 + s issues head s's products, so that while one head's issuer waits for its
    // softmax, the other keeps the tensor pipe fed.
    const int s = warp - 9;
    if (s < n_sub) {  // all 32 lanes: warp-uniform control flow; one elected lane issues
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 128, false, true);
      // Descriptors are built once; each MMA step adds a compile-time offset (16-byte
      // units) to the start-address field, keeping the issuing thread's chain short.
      const uint64_t dq = smem_desc_sw128(smem_u32(smem + Q_OFF + s * 2 * TILE_BYTES), 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(smem_u32(smem + K_OFF), 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(smem_u32(smem + V_OFF), TILE_BYTES, 1024);
      constexpr uint64_t kSub = (2 * TILE_BYTES) >> 4;   // next K,V stage
      auto koff = [](int kk) { return (uint64_t)(((kk >> 2) * TILE_BYTES + (kk & 3) * 32) >> 4); };
      const uint32_t ts = tmem + s * 128, to = tmem + 256 + s * 128;
      bool ok = mbar_wait_warp_all(&bars->q_full, 0, err);
      tc_fence_after();
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int stage = j % NST, use = j / NST;
        if (!(ok = mbar_wait_warp_all(&bars->kv_full[stage], use & 1, err))) break;
        if (j > 0) {
          // S(j) overwrites P(j-1): wait until O += P(j-1) V has completed.
          if (!(ok = mbar_wait_warp_all(&bars->o_done[s], (j - 1) & 1, err))) break;
        }
        tc_fence_after();
        const uint64_t dk = dk0 + stage * kSub, dv = dv0 + stage * kSub;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss_w(ts, dq + koff(kk), dk + koff(kk), idesc_qk, kk > 0 ? 1u : 0u);
        mma_commit_w(&bars->s_full[s]);
        if (!(ok = mbar_wait_warp_all(&bars->p_full[s], j & 1, err))) break;
        tc_fence_after();
        // 16 keys per step: 16 swizzled 128-byte rows = 2048 bytes; the two 64-dim
        // halves of V are 16 KB apart (leading byte offset).
        mma_ts_w(to, ts, dv, idesc_pv, j > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 1; kk < 8; ++kk) mma_ts_w(to, ts + kk * 8, dv + kk * (2048 >> 4), idesc_pv, 1u);
        mma_commit_w(&bars->o_done[s]);
        mma_commit_w(&bars->kv_empty[stage]);
      }
      // Never leave an MMA in flight when the block frees TMEM and exits (also after
      // giving up on a wait).
      mma_commit_w(&bars->drain[s]);
      mbar_wait_drain_warp_all(&bars->drain[s], 0, err);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int s = warp >> 2;
    if (s < n_sub) {
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
      g.j0 = j0;
      const int h = heads[s];
      uint64_t* p_full = &bars->p_full[s];
      auto signal = [p_full]() { mbar_arrive(p_full); };
      __nv_bfloat16* orow = out + (g.row * geo.hq + h) * 128;
      float* lrow = lse + (int64_t)h * lse_rows + g.row;
      float* prow = nullptr;
      float* plse = nullptr;
      if (kSplit && slot_base >= 0) {
        const int64_t slot = slot_base + (int64_t)h * slot_stride;
        prow = part_o + (slot * kFwdPartRows + r_local) * 128;
        plse = part_lse + slot * kFwdPartRows + r_local;
      }
      if (kFwdPingPong && n_sub == 2) {
        const PingPong turn{&bars->turn[s], &bars->turn[s ^ 1], s == 0 ? 1 : 0};
        fwd_softmax_row<kSplit>(tmem + s * 128 + lane_off, tmem + 256 + s * 128 + lane_off, g, n_tiles,
                                geo.scale_log2, &bars->s_full[s], &bars->o_done[s], signal, orow, lrow, err, turn,
                                prow, plse);
      } else {
        fwd_softmax_row<kSplit>(tmem + s * 128 + lane_off, tmem + 256 + s * 128 + lane_off, g, n_tiles,
                                geo.scale_log2, &bars->s_full[s], &bars->o_done[s], signal, orow, lrow, err, NoTurn(),
                                prow, plse);
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
  const int paired = p->paired[op];
  const size_t units = paired ? p->n_items[op] / 2 : p->n_items[op];
  kern<<<(unsigned)units, FWD_THREADS, FWD_SMEM, st>>>(mq, mkp, mvp, mkr, mvr, geometry(p), p->queue_d[op], paired,
                                                       p->bm[op], p->bn[op], (__nv_bfloat16*)o, lse, q_rows, p->err_d,
                                                       part_o, part_lse);
  return cudaGetLastError();
}

}  // namespace augtree
