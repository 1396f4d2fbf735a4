// SIMT (fp32 FMA) kernels of the tree-attention path: the forward of the prompt
// prefill and the response replay, and the KV-stationary backward.  They serve the
// fp32 mode (any dtype works; accumulation is fp32) and are the plain, easily checked
// counterpart of the tensor-core kernels.
//
// AugTree paper, "Splitting Prompt Prefill from Response Replay ...":
//   Sec. 2.2  attention as Q-KV block interactions with an online softmax state;
//   Sec. 3.2  prefill: causal over the prompt; replay, Eq. 1: a response row sees
//             every prompt key of its group and its own branch's keys up to itself;
//             Eq. 2: the prompt K/V gradient is summed over all branches;
//   Sec. 3.3  the prompt part and the own-branch part of a row's softmax are merged
//             as partial states (here inside one running online softmax).
//
// Tiles: 64 query rows x 64 keys; 256 threads; 4 threads share a row.
#include <cmath>

#include "common.cuh"

namespace augtree {
namespace {

constexpr int SB = 64;        // tile edge (rows and keys)
constexpr int SIMT_THREADS = 256;

template <int D>
struct SimtFwdSmem {
  float q[SB][D + 1];
  float k[SB][D + 1];
  float v[SB][D + 1];
  float p[SB][SB + 1];
};

template <typename T, int D>
__device__ void load_rows(float (*dst)[D + 1], const T* __restrict__ src, int64_t row0, int64_t row_end,
                          int heads, int head, float mul) {
  for (int idx = threadIdx.x; idx < SB * D; idx += SIMT_THREADS) {
    const int i = idx / D, c = idx % D;
    const int64_t row = row0 + i;
    float x = 0.f;
    if (row < row_end) x = to_f32(src[(row * heads + head) * D + c]) * mul;
    dst[i][c] = x;
  }
}

// One block per work item (PREFILL_Q or REPLAY_Q).
template <typename T, int D>
__global__ void __launch_bounds__(SIMT_THREADS) simt_fwd_kernel(
    Geometry geo, const int32_t* __restrict__ queue, int bm, int bn, const T* __restrict__ q,
    const T* __restrict__ kp, const T* __restrict__ vp, const T* __restrict__ kr, const T* __restrict__ vr,
    T* __restrict__ o, float* __restrict__ lse, int64_t lse_rows, uint32_t* __restrict__ err) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtFwdSmem<D>& sm = *reinterpret_cast<SimtFwdSmem<D>*>(smem_raw);
  const WorkItem it = load_item(queue, blockIdx.x);
  if (kChecked && !query_item_ok(it, geo, bm, bn)) {  // checked build only; block-uniform
    if (threadIdx.x == 0) atomicOr(err, kErrCheck);
    return;
  }
  const GroupInfo G = geo.groups[it.group];
  const int r = geo.hq / geo.hkv;
  const int h = it.head, kvh = h / r;
  const bool prefill = it.kind == K_PREFILL_Q;
  const int64_t base = prefill ? G.p0 : G.r0;
  const int64_t len = prefill ? G.lp : G.lr;
  const int64_t row0 = base + (int64_t)it.tile * bm;
  const int64_t row_end = min(row0 + bm, base + len);

  const int tid = threadIdx.x;
  const int my_row = tid >> 2, sub = tid & 3;
  const int64_t grow = row0 + my_row;
  const bool row_ok = grow < row_end;
  const int64_t my_bstart = (!prefill && row_ok) ? geo.row_bstart[grow] : 0;

  load_rows<T, D>(sm.q, q, row0, row_end, geo.hq, h, geo.scale_log2);

  float m = -INFINITY, l = 0.f;
  float acc[D / 4];
#pragma unroll
  for (int k = 0; k < D / 4; ++k) acc[k] = 0.f;

  const int n_prompt_tiles = it.a;
  const int n_own_tiles = prefill ? 0 : it.b;
  const int64_t own0 = prefill ? 0 : geo.row_bstart[row0];
  for (int t = 0; t < n_prompt_tiles + n_own_tiles; ++t) {
    const bool own = t >= n_prompt_tiles;
    const int64_t key0 = own ? own0 + (int64_t)(t - n_prompt_tiles) * bn : G.p0 + (int64_t)t * bn;
    const int64_t key_end = own ? (int64_t)G.r0 + G.lr : (int64_t)G.p0 + G.lp;
    const T* K = own ? kr : kp;
    const T* V = own ? vr : vp;
    __syncthreads();
    load_rows<T, D>(sm.k, K, key0, key_end, geo.hkv, kvh, 1.f);
    load_rows<T, D>(sm.v, V, key0, key_end, geo.hkv, kvh, 1.f);
    __syncthreads();
    float s[SB / 4];
    float tmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < SB / 4; ++j) {
      const int c = sub + 4 * j;
      const int64_t key = key0 + c;
      bool ok = row_ok && key < key_end;
      if (prefill) ok = ok && key <= grow;
      else if (own) ok = ok && key >= my_bstart && key <= grow;
      float x = -INFINITY;
      if (ok) {
        float a = 0.f;
#pragma unroll 8
        for (int d = 0; d < D; ++d) a = fmaf(sm.q[my_row][d], sm.k[c][d], a);
        x = a;
      }
      s[j] = x;
      tmax = fmaxf(tmax, x);
    }
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
    const float m_new = fmaxf(m, tmax);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = (m == -INFINITY) ? 0.f : exp2f(m - m_use);
    float psum = 0.f;
#pragma unroll
    for (int j = 0; j < SB / 4; ++j) {
      const float p = (s[j] == -INFINITY) ? 0.f : exp2f(s[j] - m_use);
      sm.p[my_row][sub + 4 * j] = p;
      psum += p;
    }
    psum += __shfl_xor_sync(0xffffffffu, psum, 1);
    psum += __shfl_xor_sync(0xffffffffu, psum, 2);
    l = l * alpha + psum;
    m = m_new;
    __syncwarp();
#pragma unroll
    for (int k = 0; k < D / 4; ++k) acc[k] *= alpha;
    for (int c = 0; c < SB; ++c) {
      const float p = sm.p[my_row][c];
#pragma unroll
      for (int k = 0; k < D / 4; ++k) acc[k] = fmaf(p, sm.v[c][sub + 4 * k], acc[k]);
    }
  }
  if (row_ok) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    T* dst = o + (grow * geo.hq + h) * D;
#pragma unroll
    for (int k = 0; k < D / 4; ++k) dst[sub + 4 * k] = from_f32<T>(acc[k] * inv);
    if (sub == 0) lse[(int64_t)h * lse_rows + grow] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
  }
}

template <int D>
struct SimtBwdSmem {
  float k[SB][D + 1];
  float v[SB][D + 1];
  float q[SB][D + 1];
  float dO[SB][D + 1];
  float p[SB][SB + 1];
  float ds[SB][SB + 1];
  float lse2[SB];
  float delta[SB];
};

// One block per KV work item (PROMPT_KV, RESP_KV or PREFILL_KV): the block keeps its
// 64 keys' dK/dV in registers and walks the query tiles [a, b) of every query head of
// its KV head; dQ contributions go to the fp32 accumulator with atomic adds.
template <typename T, int D>
__global__ void __launch_bounds__(SIMT_THREADS) simt_bwd_kernel(
    Geometry geo, const int32_t* __restrict__ queue, int bm, int bn, const T* __restrict__ q,
    const T* __restrict__ kp, const T* __restrict__ vp, const T* __restrict__ kr, const T* __restrict__ vr,
    const float* __restrict__ lse, const T* __restrict__ dO, const float* __restrict__ delta,
    float* __restrict__ dq_acc, T* __restrict__ dk_out, T* __restrict__ dv_out, float* __restrict__ dk_part,
    float* __restrict__ dv_part, float* __restrict__ dk_sum, float* __restrict__ dv_sum,
    const float* __restrict__ dk_add, const float* __restrict__ dv_add, uint32_t* __restrict__ err) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtBwdSmem<D>& sm = *reinterpret_cast<SimtBwdSmem<D>*>(smem_raw);
  const WorkItem it = load_item(queue, blockIdx.x);
  if (kChecked && !key_item_ok(it, geo, bm, bn)) {  // checked build only; block-uniform
    if (threadIdx.x == 0) atomicOr(err, kErrCheck);
    return;
  }
  const GroupInfo G = geo.groups[it.group];
  const int r = geo.hq / geo.hkv;
  const int kvh = it.head;
  const bool resp_keys = it.kind == K_RESP_KV;
  const bool prefill = it.kind == K_PREFILL_KV;
  const int64_t kbase = resp_keys ? G.r0 : G.p0;
  const int64_t klen = resp_keys ? G.lr : G.lp;
  const int64_t key0 = kbase + (int64_t)it.tile * bn;
  const int64_t key_end = min(key0 + bn, kbase + klen);
  const int64_t qbase = prefill ? G.p0 : G.r0;
  const int64_t qlen = prefill ? G.lp : G.lr;
  const int64_t q_rows_total = prefill ? geo.total_prompt : geo.total_resp;

  load_rows<T, D>(sm.k, resp_keys ? kr : kp, key0, key_end, geo.hkv, kvh, 1.f);
  load_rows<T, D>(sm.v, resp_keys ? vr : vp, key0, key_end, geo.hkv, kvh, 1.f);

  const int tid = threadIdx.x;
  const int mine = tid >> 2, sub = tid & 3;  // key row (dK/dV) or query row (scores, dQ)
  float dk[D / 4], dv[D / 4];
#pragma unroll
  for (int k = 0; k < D / 4; ++k) dk[k] = dv[k] = 0.f;

  for (int hh = 0; hh < r; ++hh) {
    const int h = kvh * r + hh;
    for (int qt = it.a; qt < it.b; ++qt) {
      const int64_t row0 = qbase + (int64_t)qt * bm;
      const int64_t row_end = min(row0 + bm, qbase + qlen);
      __syncthreads();
      load_rows<T, D>(sm.q, q, row0, row_end, geo.hq, h, 1.f);
      load_rows<T, D>(sm.dO, dO, row0, row_end, geo.hq, h, 1.f);
      if (tid < SB) {
        const int64_t row = row0 + tid;
        const bool ok = row < row_end;
        sm.lse2[tid] = ok ? lse[(int64_t)h * q_rows_total + row] * 1.4426950408889634f : 0.f;
        sm.delta[tid] = ok ? delta[(int64_t)h * q_rows_total + row] : 0.f;
      }
      __syncthreads();
      // scores / dS for query row `mine`, keys sub + 4j
      {
        const int64_t row = row0 + mine;
        const bool row_ok = row < row_end;
        const int64_t bs = (resp_keys && row_ok) ? geo.row_bstart[row] : 0;
#pragma unroll 1
        for (int j = 0; j < SB / 4; ++j) {
          const int c = sub + 4 * j;
          const int64_t key = key0 + c;
          bool ok = row_ok && key < key_end;
          if (prefill) ok = ok && key <= row;
          if (resp_keys) ok = ok && key >= bs && key <= row;
          float p = 0.f, ds = 0.f;
          if (ok) {
            float s = 0.f, dp = 0.f;
#pragma unroll 8
            for (int d = 0; d < D; ++d) {
              s = fmaf(sm.q[mine][d], sm.k[c][d], s);
              dp = fmaf(sm.dO[mine][d], sm.v[c][d], dp);
            }
            p = exp2f(s * geo.scale_log2 - sm.lse2[mine]);
            ds = p * (dp - sm.delta[mine]);
          }
          sm.p[mine][c] = p;
          sm.ds[mine][c] = ds;
        }
      }
      __syncthreads();
      // dV[key] += P^T dO ; dK[key] += dS^T Q   (key = mine)
      for (int i = 0; i < SB; ++i) {
        const float p = sm.p[i][mine], ds = sm.ds[i][mine];
#pragma unroll
        for (int k = 0; k < D / 4; ++k) {
          dv[k] = fmaf(p, sm.dO[i][sub + 4 * k], dv[k]);
          dk[k] = fmaf(ds, sm.q[i][sub + 4 * k], dk[k]);
        }
      }
      // dQ[row] += s dS K   (row = mine)
      {
        const int64_t row = row0 + mine;
        if (row < row_end) {
          float a[D / 4];
#pragma unroll
          for (int k = 0; k < D / 4; ++k) a[k] = 0.f;
          for (int c = 0; c < SB; ++c) {
            const float ds = sm.ds[mine][c];
#pragma unroll
            for (int k = 0; k < D / 4; ++k) a[k] = fmaf(ds, sm.k[c][sub + 4 * k], a[k]);
          }
          float* dst = dq_acc + (row * geo.hq + h) * D;
#pragma unroll
          for (int k = 0; k < D / 4; ++k) atomicAdd(dst + sub + 4 * k, a[k] * geo.scale);
        }
      }
    }
  }
  const int64_t key = key0 + mine;
  if (key >= key_end) return;
  const int64_t off = (key * geo.hkv + kvh) * D;
  if (it.kind == K_PROMPT_KV) {
    const SplitInfo s = geo.splits[it.group];
    float* tk = dk_sum;
    float* tv = dv_sum;
    int64_t o2 = off;
    if (s.nsplit > 1) {
      tk = dk_part;
      tv = dv_part;
      o2 = ((s.part_row0 + (int64_t)it.split * G.lp + (key - G.p0)) * geo.hkv + kvh) * D;
    }
#pragma unroll
    for (int k = 0; k < D / 4; ++k) {
      tk[o2 + sub + 4 * k] = dk[k] * geo.scale;
      tv[o2 + sub + 4 * k] = dv[k];
    }
  } else {
#pragma unroll
    for (int k = 0; k < D / 4; ++k) {
      float a = dk[k] * geo.scale, b = dv[k];
      if (dk_add) {
        a += dk_add[off + sub + 4 * k];
        b += dv_add[off + sub + 4 * k];
      }
      dk_out[off + sub + 4 * k] = from_f32<T>(a);
      dv_out[off + sub + 4 * k] = from_f32<T>(b);
    }
  }
}

template <typename T, int D>
cudaError_t fwd_launch(const augtree_plan* p, int op, const void* q, const void* kp, const void* vp, const void* kr,
                       const void* vr, void* o, float* lse, cudaStream_t st) {
  const size_t smem = sizeof(SimtFwdSmem<D>);
  cudaError_t e = cudaFuncSetAttribute(simt_fwd_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t rows = op == AUGTREE_OP_PREFILL_FWD ? p->total_prompt : p->total_resp;
  simt_fwd_kernel<T, D><<<(unsigned)p->n_items[op], SIMT_THREADS, smem, st>>>(
      geometry(p), p->queue_d[op], p->bm[op], p->bn[op], (const T*)q, (const T*)kp, (const T*)vp, (const T*)kr,
      (const T*)vr, (T*)o, lse, rows, p->err_d);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t bwd_launch(const augtree_plan* p, int op, const void* q, const void* kp, const void* vp, const void* kr,
                       const void* vr, const float* lse, const void* dO, const float* delta, float* dq_acc,
                       void* dk_out, void* dv_out, float* dk_part, float* dv_part, float* dk_sum, float* dv_sum,
                       const float* dk_add, const float* dv_add, cudaStream_t st) {
  const size_t smem = sizeof(SimtBwdSmem<D>);
  cudaError_t e = cudaFuncSetAttribute(simt_bwd_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  simt_bwd_kernel<T, D><<<(unsigned)p->n_items[op], SIMT_THREADS, smem, st>>>(
      geometry(p), p->queue_d[op], p->bm[op], p->bn[op], (const T*)q, (const T*)kp, (const T*)vp, (const T*)kr,
      (const T*)vr, lse, (const T*)dO, delta, dq_acc, (T*)dk_out, (T*)dv_out, dk_part, dv_part, dk_sum, dv_sum,
      dk_add, dv_add, p->err_d);
  return cudaGetLastError();
}

}  // namespace

cudaError_t simt_fwd(const augtree_plan* p, int op, const void* q, const void* kp, const void* vp, const void* kr,
                     const void* vr, void* o, float* lse, cudaStream_t st) {
  const bool bf = p->cfg.dtype == AUGTREE_BF16;
  if (p->cfg.head_dim == 64)
    return bf ? fwd_launch<__nv_bfloat16, 64>(p, op, q, kp, vp, kr, vr, o, lse, st)
              : fwd_launch<float, 64>(p, op, q, kp, vp, kr, vr, o, lse, st);
  return bf ? fwd_launch<__nv_bfloat16, 128>(p, op, q, kp, vp, kr, vr, o, lse, st)
            : fwd_launch<float, 128>(p, op, q, kp, vp, kr, vr, o, lse, st);
}

cudaError_t simt_bwd(const augtree_plan* p, int op, const void* q, const void* kp, const void* vp, const void* kr,
                     const void* vr, const float* lse, const void* dO, const float* delta, float* dq_acc,
                     void* dk_out, void* dv_out, float* dk_part, float* dv_part, float* dk_sum, float* dv_sum,
                     const float* dk_add, const float* dv_add, cudaStream_t st) {
  const bool bf = p->cfg.dtype == AUGTREE_BF16;
#define AUGTREE_BWD_ARGS p, op, q, kp, vp, kr, vr, lse, dO, delta, dq_acc, dk_out, dv_out, dk_part, dv_part, dk_sum, \
                         dv_sum, dk_add, dv_add, st
  if (p->cfg.head_dim == 64)
    return bf ? bwd_launch<__nv_bfloat16, 64>(AUGTREE_BWD_ARGS) : bwd_launch<float, 64>(AUGTREE_BWD_ARGS);
  return bf ? bwd_launch<__nv_bfloat16, 128>(AUGTREE_BWD_ARGS) : bwd_launch<float, 128>(AUGTREE_BWD_ARGS);
#undef AUGTREE_BWD_ARGS
}

}  // namespace augtree
