// Memory-bound kernels of the path: the backward preprocess (Delta, the SIMT family's
// zeroed fp32 dQ accumulator, the tensor-core family's tiled row statistics), the dQ
// conversion, the merge's backward, the fixed-order split-K reduction of the prompt
// K/V gradient (Eq. 2), the partial-state merge of Sec. 3.3 (standalone, and the
// n-way merge of the replay forward's split-KV partials) and the split-KV dQ sum.
//
// AugTree paper, Sec. 3.2 (Eq. 2: the prompt K/V gradient is the sum over branches,
// aggregated exactly from all of them into the one prompt) and Sec. 3.3 (partial online-softmax
// states S = (m, l, O_acc) merge associatively; here in (O, lse) form).
#include <cmath>
#include <type_traits>

#include "common.cuh"

namespace augtree {
namespace {

// One warp per (row, head): Delta = sum_d dO * O in fp32; also zeroes the fp32 dQ
// accumulator row.  delta layout [Hq, rows].
template <typename T>
__global__ void preprocess_kernel(const T* __restrict__ o, const T* __restrict__ dO, int64_t rows, int hq, int d,
                                  float* __restrict__ delta, float* __restrict__ dq_acc) {
  const int64_t warp = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (warp >= rows * hq) return;
  const int64_t row = warp / hq;
  const int h = (int)(warp % hq);
  const int64_t base = warp * d;
  float acc = 0.f;
  for (int c = lane; c < d; c += 32) acc += to_f32(o[base + c]) * to_f32(dO[base + c]);
  acc = warp_sum(acc);
  if (lane == 0) delta[(int64_t)h * rows + row] = acc;
  for (int c = lane; c < d; c += 32) dq_acc[base + c] = 0.f;
}

// Rounds to bf16 (nearest even) and returns the bits.
__device__ __forceinline__ uint16_t bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
// x as hi + mid + lo, three bf16 values (the sum carries about 24 significant bits).
__device__ __forceinline__ uint4 split3_row(float x) {
  const uint16_t h = bf16_bits(x);
  const float r1 = x - __bfloat162float(__ushort_as_bfloat16(h));
  const uint16_t m = bf16_bits(r1);
  const float r2 = r1 - __bfloat162float(__ushort_as_bfloat16(m));
  const uint16_t l = bf16_bits(r2);
  return make_uint4((uint32_t)h | ((uint32_t)m << 16), (uint32_t)l, 0u, 0u);
}

// One block (4 warps) per (128-row query tile, head); tiles of all groups are numbered
// consecutively (GroupInfo::tp0 / tr0).  Writes
//   stats[h][tile] = {lse*log2e [128], Delta [128]}  (fp32, for the query-side kernel)
//   aug[h][tile]   = {L [128][8], D [128][8]}        (bf16, for the key-side kernel)
// where row r of L holds -lse/s and row r of D holds -Delta, each split into three
// bf16 values in columns 0-2 (columns 3-7 zero).  The key-side kernel multiplies these
// rows by a constant ones operand in one extra K=16 MMA step, so its accumulators hold
// S - lse/s and dP - Delta directly.  Rows past the group's end are zero.
__global__ void preprocess_tiled_kernel(const GroupInfo* __restrict__ groups, int n_groups, bool prompt_side,
                                        int ntiles, const __nv_bfloat16* __restrict__ o,
                                        const __nv_bfloat16* __restrict__ dO, const float* __restrict__ lse,
                                        int64_t rows_total, int hq, float inv_scale, float* __restrict__ stats,
                                        uint4* __restrict__ aug) {
  const int tile = blockIdx.x;
  const int h = blockIdx.y;
  // group holding this tile: last group whose first tile is <= tile and that has tiles
  int lo = 0, hi = n_groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    const int t0 = prompt_side ? groups[mid].tp0 : groups[mid].tr0;
    if (t0 <= tile) lo = mid; else hi = mid - 1;
  }
  const GroupInfo G = groups[lo];
  const int64_t base = prompt_side ? G.p0 : G.r0;
  const int64_t len = prompt_side ? G.lp : G.lr;
  const int64_t row0 = base + (int64_t)(tile - (prompt_side ? G.tp0 : G.tr0)) * kStatRows;
  const int64_t blk = (int64_t)h * ntiles + tile;
  float* out = stats + blk * 2 * kStatRows;
  uint4* aug_l = aug + blk * 2 * kStatRows;  // one 16-byte row per query row
  uint4* aug_d = aug_l + kStatRows;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = warp; r < kStatRows; r += 4) {
    const int64_t row = row0 + r;
    float dl = 0.f, l2 = 0.f, ln = 0.f;
    const bool valid = row < base + len;
    if (valid) {
      const int64_t off = (row * hq + h) * 128 + lane * 4;
      const uint2 a = *reinterpret_cast<const uint2*>(o + off);
      const uint2 b = *reinterpret_cast<const uint2*>(dO + off);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float2 x = __bfloat1622float2(a2[i]), y = __bfloat1622float2(b2[i]);
        acc += x.x * y.x + x.y * y.y;
      }
      dl = warp_sum(acc);
      ln = lse[(int64_t)h * rows_total + row];
      l2 = ln * 1.4426950408889634f;
    }
    if (lane == 0) {
      out[r] = l2;
      out[kStatRows + r] = dl;
      aug_l[r] = valid ? split3_row(-ln * inv_scale) : make_uint4(0u, 0u, 0u, 0u);
      aug_d[r] = valid ? split3_row(-dl) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
}


template <typename T>
__global__ void convert_kernel(const float* __restrict__ src, T* __restrict__ dst, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = from_f32<T>(src[i]);
}

// Per prompt row (one block per row, Hkv*D columns): groups with several splits sum
// their partials in ascending split order; groups without prompt-KV items (no
// responses) get zeros; single-split groups were written in place by the backward.
// Out = float: the replay sums (an unsplit group was written by the key side, a group
// with no prompt-KV items gets zeros).  Out = bf16: the fused backward's final prompt
// gradient, for split groups only (the key side wrote the others).
template <typename Out>
__global__ void split_reduce_kernel(const GroupInfo* __restrict__ groups, const SplitInfo* __restrict__ splits,
                                    int n_groups, int cols, const float* __restrict__ dk_part,
                                    const float* __restrict__ dv_part, Out* __restrict__ dk_sum,
                                    Out* __restrict__ dv_sum, int total_prompt) {
  constexpr bool kFinal = !std::is_same<Out, float>::value;
  const int row = blockIdx.x;
  if (row >= total_prompt) return;
  // group of this row: binary search over p0
  int lo = 0, hi = n_groups - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (groups[mid].p0 <= row) lo = mid; else hi = mid - 1;
  }
  // skip empty groups that share p0 with the holder
  int g = lo;
  while (g > 0 && groups[g].lp == 0) --g;
  while (g < n_groups && !(groups[g].p0 <= row && row < groups[g].p0 + groups[g].lp)) ++g;
  if (g >= n_groups) return;
  const SplitInfo s = splits[g];
  const int64_t out = (int64_t)row * cols;
  if (s.nsplit == 1 || (kFinal && s.nsplit == 0)) return;
  if (s.nsplit == 0) {
    for (int c = threadIdx.x; c < cols; c += blockDim.x) {
      dk_sum[out + c] = Out(0.f);
      dv_sum[out + c] = Out(0.f);
    }
    return;
  }
  const int lp = groups[g].lp;
  const int64_t local = row - groups[g].p0;
  for (int c = threadIdx.x; c < cols; c += blockDim.x) {
    float ak = 0.f, av = 0.f;
    for (int k = 0; k < s.nsplit; ++k) {
      const int64_t pr = (s.part_row0 + (int64_t)k * lp + local) * cols + c;
      ak += dk_part[pr];
      av += dv_part[pr];
    }
    if constexpr (kFinal) {
      dk_sum[out + c] = __float2bfloat16_rn(ak);
      dv_sum[out + c] = __float2bfloat16_rn(av);
    } else {
      dk_sum[out + c] = ak;
      dv_sum[out + c] = av;
    }
  }
}

// Replay forward split-KV: one warp per (row, head) of a split query tile (block
// (tile, head, group of 8 rows)), four head dimensions per lane (D = 128).  The tile's
// nsplit <= 64 partial states (O_k = O over the chunk's keys / l_k, lse_k) merge as the
// n-way form of the state merge (+) of Sec. 3.3: lse = log sum_k exp(lse_k),
// O = sum_k exp(lse_k - lse) O_k, summed in ascending split order (deterministic).
// Lane k holds lse_k and lse_{k+32}; the weights reach every lane by shuffles.  A row
// whose splits all saw no valid key gets O = 0 and lse = -inf.
__global__ void fwd_split_merge_kernel(const GroupInfo* __restrict__ groups, const FwdSplit* __restrict__ fsplit,
                                       const int32_t* __restrict__ tiles, int hq, const float* __restrict__ part_o,
                                       const float* __restrict__ part_lse, __nv_bfloat16* __restrict__ o,
                                       float* __restrict__ lse, int64_t total_resp) {
  const GroupInfo G = groups[tiles[2 * blockIdx.x]];
  const int t = tiles[2 * blockIdx.x + 1];
  const FwdSplit fs = fsplit[G.tr0 + t];
  const int h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.z * (blockDim.x >> 5) + warp;
  const int64_t row0 = (int64_t)G.r0 + (int64_t)t * kFwdPartRows;
  if (r >= kFwdPartRows || row0 + r >= (int64_t)G.r0 + G.lr) return;
  const int64_t slot0 = fs.slot0 + (int64_t)h * fs.nsplit;
  const int n = fs.nsplit;
  const float l0 = lane < n ? part_lse[(slot0 + lane) * kFwdPartRows + r] : -INFINITY;
  const float l1 = lane + 32 < n ? part_lse[(slot0 + lane + 32) * kFwdPartRows + r] : -INFINITY;
  const float m = warp_max(fmaxf(l0, l1));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float out_lse = -INFINITY;
  if (m != -INFINITY) {
    const float s = warp_sum((l0 == -INFINITY ? 0.f : expf(l0 - m)) + (l1 == -INFINITY ? 0.f : expf(l1 - m)));
    out_lse = m + logf(s);
    const float w0 = l0 == -INFINITY ? 0.f : expf(l0 - out_lse);
    const float w1 = l1 == -INFINITY ? 0.f : expf(l1 - out_lse);
    const float* src = part_o + (slot0 * kFwdPartRows + r) * 128 + lane * 4;
    const int64_t step = (int64_t)kFwdPartRows * 128;
#pragma unroll 4
    for (int k = 0; k < n; ++k) {
      const float w = __shfl_sync(0xffffffffu, k < 32 ? w0 : w1, k & 31);
      const float4 x = *reinterpret_cast<const float4*>(src + k * step);
      acc.x = fmaf(w, x.x, acc.x);
      acc.y = fmaf(w, x.y, acc.y);
      acc.z = fmaf(w, x.z, acc.z);
      acc.w = fmaf(w, x.w, acc.w);
    }
  }
  const int64_t row = row0 + r;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(o + (row * hq + h) * 128 + lane * 4) = pk;
  if (lane == 0) lse[(int64_t)h * total_resp + row] = out_lse;
}

// Replay query-side backward split-KV: dQ of a split tile's row is the sum of its
// splits' fp32 partials, in ascending split order; one warp per (row, head), blocks as
// in the merge.
__global__ void dq_split_reduce_kernel(const GroupInfo* __restrict__ groups, const FwdSplit* __restrict__ fsplit,
                                       const int32_t* __restrict__ tiles, int hq, const float* __restrict__ dq_part,
                                       __nv_bfloat16* __restrict__ dq) {
  const GroupInfo G = groups[tiles[2 * blockIdx.x]];
  const int t = tiles[2 * blockIdx.x + 1];
  const FwdSplit fs = fsplit[G.tr0 + t];
  const int h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.z * (blockDim.x >> 5) + warp;
  const int64_t row0 = (int64_t)G.r0 + (int64_t)t * kFwdPartRows;
  if (r >= kFwdPartRows || row0 + r >= (int64_t)G.r0 + G.lr) return;
  const int64_t slot0 = fs.slot0 + (int64_t)h * fs.nsplit;
  const float* src = dq_part + (slot0 * kFwdPartRows + r) * 128 + lane * 4;
  const int64_t step = (int64_t)kFwdPartRows * 128;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int k = 0; k < fs.nsplit; ++k) {
    const float4 x = *reinterpret_cast<const float4*>(src + k * step);
    acc.x += x.x;
    acc.y += x.y;
    acc.z += x.z;
    acc.w += x.w;
  }
  const int64_t row = row0 + r;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(dq + (row * hq + h) * 128 + lane * 4) = pk;
}

// (O, lse) merge, one thread per (row, head) pair looping over d.
__global__ void lse_merge_kernel(int64_t rows, int h, int d, const float* __restrict__ oa,
                                 const float* __restrict__ la, const float* __restrict__ ob,
                                 const float* __restrict__ lb, float* __restrict__ o, float* __restrict__ l) {
  const int64_t warp = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (warp >= rows * h) return;
  const int64_t row = warp / h;
  const int head = (int)(warp % h);
  const int64_t li = (int64_t)head * rows + row;
  const float a = la[li], b = lb[li];
  const float m = fmaxf(a, b);
  float wa = 0.f, wb = 0.f, lse = -INFINITY;
  if (m != -INFINITY) {
    const float ea = (a == -INFINITY) ? 0.f : expf(a - m);
    const float eb = (b == -INFINITY) ? 0.f : expf(b - m);
    const float s = ea + eb;
    lse = m + logf(s);
    wa = ea / s;
    wb = eb / s;
  }
  const int64_t base = warp * d;
  for (int c = lane; c < d; c += 32) {
    const float x = oa[base + c], y = ob[base + c];
    o[base + c] = wa * x + wb * y;
  }
  __syncwarp();
  if (lane == 0) l[li] = lse;
}

// Backward of the state merge: one warp per (row, head).  With w_a = e^(lse_a - lse),
// w_b = e^(lse_b - lse): doa = w_a do, dob = w_b do,
// dlse_a = w_a w_b <do, oa - ob> + w_a dlse, dlse_b = w_a w_b <do, ob - oa> + w_b dlse.
__global__ void lse_merge_bwd_kernel(int64_t rows, int h, int d, const float* __restrict__ oa,
                                     const float* __restrict__ la, const float* __restrict__ ob,
                                     const float* __restrict__ lb, const float* __restrict__ dout,
                                     const float* __restrict__ dl, float* __restrict__ doa,
                                     float* __restrict__ dla, float* __restrict__ dob, float* __restrict__ dlb) {
  const int64_t warp = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (warp >= rows * h) return;
  const int64_t row = warp / h;
  const int head = (int)(warp % h);
  const int64_t li = (int64_t)head * rows + row;
  const float a = la[li], b = lb[li];
  const float m = fmaxf(a, b);
  float wa = 0.f, wb = 0.f;
  if (m != -INFINITY) {
    const float ea = (a == -INFINITY) ? 0.f : expf(a - m);
    const float eb = (b == -INFINITY) ? 0.f : expf(b - m);
    const float s = ea + eb;
    wa = ea / s;
    wb = eb / s;
  }
  const int64_t base = warp * d;
  float sa = 0.f, sb = 0.f;
  for (int c = lane; c < d; c += 32) {
    const float g = dout[base + c];
    sa = fmaf(g, oa[base + c], sa);
    sb = fmaf(g, ob[base + c], sb);
    doa[base + c] = wa * g;
    dob[base + c] = wb * g;
  }
  sa = warp_sum(sa);
  sb = warp_sum(sb);
  if (lane == 0) {
    const float g = dl ? dl[li] : 0.f;
    const float ww = wa * wb;
    dla[li] = ww * (sa - sb) + wa * g;
    dlb[li] = ww * (sb - sa) + wb * g;
  }
}

}  // namespace

cudaError_t launch_preprocess(const void* o, const void* dO, int dtype, int64_t rows, int hq, int d, float* delta,
                              float* dq_acc, cudaStream_t st) {
  const int64_t warps = rows * hq;
  if (warps == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (warps + 7) / 8;
  if (dtype == AUGTREE_BF16)
    preprocess_kernel<__nv_bfloat16><<<(unsigned)blocks, threads, 0, st>>>(
        (const __nv_bfloat16*)o, (const __nv_bfloat16*)dO, rows, hq, d, delta, dq_acc);
  else
    preprocess_kernel<float><<<(unsigned)blocks, threads, 0, st>>>((const float*)o, (const float*)dO, rows, hq, d,
                                                                   delta, dq_acc);
  return cudaGetLastError();
}

cudaError_t launch_preprocess_tiled(const augtree_plan* p, bool prompt_side, const void* o, const void* dO,
                                    const float* lse, float* stats, void* aug, cudaStream_t st) {
  const int ntiles = prompt_side ? p->ntiles_p : p->ntiles_r;
  if (ntiles == 0) return cudaSuccess;
  dim3 grid(ntiles, p->cfg.hq);
  preprocess_tiled_kernel<<<grid, 128, 0, st>>>(p->groups_d, p->n_groups, prompt_side, ntiles,
                                                (const __nv_bfloat16*)o, (const __nv_bfloat16*)dO, lse,
                                                prompt_side ? p->total_prompt : p->total_resp, p->cfg.hq,
                                                1.0f / geometry(p).scale, stats, (uint4*)aug);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const float* dq_acc, void* dq, int dtype, int64_t n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (n + threads - 1) / threads;
  if (blocks > 152 * 32) blocks = 152 * 32;
  if (dtype == AUGTREE_BF16)
    convert_kernel<__nv_bfloat16><<<(unsigned)blocks, threads, 0, st>>>(dq_acc, (__nv_bfloat16*)dq, n);
  else
    convert_kernel<float><<<(unsigned)blocks, threads, 0, st>>>(dq_acc, (float*)dq, n);
  return cudaGetLastError();
}

cudaError_t launch_split_reduce(const augtree_plan* p, const float* dk_part, const float* dv_part, float* dk_sum,
                                float* dv_sum, cudaStream_t st) {
  if (p->total_prompt == 0 || p->n_groups == 0) return cudaSuccess;
  const int cols = p->cfg.hkv * p->cfg.head_dim;
  split_reduce_kernel<float><<<p->total_prompt, 256, 0, st>>>(p->groups_d, p->splits_d, p->n_groups, cols, dk_part,
                                                              dv_part, dk_sum, dv_sum, p->total_prompt);
  return cudaGetLastError();
}

cudaError_t launch_split_reduce_final(const augtree_plan* p, const float* dk_part, const float* dv_part, void* dkp,
                                      void* dvp, cudaStream_t st) {
  if (p->total_prompt == 0 || p->n_groups == 0 || p->part_rows == 0) return cudaSuccess;
  const int cols = p->cfg.hkv * p->cfg.head_dim;
  split_reduce_kernel<__nv_bfloat16><<<p->total_prompt, 256, 0, st>>>(
      p->groups_d, p->splits_d, p->n_groups, cols, dk_part, dv_part, (__nv_bfloat16*)dkp, (__nv_bfloat16*)dvp,
      p->total_prompt);
  return cudaGetLastError();
}

cudaError_t launch_fwd_split_merge(const augtree_plan* p, const float* part_o, const float* part_lse, void* o,
                                   float* lse, cudaStream_t st) {
  const size_t n_tiles = p->fsplit_tiles_h.size() / 2;
  if (n_tiles == 0) return cudaSuccess;
  if (p->cfg.head_dim != 128 || !part_o || !part_lse) return cudaErrorInvalidValue;
  dim3 grid((unsigned)n_tiles, p->cfg.hq, kFwdPartRows / 8);
  fwd_split_merge_kernel<<<grid, 256, 0, st>>>(p->groups_d, p->fsplit_d, p->fsplit_tiles_d, p->cfg.hq, part_o,
                                               part_lse, (__nv_bfloat16*)o, lse, p->total_resp);
  return cudaGetLastError();
}

cudaError_t launch_dq_split_reduce(const augtree_plan* p, const float* dq_part, void* dq, cudaStream_t st) {
  const size_t n_tiles = p->fsplit_tiles_h.size() / 2;
  if (n_tiles == 0) return cudaSuccess;
  if (p->cfg.head_dim != 128 || !dq_part) return cudaErrorInvalidValue;
  dim3 grid((unsigned)n_tiles, p->cfg.hq, kFwdPartRows / 8);
  dq_split_reduce_kernel<<<grid, 256, 0, st>>>(p->groups_d, p->fsplit_d, p->fsplit_tiles_d, p->cfg.hq, dq_part,
                                               (__nv_bfloat16*)dq);
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(int64_t rows, int h, int d, const float* oa, const float* la, const float* ob,
                             const float* lb, float* o, float* l, cudaStream_t st) {
  const int64_t warps = rows * h;
  const int64_t blocks = (warps + 7) / 8;
  lse_merge_kernel<<<(unsigned)blocks, 256, 0, st>>>(rows, h, d, oa, la, ob, lb, o, l);
  return cudaGetLastError();
}

}  // namespace augtree

namespace augtree {
cudaError_t launch_lse_merge_bwd(int64_t rows, int h, int d, const float* oa, const float* la, const float* ob,
                                 const float* lb, const float* dout, const float* dl, float* doa, float* dla,
                                 float* dob, float* dlb, cudaStream_t st) {
  const int64_t warps = rows * h;
  if (warps == 0) return cudaSuccess;
  const int64_t blocks = (warps + 7) / 8;
  lse_merge_bwd_kernel<<<(unsigned)blocks, 256, 0, st>>>(rows, h, d, oa, la, ob, lb, dout, dl, doa, dla, dob, dlb);
  return cudaGetLastError();
}
}  // namespace augtree
