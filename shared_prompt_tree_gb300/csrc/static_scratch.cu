// augtree_prefill_bwd_static: the prefill backward with its scratch memory in a
// fixed-size array that the library itself defines, for callers that cannot
// allocate device memory at call time.
//
// Who needs this: code that runs where cudaMalloc is off limits - inside a custom
// allocator or memory-pool callback (allocating there would recurse), in a host
// callback or a real-time loop that must not take the driver's allocation lock or risk
// an out-of-memory failure mid-step, or in an embedding framework that hands out
// only its own buffers for inputs and outputs.  Such a caller still passes every input
// and output; the plan must have been created beforehand (augtree_plan_create does
// allocate), and only the call itself allocates nothing.
//
// The scratch is the file-scope device array below, 64 MiB.  What it holds per prompt
// row and query head (the prefill backward's workspace layout):
//   tensor-core kernels: 8 bytes of row statistics {lse*log2(e), Delta} and 32 bytes of
//     the key side's extra-MMA rows, 40 bytes in all, plus 32 MiB of per-SM fp32 dK/dV
//     flush slots: prompt rows x query heads up to about 838,000;
//   SIMT kernels: Delta (4 bytes) and the fp32 dQ accumulator (4 * head_dim bytes), 516
//     bytes at head_dim 128 and 260 at 64: up to about 130,000 (resp. 258,000).
//
// Address lookup: in host code the array's name is a host-side stand-in, not a device
// address.  augtree_plan_create calls static_scratch_address() with the plan's device
// current and keeps the result in the plan, so the lookup (which loads this file's
// module and with it reserves the array on that device, under lazy module loading)
// happens at plan creation, and the entry point itself neither looks anything up nor
// allocates.  A plan is tied to its device and its context, so the address can never
// outlive the context it was taken in.
//
// Every GPU that loads this library's module reserves the array until the process
// exits.  All calls share it and it keeps the last call's contents; the call
// re-initializes everything it reads (row statistics are overwritten, the SIMT dQ
// accumulator is zeroed by the call's first kernel, and the flush slots are stored
// before they are added to), so nothing carries over between calls.  Calls that can
// overlap on the GPU (different streams without ordering between them) race on the
// array.
#include "internal.h"

static __device__ __align__(256) unsigned char g_prefill_bwd_scratch[augtree::kStaticScratchBytes];

namespace augtree {

// Device address of the array on the current device.
cudaError_t static_scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_prefill_bwd_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

}  // namespace augtree

extern "C" augtree_status augtree_prefill_bwd_static(const augtree_plan* plan, const void* qp, const void* kp,
                                                     const void* vp, const void* op, const float* lse_p,
                                                     const void* dop, const float* dkp_acc, const float* dvp_acc,
                                                     void* dqp, void* dkp, void* dvp, void* stream) {
  if (!plan) return AUGTREE_ERR_INVALID_ARG;
  size_t need = 0;
  augtree_status st = augtree_plan_workspace_bytes(plan, AUGTREE_OP_PREFILL_BWD, &need);
  if (st != AUGTREE_OK) return st;
  if (need > augtree::kStaticScratchBytes) return AUGTREE_ERR_WORKSPACE_TOO_SMALL;
  // Null when the lookup at plan creation failed (the device could not reserve it).
  if (!plan->static_scratch) return AUGTREE_ERR_CUDA;
  return augtree_prefill_bwd(plan, qp, kp, vp, op, lse_p, dop, dkp_acc, dvp_acc, dqp, dkp, dvp, plan->static_scratch,
                             augtree::kStaticScratchBytes, stream);
}
