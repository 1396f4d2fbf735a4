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
// The scratch (the backward's row statistics, the fp32 dQ accumulator [P, Hq, D] and,
// for the tensor-core kernels, 32 MiB of per-SM fp32 dK/dV flush slots) is the
// file-scope device array below, 64 MiB: enough for P * Hq up to about 60,000 at
// D = 128 with the tensor-core kernels (about 520 bytes per prompt row and query head).
// The first call on a device looks up the array's device address (cudaGetSymbolAddress,
// which may load this module); make that first call before any stream capture.  Every
// GPU that loads this library reserves the array until the process exits.  All calls share it and it keeps the last call's contents; the call
// re-initializes everything it reads (Delta is overwritten, the dQ accumulator is
// zeroed by the first kernel of the call), so nothing carries over between calls.
// Calls that can overlap on the GPU (different streams without ordering between them)
// race on the array.
#include <mutex>

#include "internal.h"

#define AUGTREE_STATIC_SCRATCH_BYTES (64ull << 20)

static __device__ __align__(256) unsigned char g_prefill_bwd_scratch[AUGTREE_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the array on device `dev` (which must be current).  In host code
// the array's name is only a host-side stand-in, so the address comes from the runtime.
cudaError_t scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_prefill_bwd_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" augtree_status augtree_prefill_bwd_static(const augtree_plan* plan, const void* qp, const void* kp,
                                                     const void* vp, const void* op, const float* lse_p,
                                                     const void* dop, const float* dkp_acc, const float* dvp_acc,
                                                     void* dqp, void* dkp, void* dvp, void* stream) {
  if (!plan) return AUGTREE_ERR_INVALID_ARG;
  size_t need = 0;
  augtree_status st = augtree_plan_workspace_bytes(plan, AUGTREE_OP_PREFILL_BWD, &need);
  if (st != AUGTREE_OK) return st;
  if (need > (size_t)AUGTREE_STATIC_SCRATCH_BYTES) return AUGTREE_ERR_WORKSPACE_TOO_SMALL;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return AUGTREE_ERR_CUDA;
  void* scratch = nullptr;
  if (scratch_address(dev, &scratch) != cudaSuccess) {
    cudaGetLastError();
    return AUGTREE_ERR_CUDA;
  }
  return augtree_prefill_bwd(plan, qp, kp, vp, op, lse_p, dop, dkp_acc, dvp_acc, dqp, dkp, dvp, scratch,
                             (size_t)AUGTREE_STATIC_SCRATCH_BYTES, stream);
}
