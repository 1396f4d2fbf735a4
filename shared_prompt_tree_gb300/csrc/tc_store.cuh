// Wide global stores of the tensor-core kernels' epilogues.
#pragma once

#include <stdint.h>

namespace augtree {
namespace tc {

// One 32-byte store of eight words (sm_100 and later); p must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* r) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(r[0]), "r"(r[1]), "r"(r[2]),
               "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

}  // namespace tc
}  // namespace augtree
