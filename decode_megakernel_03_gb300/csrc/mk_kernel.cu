// The interpreter's generic instantiations (head shape read at run time), and
// the lookup of the kernel a step runs.
#include "mk_interp.cuh"
#include "mk_kernels.h"
#include "mk_sched.h"

namespace mk {

const void* kernel_generic(int B) {
  switch (B) {
    case 1: return reinterpret_cast<const void*>(&interp_kernel<1, 0, 0, 0, 0>);
    case 2: return reinterpret_cast<const void*>(&interp_kernel<2, 0, 0, 0, 0>);
    case 4: return reinterpret_cast<const void*>(&interp_kernel<4, 0, 0, 0, 0>);
    case 8: return reinterpret_cast<const void*>(&interp_kernel<8, 0, 0, 0, 0>);
    default: return nullptr;
  }
}

const void* kernel_for(const Shape& s, bool generic) {
  if (!generic) {
    if (const void* f = kernel_fixed_a(s)) return f;
    if (const void* f = kernel_fixed_b(s)) return f;
  }
  return kernel_generic(s.B);
}

int misc_bytes() { return (int)sizeof(Misc); }

cudaError_t allow_max_smem(const void* fn, int optin) {
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
}

}  // namespace mk
