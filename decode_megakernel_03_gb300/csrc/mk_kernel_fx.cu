// The interpreter's instantiations with the paged-KV-cache and greedy-decode
// code (feature bit kFxPaged): the generic ones, and those of the Llama-1B shape at batch 1
// and 8 and of the Llama-8B shape. Handles launch these only for paged caches
// and greedy decode; every other step runs a kernel without that code.
#include "mk_interp.cuh"
#include "mk_kernels.h"
#include "mk_sched.h"

namespace mk {

const void* kernel_features(const Shape& s) {
  if (s.B == 1 && s.D == 64 && s.G() == 4 && s.H == 2048 && s.QD() == 2048 && s.Fc() == 2048)
    return reinterpret_cast<const void*>(&interp_kernel<1, 64, 4, 2048, kFxPaged>);
  if (s.B == 8 && s.D == 64 && s.G() == 4) return reinterpret_cast<const void*>(&interp_kernel<8, 64, 4, 0, kFxPaged>);
  if (s.B == 1 && s.D == 128 && s.G() == 4) return reinterpret_cast<const void*>(&interp_kernel<1, 128, 4, 0, kFxPaged>);
  switch (s.B) {
    case 1: return reinterpret_cast<const void*>(&interp_kernel<1, 0, 0, 0, kFxPaged>);
    case 2: return reinterpret_cast<const void*>(&interp_kernel<2, 0, 0, 0, kFxPaged>);
    case 4: return reinterpret_cast<const void*>(&interp_kernel<4, 0, 0, 0, kFxPaged>);
    case 8: return reinterpret_cast<const void*>(&interp_kernel<8, 0, 0, 0, kFxPaged>);
    default: return nullptr;
  }
}

}  // namespace mk
