// The interpreter's instantiations with dynamic work distribution (feature
// bit kFxDyn): the LM head's row blocks taken from a per-step ticket counter.
// Only handles with a dynamic flag launch these (plain steps and the
// multi-launch build); every other step runs a kernel without that code.
#include "mk_interp.cuh"
#include "mk_kernels.h"
#include "mk_sched.h"

namespace mk {

const void* kernel_dynamic(const Shape& s) {
  if (s.B == 1 && s.D == 64 && s.G() == 4 && s.H == 2048 && s.QD() == 2048 && s.Fc() == 2048)
    return reinterpret_cast<const void*>(&interp_kernel<1, 64, 4, 2048, kFxDyn>);
  if (s.B == 8 && s.D == 64 && s.G() == 4) return reinterpret_cast<const void*>(&interp_kernel<8, 64, 4, 0, kFxDyn>);
  if (s.B == 1 && s.D == 128 && s.G() == 4) return reinterpret_cast<const void*>(&interp_kernel<1, 128, 4, 0, kFxDyn>);
  if (s.B == 1 && s.D == 64 && s.G() == 2) return reinterpret_cast<const void*>(&interp_kernel<1, 64, 2, 0, kFxDyn>);
  return nullptr;
}

}  // namespace mk
