// Interpreter instantiations specialised to a head shape: one sequence with
// 64-dimensional heads, four or two q-heads per kv-head (the Llama-3.2-1B
// shape and the small test shape).
#include "mk_interp.cuh"
#include "mk_kernels.h"

namespace mk {

const void* kernel_fixed_a(int B, int D, int G) {
  if (B == 1 && D == 64 && G == 4) return reinterpret_cast<const void*>(&interp_kernel<1, 64, 4>);
  if (B == 1 && D == 64 && G == 2) return reinterpret_cast<const void*>(&interp_kernel<1, 64, 2>);
  return nullptr;
}

}  // namespace mk
