// Interpreter instantiations specialised to a head shape: one sequence with
// 128-dimensional heads and four q-heads per kv-head (the Llama-3.1-8B shape),
// and eight sequences with the Llama-3.2-1B head shape.
#include "mk_interp.cuh"
#include "mk_kernels.h"

namespace mk {

const void* kernel_fixed_b(int B, int D, int G) {
  if (B == 1 && D == 128 && G == 4) return reinterpret_cast<const void*>(&interp_kernel<1, 128, 4>);
  if (B == 8 && D == 64 && G == 4) return reinterpret_cast<const void*>(&interp_kernel<8, 64, 4>);
  return nullptr;
}

}  // namespace mk
