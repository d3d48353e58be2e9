// Interpreter instantiations specialised to a head shape: one sequence with
// 128-dimensional heads and four q-heads per kv-head (the Llama-3.1-8B shape),
// and eight sequences with the Llama-3.2-1B head shape.
#include "mk_interp.cuh"
#include "mk_kernels.h"
#include "mk_sched.h"

namespace mk {

const void* kernel_fixed_b(const Shape& s) {
  if (s.B == 1 && s.D == 128 && s.G() == 4) return reinterpret_cast<const void*>(&interp_kernel<1, 128, 4, 0, 0>);
  if (s.B == 8 && s.D == 64 && s.G() == 4) return reinterpret_cast<const void*>(&interp_kernel<8, 64, 4, 0, 0>);
  return nullptr;
}

}  // namespace mk
