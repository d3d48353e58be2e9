// Interpreter instantiations specialised to a shape: one sequence with
// 64-dimensional heads and four q-heads per kv-head whose GEMV rows are all
// 2048 wide (the Llama-3.2-1B shape), or two q-heads per kv-head (the small
// test shape).
#include "mk_interp.cuh"
#include "mk_kernels.h"
#include "mk_sched.h"

namespace mk {

const void* kernel_fixed_a(const Shape& s) {
  if (s.B == 1 && s.D == 64 && s.G() == 4 && s.H == 2048 && s.QD() == 2048 && s.Fc() == 2048)
    return reinterpret_cast<const void*>(&interp_kernel<1, 64, 4, 2048, 0>);
  if (s.B == 1 && s.D == 64 && s.G() == 2) return reinterpret_cast<const void*>(&interp_kernel<1, 64, 2, 0, 0>);
  return nullptr;
}

}  // namespace mk
