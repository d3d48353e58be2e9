// Entry points of the interpreter kernel's instantiations (host side).
#pragma once

#include <cuda_runtime_api.h>

namespace mk {

struct Shape;

// interp_kernel<B, DS, GS, KW, FX>: batch, head dimension (0: read at run
// time), q-heads per kv-head (0: run time), GEMV width (2048, or 0: any),
// and the feature bits FX: kFxPaged for the build with the paged-cache and
// greedy-decode code, kFxDyn for the one with the dynamic LM head.
// interp_kernel<B, 0, 0, 0, 0>: head dimension and q-heads per kv-head read at
// run time, any GEMV width (B = 1, 2, 4 or 8).
const void* kernel_generic(int B);
// Instantiations specialised to a model's shape, or nullptr when the shape
// has none in that translation unit.
const void* kernel_fixed_a(const Shape& s);
const void* kernel_fixed_b(const Shape& s);
// The kernel a step of this shape runs: the specialised one when there is
// one (unless `generic`), else the generic one.
const void* kernel_for(const Shape& s, bool generic);
// The instantiation with the paged-cache and greedy-decode code for this
// shape (specialised for the Llama-1B shape at batch 1 and 8 and the Llama-8B
// shape, else generic).
const void* kernel_features(const Shape& s);
// The instantiation with dynamic work distribution for this shape (the
// Llama-1B shape at batch 1 and 8, the Llama-8B shape, and one sequence with
// head_dim 64 and two q-heads per kv-head), or nullptr.
const void* kernel_dynamic(const Shape& s);
// Size of the kernel's shared-memory barrier block.
int misc_bytes();

// Lets `fn` launch with up to `optin` bytes of dynamic shared memory (the
// device's opt-in maximum). The limit is a property of the kernel function,
// shared by every handle and call that launches it, so it is always raised to
// the device maximum and never set to one shape's size: a smaller shape must
// not lower it under a larger one that launches the same function.
cudaError_t allow_max_smem(const void* fn, int optin);

}  // namespace mk
