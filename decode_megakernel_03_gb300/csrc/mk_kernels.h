// Entry points of the interpreter kernel's instantiations (host side).
#pragma once

namespace mk {

// interp_kernel<B, 0, 0>: head dimension and q-heads per kv-head read at run
// time (B = 1, 2, 4 or 8).
const void* kernel_generic(int B);
// interp_kernel<B, D, G> specialised to a model's head shape, or nullptr when
// (B, D, G) has no specialisation in that translation unit.
const void* kernel_fixed_a(int B, int D, int G);
const void* kernel_fixed_b(int B, int D, int G);
// The kernel a step of this shape runs: the specialised one when there is
// one (unless `generic`), else the generic one.
const void* kernel_for(int B, int D, int G, bool generic);
// Size of the kernel's shared-memory barrier block.
int misc_bytes();

}  // namespace mk
