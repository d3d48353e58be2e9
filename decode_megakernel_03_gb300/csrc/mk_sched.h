// Host scheduler: turns (model shape, batch, positions, SM count) into one
// pre-planned instruction queue per SM plus the counter targets
// ("3 · L'interpréteur sur GPU", §3.2: every SM receives a pre-planned
// sequence of instructions; §3.4: counters start at zero, producers bump them,
// consumers wait for a target).
#pragma once

#include <string>
#include <vector>

#include "mk_isa.h"

namespace mk {

struct Shape {
  int L, H, nh, nkv, D, F, V, B, S;
  int G() const { return nh / nkv; }
  int QD() const { return nh * D; }
  int Fc() const { return F / kChunks; }
  int pairs_per_group() const { return (G() + 2) * (D / 2); }
  int pairs() const { return nkv * pairs_per_group(); }
};

// Counter ids. Every counter counts produced items and is awaited at its full
// target, so its final value after a step equals the target.
struct CounterMap {
  int L, nkv, B;
  int xout(int l) const { return l; }                         // target H
  int omid(int l) const { return L + l; }                     // target H
  int qkv(int l, int g) const { return 2 * L + l * nkv + g; } // pairs per group
  int att(int l, int b, int g) const { return 2 * L + L * nkv + (l * B + b) * nkv + g; }
  int red(int l) const { return 2 * L + L * nkv + L * B * nkv + l; }   // B * nkv
  int hch(int l, int c) const { return 3 * L + L * nkv + L * B * nkv + l * kChunks + c; }
  int lm() const { return 3 * L + L * nkv + L * B * nkv + L * kChunks; }
  int dyn() const { return lm() + 1; }  // ticket counter of a dynamic LM head
  int count() const { return lm() + 2; }
};

struct Phase {                 // one kernel of the multi-launch build
  int op, layer;
  std::vector<Instr> instrs;   // SM-major
  std::vector<int> sm_off;     // n_sm + 1
};

struct Plan {
  int n_sm = 0;
  int parts[kMaxBatch] = {0};
  std::vector<Instr> instrs;   // SM-major, each SM in execution order
  std::vector<int> sm_off;     // n_sm + 1
  std::vector<int> targets;    // per counter
  std::vector<Phase> phases;   // multi-launch build, in launch order
};

// Validates a configuration; returns an empty string when supported.
std::string check_shape(const Shape& s);

// Split-KV partitions per sequence for these positions. Lengths are bucketed
// to multiples of 256 so that the plan (and its upload) changes rarely; the
// token range of each partition is recomputed on the device from the exact
// position.
void choose_partitions(const Shape& s, int n_sm, const int* positions, int* parts);

// One sequence: the O-projection reduces the attention partials while it
// stages its input (no reduction instruction between them). Every SM then
// reads all partitions of all heads (P x n_heads x head_dim floats), so
// beyond 2048 attention columns the separate reduction instruction is
// cheaper despite its extra hop (8B shape: 3520 -> 3478 us/step).
inline bool fused_reduction(const Shape& s) { return s.B == 1 && s.QD() <= 2048; }

// Several sequences, or rows wider than 2048 columns: the storers of the
// chunk-3 down-projection instructions write the layer output x whole
// (the interpreter's x_whole); otherwise its readers sum xa and the four
// down-projection shares.
inline bool x_written_whole(const Shape& s) { return s.B > 1 || s.H > 2048; }

// Items (rows or row pairs) per GEMV instruction, bounded by the result
// buffer the storer drains.
int item_cap_for(const Shape& s);

// dyn_flags: MK_DYN_* (0: every instruction a fixed work range)
bool build_plan(const Shape& s, int n_sm, const int* parts, Plan* out, std::string* why,
                int dyn_flags = 0);

// k greedy steps in one launch (1 <= k <= kMaxLaunchSteps): the plans of the
// steps (parts: k rows of kMaxBatch partition counts), each SM's queues
// concatenated in step order; instructions carry their step in the layer
// field, counters of step s are offset by s times the per-step count, and
// step s > 0's layer-0 QKV instructions wait for step s - 1's LM head (their
// token is its argmax). No multi-launch phases.
bool build_plan_steps(const Shape& s, int n_sm, const int* parts, int k, Plan* out,
                      std::string* why, int dyn_flags = 0);

// Shared-memory layout of the interpreter for this shape: fills the n_pages,
// off_*, *_floats and alias_xh fields of p and returns the dynamic shared
// memory size in bytes, or 0 (with *why set) when fewer than kComputeWarps
// pages fit in `optin` bytes. misc_bytes is the size of the kernel's barrier
// block.
int smem_layout(const Shape& s, int n_sm, int optin, int misc_bytes, Params* p, std::string* why);

}  // namespace mk
