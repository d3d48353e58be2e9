// Instruction set and kernel parameters of the decode interpreter, shared by
// the host scheduler and the device code (plain C++ structs, no CUDA types).
//
// The interpreter follows "3 · L'interpréteur sur GPU": every SM runs a
// pre-planned queue of fused instructions (§3.2), weights stream through
// 16 KB shared-memory pages (§3.3), and dependencies are global counters that
// start at zero and are bumped by producers and awaited by consumers (§3.4).
#pragma once

#include <stdint.h>
#include <vector_types.h>  // float2 (a plain C header of the CUDA toolkit)

#include "mk.h"  // include/ is on the include path

namespace mk {

constexpr int kPageBytes = 16384;   // one shared-memory page (§3.3: 16 KB pages)
constexpr int kComputeWarps = 6;    // warps in the compute role (8 warps per CTA: 255 registers each)
constexpr int kThreads = (kComputeWarps + 2) * 32;  // + loader warp + storer warp
// Warp w runs on SM sub-partition w % 4. The loader and the storer share
// sub-partition 2 so that no compute warp competes with the loader for issue
// slots; the six compute warps fill sub-partitions 0, 1 and 3.
constexpr int kLoaderWarp = 2;
constexpr int kStorerWarp = 6;
constexpr int kMaxBatch = 8;
constexpr int kMaxPartitions = 64;  // split-KV partitions per (sequence, kv-head)
constexpr int kChunks = 4;          // MLP hidden state chunks (§3.4: four pieces)
constexpr int kMaxPages = 14;
constexpr int kMaxLayers = 64;    // the layer table travels in the kernel parameters
constexpr int kResBufs = 4;      // result hand-offs in flight between compute and storer

using Instr = mk_instr;
static_assert(sizeof(Instr) == 32, "instruction descriptor is 32 bytes");

// Per-layer weight and cache pointers (they travel in the kernel parameters).
struct LayerPtrs {
  const uint16_t* attn_norm;
  const uint16_t* wq;
  const uint16_t* wk;
  const uint16_t* wv;
  const uint16_t* wo;
  const uint16_t* mlp_norm;
  const uint16_t* wgate;
  const uint16_t* wup;
  const uint16_t* wdown;
  uint16_t* kc;  // [B][nkv][S][D]
  uint16_t* vc;
};

// Everything a launch needs, passed by value.
struct Params {
  // model
  int L, H, nh, nkv, D, F, V, B, S, G, Fc, QD;  // QD = nh * D
  float eps;
  LayerPtrs layers[kMaxLayers]; // per-layer pointers (constant bank: no global load)
  const uint16_t* embed;
  const uint16_t* lm;          // == embed when tied
  const uint16_t* final_norm;
  const float2* rope;          // [S][D/2] (cos, sin) of pos * theta^(-2i/D)
  // library scratch (fp32 activations). The buffers marked "stamped" hand
  // values from one instruction to another within a step: the lowest
  // mantissa bit of every word carries the step's stamp (see stamp below).
  float* xa;     // [B][H] residual after the attention block (stamped)
  float* q;      // [B][nh*D] rotated queries (stamped)
  float* kvn;    // [B][nkv][2][D] this step's k (0) and v (1) rows as they
                 // were appended to the cache: bf16 bits << 16 | stamp
  float* part;   // [B][nh][kMaxPartitions][D] attention partials: o
  float* part_ml; // [B][nh][kMaxPartitions][2] attention partials: (m, l)
  float* attn;   // [B][nh*D] reduced attention output (stamped)
  float* h;      // [B][F] SwiGLU hidden state (stamped)
  float* xpart;  // [kChunks][B][H] down-projection of each chunk of h (stamped)
  float* x;      // [B][H] the layer's output x = xa + xpart[0] + ... + xpart[3]
                 // (stamped). With several sequences, or rows wider than 2048
                 // columns, the storer of the row's chunk-3 instruction sums it
                 // (its own share in place of xpart[3]) and writes it here;
                 // otherwise every reader sums the five sources itself
  // stamp of layer 0 of step 0 of this launch (0 or 1); layer l of step s
  // stamps with (stamp + s * L + l) & 1. Every stamped word is written
  // exactly once per layer, so before a layer's write it holds the previous
  // layer's stamp and a reader can tell the two apart word by word.
  unsigned stamp;
  float* logits; // [B][V] caller-owned
  int* ctr;      // counters of this step (zero at launch)
  int* ctr_zero; // counters of the next step, zeroed by this launch
  int n_ctr;
  int* err;      // device error word (0 = fine)
  int* err_host; // mapped pinned host mirror of the error word (may be null)
  const Instr* instrs;
  const int* sm_off;           // [gridDim.x + 1]
  mk_trace_record* trace;
  int trace_cap;
  int trace_base;              // record index of instrs[0] for this launch
  unsigned long long timeout_ns;
  int no_waits;                // multi-launch build: kernel boundaries order the work
  // shared-memory layout (bytes from the dynamic smem base)
  int n_pages;
  int off_x, off_h, off_res, off_misc;
  int x_floats, h_floats, res_floats;
  int alias_xh;                // x and h staging share one buffer
  int fused_red;               // one sequence: the O-projection's staging reduces the
                               // attention partials itself (no reduction instruction)
  // paged KV cache (block_table null: each layer's cache is [B][nkv][S][D]):
  // each layer's pool is [n_blocks][nkv][kv_block][D]; position t of
  // sequence b lives in block block_table[b * max_blocks + t / kv_block]
  const int* block_table;
  int max_blocks, kv_block;
  // greedy decode (both may be null): the previous step's argmax keys, read
  // as this step's tokens instead of tok[]; this step's argmax keys, raised
  // with atomicMax by the LM head (key = ordered(logit) << 32 | ~index, so the
  // largest logit wins and the lowest index among equal ones)
  const unsigned long long* tok_keys;
  unsigned long long* argmax_out;
  // several greedy steps in one launch (instructions carry their step,
  // layer = step << 10 | layer): step s > 0 reads its token from
  // argmax_out[(s - 1) * B + b]; counters of step s are offset by
  // s * n_ctr_step; lm_ctr is the LM head's counter of step 0
  int n_ctr_step, lm_ctr;
  // prefill: the B rows are consecutive tokens of ONE sequence (cache
  // sequence 0, positions pos[0] < pos[1] < ...), each attending causally
  // to the keys before it, the chunk's own included; the loader fetches an
  // attention unit's keys after the unit's counter (they may be this step's)
  int prefill;
  // per step
  int tok[kMaxBatch];
  int pos[kMaxBatch];
};

// Error word layout: code << 24 | where. Codes match MK_ERR_*.
constexpr int kErrTimeoutCounter = (MK_ERR_TIMEOUT << 24) | 1;
constexpr int kErrTimeoutPage = (MK_ERR_TIMEOUT << 24) | 2;
constexpr int kErrTimeoutRes = (MK_ERR_TIMEOUT << 24) | 3;
constexpr int kErrTimeoutStamp = (MK_ERR_TIMEOUT << 24) | 5;

// ---- geometry of the GEMV-shaped instructions -----------------------------
// A GEMV instruction walks "items": one weight row, or a pair of rows whose
// results are combined in the epilogue (q/k/v RoPE pairs, gate/up pairs).
// Each row contributes a K-long slice (the whole row, or one chunk of it).
// A page holds `ipp` items laid out [row kind r][item].
struct Geom {
  int K;      // columns of each row slice
  int R;      // rows per item (1 or 2)
  int ipp;    // items per page
};

#if defined(__CUDACC__)
#define MK_HD __host__ __device__ __forceinline__
#else
#define MK_HD inline
#endif

// layer and greedy step of an instruction (Instr::layer = step << 10 | layer)
constexpr int kStepShift = 10;
constexpr int kMaxLaunchSteps = 32;
MK_HD int layer_of(const Instr& in) { return in.layer & ((1 << kStepShift) - 1); }
MK_HD int step_of(const Instr& in) { return (in.layer >> kStepShift) & (kMaxLaunchSteps - 1); }

// token id of a greedy-decode argmax key (Params::argmax_out)
MK_HD int key_token(unsigned long long key) { return (int)(0xffffffffu - (uint32_t)key); }

MK_HD bool is_gemv(int op) {
  return op == MK_OP_QKV || op == MK_OP_OPROJ || op == MK_OP_GATEUP || op == MK_OP_DOWN ||
         op == MK_OP_LMHEAD;
}

MK_HD Geom geom_of(int op, int H, int QD, int Fc) {
  Geom g;
  g.K = (op == MK_OP_OPROJ) ? QD : (op == MK_OP_DOWN ? Fc : H);
  g.R = (op == MK_OP_QKV || op == MK_OP_GATEUP) ? 2 : 1;
  g.ipp = kPageBytes / (g.R * g.K * 2);
  return g;
}

// One split-KV attention unit: keys [t0, t1) of the keys 0..pos of its
// sequence, partition pidx of P (the host picks P; the device recomputes the
// range from the exact position). The new key (pos), whose k/v row this step
// writes, is taken from the stamped copy the QKV instruction writes beside
// its cache append (Params::kvn); the other nc = |[t0, min(t1, pos))| keys
// are cached already and stream through shared-memory pages before the
// unit's inputs arrive, kpp keys per page: K rows in the page's first half,
// V rows in its second.
struct AttnSpan {
  int t0, t1;   // the unit's keys
  int nc;       // cached keys [t0, t0 + nc), all below pos
  int kpp;      // keys per page
  int npages;   // pages of cached keys
};

MK_HD AttnSpan attn_span(int pos, int pidx, int P, int D) {
  const int len = pos + 1;
  AttnSpan s;
  // 32-bit arithmetic (the host checks kv_capacity * kMaxPartitions < 2^31);
  // a 64-bit division would cost far more code and time
  s.t0 = pidx * len / P;
  s.t1 = (pidx + 1) * len / P;
  const int end = s.t1 < pos ? s.t1 : pos;
  s.nc = end > s.t0 ? end - s.t0 : 0;
  s.kpp = kPageBytes / (4 * D);
  s.npages = (s.nc + s.kpp - 1) / s.kpp;
  return s;
}

// q/k/v row pairs are numbered group-major: for kv-head g, the G q-heads of the
// group, then k-head g, then v-head g; inside a head, pair i holds rows i and
// i + D/2 (the rotate-half RoPE partners).
struct PairRows {
  int which;  // 0 = q, 1 = k, 2 = v
  int head;   // q-head or kv-head index
  int i;      // first dimension of the pair (second is i + D/2)
  int g;      // kv-head group
};

MK_HD PairRows pair_rows(int j, int G, int D) {
  int half = D / 2;
  int per_group = (G + 2) * half;
  PairRows p;
  p.g = j / per_group;
  int jj = j - p.g * per_group;
  int slot = jj / half;
  p.i = jj - slot * half;
  if (slot < G) {
    p.which = 0;
    p.head = p.g * G + slot;
  } else {
    p.which = slot - G + 1;
    p.head = p.g;
  }
  return p;
}

}  // namespace mk
