// The decode interpreter: one persistent CTA per SM walks its pre-planned
// instruction queue ("3 · L'interpréteur sur GPU", §3.2). Every instruction is
// split over three warp roles that walk the same queue independently:
//
//   loader  (1 warp)   streams the instruction's bf16 weight rows (and an
//                      attention unit's cached keys) into 16 KB shared-memory
//                      pages with bulk asynchronous copies; it waits for free
//                      pages, and for a counter only where a copy would read
//                      this launch's own writes, so the next instruction's
//                      weights load while the current one still waits or
//                      computes (§3.3, the page allocator);
//   compute (6 warps)  waits for the instruction's input (its counter, or for
//                      small stamped inputs the words themselves), stages the
//                      activations, and runs the dot products / attention;
//                      each page is handed back as soon as it has been read;
//   storer  (1 warp)   applies the epilogue (RoPE + KV append, residual adds,
//                      SiLU, the layer output), writes the outputs as stamped
//                      words and bumps the output counter (§3.4, counters in
//                      global memory): a scheduling hint without a fence, or
//                      a release where a reader reads plain words after an
//                      acquire (see "stamped hand-offs" below).
//
// The same kernel also serves the multi-launch comparison build: launched once
// per (layer, instruction type) with counter waits switched off, kernel
// boundaries order the work instead.
//
// Every wait (counter, page, result buffer, stamped word) is bounded by a
// %globaltimer deadline; on expiry the kernel records MK_ERR_TIMEOUT in the
// error word, the other CTAs notice it and all of them drain their copies
// and return.
//
// The kernel is a template over the batch B and, optionally, the head
// dimension DS and the q-heads per kv-head GS (0: read from the parameters
// at run time), and KW: 2048 when every GEMV row (hidden, n_heads*head_dim
// and ffn/4 columns) is 2048 wide, so only the full-page register path is
// compiled (0: any width). An interpreter that carries every attention variant is about
// twice the size of one specialised to its model's shape, and the SM's
// instruction cache cannot hold it: the code of the instructions that run
// together (loader, staging, pages, attention, epilogues) must fit, or the
// warps stall on instruction fetches that queue behind the weight stream.
// This header is included by the translation units that instantiate it.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mk_isa.h"
#include "mk_ptx.cuh"

namespace mk {

constexpr int kBtCache = 256;  // block-table entries of one attention unit (paged cache)
constexpr int kTk = 4;         // ticket slots between the loader and the compute warps and storer
constexpr int kFxPaged = 1;    // feature bit: paged KV cache and greedy decode
constexpr int kFxDyn = 2;      // feature bit: dynamic work distribution

struct Misc {
  uint64_t full[kMaxPages];
  uint64_t empty[kMaxPages];
  uint64_t res_full[kResBufs];
  uint64_t res_empty[kResBufs];
  uint64_t tk_full[kTk];   // dynamic instructions: the loader published a ticket
  uint64_t tk_empty[kTk];  // compute warp 0 and the storer have read it
  int tk[kTk];             // the tickets (-1: none left)
  int tk_cur[2];           // compute warp 0 passes each ticket to the other compute warps
  uint64_t bt_full;    // paged cache: the unit's block-table entries landed
  alignas(16) int bt[kBtCache];  // paged cache: a window of the block table (bulk-copy target)
  float red[2][kComputeWarps][kMaxBatch];  // RMSNorm partial sums, double-buffered
  int abort;
  int hold;       // queue index of the latency-critical instruction being computed (-1: none)
  int published;  // instructions the storer has published (queue order)
};

constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kBarCompute = 1;

// Index of this warp among the compute warps (all warps but loader and storer).
__device__ __forceinline__ int compute_warp() {
  const int w = threadIdx.x >> 5;
  return w < kLoaderWarp ? w : (w < kStorerWarp ? w - 1 : w - 2);
}
__device__ __forceinline__ int compute_tid() { return compute_warp() * 32 + (threadIdx.x & 31); }

__device__ __forceinline__ void compute_bar() { named_bar(kBarCompute, kComputeThreads); }
// the compute warps' barrier, returning whether any of their threads passed v
__device__ __forceinline__ bool compute_bar_or(bool v) {
  return named_bar_or(kBarCompute, kComputeThreads, v);
}

__device__ __forceinline__ bool aborted(const Misc* m) {
  return *reinterpret_cast<const volatile int*>(&m->abort) != 0;
}

__device__ __forceinline__ void raise_error(const Params& p, Misc* m, int code) {
  if (atomicCAS(p.err, 0, code) == 0 && p.err_host)
    *reinterpret_cast<volatile int*>(p.err_host) = code;  // lets the host see it without a sync
  *reinterpret_cast<volatile int*>(&m->abort) = 1;
}

// Bounded mbarrier wait. Returns false (without waiting) once the CTA aborts.
__device__ __forceinline__ bool wait_mbar(const Params& p, Misc* m, uint64_t* bar,
                                          uint32_t parity, int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15) == 0) {
      if (aborted(m)) return false;
      if (ld_volatile(p.err) != 0) {
        *reinterpret_cast<volatile int*>(&m->abort) = 1;
        return false;
      }
      if (globaltimer() - t0 > p.timeout_ns) {
        raise_error(p, m, code);
        return false;
      }
    }
  }
}

// The latency-critical instruction whose output still goes out behind a
// release fence: the attention unit (its partials are read as plain words
// after an acquire of its counter). While the compute warps run one, the
// loader issues no copy for a later instruction: the storer's release fence
// waits for the SM's bulk copies in flight, so with nothing new in flight it
// publishes sooner. The other hand-offs are stamped words and publish
// without a fence, so they need no hold.
__device__ __forceinline__ bool critical_op(const Instr& in) { return in.op == MK_OP_ATTN; }

// Loader: before issuing a copy for queue entry j, wait while an earlier
// critical instruction is computing and not yet published (bounded).
__device__ __forceinline__ bool hold_wait(const Params& p, Misc* m, int j) {
  const volatile int* vh = &m->hold;
  const volatile int* vp = &m->published;
  int h = *vh;
  if (h < 0 || j <= h || *vp > h) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    h = *vh;
    if (h < 0 || j <= h || *vp > h) return true;
    if ((it & 15) == 0) {
      if (aborted(m)) return false;
      if (ld_volatile(p.err) != 0) {
        *reinterpret_cast<volatile int*>(&m->abort) = 1;
        return false;
      }
      if (globaltimer() - t0 > p.timeout_ns) {
        raise_error(p, m, kErrTimeoutPage);
        return false;
      }
    }
  }
}

// Bounded wait for counter >= target (acquire). One thread polls.
__device__ __forceinline__ bool wait_counter(const Params& p, Misc* m, int ctr, int target) {
  const int* a = p.ctr + ctr;
  if (ld_acquire(a) >= target) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (ld_acquire(a) >= target) return true;
    if ((it & 7) == 0) {
      if (aborted(m)) return false;
      if (ld_volatile(p.err) != 0) {
        *reinterpret_cast<volatile int*>(&m->abort) = 1;
        return false;
      }
      if (globaltimer() - t0 > p.timeout_ns) {
        raise_error(p, m, kErrTimeoutCounter);
        return false;
      }
    }
  }
}

// ---- stamped hand-offs ------------------------------------------------------
// A value one instruction hands to another within a step (q, the new k/v
// rows, the attention output, xa, h, the down-projection shares, the layer
// output x where it is written whole) is an fp32
// word whose lowest mantissa bit holds a stamp, written with a relaxed
// store. Each such word is written exactly once per layer, and the stamp is
// the parity of its layer's index in the launch sequence (layer l of step s
// of a launch: stamp + s * L + l), so every write flips it: until a layer's
// write lands, the word holds the previous layer's stamp, and a reader
// checks the stamp of every word it loads and loads again if one is stale.
// The producer then needs no release fence, which would wait for its SM's
// weight copies in flight (about 2 us per hand-off); the counters stay as
// scheduling hints, bumped without a fence. A reader clears the stamp bit,
// so every value is used rounded toward zero to 22 mantissa bits whatever
// its stamp, and the results do not depend on it.

// the stamp of the words layer `layer` of step `step` of this launch writes
__device__ __forceinline__ uint32_t stamp_of(const Params& p, int step, int layer) {
  return (p.stamp + (uint32_t)step * (uint32_t)p.L + (uint32_t)layer) & 1u;
}

// Whether the layer output x is written whole by the storers of the chunk-3
// down-projection instructions (several sequences, or rows wider than 2048
// columns), or left as xa and four shares that every reader adds up (one
// sequence of 2048 columns: five sources still stage in two round trips,
// and the extra poll in the chunk-3 storer costs as much as it saves; and
// the multi-launch build, whose kernel boundaries leave nothing to poll).
// Both forms give the same bits: x = ((((xa + s0) + s1) + s2) + s3), each
// term and the sum rounded toward zero to 22 mantissa bits.
template <int B>
__device__ __forceinline__ bool x_whole(const Params& p) {
  return !p.no_waits && (B > 1 || p.H > 2048);
}

__device__ __forceinline__ float stamped(float v, uint32_t s) {
  return __uint_as_float((__float_as_uint(v) & ~1u) | s);
}

// A reader loads every word of a batch first, then tests the whole batch
// (stale*), and only when some word is stale takes the slow path that
// reloads the stale ones: a call between two loads would keep the compiler
// from issuing the second before the first returned.
__device__ __forceinline__ bool stale4(const float4& v, uint32_t s) {
  return (((__float_as_uint(v.x) ^ s) | (__float_as_uint(v.y) ^ s) | (__float_as_uint(v.z) ^ s) |
           (__float_as_uint(v.w) ^ s)) & 1u) != 0u;
}

__device__ __forceinline__ bool stale2(const float2& v, uint32_t s) {
  return (((__float_as_uint(v.x) ^ s) | (__float_as_uint(v.y) ^ s)) & 1u) != 0u;
}

__device__ __forceinline__ bool stale1(float v, uint32_t s) {
  return ((__float_as_uint(v) ^ s) & 1u) != 0u;
}

__device__ __forceinline__ float clear1(float v) { return __uint_as_float(__float_as_uint(v) & ~1u); }

__device__ __forceinline__ float4 clear4(const float4& v) {
  return make_float4(clear1(v.x), clear1(v.y), clear1(v.z), clear1(v.w));
}

// A batch of loads that found a stale word is loaded again, whole: no
// per-word slow path, so the batch's code appears once (after a counter
// wait it is almost never repeated, the counter being bumped after the words
// were stored; an instruction that polls its input words instead repeats it
// until they land). Whether to try again: false on an abort, an error raised by
// another CTA, or after the timeout (the step's results are then void).
static __device__ __noinline__ bool retry_stale(const Params& p, Misc* m, uint32_t& it,
                                                uint64_t& t0) {
  if (it++ == 0) {
    t0 = globaltimer();
    return true;
  }
  if ((it & 7) == 0) {
    if (aborted(m)) return false;
    if (ld_volatile(p.err) != 0) {
      *reinterpret_cast<volatile int*>(&m->abort) = 1;
      return false;
    }
    if (globaltimer() - t0 > p.timeout_ns) {
      raise_error(p, m, kErrTimeoutStamp);
      return false;
    }
  }
  return true;
}

// Instruction descriptors are read-only for the whole launch: two 16-byte
// loads through the non-coherent path. Every role fetches the next descriptor
// while it works on the current one, so no role stalls on a dependent global
// load at an instruction boundary.
__device__ __forceinline__ Instr load_instr(const Instr* q) {
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(q));
  const uint4 b = __ldg(reinterpret_cast<const uint4*>(q) + 1);
  Instr in;
  in.op = (int16_t)(a.x & 0xffffu);
  in.layer = (int16_t)(a.x >> 16);
  in.a0 = (int32_t)a.y;
  in.a1 = (int32_t)a.z;
  in.a2 = (int32_t)a.w;
  in.wait_ctr = (int32_t)b.x;
  in.wait_target = (int32_t)b.y;
  in.sig_ctr = (int32_t)b.z;
  in.sig_amount = (int32_t)b.w;
  return in;
}

// ---------------------------------------------------------------------------
// dynamic work distribution
// ---------------------------------------------------------------------------
// A dynamic instruction (the LM head with a2 > 0) is not a fixed row range:
// every SM's queue holds one, and the SMs take row blocks of a0 rows out of
// [0, a1) from a per-step ticket counter (counter a2 - 1, zero at launch)
// until none is left, so an SM that reaches the LM head early takes more of
// it ("3 · L'interpréteur sur GPU", §3.6: instructions distributed over the
// SMs dynamically). The loader takes each ticket (before it streams the
// block's rows) and publishes it through a small ring to the compute warps
// and the storer, which then run the block as a plain instruction.

// (compiled into the kernels with feature bit kFxDyn only)
__device__ __forceinline__ bool is_dyn(const Instr& in) { return in.op == MK_OP_LMHEAD && in.a2 > 0; }

// the plain instruction of ticket t of dynamic instruction `in`
__device__ __forceinline__ Instr dyn_item(const Instr& in, int t) {
  Instr it = in;
  it.a0 = t * in.a0;
  it.a1 = min(in.a1, it.a0 + in.a0);
  it.a2 = 0;
  it.sig_amount = it.a1 - it.a0;
  return it;
}

// Loader: the next ticket of `in` (-1: none left), published to the ring.
__device__ __forceinline__ int loader_ticket(const Params& p, Misc* m, const Instr& in,
                                             uint32_t& tk_n, bool& ok) {
  const int slot = (int)(tk_n % kTk);
  if (!wait_mbar(p, m, &m->tk_empty[slot], ((tk_n / kTk) & 1u) ^ 1u, kErrTimeoutRes)) {
    ok = false;
    return -1;
  }
  const int t = atomicAdd(p.ctr + in.a2 - 1, 1);
  const int v = (long)t * in.a0 < (long)in.a1 ? t : -1;
  *reinterpret_cast<volatile int*>(&m->tk[slot]) = v;
  mbar_arrive(&m->tk_full[slot]);  // release (CTA scope) of the ticket to its readers
  ++tk_n;
  return v;
}

// ---------------------------------------------------------------------------
// weight rows of a GEMV item
// ---------------------------------------------------------------------------

// The weight matrices of one instruction, read from the layer table once per
// instruction so that per-row addresses are pure arithmetic.
struct RowSrc {
  const uint16_t* w[3];
  int op, G, D, H, QD, F;
  // w[i] without a dynamically indexed array (which would live in local memory)
  __device__ __forceinline__ const uint16_t* at(int i) const {
    return i == 0 ? w[0] : (i == 1 ? w[1] : w[2]);
  }
};

__device__ __forceinline__ RowSrc row_src_of(const Params& p, const Instr& in) {
  RowSrc s;
  s.op = in.op;
  s.G = p.G;
  s.D = p.D;
  s.H = p.H;
  s.QD = p.QD;
  s.F = p.F;
  s.w[0] = s.w[1] = s.w[2] = nullptr;
  if (in.op == MK_OP_LMHEAD) {
    s.w[0] = p.lm;
    return s;
  }
  const LayerPtrs* L = p.layers + layer_of(in);
  switch (in.op) {
    case MK_OP_QKV: s.w[0] = L->wq; s.w[1] = L->wk; s.w[2] = L->wv; break;
    case MK_OP_OPROJ: s.w[0] = L->wo; break;
    case MK_OP_GATEUP: s.w[0] = L->wgate; s.w[1] = L->wup; break;
    default: s.w[0] = L->wdown + (size_t)in.a2 * p.Fc; break;  // MK_OP_DOWN: chunk a2
  }
  return s;
}

// element offset of key/value row t of (sequence b, kv-head g) in a layer's
// cache, contiguous or paged; rows of one block are contiguous
// FX: feature bits of the interpreter build (kernels without a feature carry
// none of its code: the instruction cache). kFxPaged: the paged-cache and
// greedy-decode code; kFxDyn: dynamic work distribution.
template <int FX>
__device__ __forceinline__ size_t kv_row(const Params& p, int b, int g, int t) {
  if (p.prefill) b = 0;  // every row of a prefill chunk is sequence 0
  if (!(FX & kFxPaged) || !p.block_table) return (((size_t)b * p.nkv + g) * (size_t)p.S + t) * p.D;
  const int blk = __ldg(p.block_table + b * p.max_blocks + t / p.kv_block);
  return (((size_t)blk * p.nkv + g) * p.kv_block + t % p.kv_block) * p.D;
}

// ---------------------------------------------------------------------------
// loader role
// ---------------------------------------------------------------------------

// Issues the bulk copies of one page: items [i0, i1) of the instruction, laid
// out [row kind r][item]. Rows are affine in the item (row = base + item *
// stride) except for q/k/v pairs, which are affine within one head; runs of
// rows that follow each other in memory go out as one copy.
__device__ __forceinline__ void issue_page(const Params& p, const Instr& in, const Geom& g,
                                           const RowSrc& rs, int i0, int i1, uint8_t* dst,
                                           uint64_t* bar, uint64_t pol) {
  const uint32_t row_bytes = (uint32_t)g.K * 2u;
  if (in.op == MK_OP_QKV) {
    // pair j holds rows (head*D + i, head*D + i + D/2); consecutive pairs of one
    // head are consecutive rows, so a page splits at most at head boundaries
    const int half = p.D / 2;
    for (int r = 0; r < 2; ++r) {
      int it = i0;
      while (it < i1) {
        const PairRows pr = pair_rows(in.a0 + it, p.G, p.D);
        const int n = min(i1 - it, half - pr.i);
        const uint16_t* src = rs.at(pr.which) + (size_t)(pr.head * p.D + pr.i + r * half) * p.H;
        bulk_g2s_hint(dst, src, row_bytes * (uint32_t)n, bar, pol);
        dst += row_bytes * (uint32_t)n;
        it += n;
      }
    }
    return;
  }
  // OPROJ / GATEUP / DOWN / LMHEAD: row of item j = w[r] + j * stride
  const size_t stride = in.op == MK_OP_OPROJ ? (size_t)p.QD : (in.op == MK_OP_DOWN ? (size_t)p.F : (size_t)p.H);
  for (int r = 0; r < g.R; ++r) {
    const uint16_t* src = rs.at(r) + (size_t)(in.a0 + i0) * stride;
    if (stride * 2 == row_bytes) {  // whole rows: one contiguous run
      bulk_g2s_hint(dst, src, row_bytes * (uint32_t)(i1 - i0), bar, pol);
      dst += row_bytes * (uint32_t)(i1 - i0);
    } else {  // row slices (down-projection chunks): one copy per row
      for (int it = i0; it < i1; ++it) {
        bulk_g2s_hint(dst, src, row_bytes, bar, pol);
        dst += row_bytes;
        src += stride;
      }
    }
  }
}

template <int FX>
static __device__ void loader_role(const Params& p, Misc* m, uint8_t* smem, const Instr* q, int n) {
  const int lane = threadIdx.x & 31;
  if (lane != 0) return;
  const uint64_t pol = policy_evict_first();
  uint32_t page_cnt = 0;  // pages issued
  int slot = 0;           // page_cnt % n_pages
  uint32_t round = 0;     // page_cnt / n_pages
  int acq_step = 0;       // greedy steps whose LM head this loader has acquired
  uint32_t bt_par = 0;    // parity of the next block-table copy
  bool bt_pending = false;  // a block-table copy was issued and has not been seen landing
  bool ok = true;
  // trace: when this instruction's first and last copies went out
  const int rec0 = p.trace_base + (int)(q - p.instrs);
  auto trace_issue = [&](int i, uint64_t t_first) {
    if (p.trace != nullptr && rec0 + i < p.trace_cap) {
      p.trace[rec0 + i].t_issue_first = t_first;
      p.trace[rec0 + i].t_issue_last = globaltimer();
    }
  };
  uint32_t tk_n = 0;      // tickets published (dynamic instructions)
  Instr nxt = n > 0 ? load_instr(q) : Instr{};
  Instr in0 = nxt;
  int adv = 1;  // 0 while a dynamic instruction still has tickets
  for (int i = 0; i < n && ok; i += adv) {
    if (adv) {
      in0 = nxt;
      if (i + 1 < n) nxt = load_instr(q + i + 1);
    }
    // a dynamic instruction is entered once per ticket it takes (the queue
    // index stays), a plain one once
    Instr in = in0;
    adv = 1;
    if ((FX & kFxDyn) && is_dyn(in0)) {
      const int t = loader_ticket(p, m, in0, tk_n, ok);
      if (t < 0) continue;  // none left (or an abort): the next entry
      in = dyn_item(in0, t);
      adv = 0;
    }
    uint64_t t_first = 0;
    if (in.op == MK_OP_ATTN) {
      // the unit's cached keys, K and V rows of kpp keys per page; they do
      // not depend on this step's outputs, so they stream in while the unit
      // still waits for its queries
      const AttnSpan sp = attn_span(p.pos[in.a0] + step_of(in), in.a2 >> 16, in.a2 & 0xffff, p.D);
      const LayerPtrs& L = p.layers[layer_of(in)];
      if constexpr ((FX & kFxPaged) != 0) {
        // keys written by an earlier step of this launch: every write of step
        // s - 1 is ordered before its LM head's count (and the bulk copies
        // below after this acquire)
        const int st = step_of(in);
        if (st > acq_step) {
          if (!p.no_waits &&
              !wait_counter(p, m, p.lm_ctr + (st - 1) * p.n_ctr_step, p.V)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
          acq_step = st;
        }
      }
      // prefill: the unit's keys include the chunk's own, which this step's
      // QKV instructions write: fetch them after the unit's counter (every
      // QKV instruction precedes this one in every SM's queue, so the wait
      // ends), then order the acquire before the bulk copies' reads
      if (p.prefill && !p.no_waits && sp.nc > 0) {
        if (!wait_counter(p, m, in.wait_ctr, in.wait_target)) {
          ok = false;
          break;
        }
        fence_proxy_async_global();
      }
      // paged cache: the table entries of the unit's cached keys, in one
      // bulk copy (a 16-byte aligned window of at most kBtCache entries;
      // every earlier page of this loader has been issued, so the slice is
      // not in use by a copy still going out)
      int bt_base = -1;
      if ((FX & kFxPaged) && p.block_table && sp.nc > 0) {
        const int e0 = in.a0 * p.max_blocks + sp.t0 / p.kv_block;
        const int e1 = in.a0 * p.max_blocks + (sp.t0 + sp.nc - 1) / p.kv_block;
        const int w0 = e0 & ~3;
        const int nw = (e1 + 1 - w0 + 3) & ~3;
        if (nw <= kBtCache) {
          // this thread's reads of the previous window are done; order them
          // before the copy's writes (generic then async proxy)
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          bt_pending = true;
          mbar_arrive_expect_tx(&m->bt_full, (uint32_t)nw * 4u);
          bulk_g2s(m->bt, p.block_table + w0, (uint32_t)nw * 4u, &m->bt_full);
          if (!wait_mbar(p, m, &m->bt_full, bt_par, kErrTimeoutPage)) {
            ok = false;
            break;
          }
          bt_pending = false;
          bt_par ^= 1u;
          bt_base = w0;
        }
      }
      for (int pg = 0; pg < sp.npages; ++pg) {
        if (!wait_mbar(p, m, &m->empty[slot], (round & 1u) ^ 1u, kErrTimeoutPage) ||
            !hold_wait(p, m, i)) {
          ok = false;
          break;
        }
        if (pg == 0 && p.trace != nullptr) t_first = globaltimer();
        const int k0 = sp.t0 + pg * sp.kpp;
        const int nk = min(sp.kpp, sp.nc - pg * sp.kpp);
        const uint32_t bytes = (uint32_t)nk * (uint32_t)p.D * 2u;
        uint8_t* dst = smem + (size_t)slot * kPageBytes;
        mbar_arrive_expect_tx(&m->full[slot], 2u * bytes);
        if (!(FX & kFxPaged) || !p.block_table) {
          // the page's keys are one contiguous run of the cache
          const size_t row = kv_row<FX>(p, in.a0, in.a1, k0);
          bulk_g2s_hint(dst, L.kc + row, bytes, &m->full[slot], pol);
          bulk_g2s_hint(dst + kPageBytes / 2, L.vc + row, bytes, &m->full[slot], pol);
        } else {
          // a paged cache: one copy per run of keys inside one block, its
          // block from the table slice in shared memory (or, for a unit
          // wider than the slice, from the table itself)
          const int* bt = p.block_table + (size_t)in.a0 * p.max_blocks;
          for (int t = k0, off = 0; t < k0 + nk;) {
            const int run = min(k0 + nk - t, p.kv_block - t % p.kv_block);
            const int e = in.a0 * p.max_blocks + t / p.kv_block - bt_base;
            const int blk = bt_base >= 0 && e < kBtCache ? m->bt[e] : __ldg(bt + t / p.kv_block);
            const size_t row = (((size_t)blk * p.nkv + in.a1) * p.kv_block + t % p.kv_block) * p.D;
            const uint32_t rb = (uint32_t)run * (uint32_t)p.D * 2u;
            bulk_g2s_hint(dst + off, L.kc + row, rb, &m->full[slot], pol);
            bulk_g2s_hint(dst + kPageBytes / 2 + off, L.vc + row, rb, &m->full[slot], pol);
            t += run;
            off += (int)rb;
          }
        }
        ++page_cnt;
        if (++slot == p.n_pages) {
          slot = 0;
          ++round;
        }
      }
      if (ok && sp.npages > 0) trace_issue(i, t_first);
      continue;
    }
    if (!is_gemv(in.op)) continue;
    const Geom g = geom_of(in.op, p.H, p.QD, p.Fc);
    const int items = in.a1 - in.a0;
    const uint32_t row_bytes = (uint32_t)g.K * 2u;
    const RowSrc rs = row_src_of(p, in);
    for (int i0 = 0; i0 < items; i0 += g.ipp) {
      if (!wait_mbar(p, m, &m->empty[slot], (round & 1u) ^ 1u, kErrTimeoutPage) ||
          !hold_wait(p, m, i)) {
        ok = false;
        break;
      }
      const int i1 = min(items, i0 + g.ipp);
      if (i0 == 0 && p.trace != nullptr) t_first = globaltimer();
      mbar_arrive_expect_tx(&m->full[slot], (uint32_t)((i1 - i0) * g.R) * row_bytes);
      issue_page(p, in, g, rs, i0, i1, smem + (size_t)slot * kPageBytes, &m->full[slot], pol);
      ++page_cnt;
      if (++slot == p.n_pages) {
        slot = 0;
        ++round;
      }
    }
    if (ok && items > 0) trace_issue(i, t_first);
  }
  if (!ok) {
    // drain: every issued copy must land before the CTA's shared memory goes away
    if (bt_pending) {
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(&m->bt_full, bt_par)) {
        if (globaltimer() - t0 > p.timeout_ns) break;
      }
    }
    const uint32_t first = page_cnt > (uint32_t)p.n_pages ? page_cnt - p.n_pages : 0u;
    for (uint32_t k = first; k < page_cnt; ++k) {
      const int sl = (int)(k % (uint32_t)p.n_pages);
      const uint32_t par = (k / (uint32_t)p.n_pages) & 1u;
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(&m->full[sl], par)) {
        if (globaltimer() - t0 > p.timeout_ns) break;
      }
    }
  }
}

// Four floats as bf16 pairs {hi(a, b), lo(a, b), hi(c, d), lo(c, d)} with
// v = hi + lo: a tensor-core operand that keeps about 16 bits of each value.
__device__ __forceinline__ uint4 split_hi_lo(float a, float b, float c, float d) {
  const uint32_t h01 = bf16x2_rn(a, b), h23 = bf16x2_rn(c, d);
  return make_uint4(h01, bf16x2_rn(a - bf_lo(h01), b - bf_hi(h01)), h23,
                    bf16x2_rn(c - bf_lo(h23), d - bf_hi(h23)));
}

// One sequence, 2048-column rows: the staged activations are kept as the B
// fragments of the tensor-core GEMV (rows4_mma), built once per staging and
// shared by the compute warps. Lane l of a warp takes the 64 words at
// l * 64 .. + 63 of the buffer: word 4 tp + q is its B register for the step
// pair tp (q = 0, 1: step 2 tp; q = 2, 3: step 2 tp + 1). The 16-byte chunks
// of lane l are stored rotated by l % 8, so that the 8 lanes of one
// shared-memory phase read different banks.
__device__ __forceinline__ int frag_word(int l, int tp, int q) { return l * 64 + 4 * (tp ^ (l & 7)) + q; }

// Writes columns c .. c + 3 (c % 4 == 0) of a 2048-column activation vector
// into the fragment buffer: column c of segment sg = c / 512, u = c % 512,
// sits in step pair tp = (u / 32) ^ sg of lane 8 sg + (u / 8) % 4 (its bf16 hi
// part) and of lane 8 sg + 4 + (u / 8) % 4 (its lo part), word q = (u % 8) / 2.
__device__ __forceinline__ void put_frag(uint32_t* fb, int c, float4 x) {
  const int sg = c >> 9, u = c & 511;
  const int tp = (u >> 5) ^ sg, tig = (u >> 3) & 3, q = (u & 7) >> 1;
  const uint4 f = split_hi_lo(x.x, x.y, x.z, x.w);  // {hi01, lo01, hi23, lo23}
  const int lh = 8 * sg + tig;
  *reinterpret_cast<uint2*>(fb + frag_word(lh, tp, q)) = make_uint2(f.x, f.z);
  *reinterpret_cast<uint2*>(fb + frag_word(lh + 4, tp, q)) = make_uint2(f.y, f.w);
}

// This lane's 64 B fragment registers from the fragment buffer.
__device__ __forceinline__ void load_frag(float (&bx)[64], const uint32_t* fb) {
  const int l = threadIdx.x & 31;
#pragma unroll
  for (int tp = 0; tp < 16; ++tp) {
    const uint4 v = lds128(fb + frag_word(l, tp, 0));
    bx[4 * tp + 0] = __uint_as_float(v.x);
    bx[4 * tp + 1] = __uint_as_float(v.y);
    bx[4 * tp + 2] = __uint_as_float(v.z);
    bx[4 * tp + 3] = __uint_as_float(v.w);
  }
}

// ---------------------------------------------------------------------------
// compute role: activation staging
// ---------------------------------------------------------------------------

enum ActKind { kActNone = 0, kActAttnNorm, kActMlpNorm, kActFinalNorm, kActAttnOut, kActH };

__device__ __forceinline__ int act_kind(int op) {
  switch (op) {
    case MK_OP_QKV: return kActAttnNorm;
    case MK_OP_OPROJ: return kActAttnOut;
    case MK_OP_GATEUP: return kActMlpNorm;
    case MK_OP_DOWN: return kActH;
    case MK_OP_LMHEAD: return kActFinalNorm;
    default: return kActNone;
  }
}

struct InvScale {
  float v[kMaxBatch];  // 1/rms per sequence (1 for activations without a norm)
};

struct Staged {
  int key_x = -1;     // what the x buffer holds
  int key_h = -1;     // what the h buffer holds
  int stage_cnt = 0;  // parity of the RMSNorm partial-sum buffer
  InvScale inv_x;     // scale of the x buffer's contents
};

// the token of sequence b: from the parameters, or (greedy decode) from the
// previous step's argmax
template <int FX>
__device__ __forceinline__ int token_of(const Params& p, int b, int step) {
  if ((FX & kFxPaged) && step > 0)
    return key_token(__ldcg(p.argmax_out + (size_t)(step - 1) * p.B + b));
  return (FX & kFxPaged) && p.tok_keys ? key_token(__ldcg(p.tok_keys + b)) : p.tok[b];
}

__device__ __forceinline__ int act_key(int kind, int layer, int chunk) {
  return (kind << 20) | (layer << 4) | chunk;
}

__device__ __forceinline__ const uint16_t* norm_weight(const Params& p, int kind, int layer) {
  if (kind == kActAttnNorm) return p.layers[layer].attn_norm;
  if (kind == kActMlpNorm) return p.layers[layer].mlp_norm;
  if (kind == kActFinalNorm) return p.final_norm;
  return nullptr;
}

// One pass of the staging over sequences [b0, b0 + NB): NS source rows per
// sequence are added left to right (NS = 5: the previous layer's output x =
// xa + its four down-projection shares; NS = 1: one row), the RMSNorm gain is
// applied, and the result is stored in the staging layout. Every thread
// issues all of its loads of a column pass before using any, so a pass costs
// one L2 round trip. The source rows are stamped words: the pass uses them
// as loaded and sets `bad` if one was stale, and the caller then stages the
// whole vector again. Returns the sums of squares per sequence in ss.
template <int B, int NS, int NB, int KU, int FX>
__device__ __forceinline__ void stage_pass(const Params& p, float* dst, int K, int Ks,
                                           const uint16_t* normw, bool from_embed,
                                           const float* base, size_t stride, int b0, int step,
                                           uint32_t st, float (&ss)[NB], bool frag, bool& bad) {
  constexpr bool kFrag = B > 1;
  constexpr int kPass = kComputeThreads * 4 * KU;  // columns per pass
  const int tid = compute_tid();
  const size_t cs = (size_t)p.B * p.H;  // distance between two down-projection shares
#pragma unroll
  for (int bb = 0; bb < NB; ++bb) ss[bb] = 0.f;
  for (int c0 = tid * 4; c0 < K; c0 += kPass) {
    float4 v[NS][NB][KU];
    uint2 wv[KU];
#pragma unroll
    for (int u = 0; u < KU; ++u) {
      const int c = c0 + u * kComputeThreads * 4;
      if (c < K) {
        if (normw) wv[u] = __ldg(reinterpret_cast<const uint2*>(normw + c));
#pragma unroll
        for (int bb = 0; bb < NB; ++bb) {
          if (b0 + bb >= B) continue;
          if (from_embed) {
            const uint16_t* erow = p.embed + (size_t)token_of<FX>(p, b0 + bb, step) * p.H;
            const uint2 e = *reinterpret_cast<const uint2*>(erow + c);
            v[0][bb][u] = make_float4(bf_lo(e.x), bf_hi(e.x), bf_lo(e.y), bf_hi(e.y));
          } else {
#pragma unroll
            for (int sidx = 0; sidx < NS; ++sidx) {
              const float* src = sidx == 0 ? base : p.xpart + (size_t)(sidx - 1) * cs;
              v[sidx][bb][u] = ld_relaxed4(src + (b0 + bb) * stride + c);
            }
          }
        }
      }
    }
    if (!from_embed) {
#pragma unroll
      for (int u = 0; u < KU; ++u)
#pragma unroll
        for (int bb = 0; bb < NB; ++bb)
#pragma unroll
          for (int sidx = 0; sidx < NS; ++sidx) {
            if (c0 + u * kComputeThreads * 4 < K && b0 + bb < B) bad |= stale4(v[sidx][bb][u], st);
            v[sidx][bb][u] = clear4(v[sidx][bb][u]);
          }
    }
#pragma unroll
    for (int u = 0; u < KU; ++u) {
      const int c = c0 + u * kComputeThreads * 4;
      if (c < K) {
#pragma unroll
        for (int bb = 0; bb < NB; ++bb) {
          if (b0 + bb >= B) continue;
          float4 x = v[0][bb][u];
          if (!from_embed) {
#pragma unroll
            for (int sidx = 1; sidx < NS; ++sidx) {
              x.x += v[sidx][bb][u].x;
              x.y += v[sidx][bb][u].y;
              x.z += v[sidx][bb][u].z;
              x.w += v[sidx][bb][u].w;
            }
            // the layer output as the chunk-3 storer would have written it
            if (NS > 1) x = clear4(x);
          }
          ss[bb] += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
          if (normw) {
            x.x *= bf_lo(wv[u].x);
            x.y *= bf_hi(wv[u].x);
            x.z *= bf_lo(wv[u].y);
            x.w *= bf_hi(wv[u].y);
          }
          float* d = dst + (size_t)(b0 + bb) * Ks + c;
          if (B == 1 && frag) {
            put_frag(reinterpret_cast<uint32_t*>(dst), c, x);
          } else if (kFrag) {
            const uint32_t h01 = bf16x2_rn(x.x, x.y), h23 = bf16x2_rn(x.z, x.w);
            const uint32_t l01 = bf16x2_rn(x.x - bf_lo(h01), x.y - bf_hi(h01));
            const uint32_t l23 = bf16x2_rn(x.z - bf_lo(h23), x.w - bf_hi(h23));
            *reinterpret_cast<uint4*>(d) = make_uint4(h01, l01, h23, l23);
          } else {
            *reinterpret_cast<float4*>(d) = x;
          }
        }
      }
    }
  }
}

// Stages the activation vector(s) of `kind` for all B sequences into the x or
// h buffer. For the RMSNorm kinds the buffer holds x * w (the gain already
// applied) and 1/rms(x) per sequence is returned in st.inv_x. The RMSNorm
// inputs of layer l > 0 and of the LM head are the previous layer's output,
// x = xa + the four down-projection shares, summed here.
// Several sequences (B > 1): sequence b's row starts at word b * (K + 4), and
// each group of four columns c .. c + 3 is stored in place as the bf16 split
// v = hi + lo of its values, {hi(c, c+1), lo(c, c+1), hi(c+2, c+3),
// lo(c+2, c+3)}: the A fragment of the tensor-core product (page_rows_mma).
// kWide: rows may be wider than 3072 columns (one sequence): six column groups
// per thread, so that 4608 columns still take one L2 round trip
template <int B, int FX, bool kWide, int KW>
__device__ __forceinline__ void stage(const Params& p, Misc* m, uint8_t* smem, Staged& st, int kind,
                                      int layer, int chunk, int key, int step) {
  constexpr bool kFrag = B > 1;
  const int tid = compute_tid();  // 0..kComputeThreads-1
  const int warp = tid >> 5, lane = tid & 31;
  const bool to_h = kind == kActH;
  float* dst = reinterpret_cast<float*>(smem + (to_h ? p.off_h : p.off_x));
  const int K = kind == kActAttnOut ? p.QD : (to_h ? p.Fc : p.H);
  const int Ks = kFrag ? K + 4 : K;  // row stride of the buffer, in words
  // one sequence, 2048 columns: the buffer holds the GEMV's B fragments
  const bool frag = B == 1 && (KW == 2048 || K == 2048);
  const uint16_t* normw = norm_weight(p, kind, layer);
  const bool from_embed = kind == kActAttnNorm && layer == 0;
  // x = xa + the four down-projection shares of the previous layer
  const bool sum_x = (kind == kActAttnNorm && layer > 0) || kind == kActFinalNorm;
  // sequence b's source row: base + b * stride
  const float* base;
  size_t stride;
  const bool whole = x_whole<B>(p);
  if (sum_x) base = whole ? p.x : p.xa, stride = p.H;
  else if (kind == kActMlpNorm) base = p.xa, stride = p.H;
  else if (kind == kActAttnOut) base = p.attn, stride = p.QD;
  else base = p.h + (size_t)chunk * p.Fc, stride = p.F;
  const int par = st.stage_cnt & 1;
  // the stamp of the source words: the previous layer's output for the
  // attention norm, the last layer's for the final norm, else this layer's
  const uint32_t wst =
      stamp_of(p, step, kind == kActAttnNorm ? layer - 1 : (kind == kActFinalNorm ? p.L - 1 : layer));
  compute_bar();  // everyone is done reading the buffer's previous contents
  // one sequence: four (six if rows may be wider than 3072 columns) column
  // groups per thread and pass, so 2048 (4608) columns take one L2 round
  // trip; with five sources (x not written whole) two (one if wide), for
  // the register budget. Several sequences: all of them and three groups per
  // pass; with five sources, two sequences and one group
  constexpr int kNB1 = B, kU1 = B == 1 ? (kWide ? 6 : 4) : 3;
  constexpr int kNB5 = B == 1 ? 1 : 2, kU5 = B == 1 && !kWide ? 2 : 1;
  const bool five = sum_x && !whole;  // x = xa + the four shares, summed here
  // the whole vector is staged again if any compute thread loaded a stale
  // word (the decision is taken at the barrier, so it is uniform)
  uint32_t tries = 0;
  uint64_t t0 = 0;
  for (;;) {
    bool bad = false;
    if (five) {
      for (int b0 = 0; b0 < B; b0 += kNB5) {
        float ss[kNB5];
        stage_pass<B, 5, kNB5, kU5, FX>(p, dst, K, Ks, normw, false, base, stride, b0, step, wst,
                                        ss, frag, bad);
        if (normw) {
#pragma unroll
          for (int bb = 0; bb < kNB5; ++bb) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss[bb] += __shfl_xor_sync(0xffffffffu, ss[bb], o);
            if (lane == 0 && b0 + bb < B) m->red[par][warp][b0 + bb] = ss[bb];
          }
        }
      }
    } else {
      float ss[kNB1];
      stage_pass<B, 1, kNB1, kU1, FX>(p, dst, K, Ks, normw, from_embed, base, stride, 0, step, wst,
                                      ss, frag, bad);
      if (normw) {
#pragma unroll
        for (int bb = 0; bb < kNB1; ++bb) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) ss[bb] += __shfl_xor_sync(0xffffffffu, ss[bb], o);
          if (lane == 0) m->red[par][warp][bb] = ss[bb];
        }
      }
    }
    if (!compute_bar_or(bad)) break;
    // some word was stale: stage again, unless this thread gives up (abort,
    // error, timeout), in which case every thread does
    if (compute_bar_or(!retry_stale(p, m, tries, t0))) break;
  }
  InvScale inv;
#pragma unroll
  for (int b = 0; b < kMaxBatch; ++b) {
    inv.v[b] = 1.f;
    if (normw && b < B) {
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kComputeWarps; ++w) sum += m->red[par][w][b];
      inv.v[b] = rsqrtf(sum / (float)p.H + p.eps);
    }
  }
  st.stage_cnt++;
  if (to_h) {
    st.key_h = key;
    if (p.alias_xh) st.key_x = -1;
  } else {
    st.key_x = key;
    st.inv_x = inv;
    if (p.alias_xh) st.key_h = -1;
  }
}

// One sequence: the O-projection's input, every head's attention output,
// reduced from the split-KV partials as it is staged (the reduction
// instruction fused into the O-projection). Thread t takes the 4-dimension
// column groups t + i * kComputeThreads (i < kG), so the LPH lanes of a warp
// that cover one head's columns form an aligned group. Per round of kR
// partitions every load is issued first: each lane the o of its groups for
// the round's partitions, and the (m, l) of one partition of its head, which
// the head's lanes then share by shuffles; weights e^(m_k - M) rescale online
// across rounds. P: partitions per head.
template <int D>
__device__ __forceinline__ void stage_attn_fused(const Params& p, uint8_t* smem, Staged& st,
                                                 int layer, int P, int key) {
  constexpr int kG = 1;  // column groups per thread per pass (768 columns: smaller code, as fast)
  constexpr int kR = 6;  // partitions per round
  constexpr int LPH = D / 4 < 32 ? D / 4 : 32;  // lanes covering one head
  const int tid = compute_tid(), lane = threadIdx.x & 31;
  const int lead = lane & ~(LPH - 1);
  float* dst = reinterpret_cast<float*>(smem + p.off_x);
  compute_bar();  // everyone is done reading the buffer's previous contents
  for (int q0 = tid; q0 * 4 < p.QD; q0 += kComputeThreads * kG) {
    float M[kG], den[kG];
    float4 acc[kG];
#pragma unroll
    for (int i = 0; i < kG; ++i) {
      M[i] = -INFINITY;
      den[i] = 0.f;
      acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int k0 = 0; k0 < P; k0 += kR) {
      float4 o[kG][kR];
      float2 ml[kG];
#pragma unroll
      for (int i = 0; i < kG; ++i) {
        const int c = (q0 + i * kComputeThreads) * 4;  // the whole warp agrees on c < QD
        if (c < p.QD) {
          const int h = c / D;
          const float* ob = p.part + ((size_t)h * kMaxPartitions + k0) * D + (c - h * D);
#pragma unroll
          for (int k = 0; k < kR; ++k)
            if (k0 + k < P) o[i][k] = __ldcg(reinterpret_cast<const float4*>(ob + (size_t)k * D));
          const int kk = k0 + (lane & (LPH - 1));
          ml[i] = kk < P && (lane & (LPH - 1)) < kR
                      ? __ldcg(reinterpret_cast<const float2*>(p.part_ml + ((size_t)h * kMaxPartitions + kk) * 2))
                      : make_float2(-INFINITY, 0.f);
        }
      }
#pragma unroll
      for (int i = 0; i < kG; ++i) {
        const int c = (q0 + i * kComputeThreads) * 4;
        if (c >= p.QD) continue;  // warp-uniform
        float mr = ml[i].x;
#pragma unroll
        for (int off = 1; off < LPH; off <<= 1) mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, off));
        const float Mn = fmaxf(M[i], mr);
        const float sc = M[i] == -INFINITY ? 0.f : fast_exp2(M[i] - Mn);
        den[i] *= sc;
        acc[i].x *= sc; acc[i].y *= sc; acc[i].z *= sc; acc[i].w *= sc;
#pragma unroll
        for (int k = 0; k < kR; ++k) {
          const float mk = __shfl_sync(0xffffffffu, ml[i].x, lead | k);
          const float lk = __shfl_sync(0xffffffffu, ml[i].y, lead | k);
          if (k0 + k < P && mk != -INFINITY) {
            const float w = fast_exp2(mk - Mn);
            den[i] = fmaf(w, lk, den[i]);
            acc[i].x = fmaf(w, o[i][k].x, acc[i].x);
            acc[i].y = fmaf(w, o[i][k].y, acc[i].y);
            acc[i].z = fmaf(w, o[i][k].z, acc[i].z);
            acc[i].w = fmaf(w, o[i][k].w, acc[i].w);
          }
        }
        M[i] = Mn;
      }
    }
#pragma unroll
    for (int i = 0; i < kG; ++i) {
      const int c = (q0 + i * kComputeThreads) * 4;
      if (c < p.QD) {
        const float inv = 1.f / den[i];
        const float4 o4 = make_float4(acc[i].x * inv, acc[i].y * inv, acc[i].z * inv, acc[i].w * inv);
        // 2048 attention columns: the O-projection's B fragments
        if (p.QD == 2048) put_frag(reinterpret_cast<uint32_t*>(dst), c, o4);
        else *reinterpret_cast<float4*>(dst + c) = o4;
      }
    }
  }
  compute_bar();
  st.stage_cnt++;
  st.key_x = key;
#pragma unroll
  for (int b = 0; b < kMaxBatch; ++b) st.inv_x.v[b] = 1.f;
  if (p.alias_xh) st.key_h = -1;
}

// One sequence, rows narrower than 2048 columns: each compute warp copies the
// staged vector into registers in the layout of the page dot products (lane
// l, block j: columns j*256 + l*8 .. +8), scaled by 1/rms for the norms.
__device__ __forceinline__ void load_regs(float (&a)[64], const float* act, float scale, int K) {
  const int lane = threadIdx.x & 31;
  const int nblk = K / 256;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < nblk) {
      const float* src = act + j * 256 + lane * 8;
      const float4 x0 = *reinterpret_cast<const float4*>(src);
      const float4 x1 = *reinterpret_cast<const float4*>(src + 4);
      a[j * 8 + 0] = x0.x * scale; a[j * 8 + 1] = x0.y * scale;
      a[j * 8 + 2] = x0.z * scale; a[j * 8 + 3] = x0.w * scale;
      a[j * 8 + 4] = x1.x * scale; a[j * 8 + 5] = x1.y * scale;
      a[j * 8 + 6] = x1.z * scale; a[j * 8 + 7] = x1.w * scale;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) a[j * 8 + e] = 0.f;
    }
  }
}

// ---------------------------------------------------------------------------
// One sequence, 2048-column rows, on the tensor cores (mma.sync m16n8k16,
// bf16 in, fp32 accumulate). A page holds 4 rows of 2048 columns; the
// product sees it as 16 "virtual rows", row m = page row m / 4 restricted to
// column segment s = m % 4 (512 columns each): the A operand. The B operand
// has 8 columns, column n = the bf16 hi (n even) or lo (n odd) part of the
// activations' segment n / 2, so x = hi + lo enters at about 16-bit
// precision per term. D[m][n] is a partial dot product when the segments of
// m and n agree (m % 4 == n / 2); the other entries are never used. A page
// is 32 products over the segment's 512 columns; its 4 row results are the
// sums of 4 segment partials. Inside a segment the order of the 16 columns
// of one product is free as long as A and B follow it: step t of segment s
// takes column pairs (tig) from P, P + 1 and (tig + 4) from P + 2, P + 3,
// P = 32 ((t / 2) ^ s) + 8 tig + 4 (t % 2), so one 16-byte load of a page row
// feeds two steps, and the XOR by s puts the two virtual rows that one
// shared-memory phase reads (segments s and s ^ 1 of one page row) on
// different banks.

// The 4 rows of one page (rows past n_rows hold an earlier page's data, stay
// inside the slot and are never stored): page row pr's result goes to
// res_page[(k * R + r)], pr = r * n_in + k.
__device__ __forceinline__ void rows4_mma(const uint8_t* page, int n_rows, int n_in, int R,
                                          const float (&bx)[64], float scale, float* res_page,
                                          int lane) {
  const int grp = lane >> 2, tig = lane & 3;
  const int sg = grp & 3;        // segment of virtual rows grp and grp + 8
  const int ra = grp >> 2;       // page row of virtual row grp (grp + 8: ra + 2)
  const uint8_t* pa = page + ra * 4096 + sg * 1024 + 16 * tig;
  const uint8_t* pb = pa + 2 * 4096;
  // four independent accumulator chains (an mma.sync waits for the previous
  // one on the same accumulator), summed at the end
  float d4[4][4];
#pragma unroll
  for (int c = 0; c < 4; ++c) d4[c][0] = d4[c][1] = d4[c][2] = d4[c][3] = 0.f;
#pragma unroll
  for (int tp = 0; tp < 16; ++tp) {
    const int off = 64 * (tp ^ sg);
    const uint4 ua = lds128(pa + off), ub = lds128(pb + off);
    const int c = 2 * (tp & 1);
    mma_bf16_16816(d4[c], make_uint4(ua.x, ub.x, ua.y, ub.y), __float_as_uint(bx[4 * tp]),
                   __float_as_uint(bx[4 * tp + 1]));
    mma_bf16_16816(d4[c + 1], make_uint4(ua.z, ub.z, ua.w, ub.w), __float_as_uint(bx[4 * tp + 2]),
                   __float_as_uint(bx[4 * tp + 3]));
  }
  float d[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) d[e] = (d4[0][e] + d4[1][e]) + (d4[2][e] + d4[3][e]);
  // the useful columns 2 sg (hi) and 2 sg + 1 (lo) sit in the lanes with
  // tig == sg: lanes 0, 5, 10, 15 (page rows 0 and 2) and 16, 21, 26, 31
  // (rows 1 and 3), one segment each
  float v01 = tig == sg ? d[0] + d[1] : 0.f;  // page row ra
  float v23 = tig == sg ? d[2] + d[3] : 0.f;  // page row ra + 2
  v01 += __shfl_xor_sync(0xffffffffu, v01, 5);
  v23 += __shfl_xor_sync(0xffffffffu, v23, 5);
  v01 += __shfl_xor_sync(0xffffffffu, v01, 10);
  v23 += __shfl_xor_sync(0xffffffffu, v23, 10);
  if ((lane & 15) == 0) {
    const int r0 = lane >> 4;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int pr = r0 + 2 * e;
      if (pr < n_rows) {
        const int r = pr / n_in, k = pr - r * n_in;
        res_page[k * R + r] = (e == 0 ? v01 : v23) * scale;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// compute role: GEMV pages
// ---------------------------------------------------------------------------
// Each compute warp owns whole pages, dealt round-robin over the CTA's page
// stream, and dots every row of its page with the activations of all B
// sequences. One sequence with 2048-column rows runs on the tensor cores
// (rows4_mma: the activations' B fragments in registers). One sequence with
// other widths runs on the CUDA cores: lane l covers columns j*256 + l*8 ..
// +8 of each 256-column block, i.e. every block is one 512-byte contiguous
// read of the row per warp, and four rows are in flight at once (two
// accumulator chains each) for ILP; with rows narrower than 2048 columns the
// activations sit in registers, with wider rows they are read from the
// staged buffer block by block. Several sequences run on the tensor cores
// (page_rows_mma): there every weight meets B activations, which the FMA
// pipes and the shared-memory reads of fp32 activations could not keep up
// with at the weight stream's rate.

__device__ __forceinline__ void warp_sum4(float (&v)[4]) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] += __shfl_xor_sync(0xffffffffu, v[q], o);
  }
}

// B == 1, K < 2048: activations a[j*8 + e] in registers. Rows 0..n_rows-1
// (n_rows <= 4) of the page starting at `rows`; lane q < n_rows stores row
// q's result to *dst (every lane passes its own row's destination, so no
// array of pointers is needed).
__device__ __forceinline__ void rows4_reg(const uint8_t* rows, int n_rows, int row_bytes,
                                          int nblk, const float (&a)[64], float* dst,
                                          int lane) {
  // two accumulator chains per row, each a packed pair of fp32 lanes (even
  // and odd columns), so one fma.rn.f32x2 covers two weights
  unsigned long long acc[4][2];
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q][0] = acc[q][1] = 0ull;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < nblk) {
      uint4 w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        w[q] = q < n_rows
                   ? *reinterpret_cast<const uint4*>(rows + (size_t)q * row_bytes + j * 512 + lane * 16)
                   : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t ws[4] = {w[q].x, w[q].y, w[q].z, w[q].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          ffma2(acc[q][j & 1], pack2(bf_lo(ws[e]), bf_hi(ws[e])),
                pack2(a[j * 8 + 2 * e], a[j * 8 + 2 * e + 1]));
      }
    }
  }
  float v[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 x = unpack2(acc[q][0]), y = unpack2(acc[q][1]);
    v[q] = (x.x + x.y) + (y.x + y.y);
  }
  warp_sum4(v);
  if (lane < 4 && lane < n_rows) {
    float mine = v[0];
#pragma unroll
    for (int q = 1; q < 4; ++q) mine = lane == q ? v[q] : mine;
    *dst = mine;
  }
}

// One sequence, rows wider than 2048 columns (a page holds at most three):
// rows4_reg with the activations read from the staged buffer block by block,
// each read serving every row of the page; the 1/rms scale multiplies the
// sums. Lane q < n_rows stores row q's result to *dst.
__device__ __forceinline__ void rows4_smem(const uint8_t* rows, int n_rows, int row_bytes,
                                           int nblk, const float* act, float scale, float* dst,
                                           int lane) {
  unsigned long long acc[4][2];
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q][0] = acc[q][1] = 0ull;
#pragma unroll 2
  for (int j = 0; j < nblk; ++j) {
    const float4 x0 = *reinterpret_cast<const float4*>(act + j * 256 + lane * 8);
    const float4 x1 = *reinterpret_cast<const float4*>(act + j * 256 + lane * 8 + 4);
    const unsigned long long a[4] = {pack2(x0.x, x0.y), pack2(x0.z, x0.w), pack2(x1.x, x1.y),
                                     pack2(x1.z, x1.w)};
    uint4 w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      w[q] = q < n_rows ? *reinterpret_cast<const uint4*>(rows + (size_t)q * row_bytes + j * 512 + lane * 16)
                        : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t ws[4] = {w[q].x, w[q].y, w[q].z, w[q].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) ffma2(acc[q][j & 1], pack2(bf_lo(ws[e]), bf_hi(ws[e])), a[e]);
    }
  }
  float v[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 x = unpack2(acc[q][0]), y = unpack2(acc[q][1]);
    v[q] = (x.x + x.y) + (y.x + y.y);
  }
  warp_sum4(v);
  if (lane < 4 && lane < n_rows) {
    float mine = v[0];
#pragma unroll
    for (int q = 1; q < 4; ++q) mine = lane == q ? v[q] : mine;
    *dst = mine * scale;
  }
}

// Several sequences: the tensor-core product of a page's rows with the staged
// activations of all B sequences. One mma.sync m16n8k16 multiplies 16
// activation rows (the bf16 hi parts of sequences 0..7 in rows 0..7, their lo
// parts in rows 8..15) by 16 columns of 8 page rows, so hi and lo products add
// up to an fp32-accurate dot product. The order of the 16 columns inside one
// product is free as long as both operands follow it: step s takes column
// pair tig from the columns P, P + 1 and pair tig + 4 from P + 2, P + 3, with
// P = 32 (s / 2) + 8 tig + 4 (s % 2). Then one 16-byte load of a page row
// feeds two steps, and the 16 staged bytes at column P are exactly one A
// fragment. Odd page rows load the two 64-byte halves of a 64-column chunk
// in swapped order, so that even and odd rows fall on disjoint banks; the
// staged rows are padded by 4 words for the same reason.
template <int B>
__device__ __forceinline__ void page_rows_mma(const uint8_t* page, int n_rows, int row_bytes,
                                              int K, const uint32_t* act, const InvScale& inv,
                                              float* res_page, int n_in, int R, int lane) {
  const int grp = lane >> 2, tig = lane & 3, odd = grp & 1;
  // lanes past the last sequence repeat it; their product rows are not stored
  const uint32_t* arow = act + (size_t)min(grp, B - 1) * (K + 4) + 8 * tig;
  float sc = inv.v[0];
#pragma unroll
  for (int b = 1; b < B; ++b) sc = grp == b ? inv.v[b] : sc;
  for (int r0 = 0; r0 < n_rows; r0 += 8) {
    const int nv = min(8, n_rows - r0);
    // B column grp = page row r0 + grp; lanes past the valid rows repeat a
    // valid row of the same parity, i.e. another lane's addresses
    const int rr = grp < nv ? grp : (nv > 1 ? odd : 0);
    const uint8_t* w0 = page + (size_t)(r0 + rr) * row_bytes + 16 * tig + 64 * odd;
    const uint8_t* w1 = page + (size_t)(r0 + rr) * row_bytes + 16 * tig + 64 * (odd ^ 1);
    // four accumulator chains; plain loads, so that the compiler can issue
    // the next chunks' loads ahead of this chunk's products
    float d[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) d[q][0] = d[q][1] = d[q][2] = d[q][3] = 0.f;
#pragma unroll 4
    for (int c = 0; c < K; c += 64) {
      const uint4 wa = *reinterpret_cast<const uint4*>(w0 + 2 * c);
      const uint4 wb = *reinterpret_cast<const uint4*>(w1 + 2 * c);
      const uint4 a0 = *reinterpret_cast<const uint4*>(arow + c);
      const uint4 a1 = *reinterpret_cast<const uint4*>(arow + c + 4);
      const uint4 a2 = *reinterpret_cast<const uint4*>(arow + c + 32);
      const uint4 a3 = *reinterpret_cast<const uint4*>(arow + c + 36);
      const uint4 wl = odd ? wb : wa;  // columns c + 8 tig .. + 7
      const uint4 wh = odd ? wa : wb;  // columns c + 32 + 8 tig .. + 7
      mma_bf16_16816(d[0], a0, wl.x, wl.y);
      mma_bf16_16816(d[1], a1, wl.z, wl.w);
      mma_bf16_16816(d[2], a2, wh.x, wh.y);
      mma_bf16_16816(d[3], a3, wh.z, wh.w);
    }
    if (grp < B) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int pr = 2 * tig + e;
        if (pr < nv) {
          const int row = r0 + pr, r = row / n_in, k = row - r * n_in;
          const float hi = (d[0][e] + d[1][e]) + (d[2][e] + d[3][e]);
          const float lo = (d[0][2 + e] + d[1][2 + e]) + (d[2][2 + e] + d[3][2 + e]);
          res_page[((size_t)k * R + r) * B + grp] = (hi + lo) * sc;
        }
      }
    }
  }
}

// kRegs: the activations are in the caller's registers a[] (B == 1, rows of at
// most 2048 columns); otherwise they are read from the staged buffer `act`
// (fp32 for one sequence, tensor-core fragments for several).
// KW == 2048: every row is 2048 wide (only the full-page code is compiled).
template <int B, bool kRegs, int KW>
__device__ __forceinline__ void gemv_run(const Params& p, Misc* m, uint8_t* smem, const Instr& in,
                                         const Geom& g, const float* act, const InvScale& inv,
                                         const float (&a)[64], float* res, uint32_t page_base,
                                         uint64_t& pwait) {
  const int warp = compute_warp(), lane = threadIdx.x & 31;
  const int items = in.a1 - in.a0;
  const int npages = (items + g.ipp - 1) / g.ipp;
  const int row_bytes = g.K * 2;
  const int nblk = g.K / 256;
  // the pages of this warp: global page index congruent to the warp index.
  // n_pages is a multiple of kComputeWarps, so every slot this warp waits on
  // was last used by this warp's own previous page (already consumed): the
  // parity wait below cannot alias an older phase.
  int pg = (int)(((uint32_t)warp + kComputeWarps - page_base % kComputeWarps) % kComputeWarps);
  // slot and phase of this warp's first page, then advanced incrementally
  const uint32_t pc0 = page_base + (uint32_t)pg;
  int slot = (int)(pc0 % (uint32_t)p.n_pages);
  uint32_t round = pc0 / (uint32_t)p.n_pages;
  for (; pg < npages; pg += kComputeWarps) {
    const uint64_t tw = p.trace != nullptr ? globaltimer() : 0;
    const bool ok = wait_mbar(p, m, &m->full[slot], round & 1u, kErrTimeoutPage);
    if (p.trace != nullptr) pwait += globaltimer() - tw;
    if (ok) {
      const int n_in = min(g.ipp, items - pg * g.ipp);  // items on this page
      const uint8_t* page = smem + (size_t)slot * kPageBytes;
      // page row pr = r * n_in + k holds row r of item pg*ipp + k; its result
      // goes to res[((item * R) + r) * B + b]
      const int n_rows = n_in * g.R;
      float* const res_page = res + (size_t)(pg * g.ipp) * g.R * B;
      if (kRegs) {
        if (KW == 2048 || nblk == 8) {
          // pages of 2048-column rows, full or the short last page of an
          // instruction, on the tensor cores (a[] holds the B fragments)
          rows4_mma(page, n_rows, n_in, g.R, a, inv.v[0], res_page, lane);
        } else if constexpr (KW == 0) {
          for (int r0 = 0; r0 < n_rows; r0 += 4) {
            const int pr = min(r0 + (lane & 3), n_rows - 1);
            const int r = pr / n_in, k = pr - r * n_in;
            rows4_reg(page + (size_t)r0 * row_bytes, n_rows - r0, row_bytes, nblk, a,
                      res_page + ((size_t)k * g.R + r) * B, lane);
          }
        }
      } else if constexpr (B > 1) {
        page_rows_mma<B>(page, n_rows, row_bytes, g.K, reinterpret_cast<const uint32_t*>(act), inv,
                         res_page, n_in, g.R, lane);
      } else {
        const int pr = min(lane & 3, n_rows - 1);
        const int r = pr / n_in, k = pr - r * n_in;
        rows4_smem(page, n_rows, row_bytes, nblk, act, inv.v[0], res_page + ((size_t)k * g.R + r) * B,
                   lane);
      }
    }
    // a page whose copy has not landed (after an abort) is never handed back,
    // so the loader cannot start a second copy into a slot still being filled
    __syncwarp();
    if (lane == 0 && ok) mbar_arrive_cnt(&m->empty[slot], kComputeWarps);
    slot += kComputeWarps;
    if (slot >= p.n_pages) {
      slot -= p.n_pages;
      ++round;
    }
  }
}

// ---------------------------------------------------------------------------
// compute role: split-KV attention partial (instruction 2)
// ---------------------------------------------------------------------------
// Unit (b, g, p): the G <= 8 q-heads of kv-head g over keys [t0, t1) of
// sequence b, on the tensor cores. Every compute warp takes whole pages of the
// unit (the pages it owns in the SM's page stream, as for GEMV pages) and
// keeps its own online softmax in the log2 domain (q is pre-scaled by
// log2(e)/sqrt(D)):
//   scores   S = Q K^T, one mma.sync per 16 dimensions and 8 keys: rows
//            0..7 the bf16 hi parts of the queries, rows 8..15 their lo
//            parts (query rows past G repeat the last one), the dimensions
//            in the permuted order of the GEMV products, so that one 16-byte
//            load of a key row feeds two steps;
//   weights  p = 2^(s - m), split into bf16 hi and lo the same way: the score
//            fragments of two 8-key blocks are exactly the A fragment of a
//            16-key step of
//   output   O += P V, V read transposed from the page with ldmatrix.
// The hi and lo rows add up at the end, and the warps' (o, m, l) combine
// through shared memory in a fixed order. The new key (position pos, written
// by this step's QKV instruction after the pages were fetched) starts the
// softmax of the warp that takes the unit's first page: a single key's
// partial is (o, m, l) = (v, q.k, 1); its k and v rows load from global
// memory together with the queries.


template <int D, int FX>
__device__ void attn_unit(const Params& p, Misc* m, uint8_t* smem, const Instr& in,
                          uint32_t page_base, uint64_t& pwait) {
  constexpr int KS = D / 16;                   // product steps over the head dimension
  constexpr int NB = D / 8;                    // 8-column blocks of the output
  constexpr int KPP = kPageBytes / (4 * D);    // keys per page (K, then V)
  constexpr int NKB = KPP / 8;                 // 8-key blocks per page
  const int warp = compute_warp(), lane = threadIdx.x & 31;
  const int grp = lane >> 2, tig = lane & 3, odd = grp & 1;
  const int b = in.a0, g = in.a1, pidx = in.a2 >> 16, P = in.a2 & 0xffff;
  const int G = p.G, pos = p.pos[b] + step_of(in);
  const AttnSpan sp = attn_span(pos, pidx, P, D);
  const float qscale = 1.4426950408889634f * rsqrtf((float)D);
  const float* qhead = p.q + (size_t)b * p.QD + (size_t)g * G * D;

  // this warp's pages are the unit's pages r0, r0 + kComputeWarps, ... (it
  // owns the slots congruent to its index; n_pages is a multiple of
  // kComputeWarps, see gemv_run). The residue r0, not the warp, names the
  // warp's share in the combination, so that the result does not depend on
  // where the unit starts in the SM's page stream.
  const int r0 = (int)(((uint32_t)warp + kComputeWarps - page_base % kComputeWarps) % kComputeWarps);
  // the new key, if in this unit, goes with share 0: k row as the B fragment
  // of key column 0 (lanes grp == 0), v columns 8 nb + 2 tig, +1 of every lane
  const bool new_here = r0 == 0 && sp.t0 <= pos && pos < sp.t1;
  const uint32_t st = stamp_of(p, step_of(in), layer_of(in));
  // The queries and (if in this unit) the new key and value: stamped words,
  // all loaded first, then tested, the stale ones reloaded. The new rows are
  // the stamped copy of what the QKV instruction appended (bf16 bits in the
  // upper half of each word; two words make one bf16 pair).
  const float* qs = qhead + (size_t)min(grp, G - 1) * D + 8 * tig;
  const float* kr = p.kvn + ((size_t)(b * p.nkv + g) * 2) * D;
  const float* vr = kr + D;
  float4 qw[KS];      // dimensions 32 (j / 2) + 8 tig + 4 (j % 2) .. + 3
  float4 kw[D / 32][2];  // k columns 32 i + 8 tig .. + 7 (lanes grp == 0)
  float2 vw[NB];      // v columns 8 nb + 2 tig, + 1
  const bool kload = new_here && grp == 0;
  {
    uint32_t tries = 0;
    uint64_t t0 = 0;
    for (;;) {
#pragma unroll
      for (int j = 0; j < KS; ++j) qw[j] = ld_relaxed4(qs + 32 * (j / 2) + 4 * (j % 2));
#pragma unroll
      for (int i = 0; i < D / 32; ++i) {
        kw[i][0] = kw[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (kload) {
          kw[i][0] = ld_relaxed4(kr + 32 * i + 8 * tig);
          kw[i][1] = ld_relaxed4(kr + 32 * i + 8 * tig + 4);
        }
      }
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
        vw[nb] = new_here ? ld_relaxed2(vr + 8 * nb + 2 * tig) : make_float2(0.f, 0.f);
      bool bad = false;
#pragma unroll
      for (int j = 0; j < KS; ++j) bad |= stale4(qw[j], st);
#pragma unroll
      for (int i = 0; i < D / 32; ++i) bad |= kload && (stale4(kw[i][0], st) || stale4(kw[i][1], st));
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) bad |= new_here && stale2(vw[nb], st);
      if (!bad || !retry_stale(p, m, tries, t0)) break;
    }
  }
  // the new key as B fragments of key column 0 (lanes grp == 0), the new
  // value's columns 8 nb + 2 tig, +1 of every lane
  uint4 kn[D / 64][2];
  uint32_t vn[NB];
#pragma unroll
  for (int j2 = 0; j2 < D / 64; ++j2)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const float4 a = kw[2 * j2 + hf][0], c = kw[2 * j2 + hf][1];
      kn[j2][hf] = make_uint4(__byte_perm(__float_as_uint(a.x), __float_as_uint(a.y), 0x7632),
                              __byte_perm(__float_as_uint(a.z), __float_as_uint(a.w), 0x7632),
                              __byte_perm(__float_as_uint(c.x), __float_as_uint(c.y), 0x7632),
                              __byte_perm(__float_as_uint(c.z), __float_as_uint(c.w), 0x7632));
    }
#pragma unroll
  for (int nb = 0; nb < NB; ++nb)
    vn[nb] = __byte_perm(__float_as_uint(vw[nb].x), __float_as_uint(vw[nb].y), 0x7632);
  // query fragments of head min(grp, G - 1): step s covers dimensions
  // 32 (s / 2) + 8 tig + 4 (s % 2) .. + 3
  uint4 qa[KS];
#pragma unroll
  for (int j = 0; j < KS; ++j) {
    const float4 x = clear4(qw[j]);
    qa[j] = split_hi_lo(x.x * qscale, x.y * qscale, x.z * qscale, x.w * qscale);
  }
  float mrow = -INFINITY;  // running maximum of head grp (equal in the group's 4 lanes)
  float lsum = 0.f;        // this lane's share of the running sum
  float o[NB][4];          // rows grp (hi weights) and grp + 8 (lo), columns 8 nb + 2 tig, +1
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
  if (new_here) {
    float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j2 = 0; j2 < D / 64; ++j2) {
      mma_bf16_16816(d0, qa[4 * j2], kn[j2][0].x, kn[j2][0].y);
      mma_bf16_16816(d1, qa[4 * j2 + 1], kn[j2][0].z, kn[j2][0].w);
      mma_bf16_16816(d0, qa[4 * j2 + 2], kn[j2][1].x, kn[j2][1].y);
      mma_bf16_16816(d1, qa[4 * j2 + 3], kn[j2][1].z, kn[j2][1].w);
    }
    // key column 0 sits in lane 4 grp of the group
    mrow = __shfl_sync(0xffffffffu, (d0[0] + d1[0]) + (d0[2] + d1[2]), lane & ~3);
    lsum = tig == 0 ? 1.f : 0.f;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      o[nb][0] = bf_lo(vn[nb]);
      o[nb][1] = bf_hi(vn[nb]);
    }
  }

  int pg = r0;
  const uint32_t pc0 = page_base + (uint32_t)pg;
  int slot = (int)(pc0 % (uint32_t)p.n_pages);
  uint32_t round = pc0 / (uint32_t)p.n_pages;
  for (; pg < sp.npages; pg += kComputeWarps) {
    // the products need the whole warp: the lanes agree on the page
    const uint64_t tw = p.trace != nullptr ? globaltimer() : 0;
    const bool ok =
        __all_sync(0xffffffffu, wait_mbar(p, m, &m->full[slot], round & 1u, kErrTimeoutPage));
    if (p.trace != nullptr) pwait += globaltimer() - tw;
    if (ok) {
      const uint8_t* kp = smem + (size_t)slot * kPageBytes;
      const uint8_t* vp = kp + kPageBytes / 2;
      const int nk = min(KPP, sp.nc - pg * KPP);
      float sc[NKB][2];
#pragma unroll
      for (int kb = 0; kb < NKB; ++kb) {
        sc[kb][0] = sc[kb][1] = -INFINITY;
        if (kb * 8 < nk) {
          // key kb*8 + grp is column grp; odd keys load the two 64-byte halves
          // of each 128-byte stretch swapped (disjoint banks)
          const uint8_t* kr = kp + (size_t)(kb * 8 + grp) * (D * 2) + 16 * tig;
          float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j2 = 0; j2 < D / 64; ++j2) {
            const uint4 x = *reinterpret_cast<const uint4*>(kr + 128 * j2 + 64 * odd);
            const uint4 y = *reinterpret_cast<const uint4*>(kr + 128 * j2 + 64 * (odd ^ 1));
            const uint4 wl = odd ? y : x, wh = odd ? x : y;
            mma_bf16_16816(d0, qa[4 * j2], wl.x, wl.y);
            mma_bf16_16816(d1, qa[4 * j2 + 1], wl.z, wl.w);
            mma_bf16_16816(d0, qa[4 * j2 + 2], wh.x, wh.y);
            mma_bf16_16816(d1, qa[4 * j2 + 3], wh.z, wh.w);
          }
#pragma unroll
          for (int e = 0; e < 2; ++e)
            if (kb * 8 + 2 * tig + e < nk) sc[kb][e] = (d0[e] + d1[e]) + (d0[2 + e] + d1[2 + e]);
        }
      }
      // online softmax over the page (every page holds at least one key)
      float mx = -INFINITY;
#pragma unroll
      for (int kb = 0; kb < NKB; ++kb) mx = fmaxf(mx, fmaxf(sc[kb][0], sc[kb][1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float mnew = fmaxf(mrow, mx);
      const float alpha = fast_exp2(mrow - mnew);
      mrow = mnew;
      lsum *= alpha;
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[nb][e] *= alpha;
#pragma unroll
      for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          sc[kb][e] = fast_exp2(sc[kb][e] - mnew);  // -inf (no key): 0
          lsum += sc[kb][e];
        }
      // O += P V, 16 keys per step; V blocks of 8 keys x 8 columns transposed
      // by ldmatrix (lane l addresses row l % 8 of block l / 8). Rows past the
      // page's keys hold whatever the slot held before (possibly not a finite
      // number): their halves of the B fragments are zeroed, since a zero
      // weight would not cancel them.
#pragma unroll
      for (int t = 0; t < NKB / 2; ++t) {
        if (16 * t < nk) {
          const uint4 pa = split_hi_lo(sc[2 * t][0], sc[2 * t][1], sc[2 * t + 1][0], sc[2 * t + 1][1]);
          const uint8_t* vr = vp + (size_t)(16 * t + (lane & 7)) * (D * 2) + 16 * (lane >> 3);
          const int k0 = 16 * t + 2 * tig;  // this lane's keys: k0, k0 + 1, k0 + 8, k0 + 9
          const uint32_t m0 = (k0 < nk ? 0xffffu : 0u) | (k0 + 1 < nk ? 0xffff0000u : 0u);
          const uint32_t m1 = (k0 + 8 < nk ? 0xffffu : 0u) | (k0 + 9 < nk ? 0xffff0000u : 0u);
#pragma unroll
          for (int nq = 0; nq < NB / 4; ++nq) {
            uint32_t b0[4], b1[4];
            ldsm_x4_trans(b0, vr + 64 * nq);                  // keys 16t .. +7
            ldsm_x4_trans(b1, vr + 64 * nq + 8 * (D * 2));    // keys 16t + 8 .. +15
#pragma unroll
            for (int i = 0; i < 4; ++i) mma_bf16_16816(o[4 * nq + i], pa, b0[i] & m0, b1[i] & m1);
          }
        }
      }
    }
    // a page whose copy has not landed (after an abort) is never handed back
    __syncwarp();
    if (lane == 0 && ok) mbar_arrive_cnt(&m->empty[slot], kComputeWarps);
    slot += kComputeWarps;
    if (slot >= p.n_pages) {
      slot -= p.n_pages;
      ++round;
    }
  }
  lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
  lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);

  // scratch [share][h][D + 2] in the activation staging area
  float* scr = reinterpret_cast<float*>(smem + p.off_x);
  compute_bar();  // previous readers of the staging area are done
  if (grp < G) {
    float* e = scr + ((size_t)r0 * G + grp) * (D + 2);
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      e[8 * nb + 2 * tig] = o[nb][0] + o[nb][2];
      e[8 * nb + 2 * tig + 1] = o[nb][1] + o[nb][3];
    }
    if (tig == 0) {
      e[D] = mrow;
      e[D + 1] = lsum;
    }
  }
  compute_bar();
  const int tid = compute_tid();
  for (int idx = tid; idx < G * D; idx += kComputeThreads) {
    const int h = idx / D, d = idx - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kComputeWarps; ++w) M = fmaxf(M, scr[((size_t)w * G + h) * (D + 2) + D]);
    float acc = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < kComputeWarps; ++w) {
      const float* e = scr + ((size_t)w * G + h) * (D + 2);
      const float wt = e[D] == -INFINITY ? 0.f : fast_exp2(e[D] - M);
      acc = fmaf(wt, e[d], acc);
      den = fmaf(wt, e[D + 1], den);
    }
    const size_t prow = ((size_t)b * p.nh + g * G + h) * kMaxPartitions + pidx;
    p.part[prow * D + d] = acc;
    if (d == 0) {
      p.part_ml[prow * 2] = M;
      p.part_ml[prow * 2 + 1] = den;
    }
  }
}

// ---------------------------------------------------------------------------
// compute role: attention partial reduction (instruction 3)
// ---------------------------------------------------------------------------

template <int D>
__device__ __forceinline__ void attn_reduce(const Params& p, const Instr& in) {
  constexpr int PL = D / 32;  // dims per lane
  constexpr int kU = 8;       // partitions whose o rows load together
  const int warp = compute_warp(), lane = threadIdx.x & 31;
  const int b = in.a0, g = in.a1, P = in.a2;
  for (int hl = warp; hl < p.G; hl += kComputeWarps) {
    const int h = g * p.G + hl;
    const float* base = p.part + ((size_t)b * p.nh + h) * kMaxPartitions * D;
    const float* ml = p.part_ml + ((size_t)b * p.nh + h) * kMaxPartitions * 2;
    // lane k (and k + 32) holds partition k's (m, l); P <= kMaxPartitions = 64
    float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;
    if (lane < P) {
      const float2 v = __ldcg(reinterpret_cast<const float2*>(ml + 2 * lane));
      m0 = v.x;
      l0 = v.y;
    }
    if (lane + 32 < P) {
      const float2 v = __ldcg(reinterpret_cast<const float2*>(ml + 2 * (lane + 32)));
      m1 = v.x;
      l1 = v.y;
    }
    float M = fmaxf(m0, m1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float w0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - M);
    const float w1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - M);
    float den = w0 * l0 + w1 * l1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    float acc[PL];
#pragma unroll
    for (int e = 0; e < PL; ++e) acc[e] = 0.f;
    for (int k0 = 0; k0 < P; k0 += kU) {
      float o[kU][PL];
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int e = 0; e < PL; ++e)
          o[u][e] = k0 + u < P ? __ldcg(base + (size_t)(k0 + u) * D + lane * PL + e) : 0.f;
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int k = k0 + u;  // its weight sits in lane k % 32 of w0 (k < 32) or w1
        const float wa = __shfl_sync(0xffffffffu, w0, k & 31);
        const float wb = __shfl_sync(0xffffffffu, w1, k & 31);
        const float wt = k < P ? (k < 32 ? wa : wb) : 0.f;
#pragma unroll
        for (int e = 0; e < PL; ++e) acc[e] = fmaf(wt, o[u][e], acc[e]);
      }
    }
    const float inv = 1.f / den;
    float* dst = p.attn + (size_t)b * p.QD + (size_t)h * D + lane * PL;
    const uint32_t st = stamp_of(p, step_of(in), layer_of(in));
#pragma unroll
    for (int e = 0; e < PL; ++e) st_relaxed(dst + e, stamped(acc[e] * inv, st));
  }
}

// ---------------------------------------------------------------------------
// compute role: the instruction loop
// ---------------------------------------------------------------------------

template <int B, int DS, int GS, int KW, int FX>
__device__ void compute_role(const Params& p, Misc* m, uint8_t* smem, const Instr* q, int n,
                             int qbase) {
  const int warp = compute_warp(), lane = threadIdx.x & 31;
  Staged st;
  // per-warp activation registers (one sequence, rows <= 2048 columns),
  // reloaded from the staged smem vector at every instruction
  float ax[64];
  uint32_t page_cnt = 0;
  uint32_t seq = 0;   // instructions (dynamic tickets included) handed to the storer
  uint32_t tk_n = 0;  // tickets read
  int known_ctr = -1, known_tgt = 0;
  Instr nxt = n > 0 ? load_instr(q) : Instr{};
  Instr in0 = nxt;
  int adv = 1;  // 0 while a dynamic instruction still has tickets
  for (int i = 0; i < n; i += adv) {
    if (adv) {
      in0 = nxt;
      if (i + 1 < n) nxt = load_instr(q + i + 1);
    }
    Instr in = in0;
    adv = 1;
    if ((FX & kFxDyn) && is_dyn(in0)) {
      // warp 0 reads the loader's ticket and passes it to the other warps
      const int slot = (int)(tk_n % kTk);
      if (warp == 0 && lane == 0) {
        int t = -1;
        if (wait_mbar(p, m, &m->tk_full[slot], (tk_n / kTk) & 1u, kErrTimeoutRes))
          t = *reinterpret_cast<volatile int*>(&m->tk[slot]);
        *reinterpret_cast<volatile int*>(&m->tk_cur[tk_n & 1u]) = t;
        mbar_arrive(&m->tk_empty[slot]);
      }
      compute_bar();
      const int t = *reinterpret_cast<volatile int*>(&m->tk_cur[tk_n & 1u]);
      ++tk_n;
      if (t < 0) continue;
      in = dyn_item(in0, t);
      adv = 0;
    }
    const int buf = (int)(seq % kResBufs);
    const uint32_t rpar = (seq / kResBufs) & 1u;
    ++seq;
    uint64_t t_start = 0, t_ready = 0, pwait = 0;
    const bool tracing = p.trace != nullptr && warp == 0 && lane == 0;
    if (tracing) t_start = globaltimer();
    if (warp == 0 && lane == 0 && critical_op(in))
      *reinterpret_cast<volatile int*>(&m->hold) = i;
    // 1. dependency: one thread polls, the other compute warps meet it at a
    // barrier. An instruction whose inputs are all stamped words and small
    // polls the words themselves instead (the attention's q and new k/v rows;
    // with one sequence also the gate/up's xa, the down-projection's chunk of
    // h, and the QKV staging's x where it is written whole): the counter
    // would only add a round trip. (Polling x's five sources, or eight
    // sequences' x, was slower: 613.5 vs 607.0 and 1491.1 vs 1426.7 us/step.)
    const bool polls_inputs =
        in.op == MK_OP_ATTN || (B == 1 && (in.op == MK_OP_GATEUP || in.op == MK_OP_DOWN)) ||
        (B == 1 && in.op == MK_OP_QKV && layer_of(in) > 0 && x_whole<B>(p) && !(FX & kFxPaged));
    if (!p.no_waits && in.wait_ctr >= 0 && !polls_inputs &&
        !(in.wait_ctr == known_ctr && in.wait_target <= known_tgt)) {
      if (warp == 0 && lane == 0) wait_counter(p, m, in.wait_ctr, in.wait_target);
      compute_bar();
      known_ctr = in.wait_ctr;
      known_tgt = in.wait_target;
    }
    if (tracing) t_ready = globaltimer();
    // 2. the result buffer this instruction hands to the storer must be free
    const bool res_ok = wait_mbar(p, m, &m->res_empty[buf], rpar ^ 1u, kErrTimeoutRes);
    const uint64_t t_res = tracing ? globaltimer() : 0;
    uint64_t t_staged = t_res;
    float* res = reinterpret_cast<float*>(smem + p.off_res) + (size_t)buf * p.res_floats;

    if (is_gemv(in.op)) {
      const int kind = act_kind(in.op);
      const int chunk = in.op == MK_OP_DOWN ? in.a2 : 0;
      const int key = act_key(kind, in.layer, chunk);
      const bool to_h = kind == kActH;
      const Geom g = geom_of(in.op, p.H, p.QD, p.Fc);
      const bool regs = B == 1 && g.K <= 2048;
      const bool norm = kind == kActAttnNorm || kind == kActMlpNorm || kind == kActFinalNorm;
      const float* act;
      {
        if ((to_h ? st.key_h : st.key_x) != key) {
          bool staged = false;
          if constexpr (B == 1) {  // one sequence: the O-projection reduces while staging
            if (kind == kActAttnOut && p.fused_red) {
              if constexpr (DS > 0) stage_attn_fused<DS>(p, smem, st, layer_of(in), in.a2, key);
              else if (p.D == 64) stage_attn_fused<64>(p, smem, st, layer_of(in), in.a2, key);
              else stage_attn_fused<128>(p, smem, st, layer_of(in), in.a2, key);
              staged = true;
            }
          }
          if (!staged)
            stage<B, FX, (B == 1 && KW == 0), KW>(p, m, smem, st, kind, layer_of(in), chunk, key,
                                               step_of(in));
        }
        act = reinterpret_cast<const float*>(smem + (to_h ? p.off_h : p.off_x));
      }
      if (tracing) t_staged = globaltimer();
      InvScale one;
#pragma unroll
      for (int b = 0; b < kMaxBatch; ++b) one.v[b] = 1.f;
      if (regs) {
        // 2048 columns: the staged B fragments (the 1/rms of the norms
        // scales the results); narrower rows: fp32 values scaled here
        const bool mma = KW == 2048 || g.K == 2048;
        if (mma) load_frag(ax, reinterpret_cast<const uint32_t*>(act));
        else load_regs(ax, act, norm ? st.inv_x.v[0] : 1.f, g.K);
        gemv_run<B, true, KW>(p, m, smem, in, g, act, mma && norm ? st.inv_x : one, ax, res,
                              page_cnt, pwait);
      } else {
        if constexpr (KW == 0)
          gemv_run<B, false, KW>(p, m, smem, in, g, act, to_h ? one : st.inv_x, ax, res, page_cnt,
                                  pwait);
      }
      page_cnt += (uint32_t)((in.a1 - in.a0 + g.ipp - 1) / g.ipp);
    } else if (in.op == MK_OP_ATTN) {
      st.key_x = -1;  // the staging area becomes scratch
      st.key_h = -1;
      // runs even after an abort: its loads stay in bounds and its barriers
      // must be met by every compute warp
      if constexpr (DS > 0) attn_unit<DS, FX>(p, m, smem, in, page_cnt, pwait);
      else if (p.D == 64) attn_unit<64, FX>(p, m, smem, in, page_cnt, pwait);
      else attn_unit<128, FX>(p, m, smem, in, page_cnt, pwait);
      page_cnt += (uint32_t)attn_span(p.pos[in.a0] + step_of(in), in.a2 >> 16, in.a2 & 0xffff, p.D)
                      .npages;
    } else if (in.op == MK_OP_RED) {
      // the reduction instruction: several sequences, or one sequence with
      // more than 2048 attention columns (the one-sequence kernel of head
      // dimension 64 reduces in the O-projection's staging and omits it)
      if constexpr (B > 1 || DS != 64) if (!aborted(m)) {
        if constexpr (DS > 0) attn_reduce<DS>(p, in);
        else if (p.D == 64) attn_reduce<64>(p, in);
        else attn_reduce<128>(p, in);
      }
    }
    (void)res_ok;
    // 3. hand the instruction to the storer
    __syncwarp();
    if (lane == 0) mbar_arrive(&m->res_full[buf]);
    if (tracing) {
      const int rec = p.trace_base + qbase + i;
      if (rec < p.trace_cap) {
        // field by field: the storer writes t_stored of the same record
        mk_trace_record* r = p.trace + rec;
        r->sm = blockIdx.x;
        r->index = (uint32_t)i;
        r->op = in.op;
        r->layer = in.layer;
        r->t_start = t_start;
        r->t_ready = t_ready;
        r->t_end = globaltimer();
        r->res_wait_ns = (uint32_t)(t_res - t_ready);
        r->stage_ns = (uint32_t)(t_staged - t_res);
        r->page_wait_ns = (uint32_t)pwait;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// storer role
// ---------------------------------------------------------------------------

__device__ __forceinline__ float silu(float z) { return z / (1.f + expf(-z)); }

// What an epilogue reads from global memory, loaded by the storer while the
// compute warps still work on the instruction: the RoPE (cos, sin) of the
// q/k/v pairs, and the residual rows of the o-projection (the previous
// layer's output x = xa + its four down-projection shares, or the embedding
// row). Lane l holds items l and l + 32 (at most 64 items).
template <int B>
struct EpiPre {
  float2 v[2][B];
};

// The storer's rows j = in.a0 + lane (+ 32) of every sequence: the sum of NS
// stamped sources, xa and xpart[0..NS-2] (NS > 1) or x alone (NS = 1), left
// to right, into pre.v[k][b].x. All loads are issued first, then the stamps
// are tested, and the whole set is loaded again if one was stale.
template <int B, int NS>
__device__ __forceinline__ void load_stamped_rows(const Params& p, Misc* m, const Instr& in,
                                                  int items, uint32_t st, EpiPre<B>& pre) {
  const int lane = threadIdx.x & 31;
  const size_t cs = (size_t)p.B * p.H;
  float r[2][B][NS];
  uint32_t tries = 0;
  uint64_t t0 = 0;
  for (;;) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int it = lane + 32 * k;
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const size_t o = (size_t)b * p.H + in.a0 + it;
#pragma unroll
        for (int c = 0; c < NS; ++c) {
          r[k][b][c] = 0.f;
          if (it < items)
            r[k][b][c] = ld_relaxed(NS == 1 ? p.x + o : (c == 0 ? p.xa + o : p.xpart + (c - 1) * cs + o));
        }
      }
    }
    bool bad = false;
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
      for (int b = 0; b < B; ++b)
#pragma unroll
        for (int c = 0; c < NS; ++c)
          if (lane + 32 * k < items) bad |= stale1(r[k][b][c], st);
    if (!bad || !retry_stale(p, m, tries, t0)) break;
  }
#pragma unroll
  for (int k = 0; k < 2; ++k)
#pragma unroll
    for (int b = 0; b < B; ++b) {
      float acc = clear1(r[k][b][0]);
#pragma unroll
      for (int c = 1; c < NS; ++c) acc += clear1(r[k][b][c]);
      pre.v[k][b].x = acc;
    }
}

template <int B, int FX>
__device__ __forceinline__ void epilogue_prefetch(const Params& p, Misc* m, const Instr& in,
                                                  EpiPre<B>& pre) {
  const int lane = threadIdx.x & 31;
  const int items = in.a1 - in.a0;
  if (in.op == MK_OP_QKV) {
    const int half = p.D / 2;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int it = lane + 32 * k;
      if (it < items) {
        const PairRows pr = pair_rows(in.a0 + it, p.G, p.D);
        if (pr.which < 2) {
#pragma unroll
          for (int b = 0; b < B; ++b)
            pre.v[k][b] = __ldg(p.rope + (size_t)(p.pos[b] + step_of(in)) * half + pr.i);
        }
      }
    }
  } else if (in.op == MK_OP_OPROJ) {
    const bool from_embed = layer_of(in) == 0;
    if (from_embed && (FX & kFxPaged) && step_of(in) > 0 && !p.no_waits && in.wait_ctr >= 0) {
      // greedy decode: the token is the previous step's argmax, complete
      // once that step's LM head is (the instruction's input counter follows
      // it); acquire that counter (the compute warps wait on it too)
      bool ok = true;
      if (lane == 0) ok = wait_counter(p, m, in.wait_ctr, in.wait_target);
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) return;
      __syncwarp();  // lane 0's acquire, then every lane's loads
    }
    // the residual, the previous layer's output x: stamped words, complete
    // before this layer's QKV instructions started, so read without waiting
    // on a counter (all loads first, then the stamp test, again if stale)
    if (from_embed) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int it = lane + 32 * k;
        if (it < items) {
#pragma unroll
          for (int b = 0; b < B; ++b)
            pre.v[k][b].x =
                bf16f(p.embed[(size_t)token_of<FX>(p, b, step_of(in)) * p.H + in.a0 + it]);
        }
      }
    } else {
      const uint32_t st = stamp_of(p, step_of(in), layer_of(in) - 1);
      if (x_whole<B>(p)) {
        load_stamped_rows<B, 1>(p, m, in, items, st, pre);
      } else {
        load_stamped_rows<B, 1 + kChunks>(p, m, in, items, st, pre);
        // the layer output as the chunk-3 storer would have written it
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
          for (int b = 0; b < B; ++b) pre.v[k][b].x = clear1(pre.v[k][b].x);
      }
    }
  } else if (in.op == MK_OP_DOWN && in.a2 == kChunks - 1 && x_whole<B>(p)) {
    // chunk 3: its rows' xa and shares of chunks 0..2, written this layer
    // by other SMs' storers (polled), summed in order; the epilogue adds
    // this instruction's share and writes x
    load_stamped_rows<B, kChunks>(p, m, in, items, stamp_of(p, step_of(in), layer_of(in)), pre);
  }
}

template <int B, int FX>
__device__ __forceinline__ void epilogue(const Params& p, const Instr& in, const float* res,
                                         const EpiPre<B>& pre) {
  const int lane = threadIdx.x & 31;
  const Geom g = geom_of(in.op, p.H, p.QD, p.Fc);
  const int items = in.a1 - in.a0;
  const LayerPtrs& L = p.layers[layer_of(in)];
  const uint32_t st = stamp_of(p, step_of(in), layer_of(in));
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int it = lane + 32 * k;
    if (it >= items) continue;
    const int j = in.a0 + it;
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const float v0 = res[((size_t)it * g.R) * B + b];
      const float v1 = g.R == 2 ? res[((size_t)it * g.R + 1) * B + b] : 0.f;
      switch (in.op) {
        case MK_OP_QKV: {
          const PairRows pr = pair_rows(j, p.G, p.D);
          const int pos = p.pos[b] + step_of(in);
          const int half = p.D / 2;
          float o0 = v0, o1 = v1;
          if (pr.which < 2) {
            const float2 cs = pre.v[k][b];
            o0 = v0 * cs.x - v1 * cs.y;
            o1 = v1 * cs.x + v0 * cs.y;
          }
          if (pr.which == 0) {
            float* qd = p.q + (size_t)b * p.QD + (size_t)pr.head * p.D + pr.i;
            st_relaxed(qd, stamped(o0, st));
            st_relaxed(qd + half, stamped(o1, st));
          } else {
            uint16_t* c = (pr.which == 1 ? L.kc : L.vc) + kv_row<FX>(p, b, pr.head, pos) + pr.i;
            const uint16_t k0 = __bfloat16_as_ushort(__float2bfloat16_rn(o0));
            const uint16_t k1 = __bfloat16_as_ushort(__float2bfloat16_rn(o1));
            c[0] = k0;
            c[half] = k1;
            // the stamped copy the attention units of this step read
            float* w = p.kvn + ((size_t)(b * p.nkv + pr.head) * 2 + (pr.which - 1)) * p.D + pr.i;
            st_relaxed(w, __uint_as_float(((uint32_t)k0 << 16) | st));
            st_relaxed(w + half, __uint_as_float(((uint32_t)k1 << 16) | st));
          }
          break;
        }
        case MK_OP_OPROJ:
          st_relaxed(p.xa + (size_t)b * p.H + j, stamped(pre.v[k][b].x + v0, st));
          break;
        case MK_OP_GATEUP:
          st_relaxed(p.h + (size_t)b * p.F + j, stamped(silu(v0) * v1, st));
          break;
        case MK_OP_DOWN:
          // this chunk's share of row j, or (chunk 3, x written whole) the row of x
          if (in.a2 == kChunks - 1 && x_whole<B>(p))
            st_relaxed(p.x + (size_t)b * p.H + j, stamped(pre.v[k][b].x + clear1(v0), st));
          else
            st_relaxed(p.xpart + ((size_t)in.a2 * p.B + b) * p.H + j, stamped(v0, st));
          break;
        default:  // MK_OP_LMHEAD
          p.logits[(size_t)b * p.V + j] = v0;
          break;
      }
    }
  }
  if ((FX & kFxPaged) && in.op == MK_OP_LMHEAD && p.argmax_out) {
    // greedy decode: the instruction's best row per sequence joins the
    // step's argmax (atomicMax of order-preserving keys: any order of the
    // SMs gives the same result)
#pragma unroll
    for (int b = 0; b < B; ++b) {
      unsigned long long best = 0ull;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int it = lane + 32 * k;
        if (it < items) {
          const uint32_t u = __float_as_uint(res[((size_t)it * g.R) * B + b]);
          const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
          const unsigned long long key =
              ((unsigned long long)ord << 32) | (0xffffffffu - (uint32_t)(in.a0 + it));
          best = key > best ? key : best;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
        best = o > best ? o : best;
      }
      if (lane == 0) atomicMax(p.argmax_out + (size_t)step_of(in) * B + b, best);
    }
  }
}

// The storer drains finished instructions in order: epilogue, then lane 0
// bumps the instruction's counter, with a release-add where a reader reads
// plain words after acquiring it and as a relaxed hint where the outputs are
// stamped words. What the epilogue needs from global memory is fetched
// before waiting for the compute warps, so the epilogue itself touches only
// registers and shared memory.
// (Publishing several instructions behind one fence was measured slower: it
// delays the first counter of each batch, which sits on the critical path.)
template <int B, int FX>
__device__ void storer_role(const Params& p, Misc* m, uint8_t* smem, const Instr* q, int n) {
  const int lane = threadIdx.x & 31;
  uint32_t seq = 0;   // instructions (dynamic tickets included) taken from the compute warps
  uint32_t tk_n = 0;  // tickets read
  Instr nxt = n > 0 ? load_instr(q) : Instr{};
  Instr in0 = nxt;
  int adv = 1;  // 0 while a dynamic instruction still has tickets
  for (int i = 0; i < n; i += adv) {
    if (adv) {
      in0 = nxt;
      if (i + 1 < n) nxt = load_instr(q + i + 1);
    }
    Instr in = in0;
    adv = 1;
    if ((FX & kFxDyn) && is_dyn(in0)) {
      const int slot = (int)(tk_n % kTk);
      int t = -1;
      if (lane == 0) {
        if (wait_mbar(p, m, &m->tk_full[slot], (tk_n / kTk) & 1u, kErrTimeoutRes))
          t = *reinterpret_cast<volatile int*>(&m->tk[slot]);
        mbar_arrive(&m->tk_empty[slot]);
      }
      t = __shfl_sync(0xffffffffu, t, 0);
      ++tk_n;
      if (t < 0) continue;
      in = dyn_item(in0, t);
      adv = 0;
    }
    const int buf = (int)(seq % kResBufs);
    const uint32_t par = (seq / kResBufs) & 1u;
    ++seq;
    EpiPre<B> pre;
    if (is_gemv(in.op) && !aborted(m)) epilogue_prefetch<B, FX>(p, m, in, pre);
    const bool ok = wait_mbar(p, m, &m->res_full[buf], par, kErrTimeoutRes);
    if (ok && !aborted(m)) {
      const float* res = reinterpret_cast<const float*>(smem + p.off_res) + (size_t)buf * p.res_floats;
      if (is_gemv(in.op)) epilogue<B, FX>(p, in, res, pre);
      if (in.sig_ctr >= 0) {
        // Outputs read as plain words after an acquire of this counter go
        // out with a release-add: the warp barrier orders the other lanes'
        // stores (and, through the result mbarrier, the compute warps'
        // stores) before lane 0's release, which publishes them at GPU scope.
        // Those are the attention partials; with the paged-cache / greedy
        // code also the KV rows a later step of the same launch fetches with
        // bulk copies (after acquiring the LM head's count, released too),
        // and in a prefill step the chunk's KV rows, which the loader fetches
        // after the QKV counter. Every other output is stamped words, and its
        // count is a scheduling hint bumped without the release, whose fence
        // would wait for this SM's weight copies in flight.
        const bool release = in.op == MK_OP_ATTN ||
                             ((FX & kFxPaged) && (in.op == MK_OP_QKV || in.op == MK_OP_LMHEAD)) ||
                             (in.op == MK_OP_QKV && p.prefill);
        __syncwarp();
        if (lane == 0) {
          if (release) red_release_add(p.ctr + in.sig_ctr, in.sig_amount);
          else red_relaxed_add(p.ctr + in.sig_ctr, in.sig_amount);
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&m->res_empty[buf]);
      *reinterpret_cast<volatile int*>(&m->published) = i + 1;
      if (p.trace) {
        const int rec = p.trace_base + (int)(q - p.instrs) + i;
        if (rec < p.trace_cap) p.trace[rec].t_stored = globaltimer();
      }
    }
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

template <int B, int DS, int GS, int KW, int FX>
__global__ void __launch_bounds__(kThreads, 1) interp_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Misc* m = reinterpret_cast<Misc*>(smem + p.off_misc);
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.n_pages; ++i) {
      mbar_init(&m->full[i], 1);
      // a GEMV page's owner warp releases it with all kComputeWarps arrivals;
      // an attention page is released by every compute warp, one each
      mbar_init(&m->empty[i], kComputeWarps);
    }
    for (int i = 0; i < kResBufs; ++i) {
      mbar_init(&m->res_full[i], kComputeWarps);
      mbar_init(&m->res_empty[i], 1);
    }
    mbar_init(&m->bt_full, 1);
    for (int i = 0; i < kTk; ++i) {
      mbar_init(&m->tk_full[i], 1);   // the loader
      mbar_init(&m->tk_empty[i], 2);  // compute warp 0 and the storer
    }
    m->abort = 0;
    m->hold = -1;
    m->published = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // counters are zero before the launch that uses them (§3.4): this launch
  // clears the set the next step will use
  if (p.ctr_zero)
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < p.n_ctr; i += gridDim.x * blockDim.x)
      p.ctr_zero[i] = 0;
  __syncthreads();
  const int q0 = p.sm_off[blockIdx.x];
  const int n = p.sm_off[blockIdx.x + 1] - q0;
  const Instr* q = p.instrs + q0;
  const int warp = threadIdx.x >> 5;
  if (warp == kLoaderWarp) loader_role<FX>(p, m, smem, q, n);
  else if (warp == kStorerWarp) storer_role<B, FX>(p, m, smem, q, n);
  else compute_role<B, DS, GS, KW, FX>(p, m, smem, q, n, q0);
}

}  // namespace mk
