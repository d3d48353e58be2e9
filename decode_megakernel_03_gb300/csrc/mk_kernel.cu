// The decode interpreter: one persistent CTA per SM walks its pre-planned
// instruction queue ("3 · L'interpréteur sur GPU", §3.2). Every instruction is
// split over three warp roles that walk the same queue independently:
//
//   loader  (1 warp)   streams the instruction's bf16 weight rows into 16 KB
//                      shared-memory pages with bulk asynchronous copies; it
//                      waits only for free pages, never for counters, so the
//                      next instruction's weights load while the current one
//                      still waits or computes (§3.3, the page allocator);
//   compute (6 warps)  waits for the instruction's input counter, stages the
//                      activations, and runs the dot products / attention;
//                      each page is handed back as soon as it has been read;
//   storer  (1 warp)   applies the epilogue (RoPE + KV append, residual adds,
//                      SiLU, chunk accumulation), writes the outputs, then
//                      fences and bumps the output counter with release
//                      semantics (§3.4, counters in global memory).
//
// The same kernel also serves the multi-launch comparison build: launched once
// per (layer, instruction type) with counter waits switched off, kernel
// boundaries order the work instead.
//
// Every wait (counter, page, result buffer) is bounded by a %globaltimer
// deadline; on expiry the kernel records MK_ERR_TIMEOUT in the error word,
// the other CTAs notice it and all of them drain their copies and return.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mk_isa.h"
#include "mk_ptx.cuh"

namespace mk {

struct Misc {
  uint64_t full[kMaxPages];
  uint64_t empty[kMaxPages];
  uint64_t res_full[2];
  uint64_t res_empty[2];
  float red[2][kComputeWarps][kMaxBatch];  // RMSNorm partial sums, double-buffered
  int abort;
};

constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kBarCompute = 1;

__device__ __forceinline__ void compute_bar() { named_bar(kBarCompute, kComputeThreads); }

__device__ __forceinline__ bool aborted(const Misc* m) {
  return *reinterpret_cast<const volatile int*>(&m->abort) != 0;
}

__device__ __noinline__ void raise_error(const Params& p, Misc* m, int code) {
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

// Bounded wait for counter >= target (acquire). One thread polls.
__device__ __noinline__ bool wait_counter(const Params& p, Misc* m, int ctr, int target) {
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

// ---------------------------------------------------------------------------
// weight rows of a GEMV item
// ---------------------------------------------------------------------------

__device__ __forceinline__ const uint16_t* row_src(const Params& p, const Instr& in, int item,
                                                   int r) {
  const LayerPtrs& L = p.layers[in.layer];
  switch (in.op) {
    case MK_OP_QKV: {
      PairRows pr = pair_rows(item, p.G, p.D);
      const uint16_t* W = pr.which == 0 ? L.wq : (pr.which == 1 ? L.wk : L.wv);
      int row = pr.head * p.D + pr.i + r * (p.D / 2);
      return W + (size_t)row * p.H;
    }
    case MK_OP_OPROJ:
      return L.wo + (size_t)item * p.QD;
    case MK_OP_GATEUP:
      return (r == 0 ? L.wgate : L.wup) + (size_t)item * p.H;
    case MK_OP_DOWN:
      return L.wdown + (size_t)item * p.F + (size_t)in.a2 * p.Fc;
    default:  // MK_OP_LMHEAD
      return p.lm + (size_t)item * p.H;
  }
}

// ---------------------------------------------------------------------------
// loader role
// ---------------------------------------------------------------------------

__device__ void loader_role(const Params& p, Misc* m, uint8_t* smem, const Instr* q, int n) {
  const int lane = threadIdx.x & 31;
  if (lane != 0) return;
  const uint64_t pol = policy_evict_first();
  uint32_t page_cnt = 0;
  bool ok = true;
  for (int i = 0; i < n && ok; ++i) {
    const Instr in = q[i];
    if (!is_gemv(in.op)) continue;
    const Geom g = geom_of(in.op, p.H, p.QD, p.Fc, p.B);
    const int items = in.a1 - in.a0;
    const int npages = (items + g.ipp - 1) / g.ipp;
    const uint32_t row_bytes = (uint32_t)g.K * 2u;
    for (int pg = 0; pg < npages; ++pg, ++page_cnt) {
      const int slot = (int)(page_cnt % (uint32_t)p.n_pages);
      const uint32_t round = page_cnt / (uint32_t)p.n_pages;
      if (!wait_mbar(p, m, &m->empty[slot], (round & 1u) ^ 1u, kErrTimeoutPage)) {
        ok = false;
        break;
      }
      const int i0 = pg * g.ipp;
      const int i1 = min(items, i0 + g.ipp);
      mbar_arrive_expect_tx(&m->full[slot], (uint32_t)((i1 - i0) * g.R) * row_bytes);
      uint8_t* dst = smem + (size_t)slot * kPageBytes;
      for (int it = i0; it < i1; ++it)
        for (int r = 0; r < g.R; ++r) {
          bulk_g2s_hint(dst, row_src(p, in, in.a0 + it, r), row_bytes, &m->full[slot], pol);
          dst += row_bytes;
        }
    }
  }
  if (!ok) {
    // drain: every issued copy must land before the CTA's shared memory goes away
    const uint32_t first = page_cnt > (uint32_t)p.n_pages ? page_cnt - p.n_pages : 0u;
    for (uint32_t k = first; k < page_cnt; ++k) {
      const int slot = (int)(k % (uint32_t)p.n_pages);
      const uint32_t par = (k / (uint32_t)p.n_pages) & 1u;
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(&m->full[slot], par)) {
        if (globaltimer() - t0 > p.timeout_ns) break;
      }
    }
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

struct Staged {
  int key_x = -1;     // what the x buffer holds
  int key_h = -1;     // what the h buffer holds
  int stage_cnt = 0;  // parity of the RMSNorm partial-sum buffer
  float inv[kMaxBatch];
};

__device__ __forceinline__ int act_key(int kind, int layer, int chunk) {
  return (kind << 20) | (layer << 4) | chunk;
}

// Stages the activation vector(s) of `kind` for all B sequences into the x or
// h buffer; for the RMSNorm kinds also computes 1/rms per sequence.
__device__ __forceinline__ void stage(const Params& p, Misc* m, uint8_t* smem, Staged& st, int kind, int layer,
                      int chunk) {
  const int tid = threadIdx.x;  // 0..255 within the compute warps
  const int warp = tid >> 5, lane = tid & 31;
  const bool to_h = kind == kActH;
  float* dst = reinterpret_cast<float*>(smem + (to_h ? p.off_h : p.off_x));
  const int K = kind == kActAttnOut ? p.QD : (to_h ? p.Fc : p.H);
  const bool norm = kind == kActAttnNorm || kind == kActMlpNorm || kind == kActFinalNorm;
  const int par = st.stage_cnt & 1;
  compute_bar();  // everyone is done reading the buffer's previous contents
  for (int b = 0; b < p.B; ++b) {
    float ss = 0.f;
    for (int c = tid * 4; c < K; c += kComputeThreads * 4) {
      float4 v;
      if (kind == kActAttnNorm && layer == 0) {
        const uint2 e = *reinterpret_cast<const uint2*>(p.embed + (size_t)p.tok[b] * p.H + c);
        v = make_float4(bf_lo(e.x), bf_hi(e.x), bf_lo(e.y), bf_hi(e.y));
      } else {
        const float* src;
        if (kind == kActAttnNorm || kind == kActFinalNorm) src = p.x + (size_t)b * p.H;
        else if (kind == kActMlpNorm) src = p.xa + (size_t)b * p.H;
        else if (kind == kActAttnOut) src = p.attn + (size_t)b * p.QD;
        else src = p.h + (size_t)b * p.F + (size_t)chunk * p.Fc;
        v = __ldcg(reinterpret_cast<const float4*>(src + c));
      }
      *reinterpret_cast<float4*>(dst + (size_t)b * K + c) = v;
      ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    if (norm) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) m->red[par][warp][b] = ss;
    }
  }
  compute_bar();
  if (norm) {
    for (int b = 0; b < p.B; ++b) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kComputeWarps; ++w) s += m->red[par][w][b];
      st.inv[b] = rsqrtf(s / (float)p.H + p.eps);
    }
  }
  st.stage_cnt++;
  const int key = act_key(kind, layer, chunk);
  if (to_h) {
    st.key_h = key;
    if (p.alias_xh) st.key_x = -1;
  } else {
    st.key_x = key;
    if (p.alias_xh) st.key_h = -1;
  }
}

// ---------------------------------------------------------------------------
// compute role: GEMV pieces
// ---------------------------------------------------------------------------
// A "piece" is (item, row of the item, segment): one warp dots one 256*J-long
// segment of one weight row with the matching activations of all B sequences.
// Lane l holds columns seg*256J + j*256 + l*8 + e (e < 8) in registers, so each
// j reads 512 contiguous bytes of the page per warp. Pieces are dealt to warps
// round-robin; every warp walks every page in order (wait full -> its pieces
// -> arrive empty) so a page is released as soon as all warps are past it.

// J (256-column blocks per warp segment) is a runtime value <= JM = 8 / B;
// the loops below are unrolled to JM and predicated on J so the activation
// registers stay statically indexed and one body serves every row length.
template <int B>
__device__ __forceinline__ void load_act(float (&a)[B][64 / B], int J, const float* buf, int K,
                                         int seg, const uint16_t* normw, const float* inv,
                                         int lane) {
  constexpr int JM = 8 / B;
#pragma unroll
  for (int j = 0; j < JM; ++j) {
    if (j < J) {
      const int col = seg * 256 * J + j * 256 + lane * 8;
      float w8[8] = {1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f};
      if (normw) {
        const uint4 wv = __ldg(reinterpret_cast<const uint4*>(normw + col));
        w8[0] = bf_lo(wv.x); w8[1] = bf_hi(wv.x); w8[2] = bf_lo(wv.y); w8[3] = bf_hi(wv.y);
        w8[4] = bf_lo(wv.z); w8[5] = bf_hi(wv.z); w8[6] = bf_lo(wv.w); w8[7] = bf_hi(wv.w);
      }
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const float4 x0 = *reinterpret_cast<const float4*>(buf + (size_t)b * K + col);
        const float4 x1 = *reinterpret_cast<const float4*>(buf + (size_t)b * K + col + 4);
        const float sc = normw ? inv[b] : 1.f;
        a[b][j * 8 + 0] = x0.x * sc * w8[0];
        a[b][j * 8 + 1] = x0.y * sc * w8[1];
        a[b][j * 8 + 2] = x0.z * sc * w8[2];
        a[b][j * 8 + 3] = x0.w * sc * w8[3];
        a[b][j * 8 + 4] = x1.x * sc * w8[4];
        a[b][j * 8 + 5] = x1.y * sc * w8[5];
        a[b][j * 8 + 6] = x1.z * sc * w8[6];
        a[b][j * 8 + 7] = x1.w * sc * w8[7];
      }
    } else {
#pragma unroll
      for (int b = 0; b < B; ++b)
#pragma unroll
        for (int e = 0; e < 8; ++e) a[b][j * 8 + e] = 0.f;
    }
  }
}

template <int B>
__device__ __forceinline__ void gemv_run(const Params& p, Misc* m, uint8_t* smem, const Instr& in,
                                         const Geom& g, const float* act, const uint16_t* normw,
                                         const float* inv, float* res, uint32_t page_base) {
  constexpr int JM = 8 / B;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int J = g.J;
  const int items = in.a1 - in.a0;
  const int npages = (items + g.ipp - 1) / g.ipp;
  const int ppi = g.R * g.nseg;  // pieces per item
  const int npieces = items * ppi;
  const int row_bytes = g.K * 2;
  float a[B][64 / B];
  int loaded = -1;
  int piece = warp;
  for (int pg = 0; pg < npages; ++pg) {
    const uint32_t pc = page_base + (uint32_t)pg;
    const int slot = (int)(pc % (uint32_t)p.n_pages);
    const bool ok = wait_mbar(p, m, &m->full[slot], (pc / (uint32_t)p.n_pages) & 1u,
                              kErrTimeoutPage);
    const int piece_end = min(npieces, (pg + 1) * g.ipp * ppi);
    const uint8_t* page = smem + (size_t)slot * kPageBytes;
    for (; piece < piece_end; piece += kComputeWarps) {
      if (!ok) continue;
      const int item = piece / ppi;
      const int rr = piece - item * ppi;
      const int r = rr / g.nseg;
      const int seg = rr - r * g.nseg;
      if (seg != loaded) {
        load_act<B>(a, J, act, g.K, seg, normw, inv, lane);
        loaded = seg;
      }
      const uint8_t* rowp =
          page + (size_t)((item - pg * g.ipp) * g.R + r) * row_bytes + (size_t)seg * J * 512;
      uint4 wv[JM];
#pragma unroll
      for (int j = 0; j < JM; ++j)
        wv[j] = j < J ? *reinterpret_cast<const uint4*>(rowp + j * 512 + lane * 16)
                      : make_uint4(0, 0, 0, 0);
      float acc[B];
#pragma unroll
      for (int b = 0; b < B; ++b) acc[b] = 0.f;
#pragma unroll
      for (int j = 0; j < JM; ++j) {
        const float wf[8] = {bf_lo(wv[j].x), bf_hi(wv[j].x), bf_lo(wv[j].y), bf_hi(wv[j].y),
                             bf_lo(wv[j].z), bf_hi(wv[j].z), bf_lo(wv[j].w), bf_hi(wv[j].w)};
#pragma unroll
        for (int e = 0; e < 8; ++e)
#pragma unroll
          for (int b = 0; b < B; ++b) acc[b] = fmaf(wf[e], a[b][j * 8 + e], acc[b]);
      }
#pragma unroll
      for (int b = 0; b < B; ++b) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], o);
      }
      if (lane == 0) {
#pragma unroll
        for (int b = 0; b < B; ++b) res[(size_t)piece * B + b] = acc[b];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&m->empty[slot]);
  }
}

// ---------------------------------------------------------------------------
// compute role: split-KV attention partial (instruction 2)
// ---------------------------------------------------------------------------
// Unit (b, g, p): the G q-heads of kv-head g over keys [t0, t1) of sequence b.
// A key row of D bf16 is read by D/8 lanes with one 16-byte load each, so a
// warp covers 256/D keys per load; per (lane group, head) an online softmax
// keeps (m, l, o) in the log2 domain (q is pre-scaled by log2(e)/sqrt(D)).
// Warps combine through shared memory and write (o, m, l) for the partition.

__device__ __forceinline__ void softmax_merge(float& m, float& l, float* o, float m2, float l2,
                                              const float* o2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  const float s1 = exp2f(m - M), s2 = exp2f(m2 - M);
  l = l * s1 + l2 * s2;
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = o[e] * s1 + o2[e] * s2;
  m = M;
}

// GH heads per pass (G = 8 runs two passes over the same keys, which the
// second pass finds in L2).
template <int D, int GH>
__device__ __forceinline__ void attn_partial(const Params& p, uint8_t* smem, const Instr& in, int h0) {
  constexpr int LPT = D / 8;       // lanes per key row
  constexpr int TPI = 32 / LPT;    // keys per warp load
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = in.a0, g = in.a1, pidx = in.a2 >> 16, P = in.a2 & 0xffff;
  const int len = p.pos[b] + 1;
  const int t0 = (int)((long)pidx * len / P), t1 = (int)((long)(pidx + 1) * len / P);
  const int sub = lane % LPT, ti = lane / LPT;
  const LayerPtrs& L = p.layers[in.layer];
  const size_t kvbase = ((size_t)b * p.nkv + g) * (size_t)p.S * D;
  const uint16_t* Kc = L.kc + kvbase;
  const uint16_t* Vc = L.vc + kvbase;
  const float qscale = 1.4426950408889634f * rsqrtf((float)D);

  float qf[GH][8], o[GH][8], mm[GH], ll[GH];
#pragma unroll
  for (int h = 0; h < GH; ++h) {
    const float* qs = p.q + (size_t)b * p.QD + (size_t)(g * p.G + h0 + h) * D + sub * 8;
    const float4 a0 = __ldcg(reinterpret_cast<const float4*>(qs));
    const float4 a1 = __ldcg(reinterpret_cast<const float4*>(qs + 4));
    qf[h][0] = a0.x * qscale; qf[h][1] = a0.y * qscale; qf[h][2] = a0.z * qscale;
    qf[h][3] = a0.w * qscale; qf[h][4] = a1.x * qscale; qf[h][5] = a1.y * qscale;
    qf[h][6] = a1.z * qscale; qf[h][7] = a1.w * qscale;
    mm[h] = -INFINITY;
    ll[h] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[h][e] = 0.f;
  }

  constexpr int U = 2;  // key rows in flight per lane
  const int stride = kComputeWarps * TPI;
  for (int base = t0 + warp * TPI; base < t1; base += U * stride) {
    uint4 kv[U], vv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = base + u * stride + ti;
      if (t < t1) {
        kv[u] = __ldcg(reinterpret_cast<const uint4*>(Kc + (size_t)t * D + sub * 8));
        vv[u] = __ldcg(reinterpret_cast<const uint4*>(Vc + (size_t)t * D + sub * 8));
      } else {
        kv[u] = make_uint4(0, 0, 0, 0);
        vv[u] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const bool valid = base + u * stride + ti < t1;
      float s[GH];
#pragma unroll
      for (int h = 0; h < GH; ++h) {
        float acc = qf[h][0] * bf_lo(kv[u].x);
        acc = fmaf(qf[h][1], bf_hi(kv[u].x), acc);
        acc = fmaf(qf[h][2], bf_lo(kv[u].y), acc);
        acc = fmaf(qf[h][3], bf_hi(kv[u].y), acc);
        acc = fmaf(qf[h][4], bf_lo(kv[u].z), acc);
        acc = fmaf(qf[h][5], bf_hi(kv[u].z), acc);
        acc = fmaf(qf[h][6], bf_lo(kv[u].w), acc);
        acc = fmaf(qf[h][7], bf_hi(kv[u].w), acc);
        s[h] = acc;
      }
#pragma unroll
      for (int off = 1; off < LPT; off <<= 1)
#pragma unroll
        for (int h = 0; h < GH; ++h) s[h] += __shfl_xor_sync(0xffffffffu, s[h], off);
      if (valid) {
        const float vf[8] = {bf_lo(vv[u].x), bf_hi(vv[u].x), bf_lo(vv[u].y), bf_hi(vv[u].y),
                             bf_lo(vv[u].z), bf_hi(vv[u].z), bf_lo(vv[u].w), bf_hi(vv[u].w)};
#pragma unroll
        for (int h = 0; h < GH; ++h) {
          const float mn = fmaxf(mm[h], s[h]);
          const float sc = exp2f(mm[h] - mn);
          const float pe = exp2f(s[h] - mn);
          ll[h] = ll[h] * sc + pe;
#pragma unroll
          for (int e = 0; e < 8; ++e) o[h][e] = fmaf(pe, vf[e], o[h][e] * sc);
          mm[h] = mn;
        }
      }
    }
  }
  // merge the key groups of the warp (lanes with the same `sub`)
#pragma unroll
  for (int off = LPT; off < 32; off <<= 1) {
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      const float m2 = __shfl_xor_sync(0xffffffffu, mm[h], off);
      const float l2 = __shfl_xor_sync(0xffffffffu, ll[h], off);
      float o2[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) o2[e] = __shfl_xor_sync(0xffffffffu, o[h][e], off);
      softmax_merge(mm[h], ll[h], o[h], m2, l2, o2);
    }
  }
  // scratch [warp][h][D + 2] in the activation staging area
  float* scr = reinterpret_cast<float*>(smem + p.off_x);
  compute_bar();  // previous readers of the staging area are done
  if (ti == 0) {
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      float* sp = scr + ((size_t)warp * GH + h) * (D + 2);
#pragma unroll
      for (int e = 0; e < 8; ++e) sp[sub * 8 + e] = o[h][e];
      if (sub == 0) {
        sp[D] = mm[h];
        sp[D + 1] = ll[h];
      }
    }
  }
  compute_bar();
  const int tid = threadIdx.x;
  for (int idx = tid; idx < GH * D; idx += kComputeThreads) {
    const int h = idx / D, d = idx - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kComputeWarps; ++w) M = fmaxf(M, scr[((size_t)w * GH + h) * (D + 2) + D]);
    float acc = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < kComputeWarps; ++w) {
      const float* sp = scr + ((size_t)w * GH + h) * (D + 2);
      const float wt = sp[D] == -INFINITY ? 0.f : exp2f(sp[D] - M);
      acc = fmaf(wt, sp[d], acc);
      den = fmaf(wt, sp[D + 1], den);
    }
    float* dst = p.part + (((size_t)b * p.nh + g * p.G + h0 + h) * kMaxPartitions + pidx) * (D + 2);
    dst[d] = acc;
    if (d == 0) {
      dst[D] = M;
      dst[D + 1] = den;
    }
  }
}

template <int D>
__device__ void attn_unit(const Params& p, uint8_t* smem, const Instr& in) {
  switch (p.G) {
    case 1: attn_partial<D, 1>(p, smem, in, 0); break;
    case 2: attn_partial<D, 2>(p, smem, in, 0); break;
    case 4: attn_partial<D, 4>(p, smem, in, 0); break;
    default:
      for (int h0 = 0; h0 < p.G; h0 += 4) attn_partial<D, 4>(p, smem, in, h0);
      break;
  }
}

// ---------------------------------------------------------------------------
// compute role: attention partial reduction (instruction 3)
// ---------------------------------------------------------------------------

template <int D>
__device__ __forceinline__ void attn_reduce(const Params& p, const Instr& in) {
  constexpr int PL = D / 32;  // dims per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = in.a0, g = in.a1, P = in.a2;
  for (int hl = warp; hl < p.G; hl += kComputeWarps) {
    const int h = g * p.G + hl;
    const float* base = p.part + ((size_t)b * p.nh + h) * kMaxPartitions * (D + 2);
    float M = -INFINITY;
    for (int k = lane; k < P; k += 32) M = fmaxf(M, __ldcg(base + (size_t)k * (D + 2) + D));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float acc[PL], den = 0.f;
#pragma unroll
    for (int e = 0; e < PL; ++e) acc[e] = 0.f;
    for (int k = 0; k < P; ++k) {
      const float* s = base + (size_t)k * (D + 2);
      const float mk = __ldcg(s + D);
      const float wt = mk == -INFINITY ? 0.f : exp2f(mk - M);
      den = fmaf(wt, __ldcg(s + D + 1), den);
#pragma unroll
      for (int e = 0; e < PL; ++e) acc[e] = fmaf(wt, __ldcg(s + lane * PL + e), acc[e]);
    }
    const float inv = 1.f / den;
    float* dst = p.attn + (size_t)b * p.QD + (size_t)h * D + lane * PL;
#pragma unroll
    for (int e = 0; e < PL; ++e) dst[e] = acc[e] * inv;
  }
}

// ---------------------------------------------------------------------------
// compute role: the instruction loop
// ---------------------------------------------------------------------------

template <int B>
__device__ void compute_role(const Params& p, Misc* m, uint8_t* smem, const Instr* q, int n,
                             int qbase) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Staged st;
  uint32_t page_cnt = 0;
  int known_ctr = -1, known_tgt = 0;
  for (int i = 0; i < n; ++i) {
    const Instr in = q[i];
    const int buf = i & 1;
    const uint32_t rpar = ((uint32_t)i >> 1) & 1u;
    uint64_t t_start = 0, t_ready = 0;
    const bool tracing = p.trace != nullptr && warp == 0 && lane == 0;
    if (tracing) t_start = globaltimer();
    // 1. dependency: one thread polls, the other compute warps meet it at a barrier
    if (!p.no_waits && in.wait_ctr >= 0 &&
        !(in.wait_ctr == known_ctr && in.wait_target <= known_tgt)) {
      if (warp == 0 && lane == 0) wait_counter(p, m, in.wait_ctr, in.wait_target);
      compute_bar();
      known_ctr = in.wait_ctr;
      known_tgt = in.wait_target;
    }
    if (tracing) t_ready = globaltimer();
    // 2. the result buffer this instruction hands to the storer must be free
    const bool res_ok = wait_mbar(p, m, &m->res_empty[buf], rpar ^ 1u, kErrTimeoutRes);
    float* res = reinterpret_cast<float*>(smem + p.off_res) + (size_t)buf * p.res_floats;

    if (is_gemv(in.op)) {
      const int kind = act_kind(in.op);
      const int chunk = in.op == MK_OP_DOWN ? in.a2 : 0;
      const int key = act_key(kind, in.layer, chunk);
      const bool to_h = kind == kActH;
      if ((to_h ? st.key_h : st.key_x) != key) stage(p, m, smem, st, kind, in.layer, chunk);
      const Geom g = geom_of(in.op, p.H, p.QD, p.Fc, p.B);
      const float* act = reinterpret_cast<const float*>(smem + (to_h ? p.off_h : p.off_x));
      const LayerPtrs& L = p.layers[in.layer];
      const uint16_t* normw = kind == kActAttnNorm ? L.attn_norm
                              : kind == kActMlpNorm ? L.mlp_norm
                              : kind == kActFinalNorm ? p.final_norm
                                                      : nullptr;
      gemv_run<B>(p, m, smem, in, g, act, normw, st.inv, res, page_cnt);
      page_cnt += (uint32_t)((in.a1 - in.a0 + g.ipp - 1) / g.ipp);
    } else if (in.op == MK_OP_ATTN) {
      st.key_x = -1;  // the staging area becomes scratch
      st.key_h = -1;
      // runs even after an abort: its loads stay in bounds and its barriers
      // must be met by every compute warp
      if (p.D == 64) attn_unit<64>(p, smem, in);
      else attn_unit<128>(p, smem, in);
    } else if (in.op == MK_OP_RED) {
      if (!aborted(m)) {
        if (p.D == 64) attn_reduce<64>(p, in);
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
        mk_trace_record r;
        r.sm = blockIdx.x;
        r.index = (uint32_t)i;
        r.op = in.op;
        r.layer = in.layer;
        r.t_start = t_start;
        r.t_ready = t_ready;
        r.t_end = globaltimer();
        p.trace[rec] = r;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// storer role
// ---------------------------------------------------------------------------

__device__ __forceinline__ float silu(float z) { return z / (1.f + expf(-z)); }

__device__ __forceinline__ void epilogue(const Params& p, const Instr& in, const float* res) {
  const int lane = threadIdx.x & 31;
  const Geom g = geom_of(in.op, p.H, p.QD, p.Fc, p.B);
  const int items = in.a1 - in.a0;
  const int B = p.B;
  const LayerPtrs& L = p.layers[in.layer];
  for (int it = lane; it < items; it += 32) {
    const int j = in.a0 + it;
    for (int b = 0; b < B; ++b) {
      float v[2] = {0.f, 0.f};
      for (int r = 0; r < g.R; ++r)
        for (int s = 0; s < g.nseg; ++s) v[r] += res[((size_t)(it * g.R + r) * g.nseg + s) * B + b];
      switch (in.op) {
        case MK_OP_QKV: {
          const PairRows pr = pair_rows(j, p.G, p.D);
          const int pos = p.pos[b];
          const int half = p.D / 2;
          float o0 = v[0], o1 = v[1];
          if (pr.which < 2) {
            const float2 cs = p.rope[(size_t)pos * half + pr.i];
            o0 = v[0] * cs.x - v[1] * cs.y;
            o1 = v[1] * cs.x + v[0] * cs.y;
          }
          if (pr.which == 0) {
            float* qd = p.q + (size_t)b * p.QD + (size_t)pr.head * p.D + pr.i;
            qd[0] = o0;
            qd[half] = o1;
          } else {
            uint16_t* c = (pr.which == 1 ? L.kc : L.vc) +
                          (((size_t)b * p.nkv + pr.head) * p.S + pos) * p.D + pr.i;
            c[0] = __bfloat16_as_ushort(__float2bfloat16_rn(o0));
            c[half] = __bfloat16_as_ushort(__float2bfloat16_rn(o1));
          }
          break;
        }
        case MK_OP_OPROJ: {
          const float base = in.layer == 0 ? bf16f(p.embed[(size_t)p.tok[b] * p.H + j])
                                           : __ldcg(p.x + (size_t)b * p.H + j);
          p.xa[(size_t)b * p.H + j] = base + v[0];
          break;
        }
        case MK_OP_GATEUP:
          p.h[(size_t)b * p.F + j] = silu(v[0]) * v[1];
          break;
        case MK_OP_DOWN: {
          float* acc = p.dacc + (size_t)b * p.H + j;
          float d = in.a2 == 0 ? v[0] : __ldcg(acc) + v[0];
          if (in.a2 == kChunks - 1) p.x[(size_t)b * p.H + j] = __ldcg(p.xa + (size_t)b * p.H + j) + d;
          else *acc = d;
          break;
        }
        default:  // MK_OP_LMHEAD
          p.logits[(size_t)b * p.V + j] = v[0];
          break;
      }
    }
  }
}

__device__ void storer_role(const Params& p, Misc* m, uint8_t* smem, const Instr* q, int n) {
  const int lane = threadIdx.x & 31;
  for (int i = 0; i < n; ++i) {
    const Instr in = q[i];
    const int buf = i & 1;
    const uint32_t par = ((uint32_t)i >> 1) & 1u;
    const bool ok = wait_mbar(p, m, &m->res_full[buf], par, kErrTimeoutRes);
    if (ok && !aborted(m)) {
      const float* res = reinterpret_cast<const float*>(smem + p.off_res) + (size_t)buf * p.res_floats;
      if (is_gemv(in.op)) epilogue(p, in, res);
      if (in.sig_ctr >= 0) {
        __threadfence();
        __syncwarp();
        if (lane == 0) red_release_add(p.ctr + in.sig_ctr, in.sig_amount);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&m->res_empty[buf]);
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

template <int B>
__global__ void __launch_bounds__(kThreads, 1) interp_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Misc* m = reinterpret_cast<Misc*>(smem + p.off_misc);
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.n_pages; ++i) {
      mbar_init(&m->full[i], 1);
      mbar_init(&m->empty[i], kComputeWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&m->res_full[i], kComputeWarps);
      mbar_init(&m->res_empty[i], 1);
    }
    m->abort = 0;
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
  if (warp == kLoaderWarp) loader_role(p, m, smem, q, n);
  else if (warp == kStorerWarp) storer_role(p, m, smem, q, n);
  else compute_role<B>(p, m, smem, q, n, q0);
}

// host-side accessor for the kernel entry of a batch size
const void* kernel_for_batch(int B) {
  switch (B) {
    case 1: return reinterpret_cast<const void*>(&interp_kernel<1>);
    case 2: return reinterpret_cast<const void*>(&interp_kernel<2>);
    case 4: return reinterpret_cast<const void*>(&interp_kernel<4>);
    case 8: return reinterpret_cast<const void*>(&interp_kernel<8>);
    default: return nullptr;
  }
}

int misc_bytes() { return (int)sizeof(Misc); }

}  // namespace mk
