// mk_decode_step_noalloc: the decode step for callers that cannot allocate
// device memory.
//
// Some callers may not call cudaMalloc at all: code running inside a memory
// pool or arena that owns every device byte of the process, plugins whose
// host forbids device allocations after start-up, or callers that must not
// take the allocator's locks or risk an allocation failure on their serving
// path. For them this entry point runs the same persistent interpreter kernel
// as mk_decode_step, but without a handle: all of its scratch (activations,
// attention partials, counters, error word, RoPE table and the per-SM
// instruction queues) lives in one file-scope device array of fixed size that
// the library reserves when it is loaded. Nothing is allocated per call: no
// cudaMalloc, cudaFree, pinned host memory or allocating library routine.
//
// Sharing rules: every call on a device uses the same array and leaves its
// contents behind. Each call clears what must start at zero (the counters,
// the error word and the values handed between instructions) before it
// launches, and uploads its queue and the RoPE rows of its positions.
// Calls that overlap on the GPU (on different streams, or from several host
// threads) race on the array; serialise them.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "mk_isa.h"
#include "mk_kernels.h"
#include "mk_sched.h"


using namespace mk;

// 16 MiB is the stated maximum: enough for every workload in the test and
// benchmark set (Llama-1B shape at batch 8 or with an 8K-token KV capacity,
// Llama-8B shape at 2K), small next to the GPU's memory. Every GPU that loads
// the library holds this array until the process exits.
constexpr size_t kStaticScratchBytes = 16u << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kStaticScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
struct DeviceSetup {
  bool done = false;
  unsigned char* base = nullptr;  // device address of g_noalloc_scratch
  int n_sm = 0;
  int optin = 0;
};
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mutex;

size_t align256(size_t n) { return (n + 255) / 256 * 256; }

int set_error(char* msg, size_t cap, const char* text) {
  if (msg && cap) std::snprintf(msg, cap, "%s", text);
  return MK_ERR_INVALID;
}

// Once per device, with that device current: resolve the device address of
// the static array (host code may not use the symbol itself as a pointer) and
// raise the kernel's shared-memory limit.
int setup_device(int dev, DeviceSetup** out, std::string* why) {
  if (dev < 0 || dev >= kMaxDevices) {
    *why = "device ordinal beyond the supported range";
    return MK_ERR_INVALID;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceSetup& s = g_setup[dev];
  if (!s.done) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) {
      *why = std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e);
      return MK_ERR_CUDA;
    }
    e = cudaDeviceGetAttribute(&s.n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&s.optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) {
      *why = std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e);
      return MK_ERR_CUDA;
    }
    s.base = static_cast<unsigned char*>(ptr);
    s.done = true;
  }
  *out = &s;
  return MK_OK;
}

}  // namespace

extern "C" int mk_decode_step_noalloc(const mk_config* cfg, const mk_weights* w,
                                      void* const* k_cache, void* const* v_cache,
                                      const int32_t* token_ids, const int32_t* positions,
                                      float* logits_out, void* stream, char* errmsg,
                                      size_t errmsg_cap) {
  // ---- host-side validation (before any CUDA call)
  if (!cfg || !w || !k_cache || !v_cache || !token_ids || !positions || !logits_out)
    return set_error(errmsg, errmsg_cap, "a required argument is NULL");
  Shape s{cfg->n_layers, cfg->hidden, cfg->n_heads, cfg->n_kv_heads, cfg->head_dim,
          cfg->ffn, cfg->vocab, cfg->batch, cfg->kv_capacity};
  std::string why = check_shape(s);
  if (!why.empty()) return set_error(errmsg, errmsg_cap, why.c_str());
  if (!(cfg->rms_eps >= 0.f) || !(cfg->rope_theta > 0.f))
    return set_error(errmsg, errmsg_cap, "rms_eps must be >= 0 and rope_theta > 0");
  if (cfg->tied_embeddings ? (w->lm_head != nullptr) : (w->lm_head == nullptr))
    return set_error(errmsg, errmsg_cap, "lm_head must be NULL iff tied_embeddings");
  for (int b = 0; b < s.B; ++b) {
    if (token_ids[b] < 0 || token_ids[b] >= s.V)
      return set_error(errmsg, errmsg_cap, "token id out of range [0, vocab)");
    if (positions[b] < 0 || positions[b] >= s.S)
      return set_error(errmsg, errmsg_cap, "position out of range [0, kv_capacity)");
  }
  auto al16 = [](const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  bool aligned = al16(w->embed) && al16(w->final_norm) && al16(logits_out) &&
                 (!w->lm_head || al16(w->lm_head));
  for (int l = 0; l < s.L && aligned; ++l)
    aligned = al16(w->attn_norm[l]) && al16(w->wq[l]) && al16(w->wk[l]) && al16(w->wv[l]) &&
              al16(w->wo[l]) && al16(w->mlp_norm[l]) && al16(w->wgate[l]) && al16(w->wup[l]) &&
              al16(w->wdown[l]) && al16(k_cache[l]) && al16(v_cache[l]);
  if (!aligned)
    return set_error(errmsg, errmsg_cap, "every pointer must be non-NULL and 16-byte aligned");

  // ---- per-device set-up (first call on this device)
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) {
    if (errmsg && errmsg_cap) std::snprintf(errmsg, errmsg_cap, "cudaGetDevice: %s", cudaGetErrorString(ce));
    return MK_ERR_CUDA;
  }
  DeviceSetup* ds = nullptr;
  int rc = setup_device(dev, &ds, &why);
  if (rc != MK_OK) {
    if (errmsg && errmsg_cap) std::snprintf(errmsg, errmsg_cap, "%s", why.c_str());
    return rc;
  }

  // ---- the schedule for these positions (host memory only)
  int parts[kMaxBatch];
  choose_partitions(s, ds->n_sm, positions, parts);
  Plan plan;
  if (!build_plan(s, ds->n_sm, parts, &plan, &why))
    return set_error(errmsg, errmsg_cap, why.c_str());

  // ---- carve the static array
  const int B = s.B;
  CounterMap cm{s.L, s.nkv, s.B};
  const int n_ctr = cm.count();
  // pieces 0..6 hold the stamped hand-off words (cleared before each call,
  // which then runs with stamp 1)
  const size_t sizes[] = {
      sizeof(float) * (size_t)kChunks * B * s.H,                      // down-projection shares
      sizeof(float) * (size_t)B * s.H,                                // xa
      sizeof(float) * (size_t)B * s.QD(),                             // q
      sizeof(float) * (size_t)B * s.QD(),                             // attention output
      sizeof(float) * (size_t)B * s.F,                                // h
      sizeof(float) * (size_t)B * s.nkv * 2 * s.D,                    // new k/v rows
      sizeof(float) * (size_t)B * s.H,                                // layer output x
      sizeof(float) * (size_t)B * s.nh * kMaxPartitions * (s.D + 2),  // attention partials
      sizeof(float2) * (size_t)s.S * (s.D / 2),                       // RoPE table
      sizeof(int) * (size_t)n_ctr,                                    // counters
      sizeof(int) * 64,                                               // error word
      sizeof(Instr) * plan.instrs.size(),                             // queues
      sizeof(int) * plan.sm_off.size(),                               // queue offsets
  };
  constexpr int kPieces = sizeof(sizes) / sizeof(sizes[0]);
  size_t offs[kPieces], total = 0;
  for (int i = 0; i < kPieces; ++i) {
    offs[i] = total;
    total += align256(sizes[i]);
  }
  if (total > kStaticScratchBytes) {
    if (errmsg && errmsg_cap)
      std::snprintf(errmsg, errmsg_cap,
                    "this configuration needs %zu bytes of scratch; the static array holds %zu",
                    total, kStaticScratchBytes);
    return MK_ERR_INVALID;
  }
  unsigned char* base = ds->base;

  // ---- launch parameters (same layout rules as mk_create)
  Params p{};
  p.L = s.L; p.H = s.H; p.nh = s.nh; p.nkv = s.nkv; p.D = s.D; p.F = s.F; p.V = s.V;
  p.B = s.B; p.S = s.S; p.G = s.G(); p.Fc = s.Fc(); p.QD = s.QD();
  p.eps = cfg->rms_eps;
  p.embed = static_cast<const uint16_t*>(w->embed);
  p.lm = static_cast<const uint16_t*>(cfg->tied_embeddings ? w->embed : w->lm_head);
  p.final_norm = static_cast<const uint16_t*>(w->final_norm);
  for (int l = 0; l < s.L; ++l) {
    LayerPtrs& lp = p.layers[l];
    lp.attn_norm = static_cast<const uint16_t*>(w->attn_norm[l]);
    lp.wq = static_cast<const uint16_t*>(w->wq[l]);
    lp.wk = static_cast<const uint16_t*>(w->wk[l]);
    lp.wv = static_cast<const uint16_t*>(w->wv[l]);
    lp.wo = static_cast<const uint16_t*>(w->wo[l]);
    lp.mlp_norm = static_cast<const uint16_t*>(w->mlp_norm[l]);
    lp.wgate = static_cast<const uint16_t*>(w->wgate[l]);
    lp.wup = static_cast<const uint16_t*>(w->wup[l]);
    lp.wdown = static_cast<const uint16_t*>(w->wdown[l]);
    lp.kc = static_cast<uint16_t*>(k_cache[l]);
    lp.vc = static_cast<uint16_t*>(v_cache[l]);
  }
  p.xpart = reinterpret_cast<float*>(base + offs[0]);
  p.xa = reinterpret_cast<float*>(base + offs[1]);
  p.q = reinterpret_cast<float*>(base + offs[2]);
  p.attn = reinterpret_cast<float*>(base + offs[3]);
  p.h = reinterpret_cast<float*>(base + offs[4]);
  p.kvn = reinterpret_cast<float*>(base + offs[5]);
  p.x = reinterpret_cast<float*>(base + offs[6]);
  p.stamp = 1u;  // the cleared words carry stamp 0
  p.part = reinterpret_cast<float*>(base + offs[7]);
  // (m, l) after the o rows, in the same piece
  p.part_ml = p.part + (size_t)B * s.nh * kMaxPartitions * s.D;
  p.rope = reinterpret_cast<const float2*>(base + offs[8]);
  p.ctr = reinterpret_cast<int*>(base + offs[9]);
  p.ctr_zero = nullptr;  // cleared by the memset below instead
  p.n_ctr = n_ctr;
  p.err = reinterpret_cast<int*>(base + offs[10]);
  p.err_host = nullptr;
  p.instrs = reinterpret_cast<const Instr*>(base + offs[11]);
  p.sm_off = reinterpret_cast<const int*>(base + offs[12]);
  p.logits = logits_out;
  p.trace = nullptr;
  p.trace_cap = 0;
  p.trace_base = 0;
  p.timeout_ns = 2000000000ull;
  p.no_waits = 0;
  for (int b = 0; b < kMaxBatch; ++b) {
    p.tok[b] = b < B ? token_ids[b] : 0;
    p.pos[b] = b < B ? positions[b] : 0;
  }
  // shared-memory layout (the same rules as mk_create)
  const int smem_bytes = smem_layout(s, ds->n_sm, ds->optin, misc_bytes(), &p, &why);
  if (!smem_bytes) return set_error(errmsg, errmsg_cap, why.c_str());

  // ---- uploads, clears, launch: no allocation anywhere below
  // The step reads the RoPE table only at the B positions it decodes: those
  // rows alone are computed (angle = pos * theta^(-2i/D), in double, rounded
  // to fp32, as mk_create does for the whole table) and copied to their
  // offsets in the table piece.
  const int half = s.D / 2;
  std::vector<float2> rope((size_t)B * half);
  for (int b = 0; b < B; ++b)
    for (int i = 0; i < half; ++i) {
      double ang = (double)positions[b] * std::pow((double)cfg->rope_theta, -2.0 * i / (double)s.D);
      rope[(size_t)b * half + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
    }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const void* fn = kernel_for(s, false);
  // pageable-source copies are staged by the driver before they return, so
  // the host vectors may go out of scope right after the calls
  ce = allow_max_smem(fn, ds->optin);
  for (int b = 0; b < B && ce == cudaSuccess; ++b)
    ce = cudaMemcpyAsync(base + offs[8] + sizeof(float2) * (size_t)positions[b] * half,
                         rope.data() + (size_t)b * half, sizeof(float2) * half,
                         cudaMemcpyHostToDevice, st);
  if (ce == cudaSuccess)
    ce = cudaMemcpyAsync(base + offs[11], plan.instrs.data(), sizes[11], cudaMemcpyHostToDevice, st);
  if (ce == cudaSuccess)
    ce = cudaMemcpyAsync(base + offs[12], plan.sm_off.data(), sizes[12], cudaMemcpyHostToDevice, st);
  if (ce == cudaSuccess) ce = cudaMemsetAsync(base, 0, offs[7], st);  // stamped words
  if (ce == cudaSuccess) ce = cudaMemsetAsync(base + offs[9], 0, sizes[9], st);  // counters
  if (ce == cudaSuccess) ce = cudaMemsetAsync(base + offs[10], 0, sizes[10], st);  // error word
  if (ce == cudaSuccess) {
    void* args[] = {&p};
    ce = cudaLaunchCooperativeKernel(fn, dim3(ds->n_sm), dim3(kThreads), args, (size_t)smem_bytes, st);
  }
  // the call is synchronous: it waits for the step and reports a device timeout
  int err_word = 0;
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(st);
  if (ce == cudaSuccess)
    ce = cudaMemcpy(&err_word, base + offs[10], sizeof(int), cudaMemcpyDeviceToHost);
  if (ce != cudaSuccess) {
    if (errmsg && errmsg_cap) std::snprintf(errmsg, errmsg_cap, "CUDA: %s", cudaGetErrorString(ce));
    return MK_ERR_CUDA;
  }
  if (err_word != 0) {
    if (errmsg && errmsg_cap)
      std::snprintf(errmsg, errmsg_cap, "device error word 0x%08x", err_word);
    const int code = (err_word >> 24) & 0xff;
    return code ? code : MK_ERR_CUDA;
  }
  if (errmsg && errmsg_cap) errmsg[0] = '\0';
  return MK_OK;
}
