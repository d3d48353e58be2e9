// C ABI of libmk.so (declared in include/mk.h): handle lifetime, scratch
// allocation, the plan cache, and the launches of the persistent interpreter
// (one per decode step) and of the multi-launch comparison build.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <memory>
#include <random>
#include <string>
#include <vector>

#include "mk_isa.h"
#include "mk_kernels.h"
#include "mk_sched.h"


using namespace mk;

namespace {

thread_local std::string g_create_error;

struct PlanEntry {
  int key[kMaxBatch + 3];  // partitions per sequence, injection flag, permutation seed, dynamic flags
  Plan plan;
  Instr* d_instrs = nullptr;
  int* d_sm_off = nullptr;
  Instr* d_phase_instrs = nullptr;  // all multi-launch phases, concatenated
  int* d_phase_off = nullptr;
  std::vector<int> phase_instr_base, phase_off_base;
  cudaGraphExec_t gexec = nullptr;
  cudaGraph_t graph = nullptr;
  std::vector<cudaGraphNode_t> nodes;
  unsigned long long last_use = 0;
};

}  // namespace

struct mk_handle {
  mk_config cfg;
  Shape shape;
  int device = 0;
  int n_sm = 0;
  int smem_bytes = 0;
  int smem_optin = 0;     // the device's opt-in maximum of dynamic shared memory per block
  const void* fn = nullptr;  // the interpreter instantiation this handle launches
  const void* fn_fx = nullptr;  // the one with the paged-cache / greedy-decode code
  const void* fn_dyn = nullptr; // the one with dynamic work distribution (or nullptr)
  Params base{};          // launch parameters without the per-step fields
  void* d_scratch = nullptr;
  float2* d_rope = nullptr;
  int* d_ctr = nullptr;   // two counter sets
  int n_ctr = 0;
  int* d_err = nullptr;
  unsigned long long* d_keys = nullptr;  // greedy decode: argmax keys [kMaxGreedySteps][B]
  int kv_block = 0;       // paged KV cache: positions per block (0: contiguous caches)
  int n_blocks = 0;       // paged KV cache: blocks in each layer's pool
  int max_blocks = 0;     // paged KV cache: block-table entries per sequence
  int* d_table = nullptr; // paged KV cache: the step's block table [B][max_blocks]
  int* d_ctr_steps = nullptr;  // counters of a several-step launch [kMaxLaunchSteps][n_ctr]
  float* d_plogits = nullptr;  // prefill: the logits of every row of a chunk [B][V]
  // stamped hand-off words: the first stamped_bytes of the scratch; layer l
  // of the next step stamps with (stamp_serial + l) & 1 (each step adds L)
  size_t stamped_bytes = 0;
  uint32_t stamp_serial = 1;
  struct StepsPlan {
    std::vector<int> key;  // steps, then each step's partition counts
    Instr* d_instrs = nullptr;
    int* d_sm_off = nullptr;
  };
  std::vector<StepsPlan> steps_plans;
  int* h_err_mirror = nullptr;  // mapped pinned host memory the kernel writes on error
  std::vector<PlanEntry*> plans;
  unsigned long long use_clock = 0;
  unsigned long long steps = 0;
  int cur_set = 0;        // counter set used by the most recent step
  int inject = 0;
  uint32_t perm_seed = 0; // test hook: queues handed to the CTAs in a seeded order
  int dyn = 0;            // MK_DYN_* flags of the plans
  std::string err;
};

namespace {

int fail(mk_handle* h, int code, const std::string& msg) {
  if (h) h->err = msg;
  else g_create_error = msg;
  return code;
}

int cuda_fail(mk_handle* h, cudaError_t e, const char* what) {
  std::string msg = std::string(what) + ": " + cudaGetErrorString(e);
  int code = (e == cudaErrorMemoryAllocation) ? MK_ERR_OOM : MK_ERR_CUDA;
  return fail(h, code, msg);
}

#define MK_CUDA(h, call)                                   \
  do {                                                     \
    cudaError_t e_ = (call);                               \
    if (e_ != cudaSuccess) return cuda_fail((h), e_, #call); \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

Shape shape_of(const mk_config& c) {
  Shape s;
  s.L = c.n_layers;
  s.H = c.hidden;
  s.nh = c.n_heads;
  s.nkv = c.n_kv_heads;
  s.D = c.head_dim;
  s.F = c.ffn;
  s.V = c.vocab;
  s.B = c.batch;
  s.S = c.kv_capacity;
  return s;
}

int check_config(const mk_config* c, mk_handle* h) {
  if (!c) return fail(h, MK_ERR_INVALID, "config is NULL");
  std::string e = check_shape(shape_of(*c));
  if (!e.empty()) return fail(h, MK_ERR_INVALID, e);
  if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f))
    return fail(h, MK_ERR_INVALID, "rms_eps must be >= 0 and rope_theta > 0");
  return MK_OK;
}

int check_steps(mk_handle* h, const int32_t* tok, const int32_t* pos) {
  if (!tok || !pos) return fail(h, MK_ERR_INVALID, "token_ids / positions must be non-NULL");
  for (int b = 0; b < h->shape.B; ++b) {
    if (tok[b] < 0 || tok[b] >= h->shape.V)
      return fail(h, MK_ERR_INVALID, "token id out of range [0, vocab)");
    if (pos[b] < 0 || pos[b] >= h->shape.S)
      return fail(h, MK_ERR_INVALID, "position out of range [0, kv_capacity)");
  }
  return MK_OK;
}

void free_plan(PlanEntry* e) {
  if (e->gexec) cudaGraphExecDestroy(e->gexec);
  if (e->graph) cudaGraphDestroy(e->graph);
  cudaFree(e->d_instrs);
  cudaFree(e->d_sm_off);
  cudaFree(e->d_phase_instrs);
  cudaFree(e->d_phase_off);
  delete e;
}

// Returns the plan for these positions, building and uploading it if needed
// (dyn: MK_DYN_* flags of the plan; greedy decode and paged steps run
// kernels without dynamic distribution and pass 0).
int get_plan(mk_handle* h, const int32_t* pos, PlanEntry** out, int dyn) {
  int parts[kMaxBatch];
  choose_partitions(h->shape, h->n_sm, pos, parts);
  int key[kMaxBatch + 3];
  for (int b = 0; b < kMaxBatch; ++b) key[b] = b < h->shape.B ? parts[b] : 0;
  key[kMaxBatch] = h->inject;
  key[kMaxBatch + 1] = (int)h->perm_seed;
  key[kMaxBatch + 2] = dyn;
  for (PlanEntry* e : h->plans)
    if (std::memcmp(e->key, key, sizeof key) == 0) {
      e->last_use = ++h->use_clock;
      *out = e;
      return MK_OK;
    }
  // on an error below, the deleter frees what was already uploaded
  std::unique_ptr<PlanEntry, void (*)(PlanEntry*)> e(new PlanEntry(), free_plan);
  std::memcpy(e->key, key, sizeof key);
  std::string why;
  if (!build_plan(h->shape, h->n_sm, parts, &e->plan, &why, dyn))
    return fail(h, MK_ERR_INVALID, why);
  Plan& P = e->plan;
  if (h->inject) {
    // raise the first wait of the last SM's queue past what can ever be produced
    int s = h->n_sm - 1;
    for (int i = P.sm_off[s]; i < P.sm_off[s + 1]; ++i)
      if (P.instrs[i].wait_ctr >= 0) {
        P.instrs[i].wait_target += 1;
        break;
      }
  }
  if (h->perm_seed) {
    // CTA k runs the queue built for SM perm[k]
    std::vector<int> perm(h->n_sm);
    for (int k = 0; k < h->n_sm; ++k) perm[k] = k;
    std::mt19937 rng(h->perm_seed);
    std::shuffle(perm.begin(), perm.end(), rng);
    std::vector<Instr> q;
    std::vector<int> off(h->n_sm + 1, 0);
    for (int k = 0; k < h->n_sm; ++k) {
      off[k] = (int)q.size();
      q.insert(q.end(), P.instrs.begin() + P.sm_off[perm[k]], P.instrs.begin() + P.sm_off[perm[k] + 1]);
    }
    off[h->n_sm] = (int)q.size();
    P.instrs.swap(q);
    P.sm_off.swap(off);
  }
  // upload (plans change every few hundred tokens, so a synchronous copy is fine)
  MK_CUDA(h, cudaMalloc(&e->d_instrs, sizeof(Instr) * std::max<size_t>(1, P.instrs.size())));
  MK_CUDA(h, cudaMalloc(&e->d_sm_off, sizeof(int) * P.sm_off.size()));
  MK_CUDA(h, cudaMemcpy(e->d_instrs, P.instrs.data(), sizeof(Instr) * P.instrs.size(),
                        cudaMemcpyHostToDevice));
  MK_CUDA(h, cudaMemcpy(e->d_sm_off, P.sm_off.data(), sizeof(int) * P.sm_off.size(),
                        cudaMemcpyHostToDevice));
  std::vector<Instr> all;
  std::vector<int> offs;
  for (auto& ph : P.phases) {
    e->phase_instr_base.push_back((int)all.size());
    e->phase_off_base.push_back((int)offs.size());
    all.insert(all.end(), ph.instrs.begin(), ph.instrs.end());
    offs.insert(offs.end(), ph.sm_off.begin(), ph.sm_off.end());
  }
  MK_CUDA(h, cudaMalloc(&e->d_phase_instrs, sizeof(Instr) * std::max<size_t>(1, all.size())));
  MK_CUDA(h, cudaMalloc(&e->d_phase_off, sizeof(int) * std::max<size_t>(1, offs.size())));
  MK_CUDA(h, cudaMemcpy(e->d_phase_instrs, all.data(), sizeof(Instr) * all.size(),
                        cudaMemcpyHostToDevice));
  MK_CUDA(h, cudaMemcpy(e->d_phase_off, offs.data(), sizeof(int) * offs.size(),
                        cudaMemcpyHostToDevice));
  // keep a handful of plans; evicting one waits for the device to be idle
  if (h->plans.size() >= 6) {
    size_t victim = 0;
    for (size_t i = 1; i < h->plans.size(); ++i)
      if (h->plans[i]->last_use < h->plans[victim]->last_use) victim = i;
    MK_CUDA(h, cudaDeviceSynchronize());
    free_plan(h->plans[victim]);
    h->plans.erase(h->plans.begin() + victim);
  }
  e->last_use = ++h->use_clock;
  *out = e.release();
  h->plans.push_back(*out);
  return MK_OK;
}

Params step_params(mk_handle* h, const int32_t* tok, const int32_t* pos, float* logits) {
  Params p = h->base;
  for (int b = 0; b < kMaxBatch; ++b) {
    p.tok[b] = b < h->shape.B ? tok[b] : 0;
    p.pos[b] = b < h->shape.B ? pos[b] : 0;
  }
  p.logits = logits;
  p.tok_keys = nullptr;
  p.argmax_out = nullptr;
  const int set = (int)(h->steps & 1ull);
  p.ctr = h->d_ctr + (size_t)set * h->n_ctr;
  p.ctr_zero = h->d_ctr + (size_t)(set ^ 1) * h->n_ctr;
  p.stamp = h->stamp_serial & 1u;
  return p;
}

// A device timeout of an earlier step, seen through the mapped host mirror of
// the error word without synchronising; sticky until mk_get_status.
int check_sticky(mk_handle* h) {
  if (h->h_err_mirror && *reinterpret_cast<volatile int*>(h->h_err_mirror) != 0)
    return fail(h, MK_ERR_TIMEOUT, "an earlier step reported a device timeout; call mk_get_status");
  return MK_OK;
}

static_assert(MK_MAX_STEPS_PER_LAUNCH == kMaxLaunchSteps, "steps per launch");

// greedy decode: argmax keys -> token ids
__global__ void keys_to_tokens(const unsigned long long* keys, int n, int32_t* tokens) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) tokens[i] = key_token(keys[i]);
}

}  // namespace

extern "C" {

const char* mk_last_error(const mk_handle* h) {
  return h ? h->err.c_str() : g_create_error.c_str();
}

namespace {

// mk_create and mk_create_paged (kv_block > 0: the caches are block pools)
int create_impl(const mk_config* cfg, const mk_weights* w, void* const* k_cache,
                void* const* v_cache, int kv_block, int n_blocks, mk_handle** out) {
  if (!out) return fail(nullptr, MK_ERR_INVALID, "out is NULL");
  *out = nullptr;
  int rc = check_config(cfg, nullptr);
  if (rc) return rc;
  if (kv_block < 0 || (kv_block > 0 && n_blocks < 1))
    return fail(nullptr, MK_ERR_INVALID, "block_size must be >= 1 and n_blocks >= 1");
  if (!w || !k_cache || !v_cache) return fail(nullptr, MK_ERR_INVALID, "weights / caches NULL");
  const int L = cfg->n_layers;
  if (!w->embed || !w->final_norm || !w->attn_norm || !w->wq || !w->wk || !w->wv || !w->wo ||
      !w->mlp_norm || !w->wgate || !w->wup || !w->wdown)
    return fail(nullptr, MK_ERR_INVALID, "a weight pointer is NULL");
  if (cfg->tied_embeddings ? (w->lm_head != nullptr) : (w->lm_head == nullptr))
    return fail(nullptr, MK_ERR_INVALID, "lm_head must be NULL iff tied_embeddings");
  std::vector<const void*> ptrs = {w->embed, w->final_norm};
  if (w->lm_head) ptrs.push_back(w->lm_head);
  for (int l = 0; l < L; ++l) {
    for (const void* p : {w->attn_norm[l], w->wq[l], w->wk[l], w->wv[l], w->wo[l], w->mlp_norm[l],
                          w->wgate[l], w->wup[l], w->wdown[l], (const void*)k_cache[l],
                          (const void*)v_cache[l]})
      ptrs.push_back(p);
  }
  for (const void* p : ptrs) {
    if (!p) return fail(nullptr, MK_ERR_INVALID, "a weight or cache pointer is NULL");
    if (!aligned16(p)) return fail(nullptr, MK_ERR_INVALID, "pointers must be 16-byte aligned");
  }

  std::unique_ptr<mk_handle> h(new mk_handle());
  h->cfg = *cfg;
  h->shape = shape_of(*cfg);
  h->kv_block = kv_block;
  h->n_blocks = n_blocks;
  h->max_blocks = kv_block > 0 ? (cfg->kv_capacity + kv_block - 1) / kv_block : 0;
  const Shape& s = h->shape;
  cudaError_t ce = cudaGetDevice(&h->device);
  if (ce != cudaSuccess) return cuda_fail(nullptr, ce, "cudaGetDevice");
  int optin = 0;
  ce = cudaDeviceGetAttribute(&h->n_sm, cudaDevAttrMultiProcessorCount, h->device);
  if (ce == cudaSuccess)
    ce = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device);
  if (ce != cudaSuccess) return cuda_fail(nullptr, ce, "cudaDeviceGetAttribute");
  h->smem_optin = optin;

  // ---- shared-memory layout
  const int B = s.B;
  Params& p = h->base;
  {
    std::string why;
    h->smem_bytes = smem_layout(s, h->n_sm, optin, misc_bytes(), &p, &why);
    if (!h->smem_bytes) return fail(nullptr, MK_ERR_INVALID, why);
  }

  // ---- model constants
  p.L = s.L; p.H = s.H; p.nh = s.nh; p.nkv = s.nkv; p.D = s.D; p.F = s.F; p.V = s.V;
  p.B = s.B; p.S = s.S; p.G = s.G(); p.Fc = s.Fc(); p.QD = s.QD();
  p.eps = cfg->rms_eps;
  p.embed = static_cast<const uint16_t*>(w->embed);
  p.lm = static_cast<const uint16_t*>(cfg->tied_embeddings ? w->embed : w->lm_head);
  p.final_norm = static_cast<const uint16_t*>(w->final_norm);
  p.timeout_ns = 2000000000ull;

  // ---- scratch: one allocation, 256-byte aligned pieces
  CounterMap cm{s.L, s.nkv, s.B};
  h->n_ctr = cm.count();
  // pieces 0..6 hold the stamped hand-off words (cleared here and after a
  // failed step; the next step then runs with stamp 1)
  size_t sizes[] = {
      sizeof(float) * (size_t)kChunks * B * s.H,                          // xpart
      sizeof(float) * (size_t)B * s.H,                                    // xa
      sizeof(float) * (size_t)B * s.QD(),                                 // q
      sizeof(float) * (size_t)B * s.QD(),                                 // attn
      sizeof(float) * (size_t)B * s.F,                                    // h
      sizeof(float) * (size_t)B * s.nkv * 2 * s.D,                        // new k/v rows
      sizeof(float) * (size_t)B * s.H,                                    // x
      sizeof(float) * (size_t)B * s.nh * kMaxPartitions * (s.D + 2),      // part
      sizeof(float2) * (size_t)s.S * (s.D / 2),                           // rope
      sizeof(int) * (size_t)2 * h->n_ctr,                                 // counters
      sizeof(int) * 64,                                                   // error word
      sizeof(unsigned long long) * (size_t)MK_MAX_GREEDY_STEPS * B,      // argmax keys
      sizeof(int) * (size_t)B * std::max(1, h->max_blocks),               // block table
      sizeof(int) * (size_t)kMaxLaunchSteps * h->n_ctr,                   // several-step counters
      sizeof(float) * (size_t)B * s.V,                                    // prefill logits
  };
  const int npieces = sizeof(sizes) / sizeof(sizes[0]);
  size_t offs[npieces], total = 0;
  for (int i = 0; i < npieces; ++i) {
    offs[i] = total;
    total += (sizes[i] + 255) / 256 * 256;
  }
  ce = cudaMalloc(&h->d_scratch, total);
  if (ce != cudaSuccess) return cuda_fail(nullptr, ce, "cudaMalloc(scratch)");
  char* base = static_cast<char*>(h->d_scratch);
  p.xpart = reinterpret_cast<float*>(base + offs[0]);
  p.xa = reinterpret_cast<float*>(base + offs[1]);
  p.q = reinterpret_cast<float*>(base + offs[2]);
  p.attn = reinterpret_cast<float*>(base + offs[3]);
  p.h = reinterpret_cast<float*>(base + offs[4]);
  p.kvn = reinterpret_cast<float*>(base + offs[5]);
  p.x = reinterpret_cast<float*>(base + offs[6]);
  h->stamped_bytes = offs[7];
  h->stamp_serial = 1;  // the cleared words carry stamp 0
  p.part = reinterpret_cast<float*>(base + offs[7]);
  // (m, l) after the o rows, in the same piece
  p.part_ml = p.part + (size_t)B * s.nh * kMaxPartitions * s.D;
  h->d_rope = reinterpret_cast<float2*>(base + offs[8]);
  h->d_ctr = reinterpret_cast<int*>(base + offs[9]);
  h->d_err = reinterpret_cast<int*>(base + offs[10]);
  h->d_keys = reinterpret_cast<unsigned long long*>(base + offs[11]);
  h->d_table = reinterpret_cast<int*>(base + offs[12]);
  h->d_ctr_steps = reinterpret_cast<int*>(base + offs[13]);
  h->d_plogits = reinterpret_cast<float*>(base + offs[14]);
  p.block_table = nullptr;  // set per step (paged handles)
  p.max_blocks = h->max_blocks;
  p.kv_block = kv_block;
  p.rope = h->d_rope;
  p.err = h->d_err;
  p.n_ctr = h->n_ctr;

  // what a failure below must give back before the handle goes away
  auto release = [&h]() {
    if (h->h_err_mirror) cudaFreeHost(h->h_err_mirror);
    cudaFree(h->d_scratch);
  };
  ce = cudaMemset(h->d_scratch, 0, total);
  if (ce != cudaSuccess) {
    release();
    return cuda_fail(nullptr, ce, "cudaMemset(scratch)");
  }
  ce = cudaHostAlloc(reinterpret_cast<void**>(&h->h_err_mirror), sizeof(int), cudaHostAllocMapped);
  if (ce != cudaSuccess) h->h_err_mirror = nullptr;
  if (ce == cudaSuccess) {
    *h->h_err_mirror = 0;
    ce = cudaHostGetDevicePointer(reinterpret_cast<void**>(&p.err_host), h->h_err_mirror, 0);
  }
  if (ce != cudaSuccess) {
    release();
    return cuda_fail(nullptr, ce, "cudaHostAlloc(error mirror)");
  }
  // RoPE table: angle = pos * theta^(-2i/D), in double, rounded to fp32
  std::vector<float2> rope((size_t)s.S * (s.D / 2));
  for (int pos = 0; pos < s.S; ++pos)
    for (int i = 0; i < s.D / 2; ++i) {
      double ang = (double)pos * std::pow((double)cfg->rope_theta, -2.0 * i / (double)s.D);
      rope[(size_t)pos * (s.D / 2) + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
    }
  LayerPtrs* lp = p.layers;
  for (int l = 0; l < L; ++l) {
    lp[l].attn_norm = static_cast<const uint16_t*>(w->attn_norm[l]);
    lp[l].wq = static_cast<const uint16_t*>(w->wq[l]);
    lp[l].wk = static_cast<const uint16_t*>(w->wk[l]);
    lp[l].wv = static_cast<const uint16_t*>(w->wv[l]);
    lp[l].wo = static_cast<const uint16_t*>(w->wo[l]);
    lp[l].mlp_norm = static_cast<const uint16_t*>(w->mlp_norm[l]);
    lp[l].wgate = static_cast<const uint16_t*>(w->wgate[l]);
    lp[l].wup = static_cast<const uint16_t*>(w->wup[l]);
    lp[l].wdown = static_cast<const uint16_t*>(w->wdown[l]);
    lp[l].kc = static_cast<uint16_t*>(k_cache[l]);
    lp[l].vc = static_cast<uint16_t*>(v_cache[l]);
  }
  h->fn = kernel_for(s, false);
  h->fn_fx = kernel_features(s);
  h->fn_dyn = kernel_dynamic(s);
  ce = cudaMemcpy(h->d_rope, rope.data(), sizeof(float2) * rope.size(), cudaMemcpyHostToDevice);
  if (ce == cudaSuccess)
    ce = allow_max_smem(h->fn, optin);
  if (ce == cudaSuccess)
    ce = allow_max_smem(h->fn_fx, optin);
  if (ce == cudaSuccess && h->fn_dyn) ce = allow_max_smem(h->fn_dyn, optin);
  if (ce != cudaSuccess) {
    release();
    return cuda_fail(nullptr, ce, "mk_create upload");
  }
  *out = h.release();
  return MK_OK;
}

}  // namespace

int mk_create(const mk_config* cfg, const mk_weights* w, void* const* k_cache,
              void* const* v_cache, mk_handle** out) {
  return create_impl(cfg, w, k_cache, v_cache, 0, 0, out);
}

int mk_create_paged(const mk_config* cfg, const mk_weights* w, void* const* k_pool,
                    void* const* v_pool, int block_size, int n_blocks, mk_handle** out) {
  if (block_size < 1) return fail(nullptr, MK_ERR_INVALID, "block_size must be >= 1");
  return create_impl(cfg, w, k_pool, v_pool, block_size, n_blocks, out);
}

int mk_destroy(mk_handle* h) {
  if (!h) return MK_OK;
  cudaDeviceSynchronize();
  for (PlanEntry* e : h->plans) free_plan(e);
  for (auto& sp : h->steps_plans) {
    cudaFree(sp.d_instrs);
    cudaFree(sp.d_sm_off);
  }
  cudaFree(h->d_scratch);
  if (h->h_err_mirror) cudaFreeHost(h->h_err_mirror);
  delete h;
  return MK_OK;
}

int mk_set_timeout(mk_handle* h, uint64_t ns) {
  if (!h) return MK_ERR_INVALID;
  if (ns == 0) return fail(h, MK_ERR_INVALID, "timeout must be positive");
  h->base.timeout_ns = ns;
  return MK_OK;
}

int mk_set_trace(mk_handle* h, mk_trace_record* buf, int capacity) {
  if (!h) return MK_ERR_INVALID;
  if (buf && capacity <= 0) return fail(h, MK_ERR_INVALID, "trace capacity must be positive");
  h->base.trace = buf;
  h->base.trace_cap = buf ? capacity : 0;
  return MK_OK;
}

int mk_debug_use_generic_kernel(mk_handle* h, int enable) {
  if (!h) return MK_ERR_INVALID;
  const Shape& s = h->shape;
  const void* fn = kernel_for(s, enable != 0);
  MK_CUDA(h, allow_max_smem(fn, h->smem_optin));
  h->fn = fn;
  return MK_OK;
}

int mk_set_dynamic(mk_handle* h, int flags) {
  if (!h) return MK_ERR_INVALID;
  if (flags & ~MK_DYN_LMHEAD) return fail(h, MK_ERR_INVALID, "unknown dynamic distribution flag");
  if (flags && !h->fn_dyn)
    return fail(h, MK_ERR_INVALID, "dynamic distribution is not built for this model shape");
  h->dyn = flags;
  return MK_OK;
}

int mk_debug_permute_queues(mk_handle* h, uint32_t seed) {
  if (!h) return MK_ERR_INVALID;
  h->perm_seed = seed;
  return MK_OK;
}

int mk_debug_inject_unsatisfiable_wait(mk_handle* h, int enable) {
  if (!h) return MK_ERR_INVALID;
  h->inject = enable ? 1 : 0;
  return MK_OK;
}

int mk_decode_step_paged(mk_handle* h, const int32_t* tok, const int32_t* pos,
                         const int32_t* block_table, float* logits, void* stream) {
  if (!h) return MK_ERR_INVALID;
  if (h->kv_block == 0) return fail(h, MK_ERR_INVALID, "not a paged handle (mk_create_paged)");
  int rc = check_steps(h, tok, pos);
  if (rc) return rc;
  if (!block_table) return fail(h, MK_ERR_INVALID, "block_table is NULL");
  for (int b = 0; b < h->shape.B; ++b)
    for (int i = 0; i <= pos[b] / h->kv_block; ++i) {
      const int e = block_table[b * h->max_blocks + i];
      if (e < 0 || e >= h->n_blocks)
        return fail(h, MK_ERR_INVALID, "block_table entry out of range [0, n_blocks)");
    }
  if (!logits || !aligned16(logits)) return fail(h, MK_ERR_INVALID, "logits must be 16-byte aligned");
  rc = check_sticky(h);
  if (rc) return rc;
  PlanEntry* e = nullptr;
  rc = get_plan(h, pos, &e, 0);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // pageable source: the copy has read the table when the call returns
  MK_CUDA(h, cudaMemcpyAsync(h->d_table, block_table,
                             sizeof(int) * (size_t)h->shape.B * h->max_blocks,
                             cudaMemcpyHostToDevice, st));
  Params p = step_params(h, tok, pos, logits);
  p.block_table = h->d_table;
  p.instrs = e->d_instrs;
  p.sm_off = e->d_sm_off;
  p.no_waits = 0;
  p.trace_base = 0;
  void* args[] = {&p};
  cudaError_t ce = cudaLaunchCooperativeKernel(h->fn_fx, dim3(h->n_sm), dim3(kThreads), args,
                                               (size_t)h->smem_bytes, st);
  if (ce != cudaSuccess) return cuda_fail(h, ce, "cudaLaunchCooperativeKernel");
  h->cur_set = (int)(h->steps & 1ull);
  h->steps++;
  h->stamp_serial += (uint32_t)h->shape.L;
  return MK_OK;
}

int mk_decode_step(mk_handle* h, const int32_t* tok, const int32_t* pos, float* logits,
                   void* stream) {
  if (!h) return MK_ERR_INVALID;
  if (h->kv_block) return fail(h, MK_ERR_INVALID, "paged handle: use mk_decode_step_paged");
  int rc = check_steps(h, tok, pos);
  if (rc) return rc;
  if (!logits || !aligned16(logits)) return fail(h, MK_ERR_INVALID, "logits must be 16-byte aligned");
  rc = check_sticky(h);
  if (rc) return rc;
  PlanEntry* e = nullptr;
  rc = get_plan(h, pos, &e, h->dyn);
  if (rc) return rc;
  Params p = step_params(h, tok, pos, logits);
  p.instrs = e->d_instrs;
  p.sm_off = e->d_sm_off;
  p.no_waits = 0;
  p.trace_base = 0;
  void* args[] = {&p};
  // dynamic distribution is compiled into its own instantiations
  cudaError_t ce = cudaLaunchCooperativeKernel(h->dyn ? h->fn_dyn : h->fn, dim3(h->n_sm),
                                               dim3(kThreads), args, (size_t)h->smem_bytes,
                                               static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess) return cuda_fail(h, ce, "cudaLaunchCooperativeKernel");
  h->cur_set = (int)(h->steps & 1ull);
  h->steps++;
  h->stamp_serial += (uint32_t)h->shape.L;
  return MK_OK;
}

int mk_prefill(mk_handle* h, const int32_t* tokens, int n_tokens, int start_pos,
               float* logits_out, void* stream) {
  if (!h) return MK_ERR_INVALID;
  if (h->kv_block) return fail(h, MK_ERR_INVALID, "paged handle: prefill needs contiguous caches");
  const int B = h->shape.B;
  if (!tokens || n_tokens < 1) return fail(h, MK_ERR_INVALID, "tokens must be non-NULL, n_tokens >= 1");
  const int chunks = (n_tokens + B - 1) / B;
  if (start_pos < 0 || (long)start_pos + (long)chunks * B > h->shape.S)
    return fail(h, MK_ERR_INVALID,
                "start_pos + n_tokens rounded up to whole chunks of batch rows must fit kv_capacity");
  for (int i = 0; i < n_tokens; ++i)
    if (tokens[i] < 0 || tokens[i] >= h->shape.V)
      return fail(h, MK_ERR_INVALID, "token id out of range [0, vocab)");
  if (!logits_out || !aligned16(logits_out))
    return fail(h, MK_ERR_INVALID, "logits must be 16-byte aligned");
  int rc = check_sticky(h);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int c = 0; c < chunks; ++c) {
    // row b: token c * B + b at position start_pos + c * B + b; the rows past
    // the last token (a partial last chunk) repeat it at the positions after
    // the prompt, whose cache slots the decode steps that follow overwrite
    // before anything reads them
    int32_t tk[kMaxBatch], ps[kMaxBatch];
    for (int b = 0; b < B; ++b) {
      const int i = std::min(c * B + b, n_tokens - 1);
      tk[b] = tokens[i];
      ps[b] = start_pos + c * B + b;
    }
    PlanEntry* e = nullptr;
    rc = get_plan(h, ps, &e, 0);
    if (rc) return rc;
    Params p = step_params(h, tk, ps, h->d_plogits);
    p.prefill = 1;
    p.instrs = e->d_instrs;
    p.sm_off = e->d_sm_off;
    p.no_waits = 0;
    p.trace_base = 0;
    void* args[] = {&p};
    cudaError_t ce = cudaLaunchCooperativeKernel(h->fn, dim3(h->n_sm), dim3(kThreads), args,
                                                 (size_t)h->smem_bytes, st);
    if (ce != cudaSuccess) return cuda_fail(h, ce, "cudaLaunchCooperativeKernel");
    h->cur_set = (int)(h->steps & 1ull);
    h->steps++;
    h->stamp_serial += (uint32_t)h->shape.L;
  }
  // the last prompt token's row of the last chunk
  const int last_row = (n_tokens - 1) - (chunks - 1) * B;
  MK_CUDA(h, cudaMemcpyAsync(logits_out, h->d_plogits + (size_t)last_row * h->shape.V,
                             sizeof(float) * (size_t)h->shape.V, cudaMemcpyDeviceToDevice, st));
  return MK_OK;
}

int mk_decode_greedy(mk_handle* h, const int32_t* tok, const int32_t* pos, int n_steps,
                     int32_t* tokens_out, float* logits, void* stream) {
  if (!h) return MK_ERR_INVALID;
  if (h->kv_block) return fail(h, MK_ERR_INVALID, "paged handle: greedy decode needs contiguous caches");
  int rc = check_steps(h, tok, pos);
  if (rc) return rc;
  if (n_steps < 1 || n_steps > MK_MAX_GREEDY_STEPS)
    return fail(h, MK_ERR_INVALID, "n_steps must be in [1, MK_MAX_GREEDY_STEPS]");
  for (int b = 0; b < h->shape.B; ++b)
    if (pos[b] + n_steps - 1 >= h->shape.S)
      return fail(h, MK_ERR_INVALID, "positions + n_steps - 1 must be < kv_capacity");
  if (!tokens_out || !aligned16(tokens_out))
    return fail(h, MK_ERR_INVALID, "tokens_out must be 16-byte aligned");
  if (!logits || !aligned16(logits)) return fail(h, MK_ERR_INVALID, "logits must be 16-byte aligned");
  rc = check_sticky(h);
  if (rc) return rc;
  const int B = h->shape.B;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MK_CUDA(h, cudaMemsetAsync(h->d_keys, 0, sizeof(unsigned long long) * (size_t)n_steps * B, st));
  int32_t ps[kMaxBatch];
  for (int s = 0; s < n_steps; ++s) {
    for (int b = 0; b < B; ++b) ps[b] = pos[b] + s;
    PlanEntry* e = nullptr;
    rc = get_plan(h, ps, &e, 0);
    if (rc) return rc;
    Params p = step_params(h, tok, ps, logits);
    p.tok_keys = s > 0 ? h->d_keys + (size_t)(s - 1) * B : nullptr;
    p.argmax_out = h->d_keys + (size_t)s * B;
    p.instrs = e->d_instrs;
    p.sm_off = e->d_sm_off;
    p.no_waits = 0;
    p.trace_base = 0;
    void* args[] = {&p};
    cudaError_t ce = cudaLaunchCooperativeKernel(h->fn_fx, dim3(h->n_sm), dim3(kThreads), args,
                                                 (size_t)h->smem_bytes, st);
    if (ce != cudaSuccess) return cuda_fail(h, ce, "cudaLaunchCooperativeKernel");
    h->cur_set = (int)(h->steps & 1ull);
    h->steps++;
    h->stamp_serial += (uint32_t)h->shape.L;
  }
  const int n = n_steps * B;
  keys_to_tokens<<<(n + 255) / 256, 256, 0, st>>>(h->d_keys, n, tokens_out);
  MK_CUDA(h, cudaGetLastError());
  return MK_OK;
}

int mk_decode_greedy_persistent(mk_handle* h, const int32_t* tok, const int32_t* pos,
                                int n_steps, int32_t* tokens_out, float* logits, void* stream) {
  if (!h) return MK_ERR_INVALID;
  if (h->kv_block) return fail(h, MK_ERR_INVALID, "paged handle: greedy decode needs contiguous caches");
  int rc = check_steps(h, tok, pos);
  if (rc) return rc;
  if (n_steps < 1 || n_steps > MK_MAX_STEPS_PER_LAUNCH)
    return fail(h, MK_ERR_INVALID, "n_steps must be in [1, MK_MAX_STEPS_PER_LAUNCH]");
  const int B = h->shape.B;
  for (int b = 0; b < B; ++b)
    if (pos[b] + n_steps - 1 >= h->shape.S)
      return fail(h, MK_ERR_INVALID, "positions + n_steps - 1 must be < kv_capacity");
  if (!tokens_out || !aligned16(tokens_out))
    return fail(h, MK_ERR_INVALID, "tokens_out must be 16-byte aligned");
  if (!logits || !aligned16(logits)) return fail(h, MK_ERR_INVALID, "logits must be 16-byte aligned");
  rc = check_sticky(h);
  if (rc) return rc;
  // the plan: every step's partitions (cached by them)
  std::vector<int> parts((size_t)n_steps * kMaxBatch, 0);
  std::vector<int> key(1, n_steps);
  for (int s = 0; s < n_steps; ++s) {
    int32_t ps[kMaxBatch] = {0};
    for (int b = 0; b < B; ++b) ps[b] = pos[b] + s;
    choose_partitions(h->shape, h->n_sm, ps, parts.data() + (size_t)s * kMaxBatch);
    key.insert(key.end(), parts.begin() + (size_t)s * kMaxBatch,
               parts.begin() + (size_t)(s + 1) * kMaxBatch);
  }
  mk_handle::StepsPlan* sp = nullptr;
  for (auto& c : h->steps_plans)
    if (c.key == key) sp = &c;
  if (!sp) {
    Plan P;
    std::string why;
    if (!build_plan_steps(h->shape, h->n_sm, parts.data(), n_steps, &P, &why))
      return fail(h, MK_ERR_INVALID, why);
    if (h->steps_plans.size() >= 4) {
      MK_CUDA(h, cudaDeviceSynchronize());
      cudaFree(h->steps_plans.front().d_instrs);
      cudaFree(h->steps_plans.front().d_sm_off);
      h->steps_plans.erase(h->steps_plans.begin());
    }
    mk_handle::StepsPlan c;
    c.key = key;
    cudaError_t ue = cudaMalloc(&c.d_instrs, sizeof(Instr) * std::max<size_t>(1, P.instrs.size()));
    if (ue == cudaSuccess) ue = cudaMalloc(&c.d_sm_off, sizeof(int) * P.sm_off.size());
    if (ue == cudaSuccess)
      ue = cudaMemcpy(c.d_instrs, P.instrs.data(), sizeof(Instr) * P.instrs.size(),
                      cudaMemcpyHostToDevice);
    if (ue == cudaSuccess)
      ue = cudaMemcpy(c.d_sm_off, P.sm_off.data(), sizeof(int) * P.sm_off.size(),
                      cudaMemcpyHostToDevice);
    if (ue != cudaSuccess) {
      cudaFree(c.d_instrs);
      cudaFree(c.d_sm_off);
      return cuda_fail(h, ue, "uploading the several-step plan");
    }
    h->steps_plans.push_back(c);
    sp = &h->steps_plans.back();
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MK_CUDA(h, cudaMemsetAsync(h->d_ctr_steps, 0, sizeof(int) * (size_t)n_steps * h->n_ctr, st));
  MK_CUDA(h, cudaMemsetAsync(h->d_keys, 0, sizeof(unsigned long long) * (size_t)n_steps * B, st));
  Params p = step_params(h, tok, pos, logits);
  p.ctr = h->d_ctr_steps;
  p.ctr_zero = nullptr;  // this launch's counters were cleared just above
  p.n_ctr_step = h->n_ctr;
  p.lm_ctr = CounterMap{h->shape.L, h->shape.nkv, B}.lm();
  p.argmax_out = h->d_keys;
  p.instrs = sp->d_instrs;
  p.sm_off = sp->d_sm_off;
  p.no_waits = 0;
  p.trace_base = 0;
  void* args[] = {&p};
  cudaError_t ce = cudaLaunchCooperativeKernel(h->fn_fx, dim3(h->n_sm), dim3(kThreads), args,
                                               (size_t)h->smem_bytes, st);
  if (ce != cudaSuccess) return cuda_fail(h, ce, "cudaLaunchCooperativeKernel");
  h->stamp_serial += (uint32_t)n_steps * (uint32_t)h->shape.L;
  const int n = n_steps * B;
  keys_to_tokens<<<(n + 255) / 256, 256, 0, st>>>(h->d_keys, n, tokens_out);
  MK_CUDA(h, cudaGetLastError());
  return MK_OK;
}

int mk_decode_step_multilaunch(mk_handle* h, const int32_t* tok, const int32_t* pos,
                               float* logits, void* stream, int use_graph) {
  if (!h) return MK_ERR_INVALID;
  if (h->kv_block) return fail(h, MK_ERR_INVALID, "paged handle: the multi-launch build needs contiguous caches");
  int rc = check_steps(h, tok, pos);
  if (rc) return rc;
  if (!logits || !aligned16(logits)) return fail(h, MK_ERR_INVALID, "logits must be 16-byte aligned");
  rc = check_sticky(h);
  if (rc) return rc;
  PlanEntry* e = nullptr;
  rc = get_plan(h, pos, &e, h->dyn);
  if (rc) return rc;
  Params p = step_params(h, tok, pos, logits);
  p.no_waits = 1;
  p.trace = nullptr;
  p.trace_cap = 0;
  const void* fn = h->dyn ? h->fn_dyn : h->fn;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t nph = e->plan.phases.size();
  std::vector<Params> ps(nph, p);
  for (size_t k = 0; k < nph; ++k) {
    ps[k].instrs = e->d_phase_instrs + e->phase_instr_base[k];
    ps[k].sm_off = e->d_phase_off + e->phase_off_base[k];
    if (k > 0) ps[k].ctr_zero = nullptr;
  }
  if (!use_graph) {
    for (size_t k = 0; k < nph; ++k) {
      void* args[] = {&ps[k]};
      cudaError_t ce = cudaLaunchKernel(fn, dim3(h->n_sm), dim3(kThreads), args,
                                        (size_t)h->smem_bytes, st);
      if (ce != cudaSuccess) return cuda_fail(h, ce, "cudaLaunchKernel");
    }
  } else {
    if (!e->gexec) {
      MK_CUDA(h, cudaGraphCreate(&e->graph, 0));
      cudaGraphNode_t prev = nullptr;
      for (size_t k = 0; k < nph; ++k) {
        cudaKernelNodeParams kp{};
        void* args[] = {&ps[k]};
        kp.func = const_cast<void*>(fn);
        kp.gridDim = dim3(h->n_sm);
        kp.blockDim = dim3(kThreads);
        kp.sharedMemBytes = (unsigned)h->smem_bytes;
        kp.kernelParams = args;
        cudaGraphNode_t node;
        MK_CUDA(h, cudaGraphAddKernelNode(&node, e->graph, prev ? &prev : nullptr, prev ? 1 : 0, &kp));
        e->nodes.push_back(node);
        prev = node;
      }
      MK_CUDA(h, cudaGraphInstantiate(&e->gexec, e->graph, 0));
    } else {
      for (size_t k = 0; k < nph; ++k) {
        cudaKernelNodeParams kp{};
        void* args[] = {&ps[k]};
        kp.func = const_cast<void*>(fn);
        kp.gridDim = dim3(h->n_sm);
        kp.blockDim = dim3(kThreads);
        kp.sharedMemBytes = (unsigned)h->smem_bytes;
        kp.kernelParams = args;
        MK_CUDA(h, cudaGraphExecKernelNodeSetParams(e->gexec, e->nodes[k], &kp));
      }
    }
    MK_CUDA(h, cudaGraphLaunch(e->gexec, st));
  }
  h->cur_set = (int)(h->steps & 1ull);
  h->steps++;
  h->stamp_serial += (uint32_t)h->shape.L;
  return MK_OK;
}

int mk_get_status(mk_handle* h, void* stream) {
  if (!h) return MK_ERR_INVALID;
  MK_CUDA(h, cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  int e = 0;
  MK_CUDA(h, cudaMemcpy(&e, h->d_err, sizeof e, cudaMemcpyDeviceToHost));
  if (h->h_err_mirror) *reinterpret_cast<volatile int*>(h->h_err_mirror) = 0;
  if (e != 0) {
    MK_CUDA(h, cudaMemset(h->d_err, 0, sizeof e));
    // the failed step may have left stamped words unwritten: clear them all
    // so that no stale word can carry the next step's stamp
    MK_CUDA(h, cudaMemset(h->d_scratch, 0, h->stamped_bytes));
    h->stamp_serial = 1;
    int code = (e >> 24) & 0xff;
    char buf[128];
    std::snprintf(buf, sizeof buf, "device error word 0x%08x (code %d, site %d)", e, code, e & 0xffffff);
    return fail(h, code ? code : MK_ERR_CUDA, buf);
  }
  return MK_OK;
}

int mk_read_counters(mk_handle* h, int32_t* out, int capacity, int* n_out) {
  if (!h || !n_out) return MK_ERR_INVALID;
  *n_out = h->n_ctr;
  if (!out || capacity < h->n_ctr) return fail(h, MK_ERR_INVALID, "counter buffer too small");
  MK_CUDA(h, cudaDeviceSynchronize());
  MK_CUDA(h, cudaMemcpy(out, h->d_ctr + (size_t)h->cur_set * h->n_ctr, sizeof(int) * h->n_ctr,
                        cudaMemcpyDeviceToHost));
  return MK_OK;
}

int mk_schedule_build_dynamic(const mk_config* cfg, int n_sm, const int32_t* positions,
                              int dyn_flags, mk_instr* instrs, int instr_capacity, int* n_instr,
                              int32_t* sm_offsets, int32_t* targets, int counter_capacity,
                              int* n_counters) {
  int rc = check_config(cfg, nullptr);
  if (rc) return rc;
  if (n_sm < 1 || !positions) return fail(nullptr, MK_ERR_INVALID, "n_sm / positions");
  Shape s = shape_of(*cfg);
  for (int b = 0; b < s.B; ++b)
    if (positions[b] < 0 || positions[b] >= s.S)
      return fail(nullptr, MK_ERR_INVALID, "position out of range [0, kv_capacity)");
  int parts[kMaxBatch];
  choose_partitions(s, n_sm, positions, parts);
  Plan P;
  std::string why;
  if (dyn_flags & ~MK_DYN_LMHEAD) return fail(nullptr, MK_ERR_INVALID, "unknown dynamic flag");
  if (!build_plan(s, n_sm, parts, &P, &why, dyn_flags)) return fail(nullptr, MK_ERR_INVALID, why);
  if (n_instr) *n_instr = (int)P.instrs.size();
  if (n_counters) *n_counters = (int)P.targets.size();
  if (instrs) {
    if (instr_capacity < (int)P.instrs.size())
      return fail(nullptr, MK_ERR_INVALID, "instruction capacity too small");
    std::memcpy(instrs, P.instrs.data(), sizeof(Instr) * P.instrs.size());
  }
  if (sm_offsets) std::memcpy(sm_offsets, P.sm_off.data(), sizeof(int) * P.sm_off.size());
  if (targets) {
    if (counter_capacity < (int)P.targets.size())
      return fail(nullptr, MK_ERR_INVALID, "counter capacity too small");
    std::memcpy(targets, P.targets.data(), sizeof(int) * P.targets.size());
  }
  return MK_OK;
}


int mk_schedule_build_steps(const mk_config* cfg, int n_sm, const int32_t* positions, int n_steps,
                            mk_instr* instrs, int instr_capacity, int* n_instr,
                            int32_t* sm_offsets, int32_t* targets, int counter_capacity,
                            int* n_counters) {
  int rc = check_config(cfg, nullptr);
  if (rc) return rc;
  if (n_sm < 1 || !positions) return fail(nullptr, MK_ERR_INVALID, "n_sm / positions");
  if (n_steps < 1 || n_steps > MK_MAX_STEPS_PER_LAUNCH)
    return fail(nullptr, MK_ERR_INVALID, "n_steps must be in [1, MK_MAX_STEPS_PER_LAUNCH]");
  Shape s = shape_of(*cfg);
  for (int b = 0; b < s.B; ++b)
    if (positions[b] < 0 || positions[b] + n_steps - 1 >= s.S)
      return fail(nullptr, MK_ERR_INVALID, "positions + n_steps - 1 must be in [0, kv_capacity)");
  std::vector<int> parts((size_t)n_steps * kMaxBatch, 0);
  for (int st = 0; st < n_steps; ++st) {
    int32_t ps[kMaxBatch] = {0};
    for (int b = 0; b < s.B; ++b) ps[b] = positions[b] + st;
    choose_partitions(s, n_sm, ps, parts.data() + (size_t)st * kMaxBatch);
  }
  Plan P;
  std::string why;
  if (!build_plan_steps(s, n_sm, parts.data(), n_steps, &P, &why))
    return fail(nullptr, MK_ERR_INVALID, why);
  if (n_instr) *n_instr = (int)P.instrs.size();
  if (n_counters) *n_counters = (int)P.targets.size();
  if (instrs) {
    if (instr_capacity < (int)P.instrs.size())
      return fail(nullptr, MK_ERR_INVALID, "instruction capacity too small");
    std::memcpy(instrs, P.instrs.data(), sizeof(Instr) * P.instrs.size());
  }
  if (sm_offsets) std::memcpy(sm_offsets, P.sm_off.data(), sizeof(int) * P.sm_off.size());
  if (targets) {
    if (counter_capacity < (int)P.targets.size())
      return fail(nullptr, MK_ERR_INVALID, "counter capacity too small");
    std::memcpy(targets, P.targets.data(), sizeof(int) * P.targets.size());
  }
  return MK_OK;
}

int mk_schedule_build(const mk_config* cfg, int n_sm, const int32_t* positions, mk_instr* instrs,
                      int instr_capacity, int* n_instr, int32_t* sm_offsets, int32_t* targets,
                      int counter_capacity, int* n_counters) {
  return mk_schedule_build_dynamic(cfg, n_sm, positions, 0, instrs, instr_capacity, n_instr,
                                   sm_offsets, targets, counter_capacity, n_counters);
}

}  // extern "C"
