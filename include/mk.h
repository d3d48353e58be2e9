/*
 * mk.h — C ABI of the GB300 decode megakernel library (libmk.so).
 *
 * One call runs one decode step of a Llama-style decoder (batch 1..8) as ONE
 * persistent kernel: an on-GPU interpreter in which every SM executes a
 * host-prescheduled queue of fused instructions ("3 · L'interpréteur sur GPU",
 * §3.2 "La solution : un interpréteur" and its table of seven instructions),
 * each instruction split into loader / compute / storer warp roles (§3.2, the
 * instruction template), weights streamed into a paged shared-memory allocator
 * (§3.3 "La solution : un allocateur de pages"), and kernel boundaries replaced
 * by zero-initialised global-memory counters with chunked dependencies (§3.4
 * "des compteurs en mémoire globale" and "L'exemple canonique du découpage").
 *
 * Conventions shared by every entry point
 *   - Every function returns an int status: MK_OK (0) or one of MK_ERR_*.
 *     On failure mk_last_error() describes the cause. Validation failures
 *     return before anything is launched or allocated.
 *   - "stream" is a cudaStream_t passed as void*; NULL is the legacy default
 *     stream. Calls that take a stream are asynchronous on it unless stated.
 *   - The caller owns the weights, the KV cache and the logits buffer: the
 *     library never frees, copies or repacks them. The library owns its
 *     scratch (counters, activations, queues) and frees it in mk_destroy.
 *   - Weights are bf16, row-major [out][in] (the nn.Linear layout); every
 *     device pointer must be 16-byte aligned (the weight pages are filled with
 *     bulk asynchronous copies, which move 16-byte units).
 *   - A handle is not thread-safe; use one handle per host thread.
 */
#ifndef MK_H
#define MK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MK_OK 0
#define MK_ERR_INVALID 1 /* bad argument or unsupported configuration */
#define MK_ERR_CUDA 2    /* a CUDA runtime call failed (see mk_last_error) */
#define MK_ERR_TIMEOUT 3 /* a device wait ran past its deadline; the step's
                            outputs are undefined, the context stays usable */
#define MK_ERR_OOM 4     /* device or pinned host allocation failed */

typedef struct mk_handle mk_handle;

/* Model + run configuration. Supported: head_dim 64 or 128; hidden, n_heads *
   head_dim and ffn / 4 multiples of 256 and at most 4096, 4096 and 8192;
   n_heads a multiple of n_kv_heads with at most 8 q-heads per kv-head;
   batch 1, 2, 4 or 8. */
typedef struct {
  int n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab;
  int tied_embeddings; /* 1: the LM head is the embedding matrix */
  float rms_eps, rope_theta;
  int batch;           /* sequences per step, fixed per handle */
  int kv_capacity;     /* S: KV slots per sequence */
} mk_config;

/* Device pointers (bf16). The per-layer members are HOST arrays of n_layers
   device pointers; they are read during mk_create only. */
typedef struct {
  const void* embed;          /* [vocab][hidden] */
  const void* lm_head;        /* [vocab][hidden]; NULL iff tied_embeddings */
  const void* final_norm;     /* [hidden] */
  const void* const* attn_norm; /* [hidden] */
  const void* const* wq;      /* [n_heads*head_dim][hidden] */
  const void* const* wk;      /* [n_kv_heads*head_dim][hidden] */
  const void* const* wv;      /* [n_kv_heads*head_dim][hidden] */
  const void* const* wo;      /* [hidden][n_heads*head_dim] */
  const void* const* mlp_norm;  /* [hidden] */
  const void* const* wgate;   /* [ffn][hidden] */
  const void* const* wup;     /* [ffn][hidden] */
  const void* const* wdown;   /* [hidden][ffn] */
} mk_weights;

/* Creates a handle on the current CUDA device. k_cache / v_cache: host arrays
   of n_layers device pointers, each bf16 [batch][n_kv_heads][kv_capacity]
   [head_dim], caller-owned and updated in place by every decode step. The
   handle records the pointers; they must stay valid until mk_destroy.
   Allocates the scratch (cudaMalloc) and pinned host staging.
   Errors: MK_ERR_INVALID (NULL, misaligned or unsupported), MK_ERR_OOM,
   MK_ERR_CUDA. On error *out is set to NULL. */
int mk_create(const mk_config* cfg, const mk_weights* w,
              void* const* k_cache, void* const* v_cache, mk_handle** out);

/* mk_create for a paged KV cache: k_pool[l] / v_pool[l] (DEVICE, bf16,
   caller-owned, 16-byte aligned) are each layer's block pool
   [n_blocks][n_kv_heads][block_size][head_dim]; position t of sequence b
   lives in block block_table[b][t / block_size] of the table passed to
   mk_decode_step_paged, at row t % block_size. config->kv_capacity bounds
   the positions (block tables have ceil(kv_capacity / block_size) entries
   per sequence). Such a handle takes mk_decode_step_paged only (not
   mk_decode_step, mk_decode_greedy or the multi-launch build).
   Errors: as mk_create, and MK_ERR_INVALID when block_size < 1 or
   n_blocks < 1. */
int mk_create_paged(const mk_config* cfg, const mk_weights* w, void* const* k_pool,
                    void* const* v_pool, int block_size, int n_blocks, mk_handle** out);

/* mk_decode_step for a paged handle. block_table: HOST int32
   [batch][ceil(kv_capacity / block_size)], copied to the device by the call
   (the caller may reuse it on return); the entries that cover positions
   0..positions[b] must lie in [0, n_blocks) (MK_ERR_INVALID before any
   launch otherwise); the step appends sequence b's k/v row at position
   positions[b] into its block. Otherwise as mk_decode_step. */
int mk_decode_step_paged(mk_handle* h, const int32_t* token_ids, const int32_t* positions,
                         const int32_t* block_table, float* logits_out, void* stream);

/* One decode step, ONE kernel launch (the persistent interpreter).
   token_ids, positions: HOST arrays of `batch` int32. Sequence b consumes
   token_ids[b] at position positions[b]: its new k/v row is written into slot
   positions[b] of every layer's cache, and it attends to slots
   0..positions[b] inclusive. The host scheduler needs the positions to size
   the split-KV attention partitions, which is why they are host data.
   logits_out: device fp32 [batch][vocab], caller-owned.
   Asynchronous on `stream`. Returns MK_ERR_INVALID (range checks) before
   launching, MK_ERR_TIMEOUT if an earlier step on this handle reported a
   device timeout (sticky until mk_get_status), else MK_OK / MK_ERR_CUDA. */
int mk_decode_step(mk_handle* h, const int32_t* token_ids, const int32_t* positions,
                   float* logits_out, void* stream);

/* Prefill of a prompt of n_tokens tokens into sequence 0 of the handle's
   cache, at positions start_pos .. start_pos + n_tokens - 1, in chunks of
   `batch` tokens (the handle's batch size): each chunk is ONE interpreter
   launch in which the batch rows are the chunk's consecutive tokens of that
   one sequence. Every GEMV of the step is then a small GEMM over the chunk's
   tokens on the tensor cores, and each token attends causally to the keys
   before it, the chunk's own included ("9 · Quand ne pas le faire", §9.1,
   prefill; "3 · L'interpréteur sur GPU", §3.2, the same instructions).
   tokens: HOST int32 [n_tokens]. The k/v rows of every prompt token are
   written into cache sequence 0; a partial last chunk is padded with rows at
   the positions after the prompt (start_pos + n_tokens rounded up to whole
   chunks must fit kv_capacity), whose slots the next decode steps overwrite
   before reading them. logits_out: DEVICE fp32 [vocab], the logits after
   the last prompt token. Asynchronous on `stream`. Errors as
   mk_decode_step, and MK_ERR_INVALID for a paged handle or out-of-range
   arguments (before any launch). */
int mk_prefill(mk_handle* h, const int32_t* tokens, int n_tokens, int start_pos,
               float* logits_out, void* stream);

/* Greedy decode of n_steps tokens per sequence in one call, the next token
   fed back on the device (no host round trip between steps): step s
   (0 <= s < n_steps) consumes token_ids[b] (s = 0, HOST) or the argmax of
   step s - 1's logits (s > 0) at position positions[b] + s, appending its
   k/v rows there as mk_decode_step does. The LM-head instruction fuses the
   argmax (largest logit; the lowest token id among equal ones):
   tokens_out[s * batch + b] (DEVICE int32, caller-owned, 16-byte aligned)
   receives step s's argmax, logits_out (DEVICE fp32 [batch][vocab]) each
   step's logits in turn, so the last step's remain. One interpreter launch
   per step plus one small conversion launch, back to back on `stream`;
   asynchronous. Returns MK_ERR_INVALID before launching when n_steps is
   outside [1, MK_MAX_GREEDY_STEPS], a position + n_steps - 1 reaches
   kv_capacity or a range check of mk_decode_step fails; otherwise as
   mk_decode_step. */
#define MK_MAX_GREEDY_STEPS 1024
int mk_decode_greedy(mk_handle* h, const int32_t* token_ids, const int32_t* positions,
                     int n_steps, int32_t* tokens_out, float* logits_out, void* stream);

/* mk_decode_greedy with all n_steps steps in ONE persistent launch: each
   SM's queue holds the steps one after the other, every step with its own
   counters; step s + 1's first layer waits on step s's LM head (its argmax
   is the token), and each SM's loader acquires that count before it
   prefetches cached keys an earlier step of the launch wrote. Arguments,
   results and errors as mk_decode_greedy, with 1 <= n_steps <=
   MK_MAX_STEPS_PER_LAUNCH. */
#define MK_MAX_STEPS_PER_LAUNCH 32
int mk_decode_greedy_persistent(mk_handle* h, const int32_t* token_ids, const int32_t* positions,
                                int n_steps, int32_t* tokens_out, float* logits_out,
                                void* stream);

/* The same step run as the multi-launch comparison build: the same
   instruction templates and the same per-SM work units, but one kernel per
   (layer, instruction type) — kernel boundaries instead of counter waits —
   5 * n_layers + 1 launches with one sequence and at most 2048 attention
   columns (n_heads * head_dim), 6 * n_layers + 1 otherwise (a separate
   reduction instruction). use_graph != 0 replays them as one CUDA graph.
   Results are bit-identical to mk_decode_step. */
int mk_decode_step_multilaunch(mk_handle* h, const int32_t* token_ids,
                               const int32_t* positions, float* logits_out,
                               void* stream, int use_graph);

/* Synchronises `stream`, reads the device error word and clears it.
   Returns MK_OK, MK_ERR_TIMEOUT or MK_ERR_CUDA. The error word is
   code << 24 | site (reported in mk_last_error): site 1 a counter wait,
   2 a page or block-table copy, 3 a result buffer or ticket, 5 a value
   handed between instructions that kept its previous layer's stamp. After
   an error the handle also clears those hand-off values, so the next step
   starts from a known state. */
int mk_get_status(mk_handle* h, void* stream);

/* Frees everything the handle owns (synchronising the device first).
   Accepts NULL. */
int mk_destroy(mk_handle* h);

/* Human-readable description of the last error on h (or of the last
   mk_create failure in this thread when h is NULL). Never NULL. */
const char* mk_last_error(const mk_handle* h);

/* ---- test / benchmark helpers ------------------------------------------ */

/* Copies the counter array of the most recent step into host_out
   (synchronising the device). *n_out receives the number of counters; if
   capacity is too small nothing is copied and MK_ERR_INVALID is returned. */
int mk_read_counters(mk_handle* h, int32_t* host_out, int capacity, int* n_out);

/* Deadline of every device wait, in nanoseconds (default 2 s). */
int mk_set_timeout(mk_handle* h, uint64_t timeout_ns);

/* Test-only fault injection on the host schedule: while `enable` is non-zero,
   the wait target of the first counter wait on the last SM's queue is raised
   by one, so that wait can never be satisfied and the step ends with
   MK_ERR_TIMEOUT (device waits are bounded; nothing faults). */
int mk_debug_inject_unsatisfiable_wait(mk_handle* h, int enable);

/* Test-only: with a non-zero seed the handle's plans hand the per-SM queues
   to the CTAs in a seeded random order (CTA k runs the queue the schedule
   built for SM perm[k]); 0 restores the identity. Every CTA is co-resident,
   so any assignment runs, and the results must not depend on it. */
int mk_debug_permute_queues(mk_handle* h, uint32_t seed);

/* Test-only: with `enable` non-zero the handle launches the interpreter
   instantiation that reads the head dimension and q-heads per kv-head at run
   time, instead of one specialised to the model's head shape (the default
   whenever the library has one). Both compute the same results. */
int mk_debug_use_generic_kernel(mk_handle* h, int enable);

/* Per-instruction trace. When dev_buf (device memory holding `capacity`
   mk_trace_record) is non-NULL, the compute warps of every SM write one record
   per instruction they run, timestamped with %globaltimer; record k belongs to
   the k-th instruction of the step in the schedule's SM-major order, so the
   buffer needs at least as many records as the schedule has instructions
   (mk_schedule_build reports that count). Records past `capacity` are dropped.
   Pass NULL to disable. The idle gap between two instructions of one SM is
   t_start(next) - t_end(prev); the dependency stall is t_ready - t_start. The
   storer fills t_stored after the compute warps' record, so read the buffer
   only after the step has completed. */
typedef struct {
  uint32_t sm, index;       /* SM and position in its queue */
  int32_t op, layer;        /* MK_OP_* and layer (-1 for the LM head) */
  uint64_t t_start;         /* compute warps start the instruction */
  uint64_t t_ready;         /* its counter wait (if any) is satisfied */
  uint64_t t_end;           /* compute warps finish it */
  uint64_t t_stored;        /* the storer has published it (counter bumped) */
  uint32_t res_wait_ns;     /* compute warp 0: waiting for a free result buffer */
  uint32_t stage_ns;        /* compute warp 0: staging the activations */
  uint64_t t_issue_first;   /* the loader issues the instruction's first copy
                               (0: the instruction has no pages) */
  uint64_t t_issue_last;    /* the loader issues its last copy */
  uint32_t page_wait_ns;    /* compute warp 0: waiting for its pages to land */
  uint32_t reserved;
} mk_trace_record;
int mk_set_trace(mk_handle* h, mk_trace_record* dev_buf, int capacity);

/* Instruction opcodes (the seven fused instructions of the pages, with the
   embedding lookup folded into layer 0's first instruction). */
#define MK_OP_QKV 1   /* RMSNorm + QKV + RoPE + KV append      (instr. 1) */
#define MK_OP_ATTN 2  /* split-KV attention partial            (instr. 2) */
#define MK_OP_RED 3   /* attention partial reduction           (instr. 3) */
#define MK_OP_OPROJ 4 /* O-projection + residual               (instr. 4) */
#define MK_OP_GATEUP 5 /* RMSNorm + up/gate + SiLU, one chunk  (instr. 5) */
#define MK_OP_DOWN 6  /* down-projection share of one chunk of h (instr. 6) */
#define MK_OP_LMHEAD 7 /* final RMSNorm + LM head              (instr. 7) */

/* One queue entry as the host scheduler emits it (32 bytes). Exported for
   the schedule checks; the meaning of a0..a2 depends on op:
     QKV:    items [a0, a1) of the layer's (q|k|v) row pairs, group-major
     ATTN:   a0 = sequence, a1 = kv-head, a2 = partition << 16 | n_partitions
     RED:    a0 = sequence, a1 = kv-head, a2 = n_partitions
     OPROJ:  output rows [a0, a1)
     GATEUP: hidden units [a0, a1) of chunk a2
     DOWN:   output rows [a0, a1), input chunk a2
     LMHEAD: vocabulary rows [a0, a1) (a2 = 0), or, dynamic (a2 > 0): row
             blocks of a0 rows out of [0, a1), taken from ticket counter
             a2 - 1 by whichever SM reaches the instruction first
             (sig_amount is then the rows of each block it runs)
   wait_ctr < 0 means no wait; sig_ctr < 0 means no signal. */
typedef struct {
  int16_t op, layer;
  int32_t a0, a1, a2;
  int32_t wait_ctr, wait_target;
  int32_t sig_ctr, sig_amount;
} mk_instr;

/* Dynamic work distribution ("3 · L'interpréteur sur GPU", §3.6: the
   instructions dealt to the SMs at run time instead of by a fixed plan).
   MK_DYN_LMHEAD: the LM head's row blocks are taken from a per-step atomic
   ticket counter by the SMs as they reach it. Off by default (the static
   plan); the results are the same either way (each row's arithmetic does
   not depend on which SM computes it). Steps of a handle with a flag set
   (mk_decode_step and the multi-launch build) run an interpreter build of
   their own that carries the ticket code; every other step runs one without
   it. */
#define MK_DYN_LMHEAD 1
int mk_set_dynamic(mk_handle* h, int flags);

/* mk_schedule_build with dynamic work distribution flags (MK_DYN_*). */
int mk_schedule_build_dynamic(const mk_config* cfg, int n_sm, const int32_t* positions,
                              int dyn_flags, mk_instr* instrs, int instr_capacity, int* n_instr,
                              int32_t* sm_offsets, int32_t* targets, int counter_capacity,
                              int* n_counters);

/* Host-only (no CUDA call): builds the schedule that mk_decode_step would run
   for `cfg` on n_sm SMs at these positions (host array of cfg->batch).
   Outputs, each optional (NULL to skip) and bounded by its capacity:
     instrs[*n_instr]          all queues, SM-major, each in execution order
     sm_offsets[n_sm + 1]      queue of SM s = instrs[sm_offsets[s] .. s+1)
     targets[*n_counters]      the value each counter holds after a step
   Returns MK_ERR_INVALID if cfg is unsupported or a capacity is too small
   (the required sizes are still written to *n_instr / *n_counters). */
int mk_schedule_build(const mk_config* cfg, int n_sm, const int32_t* positions,
                      mk_instr* instrs, int instr_capacity, int* n_instr,
                      int32_t* sm_offsets, int32_t* targets, int counter_capacity,
                      int* n_counters);

/* Host-only (no CUDA call): the schedule that mk_decode_greedy_persistent
   runs for n_steps steps (1 <= n_steps <= MK_MAX_STEPS_PER_LAUNCH) from these
   positions: each SM's queue holds the steps one after the other; an
   instruction's step is (layer >> 10) & 31 and its layer layer & 1023;
   counters of step s are those of one step offset by s times the per-step
   count (targets has n_steps times that many entries); step s > 0's layer-0
   QKV instructions wait for step s - 1's LM head. Outputs, capacities and
   errors as for mk_schedule_build; MK_ERR_INVALID also when n_steps is out of
   range or a position + n_steps - 1 reaches kv_capacity. */
int mk_schedule_build_steps(const mk_config* cfg, int n_sm, const int32_t* positions, int n_steps,
                            mk_instr* instrs, int instr_capacity, int* n_instr,
                            int32_t* sm_offsets, int32_t* targets, int counter_capacity,
                            int* n_counters);

/* ---- decode step without any allocation -------------------------------- */

/* The pages have no counterpart of this call; it exists for callers that may
   not allocate device memory: code running inside a memory pool or arena that
   owns every device byte, plugins whose host forbids device allocations after
   start-up, serving paths that must not take the allocator's locks or risk an
   allocation failure.

   Runs the same decode step as mk_decode_step (same kernel, same schedule,
   same results) without a handle. All scratch -- activations, attention
   partials, counters, error word, RoPE table and instruction queues -- lives
   in ONE file-scope device array of 16 MiB that the library reserves on every
   GPU that loads it, until the process exits. The call performs no cudaMalloc,
   cudaFree, pinned-memory or other device allocation (host-side schedule
   building uses ordinary heap memory).

   cfg, w, k_cache, v_cache: as for mk_create (host structs and host arrays of
   device pointers; the caches are updated in place). token_ids, positions:
   host arrays of cfg->batch, as for mk_decode_step. logits_out: device fp32
   [batch][vocab]. stream: cudaStream_t as void*. errmsg / errmsg_cap: optional
   host buffer for a description of a failure (may be NULL / 0).

   The first call on a device resolves the array's device address
   (cudaGetSymbolAddress) and the device attributes; make that first call
   before any stream capture on the device.
   The call is synchronous: it waits for the step on `stream` and returns
   MK_ERR_TIMEOUT if a device wait expired.
   Every call shares the array and leaves its contents behind; each call
   clears the counters, the error word and the values handed between
   instructions itself. Calls that overlap on the
   GPU (several streams or host threads) race on the array: serialise them.
   Errors: MK_ERR_INVALID (bad or unsupported arguments, or a configuration
   whose scratch exceeds the 16 MiB array, reported with the size it needs),
   MK_ERR_CUDA, MK_ERR_TIMEOUT. */
int mk_decode_step_noalloc(const mk_config* cfg, const mk_weights* w,
                           void* const* k_cache, void* const* v_cache,
                           const int32_t* token_ids, const int32_t* positions,
                           float* logits_out, void* stream, char* errmsg, size_t errmsg_cap);

#ifdef __cplusplus
}
#endif
#endif /* MK_H */
