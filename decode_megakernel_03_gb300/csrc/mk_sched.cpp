// Host scheduler (see mk_sched.h).
//
// The queues of all SMs are cut from ONE global order of the step:
//
//   for each layer l:
//     QKV(l)  ATTN(l)  RED(l)  OPROJ(l)   (one sequence: no RED; OPROJ reduces)
//     GATEUP(l,0)  GATEUP(l,1)  GATEUP(l,2)  GATEUP(l,3)  DOWN(l)
//   LMHEAD
//
// and every instruction waits only on counters produced by instructions that
// precede it in that order. Each SM's queue is that order filtered to the SM,
// so with all SMs co-resident the step cannot deadlock. The hidden state h is
// produced in four chunks with one counter each, and the down-projection is
// cut along the same chunks: an instruction reading chunk c waits for chunk
// c only (§3.4, the four-chunk MLP: the granularity of a dependency follows
// the granularity of its production).
#include "mk_sched.h"

#include <algorithm>
#include <cstdio>

namespace mk {

std::string check_shape(const Shape& s) {
  char buf[256];
  auto bad = [&](const char* what) {
    std::snprintf(buf, sizeof buf, "unsupported configuration: %s", what);
    return std::string(buf);
  };
  if (s.L < 1 || s.L > kMaxLayers) return bad("n_layers must be in 1..64");
  if (s.H < 256 || s.H % 256 || s.H > 4096) return bad("hidden must be a multiple of 256 in 256..4096");
  if (s.D != 64 && s.D != 128) return bad("head_dim must be 64 or 128");
  if (s.nh < 1 || s.nkv < 1 || s.nh % s.nkv) return bad("n_heads must be a multiple of n_kv_heads");
  if (s.G() > 8) return bad("at most 8 query heads per kv head");
  if (s.QD() % 256 || s.QD() > 4096) return bad("n_heads*head_dim must be a multiple of 256, <= 4096");
  if (s.F < 256 * kChunks || s.F % (256 * kChunks) || s.Fc() > 8192)
    return bad("ffn must be a multiple of 1024 with ffn/4 <= 8192");
  if (s.V < 1) return bad("vocab must be positive");
  if (s.B != 1 && s.B != 2 && s.B != 4 && s.B != 8) return bad("batch must be 1, 2, 4 or 8");
  if (s.S < 1) return bad("kv_capacity must be positive");
  if ((long)s.S * kMaxPartitions >= (1L << 31)) return bad("kv_capacity must be below 2^31 / 64");
  return std::string();
}

int item_cap_for(const Shape& s) { return s.B == 1 ? 64 : (s.B == 2 ? 32 : 16); }

void choose_partitions(const Shape& s, int n_sm, const int* positions, int* parts) {
  long bucket[kMaxBatch];
  long work = 0;
  for (int b = 0; b < s.B; ++b) {
    long len = (long)positions[b] + 1;
    bucket[b] = (len + 255) / 256 * 256;
    work += bucket[b] * s.nkv;
  }
  // about one partition per SM over all (sequence, kv-head) pairs, and at
  // least 64 keys per partition so each stays worth a queue entry. With one
  // sequence the O-projection reduces the partials while staging, so fewer,
  // longer partitions (at least 128 keys: two pages) keep that cheap; the
  // keys stream through pages ahead of the unit, so a longer one costs little
  const long min_keys = fused_reduction(s) ? 128 : 64;
  for (int b = 0; b < kMaxBatch; ++b) parts[b] = 0;
  if (!fused_reduction(s)) {
    // several sequences: at most one unit per SM over all (sequence,
    // kv-head, partition) triples (a second unit on some SMs would double
    // their attention time), dealt one partition at a time to the sequence
    // with the most keys per partition, since the longest unit bounds the
    // layer; no partition drops below min_keys
    const long budget = std::max<long>(s.B, n_sm / std::max(1, s.nkv));
    long total = s.B;
    for (int b = 0; b < s.B; ++b) parts[b] = 1;
    while (total < budget) {
      int best = -1;
      long best_num = 0, best_den = 1;  // keys per partition, as a fraction
      for (int b = 0; b < s.B; ++b) {
        const long len = (long)positions[b] + 1;
        if (parts[b] >= kMaxPartitions || parts[b] >= len) continue;
        if (bucket[b] / (parts[b] + 1) < min_keys) continue;
        if (best < 0 || bucket[b] * best_den > best_num * parts[b]) {
          best = b;
          best_num = bucket[b];
          best_den = parts[b];
        }
      }
      if (best < 0) break;
      ++parts[best];
      ++total;
    }
    return;
  }
  long per = std::max<long>(min_keys, (work + n_sm - 1) / std::max(1, n_sm));
  for (int b = 0; b < s.B; ++b) {
    long p = (bucket[b] + per - 1) / per;
    long len = (long)positions[b] + 1;
    p = std::min<long>(p, len);  // every partition keeps at least one key
    // every SM's O-projection reduces all partitions of all heads while it
    // stages (P x n_heads x head_dim floats per SM), so that cost grows with
    // P while a unit's shrinks: at most 12 (measured on the 1B shape at 8192
    // keys and the 8B shape at 2048: 852 -> 806 and 3637 -> 3532 us/step
    // against the uncapped count; a cap of 8 was slower on both)
    p = std::min<long>(p, 12);
    p = std::max<long>(1, std::min<long>(p, kMaxPartitions));
    parts[b] = (int)p;
  }
}

namespace {

struct Builder {
  const Shape& s;
  int n_sm;
  CounterMap cm;
  int cap;
  // global order: a list of steps, each a list of (sm, instr)
  struct Step {
    int op, layer;
    std::vector<std::pair<int, Instr>> items;
  };
  std::vector<Step> steps;

  Builder(const Shape& sh, int n) : s(sh), n_sm(n), cm{sh.L, sh.nkv, sh.B}, cap(item_cap_for(sh)) {}

  int rot_of(int layer, int step) const {
    return (int)(((long)layer * 61 + (long)step * 23) % n_sm);
  }

  static Instr make(int op, int layer, int a0, int a1, int a2, int wc, int wt, int sc, int sa) {
    Instr in;
    in.op = (int16_t)op;
    in.layer = (int16_t)layer;
    in.a0 = a0;
    in.a1 = a1;
    in.a2 = a2;
    in.wait_ctr = wc;
    in.wait_target = wt;
    in.sig_ctr = sc;
    in.sig_amount = sa;
    return in;
  }

  // Splits [0, n) into n_sm near-equal contiguous ranges, then each range at
  // `cap` items and at multiples of `align` (0 = no alignment cut). Range k
  // goes to SM (k + rot) % n_sm: rotating per step moves the ranges that get
  // one item more around the SMs, so their totals over the step stay level.
  template <class F>
  void spread(int n, int align, int rot, F emit, int item_cap = 0) {
    const int cap = item_cap > 0 ? item_cap : this->cap;
    for (int k = 0; k < n_sm; ++k) {
      int sm = (k + rot) % n_sm;
      int lo = (int)((long)n * k / n_sm);
      int hi = (int)((long)n * (k + 1) / n_sm);
      int a = lo;
      while (a < hi) {
        int b = std::min(hi, a + cap);
        if (align > 0) b = std::min(b, (a / align + 1) * align);
        emit(sm, a, b);
        a = b;
      }
    }
  }

  void add_layer(int l, const int* parts, int rot) {
    const int H = s.H, G = s.G(), Fc = s.Fc();
    const bool fused = fused_reduction(s);
    const int ppg = s.pairs_per_group();
    // 1. RMSNorm + QKV + RoPE + KV append
    {
      Step st{MK_OP_QKV, l, {}};
      int wc = l == 0 ? -1 : cm.xout(l - 1);
      int wt = l == 0 ? 0 : kChunks * H;
      spread(s.pairs(), ppg, rot_of(l, 0), [&](int sm, int a, int b) {
        int g = a / ppg;
        st.items.push_back({sm, make(MK_OP_QKV, l, a, b, 0, wc, wt, cm.qkv(l, g), b - a)});
      });
      steps.push_back(std::move(st));
    }
    // 2. split-KV attention: one unit per (sequence, kv-head, partition)
    {
      Step st{MK_OP_ATTN, l, {}};
      int k = 0;
      for (int b = 0; b < s.B; ++b)
        for (int g = 0; g < s.nkv; ++g)
          for (int p = 0; p < parts[b]; ++p, ++k) {
            int sm = (rot + k) % n_sm;
            st.items.push_back({sm, make(MK_OP_ATTN, l, b, g, (p << 16) | parts[b], cm.qkv(l, g),
                                         ppg, fused ? cm.red(l) : cm.att(l, b, g), 1)});
          }
      steps.push_back(std::move(st));
    }
    // 3. attention reduction: one unit per (sequence, kv-head); one sequence:
    // none, the O-projection reduces while staging
    if (!fused) {
      Step st{MK_OP_RED, l, {}};
      int k = 0;
      for (int b = 0; b < s.B; ++b)
        for (int g = 0; g < s.nkv; ++g, ++k) {
          int sm = (rot + n_sm / 2 + k) % n_sm;
          st.items.push_back({sm, make(MK_OP_RED, l, b, g, parts[b], cm.att(l, b, g), parts[b],
                                       cm.red(l), 1)});
        }
      steps.push_back(std::move(st));
    }
    // 4. O-projection + residual
    {
      Step st{MK_OP_OPROJ, l, {}};
      // fused: a2 = partitions per head, and the wait is for every unit
      const int red_target = fused ? s.nkv * parts[0] : s.B * s.nkv;
      spread(H, 0, rot_of(l, 1), [&](int sm, int a, int b) {
        st.items.push_back({sm, make(MK_OP_OPROJ, l, a, b, fused ? parts[0] : 0, cm.red(l),
                                     red_target, cm.omid(l), b - a)});
      });
      steps.push_back(std::move(st));
    }
    // 5. the four gate/up chunks
    auto gateup = [&](int c) {
      Step st{MK_OP_GATEUP, l, {}};
      spread(Fc, 0, rot_of(l, 2 + c), [&](int sm, int a, int b) {
        st.items.push_back({sm, make(MK_OP_GATEUP, l, c * Fc + a, c * Fc + b, c, cm.omid(l), H,
                                     cm.hch(l, c), b - a)});
      });
      steps.push_back(std::move(st));
    };
    for (int c = 0; c < kChunks; ++c) gateup(c);
    // 6. the down-projection over the (chunk, row) units of the layer: every
    // SM takes one contiguous range of them, so it reads one chunk of h (two
    // where its range crosses a chunk boundary) once, and its instructions
    // wait for that chunk alone. Chunks 0..2 write their rows' shares to
    // xpart[c]; with several sequences or rows wider than 2048 columns the
    // storer of a chunk-3 instruction reads those shares of its rows
    // (stamped words, polled) and writes x = xa + the four shares, so the
    // layer's readers load one vector instead of five (else chunk 3 writes
    // its share too and the readers add them up). The weights of
    // an SM's range do not depend on anything, so they stream in while the
    // gate/up chunks still run. When x is written whole, chunk 3 is its own
    // step (after the others in every queue); the multi-launch build, where
    // the readers add the shares up, still runs them as one kernel.
    {
      const bool whole = x_written_whole(s);
      Step st{MK_OP_DOWN, l, {}}, st3{MK_OP_DOWN, l, {}};
      spread(kChunks * H, H, rot_of(l, 2 + kChunks), [&](int sm, int a, int b) {
        const int c = a / H;
        (whole && c == kChunks - 1 ? st3 : st)
            .items.push_back({sm, make(MK_OP_DOWN, l, a - c * H, b - c * H, c, cm.hch(l, c), Fc,
                                       cm.xout(l), b - a)});
      });
      steps.push_back(std::move(st));
      if (whole) steps.push_back(std::move(st3));
    }
  }

  void add_lm_head(bool dyn) {
    Step st{MK_OP_LMHEAD, -1, {}};
    if (dyn) {
      // one dynamic instruction per SM: row blocks of the static item size,
      // taken from the ticket counter (its count is set to V below)
      const int rows = std::min(64, 2 * cap);
      for (int sm = 0; sm < n_sm; ++sm)
        st.items.push_back({sm, make(MK_OP_LMHEAD, s.L - 1, rows, s.V, cm.dyn() + 1,
                                     cm.xout(s.L - 1), kChunks * s.H, cm.lm(), 0)});
      steps.push_back(std::move(st));
      return;
    }
    // one row per item: twice the items of a row-pair instruction fit the
    // result buffer, up to the 64 the storer's epilogue takes (fewer
    // instructions for the longest GEMV of the step)
    spread(s.V, 0, rot_of(s.L, 0), [&](int sm, int a, int b) {
      st.items.push_back({sm, make(MK_OP_LMHEAD, s.L - 1, a, b, 0, cm.xout(s.L - 1),
                                   kChunks * s.H, cm.lm(), b - a)});
    }, std::min(64, 2 * cap));
    steps.push_back(std::move(st));
  }
};

void cut_queues(const std::vector<const std::vector<std::pair<int, Instr>>*>& lists, int n_sm,
                std::vector<Instr>* instrs, std::vector<int>* sm_off) {
  std::vector<std::vector<Instr>> per(n_sm);
  for (auto* lst : lists)
    for (auto& it : *lst) per[it.first].push_back(it.second);
  instrs->clear();
  sm_off->assign(n_sm + 1, 0);
  for (int sm = 0; sm < n_sm; ++sm) {
    (*sm_off)[sm] = (int)instrs->size();
    instrs->insert(instrs->end(), per[sm].begin(), per[sm].end());
  }
  (*sm_off)[n_sm] = (int)instrs->size();
}

}  // namespace

bool build_plan(const Shape& s, int n_sm, const int* parts, Plan* out, std::string* why,
                int dyn_flags) {
  std::string e = check_shape(s);
  if (!e.empty()) {
    if (why) *why = e;
    return false;
  }
  if (n_sm < 1) {
    if (why) *why = "n_sm must be positive";
    return false;
  }
  for (int b = 0; b < s.B; ++b)
    if (parts[b] < 1 || parts[b] > kMaxPartitions) {
      if (why) *why = "partition count out of range";
      return false;
    }
  Builder bld(s, n_sm);
  for (int l = 0; l < s.L; ++l) bld.add_layer(l, parts, (l * 37) % n_sm);
  bld.add_lm_head((dyn_flags & MK_DYN_LMHEAD) != 0);

  out->n_sm = n_sm;
  for (int b = 0; b < kMaxBatch; ++b) out->parts[b] = b < s.B ? parts[b] : 0;
  std::vector<const std::vector<std::pair<int, Instr>>*> all;
  for (auto& st : bld.steps) all.push_back(&st.items);
  cut_queues(all, n_sm, &out->instrs, &out->sm_off);

  // counter targets = what the producers add up to
  const CounterMap& cm = bld.cm;
  out->targets.assign(cm.count(), 0);
  for (auto& in : out->instrs)
    if (in.sig_ctr >= 0) out->targets[in.sig_ctr] += in.sig_amount;
  // a dynamic LM head counts the rows of the tickets it runs: all V of them
  if (dyn_flags & MK_DYN_LMHEAD) out->targets[cm.lm()] = s.V;
  for (auto& in : out->instrs)
    if (in.wait_ctr >= 0 && in.wait_target != out->targets[in.wait_ctr]) {
      if (why) *why = "internal: a wait target differs from its counter's production";
      return false;
    }

  // multi-launch build: one kernel per (layer, instruction type); the gate/up
  // chunks form one kernel and the down-projection chunks the next
  out->phases.clear();
  size_t i = 0;
  while (i < bld.steps.size()) {
    int op = bld.steps[i].op, layer = bld.steps[i].layer;
    std::vector<const std::vector<std::pair<int, Instr>>*> lists;
    if (op == MK_OP_GATEUP || op == MK_OP_DOWN) {
      // collect all GATEUP (DOWN) steps of this layer into one kernel
      size_t j = i;
      std::vector<const std::vector<std::pair<int, Instr>>*> gu;
      while (j < bld.steps.size() && bld.steps[j].layer == layer && bld.steps[j].op == op) {
        gu.push_back(&bld.steps[j].items);
        ++j;
      }
      Phase p1{op, layer, {}, {}};
      cut_queues(gu, n_sm, &p1.instrs, &p1.sm_off);
      out->phases.push_back(std::move(p1));
      i = j;
      continue;
    }
    lists.push_back(&bld.steps[i].items);
    Phase p{op, layer, {}, {}};
    cut_queues(lists, n_sm, &p.instrs, &p.sm_off);
    out->phases.push_back(std::move(p));
    ++i;
  }
  if (why) why->clear();
  return true;
}

bool build_plan_steps(const Shape& s, int n_sm, const int* parts, int k, Plan* out,
                      std::string* why, int dyn_flags) {
  if (k < 1 || k > kMaxLaunchSteps) {
    if (why) *why = "steps per launch out of range";
    return false;
  }
  if (s.L > (1 << kStepShift)) {
    if (why) *why = "too many layers for steps in one launch";
    return false;
  }
  std::vector<Plan> pl(k);
  for (int st = 0; st < k; ++st)
    if (!build_plan(s, n_sm, parts + st * kMaxBatch, &pl[st], why, dyn_flags)) return false;
  const int nc = (int)pl[0].targets.size();  // counters per step
  const CounterMap cm{s.L, s.nkv, s.B};
  out->n_sm = n_sm;
  for (int b = 0; b < kMaxBatch; ++b) out->parts[b] = pl[0].parts[b];
  out->instrs.clear();
  out->targets.clear();
  out->phases.clear();
  out->sm_off.assign(n_sm + 1, 0);
  for (int st = 0; st < k; ++st)
    out->targets.insert(out->targets.end(), pl[st].targets.begin(), pl[st].targets.end());
  for (int sm = 0; sm < n_sm; ++sm) {
    out->sm_off[sm] = (int)out->instrs.size();
    for (int st = 0; st < k; ++st) {
      for (int i = pl[st].sm_off[sm]; i < pl[st].sm_off[sm + 1]; ++i) {
        Instr in = pl[st].instrs[i];
        in.layer = (int16_t)(in.layer | (st << kStepShift));
        if (in.wait_ctr >= 0) in.wait_ctr += st * nc;
        if (in.sig_ctr >= 0) in.sig_ctr += st * nc;
        if (in.op == MK_OP_LMHEAD && in.a2 > 0) in.a2 += st * nc;  // its ticket counter
        if (st > 0 && in.op == MK_OP_QKV && layer_of(in) == 0) {
          // the token is the previous step's argmax
          in.wait_ctr = cm.lm() + (st - 1) * nc;
          in.wait_target = pl[st - 1].targets[cm.lm()];
        }
        out->instrs.push_back(in);
      }
    }
  }
  out->sm_off[n_sm] = (int)out->instrs.size();
  return true;
}

int smem_layout(const Shape& s, int n_sm, int optin, int misc_bytes, Params* p, std::string* why) {
  // pages | x staging | h staging | results | barriers; the attention
  // scratch reuses the staging area
  (void)n_sm;
  const int B = s.B;
  // several sequences: each staged row is padded by 4 words (bank spread of
  // the tensor-core fragments)
  const int pad = B > 1 ? 4 : 0;
  p->x_floats = B * (std::max(s.H, s.QD()) + pad);
  p->h_floats = B * (s.Fc() + pad);
  p->alias_xh = B > 1 ? 1 : 0;
  p->fused_red = fused_reduction(s) ? 1 : 0;
  p->res_floats = item_cap_for(s) * 2 * B;
  const int att_scratch = kComputeWarps * s.G() * (s.D + 2);
  int xh = p->alias_xh ? std::max(p->x_floats, p->h_floats) : p->x_floats + p->h_floats;
  xh = std::max(xh, att_scratch);
  const int staging_floats = (xh + 3) / 4 * 4;
  // A page slot is always owned by compute warp (slot % kComputeWarps): with
  // the slot count a multiple of the warp count, page k and page k + n_pages
  // (same slot) have the same owner, which consumes them in order, so no warp
  // can wait on a slot two mbarrier phases ahead of its contents.
  const int fixed = staging_floats * 4 + kResBufs * p->res_floats * 4 + ((misc_bytes + 127) / 128) * 128;
  int n_pages = std::min(kMaxPages, (optin - fixed) / kPageBytes);
  n_pages -= n_pages % kComputeWarps;
  if (n_pages < kComputeWarps) {
    if (why) *why = "configuration leaves too few shared-memory pages";
    return 0;
  }
  p->n_pages = n_pages;
  p->off_x = n_pages * kPageBytes;
  p->off_h = p->alias_xh ? p->off_x : p->off_x + p->x_floats * 4;
  p->off_res = p->off_x + staging_floats * 4;
  p->off_misc = (p->off_res + kResBufs * p->res_floats * 4 + 127) / 128 * 128;
  return p->off_misc + misc_bytes;
}

}  // namespace mk
