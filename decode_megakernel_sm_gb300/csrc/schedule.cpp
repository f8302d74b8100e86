// schedule.cpp -- host-side schedule builder and checker (plain C++, no CUDA).
//
// "Megakernels: Deleting the Kernel Boundary", section "One launch, one
// interpreter": the per-SM instruction queues are computed on the host ahead
// of time and reused for many forward passes.  Section "Correctness without
// the free barrier": every dependency is a counter that producers increment
// and consumers wait on, at a finer grain than a kernel boundary (per kv
// head after QKV, per kv head after attention, per layer after O-proj/MLP).
//
// Balance: every phase is cut into n_sm contiguous row ranges of (nearly)
// equal bytes, so no SM carries a wave-quantisation tail ("Where the
// microseconds go": 512 blocks on 148 SMs leave a 68-SM last wave).
#include <algorithm>
#include <cstring>
#include <vector>

#include "mk_internal.h"

namespace mk {

static long cut(long total, int n, int i, int align) {
  long v = total * (long)i / n;
  return v / align * align;
}

int plan_shape_ok(const mk_model_desc& d) {
  if (d.n_layers <= 0 || d.hidden <= 0 || d.n_q_heads <= 0 || d.n_kv_heads <= 0 ||
      d.head_dim <= 0 || d.vocab <= 0 || d.max_batch <= 0 || d.max_seq <= 0)
    return MK_ERR_INVALID_ARG;
  if (d.n_q_heads % d.n_kv_heads) return MK_ERR_INVALID_ARG;
  if (!(d.rms_eps >= 0.f) || !(d.rope_theta > 0.f)) return MK_ERR_INVALID_ARG;
  if (d.n_experts < 0 || d.top_k < 0 || d.expert_ffn < 0 || d.shared_ffn < 0 || d.ffn < 0)
    return MK_ERR_INVALID_ARG;
  if (d.n_experts == 0 && d.ffn <= 0) return MK_ERR_INVALID_ARG;
  if (d.batched_variant != 0 && d.batched_variant != 1) return MK_ERR_INVALID_ARG;
  if (d.n_experts > 0 && (d.top_k <= 0 || d.top_k > d.n_experts || d.expert_ffn <= 0))
    return MK_ERR_INVALID_ARG;
  if (d.hidden % 256 || d.hidden > 16384) return MK_ERR_UNSUPPORTED;
  if (d.head_dim != 64 && d.head_dim != 128) return MK_ERR_UNSUPPORTED;
  if (d.n_q_heads / d.n_kv_heads > 8) return MK_ERR_UNSUPPORTED;
  // the last router of a layer ranks up to 256 logits in shared memory
  if (d.n_experts > 256 || d.top_k > 16) return MK_ERR_UNSUPPORTED;
  return MK_OK;
}

// The common end of a plan: hold marks, counter targets, the flattened
// HALT-padded queues and their statistics (all but weight_bytes).
static void finish_plan(std::vector<std::vector<Instr>>& qs, const std::vector<double>& bytes,
                        const CtrMap& cm, unsigned hold_mask, int S, int n_lm, PlanOut& out) {
  const int n_sm = (int)qs.size();
  Instr halt;
  std::memset(&halt, 0, sizeof halt);
  halt.op = OP_HALT;
  halt.wait_ctr = NO_CTR;
  halt.sig_ctr = NO_CTR;
  // ---- hold marks: the first instruction of each run of a held op on an SM
  auto hold_bit = [](uint8_t op) -> unsigned {
    switch (op) {
      case OP_QKV: return HOLD_QKV;
      case OP_ATTN: return HOLD_ATTN;
      case OP_OPROJ: return HOLD_OPROJ;
      case OP_MLP: case OP_MLP_UP: case OP_ROUTER: return HOLD_MLP;
      case OP_MLP_DOWN: return HOLD_DOWN;
      case OP_LMHEAD: return HOLD_LM;
      default: return 0;
    }
  };
  for (auto& q : qs)
    for (size_t k = 1; k < q.size(); k++)
      if ((hold_mask & hold_bit(q[k].op)) &&
          (q[k - 1].op != q[k].op || q[k - 1].layer != q[k].layer))
        q[k].flags |= F_HOLD;

  // ---- counter targets: a wait is for every signal of its counter
  const int n_ctr = cm.count();
  std::vector<uint32_t> cnt(n_ctr, 0);
  for (auto& q : qs)
    for (auto& I : q)
      if (I.sig_ctr != NO_CTR) cnt[I.sig_ctr]++;
  for (auto& q : qs)
    for (auto& I : q) {
      if (I.wait_ctr != NO_CTR) I.wait_cnt = cnt[I.wait_ctr];
    }

  // ---- flatten, HALT-padded
  size_t mx = 0, total = 0;
  for (auto& q : qs) {
    mx = std::max(mx, q.size());
    total += q.size();
  }
  out.max_pc = (int)mx + 1;
  out.q.assign((size_t)n_sm * out.max_pc, halt);
  for (int i = 0; i < n_sm; i++)
    std::copy(qs[i].begin(), qs[i].end(), out.q.begin() + (size_t)i * out.max_pc);
  out.n_ctr = n_ctr;
  out.splits = S;
  out.n_lm = n_lm;
  out.n_instr = (int)total;
  double sum = 0, m = 0;
  for (double v : bytes) {
    sum += v;
    m = std::max(m, v);
  }
  out.max_sm_bytes = m;
  out.mean_sm_bytes = sum / n_sm;
}

// ---------------------------------------------------------- wide batch ----
// 2 .. 32 sequences on the shapes of wide_path ("Megakernels in LLM Inference When Fusion Actually
// Wins", sections "Core Tradeoff" and "When Megakernels Win": the batch range
// where one fused launch meets skinny GEMMs).  Per layer:
//   NORM (attention input) -> QKV rows -> attention items -> O-proj rows ->
//   NORM (MLP input) -> gate/up columns -> down (row block, FFN chunks),
// then the final NORM and the LM head rows.  The norms are one instruction
// per sequence (padded to Bp = B rounded up to 8), spread over the SMs; every
// GEMV instruction holds at most 128 weight rows (the MMA's M) starting on a
// multiple of 8 (the operand atoms); an O-projection instruction covers all
// query heads of one kv group (one K chunk per head).
static int plan_build_wide(const mk_model_desc& d, int B, int max_ctx, int n_sm, PlanOut& out,
                           unsigned hold_mask) {
  const int L = d.n_layers, H = d.hidden, Hq = d.n_q_heads, Hkv = d.n_kv_heads;
  const int D = d.head_dim, HPG = Hq / Hkv, V = d.vocab;
  const long F = d.ffn;
  if (d.n_experts > 0 || B > WIDE_NB || D != WIDE_KC || H % WIDE_KC || F % WIDE_KC)
    return MK_ERR_UNSUPPORTED;
  const int GR = (HPG + 2) * D;
  const long R = (long)Hkv * GR;
  const int Bp = wide_bp(B);
  CtrMap cm{Hkv, L};
  // split-KV: as many slices per (sequence, kv head) pair as keep the items
  // at one per SM (an SM's second item doubles the phase; whole sequences
  // once the pairs number the SMs), at most 4 (each slice adds to the
  // merge), at least 16 positions per slice at max_ctx.  Measured per step
  // with 8 kv heads (ms, slices 1 / 2 / 3 / 4): 4 sequences 0.898 / 0.882 /
  // 0.873 / 0.861, 8 sequences 0.955 / 0.940 / 1.020 / 0.984, 12 sequences
  // 1.022 / 1.127 / 1.086 / 1.132; 2 sequences with 4 / 6 / 9 slices 0.837 /
  // 0.844 / 0.848.  Items are dealt out slice-major and round-robin, so that
  // each SM's items come from different sequences.
  const int pairs = B * Hkv;
  int S = std::min(4, std::max(1, n_sm / pairs));
  S = std::min(S, std::max(1, max_ctx / 16));
  const int n_items = B * Hkv * S;
  std::vector<std::vector<Instr>> qs(n_sm);
  std::vector<double> bytes(n_sm, 0.0);
  auto mk = [](uint8_t op, int layer) {
    Instr I;
    std::memset(&I, 0, sizeof I);
    I.op = op;
    I.layer = (uint16_t)layer;
    I.wait_ctr = NO_CTR;
    I.sig_ctr = NO_CTR;
    return I;
  };
  const double ab = 2.0 * Bp * 128;  // operand bytes of one K chunk
  auto norms = [&](int layer, int which, uint32_t wait, uint32_t sig) {
    for (int b = 0; b < Bp; b++) {
      Instr I = mk(OP_NORM, layer);
      I.g = (uint16_t)which;
      I.r0 = (uint32_t)b;
      I.r1 = (uint32_t)b + 1;
      I.wait_ctr = wait;
      I.sig_ctr = sig;
      qs[(size_t)((long)b * n_sm / Bp)].push_back(I);
    }
  };
  int n_lm = 0;
  for (int l = 0; l < L; l++) {
    norms(l, 0, l > 0 ? cm.mlp(l - 1) : NO_CTR, cm.norm_a(l));
    // ---- QKV rows: per kv head group, cut at multiples of 8 rows
    for (int i = 0; i < n_sm; i++) {
      long a, b;
      if (n_sm >= Hkv) {
        const int g = (int)((long)i * Hkv / n_sm);
        const long s0 = ((long)g * n_sm + Hkv - 1) / Hkv;
        const long s1 = ((long)(g + 1) * n_sm + Hkv - 1) / Hkv;
        const int m = (int)(s1 - s0), k = (int)(i - s0);
        a = (long)g * GR + cut(GR, m, k, 8);
        b = (long)g * GR + (k == m - 1 ? GR : cut(GR, m, k + 1, 8));
      } else {
        a = cut(R, n_sm, i, 8);
        b = (i == n_sm - 1) ? R : cut(R, n_sm, i + 1, 8);
      }
      while (a < b) {
        const long g = a / GR;
        const long e = std::min(std::min(b, (g + 1) * GR), a + (long)WIDE_ROWS);
        Instr I = mk(OP_QKV, l);
        I.g = (uint16_t)g;
        I.r0 = (uint32_t)a;
        I.r1 = (uint32_t)e;
        I.wait_ctr = cm.norm_a(l);
        I.sig_ctr = cm.qkv(l, (int)g);
        qs[i].push_back(I);
        bytes[i] += (double)(e - a) * H * 2 + (double)(H / WIDE_KC) * ab;
        a = e;
      }
    }
    // ---- attention items: item k = slice k / (B Hkv) of pair k % (B Hkv)
    for (int k = 0; k < n_items; k++) {
      const int sm = k % n_sm, pr = k % (B * Hkv);
      Instr I = mk(OP_ATTN, l);
      I.b = (uint16_t)(pr / Hkv);
      I.g = (uint16_t)(pr % Hkv);
      I.r0 = (uint32_t)(k / (B * Hkv));
      I.r1 = (uint32_t)S;
      I.wait_ctr = cm.qkv(l, I.g);
      I.sig_ctr = cm.attn(l, I.g);
      qs[sm].push_back(I);
      bytes[sm] += (double)max_ctx / S * D * 4;
    }
    // ---- O-projection: per kv group, its query heads' Wo columns for a row
    // range (multiples of 8, at most 128 rows); the SMs split evenly over
    // the groups
    for (int i = 0; i < n_sm; i++) {
      int g;
      long a, b;
      if (n_sm >= Hkv) {
        g = (int)((long)i * Hkv / n_sm);
        const long s0 = ((long)g * n_sm + Hkv - 1) / Hkv;
        const long s1 = ((long)(g + 1) * n_sm + Hkv - 1) / Hkv;
        const int m = (int)(s1 - s0), k = (int)(i - s0);
        a = cut(H, m, k, 8);
        b = k == m - 1 ? H : cut(H, m, k + 1, 8);
      } else {  // fewer SMs than groups: SM i takes whole groups
        g = -1;
        a = b = 0;
      }
      auto push = [&](int grp, long a0, long b0) {
        while (a0 < b0) {
          const long e = std::min(b0, a0 + (long)WIDE_ROWS);
          Instr I = mk(OP_OPROJ, l);
          I.g = (uint16_t)grp;
          I.r0 = (uint32_t)a0;
          I.r1 = (uint32_t)e;
          I.flags = grp == 0 ? F_RESIDUAL : 0;
          I.wait_ctr = cm.attn(l, grp);
          I.sig_ctr = cm.oproj(l);
          qs[i].push_back(I);
          bytes[i] += (double)(e - a0) * HPG * D * 2 + HPG * ab;
          a0 = e;
        }
      };
      if (g >= 0) {
        push(g, a, b);
      } else {
        for (int grp = i; grp < Hkv; grp += n_sm) push(grp, 0, H);
      }
    }
    norms(l, 1, cm.oproj(l), cm.norm_m(l));
    // ---- gate/up columns: multiples of 4 (8 interleaved rows), at most 64
    for (int i = 0; i < n_sm; i++) {
      long a = cut(F / 4, n_sm, i, 1) * 4;
      const long b = (i == n_sm - 1) ? F : cut(F / 4, n_sm, i + 1, 1) * 4;
      while (a < b) {
        const long e = std::min(b, a + (long)WIDE_ROWS / 2);
        Instr I = mk(OP_MLP_UP, l);
        I.r0 = (uint32_t)a;
        I.r1 = (uint32_t)e;
        I.wait_ctr = cm.norm_m(l);
        I.sig_ctr = cm.mlp_up(l);
        qs[i].push_back(I);
        bytes[i] += (double)(e - a) * 2 * H * 2 + (double)(H / WIDE_KC) * ab;
        a = e;
      }
    }
    // ---- down: per 128-row block of x, its FFN chunks cut into K ranges,
    // the SMs split evenly over the row blocks (one instruction per SM, so
    // one epilogue of reductions each)
    const long nrb = (H + WIDE_ROWS - 1) / WIDE_ROWS, nch = F / WIDE_KC;
    auto push_down = [&](int i, long rb, long k0, long k1) {
      if (k0 >= k1) return;
      Instr I = mk(OP_MLP_DOWN, l);
      I.r0 = (uint32_t)(rb * WIDE_ROWS);
      I.r1 = (uint32_t)std::min((long)H, (rb + 1) * WIDE_ROWS);
      I.b = (uint16_t)k0;
      I.g = (uint16_t)k1;
      I.wait_ctr = cm.mlp_up(l);
      I.sig_ctr = cm.mlp(l);
      qs[i].push_back(I);
      bytes[i] += (double)(k1 - k0) * ((double)(I.r1 - I.r0) * WIDE_KC * 2 + ab);
    };
    for (int i = 0; i < n_sm; i++) {
      if (n_sm >= nrb) {
        const long rb = (long)i * nrb / n_sm;
        const long s0 = (rb * n_sm + nrb - 1) / nrb, s1 = ((rb + 1) * n_sm + nrb - 1) / nrb;
        const int m = (int)(s1 - s0), k = (int)(i - s0);
        push_down(i, rb, cut(nch, m, k, 1), k == m - 1 ? nch : cut(nch, m, k + 1, 1));
      } else {  // fewer SMs than row blocks: SM i takes whole row blocks
        for (long rb = i; rb < nrb; rb += n_sm) push_down(i, rb, 0, nch);
      }
    }
  }
  norms(L, 2, cm.mlp(L - 1), cm.norm_f());
  // ---- LM head rows: multiples of 8, at most 128 per instruction; an SM's
  // instructions are one argmax slice (aux), the first (b bit 0) and last
  // (bit 1) of them marked
  for (int i = 0; i < n_sm; i++) {
    long a = cut(V, n_sm, i, 8);
    const long b = (i == n_sm - 1) ? V : cut(V, n_sm, i + 1, 8);
    if (a >= b) continue;
    const size_t k0 = qs[i].size();
    while (a < b) {
      const long e = std::min(b, a + (long)WIDE_ROWS);
      Instr I = mk(OP_LMHEAD, L);
      I.r0 = (uint32_t)a;
      I.r1 = (uint32_t)e;
      I.wait_ctr = cm.norm_f();
      I.aux = (uint32_t)n_lm;
      qs[i].push_back(I);
      bytes[i] += (double)(e - a) * H * 2 + (double)(H / WIDE_KC) * ab;
      a = e;
    }
    qs[i][k0].b |= 1;
    qs[i].back().b |= 2;
    n_lm++;
  }
  finish_plan(qs, bytes, cm, hold_mask, S, n_lm, out);
  out.n_ctr += L * B * Hkv;  // the attention-arrival counters (after cm's)
  out.weight_bytes = (double)L * ((double)R * H * 2 + (double)Hq * D * H * 2 + (double)F * H * 6 +
                                  2.0 * H * 2) +
                     (double)V * H * 2 + (double)H * 2;
  return MK_OK;
}

// Coverage check of a wide plan (plan_verify's counterpart).
static int plan_verify_wide(const mk_model_desc& d, int B, const PlanOut& p) {
  const int L = d.n_layers, H = d.hidden, Hq = d.n_q_heads, Hkv = d.n_kv_heads;
  const int D = d.head_dim, HPG = Hq / Hkv, V = d.vocab, GR = (HPG + 2) * D;
  const long R = (long)Hkv * GR, F = d.ffn, nch = F / WIDE_KC;
  const int S = p.splits, Bp = wide_bp(B);
  std::vector<uint8_t> qkv((size_t)L * R, 0), att((size_t)L * B * Hkv * S, 0);
  std::vector<uint8_t> op((size_t)L * Hq * H, 0), up((size_t)L * F, 0);
  std::vector<uint8_t> dn((size_t)L * H * nch, 0), lm(V, 0), slot(p.n_lm, 0);
  std::vector<uint8_t> nrm((size_t)(2 * L + 1) * Bp, 0);
  auto mark = [](std::vector<uint8_t>& v, size_t i) {
    if (i >= v.size() || v[i]) return false;
    v[i] = 1;
    return true;
  };
  for (const Instr& I : p.q) {
    const int l = I.layer;
    if (I.op != OP_HALT && (I.flags & (F_TAG_WAIT | F_RELAXED_SIG))) return 29;
    switch (I.op) {
      case OP_HALT: break;
      case OP_NORM:
        if (I.g > 2 || (I.g == 2) != (l == L) || l > L || I.r1 != I.r0 + 1 || (int)I.r0 >= Bp)
          return 40;
        if (!mark(nrm, (size_t)(I.g == 2 ? 2 * L : 2 * l + I.g) * Bp + I.r0)) return 41;
        break;
      case OP_QKV:
        if (l >= L || I.r0 >= I.r1 || I.r1 > R || I.r1 - I.r0 > (uint32_t)WIDE_ROWS) return 1;
        if (I.r0 / GR != I.g || (I.r1 - 1) / GR != I.g || (I.r0 % 8) || (I.r1 % 2)) return 2;
        for (uint32_t r = I.r0; r < I.r1; r++)
          if (!mark(qkv, (size_t)l * R + r)) return 3;
        break;
      case OP_ATTN:
        if (l >= L || I.b >= B || I.g >= Hkv || (int)I.r1 != S || (int)I.r0 >= S) return 4;
        if (!mark(att, (((size_t)l * B + I.b) * Hkv + I.g) * S + I.r0)) return 5;
        break;
      case OP_OPROJ:  // a kv group's query heads
        if (l >= L || I.g >= Hkv || I.r0 >= I.r1 || (int)I.r1 > H || (I.r0 % 8) ||
            I.r1 - I.r0 > (uint32_t)WIDE_ROWS)
          return 6;
        if (((I.flags & F_RESIDUAL) != 0) != (I.g == 0)) return 7;
        for (int hh = 0; hh < HPG; hh++)
          for (uint32_t r = I.r0; r < I.r1; r++)
            if (!mark(op, ((size_t)l * Hq + (size_t)I.g * HPG + hh) * H + r)) return 8;
        break;
      case OP_MLP_UP:
        if (l >= L || I.r0 >= I.r1 || (long)I.r1 > F || (I.r0 % 4) ||
            2 * (I.r1 - I.r0) > (uint32_t)WIDE_ROWS)
          return 23;
        for (uint32_t c = I.r0; c < I.r1; c++)
          if (!mark(up, (size_t)l * F + c)) return 24;
        break;
      case OP_MLP_DOWN:
        if (l >= L || I.r0 >= I.r1 || (int)I.r1 > H || (I.r0 % 8) ||
            I.r1 - I.r0 > (uint32_t)WIDE_ROWS || I.b >= I.g || (long)I.g > nch)
          return 25;
        for (uint32_t r = I.r0; r < I.r1; r++)
          for (uint32_t k = I.b; k < I.g; k++)
            if (!mark(dn, ((size_t)l * H + r) * nch + k)) return 26;
        break;
      case OP_LMHEAD:
        if (I.r0 >= I.r1 || (int)I.r1 > V || (I.r0 % 8) || I.r1 - I.r0 > (uint32_t)WIDE_ROWS ||
            (int)I.aux >= p.n_lm || I.b > 3)
          return 17;
        if ((I.b & 2) && !mark(slot, I.aux)) return 18;  // one last instruction per slice
        for (uint32_t r = I.r0; r < I.r1; r++)
          if (!mark(lm, r)) return 19;
        break;
      default:
        return 20;
    }
  }
  for (auto* v : {&qkv, &att, &op, &up, &dn, &lm, &slot, &nrm})
    for (uint8_t x : *v)
      if (!x) return 21;
  return 0;
}

int plan_build(const mk_model_desc& d, int B, int max_ctx, int n_sm, PlanOut& out,
               unsigned hold_mask, int wb) {
  int rc = plan_shape_ok(d);
  if (rc) return rc;
  if (B <= 0 || B > d.max_batch || max_ctx <= 0 || max_ctx > d.max_seq || n_sm <= 0)
    return MK_ERR_INVALID_ARG;
  if (wb != 1 && wb != 2) return MK_ERR_INVALID_ARG;
  if (wide_path(d)) return wb == 2 ? plan_build_wide(d, B, max_ctx, n_sm, out, hold_mask)
                                   : MK_ERR_UNSUPPORTED;
  // int8 weights: an LM-head instruction's row scales fit the kernel's
  // hidden-sized scale buffer
  if (wb == 1 && ((long)d.vocab + n_sm - 1) / n_sm > d.hidden) return MK_ERR_UNSUPPORTED;
  const int L = d.n_layers, H = d.hidden, Hq = d.n_q_heads, Hkv = d.n_kv_heads;
  const int D = d.head_dim, HPG = Hq / Hkv, V = d.vocab;
  const bool moe = d.n_experts > 0;
  const int GR = (HPG + 2) * D;  // packed QKV rows per kv head
  const long R = (long)Hkv * GR;
  CtrMap cm{Hkv, L};

  // split-KV slices per (sequence, kv head): about one work item per SM, at
  // least 16 positions per slice on average at max_ctx, and few enough that
  // one head's partials of every sequence fit the smallest ring stage (the
  // O-projection copies them in with one bulk copy per sequence).
  int S = std::max(1, n_sm / (B * Hkv));
  S = std::min(S, std::max(1, max_ctx / 16));
  S = std::min(S, STAGE_UNIT / (B * part_stride(D) * 4));
  if (S < 1) return MK_ERR_UNSUPPORTED;
  const int n_items = B * Hkv * S;

  std::vector<std::vector<Instr>> qs(n_sm);
  std::vector<double> bytes(n_sm, 0.0);
  auto mk = [](uint8_t op, int layer) {
    Instr I;
    std::memset(&I, 0, sizeof I);
    I.op = op;
    I.layer = (uint16_t)layer;
    I.wait_ctr = NO_CTR;
    I.sig_ctr = NO_CTR;
    return I;
  };

  // MoE virtual FFN: shared-expert columns [0, Fs) then top_k routed slots
  // of expert_ffn columns each; dense: the ffn columns.
  const long Fs = moe ? d.shared_ffn : 0;
  const long Fv = moe ? Fs + (long)d.top_k * d.expert_ffn : d.ffn;

  int n_lm = 0;
  for (int l = 0; l < L; l++) {
    // ---- QKV rows: with at least one SM per kv head, every SM works inside
    // one group (so no SM runs two pieces); otherwise contiguous ranges.
    for (int i = 0; i < n_sm; i++) {
      long a, b;
      if (n_sm >= Hkv) {
        const int g = (int)((long)i * Hkv / n_sm);
        const long s0 = ((long)g * n_sm + Hkv - 1) / Hkv;   // first SM of group g
        const long s1 = ((long)(g + 1) * n_sm + Hkv - 1) / Hkv;
        const int m = (int)(s1 - s0), k = (int)(i - s0);
        a = (long)g * GR + cut(GR, m, k, 2);
        b = (long)g * GR + (k == m - 1 ? GR : cut(GR, m, k + 1, 2));
      } else {
        a = cut(R, n_sm, i, 2);
        b = (i == n_sm - 1) ? R : cut(R, n_sm, i + 1, 2);
      }
      bool first = true;
      while (a < b) {
        long g = a / GR;
        long e = std::min(std::min(b, (g + 1) * GR), a + MAX_ROWS);
        Instr I = mk(OP_QKV, l);
        I.g = (uint16_t)g;
        I.r0 = (uint32_t)a;
        I.r1 = (uint32_t)e;
        I.flags = first ? 0 : F_NORM_CACHED;
        if (l > 0) I.wait_ctr = cm.mlp(l - 1);
        // split MLP: the previous layer's down rows arrive as tagged words
        if (l > 0 && mlp_split(d)) I.flags |= F_TAG_WAIT;
        I.sig_ctr = cm.qkv(l, (int)g);
        qs[i].push_back(I);
        bytes[i] += (double)(e - a) * H * wb;
        first = false;
        a = e;
      }
    }
    // ---- attention items
    for (int k = 0; k < n_items; k++) {
      int sm = (int)((long)k * n_sm / n_items);
      int b = k / (Hkv * S), g = (k / S) % Hkv, s = k % S;
      Instr I = mk(OP_ATTN, l);
      I.b = (uint16_t)b;
      I.g = (uint16_t)g;
      I.r0 = (uint32_t)s;
      I.r1 = (uint32_t)S;
      I.wait_ctr = cm.qkv(l, g);
      I.sig_ctr = cm.attn(l, g);
      qs[sm].push_back(I);
      bytes[sm] += (double)max_ctx / S * D * 4;
    }
    // ---- O-projection: with at least one SM per query head every SM takes
    // rows of a single head; otherwise the (head, row) space is cut evenly.
    // (the batched variants' tensor-core O-projection takes 8-row tiles and
    // adds row pairs with 8-byte reductions: cut at multiples of 8 rows)
    const long OR = (long)Hq * H;
    const int oal = d.max_batch > 1 ? 8 : 1;
    for (int i = 0; i < n_sm; i++) {
      long a, b;
      if (n_sm >= Hq) {
        const int h = (int)((long)i * Hq / n_sm);
        const long s0 = ((long)h * n_sm + Hq - 1) / Hq;
        const long s1 = ((long)(h + 1) * n_sm + Hq - 1) / Hq;
        const int m = (int)(s1 - s0), k = (int)(i - s0);
        a = (long)h * H + cut(H, m, k, oal);
        b = (long)h * H + (k == m - 1 ? H : cut(H, m, k + 1, oal));
      } else {
        a = cut(OR, n_sm, i, oal);
        b = (i == n_sm - 1) ? OR : cut(OR, n_sm, i + 1, oal);
      }
      while (a < b) {
        long h = a / H;
        long e = std::min(b, (h + 1) * H);
        Instr I = mk(OP_OPROJ, l);
        I.g = (uint16_t)h;
        I.r0 = (uint32_t)(a - h * H);
        I.r1 = (uint32_t)(e - h * H);
        I.flags = h == 0 ? F_RESIDUAL : 0;
        I.wait_ctr = cm.attn(l, (int)(h / HPG));
        I.sig_ctr = cm.oproj(l);
        qs[i].push_back(I);
        bytes[i] += (double)(e - a) * D * wb;
        a = e;
      }
    }
    // ---- MoE router rows; aux of each router instruction = how many there
    // are in the layer (the last to arrive signals the counter for all)
    if (moe) {
      const long E = d.n_experts;
      std::vector<std::pair<int, size_t>> routers;
      for (int i = 0; i < n_sm; i++) {
        long a = cut(E, n_sm, i, 1), b = (i == n_sm - 1) ? E : cut(E, n_sm, i + 1, 1);
        while (a < b) {
          long e = std::min(b, a + MAX_ROWS);
          Instr I = mk(OP_ROUTER, l);
          I.r0 = (uint32_t)a;
          I.r1 = (uint32_t)e;
          I.wait_ctr = cm.oproj(l);
          I.sig_ctr = cm.router(l);
          qs[i].push_back(I);
          routers.push_back({i, qs[i].size() - 1});
          bytes[i] += (double)(e - a) * H * 2;
          a = e;
        }
      }
      for (auto& rp : routers) qs[rp.first][rp.second].aux = (uint32_t)routers.size();
    }
    // ---- split MLP (dense, batch 1): gate/up column slices, then down rows
    if (mlp_split(d) || mlp_split_batched(d)) {
      // batched: gate/up slices in whole 16-column k-tiles of h, down runs of
      // (row block, column chunk) units
      const bool bat = mlp_split_batched(d);
      const long F = d.ffn, cu = bat ? 16 : 1;
      for (int i = 0; i < n_sm; i++) {
        long a = cut(F / cu, n_sm, i, 1) * cu;
        long b = (i == n_sm - 1) ? F : cut(F / cu, n_sm, i + 1, 1) * cu;
        bool first = true;
        while (a < b) {
          const long e = std::min(b, a + MAX_COLS);
          Instr I = mk(OP_MLP_UP, l);
          I.r0 = (uint32_t)a;
          I.r1 = (uint32_t)e;
          I.flags = first ? 0 : F_NORM_CACHED;
          I.wait_ctr = cm.oproj(l);
          I.sig_ctr = cm.mlp_up(l);
          qs[i].push_back(I);
          bytes[i] += (double)(e - a) * H * 2 * wb;
          first = false;
          a = e;
        }
      }
      // batch 1: rows [r0, r1) of x_{2l+2}, one owner per row; batched: a
      // run [r0, r1) of chunk-major down units (r0 / NRB is the first chunk)
      const long NRB = H / BD_ROWS, NU = bat ? NRB * (F / BD_KC) : H;
      for (int i = 0; i < n_sm; i++) {
        long a = cut(NU, n_sm, i, 1);
        long b = (i == n_sm - 1) ? NU : cut(NU, n_sm, i + 1, 1);
        while (a < b) {
          long e = std::min(b, a + (bat ? (long)BD_MAX_UNITS : (long)MAX_DOWN_ROWS));
          if (bat) e = std::min(e, (a / NRB + 2) * NRB);  // at most two chunks of h
          Instr I = mk(OP_MLP_DOWN, l);
          I.r0 = (uint32_t)a;
          I.r1 = (uint32_t)e;
          // batch 1: its rows of x_{2l+2} leave as tagged words, polled by
          // their consumers, so the signal needs no release
          I.flags = bat ? 0 : F_RELAXED_SIG;
          I.wait_ctr = cm.mlp_up(l);
          I.sig_ctr = cm.mlp(l);
          qs[i].push_back(I);
          bytes[i] += bat ? (double)(e - a) * BD_ROWS * BD_KC * 2 : (double)(e - a) * F * wb;
          a = e;
        }
      }
      continue;
    }
    // ---- MLP column slices (dense FFN, or MoE shared + routed slots)
    std::vector<std::pair<int, size_t>> mlp_at;  // (sm, index in qs[sm])
    // MoE: every SM takes a slice of the shared columns first (their weights
    // stream while the router resolves), then a slice of the routed columns.
    std::vector<std::pair<long, long>> fsegs;
    if (moe) {
      if (Fs > 0) fsegs.push_back({0, Fs});
      fsegs.push_back({Fs, Fv});
    } else {
      fsegs.push_back({0, Fv});
    }
    for (int i = 0; i < n_sm; i++)
      for (auto& fs : fsegs) {
      const long span = fs.second - fs.first;
      long a = fs.first + cut(span, n_sm, i, 1);
      long b = fs.first + ((i == n_sm - 1) ? span : cut(span, n_sm, i + 1, 1));
      while (a < b) {
        long seg_end = Fv;
        int slot = -1;
        if (moe) {
          if (a < Fs) {
            seg_end = Fs;
          } else {
            slot = (int)((a - Fs) / d.expert_ffn);
            seg_end = Fs + (long)(slot + 1) * d.expert_ffn;
          }
        }
        long e = std::min(std::min(b, seg_end), a + MAX_COLS);
        Instr I = mk(OP_MLP, l);
        if (!moe) {
          I.r0 = (uint32_t)a;
          I.r1 = (uint32_t)e;
          I.wait_ctr = cm.oproj(l);
        } else if (slot < 0) {
          I.flags = F_SHARED;
          I.r0 = (uint32_t)a;
          I.r1 = (uint32_t)e;
          I.wait_ctr = cm.oproj(l);
        } else {
          long base = Fs + (long)slot * d.expert_ffn;
          I.g = (uint16_t)slot;
          I.r0 = (uint32_t)(a - base);
          I.r1 = (uint32_t)(e - base);
          I.wait_ctr = cm.router(l);
        }
        I.sig_ctr = cm.mlp(l);
        I.flags |= F_RESIDUAL;
        qs[i].push_back(I);
        mlp_at.push_back({i, qs[i].size() - 1});
        bytes[i] += (double)(e - a) * H * 6;
        a = e;
      }
      }
    // residual rows [k*H/n, (k+1)*H/n) go to MLP instruction k of this layer
    const int n_mlp = (int)mlp_at.size();
    for (int k = 0; k < n_mlp; k++) {
      Instr& I = qs[mlp_at[k].first][mlp_at[k].second];
      uint32_t rs0 = (uint32_t)cut(H, n_mlp, k, 1);
      uint32_t rs1 = (k == n_mlp - 1) ? (uint32_t)H : (uint32_t)cut(H, n_mlp, k + 1, 1);
      I.aux = rs0 | (rs1 << 16);
    }
  }
  // ---- LM head rows (+ argmax by the last arriver)
  for (int i = 0; i < n_sm; i++) {
    long a = cut(V, n_sm, i, 1), b = (i == n_sm - 1) ? V : cut(V, n_sm, i + 1, 1);
    if (a >= b) continue;
    Instr I = mk(OP_LMHEAD, L);
    I.r0 = (uint32_t)a;
    I.r1 = (uint32_t)b;
    I.wait_ctr = cm.mlp(L - 1);
    if (mlp_split(d)) I.flags |= F_TAG_WAIT;
    I.aux = (uint32_t)n_lm++;
    qs[i].push_back(I);
    bytes[i] += (double)(b - a) * H * wb;
  }

  finish_plan(qs, bytes, cm, hold_mask, S, n_lm, out);
  const double router_rows = moe ? (double)d.n_experts : 0.0;
  // weights read per step (int8: codes plus one fp32 scale per row; the
  // norm gains stay bf16)
  out.weight_bytes = (double)L * ((double)R * H * wb + (double)Hq * D * H * wb +
                                  router_rows * H * wb + (double)Fv * H * 3 * wb + 2.0 * H * 2) +
                     (double)V * H * wb + (double)H * 2;
  if (wb == 1) out.weight_bytes += 4.0 * ((double)L * ((double)R + 2.0 * H + 2.0 * Fv) + V);
  return MK_OK;
}

// Coverage check of a built plan: every output row / column / work item of
// every phase is produced by exactly one instruction, pieces respect the
// group / pair / size limits the kernel relies on, and every residual row is
// added exactly once per layer.
int plan_verify(const mk_model_desc& d, int B, const PlanOut& p) {
  if (wide_path(d)) return plan_verify_wide(d, B, p);
  const int L = d.n_layers, H = d.hidden, Hq = d.n_q_heads, Hkv = d.n_kv_heads;
  const int D = d.head_dim, HPG = Hq / Hkv, V = d.vocab, GR = (HPG + 2) * D;
  const bool moe = d.n_experts > 0;
  const long R = (long)Hkv * GR, Fs = moe ? d.shared_ffn : 0;
  const long Fv = moe ? Fs + (long)d.top_k * d.expert_ffn : d.ffn;
  const int S = p.splits;
  // one head's partials of every sequence fill at most the smallest ring stage
  if (S < 1 || (long)B * S * part_stride(D) * 4 > STAGE_UNIT) return 32;
  std::vector<uint8_t> qkv((size_t)L * R, 0), att((size_t)L * B * Hkv * S, 0);
  std::vector<uint8_t> op((size_t)L * Hq * H, 0), mlp((size_t)L * Fv, 0), res((size_t)L * H, 0);
  std::vector<uint8_t> rt((size_t)L * (moe ? d.n_experts : 1), 0), lm(V, 0), slot(p.n_lm, 0);
  // batched split MLP: down units (row block, column chunk)
  std::vector<uint8_t> dunit(mlp_split_batched(d) ? (size_t)L * (H / BD_ROWS) * (d.ffn / BD_KC) : 0, 0);
  auto mark = [](std::vector<uint8_t>& v, size_t i) {
    if (i >= v.size() || v[i]) return false;
    v[i] = 1;
    return true;
  };
  const CtrMap cm{Hkv, L};
  // signals per counter, and whether any signaller of it signals without
  // release (F_RELAXED_SIG): such a counter orders no data, so only waiters
  // that poll tagged inputs may use it
  std::vector<uint32_t> sig_count(p.n_ctr, 0);
  std::vector<uint8_t> silent(p.n_ctr, 0);
  for (const Instr& I : p.q) {
    if (I.op == OP_HALT || I.sig_ctr == NO_CTR) continue;
    if (I.sig_ctr >= (uint32_t)p.n_ctr) return 28;
    sig_count[I.sig_ctr]++;
    if (I.flags & F_RELAXED_SIG) silent[I.sig_ctr] = 1;
  }
  for (const Instr& I : p.q) {
    if (I.op == OP_HALT) continue;
    const bool tag_wait = (I.flags & F_TAG_WAIT) != 0;
    // only these consumers poll tagged inputs, and only in the split MLP
    if (tag_wait && !(mlp_split(d) && (I.op == OP_QKV || I.op == OP_LMHEAD))) return 29;
    if ((I.flags & F_RELAXED_SIG) && !(mlp_split(d) && I.op == OP_MLP_DOWN)) return 29;
    if (!tag_wait && I.wait_ctr != NO_CTR && I.wait_ctr < (uint32_t)p.n_ctr && silent[I.wait_ctr])
      return 30;
  }
  for (const Instr& I : p.q) {
    const int l = I.layer;
    switch (I.op) {
      case OP_HALT: break;
      case OP_QKV:
        if (l >= L || I.r0 >= I.r1 || I.r1 > R || I.r1 - I.r0 > (uint32_t)MAX_ROWS) return 1;
        if (I.r0 / GR != I.g || (I.r1 - 1) / GR != I.g || (I.r0 % 2) || (I.r1 % 2)) return 2;
        for (uint32_t r = I.r0; r < I.r1; r++)
          if (!mark(qkv, (size_t)l * R + r)) return 3;
        break;
      case OP_ATTN:
        if (l >= L || I.b >= B || I.g >= Hkv || (int)I.r1 != S || (int)I.r0 >= S) return 4;
        if (!mark(att, (((size_t)l * B + I.b) * Hkv + I.g) * S + I.r0)) return 5;
        break;
      case OP_OPROJ:
        if (l >= L || I.g >= Hq || I.r0 >= I.r1 || (int)I.r1 > H) return 6;
        if (((I.flags & F_RESIDUAL) != 0) != (I.g == 0)) return 7;
        for (uint32_t r = I.r0; r < I.r1; r++)
          if (!mark(op, ((size_t)l * Hq + I.g) * H + r)) return 8;
        break;
      case OP_ROUTER:
        if (!moe || l >= L || I.r0 >= I.r1 || (int)I.r1 > d.n_experts ||
            I.r1 - I.r0 > (uint32_t)MAX_ROWS)
          return 9;
        for (uint32_t r = I.r0; r < I.r1; r++)
          if (!mark(rt, (size_t)l * d.n_experts + r)) return 10;
        // the last router to arrive signals for all: aux = their number
        if (I.sig_ctr != cm.router(l) || I.aux == 0 || I.aux != sig_count[I.sig_ctr]) return 31;
        break;
      case OP_MLP: {
        if (l >= L || I.r0 >= I.r1 || I.r1 - I.r0 > (uint32_t)MAX_COLS) return 11;
        long base = 0, width = Fv;
        if (moe) {
          if (I.flags & F_SHARED) {
            width = Fs;
          } else {
            if (I.g >= d.top_k) return 12;
            base = Fs + (long)I.g * d.expert_ffn;
            width = d.expert_ffn;
          }
        }
        if ((long)I.r1 > width) return 13;
        for (uint32_t c = I.r0; c < I.r1; c++)
          if (!mark(mlp, (size_t)l * Fv + base + c)) return 14;
        uint32_t rs0 = I.aux & 0xFFFF, rs1 = I.aux >> 16;
        if (rs1 > (uint32_t)H || rs0 > rs1) return 15;
        for (uint32_t r = rs0; r < rs1; r++)
          if (!mark(res, (size_t)l * H + r)) return 16;
        break;
      }
      case OP_MLP_UP:
        if (!(mlp_split(d) || mlp_split_batched(d)) || l >= L || I.r0 >= I.r1 ||
            I.r1 - I.r0 > (uint32_t)MAX_COLS || (long)I.r1 > Fv)
          return 23;
        if (mlp_split_batched(d) && ((I.r0 % 16) || (I.r1 % 16))) return 23;
        for (uint32_t c = I.r0; c < I.r1; c++)
          if (!mark(mlp, (size_t)l * Fv + c)) return 24;
        break;
      case OP_MLP_DOWN:
        if (!(mlp_split(d) || mlp_split_batched(d)) || l >= L || I.r0 >= I.r1) return 25;
        if (mlp_split_batched(d)) {
          // a run of chunk-major units spanning at most two chunks; the
          // chunk-0 units add the residual rows of their row blocks
          const uint32_t nrb = (uint32_t)(H / BD_ROWS), nu = nrb * (uint32_t)(d.ffn / BD_KC);
          if (I.r1 > nu || I.r1 - I.r0 > (uint32_t)BD_MAX_UNITS || (I.r1 - 1) / nrb > I.r0 / nrb + 1)
            return 25;
          for (uint32_t u = I.r0; u < I.r1; u++) {
            if (!mark(dunit, (size_t)l * nu + u)) return 26;
            if (u < nrb)
              for (uint32_t r = u * BD_ROWS; r < (u + 1) * BD_ROWS; r++)
                if (!mark(res, (size_t)l * H + r)) return 26;
          }
          break;
        }
        if ((int)I.r1 > H || I.r1 - I.r0 > (uint32_t)MAX_DOWN_ROWS) return 25;
        for (uint32_t r = I.r0; r < I.r1; r++)
          if (!mark(res, (size_t)l * H + r)) return 26;
        break;
      case OP_LMHEAD:
        if (I.r0 >= I.r1 || (int)I.r1 > V || (int)I.aux >= p.n_lm) return 17;
        if (!mark(slot, I.aux)) return 18;
        for (uint32_t r = I.r0; r < I.r1; r++)
          if (!mark(lm, r)) return 19;
        break;
      default:
        return 20;
    }
  }
  for (auto* v : {&qkv, &att, &op, &mlp, &res, &lm, &slot, &dunit})
    for (uint8_t x : *v)
      if (!x) return 21;
  if (moe)
    for (uint8_t x : rt)
      if (!x) return 22;
  return 0;
}

// In-order execution of every queue under the wait semantics: an
// instruction runs once its counter has received wait_cnt signals.  Two
// counts are kept per counter: every signal, which is what a consumer of
// tagged inputs (F_TAG_WAIT) waits for, and the release signals only (not
// F_RELAXED_SIG), the only ones that order the data a plain counter wait
// then reads -- a plain wait that needs a relaxed signal never completes
// here.  A deadlock is any state where no queue can advance before all
// reach HALT.
int plan_check(const Instr* q, int n_sm, int max_pc, int n_ctr) {
  if (!q || n_sm <= 0 || max_pc <= 0 || n_ctr <= 0) return MK_ERR_INVALID_ARG;
  std::vector<int> pc(n_sm, 0);
  std::vector<uint64_t> cnt(n_ctr, 0), dev(n_ctr, 0);
  for (;;) {
    bool progress = false, done = true;
    for (int s = 0; s < n_sm; s++) {
      for (;;) {
        if (pc[s] >= max_pc) break;
        const Instr& I = q[(size_t)s * max_pc + pc[s]];
        if (I.op == OP_HALT) break;
        const bool tag_wait = (I.flags & F_TAG_WAIT) != 0;
        if (I.wait_ctr != NO_CTR) {
          if (I.wait_ctr >= (uint32_t)n_ctr) return MK_ERR_SCHEDULE;
          if ((tag_wait ? cnt : dev)[I.wait_ctr] < I.wait_cnt) break;
        }
        if (I.sig_ctr != NO_CTR) {
          if (I.sig_ctr >= (uint32_t)n_ctr) return MK_ERR_SCHEDULE;
          cnt[I.sig_ctr]++;
          if (!(I.flags & F_RELAXED_SIG)) dev[I.sig_ctr]++;
        }
        pc[s]++;
        progress = true;
      }
      if (pc[s] < max_pc && q[(size_t)s * max_pc + pc[s]].op != OP_HALT) done = false;
    }
    if (done) return MK_OK;
    if (!progress) return MK_ERR_SCHEDULE;
  }
}

}  // namespace mk

extern "C" int mk_plan(const mk_model_desc* desc, int batch, int max_ctx, int n_sm,
                       mk_plan_stats* stats, mk_instr* out, size_t out_cap) {
  if (!desc) return MK_ERR_INVALID_ARG;
  mk::PlanOut p;
  int rc = mk::plan_build(*desc, batch, max_ctx, n_sm, p);
  if (rc) return rc;
  if (mk::plan_verify(*desc, batch, p)) return MK_ERR_SCHEDULE;
  if (mk::plan_check(p.q.data(), n_sm, p.max_pc, p.n_ctr)) return MK_ERR_SCHEDULE;
  if (stats) {
    stats->n_sm = n_sm;
    stats->max_pc = p.max_pc;
    stats->n_instr = p.n_instr;
    stats->n_counters = p.n_ctr;
    stats->attn_splits = p.splits;
    stats->n_lm = p.n_lm;
    stats->max_sm_bytes = p.max_sm_bytes;
    stats->mean_sm_bytes = p.mean_sm_bytes;
  }
  if (out) {
    if (out_cap < p.q.size()) return MK_ERR_INVALID_ARG;
    std::memcpy(out, p.q.data(), p.q.size() * sizeof(mk_instr));
  }
  return MK_OK;
}

extern "C" int mk_plan_check(const mk_instr* q, int n_sm, int max_pc, int n_counters) {
  return mk::plan_check(q, n_sm, max_pc, n_counters);
}
