// megakernel.cuh -- the persistent decode interpreter for sm_103a.
//
// One CTA per SM runs its queue of opcoded instructions in order ("Megakernels:
// Deleting the Kernel Boundary", section "One launch, one interpreter").
// The CTA has NCW consumer warps and one producer warp.  The producer walks
// the same queue ahead of the consumers and issues non-multicast TMA bulk
// copies (cp.async.bulk) of every instruction's weight rows -- and of the
// cached K/V rows of attention work items -- into a ring of shared-memory
// stages guarded by full/empty mbarriers.  Weight loads never wait on a
// counter, so the ring keeps HBM busy while the consumers wait for the
// activations of their next instruction; this is the GB300 form of the
// pages' paged shared memory and load/compute/store/finish overlap (section
// "Correctness without the free barrier", last paragraph, and the hook
// template of "One launch, one interpreter").
//
// Template parameters: HT hidden size, D head dim, HPG query heads per kv
// head, NB batch capacity of the compiled variant (rows b >= B are masked).
#pragma once
#include "attn_tc.cuh"
#include "mk_tc.cuh"
#include "mk_device.cuh"

namespace mk {

// The batched variants with 64-dim heads and 2 or 4 query heads per kv head
// run attention on the tensor cores over TMA-swizzled K / V tiles (when the
// cache is contiguous; a paged cache keeps the CUDA-core body).
template <int D, int HPG, int NB>
MK_HD constexpr bool attn_tc_path() {
  return NB > 1 && D == 64 && (HPG == 2 || HPG == 4);
}

template <int HT, int D, int HPG, int NB, int WB>
struct Ctx {
  float* xn;    // [NB][HT] normalised activation of the current instruction
  float* yrow;  // [NB][MAX_ROWS] row outputs / attention merge scratch
  float* hbuf;  // [NB][MAX_COLS] SiLU(gate)*up of an MLP slice
  float* mpart; // NB > 1: [NCW][MMA_FLUSH][NB] per-warp partial sums of the batched GEMV
  float* attn;  // [NB][D] reduced attention output of one head
  float* red;   // reduction scratch
  float* sc;    // int8 weights: row scales of the current O-proj / LM-head instruction [HT]
  int* tok;     // [NB]
  int* pos;     // [NB]
  int* topk;    // [NB][K] routed expert ids
  float* topw;  // [NB][K] routed expert weights
  int* flag;    // [0] bad launch input, [2] a tagged-input poll failed, [3] / [4] key of
                // the instruction whose counter was seen / whose wait failed
                // (both shared by the consumer warps; [1] belongs to the producer),
                // [5] a router's arrival count, [6] wide batch: this attention
                // item arrived last for its (sequence, kv head), [7] this LM-head
                // slice arrived last
  Ring ring;
  int tid, warp, lane;
  int pc;
  int step;         // step of this launch (0 .. n_steps - 1)
  uint32_t epoch;   // g.epoch + step: counter targets, tags, residual parity
  unsigned long long tw0, tw1;  // trace: wait start / end (thread 0)
  unsigned long long tm[2];     // trace: after the prologue phase, after the ring loop
  // wide batch: tensor-memory base, MMA-done mbarrier (shared address) and
  // the parity of its next phase
  uint32_t tmem, mma_bar, mma_par;
  MK_DEV void mark(const Globals& g, int k) {
    if (g.trace && tid == 0) tm[k] = gtimer();
  }
};

// The dependency wait of one instruction: thread 0 spins on the counter,
// then all consumer warps meet; false if the grid has failed.  Every op
// calls it exactly once, after issuing its dependency-free loads.
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool dep_wait(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Instr& I) {
  // the first lanes of n_pollers warps poll the counter, staggered (flag[3]:
  // key of the instruction whose counter was seen; flag[4]: key of a failed
  // wait).  A met counter means complete inputs; errors elsewhere in the
  // grid surface in this and the later bounded waits (no extra L2 round
  // trip).  F_TAG_WAIT: the op polls its tagged inputs itself.
  const int key = c.pc + 1;
  if (c.tid == 0 && g.trace) c.tw0 = gtimer();
  if (!(I.flags & F_TAG_WAIT) && I.wait_ctr != NO_CTR && c.lane == 0 && c.warp < g.n_pollers) {
    if (!poll_counter_shared(g, I.wait_ctr, c.epoch * I.wait_cnt,
                             (uint64_t)c.warp * g.poll_stagger_ns, c.flag + 3, key, c.pc, I.op))
      ((volatile int*)c.flag)[4] = key;
  }
  if (c.tid == 0) {
    c.flag[2] = 0;
    if (g.trace) c.tw1 = gtimer();
  }
  consumer_bar();
  return ((volatile int*)c.flag)[4] != key;
}

// Residual stream x_j, j in [1, 2L] (x_0 is the embedding row), held as
// g.kc partial copies that add up to x_j: an SM accumulates its atomics into
// copy (SM index mod kc), which spreads the contention on each L2 line over
// kc lines; readers sum the copies.
// The buffers alternate with the step's parity (epoch & 1): a step zeroes
// the other parity's copies for the next one.
MK_DEV float* xres(const Globals& g, uint32_t ep, int j, int b, int copy = 0) {
  return g.xbuf +
         ((((size_t)(ep & 1u) * 2 * g.L + (size_t)(j - 1)) * g.kc + copy) * g.B + b) * (size_t)g.H;
}

MK_DEV float* xres_mine(const Globals& g, uint32_t ep, int j, int b) {
  return xres(g, ep, j, b, (int)(blockIdx.x % (unsigned)g.kc));
}

// x_j[b][r], summed over the copies.
MK_DEV float xres_sum(const Globals& g, uint32_t ep, int j, int b, int r) {
  float v = 0.f;
  for (int c = 0; c < g.kc; c++) v += __ldcg(xres(g, ep, j, b, c) + r);
  return v;
}

// The weight / cache byte ranges an instruction streams, in ring order.
// The producer issues exactly these copies; the consumers consume exactly
// these stages.  Returns the number of segments (0..2).
template <int HT, int D, int WB, int NB>
MK_DEV int get_segs(const Globals& g, const Instr& I, const int* pos, const int* topk, Seg* s) {
  // WB bytes per weight: 2 (bf16) or 1 (int8 codes, dense batch-1 shapes only)
  constexpr uint32_t ROW = HT * WB;
  const uint32_t SBY = (uint32_t)g.stage_bytes;
  const uint32_t RPS = SBY / ROW;
  const LayerPtrs* Lp = g.layers + (I.op == OP_LMHEAD ? 0 : I.layer);
  const uint32_t n = I.r1 - I.r0;
  if constexpr (NB > 8) {
    // wide batch: K chunks of the instruction's rows (K-chunk-major packed
    // matrices, [K / 64][R8][64] with R8 = R rounded up to 8 rows) next to
    // the operand's chunks; QKV / gate-up / LM head take every chunk of
    // their normalised operand, a down instruction the chunks [b, g) of h
    if (I.op == OP_QKV || I.op == OP_MLP_UP || I.op == OP_MLP_DOWN || I.op == OP_LMHEAD) {
      const uint32_t ab = 2u * (uint32_t)g.Bp * 128u;
      const size_t abuf = (size_t)(HT / WIDE_KC) * ab;
      const unsigned char* w;
      const unsigned char* a;
      uint32_t R, r0, rows, k0 = 0, nk = HT / WIDE_KC;
      if (I.op == OP_QKV) {
        w = (const unsigned char*)Lp->wqkv;
        a = g.act;
        R = (uint32_t)(g.Hq + 2 * g.Hkv) * D;
        r0 = I.r0;
        rows = n;
      } else if (I.op == OP_MLP_UP) {
        w = (const unsigned char*)Lp->wgu;
        a = g.act + abuf;
        R = 2u * (uint32_t)g.F;
        r0 = 2u * I.r0;
        rows = 2u * n;
      } else if (I.op == OP_MLP_DOWN) {
        w = (const unsigned char*)Lp->wdT;
        a = (const unsigned char*)g.hglob;
        R = (uint32_t)g.H;
        r0 = I.r0;
        rows = n;
        k0 = I.b;
        nk = (uint32_t)I.g - I.b;
      } else {
        w = (const unsigned char*)g.lm_head;
        a = g.act + 2 * abuf;
        R = (uint32_t)g.V;
        r0 = I.r0;
        rows = n;
      }
      const uint32_t R8 = (R + 7u) / 8u * 8u, unit = (rows + 7u) / 8u * 8u * 128u;
      s[0] = {w + ((size_t)k0 * R8 + r0) * 128u, a + (size_t)k0 * ab, unit, nk, SBY / (unit + ab),
              seg_wide_tag(R8 * 128u, ab)};
      return 1;
    }
    if (I.op == OP_OPROJ) {
      // rows [r0, r1) of Wo for each of kv group I.g's query heads (one K
      // chunk per head, [Hq][H][64] packed, H rows apart), next to those
      // heads' merged attention outputs (the fourth operand buffer, one
      // chunk per query head)
      const uint32_t ab = 2u * (uint32_t)g.Bp * 128u;
      const uint32_t unit = (n + 7u) / 8u * 8u * 128u;
      const int hpg = g.Hq / g.Hkv;
      s[0] = {(const unsigned char*)Lp->wo + ((size_t)I.g * hpg * HT + I.r0) * 128u,
              g.act + (3 * (size_t)(HT / WIDE_KC) + (size_t)I.g * hpg) * ab, unit, (uint32_t)hpg,
              SBY / (unit + ab), seg_wide_tag((uint32_t)HT * 128u, ab)};
      return 1;
    }
    if (I.op == OP_NORM) return 0;
  }
  switch (I.op) {
    case OP_QKV:
      s[0] = {(const unsigned char*)Lp->wqkv + (size_t)I.r0 * ROW, nullptr, ROW, n, RPS, I.r0};
      return 1;
    case OP_OPROJ: {
      // rows of Wo; with staged partials (heads of 128+ dims), first head
      // I.g's split-KV partials of every sequence, copied in by the consumers
      // once attention is done (one stage)
      const Seg wo = {(const unsigned char*)Lp->wo + ((size_t)I.g * HT + I.r0) * D * WB, nullptr,
                      D * WB, n, SBY / (D * WB)};
      if constexpr (D >= 128) {
        if (g.part_staged) {
          const uint32_t pb = (uint32_t)(g.B * g.splits * part_stride(D) * 4);
          s[0] = {(const unsigned char*)g.part, nullptr, 16u, pb / 16u, SBY / 16u, SEG_CFILL};
          s[1] = wo;
          return 2;
        }
      }
      s[0] = wo;
      return 1;
    }
    case OP_ROUTER:
      s[0] = {(const unsigned char*)(Lp->router + (size_t)I.r0 * HT), nullptr, ROW, n, RPS, I.r0};
      return 1;
    case OP_MLP: {
      const uint16_t *gu, *dT;
      uint32_t row0;  // first gate/up row, the swizzle key of the packed tensor
      if (g.E == 0) {
        gu = Lp->wgu + (size_t)I.r0 * 2 * HT;
        dT = Lp->wdT + (size_t)I.r0 * HT;
        row0 = 2 * I.r0;
      } else if (I.flags & F_SHARED) {
        gu = Lp->sh_gu + (size_t)I.r0 * 2 * HT;
        dT = Lp->sh_dT + (size_t)I.r0 * HT;
        row0 = 2 * I.r0;
      } else {
        const size_t e = (size_t)topk[I.g];
        gu = Lp->ex_gu + (e * g.Fe + I.r0) * 2 * HT;
        dT = Lp->ex_dT + (e * g.Fe + I.r0) * HT;
        row0 = (uint32_t)(2 * (e * g.Fe + I.r0));
      }
      s[0] = {(const unsigned char*)gu, nullptr, ROW, 2 * n, RPS, row0};
      s[1] = {(const unsigned char*)dT, nullptr, ROW, n, RPS};
      return 2;
    }
    case OP_LMHEAD:
      s[0] = {(const unsigned char*)g.lm_head + (size_t)I.r0 * ROW, nullptr, ROW, n, RPS, I.r0};
      return 1;
    case OP_MLP_UP:
      s[0] = {(const unsigned char*)Lp->wgu + (size_t)I.r0 * 2 * ROW, nullptr, ROW, 2 * n, RPS,
              2 * I.r0};
      return 1;
    case OP_MLP_DOWN:
      if (g.bsplit) {
        // the run [r0, r1) of chunk-major weight units (BD_ROWS x BD_KC, 16 KB)
        const uint32_t unit = BD_ROWS * BD_KC * 2u;
        s[0] = {(const unsigned char*)Lp->wdT + (size_t)I.r0 * unit, nullptr, unit, n, SBY / unit};
        return 1;
      }
      // rows of the row-major [H][F] down projection
      s[0] = {(const unsigned char*)Lp->wdT + (size_t)I.r0 * g.F * WB, nullptr, (uint32_t)g.F * WB,
              n, SBY / ((uint32_t)g.F * WB)};
      return 1;
    case OP_ATTN: {
      // slice s of S over positions [0, P]: [s*C/S, (s+1)*C/S), C = P + 1.
      // Rows below P come from the cache through the ring; row P (written by
      // this step's QKV instructions) is read directly after the wait.
      const int P = pos[I.b];
      const long C = (long)P + 1;
      const int p0 = (int)(C * I.r0 / I.r1);
      const int p1 = (int)(C * (I.r0 + 1) / I.r1);
      const int pe = p1 < P ? p1 : P;
      const uint32_t cnt = pe > p0 ? (uint32_t)(pe - p0) : 0u;
      const size_t base = (((size_t)I.b * g.Hkv + I.g) * g.max_seq + (size_t)p0) * D;
      s[0] = {(const unsigned char*)(Lp->kc + base), (const unsigned char*)(Lp->vc + base), D * 2,
              cnt, (SBY / 2) / (D * 2)};
      return 1;
    }
    default:
      return 0;
  }
}

// Units of a segment in the stage that starts at unit u0, checked in the
// bounds build against the room the stage (or its half) has for them: a
// violation records MK_ERR_BOUNDS and the consumer reads none of them.
MK_DEV uint32_t stage_units(const Globals& g, const Seg& sg, uint32_t u0, uint32_t room, int pc,
                            int op) {
  const uint32_t n = min(sg.ups, sg.n - u0);
  return MK_IN(g, n * sg.unit <= room, pc, op) ? n : 0u;
}

// ---------------------------------------------------------------- norms ----
// xn[b][k] = x[b][k] * rsqrt(mean(x^2) + eps) * gain[k] for the residual
// x_j (j = 0: the embedding row of the token).  The gain slice of each
// thread is loaded before the dependency wait (norm_gain), the rest after
// it (norm_apply).  All consumer threads.
template <int HT, int NB>
struct NormGain {
  static constexpr int GROUPS = HT / 8;
  static constexpr int GPT = (GROUPS + NCT - 1) / NCT;
  static constexpr int KPT = (HT + NCT - 1) / NCT;  // batched: columns tid + q * NCT
  uint4 w[NB == 1 ? GPT : 1];       // batch 1: 8 packed bf16 gains per 8-column group
  uint16_t gw[NB == 1 ? 1 : KPT];   // batched: this thread's columns' bf16 gains (widened
                                    // at use, so the loads do not stall the wait)
};

template <int HT, int NB>
MK_DEV void norm_gain(NormGain<HT, NB>& ng, const uint16_t* gain, int tid) {
  if constexpr (NB == 1) {
#pragma unroll
    for (int q = 0; q < NormGain<HT, NB>::GPT; q++) {
      const int gi = tid + q * NCT;
      if (gi < NormGain<HT, NB>::GROUPS) ng.w[q] = __ldg((const uint4*)gain + gi);
    }
  } else {
#pragma unroll
    for (int q = 0; q < NormGain<HT, NB>::KPT; q++) {
      const int k = tid + q * NCT;
      ng.gw[q] = k < HT ? __ldg(gain + k) : (uint16_t)0;
    }
  }
}

// RMSNorm for the batched variants (NB = 8), straight into the tensor-core
// A-fragment layout the batched GEMV reads.  Pass 1: thread t takes columns
// k = t + q*NCT of all 8 sequences and stores each column k-major (32 bytes;
// adjacent lanes write adjacent columns, so the stores do not conflict),
// summing squares on the way.  Pass 2 scales column k by gain[k] / rms(x_b).
// Pass 3 turns every 16-column k-tile (512 bytes, k-major) into its 32 lanes'
// fragments in place: lane 4g + t holds bf16 hi / lo of sequence g at
// columns 2t, 2t+1 and 2t+8, 2t+9.
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool norm_apply_batched(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, int j,
                               const NormGain<HT, NB>& ng) {
  static_assert(NB == 8, "k-tile blocks of 16 columns x 8 sequences");
  constexpr int KPT = (HT + NCT - 1) / NCT;  // columns per thread
  // every load of the pass in flight at once: under a streaming ring each L2
  // round trip costs microseconds, so the pass takes one
  constexpr int CH = KPT;
  float ss[NB];
#pragma unroll
  for (int b = 0; b < NB; b++) ss[b] = 0.f;
  // the per-sequence source rows (and the case) are fixed for the whole pass,
  // so the column loop below is a straight run of independent loads
  const bool emb = j == 0;
  const float* xb[NB];
  int tk[NB];
#pragma unroll
  for (int b = 0; b < NB; b++) {
    const bool live = b < g.B;
    tk[b] = live ? c.tok[b] : 0;
    xb[b] = (!emb && live) ? xres(g, c.epoch, j, b, 0) : nullptr;
  }
#pragma unroll
  for (int q0 = 0; q0 < KPT; q0 += CH) {
    float v[CH][NB];
#pragma unroll
    for (int u = 0; u < CH; u++) {
      const int k = c.tid + (q0 + u) * NCT;
      const bool kin = q0 + u < KPT && k < HT;
#pragma unroll
      for (int b = 0; b < NB; b++) {
        float x = 0.f;
        if (kin && b < g.B) {
          if (emb)  // embedding rows are chunk-swizzled by token id
            x = bf1(__ldg(g.embed + (size_t)tk[b] * HT + ((((k >> 3) ^ (tk[b] & 7)) << 3) | (k & 7))));
          else
            x = __ldcg(xb[b] + k);
        }
        v[u][b] = x;
      }
    }
    if (g.kc > 1 && !emb) {  // further partial copies of the residual vector
      for (int cp = 1; cp < g.kc; cp++)
#pragma unroll
        for (int u = 0; u < CH; u++) {
          const int k = c.tid + (q0 + u) * NCT;
#pragma unroll
          for (int b = 0; b < NB; b++)
            if (q0 + u < KPT && k < HT && b < g.B) v[u][b] += __ldcg(xres(g, c.epoch, j, b, cp) + k);
        }
    }
#pragma unroll
    for (int u = 0; u < CH; u++) {
      const int k = c.tid + (q0 + u) * NCT;
      if (q0 + u < KPT && k < HT) {
        st_shared_f4(c.xn + (size_t)k * NB, v[u][0], v[u][1], v[u][2], v[u][3]);
        st_shared_f4(c.xn + (size_t)k * NB + 4, v[u][4], v[u][5], v[u][6], v[u][7]);
#pragma unroll
        for (int b = 0; b < NB; b++) ss[b] = fmaf(v[u][b], v[u][b], ss[b]);
      }
    }
  }
  float gw[KPT];  // loaded before the dependency wait
#pragma unroll
  for (int q = 0; q < KPT; q++) gw[q] = bf1(ng.gw[q]);
#pragma unroll
  for (int b = 0; b < NB; b++) {
    const float t = warp_sum(ss[b]);
    if (c.lane == 0) c.red[c.warp * NB + b] = t;
  }
  consumer_bar();
  float rs[NB];
#pragma unroll
  for (int b = 0; b < NB; b++) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < NCW; w++) t += c.red[w * NB + b];
    rs[b] = rsqrtf(t / (float)HT + g.eps);
  }
#pragma unroll
  for (int q = 0; q < KPT; q++) {
    const int k = c.tid + q * NCT;
    if (k < HT) {
      float4* o = (float4*)(c.xn + (size_t)k * NB);
      float4 a0 = o[0], a1 = o[1];
      a0.x *= rs[0] * gw[q]; a0.y *= rs[1] * gw[q]; a0.z *= rs[2] * gw[q]; a0.w *= rs[3] * gw[q];
      a1.x *= rs[4] * gw[q]; a1.y *= rs[5] * gw[q]; a1.z *= rs[6] * gw[q]; a1.w *= rs[7] * gw[q];
      o[0] = a0;
      o[1] = a1;
    }
  }
  consumer_bar();
  const int gq = c.lane >> 2, tq = c.lane & 3;
  for (int kt = c.warp; kt < HT / 16; kt += NCW) {
    const float* blk = c.xn + (size_t)kt * 16 * NB;
    const float v0 = blk[(2 * tq) * NB + gq], v1 = blk[(2 * tq + 1) * NB + gq];
    const float v2 = blk[(2 * tq + 8) * NB + gq], v3 = blk[(2 * tq + 9) * NB + gq];
    uint4 f;
    split2(v0, v1, f.x, f.y);
    split2(v2, v3, f.z, f.w);
    __syncwarp();
    ((uint4*)c.xn)[(size_t)kt * 32 + c.lane] = f;
  }
  consumer_bar();
  return true;
}

template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool norm_apply(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, int j,
                       const NormGain<HT, NB>& ng) {
  if constexpr (NB > 1) {
    return norm_apply_batched(c, g, j, ng);
  } else {
  constexpr int GROUPS = NormGain<HT, NB>::GROUPS, GPT = NormGain<HT, NB>::GPT;
  bool ok = true;
  // bounds build: the residual vector must lie inside its buffer, else the
  // instruction fails (and reads x_1 meanwhile, which does)
  if (j > 0 && !MK_IN(g,
                      (g.xtag && (j & 1) == 0)
                          ? (size_t)(j / 2) * g.B * HT <= g.n_xt
                          : (size_t)(xres(g, c.epoch, j, g.B - 1, g.kc - 1) - g.xbuf) + HT <= g.n_xbuf,
                      c.pc, -1)) {
    ok = false;
    j = 1;
  }
  // split MLP: x_{2l+2} (j even, j > 0) arrives as tagged words from the
  // down rows' owners; each thread polls its own 8-element groups
  const bool tagged = g.xtag && j > 0 && (j & 1) == 0;
  if constexpr (NB == 1) {
    if (tagged) {  // this thread's groups, polled together straight into xn
      uint32_t valid = 0;
#pragma unroll
      for (int q = 0; q < GPT; q++)
        if (c.tid + q * NCT < GROUPS) valid |= 1u << q;
      ok = ok && poll_tag_groups_to<GPT, 4>(g, g.xt + (size_t)(j / 2 - 1) * HT + 8 * c.tid,
                                      (size_t)NCT * 8, valid, c.epoch, c.xn + 8 * c.tid, NCT * 8,
                                      c.pc, OP_QKV);
    }
  }
  float ss[NB];
#pragma unroll
  for (int b = 0; b < NB; b++) ss[b] = 0.f;
#pragma unroll
  for (int q = 0; q < GPT; q++) {
    const int gi = c.tid + q * NCT;
    if (gi >= GROUPS) continue;
    // every sequence's loads of this group first, then the shared-memory
    // stores: the stores may alias (as far as the compiler can tell) and
    // would otherwise hold each next load back by a whole round trip
    float v[NB][8];
#pragma unroll
    for (int b = 0; b < NB; b++) {
      if (b < g.B) {
        if (j == 0) {
          // embedding rows are chunk-swizzled by token id
          const uint4 w =
              __ldg((const uint4*)(g.embed + (size_t)c.tok[b] * HT) + (gi ^ (c.tok[b] & 7)));
          unpack8(w, v[b]);
        } else if (tagged) {  // polled into xn above (batch 1 only: the split MLP)
          const float4* p = (const float4*)(c.xn + (size_t)b * HT) + 2 * gi;
          const float4 a0 = p[0], a1 = p[1];
          v[b][0] = a0.x; v[b][1] = a0.y; v[b][2] = a0.z; v[b][3] = a0.w;
          v[b][4] = a1.x; v[b][5] = a1.y; v[b][6] = a1.z; v[b][7] = a1.w;
        } else if (g.kc == 1) {
          const float4* p = (const float4*)xres(g, c.epoch, j, b, 0) + 2 * gi;
          const float4 a0 = __ldcg(p), a1 = __ldcg(p + 1);
          v[b][0] = a0.x; v[b][1] = a0.y; v[b][2] = a0.z; v[b][3] = a0.w;
          v[b][4] = a1.x; v[b][5] = a1.y; v[b][6] = a1.z; v[b][7] = a1.w;
        } else {
#pragma unroll
          for (int k = 0; k < 8; k++) v[b][k] = 0.f;
          for (int cp = 0; cp < g.kc; cp++) {
            const float4* p = (const float4*)xres(g, c.epoch, j, b, cp) + 2 * gi;
            const float4 a0 = __ldcg(p), a1 = __ldcg(p + 1);
            v[b][0] += a0.x; v[b][1] += a0.y; v[b][2] += a0.z; v[b][3] += a0.w;
            v[b][4] += a1.x; v[b][5] += a1.y; v[b][6] += a1.z; v[b][7] += a1.w;
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < 8; k++) v[b][k] = 0.f;
      }
    }
    {
      float4* o = (float4*)c.xn + 2 * gi;
      o[0] = make_float4(v[0][0], v[0][1], v[0][2], v[0][3]);
      o[1] = make_float4(v[0][4], v[0][5], v[0][6], v[0][7]);
    }
#pragma unroll
    for (int b = 0; b < NB; b++)
#pragma unroll
      for (int k = 0; k < 8; k++) ss[b] = fmaf(v[b][k], v[b][k], ss[b]);
  }
#pragma unroll
  for (int b = 0; b < NB; b++) {
    const float t = warp_sum(ss[b]);
    if (c.lane == 0) c.red[c.warp * NB + b] = t;
  }
  if (!ok) c.flag[2] = 1;  // read by every consumer thread after the barrier
  consumer_bar();
  if (c.flag[2]) return false;
  float rs[NB];
#pragma unroll
  for (int b = 0; b < NB; b++) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < NCW; w++) t += c.red[w * NB + b];
    rs[b] = rsqrtf(t / (float)HT + g.eps);
  }
#pragma unroll
  for (int q = 0; q < GPT; q++) {
    const int gi = c.tid + q * NCT;
    if (gi >= GROUPS) continue;
    float gw[8];
    unpack8(ng.w[q], gw);
    {
      float4* o = (float4*)c.xn + 2 * gi;
      float4 a0 = o[0], a1 = o[1];
      a0.x *= rs[0] * gw[0]; a0.y *= rs[0] * gw[1]; a0.z *= rs[0] * gw[2]; a0.w *= rs[0] * gw[3];
      a1.x *= rs[0] * gw[4]; a1.y *= rs[0] * gw[5]; a1.z *= rs[0] * gw[6]; a1.w *= rs[0] * gw[7];
      o[0] = a0;
      o[1] = a1;
    }
  }
  consumer_bar();
  return true;
  }
}

// ----------------------------------------------------------------- GEMV ----
// Lane l of a warp owns the columns of its 16-byte chunks of a row: bf16
// rows {it*256 + l*8 + k}, int8 rows {it*512 + l*16 + k}; for NB == 1 its
// slice of xn lives in registers.
template <int HT, int WB>
MK_DEV void load_xr(const float* xn, int lane, float (&xr)[HT / 32]) {
  if constexpr (WB == 1) {
#pragma unroll
    for (int it = 0; it < HT / 512; it++) {
      const float4* p = (const float4*)(xn + it * 512 + lane * 16);
#pragma unroll
      for (int q = 0; q < 4; q++) {
        const float4 a = p[q];
        xr[it * 16 + 4 * q] = a.x; xr[it * 16 + 4 * q + 1] = a.y;
        xr[it * 16 + 4 * q + 2] = a.z; xr[it * 16 + 4 * q + 3] = a.w;
      }
    }
  } else {
#pragma unroll
    for (int it = 0; it < HT / 256; it++) {
      const float4* p = (const float4*)(xn + it * 256 + lane * 8);
      const float4 a = p[0], b = p[1];
      xr[it * 8 + 0] = a.x; xr[it * 8 + 1] = a.y; xr[it * 8 + 2] = a.z; xr[it * 8 + 3] = a.w;
      xr[it * 8 + 4] = b.x; xr[it * 8 + 5] = b.y; xr[it * 8 + 6] = b.z; xr[it * 8 + 7] = b.w;
    }
  }
}

// Partial dot of one row (in shared memory) with the activation(s); the
// caller reduces across the warp.  int8 rows give the dot with the codes
// (the caller applies the row's scale).
template <int HT, int NB, int WB>
MK_DEV void row_dot(const unsigned char* row, const float (&xr)[HT / 32], const float* xn,
                    int lane, int key, float (&acc)[NB]) {
  // the row is chunk-swizzled: this lane's chunk it*32 + lane sits at slot
  // it*32 + (lane ^ key), key = row index & 7
  const uint4* w4 = (const uint4*)row;
  const int sl = lane ^ key;
  static_assert(NB == 1, "batched variants use the tensor-core GEMV");
  if constexpr (WB == 1) {
    // eight chains (element e of a word pair), two per packed FMA
    float2 a[4];
#pragma unroll
    for (int k = 0; k < 4; k++) a[k] = make_float2(0.f, 0.f);
#pragma unroll
    for (int it = 0; it < HT / 512; it++) {
      const uint4 w = w4[it * 32 + sl];
      const float* x = xr + it * 16;
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int q = 0; q < 4; q++)
#pragma unroll
        for (int e = 0; e < 4; e += 2)
          a[((4 * q + e) & 7) >> 1] = ffma2(i8_pair(ws[q], e), make_float2(x[4 * q + e], x[4 * q + e + 1]),
                                           a[((4 * q + e) & 7) >> 1]);
    }
    acc[0] = ((a[0].x + a[0].y) + (a[1].x + a[1].y)) + ((a[2].x + a[2].y) + (a[3].x + a[3].y));
  } else {
    // eight independent chains (one per element of a 16-byte chunk): the
    // dependent-FMA depth is HT/256 instead of HT/64
    float a[8];
#pragma unroll
    for (int k = 0; k < 8; k++) a[k] = 0.f;
#pragma unroll
    for (int it = 0; it < HT / 256; it++) {
      const uint4 w = w4[it * 32 + sl];
      const float* x = xr + it * 8;
      a[0] = fmaf(bf_lo(w.x), x[0], a[0]); a[1] = fmaf(bf_hi(w.x), x[1], a[1]);
      a[2] = fmaf(bf_lo(w.y), x[2], a[2]); a[3] = fmaf(bf_hi(w.y), x[3], a[3]);
      a[4] = fmaf(bf_lo(w.z), x[4], a[4]); a[5] = fmaf(bf_hi(w.z), x[5], a[5]);
      a[6] = fmaf(bf_lo(w.w), x[6], a[6]); a[7] = fmaf(bf_hi(w.w), x[7], a[7]);
    }
    acc[0] = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
  }
}


// Stream the rows of one segment through the ring; warp w computes rows
// w, w + NCW, ... of each stage and hands (row index, per-sequence dot) to
// fn on every lane.  Returns false if a wait gave up.
template <int HT, int D, int HPG, int NB, int WB, class Fn>
MK_DEV bool gemv_rows(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Seg& s,
                      const float (&xr)[HT / 32], Fn&& fn) {
  float pend = 0.f;  // NB == 1: this lane's partial of the row not yet reduced
  int prow = -1;
  for (uint32_t u0 = 0; u0 < s.n; u0 += s.ups) {
    const uint32_t n = stage_units(g, s, u0, (uint32_t)g.stage_bytes, c.pc, -1);
    if (!c.ring.acquire(g)) return false;
    const unsigned char* st = c.ring.stage_ptr();
    // segment row u0 + r goes to warp (u0 + r) mod NCW, so a short segment
    // spreads its rows over all warps rather than over one stage's worth
    for (uint32_t r = (uint32_t)(c.warp + NCW - (int)(u0 % NCW)) % NCW; r < n; r += NCW) {
      float acc[NB];
      if constexpr (NB == 1) {
        // the previous row's cross-lane sum is issued in the same block as
        // this row's loads and FMAs, so its shuffle latency hides behind them
        float prev[1] = {warp_sum(pend)};
        row_dot<HT, NB, WB>(st + (size_t)r * HT * WB, xr, c.xn, c.lane, (int)((s.row0 + u0 + r) & 7u),
                        acc);
        if (prow >= 0) fn((uint32_t)prow, prev);
        pend = acc[0];
        prow = (int)(u0 + r);
      } else {
        row_dot<HT, NB, WB>(st + (size_t)r * HT * WB, xr, c.xn, c.lane, (int)((s.row0 + u0 + r) & 7u),
                        acc);
#pragma unroll
        for (int b = 0; b < NB; b++) acc[b] = warp_sum(acc[b]);
        fn(u0 + r, acc);
      }
    }
    c.ring.release(c.lane);
  }
  if constexpr (NB == 1) {
    if (prow >= 0) {
      float last[1] = {warp_sum(pend)};
      fn((uint32_t)prow, last);
    }
  }
  return true;
}

// Batched GEMV on the tensor cores (NB > 1): y[b][row] = sum_k W[row][k] x[b][k]
// with mma.sync m16n8k16 (bf16 in, f32 accumulate), A = the activations and
// B = 8 weight rows.  A's rows 0..7 hold bf16(x[b]) and rows 8..15 the bf16 of
// the remainder x[b] - bf16(x[b]); the two halves' products are added, so the
// activation keeps about 16 mantissa bits; the A fragments are built once per
// normalisation, in shared memory (norm_apply).  The k range is split over the
// consumer warps: warp w reads only its k-tile pairs of every ring stage, 8
// rows at a time with ldmatrix (rows are chunk-swizzled, so the 8 row reads
// hit 8 bank groups), with the matching A fragments.  Per-warp
// partial sums meet in shared memory every MMA_FLUSH rows, where fe(row, b,
// y) receives each output once.  Every warp runs the same loop and barriers;
// a warp whose ring wait gave up stops touching the ring (it neither reads
// nor releases stages) and the failure is broadcast, so all return alike.
template <int HT, int D, int HPG, int NB, int WB, class Fe>
MK_DEV bool gemv_rows_mma(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Seg& s, Fe&& fe) {
  static_assert(NB > 1 && NB <= 8, "one m16n8k16 A tile holds up to 8 sequences");
  static_assert(NCT % NB == 0 && (NB & (NB - 1)) == 0, "a thread's outputs share one sequence");
  static_assert(MAX_STAGE_BYTES / (HT * 2) <= MMA_FLUSH, "a stage's rows fit one flush window");
  static_assert(NB == 8, "the fragment layout packs 8 sequences per k-tile");
  constexpr int NPAIR = HT / 32;  // pairs of 16-column k-tiles
  constexpr int PPW = (NPAIR + NCW - 1) / NCW;
  const int p0 = c.warp * NPAIR / NCW, np = (c.warp + 1) * NPAIR / NCW - p0;
  const int gq = c.lane >> 2, tq = c.lane & 3;
  // A fragments of k-tile kt: ((uint4*)xn)[kt * 32 + lane], built by norm_apply
  const uint4* af = (const uint4*)c.xn + c.lane;
  float* part = c.mpart;
  bool bad = false;
  uint32_t prow0 = 0, pending = 0;  // rows held in part since the last flush
  const uint32_t li = (uint32_t)c.lane & 7u, lm = (uint32_t)c.lane >> 3;
  for (uint32_t u0 = 0; u0 < s.n; u0 += s.ups) {
    const uint32_t n = stage_units(g, s, u0, (uint32_t)g.stage_bytes, c.pc, -1);
    if (!bad && !c.ring.acquire(g)) bad = true;
    if (!bad) {
      const uint32_t sbase = smem_u32(c.ring.stage_ptr());
      for (uint32_t nt = 0; nt < n; nt += 8) {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t rr = nt + li < n ? nt + li : nt;  // rows past the stage repeat row nt
        const uint32_t key = (s.row0 + u0 + rr) & 7u;
        const uint32_t rowaddr = sbase + rr * (uint32_t)(HT * 2);
#pragma unroll
        for (int pp = 0; pp < PPW; pp++) {
          if (pp < np) {
            const uint32_t ch = (uint32_t)(p0 + pp) * 4u + lm;  // 16-byte chunk of this lane's matrix
            uint32_t b0, b1, b2, b3;
            ldsm_x4(rowaddr + ((ch ^ key) << 4), b0, b1, b2, b3);
            const uint4 fa = af[(size_t)(p0 + pp) * 64], fb = af[(size_t)(p0 + pp) * 64 + 32];
            const uint32_t a0[4] = {fa.x, fa.y, fa.z, fa.w}, a1[4] = {fb.x, fb.y, fb.z, fb.w};
            mma_16816(d, a0, b0, b1);
            mma_16816(d, a1, b2, b3);
          }
        }
        // d[0], d[1]: hi products of sequence gq, rows nt + 2tq, +1; d[2], d[3]: lo
        const uint32_t r = nt + 2u * (uint32_t)tq;
        float* pw = part + ((size_t)c.warp * MMA_FLUSH + (u0 + r - prow0)) * NB + gq;
        if (gq < NB && r < n) pw[0] = d[0] + d[2];
        if (gq < NB && r + 1 < n) pw[NB] = d[1] + d[3];
      }
      c.ring.release(c.lane);
    }
    pending += n;
    if (u0 + s.ups >= s.n || pending + s.ups > (uint32_t)MMA_FLUSH) {
      consumer_bar();
      for (int it = c.tid; it < (int)pending * NB; it += NCT) {
        const int r = it / NB, b = it % NB;
        float y = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; w++) y += part[((size_t)w * MMA_FLUSH + r) * NB + b];
        if (b < g.B) fe(prow0 + (uint32_t)r, b, y);
      }
      consumer_bar();
      prow0 += pending;
      pending = 0;
    }
  }
  if (bad) c.flag[2] = 1;
  consumer_bar();
  return c.flag[2] == 0;
}

// The GEMV of the row-dotted matrices: fe(row, b, y) is called exactly once
// per output.  Batch 1 runs on the FP32 pipes (lane 0 of the row's warp
// calls fe); batched variants run on the tensor cores.
template <int HT, int D, int HPG, int NB, int WB, class Fe>
MK_DEV bool gemv(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Seg& s,
                 const float (&xr)[HT / 32], Fe&& fe) {
  if constexpr (NB > 1) {
    return gemv_rows_mma(c, g, s, fe);
  } else {
    const int lane = c.lane;
    return gemv_rows(c, g, s, xr, [&](uint32_t r, float(&acc)[NB]) {
      if (lane == 0) fe(r, 0, acc[0]);
    });
  }
}

}  // namespace mk

namespace mk {

// ------------------------------------------------- OP_QKV (RMS+QKV+RoPE) ----
// Rows [r0, r1) of the layer's packed QKV matrix, all inside kv head I.g's
// group [q heads of the group][k][v]; inside a head, packed rows 2t and 2t+1
// hold head dims t and t + D/2, so each rotary pair is produced by one SM.
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool op_qkv(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Instr& I) {
  static_assert(MAX_ROWS <= 2 * NCT, "one rotary pair per thread");
  const LayerPtrs& Lp = g.layers[I.layer];
  const bool cached = (I.flags & F_NORM_CACHED) != 0;
  NormGain<HT, NB> ng;
  if (!cached) norm_gain(ng, Lp.attn_norm, c.tid);
  // this thread's rotary pair: head slot hs, dims (t, t + D/2), and its
  // cos/sin at P -- none of it depends on the wait
  constexpr int GR = (HPG + 2) * D;
  const uint32_t n = I.r1 - I.r0;
  const uint32_t i = 2u * (uint32_t)c.tid;
  int hs = 0, t = 0;
  float2 cs[NB];
  float2 rsc = make_float2(1.f, 1.f);  // int8: the pair's row scales
  if (i < n) {
    if constexpr (WB == 1) rsc = *(const float2*)(Lp.sqkv + I.r0 + i);  // r0, i even
    const int lr = (int)(I.r0 + i) - (int)I.g * GR;
    hs = lr / D;
    t = (lr % D) >> 1;
    if (hs <= HPG)
#pragma unroll
      for (int b = 0; b < NB; b++)
        if (b < g.B) cs[b] = ((const float2*)g.rope)[(size_t)c.pos[b] * (D / 2) + t];
  }
  if (!dep_wait(c, g, I)) return false;
  if (!cached && !norm_apply(c, g, 2 * I.layer, ng)) return false;
  c.mark(g, 0);
  float xr[HT / 32];
  if constexpr (NB == 1) load_xr<HT, WB>(c.xn, c.lane, xr);
  Seg s[2];
  get_segs<HT, D, WB, NB>(g, I, c.pos, c.topk, s);
  float* yrow = c.yrow;
  const int lane = c.lane;
  gemv(c, g, s[0], xr, [&](uint32_t r, int b, float y) { yrow[b * MAX_ROWS + r] = y; });
  c.mark(g, 1);
  consumer_bar();
  if (i < n) {
#pragma unroll
    for (int b = 0; b < NB; b++) {
      if (b >= g.B) break;
      float y0 = yrow[b * MAX_ROWS + i], y1 = yrow[b * MAX_ROWS + i + 1];
      if constexpr (WB == 1) {
        y0 *= rsc.x;
        y1 *= rsc.y;
      }
      const int P = c.pos[b];
      if (hs <= HPG) {  // q heads and k: rotate (t, t + D/2) by P * theta^(-2t/D)
        const float a = y0 * cs[b].x - y1 * cs[b].y;
        const float bb = y0 * cs[b].y + y1 * cs[b].x;
        y0 = a;
        y1 = bb;
      }
      if (hs < HPG) {
        const size_t qo = (((size_t)I.layer * g.B + b) * g.Hq + (size_t)I.g * HPG + hs) * D;
        if (MK_IN(g, qo + D <= g.n_q, c.pc, I.op)) {
          float* q = g.qbuf + qo;
          q[t] = y0;
          q[t + D / 2] = y1;
        }
      } else {
        const long long off = kv_row(g, b, I.g, P);
        if (off < 0) {
          set_err(g, MK_ERR_INVALID_ARG, c.pc, I.op);  // a block outside the pool
        } else if (MK_IN(g, (size_t)off + D <= g.kv_elems, c.pc, I.op)) {
          uint16_t* row = (hs == HPG ? Lp.kc : Lp.vc) + off;
          row[t] = to_bf16(y0);
          row[t + D / 2] = to_bf16(y1);
        }
      }
    }
  }
  consumer_bar();
  return true;
}

// ------------------------------------------ OP_ATTN (split-KV partial) ----
// Work item (b, kv head g, slice s of S): for the HPG query heads of the
// group, the partial softmax state over positions [s*C/S, (s+1)*C/S) of
// [0, P]: running max m, sum l of 2^(score - m) and o = sum 2^(score - m) v,
// with scores in log2 units (q pre-scaled by log2(e)/sqrt(D)).  Rows stream
// through the ring K-half / V-half per stage; every slot of LPR lanes handles
// one position at a time with an online-softmax update, then slots, warps
// and finally the CTA merge their states.

template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool attn_merge_wide(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Instr& I);

// The end of an attention item: every warp has put its per-head state (o,
// m, l) into sc = yrow [NCW][HPG][D + 2]; merge the warps and write the
// item's partial record (o, m, l of each head) for the O-projection (or, wide
// batch, for the last arriving item's merge).
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool attn_cta_merge(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Instr& I) {
  const int b = I.b;
  const float* sc = c.yrow;
  consumer_bar();
  for (int t = c.tid; t < HPG * D; t += NCT) {
    const int h = t / D, dim = t % D;
    float M = NEG_BIG;
#pragma unroll
    for (int w = 0; w < NCW; w++) M = fmaxf(M, sc[(w * HPG + h) * (D + 2) + D]);
    float Ls = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < NCW; w++) {
      const float* p = sc + (w * HPG + h) * (D + 2);
      const float f = exp2f(p[D] - M);
      Ls = fmaf(p[D + 1], f, Ls);
      O = fmaf(p[dim], f, O);
    }
    if constexpr (NB > 8) {
      if (g.splits == 1) {
        // wide batch, one slice per (sequence, kv head): the item's output
        // goes straight into the O-projection's operand (bf16 high part and
        // remainder, rows 2b, 2b + 1 of the head's chunk)
        const uint32_t ab = 2u * (uint32_t)g.Bp * 128u;
        const uint32_t col = (uint32_t)((I.g * HPG + h) * D + dim);
        unsigned char* out = g.act + 3 * (size_t)(HT / WIDE_KC) * ab + (size_t)(col / WIDE_KC) * ab;
        const float x = O / Ls;
        const uint16_t hi = to_bf16(x), lo = to_bf16(x - bf1(hi));
        *(uint16_t*)(out + sw128_off(2u * b, col % WIDE_KC)) = hi;
        *(uint16_t*)(out + sw128_off(2u * b + 1u, col % WIDE_KC)) = lo;
        continue;
      }
    }
    const size_t po = ((((size_t)I.layer * g.B + b) * g.Hq + (size_t)I.g * HPG + h) * g.splits +
                       I.r0) * part_stride(D);
    if (MK_IN(g, po + D + 2 <= g.n_part, c.pc, I.op)) {
      float* dst = g.part + po;
      dst[dim] = O;
      if (dim == 0) {
        dst[D] = M;
        dst[D + 1] = Ls;
      }
    }
  }
  consumer_bar();
  if constexpr (NB > 8) return attn_merge_wide(c, g, I);
  return true;
}

// Attention item (b, kv group g, slice) on the tensor cores (attn_tc.cuh):
// the K / V stages arrive as swizzled TMA tiles; each warp takes 16-position
// chunks of every stage (rotating with the stage, so that the short last
// chunk moves between warps), and warp 0 of the item's last slice also runs
// row P from a zero-padded 16-row tile.  The V rows past a stage's last
// position in its last chunk are zeroed first (those rows may hold anything).
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool op_attn_tc(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Instr& I) {
  const int b = I.b, P = c.pos[b];
  const LayerPtrs& Lp = g.layers[I.layer];
  const bool last = I.r0 + 1 == I.r1 && c.warp == 0;
  if (!dep_wait(c, g, I)) return false;
  constexpr float QS = 0.125f * 1.4426950408889634f;  // log2(e) / sqrt(64)
  AttnTC<HPG> st;
  {
    const size_t qo = (((size_t)I.layer * g.B + b) * g.Hq + (size_t)I.g * HPG) * D;
    st.init(g.qbuf + (MK_IN(g, qo + HPG * D <= g.n_q, c.pc, I.op) ? qo : 0), QS, c.lane);
  }
  c.mark(g, 0);
  Seg s[2];
  get_segs<HT, D, WB, NB>(g, I, c.pos, c.topk, s);
  uint32_t rot = 0;  // chunks of earlier stages (round-robin offset)
  for (uint32_t u0 = 0; u0 < s[0].n; u0 += s[0].ups) {
    const uint32_t n = stage_units(g, s[0], u0, (uint32_t)g.stage_bytes / 2, c.pc, OP_ATTN);
    if (!c.ring.acquire(g)) {
      c.flag[2] = 1;
      break;
    }
    const uint32_t kt = smem_u32(c.ring.stage_ptr()), vt = kt + c.ring.sb / 2;
    const uint32_t nch = (n + 15u) / 16u;
    for (uint32_t ch = (uint32_t)(c.warp + NCW - (int)(rot % NCW)) % NCW; ch < nch; ch += NCW) {
      const int nv = (int)min(16u, n - 16u * ch);
      if (nv < 16) {  // zero V rows nv .. 15 of this chunk (generic stores, then a proxy fence
                      // before the stage goes back to the bulk-copy engine)
        unsigned char* vr = (unsigned char*)c.ring.stage_ptr() + c.ring.sb / 2 +
                            (size_t)(16u * ch + (uint32_t)nv) * 128u;
        for (int i = c.lane; i < (16 - nv) * 8; i += 32) ((uint4*)vr)[i] = make_uint4(0, 0, 0, 0);
        __syncwarp();
      }
      st.chunk(kt, vt, 16u * ch, nv, c.lane);
      if (nv < 16) fence_async_smem();
    }
    rot += nch;
    c.ring.release(c.lane);
  }
  if (last) {
    // row P in a 16-row tile (1024-byte aligned, inside xn, free during
    // attention): rows 1..15 zero, row 0 unswizzled
    unsigned char* mt = (unsigned char*)(((uintptr_t)c.xn + 1023) & ~(uintptr_t)1023);
    for (int i = c.lane; i < 256; i += 32) ((uint4*)mt)[i] = make_uint4(0, 0, 0, 0);
    __syncwarp();
    const long long off = kv_row(g, b, I.g, P);
    if (c.lane < 16 && off >= 0 && MK_IN(g, (size_t)off + D <= g.kv_elems, c.pc, I.op)) {
      const uint16_t* src = (c.lane < 8 ? Lp.kc : Lp.vc) + off + (c.lane & 7) * 8;
      ((uint4*)(mt + (c.lane < 8 ? 0 : 2048)))[c.lane & 7] = __ldcg((const uint4*)src);
    }
    __syncwarp();
    st.chunk(smem_u32(mt), smem_u32(mt) + 2048u, 0u, 1, c.lane);
  }
  st.finish();
  c.mark(g, 1);
  consumer_bar();  // (every warp is past its last use of xn's tile and of the ring)
  if (c.flag[2]) return false;
  float* sc = c.yrow;  // [NCW][HPG][D + 2]
  const int gq = c.lane >> 2, tq = c.lane & 3;
  if (gq < HPG) {
    float* p = sc + ((size_t)c.warp * HPG + gq) * (D + 2);
#pragma unroll
    for (int dt = 0; dt < 8; dt++) {
      p[8 * dt + 2 * tq] = st.o[dt][0];
      p[8 * dt + 2 * tq + 1] = st.o[dt][1];
    }
    if (tq == 0) {
      p[D] = st.m;
      p[D + 1] = st.l;
    }
  }
  return attn_cta_merge(c, g, I);
}

template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool op_attn(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Instr& I) {
  if constexpr (attn_tc_path<D, HPG, NB>())
    if (g.tmaps && !g.kv_block) return op_attn_tc(c, g, I);
  constexpr int LPR = D / 8, SPW = 32 / LPR;
  const int slot = c.lane / LPR, dsl = c.lane % LPR;
  const int b = I.b, P = c.pos[b];
  const LayerPtrs& Lp = g.layers[I.layer];
  const bool last = I.r0 + 1 == I.r1 && c.warp == 0;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  if (!dep_wait(c, g, I)) return false;
  // row P (appended by this step's QKV) is fetched together with q
  uint4 kP = zero, vP = zero;
  if (last && slot == 0) {
    const long long off = kv_row(g, b, I.g, P);
    if (off >= 0 && MK_IN(g, (size_t)off + D <= g.kv_elems, c.pc, I.op)) {  // (a bad block was
                                                                            // reported by the append)
      kP = __ldcg((const uint4*)(Lp.kc + off + dsl * 8));
      vP = __ldcg((const uint4*)(Lp.vc + off + dsl * 8));
    }
  }
  constexpr float QS = (D == 64 ? 0.125f : 0.08838834764831845f) * 1.4426950408889634f;
  float q[HPG][8], m[HPG], l[HPG], o[HPG][8];
#pragma unroll
  for (int h = 0; h < HPG; h++) {
    const size_t qo = (((size_t)I.layer * g.B + b) * g.Hq + (size_t)I.g * HPG + h) * D + dsl * 8;
    const float4* qp = (const float4*)(g.qbuf + (MK_IN(g, qo + 8 <= g.n_q, c.pc, I.op) ? qo : 0));
    const float4 a0 = __ldcg(qp), a1 = __ldcg(qp + 1);
    q[h][0] = a0.x * QS; q[h][1] = a0.y * QS; q[h][2] = a0.z * QS; q[h][3] = a0.w * QS;
    q[h][4] = a1.x * QS; q[h][5] = a1.y * QS; q[h][6] = a1.z * QS; q[h][7] = a1.w * QS;
    m[h] = NEG_BIG;
    l[h] = 0.f;
#pragma unroll
    for (int j = 0; j < 8; j++) o[h][j] = 0.f;
  }
  auto process = [&](const uint4& kw, const uint4& vw, bool valid) {
    float kf[8], vf[8], sc[HPG];
    unpack8(kw, kf);
    unpack8(vw, vf);
#pragma unroll
    for (int h = 0; h < HPG; h++) {
      float a = 0.f;
#pragma unroll
      for (int j = 0; j < 8; j++) a = fmaf(q[h][j], kf[j], a);
      sc[h] = a;
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1)
#pragma unroll
      for (int h = 0; h < HPG; h++) sc[h] += __shfl_xor_sync(0xFFFFFFFFu, sc[h], off);
    if (valid) {
#pragma unroll
      for (int h = 0; h < HPG; h++) {
        const float mn = fmaxf(m[h], sc[h]);
        const float cr = exp2f(m[h] - mn), p = exp2f(sc[h] - mn);
        l[h] = fmaf(l[h], cr, p);
#pragma unroll
        for (int j = 0; j < 8; j++) o[h][j] = fmaf(o[h][j], cr, p * vf[j]);
        m[h] = mn;
      }
    }
  };
  // Two positions per slot and pass (j and j + NCW * SPW): their scores,
  // shuffles and exponentials are independent chains, so each hides the
  // other's latency, and one running-max update covers both.  An absent
  // position scores -inf and contributes 2^-inf = 0.
  auto process2 = [&](const uint4& ka, const uint4& va, bool oka, const uint4& kb,
                      const uint4& vb, bool okb) {
    float kfa[8], kfb[8], sa[HPG], sb[HPG];
    unpack8(ka, kfa);
    unpack8(kb, kfb);
#pragma unroll
    for (int h = 0; h < HPG; h++) {
      float a = 0.f, b = 0.f;
#pragma unroll
      for (int j = 0; j < 8; j++) {
        a = fmaf(q[h][j], kfa[j], a);
        b = fmaf(q[h][j], kfb[j], b);
      }
      sa[h] = a;
      sb[h] = b;
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1)
#pragma unroll
      for (int h = 0; h < HPG; h++) {
        sa[h] += __shfl_xor_sync(0xFFFFFFFFu, sa[h], off);
        sb[h] += __shfl_xor_sync(0xFFFFFFFFu, sb[h], off);
      }
    float vfa[8], vfb[8];
    unpack8(va, vfa);
    unpack8(vb, vfb);
#pragma unroll
    for (int h = 0; h < HPG; h++) {
      const float xa = oka ? sa[h] : -INFINITY, xb = okb ? sb[h] : -INFINITY;
      const float mn = fmaxf(m[h], fmaxf(xa, xb));
      const float cr = exp2f(m[h] - mn), pa = exp2f(xa - mn), pb = exp2f(xb - mn);
      l[h] = fmaf(l[h], cr, pa + pb);
#pragma unroll
      for (int j = 0; j < 8; j++) o[h][j] = fmaf(o[h][j], cr, fmaf(pa, vfa[j], pb * vfb[j]));
      m[h] = mn;
    }
  };
  c.mark(g, 0);
  Seg s[2];
  get_segs<HT, D, WB, NB>(g, I, c.pos, c.topk, s);
  constexpr uint32_t STEP = NCW * SPW;  // positions per pass of all warps' slots
  for (uint32_t u0 = 0; u0 < s[0].n; u0 += s[0].ups) {
    const uint32_t n = stage_units(g, s[0], u0, (uint32_t)g.stage_bytes / 2, c.pc, OP_ATTN);
    if (!c.ring.acquire(g)) break;
    const unsigned char* st = c.ring.stage_ptr();
    const unsigned char* vs = st + c.ring.sb / 2;
    for (uint32_t jb = (uint32_t)c.warp * SPW; jb < n; jb += 2 * STEP) {
      const uint32_t ja = jb + slot, jc = ja + STEP;
      const bool oka = ja < n, okb = jc < n;
      const size_t oa = (size_t)ja * D * 2 + dsl * 16, ob = (size_t)jc * D * 2 + dsl * 16;
      const uint4 ka = oka ? *(const uint4*)(st + oa) : zero, va = oka ? *(const uint4*)(vs + oa) : zero;
      const uint4 kb = okb ? *(const uint4*)(st + ob) : zero, vb = okb ? *(const uint4*)(vs + ob) : zero;
      if (jb + STEP < n)
        process2(ka, va, oka, kb, vb, okb);
      else
        process(ka, va, oka);  // (warp-uniform: no slot of this pass has a second position)
    }
    c.ring.release(c.lane);
  }
  if (last) process(kP, vP, slot == 0);
  c.mark(g, 1);
  // merge the slots of the warp
#pragma unroll
  for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
    for (int h = 0; h < HPG; h++) {
      const float mo = __shfl_xor_sync(0xFFFFFFFFu, m[h], off);
      const float lo = __shfl_xor_sync(0xFFFFFFFFu, l[h], off);
      const float mn = fmaxf(m[h], mo);
      const float fa = exp2f(m[h] - mn), fb = exp2f(mo - mn);
      l[h] = l[h] * fa + lo * fb;
#pragma unroll
      for (int j = 0; j < 8; j++) {
        const float oo = __shfl_xor_sync(0xFFFFFFFFu, o[h][j], off);
        o[h][j] = o[h][j] * fa + oo * fb;
      }
      m[h] = mn;
    }
  }
  float* sc = c.yrow;  // [NCW][HPG][D + 2]
  if (slot == 0) {
#pragma unroll
    for (int h = 0; h < HPG; h++) {
      float* p = sc + ((size_t)c.warp * HPG + h) * (D + 2);
#pragma unroll
      for (int j = 0; j < 8; j++) p[dsl * 8 + j] = o[h][j];
      if (dsl == 0) {
        p[D] = m[h];
        p[D + 1] = l[h];
      }
    }
  }
  return attn_cta_merge(c, g, I);
}

// Residual input x_j[b][r] (j = 0: the embedding row of the token).
MK_DEV float x_in(const Globals& g, uint32_t ep, int j, const int* tok, int b, int r) {
  if (j == 0)  // embedding rows are chunk-swizzled by token id
    return bf1(g.embed[(size_t)tok[b] * g.H + ((((r >> 3) ^ (tok[b] & 7)) << 3) | (r & 7))]);
  return xres_sum(g, ep, j, b, r);
}

// The SG partial merges of each (b, dim) of one head into its attention
// output (c.attn).  All consumer threads.
template <int D, int NB, int SG, class C>
MK_DEV void merge_heads(C& c, const Globals& g, const float* pm, const float* pl, const float* po) {
  for (int it = c.tid; it < NB * D; it += NCT) {
    const int b = it / D, dim = it % D;
    float M = NEG_BIG;
#pragma unroll
    for (int sg = 0; sg < SG; sg++) M = fmaxf(M, pm[(b * SG + sg) * D + dim]);
    float Ls = 0.f, O = 0.f;
#pragma unroll
    for (int sg = 0; sg < SG; sg++) {
      const int k = (b * SG + sg) * D + dim;
      const float f = exp2f(pm[k] - M);
      Ls = fmaf(pl[k], f, Ls);
      O = fmaf(po[k], f, O);
    }
    c.attn[b * D + dim] = b < g.B ? O / Ls : 0.f;
  }
}

// --------------------------------- OP_OPROJ (split reduce + O-proj rows) ----
// Head h's partials are merged (M = max m_s, L = sum l_s 2^(m_s - M),
// o = sum o_s 2^(m_s - M) / L), then rows [r0, r1) of Wo[:, h*D:(h+1)*D]
// (packed [Hq][H][D]) are applied and accumulated into x_{2l+1} with float
// atomics; the head-0 instructions also add the residual x_{2l}.
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool op_oproj(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Instr& I) {
  constexpr int SG = (NCT / (NB * D)) > 0 ? NCT / (NB * D) : 1;  // slice groups per (b, dim)
  const int h = I.g, l = I.layer;
  const int S = g.splits;
  constexpr int PS = part_stride(D);  // partial record stride
  if constexpr (WB == 1) {
    // int8: the Wo rows' scales, copied in while the wait runs
    const float* so = g.layers[l].so + I.r0;
    for (int t = c.tid; t < (int)(I.r1 - I.r0); t += NCT) cp_async4(c.sc + t, so + t);
  }
  const bool waited = dep_wait(c, g, I);
  if constexpr (WB == 1) cp_async_wait_all();
  if (!waited) return false;
  Seg s[2];
  bool staged = false;
  float* pm = c.yrow;                    // [NB][SG][D] partial max
  float* pl = pm + NB * SG * D;          // partial sum
  float* po = pl + NB * SG * D;          // partial o
  if constexpr (D >= 128) {
    // heads of 128+ dims, many slices: the head's partials of every
    // sequence land in the instruction's first ring stage, one bulk copy per
    // sequence, issued now that attention is done (the producer armed the
    // stage; every earlier stage is released); the residual loads below
    // overlap them
    staged = g.part_staged != 0;
    if (staged) {
      get_segs<HT, D, WB, NB>(g, I, c.pos, c.topk, s);
      if (c.tid == 0) {
        asm volatile("fence.proxy.async.global;" ::: "memory");  // written by generic stores
        const uint64_t pol = policy_evict_normal();
        const uint32_t blk = (uint32_t)(S * PS * 4);
        for (int b = 0; b < g.B; b++)
          bulk_g2s(smem_u32(c.ring.ahead_ptr(0)) + (uint32_t)b * blk,
                   g.part + (((size_t)l * g.B + b) * g.Hq + h) * S * PS, blk, c.ring.ahead_full(0),
                   pol);
      }
    }
  }
  if (!staged) {
    // Work item (b, dim, sg) merges slices sg, sg + SG, ... straight from L2;
    // all its loads are independent (about one round trip per four slices)
    for (int it = c.tid; it < NB * SG * D; it += NCT) {
      const int dim = it % D, sg = (it / D) % SG, b = it / (D * SG);
      float M = NEG_BIG, Ls = 0.f, O = 0.f;
      if (b < g.B && MK_IN(g, (((size_t)l * g.B + b) * g.Hq + h + 1) * S * PS <= g.n_part, c.pc,
                           I.op)) {
        const float* base = g.part + (((size_t)l * g.B + b) * g.Hq + h) * S * PS;
#pragma unroll 4
        for (int s2 = sg; s2 < S; s2 += SG) {
          const float* p = base + (size_t)s2 * PS;
          const float ms = __ldcg(p + D), ls = __ldcg(p + D + 1), os = __ldcg(p + dim);
          const float mn = fmaxf(M, ms);
          const float fa = exp2f(M - mn), fb = exp2f(ms - mn);
          Ls = Ls * fa + ls * fb;
          O = O * fa + os * fb;
          M = mn;
        }
      }
      pm[it] = M;
      pl[it] = Ls;
      po[it] = O;
    }
    consumer_bar();
    merge_heads<D, NB, SG>(c, g, pm, pl, po);
  }
  const bool resid = (I.flags & F_RESIDUAL) != 0;
  float* xr_s = c.xn;  // residual rows of this slice, [NB][nr] with nr <= H (head-0 slices)
  if (resid) {
    const int nr = (int)(I.r1 - I.r0);
    const bool tagged = g.xtag && l > 0;  // x_{2l} from the down rows' owners
    bool okr = true;
    if (tagged) {
      for (int t = c.tid; t < NB * nr; t += NCT) {
        const int b = t / nr, r = t % nr;
        float v = 0.f;
        const size_t xo = ((size_t)(l - 1) * g.B + b) * g.H + I.r0 + r;
        if (b < g.B && MK_IN(g, xo < g.n_xt, c.pc, I.op)) {
          if (!poll_tag1(g, g.xt + xo, c.epoch, v, c.pc, I.op)) okr = false;
        }
        xr_s[t] = v;
      }
    } else {
      // eight rows' loads in flight before their shared-memory stores
      for (int t0 = c.tid; t0 < NB * nr; t0 += 8 * NCT) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; u++) {
          const int t = t0 + u * NCT, b = t / nr, r = t % nr;
          v[u] = t < NB * nr && b < g.B ? x_in(g, c.epoch, 2 * l, c.tok, b, (int)I.r0 + r) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; u++)
          if (t0 + u * NCT < NB * nr) xr_s[t0 + u * NCT] = v[u];
      }
    }
    if (!okr) c.flag[2] = 1;
  }
  if constexpr (D >= 128) {
    if (staged) {  // the same merge from the stage, once the copies land
      if (c.ring.acquire(g)) {
        const float* part = (const float*)c.ring.stage_ptr();
        for (int it = c.tid; it < NB * SG * D; it += NCT) {
          const int dim = it % D, sg = (it / D) % SG, b = it / (D * SG);
          float M = NEG_BIG, Ls = 0.f, O = 0.f;
          if (b < g.B) {
            const float* base = part + (size_t)b * S * PS;
            for (int s2 = sg; s2 < S; s2 += SG) {
              const float* p = base + (size_t)s2 * PS;
              const float ms = p[D], ls = p[D + 1], os = p[dim];
              const float mn = fmaxf(M, ms);
              const float fa = exp2f(M - mn), fb = exp2f(ms - mn);
              Ls = Ls * fa + ls * fb;
              O = O * fa + os * fb;
              M = mn;
            }
          }
          pm[it] = M;
          pl[it] = Ls;
          po[it] = O;
        }
        c.ring.release(c.lane);
      } else {
        c.flag[2] = 1;
      }
      consumer_bar();
      merge_heads<D, NB, SG>(c, g, pm, pl, po);
    }
  }
  c.mark(g, 0);
  consumer_bar();
  if (c.flag[2]) return false;
  if (!staged) get_segs<HT, D, WB, NB>(g, I, c.pos, c.topk, s);
  const Seg& wseg = s[staged ? 1 : 0];  // the Wo rows
  const uint4 zero = make_uint4(0, 0, 0, 0);
  const int nr = (int)(I.r1 - I.r0);
  if constexpr (NB == 1) {
    // One lane per Wo row: the lane dots its row's D columns with the head's
    // attention output (registers for D = 64, shared-memory broadcasts for
    // D = 128), so there is no cross-lane reduction, and a warp's 32
    // consecutive rows leave as one coalesced reduction.  The packed rows are
    // chunk-swizzled (chunk k of row r at slot k ^ (r & 7)), which keeps the
    // 32 lanes' row reads free of bank conflicts.
    constexpr int CPR = D / 8;
    constexpr bool REG = D <= 64;
    float av[REG ? D : 1];
    if constexpr (REG) {
#pragma unroll
      for (int k = 0; k < D / 4; k++) {
        const float4 t = ((const float4*)c.attn)[k];
        av[4 * k] = t.x; av[4 * k + 1] = t.y; av[4 * k + 2] = t.z; av[4 * k + 3] = t.w;
      }
    }
    float* dst = xres_mine(g, c.epoch, 2 * l + 1, 0);
    uint32_t bc = 0;  // 32-row blocks of earlier stages (round-robin offset)
    for (uint32_t u0 = 0; u0 < wseg.n; u0 += wseg.ups) {
      const uint32_t n = stage_units(g, wseg, u0, (uint32_t)g.stage_bytes, c.pc, OP_OPROJ);
      if (!c.ring.acquire(g)) break;
      const unsigned char* st = c.ring.stage_ptr();
      const uint32_t nblk = (n + 31) / 32;
      for (uint32_t blk = (uint32_t)(c.warp + NCW - (int)(bc % NCW)) % NCW; blk < nblk;
           blk += NCW) {
        const uint32_t j = blk * 32 + (uint32_t)c.lane;
        const bool valid = j < n;
        const uint32_t row = I.r0 + u0 + j;
        const unsigned char* rp = st + (size_t)j * D * WB;
        float a[8];
#pragma unroll
        for (int e = 0; e < 8; e++) a[e] = 0.f;
        if constexpr (WB == 1) {
          // int8 rows of 64 codes, 4 chunks; chunk k of row r sits at slot
          // k ^ ((r >> 1) & 3): 8 consecutive rows (two per 128 bytes) hit 8
          // different bank groups
          static_assert(D == 64 && REG, "int8 Wo rows hold 64 codes");
          float2 a2[4];
#pragma unroll
          for (int e = 0; e < 4; e++) a2[e] = make_float2(0.f, 0.f);
#pragma unroll
          for (int k = 0; k < D / 16; k++) {
            const uint4 w = valid ? *(const uint4*)(rp + ((k ^ ((row >> 1) & 3u)) * 16)) : zero;
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 16; e += 2)
              a2[(e & 7) >> 1] = ffma2(i8_pair(ws[e >> 2], e & 3),
                                       make_float2(av[k * 16 + e], av[k * 16 + e + 1]),
                                       a2[(e & 7) >> 1]);
          }
#pragma unroll
          for (int e = 0; e < 4; e++) {
            a[2 * e] = a2[e].x;
            a[2 * e + 1] = a2[e].y;
          }
        }
#pragma unroll
        for (int k = 0; k < (WB == 1 ? 0 : CPR); k++) {
          const uint4 w = valid ? *(const uint4*)(rp + ((k ^ (row & 7u)) * 16)) : zero;
          float wf[8];
          unpack8(w, wf);
          float xv[8];
          if constexpr (REG) {
#pragma unroll
            for (int e = 0; e < 8; e++) xv[e] = av[k * 8 + e];
          } else {
            const float4 x0 = ((const float4*)c.attn)[2 * k], x1 = ((const float4*)c.attn)[2 * k + 1];
            xv[0] = x0.x; xv[1] = x0.y; xv[2] = x0.z; xv[3] = x0.w;
            xv[4] = x1.x; xv[5] = x1.y; xv[6] = x1.z; xv[7] = x1.w;
          }
#pragma unroll
          for (int e = 0; e < 8; e++) a[e] = fmaf(wf[e], xv[e], a[e]);
        }
        if (valid && MK_IN(g, (size_t)(dst - g.xbuf) + row < g.n_xbuf, c.pc, I.op)) {
          float v = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
          if constexpr (WB == 1) v *= c.sc[row - I.r0];
          if (resid) v += xr_s[row - I.r0];
          red_add_f32(dst + row, v);
        }
      }
      bc += nblk;
      c.ring.release(c.lane);
    }
  } else {
    // Batched (8 sequences): y[b][row] = Wo_h[row] . attn_h[b] on the tensor
    // cores, mma.sync m16n8k16 with f32 accumulators.  A = the head's
    // attention output as the batched GEMV holds activations (rows 0-7 the
    // bf16 high parts of the 8 sequences, rows 8-15 the bf16 remainders, so
    // the sum of the two halves keeps about 16 mantissa bits), built once in
    // registers for the D / 16 k-tiles; B = 8 Wo rows per n-tile, loaded with
    // ldmatrix from the chunk-swizzled stage (chunk k of row r at slot
    // k ^ (r & 7): the 8 row reads of a matrix hit 8 bank groups).  Lane
    // 4g + t ends with sequence g's outputs of rows 2t, 2t + 1 of the n-tile
    // and adds them into x_{2l+1} with one 8-byte reduction (the planner cuts
    // batched O-projection rows at multiples of 8, so the pair is aligned).
    static_assert(NB == 8 && D == 64, "fragments of 8 sequences, 4 k-tiles");
    constexpr int KT = D / 16;
    const int gq = c.lane >> 2, tq = c.lane & 3;
    uint32_t af[KT][4];
#pragma unroll
    for (int kt = 0; kt < KT; kt++) {
      const float* ap = c.attn + gq * D + kt * 16 + 2 * tq;
      split2(ap[0], ap[1], af[kt][0], af[kt][1]);
      split2(ap[8], ap[9], af[kt][2], af[kt][3]);
    }
    const bool live = gq < g.B;
    float* dst = xres_mine(g, c.epoch, 2 * l + 1, live ? gq : 0);
    const uint32_t li = (uint32_t)c.lane & 7u, mi = (uint32_t)c.lane >> 3;
    uint32_t tc = 0;  // 8-row tiles of earlier stages (round-robin offset)
    for (uint32_t u0 = 0; u0 < wseg.n; u0 += wseg.ups) {
      const uint32_t n = stage_units(g, wseg, u0, (uint32_t)g.stage_bytes, c.pc, OP_OPROJ);
      if (!c.ring.acquire(g)) break;
      const uint32_t sbase = smem_u32(c.ring.stage_ptr());
      const uint32_t nt = (n + 7) / 8;
      for (uint32_t t = (uint32_t)(c.warp + NCW - (int)(tc % NCW)) % NCW; t < nt; t += NCW) {
        // rows past the stage's last repeat row 8t (their outputs are dropped)
        const uint32_t rr = t * 8 + li < n ? t * 8 + li : t * 8;
        const uint32_t key = (I.r0 + u0 + rr) & 7u;
        const uint32_t ra = sbase + rr * (uint32_t)(D * 2);
        uint32_t b[8];
        ldsm_x4(ra + ((mi ^ key) << 4), b[0], b[1], b[2], b[3]);
        ldsm_x4(ra + (((mi + 4u) ^ key) << 4), b[4], b[5], b[6], b[7]);
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kt = 0; kt < KT; kt++) mma_16816(d, af[kt], b[2 * kt], b[2 * kt + 1]);
        const uint32_t r = t * 8 + 2u * (uint32_t)tq;  // stage row of this lane's pair
        if (live && r < n &&
            MK_IN(g, (size_t)(dst - g.xbuf) + I.r0 + u0 + r + 2 <= g.n_xbuf, c.pc, I.op)) {
          const int row = (int)(I.r0 + u0 + r);
          float v0 = d[0] + d[2], v1 = d[1] + d[3];
          if (resid) {
            v0 += xr_s[gq * nr + (row - (int)I.r0)];
            if (r + 1 < n) v1 += xr_s[gq * nr + (row + 1 - (int)I.r0)];
          }
          if (r + 1 < n)
            red_add_v2f32(dst + row, v0, v1);
          else
            red_add_f32(dst + row, v0);
        }
      }
      tc += nt;
      c.ring.release(c.lane);
    }
  }
  c.mark(g, 1);
  consumer_bar();
  return true;
}

// ------------------------------------------------- OP_ROUTER (MoE only) ----
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool op_router(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Instr& I) {
  const LayerPtrs& Lp = g.layers[I.layer];
  NormGain<HT, NB> ng;
  norm_gain(ng, Lp.mlp_norm, c.tid);
  if (!dep_wait(c, g, I)) return false;
  if (!norm_apply(c, g, 2 * I.layer + 1, ng)) return false;
  float xr[HT / 32];
  if constexpr (NB == 1) load_xr<HT, WB>(c.xn, c.lane, xr);
  Seg s[2];
  get_segs<HT, D, WB, NB>(g, I, c.pos, c.topk, s);
  float* rl = g.rlog + (size_t)I.layer * g.B * g.E + I.r0;
  const int E = g.E;
  gemv(c, g, s[0], xr, [&](uint32_t r, int b, float y) { rl[(size_t)b * E + r] = y; });
  consumer_bar();
  // Every router instruction of the layer arrives once; the last to arrive
  // ranks all E logits and publishes the routing, then signals the router
  // counter once for all of them (I.aux of them).  Softmax is monotonic, so
  // the top-K by probability are the K largest logits; rank i = number of
  // logits above logit i, equal ones with a lower id counting as above.
  // Weights are the probabilities renormalised over the K chosen,
  // exp(l - l_max) / sum.  Batch 1 (sequence 0).
  // (its own slot: flag[3] holds the dependency-wait key of the instruction
  // whose counter was seen, and an arrival count equal to the next
  // instruction's key would let that instruction skip its wait)
  int* arrived = c.flag + 5;
  if (c.tid == 0)
    *arrived = (int)atom_add_acq_rel(g.ctr + CtrMap{g.Hkv, g.L}.router_arrive(I.layer), 1u);
  consumer_bar();
  if ((uint32_t)*arrived != c.epoch * I.aux - 1u) return true;
  float* ys = c.yrow;               // [E <= 256] logits
  int* sel = (int*)(c.yrow + 256);  // [K <= 16] ids by rank
  float* sv = c.yrow + 256 + 16;    // [K] their logits
  const float* lg = g.rlog + (size_t)I.layer * g.B * g.E;
  for (int i = c.tid; i < E; i += NCT) ys[i] = __ldcg(lg + i);
  if (c.tid < g.K) {
    sel[c.tid] = 0;
    sv[c.tid] = -INFINITY;
  }
  consumer_bar();
  for (int i = c.tid; i < E; i += NCT) {
    const float li = ys[i];
    int rank = 0;
    for (int j = 0; j < E; j++) {
      const float lj = ys[j];
      rank += (lj > li || (lj == li && j < i)) ? 1 : 0;
    }
    if (rank < g.K) {
      sel[rank] = i;
      sv[rank] = li;
    }
  }
  consumer_bar();
  if (c.tid == 0) {
    const float top = sv[0];
    float sum = 0.f;
    for (int r = 0; r < g.K; r++) sum += expf(sv[r] - top);
    for (int r = 0; r < g.K; r++) {
      g.routes[(size_t)I.layer * g.K + r] = sel[r];
      g.rweight[(size_t)I.layer * g.K + r] = expf(sv[r] - top) / sum;
    }
    red_release(g.ctr + I.sig_ctr, I.aux);
  }
  return true;
}

// ---------------------------------------- OP_MLP (one FFN column slice) ----
// h_c = SiLU(gate_c . xn) * (up_c . xn) for the slice's columns c, then
// x_{2l+2} += sum_c h_c * Wd[:, c] (down stored transposed, one contiguous
// row per column) with float4 atomics; the instruction also adds x_{2l+1}
// for its residual rows.  MoE: routed slices scale h by the slot's router
// weight and read expert topk[slot]'s rows; shared slices use weight 1.
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool op_mlp(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Instr& I) {
  const int l = I.layer;
  const LayerPtrs& Lp = g.layers[l];
  const bool routed = g.E > 0 && !(I.flags & F_SHARED);
  const bool cached = (I.flags & F_NORM_CACHED) != 0;
  NormGain<HT, NB> ng;
  if (!cached) norm_gain(ng, Lp.mlp_norm, c.tid);
  if (!dep_wait(c, g, I)) return false;
  if (!cached && !norm_apply(c, g, 2 * l + 1, ng)) return false;
  c.mark(g, 0);
  if (routed) {  // the routing this layer's last router published (ids clamped to [0, E))
    if (c.warp == 0 && c.lane < g.K) {
      const int e = __ldcg(g.routes + (size_t)l * g.K + c.lane);
      c.topk[c.lane] = min(max(e, 0), g.E - 1);
      c.topw[c.lane] = __ldcg(g.rweight + (size_t)l * g.K + c.lane);
    }
    consumer_bar();
  }
  const float scale = routed ? c.topw[I.g] : 1.f;
  float xr[HT / 32];
  if constexpr (NB == 1) load_xr<HT, WB>(c.xn, c.lane, xr);
  Seg s[2];
  get_segs<HT, D, WB, NB>(g, I, c.pos, c.topk, s);
  float* yrow = c.yrow;
  const int lane = c.lane;
  gemv(c, g, s[0], xr, [&](uint32_t r, int b, float y) { yrow[b * MAX_ROWS + r] = y; });
  consumer_bar();
  const int ncol = (int)(I.r1 - I.r0);
  for (int t = c.tid; t < NB * ncol; t += NCT) {
    const int b = t / ncol, j = t % ncol;
    const float gt = yrow[b * MAX_ROWS + 2 * j], up = yrow[b * MAX_ROWS + 2 * j + 1];
    c.hbuf[b * MAX_COLS + j] = scale * (gt / (1.f + expf(-gt))) * up;
  }
  consumer_bar();
  // Down columns as an axpy over the output in 4-row quads (8 bytes of a
  // transposed down row): HT / 4 quads over the consumer threads, so the
  // busiest thread holds ceil(HT / 4 / NCT) quads (12 rows at H = 2048)
  // rather than two 8-row groups; one 16-byte reduction per quad.
  constexpr int NQ = HT / 4;                   // 4-row quads of the output
  constexpr int QPT = (NQ + NCT - 1) / NCT;    // quads per consumer thread (at most)
  float acc[QPT][NB][4];
#pragma unroll
  for (int q = 0; q < QPT; q++)
#pragma unroll
    for (int b = 0; b < NB; b++)
#pragma unroll
      for (int k = 0; k < 4; k++) acc[q][b][k] = 0.f;
  for (uint32_t u0 = 0; u0 < s[1].n; u0 += s[1].ups) {
    const uint32_t n = stage_units(g, s[1], u0, (uint32_t)g.stage_bytes, c.pc, OP_MLP);
    if (!c.ring.acquire(g)) break;
    const unsigned char* st = c.ring.stage_ptr();
    for (uint32_t j = 0; j < n; j++) {
      float hv[NB];
#pragma unroll
      for (int b = 0; b < NB; b++) hv[b] = c.hbuf[b * MAX_COLS + u0 + j];
#pragma unroll
      for (int q = 0; q < QPT; q++) {
        const int k = c.tid + q * NCT;
        if (k < NQ) {
          const uint2 w = *(const uint2*)(st + (size_t)j * HT * 2 + k * 8);
          const float wf[4] = {bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y)};
#pragma unroll
          for (int b = 0; b < NB; b++)
#pragma unroll
            for (int e = 0; e < 4; e++) acc[q][b][e] = fmaf(hv[b], wf[e], acc[q][b][e]);
        }
      }
    }
    c.ring.release(c.lane);
  }
  c.mark(g, 1);
  const int rs0 = (int)(I.aux & 0xFFFFu), rs1 = (int)(I.aux >> 16);
#pragma unroll
  for (int q = 0; q < QPT; q++) {
    const int k = c.tid + q * NCT;
    if (k < NQ) {
      const int r0 = k * 4;
      for (int b = 0; b < g.B && b < NB; b++) {
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; e++) {
          v[e] = acc[q][b][e];
          if (r0 + e >= rs0 && r0 + e < rs1) v[e] += xres_sum(g, c.epoch, 2 * l + 1, b, r0 + e);
        }
        red_add_v4f32(xres_mine(g, c.epoch, 2 * l + 2, b) + r0, v[0], v[1], v[2], v[3]);
      }
    }
  }
  consumer_bar();
  return true;
}

// ------------------------------------- OP_MLP_UP (gate/up column slice) ----
// h_c = SiLU(gate_c . xn) * (up_c . xn) for the slice's FFN columns, written
// to the layer's h vector in global memory for the down instructions.
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool op_mlp_up(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Instr& I) {
  const int l = I.layer;
  const LayerPtrs& Lp = g.layers[l];
  const bool cached = (I.flags & F_NORM_CACHED) != 0;
  NormGain<HT, NB> ng;
  if (!cached) norm_gain(ng, Lp.mlp_norm, c.tid);
  // int8: the gate / up row scales of this thread's FFN column (NB == 1:
  // one column per thread)
  float2 usc = make_float2(1.f, 1.f);
  if constexpr (WB == 1) {
    static_assert(NB == 1 && MAX_COLS <= NCT, "one column per thread");
    if (c.tid < (int)(I.r1 - I.r0)) usc = *(const float2*)(Lp.sgu + 2 * (I.r0 + c.tid));
  }
  if (!dep_wait(c, g, I)) return false;
  if (!cached && !norm_apply(c, g, 2 * l + 1, ng)) return false;
  c.mark(g, 0);
  float xr[HT / 32];
  if constexpr (NB == 1) load_xr<HT, WB>(c.xn, c.lane, xr);
  Seg s[2];
  get_segs<HT, D, WB, NB>(g, I, c.pos, c.topk, s);
  float* yrow = c.yrow;
  const int lane = c.lane;
  gemv(c, g, s[0], xr, [&](uint32_t r, int b, float y) { yrow[b * MAX_ROWS + r] = y; });
  c.mark(g, 1);
  consumer_bar();
  const int ncol = (int)(I.r1 - I.r0);
  if constexpr (NB > 1) {
    // h into shared memory (0 for sequences past the batch), then out as the
    // down rows' tensor-core A fragments, one 16-byte word per (16-column
    // k-tile, lane 4g + t): bf16 hi / lo of sequence g at columns 2t, 2t+1
    // and 2t+8, 2t+9 of the k-tile (the slice is whole k-tiles)
    float* hs = c.hbuf;  // [NB][MAX_COLS]
    for (int t = c.tid; t < NB * ncol; t += NCT) {
      const int b = t / ncol, j = t % ncol;
      float h = 0.f;
      if (b < g.B) {
        const float gt = yrow[b * MAX_ROWS + 2 * j], up = yrow[b * MAX_ROWS + 2 * j + 1];
        h = (gt / (1.f + expf(-gt))) * up;
      }
      hs[b * MAX_COLS + j] = h;
    }
    consumer_bar();
    uint4* hf = (uint4*)g.hglob + ((size_t)l * (g.F / 16) + I.r0 / 16) * 32;
    for (int it = c.tid; it < (ncol / 16) * 32; it += NCT) {
      const int kt = it / 32, ln = it % 32, gq = ln >> 2, tq = ln & 3;
      const float* hp = hs + gq * MAX_COLS + kt * 16 + 2 * tq;
      uint4 f;
      split2(hp[0], hp[1], f.x, f.y);
      split2(hp[8], hp[9], f.z, f.w);
      hf[it] = f;
    }
  } else {
    for (int t = c.tid; t < NB * ncol; t += NCT) {
      const int b = t / ncol, j = t % ncol;
      if (b < g.B) {
        float gt = yrow[b * MAX_ROWS + 2 * j], up = yrow[b * MAX_ROWS + 2 * j + 1];
        if constexpr (WB == 1) {
          gt *= usc.x;
          up *= usc.y;
        }
        const size_t ho = ((size_t)l * g.B + b) * g.F + I.r0 + j;
        if (MK_IN(g, ho < g.n_h, c.pc, I.op)) g.hglob[ho] = (gt / (1.f + expf(-gt))) * up;
      }
    }
  }
  consumer_bar();
  return true;
}

// --------------------------------------- OP_MLP_DOWN (down rows, batch 1) ----
// Rows [r0, r1) of x_{2l+2} = x_{2l+1} + Wd h: each consumer thread holds
// its 16-byte chunks of h in registers and dots them with the same chunks of
// every down row streamed through the ring; per-warp partials meet in shared
// memory.  Plain stores: no atomics, no other SM touches these rows.
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool op_mlp_down(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Instr& I) {
  if constexpr (NB != 1) {
    // Batched (8 sequences): a run [r0, r1) of chunk-major units (chunk q,
    // row block rb) = unit q * NRB + rb, spanning chunks q0 and at most q0 + 1.
    // After the gate/up counter the consumers copy those chunks' h fragments
    // (A fragments as the gate/up slices wrote them: rows 0-7 the hi parts of
    // 8 sequences, rows 8-15 the lo parts) into shared memory with cp.async,
    // and the residual rows of any chunk-0 unit; the units' weights stream
    // through the ring (chunk q' of unit row i at slot q' ^ (i & 7)).  Warp
    // w takes the run's units w, w + NCW, ... whole: 32 k-tiles, B = 8
    // weight rows by ldmatrix, two accumulators for rows 0-7 and 8-15, so no
    // cross-warp sum is needed.  Each lane then adds sequence g's outputs of
    // two row pairs into x_{2l+2} with 8-byte float reductions.
    static_assert(NB == 8, "fragments of 8 sequences");
    constexpr int KT = BD_KC / 16;                        // k-tiles per chunk
    constexpr uint32_t UNIT = BD_ROWS * BD_KC * 2u;       // bytes of a weight unit
    constexpr int RES_MAX = BD_MAX_UNITS * BD_ROWS * NB;  // residual values of chunk-0 units
    static_assert(2 * KT * 32 * 16 + RES_MAX * 4 <= NB * HT * 4, "h + residual fit xn");
    const int l = I.layer;
    const uint32_t NRB = (uint32_t)g.H / BD_ROWS;
    const uint32_t u0 = I.r0, u1 = I.r1, q0 = u0 / NRB;
    const uint32_t nq = (u1 - 1) / NRB - q0 + 1;  // 1 or 2 chunks of h
    if (!dep_wait(c, g, I)) return false;
    uint4* hs = (uint4*)c.xn;                      // [nq][KT][32 lanes] A fragments
    float* res = c.xn + 2 * KT * 32 * 4;           // [units of chunk 0][BD_ROWS][NB]
    {
      const uint4* src = (const uint4*)g.hglob + ((size_t)l * (g.F / 16) + (size_t)q0 * KT) * 32;
      for (int i = c.tid; i < (int)(nq * KT * 32); i += NCT) cp_async16(hs + i, src + i);
      // chunk-0 units add the residual x_{2l+1} of their rows
      const int n0 = q0 == 0 ? (int)(min(u1, NRB) - u0) : 0;
      for (int t = c.tid; t < n0 * BD_ROWS * NB; t += NCT) {
        const int j = t / (BD_ROWS * NB), r = (t / NB) % BD_ROWS, b = t % NB;
        res[t] = b < g.B ? xres_sum(g, c.epoch, 2 * l + 1, b, (int)(u0 + j) * BD_ROWS + r) : 0.f;
      }
      cp_async_wait_all();
    }
    consumer_bar();
    c.mark(g, 0);
    const int gq = c.lane >> 2, tq = c.lane & 3;
    // ldmatrix lanes: matrix m = lane / 8 is rows 8 (m / 2) .. +7, k half m % 2
    const uint32_t li = (uint32_t)c.lane & 7u, mi = (uint32_t)c.lane >> 3;
    const uint32_t roff = (li + 8u * (mi >> 1)) * (BD_KC * 2u);
    const bool live = gq < g.B;
    float* dst = xres_mine(g, c.epoch, 2 * l + 2, live ? gq : 0);
    Seg s[2];
    get_segs<HT, D, WB, NB>(g, I, c.pos, c.topk, s);
    bool bad = false;
    for (uint32_t v0 = 0; v0 < s[0].n; v0 += s[0].ups) {
      const uint32_t n = stage_units(g, s[0], v0, (uint32_t)g.stage_bytes, c.pc, OP_MLP_DOWN);
      if (!c.ring.acquire(g)) {
        bad = true;
        break;
      }
      const uint32_t wb = smem_u32(c.ring.stage_ptr());
      for (uint32_t j = 0; j < n; j++) {
        const uint32_t u = u0 + v0 + j;
        if ((int)((v0 + j) % NCW) != c.warp) continue;
        const uint32_t q = u / NRB, rb = u % NRB;
        const uint4* af = hs + (size_t)(q - q0) * KT * 32 + c.lane;
        const uint32_t wu = wb + j * UNIT + roff;
        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int kt = 0; kt < KT; kt++) {
          const uint4 fa = af[kt * 32];
          const uint32_t a[4] = {fa.x, fa.y, fa.z, fa.w};
          uint32_t b0, b1, b2, b3;
          ldsm_x4(wu + ((((uint32_t)(2 * kt) + (mi & 1u)) ^ li) << 4), b0, b1, b2, b3);
          mma_16816(d0, a, b0, b1);
          mma_16816(d1, a, b2, b3);
        }
        if (live) {
          // rows 2t, 2t + 1 (d0) and 8 + 2t, 9 + 2t (d1) of the unit, sequence gq
          float v[4] = {d0[0] + d0[2], d0[1] + d0[3], d1[0] + d1[2], d1[1] + d1[3]};
          if (q == 0) {
            const float* rr = res + (size_t)(u - u0) * BD_ROWS * NB + gq;
            v[0] += rr[(2 * tq) * NB];
            v[1] += rr[(2 * tq + 1) * NB];
            v[2] += rr[(8 + 2 * tq) * NB];
            v[3] += rr[(9 + 2 * tq) * NB];
          }
          const int row = (int)rb * BD_ROWS + 2 * tq;
          red_add_v2f32(dst + row, v[0], v[1]);
          red_add_v2f32(dst + row + 8, v[2], v[3]);
        }
      }
      c.ring.release(c.lane);
    }
    c.mark(g, 1);
    if (bad) c.flag[2] = 1;
    consumer_bar();
    if (c.flag[2]) return false;
    return true;
  } else {
    // a 16-byte chunk of a down row covers CW columns (8 bf16 or 16 int8)
    constexpr int CW = 16 / WB;
    constexpr int CPT = (DOWN_ROW_MAX / 2 / CW + NCT - 1) / NCT;  // h chunks per thread (F <= 8192)
    const int l = I.layer, F = g.F, nch = F / CW;
    const int nrows = (int)(I.r1 - I.r0);
    float dsc = 1.f;  // int8: this thread's output row scale
    if constexpr (WB == 1)
      if (c.tid < nrows) dsc = __ldg(g.layers[l].sd + I.r0 + c.tid);
    if (!dep_wait(c, g, I)) return false;
    float h[CPT][CW];
    // (the whole row of h this layer's down rows read)
    const float* hp =
        g.hglob + (MK_IN(g, ((size_t)l + 1) * F <= g.n_h, c.pc, I.op) ? (size_t)l * F : 0);
#pragma unroll
    for (int q = 0; q < CPT; q++) {
      const int k = c.tid + q * NCT;
#pragma unroll
      for (int e4 = 0; e4 < CW / 4; e4++) {
        const float4 a = k < nch ? __ldcg((const float4*)(hp + (size_t)k * CW) + e4)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        h[q][4 * e4] = a.x; h[q][4 * e4 + 1] = a.y; h[q][4 * e4 + 2] = a.z; h[q][4 * e4 + 3] = a.w;
      }
    }
    const float res = c.tid < nrows ? xres_sum(g, c.epoch, 2 * l + 1, 0, (int)I.r0 + c.tid) : 0.f;
    c.mark(g, 0);
    float* part = c.yrow;  // [NCW][MAX_DOWN_ROWS]
    const uint4 zero = make_uint4(0, 0, 0, 0);
    float pend = 0.f;
    int prow = -1;
    Seg s[2];
    get_segs<HT, D, WB, NB>(g, I, c.pos, c.topk, s);
    for (uint32_t u0 = 0; u0 < s[0].n; u0 += s[0].ups) {
      const uint32_t n = stage_units(g, s[0], u0, (uint32_t)g.stage_bytes, c.pc, OP_MLP_DOWN);
      if (!c.ring.acquire(g)) break;
      const unsigned char* st = c.ring.stage_ptr();
      for (uint32_t j = 0; j < n; j++) {
        const float prev = warp_sum(pend);  // overlaps this row's FMAs
        float a[CPT];
#pragma unroll
        for (int q = 0; q < CPT; q++) {
          const int k = c.tid + q * NCT;
          const uint4 wv = k < nch ? *(const uint4*)(st + (size_t)j * F * WB + (size_t)k * 16) : zero;
          float a0 = 0.f, a1 = 0.f;
          if constexpr (WB == 1) {
            const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
            float2 a01 = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 16; e += 2)
              a01 = ffma2(i8_pair(ws[e >> 2], e & 3), make_float2(h[q][e], h[q][e + 1]), a01);
            a0 = a01.x;
            a1 = a01.y;
          } else {
            float w[8];
            unpack8(wv, w);
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              a0 = fmaf(w[e], h[q][e], a0);
              a1 = fmaf(w[e + 1], h[q][e + 1], a1);
            }
          }
          a[q] = a0 + a1;
        }
        if (prow >= 0 && c.lane == 0) part[c.warp * MAX_DOWN_ROWS + prow] = prev;
        float t = 0.f;
#pragma unroll
        for (int q = 0; q < CPT; q++) t += a[q];
        pend = t;
        prow = (int)(u0 + j);
      }
      c.ring.release(c.lane);
    }
    if (prow >= 0) {
      const float last = warp_sum(pend);
      if (c.lane == 0) part[c.warp * MAX_DOWN_ROWS + prow] = last;
    }
    c.mark(g, 1);
    consumer_bar();
    if (c.tid < nrows) {
      float y = 0.f;
#pragma unroll
      for (int w = 0; w < NCW; w++) y += part[w * MAX_DOWN_ROWS + c.tid];
      if constexpr (WB == 1) y *= dsc;
      const size_t xo = (size_t)l * g.B * g.H + I.r0 + c.tid;
      if (MK_IN(g, xo < g.n_xt, c.pc, I.op)) st_tag(g.xt + xo, res + y, c.epoch);
    }
    consumer_bar();
    return true;
  }
}

// ------------------------------------ OP_LMHEAD (final norm + head rows) ----
// Logits rows [r0, r1) and this slice's (max, first index); the slice that
// arrives last on the argmax counter reduces all slices into argmax[b].
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool op_lmhead(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Instr& I) {
  if (g.zero_next) {
    // this slice's share of the next step's residual buffers (the other
    // parity): every step of this and earlier launches that read them is
    // done, and the next step accumulates into them only after the argmax
    // counter below, which waits for every LM head slice
    const size_t total = (size_t)2 * g.L * g.kc * g.B * g.H;
    const size_t a = total * I.aux / (size_t)g.n_lm, e = total * (I.aux + 1) / (size_t)g.n_lm;
    float* nx = g.xbuf + (size_t)((c.epoch + 1u) & 1u) * total;
    if (MK_IN(g, 2 * total <= g.n_xbuf, c.pc, I.op))
      for (size_t i = a + c.tid; i < e; i += NCT) nx[i] = 0.f;
  }
  NormGain<HT, NB> ng;
  norm_gain(ng, g.final_norm, c.tid);
  if constexpr (WB == 1)  // int8: the rows' scales (at most HT rows), copied in while the wait runs
    for (int t = c.tid; t < (int)(I.r1 - I.r0); t += NCT) cp_async4(c.sc + t, g.lm_scale + I.r0 + t);
  const bool waited = dep_wait(c, g, I);
  if constexpr (WB == 1) cp_async_wait_all();
  if (!waited) return false;
  if (!norm_apply(c, g, 2 * g.L, ng)) return false;
  c.mark(g, 0);
  float xr[HT / 32];
  if constexpr (NB == 1) load_xr<HT, WB>(c.xn, c.lane, xr);
  Seg s[2];
  get_segs<HT, D, WB, NB>(g, I, c.pos, c.topk, s);
  // each thread only ever sees one sequence, b = tid % NB (both GEMV paths);
  // it keeps that sequence's best (value, lowest row) of this slice
  float best = -INFINITY;
  int bidx = 0x7FFFFFFF;
  const int lane = c.lane, B = g.B, V = g.V;
  float* logits = g.logits;
  const uint32_t r0 = I.r0;
  const float* rsc = c.sc;
  const int pcI = c.pc;
  gemv(c, g, s[0], xr, [&](uint32_t r, int b, float y) {
    if constexpr (WB == 1) y *= rsc[r];
    const int row = (int)(r0 + r);
    if (MK_IN(g, row < V, pcI, OP_LMHEAD)) logits[(size_t)b * V + row] = y;
    if (y > best || (y == best && row < bidx)) {
      best = y;
      bidx = row;
    }
  });
  // lanes with equal lane % NB hold the same sequence: reduce them into
  // lanes 0 .. NB-1, one per sequence
#pragma unroll
  for (int o = NB; o < 32; o <<= 1) {
    const float ov = __shfl_xor_sync(0xFFFFFFFFu, best, o);
    const int oi = __shfl_xor_sync(0xFFFFFFFFu, bidx, o);
    if (ov > best || (ov == best && oi < bidx)) {
      best = ov;
      bidx = oi;
    }
  }
  float* rv = c.red;
  int* ri = (int*)(c.red + NCW * NB);
  if (lane < NB) {
    rv[c.warp * NB + lane] = best;
    ri[c.warp * NB + lane] = bidx;
  }
  consumer_bar();
  if (c.tid == 0 && MK_IN(g, ((size_t)I.aux + 1) * B <= g.n_lmv, c.pc, I.op)) {
    for (int b = 0; b < B && b < NB; b++) {
      float v = -INFINITY;
      int ix = 0x7FFFFFFF;
      for (int w = 0; w < NCW; w++) {
        const float ov = rv[w * NB + b];
        const int oi = ri[w * NB + b];
        if (ov > v || (ov == v && oi < ix)) {
          v = ov;
          ix = oi;
        }
      }
      g.lm_val[(size_t)I.aux * B + b] = v;
      g.lm_idx[(size_t)I.aux * B + b] = ix;
    }
  }
  lm_reduce(c, g);
  return true;
}

// The LM-head slices' last step (all consumer threads, once this slice's
// (max, first index) per sequence is in lm_val / lm_idx): count the slice in;
// the CTA whose slice arrives last reduces all slices into argmax[b], one
// sequence per warp with four slices' loads in flight per lane, and signals
// the step done.
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV void lm_reduce(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g) {
  const int lane = c.lane, B = g.B;
  consumer_bar();  // every slice value this CTA writes is written
  if (c.tid == 0)
    c.flag[7] = atom_add_acq_rel(g.ctr + g.lm_ctr, 1u) == c.epoch * (uint32_t)g.n_lm - 1u;
  consumer_bar();
  if (!c.flag[7]) return;
  for (int b = c.warp; b < B && b < NB; b += NCW) {
    float v = -INFINITY;
    int ix = 0x7FFFFFFF;
    for (int k0 = lane; k0 < g.n_lm; k0 += 4 * 32) {
      float ov[4];
      int oi[4];
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const int k = k0 + 32 * u;
        ov[u] = k < g.n_lm ? __ldcg(g.lm_val + (size_t)k * B + b) : -INFINITY;
        oi[u] = k < g.n_lm ? __ldcg(g.lm_idx + (size_t)k * B + b) : 0x7FFFFFFF;
      }
#pragma unroll
      for (int u = 0; u < 4; u++)
        if (ov[u] > v || (ov[u] == v && oi[u] < ix)) {
          v = ov[u];
          ix = oi[u];
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, v, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, ix, o);
      if (ov > v || (ov == v && oi < ix)) {
        v = ov;
        ix = oi;
      }
    }
    if (lane == 0) g.argmax[(size_t)c.step * B + b] = ix;
  }
  // every SM is done with this step once its argmax is out: a multi-step
  // launch starts the next step behind this signal
  consumer_bar();
  if (c.tid == 0) red_release(g.ctr + g.lm_done_ctr, 1u);
}

}  // namespace mk

#include "megakernel_wide.cuh"

namespace mk {

// ------------------------------------------------------------ interpreter ----
MK_DEV Instr load_instr(const Globals& g, int sm, int pc) {
  const uint4* p = (const uint4*)(g.sched + (size_t)sm * g.max_pc + pc);
  const uint4 a = __ldg(p), b = __ldg(p + 1);
  Instr I;
  *(uint4*)&I = a;
  *((uint4*)&I + 1) = b;
  return I;
}

// Second cursor of the producer: walks the same chunk sequence as the ring
// cursor.  Only while the ring is full (the consumers are waiting on a
// dependency and the producer is blocked) does it warm L2 with the chunks
// that lie up to l2_ahead bytes beyond the ring cursor, so that HBM keeps
// streaming the SM's upcoming weights during the wait and the ring then
// refills from L2; chunks the ring has already issued are skipped.  The
// prefetches are per-line LSU prefetches spread over the producer warp's 32
// lanes (the TMA engine stays free for the ring copies); every lane runs the
// cursor in lockstep.
template <int HT, int D, int NB, int WB>
struct L2Cursor {
  int pc = 0, k = 0, nseg = 0;
  uint32_t u0 = 0;
  unsigned long long bytes = 0;
  bool done = false;
  Seg s[2];

  // Advance over chunks ending at or before `from` without prefetching, then
  // prefetch at most `budget` chunks that start below `limit`.
  MK_DEV void run(const Globals& g, unsigned long long limit, unsigned long long from,
                  const int* ptopk, int routed_layer, int budget) {
    while (!done && bytes < limit && budget > 0) {
      if (k >= nseg) {
        if (pc >= g.max_pc) {
          done = true;
          return;
        }
        const Instr I = load_instr(g, queue_id(g), pc);
        if (I.op == OP_HALT) {
          done = true;
          return;
        }
        if (I.op == OP_NOP) {
          pc++;
          continue;
        }
        const bool routed = I.op == OP_MLP && g.E > 0 && !(I.flags & F_SHARED);
        if (routed && routed_layer != (int)I.layer) return;  // addresses not known yet
        int pos[NB];
        if (I.op == OP_ATTN) {
          if (g.pdl) {  // positions may still be written by the previous launch
            pc++;
            continue;
          }
          const int P = __ldg(g.positions + I.b);
          if (P < 0 || P >= g.max_ctx) {
            done = true;
            return;
          }
          pos[I.b] = P;
        }
        nseg = get_segs<HT, D, WB, NB>(g, I, pos, ptopk, s);
        k = 0;
        u0 = 0;
        pc++;
        continue;
      }
      if (u0 >= s[k].n) {
        k++;
        u0 = 0;
        continue;
      }
      const uint32_t n = min(s[k].ups, s[k].n - u0);
      const uint32_t b = n * s[k].unit;
      const bool wseg = NB > 8 && s[k].wide();
      const unsigned long long cb = wseg ? (unsigned long long)n * (s[k].unit + s[k].unit2())
                                         : (s[k].src2 ? 2ull * b : b);
      if (bytes + cb > from && !s[k].cfill() && !wseg && !(g.kv_block && s[k].src2)) {
        if ((threadIdx.x & 31) == 0) {
          bulk_prefetch_l2(s[k].src + (size_t)u0 * s[k].unit, b);
          if (s[k].src2) bulk_prefetch_l2(s[k].src2 + (size_t)u0 * s[k].unit, b);
        }
        budget--;
      }
      bytes += cb;
      u0 += n;
    }
  }
};

// The source of a bulk copy, checked in the bounds build: it must lie in the
// packed weights, the scratch or the instruction's layer of K / V cache;
// otherwise MK_ERR_BOUNDS is recorded and the copy reads the first bytes of
// the packed weights instead, so the stage still completes (the step has
// failed by then).
MK_DEV const unsigned char* copy_src(const Globals& g, const Instr& I, const unsigned char* p,
                                     uint32_t bytes, int pc) {
#ifdef MK_BOUNDS
  const LayerPtrs* Lp = g.layers + (I.op == OP_LMHEAD ? 0 : I.layer);
  const size_t kvb = g.kv_elems * 2;
  const bool ok = span_in(p, bytes, g.pk_lo, g.pk_bytes) || span_in(p, bytes, g.sc_lo, g.sc_bytes) ||
                  span_in(p, bytes, Lp->kc, kvb) || span_in(p, bytes, Lp->vc, kvb);
  if (!MK_IN(g, ok, pc, I.op)) return g.pk_lo;
#endif
  return p;
}

// Producer warp: walks the queue and streams every instruction's segments
// into the ring (lane 0 issues).  It waits for free stages, and besides:
// a routed MoE slice needs the router result for its weight addresses, a
// batched down unit's activation half needs the gate/up counter, and a held
// instruction issues its later stages only once the consumers have finished
// the instructions before it.  On any error it stops issuing and waits for
// its copies in flight before the CTA may exit.
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV void producer(const Globals& g, unsigned char* ring, uint32_t full0, uint32_t empty0,
                     int* ppos, int* ptopk, float* ptopw, const int* done, int lane) {
  const uint64_t pol_w = policy_evict_first();
  const uint64_t pol_kv = policy_evict_normal();
  const int ns = g.n_stages;
  const uint32_t ring_s = smem_u32(ring);
  uint32_t issued = 0;
  int st = 0;
  uint32_t par = 0;
  bool grid_waited = !g.pdl;
  int routed_layer = -1;
  int seq = 0;  // instructions of this launch before the current one (consumer order)
  unsigned long long issued_bytes = 0;
  L2Cursor<HT, D, NB, WB> l2;
  const int qid = queue_id(g);
  int t = 0;               // step of this launch: the queue runs once per step
  uint32_t ep = g.epoch;   // its epoch
  bool step_ready = true;  // this step's copies may read rows written by earlier steps
  for (int pc = 0;; pc++) {
    Instr I;
    if (pc < g.max_pc) I = load_instr(g, qid, pc);
    if (pc >= g.max_pc || I.op == OP_HALT) {
      if (++t >= g.n_steps) break;
      pc = -1;
      ep = g.epoch + (uint32_t)t;
      routed_layer = -1;
      step_ready = false;
      continue;
    }
    if (I.op == OP_NOP) continue;
    if (g.stress_ns) {
      if (lane == 0) stress_delay(g, qid, pc, t, 0x5EEDu);
      __syncwarp();
    }
    // every branch below is warp-uniform: lane 0 decides, the warp follows
    // (errors elsewhere in the grid are seen in the bounded waits below)
    const bool routed = I.op == OP_MLP && g.E > 0 && !(I.flags & F_SHARED);
    if ((I.op == OP_ATTN || routed) && !grid_waited) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      grid_waited = true;
    }
    if (I.op == OP_ATTN && !step_ready) {
      // the cache rows that earlier steps of this launch appended come
      // through the ring: wait until the previous step is done (its argmax
      // is out), then order their generic stores before the bulk copies
      bool ok = true;
      if (lane == 0) {
        ok = wait_counter(g, g.lm_done_ctr, ep - 1u, pc, I.op);
        if (ok) asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) goto drain;
      step_ready = true;
    }
    if (I.op == OP_ATTN) {
      const int P = __shfl_sync(0xFFFFFFFFu, __ldg(g.positions + I.b), 0) + t;
      if (P < 0 || P >= g.max_ctx) {
        if (lane == 0) set_err(g, MK_ERR_INVALID_ARG, pc, I.op);
        goto drain;
      }
      if (lane == 0) ppos[I.b] = P;
    }
    if (routed && routed_layer != I.layer) {
      bool ok = true;
      if (lane == 0) ok = wait_counter(g, I.wait_ctr, ep * I.wait_cnt, pc, I.op);
      if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) goto drain;
      __syncwarp();
      if (lane < g.K) {  // the routing published by the layer's last router
        const int e = __ldcg(g.routes + (size_t)I.layer * g.K + lane);
        ptopk[lane] = min(max(e, 0), g.E - 1);
        ptopw[lane] = __ldcg(g.rweight + (size_t)I.layer * g.K + lane);
      }
      __syncwarp();
      routed_layer = I.layer;
    }
    __syncwarp();
    Seg s[2];
    const int nseg = get_segs<HT, D, WB, NB>(g, I, ppos, ptopk, s);
    const int my_seq = seq++;
    if constexpr (NB > 8) {
      // wide batch: the operand pieces are this step's input, written with
      // generic stores by other SMs -- wait for the dependency, then order
      // those stores before the bulk copies that read them
      if (nseg > 0 && s[0].wide() && s[0].unit2() && I.wait_ctr != NO_CTR) {
        bool ok = true;
        if (lane == 0) {
          ok = wait_counter(g, I.wait_ctr, ep * I.wait_cnt, pc, I.op);
          if (ok) asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) goto drain;
      }
    }
    // a held instruction: stages from hold_k on wait until the consumers
    // have finished (and signalled) every earlier instruction of this launch
    const uint32_t hold_k =
        (I.flags & F_HOLD) ? (uint32_t)(g.hold_early / (unsigned)g.stage_bytes) : 0xFFFFFFFFu;
    auto held_back = [&]() { return *(volatile const int*)done < my_seq; };
    uint32_t nst_i = 0;  // stages of this instruction issued so far
    for (int k = 0; k < nseg; k++) {
      for (uint32_t u0 = 0; u0 < s[k].n; u0 += s[k].ups) {
        const uint32_t n = min(s[k].ups, s[k].n - u0);
        if (nst_i++ == hold_k) {
          int bad = 0;
          if (lane == 0) {
            const uint64_t t0 = gtimer();
            for (uint32_t it = 1; held_back(); it++) {
              if ((it & 63) == 0) {
                if (peek_err(g)) {
                  bad = 1;
                  break;
                }
                if (gtimer() - t0 > g.timeout_ns) {
                  set_err(g, MK_ERR_TIMEOUT, pc, I.op);
                  bad = 1;
                  break;
                }
              }
            }
          }
          if (__shfl_sync(0xFFFFFFFFu, bad, 0)) goto drain;
        }
        // wait for a free stage; while the ring is full, warm L2 ahead
        const uint32_t empty = empty0 + 8u * st;
        if (!__shfl_sync(0xFFFFFFFFu, mbar_try(empty, par ^ 1u), 0)) {
          const uint64_t t0 = gtimer();
          for (uint32_t it = 1;; it++) {
            if (g.l2_ahead)
              l2.run(g, issued_bytes + g.l2_ahead, issued_bytes, ptopk, routed_layer, 1);
            if (__shfl_sync(0xFFFFFFFFu, mbar_try(empty, par ^ 1u), 0)) break;
            if ((it & 63) == 0) {
              int bad = 0;
              if (lane == 0) {
                if (peek_err(g)) {
                  bad = 1;
                } else if (gtimer() - t0 > g.timeout_ns) {
                  set_err(g, MK_ERR_TIMEOUT, pc, I.op);
                  bad = 1;
                }
              }
              if (__shfl_sync(0xFFFFFFFFu, bad, 0)) goto drain;
            }
          }
        }
#ifdef MK_BOUNDS
        {  // the stage (or each half) must hold what the segment puts there
          const uint32_t room = s[k].src2 ? (uint32_t)g.stage_bytes / 2 : (uint32_t)g.stage_bytes;
          const bool fits = (NB > 8 && s[k].wide())
                                ? n * (s[k].unit + s[k].unit2()) <= (uint32_t)g.stage_bytes
                                : n * s[k].unit <= room;
          int bad = 0;
          if (lane == 0 && !MK_IN(g, fits, pc, I.op)) bad = 1;
          if (__shfl_sync(0xFFFFFFFFu, bad, 0)) goto drain;
        }
#endif
        if (lane == 0) {
          if (g.trace && k == 0 && u0 == 0)
            g.trace[((size_t)qid * g.max_pc + pc) * 8] = gtimer();
          const uint32_t bytes = n * s[k].unit;
          const uint32_t full = full0 + 8u * st;
          const uint32_t dst = ring_s + (uint32_t)st * (uint32_t)g.stage_bytes;
          const bool wseg = NB > 8 && s[k].wide();
          if (wseg) {
            // chunk j: its weight piece at j * unit; the stage's operand
            // pieces (if the operand is streamed; unit2 > 0) are contiguous
            // at both ends, one copy to ups * unit
            const uint32_t u2 = s[k].unit2();
            mbar_expect_tx(full, n * (s[k].unit + u2));
            if (u2)
              bulk_g2s(dst + s[k].ups * s[k].unit,
                       copy_src(g, I, s[k].src2 + (size_t)u0 * u2, n * u2, pc), n * u2, full, pol_kv);
            for (uint32_t j = 0; j < n; j++)
              bulk_g2s(dst + j * s[k].unit,
                       copy_src(g, I, s[k].src + (size_t)(u0 + j) * s[k].pitch(), s[k].unit, pc),
                       s[k].unit, full, pol_w);
          } else if (attn_tc_path<D, HPG, NB>() && g.tmaps && I.op == OP_ATTN && !g.kv_block) {
            // tensor-core attention: the K and V rows as tiled TMA boxes of
            // 64 rows in the 128-byte swizzle (the box past the item's last
            // row loads neighbouring rows, or zeros past the cache's end)
            const uint32_t nbox = (n + 63u) / 64u;
            mbar_expect_tx(full, 2u * nbox * 8192u);
            const LayerPtrs* Lp = g.layers + I.layer;
            const int row = (int)((s[k].src - (const unsigned char*)Lp->kc) / 128) + (int)u0;
            const unsigned char* tm = (const unsigned char*)g.tmaps + (size_t)I.layer * 256;
            for (uint32_t x = 0; x < nbox; x++) {
              tma_load_2d(dst + 8192u * x, tm, 0, row + 64 * (int)x, full, pol_kv);
              tma_load_2d(dst + (uint32_t)g.stage_bytes / 2 + 8192u * x, tm + 128, 0,
                          row + 64 * (int)x, full, pol_kv);
            }
          } else {
            mbar_expect_tx(full, s[k].src2 ? 2u * bytes : bytes);
          }
          if (wseg || (attn_tc_path<D, HPG, NB>() && g.tmaps && I.op == OP_ATTN && !g.kv_block)) {
            // issued above
          } else if (s[k].cfill()) {
            // the consumers copy this stage in after their dependency wait
          } else if (s[k].src2 && g.kv_block && I.op == OP_ATTN) {
            // paged cache: the stage's rows, one copy per block piece (K in
            // the lower half, V in the upper)
            const LayerPtrs* Lp = g.layers + I.layer;
            const int P = ppos[I.b];
            const int p0 = (int)((long)(P + 1) * I.r0 / I.r1) + (int)u0;
            for (int r = p0; r < p0 + (int)n;) {
              const int re = min(p0 + (int)n, (r / g.kv_block + 1) * g.kv_block);
              long long off = kv_row(g, I.b, I.g, r);
              if (off < 0) {  // a block outside the pool: fail the step, still fill the stage
                set_err(g, MK_ERR_INVALID_ARG, pc, I.op);
                off = 0;
              }
              const uint32_t pb = (uint32_t)(re - r) * (uint32_t)(D * 2);
              const uint32_t at = (uint32_t)(r - p0) * (uint32_t)(D * 2);
              bulk_g2s(dst + at, copy_src(g, I, (const unsigned char*)(Lp->kc + off), pb, pc), pb, full,
                       pol_kv);
              bulk_g2s(dst + (uint32_t)g.stage_bytes / 2 + at,
                       copy_src(g, I, (const unsigned char*)(Lp->vc + off), pb, pc), pb, full, pol_kv);
              r = re;
            }
          } else if (s[k].src2) {
            bulk_g2s(dst, copy_src(g, I, s[k].src + (size_t)u0 * s[k].unit, bytes, pc), bytes, full,
                     pol_kv);
            bulk_g2s(dst + (uint32_t)g.stage_bytes / 2,
                     copy_src(g, I, s[k].src2 + (size_t)u0 * s[k].unit, bytes, pc), bytes, full, pol_kv);
          } else {
            bulk_g2s(dst, copy_src(g, I, s[k].src + (size_t)u0 * s[k].unit, bytes, pc), bytes, full,
                     pol_w);
          }
        }
        issued_bytes += (NB > 8 && s[k].wide()) ? (unsigned long long)n * (s[k].unit + s[k].unit2())
                                                 : (s[k].src2 ? 2ull : 1ull) * n * s[k].unit;
        __syncwarp();
        issued++;
        if (++st == ns) {
          st = 0;
          par ^= 1u;
        }
      }
    }
  }
  return;
drain:
  // The latest arming of each stage is among the last ns issued; wait for
  // those copies to land so that no bulk copy outlives the CTA.
  if (lane != 0) return;
  for (uint32_t k = 1; k <= issued && k <= (uint32_t)ns; k++) {
    const uint32_t j = issued - k;
    wait_mbar(g, full0 + 8u * (j % (uint32_t)ns), (j / (uint32_t)ns) & 1u, false);
  }
}

template <int HT, int D, int HPG, int NB, int WB>
MK_DEV void consumer_steps(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, int* misc);

template <int HT, int D, int HPG, int NB, int WB>
__global__ void __launch_bounds__(NTHREADS, 1) mk_decode_kernel(const __grid_constant__ Globals g) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const SmemLayout Ls = smem_layout(g.n_stages, g.stage_bytes, NB, HT, D, HPG, g.K, WB);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t full0 = smem_u32(smem + Ls.full), empty0 = smem_u32(smem + Ls.empty);
  const int KM = g.K > 0 ? g.K : 1;
  int* misc = (int*)(smem + Ls.misc);
  int* flag = misc;
  int* tok = misc + 8;
  int* pos = tok + NB;
  int* topk = pos + NB;
  int* ptopk = topk + NB * KM;
  float* topw = (float*)(ptopk + NB * KM);
  float* ptopw = topw + NB * KM;
  int* ppos = (int*)(ptopw + NB * KM);
  if (tid == 0) {
    for (int s = 0; s < g.n_stages; s++) {
      mbar_init(full0 + 8u * s, 1u);
      mbar_init(empty0 + 8u * s, (uint32_t)NCW);
    }
    if constexpr (NB > 8) mbar_init(smem_u32(smem + Ls.tcw + 8), (uint32_t)WIDE_NI);  // MMA done
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    *flag = 0;
    misc[1] = 0;  // instructions the consumers have finished (read by the producer)
    misc[3] = misc[4] = 0;  // dependency-wait keys (never 0 once in use)
  }
  __syncthreads();

  if (warp == NCW) {
    producer<HT, D, HPG, NB, WB>(g, smem + Ls.ring, full0, empty0, ppos, ptopk, ptopw, misc + 1,
                             lane);
    return;
  }

  // ---- consumers
  if (g.pdl) asm volatile("griddepcontrol.wait;" ::: "memory");
  Ctx<HT, D, HPG, NB, WB> c;
  c.xn = (float*)(smem + Ls.xn);
  c.yrow = (float*)(smem + Ls.yrow);
  c.hbuf = (float*)(smem + Ls.hbuf);
  c.mpart = (float*)(smem + Ls.mpart);
  c.attn = (float*)(smem + Ls.attn);
  c.red = (float*)(smem + Ls.red);
  c.sc = WB == 1 ? (float*)(smem + Ls.sc) : nullptr;
  c.tok = tok;
  c.pos = pos;
  c.topk = topk;
  c.topw = topw;
  c.ring = Ring{smem + Ls.ring, full0, empty0, g.n_stages, 0, 0u, 0ull, g.trace != nullptr,
                (uint32_t)g.stage_bytes};
  c.tid = tid;
  c.warp = warp;
  c.lane = lane;
  c.flag = flag;
  c.tw0 = c.tw1 = 0;
  c.tm[0] = c.tm[1] = 0;
  c.tmem = c.mma_bar = c.mma_par = 0;
  if constexpr (NB > 8) {
    // wide batch: the accumulators' tensor memory, held for the whole kernel
    c.mma_bar = smem_u32(smem + Ls.tcw + 8);
    if (warp == 0) tmem_alloc(smem_u32(smem + Ls.tcw), (uint32_t)WIDE_TMEM_COLS);
    tc_fence_before();
    consumer_bar();
    tc_fence_after();
    c.tmem = *(volatile uint32_t*)(smem + Ls.tcw);
  }
  consumer_steps(c, g, misc);
  if constexpr (NB > 8) {
    // every exit: once the MMAs issued so far have completed (each issuing
    // warp commits; a commit with none outstanding arrives at once), warp 0
    // frees the tensor memory
    tc_fence_before();
    consumer_bar();
    if (warp < WIDE_NI && lane == 0) tc_commit(c.mma_bar);
    if (warp == 0) {
      if (lane == 0) wait_mbar(g, c.mma_bar, c.mma_par, false);
      __syncwarp();
      tc_fence_after();
      tmem_dealloc(c.tmem, (uint32_t)WIDE_TMEM_COLS);
    }
  }
}

// The consumer warps' work: every step of the launch, every instruction of
// the CTA's queue, in order.  Returns on completion or on the first failure
// (the error word is set by then).
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV void consumer_steps(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, int* misc) {
  const int tid = c.tid;
  int* flag = c.flag;
  int* tok = c.tok;
  int* pos = c.pos;
  int finished = 0;
  const int qid = queue_id(g);
  for (int step = 0; step < g.n_steps; step++) {
    c.step = step;
    c.epoch = g.epoch + (uint32_t)step;
    if (step > 0) {
      // step t decodes step t - 1's argmax, once every SM is done with
      // step t - 1 (its argmax is out)
      if (tid == 0) *flag = wait_counter(g, g.lm_done_ctr, c.epoch - 1u, -1, OP_LMHEAD) ? 0 : 2;
      consumer_bar();
      if (*flag) return;  // the error word is set
    }
    if (tid < g.B && tid < NB) {
      const int t = step == 0 ? g.tokens[tid] : __ldcg(g.argmax + (size_t)(step - 1) * g.B + tid);
      const int p = g.positions[tid] + step;
      tok[tid] = t;
      pos[tid] = p;
      if (t < 0 || t >= g.V || p < 0 || p >= g.max_ctx) *flag = 1;
    }
    consumer_bar();
    if (*flag) {
      if (tid == 0) set_err(g, MK_ERR_INVALID_ARG, -1, -1);
      return;
    }
    if (step == 0 && g.pdl && tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    consumer_bar();  // everyone has read *flag before it is reused

    Instr next = load_instr(g, qid, 0);
    for (int pc = 0; pc < g.max_pc; pc++) {
      const Instr I = next;
      if (I.op == OP_HALT) break;
      if (pc + 1 < g.max_pc) next = load_instr(g, qid, pc + 1);
      if (I.op == OP_NOP) continue;
      c.pc = pc;
      // race stress: thread 0 starts late; the op's dependency wait holds the rest
      if (g.stress_ns && tid == 0) stress_delay(g, qid, pc, step, 0xC0DEu);
      bool ok;
      if constexpr (NB > 8) {
        switch (I.op) {
          case OP_NORM: ok = op_norm_wide(c, g, I); break;
          case OP_QKV: ok = op_qkv_wide(c, g, I); break;
          case OP_ATTN: ok = op_attn(c, g, I); break;
          case OP_OPROJ: ok = op_oproj_wide(c, g, I); break;
          case OP_MLP_UP: ok = op_mlp_up_wide(c, g, I); break;
          case OP_MLP_DOWN: ok = op_mlp_down_wide(c, g, I); break;
          case OP_LMHEAD: ok = op_lmhead_wide(c, g, I); break;
          default:
            if (tid == 0) set_err(g, MK_ERR_DEVICE, pc, I.op);
            ok = false;
            break;
        }
      } else {
        switch (I.op) {
          case OP_QKV: ok = op_qkv(c, g, I); break;
          case OP_ATTN: ok = op_attn(c, g, I); break;
          case OP_OPROJ: ok = op_oproj(c, g, I); break;
          case OP_ROUTER: ok = op_router(c, g, I); break;
          case OP_MLP: ok = op_mlp(c, g, I); break;
          case OP_MLP_UP: ok = op_mlp_up(c, g, I); break;
          case OP_MLP_DOWN: ok = op_mlp_down(c, g, I); break;
          case OP_LMHEAD: ok = op_lmhead(c, g, I); break;
          default:
            if (tid == 0) set_err(g, MK_ERR_DEVICE, pc, I.op);
            ok = false;
            break;
        }
      }
      if (!ok) return;
      if (tid == 0) {
        if (g.trace) {
          unsigned long long* t = g.trace + ((size_t)qid * g.max_pc + pc) * 8;
          t[1] = c.tw0;
          t[2] = c.tw1;
          t[3] = c.tm[0];
          t[4] = c.tm[1];
          t[5] = gtimer();
          t[6] = c.ring.waited;  // warp 0's time blocked on ring data during this instruction
          c.ring.waited = 0;
        }
        if (I.sig_ctr != NO_CTR && I.op != OP_ROUTER) {  // routers: the last arriver signals
          if (I.flags & F_RELAXED_SIG)
            red_relaxed(g.ctr + I.sig_ctr, 1u);
          else
            red_release(g.ctr + I.sig_ctr, 1u);
        }
        if (g.trace) g.trace[((size_t)qid * g.max_pc + pc) * 8 + 7] = gtimer();
        *(volatile int*)(misc + 1) = ++finished;
      }
    }
  }  // steps
}

}  // namespace mk
