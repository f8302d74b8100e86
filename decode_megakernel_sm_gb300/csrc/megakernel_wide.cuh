// megakernel_wide.cuh -- op bodies of the wide-batch variant (2 .. 32
// sequences on the shapes it takes, see wide_path), included by
// megakernel.cuh.
//
// Every contraction runs on the fifth-generation tensor cores: elected
// threads issue tcgen05.mma (kind::f16, bf16 x bf16 -> f32) with A = 128
// weight rows of a ring stage and B = the activation operand, 2 Bp rows: the
// bf16 high part of sequence b's activation in row 2b and the bf16 remainder
// in row 2b + 1, so that the two products together keep about 16 mantissa
// bits of the activation ("Megakernels in LLM Inference When Fusion
// Actually Wins", sections "Core Tradeoff" and "When Megakernels Win": the
// batch range where the contraction turns from a GEMV into a skinny GEMM).
// Consumer warps 0 .. WIDE_NI - 1 each issue the MMAs of every WIDE_NI-th K
// chunk into an accumulator of their own in tensor memory (64 columns each,
// allocated once per CTA for the life of the kernel); consumer warps 0-3 read
// them back with tcgen05.ld, one accumulator row (one weight row) per
// thread, sum the accumulators and add the high and low columns of each
// sequence.
//
// A stage is released to the producer by a tcgen05.commit of each issuing
// warp on its empty barrier (that warp's arrival), which fires once the
// warp's MMAs have read it; the other consumer warps arrive as usual.  The
// accumulators are complete when each issuing warp's commit on the CTA's
// MMA-done barrier has fired.
#pragma once
#include "mk_tc.cuh"

namespace mk {

// bf16 high part and remainder of x (x = hi + lo to about 16 mantissa bits).
MK_DEV void split_hl8(const float (&x)[8], uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; i++) split2(x[2 * i], x[2 * i + 1], h[i], l[i]);
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// Byte offset of (operand row, column k) in an operand buffer of K chunks:
// chunk k / 64 is a tile of 2 Bp rows x 64 columns (ab bytes).
MK_DEV size_t opnd_off(uint32_t ab, uint32_t row, uint32_t k) {
  return (size_t)(k / WIDE_KC) * ab + sw128_off(row, k % WIDE_KC);
}

// Wait for the MMAs committed so far on the MMA-done barrier (all consumer
// threads; bounded).  False if the wait gave up.  The wait does not give up
// on an error elsewhere in the grid: the committed MMAs complete regardless,
// so every thread returns the same value and the warps leave the op together
// (the next dependency wait sees the error).
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool wide_mma_wait(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g) {
  const bool ok = wait_mbar(g, c.mma_bar, c.mma_par, false);
  c.mma_par ^= 1u;
  tc_fence_after();
  return ok;
}

// Stream a wide segment through the ring into the accumulators: chunk by
// chunk, D_w (+)= W_chunk (128 rows from the weight piece) x operand_chunk^T,
// where consumer warp w < WIDE_NI issues (lane 0) the MMAs of chunks i with
// i % WIDE_NI == w into its own accumulator at column 64 w and releases each
// stage with a commit once its MMAs have read it; wide_tile_out sums the
// accumulators.  Rows past the piece's own read the bytes that follow it (the
// rest of the stage, or the shared memory after the ring); their outputs are
// never read.  All consumer warps call; false (on every thread) if a ring
// wait gave up.
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool wide_mma_stream(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Seg& s) {
  const uint32_t N = s.unit2() / 128u;
  const uint32_t idesc = idesc_bf16(128, (int)N);
  const uint32_t NI = (uint32_t)WIDE_NI;
  bool bad = false, first = true;  // first: this warp's accumulator not written yet
  for (uint32_t u0 = 0; u0 < s.n; u0 += s.ups) {
    uint32_t n = min(s.ups, s.n - u0);
    if (!MK_IN(g, n * (s.unit + s.unit2()) <= (uint32_t)g.stage_bytes, c.pc, -1)) n = 0;
    if (!bad && !c.ring.acquire(g)) bad = true;
    if (bad) continue;
    if ((uint32_t)c.warp < NI) {
      // warp w: the stage's chunks u0 + j with (u0 + j) % NI == w
      if (c.lane == 0) {
        tc_fence_after();
        const uint32_t sb = smem_u32(c.ring.stage_ptr());
        const uint32_t acc = c.tmem + 64u * (uint32_t)c.warp;
        for (uint32_t j = ((uint32_t)c.warp + NI - u0 % NI) % NI; j < n; j += NI) {
          const uint32_t wa = sb + j * s.unit, aa = sb + s.ups * s.unit + j * s.unit2();
#pragma unroll
          for (uint32_t k = 0; k < 4; k++)
            tc_mma_bf16(acc, sw128_desc(wa + 32u * k), sw128_desc(aa + 32u * k), idesc,
                        !first || k > 0);
          first = false;
        }
        tc_commit(c.ring.empty_bar());  // the warp's arrival, once its MMAs have read the stage
      }
      __syncwarp();
      c.ring.advance();
    } else {
      c.ring.release(c.lane);
    }
  }
  if (bad) c.flag[2] = 1;
  consumer_bar();
  if (c.flag[2]) return false;
  if ((uint32_t)c.warp < NI && c.lane == 0) tc_commit(c.mma_bar);  // WIDE_NI arrivals
  return wide_mma_wait(c, g);
}

// Accumulators a segment writes: one per issuing warp that has a chunk.
MK_DEV uint32_t wide_nacc(const Seg& s) { return min((uint32_t)WIDE_NI, s.n); }

// Read the accumulators back (128 weight rows, N = 2 Bp columns each; nacc
// of them written, wide_nacc) into yrow[b][m], b < Bp, m < 128: consumer warp
// w < 4 reads lanes 32 w .. 32 w + 31, sums the accumulators and adds each
// sequence's high and low columns.  Ends with the
// tensor-memory reads ordered before a CTA barrier, after which yrow is
// complete (and the next MMAs may overwrite the accumulator).
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV void wide_tile_out(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, uint32_t N, uint32_t nacc) {
  static_assert(NB <= 32, "64 accumulator columns per tile");
  if (c.warp < 4) {
    float* y = c.yrow + 32 * c.warp + c.lane;
    for (uint32_t q = 0; 16u * q < N; q++) {  // 16 columns: sequences 8q .. 8q + 7
      float v[16], w[16];
      const uint32_t ta = c.tmem + ((uint32_t)(32 * c.warp) << 16) + 16u * q;
      tmem_ld16(ta, v);
      for (uint32_t a = 1; a < nacc; a++) {  // the other issuers' accumulators
        tmem_ld16(ta + 64u * a, w);
#pragma unroll
        for (int e = 0; e < 16; e++) v[e] += w[e];
      }
#pragma unroll
      for (int e = 0; e < 8; e++) y[(8 * q + e) * WIDE_ROWS] = v[2 * e] + v[2 * e + 1];
    }
  }
  tc_fence_before();
  consumer_bar();
}

// ------------------------------------------- OP_NORM (operand of a GEMV) ----
// Sequences [r0, r1) of x_j -> rows 2b, 2b + 1 of operand buffer I.g (0: the
// QKV input, x_{2l} with the attention-norm gain; 1: the MLP input, x_{2l+1}
// with the MLP-norm gain; 2: the LM head's input, x_{2L} with the final
// gain).  Sequences b >= B (up to Bp) get zero rows.
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool op_norm_wide(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Instr& I) {
  constexpr int GROUPS = HT / 8, GPT = (GROUPS + NCT - 1) / NCT;
  const int which = I.g, l = I.layer;
  const int j = which == 0 ? 2 * l : which == 1 ? 2 * l + 1 : 2 * g.L;
  const uint16_t* gain = which == 2 ? g.final_norm
                                    : (which == 0 ? g.layers[l].attn_norm : g.layers[l].mlp_norm);
  uint4 gw[GPT];
#pragma unroll
  for (int q = 0; q < GPT; q++) {
    const int gi = c.tid + q * NCT;
    gw[q] = gi < GROUPS ? __ldg((const uint4*)gain + gi) : make_uint4(0, 0, 0, 0);
  }
  if (!dep_wait(c, g, I)) return false;
  const uint32_t ab = 2u * (uint32_t)g.Bp * 128u;
  unsigned char* out = g.act + (size_t)which * (HT / WIDE_KC) * ab;
  for (int b = (int)I.r0; b < (int)I.r1; b++) {
    float v[GPT][8];
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < GPT; q++) {
      const int gi = c.tid + q * NCT;
#pragma unroll
      for (int e = 0; e < 8; e++) v[q][e] = 0.f;
      if (gi >= GROUPS || b >= g.B) continue;
      if (j == 0) {  // embedding rows are chunk-swizzled by token id
        const int tk = c.tok[b];
        unpack8(__ldg((const uint4*)(g.embed + (size_t)tk * HT) + (gi ^ (tk & 7))), v[q]);
      } else {
        for (int cp = 0; cp < g.kc; cp++) {
          const float4* p = (const float4*)xres(g, c.epoch, j, b, cp) + 2 * gi;
          const float4 a0 = __ldcg(p), a1 = __ldcg(p + 1);
          v[q][0] += a0.x; v[q][1] += a0.y; v[q][2] += a0.z; v[q][3] += a0.w;
          v[q][4] += a1.x; v[q][5] += a1.y; v[q][6] += a1.z; v[q][7] += a1.w;
        }
      }
#pragma unroll
      for (int e = 0; e < 8; e++) ss = fmaf(v[q][e], v[q][e], ss);
    }
    ss = warp_sum(ss);
    if (c.lane == 0) c.red[c.warp] = ss;
    consumer_bar();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < NCW; w++) t += c.red[w];
    const float rs = rsqrtf(t / (float)HT + g.eps);
#pragma unroll
    for (int q = 0; q < GPT; q++) {
      const int gi = c.tid + q * NCT;
      if (gi >= GROUPS) continue;
      float gf[8], x[8];
      unpack8(gw[q], gf);
#pragma unroll
      for (int e = 0; e < 8; e++) x[e] = b < g.B ? v[q][e] * rs * gf[e] : 0.f;
      uint4 hi, lo;
      split_hl8(x, hi, lo);
      *(uint4*)(out + opnd_off(ab, 2u * b, 8u * gi)) = hi;
      *(uint4*)(out + opnd_off(ab, 2u * b + 1u, 8u * gi)) = lo;
    }
    consumer_bar();  // c.red is reused by the next sequence
  }
  return true;
}

// ------------------------------------------------- OP_QKV (wide batch) ----
// Rows [r0, r1) (at most 128, starting on a multiple of 8) of kv head I.g's
// packed QKV rows; then RoPE on the (t, t + D/2) pairs of q and k, q to the
// query buffer, k and v appended to the cache at each sequence's position.
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool op_qkv_wide(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Instr& I) {
  const LayerPtrs& Lp = g.layers[I.layer];
  if (!dep_wait(c, g, I)) return false;
  c.mark(g, 0);
  Seg s[2];
  get_segs<HT, D, WB, NB>(g, I, c.pos, c.topk, s);
  if (!wide_mma_stream(c, g, s[0])) return false;
  c.mark(g, 1);
  const uint32_t n = I.r1 - I.r0;
  float* yrow = c.yrow;  // [NB][WIDE_ROWS]
  wide_tile_out(c, g, s[0].unit2() / 128u, wide_nacc(s[0]));
  constexpr int GR = (HPG + 2) * D;
  const int np = (int)n / 2;
  for (int it = c.tid; it < np * g.B; it += NCT) {
    const int b = it / np, i = 2 * (it % np);
    float y0 = yrow[b * WIDE_ROWS + i], y1 = yrow[b * WIDE_ROWS + i + 1];
    const int lr = (int)(I.r0 + i) - (int)I.g * GR;
    const int hs = lr / D, t = (lr % D) >> 1;
    const int P = c.pos[b];
    if (hs <= HPG) {  // q heads and k: rotate (t, t + D/2) by P * theta^(-2t/D)
      const float2 cs = ((const float2*)g.rope)[(size_t)P * (D / 2) + t];
      const float a = y0 * cs.x - y1 * cs.y;
      const float bb = y0 * cs.y + y1 * cs.x;
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
        set_err(g, MK_ERR_INVALID_ARG, c.pc, I.op);
      } else if (MK_IN(g, (size_t)off + D <= g.kv_elems, c.pc, I.op)) {
        uint16_t* row = (hs == HPG ? Lp.kc : Lp.vc) + off;
        row[t] = to_bf16(y0);
        row[t + D / 2] = to_bf16(y1);
      }
    }
  }
  consumer_bar();
  return true;
}

// The rows [r0, r1) of yrow (one per weight row; r0 and r1 - r0 multiples of
// 8) added into the residual x_out with 16-byte float reductions, four rows
// of one sequence each; with `resid`, the instruction also adds x_in of its
// rows (the residual input of the phase).
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV void wide_residual_add(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Instr& I,
                              int j_in, int j_out, bool resid) {
  const int n4 = (int)(I.r1 - I.r0) / 4;
  for (int it = c.tid; it < g.B * n4; it += NCT) {
    const int b = it / n4, m = 4 * (it % n4);
    const int row = (int)I.r0 + m;
    const float* y = c.yrow + b * WIDE_ROWS + m;
    float v[4] = {y[0], y[1], y[2], y[3]};
    if (resid)
#pragma unroll
      for (int e = 0; e < 4; e++) v[e] += x_in(g, c.epoch, j_in, c.tok, b, row + e);
    float* dst = xres_mine(g, c.epoch, j_out, b);
    if (MK_IN(g, (size_t)(dst - g.xbuf) + row + 4 <= g.n_xbuf, c.pc, I.op))
      red_add_v4f32(dst + row, v[0], v[1], v[2], v[3]);
  }
  consumer_bar();
}

// ------------------------------------- attention merge (wide batch) ----
// After an attention item has written its partial (o, m, l) records: count
// the item in for its (layer, sequence, kv head); the item that arrives last
// merges the S slices of each of the group's query heads (M = max m_s,
// L = sum l_s 2^(m_s - M), o = sum o_s 2^(m_s - M) / L) and writes the heads'
// outputs, bf16 high part and remainder, as rows 2b, 2b + 1 of their chunks
// of the O-projection's operand buffer.  Its completion signal (a release)
// follows, so a met attention counter means merged outputs.
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool attn_merge_wide(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Instr& I) {
  const int b = I.b, S = (int)I.r1;
  constexpr int PS = part_stride(D);
  if (S == 1) return true;  // (a whole-sequence item wrote its outputs itself: attn_cta_merge)
  if (c.tid == 0) {
    uint32_t* arr = g.ctr + g.arr_ctr + ((size_t)I.layer * g.B + b) * g.Hkv + I.g;
    const uint32_t old = atom_add_acq_rel(arr, 1u);
    c.flag[6] = old == c.epoch * (uint32_t)S - 1u;
  }
  consumer_bar();
  const bool last = c.flag[6] != 0;
  if (!last) return true;
  const uint32_t ab = 2u * (uint32_t)g.Bp * 128u;
  unsigned char* out = g.act + 3 * (size_t)(HT / WIDE_KC) * ab;
  for (int t = c.tid; t < HPG * D; t += NCT) {
    const int h = t / D, dim = t % D, hq = I.g * HPG + h;
    const size_t r = (((size_t)I.layer * g.B + b) * g.Hq + hq) * S;
    float M = NEG_BIG, Ls = 0.f, O = 0.f;
    if (MK_IN(g, (r + S) * PS <= g.n_part, c.pc, I.op)) {
      for (int s2 = 0; s2 < S; s2++) {
        const float* p = g.part + (r + s2) * PS;
        const float ms = __ldcg(p + D), ls = __ldcg(p + D + 1), os = __ldcg(p + dim);
        const float mn = fmaxf(M, ms);
        const float fa = exp2f(M - mn), fb = exp2f(ms - mn);
        Ls = Ls * fa + ls * fb;
        O = O * fa + os * fb;
        M = mn;
      }
    }
    const float x = O / Ls;
    const uint16_t hi = to_bf16(x), lo = to_bf16(x - bf1(hi));
    *(uint16_t*)(out + opnd_off(ab, 2u * b, (uint32_t)(hq * D + dim))) = hi;
    *(uint16_t*)(out + opnd_off(ab, 2u * b + 1u, (uint32_t)(hq * D + dim))) = lo;
  }
  consumer_bar();
  return true;
}

// --------------------------------------------- OP_OPROJ (wide batch) ----
// Rows [r0, r1) (at most 128, from a multiple of 8) of Wo over kv group I.g's
// HPG * D columns, against the group's merged attention outputs (streamed
// with the weights, one K chunk per query head), added into x_{2l+1} with
// float reductions: one contribution per group and element rather than one
// per head.  The group-0 instructions also add x_{2l}.
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool op_oproj_wide(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Instr& I) {
  static_assert(D == WIDE_KC, "one head is one K chunk");
  const int l = I.layer;
  if (!dep_wait(c, g, I)) return false;
  c.mark(g, 0);
  Seg s[2];
  get_segs<HT, D, WB, NB>(g, I, c.pos, c.topk, s);
  if (!wide_mma_stream(c, g, s[0])) return false;
  c.mark(g, 1);
  wide_tile_out(c, g, s[0].unit2() / 128u, wide_nacc(s[0]));
  wide_residual_add(c, g, I, 2 * l, 2 * l + 1, (I.flags & F_RESIDUAL) != 0);
  return true;
}

// ---------------------------------------------- OP_MLP_UP (wide batch) ----
// FFN columns [r0, r1) (at most 64, starting on a multiple of 4): gate and up
// rows 2c, 2c + 1, then h = SiLU(gate) * up written into h's operand buffer
// (rows 2b, 2b + 1 of the column's chunk).
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool op_mlp_up_wide(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Instr& I) {
  if (!dep_wait(c, g, I)) return false;
  c.mark(g, 0);
  Seg s[2];
  get_segs<HT, D, WB, NB>(g, I, c.pos, c.topk, s);
  if (!wide_mma_stream(c, g, s[0])) return false;
  c.mark(g, 1);
  const int ncol = (int)(I.r1 - I.r0);
  float* yrow = c.yrow;  // [NB][WIDE_ROWS]
  wide_tile_out(c, g, s[0].unit2() / 128u, wide_nacc(s[0]));
  const uint32_t ab = 2u * (uint32_t)g.Bp * 128u;
  unsigned char* hb = (unsigned char*)g.hglob;
  for (int it = c.tid; it < ncol * g.Bp; it += NCT) {
    const int b = it / ncol, j = it % ncol;
    float h = 0.f;
    if (b < g.B) {
      const float gt = yrow[b * WIDE_ROWS + 2 * j], up = yrow[b * WIDE_ROWS + 2 * j + 1];
      h = (gt / (1.f + expf(-gt))) * up;
    }
    const uint16_t hi = to_bf16(h), lo = to_bf16(h - bf1(hi));
    const uint32_t col = I.r0 + (uint32_t)j;
    *(uint16_t*)(hb + opnd_off(ab, 2u * b, col)) = hi;
    *(uint16_t*)(hb + opnd_off(ab, 2u * b + 1u, col)) = lo;
  }
  consumer_bar();
  return true;
}

// -------------------------------------------- OP_MLP_DOWN (wide batch) ----
// Rows [r0, r1) (at most 128, starting on a multiple of 8) of x_{2l+2} over
// the FFN chunks [b, g) of h, added with float reductions; the instructions
// of chunk 0 also add the residual x_{2l+1}.
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool op_mlp_down_wide(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Instr& I) {
  const int l = I.layer;
  if (!dep_wait(c, g, I)) return false;
  c.mark(g, 0);
  Seg s[2];
  get_segs<HT, D, WB, NB>(g, I, c.pos, c.topk, s);
  if (!wide_mma_stream(c, g, s[0])) return false;
  c.mark(g, 1);
  wide_tile_out(c, g, s[0].unit2() / 128u, wide_nacc(s[0]));
  wide_residual_add(c, g, I, 2 * l + 1, 2 * l + 2, I.b == 0);
  return true;
}

// ----------------------------------------------- OP_LMHEAD (wide batch) ----
// Rows [r0, r1) (at most 128) of the LM head over the final operand: the
// logits and, per sequence, the first maximum of the rows, folded into the
// SM's running (max, lowest row) in shared memory.  An SM's LM-head
// instructions form one slice (aux): the first of them (I.b bit 0) starts the
// running maxima and zeroes the slice's share of the next step's residual
// buffers, the last (bit 1) writes the slice's values and joins the
// last-arriver argmax over all slices (lm_reduce).
template <int HT, int D, int HPG, int NB, int WB>
MK_DEV bool op_lmhead_wide(Ctx<HT, D, HPG, NB, WB>& c, const Globals& g, const Instr& I) {
  const bool first = (I.b & 1) != 0, last = (I.b & 2) != 0;
  if (g.zero_next && first) {  // as in op_lmhead, once per slice
    const size_t total = (size_t)2 * g.L * g.kc * g.B * g.H;
    const size_t a = total * I.aux / (size_t)g.n_lm, e = total * (I.aux + 1) / (size_t)g.n_lm;
    float* nx = g.xbuf + (size_t)((c.epoch + 1u) & 1u) * total;
    if (MK_IN(g, 2 * total <= g.n_xbuf, c.pc, I.op))
      for (size_t i = a + c.tid; i < e; i += NCT) nx[i] = 0.f;
  }
  if (!dep_wait(c, g, I)) return false;
  c.mark(g, 0);
  Seg s[2];
  get_segs<HT, D, WB, NB>(g, I, c.pos, c.topk, s);
  if (!wide_mma_stream(c, g, s[0])) return false;
  c.mark(g, 1);
  const int n = (int)(I.r1 - I.r0), B = g.B, V = g.V;
  float* yrow = c.yrow;  // [NB][WIDE_ROWS]
  wide_tile_out(c, g, s[0].unit2() / 128u, wide_nacc(s[0]));
  for (int it = c.tid; it < B * n; it += NCT) {
    const int b = it / n, m = it % n;
    const int row = (int)I.r0 + m;
    if (MK_IN(g, row < V, c.pc, I.op)) g.logits[(size_t)b * V + row] = yrow[b * WIDE_ROWS + m];
  }
  // this instruction's (max, lowest row) per sequence, folded into the SM's
  // running values: warp w takes sequences w, w + NCW, ...
  float* runv = c.red + 2 * NCW * NB + 4;
  int* runi = (int*)(runv + NB);
  for (int b = c.warp; b < B; b += NCW) {
    float best = -INFINITY;
    int bidx = 0x7FFFFFFF;
    for (int m = c.lane; m < n; m += 32) {
      const float y = yrow[b * WIDE_ROWS + m];
      if (y > best) {  // rows ascend along a lane: the first maximum wins
        best = y;
        bidx = (int)I.r0 + m;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, best, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bidx, o);
      if (ov > best || (ov == best && oi < bidx)) {
        best = ov;
        bidx = oi;
      }
    }
    if (c.lane == 0) {
      if (!first && (runv[b] > best || (runv[b] == best && runi[b] < bidx))) {
        best = runv[b];
        bidx = runi[b];
      }
      runv[b] = best;
      runi[b] = bidx;
      if (last && MK_IN(g, ((size_t)I.aux + 1) * B <= g.n_lmv, c.pc, I.op)) {
        g.lm_val[(size_t)I.aux * B + b] = best;
        g.lm_idx[(size_t)I.aux * B + b] = bidx;
      }
    }
  }
  consumer_bar();
  if (last) lm_reduce(c, g);
  return true;
}

}  // namespace mk
