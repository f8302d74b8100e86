// mk_internal.h -- records shared by the host planner, the C-ABI layer and the
// device interpreter.  Plain C++ (no CUDA types) so the planner builds with g++.
#pragma once
#include <stddef.h>
#include <stdint.h>

#include <vector>

#include "../../include/mk.h"

#ifdef __CUDACC__
#define MK_HD __host__ __device__
#else
#define MK_HD
#endif

namespace mk {

// Opcodes of the interpreter ("Megakernels: Deleting the Kernel Boundary",
// section "One launch, one interpreter", re-cut for GB300: the attention
// reduce is folded into the O-projection, up/gate and down are one
// instruction over an FFN column slice, ROUTER serves the MoE MLP).
enum Op : uint8_t {
  OP_HALT = 0,
  OP_QKV = 1,     // RMSNorm + QKV rows + RoPE + KV append
  OP_ATTN = 2,    // split-KV GQA partial softmax over a slice of positions
  OP_OPROJ = 3,   // split reduce + O-projection rows of one head + residual
  OP_MLP = 4,     // RMSNorm + gate/up rows + SiLU*mul + down columns + residual
  OP_LMHEAD = 5,  // final RMSNorm + LM-head rows + argmax (last arriver)
  OP_ROUTER = 6,  // MoE: RMSNorm + router rows
  OP_NOP = 7,     // does nothing (fault-injection stand-in)
  OP_MLP_UP = 8,  // RMSNorm + gate/up rows + SiLU*mul of an FFN column slice -> h (split MLP)
  OP_MLP_DOWN = 9,  // down-projection rows over the whole h + residual (split MLP)
  OP_NORM = 10,     // wide batch: RMSNorm of a range of sequences -> tensor-core operand
};

// Ablation phases: one launch per (layer, phase), each over queues that hold
// only that phase's instructions.  No instruction waits on a counter
// signalled by an instruction of its own phase.  (The wide-batch norms run
// before QKV and before the MLP; the final norm and the LM head are keyed
// to layer L.)
enum Phase : int {
  PH_NORM_A = 0, PH_QKV = 1, PH_ATTN = 2, PH_OPROJ = 3, PH_ROUTER = 4, PH_NORM_M = 5,
  PH_MLP = 6, PH_DOWN = 7, N_PHASES = 8
};

enum Flag : uint8_t {
  F_RESIDUAL = 1,    // this instruction also adds the residual input for its rows
  F_NORM_CACHED = 2, // the normalised input left in shared memory is still valid
  F_SHARED = 4,      // MoE MLP: shared-expert columns (weight 1, no routing)
  F_HOLD = 8,        // producer: issue at most hold_early bytes of this instruction's ring
                     // copies before the consumers have finished every earlier instruction
  F_TAG_WAIT = 16,   // inputs arrive as tagged words: poll them, not the wait counter
                     // (which still models the dependency for the schedule checker)
  F_RELAXED_SIG = 32,// every consumer polls tagged outputs: signal with a relaxed reduction,
                     // which does not wait for this SM's earlier memory operations
};

// Which instructions the planner marks F_HOLD (first of a run of the op on
// an SM).  A release fence waits for every memory operation the SM has in
// flight -- bulk copies and L2 prefetches included -- so the next
// instruction's copies issued in the last microseconds before a fence sit
// on the critical path.  A held instruction gets its first hold_early bytes
// of copies early (they land before the fence) and the rest right after the
// previous instruction's signal, while the dependency hop runs.
enum HoldBit : unsigned {
  HOLD_QKV = 1, HOLD_ATTN = 2, HOLD_OPROJ = 4, HOLD_MLP = 8, HOLD_DOWN = 16, HOLD_LM = 32,
};
// Default: the gate/up and down instructions, whose predecessors (O-proj and
// gate/up) end with the fences that have the most copies in flight behind them.
constexpr unsigned DEFAULT_HOLD = HOLD_MLP | HOLD_DOWN;
constexpr unsigned DEFAULT_HOLD_EARLY = 128u << 10;

constexpr uint32_t NO_CTR = 0xFFFFFFFFu;

using Instr = mk_instr;  // 32-byte record, layout fixed by mk.h
static_assert(sizeof(Instr) == 32, "instruction record must be 32 bytes");

MK_HD inline int phase_of(const Instr& I) {
  switch (I.op) {
    case OP_QKV: return PH_QKV;
    case OP_ATTN: return PH_ATTN;
    case OP_OPROJ: return PH_OPROJ;
    case OP_ROUTER: return PH_ROUTER;
    case OP_MLP_DOWN: return PH_DOWN;
    case OP_NORM: return I.g == 1 ? PH_NORM_M : PH_NORM_A;
    default: return PH_MLP;
  }
}

// Counter ids: per layer l, base l*stride:
//   qkv[g] (g < Hkv), attn[g], oproj, mlp, router, mlp_up, router arrivals;
//   then the argmax counter, the step counter, and (wide batch) norm_a and
//   norm_m of every layer and norm_f.
struct CtrMap {
  int Hkv, L;
  MK_HD int stride() const { return 2 * Hkv + 5; }
  MK_HD uint32_t qkv(int l, int g) const { return (uint32_t)(l * stride() + g); }
  MK_HD uint32_t attn(int l, int g) const { return (uint32_t)(l * stride() + Hkv + g); }
  MK_HD uint32_t oproj(int l) const { return (uint32_t)(l * stride() + 2 * Hkv); }
  MK_HD uint32_t mlp(int l) const { return (uint32_t)(l * stride() + 2 * Hkv + 1); }
  MK_HD uint32_t router(int l) const { return (uint32_t)(l * stride() + 2 * Hkv + 2); }
  MK_HD uint32_t mlp_up(int l) const { return (uint32_t)(l * stride() + 2 * Hkv + 3); }
  // router instructions arriving (not a dependency: the last arriver ranks
  // the logits, then signals router(l) on behalf of all of them)
  MK_HD uint32_t router_arrive(int l) const { return (uint32_t)(l * stride() + 2 * Hkv + 4); }
  MK_HD uint32_t lm() const { return (uint32_t)(L * stride()); }
  // one signal per step, by the LM head's last arriver once the step's
  // argmax is written: a multi-step launch starts step t + 1 behind it
  MK_HD uint32_t lm_done() const { return (uint32_t)(L * stride() + 1); }
  // wide batch: the normalised operand of QKV / of the MLP of layer l, and of
  // the LM head, is complete
  MK_HD uint32_t norm_a(int l) const { return (uint32_t)(L * stride() + 2 + 2 * l); }
  MK_HD uint32_t norm_m(int l) const { return (uint32_t)(L * stride() + 3 + 2 * l); }
  MK_HD uint32_t norm_f() const { return (uint32_t)(L * stride() + 2 + 2 * L); }
  MK_HD int count() const { return L * stride() + 3 + 2 * L; }
};

// Kernel-shape constants.
constexpr int NCW = 7;               // consumer warps (8 warps per CTA: two per scheduler partition, 255 registers)
constexpr int NCT = NCW * 32;        // consumer threads
constexpr int NTHREADS = NCT + 32;   // + one producer warp
// Ring stages are a runtime size: a multiple of STAGE_UNIT up to
// MAX_STAGE_BYTES (bigger stages hold more rows, so all consumer warps have a
// row in every stage and the per-stage barrier cost is spread wider).
constexpr int STAGE_UNIT = 16384;
constexpr int MAX_STAGE_BYTES = 65536;
constexpr int DEFAULT_STAGE_BYTES = 32768;
// The wide-batch variant's default: its consumer issues a tensor-core MMA per
// 16-deep K step of a chunk plus a commit per stage, and bigger stages hold
// more chunks per stage and per ring (a 128-row chunk with its operand takes
// 18-24 KB, so 32 KB stages leave a quarter to half of each unused).
constexpr int WIDE_STAGE_BYTES = 65536;
// The one-sequence bf16 default: a weight row of 4 KB fills a 32 KB stage
// with only 8 rows, so the 7 consumer warps take one or two rows each and
// wait on a stage hand-off for every 8 rows; 64 KB stages (three in the ring)
// halve those hand-offs.  Measured 0.8 % faster on a 1K cache and 2.3 % on
// an 8K cache; int8 handles (half the bytes per row) keep 32 KB, where 64 KB
// was 1.4 % slower, and so does the batched mma.sync variant (2.8 % slower).
constexpr int BATCH1_STAGE_BYTES = 65536;
constexpr int MAX_STAGES = 16;
constexpr int DOWN_ROW_MAX = 16384;  // bytes of one down row (F <= 8192) in the split MLP
constexpr int MAX_ROWS = 256;        // rows of one QKV / gate-up / router instruction
constexpr int MAX_COLS = MAX_ROWS / 2;
constexpr int MAX_DOWN_ROWS = 64;    // output rows of one split-MLP down instruction
// One split-KV partial record: o[D], m, l; for heads of 128+ dims padded to
// 16 bytes, so that an O-projection instruction can copy its head's partials
// of every sequence in one bulk copy per sequence (they must then fit the
// smallest ring stage).
MK_HD inline constexpr int part_stride(int D) { return D >= 128 ? D + 4 : D + 2; }
// The O-projection merges each (sequence, dim) of its head over the S slices
// with SG = NCT / (NB * D) threads, four slices' loads at a time.  For heads
// of 128 or more dims (one thread per dim), beyond two such rounds of L2
// round trips it copies the partials into a ring stage first (one bulk copy
// per sequence) and merges them from shared memory.  Smaller heads merge
// straight from L2: there the staged variant measured slower.
MK_HD inline bool part_staged(int S, int NB, int D) {
  const int sg = NCT / (NB * D) > 0 ? NCT / (NB * D) : 1;
  return D >= 128 && S > 8 * sg;
}
constexpr int MMA_FLUSH = 32;        // batched GEMV: rows per cross-warp sum of partials

// Dense batch-1 models run the MLP as two ops (gate/up column slices, then
// row-split down projection over the whole h) when one down row fits a ring
// stage; otherwise one fused op per FFN column slice with float atomics.
// Batched split MLP (dense, 2..8 sequences): gate/up column slices (multiples
// of 16 columns) write h in tensor-core A-fragment form; the down projection
// is cut into units of BD_ROWS rows x BD_KC columns (16 KB), numbered
// chunk-major, and a down instruction takes a run of at most BD_MAX_UNITS
// consecutive units that spans at most two chunks.  It loads those chunks'
// h fragments (16 KB each) once, streams its units through the ring and adds
// each unit's partial rows into the residual with float reductions (the
// chunk-0 units also add x_{2l+1}).
// Wide batch (8 .. WIDE_NB sequences, dense FFN, 64-dim heads).  Every
// contraction runs on the fifth-generation tensor cores: tcgen05.mma with
// M = 128 weight rows (A, from the ring) and N = 2 * Bp activation rows (B:
// the bf16 high and low parts of each sequence's activation, rows 2b and
// 2b + 1, Bp = the batch rounded up to 8), the f32 accumulator in tensor
// memory.  Both operands are K-major tiles of 64 columns in the 128-byte
// swizzle.  The normalised activations are written once per step and norm
// point by OP_NORM instructions, into operand buffers in that layout; the
// QKV, gate/up, down and LM-head instructions stream them through the ring
// K chunk by K chunk next to their weights.  The attention items that finish
// a (sequence, kv head) last merge its split-KV slices into a fourth operand
// buffer, which the O-projection (one kv group's query heads, one K chunk
// per head) streams the same way.
constexpr int WIDE_NB = 32;          // batch capacity of the wide variant
constexpr int WIDE_KC = 64;          // columns of one K chunk (a 128-byte row of bf16)
constexpr int WIDE_ROWS = 128;       // weight rows of one instruction (the MMA's M)
// Consumer warps 0 .. WIDE_NI - 1 each issue the MMAs of every WIDE_NI-th K
// chunk into an accumulator of their own (64 columns apart): one thread
// issues a tcgen05.mma about every 40 ns whatever its shape, so the issue
// rate, not the tensor pipe, bounds a GEMV with a handful of operand rows
// (measured at 8 / 16 / 32 sequences, 1 / 2 / 4 / 7 issuers: 0.993 / 0.952 /
// 0.937 / 0.938, 1.111 / 1.076 / 1.053 / 1.061, 1.451 / 1.404 / 1.397 /
// 1.408 ms per step).
constexpr int WIDE_NI = 4;
// tensor-memory columns a CTA allocates (a power of two >= 32)
constexpr int WIDE_TMEM_COLS = WIDE_NI <= 1 ? 64 : WIDE_NI <= 2 ? 128 : WIDE_NI <= 4 ? 256 : 512;
// Used from 9 sequences on, and from 2 when the shape allows it unless the
// descriptor asks for the batched variant (measured at 2 / 4 / 7 sequences:
// 0.832 / 0.882 / 0.904 ms per step against the batched variant's 0.953 /
// 1.013 / 1.125).
MK_HD inline bool wide_path(const mk_model_desc& d) {
  return d.n_experts == 0 &&
         (d.max_batch > 8 ||
          (d.max_batch >= 2 && d.batched_variant == 0 && d.ffn % WIDE_KC == 0 &&
           d.hidden % WIDE_KC == 0 && d.head_dim == WIDE_KC && d.n_q_heads == 4 * d.n_kv_heads));
}
MK_HD inline int wide_bp(int B) { return (B + 7) / 8 * 8; }

constexpr int BD_KC = 512;
constexpr int BD_ROWS = 16;
constexpr int BD_MAX_UNITS = 32;
MK_HD inline bool mlp_split_batched(const mk_model_desc& d) {
  return d.n_experts == 0 && d.max_batch > 1 && d.max_batch <= 8 && !wide_path(d) &&
         d.ffn % BD_KC == 0 && d.hidden % BD_ROWS == 0;
}

inline bool mlp_split(const mk_model_desc& d) {
  return d.n_experts == 0 && d.max_batch == 1 && d.ffn % 8 == 0 && d.ffn * 2 <= DOWN_ROW_MAX;
}



// Device pointers of one layer inside the packed weight buffer.
struct LayerPtrs {
  const uint16_t* attn_norm;  // [H]
  const uint16_t* mlp_norm;   // [H]
  const uint16_t* wqkv;       // [Hkv][(HPG+2)*D][H]; per head rows (t, t+D/2) adjacent
  const uint16_t* wo;         // [Hq][H][D]
  const uint16_t* wgu;        // dense: [F][2][H]      (gate row, up row)
  const uint16_t* wdT;        // dense: down, [F][H] transposed (fused MLP) or [H][F] (split MLP)
  const uint16_t* router;     // MoE:   [E][H]
  const uint16_t* ex_gu;      // MoE:   [E][Fe][2][H]
  const uint16_t* ex_dT;      // MoE:   [E][Fe][H]
  const uint16_t* sh_gu;      // MoE:   [Fs][2][H]
  const uint16_t* sh_dT;      // MoE:   [Fs][H]
  uint16_t* kc;               // caller cache [maxB][Hkv][max_seq][D]
  uint16_t* vc;
  // int8 weights (dense batch 1): wqkv, wo, wgu, wdT then hold int8 codes,
  // biased by 128 (byte q + 128), in the same layouts (Wo: chunk k of row r
  // at slot k ^ ((r >> 1) & 3)), and these fp32 scales, one per packed row,
  // multiply each row's dot product
  const float* sqkv;          // [Hkv][(HPG+2)*D], packed row order
  const float* so;            // [H]: Wo output row r (shared by every head's piece)
  const float* sgu;           // [F][2]: gate row c, up row c
  const float* sd;            // [H]: down output row
};

// A value that one writer produces once per step, with that step's tag
// (the epoch); read and written as one aligned 64-bit word.
struct alignas(8) TagWord {
  uint32_t bits;  // the f32 value's bits
  uint32_t tag;   // epoch of the step that wrote it (0: never written)
};

// Kernel parameter block (passed by value as __grid_constant__).
struct Globals {
  const Instr* sched;
  const LayerPtrs* layers;
  const uint16_t* embed;
  const uint16_t* lm_head;    // int8 weights: biased int8 codes [V][H], scales lm_scale [V]
  const float* lm_scale;
  const uint16_t* final_norm;
  const float* rope;       // [max_seq][D/2][2] (cos, sin)
  float* xbuf;             // [2][2L][kc][B][H] residual stream x_1 .. x_2L, kc partial copies
  float* qbuf;             // [L][B][Hq][D]
  float* part;             // [L][B][Hq][splits][part_stride(D)]: o[D], m, l (log2 domain)
  float* rlog;             // [L][B][E] router logits
  float* hglob;            // [L][B][F] SiLU(gate)*up (split MLP)
  TagWord* xt;             // [L][B][H] tagged x_{2l+2} (split MLP: written once, by row owners)
  int* routes;             // [L][K] expert ids of the current step (MoE, batch 1), by rank
  float* rweight;          // [L][K] their router probabilities renormalised over the K chosen
  float* lm_val;           // [n_lm][B]
  int* lm_idx;             // [n_lm][B]
  uint32_t* ctr;           // dependency counters
  int* err;                // [4]: status, sm, pc, op
  const int* tokens;
  const int* positions;
  float* logits;
  int* argmax;
  unsigned long long timeout_ns;
  int n_pollers;           // warps that poll a dependency counter (1..NCW)
  unsigned poll_stagger_ns;// delay between the pollers' first polls
  int max_pc, n_sm, n_stages;
  int stage_bytes;  // bytes per ring stage (multiple of STAGE_UNIT)
  int B, H, Hq, Hkv, D, F, V, L, max_seq, max_ctx, splits;
  int E, K, Fe, Fs;
  int kc;                  // partial copies of each residual vector (1..8)
  float eps;
  uint32_t epoch;          // step number (>= 1); counter targets are epoch * count, and
                           // tagged words written in this step carry tag == epoch
  int xtag;                // x_{2l+2} lives in xt (split MLP) rather than in xbuf
  int bsplit;              // batched split MLP (hglob holds h as A fragments)
  uint32_t lm_ctr;
  uint32_t lm_done_ctr;     // signalled once per step after the argmax is written
  int part_staged;          // O-projection: partials through a ring stage (part_staged())
  int kv_block;             // 0: KV cache [B][Hkv][max_seq][D]; else paged, blocks of kv_block rows:
  int kv_blocks;            //   pool [kv_blocks][Hkv][kv_block][D], block of (b, j) =
  const int* kv_table;      //   kv_table[b * kv_stride + j]
  int kv_stride;
  int n_steps;              // greedy decode steps in this launch (1: one step)
  // race stress (mk_set_race_stress; off: 0 / nullptr): a hashed delay below
  // stress_ns before each instruction, on the producer and the consumers,
  // and queue qperm[blockIdx.x] run by CTA blockIdx.x
  uint32_t stress_ns, stress_seed;
  const int* qperm;
  int n_lm;
  int zero_next;           // the LM head slices zero the next step's residual buffers (the
                           // other parity, epoch + 1 & 1) while they wait for their input
  int pdl;                 // ablation with programmatic dependent launch
  unsigned long long* trace;  // optional [n_sm][max_pc][8] %globaltimer stamps (NULL: off)
  unsigned long long l2_ahead;  // bytes of the SM's stream warmed in L2 ahead of the ring (0: off)
  unsigned hold_early;          // bytes of a held instruction's copies issued before the
                                // consumers finish the previous instruction (whole stages)
  // extents, for the bounds-checked build (MK_BOUNDS): the library's scratch
  // and packed-weight allocations, one layer's K (or V) cache, and the
  // element counts of the scratch buffers the ops index
  const unsigned char* sc_lo;
  size_t sc_bytes;
  const unsigned char* pk_lo;
  size_t pk_bytes;
  size_t kv_elems;              // bf16 elements of one layer's K (or V) cache or pool
  size_t n_xbuf, n_q, n_part, n_h, n_xt, n_lmv;  // n_lmv: lm_val / lm_idx elements
  // wide batch: the three normalised operands (attention input, MLP input,
  // final), each [H / 64][2 Bp][64] bf16 in the swizzled K-major layout; h
  // (in hglob) is [F / 64][2 Bp][64] likewise
  unsigned char* act;      // (then a fourth, [Hq][2 Bp][64]: the merged attention outputs)
  int Bp;                  // batch rounded up to 8 (the operand holds 2 Bp rows)
  uint32_t arr_ctr;        // first of the [L][B][Hkv] attention-arrival counters
  // batched variants: [L][K, V] tensor maps (128 bytes each) of the contiguous
  // K / V caches for the tensor-core attention; nullptr: the CUDA-core body
  const void* tmaps;
};

// Shared-memory layout (bytes from the dynamic shared memory base).
struct SmemLayout {
  int ring, full, empty, xn, yrow, hbuf, attn, red, misc, mpart, sc, tcw, total;
};

// WB: bytes per weight (2 bf16, 1 int8; int8 adds the row-scale region sc)
MK_HD inline SmemLayout smem_layout(int n_stages, int stage_bytes, int NB, int H, int D, int HPG,
                                     int K, int WB) {
  SmemLayout s;
  int o = 0;
  s.ring = o;   o += n_stages * stage_bytes;
  s.full = o;   o += 8 * n_stages;
  s.empty = o;  o += 8 * n_stages;
  o = (o + 15) / 16 * 16;
  if (NB > 8) {
    // wide batch: no normalised vector in shared memory (it is an operand
    // buffer in global memory); the M = 128 MMAs read up to 16 KB from the
    // start of a weight piece, so at least that much shared memory follows
    // the ring (yrow comes first)
    s.xn = o;
    s.yrow = o;
    const int yb = 4 * NB * WIDE_ROWS, ab = 4 * NCW * HPG * (D + 2);
    int m = yb > ab ? yb : ab;
    m = m > 16384 ? m : 16384;
    o += (m + 15) / 16 * 16;
    s.hbuf = o;
    s.attn = o;
    s.red = o;    o += 4 * 2 * NCW * NB + 16 + 4 * 2 * NB;  // + an LM-head slice's running maxima
    s.misc = o;   o += 4 * (8 + 3 * NB + 4 * NB);
    s.tcw = o;    o += 16;  // tensor-memory base address, MMA-done mbarrier
    s.mpart = o;
    s.sc = o;
    s.total = (o + 127) / 128 * 128;
    return s;
  }
  s.xn = o;     o += 4 * NB * H;
  s.yrow = o;
  int yb = 4 * NB * MAX_ROWS;
  int mb = 4 * NCW * HPG * (D + 2);
  o += ((yb > mb ? yb : mb) + 15) / 16 * 16;
  s.hbuf = o;   o += 4 * NB * MAX_COLS;
  s.attn = o;   o += 4 * NB * D;
  s.red = o;    o += 4 * 2 * NCW * NB + 16;
  s.misc = o;   o += 4 * (8 + 3 * NB + 4 * NB * (K > 0 ? K : 1));
  o = (o + 15) / 16 * 16;
  s.mpart = o;  o += NB > 1 ? 4 * NCW * MMA_FLUSH * NB : 0;  // batched GEMV partial sums
  s.sc = o;     o += WB == 1 ? 4 * H : 0;  // row scales of one O-proj / LM-head instruction
  s.tcw = o;
  s.total = (o + 127) / 128 * 128;
  return s;
}

// One compiled instantiation of the interpreter.
struct Variant {
  int H, D, HPG, NB, WB;  // WB: bytes per weight, 2 (bf16) or 1 (int8 codes)
  const void* kernel;     // host stub of mk_decode_kernel<H, D, HPG, NB, WB>
};

// A built schedule: queues [n_sm][max_pc] (HALT-padded) and their statistics.
struct PlanOut {
  std::vector<Instr> q;
  int max_pc = 0, n_ctr = 0, splits = 0, n_lm = 0, n_instr = 0;
  double max_sm_bytes = 0, mean_sm_bytes = 0, weight_bytes = 0;
};
int plan_shape_ok(const mk_model_desc& d);
// wb: bytes per weight of the packed matrices (2 bf16, 1 int8)
int plan_build(const mk_model_desc& d, int B, int max_ctx, int n_sm, PlanOut& out,
               unsigned hold_mask = DEFAULT_HOLD, int wb = 2);
int plan_verify(const mk_model_desc& d, int B, const PlanOut& p);
int plan_check(const Instr* q, int n_sm, int max_pc, int n_ctr);

}  // namespace mk
