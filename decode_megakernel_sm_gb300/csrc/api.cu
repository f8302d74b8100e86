// api.cu -- the C ABI of libmk.so (declared in include/mk.h): handle life
// cycle, weight packing, schedule upload, the one-launch decode step, the
// host-buffer step, the per-phase ablation launcher and error reporting.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <tuple>
#include <vector>

#include "mk_internal.h"

namespace mk {
cudaError_t pack_qkv(uint16_t* dst, const void* wq, const void* wk, const void* wv, int H, int Hkv,
                     int HPG, int D, cudaStream_t s);
cudaError_t pack_interleave(uint16_t* dst, const void* a, const void* b, long rows, int H,
                            cudaStream_t s);
cudaError_t pack_wo(uint16_t* dst, const void* wo, int H, int Hq, int D, cudaStream_t s);
cudaError_t pack_rows(uint16_t* dst, const void* src, long rows, int H, cudaStream_t s);
cudaError_t pack_down_tiles(uint16_t* dst, const void* src, int H, int F, cudaStream_t s);
cudaError_t pack_transpose(uint16_t* dst, const void* src, int R, int C, int batch,
                           cudaStream_t s);
cudaError_t quantize_rows_int8(int8_t* codes, float* scales, const void* w, long rows, int cols,
                               cudaStream_t s);
cudaError_t pack_qkv_scales(float* dst, const float* sq, const float* sk, const float* sv, int Hkv,
                            int HPG, int D, cudaStream_t s);
cudaError_t interleave_scales(float* dst, const float* a, const float* b, int n, cudaStream_t s);
cudaError_t pack_wo_i8(void* dst, const void* wo_codes, int H, int Hq, cudaStream_t s);
cudaError_t bias_codes(void* p, size_t bytes, cudaStream_t s);
cudaError_t pack_kchunk(uint16_t* dst, const uint16_t* src, long R, int K, cudaStream_t s);

extern const Variant variant_h256_d64_g2_b1;
#ifndef MK_BOUNDS
extern const Variant variant_h2048_d64_g4_b1;
extern const Variant variant_h2048_d64_g4_b8;
extern const Variant variant_h2048_d64_g4_b32;
extern const Variant variant_h2048_d128_g4_b1;
extern const Variant variant_h2048_d64_g4_b1_w8;
#endif
}  // namespace mk

using namespace mk;

// Per-schedule device scratch, carved from one allocation (or from the
// library's fixed array on the no-alloc path).  The tagged block holds the
// words that carry a step tag; it must read as tag 0 (never a valid epoch)
// whenever a step is about to run with an epoch that earlier contents may
// already carry.
struct Scratch {
  float *xbuf, *qbuf, *part, *rlog, *lm_val;
  int *lm_idx, *routes, *err;
  float* rweight;
  uint32_t* ctr;
  float* hglob;             // SiLU(gate)*up (split MLP)
  TagWord* xt;              // tagged block: x_{2l+2} (split MLP)
  unsigned char* act;       // wide batch: the three normalised operands
  size_t xbuf_bytes, ctr_bytes, err_bytes, tag_bytes, total;
  size_t n_q, n_part, n_h, n_xt, n_lm;  // element counts (bounds checks)
};

static size_t al256(size_t n) { return (n + 255) / 256 * 256; }

// Sizes (and, when base != nullptr, pointers) of the scratch for one schedule.
static Scratch carve_scratch(const mk_model_desc& d, size_t B, size_t kc, size_t splits,
                             size_t n_lm, size_t n_ctr, char* base) {
  const size_t L = d.n_layers, H = d.hidden, Hq = d.n_q_heads, D = d.head_dim;
  const size_t E = d.n_experts > 0 ? d.n_experts : 1;
  const size_t F = d.ffn > 0 ? d.ffn : 1;
  const size_t sx = al256(2 * 2 * L * kc * B * H * 4), sq = al256(L * B * Hq * D * 4);
  const size_t sp = al256(L * B * Hq * splits * part_stride((int)D) * 4);
  const size_t sr = al256(L * B * E * 4), sl = al256(n_lm * B * 4);
  const size_t sc = al256(n_ctr * 4), se = 256;
  const size_t sroute = al256(L * (size_t)(d.top_k > 0 ? d.top_k : 1) * 4);  // ids, then weights
  // h: batch-1 split [L][B][F] floats; batched split [L][F/16][32] A-fragment
  // words of 16 bytes (8 sequences x 4 bytes per column); wide batch one
  // operand buffer [F/64][2 Bp][64] bf16 (every layer reuses it).  The wide
  // normalised operands: three buffers [H/64][2 Bp][64] bf16, then the merged
  // attention outputs [Hq][2 Bp][64].
  const bool wide = wide_path(d);
  const size_t Bp = (size_t)wide_bp((int)B);
  const size_t hB = mlp_split_batched(d) ? 8 : B;
  const size_t sxt = al256(L * B * H * 8);
  const size_t sh = wide ? al256(F * 2 * Bp * 2) : al256(L * hB * F * 4);
  const size_t sa = wide ? al256((3 * H + Hq * D) * 2 * Bp * 2) : 0;
  Scratch s{};
  s.xbuf_bytes = sx;
  s.ctr_bytes = sc;
  s.err_bytes = se;
  s.tag_bytes = sxt;
  s.n_q = sq / 4;
  s.n_part = sp / 4;
  s.n_h = sh / 4;
  s.n_xt = sxt / 8;
  s.n_lm = sl / 4;
  s.total = sx + sq + sp + sr + 2 * sl + sc + se + 2 * sroute + sh + sxt + sa;
  if (!base) return s;
  char* q = base;
  s.xbuf = (float*)q; q += sx;
  s.qbuf = (float*)q; q += sq;
  s.part = (float*)q; q += sp;
  s.rlog = (float*)q; q += sr;
  s.lm_val = (float*)q; q += sl;
  s.lm_idx = (int*)q; q += sl;
  s.ctr = (uint32_t*)q; q += sc;
  s.err = (int*)q; q += se;
  s.routes = (int*)q; q += sroute;
  s.rweight = (float*)q; q += sroute;
  s.hglob = (float*)q; q += sh;
  s.xt = (TagWord*)q; q += sxt;
  s.act = sa ? (unsigned char*)q : nullptr;
  return s;
}

struct mk_handle {
  mk_model_desc d{};
  int dev = 0, n_sm = 0;
  const Variant* var = nullptr;
  int n_stages = 0, smem_bytes = 0;
  int stage_bytes = DEFAULT_STAGE_BYTES;
  int max_stages = 0;  // 0: as many as fit
  int kv_block = 0, kv_blocks = 0, kv_stride = 0;  // paged KV cache (0: contiguous)
  const int32_t* kv_table = nullptr;
  unsigned stress_ns = 0, stress_seed = 0;  // race stress (0: off)
  int* qperm = nullptr;                     // device queue permutation, or nullptr
  void* packed = nullptr;
  size_t packed_bytes = 0;
  std::vector<LayerPtrs> layers_h;
  LayerPtrs* layers_d = nullptr;
  const uint16_t *embed = nullptr, *lm_head = nullptr, *final_norm = nullptr;
  int wfmt = MK_WEIGHTS_BF16;
  const float* lm_scale = nullptr;  // int8 weights
  float* rope = nullptr;
  // batched variants: per layer, tensor maps of the K and V caches (tiled
  // TMA loads for the tensor-core attention), or nullptr
  void* tmaps = nullptr;
  // schedule and scratch
  int batch = 0, max_ctx = 0;
  PlanOut plan;
  Instr* sched = nullptr;
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
  Scratch sc{};
  // ablation: one launch per (layer, phase) key that owns instructions, each
  // over compacted queues holding only that key's instructions
  struct AblLaunch {
    size_t off;   // first record of its queues in abl_sched
    int n_q;      // queues (= CTAs of the launch): the SMs that own such instructions
    int max_pc;   // records per queue, HALT included
  };
  std::vector<AblLaunch> abl;
  Instr* abl_sched = nullptr;
  uint32_t epoch = 0;
  unsigned long long timeout_ns = 2000000000ull;
  int n_pollers = 1;
  unsigned poll_stagger_ns = 0;
  unsigned long long l2_ahead = 0;
  int kc = 1;  // partial copies of each residual vector
  unsigned hold_mask = DEFAULT_HOLD;
  unsigned hold_early = DEFAULT_HOLD_EARLY;
  // host-buffer step
  cudaStream_t own = nullptr;
  int32_t *d_tok = nullptr, *d_pos = nullptr, *d_am = nullptr;
  float* d_logits = nullptr;
  int* h_err = nullptr;  // pinned [4]
  unsigned long long* trace = nullptr;  // [n_sm][max_pc][8] when tracing is on
  // graph-mode ablation cache
  std::map<std::tuple<const void*, const void*, const void*, const void*, const void*>,
           cudaGraphExec_t>
      graphs;
};

#define CK(x)                                \
  do {                                       \
    cudaError_t e_ = (x);                    \
    if (e_ != cudaSuccess) return MK_ERR_CUDA; \
  } while (0)


static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

static const Variant* pick_variant(const mk_model_desc& d, int wb) {
#ifdef MK_BOUNDS
  // the bounds-checked library carries the small variant only
  const Variant* all[] = {&variant_h256_d64_g2_b1};
#else
  const Variant* all[] = {&variant_h256_d64_g2_b1, &variant_h2048_d64_g4_b1,
                          &variant_h2048_d64_g4_b8, &variant_h2048_d128_g4_b1,
                          &variant_h2048_d64_g4_b1_w8, &variant_h2048_d64_g4_b32};
#endif
  const int HPG = d.n_q_heads / d.n_kv_heads;
  const Variant* best = nullptr;
  for (const Variant* v : all) {
    if (v->H != d.hidden || v->D != d.head_dim || v->HPG != HPG || v->WB != wb) continue;
    if (v->NB < d.max_batch) continue;
    if (wide_path(d) != (v->NB == WIDE_NB)) continue;  // the wide variant exactly on its path
    if (!best || v->NB < best->NB) best = v;
  }
  if (best && d.n_experts > 0 && best->NB != 1) return nullptr;  // MoE routing is per token
  return best;
}

static void free_schedule(mk_handle* h) {
  if (h->trace) cudaFree(h->trace);
  h->trace = nullptr;
  for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second);
  h->graphs.clear();
  if (h->sched) cudaFree(h->sched);
  if (h->abl_sched) cudaFree(h->abl_sched);
  if (h->scratch) cudaFree(h->scratch);
  h->sched = nullptr;
  h->abl_sched = nullptr;
  h->abl.clear();
  h->scratch = nullptr;
  if (h->d_tok) cudaFree(h->d_tok);
  h->d_tok = h->d_pos = h->d_am = nullptr;
  h->d_logits = nullptr;
  h->batch = 0;
}

static void free_all(mk_handle* h) {
  if (!h) return;
  free_schedule(h);
  if (h->packed) cudaFree(h->packed);
  if (h->layers_d) cudaFree(h->layers_d);
  if (h->rope) cudaFree(h->rope);
  if (h->tmaps) cudaFree(h->tmaps);
  if (h->qperm) cudaFree(h->qperm);
  if (h->h_err) cudaFreeHost(h->h_err);
  if (h->own) cudaStreamDestroy(h->own);
  delete h;
}

// Packed-buffer sizes (elements) of one layer, in carve order.
struct LayerSizes {
  size_t norm, qkv, wo, gu, dT, router, ex_gu, ex_dT, sh_gu, sh_dT;
};

static LayerSizes layer_sizes(const mk_model_desc& d) {
  const size_t H = d.hidden, D = d.head_dim, Hq = d.n_q_heads, Hkv = d.n_kv_heads;
  const size_t HPG = Hq / Hkv;
  LayerSizes s{};
  s.norm = H;
  s.qkv = Hkv * (HPG + 2) * D * H;
  s.wo = Hq * H * D;
  if (d.n_experts == 0) {
    s.gu = 2 * (size_t)d.ffn * H;
    s.dT = (size_t)d.ffn * H;
  } else {
    s.router = (size_t)d.n_experts * H;
    s.ex_gu = 2 * (size_t)d.n_experts * d.expert_ffn * H;
    s.ex_dT = (size_t)d.n_experts * d.expert_ffn * H;
    s.sh_gu = 2 * (size_t)d.shared_ffn * H;
    s.sh_dT = (size_t)d.shared_ffn * H;
  }
  return s;
}

// Ring depth for `stage_bytes`: as many stages (2..MAX_STAGES) as the
// opt-in shared memory holds next to the fixed buffers; sets the kernel's
// dynamic shared-memory size and checks that one CTA still fits per SM.
static int size_ring(mk_handle* h, int stage_bytes) {
  const mk_model_desc& d = h->d;
  const int K = d.n_experts > 0 ? d.top_k : 0;
  const int HPG = d.n_q_heads / d.n_kv_heads;
  int optin = 0;
  CK(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->dev));
  int ns = 0;
  const int cap = h->max_stages > 0 ? h->max_stages : MAX_STAGES;
  for (int n = 2; n <= cap; n++)
    if (smem_layout(n, stage_bytes, h->var->NB, d.hidden, d.head_dim, HPG, K, h->var->WB).total <= optin)
      ns = n;
  if (ns < 2) return MK_ERR_UNSUPPORTED;
  const int bytes = smem_layout(ns, stage_bytes, h->var->NB, d.hidden, d.head_dim, HPG, K, h->var->WB).total;
  CK(cudaFuncSetAttribute(h->var->kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
  int per_sm = 0;
  CK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, h->var->kernel, NTHREADS, bytes));
  if (per_sm < 1) return MK_ERR_UNSUPPORTED;
  h->stage_bytes = stage_bytes;
  h->n_stages = ns;
  h->smem_bytes = bytes;
  return MK_OK;
}

static int pack_int8(mk_handle* h, const mk_weights* w, const mk_kv* kv, cudaStream_t s);
static int pack_bf16(mk_handle* h, const mk_weights* w, const mk_kv* kv, cudaStream_t s);

// Tensor maps of every layer's K and V cache for the tensor-core attention
// of the batched variants (64-dim heads, 2 or 4 query heads per kv head): the
// cache [max_batch][Hkv][max_seq][64] as a 2-D bf16 tensor of
// max_batch * Hkv * max_seq rows, loaded in boxes of 64 rows x 64 columns in
// the 128-byte swizzle.  Other shapes get none (the CUDA-core attention).
static int make_kv_tmaps(mk_handle* h, const mk_kv* kv) {
  const mk_model_desc& d = h->d;
  const int HPG = d.n_q_heads / d.n_kv_heads;
  if (h->var->NB == 1 || d.head_dim != 64 || (HPG != 2 && HPG != 4)) return MK_OK;
  static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if (!enc) {
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", (void**)&enc, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !enc) {
      enc = nullptr;
      return MK_ERR_CUDA;
    }
  }
  const int L = d.n_layers;
  std::vector<CUtensorMap> maps(2 * (size_t)L);
  const cuuint64_t dims[2] = {64, (cuuint64_t)d.max_batch * d.n_kv_heads * d.max_seq};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {64, 64}, es[2] = {1, 1};
  for (int l = 0; l < L; l++)
    for (int kvi = 0; kvi < 2; kvi++) {
      void* base = kvi == 0 ? kv->k[l] : kv->v[l];
      if (enc(&maps[2 * l + kvi], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return MK_ERR_CUDA;
    }
  CK(cudaMalloc(&h->tmaps, maps.size() * sizeof(CUtensorMap)));
  CK(cudaMemcpy(h->tmaps, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice));
  return MK_OK;
}

static int create_impl(const mk_model_desc* desc, const mk_weights* w, const mk_kv* kv,
                       mk_handle* h, int wfmt) {
  const mk_model_desc& d = *desc;
  h->d = d;
  int rc = plan_shape_ok(d);
  if (rc) return rc;
  if (wfmt != MK_WEIGHTS_BF16 && wfmt != MK_WEIGHTS_INT8) return MK_ERR_INVALID_ARG;
  // int8 weights: dense batch-1 shapes with the split MLP and 64-dim heads
  if (wfmt == MK_WEIGHTS_INT8 && (!mlp_split(d) || d.ffn % 16 || d.head_dim != 64))
    return MK_ERR_UNSUPPORTED;
  h->wfmt = wfmt;
  // wide batch (2 .. 32 sequences, see wide_path): dense FFN in whole
  // 64-column chunks, 64-dim heads, bf16 weights
  if (d.max_batch > 8 && (d.n_experts > 0 || d.max_batch > WIDE_NB || d.ffn % WIDE_KC ||
                          d.hidden % WIDE_KC || d.head_dim != WIDE_KC))
    return MK_ERR_UNSUPPORTED;
  if (wide_path(d) && wfmt != MK_WEIGHTS_BF16) return MK_ERR_UNSUPPORTED;
  h->var = pick_variant(d, wfmt == MK_WEIGHTS_INT8 ? 1 : 2);
  if (!h->var) return MK_ERR_UNSUPPORTED;
  const int L = d.n_layers, D = d.head_dim;
  const bool moe = d.n_experts > 0;
  // ---- argument checks (pointers present and 16-byte aligned)
  if (!w || !kv || !kv->k || !kv->v || !w->embed || !w->final_norm || !w->attn_norm || !w->wq ||
      !w->wk || !w->wv || !w->wo || !w->mlp_norm)
    return MK_ERR_INVALID_ARG;
  if (!d.tied_lm_head && !w->lm_head) return MK_ERR_INVALID_ARG;
  if (!moe && (!w->w_gate || !w->w_up || !w->w_down)) return MK_ERR_INVALID_ARG;
  if (moe && (!w->router || !w->ex_gate || !w->ex_up || !w->ex_down)) return MK_ERR_INVALID_ARG;
  if (moe && d.shared_ffn > 0 && (!w->sh_gate || !w->sh_up || !w->sh_down))
    return MK_ERR_INVALID_ARG;
  auto okp = [](const void* p) { return p && aligned16(p); };
  if (!okp(w->embed) || !okp(w->final_norm) || (!d.tied_lm_head && !okp(w->lm_head)))
    return MK_ERR_INVALID_ARG;
  for (int l = 0; l < L; l++) {
    if (!okp(w->attn_norm[l]) || !okp(w->wq[l]) || !okp(w->wk[l]) || !okp(w->wv[l]) ||
        !okp(w->wo[l]) || !okp(w->mlp_norm[l]) || !okp(kv->k[l]) || !okp(kv->v[l]))
      return MK_ERR_INVALID_ARG;
    if (!moe && (!okp(w->w_gate[l]) || !okp(w->w_up[l]) || !okp(w->w_down[l])))
      return MK_ERR_INVALID_ARG;
    if (moe && (!okp(w->router[l]) || !okp(w->ex_gate[l]) || !okp(w->ex_up[l]) ||
                !okp(w->ex_down[l])))
      return MK_ERR_INVALID_ARG;
    if (moe && d.shared_ffn > 0 &&
        (!okp(w->sh_gate[l]) || !okp(w->sh_up[l]) || !okp(w->sh_down[l])))
      return MK_ERR_INVALID_ARG;
  }
  // int8 weights: a 4-stage ring by default (fewer copies in flight shorten
  // the dependency hops; half the bytes per row keep the bodies fed)
  if (wfmt == MK_WEIGHTS_INT8) h->max_stages = 4;
  if (h->var->NB > 8) h->stage_bytes = WIDE_STAGE_BYTES;
  if (h->var->NB == 1 && wfmt != MK_WEIGHTS_INT8) h->stage_bytes = BATCH1_STAGE_BYTES;
  // ---- device
  CK(cudaGetDevice(&h->dev));
  CK(cudaDeviceGetAttribute(&h->n_sm, cudaDevAttrMultiProcessorCount, h->dev));
  {
    int st = size_ring(h, h->stage_bytes);
    // a one-sequence shape whose fixed buffers leave no room for two 64 KB
    // stages takes the general default
    if (st == MK_ERR_UNSUPPORTED && h->var->NB == 1 && h->stage_bytes > DEFAULT_STAGE_BYTES)
      st = size_ring(h, DEFAULT_STAGE_BYTES);
    if (st != MK_OK) return st;
  }
  CK(cudaStreamCreateWithFlags(&h->own, cudaStreamNonBlocking));
  CK(cudaMallocHost(&h->h_err, 4 * sizeof(int)));
  cudaStream_t s = h->own;
  if (wfmt == MK_WEIGHTS_INT8) {
    rc = pack_int8(h, w, kv, s);
    if (rc) return rc;
  } else {
    rc = pack_bf16(h, w, kv, s);
    if (rc) return rc;
  }
  CK(cudaMalloc(&h->layers_d, sizeof(LayerPtrs) * L));
  CK(cudaMemcpyAsync(h->layers_d, h->layers_h.data(), sizeof(LayerPtrs) * L,
                     cudaMemcpyHostToDevice, s));
  // rotary table: angle p * theta^(-2t/D) evaluated in double, stored fp32
  std::vector<float> rope((size_t)d.max_seq * D);
  for (int pp = 0; pp < d.max_seq; pp++)
    for (int t = 0; t < D / 2; t++) {
      const double ang = (double)pp * std::pow((double)d.rope_theta, -2.0 * t / (double)D);
      rope[((size_t)pp * (D / 2) + t) * 2 + 0] = (float)std::cos(ang);
      rope[((size_t)pp * (D / 2) + t) * 2 + 1] = (float)std::sin(ang);
    }
  CK(cudaMalloc(&h->rope, rope.size() * sizeof(float)));
  {
    const int rc2 = make_kv_tmaps(h, kv);
    if (rc2 != MK_OK) return rc2;
  }
  CK(cudaMemcpyAsync(h->rope, rope.data(), rope.size() * sizeof(float), cudaMemcpyHostToDevice,
                     s));
  CK(cudaStreamSynchronize(s));
  return MK_OK;
}

// bf16 packing: every matrix re-laid out for the ring (the layouts in pack.cu).
static int pack_bf16(mk_handle* h, const mk_weights* w, const mk_kv* kv, cudaStream_t s) {
  const mk_model_desc& d = h->d;
  const int L = d.n_layers, H = d.hidden, Hq = d.n_q_heads, Hkv = d.n_kv_heads;
  const int D = d.head_dim, HPG = Hq / Hkv;
  const bool moe = d.n_experts > 0;
  const LayerSizes ls = layer_sizes(d);
  const size_t V = d.vocab;
  // wide batch: every streamed matrix but Wo K-chunk-major ([K/64][R8][64],
  // pack_kchunk) from its standard packed form, staged in `tmp`
  const bool wide = wide_path(d);
  const size_t V8 = (V + 7) / 8 * 8;
  size_t per_layer = 0;
  for (size_t e : {ls.norm, ls.norm, ls.qkv, ls.wo, ls.gu, ls.dT, ls.router, ls.ex_gu, ls.ex_dT,
                   ls.sh_gu, ls.sh_dT})
    per_layer += al256(e * 2);
  const size_t lm_bytes = wide ? al256(V8 * H * 2) : al256(V * H * 2);
  const size_t total =
      per_layer * L + al256(V * H * 2) + (d.tied_lm_head && !wide ? 0 : lm_bytes) + al256(H * 2);
  uint16_t* tmp = nullptr;
  if (wide) {
    const size_t mx = std::max({ls.qkv, ls.gu, ls.dT, V * (size_t)H});
    CK(cudaMalloc(&tmp, mx * 2));
  }
  struct TmpFree {
    uint16_t* p;
    cudaStream_t s;
    ~TmpFree() {
      if (p) {
        cudaStreamSynchronize(s);
        cudaFree(p);
      }
    }
  } tmp_free{tmp, s};
  CK(cudaMalloc(&h->packed, total));
  h->packed_bytes = total;
  char* p = (char*)h->packed;
  auto take = [&](size_t elems) {
    uint16_t* r = (uint16_t*)p;
    p += al256(elems * 2);
    return r;
  };
  h->layers_h.resize(L);
  for (int l = 0; l < L; l++) {
    LayerPtrs& lp = h->layers_h[l];
    std::memset(&lp, 0, sizeof lp);
    uint16_t* an = take(ls.norm);
    uint16_t* mn = take(ls.norm);
    uint16_t* qkv = take(ls.qkv);
    uint16_t* wo = take(ls.wo);
    uint16_t* gu = take(ls.gu);
    uint16_t* dT = take(ls.dT);
    uint16_t* rt = take(ls.router);
    uint16_t* egu = take(ls.ex_gu);
    uint16_t* edT = take(ls.ex_dT);
    uint16_t* sgu = take(ls.sh_gu);
    uint16_t* sdT = take(ls.sh_dT);
    CK(cudaMemcpyAsync(an, w->attn_norm[l], ls.norm * 2, cudaMemcpyDeviceToDevice, s));
    CK(cudaMemcpyAsync(mn, w->mlp_norm[l], ls.norm * 2, cudaMemcpyDeviceToDevice, s));
    CK(pack_wo(wo, w->wo[l], H, Hq, D, s));
    if (wide) {
      CK(pack_qkv(tmp, w->wq[l], w->wk[l], w->wv[l], H, Hkv, HPG, D, s));
      CK(pack_kchunk(qkv, tmp, (long)Hkv * (HPG + 2) * D, H, s));
      CK(pack_interleave(tmp, w->w_gate[l], w->w_up[l], d.ffn, H, s));
      CK(pack_kchunk(gu, tmp, 2L * d.ffn, H, s));
      CK(pack_rows(tmp, w->w_down[l], H, d.ffn, s));
      CK(pack_kchunk(dT, tmp, H, d.ffn, s));
    } else {
      CK(pack_qkv(qkv, w->wq[l], w->wk[l], w->wv[l], H, Hkv, HPG, D, s));
    }
    if (wide) {
      // packed above
    } else if (!moe) {
      CK(pack_interleave(gu, w->w_gate[l], w->w_up[l], d.ffn, H, s));
      if (mlp_split(d))  // the down rows are streamed as they are
        CK(cudaMemcpyAsync(dT, w->w_down[l], ls.dT * 2, cudaMemcpyDeviceToDevice, s));
      else if (mlp_split_batched(d))  // units of BD_ROWS rows x BD_KC columns
        CK(pack_down_tiles(dT, w->w_down[l], H, d.ffn, s));
      else
        CK(pack_transpose(dT, w->w_down[l], H, d.ffn, 1, s));
    } else {
      CK(pack_rows(rt, w->router[l], d.n_experts, H, s));
      CK(pack_interleave(egu, w->ex_gate[l], w->ex_up[l], (long)d.n_experts * d.expert_ffn, H,
                         s));
      CK(pack_transpose(edT, w->ex_down[l], H, d.expert_ffn, d.n_experts, s));
      if (d.shared_ffn > 0) {
        CK(pack_interleave(sgu, w->sh_gate[l], w->sh_up[l], d.shared_ffn, H, s));
        CK(pack_transpose(sdT, w->sh_down[l], H, d.shared_ffn, 1, s));
      }
    }
    lp.attn_norm = an;
    lp.mlp_norm = mn;
    lp.wqkv = qkv;
    lp.wo = wo;
    lp.wgu = moe ? nullptr : gu;
    lp.wdT = moe ? nullptr : dT;
    lp.router = moe ? rt : nullptr;
    lp.ex_gu = moe ? egu : nullptr;
    lp.ex_dT = moe ? edT : nullptr;
    lp.sh_gu = moe && d.shared_ffn > 0 ? sgu : nullptr;
    lp.sh_dT = moe && d.shared_ffn > 0 ? sdT : nullptr;
    lp.kc = (uint16_t*)kv->k[l];
    lp.vc = (uint16_t*)kv->v[l];
  }
  uint16_t* emb = take(V * H);
  CK(pack_rows(emb, w->embed, (long)V, H, s));
  h->embed = emb;
  if (wide) {  // its own K-chunk-major copy, tied or not
    uint16_t* lm = take(V8 * H);
    CK(pack_rows(tmp, d.tied_lm_head ? w->embed : w->lm_head, (long)V, H, s));
    CK(pack_kchunk(lm, tmp, (long)V, H, s));
    h->lm_head = lm;
  } else if (d.tied_lm_head) {
    h->lm_head = emb;
  } else {
    uint16_t* lm = take(V * H);
    CK(pack_rows(lm, w->lm_head, (long)V, H, s));
    h->lm_head = lm;
  }
  uint16_t* fn = take(H);
  CK(cudaMemcpyAsync(fn, w->final_norm, (size_t)H * 2, cudaMemcpyDeviceToDevice, s));
  h->final_norm = fn;
  return MK_OK;
}

// int8 packing: every streamed matrix quantised per row (quantize_rows_int8),
// then laid out like its bf16 counterpart with 16-code chunks, codes stored
// biased by 128.  The
// embedding stays bf16 for the token gather; the LM head (the embedding
// when tied) gets its own int8 copy.
static int pack_int8(mk_handle* h, const mk_weights* w, const mk_kv* kv, cudaStream_t s) {
  const mk_model_desc& d = h->d;
  const int L = d.n_layers, H = d.hidden, Hq = d.n_q_heads, Hkv = d.n_kv_heads;
  const int D = d.head_dim, HPG = Hq / Hkv, F = d.ffn;
  const size_t V = d.vocab, R = (size_t)Hkv * (HPG + 2) * D;
  const size_t per_layer = 2 * al256((size_t)H * 2) + al256(R * H) + al256((size_t)Hq * D * H) +
                           al256(2 * (size_t)F * H) + al256((size_t)F * H) + al256(R * 4) +
                           2 * al256((size_t)H * 4) + al256(2 * (size_t)F * 4);
  const size_t total = per_layer * L + al256(V * H * 2) + al256(V * H) + al256(V * 4) + al256(H * 2);
  CK(cudaMalloc(&h->packed, total));
  h->packed_bytes = total;
  // codes and scales of the matrices being packed (the largest: QKV, gate +
  // up, or the LM head)
  const size_t tcodes = std::max(std::max(R * H, 2 * (size_t)F * H), V * H);
  const size_t tscales = std::max(std::max(R, 2 * (size_t)F), V);
  struct Tmp {
    void* p = nullptr;
    ~Tmp() {
      if (p) cudaFree(p);
    }
  } tmp;
  CK(cudaMalloc(&tmp.p, al256(tcodes) + tscales * 4));
  int8_t* tc = (int8_t*)tmp.p;
  float* ts = (float*)((char*)tmp.p + al256(tcodes));
  char* p = (char*)h->packed;
  auto take = [&](size_t bytes) {
    char* r = p;
    p += al256(bytes);
    return r;
  };
  h->layers_h.resize(L);
  for (int l = 0; l < L; l++) {
    LayerPtrs& lp = h->layers_h[l];
    std::memset(&lp, 0, sizeof lp);
    uint16_t* an = (uint16_t*)take((size_t)H * 2);
    uint16_t* mn = (uint16_t*)take((size_t)H * 2);
    char* qkv = take(R * H);
    char* wo = take((size_t)Hq * D * H);
    char* gu = take(2 * (size_t)F * H);
    char* dn = take((size_t)F * H);
    float* sqkv = (float*)take(R * 4);
    float* so = (float*)take((size_t)H * 4);
    float* sd = (float*)take((size_t)H * 4);
    float* sgu = (float*)take(2 * (size_t)F * 4);
    CK(cudaMemcpyAsync(an, w->attn_norm[l], (size_t)H * 2, cudaMemcpyDeviceToDevice, s));
    CK(cudaMemcpyAsync(mn, w->mlp_norm[l], (size_t)H * 2, cudaMemcpyDeviceToDevice, s));
    // QKV: q, k, v codes side by side, then the bf16 packer on 2-code units
    const size_t nq = (size_t)Hq * D, nk = (size_t)Hkv * D;
    CK(quantize_rows_int8(tc, ts, w->wq[l], (long)nq, H, s));
    CK(quantize_rows_int8(tc + nq * H, ts + nq, w->wk[l], (long)nk, H, s));
    CK(quantize_rows_int8(tc + (nq + nk) * H, ts + nq + nk, w->wv[l], (long)nk, H, s));
    CK(pack_qkv((uint16_t*)qkv, tc, tc + nq * H, tc + (nq + nk) * H, H / 2, Hkv, HPG, D, s));
    CK(pack_qkv_scales(sqkv, ts, ts + nq, ts + nq + nk, Hkv, HPG, D, s));
    CK(quantize_rows_int8(tc, so, w->wo[l], H, Hq * D, s));
    CK(pack_wo_i8(wo, tc, H, Hq, s));
    CK(quantize_rows_int8(tc, ts, w->w_gate[l], F, H, s));
    CK(quantize_rows_int8(tc + (size_t)F * H, ts + F, w->w_up[l], F, H, s));
    CK(pack_interleave((uint16_t*)gu, tc, tc + (size_t)F * H, F, H / 2, s));
    CK(interleave_scales(sgu, ts, ts + F, F, s));
    CK(quantize_rows_int8((int8_t*)dn, sd, w->w_down[l], H, F, s));  // rows as they are
    // the kernel reads codes biased by 128
    CK(bias_codes(qkv, R * H, s));
    CK(bias_codes(wo, (size_t)Hq * D * H, s));
    CK(bias_codes(gu, 2 * (size_t)F * H, s));
    CK(bias_codes(dn, (size_t)F * H, s));
    lp.attn_norm = an;
    lp.mlp_norm = mn;
    lp.wqkv = (const uint16_t*)qkv;
    lp.wo = (const uint16_t*)wo;
    lp.wgu = (const uint16_t*)gu;
    lp.wdT = (const uint16_t*)dn;
    lp.sqkv = sqkv;
    lp.so = so;
    lp.sgu = sgu;
    lp.sd = sd;
    lp.kc = (uint16_t*)kv->k[l];
    lp.vc = (uint16_t*)kv->v[l];
  }
  uint16_t* emb = (uint16_t*)take(V * H * 2);
  CK(pack_rows(emb, w->embed, (long)V, H, s));
  h->embed = emb;
  char* lm = take(V * H);
  float* lms = (float*)take(V * 4);
  CK(quantize_rows_int8(tc, lms, d.tied_lm_head ? w->embed : w->lm_head, (long)V, H, s));
  CK(pack_rows((uint16_t*)lm, tc, (long)V, H / 2, s));
  CK(bias_codes(lm, V * H, s));
  h->lm_head = (const uint16_t*)lm;
  h->lm_scale = lms;
  uint16_t* fn = (uint16_t*)take((size_t)H * 2);
  CK(cudaMemcpyAsync(fn, w->final_norm, (size_t)H * 2, cudaMemcpyDeviceToDevice, s));
  h->final_norm = fn;
  CK(cudaStreamSynchronize(s));  // before the temporary codes are freed
  return MK_OK;
}

static int create_checked(const mk_model_desc* desc, const mk_weights* w, const mk_kv* kv,
                          int wfmt, mk_handle** out) {
  if (!out) return MK_ERR_INVALID_ARG;
  *out = nullptr;
  if (!desc) return MK_ERR_INVALID_ARG;
  mk_handle* h = new (std::nothrow) mk_handle();
  if (!h) return MK_ERR_INVALID_ARG;
  const int rc = create_impl(desc, w, kv, h, wfmt);
  if (rc != MK_OK) {
    free_all(h);
    cudaGetLastError();
    return rc;
  }
  *out = h;
  return MK_OK;
}

extern "C" int mk_create_ex(const mk_model_desc* desc, const mk_weights* w, const mk_kv* kv,
                            int weight_format, mk_handle** out) {
  return create_checked(desc, w, kv, weight_format, out);
}

extern "C" int mk_quantize_rows_int8(const void* d_w, long rows, int cols, int8_t* d_codes,
                                     float* d_scales, void* stream) {
  if (rows < 0 || cols <= 0 || (rows > 0 && (!d_w || !d_codes || !d_scales)))
    return MK_ERR_INVALID_ARG;
  CK(quantize_rows_int8(d_codes, d_scales, d_w, rows, cols, (cudaStream_t)stream));
  return MK_OK;
}

extern "C" int mk_create(const mk_model_desc* desc, const mk_weights* w, const mk_kv* kv,
                         mk_handle** out) {
  return create_checked(desc, w, kv, MK_WEIGHTS_BF16, out);
}

// ------------------------------------------------------------- schedule ----
extern "C" int mk_build_schedule(mk_handle* h, int batch, int max_ctx) {
  if (!h) return MK_ERR_INVALID_ARG;
  CK(cudaStreamSynchronize(h->own));
  free_schedule(h);
  PlanOut p;
  int rc = plan_build(h->d, batch, max_ctx, h->n_sm, p, h->hold_mask, h->var->WB);
  if (rc) return rc;
  if (plan_verify(h->d, batch, p)) return MK_ERR_SCHEDULE;
  if (plan_check(p.q.data(), h->n_sm, p.max_pc, p.n_ctr)) return MK_ERR_SCHEDULE;
  const mk_model_desc& d = h->d;
  const size_t L = d.n_layers, B = batch;
  const size_t total = carve_scratch(d, B, h->kc, p.splits, p.n_lm, p.n_ctr, nullptr).total;
  CK(cudaMalloc(&h->scratch, total));
  h->scratch_bytes = total;
  h->sc = carve_scratch(d, B, h->kc, p.splits, p.n_lm, p.n_ctr, (char*)h->scratch);
  CK(cudaMemsetAsync(h->scratch, 0, total, h->own));
  CK(cudaMalloc(&h->sched, p.q.size() * sizeof(Instr)));
  CK(cudaMemcpyAsync(h->sched, p.q.data(), p.q.size() * sizeof(Instr), cudaMemcpyHostToDevice,
                     h->own));
  // staging of the host-buffer step: tokens, positions, argmax, logits
  const size_t st = al256(B * 4) * 3 + al256(B * (size_t)d.vocab * 4);
  CK(cudaMalloc(&h->d_tok, st));
  h->d_pos = (int32_t*)((char*)h->d_tok + al256(B * 4));
  h->d_am = (int32_t*)((char*)h->d_pos + al256(B * 4));
  h->d_logits = (float*)((char*)h->d_am + al256(B * 4));
  // ablation queues: for every (layer, phase) key in step order, each SM's
  // instructions of that key alone (in queue order), one queue per SM that
  // owns any, HALT-padded -- so a launch walks only its own work
  {
    // (the LM head and the final norm carry layer L)
    auto key_of = [&](const Instr& I) { return (size_t)I.layer * N_PHASES + phase_of(I); };
    Instr halt;
    std::memset(&halt, 0, sizeof halt);
    halt.op = OP_HALT;
    std::vector<Instr> flat;
    for (size_t k = 0; k < (L + 1) * N_PHASES; k++) {
      std::vector<std::vector<Instr>> qs;
      for (int sm = 0; sm < h->n_sm; sm++) {
        std::vector<Instr> q;
        for (int pc = 0; pc < p.max_pc; pc++) {
          const Instr& I = p.q[(size_t)sm * p.max_pc + pc];
          if (I.op == OP_HALT) break;
          if (I.op != OP_NOP && key_of(I) == k) q.push_back(I);
        }
        if (!q.empty()) qs.push_back(std::move(q));
      }
      if (qs.empty()) continue;
      size_t mx = 0;
      for (auto& q : qs) mx = std::max(mx, q.size());
      mk_handle::AblLaunch a{flat.size(), (int)qs.size(), (int)mx + 1};
      for (auto& q : qs) {
        q.resize(mx + 1, halt);
        flat.insert(flat.end(), q.begin(), q.end());
      }
      h->abl.push_back(a);
    }
    CK(cudaMalloc(&h->abl_sched, flat.size() * sizeof(Instr)));
    CK(cudaMemcpyAsync(h->abl_sched, flat.data(), flat.size() * sizeof(Instr),
                       cudaMemcpyHostToDevice, h->own));
    CK(cudaStreamSynchronize(h->own));  // before `flat` goes out of scope
  }
  h->plan = std::move(p);
  h->batch = batch;
  h->max_ctx = max_ctx;
  h->epoch = 0;
  CK(cudaStreamSynchronize(h->own));
  return MK_OK;
}

static Globals make_globals(const mk_handle* h, const int32_t* tok, const int32_t* pos,
                            float* logits, int32_t* am) {
  const mk_model_desc& d = h->d;
  Globals g;
  std::memset(&g, 0, sizeof g);
  g.sched = h->sched;
  g.layers = h->layers_d;
  g.embed = h->embed;
  g.lm_scale = h->lm_scale;
  g.lm_head = h->lm_head;
  g.final_norm = h->final_norm;
  g.rope = h->rope;
  g.xbuf = h->sc.xbuf;
  g.qbuf = h->sc.qbuf;
  g.part = h->sc.part;
  g.rlog = h->sc.rlog;
  g.xt = h->sc.xt;
  g.hglob = h->sc.hglob;
  g.act = h->sc.act;
  g.tmaps = h->kv_block ? nullptr : h->tmaps;  // (a paged cache: the CUDA-core attention)
  g.Bp = wide_bp(h->batch);
  g.arr_ctr = (uint32_t)CtrMap{d.n_kv_heads, d.n_layers}.count();
  g.routes = h->sc.routes;
  g.rweight = h->sc.rweight;
  g.lm_val = h->sc.lm_val;
  g.lm_idx = h->sc.lm_idx;
  g.ctr = h->sc.ctr;
  g.err = h->sc.err;
  g.tokens = tok;
  g.positions = pos;
  g.logits = logits;
  g.argmax = am;
  g.timeout_ns = h->timeout_ns;
  g.n_pollers = h->n_pollers;
  g.poll_stagger_ns = h->poll_stagger_ns;
  g.max_pc = h->plan.max_pc;
  g.n_sm = h->n_sm;
  g.n_stages = h->n_stages;
  g.stage_bytes = h->stage_bytes;
  g.B = h->batch;
  g.H = d.hidden;
  g.Hq = d.n_q_heads;
  g.Hkv = d.n_kv_heads;
  g.D = d.head_dim;
  g.F = d.ffn;
  g.V = d.vocab;
  g.L = d.n_layers;
  g.max_seq = d.max_seq;
  g.max_ctx = h->max_ctx;
  g.splits = h->plan.splits;
  g.E = d.n_experts;
  g.K = d.n_experts > 0 ? d.top_k : 0;
  g.Fe = d.expert_ffn;
  g.Fs = d.shared_ffn;
  g.kc = h->kc;
  g.xtag = mlp_split(d) ? 1 : 0;
  g.bsplit = mlp_split_batched(d) ? 1 : 0;
  g.eps = d.rms_eps;
  g.lm_ctr = CtrMap{d.n_kv_heads, d.n_layers}.lm();
  g.lm_done_ctr = CtrMap{d.n_kv_heads, d.n_layers}.lm_done();
  g.part_staged = part_staged(h->plan.splits, h->var->NB, d.head_dim) ? 1 : 0;
  g.kv_block = h->kv_block;
  g.kv_blocks = h->kv_blocks;
  g.kv_table = h->kv_table;
  g.kv_stride = h->kv_stride;
  g.stress_ns = h->stress_ns;
  g.stress_seed = h->stress_seed;
  g.qperm = h->qperm;
  g.n_steps = 1;
  g.n_lm = h->plan.n_lm;
  g.trace = h->trace;
  g.l2_ahead = h->l2_ahead;
  g.hold_early = h->hold_early;
  g.sc_lo = (const unsigned char*)h->scratch;
  g.sc_bytes = h->scratch_bytes;
  g.pk_lo = (const unsigned char*)h->packed;
  g.pk_bytes = h->packed_bytes;
  g.kv_elems = h->kv_block ? (size_t)h->kv_blocks * d.n_kv_heads * h->kv_block * d.head_dim
                           : (size_t)d.max_batch * d.n_kv_heads * d.max_seq * d.head_dim;
  g.n_xbuf = h->sc.xbuf_bytes / 4;
  g.n_q = h->sc.n_q;
  g.n_part = h->sc.n_part;
  g.n_h = h->sc.n_h;
  g.n_xt = h->sc.n_xt;
  g.n_lmv = h->sc.n_lm;
  return g;
}

static cudaError_t launch_mega(const mk_handle* h, Globals& g, cudaStream_t s) {
  void* args[] = {&g};
  return cudaLaunchCooperativeKernel(h->var->kernel, dim3(h->n_sm), dim3(NTHREADS), args,
                                     (size_t)h->smem_bytes, s);
}

extern "C" int mk_decode_step(mk_handle* h, const int32_t* d_tokens, const int32_t* d_positions,
                              float* d_logits, int32_t* d_argmax, void* stream) {
  if (!h) return MK_ERR_INVALID_ARG;
  if (!h->sched) return MK_ERR_NOT_READY;
  if (!d_tokens || !d_positions || !d_logits || !d_argmax) return MK_ERR_INVALID_ARG;
  Globals g = make_globals(h, d_tokens, d_positions, d_logits, d_argmax);
  g.epoch = ++h->epoch;
  g.zero_next = 1;
  CK(launch_mega(h, g, (cudaStream_t)stream));
  return MK_OK;
}

extern "C" int mk_decode_steps(mk_handle* h, const int32_t* d_tokens, const int32_t* d_positions,
                               int n_steps, float* d_logits, int32_t* d_argmax, void* stream) {
  if (!h) return MK_ERR_INVALID_ARG;
  if (!h->sched) return MK_ERR_NOT_READY;
  if (!d_tokens || !d_positions || !d_logits || !d_argmax || n_steps < 1) return MK_ERR_INVALID_ARG;
  Globals g = make_globals(h, d_tokens, d_positions, d_logits, d_argmax);
  g.epoch = h->epoch + 1;
  h->epoch += (uint32_t)n_steps;
  g.n_steps = n_steps;
  g.zero_next = 1;
  CK(launch_mega(h, g, (cudaStream_t)stream));
  return MK_OK;
}

static void reset_after_error(mk_handle* h) {
  cudaMemset(h->sc.ctr, 0, h->sc.ctr_bytes);
  cudaMemset(h->sc.xbuf, 0, h->sc.xbuf_bytes);
  cudaMemset(h->sc.xt, 0, h->sc.tag_bytes);  // the next step is epoch 1 again
  cudaMemset(h->sc.err, 0, h->sc.err_bytes);
  cudaDeviceSynchronize();
  h->epoch = 0;
}

extern "C" int mk_decode_step_host(mk_handle* h, const int32_t* h_tokens,
                                   const int32_t* h_positions, float* h_logits,
                                   int32_t* h_argmax) {
  if (!h) return MK_ERR_INVALID_ARG;
  if (!h->sched) return MK_ERR_NOT_READY;
  if (!h_tokens || !h_positions || !h_argmax) return MK_ERR_INVALID_ARG;
  const int B = h->batch;
  for (int b = 0; b < B; b++)
    if (h_tokens[b] < 0 || h_tokens[b] >= h->d.vocab || h_positions[b] < 0 ||
        h_positions[b] >= h->max_ctx)
      return MK_ERR_INVALID_ARG;
  cudaStream_t s = h->own;
  CK(cudaMemcpyAsync(h->d_tok, h_tokens, B * 4, cudaMemcpyHostToDevice, s));
  CK(cudaMemcpyAsync(h->d_pos, h_positions, B * 4, cudaMemcpyHostToDevice, s));
  Globals g = make_globals(h, h->d_tok, h->d_pos, h->d_logits, h->d_am);
  g.epoch = ++h->epoch;
  g.zero_next = 1;
  CK(launch_mega(h, g, s));
  if (h_logits)
    CK(cudaMemcpyAsync(h_logits, h->d_logits, (size_t)B * h->d.vocab * 4, cudaMemcpyDeviceToHost,
                       s));
  CK(cudaMemcpyAsync(h_argmax, h->d_am, B * 4, cudaMemcpyDeviceToHost, s));
  CK(cudaMemcpyAsync(h->h_err, h->sc.err, 4 * sizeof(int), cudaMemcpyDeviceToHost, s));
  CK(cudaStreamSynchronize(s));
  if (h->h_err[0] != 0) {
    const int code = h->h_err[0];
    reset_after_error(h);
    return code;
  }
  return MK_OK;
}

// ------------------------------------------------------------- ablation ----
// One launch per (layer, phase), each over its own compacted queues and with
// one CTA per queue.  Tracing and the race-stress queue permutation index the
// full schedule, so neither applies here (stress delays still do).
static cudaError_t launch_phases(mk_handle* h, Globals g, cudaStream_t s, bool pdl) {
  g.trace = nullptr;
  g.qperm = nullptr;
  for (const mk_handle::AblLaunch& a : h->abl) {
    g.sched = h->abl_sched + a.off;
    g.max_pc = a.max_pc;
    g.pdl = pdl ? 1 : 0;
    void* args[] = {&g};
    cudaError_t e;
    if (pdl) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(a.n_q);
      cfg.blockDim = dim3(NTHREADS);
      cfg.dynamicSmemBytes = (size_t)h->smem_bytes;
      cfg.stream = s;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      at[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      e = cudaLaunchKernelExC(&cfg, h->var->kernel, args);
    } else {
      e = cudaLaunchKernel(h->var->kernel, dim3(a.n_q), dim3(NTHREADS), args,
                           (size_t)h->smem_bytes, s);
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

extern "C" int mk_decode_step_ablation(mk_handle* h, int mode, const int32_t* d_tokens,
                                       const int32_t* d_positions, float* d_logits,
                                       int32_t* d_argmax, void* stream) {
  if (!h) return MK_ERR_INVALID_ARG;
  if (!h->sched) return MK_ERR_NOT_READY;
  if (!d_tokens || !d_positions || !d_logits || !d_argmax) return MK_ERR_INVALID_ARG;
  if (mode != MK_ABL_STREAM && mode != MK_ABL_GRAPH && mode != MK_ABL_PDL)
    return MK_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  Globals g = make_globals(h, d_tokens, d_positions, d_logits, d_argmax);
  if (mode != MK_ABL_GRAPH) {
    g.epoch = ++h->epoch;
    g.zero_next = 1;
    CK(launch_phases(h, g, s, mode == MK_ABL_PDL));
    return MK_OK;
  }
  // Graph mode: a self-contained replay -- zero the counters and both
  // residual sets, then run the step as epoch 1 (parity 1).
  auto key = std::make_tuple((const void*)d_tokens, (const void*)d_positions, (const void*)d_logits,
                             (const void*)d_argmax, (const void*)h->sched);
  auto it = h->graphs.find(key);
  if (it == h->graphs.end()) {
    CK(cudaStreamSynchronize(h->own));
    g.epoch = 1;
    g.zero_next = 0;
    cudaGraph_t graph = nullptr;
    CK(cudaStreamBeginCapture(h->own, cudaStreamCaptureModeThreadLocal));
    cudaError_t e1 = cudaMemsetAsync(h->sc.ctr, 0, h->sc.ctr_bytes, h->own);
    cudaError_t e2 = cudaMemsetAsync(h->sc.xbuf, 0, h->sc.xbuf_bytes, h->own);
    // every replay runs as epoch 1: clear the previous replay's step tags
    if (!e2) e2 = cudaMemsetAsync(h->sc.xt, 0, h->sc.tag_bytes, h->own);
    cudaError_t e3 = launch_phases(h, g, h->own, false);
    cudaError_t e4 = cudaStreamEndCapture(h->own, &graph);
    if (e1 || e2 || e3 || e4) {
      if (graph) cudaGraphDestroy(graph);
      cudaGetLastError();
      return MK_ERR_CUDA;
    }
    cudaGraphExec_t exec = nullptr;
    cudaError_t e5 = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e5 != cudaSuccess) return MK_ERR_CUDA;
    it = h->graphs.emplace(key, exec).first;
  }
  CK(cudaGraphLaunch(it->second, s));
  h->epoch = 1;  // counters now stand at one step; parity-0 residuals are zero
  return MK_OK;
}

// --------------------------------------------------------------- status ----
extern "C" int mk_sync_status(mk_handle* h, void* stream) {
  if (!h) return MK_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MK_ERR_CUDA;
  if (!h->sc.err) return MK_OK;
  if (cudaMemcpy(h->h_err, h->sc.err, 4 * sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MK_ERR_CUDA;
  if (h->h_err[0] != 0) {
    const int code = h->h_err[0];
    reset_after_error(h);
    return code;
  }
  return MK_OK;
}

extern "C" int mk_set_wait_timeout(mk_handle* h, uint64_t ns) {
  if (!h || ns < 1000) return MK_ERR_INVALID_ARG;
  h->timeout_ns = ns;
  for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second);
  h->graphs.clear();
  return MK_OK;
}

// ------------------------------------------------- no-allocation step ----
// Some callers cannot allocate device memory at the moment they decode: a
// serving loop whose device memory is owned by another allocator (a pooled
// or budgeted arena that forbids stray cudaMalloc calls), code that must not
// hit the synchronising cudaMalloc/cudaFree paths on a latency-critical
// thread, or a host that hands this library a handle built earlier but no
// memory of its own.  For them, mk_decode_step_noalloc runs the very same
// decode kernel with its scratch (residual stream, q, attention partials,
// router logits, argmax slots, counters and error word) carved out of the
// fixed array below instead of the handle's scratch.  The array is a
// file-scope __device__ object: every GPU that loads this library holds it
// until the process exits.
#define MK_NOALLOC_SCRATCH_BYTES (16u << 20)
static __device__ __align__(256) unsigned char mk_noalloc_scratch[MK_NOALLOC_SCRATCH_BYTES];

static std::mutex g_noalloc_mu;
static void* g_noalloc_base[64];  // device address of the array, per device

extern "C" int mk_decode_step_noalloc(mk_handle* h, const int32_t* d_tokens,
                                      const int32_t* d_positions, float* d_logits,
                                      int32_t* d_argmax, int32_t* d_status, void* stream) {
  if (!h) return MK_ERR_INVALID_ARG;
  if (!h->sched) return MK_ERR_NOT_READY;
  if (!d_tokens || !d_positions || !d_logits || !d_argmax) return MK_ERR_INVALID_ARG;
  int dev = -1;
  CK(cudaGetDevice(&dev));
  if (dev != h->dev || dev < 0 || dev >= 64) return MK_ERR_INVALID_ARG;
  // the same carve as the handle's scratch, sized for this handle's schedule
  const mk_model_desc& d = h->d;
  const size_t need =
      carve_scratch(d, h->batch, h->kc, h->plan.splits, h->plan.n_lm, h->plan.n_ctr, nullptr).total;
  if (need > MK_NOALLOC_SCRATCH_BYTES) return MK_ERR_SCRATCH;
  // set-up, once per device, with that device current: the host-side name of
  // the array is not a device address, so look the address up
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_base[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, mk_noalloc_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return MK_ERR_CUDA;
      }
      g_noalloc_base[dev] = p;
    }
    base = g_noalloc_base[dev];
  }
  cudaStream_t s = (cudaStream_t)stream;
  const Scratch sc =
      carve_scratch(d, h->batch, h->kc, h->plan.splits, h->plan.n_lm, h->plan.n_ctr, (char*)base);
  Globals g = make_globals(h, d_tokens, d_positions, d_logits, d_argmax);
  g.xbuf = sc.xbuf;
  g.qbuf = sc.qbuf;
  g.part = sc.part;
  g.rlog = sc.rlog;
  g.lm_val = sc.lm_val;
  g.lm_idx = sc.lm_idx;
  g.ctr = sc.ctr;
  g.err = sc.err;
  g.xt = sc.xt;
  g.hglob = sc.hglob;
  g.routes = sc.routes;    // MoE routing of this call, in the array as well
  g.rweight = sc.rweight;
  g.act = sc.act;          // wide batch: the tensor-core operands, likewise
  g.sc_lo = (const unsigned char*)base;
  g.sc_bytes = need;
  // the array keeps the previous call's contents: clear what must start at
  // zero (residual accumulators of both parities, counters, error word, step
  // tags) and run the step as epoch 1
  CK(cudaMemsetAsync(g.xbuf, 0, sc.xbuf_bytes, s));
  CK(cudaMemsetAsync(g.ctr, 0, sc.ctr_bytes, s));
  CK(cudaMemsetAsync(g.err, 0, sc.err_bytes, s));
  CK(cudaMemsetAsync(g.xt, 0, sc.tag_bytes, s));
  g.epoch = 1;
  g.zero_next = 0;
  g.trace = nullptr;
  CK(launch_mega(h, g, s));
  if (d_status) CK(cudaMemcpyAsync(d_status, g.err, sizeof(int32_t), cudaMemcpyDeviceToDevice, s));
  return MK_OK;
}

extern "C" int mk_set_hold_policy(mk_handle* h, unsigned mask, uint64_t early_bytes) {
  if (!h || mask > 63u || early_bytes > (64ull << 20)) return MK_ERR_INVALID_ARG;
  h->hold_mask = mask;
  h->hold_early = (unsigned)early_bytes;
  return MK_OK;
}

extern "C" int mk_set_poll_policy(mk_handle* h, int pollers, unsigned stagger_ns) {
  if (!h || pollers < 1 || pollers > NCW || stagger_ns > 100000u) return MK_ERR_INVALID_ARG;
  h->n_pollers = pollers;
  h->poll_stagger_ns = stagger_ns;
  for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second);
  h->graphs.clear();
  return MK_OK;
}

extern "C" int mk_debug_read(mk_handle* h, int what, int layer, float* out, size_t n) {
  if (!h || !out) return MK_ERR_INVALID_ARG;
  if (!h->scratch || h->batch <= 0 || h->epoch == 0) return MK_ERR_NOT_READY;
  const mk_model_desc& d = h->d;
  const size_t B = h->batch, L = d.n_layers, H = d.hidden, F = d.ffn > 0 ? d.ffn : 0;
  const size_t HqD = (size_t)d.n_q_heads * d.head_dim;
  CK(cudaDeviceSynchronize());  // the step may have run on any stream
  switch (what) {
    case MK_DBG_Q: {
      if (layer < 0 || (size_t)layer >= L || n < B * HqD) return MK_ERR_INVALID_ARG;
      CK(cudaMemcpy(out, h->sc.qbuf + (size_t)layer * B * HqD, B * HqD * 4,
                    cudaMemcpyDeviceToHost));
      return MK_OK;
    }
    case MK_DBG_X: {
      if (layer < 1 || (size_t)layer > 2 * L || n < B * H) return MK_ERR_INVALID_ARG;
      const size_t j = (size_t)layer;
      if (j % 2 == 0 && mlp_split(d)) {  // x_{2l+2} as the down rows' tagged words
        std::vector<TagWord> t(B * H);
        CK(cudaMemcpy(t.data(), h->sc.xt + (j / 2 - 1) * B * H, t.size() * sizeof(TagWord),
                      cudaMemcpyDeviceToHost));
        for (size_t i = 0; i < t.size(); i++) std::memcpy(out + i, &t[i].bits, 4);
        return MK_OK;
      }
      // the step's parity, summed over the partial copies
      const size_t kc = (size_t)h->kc, par = h->epoch & 1u;
      std::vector<float> v(kc * B * H);
      CK(cudaMemcpy(v.data(), h->sc.xbuf + ((par * 2 * L + (j - 1)) * kc) * B * H, v.size() * 4,
                    cudaMemcpyDeviceToHost));
      for (size_t i = 0; i < B * H; i++) {
        float s = 0.f;
        for (size_t c = 0; c < kc; c++) s += v[c * B * H + i];
        out[i] = s;
      }
      return MK_OK;
    }
    case MK_DBG_H: {
      if (!mlp_split(d)) return MK_ERR_UNSUPPORTED;
      if (layer < 0 || (size_t)layer >= L || n < B * F) return MK_ERR_INVALID_ARG;
      CK(cudaMemcpy(out, h->sc.hglob + (size_t)layer * B * F, B * F * 4, cudaMemcpyDeviceToHost));
      return MK_OK;
    }
    default:
      return MK_ERR_INVALID_ARG;
  }
}

extern "C" int mk_set_race_stress(mk_handle* h, unsigned max_delay_ns, unsigned seed,
                                  int permute_queues) {
  if (!h || max_delay_ns > 100000u || (permute_queues != 0 && permute_queues != 1))
    return MK_ERR_INVALID_ARG;
  CK(cudaStreamSynchronize(h->own));
  if (h->qperm) {
    CK(cudaFree(h->qperm));
    h->qperm = nullptr;
  }
  if (permute_queues) {
    // a seeded Fisher-Yates shuffle of the queues over the CTAs
    std::vector<int> perm(h->n_sm);
    for (int i = 0; i < h->n_sm; i++) perm[i] = i;
    uint64_t x = 0x9E3779B97F4A7C15ull ^ seed;
    for (int i = h->n_sm - 1; i > 0; i--) {
      x ^= x << 13;
      x ^= x >> 7;
      x ^= x << 17;
      std::swap(perm[i], perm[(int)(x % (uint64_t)(i + 1))]);
    }
    CK(cudaMalloc(&h->qperm, perm.size() * sizeof(int)));
    CK(cudaMemcpy(h->qperm, perm.data(), perm.size() * sizeof(int), cudaMemcpyHostToDevice));
  }
  h->stress_ns = max_delay_ns;
  h->stress_seed = seed;
  for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second);
  h->graphs.clear();
  return MK_OK;
}

extern "C" int mk_set_kv_pages(mk_handle* h, int block, int n_blocks, const int32_t* d_table,
                               int table_stride) {
  if (!h) return MK_ERR_INVALID_ARG;
  if (block == 0) {  // back to the contiguous cache
    h->kv_block = h->kv_blocks = h->kv_stride = 0;
    h->kv_table = nullptr;
  } else {
    if (block < 16 || block > 4096 || (block & (block - 1)) || n_blocks < 1 || !d_table ||
        table_stride < 1 || (long)table_stride * block < h->d.max_seq)
      return MK_ERR_INVALID_ARG;
    h->kv_block = block;
    h->kv_blocks = n_blocks;
    h->kv_table = d_table;
    h->kv_stride = table_stride;
  }
  for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second);
  h->graphs.clear();
  return MK_OK;
}

extern "C" int mk_set_ring_depth(mk_handle* h, int max_stages) {
  if (!h || max_stages < 0 || max_stages == 1 || max_stages > MAX_STAGES) return MK_ERR_INVALID_ARG;
  const int old = h->max_stages;
  h->max_stages = max_stages;
  const int st = size_ring(h, h->stage_bytes);
  if (st != MK_OK) {
    h->max_stages = old;
    size_ring(h, h->stage_bytes);
    return st;
  }
  for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second);
  h->graphs.clear();
  return MK_OK;
}

extern "C" int mk_set_stage_bytes(mk_handle* h, int stage_bytes) {
  if (!h || stage_bytes < STAGE_UNIT || stage_bytes > MAX_STAGE_BYTES ||
      stage_bytes % STAGE_UNIT != 0)
    return MK_ERR_INVALID_ARG;
  // wide batch: a stage holds a 128-row K chunk of weights (16 KB) and the
  // operand's chunk (up to 8 KB)
  if (h->var->NB > 8 && stage_bytes < 2 * STAGE_UNIT) return MK_ERR_UNSUPPORTED;
  const int old = h->stage_bytes;
  const int st = size_ring(h, stage_bytes);
  if (st != MK_OK) {
    size_ring(h, old);
    return st;
  }
  for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second);
  h->graphs.clear();
  return MK_OK;
}

extern "C" int mk_set_residual_copies(mk_handle* h, int copies) {
  if (!h || copies < 1 || copies > 8) return MK_ERR_INVALID_ARG;
  h->kc = copies;
  return MK_OK;
}

extern "C" int mk_set_l2_prefetch(mk_handle* h, uint64_t bytes_ahead) {
  if (!h) return MK_ERR_INVALID_ARG;
  h->l2_ahead = bytes_ahead;
  for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second);
  h->graphs.clear();
  return MK_OK;
}

extern "C" int mk_get_info(const mk_handle* h, mk_info* out) {
  if (!h || !out) return MK_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof *out);
  out->n_sm = h->n_sm;
  out->stage_bytes = h->stage_bytes;
  out->n_stages = h->n_stages;
  out->smem_bytes = h->smem_bytes;
  out->max_pc = h->plan.max_pc;
  out->n_instr = h->plan.n_instr;
  out->n_counters = h->plan.n_ctr;
  out->attn_splits = h->plan.splits;
  out->launches_per_step = 1;
  out->ablation_launches = (int)h->abl.size();
  out->batch = h->batch;
  out->max_ctx = h->max_ctx;
  out->packed_bytes = h->packed_bytes;
  out->scratch_bytes = h->scratch_bytes;
  out->weight_bytes_per_step = h->plan.weight_bytes;
  return MK_OK;
}

extern "C" int mk_set_trace(mk_handle* h, int on) {
  if (!h) return MK_ERR_INVALID_ARG;
  if (!h->sched) return MK_ERR_NOT_READY;
  CK(cudaStreamSynchronize(h->own));
  for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second);
  h->graphs.clear();
  if (!on) {
    if (h->trace) cudaFree(h->trace);
    h->trace = nullptr;
    return MK_OK;
  }
  if (!h->trace) {
    const size_t n = (size_t)h->n_sm * h->plan.max_pc * 8;
    CK(cudaMalloc(&h->trace, n * sizeof(unsigned long long)));
    CK(cudaMemset(h->trace, 0, n * sizeof(unsigned long long)));
  }
  return MK_OK;
}

extern "C" int mk_get_trace(mk_handle* h, uint64_t* out, size_t n) {
  if (!h || !out) return MK_ERR_INVALID_ARG;
  if (!h->trace) return MK_ERR_NOT_READY;
  const size_t need = (size_t)h->n_sm * h->plan.max_pc * 8;
  if (n < need) return MK_ERR_INVALID_ARG;
  CK(cudaDeviceSynchronize());
  CK(cudaMemcpy(out, h->trace, need * sizeof(uint64_t), cudaMemcpyDeviceToHost));
  return MK_OK;
}

extern "C" int mk_get_routes(mk_handle* h, int32_t* out, size_t n) {
  if (!h || !out) return MK_ERR_INVALID_ARG;
  if (!h->sched) return MK_ERR_NOT_READY;
  if (h->d.n_experts == 0) return MK_ERR_UNSUPPORTED;
  const size_t need = (size_t)h->d.n_layers * h->d.top_k;
  if (n < need) return MK_ERR_INVALID_ARG;
  CK(cudaDeviceSynchronize());
  CK(cudaMemcpy(out, h->sc.routes, need * sizeof(int32_t), cudaMemcpyDeviceToHost));
  return MK_OK;
}

extern "C" int mk_debug_drop_instruction(mk_handle* h, int sm, int pc) {
  if (!h) return MK_ERR_INVALID_ARG;
  if (!h->sched) return MK_ERR_NOT_READY;
  if (sm < 0 || sm >= h->n_sm || pc < 0 || pc >= h->plan.max_pc) return MK_ERR_INVALID_ARG;
  const size_t i = (size_t)sm * h->plan.max_pc + pc;
  Instr& I = h->plan.q[i];
  if (I.op == OP_HALT) return MK_ERR_INVALID_ARG;
  I.op = OP_NOP;
  CK(cudaMemcpy(h->sched + i, &I, sizeof(Instr), cudaMemcpyHostToDevice));
  return MK_OK;
}

extern "C" int mk_destroy(mk_handle* h) {
  if (!h) return MK_ERR_INVALID_ARG;
  if (h->own) cudaStreamSynchronize(h->own);
  free_all(h);
  return MK_OK;
}

extern "C" const char* mk_status_string(int status) {
  switch (status) {
    case MK_OK: return "ok";
    case MK_ERR_INVALID_ARG: return "invalid argument";
    case MK_ERR_CUDA: return "CUDA runtime error";
    case MK_ERR_UNSUPPORTED: return "unsupported shape (no compiled kernel variant)";
    case MK_ERR_SCHEDULE: return "schedule failed its deadlock or coverage check";
    case MK_ERR_TIMEOUT: return "a device wait exceeded its time limit";
    case MK_ERR_NOT_READY: return "no schedule built";
    case MK_ERR_DEVICE: return "device reported an internal inconsistency";
    case MK_ERR_SCRATCH:
      return "workload needs more scratch than the 16 MiB no-allocation array holds";
    case MK_ERR_BOUNDS:
      return "bounds-checked build: an access fell outside its buffer";
    default: return "unknown status";
  }
}
