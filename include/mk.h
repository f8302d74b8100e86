/*
 * mk.h -- C ABI of the GB300 decode megakernel library (libmk.so).
 *
 * One low-batch transformer decode step runs as ONE persistent CUDA kernel
 * (one CTA per SM) that interprets a per-SM queue of opcoded instructions,
 * replaces kernel boundaries with a global-memory counter array, and streams
 * weights through a TMA bulk-copy shared-memory ring.  The design follows
 * "Megakernels: Deleting the Kernel Boundary to Win Back Microseconds"
 * (sections "One launch, one interpreter", "Correctness without the free
 * barrier"), re-planned for sm_103a.
 *
 * Conventions
 *  - Every pointer named d_* is a CUDA device pointer; h_* is host memory.
 *  - Weights are bf16 (IEEE binary32 upper halves), row-major [out][in].
 *  - All calls return MK_OK (0) or a negative MK_ERR_* code; no call aborts
 *    the process, and no kernel traps: device-side faults in the schedule
 *    (a wait that never completes) or in the inputs (a token or position
 *    out of range) set a device error word that mk_sync_status() returns.
 *  - A handle is not thread-safe; use one handle per host thread.
 *  - `stream` arguments are cudaStream_t values passed as void* (NULL is the
 *    legacy default stream).
 */
#ifndef MK_H
#define MK_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MK_OK 0
#define MK_ERR_INVALID_ARG (-1) /* bad pointer, shape, token or position          */
#define MK_ERR_CUDA (-2)        /* a CUDA runtime call failed                      */
#define MK_ERR_UNSUPPORTED (-3) /* shape with no compiled kernel variant           */
#define MK_ERR_SCHEDULE (-4)    /* schedule failed its deadlock / coverage check   */
#define MK_ERR_TIMEOUT (-5)     /* a device wait ran past its time limit           */
#define MK_ERR_NOT_READY (-6)   /* mk_build_schedule has not succeeded yet         */
#define MK_ERR_DEVICE (-7)      /* device reported an internal inconsistency       */
#define MK_ERR_SCRATCH (-8)     /* scratch need exceeds the fixed no-allocation array */
#define MK_ERR_BOUNDS (-9)      /* bounds-checked build only: an access fell outside its buffer */

typedef struct mk_handle mk_handle;

/* Decoder shape.  Dense MLP when n_experts == 0 (ffn used); otherwise a
 * routed MoE MLP with n_experts experts of width expert_ffn, top_k of them
 * per token, plus an always-on shared expert of width shared_ffn (0: none).
 * "Gemma 4 TPU megakernel", section "Megakernels for Gemma 4", lists the
 * router / experts / shared MLP components of that MoE step.  Supported:
 * n_experts <= 256, top_k <= 16 (MK_ERR_UNSUPPORTED otherwise).
 * batched_variant picks the kernel for max_batch 2..8 on a dense shape with
 * 64-dim heads, four query heads per kv head and hidden / ffn multiples of
 * 64: 0 (default) the wide-batch variant (every contraction on tcgen05 with
 * tensor-memory accumulators; measured 14-21 % faster per step at 2, 4 and
 * 7 sequences), 1 the batched variant (warp-level mma.sync).  Other shapes
 * and max_batch 9..32 ignore it (the wide-batch variant).  "Megakernels in LLM Inference When Fusion
 * Actually Wins", section "Core Tradeoff", frames the batch ranges.        */
typedef struct {
  int n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
  float rms_eps, rope_theta;
  int tied_lm_head;                 /* 1: the LM head is the embedding matrix */
  int n_experts, top_k, expert_ffn, shared_ffn;
  int max_batch, max_seq;           /* KV cache capacity (rows per kv head)   */
  int batched_variant;              /* 2..8 sequences: 0 tcgen05, 1 mma.sync  */
} mk_model_desc;

/* Weight pointers (device, bf16).  Per-layer fields are HOST arrays of
 * n_layers device pointers.  mk_create copies (and re-lays-out) every weight
 * into a library-owned buffer, so the caller may free its copies after
 * mk_create returns.  Fields a model does not use may be NULL.
 *   embed [vocab][hidden], lm_head [vocab][hidden] (NULL when tied),
 *   final_norm [hidden], attn_norm/mlp_norm [hidden],
 *   wq [n_q_heads*head_dim][hidden], wk/wv [n_kv_heads*head_dim][hidden],
 *   wo [hidden][n_q_heads*head_dim],
 *   dense: w_gate/w_up [ffn][hidden], w_down [hidden][ffn],
 *   MoE:   router [n_experts][hidden], ex_gate/ex_up [n_experts][expert_ffn][hidden],
 *          ex_down [n_experts][hidden][expert_ffn],
 *          sh_gate/sh_up [shared_ffn][hidden], sh_down [hidden][shared_ffn].   */
typedef struct {
  const void* embed;
  const void* lm_head;
  const void* final_norm;
  const void* const* attn_norm;
  const void* const* wq;
  const void* const* wk;
  const void* const* wv;
  const void* const* wo;
  const void* const* mlp_norm;
  const void* const* w_gate;
  const void* const* w_up;
  const void* const* w_down;
  const void* const* router;
  const void* const* ex_gate;
  const void* const* ex_up;
  const void* const* ex_down;
  const void* const* sh_gate;
  const void* const* sh_up;
  const void* const* sh_down;
} mk_weights;

/* KV cache, caller-owned, bf16.  k[l], v[l] (HOST arrays of n_layers device
 * pointers) each point at [max_batch][n_kv_heads][max_seq][head_dim], 16-byte
 * aligned.  Rows [0, P) of sequence b must hold the already-rotated keys and
 * the values of earlier positions; mk_decode_step writes row P in place.
 * The cache must stay allocated for the life of the handle.               */
typedef struct {
  void* const* k;
  void* const* v;
} mk_kv;

/* Create a handle on the current CUDA device: validates the shape, selects
 * the compiled kernel variant (MK_ERR_UNSUPPORTED if none), copies and packs
 * the weights on the device (synchronous), allocates counters and scratch.
 * Passage: "Megakernels: Deleting the Kernel Boundary to Win Back
 * Microseconds", opening paragraph (batch-1 decode reads every weight once
 * per forward pass, so the packed weights are laid out for one contiguous
 * stream per instruction) and section "Correctness without the free
 * barrier", last paragraph (weights prefetched into paged shared memory:
 * here a bulk-copy ring, which is why every matrix is re-laid out).
 * Ownership: the caller keeps its weights (read only during the call) and
 * its KV cache (must outlive the handle); the library owns the packed copy.
 * Batch capacity: max_batch 1 (the batch-1 variants), 2..32 (the wide-batch
 * variant: every contraction on the tcgen05 tensor cores with the
 * accumulator in tensor memory; dense FFN of whole 64-column chunks, hidden
 * size a multiple of 64, 64-dim heads, bf16 weights -- "Megakernels in LLM
 * Inference When Fusion Actually Wins", sections "Core Tradeoff" and "When
 * Megakernels Win", the batch range up to 32 where the crossover lies) or
 * 2..8 (the batched variant, warp-level mma.sync: other shapes, or
 * batched_variant 1).
 * Errors: MK_ERR_INVALID_ARG for a NULL or non-16-byte-aligned pointer or an
 * inconsistent shape, MK_ERR_UNSUPPORTED (no compiled variant, or a wide
 * batch outside the conditions above), MK_ERR_CUDA.
 * On error *out is NULL and nothing is leaked.                            */
int mk_create(const mk_model_desc* desc, const mk_weights* w, const mk_kv* kv, mk_handle** out);

/* Weight formats of mk_create_ex. */
#define MK_WEIGHTS_BF16 0 /* as mk_create */
#define MK_WEIGHTS_INT8 1 /* int8 codes with one fp32 scale per row           */

/* mk_create with a choice of streamed weight format (int8 weight
 * streaming; "Gemma 4 TPU megakernel", section "What's next":
 * the same kernel reaches a higher rate with INT8 experts, because decode is
 * bound by the weight bytes it reads).  The caller still passes bf16 weights.
 * MK_WEIGHTS_INT8 quantises every streamed matrix on the device, row by row,
 * exactly as mk_quantize_rows_int8 does: QKV, O-projection, gate, up, down
 * and the LM head (with a tied head, an int8 copy of the embedding; the
 * token gather still reads the bf16 embedding).  Norm gains and the KV cache
 * stay bf16.  The step then computes y[r] = s[r] * sum_k q[r][k] * x[k] for
 * every such matrix; everything else is as with bf16 weights.
 * An int8 handle starts with a ring of at most 4 stages (mk_set_ring_depth
 * changes it).  Supported: dense models with batch capacity 1 (max_batch ==
 * 1), hidden 2048, head_dim 64, 4 query heads per kv head, ffn a multiple
 * of 16 and at most 8192, vocab at most hidden x (SM count);
 * MK_ERR_UNSUPPORTED otherwise.  Errors and ownership as mk_create.       */
int mk_create_ex(const mk_model_desc* desc, const mk_weights* w, const mk_kv* kv,
                 int weight_format, mk_handle** out);

/* The row quantiser of MK_WEIGHTS_INT8, on its own.  d_w: device bf16
 * [rows][cols]; d_codes: device int8 [rows][cols]; d_scales: device fp32
 * [rows] (all caller-owned).  Per row: m = max |w|, s = m / 127, q =
 * round-half-even(w / s) clamped to [-127, 127], both divisions correctly
 * rounded in fp32; a row of zeros gets s = 0 and codes 0.  Weights must be
 * finite.  Asynchronous on `stream` (a cudaStream_t, NULL: the default
 * stream).  MK_ERR_INVALID_ARG for negative rows, cols <= 0 or NULL
 * pointers; MK_ERR_CUDA if the launch fails.                              */
int mk_quantize_rows_int8(const void* d_w, long rows, int cols, int8_t* d_codes, float* d_scales,
                          void* stream);

/* Paged KV cache (long-context decode over a block-table cache; the blocks of
 * vLLM-style serving).  From the next step on, kv->k[l] / kv->v[l] given to
 * mk_create point at pools [n_blocks][n_kv_heads][block][head_dim] (bf16,
 * 16-byte aligned), and cache row p of sequence b lives in block
 * d_table[b * table_stride + p / block] at row p % block.  d_table is a
 * caller-owned device int32 array [max_batch][table_stride]; the caller may
 * rewrite it between steps (e.g. to give a growing sequence a new block), and
 * it must name a block for every row a step reads or writes (rows [0, P],
 * and [0, P + n_steps - 1] for mk_decode_steps).  A block id outside
 * [0, n_blocks) fails the step with MK_ERR_INVALID_ARG at mk_sync_status().
 * block: a power of two, 16..4096; table_stride * block >= max_seq.
 * block == 0 returns to the contiguous cache.  Results are the same as with
 * the contiguous cache holding the same rows.  MK_ERR_INVALID_ARG
 * otherwise.                                                               */
int mk_set_kv_pages(mk_handle* h, int block, int n_blocks, const int32_t* d_table,
                    int table_stride);

/* Diagnostics: an intermediate of the handle's most recent step
 * (mk_decode_step, mk_decode_step_host, or the last step of
 * mk_decode_steps; not the no-allocation call), copied to host memory as
 * fp32, for per-phase checks against a reference:
 *   MK_DBG_Q: the queries of layer `layer` after RoPE, [batch][n_q_heads][head_dim];
 *   MK_DBG_X: the residual x_j for j = `layer` in [1, 2 n_layers]: x_{2l+1}
 *             after layer l's O-projection, x_{2l+2} after its MLP, [batch][hidden];
 *   MK_DBG_H: SiLU(gate) * up of layer `layer`, [batch][ffn] (dense batch 1
 *             only; MK_ERR_UNSUPPORTED otherwise).
 * n: capacity of out in floats.  Synchronises the device.
 * MK_ERR_NOT_READY before the first step; MK_ERR_INVALID_ARG for a bad
 * selector, layer or capacity.                                            */
#define MK_DBG_Q 0
#define MK_DBG_X 1
#define MK_DBG_H 2
int mk_debug_read(mk_handle* h, int what, int layer, float* out, size_t n);

/* Race stress for tests (a stress level for the counter protocol; the hazard is
 * the missing fence that "Megakernels: Deleting the Kernel Boundary",
 * section "Correctness without the free barrier", warns of).  With
 * max_delay_ns > 0 the producer warp and consumer thread 0 of every CTA
 * sleep a pseudo-random time below max_delay_ns (a function of queue, pc,
 * step and seed) before each instruction; with permute_queues = 1 the CTAs
 * run the queues in a seeded random permutation.  Only timing and placement
 * change: every wait, fence and signal stays, so results must be those of
 * an unstressed step.  max_delay_ns <= 100000; (0, *, 0) turns it off.
 * Synchronises the handle's stream; drops cached ablation graphs.
 * MK_ERR_INVALID_ARG for out-of-range arguments.                          */
int mk_set_race_stress(mk_handle* h, unsigned max_delay_ns, unsigned seed, int permute_queues);

/* Build the per-SM instruction queues for `batch` sequences whose positions
 * will stay below `max_ctx` (<= max_seq): splits every projection into
 * byte-balanced row ranges, one split-KV attention work item per
 * (sequence, kv head, split), assigns counter ids and targets, checks the
 * queues for deadlock and coverage on the host (MK_ERR_SCHEDULE), uploads
 * them and zeroes the counters.  Synchronous.  Must precede any step.
 * Passage: "Megakernels: Deleting the Kernel Boundary to Win Back
 * Microseconds", section "One launch, one interpreter" (the per-SM
 * instruction schedule is computed on the host ahead of time and reused for
 * many forward passes) and section "Correctness without the free barrier"
 * (a counter array in global memory, zeroed before the launch, replaces the
 * kernel boundaries); the byte balance answers the wave-quantisation tail of
 * section "Where the microseconds go".
 * Errors: MK_ERR_INVALID_ARG (batch outside [1, max_batch], max_ctx outside
 * [1, max_seq]), MK_ERR_UNSUPPORTED, MK_ERR_SCHEDULE, MK_ERR_CUDA; the
 * previous schedule is dropped in every case.                             */
int mk_build_schedule(mk_handle* h, int batch, int max_ctx);

/* One decode step, asynchronous on `stream`, one kernel launch.
 * Passage: "Megakernels: Deleting the Kernel Boundary to Win Back
 * Microseconds", section "One launch, one interpreter" (one persistent
 * kernel, one block per SM, runs the whole forward pass: RMSNorm + QKV +
 * RoPE, attention and its reduce, O-projection + residual, RMSNorm + gate/up
 * + SiLU, down + residual, final RMSNorm + LM head) and the page's opening
 * paragraph (a token per pass; here the argmax of the logits).
 * All buffers are caller-owned device memory; the library writes d_logits,
 * d_argmax and cache row P of every layer.
 *   d_tokens    [batch] int32: token fed at this step (may alias the d_argmax
 *               of the previous step);
 *   d_positions [batch] int32: P, the cache row written by this step; each
 *               sequence attends to rows [0, P]; must satisfy P < max_ctx;
 *   d_logits    [batch][vocab] fp32 output;
 *   d_argmax    [batch] int32 output: first index of the largest logit.
 * Out-of-range tokens or positions are detected on the device before any
 * write; the step then writes nothing and mk_sync_status() returns
 * MK_ERR_INVALID_ARG.                                                     */
int mk_decode_step(mk_handle* h, const int32_t* d_tokens, const int32_t* d_positions,
                   float* d_logits, int32_t* d_argmax, void* stream);

/* n_steps greedy decode steps in one launch ("Megakernels: Deleting the
 * Kernel Boundary", ranked next step: the argmax feeds the next step's
 * embedding on the device).  Step 0 decodes d_tokens at d_positions; step
 * t > 0 decodes step t - 1's argmax at d_positions + t.  The queues run once
 * per step; step t begins once every SM is done with step t - 1, and the
 * producer streams step t's first weights while step t - 1's LM head runs.
 *   d_argmax  [n_steps][batch] int32 output: the argmax of every step;
 *   d_logits  [batch][vocab] fp32 output: the logits of the last step.
 * Requires d_positions[b] + n_steps - 1 < max_ctx (checked on the device
 * before each step: MK_ERR_INVALID_ARG at mk_sync_status(), nothing written
 * for that step and the ones after it).  Asynchronous, one kernel launch.
 * Equivalent to n_steps calls of mk_decode_step, each fed the previous
 * argmax; results agree to float rounding.                                */
int mk_decode_steps(mk_handle* h, const int32_t* d_tokens, const int32_t* d_positions,
                    int n_steps, float* d_logits, int32_t* d_argmax, void* stream);

/* The same step from HOST buffers: copies h_tokens / h_positions to the
 * device, runs the step on the handle's own stream, copies logits (may be
 * NULL to skip) and argmax back, and waits.  Validates tokens and positions
 * on the host first.                                                       */
int mk_decode_step_host(mk_handle* h, const int32_t* h_tokens, const int32_t* h_positions,
                        float* h_logits, int32_t* h_argmax);

/* Ablation: the same instruction bodies, one kernel launch per (layer,
 * phase) instead of one persistent launch.  "Megakernels: Deleting the
 * Kernel Boundary", section "Where the microseconds go", describes the
 * per-operator launch sequence this reproduces.
 *   mode MK_ABL_STREAM: plain launches on `stream`;
 *   mode MK_ABL_GRAPH : the same launches captured once into a CUDA graph
 *                       (cached per argument set) and replayed;
 *   mode MK_ABL_PDL   : plain launches with programmatic dependent launch,
 *                       each kernel starts its weight prefetch before
 *                       waiting on its predecessor.                        */
#define MK_ABL_STREAM 0
#define MK_ABL_GRAPH 1
#define MK_ABL_PDL 2
int mk_decode_step_ablation(mk_handle* h, int mode, const int32_t* d_tokens,
                            const int32_t* d_positions, float* d_logits, int32_t* d_argmax,
                            void* stream);

/* Decode step that allocates nothing -- no counterpart in the pages; it is a
 * service to callers that must not allocate device memory while decoding
 * (their device memory belongs to another allocator or a fixed budget, or
 * they run on a latency-critical thread that must not enter the
 * synchronising cudaMalloc/cudaFree paths).  Same arguments and same kernel
 * as mk_decode_step, but the step's scratch (residual stream, q, attention
 * partials, router logits, argmax slots, counters, error word) lives in a
 * fixed file-scope device array of 16 MiB that every GPU loading this
 * library holds until exit, not in the handle's scratch.  The handle must
 * have a schedule (built earlier, by a caller that could allocate).
 *   d_status (may be NULL): [1] int32 device output that receives the step's
 *            device status (MK_OK, MK_ERR_TIMEOUT, MK_ERR_INVALID_ARG, ...).
 * Everything the step writes besides the caller's outputs and KV cache
 * (MoE routing included) stays in the array, so mk_get_routes and
 * mk_debug_read keep reporting the handle's own most recent step.
 * Returns MK_ERR_SCRATCH, with nothing launched, if the handle's schedule
 * needs more than 16 MiB of scratch.  Each call clears the parts of the
 * array that must start at zero, on `stream`, before its launch; all calls
 * share the one array, so calls that overlap on the GPU (on different
 * streams, or from different handles) race and must be serialised by the
 * caller.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Calls no cudaMalloc / cudaFree.            */
int mk_decode_step_noalloc(mk_handle* h, const int32_t* d_tokens, const int32_t* d_positions,
                           float* d_logits, int32_t* d_argmax, int32_t* d_status, void* stream);

/* Wait for `stream` and return the device error word (MK_OK if none).  A
 * non-OK result also resets the counters and scratch so that the next step
 * starts clean (the KV rows written by the failed step are unspecified).
 * Passage: "Megakernels: Deleting the Kernel Boundary to Win Back
 * Microseconds", section "Correctness without the free barrier": the
 * consumer there spins until a counter reaches its target; here every such
 * wait is bounded in time, and a wait that runs out, or a bad input, sets
 * the error word this call reads instead of hanging the GPU.
 * Errors: MK_ERR_INVALID_ARG (NULL handle), MK_ERR_CUDA (the stream failed),
 * or the device status itself (MK_ERR_TIMEOUT, MK_ERR_INVALID_ARG, ...).  */
int mk_sync_status(mk_handle* h, void* stream);

/* Limit, in nanoseconds, of every device-side wait (default 2 s). */
int mk_set_wait_timeout(mk_handle* h, uint64_t ns);

/* How far (bytes of each SM's own weight / KV stream) the kernel warms L2
 * ahead of its shared-memory ring with cp.async.bulk.prefetch.L2; 0 turns
 * the L2 lookahead off (the default).  A performance knob only: results
 * do not depend on it.                                                     */
int mk_set_l2_prefetch(mk_handle* h, uint64_t bytes_ahead);

/* Bytes per shared-memory ring stage: 16384, 32768, 49152 or 65536
 * (default 65536 on a one-sequence bf16 handle where two such stages fit,
 * and on a wide-batch handle, whose consumer pays a tensor-core commit per
 * stage; 32768 on int8 and on batched mma.sync handles).  The ring holds as many stages (2..16) as the device's
 * opt-in shared memory allows next to the kernel's fixed buffers.  Bigger
 * stages hold more weight rows, so every consumer warp has rows in each
 * stage; smaller stages give a deeper ring.  Results do not depend on it.
 * Call between steps (not while a step is in flight on another stream);
 * drops the cached ablation graphs.  MK_ERR_INVALID_ARG for other sizes,
 * MK_ERR_UNSUPPORTED if two stages no longer fit, or for 16384 on a
 * wide-batch handle (a stage holds a 128-row weight chunk and its operand
 * chunk); the old size is kept.                                            */
int mk_set_stage_bytes(mk_handle* h, int stage_bytes);

/* At most `max_stages` ring stages (2..16; 0, the default: as many as the
 * opt-in shared memory holds).  Fewer stages keep fewer bytes in flight per
 * SM, which shortens the queues every L2 access waits in while HBM streams.
 * A performance knob only: results do not depend on it.  Call between
 * steps; drops the cached ablation graphs.  MK_ERR_INVALID_ARG for 1 or out
 * of range (the old depth is kept).                                        */
int mk_set_ring_depth(mk_handle* h, int max_stages);

/* How an SM waits for a dependency counter: `pollers` warps (1..7) each
 * poll it, the k-th starting k * stagger_ns after the first, and all stop
 * once one has seen it complete.  A poll is an L2 round trip; staggered
 * pollers see the counter complete sooner after the last signal.  Takes
 * effect at the next step.  Results do not depend on it.
 * MK_ERR_INVALID_ARG for other pollers or stagger_ns > 100000.            */
int mk_set_poll_policy(mk_handle* h, int pollers, unsigned stagger_ns);

/* Number of partial copies (1..8, default 1) that each residual-stream
 * vector is accumulated into: SM i adds its float atomics into copy
 * i mod copies and readers sum the copies, which spreads the atomic traffic
 * of the O-projection and MLP slices over more L2 lines.  Takes effect at
 * the next mk_build_schedule.  Results agree to float rounding.            */
int mk_set_residual_copies(mk_handle* h, int copies);

/* Fetch policy at instruction boundaries.  A release fence waits for every
 * memory operation the SM has in flight (bulk copies and L2 prefetches
 * included), so ring copies of the next instruction issued just before the
 * fence that ends the current one slow that fence, and every SM waiting on
 * it.  Instructions of the ops in `mask` (bits: 1 QKV, 2 attention,
 * 4 O-projection, 8 MLP gate/up or fused MLP or router, 16 MLP down rows,
 * 32 LM head) that follow another op on their SM are "held": the producer
 * issues their first `early_bytes` of ring copies (whole stages; 0: none) as
 * usual and the rest only after the consumers have finished, and signalled,
 * every earlier instruction.  Default mask 24 (gate/up and down), 128 KiB.
 * Takes effect at the next mk_build_schedule.  Results do not depend on it.
 * MK_ERR_INVALID_ARG for mask > 63 or early_bytes > 64 MiB.               */
int mk_set_hold_policy(mk_handle* h, unsigned mask, uint64_t early_bytes);

typedef struct {
  int n_sm;               /* CTAs of the persistent kernel (= SMs)          */
  int stage_bytes;        /* bytes per shared-memory ring stage             */
  int n_stages;           /* ring stages                                    */
  int smem_bytes;         /* dynamic shared memory per CTA                  */
  int max_pc;             /* instructions per SM queue (incl. HALT)         */
  int n_instr;            /* instructions in the schedule                   */
  int n_counters;         /* counters in the dependency array               */
  int attn_splits;        /* split-KV slices per (sequence, kv head)        */
  int launches_per_step;  /* megakernel: 1                                  */
  int ablation_launches;  /* launches per step in the ablation modes        */
  int batch, max_ctx;
  size_t packed_bytes;    /* library-owned weight copy                      */
  size_t scratch_bytes;   /* counters + activations + partials              */
  double weight_bytes_per_step; /* weights one step must read (routed MoE: active experts) */
} mk_info;
int mk_get_info(const mk_handle* h, mk_info* out);

/* MoE only: the expert ids the router chose at the most recent step,
 * [n_layers][top_k] int32 in selection order (largest router logit first,
 * lower id first on ties; "Gemma 4 TPU megakernel", section "Megakernels
 * for Gemma 4", component "Router").  Waits for the device.  n = capacity.
 * "Most recent step" means the handle's own steps (mk_decode_step, the
 * host-buffer step, the last step of mk_decode_steps, the ablation): a
 * mk_decode_step_noalloc call keeps its routing in the library's fixed
 * array, so this call does not see it.                                     */
int mk_get_routes(mk_handle* h, int32_t* out, size_t n);

/* Replace instruction `pc` of SM `sm` by a no-op that neither waits nor
 * signals -- a fault-injection aid for tests: every instruction waiting on
 * the dropped one's counter then runs into its time limit and the step
 * fails with MK_ERR_TIMEOUT instead of hanging.  Undone by the next
 * mk_build_schedule.                                                       */
int mk_debug_drop_instruction(mk_handle* h, int sm, int pc);

/* Tracing: when on, every launch records %globaltimer stamps (ns) per
 * instruction into a device buffer [n_sm][max_pc][8]: [0] the producer's
 * first bulk copy of the instruction, [1] the consumers' wait start, [2]
 * wait end, [3] end of the op's prologue phase (norm / split combine), [4]
 * end of its ring loop, [5] body end, [6] nanoseconds warp 0 spent waiting
 * for ring data during the instruction, [7] the moment the instruction's
 * completion signal (a release reduction, which first waits for the SM's
 * earlier memory operations) retired.  Slots of instructions that did not
 * run keep their old values.
 * mk_set_trace(h, 1) allocates the buffer (after mk_build_schedule; a new
 * schedule turns tracing off); mk_get_trace waits for the device and copies
 * the n_sm * max_pc * 8 values to `out` (n = capacity in values).         */
int mk_set_trace(mk_handle* h, int on);
int mk_get_trace(mk_handle* h, uint64_t* out, size_t n);

/* Release everything the library owns for the handle (packed weights,
 * schedule, scratch, streams), after waiting for the handle's own stream.
 * The pages have no counterpart: it ends the life cycle that mk_create
 * starts.  The caller's weights, KV cache and buffers are untouched.
 * MK_ERR_INVALID_ARG for a NULL handle.                                    */
int mk_destroy(mk_handle* h);

/* A static, NUL-terminated English description of a status code (never
 * NULL; "unknown status" for codes this library does not define).  No
 * counterpart in the pages: the library's own error reporting.             */
const char* mk_status_string(int status);

/* ---- host-only planning (no GPU needed) ---------------------------------
 * The schedule builder and its checker, exposed for inspection and tests.
 * Instructions are 32-byte records:
 *   op, flags (u8), layer (u16), b, g (u16), r0, r1, wait_ctr, wait_cnt,
 *   sig_ctr, aux (u32).  op: 0 HALT, 1 QKV, 2 ATTN, 3 OPROJ, 4 MLP (fused
 *   column slice), 5 LMHEAD, 6 ROUTER, 7 NOP, 8 MLP_UP (gate/up column
 *   slice), 9 MLP_DOWN (down rows), 10 NORM (wide batch: RMSNorm of the
 *   sequences [r0, r1) into the tensor-core operand g: 0 attention input,
 *   1 MLP input, 2 LM-head input).  Wide-batch MLP_DOWN: rows [r0, r1) over
 *   the 64-column FFN chunks [b, g); wide-batch OPROJ: kv group g's query
 *   heads; wide-batch LMHEAD: b bit 0 / bit 1 mark the first / last
 *   instruction of an SM's slice aux.  wait_ctr / sig_ctr 0xFFFFFFFF: none. */
typedef struct {
  uint8_t op, flags;
  uint16_t layer;
  uint16_t b, g;
  uint32_t r0, r1;
  uint32_t wait_ctr, wait_cnt;
  uint32_t sig_ctr, aux;
} mk_instr;

typedef struct {
  int n_sm, max_pc, n_instr, n_counters, attn_splits, n_lm;
  double max_sm_bytes, mean_sm_bytes; /* streamed bytes per SM (weights + KV at max_ctx) */
} mk_plan_stats;

/* Build the schedule for `n_sm` SMs on the host.  If `out` is non-NULL and
 * `out_cap` >= n_sm * max_pc records, the queues are written there
 * ([n_sm][max_pc], HALT-padded).  Returns MK_OK or an MK_ERR_* code.     */
int mk_plan(const mk_model_desc* desc, int batch, int max_ctx, int n_sm, mk_plan_stats* stats,
            mk_instr* out, size_t out_cap);

/* Check queues [n_sm][max_pc] against n_counters counters: simulates
 * in-order execution of every queue under the wait semantics; MK_OK if all
 * queues run to HALT, MK_ERR_SCHEDULE on a deadlock (some wait can never be
 * met) or an out-of-range counter id.                                      */
int mk_plan_check(const mk_instr* q, int n_sm, int max_pc, int n_counters);

#ifdef __cplusplus
}
#endif
#endif
