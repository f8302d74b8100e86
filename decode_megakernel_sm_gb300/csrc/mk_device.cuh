// mk_device.cuh -- device helpers of the interpreter: inline PTX for mbarriers,
// bulk copies and release/acquire counters, bounded waits, bf16 unpacking.
//
// Counter protocol ("Megakernels: Deleting the Kernel Boundary", section
// "Correctness without the free barrier"): a producer makes its stores
// visible device-wide and then increments a counter; a consumer spins until
// the counter reaches its target.  Here the increment is a release pattern
// (fence.release.gpu, then a relaxed reduction) issued by one thread after a
// CTA barrier, the
// spin is an acquire load (ld.acquire.gpu), and every spin is bounded by
// %globaltimer so that a missing producer turns into an error status, never
// a hung GPU.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "mk_internal.h"

namespace mk {

#define MK_DEV __device__ __forceinline__

MK_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Start value of a running softmax maximum (finite, so that max - start
// never forms inf - inf).
constexpr float NEG_BIG = -1e30f;

MK_DEV uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Generic-proxy shared-memory stores ordered before later async-proxy
// accesses of the same bytes (tensor-core operand reads, bulk-copy writes).
MK_DEV void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

MK_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

MK_DEV bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

MK_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

MK_DEV void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

MK_DEV uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

MK_DEV uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Non-multicast bulk copy global -> this CTA's shared memory, completing on
// the mbarrier's transaction count.  dst, src and bytes are multiples of 16.
MK_DEV void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                     uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Warm L2 with a global range ahead of its bulk copy (no shared memory, no
// completion tracking).  src and bytes are multiples of 16.
MK_DEV void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Warm L2 with one 128-byte line through the load/store unit.
MK_DEV void prefetch_l2_line(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Fire-and-forget float reductions into global memory (no return value, so
// the issuing thread never waits for the L2 round trip).
MK_DEV void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

MK_DEV void red_add_v2f32(float* p, float a, float b) {
  asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(p), "f"(a), "f"(b) : "memory");
}

MK_DEV void red_add_v4f32(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

MK_DEV uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

MK_DEV uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// A reduction with no release semantics: it orders nothing before it, and
// so does not wait for this SM's outstanding memory operations.
MK_DEV void red_relaxed(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Release pattern: a release fence, then a relaxed reduction.  While bulk
// copies are in flight on the SM this waits about half as long as a
// red.release (which orders the thread's earlier loads as well).
MK_DEV void red_release(uint32_t* p, uint32_t v) {
  asm volatile("fence.release.gpu;" ::: "memory");
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Acquire-release increment: a release fence, then an acquiring atomic.
MK_DEV uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("fence.release.gpu;" ::: "memory");
  asm volatile("atom.acquire.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

// Barrier among the consumer warps only (the producer warp never joins).
MK_DEV void consumer_bar() { asm volatile("bar.sync 1, %0;" ::"n"(NCT) : "memory"); }

MK_DEV float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
MK_DEV float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
MK_DEV float bf1(uint16_t h) { return __uint_as_float(((uint32_t)h) << 16); }
MK_DEV uint16_t to_bf16(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

// Shared-memory store that the compiler does not treat as touching other
// memory, so global loads around it may still be issued early (ordering
// against later shared-memory reads comes from the barrier between them).
MK_DEV void st_shared_f4(const void* p, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(p)), "f"(a), "f"(b),
               "f"(c), "f"(d));
}

// Two floats as bf16x2 pairs: hi = bf16(v) (nearest), lo = bf16(v - hi), so
// hi + lo carries ~16 mantissa bits of v (lower column in the low half).
MK_DEV void split2(float v0, float v1, uint32_t& hi, uint32_t& lo) {
  const uint16_t h0 = to_bf16(v0), h1 = to_bf16(v1);
  const uint16_t l0 = to_bf16(v0 - bf1(h0)), l1 = to_bf16(v1 - bf1(h1));
  hi = (uint32_t)h0 | ((uint32_t)h1 << 16);
  lo = (uint32_t)l0 | ((uint32_t)l1 << 16);
}

// Four 8x8 b16 matrices from shared memory; lane 8m + i gives row i of
// matrix m, and register m receives this lane's pair of matrix m (row
// lane / 4, columns 2 (lane % 4), +1).
MK_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// d += A (16x16 bf16, row-major fragment a) x B (16x8 bf16, column-major
// fragment b0, b1), f32 accumulate.
MK_DEV void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 4-byte asynchronous global -> shared copy (the LSU path, not the bulk-copy
// engine); cp_async_wait_all waits for this thread's copies.
MK_DEV void cp_async4(float* sdst, const float* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(sdst)), "l"(gsrc)
               : "memory");
}
MK_DEV void cp_async16(void* sdst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(sdst)), "l"(gsrc)
               : "memory");
}
MK_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Two fp32 lanes in one 64-bit register, and the packed f32x2 arithmetic of
// sm_100+ (two IEEE fp32 operations per instruction, each rounded as the
// scalar one).
MK_DEV unsigned long long f2_bits(float2 v) {
  return ((unsigned long long)__float_as_uint(v.y) << 32) | __float_as_uint(v.x);
}
MK_DEV float2 bits_f2(unsigned long long u) {
  return make_float2(__uint_as_float((uint32_t)u), __uint_as_float((uint32_t)(u >> 32)));
}
MK_DEV float2 ffma2(float2 a, float2 b, float2 c) {  // a * b + c
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)), "l"(f2_bits(c)));
  return bits_f2(d);
}
MK_DEV float2 fadd2(float2 a, float2 b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(d);
}

// int8 weight codes, stored biased by 128 (byte u = q + 128, 1..255).  Byte
// k of a word as the low mantissa byte of 2^23 (bits 0x4B0000uu) is exactly
// 2^23 + u; subtracting 2^23 + 128 leaves q exactly.  i8_pair gives codes
// k, k + 1 of a word: two byte permutes and one packed add.
MK_DEV float2 i8_pair(uint32_t biased, int k) {
  const float2 m = make_float2(
      __uint_as_float(__byte_perm(biased, 0x4B000000u, 0x7440u | (uint32_t)k)),
      __uint_as_float(__byte_perm(biased, 0x4B000000u, 0x7440u | (uint32_t)(k + 1))));
  return fadd2(m, make_float2(-8388736.f, -8388736.f));
}

MK_DEV void unpack8(const uint4& w, float* f) {
  f[0] = bf_lo(w.x); f[1] = bf_hi(w.x);
  f[2] = bf_lo(w.y); f[3] = bf_hi(w.y);
  f[4] = bf_lo(w.z); f[5] = bf_hi(w.z);
  f[6] = bf_lo(w.w); f[7] = bf_hi(w.w);
}

MK_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

MK_DEV int peek_err(const Globals& g) { return *(volatile const int*)g.err; }

// The queue this CTA runs (a permutation of the CTAs under race stress).
MK_DEV int queue_id(const Globals& g) { return g.qperm ? __ldg(g.qperm + blockIdx.x) : (int)blockIdx.x; }

// Race stress: sleep a pseudo-random time below g.stress_ns, a function of
// (queue, pc, step, seed, side).  Only timing changes: no wait is skipped.
MK_DEV void stress_delay(const Globals& g, int q, int pc, int step, uint32_t side) {
  uint32_t h = (uint32_t)q * 0x9E3779B1u ^ (uint32_t)pc * 0x85EBCA6Bu ^
               (uint32_t)step * 0xC2B2AE35u ^ g.stress_seed ^ side;
  h ^= h >> 15;
  h *= 0x2C1B3C6Du;
  h ^= h >> 12;
  __nanosleep(h % g.stress_ns);
}

MK_DEV void set_err(const Globals& g, int code, int pc, int op) {
  if (atomicCAS(g.err, 0, code) == 0) {
    g.err[1] = (int)blockIdx.x;
    g.err[2] = pc;
    g.err[3] = op;
  }
}

// ---- bounds-checked build -------------------------------------------------
// With MK_BOUNDS defined (the libmk_bounds.so build), MK_IN(g, cond, pc, op)
// checks an access before it happens: a violation records MK_ERR_BOUNDS (with
// the SM, pc and op) in the error word, and the caller skips the access, so
// nothing traps and no out-of-range address is ever touched.  Without it the
// check is the constant true and compiles away.
#ifdef MK_BOUNDS
MK_DEV bool mk_in(const Globals& g, bool ok, int pc, int op) {
  if (!ok) set_err(g, MK_ERR_BOUNDS, pc, op);
  return ok;
}
#define MK_IN(g, cond, pc, op) mk_in((g), (cond), (pc), (op))
#else
#define MK_IN(g, cond, pc, op) true
#endif

// [p, p + bytes) inside [lo, lo + n)
MK_DEV bool span_in(const void* p, size_t bytes, const void* lo, size_t n) {
  const unsigned char *a = (const unsigned char*)p, *b = (const unsigned char*)lo;
  return a >= b && a + bytes <= b + n;
}

// ---- KV cache rows -------------------------------------------------------
// Element offset of cache row p of (sequence b, kv head h): contiguous
// [B][Hkv][max_seq][D], or paged -- block kv_table[b][p / blk] of the pool
// [blocks][Hkv][blk][D] (the layout keeps a block's rows of one kv head
// contiguous, one bulk copy per block).  -1 if the table names a block
// outside the pool (the caller turns that into MK_ERR_INVALID_ARG).
MK_DEV long long kv_row(const Globals& g, int b, int h, int p) {
  if (g.kv_block == 0) return (((long long)b * g.Hkv + h) * g.max_seq + p) * g.D;
  const int j = p / g.kv_block;
  if (j >= g.kv_stride) return -1;
  const int blk = __ldg(g.kv_table + (size_t)b * g.kv_stride + j);
  if (blk < 0 || blk >= g.kv_blocks) return -1;
  return (((long long)blk * g.Hkv + h) * g.kv_block + (p - j * g.kv_block)) * g.D;
}

// ---- tagged words --------------------------------------------------------
// A value produced by exactly one writer per step travels as a 64-bit word
// {f32 value, u32 tag}, tag = the step's epoch, written with one relaxed
// 64-bit store.  Aligned 64-bit accesses are single-copy atomic, so a
// reader that sees this step's tag sees the value stored with it: the writer
// needs no release fence, and the reader needs no counter round trip before
// it loads the data -- it polls the data itself.
MK_DEV void st_tag(TagWord* p, float v, uint32_t tag) {
  const unsigned long long w = ((unsigned long long)tag << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}

MK_DEV void ld_tag2(const TagWord* p, TagWord& a, TagWord& b) {
  unsigned long long x, y;
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(x), "=l"(y) : "l"(p) : "memory");
  a = TagWord{(uint32_t)x, (uint32_t)(x >> 32)};
  b = TagWord{(uint32_t)y, (uint32_t)(y >> 32)};
}

MK_DEV TagWord ld_tag1(const TagWord* p) {
  unsigned long long x;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(x) : "l"(p) : "memory");
  return TagWord{(uint32_t)x, (uint32_t)(x >> 32)};
}

// G groups of NP tagged pairs, group q at p + q * stride (in words); only
// the groups whose bit is set in `valid` are read, and their values land in
// memory (shared memory, as a rule): group q's 2*NP floats at
// dst + q * dst_stride.  Every first read is issued before any tag is
// checked, so a thread's whole input costs one round trip once the last
// writer has stored; only stale pairs are re-read.  Bounded like every
// wait: false if the grid has failed or the deadline passed (then the
// error word is set).
template <int G, int NP>
MK_DEV bool poll_tag_groups_to(const Globals& g, const TagWord* p, size_t stride, uint32_t valid,
                               uint32_t tag, float* dst, int dst_stride, int pc, int op) {
  static_assert(G * NP <= 32, "one bit per pair");
  uint32_t miss = 0;
#pragma unroll
  for (int q = 0; q < G; q++)
#pragma unroll
    for (int i = 0; i < NP; i++) {
      if (valid & (1u << q)) {
        TagWord a, b;
        ld_tag2(p + q * stride + 2 * i, a, b);
        dst[q * dst_stride + 2 * i] = __uint_as_float(a.bits);
        dst[q * dst_stride + 2 * i + 1] = __uint_as_float(b.bits);
        if (a.tag != tag || b.tag != tag) miss |= 1u << (q * NP + i);
      }
    }
  if (miss == 0) return true;
  const uint64_t t0 = gtimer();
  for (uint32_t it = 1;; it++) {
    for (int k = 0; k < G * NP; k++) {
      const uint32_t bit = 1u << k;
      if (miss & bit) {
        const int q = k / NP, i = k % NP;
        TagWord a, b;
        ld_tag2(p + q * stride + 2 * i, a, b);
        dst[q * dst_stride + 2 * i] = __uint_as_float(a.bits);
        dst[q * dst_stride + 2 * i + 1] = __uint_as_float(b.bits);
        if (a.tag == tag && b.tag == tag) miss &= ~bit;
      }
    }
    if (miss == 0) return true;
    if ((it & 15) == 0) {
      if (peek_err(g)) return false;
      if (gtimer() - t0 > g.timeout_ns) {
        set_err(g, MK_ERR_TIMEOUT, pc, op);
        return false;
      }
    }
  }
}

// One tagged float, polled the same way.
MK_DEV bool poll_tag1(const Globals& g, const TagWord* p, uint32_t tag, float& v, int pc, int op) {
  TagWord a = ld_tag1(p);
  if (a.tag != tag) {
    const uint64_t t0 = gtimer();
    for (uint32_t it = 1; (a = ld_tag1(p)).tag != tag; it++) {
      if ((it & 15) == 0) {
        if (peek_err(g)) return false;
        if (gtimer() - t0 > g.timeout_ns) {
          set_err(g, MK_ERR_TIMEOUT, pc, op);
          return false;
        }
      }
    }
  }
  v = __uint_as_float(a.bits);
  return true;
}

// Spin (acquire) until ctr[idx] has reached `target` (wrap-safe).  Returns
// false after an error anywhere in the grid or after the time limit.
template <bool ACQUIRE = true>
MK_DEV bool wait_counter(const Globals& g, uint32_t idx, uint32_t target, int pc, int op) {
  const uint32_t* p = g.ctr + idx;
  auto ld = [](const uint32_t* a) { return ACQUIRE ? ld_acquire(a) : ld_relaxed(a); };
  if ((int32_t)(ld(p) - target) >= 0) return true;
  const uint64_t t0 = gtimer();
  for (uint32_t it = 1;; it++) {
    if ((int32_t)(ld(p) - target) >= 0) return true;
    if ((it & 15) == 0) {
      if (peek_err(g)) return false;
      if (gtimer() - t0 > g.timeout_ns) {
        set_err(g, MK_ERR_TIMEOUT, pc, op);
        return false;
      }
    }
  }
}

// One of several staggered pollers of a counter (one lane per warp): it
// starts after `delay_ns` and stops as soon as any poller has seen the
// counter at `target` (the shared word `seen` then holds `key`).  Each poll
// is an L2 round trip, so n pollers spaced a fraction of a round trip apart
// see the counter complete that much sooner than one.  The poller that
// sees it has acquired; the others are ordered after it by the CTA barrier
// that follows.  Bounded like every wait.
MK_DEV bool poll_counter_shared(const Globals& g, uint32_t idx, uint32_t target, uint64_t delay_ns,
                                volatile int* seen, int key, int pc, int op) {
  const uint32_t* p = g.ctr + idx;
  const uint64_t t0 = gtimer();
  while (delay_ns && gtimer() - t0 < delay_ns)
    if (*seen == key) return true;
  for (uint32_t it = 1;; it++) {
    if (*seen == key) return true;
    if ((int32_t)(ld_acquire(p) - target) >= 0) {
      *seen = key;
      return true;
    }
    if ((it & 15) == 0) {
      if (peek_err(g)) return false;
      if (gtimer() - t0 > g.timeout_ns) {
        set_err(g, MK_ERR_TIMEOUT, pc, op);
        return false;
      }
    }
  }
}

// Wait for a phase of an mbarrier.  abort_on_err: also give up when the
// grid has failed (consumers); the producer's drain passes false so that it
// always waits for its own copies in flight.
MK_DEV bool wait_mbar(const Globals& g, uint32_t bar, uint32_t parity, bool abort_on_err) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  for (uint32_t it = 1;; it++) {
    if (mbar_try(bar, parity)) return true;
    if ((it & 63) == 0) {
      if (abort_on_err && peek_err(g)) return false;
      if (gtimer() - t0 > g.timeout_ns) {
        set_err(g, MK_ERR_TIMEOUT, -1, -1);
        return false;
      }
    }
  }
}

// One contiguous run of equal-sized units (weight rows, or cache rows of K
// with the matching V rows in src2) streamed through the ring, `ups` units
// per stage.  src2 lands in the upper half of the stage.
constexpr uint32_t SEG_CFILL = 0x80000000u;
// A wide-batch segment: unit i (a K chunk) is a weight piece of `unit` bytes
// at src + i * pitch and an operand piece of `unit2` bytes at src2 + i * unit2;
// a stage holds `ups` chunks, the weight pieces first (unit apart), then the
// operand pieces (unit2 apart, from offset ups * unit).  The operand is an
// input of this step: the producer waits for the instruction's dependency
// before it issues any of the segment's copies.  row0 carries the flag, the
// pitch in 128-byte rows in bits [8, 30) and unit2 / 128 in bits [0, 8).
constexpr uint32_t SEG_WIDE = 0x40000000u;
MK_HD inline uint32_t seg_wide_tag(uint32_t pitch, uint32_t unit2) {
  return SEG_WIDE | ((pitch / 128u) << 8) | (unit2 / 128u);
}

struct Seg {
  const unsigned char* src;
  const unsigned char* src2;
  uint32_t unit;
  uint32_t n;
  uint32_t ups;
  uint32_t row0;  // swizzled GEMV matrices: index of the first row in its tensor (key = row & 7);
                  // SEG_CFILL set: an input of this step, whose stages the producer only arms
                  // and the consumers fill once their dependency wait has passed
  MK_DEV bool cfill() const { return (row0 & SEG_CFILL) != 0; }
  MK_DEV bool wide() const { return (row0 & SEG_WIDE) != 0; }
  MK_DEV uint32_t pitch() const { return ((row0 & 0x3FFFFFFFu) >> 8) * 128u; }
  MK_DEV uint32_t unit2() const { return (row0 & 0xFFu) * 128u; }
};

// Ring cursor of one consumer warp.
struct Ring {
  unsigned char* base;
  uint32_t full0, empty0;  // shared addresses of full[0], empty[0]
  int ns;
  int st;
  uint32_t par;
  unsigned long long waited;  // ns spent blocked in acquire (measured only when tracing)
  bool timed;
  uint32_t sb;  // bytes per stage

  MK_DEV const unsigned char* stage_ptr() const { return base + (size_t)st * sb; }
  // the stage j places ahead of the cursor, and its full barrier
  MK_DEV unsigned char* ahead_ptr(int j) const { return base + (size_t)((st + j) % ns) * sb; }
  MK_DEV uint32_t ahead_full(int j) const { return full0 + 8u * (uint32_t)((st + j) % ns); }
  // All 32 lanes call; the result is the same on every lane.
  MK_DEV bool acquire(const Globals& g) {
    bool ok;
    if (timed) {  // try_wait itself may suspend the thread, so time the whole wait
      const uint64_t t0 = gtimer();
      ok = wait_mbar(g, full0 + 8u * st, par, true);
      waited += gtimer() - t0;
    } else {
      ok = wait_mbar(g, full0 + 8u * st, par, true);
    }
    return __all_sync(0xFFFFFFFFu, ok);
  }
  // All 32 lanes call; lane 0 arrives for the warp.
  MK_DEV void release(int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8u * st);
    advance();
  }
  // The cursor moves on without arriving: the warp's arrival comes from
  // elsewhere (a tensor-core commit, once its MMAs have read the stage).
  MK_DEV void advance() {
    if (++st == ns) {
      st = 0;
      par ^= 1u;
    }
  }
  MK_DEV uint32_t empty_bar() const { return empty0 + 8u * st; }
};

}  // namespace mk
