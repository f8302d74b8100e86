// attn_tc.cuh -- one split-KV attention work item on the tensor cores, for
// the batched variants (64-dim heads, 2 or 4 query heads per kv head).
//
// The producer loads each ring stage's K half and V half with tiled TMA
// copies (cp.async.bulk.tensor, 64-row boxes) in the 128-byte swizzle: in a
// 1024-byte aligned tile, 16-byte chunk j of row r sits at slot j ^ (r & 7),
// so the eight rows an ldmatrix reads at one column offset hit eight bank
// groups.  Per 16-position chunk a warp computes
//   S = [q_hi; q_lo] K^T        (mma.sync m16n8k16, bf16 in, f32 accumulate:
//                                rows h and h + HPG summed give q . k with an
//                                activation of about 16 mantissa bits)
// then the online-softmax update of each head (running max m, sum l, in
// log2 units), and
//   O += [p_hi; p_lo] V         (p as bf16 high part and remainder, the S
//                                accumulator fragment reused as the A
//                                fragment of the next MMA).
// Row P of the cache (appended this step) is run as one more chunk from a
// small zero-padded tile.  The result per warp is the same partial state as
// the CUDA-core body's: o = sum p v, m, l per head, merged across warps by
// the caller.
#pragma once
#include "mk_device.cuh"

namespace mk {

// Tiled 2-D TMA load of one box (x = column, y = row) into shared memory,
// completing on the mbarrier's transaction count.
MK_DEV void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar,
                        uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// Four 8x8 b16 matrices from shared memory, transposed: register m of lane
// 4g + t holds matrix m's elements (row 2t, column g) and (row 2t + 1,
// column g).
MK_DEV void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// Shared address of 16-byte chunk j of row r of a swizzled tile.
MK_DEV uint32_t swz(uint32_t tile, uint32_t r, uint32_t j) {
  return tile + r * 128u + (((j ^ r) & 7u) << 4);
}

MK_DEV uint32_t pack_bf16x2(float a, float b) {
  return (uint32_t)to_bf16(a) | ((uint32_t)to_bf16(b) << 16);
}

// Per-thread state of one warp's share of an item.  Lane 4g + t works on
// row g of the MMA tiles: g < HPG the high part of head g, HPG <= g < 2 HPG
// the low part of head g - HPG, larger g nothing (rows of zeros).
template <int HPG>
struct AttnTC {
  static_assert(HPG == 2 || HPG == 4, "hi and lo rows of a head in one 8-row half");
  uint32_t qa[4][4];  // A fragments of [q_hi; q_lo] per 16-dim k-step (rows g + 8: zero)
  float m, l;         // running max and this thread's share of the sum, for head g % HPG
  float o[8][4];      // O[row g][8 dt + 2t, + 1] in [dt][0, 1] ([2, 3]: rows g + 8, zero)

  // q: the item's HPG query heads, [HPG][64] f32, scaled by qs
  MK_DEV void init(const float* q, float qs, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const int h = g % HPG;
    const bool hi = g < HPG, live = g < 2 * HPG;
#pragma unroll
    for (int ks = 0; ks < 4; ks++)
#pragma unroll
      for (int half = 0; half < 2; half++) {
        const int d0 = 16 * ks + 8 * half + 2 * t;
        float v[2] = {0.f, 0.f};
        if (live) {
#pragma unroll
          for (int e = 0; e < 2; e++) {
            const float x = __ldcg(q + h * 64 + d0 + e) * qs;
            v[e] = hi ? x : x - bf1(to_bf16(x));
          }
        }
        qa[ks][2 * half] = pack_bf16x2(v[0], v[1]);
        qa[ks][2 * half + 1] = 0u;
      }
    m = NEG_BIG;
    l = 0.f;
#pragma unroll
    for (int dt = 0; dt < 8; dt++)
#pragma unroll
      for (int e = 0; e < 4; e++) o[dt][e] = 0.f;
  }

  // Positions r0 .. r0 + 15 of the K and V tiles (shared addresses of
  // 1024-byte aligned swizzled tiles), of which the first nv are valid.  V
  // rows past nv must hold finite values (callers zero them).
  MK_DEV void chunk(uint32_t kt, uint32_t vt, uint32_t r0, int nv, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const uint32_t li = (uint32_t)lane & 7u, mi = (uint32_t)lane >> 3;
    float s[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; nt++) {
      float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kq = 0; kq < 2; kq++) {
        // matrices: dims 32 kq + 8 mi .. +7 of positions r0 + 8 nt + li
        uint32_t b0, b1, b2, b3;
        ldsm_x4(swz(kt, r0 + 8u * nt + li, 4u * kq + mi), b0, b1, b2, b3);
        mma_16816(d, qa[2 * kq], b0, b1);
        mma_16816(d, qa[2 * kq + 1], b2, b3);
      }
      s[nt][0] = d[0];
      s[nt][1] = d[1];
    }
    // high + low rows of each head (rows g and g ^ HPG sit 4 HPG lanes apart)
#pragma unroll
    for (int nt = 0; nt < 2; nt++)
#pragma unroll
      for (int e = 0; e < 2; e++) {
        s[nt][e] += __shfl_xor_sync(0xFFFFFFFFu, s[nt][e], 4 * HPG);
        if (8 * nt + 2 * t + e >= nv || g >= 2 * HPG) s[nt][e] = -INFINITY;
      }
    float mx = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
    const float mn = fmaxf(m, mx);
    const float cr = exp2f(m - mn);
    m = mn;
    float p[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; nt++)
#pragma unroll
      for (int e = 0; e < 2; e++) p[nt][e] = exp2f(s[nt][e] - mn);
    l = fmaf(l, cr, (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]));
#pragma unroll
    for (int dt = 0; dt < 8; dt++) {
      o[dt][0] *= cr;
      o[dt][1] *= cr;
    }
    // A = [p_hi; p_lo]: row g, positions 2t, 2t+1 (n-tile 0) and 2t+8, 2t+9
    const bool hi = g < HPG;
    auto part = [&](float x) { return hi ? x : x - bf1(to_bf16(x)); };
    const uint32_t a[4] = {pack_bf16x2(part(p[0][0]), part(p[0][1])), 0u,
                           pack_bf16x2(part(p[1][0]), part(p[1][1])), 0u};
#pragma unroll
    for (int dq = 0; dq < 4; dq++) {
      // matrices: positions r0 + 8 (mi & 1) + li, dims 16 dq + 8 (mi >> 1) ..
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(swz(vt, r0 + 8u * (mi & 1u) + li, 2u * dq + (mi >> 1)), b0, b1, b2, b3);
      mma_16816(o[2 * dq], a, b0, b1);
      mma_16816(o[2 * dq + 1], a, b2, b3);
    }
  }

  // Lanes g < HPG end with head g's o[8 dt + 2t, + 1] (dt = 0..7), m and l
  // over this warp's positions.
  MK_DEV void finish() {
#pragma unroll
    for (int dt = 0; dt < 8; dt++) {
      o[dt][0] += __shfl_xor_sync(0xFFFFFFFFu, o[dt][0], 4 * HPG);
      o[dt][1] += __shfl_xor_sync(0xFFFFFFFFu, o[dt][1], 4 * HPG);
    }
    l += __shfl_xor_sync(0xFFFFFFFFu, l, 1);
    l += __shfl_xor_sync(0xFFFFFFFFu, l, 2);
  }
};

}  // namespace mk
