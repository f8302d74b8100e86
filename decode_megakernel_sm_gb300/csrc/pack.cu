// pack.cu -- device-side re-layout of the caller's bf16 weights into the
// instruction-contiguous layouts the interpreter streams (one run per
// instruction, one bulk copy per ring stage, no tensor map needed).
// Every matrix whose rows are dotted with the normalised activation (QKV,
// gate/up, router, experts, embedding / LM head) is chunk-swizzled: 16-byte
// chunk i of row p sits at slot i ^ (p & 7), so 8 consecutive rows read at
// the same column offset land in 8 different shared-memory bank groups
// (ldmatrix over 8 rows is conflict-free; a lane that walks one row just
// XORs its chunk index).
//   QKV   [Hkv][(HPG+2)*D][H]  per kv head: its HPG query heads, then k, then
//                              v; inside a head, rows 2t / 2t+1 = dims t / t+D/2
//   Wo    [Hq][H][D]           one head's columns as contiguous 128/256-byte rows;
//                              16-byte chunk c of row r sits at slot c ^ (r & 7),
//                              so 8 consecutive rows read chunk c from 8
//                              different shared-memory bank groups
//   gate/up [F][2][H]          gate row c, then up row c
//   down  dense batch 1: [H][F] as given (one contiguous row per output row);
//         2..8 sequences, F a multiple of 512: units of 16 rows x 512 columns
//         in chunk-major order (unit kc * (H / 16) + row block), 16-byte
//         chunk q of unit row i at slot q ^ (i & 7);
//         otherwise [F][H], transposed (one contiguous row per FFN column)
//
// int8 weights (dense batch-1 shapes): every matrix is first quantised per
// row (quantize_rows_kernel), then the codes take the same layouts with
// 16-byte chunks of 16 codes (a row of H codes is H / 16 chunks, swizzled
// the same way), except Wo, whose 64-code head rows are 4 chunks: chunk c of
// row r sits at slot c ^ ((r >> 1) & 3).  The packed codes are stored
// biased by 128 (byte q + 128; bias_codes), which the kernel's decode
// expects.  The fp32 row scales follow their rows (QKV: packed row order;
// gate/up: interleaved).
#include <cuda_runtime.h>

#include "mk_internal.h"

namespace mk {

__global__ void pack_qkv_kernel(uint4* __restrict__ dst, const uint16_t* __restrict__ wq,
                                const uint16_t* __restrict__ wk, const uint16_t* __restrict__ wv,
                                int H, int HPG, int D) {
  const int p = blockIdx.x;
  const int GR = (HPG + 2) * D;
  const int g = p / GR, lr = p % GR, hs = lr / D, e = lr % D;
  const int dim = (e & 1) ? (e >> 1) + D / 2 : (e >> 1);
  const uint16_t* src = hs < HPG   ? wq + ((size_t)(g * HPG + hs) * D + dim) * H
                        : hs == HPG ? wk + ((size_t)g * D + dim) * H
                                    : wv + ((size_t)g * D + dim) * H;
  const uint4* s4 = (const uint4*)src;
  uint4* d4 = dst + (size_t)p * (H / 8);
  for (int i = threadIdx.x; i < H / 8; i += blockDim.x) d4[i ^ (p & 7)] = s4[i];
}

// dst row 2c = a row c, dst row 2c+1 = b row c (rows of H elements), swizzled.
__global__ void pack_interleave_kernel(uint4* __restrict__ dst, const uint4* __restrict__ a,
                                       const uint4* __restrict__ b, int H) {
  const size_t c = blockIdx.x;
  const int n = H / 8;
  const int k0 = (int)((2 * c) & 7), k1 = (int)((2 * c + 1) & 7);
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    dst[(2 * c) * n + (i ^ k0)] = a[c * n + i];
    dst[(2 * c + 1) * n + (i ^ k1)] = b[c * n + i];
  }
}

// dst row r = src row r (rows of H elements), swizzled.
__global__ void pack_rows_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, int H) {
  const size_t r = blockIdx.x;
  const int n = H / 8;
  for (int i = threadIdx.x; i < n; i += blockDim.x) dst[r * n + (i ^ (int)(r & 7))] = src[r * n + i];
}

// dst[h][r][c ^ (r & 7)] = wo[r][h*D + 8c : h*D + 8c + 8] (16-byte chunks c).
__global__ void pack_wo_kernel(uint4* __restrict__ dst, const uint4* __restrict__ wo, int H, int Hq,
                               int D) {
  const size_t total = (size_t)Hq * H * (D / 8);
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t slot = i % (D / 8), hr = i / (D / 8);
    const size_t r = hr % H, h = hr / H;
    const size_t c8 = slot ^ (r & 7);
    dst[i] = wo[(r * Hq + h) * (D / 8) + c8];
  }
}

// Batched transpose of bf16 [R][C] -> [C][R]; blockIdx.z selects the matrix.
__global__ void transpose_kernel(uint16_t* __restrict__ dst, const uint16_t* __restrict__ src, int R,
                                 int C) {
  __shared__ uint16_t tile[32][33];
  const size_t off = (size_t)blockIdx.z * R * C;
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int k = threadIdx.y; k < 32; k += blockDim.y) {
    const int r = r0 + k, c = c0 + threadIdx.x;
    if (r < R && c < C) tile[k][threadIdx.x] = src[off + (size_t)r * C + c];
  }
  __syncthreads();
  for (int k = threadIdx.y; k < 32; k += blockDim.y) {
    const int c = c0 + k, r = r0 + threadIdx.x;
    if (r < R && c < C) dst[off + (size_t)c * R + r] = tile[threadIdx.x][k];
  }
}

cudaError_t pack_qkv(uint16_t* dst, const void* wq, const void* wk, const void* wv, int H, int Hkv,
                     int HPG, int D, cudaStream_t s) {
  pack_qkv_kernel<<<Hkv * (HPG + 2) * D, 128, 0, s>>>((uint4*)dst, (const uint16_t*)wq,
                                                      (const uint16_t*)wk, (const uint16_t*)wv, H,
                                                      HPG, D);
  return cudaGetLastError();
}

cudaError_t pack_interleave(uint16_t* dst, const void* a, const void* b, long rows, int H,
                            cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  pack_interleave_kernel<<<(unsigned)rows, 128, 0, s>>>((uint4*)dst, (const uint4*)a,
                                                       (const uint4*)b, H);
  return cudaGetLastError();
}

// Down projection [H][F] as units of BD_ROWS rows x BD_KC columns, unit
// (rb, kc) at ((rb * (F / BD_KC) + kc) * BD_ROWS) rows of BD_KC; inside a
// unit, 16-byte chunk q of unit row i sits at slot q ^ (i & 7).
// Units of BD_ROWS rows x BD_KC columns in chunk-major order: unit
// (chunk kc, row block rb) is unit kc * (H / BD_ROWS) + rb, so a run of
// consecutive units covers consecutive row blocks of one or two chunks.
__global__ void pack_down_tiles_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, int H,
                                       int F) {
  const int nkc = F / BD_KC, cpr = BD_KC / 8, nrb = H / BD_ROWS;
  const size_t r = blockIdx.x / nkc;
  const int kc = (int)(blockIdx.x % nkc);
  const size_t rb = r / BD_ROWS;
  const int i = (int)(r % BD_ROWS);
  uint4* d = dst + (((size_t)kc * nrb + rb) * BD_ROWS + i) * cpr;
  const uint4* sr = src + r * (F / 8) + (size_t)kc * cpr;
  for (int q = threadIdx.x; q < cpr; q += blockDim.x) d[q ^ (i & 7)] = sr[q];
}

cudaError_t pack_down_tiles(uint16_t* dst, const void* src, int H, int F, cudaStream_t s) {
  pack_down_tiles_kernel<<<(unsigned)((size_t)H * (F / BD_KC)), 128, 0, s>>>(
      (uint4*)dst, (const uint4*)src, H, F);
  return cudaGetLastError();
}

cudaError_t pack_rows(uint16_t* dst, const void* src, long rows, int H, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  pack_rows_kernel<<<(unsigned)rows, 128, 0, s>>>((uint4*)dst, (const uint4*)src, H);
  return cudaGetLastError();
}

cudaError_t pack_wo(uint16_t* dst, const void* wo, int H, int Hq, int D, cudaStream_t s) {
  pack_wo_kernel<<<2048, 256, 0, s>>>((uint4*)dst, (const uint4*)wo, H, Hq, D);
  return cudaGetLastError();
}

cudaError_t pack_transpose(uint16_t* dst, const void* src, int R, int C, int batch,
                           cudaStream_t s) {
  if (R <= 0 || C <= 0 || batch <= 0) return cudaSuccess;
  dim3 grid((C + 31) / 32, (R + 31) / 32, batch);
  transpose_kernel<<<grid, dim3(32, 8), 0, s>>>(dst, (const uint16_t*)src, R, C);
  return cudaGetLastError();
}

// Symmetric per-row int8 quantisation of a bf16 matrix [rows][cols], the
// "INT8 experts" of the Gemma 4 TPU megakernel page ("What's next") applied
// to every streamed matrix: with m = max_k |w[r][k]|, the scale is
// s = m / 127 and the code q = round-half-even(w / s) in [-127, 127], both
// divisions correctly rounded in fp32 (a zero row: s = 0, codes 0), so that
// w ~ q * s.  One block per row.
__global__ void quantize_rows_kernel(int8_t* __restrict__ codes, float* __restrict__ scales,
                                     const uint16_t* __restrict__ w, int cols) {
  __shared__ float red[32];
  const size_t r = blockIdx.x;
  const uint16_t* src = w + r * (size_t)cols;
  float m = 0.f;
  for (int k = threadIdx.x; k < cols; k += blockDim.x)
    m = fmaxf(m, fabsf(__uint_as_float((uint32_t)src[k] << 16)));
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (threadIdx.x == 0) red[0] = m;
  }
  __syncthreads();
  const float s = red[0] > 0.f ? __fdiv_rn(red[0], 127.f) : 0.f;
  int8_t* dst = codes + r * (size_t)cols;
  for (int k = threadIdx.x; k < cols; k += blockDim.x) {
    int q = 0;
    if (s > 0.f) {
      q = __float2int_rn(__fdiv_rn(__uint_as_float((uint32_t)src[k] << 16), s));
      q = min(127, max(-127, q));
    }
    dst[k] = (int8_t)q;
  }
  if (threadIdx.x == 0) scales[r] = s;
}

cudaError_t quantize_rows_int8(int8_t* codes, float* scales, const void* w, long rows, int cols,
                               cudaStream_t s) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  quantize_rows_kernel<<<(unsigned)rows, 256, 0, s>>>(codes, scales, (const uint16_t*)w, cols);
  return cudaGetLastError();
}

// Row scales of the packed QKV rows (the row order of pack_qkv_kernel).
__global__ void pack_qkv_scales_kernel(float* __restrict__ dst, const float* __restrict__ sq,
                                       const float* __restrict__ sk, const float* __restrict__ sv,
                                       int HPG, int D, int n) {
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= n) return;
  const int GR = (HPG + 2) * D;
  const int g = p / GR, lr = p % GR, hs = lr / D, e = lr % D;
  const int dim = (e & 1) ? (e >> 1) + D / 2 : (e >> 1);
  dst[p] = hs < HPG ? sq[(g * HPG + hs) * D + dim] : hs == HPG ? sk[g * D + dim] : sv[g * D + dim];
}

cudaError_t pack_qkv_scales(float* dst, const float* sq, const float* sk, const float* sv, int Hkv,
                            int HPG, int D, cudaStream_t s) {
  const int n = Hkv * (HPG + 2) * D;
  pack_qkv_scales_kernel<<<(n + 255) / 256, 256, 0, s>>>(dst, sq, sk, sv, HPG, D, n);
  return cudaGetLastError();
}

// dst[2c] = a[c], dst[2c + 1] = b[c]: gate / up row scales.
__global__ void interleave_scales_kernel(float* __restrict__ dst, const float* __restrict__ a,
                                         const float* __restrict__ b, int n) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c < n) {
    dst[2 * c] = a[c];
    dst[2 * c + 1] = b[c];
  }
}

cudaError_t interleave_scales(float* dst, const float* a, const float* b, int n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  interleave_scales_kernel<<<(n + 255) / 256, 256, 0, s>>>(dst, a, b, n);
  return cudaGetLastError();
}

// int8 Wo codes [H][Hq*64] -> [Hq][H][64]: chunk c of head row r at slot
// c ^ ((r >> 1) & 3) (4 chunks of 16 codes per row).
__global__ void pack_wo_i8_kernel(uint4* __restrict__ dst, const uint4* __restrict__ wo, int H,
                                  int Hq) {
  const size_t total = (size_t)Hq * H * 4;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t slot = i % 4, hr = i / 4;
    const size_t r = hr % H, h = hr / H;
    dst[i] = wo[(r * Hq + h) * 4 + (slot ^ ((r >> 1) & 3))];
  }
}

cudaError_t pack_wo_i8(void* dst, const void* wo_codes, int H, int Hq, cudaStream_t s) {
  pack_wo_i8_kernel<<<2048, 256, 0, s>>>((uint4*)dst, (const uint4*)wo_codes, H, Hq);
  return cudaGetLastError();
}

// Two's complement int8 codes -> biased bytes q + 128 (flip each top bit), in place.
__global__ void bias_codes_kernel(uint4* __restrict__ p, size_t n) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    uint4 v = p[i];
    v.x ^= 0x80808080u;
    v.y ^= 0x80808080u;
    v.z ^= 0x80808080u;
    v.w ^= 0x80808080u;
    p[i] = v;
  }
}

cudaError_t bias_codes(void* p, size_t bytes, cudaStream_t s) {
  if (bytes == 0) return cudaSuccess;
  bias_codes_kernel<<<2048, 256, 0, s>>>((uint4*)p, bytes / 16);
  return cudaGetLastError();
}

// Wide batch: the K-chunk-major re-layout of a chunk-swizzled row-major
// matrix [R][K] (16-byte chunk i of row p at slot i ^ (p & 7), as the
// packers above write it): dst[kc][p] = the 128 bytes of columns
// [64 kc, 64 kc + 64) of row p, for kc < K / 64 and p < R8 (R rounded up to
// 8 rows; rows past R are zero).  A row's swizzle only permutes the low three
// bits of the chunk index, so inside each 128-byte piece chunk j of row p
// already sits at slot j ^ (p & 7): the tensor cores' 128-byte swizzle of a
// K-major operand tile whose 8-row atoms start at rows that are multiples of 8.
__global__ void pack_kchunk_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, long R,
                                   long R8, int nk) {
  const size_t total = (size_t)nk * R8 * 8;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t e = i % 8, pr = i / 8;
    const size_t p = pr % R8, kc = pr / R8;
    dst[i] = p < (size_t)R ? src[(p * nk + kc) * 8 + e] : make_uint4(0, 0, 0, 0);
  }
}

cudaError_t pack_kchunk(uint16_t* dst, const uint16_t* src, long R, int K, cudaStream_t s) {
  if (R <= 0 || K <= 0 || K % 64) return cudaErrorInvalidValue;
  pack_kchunk_kernel<<<4096, 256, 0, s>>>((uint4*)dst, (const uint4*)src, R, (R + 7) / 8 * 8,
                                          K / 64);
  return cudaGetLastError();
}

}  // namespace mk
