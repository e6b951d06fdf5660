// k1_block_index.cuh -- block compression of the proxy keys.
//
// ai4snews item "Step 5 Preview bets on depth over width", Interpretation para 2: the
// indexer keys of adjacent historical positions are compressed into one representation
// per block of B = 8 tokens.  Reading: the element-wise mean of the block's token proxies;
// a partly filled block averages the tokens present.
//
// Layout: k_proxy [G, ctx_cap, P] bf16 -> k_blk [G, nb_cap, P] bf16.  Each thread owns 8
// consecutive proxy elements (one 16-byte vector) of one block, so a warp reads whole
// 512-byte token rows (P = 256) and writes a whole 512-byte block row.  The sum runs in
// fp32 in token order; full blocks multiply by 1/B (exact, B is a power of two), and a
// partial block of n tokens rounds sum / n to bf16 as if the quotient were exact
// (k1_partial_fp32_ok).
//
// The decode cache can hold the block index as FP8 E4M3 instead (the pages deploy the model
// in FP8; this cache is a variant): the same fp32 sum, rounded once to E4M3 (to nearest,
// ties to even, saturating at +-448) by the hardware conversion from the same fp32 value
// (x 1/B for full blocks, the fp32 quotient of k1_partial_fp32_ok for partial ones).
#pragma once
#include <cuda_fp8.h>
#include "ptx.cuh"

namespace sgqa {

struct K1Args {
  const __nv_bfloat16* k_proxy;
  void* k_blk;          // bf16 or E4M3 codes, [G, nb_cap, P]
  int64_t ctx_cap, nb_cap;
  int64_t tok_end;      // tokens present
  int64_t blk_begin;    // first block to build
  int64_t n_blocks;     // blocks to build per group
  int32_t G, P, B;
  // optional per-sequence mode (decode): blocks are given by (kv_off + pos) / B
  const int64_t* seq_tok_end;  // device or nullptr
};

// A partial block of n < B <= 16 tokens rounds sum / n once.  In place of a double division
// (B300's FP64 unit is slow: the partial blocks of one decode step took about 10 us), the
// fp32 quotient q = RN32(s / n) is rounded to bf16 or E4M3, which gives the same result:
// - a rounding midpoint m of either format has at most 9 significant bits, so s - n m is a
//   multiple of 2^min(e_s, e_m), e_s the last bit of s and e_m that of m; if s / n != m it
//   misses m by at least 2^e_s / n (or 2^e_m / n, larger still);
// - 2^e_s > |s| 2^-24 = n |s / n| 2^-24, and for n not a power of two the power of two
//   2^e_s exceeds n |m| 2^-24 by enough that s / n misses m by more than half of m's fp32
//   step, so q = m only when s / n = m (n a power of two divides exactly);
// - no midpoint lies strictly between s / n and q, q being the fp32 value nearest s / n.
// The argument holds while s / n is a normal fp32 number: sums of magnitude below 2^-100
// (other than zero) still divide in double.
__device__ __forceinline__ bool k1_partial_fp32_ok(float acc) { return acc == 0.f || fabsf(acc) >= 0x1p-100f; }

// The 8 means of one thread, stored as bf16 (16 bytes) or E4M3 (8 bytes) at element `e0`
// of the block row.
template <bool E4M3>
__device__ __forceinline__ void k1_store(void* row, int pv, const float (&acc)[8], int64_t n, int B) {
  const float inv_b = 1.0f / (float)B;
  const float fn = (float)n;
  if (!E4M3) {
    uint4 o;
    uint32_t* op = reinterpret_cast<uint32_t*>(&o);
    if (n == B) {
#pragma unroll
      for (int e = 0; e < 4; ++e) op[e] = pack_bf16(acc[2 * e] * inv_b, acc[2 * e + 1] * inv_b);
    } else {
      __nv_bfloat16 h[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        h[e] = k1_partial_fp32_ok(acc[e]) ? __float2bfloat16_rn(__fdiv_rn(acc[e], fn))
                                          : __double2bfloat16((double)acc[e] / (double)n);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        op[e] = (uint32_t)__bfloat16_as_ushort(h[2 * e]) | ((uint32_t)__bfloat16_as_ushort(h[2 * e + 1]) << 16);
    }
    reinterpret_cast<uint4*>(row)[pv] = o;
  } else {
    uint8_t c[8];
    if (n == B) {
#pragma unroll
      for (int e = 0; e < 8; ++e) c[e] = __nv_cvt_float_to_fp8(acc[e] * inv_b, __NV_SATFINITE, __NV_E4M3);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        c[e] = k1_partial_fp32_ok(acc[e])
                   ? __nv_cvt_float_to_fp8(__fdiv_rn(acc[e], fn), __NV_SATFINITE, __NV_E4M3)
                   : __nv_cvt_double_to_fp8((double)acc[e] / (double)n, __NV_SATFINITE, __NV_E4M3);
    }
    uint2 o;
    o.x = (uint32_t)c[0] | ((uint32_t)c[1] << 8) | ((uint32_t)c[2] << 16) | ((uint32_t)c[3] << 24);
    o.y = (uint32_t)c[4] | ((uint32_t)c[5] << 8) | ((uint32_t)c[6] << 16) | ((uint32_t)c[7] << 24);
    reinterpret_cast<uint2*>(row)[pv] = o;
  }
}

template <bool E4M3>
__global__ void __launch_bounds__(256) k1_block_index(K1Args a) {
  const int vec_per_row = a.P / 8;
  const int64_t n_vec = (int64_t)a.G * a.n_blocks * vec_per_row;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < n_vec; v += (int64_t)gridDim.x * blockDim.x) {
    const int pv = (int)(v % vec_per_row);
    const int64_t gb = v / vec_per_row;
    const int64_t g = gb / a.n_blocks;
    const int64_t b = a.blk_begin + gb % a.n_blocks;
    const int64_t first = b * a.B;
    int64_t n = a.tok_end - first;
    if (n > a.B) n = a.B;
    if (n <= 0) continue;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    const uint4* src = reinterpret_cast<const uint4*>(a.k_proxy + ((g * a.ctx_cap + first) * a.P)) + pv;
    // all (at most 16) token loads are issued before the first add, then summed in order
    uint4 wv[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) wv[j] = j < n ? __ldg(src + j * vec_per_row) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (j >= n) break;
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&wv[j]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float2 f = __bfloat1622float2(h[e]);
        acc[2 * e] += f.x;
        acc[2 * e + 1] += f.y;
      }
    }
    const int64_t row = (g * a.nb_cap + b) * a.P;
    k1_store<E4M3>(E4M3 ? (void*)(static_cast<uint8_t*>(a.k_blk) + row) : (void*)(static_cast<__nv_bfloat16*>(a.k_blk) + row),
                   pv, acc, n, a.B);
  }
}

// Decode form: for each sequence s rebuild the block holding its newest token.
struct K1SeqArgs {
  const __nv_bfloat16* k_proxy;  // [G, total, P]
  void* k_blk;                   // [G, total / B, P], bf16 or E4M3 codes
  int64_t total;
  int32_t G, P, B, batch;
  int64_t ctx_len[256];
  int64_t kv_off[256];
};

template <bool E4M3>
__global__ void __launch_bounds__(256) k1_block_index_seq(const __grid_constant__ K1SeqArgs a) {
  const int vec_per_row = a.P / 8;
  const int n_vec = a.G * a.batch * vec_per_row;
  const int64_t nb_total = a.total / a.B;
  for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < n_vec; v += gridDim.x * blockDim.x) {
    const int pv = v % vec_per_row;
    const int s = (v / vec_per_row) % a.batch;
    const int g = v / (vec_per_row * a.batch);
    const int64_t L = a.ctx_len[s];
    const int64_t bl = (L - 1) / a.B;              // block of the newest token (sequence-local)
    const int64_t first = bl * a.B;
    const int64_t n = L - first;                   // 1 .. B tokens present
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    const uint4* src =
        reinterpret_cast<const uint4*>(a.k_proxy + (((int64_t)g * a.total + a.kv_off[s] + first) * a.P)) + pv;
    // all (at most 16) token loads are issued before the first add, then summed in order
    uint4 wv[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) wv[j] = j < n ? __ldg(src + j * vec_per_row) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (j >= n) break;
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&wv[j]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float2 f = __bfloat1622float2(h[e]);
        acc[2 * e] += f.x;
        acc[2 * e + 1] += f.y;
      }
    }
    const int64_t row = ((int64_t)g * nb_total + a.kv_off[s] / a.B + bl) * a.P;
    k1_store<E4M3>(E4M3 ? (void*)(static_cast<uint8_t*>(a.k_blk) + row) : (void*)(static_cast<__nv_bfloat16*>(a.k_blk) + row),
                   pv, acc, n, a.B);
  }
}

}  // namespace sgqa
