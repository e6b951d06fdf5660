// k2d_decode_index.cuh -- indexer scores for decode: one query proxy per (sequence, group)
// against that sequence's earlier block proxies.  Same definition as the prefill indexer
// (a plain dot product, fp32 accumulation; ai4snews item, Interpretation para 2), but with
// a single query row it is a matrix-vector product that streams the block-proxy cache
// from HBM: one warp reads one 512-byte block row per load (P = 256), eight rows per step
// with the next step's eight already in flight, and the rows K2D_AHEAD steps ahead are
// prefetched into L2 (one bulk prefetch per warp and step), so that more of the stream is
// in flight than the registers hold.  Products take the bf16 operands as they are
// (mixed-precision FMA, fp32 accumulation: the same result as widening them first).
#pragma once
#include <cuda_fp16.h>
#include <type_traits>
#include <cuda_fp8.h>
#include "ptx.cuh"

namespace sgqa {

constexpr int K2D_AHEAD = 3;  // steps between a warp's L2 prefetch of its rows and their load

struct K2dArgs {
  const __nv_bfloat16* qp;    // [G, batch, P]
  const void* kblk;           // [G, nb_total, P], bf16 (k2d_decode_index) or E4M3 codes (_e4m3)
  float* scores;              // [G, batch, ld]
  int64_t ld, nb_total;
  int32_t G, P, B, batch;
  int32_t rows_per_cta;
  int64_t ctx_len[256];
  int64_t kv_off[256];
};

// c + a.lo * b.lo + a.hi * b.hi for two bf16 pairs, rounded after each product as two fp32
// FMAs would: the mixed-precision FMA (bf16 sources, fp32 addend and result) forms each
// product exactly, so this equals fmaf(a.hi, b.hi, fmaf(a.lo, b.lo, c)) on the widened
// values, without widening them.
__device__ __forceinline__ float k2d_fma2_bf16(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n\t.reg .b16 alo, ahi, blo, bhi;\n\t.reg .f32 t;\n\t"
      "mov.b32 {alo, ahi}, %1;\n\tmov.b32 {blo, bhi}, %2;\n\t"
      "fma.rn.f32.bf16 t, alo, blo, %3;\n\tfma.rn.f32.bf16 %0, ahi, bhi, t;\n\t}"
      : "=f"(d)
      : "r"(a), "r"(b), "f"(c));
  return d;
}

__global__ void __launch_bounds__(256) k2d_decode_index(const __grid_constant__ K2dArgs a) {
  const int gs = blockIdx.y;  // g * batch + s
  const int g = gs / a.batch, s = gs % a.batch;
  const int64_t n = (a.ctx_len[s] - 1) / a.B;  // candidates 0 .. b_t - 1
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = a.P / 8;
  const bool active = lane < nvec;
  uint4 qw = make_uint4(0, 0, 0, 0);  // the lane's 8 query-proxy elements, bf16 pairs
  if (active) qw = __ldg(reinterpret_cast<const uint4*>(a.qp + ((int64_t)g * a.batch + s) * a.P) + lane);
  const uint32_t* qp2 = reinterpret_cast<const uint32_t*>(&qw);
  const __nv_bfloat16* base =
      static_cast<const __nv_bfloat16*>(a.kblk) + ((int64_t)g * a.nb_total + a.kv_off[s] / a.B) * a.P;
  float* out = a.scores + (int64_t)gs * a.ld;
  const int64_t b_lo = (int64_t)blockIdx.x * a.rows_per_cta;
  int64_t b_hi = b_lo + a.rows_per_cta;
  if (b_hi > n) b_hi = n;
  // each warp takes 8 consecutive rows per step; the next step's rows are loaded before
  // this step's dot products are reduced, so 16 rows (8 KB) per warp are in flight
  constexpr int RW = 8;
  auto load = [&](int64_t b0, uint4 (&w)[RW]) {
#pragma unroll
    for (int r = 0; r < RW; ++r) {
      w[r] = make_uint4(0, 0, 0, 0);
      if (active && b0 + r < b_hi) w[r] = __ldg(reinterpret_cast<const uint4*>(base + (b0 + r) * a.P) + lane);
    }
  };
  const int64_t step = 8 * RW;  // 8 warps
  // the warp's RW rows from b (P * 2 bytes each, contiguous) into L2
  auto prefetch = [&](int64_t b) {
    if (lane == 0 && b < b_hi) {
      const int64_t nr = b_hi - b < RW ? b_hi - b : RW;
      bulk_prefetch_l2(base + b * a.P, (uint32_t)(nr * a.P * 2));
    }
  };
  uint4 cur[RW], nxt[RW];
  int64_t b0 = b_lo + warp * RW;
  if (b0 < b_hi) load(b0, cur);
#pragma unroll
  for (int d = 2; d < K2D_AHEAD; ++d) prefetch(b0 + d * step);
  for (; b0 < b_hi; b0 += step) {
    prefetch(b0 + K2D_AHEAD * step);
    if (b0 + step < b_hi) load(b0 + step, nxt);
    float acc[RW];
#pragma unroll
    for (int r = 0; r < RW; ++r) {
      const uint32_t* k2 = reinterpret_cast<const uint32_t*>(&cur[r]);
      float sum = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) sum = k2d_fma2_bf16(qp2[e], k2[e], sum);
      acc[r] = sum;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
      for (int r = 0; r < RW; ++r) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], o);
    }
    if (lane < RW && b0 + lane < b_hi) {
      float v = acc[0];
#pragma unroll
      for (int r = 1; r < RW; ++r) v = lane == r ? acc[r] : v;
      out[b0 + lane] = v;
    }
#pragma unroll
    for (int r = 0; r < RW; ++r) cur[r] = nxt[r];
  }
}

// c + a.lo * b.lo + a.hi * b.hi, rounded after each product as two fp32 FMAs would: a holds
// two f16 values, b two E4M3 codes widened exactly to f16.  The mixed-precision FMA
// (f16 sources, fp32 addend and result) forms each product exactly, so this equals
// fmaf(a.hi, b.hi, fmaf(a.lo, b.lo, c)) on the fp32 values, without widening to fp32.
__device__ __forceinline__ float k2d_fma2_f16_e4m3(uint32_t a, uint16_t codes, float c) {
  float d;
  asm("{\n\t.reg .b32 h2;\n\t.reg .b16 alo, ahi, blo, bhi;\n\t.reg .f32 t;\n\t"
      "cvt.rn.f16x2.e4m3x2 h2, %2;\n\t"
      "mov.b32 {alo, ahi}, %1;\n\tmov.b32 {blo, bhi}, h2;\n\t"
      "fma.rn.f32.f16 t, alo, blo, %3;\n\tfma.rn.f32.f16 %0, ahi, bhi, t;\n\t}"
      : "=f"(d)
      : "r"(a), "h"(codes), "f"(c));
  return d;
}

// The same scores from an E4M3 block-proxy cache: half the bytes of the bf16 cache.  A lane
// reads 16 codes (16 bytes) of a row; a row takes P / 16 lanes (4, 8 or 16), or for
// P = 192 (IDLE) 16 lanes of which four hold no codes, and a warp load covers 32 / lpr
// rows; eight loads per step with the next step's eight in flight (an L2 prefetch ahead of
// them, as in the bf16 kernel, measured slower here: 0.243 -> 0.277 ms per decode step on
// B300).  Codes are widened exactly (E4M3 -> f16) and the dot product runs in fp32: when
// every element of the query proxy is exactly an f16 value (one warp vote; the same answer
// in every warp of the CTA) the products are taken from f16 operands by mixed-precision
// FMAs, otherwise the codes are widened on to fp32 -- the same fp32 result either way.
template <bool IDLE>
__global__ void __launch_bounds__(256) k2d_decode_index_e4m3(const __grid_constant__ K2dArgs a) {
  const int gs = blockIdx.y;  // g * batch + s
  const int g = gs / a.batch, s = gs % a.batch;
  const int64_t n = (a.ctx_len[s] - 1) / a.B;  // candidates 0 .. b_t - 1
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lpr = IDLE ? 16 : a.P / 16;  // lanes per row
  const int rpl = 32 / lpr;              // rows per warp load
  const int sub = lane % lpr, rsub = lane / lpr;
  const bool active = !IDLE || sub < a.P / 16;  // lanes holding codes of a row
  float qv[16];
  uint32_t qh[8];  // the same 16 values as f16 pairs
  bool q_f16 = true;
  {
    const uint4* qs = reinterpret_cast<const uint4*>(a.qp + ((int64_t)g * a.batch + s) * a.P + 16 * sub);
#pragma unroll
    for (int hlf = 0; hlf < 2; ++hlf) {
      const uint4 w = active ? __ldg(qs + hlf) : make_uint4(0, 0, 0, 0);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h[e]);
        qv[8 * hlf + 2 * e] = f.x;
        qv[8 * hlf + 2 * e + 1] = f.y;
        const __half2 hq = __floats2half2_rn(f.x, f.y);
        const float2 back = __half22float2(hq);
        q_f16 = q_f16 && back.x == f.x && back.y == f.y;
        qh[4 * hlf + e] = *reinterpret_cast<const uint32_t*>(&hq);
      }
    }
  }
  q_f16 = __all_sync(0xffffffffu, q_f16);
  const uint8_t* base =
      static_cast<const uint8_t*>(a.kblk) + ((int64_t)g * a.nb_total + a.kv_off[s] / a.B) * a.P + 16 * sub;
  float* out = a.scores + (int64_t)gs * a.ld;
  const int64_t b_lo = (int64_t)blockIdx.x * a.rows_per_cta;
  int64_t b_hi = b_lo + a.rows_per_cta;
  if (b_hi > n) b_hi = n;
  constexpr int RW = 8;
  const int64_t wrows = (int64_t)RW * rpl;  // rows of one warp step
  auto load = [&](int64_t b0, uint4 (&w)[RW]) {
#pragma unroll
    for (int r = 0; r < RW; ++r) {
      const int64_t b = b0 + r * rpl + rsub;
      w[r] = active && b < b_hi ? __ldg(reinterpret_cast<const uint4*>(base + b * a.P)) : make_uint4(0, 0, 0, 0);
    }
  };
  const int64_t step = 8 * wrows;  // 8 warps
  // the warp's rows, eight loads per step; F16Q: products from f16 operands
  auto stream = [&](auto f16q) {
    constexpr bool F16Q = decltype(f16q)::value;
    uint4 cur[RW], nxt[RW];
    int64_t b0 = b_lo + warp * wrows;
    if (b0 < b_hi) load(b0, cur);
    for (; b0 < b_hi; b0 += step) {
      if (b0 + step < b_hi) load(b0 + step, nxt);
      float acc[RW];
#pragma unroll
      for (int r = 0; r < RW; ++r) {
        const uint16_t* c2 = reinterpret_cast<const uint16_t*>(&cur[r]);
        float sum = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (F16Q) {
            sum = k2d_fma2_f16_e4m3(qh[e], c2[e], sum);
          } else {
            const __half2 hv = __half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)c2[e], __NV_E4M3));
            const float2 f = __half22float2(hv);
            sum = fmaf(qv[2 * e], f.x, sum);
            sum = fmaf(qv[2 * e + 1], f.y, sum);
          }
        }
        acc[r] = sum;
      }
      for (int o = lpr / 2; o > 0; o >>= 1) {
#pragma unroll
        for (int r = 0; r < RW; ++r) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], o);
      }
      if (sub == 0) {
#pragma unroll
        for (int r = 0; r < RW; ++r) {
          const int64_t b = b0 + r * rpl + rsub;
          if (b < b_hi) out[b] = acc[r];
        }
      }
#pragma unroll
      for (int r = 0; r < RW; ++r) cur[r] = nxt[r];
    }
  };
  if (q_f16)
    stream(std::true_type{});
  else
    stream(std::false_type{});
}

// Bounded-wait self test: waits on an mbarrier that nothing ever arrives at.  The wait
// gives up after limit_ns and records the timeout in the device error word.
__global__ void k_selftest_wait(uint64_t limit_ns, int32_t* result) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    const bool ok = mbar_wait(smem_u32(&bar), 0, limit_ns);
    if (result) *result = ok ? 1 : 0;
  }
}

}  // namespace sgqa
