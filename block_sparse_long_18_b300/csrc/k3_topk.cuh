// k3_topk.cuh -- top-k block selection with a deterministic tie rule.
//
// ai4snews item "Step 5 Preview bets on depth over width", Interpretation para 2 (top-k
// over block representations); ai.info article, "Sparse GQA targets million-token
// context" (top-k of 4,096 tokens = 512 blocks of 8); phantomic12 entry (topk 512).
// Readings: the query's own block b_t is always kept and never scored; the other k-1
// slots go to the strictly earlier blocks in order (score descending, block index
// descending); -0 and +0 compare equal; the kept set is written in ascending order.
//
// One CTA per (group, query row).  Scores are mapped to order-preserving unsigned keys;
// a radix select over 11/11/10-bit digits (shared-memory histograms, block-wide suffix
// search) finds the key of the (k-1)-th best candidate and how many candidates equal to
// it are kept; it stops early once a digit bucket is taken whole.  Equal keys are taken
// from the largest index down by ranking them in index order.  The final pass compacts
// the kept indices in ascending order with one block-wide scan per tile of candidates.
// Rows up to NT*PER candidates keep their keys in registers (one pass over global
// memory); longer rows (contexts past 128K tokens at B = 8) stream tiles per pass.
#pragma once
#include "ptx.cuh"

namespace sgqa {

struct K3Args {
  const float* scores;  // [G, rows, ld]  (rows of this launch)
  int64_t ld;           // row stride of scores (elements)
  int64_t rows;         // rows of this launch
  int64_t pos0;         // absolute position of launch row 0 (prefill)
  int64_t out_row0;     // row offset into the [G, T_out, k] outputs
  int64_t T_out;        // rows per group of the outputs
  int32_t G, B, k;
  int32_t* sel_idx;     // [G, T_out, k]
  int32_t* sel_cnt;     // [G, T_out]
  int32_t use_pos;      // decode: positions come from pos[]
  int64_t pos[256];     // decode: absolute position of each row's query
};

__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u << 1) == 0) u = 0;  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int NT>
__device__ __forceinline__ uint32_t k3_block_excl_scan(uint32_t v, uint32_t* warp_tot, uint32_t& total) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t t = lane < NW ? warp_tot[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t s = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += s;
    }
    if (lane < NW) warp_tot[lane] = t;
  }
  __syncthreads();
  const uint32_t before = warp > 0 ? warp_tot[warp - 1] : 0u;
  total = warp_tot[NW - 1];
  __syncthreads();
  return before + incl - v;
}

template <int NT, int PER, bool STREAM>
__global__ void __launch_bounds__(NT) k3_topk(const __grid_constant__ K3Args a) {
  constexpr int NBINS = 2048;
  constexpr int BPT = NBINS / NT;  // bins per thread
  constexpr int TILE = NT * PER;
  __shared__ uint32_t hist[NBINS];
  __shared__ uint32_t warp_tot[NT / 32];
  __shared__ uint32_t sh_digit, sh_above;

  const int64_t r = blockIdx.x;
  const int64_t g = r / a.rows;
  const int64_t i = r % a.rows;
  const int64_t pos = a.use_pos ? a.pos[i] : a.pos0 + i;
  const int64_t bt = pos / a.B;
  const int64_t n = bt;                 // candidates 0 .. bt-1
  const int need = a.k - 1;
  int32_t* out = a.sel_idx + ((g * a.T_out) + a.out_row0 + i) * a.k;
  const float* row = a.scores + (g * a.rows + i) * a.ld;
  const int tid = threadIdx.x;

  if (n <= need) {  // every causal block is kept
    for (int64_t j = tid; j < a.k; j += NT) out[j] = j < n ? (int32_t)j : (j == n ? (int32_t)bt : -1);
    if (tid == 0) a.sel_cnt[g * a.T_out + a.out_row0 + i] = (int32_t)(n + 1);
    return;
  }

  const int n_tiles = STREAM ? (int)((n + TILE - 1) / TILE) : 1;
  uint32_t key[PER];
  auto load_tile = [&](int tile) {
    const int64_t base = (int64_t)tile * TILE + (int64_t)tid * PER;
#pragma unroll
    for (int j = 0; j < PER; j += 4) {
      if (base + j + 3 < n) {
        float4 f = __ldg(reinterpret_cast<const float4*>(row + base + j));
        key[j] = score_key(f.x);
        key[j + 1] = score_key(f.y);
        key[j + 2] = score_key(f.z);
        key[j + 3] = score_key(f.w);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) key[j + e] = (base + j + e < n) ? score_key(__ldg(row + base + j + e)) : 0u;
      }
    }
  };
  if (tid == 0) {
    sh_digit = 0;
    sh_above = 0;
  }
  if (!STREAM) load_tile(0);

  uint32_t prefix = 0, pmask = 0;
  uint32_t need_rem = (uint32_t)need, eq_count = 0;
#pragma unroll
  for (int p = 0; p < 3; ++p) {
    const int sh = p == 0 ? 21 : (p == 1 ? 10 : 0);
    const uint32_t wm = p == 2 ? 0x3FFu : 0x7FFu;
    for (int b = tid; b < NBINS; b += NT) hist[b] = 0;
    __syncthreads();
    for (int tile = 0; tile < n_tiles; ++tile) {
      if (STREAM) load_tile(tile);
      const int64_t base = (int64_t)tile * TILE + (int64_t)tid * PER;
#pragma unroll
      for (int j = 0; j < PER; ++j)
        if (base + j < n && (key[j] & pmask) == prefix) atomicAdd(&hist[(key[j] >> sh) & wm], 1u);
    }
    __syncthreads();
    // find the digit holding the need_rem-th largest matching key
    uint32_t loc = 0;
#pragma unroll
    for (int b = 0; b < BPT; ++b) loc += hist[tid * BPT + b];
    uint32_t total;
    const uint32_t excl = k3_block_excl_scan<NT>(loc, warp_tot, total);
    uint32_t cum = total - excl - loc;  // keys in bins above this thread's bins
#pragma unroll
    for (int b = BPT - 1; b >= 0; --b) {
      const uint32_t h = hist[tid * BPT + b];
      if (cum < need_rem && cum + h >= need_rem) {
        sh_digit = (uint32_t)(tid * BPT + b);
        sh_above = cum;
      }
      cum += h;
    }
    __syncthreads();
    const uint32_t d = sh_digit;
    need_rem -= sh_above;
    eq_count = hist[d];
    prefix |= d << sh;
    pmask |= wm << sh;
    __syncthreads();
    if (need_rem == eq_count) break;  // the whole bucket is kept: no tie to break
  }

  // ---- compaction in ascending index order ----
  const uint32_t skip = eq_count - need_rem;  // equal keys passed over, smallest indices first
  uint32_t out_base = 0, tie_base = 0;
  for (int tile = 0; tile < n_tiles; ++tile) {
    if (STREAM) load_tile(tile);
    const int64_t base = (int64_t)tile * TILE + (int64_t)tid * PER;
    uint32_t c_gt = 0, c_eq = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      if (base + j < n) {
        const uint32_t kh = key[j] & pmask;
        c_gt += kh > prefix;
        c_eq += kh == prefix;
      }
    }
    uint32_t total;
    const uint32_t ex = k3_block_excl_scan<NT>((c_gt << 16) | c_eq, warp_tot, total);
    uint32_t ties_before = tie_base + (ex & 0xFFFFu);
    // kept ties before this thread within this tile: those of global rank >= skip
    const uint32_t kept_prev = tie_base > skip ? tie_base - skip : 0u;
    uint32_t o = out_base + (ex >> 16) + (ties_before > skip ? ties_before - skip : 0u) - kept_prev;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      if (base + j < n) {
        const uint32_t kh = key[j] & pmask;
        if (kh > prefix) {
          out[o++] = (int32_t)(base + j);
        } else if (kh == prefix) {
          if (ties_before >= skip) out[o++] = (int32_t)(base + j);
          ++ties_before;
        }
      }
    }
    const uint32_t t_gt = total >> 16, t_eq = total & 0xFFFFu;
    out_base += t_gt + ((tie_base + t_eq > skip) ? (tie_base + t_eq - (tie_base > skip ? tie_base : skip)) : 0u);
    tie_base += t_eq;
  }
  if (tid == 0) {
    out[need] = (int32_t)bt;
    a.sel_cnt[g * a.T_out + a.out_row0 + i] = a.k;
  }
}

}  // namespace sgqa
