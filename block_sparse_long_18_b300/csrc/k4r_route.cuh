// k4r_route.cuh -- per 8-row unit, which attention kernel serves it.
//
// The union kernel (k4u_attention.cuh) gathers each block of a unit's union once and runs
// its MMAs over all 8 rows x 16 heads; the warp-level kernel (k4_attention.cuh) gathers a
// row's selected blocks for that row alone.  Which is cheaper depends on how much the 8
// rows' selections overlap: measured on B300 at 128K tokens, a union block costs the
// union kernel about 0.71 ns of the GPU's time and a (row, selected block) pair costs the
// warp-level kernel about 0.37 ns.  So a unit goes to the union kernel when
//     kRouteUnionCost * |union| <= kRoutePairCost * (number of (row, block) pairs)
// and to the warp-level kernel otherwise.  Both kernels compute the same quantity; the
// choice changes only which one runs (and the fp32 accumulation order).
//
// k4r_count: one warp per unit; the union size is counted with the union builder's window
// bitmap and its entry rules (counts clamped to [1, min(k, b_t + 1)], entries outside
// [0, b_t] skipped).  k4r_compact: one CTA turns the per-unit choices into two unit lists
// in ascending unit order (group-major, so both kernels keep one group's K/V in L2).
#pragma once
#include "ptx.cuh"
#include "k4u_attention.cuh"

namespace sgqa {

#ifndef SGQA_ROUTE_UNION_COST
#define SGQA_ROUTE_UNION_COST 100
#endif
#ifndef SGQA_ROUTE_PAIR_COST
#define SGQA_ROUTE_PAIR_COST 55
#endif
constexpr int kRouteUnionCost = SGQA_ROUTE_UNION_COST, kRoutePairCost = SGQA_ROUTE_PAIR_COST;

struct K4RouteArgs {
  const int32_t* sel_idx;  // [G, rows, kcap]
  const int32_t* sel_cnt;  // [G, rows]
  const int32_t* perm;     // [G, rows] row at each slot (grouped units), or null: slot = row
  int32_t* choice;         // [G * tiles]: 1 = union kernel, 0 = warp-level kernel
  int32_t* union_units;    // [G * tiles] (k4r_compact)
  int32_t* warp_units;     // [G * tiles] (k4r_compact)
  int32_t* counts;         // [2]: union units, warp-level units (k4r_compact)
  int64_t rows, pos0;
  int32_t G, kcap;
};
constexpr int K4R_WARPS = 4;

__global__ void __launch_bounds__(K4R_WARPS * 32) k4r_count(const K4RouteArgs a) {
  __shared__ uint32_t seen[K4R_WARPS][K4U_WIN / 32];
  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
  const int64_t ntiles = (a.rows + 7) / 8;
  const int64_t u = (int64_t)blockIdx.x * K4R_WARPS + warp;
  if (u >= (int64_t)a.G * ntiles) return;
  const int32_t g = (int32_t)(u / ntiles);
  const int64_t i0 = (u % ntiles) * 8;
  uint32_t* bm = seen[warp];
  int32_t cnt_l = 0, bt_l = -1;
  int64_t row_l = 0;
  if (lane < 8 && i0 + lane < a.rows) {
    const int64_t i = a.perm ? (int64_t)__ldg(a.perm + (int64_t)g * a.rows + i0 + lane) : i0 + lane;
    row_l = i;
    bt_l = (int32_t)((a.pos0 + i) >> 3);
    int32_t c = __ldg(a.sel_cnt + (int64_t)g * a.rows + i);
    const int32_t cap = a.kcap < bt_l + 1 ? a.kcap : bt_l + 1;
    if (c < 1 || c > cap) c = c < 1 ? 1 : cap;  // the attention kernels report it
    cnt_l = c;
  }
  int32_t bmax = bt_l, pairs = cnt_l;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    bmax = max(bmax, __shfl_xor_sync(0xffffffffu, bmax, o));
    pairs += __shfl_xor_sync(0xffffffffu, pairs, o);
  }
  uint32_t nU = 0;
  const int64_t windows = bmax / K4U_WIN + 1;
  for (int32_t wb = 0; wb <= bmax; wb += K4U_WIN) {
    for (int w = lane; w < K4U_WIN / 32; w += 32) bm[w] = 0u;
    __syncwarp();
#pragma unroll 1
    for (int r = 0; r < 8; ++r) {
      const int32_t cnt = __shfl_sync(0xffffffffu, cnt_l, r), bt = __shfl_sync(0xffffffffu, bt_l, r);
      const int64_t row = __shfl_sync(0xffffffffu, row_l, r);
      const int32_t* sel = a.sel_idx + ((int64_t)g * a.rows + row) * a.kcap;
      // 512 entries at a time, every load issued before the first is used
      for (int32_t j0 = 0; j0 < cnt; j0 += 512) {
        int32_t e[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int32_t j = j0 + (int32_t)lane + 32 * q;
          e[q] = j < cnt ? __ldg(sel + j) : -1;
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int32_t b = e[q], o = b - wb;
          if (b >= 0 && b <= bt && o >= 0 && o < K4U_WIN) atomicOr(&bm[o >> 5], 1u << (o & 31));
        }
      }
    }
    __syncwarp();
    uint32_t pc = 0;
    for (int w = lane; w < K4U_WIN / 32; w += 32) pc += __popc(bm[w]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pc += __shfl_xor_sync(0xffffffffu, pc, o);
    nU += pc;
    __syncwarp();
  }
  if (lane == 0)
    a.choice[u] = (int64_t)kRouteUnionCost * windows * nU <= (int64_t)kRoutePairCost * pairs ? 1 : 0;
}

// One CTA of 1024 threads: thread t takes a contiguous run of units, the block scans the
// runs' counts, and every thread writes its units into the two lists in order.
constexpr int K4R_COMPACT_THREADS = 1024;

__global__ void __launch_bounds__(K4R_COMPACT_THREADS) k4r_compact(const K4RouteArgs a) {
  __shared__ uint32_t wsum[2][K4R_COMPACT_THREADS / 32];
  const int64_t n = (int64_t)a.G * ((a.rows + 7) / 8);
  const int64_t per = (n + K4R_COMPACT_THREADS - 1) / K4R_COMPACT_THREADS;
  const int64_t b = (int64_t)threadIdx.x * per, e = b + per < n ? b + per : n;
  uint32_t cu = 0, cw = 0;
  for (int64_t u = b; u < e; ++u) (a.choice[u] ? cu : cw) += 1u;
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  // exclusive scans of (cu, cw) over the block
  uint32_t iu = cu, iw = cw;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, iu, o), y = __shfl_up_sync(0xffffffffu, iw, o);
    if (lane >= (uint32_t)o) {
      iu += x;
      iw += y;
    }
  }
  if (lane == 31) {
    wsum[0][warp] = iu;
    wsum[1][warp] = iw;
  }
  __syncthreads();
  uint32_t bu = 0, bw = 0, tu = 0, tw = 0;
  for (int w = 0; w < K4R_COMPACT_THREADS / 32; ++w) {
    if (w < (int)warp) {
      bu += wsum[0][w];
      bw += wsum[1][w];
    }
    tu += wsum[0][w];
    tw += wsum[1][w];
  }
  uint32_t ou = bu + iu - cu, ow = bw + iw - cw;
  for (int64_t u = b; u < e; ++u) {
    if (a.choice[u])
      a.union_units[ou++] = (int32_t)u;
    else
      a.warp_units[ow++] = (int32_t)u;
  }
  if (threadIdx.x == 0) {
    a.counts[0] = (int32_t)tu;
    a.counts[1] = (int32_t)tw;
  }
}


// ---------------------------------------------------------------------------------------
// Grouped units: k4g_signature (a warp per row) writes each row's sort key; k4g_sort (a CTA
// per (group, window of K4G_WIN rows)) orders the window.
// ---------------------------------------------------------------------------------------
#ifndef SGQA_GROUP_WINDOW
#define SGQA_GROUP_WINDOW 4096
#endif
constexpr int K4G_WIN = SGQA_GROUP_WINDOW;   // rows per grouping window (a power of 2, >= 1024)
constexpr int K4G_THREADS = 1024;
static_assert(K4G_WIN >= K4G_THREADS && (K4G_WIN & (K4G_WIN - 1)) == 0, "grouping window");

// The 32-bit finalizer of MurmurHash3 (Austin Appleby, public domain): a bijective mixer
// of a 32-bit word.  The two signatures hash the block index and the block index xor a
// constant.
__device__ __forceinline__ uint32_t k4g_mix(uint32_t h) {
  h ^= h >> 16;
  h *= 0x85ebca6bu;
  h ^= h >> 13;
  h *= 0xc2b2ae35u;
  h ^= h >> 16;
  return h;
}
constexpr uint32_t K4G_SEED2 = 0x5bd1e995u;

struct K4GroupArgs {
  const int32_t* sel_idx;  // [G, rows, kcap]
  const int32_t* sel_cnt;  // [G, rows]
  uint64_t* keys;          // [G, rows] sort keys (k4g_signature), read by k4g_sort
  int32_t* perm;           // [G, rows]
  int64_t rows, pos0;
  int32_t G, kcap;
};
constexpr int K4G_SIG_WARPS = 8;

// Sort key of every row, one warp per row: the least first hash over the row's valid
// selected blocks, then the high bits of the least second hash, then the row's place in its
// window.  The same entry rules as the union builder.
__global__ void __launch_bounds__(K4G_SIG_WARPS * 32) k4g_signature(const K4GroupArgs a) {
  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
  const int64_t r = (int64_t)blockIdx.x * K4G_SIG_WARPS + warp;  // (group, row)
  if (r >= (int64_t)a.G * a.rows) return;
  const int64_t g = r / a.rows, i = r % a.rows;
  const int32_t bt = (int32_t)((a.pos0 + i) >> 3);
  int32_t c = __ldg(a.sel_cnt + r);
  const int32_t cap = a.kcap < bt + 1 ? a.kcap : bt + 1;
  if (c < 1 || c > cap) c = c < 1 ? 1 : cap;
  const int32_t* sel = a.sel_idx + r * a.kcap;
  uint32_t h1 = ~0u, h2 = ~0u;
  // 512 entries at a time, every load issued before the first is used
  for (int32_t j0 = 0; j0 < c; j0 += 512) {
    int32_t e[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int32_t j = j0 + (int32_t)lane + 32 * q;
      e[q] = j < c ? __ldg(sel + j) : -1;
    }
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int32_t b = e[q];
      if (b < 0 || b > bt) continue;
      h1 = min(h1, k4g_mix((uint32_t)b));
      h2 = min(h2, k4g_mix((uint32_t)b ^ K4G_SEED2));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    h1 = min(h1, __shfl_xor_sync(0xffffffffu, h1, o));
    h2 = min(h2, __shfl_xor_sync(0xffffffffu, h2, o));
  }
  constexpr int kRowBits = __builtin_ctz(K4G_WIN);
  if (lane == 0)
    a.keys[r] = ((uint64_t)h1 << 32) | ((uint64_t)(h2 >> kRowBits) << kRowBits) | (uint64_t)(i & (K4G_WIN - 1));
  (void)g;
}

// One CTA per (group, window): bitonic sort of the window's keys in shared memory; the
// sorted keys' low bits give the row order.
__global__ void __launch_bounds__(K4G_THREADS) k4g_sort(const K4GroupArgs a) {
  __shared__ uint64_t key[K4G_WIN];
  const int64_t nwin = (a.rows + K4G_WIN - 1) / K4G_WIN;
  const int32_t g = (int32_t)(blockIdx.x / nwin);
  const int64_t w0 = (int64_t)(blockIdx.x % nwin) * K4G_WIN;
  const int nrow = (int)(a.rows - w0 < K4G_WIN ? a.rows - w0 : K4G_WIN);
  for (int t = threadIdx.x; t < K4G_WIN; t += K4G_THREADS)
    key[t] = t < nrow ? a.keys[(int64_t)g * a.rows + w0 + t] : ~0ull;
  __syncthreads();
  // ascending; thread t owns elements t, t + 1024, ...
  for (uint32_t k = 2; k <= (uint32_t)K4G_WIN; k <<= 1) {
    for (uint32_t j = k >> 1; j > 0; j >>= 1) {
      for (uint32_t t = threadIdx.x; t < (uint32_t)K4G_WIN; t += K4G_THREADS) {
        const uint32_t p = t ^ j;
        if (p > t) {
          const uint64_t x = key[t], y = key[p];
          const bool up = (t & k) == 0;
          if ((x > y) == up) {
            key[t] = y;
            key[p] = x;
          }
        }
      }
      __syncthreads();
    }
  }
  for (uint32_t t = threadIdx.x; (int)t < nrow; t += K4G_THREADS)
    a.perm[(int64_t)g * a.rows + w0 + t] = (int32_t)(w0 + (int64_t)(key[t] & (K4G_WIN - 1)));
}

}  // namespace sgqa
