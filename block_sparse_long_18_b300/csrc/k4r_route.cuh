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
  if (lane < 8 && i0 + lane < a.rows) {
    const int64_t i = i0 + lane;
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
      const int32_t* sel = a.sel_idx + ((int64_t)g * a.rows + i0 + r) * a.kcap;
      for (int32_t j = (int32_t)lane; j < cnt; j += 32) {
        const int32_t b = __ldg(sel + j);
        const int32_t o = b - wb;
        if (b >= 0 && b <= bt && o >= 0 && o < K4U_WIN) atomicOr(&bm[o >> 5], 1u << (o & 31));
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

}  // namespace sgqa
