// k2_indexer.cuh -- block indexer scores on the 5th-generation tensor cores.
//
// ai4snews item "Step 5 Preview bets on depth over width", Interpretation para 2, and the
// phantomic12 catalog entry ("sparse indexer (topk 512, proxy_dim 256)"): every query's
// proxy vector is scored against the block-compressed proxy keys.  Reading: a plain dot
// product, fp32 accumulation, no scale.
//
//   S[g, i, b] = sum_p q_proxy[g, row_base + i, p] * k_blk[g, b, p]
//
// Per group this is a GEMM (rows x P) . (P x blocks).  Only candidates b < b_t matter for
// row i (b_t = (pos0 + i) / B), so each 128-row tile stops at the last candidate of its
// last row; columns past a row's own candidates are written but never read.
//
// Design (one CTA per SM, persistent over work items):
//   warp 0      TMA producer: A tile (128 query rows x P, K-major, 128-byte swizzle) once
//               per item, B tiles (128 blocks x P) through a 2-stage ring.
//   warp 1      allocates 256 TMEM columns (two 128x128 fp32 accumulators) and issues
//               tcgen05.mma kind::f16 (M=128, N=128, K=16) from one thread; commits free
//               the B stage and publish the accumulator.
//   warps 2..9  epilogue, two warps per TMEM lane quarter, each taking two of a tile's four
//               32-column chunks: tcgen05.ld 32 lanes x 32 columns (thread = query row), then
//               by mode:
//               K2_SCORES    write a swizzled 32x32 fp32 tile to shared memory and TMA-store
//                            it (the store clips rows past the call's rows and columns past
//                            the workspace row length);
//               K2_MAXIMA    per row, the largest score key of each 8 consecutive candidates
//                            below the row's own block (a 4-byte key per 8 scores);
//               K2_SURVIVORS per row, the candidates whose score key reaches the row's bound:
//                            their keys, in place, and a mask word per 32 candidates;
//                            nothing else leaves the SM.
// The last two serve the top-k without materialising the scores: the (k-1)-th largest of a
// row's group maxima is at most its (k-1)-th largest score (those maxima are k-1 distinct
// candidates), so every block the top-k keeps, ties included, reaches that bound.
// Every wait is bounded (globaltimer); on expiry the CTA raises an abort flag, drains the
// copies and MMAs it has in flight, frees TMEM and returns.
#pragma once
#include "ptx.cuh"

namespace sgqa {

struct K2Args {
  int32_t G, P, B;
  int32_t kch;          // P / 64
  int64_t Tc;           // rows in this launch
  int64_t row_base;     // first q_proxy row of this launch (TMA y coordinate)
  int64_t pos0;         // absolute position of row 0 of this launch
  int32_t n_mtiles;     // ceil(Tc / 128)
  int32_t items_per_m;  // ceil(max n-tiles / nti)
  int32_t nti;          // n-tiles per work item
  int64_t n_items;      // G * n_mtiles * items_per_m
  int64_t ld;           // score row length of the workspace (elements)
  uint64_t wait_ns;
  int32_t mode;         // K2_SCORES, K2_MAXIMA or K2_SURVIVORS
  // K2_SCORES: with tile_flag, only the (group, 128-row tile) items whose flag is set
  const int32_t* tile_flag;  // [G, n_mtiles] or null
  // K2_MAXIMA: maxima[(g * Tc + row) * ld8 + j] = largest key of candidates gs j .. gs j +
  // gs - 1 below the row's own block, gs = 8 or 16 (only groups with at least one such
  // candidate are written; 0 for a group's candidates past it); ld8 = 4 * ceil(ld / 32)
  uint32_t* maxima;
  int64_t ld8;
  int32_t gs;
  // K2_SURVIVORS, row r = g * Tc + row: bit u of smask[r * ld32 + x / 32] set for candidate
  // x = 32 (x / 32) + u when its key reaches thr[r] (words of candidates below the row's own
  // block only), and that key at skeys[r * ld + x]
  const uint32_t* thr;
  uint32_t* smask;
  int64_t ld32;
  uint32_t* skeys;
};

enum K2Mode : int { K2_SCORES = 0, K2_MAXIMA = 1, K2_SURVIVORS = 2 };

constexpr int K2_THREADS = 320;
constexpr uint32_t K2_TILE_BYTES = 128 * 128;            // 128 rows x 128 B (64 bf16)
constexpr uint32_t K2_A_OFF = 0;                         // 4 chunks
constexpr uint32_t K2_B_OFF = 4 * K2_TILE_BYTES;         // 2 stages x 4 chunks
constexpr uint32_t K2_C_OFF = K2_B_OFF + 8 * K2_TILE_BYTES;  // 8 warps x 4 KB
constexpr uint32_t K2_BAR_OFF = K2_C_OFF + 8 * 4096;
constexpr uint32_t K2_SMEM_BYTES = K2_BAR_OFF + 128 + 1024;  // + alignment slack

struct K2Item {
  int32_t g, m, n_begin, n_end;
};

__device__ __forceinline__ bool k2_decode_item(const K2Args& a, int64_t item, K2Item& it) {
  const int64_t per_g = (int64_t)a.n_mtiles * a.items_per_m;
  it.g = (int32_t)(item / per_g);
  const int64_t rem = item % per_g;
  it.m = (int32_t)(rem / a.items_per_m);
  const int32_t c = (int32_t)(rem % a.items_per_m);
  int64_t last_row = (int64_t)it.m * 128 + 127;
  if (last_row > a.Tc - 1) last_row = a.Tc - 1;
  const int64_t ncand = (a.pos0 + last_row) / a.B;  // candidates of the tile's last row
  const int32_t nt = (int32_t)((ncand + 127) / 128);
  it.n_begin = c * a.nti;
  it.n_end = it.n_begin + a.nti < nt ? it.n_begin + a.nti : nt;
  if (a.tile_flag && a.tile_flag[(int64_t)it.g * a.n_mtiles + it.m] == 0) return false;
  return it.n_begin < it.n_end;
}

__global__ void __launch_bounds__(K2_THREADS, 1)
    k2_indexer(const K2Args a, const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmC) {
  extern __shared__ uint8_t k2_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(k2_smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + K2_BAR_OFF);
  const uint32_t bar_a_full = smem_u32(&bars[0]);
  const uint32_t bar_a_empty = smem_u32(&bars[1]);
  const uint32_t bar_b_full0 = smem_u32(&bars[2]);     // + 8 * s
  const uint32_t bar_b_empty0 = smem_u32(&bars[4]);
  const uint32_t bar_acc_full0 = smem_u32(&bars[6]);
  const uint32_t bar_acc_empty0 = smem_u32(&bars[8]);
  const uint32_t bar_final = smem_u32(&bars[10]);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + K2_BAR_OFF + 96);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + K2_BAR_OFF + 100);

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();

  if (threadIdx.x == 0) {
    mbar_init(bar_a_full, 1);
    mbar_init(bar_a_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_b_full0 + 8 * s, 1);
      mbar_init(bar_b_empty0 + 8 * s, 1);
      mbar_init(bar_acc_full0 + 8 * s, 1);
      mbar_init(bar_acc_empty0 + 8 * s, 8);
    }
    mbar_init(bar_final, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    prefetch_tensormap(&tmC);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t chunk_bytes = K2_TILE_BYTES * (uint32_t)a.kch;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t it_a = 0, it_b = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; item < a.n_items && ok; item += gridDim.x) {
        K2Item it;
        if (!k2_decode_item(a, item, it)) continue;
        if (it_a > 0 && !mbar_wait(bar_a_empty, (it_a - 1) & 1, a.wait_ns, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(bar_a_full, chunk_bytes);
        for (int kc = 0; kc < a.kch; ++kc)
          tma_load_3d(sbase + K2_A_OFF + kc * K2_TILE_BYTES, &tmA, bar_a_full, kc * 64,
                      (int32_t)(a.row_base + (int64_t)it.m * 128), it.g);
        ++it_a;
        for (int32_t n = it.n_begin; n < it.n_end; ++n) {
          const uint32_t s = it_b & 1;
          if (it_b >= 2 && !mbar_wait(bar_b_empty0 + 8 * s, ((it_b >> 1) - 1) & 1, a.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar_b_full0 + 8 * s, chunk_bytes);
          for (int kc = 0; kc < a.kch; ++kc)
            tma_load_3d(sbase + K2_B_OFF + (s * 4 + kc) * K2_TILE_BYTES, &tmB, bar_b_full0 + 8 * s, kc * 64, n * 128,
                        it.g);
          ++it_b;
        }
      }
      // Drain: the latest load issued to each buffer must land before the CTA exits.
      if (it_a > 0) mbar_wait(bar_a_full, (it_a - 1) & 1, kDrainLimitNs);
      for (uint32_t s = 0; s < 2; ++s) {
        if (it_b > s) {
          const uint32_t last = ((it_b - 1 - s) & ~1u) + s;  // last use index of stage s
          mbar_wait(bar_b_full0 + 8 * s, (last >> 1) & 1, kDrainLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, 128);
      uint32_t it_a = 0, it_b = 0, it_acc = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; item < a.n_items && ok; item += gridDim.x) {
        K2Item it;
        if (!k2_decode_item(a, item, it)) continue;
        if (!mbar_wait(bar_a_full, it_a & 1, a.wait_ns, abort_flag)) { ok = false; break; }
        ++it_a;
        for (int32_t n = it.n_begin; n < it.n_end; ++n) {
          const uint32_t s = it_b & 1;
          const uint32_t acc = it_acc & 1;
          if (!mbar_wait(bar_b_full0 + 8 * s, (it_b >> 1) & 1, a.wait_ns, abort_flag)) { ok = false; break; }
          if (it_acc >= 2 && !mbar_wait(bar_acc_empty0 + 8 * acc, ((it_acc >> 1) - 1) & 1, a.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * 128;
          for (int kc = 0; kc < a.kch; ++kc) {
            const uint64_t adesc = smem_desc_k_sw128(sbase + K2_A_OFF + kc * K2_TILE_BYTES);
            const uint64_t bdesc = smem_desc_k_sw128(sbase + K2_B_OFF + (s * 4 + kc) * K2_TILE_BYTES);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              tc_mma_f16(d_tmem, adesc + 2 * ks, bdesc + 2 * ks, idesc, (kc | ks) != 0);
          }
          tc_commit(bar_b_empty0 + 8 * s);
          tc_commit(bar_acc_full0 + 8 * acc);
          ++it_b;
          ++it_acc;
        }
        if (ok) tc_commit(bar_a_empty);
      }
      // every MMA issued so far completes before TMEM is released
      tc_commit(bar_final);
      mbar_wait(bar_final, 0, kDrainLimitNs);
    }
  } else {
    // ---------------- epilogue: TMEM -> smem -> TMA store ----------------
    const uint32_t q = warp & 3;          // TMEM lane quarter this warp may access
    const uint32_t e = warp - 2;          // staging slot
    const int c0 = 2 * (int)(e >> 2);     // first of this warp's two 32-column chunks
    uint32_t it_acc = 0, n_store = 0;
    bool ok = true;
    for (int64_t item = blockIdx.x; item < a.n_items && ok; item += gridDim.x) {
      K2Item it;
      if (!k2_decode_item(a, item, it)) continue;
      for (int32_t n = it.n_begin; n < it.n_end; ++n) {
        const uint32_t acc = it_acc & 1;
        if (!mbar_wait(bar_acc_full0 + 8 * acc, (it_acc >> 1) & 1, a.wait_ns, abort_flag)) { ok = false; break; }
        tc_fence_after();
        if (a.mode == K2_SCORES) {
          for (int c = c0; c < c0 + 2; ++c) {
            // A 32x32 box wholly past the workspace row or the call's rows is never read:
            // skip it entirely (warp-uniform), so only real stores cycle the two buffers.
            const int32_t x0 = n * 128 + c * 32, y0 = it.m * 128 + (int32_t)q * 32;
            if (x0 >= a.ld || y0 >= a.Tc) continue;
            uint32_t r[32];
            tmem_ld_32x32b_x32(tmem_base + ((q * 32) << 16) + acc * 128 + c * 32, r);
            tmem_ld_wait();
            const uint32_t stage_addr = sbase + K2_C_OFF + e * 4096;
            // this warp's previous store must have finished reading its buffer
            if (lane == 0) bulk_wait_group_read<0>();
            __syncwarp();
            const uint32_t row_addr = stage_addr + lane * 128;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const uint32_t dst = row_addr + ((u ^ (lane & 7)) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(r[4 * u]), "r"(r[4 * u + 1]),
                           "r"(r[4 * u + 2]), "r"(r[4 * u + 3])
                           : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&tmC, stage_addr, x0, y0, it.g);
              bulk_commit_group();
            }
            ++n_store;
          }
        } else {
          // thread = query row of the tile; its candidates are the blocks below its own
          const int64_t row = (int64_t)it.m * 128 + q * 32 + lane;
          const int64_t bt = row < a.Tc ? (a.pos0 + row) / a.B : 0;
          const int64_t rr = (int64_t)it.g * a.Tc + row;
          const uint32_t thr = (a.mode == K2_SURVIVORS && row < a.Tc) ? a.thr[rr] : 0u;
          for (int c = c0; c < c0 + 2; ++c) {
            const int64_t x0 = (int64_t)n * 128 + c * 32;
            if (x0 >= a.ld || (int64_t)it.m * 128 + q * 32 >= a.Tc) continue;  // warp-uniform
            uint32_t r[32];
            tmem_ld_32x32b_x32(tmem_base + ((q * 32) << 16) + acc * 128 + c * 32, r);
            tmem_ld_wait();
            if (x0 >= bt) continue;  // no candidate of this row here
            if (a.mode == K2_MAXIMA) {
              uint32_t mx[4] = {0u, 0u, 0u, 0u};
#pragma unroll
              for (int u = 0; u < 32; ++u)
                if (x0 + u < bt) mx[u >> 3] = max(mx[u >> 3], score_key(__uint_as_float(r[u])));
              if (a.gs == 16) {
                // groups 16j .. 16j+15 with j = x0/16, x0/16+1: 8-byte aligned
                *reinterpret_cast<uint2*>(a.maxima + rr * a.ld8 + x0 / 16) =
                    make_uint2(max(mx[0], mx[1]), max(mx[2], mx[3]));
              } else {
                // groups 8j .. 8j+7 with j = x0/8 .. x0/8+3; x0 is a multiple of 32, so 16-byte aligned
                *reinterpret_cast<uint4*>(a.maxima + rr * a.ld8 + x0 / 8) = make_uint4(mx[0], mx[1], mx[2], mx[3]);
              }
            } else {
              uint32_t m = 0u;
              uint32_t* krow = a.skeys + rr * a.ld;
#pragma unroll
              for (int u = 0; u < 32; ++u) {
                const uint32_t kk = score_key(__uint_as_float(r[u]));
                if (x0 + u < bt && kk >= thr) {
                  m |= 1u << u;
                  krow[x0 + u] = kk;
                }
              }
              a.smask[rr * a.ld32 + x0 / 32] = m;
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_acc_empty0 + 8 * acc);
        ++it_acc;
      }
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 256);
}

}  // namespace sgqa
