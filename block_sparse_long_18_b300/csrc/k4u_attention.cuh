// k4u_attention.cuh -- gated sparse attention for 8 query rows at a time over the union of
// their selected blocks, on the 5th-generation tensor cores (tcgen05, tensor memory).
//
// Same operation as k4_attention.cuh (ai.info article "StepFun Details Step 5 Preview's
// 92-Block Agent Design", "Why StepFun chose 92 transformer blocks": Gated GQA; ai4snews
// item "Step 5 Preview bets on depth over width", Interpretation para 2: sparse flash
// attention over the selected blocks; phantomic12 entry: 4 KV groups x 16 heads, D = 192):
//   for row i (position t), group g, head h of g:  J = { j in the row's selected blocks : j <= t }
//   o = softmax_j(scale * q_h . k_j) . v_j ;  out = o * sigmoid(gate) ;  lse = log sum exp
//
// Unit = (KV group g, 8 consecutive query rows).  Its 8 rows x 16 heads = 128 (row, head)
// pairs are the M of the MMA, one pair per tensor-memory lane.  The keys are the union U of
// the 8 rows' selections in ascending block order: every union block is gathered once per
// unit and serves every row that selected it; a row's scores outside its own selection
// (and past its position inside its own block) are masked in the softmax.
//   S [128 pairs x 128 keys]  = Q [128 x 192] (tensor memory) . K_chunk [128 keys x 192]^T
//   O [128 pairs x 192]      += P [128 x 128] (tensor memory, bf16) . V_chunk [128 keys x 192]
// Both products read A from tensor memory and B from shared memory, where each union block
// lands by one TMA copy (box {64, 8, 3}) as three 1 KB swizzle atoms [D chunk][key][64]:
// K-major for K (atoms 3 KB apart), MN-major for V.  The softmax is per thread: a (row,
// head) pair owns its TMEM lane, so maxima, sums and the rare O rescale need no exchange.
//
// Tensor memory (512 columns): Q 0..95 (bf16 pairs), O 96..287, S 288..415, P 416..479.
// Roles (one persistent CTA per SM, 12 warps, units dealt round-robin, group-major):
//   warp 0     K producer: 16 copies per 128-key chunk into a 2-slot ring
//   warp 3     V producer: the same for V
//   warp 1     allocates tensor memory; one thread issues S(c), then O(c-1)
//   warp 2     builds the next unit's union tables (double-buffered)
//   warps 4-11 softmax + epilogue: thread = (row, head) = its TMEM lane, two warps per lane
//              quarter (one per half of the keys); they also write the next unit's Q into
//              tensor memory, so its first S overlaps this epilogue
// Every wait is bounded; on expiry the CTA raises an abort flag, drains and returns.
#pragma once
#include "ptx.cuh"

namespace sgqa {

constexpr int K4U_D = 192;                          // head dimension
constexpr int K4U_CB = 16;                          // union blocks per chunk (128 keys)
constexpr uint32_t K4U_SLOT = K4U_CB * 3072;        // one chunk of K (or V): 48 KB
constexpr int K4U_MAXU = 4096;                      // union capacity: 8 rows x 512 blocks
constexpr int K4U_WIN = 16384;                      // blocks covered by one builder bitmap
constexpr int K4U_MAX_WIN = 16;                     // windows a unit's blocks may span
constexpr int K4U_MAX_BLOCKS = K4U_WIN * K4U_MAX_WIN;  // 262,144 blocks: positions below 2,097,152
// one table buffer: union entries (u16: block offset inside its window), per-row membership
// bits over union positions, meta
constexpr uint32_t K4U_TB_UBLK = 0;
constexpr uint32_t K4U_TB_RBITS = 2 * K4U_MAXU;              // uint32 [8][K4U_MAXU / 32]
constexpr uint32_t K4U_TB_META = K4U_TB_RBITS + 8 * (K4U_MAXU / 8);
// meta, int32: [0] nU, [1..8] own position per row, [9] windows used, [10..25] the union
// position at which each window's entries start (ascending; an empty window repeats the
// next start)
constexpr int K4U_META_NWIN = 9, K4U_META_WSTART = 10;
constexpr uint32_t K4U_TB = K4U_TB_META + 128;
static_assert((K4U_META_WSTART + K4U_MAX_WIN) * 4 <= 128, "k4u table meta");
constexpr uint32_t K4U_K_OFF = 0;
constexpr uint32_t K4U_V_OFF = 2 * K4U_SLOT;
constexpr uint32_t K4U_T_OFF = 4 * K4U_SLOT;
constexpr uint32_t K4U_BM_OFF = K4U_T_OFF + 2 * K4U_TB;      // uint32 [K4U_WIN / 32] window bitmap
constexpr uint32_t K4U_PRE_OFF = K4U_BM_OFF + K4U_WIN / 8;   // uint32 [K4U_WIN / 32] prefix counts
constexpr uint32_t K4U_X_OFF = K4U_PRE_OFF + K4U_WIN / 8;    // float [2][128]: row sums, reference maxima per pair
constexpr uint32_t K4U_BAR_OFF = K4U_X_OFF + 2 * 128 * 4;
constexpr uint32_t K4U_SMEM = K4U_BAR_OFF + 512 + 1024;     // + barriers, flags, alignment
constexpr int K4U_THREADS = 384;
constexpr uint32_t kSuspendNs = 20000;  // a waiting role sleeps in its polls (woken when the phase completes)
constexpr uint32_t K4U_COL_Q = 0, K4U_COL_O = 96, K4U_COL_S = 288, K4U_COL_P = 416;
static_assert(K4U_SMEM <= 232448, "k4u shared memory");

struct K4UArgs {
  const __nv_bfloat16* q;     // [rows, H, D]
  const __nv_bfloat16* gate;  // [rows, H, D] or [rows, H]
  __nv_bfloat16* out;         // [rows, H, D]
  float* lse;                 // [rows, H] or null
  const int32_t* sel_idx;     // [G, rows, kcap], ascending, -1 padded
  const int32_t* sel_cnt;     // [G, rows]
  int64_t rows, pos0, ctx_cap;
  int32_t G, H, kcap;         // 16 heads per group, blocks of 8, D = 192
  float scale_log2;
  int32_t gate_per_dim;
  uint64_t wait_ns;
  // routed mode: the units to serve are units[0 .. *n_units_dev) (unit = g * tiles + tile
  // of 8 slots); otherwise every unit of the call
  const int32_t* units;
  const int32_t* n_units_dev;
  // grouped units: perm[g * rows + s] is the row at slot s (null: slot s is row s)
  const int32_t* perm;
};

__global__ void __launch_bounds__(K4U_THREADS, 1)
    k4u_sparse_attn(const __grid_constant__ K4UArgs a, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t k4u_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(k4u_smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb0 = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + K4U_BAR_OFF);
  auto bar = [&](int idx) { return smem_u32(&bars[idx]); };
  // kKEmpty + s completes when S of the chunk in K slot s is done (the slot and the S columns
  // may be reused, the chunk's scores read; after a unit's last chunk, Q too); kVEmpty + s
  // when O += P V of the chunk in V slot s is done (the slot and the P columns free).  A
  // waiter is never two phases behind on either, so the parity of its chunk identifies it.
  enum { kKFull = 0, kKEmpty = 2, kVFull = 4, kVEmpty = 6, kTblFull = 8, kTblEmpty = 10, kSFree = 12, kPFull = 13,
         kQFull = 14, kOEmpty = 15, kFinal = 16 };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + K4U_BAR_OFF + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + K4U_BAR_OFF + 260);

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const int64_t ntiles = (a.rows + 7) / 8;
  // units of this launch: every (group, 8-row tile), or the routed list
  const int64_t n_units = a.units ? (int64_t)*a.n_units_dev : (int64_t)a.G * ntiles;
  auto unit_id = [&](int64_t u) -> int64_t { return a.units ? (int64_t)__ldg(a.units + u) : u; };
  // row at slot s of group g; a.rows (no row) for the empty slots of a ragged last tile
  auto row_at = [&](int32_t g, int64_t s) -> int64_t {
    return s >= a.rows ? a.rows : (a.perm ? (int64_t)__ldg(a.perm + (int64_t)g * a.rows + s) : s);
  };
  auto tbl = [&](uint32_t buf) { return smem + K4U_T_OFF + buf * K4U_TB; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kKFull + s), 1);
      mbar_init(bar(kKEmpty + s), 1);
      mbar_init(bar(kVFull + s), 1);
      mbar_init(bar(kVEmpty + s), 1);
      mbar_init(bar(kTblFull + s), 1);
      mbar_init(bar(kTblEmpty + s), 11);  // K and V producers, MMA thread, 8 softmax warps
    }
    mbar_init(bar(kSFree), 8);
    mbar_init(bar(kPFull), 8);
    mbar_init(bar(kQFull), 8);
    mbar_init(bar(kOEmpty), 8);
    mbar_init(bar(kFinal), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // lane 0 waits, the warp agrees on the outcome
  auto warp_wait = [&](int b, uint32_t parity) -> bool {
    bool r = true;
    if (lane == 0) r = mbar_wait(bar(b), parity, a.wait_ns, abort_flag, kSuspendNs);
    return __shfl_sync(0xffffffffu, r, 0) != 0;
  };

  if (warp == 2) {
    // ------------------------------- union builder -------------------------------
    // Per window of K4U_WIN blocks: mark every selected block in a bitmap, turn the bitmap
    // into ascending union positions (prefix popcounts), then mark each row's entries in
    // its membership bits.  The rows' own blocks are noted for the causal mask.
    uint32_t* bm = reinterpret_cast<uint32_t*>(smem + K4U_BM_OFF);
    uint32_t* pre = reinterpret_cast<uint32_t*>(smem + K4U_PRE_OFF);
    uint32_t uc = 0;
    for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x, ++uc) {
      const uint32_t buf = uc & 1;
      if (uc >= 2 && !warp_wait(kTblEmpty + buf, ((uc >> 1) - 1) & 1)) break;
      const int64_t uid = unit_id(u);
      const int32_t g = (int32_t)(uid / ntiles);
      const int64_t i0 = (uid % ntiles) * 8;
      uint8_t* T = tbl(buf);
      uint16_t* ublk = reinterpret_cast<uint16_t*>(T + K4U_TB_UBLK);
      uint32_t* rbits = reinterpret_cast<uint32_t*>(T + K4U_TB_RBITS);
      int32_t* meta = reinterpret_cast<int32_t*>(T + K4U_TB_META);
      int32_t cnt_l = 0, bt_l = -1;
      const int64_t row_l = row_at(g, i0 + (lane & 7));  // lanes 0..7: the unit's rows
      if (lane < 8 && i0 + lane < a.rows) {
        const int64_t i = row_l;
        bt_l = (int32_t)((a.pos0 + i) >> 3);
        int32_t c = __ldg(a.sel_cnt + (int64_t)g * a.rows + i);
        const int32_t cap = a.kcap < bt_l + 1 ? a.kcap : bt_l + 1;
        if (c < 1 || c > cap) {
          report_error(kErrBounds);
          c = c < 1 ? 1 : cap;
        }
        cnt_l = c;
      }
      for (int w = lane; w < 8 * (K4U_MAXU / 32); w += 32) rbits[w] = 0u;
      if (lane < 8) meta[1 + lane] = -1;
      int32_t bmax = bt_l;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) bmax = max(bmax, __shfl_xor_sync(0xffffffffu, bmax, o));
      int32_t nU = 0, nwin = 0;
      for (int32_t wb = 0; wb <= bmax; wb += K4U_WIN, ++nwin) {
        if (lane == 0) meta[K4U_META_WSTART + nwin] = nU;
        for (int w = lane; w < K4U_WIN / 32; w += 32) bm[w] = 0u;
        __syncwarp();
        for (int r0 = 0; r0 < 8; r0 += 2) {  // two rows' entries in flight at once
          int32_t e[2][16];
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int32_t cnt = __shfl_sync(0xffffffffu, cnt_l, r0 + rr);
            const int64_t row = __shfl_sync(0xffffffffu, row_l, r0 + rr);
            const int32_t* sel = a.sel_idx + ((int64_t)g * a.rows + row) * a.kcap;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const int32_t j = (int32_t)lane + 32 * k;
              e[rr][k] = j < cnt ? __ldg(sel + j) : -1;
            }
          }
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int32_t cnt = __shfl_sync(0xffffffffu, cnt_l, r0 + rr);
            const int32_t bt = __shfl_sync(0xffffffffu, bt_l, r0 + rr);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const int32_t j = (int32_t)lane + 32 * k;
              if (j >= cnt) continue;
              const int32_t b = e[rr][k];
              if (b < 0 || b > bt) {
                if (wb == 0) report_error(kErrBounds);
                continue;
              }
              const int32_t o = b - wb;
              if (o >= 0 && o < K4U_WIN) atomicOr(&bm[o >> 5], 1u << (o & 31));
            }
          }
        }
        __syncwarp();
        constexpr int WPL = K4U_WIN / 32 / 32;  // bitmap words per lane
        uint32_t pc = 0;
#pragma unroll
        for (int k = 0; k < WPL; ++k) pc += __popc(bm[WPL * lane + k]);
        uint32_t incl = pc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
          if ((int)lane >= o) incl += v;
        }
        uint32_t run = (uint32_t)nU + incl - pc;
        for (int k = 0; k < WPL; ++k) {
          const uint32_t wi = WPL * lane + k;
          uint32_t bits = bm[wi];
          pre[wi] = run;
          while (bits) {
            const uint32_t bit = __ffs(bits) - 1;
            bits &= bits - 1;
            ublk[run++] = (uint16_t)(32 * wi + bit);
          }
        }
        nU += (int32_t)__shfl_sync(0xffffffffu, incl, 31);
        __syncwarp();
        for (int r0 = 0; r0 < 8; r0 += 2) {
          int32_t e[2][16];
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int32_t cnt = __shfl_sync(0xffffffffu, cnt_l, r0 + rr);
            const int64_t row = __shfl_sync(0xffffffffu, row_l, r0 + rr);
            const int32_t* sel = a.sel_idx + ((int64_t)g * a.rows + row) * a.kcap;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const int32_t j = (int32_t)lane + 32 * k;
              e[rr][k] = j < cnt ? __ldg(sel + j) : -1;
            }
          }
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int r = r0 + rr;
            const int32_t cnt = __shfl_sync(0xffffffffu, cnt_l, r);
            const int32_t bt = __shfl_sync(0xffffffffu, bt_l, r);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const int32_t j = (int32_t)lane + 32 * k;
              const int32_t b = e[rr][k];
              if (j >= cnt || b < 0 || b > bt) continue;
              const int32_t o = b - wb;
              if (o < 0 || o >= K4U_WIN) continue;
              const uint32_t w = (uint32_t)o >> 5;
              const uint32_t pos = pre[w] + __popc(bm[w] & ((1u << (o & 31)) - 1u));
              atomicOr(&rbits[r * (K4U_MAXU / 32) + (pos >> 5)], 1u << (pos & 31));
              if (b == bt) meta[1 + r] = (int32_t)pos;
            }
          }
        }
        __syncwarp();
      }
      if (nU == 0) {  // only after bad input: one fully masked block keeps every role in step
        if (lane == 0) {
          ublk[0] = 0;
          meta[K4U_META_WSTART] = 0;
        }
        nU = 1;
        nwin = 1;
      }
      if (lane == 0) {
        meta[0] = nU;
        meta[K4U_META_NWIN] = nwin;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kTblFull + buf));
    }
  } else if (warp == 0 || warp == 3) {
    // --------------------------- TMA producers (K: warp 0, V: warp 3) ---------------------------
    const bool is_k = warp == 0;
    const CUtensorMap* map = is_k ? &tmK : &tmV;
    const int full0 = is_k ? kKFull : kVFull, empty0 = is_k ? kKEmpty : kVEmpty;
    const uint32_t base0 = sb0 + (is_k ? K4U_K_OFF : K4U_V_OFF);
    // Each union block is fetched once per unit, but neighbouring units (the CTAs in flight
    // work on adjacent rows of one group) select many of the same blocks: keep K/V in L2.
    const uint64_t keep = make_l2_evict_last();
    uint32_t uc = 0, kc = 0;
    bool ok = true;
    for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
      const uint32_t buf = uc & 1;
      if (!warp_wait(kTblFull + buf, (uc >> 1) & 1)) break;
      const int32_t g = (int32_t)(unit_id(u) / ntiles);
      const uint8_t* T = tbl(buf);
      const uint16_t* ublk = reinterpret_cast<const uint16_t*>(T + K4U_TB_UBLK);
      const int32_t* meta = reinterpret_cast<const int32_t*>(T + K4U_TB_META);
      const int32_t nU = meta[0], nwin = meta[K4U_META_NWIN];
      const int32_t nch = (nU + K4U_CB - 1) / K4U_CB;
      const int64_t row0 = (int64_t)g * a.ctx_cap;
      for (int32_t c = 0; c < nch; ++c) {
        const uint32_t slot = kc & 1;
        bool r = true;
        if (lane == 0) {
          if (kc >= 2) r = mbar_wait(bar(empty0 + slot), ((kc >> 1) - 1) & 1, a.wait_ns, abort_flag, kSuspendNs);
          if (r) mbar_arrive_expect_tx(bar(full0 + slot), K4U_SLOT);
        }
        ok = __shfl_sync(0xffffffffu, r, 0) != 0;
        if (!ok) break;
        if (lane < K4U_CB) {
          int32_t p = c * K4U_CB + (int32_t)lane;
          p = p < nU ? p : nU - 1;  // past the union: a valid block, masked
          // the window holding position p: the last one whose entries start at or before p
          int32_t w = 0;
#pragma unroll
          for (int x = 1; x < K4U_MAX_WIN; ++x) w += (x < nwin && meta[K4U_META_WSTART + x] <= p) ? 1 : 0;
          const int32_t b = w * K4U_WIN + (int32_t)ublk[p];
          tma_load_3d_hint(base0 + slot * K4U_SLOT + lane * 3072, map, bar(full0 + slot), 0,
                           (int32_t)(row0 + (int64_t)b * 8), 0, keep);
        }
        __syncwarp();
        ++kc;
      }
      if (lane == 0) mbar_arrive(bar(kTblEmpty + buf));
    }
    // drain: the latest copies into each slot land before the CTA leaves
    if (lane == 0)
      for (uint32_t b = 0; b < 2; ++b)
        if (kc > b) {
          const uint32_t last = ((kc - 1 - b) & ~1u) + b;
          mbar_wait(bar(full0 + b), (last >> 1) & 1, kDrainLimitNs);
        }
  } else if (warp == 1) {
    // ------------------------------- MMA issuer -------------------------------
    // A tcgen05.mma issue takes as long as the MMA runs (about 65 cycles at N = 128), so the
    // tensor pipe idles whenever this thread is not issuing: one commit per product, and the
    // inputs of each O are tested (without blocking) before the S ahead of it is issued.
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, 128);
      const uint32_t id_o = idesc_bf16_f32(128, 192) | (1u << 16);  // B (V) is MN-major
      uint32_t uc = 0, kc = 0;
      bool ok = true;
      auto issue_s = [&](uint32_t c) {
        tc_fence_after();
        const uint32_t kb = sb0 + K4U_K_OFF + (c & 1) * K4U_SLOT;
#pragma unroll
        for (int ks = 0; ks < 12; ++ks)
          tc_mma_ts(tmem + K4U_COL_S, tmem + K4U_COL_Q + 8 * ks,
                    smem_desc_k_sw128_sbo(kb + (ks >> 2) * 1024 + (ks & 3) * 32, 3072), id_s, ks > 0 ? 1u : 0u);
        tc_commit(bar(kKEmpty + (c & 1)));
      };
      auto issue_o = [&](uint32_t c, bool first) {
        tc_fence_after();
        const uint32_t vb = sb0 + K4U_V_OFF + (c & 1) * K4U_SLOT;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          tc_mma_ts(tmem + K4U_COL_O, tmem + K4U_COL_P + 8 * ks, smem_desc_mn_sw128(vb + ks * 6144, 1024, 3072),
                    id_o, (first && ks == 0) ? 0u : 1u);
        tc_commit(bar(kVEmpty + (c & 1)));
      };
      auto s_wait = [&](uint32_t c) -> bool {
        return mbar_wait(bar(kKFull + (c & 1)), (c >> 1) & 1, a.wait_ns, abort_flag, kSuspendNs) &&
               (c == 0 || mbar_wait(bar(kSFree), (c - 1) & 1, a.wait_ns, abort_flag, kSuspendNs));
      };
      // inputs of O(c): P(c), V(c)
      auto o_ready = [&](uint32_t c) -> bool {
        return mbar_test_wait(bar(kPFull), c & 1) & mbar_test_wait(bar(kVFull + (c & 1)), (c >> 1) & 1);
      };
      auto o_wait = [&](uint32_t c) -> bool {
        return mbar_wait(bar(kPFull), c & 1, a.wait_ns, abort_flag, kSuspendNs) &&
               mbar_wait(bar(kVFull + (c & 1)), (c >> 1) & 1, a.wait_ns, abort_flag, kSuspendNs);
      };
      for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
        const uint32_t buf = uc & 1;
        if (!mbar_wait(bar(kTblFull + buf), (uc >> 1) & 1, a.wait_ns, abort_flag, kSuspendNs)) break;
        const int32_t nU = reinterpret_cast<const int32_t*>(tbl(buf) + K4U_TB_META)[0];
        const int32_t nch = (nU + K4U_CB - 1) / K4U_CB;
        mbar_arrive(bar(kTblEmpty + buf));
        if (!mbar_wait(bar(kQFull), uc & 1, a.wait_ns, abort_flag, kSuspendNs) || !s_wait(kc)) break;
        issue_s(kc);
        // the unit's first P.V overwrites O: the previous unit's O must have been read out
        if (uc >= 1 && !mbar_wait(bar(kOEmpty), (uc - 1) & 1, a.wait_ns, abort_flag, kSuspendNs)) break;
        for (int32_t j = 1; j < nch; ++j) {
          const uint32_t c = kc + (uint32_t)j;
          // S(c), then O(c - 1); O's inputs are tested before S goes out, so that the test's
          // latency hides behind S's issue
          if (!s_wait(c)) {
            ok = false;
            break;
          }
          const bool ro = o_ready(c - 1);
          issue_s(c);
          if (!ro && !o_wait(c - 1)) {
            ok = false;
            break;
          }
          issue_o(c - 1, j == 1);
        }
        if (!ok) break;
        const uint32_t cl = kc + (uint32_t)nch - 1;
        if (!o_wait(cl)) break;
        issue_o(cl, nch == 1);
        kc += (uint32_t)nch;
      }
      tc_commit(bar(kFinal));
      mbar_wait(bar(kFinal), 0, kDrainLimitNs);
    }
    __syncwarp();
  } else {
    // ------------------------------- softmax + epilogue -------------------------------
    // Eight warps, two per TMEM lane quarter q = w & 3.  In the chunk loop warp (q, hf) owns
    // query row 2q + hf, its 16 lanes read through the .16x256b shape: every softmax
    // decision (which blocks the row selected, the maxima, the rescale) is uniform over the
    // warp and needs no exchange with other warps.  For Q and the epilogue the two warps of
    // a quarter split the columns instead (thread = pair, .32x32b).
    const uint32_t sw = warp - 4;         // 0..7
    const uint32_t q = warp & 3;          // TMEM lane quarter of this warp
    const uint32_t hf = sw >> 2;          // row within the quarter; half of Q and O columns
    const uint32_t m = q * 32 + lane;     // this thread's (row, head) pair = its TMEM lane
    const uint32_t r = m >> 4, h = m & 15;
    const uint32_t lbase = (q * 32) << 16;
    const uint32_t tQ = tmem + lbase + K4U_COL_Q + 48 * hf, tO = tmem + lbase + K4U_COL_O + 96 * hf;
    const uint32_t rr = 2 * q + hf;        // the query row this warp serves in the chunk loop
    const uint32_t hA = lane >> 2, hB = hA + 8, kq = 2 * (lane & 3);
    const uint32_t lb16 = (q * 32 + 16 * hf) << 16;  // the row's 16 TMEM lanes
    const uint32_t tS16 = tmem + lb16 + K4U_COL_S, tP16 = tmem + lb16 + K4U_COL_P, tO16 = tmem + lb16 + K4U_COL_O;
    float* xchg = reinterpret_cast<float*>(smem + K4U_X_OFF);  // row sums per pair, for the epilogue
    const float sl2 = a.scale_log2;
    // A lane's chunk sum of P past 2^16 (a reference maximum unset or far too low) sends the
    // chunk through the rescale; below it every P stays under 2^16, where bf16 P and the fp32
    // sums keep their relative precision
    constexpr float kLazySum = 65536.f;

    auto write_q = [&](int64_t u) {  // this half of the Q rows of unit u -> tensor memory
      const int64_t uid = unit_id(u);
      const int32_t g = (int32_t)(uid / ntiles);
      const int64_t i = row_at(g, (uid % ntiles) * 8 + r);
      const bool valid = i < a.rows;
      const uint4* src =
          reinterpret_cast<const uint4*>(a.q + ((i * a.H) + (int64_t)g * 16 + h) * K4U_D + 96 * hf);
      uint4 x[12];
#pragma unroll
      for (int e = 0; e < 12; ++e) x[e] = valid ? __ldg(src + e) : make_uint4(0u, 0u, 0u, 0u);
      uint32_t v[32];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        v[4 * e] = x[e].x;
        v[4 * e + 1] = x[e].y;
        v[4 * e + 2] = x[e].z;
        v[4 * e + 3] = x[e].w;
      }
      tmem_st_32x32b_x32(tQ, v);
      float w[16];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        w[4 * e] = __uint_as_float(x[8 + e].x);
        w[4 * e + 1] = __uint_as_float(x[8 + e].y);
        w[4 * e + 2] = __uint_as_float(x[8 + e].z);
        w[4 * e + 3] = __uint_as_float(x[8 + e].w);
      }
      tmem_st_32x32b_x16(tQ + 32, w);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kQFull));
    };

    // The eight warps meet on named barrier 1; a failed wait only marks the warp `bad`.
    // Each warp posts (bad || abort) before a barrier and all of them OR the eight posts
    // after it, so every warp leaves at the same barrier and none is left waiting in one.
    volatile uint32_t* post = reinterpret_cast<volatile uint32_t*>(smem + K4U_BAR_OFF + 320);  // [2][8]
    uint32_t xb = 0;
    bool bad = false;
    auto sync_stop = [&]() -> bool {
      if (lane == 0) post[(xb & 1) * 8 + sw] = (bad || *abort_flag) ? 1u : 0u;
      asm volatile("bar.sync 1, 256;" ::: "memory");
      const volatile uint32_t* pp = post + (xb & 1) * 8;
      const bool st = (pp[0] | pp[1] | pp[2] | pp[3] | pp[4] | pp[5] | pp[6] | pp[7]) != 0;
      ++xb;
      return st;
    };
    auto wait_ok = [&](int b, uint32_t parity) {  // skipped once the warp is bad
      if (!bad && !warp_wait(b, parity)) bad = true;
      return !bad;
    };

    if ((int64_t)blockIdx.x < n_units) write_q(blockIdx.x);
    uint32_t uc = 0, kc = 0;
    for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x, ++uc) {
      const uint32_t buf = uc & 1;
      wait_ok(kTblFull + buf, (uc >> 1) & 1);
      if (sync_stop()) break;
      const int64_t uid = unit_id(u);
      const int32_t g = (int32_t)(uid / ntiles);
      const int64_t i = row_at(g, (uid % ntiles) * 8 + r);
      const bool row_ok = i < a.rows;
      const uint8_t* T = tbl(buf);
      const uint32_t* rb = reinterpret_cast<const uint32_t*>(T + K4U_TB_RBITS);
      const int32_t* meta = reinterpret_cast<const int32_t*>(T + K4U_TB_META);
      const int32_t nU = meta[0];
      const int32_t nch = (nU + K4U_CB - 1) / K4U_CB;
      const int64_t hb = i * a.H + (int64_t)g * 16 + h;
      if (row_ok && a.gate_per_dim) {  // warm L2 for the epilogue's gate half-row
        const char* gp = reinterpret_cast<const char*>(a.gate + hb * K4U_D + 96 * hf);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(gp));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(gp + 128));
      }

      // chunk loop: this warp serves query row rr of the unit (TMEM lanes 16 rr .. 16 rr + 15);
      // thread t holds heads hA = t/4 and hB = hA + 8, keys kq, kq + 1 of every block
      const uint32_t* rb_row = rb + rr * (K4U_MAXU / 32);
      const int64_t ir = row_at(g, (uid % ntiles) * 8 + rr);
      const int32_t own_r = meta[1 + rr];
      const int32_t tlim_r = (int32_t)((a.pos0 + ir) & 7);
      float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;
      for (int32_t j = 0; j < nch; ++j) {
        const uint32_t c = kc + (uint32_t)j;
        const uint32_t mine = (rb_row[j >> 1] >> ((uint32_t)(j & 1) * 16)) & 0xFFFFu;  // warp-uniform
        const int32_t ownj = own_r - j * K4U_CB;  // own block's slot in this chunk, if 0..15
        float s[64];
        if (wait_ok(kKEmpty + (c & 1), (c >> 1) & 1)) {
          tc_fence_after();
          uint32_t v0[32], v1[32];
          tmem_ld_16x256b_x8(tS16, v0);
          tmem_ld_16x256b_x8(tS16 + 64, v1);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kSFree));
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            s[e] = __uint_as_float(v0[e]);
            s[32 + e] = __uint_as_float(v1[e]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e) s[e] = -INFINITY;
        }
        if (ownj >= 0 && ownj < K4U_CB) {  // the own block: keys past the row's position
#pragma unroll
          for (int k = 0; k < K4U_CB; ++k)
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (k == ownj && (int32_t)(kq + (e & 1)) > tlim_r) s[4 * k + e] = -INFINITY;
        }
        // P = 2^(scale_log2 * s - m) on the row's blocks with the current references, with no
        // branch: a block the row did not select gets the exponent offset -inf, so its P is 0.
        // A lane sum past kLazySum (some P far above 1) sends the chunk through a second pass
        // after the rescale to the chunk's true maxima.
        uint32_t pw[32];
        float lca = 0.f, lcb = 0.f;
        auto ppass = [&]() {
          lca = 0.f;
          lcb = 0.f;
          const float na = -ma, nb = -mb;
#pragma unroll
          for (int k = 0; k < K4U_CB; ++k) {
            const bool mk = ((mine >> k) & 1u) != 0u;
            const float ca = mk ? na : -INFINITY, cb = mk ? nb : -INFINITY;
            const float p0 = fast_exp2(fmaf(s[4 * k], sl2, ca)), p1 = fast_exp2(fmaf(s[4 * k + 1], sl2, ca));
            const float p2 = fast_exp2(fmaf(s[4 * k + 2], sl2, cb)), p3 = fast_exp2(fmaf(s[4 * k + 3], sl2, cb));
            lca += p0 + p1;
            lcb += p2 + p3;
            pw[2 * k] = pack_bf16(p0, p1);
            pw[2 * k + 1] = pack_bf16(p2, p3);
          }
        };
        ppass();
        if (__any_sync(0xffffffffu, !(lca <= kLazySum) || !(lcb <= kLazySum))) {
          float xa = -INFINITY, xb = -INFINITY;
#pragma unroll
          for (int k = 0; k < K4U_CB; ++k)
            if ((mine >> k) & 1u) {
              xa = fmaxf(xa, fmaxf(s[4 * k], s[4 * k + 1]));
              xb = fmaxf(xb, fmaxf(s[4 * k + 2], s[4 * k + 3]));
            }
#pragma unroll
          for (int o = 1; o <= 2; o <<= 1) {
            xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, o));
            xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, o));
          }
          const float na = fmaxf(ma, xa * sl2), nb = fmaxf(mb, xb * sl2);
          const float alpha_a = na == -INFINITY ? 1.f : fast_exp2(ma - na);
          const float alpha_b = nb == -INFINITY ? 1.f : fast_exp2(mb - nb);
          la *= alpha_a;
          lb *= alpha_b;
          ma = na;
          mb = nb;
          // O holds this unit's earlier chunks: rescale the row once O(c-1) is complete
          if (j > 0 && wait_ok(kVEmpty + ((c - 1) & 1), ((c - 1) >> 1) & 1)) {
            tc_fence_after();
#pragma unroll 1
            for (int cc = 0; cc < 6; ++cc) {
              uint32_t o[16];
              tmem_ld_16x256b_x4(tO16 + 32 * cc, o);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e)
                o[e] = __float_as_uint(__uint_as_float(o[e]) * ((e & 2) ? alpha_b : alpha_a));
              tmem_st_16x256b_x4(tO16 + 32 * cc, o);
            }
            tmem_st_wait();
          }
          ppass();
        }
        la += lca;
        lb += lcb;
        // the P columns are free once O(c-1) has read them
        if ((c == 0 || wait_ok(kVEmpty + ((c - 1) & 1), ((c - 1) >> 1) & 1)) && !bad) {
          tc_fence_after();
          tmem_st_16x128b_x16(tP16, pw);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kPFull));
        }
      }
      // row sums of the two heads over the quad; the quad leader publishes them (and the lse)
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        la += __shfl_xor_sync(0xffffffffu, la, o);
        lb += __shfl_xor_sync(0xffffffffu, lb, o);
      }
      float* xl = xchg;
      float* xm = xchg + 128;
      if ((lane & 3) == 0) {
        xl[16 * rr + hA] = la;
        xl[16 * rr + hB] = lb;
        xm[16 * rr + hA] = ma;
        xm[16 * rr + hB] = mb;
      }
      kc += (uint32_t)nch;
      // the next unit's Q goes in now: its first S overlaps this epilogue
      const int64_t un = u + gridDim.x;
      // Q is free once the unit's last S is done, which this warp waited for in the chunk loop
      if (un < n_units && !bad) {
        tc_fence_after();
        write_q(un);
      }
      // ---- epilogue: O / l, times sigmoid(gate), bf16 (thread = pair m, 96 columns) ----
      const uint4* gs = reinterpret_cast<const uint4*>(a.gate + hb * K4U_D + 96 * hf);
      float gh = 0.f;
      if (row_ok && !a.gate_per_dim) gh = __bfloat162float(a.gate[hb]);
      if (sync_stop()) break;
      const float lt = xl[m], mt = xm[m];
      if (hf == 0 && row_ok && a.lse) a.lse[hb] = (mt + __log2f(lt)) * 0.6931471805599453f;
      if (!wait_ok(kVEmpty + ((kc - 1) & 1), ((kc - 1) >> 1) & 1)) continue;  // caught at the next unit's barrier
      tc_fence_after();
      const float inv = lt > 0.f ? __frcp_rn(lt) : 0.f;
      const float kLog2e = 1.4426950408889634f;
      // O leaves tensor memory first, so the next unit's P.V can start while this one gates
      // and stores
      uint32_t o0[32], o1[32], o2[32];
      tmem_ld_32x32b_x32(tO, o0);
      tmem_ld_32x32b_x32(tO + 32, o1);
      tmem_ld_32x32b_x32(tO + 64, o2);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kOEmpty));
#pragma unroll
      for (int cc = 0; cc < 3; ++cc) {
        const uint32_t* o = cc == 0 ? o0 : cc == 1 ? o1 : o2;
        if (row_ok) {
          uint4 gv[4];
          if (a.gate_per_dim) {
#pragma unroll
            for (int e = 0; e < 4; ++e) gv[e] = __ldg(gs + cc * 4 + e);
          }
          uint32_t y[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float g0 = gh, g1 = gh;
            if (a.gate_per_dim) {
              const uint4 x = gv[e / 4];
              const uint32_t gw = (e & 3) == 0 ? x.x : (e & 3) == 1 ? x.y : (e & 3) == 2 ? x.z : x.w;
              const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw));
              g0 = f.x;
              g1 = f.y;
            }
            const float s0v = fast_rcp(1.f + fast_exp2(-g0 * kLog2e));
            const float s1v = fast_rcp(1.f + fast_exp2(-g1 * kLog2e));
            y[e] = pack_bf16(__uint_as_float(o[2 * e]) * inv * s0v, __uint_as_float(o[2 * e + 1]) * inv * s1v);
          }
          uint4* dst = reinterpret_cast<uint4*>(a.out + hb * K4U_D + 96 * hf + 32 * cc);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(y[4 * e], y[4 * e + 1], y[4 * e + 2], y[4 * e + 3]);
        }
      }
      if (lane == 0) mbar_arrive(bar(kTblEmpty + buf));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}


}  // namespace sgqa
