// k4_attention.cuh -- gated sparse attention over the selected blocks.
//
// ai.info article "StepFun Details Step 5 Preview's 92-Block Agent Design", "Why StepFun
// chose 92 transformer blocks": the full-attention path is Gated GQA; ai4snews item,
// Interpretation para 2: a sparse flash-attention operator runs over the selected blocks;
// phantomic12 entry: 64 heads in 4 KV groups, head_dim 192.
//
//   for row i (position t), group g, head h in g:  J = { j in selected blocks : j <= t }
//   o = softmax_j(scale * q_h . k_j) . v_j ;  out = o * sigmoid(gate) ;  lse = log sum exp
//
// One warp owns one (row, group) unit: its 16 heads are the M = 16 of mma.sync m16n8k16
// (bf16 in, fp32 accumulate), so every gathered K/V byte serves all 16 heads.  The warp
// walks its selection 16 keys per stage (two blocks of 8, or one of 16), two stages per
// warp: one in flight while the other is consumed.  Every 8 keys of a tensor arrive by ONE
// TMA copy of box {64, 8, 3} through a {64, tokens, 3} tensor map whose strides are
// {384 B, 128 B}: it lands the keys as three 1 KB atoms [chunk][key][64] with the 128-byte
// swizzle, whose XOR term is the key alone, so the ldmatrix addresses of a stage are six
// per-lane bases plus immediates.  The selection is read 32 entries at a time into a
// register and handed out by shuffles.  S = Q K^T (2 n-tiles x 12 k-steps), online
// softmax in fp32 (exp2 domain, masked keys -inf, reference maxima refreshed lazily), P
// goes straight from the accumulator layout into the A operand of P V (24 n-tiles over
// D).  The epilogue normalises, applies sigmoid(gate) and writes bf16 through a swizzled
// smem tile with 16-byte stores.  Blocks smaller than 8 are gathered with cp.async into
// the same layout.
//
// Units are numbered group-major, so the CTAs in flight at any moment gather from one
// group's K/V (100 MB at 128K tokens), which the 126 MB L2 can hold.
//
// Split-K (decode): unit = (row, group, split); a split walks a range of stages and
// writes fp32 partials (m, l, O) that k4_combine merges with LSE weights.
#pragma once
#include "ptx.cuh"

namespace sgqa {

constexpr int K4_D = 192;
constexpr int K4_UNITS = K4_D / 8;            // 16-byte units per row: 24
constexpr uint32_t K4_TILE = 16 * K4_D * 2;   // 16 keys x 192 bf16 = 6144 B
constexpr uint32_t K4_STAGE = 2 * K4_TILE;    // K + V
// Blocks of fewer than 8 tokens: each key row arrives by one untiled bulk copy into a
// row of its own, padded to 400 bytes (100 words: 8 consecutive rows start 4 banks apart,
// so an 8x8 ldmatrix of 16-byte row pieces touches every bank once, without a swizzle).
constexpr uint32_t K4_ROW = 400;
__host__ __device__ constexpr uint32_t k4_tile_bytes(bool tma) { return tma ? K4_TILE : 16 * K4_ROW; }
__host__ __device__ constexpr uint32_t k4_stage_bytes(bool tma) { return 2 * k4_tile_bytes(tma); }
constexpr int K4_SEL_CACHE = 512;             // selection entries a warp keeps in shared memory

struct K4Args {
  const __nv_bfloat16* q;       // [rows, H, D]
  const __nv_bfloat16* gate;    // [rows, H, D] or [rows, H]
  const __nv_bfloat16* kc;      // [G, ctx_cap, D]  (cp.async loader)
  const __nv_bfloat16* vc;
  __nv_bfloat16* out;           // [rows, H, D]
  float* lse;                   // [rows, H] or null
  const int32_t* sel_idx;       // [G, rows, kcap]
  const int32_t* sel_cnt;       // [G, rows]
  float* part_o;                // split mode: [units, 16, D]
  float* part_ml;               // split mode: [units, 16, 2]
  int64_t rows;
  int64_t pos0;
  int64_t ctx_cap;
  int32_t G, Hg, H, B, kcap;
  float scale_log2;
  int32_t dense;
  int32_t gate_per_dim;
  int32_t nsplit;
  int32_t use_pos;
  // routed mode (nsplit = 1, NW = 8): CTA b serves the 8-row unit units[b] (unit = g * tiles
  // + tile of 8 rows), one warp per row, for b < *n_units_dev
  const int32_t* units;
  const int32_t* n_units_dev;
  const int32_t* perm;  // grouped units: perm[g * rows + s] is the row at slot s (null: s itself)
  uint64_t wait_ns;
  int64_t pos[256];
  int64_t kv_off[256];
};

// Byte offset, inside a 16-row tile staged for ldmatrix (Q, gate, output), of 16-byte unit
// u (0..23) of row n (0..15): row n's 384 bytes are 128-byte lines 3n .. 3n+2, swizzled.
__device__ __forceinline__ uint32_t k4_off(uint32_t n, uint32_t u) {
  const uint32_t r = n * 3 + (u >> 3);
  return r * 128 + (((u & 7) ^ (r & 7)) << 4);
}

// Byte offset, inside a stage's K (or V) tile of 16 keys, of 16-byte unit u (0..23) of key
// n (0..15).  Keys come in two groups of 8; a group holds its three 64-wide chunks of D as
// 1 KB atoms [chunk][key][64] with the 128-byte swizzle (unit XOR key), which is what one
// TMA copy of box {64, 8, 3} through a {64, tokens, 3} map with strides {384 B, 128 B}
// writes.  The swizzle term depends on the key alone, so a lane's ldmatrix addresses are
// a few per-lane bases plus immediates.
__device__ __forceinline__ uint32_t k4_kv_off(uint32_t n, uint32_t u) {
  return (n >> 3) * 3072 + (u >> 3) * 1024 + (n & 7) * 128 + (((u & 7) ^ (n & 7)) << 4);
}

template <int NW, bool TMA>
__global__ void __launch_bounds__(NW * 32, 1)
    k4_sparse_attn(const __grid_constant__ K4Args a, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV) {
  constexpr int NSTAGE = 2;  // a stage in flight while the other is consumed
  constexpr uint32_t TILE = k4_tile_bytes(TMA), STAGE = k4_stage_bytes(TMA);
  extern __shared__ uint8_t k4_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(k4_smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const uint32_t wbase = smem_u32(smem) + warp * (NSTAGE * STAGE);
  const uint32_t bar0 = smem_u32(smem) + NW * NSTAGE * STAGE + warp * NSTAGE * 8;

  const int64_t n_units = (int64_t)a.G * a.rows * a.nsplit;
  int64_t unit = (int64_t)blockIdx.x * NW + warp;
  if (a.units) {
    static_assert(NW == 8, "a routed unit is 8 rows, one per warp");
    if ((int64_t)blockIdx.x >= (int64_t)*a.n_units_dev) return;
    const int64_t ntiles = (a.rows + 7) / 8;
    const int64_t uid = __ldg(a.units + blockIdx.x);
    const int64_t slot = (uid % ntiles) * 8 + warp;
    if (slot >= a.rows) return;
    const int64_t row = a.perm ? (int64_t)__ldg(a.perm + (uid / ntiles) * a.rows + slot) : slot;
    unit = (uid / ntiles) * a.rows + row;
  }
  if (unit >= n_units) return;
  const int32_t split = (int32_t)(unit % a.nsplit);
  const int64_t gr = unit / a.nsplit;
  const int32_t g = (int32_t)(gr / a.rows);
  const int64_t i = gr % a.rows;
  const int64_t t = a.use_pos ? a.pos[i] : a.pos0 + i;
  const int64_t kvo = a.use_pos ? a.kv_off[i] : 0;
  const int32_t bt = (int32_t)(t / a.B);
  const int32_t* sel = a.sel_idx + (g * a.rows + i) * (int64_t)a.kcap;
  int32_t cnt = a.dense ? bt + 1 : a.sel_cnt[g * a.rows + i];
  if (cnt < 1 || cnt > (a.dense ? bt + 1 : a.kcap)) {
    report_error(kErrBounds);
    cnt = cnt < 1 ? 1 : (a.dense ? bt + 1 : a.kcap);
  }
  const int bps = 16 / a.B;  // blocks per stage (B <= 16); a block of 16 is one stage
  const int32_t n_st = (cnt + bps - 1) / bps;
  const int32_t per_split = (n_st + a.nsplit - 1) / a.nsplit;
  const int32_t s_begin = split * per_split;
  const int32_t s_end = s_begin + per_split < n_st ? s_begin + per_split : n_st;
  const int64_t row_base = (int64_t)g * a.ctx_cap + kvo;  // cache row of token 0 of this unit

  // Block j of the selection: -1 past the count, -2 for an index outside 0..bt.  Rows of
  // up to K4_SEL_CACHE entries are copied once into this warp's shared-memory table, so a
  // lookup is one broadcast shared load; longer rows read the global array.
  int32_t* selc = reinterpret_cast<int32_t*>(smem + NW * NSTAGE * STAGE + NW * NSTAGE * 8) + warp * K4_SEL_CACHE;
  const uint32_t selc_s = smem_u32(selc);
  const bool cached = !a.dense && cnt <= K4_SEL_CACHE;
  if (cached) {
#pragma unroll
    for (int m = 0; m < K4_SEL_CACHE / 32; ++m) {
      const int32_t j = m * 32 + (int32_t)lane;
      const int32_t v = j < cnt ? __ldg(sel + j) : -1;
      asm volatile("st.shared.b32 [%0], %1;" ::"r"(selc_s + 4u * j), "r"(v) : "memory");
    }
  }
  __syncwarp();
  auto lookup = [&](int32_t j) -> int32_t {  // every lane calls it with the same j
    if (j >= cnt) return -1;
    int32_t v;
    if (cached)
      asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(selc_s + 4u * j) : "memory");
    else
      v = a.dense ? j : __ldg(sel + j);
    return (v >= 0 && v <= bt) ? v : -2;
  };

  // ---- Q fragments: Q[i, g*Hg + h, :] staged swizzled in slot 0, then ldmatrix ----
  const uint32_t qs = wbase;
  {
    const uint4* src = reinterpret_cast<const uint4*>(a.q + (i * a.H + (int64_t)g * a.Hg) * K4_D);
    for (int w = lane; w < 16 * K4_UNITS; w += 32) {
      const uint32_t h = w / K4_UNITS, u = w % K4_UNITS;
      uint4 v = make_uint4(0, 0, 0, 0);
      if ((int)h < a.Hg) v = __ldg(src + w);
      asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(qs + k4_off(h, u)), "r"(v.x), "r"(v.y), "r"(v.z),
                   "r"(v.w)
                   : "memory");
    }
  }
  __syncwarp();
  uint32_t qa[12][4];
#pragma unroll
  for (int ks = 0; ks < 12; ++ks) {
    // matrices: (heads 0-7, unit 2ks), (heads 8-15, unit 2ks), (0-7, 2ks+1), (8-15, 2ks+1)
    const uint32_t m = lane >> 3;
    const uint32_t h = (m & 1) * 8 + (lane & 7);
    const uint32_t u = 2 * ks + (m >> 1);
    ldsm_x4(qs + k4_off(h, u), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
  }
  __syncwarp();

  if (lane == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  __syncwarp();

  // per-lane ldmatrix bases (see k4_kv_off): K as the B operand of S = Q K^T reads key
  // nt*8 + (lane&7), unit 2kp + (lane>>3); V (transposed) reads key (lane>>3 & 1)*8 +
  // (lane&7), unit 2dp + (lane>>4).
  const uint32_t kr = lane & 7;
  const uint32_t k_lo = kr * 128 + (((lane >> 3) ^ kr) << 4);  // units with (u & 7) < 4
  const uint32_t k_hi = k_lo ^ 64u;                             // units with (u & 7) >= 4
  uint32_t v_off[4];
#pragma unroll
  for (int jx = 0; jx < 4; ++jx)
    v_off[jx] = ((lane >> 3) & 1) * 3072 + kr * 128 + (((((lane >> 4) ^ kr)) ^ (2u * jx)) << 4);
  // the padded-row layout (blocks of fewer than 8 tokens): byte n * K4_ROW + 16 u
  const uint32_t k_pad = kr * K4_ROW + (lane >> 3) * 16;
  const uint32_t v_pad = ((lane >> 3) & 1) * 8 * K4_ROW + kr * K4_ROW + (lane >> 4) * 16;

  // ---- stage loader.  TMA: lane 0 fetches stage s from blocks (b0, b1) looked up one
  // iteration earlier, so no shuffle latency sits in front of the copies.  Blocks of fewer
  // than 8 tokens: lane l copies key l & 15 of K (l < 16) or V with one bulk copy.  Both
  // complete on the stage's mbarrier. ----
  auto issue = [&](int32_t s, int32_t b0, int32_t b1) {
    const uint32_t slot = (uint32_t)(s - s_begin) % NSTAGE;
    const uint32_t ks_addr = wbase + slot * STAGE;
    const uint32_t vs_addr = ks_addr + TILE;
    if (TMA) {
      // B = 8: two blocks of 8 keys; B = 16: the two halves of one block
      if (b0 < 0) b0 = bt;  // unused / invalid slot: fetch the own block, masked below
      if (b1 < 0) b1 = bt;
      if (lane == 0) {
        const uint32_t bar = bar0 + 8 * slot;
        mbar_arrive_expect_tx(bar, K4_STAGE);
        const int32_t r0 = (int32_t)(row_base + (int64_t)b0 * a.B);
        const int32_t r1 = bps == 2 ? (int32_t)(row_base + (int64_t)b1 * a.B) : r0 + 8;
        tma_load_3d(ks_addr, &tmK, bar, 0, r0, 0);
        tma_load_3d(ks_addr + 3072, &tmK, bar, 0, r1, 0);
        tma_load_3d(vs_addr, &tmV, bar, 0, r0, 0);
        tma_load_3d(vs_addr + 3072, &tmV, bar, 0, r1, 0);
      }
    } else {
      const int64_t row_lim = (int64_t)a.G * a.ctx_cap - 1;
      const uint32_t bar = bar0 + 8 * slot;
      if (lane == 0) mbar_arrive_expect_tx(bar, STAGE - 2 * 16 * (K4_ROW - K4_D * 2));
      __syncwarp();
      const uint32_t n = lane & 15;
      const int32_t j = s * bps + (int32_t)n / a.B;
      int64_t b = j < cnt ? (a.dense ? j : __ldg(sel + j)) : -1;
      if (b < 0 || b > bt) b = bt;  // unused / invalid slot: a valid row, masked below
      int64_t row = row_base + b * a.B + (n % a.B);
      if (row > row_lim) row = row_lim;
      bulk_load_g2s((lane < 16 ? ks_addr : vs_addr) + n * K4_ROW, (lane < 16 ? a.kc : a.vc) + row * K4_D, K4_D * 2,
                    bar);
    }
  };

  float o[24][4];
#pragma unroll
  for (int d = 0; d < 24; ++d) o[d][0] = o[d][1] = o[d][2] = o[d][3] = 0.f;
  // m0/m1: reference maxima (log2 units) of rows r = lane/4 and r + 8; they may lag the
  // true running maxima by up to kLazy so that O is rescaled only when a maximum grows.
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  constexpr float kLazy = 8.f;
  const uint32_t qd = lane & 3;  // column pair within an 8-wide tile
  bool ok = true;
  int32_t issued = s_begin;

  auto wait_stage = [&](int32_t s) -> bool {
    const uint32_t slot = (uint32_t)(s - s_begin) % NSTAGE;
    return mbar_wait(bar0 + 8 * slot, (uint32_t)((s - s_begin) / NSTAGE) & 1u, a.wait_ns);
  };

  // nb0/nb1: blocks of the stage issued last (masked by the next iteration); pb0/pb1:
  // blocks of the stage to issue next
  int32_t nb0 = 0, nb1 = 0, pb0 = 0, pb1 = 0;
  auto look_stage = [&](int32_t s) {
    if (TMA && s < s_end) {
      pb0 = lookup(s * bps);
      pb1 = bps == 2 ? lookup(s * bps + 1) : pb0;
    }
  };
  look_stage(s_begin);
  if (s_begin < s_end) {
    issue(s_begin, pb0, pb1);
    nb0 = pb0;
    nb1 = pb1;
    issued = s_begin + 1;
  }
  look_stage(s_begin + 1);

  for (int32_t s = s_begin; s < s_end; ++s) {
    // blocks of this stage and whether all are valid and strictly before the own block
    const int32_t cb0 = nb0, cb1 = nb1;
    // prefetch into the slot stage s-1 has released, then look up the stage after it
    if (s + 1 < s_end) {
      issue(s + 1, pb0, pb1);
      nb0 = pb0;
      nb1 = pb1;
      issued = s + 2;
      look_stage(s + 2);
    }
    bool fast = true;
    if (TMA) {
      fast = cb0 >= 0 && cb0 < bt && cb1 >= 0 && cb1 < bt;
    } else {
      for (int bi = 0; bi < bps; ++bi) {
        const int32_t j = s * bps + bi;
        const int32_t b = j < cnt ? (a.dense ? j : __ldg(sel + j)) : -1;
        fast = fast && b >= 0 && b < bt;
      }
    }
    if (!wait_stage(s)) { ok = false; break; }
    const uint32_t ks_addr = wbase + ((uint32_t)(s - s_begin) % NSTAGE) * STAGE;
    const uint32_t vs_addr = ks_addr + TILE;

    // ---- S = Q K^T: two n-tiles x 12 k-steps as four independent chains ----
    float sc[2][4];
    {
      float acc[2][2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h) acc[nt][h][0] = acc[nt][h][1] = acc[nt][h][2] = acc[nt][h][3] = 0.f;
      const uint32_t klo = ks_addr + k_lo, khi = ks_addr + k_hi;
#pragma unroll
      for (int kp = 0; kp < 12; kp += 2) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          uint32_t b0, b1, b2, b3;
          if (TMA)
            ldsm_x4(((kp & 2) ? khi : klo) + nt * 3072 + (kp >> 2) * 1024, b0, b1, b2, b3);
          else
            ldsm_x4(ks_addr + k_pad + nt * 8 * K4_ROW + kp * 32, b0, b1, b2, b3);
          mma_bf16_16816(acc[nt][0], qa[kp], b0, b1);
          mma_bf16_16816(acc[nt][1], qa[kp + 1], b2, b3);
        }
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[nt][e] = acc[nt][0][e] + acc[nt][1][e];
    }

    // ---- mask unused slots, invalid indices and tokens after t (scores stay unscaled) ----
    if (!fast) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int key = nt * 8 + 2 * qd + c;
          int32_t b;
          if (TMA) {
            b = (nt == 1 && bps == 2) ? cb1 : cb0;
          } else {
            const int32_t j = s * bps + key / a.B;
            const int32_t raw = j < cnt ? (a.dense ? j : __ldg(sel + j)) : -1;
            b = j >= cnt ? -1 : ((raw >= 0 && raw <= bt) ? raw : -2);
          }
          const bool valid = b >= 0 && (int64_t)b * a.B + (key % a.B) <= t;
          if (b == -2) report_error(kErrBounds);
          if (!valid) {
            sc[nt][c] = -INFINITY;
            sc[nt][2 + c] = -INFINITY;
          }
        }
      }
    }

    // ---- online softmax (log2 domain), rows r = lane/4 and r + 8 ----
    // A row's quad shares its reference maximum; the quad maximum is needed only when some
    // lane's own scores pass the reference by more than kLazy, which one vote detects.
    const float sl2 = a.scale_log2;
    float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1])) * sl2;
    float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3])) * sl2;
    if (__any_sync(0xffffffffu, mx0 > m0 + kLazy || mx1 > m1 + kLazy)) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float al0 = mn0 == -INFINITY ? 1.f : fast_exp2(m0 - mn0);
      const float al1 = mn1 == -INFINITY ? 1.f : fast_exp2(m1 - mn1);
      l0 *= al0;
      l1 *= al1;
#pragma unroll
      for (int d = 0; d < 24; ++d) {
        o[d][0] *= al0;
        o[d][1] *= al0;
        o[d][2] *= al1;
        o[d][3] *= al1;
      }
      m0 = mn0;
      m1 = mn1;
    }
    const float mu0 = m0 == -INFINITY ? 0.f : m0, mu1 = m1 == -INFINITY ? 0.f : m1;
    float p[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      p[nt][0] = fast_exp2(fmaf(sc[nt][0], sl2, -mu0));
      p[nt][1] = fast_exp2(fmaf(sc[nt][1], sl2, -mu0));
      p[nt][2] = fast_exp2(fmaf(sc[nt][2], sl2, -mu1));
      p[nt][3] = fast_exp2(fmaf(sc[nt][3], sl2, -mu1));
    }
    l0 += (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
    l1 += (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]);
    uint32_t pa[4];
    pa[0] = pack_bf16(p[0][0], p[0][1]);
    pa[1] = pack_bf16(p[0][2], p[0][3]);
    pa[2] = pack_bf16(p[1][0], p[1][1]);
    pa[3] = pack_bf16(p[1][2], p[1][3]);

    // ---- O += P V ----
#pragma unroll
    for (int dp = 0; dp < 12; ++dp) {
      uint32_t v0, v1, v2, v3;
      if (TMA)
        ldsm_x4_t(vs_addr + v_off[dp & 3] + (dp >> 2) * 1024, v0, v1, v2, v3);
      else
        ldsm_x4_t(vs_addr + v_pad + dp * 32, v0, v1, v2, v3);
      mma_bf16_16816(o[2 * dp], pa, v0, v1);
      mma_bf16_16816(o[2 * dp + 1], pa, v2, v3);
    }
    __syncwarp();  // every lane is done with this stage's slot
  }

  if (!ok) {
    // drain the copies still in flight into this warp's slots, then leave
    if (lane == 0) {
      for (int32_t s = issued - NSTAGE > s_begin ? issued - NSTAGE : s_begin; s < issued; ++s) {
        const uint32_t slot = (uint32_t)(s - s_begin) % NSTAGE;
        mbar_wait(bar0 + 8 * slot, (uint32_t)((s - s_begin) / NSTAGE) & 1u, kDrainLimitNs);
      }
    }
    __syncwarp();
    return;
  }
  __syncwarp();

  // full row sums across the quad
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const uint32_t r0 = lane >> 2, r1 = r0 + 8;

  if (a.nsplit > 1) {
    float* po = a.part_o + unit * (16 * K4_D);
    float* pml = a.part_ml + unit * 32;
#pragma unroll
    for (int d = 0; d < 24; ++d) {
      const int col = d * 8 + 2 * qd;
      *reinterpret_cast<float2*>(po + r0 * K4_D + col) = make_float2(o[d][0], o[d][1]);
      *reinterpret_cast<float2*>(po + r1 * K4_D + col) = make_float2(o[d][2], o[d][3]);
    }
    if (qd == 0) {
      pml[r0 * 2] = m0;
      pml[r0 * 2 + 1] = l0;
      pml[r1 * 2] = m1;
      pml[r1 * 2 + 1] = l1;
    }
    return;
  }

  // ---- epilogue: normalise, gate, bf16, coalesced store ----
  const float inv0 = l0 > 0.f ? __frcp_rn(l0) : 0.f;
  const float inv1 = l1 > 0.f ? __frcp_rn(l1) : 0.f;
  const uint32_t ts = wbase;  // slot 0 is free: every issued stage has been consumed
  const int64_t head0 = i * a.H + (int64_t)g * a.Hg;
  if (a.gate_per_dim) {
    const uint4* src = reinterpret_cast<const uint4*>(a.gate + head0 * K4_D);
    for (int w = lane; w < a.Hg * K4_UNITS; w += 32) {
      const uint4 v = __ldg(src + w);
      asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(ts + k4_off(w / K4_UNITS, w % K4_UNITS)),
                   "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                   : "memory");
    }
  }
  __syncwarp();
  const float kLog2e = 1.4426950408889634f;
  float gh0 = 0.f, gh1 = 0.f;
  if (!a.gate_per_dim) {
    if ((int)r0 < a.Hg) gh0 = __bfloat162float(a.gate[head0 + r0]);
    if ((int)r1 < a.Hg) gh1 = __bfloat162float(a.gate[head0 + r1]);
  }
#pragma unroll
  for (int d = 0; d < 24; ++d) {
    const uint32_t col = d * 8 + 2 * qd;
    const uint32_t a0 = ts + k4_off(r0, col >> 3) + (col & 7) * 2;
    const uint32_t a1 = ts + k4_off(r1, col >> 3) + (col & 7) * 2;
    float g00 = gh0, g01 = gh0, g10 = gh1, g11 = gh1;
    if (a.gate_per_dim) {
      uint32_t w0, w1;
      asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w0) : "r"(a0));
      asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w1) : "r"(a1));
      const float2 f0 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w0));
      const float2 f1 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w1));
      g00 = f0.x; g01 = f0.y; g10 = f1.x; g11 = f1.y;
    }
    const float s00 = __frcp_rn(1.f + fast_exp2(-g00 * kLog2e));
    const float s01 = __frcp_rn(1.f + fast_exp2(-g01 * kLog2e));
    const float s10 = __frcp_rn(1.f + fast_exp2(-g10 * kLog2e));
    const float s11 = __frcp_rn(1.f + fast_exp2(-g11 * kLog2e));
    const uint32_t w0 = pack_bf16(o[d][0] * inv0 * s00, o[d][1] * inv0 * s01);
    const uint32_t w1 = pack_bf16(o[d][2] * inv1 * s10, o[d][3] * inv1 * s11);
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(a0), "r"(w0) : "memory");
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(a1), "r"(w1) : "memory");
  }
  __syncwarp();
  {
    uint4* dst = reinterpret_cast<uint4*>(a.out + head0 * K4_D);
    for (int w = lane; w < a.Hg * K4_UNITS; w += 32) {
      uint4 v;
      asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                   : "r"(ts + k4_off(w / K4_UNITS, w % K4_UNITS)));
      dst[w] = v;
    }
  }
  if (a.lse && qd == 0) {
    const float kLn2 = 0.6931471805599453f;
    if ((int)r0 < a.Hg) a.lse[head0 + r0] = (m0 + __log2f(l0)) * kLn2;
    if ((int)r1 < a.Hg) a.lse[head0 + r1] = (m1 + __log2f(l1)) * kLn2;
  }
}

// Merge split-K partials.  One warp per (row, group, head, 32-wide slice of D): lane s
// reads split s's (m, l) to form the weights, then lane d sums its column over the splits
// with every split's load issued at once (the partials sit in L2; a warp that walked the
// splits one after another would wait on each load in turn).
struct K4CombineArgs {
  const float* part_o;     // [G*rows*nsplit, 16, D]
  const float* part_ml;    // [G*rows*nsplit, 16, 2]
  const __nv_bfloat16* gate;
  __nv_bfloat16* out;
  float* lse;
  int64_t rows;
  int32_t G, Hg, H, nsplit, gate_per_dim;  // nsplit <= 32 (one lane per split)
};
constexpr int K4C_SLICES = K4_D / 32;  // warps per (row, group, head)

__global__ void __launch_bounds__(128) k4_combine(const K4CombineArgs a) {
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t lane = lane_id();
  const int64_t total = (int64_t)a.G * a.rows * a.Hg * K4C_SLICES;
  if (wid >= total) return;
  const int sl = (int)(wid % K4C_SLICES);
  const int64_t gh = wid / K4C_SLICES;
  const int h = (int)(gh % a.Hg);
  const int64_t gr = gh / a.Hg;            // = g * rows + i
  const int g = (int)(gr / a.rows);
  const int64_t i = gr % a.rows;
  // lane s holds split s (nsplit <= 32): its (m, l), the maximum over splits with mass and
  // its weight exp2(m_s - M)
  float ms = -INFINITY, ls = 0.f;
  if ((int)lane < a.nsplit) {
    const float2 ml = __ldg(reinterpret_cast<const float2*>(a.part_ml + ((gr * a.nsplit + lane) * 16 + h) * 2));
    if (ml.y > 0.f) {
      ms = ml.x;
      ls = ml.y;
    }
  }
  float M = ms;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float ws = ls > 0.f ? fast_exp2(ms - M) : 0.f;
  float L = ws * ls;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  // column d = 32 sl + lane, summed over the splits (a split that got no keys wrote zero
  // partials and has weight 0)
  const int d = 32 * sl + (int)lane;
  const float* po = a.part_o + (gr * a.nsplit * 16 + h) * K4_D + d;
  float x[32];
#pragma unroll
  for (int s = 0; s < 32; ++s) x[s] = s < a.nsplit ? __ldg(po + (int64_t)s * 16 * K4_D) : 0.f;
  float acc = 0.f;
#pragma unroll
  for (int s = 0; s < 32; ++s) acc = fmaf(__shfl_sync(0xffffffffu, ws, s), x[s], acc);
  const float inv = L > 0.f ? __frcp_rn(L) : 0.f;
  const int64_t head = i * a.H + (int64_t)g * a.Hg + h;
  const float kLog2e = 1.4426950408889634f;
  const float gv = a.gate_per_dim ? __bfloat162float(a.gate[head * K4_D + d]) : __bfloat162float(a.gate[head]);
  const float sg = __frcp_rn(1.f + fast_exp2(-gv * kLog2e));
  a.out[head * K4_D + d] = __float2bfloat16_rn(acc * inv * sg);
  if (a.lse && sl == 0 && lane == 0) a.lse[head] = (M + __log2f(L)) * 0.6931471805599453f;
}

}  // namespace sgqa
