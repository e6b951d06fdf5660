// k4tc_attention.cuh -- gated sparse attention over the selected blocks on the
// 5th-generation tensor cores (tcgen05.mma, accumulators in tensor memory).
//
// Same operation as k4_attention.cuh (ai.info article, "Why StepFun chose 92 transformer
// blocks": Gated GQA; ai4snews item, Interpretation para 2: sparse flash attention over
// the selected blocks):  for row i (position t), group g, head h of g,
//   o_h = softmax_j(scale * q_h . k_j) . v_j over the selected tokens j <= t,
//   out = o_h * sigmoid(gate),  lse_h = log sum_j exp(scale * q_h . k_j).
//
// The MMA's M must be 64 or more, so the operands are swapped: per chunk of 128 gathered
// keys (16 blocks of 8), the keys are M and the 16 heads of the group are N.
//   S^T [128 keys x 16 heads]  = K[128 x 192] . Q[16 x 192]^T      (A, B K-major)
//   O^T [192 x 16]            += V^T[192 x 128] . P[16 x 128]^T    (A MN-major, B K-major)
// O^T is accumulated as two M=128 products over d 0..127 and d 64..191 (rows 64..127 of
// the second one give d 128..191), so no M=64 shape is needed.
//
// Shared memory: every gathered block lands as three 1 KB swizzle atoms (8 tokens x 64
// of D, one per 64-wide chunk of D) -- one TMA copy each through a 3-D tensor map
// {64, 3, tokens} with box {64, 1, B}.  Region c of a chunk holds all 128 keys of D-chunk
// c, which is at once the K-major layout of K (A of the first product) and the MN-major
// layout of V^T (A of the second: 64 d per 128-byte row, 8 keys per atom, the two
// 64-wide halves 16 KB apart).
//
// Roles (one CTA per SM, persistent over (row, group) units, group-major):
//   warp 0     TMA producer: Q tile per unit (2 buffers), K and V chunks through separate
//              2-slot rings (K frees as soon as S is computed).
//   warp 1     allocates 128 TMEM columns; one thread issues S(c+1) before P.V(c).
//   warps 2-5  softmax: thread = key (TMEM lane) with its 16 head scores; masking per key;
//              row maxima refreshed lazily (only when some score exceeds the reference
//              by more than 2^8, agreed through a 4-warp barrier), O^T rescaled in TMEM
//              then; P written to shared memory in the swizzled K-major layout; epilogue
//              reads O^T (thread = d), normalises, gates and stores bf16.
// Every wait is bounded; on expiry the CTA raises an abort flag, drains and returns.
#pragma once
#include "ptx.cuh"

namespace sgqa {

constexpr uint32_t K4T_REGION = 128 * 128;     // 128 keys x 128 B (64 of D) = 16 KB
constexpr uint32_t K4T_KV = 3 * K4T_REGION;    // one tensor's chunk: 48 KB
constexpr uint32_t K4T_QB = 3 * 16 * 128;      // Q tile: 3 regions x 16 heads x 128 B
constexpr uint32_t K4T_PB = 2 * 16 * 128;      // P tile: 2 regions (64 keys) x 16 heads x 128 B
constexpr uint32_t K4T_K_OFF = 0;
constexpr uint32_t K4T_V_OFF = 2 * K4T_KV;
constexpr uint32_t K4T_Q_OFF = 4 * K4T_KV;
constexpr uint32_t K4T_P_OFF = K4T_Q_OFF + 2 * K4T_QB;
constexpr uint32_t K4T_BAR_OFF = K4T_P_OFF + 2 * K4T_PB;
constexpr uint32_t K4T_SMEM = K4T_BAR_OFF + 1024 + 1024;  // + barriers/scratch + alignment
constexpr int K4T_THREADS = 224;  // 7 warps
constexpr uint32_t K4T_TMEM_COLS = 128;
// TMEM columns: S buffers 0 and 16; O buffer ob: 32 + 32*ob (d 0..127), +16 (d 64..191)

struct K4TArgs {
  const __nv_bfloat16* gate;  // [rows, H, D] or [rows, H]
  __nv_bfloat16* out;         // [rows, H, D]
  float* lse;                 // [rows, H] or null
  const int32_t* sel_idx;     // [G, rows, kcap]
  const int32_t* sel_cnt;     // [G, rows]
  int64_t rows, pos0, ctx_cap;
  int32_t G, Hg, H, B, kcap;
  float scale_log2;
  int32_t dense, gate_per_dim;
  int32_t block_major;  // 1: one TMA copy per block lands [3 chunks][8 keys][64] (B = 8)
  int32_t g_first, g_count;  // groups handled by this launch (one launch per group keeps the
                             // CTAs of a launch on one group's K/V, which L2 holds)
  uint64_t wait_ns;
};

struct K4TUnit {
  int32_t g;
  int64_t i, t, bt, cnt, n_ch;
  const int32_t* sel;
};

__device__ __forceinline__ K4TUnit k4t_unit(const K4TArgs& a, int64_t u) {
  K4TUnit x;
  x.g = a.g_first + (int32_t)(u / a.rows);
  x.i = u % a.rows;
  x.t = a.pos0 + x.i;
  x.bt = x.t / a.B;
  x.sel = a.sel_idx + ((int64_t)x.g * a.rows + x.i) * a.kcap;
  int64_t cnt = a.dense ? x.bt + 1 : (int64_t)__ldg(a.sel_cnt + (int64_t)x.g * a.rows + x.i);
  const int64_t cap = a.dense ? x.bt + 1 : (int64_t)a.kcap;
  if (cnt < 1) cnt = 1;   // a bad count is reported by the softmax warps
  if (cnt > cap) cnt = cap;
  x.cnt = cnt;
  x.n_ch = (cnt * a.B + 127) / 128;
  return x;
}

// j-th selected block of a unit: the block, -1 past the count, -2 if out of range
__device__ __forceinline__ int64_t k4t_block(const K4TArgs& a, const K4TUnit& x, int64_t j) {
  if (j >= x.cnt) return -1;
  const int64_t b = a.dense ? j : (int64_t)__ldg(x.sel + j);
  return (b >= 0 && b <= x.bt) ? b : -2;
}

__global__ void __launch_bounds__(K4T_THREADS, 1)
    k4tc_sparse_attn(const __grid_constant__ K4TArgs a, const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t k4t_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(k4t_smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb0 = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + K4T_BAR_OFF);
  auto bar = [&](int idx) { return smem_u32(&bars[idx]); };
  // barrier indices
  enum { kKFull = 0, kKEmpty = 2, kVFull = 4, kVEmpty = 6, kQFull = 8, kQEmpty = 10, kSFull = 12, kSEmpty = 14,
         kPFull = 16, kPEmpty = 18, kOFull = 20, kOEmpty = 22, kPvDone = 24, kFinal = 25, kXBar = 26 };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + K4T_BAR_OFF + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + K4T_BAR_OFF + 260);
  volatile uint32_t* need_flag = reinterpret_cast<volatile uint32_t*>(smem + K4T_BAR_OFF + 264);  // [2][4]
  float* red = reinterpret_cast<float*>(smem + K4T_BAR_OFF + 512);                               // [4][16]
  float* red2 = reinterpret_cast<float*>(smem + K4T_BAR_OFF + 768);                              // [4][16]

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const int64_t n_units = (int64_t)a.g_count * a.rows;
  const int bpc = 128 / a.B;  // blocks per chunk

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kKFull + s), 1);
      mbar_init(bar(kKEmpty + s), 1);
      mbar_init(bar(kVFull + s), 1);
      mbar_init(bar(kVEmpty + s), 1);
      mbar_init(bar(kQFull + s), 1);
      mbar_init(bar(kQEmpty + s), 1);
      mbar_init(bar(kSFull + s), 1);
      mbar_init(bar(kSEmpty + s), 4);
      mbar_init(bar(kPFull + s), 4);
      mbar_init(bar(kPEmpty + s), 1);
      mbar_init(bar(kOFull + s), 1);
      mbar_init(bar(kOEmpty + s), 4);
    }
    mbar_init(bar(kPvDone), 1);
    mbar_init(bar(kFinal), 1);
    mbar_init(bar(kXBar), 4);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), K4T_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 || warp == 6) {
    // ---------------- TMA producers: warp 0 streams Q and K, warp 6 streams V ----------------
    // Separate streams let K run up to two chunks ahead of V: the next chunk's scores and
    // softmax overlap the flight of its V tile, which is then held only briefly.
    const bool is_k = warp == 0;
    uint32_t uc = 0, kc = 0;
    bool ok = true;
    for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
      const K4TUnit x = k4t_unit(a, u);
      if (is_k) {
        const uint32_t qb = uc & 1;
        if (lane == 0) {
          if (uc >= 2) ok = mbar_wait(bar(kQEmpty + qb), ((uc >> 1) - 1) & 1, a.wait_ns, abort_flag);
          if (ok) {
            mbar_arrive_expect_tx(bar(kQFull + qb), K4T_QB);
            for (int r = 0; r < 3; ++r)
              tma_load_3d(sb0 + K4T_Q_OFF + qb * K4T_QB + r * 2048, &tmQ, bar(kQFull + qb), 0, r,
                          (int32_t)(x.i * a.H + (int64_t)x.g * a.Hg));
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      for (int64_t c = 0; c < x.n_ch && ok; ++c, ++kc) {
        const uint32_t slot = kc & 1;
        int64_t blk = -1;
        if ((int)lane < bpc) {
          blk = k4t_block(a, x, c * bpc + lane);
          if (blk < 0) blk = x.bt;  // unused or bad slot: fetch the own block, masked later
        }
        const int32_t row = (int32_t)((int64_t)x.g * a.ctx_cap + blk * a.B);
        const int full = (is_k ? kKFull : kVFull) + slot, empty = (is_k ? kKEmpty : kVEmpty) + slot;
        const uint32_t base = sb0 + (is_k ? K4T_K_OFF : K4T_V_OFF) + slot * K4T_KV;
        if (lane == 0) {
          if (kc >= 2) ok = mbar_wait(bar(empty), ((kc >> 1) - 1) & 1, a.wait_ns, abort_flag);
          if (ok) mbar_arrive_expect_tx(bar(full), K4T_KV);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok && (int)lane < bpc) {
          if (a.block_major) {  // one copy: the block's 3 atoms, 3 KB apart per block
            tma_load_3d(base + lane * 3072, is_k ? &tmK : &tmV, bar(full), 0, row, 0);
          } else {
            for (int r = 0; r < 3; ++r)
              tma_load_3d(base + r * K4T_REGION + lane * a.B * 128, is_k ? &tmK : &tmV, bar(full), 0, r, row);
          }
        }
        __syncwarp();
      }
    }
    // drain: the latest copies into every buffer land before the CTA leaves
    if (lane == 0) {
      if (is_k)
        for (uint32_t b = 0; b < 2; ++b)
          if (uc > b) {
            const uint32_t last = ((uc - 1 - b) & ~1u) + b;
            mbar_wait(bar(kQFull + b), (last >> 1) & 1, kDrainLimitNs);
          }
      for (uint32_t b = 0; b < 2; ++b)
        if (kc > b) {
          const uint32_t last = ((kc - 1 - b) & ~1u) + b;
          mbar_wait(bar((is_k ? kKFull : kVFull) + b), (last >> 1) & 1, kDrainLimitNs);
        }
    }
  } else if (warp == 1) {
    // ------------------------------- MMA issuer -------------------------------
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16_f32(128, 16);
      const uint32_t idesc_pv = idesc_bf16_f32(128, 16) | (1u << 15);  // A (V^T) is MN-major
      uint32_t uc = 0, kc = 0;
      bool ok = true;
      auto issue_qk = [&](uint32_t c, uint32_t qb) -> bool {
        const uint32_t slot = c & 1, sbuf = c & 1;
        if (!mbar_wait(bar(kKFull + slot), (c >> 1) & 1, a.wait_ns, abort_flag)) return false;
        if (c >= 2 && !mbar_wait(bar(kSEmpty + sbuf), ((c >> 1) - 1) & 1, a.wait_ns, abort_flag)) return false;
        tc_fence_after();
        const uint32_t kbase = sb0 + K4T_K_OFF + slot * K4T_KV;
        const uint32_t qbase = sb0 + K4T_Q_OFF + qb * K4T_QB;
#pragma unroll
        for (int r = 0; r < 3; ++r) {
          const uint64_t ad = a.block_major ? smem_desc_k_sw128_sbo(kbase + r * 1024, 3072)
                                            : smem_desc_k_sw128(kbase + r * K4T_REGION);
          const uint64_t bd = smem_desc_k_sw128(qbase + r * 2048);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) tc_mma_f16(tmem + sbuf * 16, ad + 2 * ks, bd + 2 * ks, idesc_qk, (r | ks) != 0);
        }
        tc_commit(bar(kKEmpty + slot));
        tc_commit(bar(kSFull + sbuf));
        return true;
      };
      for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
        const K4TUnit x = k4t_unit(a, u);
        const uint32_t qb = uc & 1, ob = uc & 1;
        if (!mbar_wait(bar(kQFull + qb), (uc >> 1) & 1, a.wait_ns, abort_flag)) { ok = false; break; }
        if (uc >= 2 && !mbar_wait(bar(kOEmpty + ob), ((uc >> 1) - 1) & 1, a.wait_ns, abort_flag)) { ok = false; break; }
        const uint32_t c0 = kc;
        if (!issue_qk(c0, qb)) { ok = false; break; }
        const uint32_t o1 = tmem + 32 + ob * 32, o2 = o1 + 16;
        for (int64_t j = 0; j < x.n_ch; ++j) {
          if (j + 1 < x.n_ch && !issue_qk(c0 + (uint32_t)j + 1, qb)) { ok = false; break; }
          const uint32_t c = c0 + (uint32_t)j, slot = c & 1, pb = c & 1;
          if (!mbar_wait(bar(kVFull + slot), (c >> 1) & 1, a.wait_ns, abort_flag)) { ok = false; break; }
          if (!mbar_wait(bar(kPFull + pb), (c >> 1) & 1, a.wait_ns, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t vbase = sb0 + K4T_V_OFF + slot * K4T_KV;
          const uint32_t pbase = sb0 + K4T_P_OFF + pb * K4T_PB;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t a1 = a.block_major ? smem_desc_mn_sw128(vbase + ks * 6144, 1024, 3072)
                                              : smem_desc_mn_sw128(vbase + ks * 2048, K4T_REGION);  // d 0..127
            const uint64_t a2 = a.block_major ? smem_desc_mn_sw128(vbase + 1024 + ks * 6144, 1024, 3072)
                                              : smem_desc_mn_sw128(vbase + K4T_REGION + ks * 2048,
                                                                   K4T_REGION);  // d 64..191
            const uint64_t bd = smem_desc_k_sw128(pbase + (ks >> 2) * 2048) + 2 * (ks & 3);
            const uint32_t acc = (j > 0 || ks > 0) ? 1u : 0u;
            tc_mma_f16(o1, a1, bd, idesc_pv, acc);
            tc_mma_f16(o2, a2, bd, idesc_pv, acc);
          }
          tc_commit(bar(kVEmpty + slot));
          tc_commit(bar(kPEmpty + pb));
          tc_commit(bar(kPvDone));
        }
        if (!ok) break;
        tc_commit(bar(kQEmpty + qb));
        tc_commit(bar(kOFull + ob));
        kc += (uint32_t)x.n_ch;
      }
      tc_commit(bar(kFinal));
      mbar_wait(bar(kFinal), 0, kDrainLimitNs);
    }
  } else {
    // ------------------------------- softmax + epilogue -------------------------------
    // The four softmax warps meet on hardware barrier 1.  They never leave the loop on
    // their own: a failed wait only marks the warp `bad`; each warp posts (bad || abort)
    // before a barrier and all of them OR the same four posts after it, so every warp
    // takes the same exit at the same barrier.
    const uint32_t q = warp & 3;       // TMEM lane quarter of this warp
    const uint32_t sw = warp - 2;      // slot in the cross-warp scratch
    const uint32_t kq = q * 32 + lane; // this thread's key within a chunk (= its TMEM lane)
    const uint32_t lane_base = (q * 32) << 16;
    constexpr float kLazy = 8.f;
    volatile uint32_t* stop_post = need_flag + 8;  // [2][4]
    uint32_t uc = 0, kc = 0, xb = 0;
    bool bad = false, stop = false;
    auto sync128 = [&]() -> bool {  // returns true when every softmax warp must stop
      if (lane == 0) stop_post[(xb & 1) * 4 + sw] = (bad || *abort_flag) ? 1u : 0u;
      asm volatile("bar.sync 1, 128;" ::: "memory");
      const uint32_t* sp = const_cast<const uint32_t*>(stop_post) + (xb & 1) * 4;
      const bool r = (sp[0] | sp[1] | sp[2] | sp[3]) != 0;
      ++xb;
      return r;
    };
    auto lane0_wait = [&](int b, uint32_t parity) {
      bool r = true;
      if (lane == 0) r = mbar_wait(bar(b), parity, a.wait_ns, abort_flag);
      r = __shfl_sync(0xffffffffu, r, 0);
      __syncwarp();
      if (!r) bad = true;
    };
    for (int64_t u = blockIdx.x; u < n_units && !stop; u += gridDim.x, ++uc) {
      const K4TUnit x = k4t_unit(a, u);
      if (lane == 0 && sw == 0) {
        const int64_t raw = a.dense ? x.bt + 1 : (int64_t)__ldg(a.sel_cnt + (int64_t)x.g * a.rows + x.i);
        if (raw < 1 || raw > (a.dense ? x.bt + 1 : (int64_t)a.kcap)) report_error(kErrBounds);
      }
      float m[16], l[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
      }
      for (int64_t j = 0; j < x.n_ch && !stop; ++j) {
        const uint32_t c = kc + (uint32_t)j, sbuf = c & 1;
        // this thread's key: block index lookup first, its latency overlaps the wait
        const int64_t kk = j * 128 + kq;
        const int64_t b = k4t_block(a, x, kk >> 3);
        lane0_wait(kSFull + sbuf, (c >> 1) & 1);
        tc_fence_after();
        float s[16];
        tmem_ld_32x32b_x16(tmem + lane_base + sbuf * 16, s);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kSEmpty + sbuf));
        if (b == -2) report_error(kErrBounds);
        const bool valid = b >= 0 && b * 8 + (kk & 7) <= x.t;
        bool need = false;
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          s[h] = valid ? s[h] * a.scale_log2 : -INFINITY;
          need |= s[h] > m[h] + kLazy;
        }
        need = __any_sync(0xffffffffu, need);
        if (lane == 0) need_flag[(c & 1) * 4 + sw] = need ? 1u : 0u;
        if (sync128()) { stop = true; break; }
        const bool any_need = (need_flag[(c & 1) * 4 + 0] | need_flag[(c & 1) * 4 + 1] |
                               need_flag[(c & 1) * 4 + 2] | need_flag[(c & 1) * 4 + 3]) != 0;
        if (any_need) {
#pragma unroll
          for (int h = 0; h < 16; ++h) {
            float v = s[h];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) red[sw * 16 + h] = v;
          }
          if (sync128()) { stop = true; break; }
          float alpha[16];
#pragma unroll
          for (int h = 0; h < 16; ++h) {
            const float cm = fmaxf(fmaxf(red[h], red[16 + h]), fmaxf(red[32 + h], red[48 + h]));
            const float mn = fmaxf(m[h], cm);
            alpha[h] = mn == -INFINITY ? 1.f : fast_exp2(m[h] - mn);
            l[h] *= alpha[h];
            m[h] = mn;
          }
          if (j > 0) {
            // O^T holds the earlier chunks: rescale it once their P.V has completed
            lane0_wait(kPvDone, (c - 1) & 1);
            tc_fence_after();
            const uint32_t ob = uc & 1;
            const uint32_t o1 = tmem + lane_base + 32 + ob * 32, o2 = o1 + 16;
            float v1[16], v2[16];
            tmem_ld_32x32b_x16(o1, v1);
            tmem_ld_32x32b_x16(o2, v2);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < 16; ++h) {
              v1[h] *= alpha[h];
              v2[h] *= alpha[h];
            }
            tmem_st_32x32b_x16(o1, v1);
            tmem_st_32x32b_x16(o2, v2);
            tmem_st_wait();
            tc_fence_before();
          }
          if (sync128()) { stop = true; break; }  // red[] is reused next time
        }
        float p[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          p[h] = fast_exp2(s[h] - (m[h] == -INFINITY ? 0.f : m[h]));
          l[h] += p[h];
        }
        // P [16 heads][128 keys], K-major, 128-byte swizzle (two 64-key regions)
        const uint32_t pb = c & 1;
        if (c >= 2) lane0_wait(kPEmpty + pb, ((c >> 1) - 1) & 1);
        const uint32_t col = kq & 63, uu = col >> 3, e = col & 7;
        const uint32_t pbase = sb0 + K4T_P_OFF + pb * K4T_PB + (kq >> 6) * 2048 + e * 2;
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          const uint16_t bits = __bfloat16_as_ushort(__float2bfloat16_rn(p[h]));
          asm volatile("st.shared.b16 [%0], %1;" ::"r"(pbase + h * 128 + ((uu ^ (h & 7)) << 4)), "h"(bits)
                       : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kPFull + pb));
      }
      if (stop) break;
      // ---- epilogue: row sums, O^T -> out ----
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        float v = l[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red2[sw * 16 + h] = v;
      }
      if (sync128()) { stop = true; break; }
      float L[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) L[h] = (red2[h] + red2[16 + h]) + (red2[32 + h] + red2[48 + h]);
      const uint32_t ob = uc & 1;
      lane0_wait(kOFull + ob, (uc >> 1) & 1);
      tc_fence_after();
      const uint32_t o1 = tmem + lane_base + 32 + ob * 32, o2 = o1 + 16;
      float v1[16], v2[16];
      tmem_ld_32x32b_x16(o1, v1);
      if (q >= 2) tmem_ld_32x32b_x16(o2, v2);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kOEmpty + ob));
      const int64_t head0 = x.i * a.H + (int64_t)x.g * a.Hg;
      const float kLog2e = 1.4426950408889634f;
      const uint32_t d1 = kq, d2 = 64 + kq;  // d2 valid for q >= 2 (128..191)
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        if (h < a.Hg) {
          const float inv = L[h] > 0.f ? __frcp_rn(L[h]) : 0.f;
          const int64_t hb = head0 + h;
          const float g1 = a.gate_per_dim ? __bfloat162float(a.gate[hb * K4_D + d1]) : __bfloat162float(a.gate[hb]);
          a.out[hb * K4_D + d1] = __float2bfloat16_rn(v1[h] * inv * __frcp_rn(1.f + fast_exp2(-g1 * kLog2e)));
          if (q >= 2) {
            const float g2 = a.gate_per_dim ? __bfloat162float(a.gate[hb * K4_D + d2]) : g1;
            a.out[hb * K4_D + d2] = __float2bfloat16_rn(v2[h] * inv * __frcp_rn(1.f + fast_exp2(-g2 * kLog2e)));
          }
        }
      }
      if (a.lse && sw == 0) {
#pragma unroll
        for (int h = 0; h < 16; ++h)
          if ((int)lane == h && h < a.Hg) a.lse[head0 + h] = (m[h] + __log2f(L[h])) * 0.6931471805599453f;
      }
      if (sync128()) { stop = true; break; }  // red2[] is reused by the next unit
      kc += (uint32_t)x.n_ch;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, K4T_TMEM_COLS);
}

}  // namespace sgqa
