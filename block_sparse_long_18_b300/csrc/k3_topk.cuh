// k3_topk.cuh -- top-k block selection with a deterministic tie rule.
//
// ai4snews item "Step 5 Preview bets on depth over width", Interpretation para 2 (top-k
// over block representations); ai.info article, "Sparse GQA targets million-token
// context" (top-k of 4,096 tokens = 512 blocks of 8); phantomic12 entry (topk 512).
// Readings: the query's own block b_t is always kept and never scored; the other k-1
// slots go to the strictly earlier blocks in order (score descending, block index
// descending); -0 and +0 compare equal; the kept set is written in ascending order.
//
// One CTA of NT threads per (group, query row).  Scores are mapped to order-preserving
// unsigned keys.  Thread `tid` holds, for j = 0..PER/4-1, the four consecutive candidates
// 4*(j*NT + tid) .. +3, so every load is one coalesced float4 per thread and each group j
// covers 4*NT consecutive indices.  A radix select over 11/11/10-bit digits (shared-memory
// histograms, block-wide suffix search; the first pass needs no prefix test) finds the key
// of the (k-1)-th best candidate and how many candidates equal to it are kept, stopping as
// soon as a digit bucket is kept whole.  Equal keys are taken from the largest index down:
// they are ranked in index order and the first `skip` of them are passed over.  The
// compaction writes the kept indices in ascending order: per group j each warp scans its
// lanes' counts, one block-wide scan over the (j, warp) totals places the warps.  Rows up to
// NT*PER candidates keep their keys in registers.  Longer rows (contexts past 128K tokens at
// B = 8) take two levels: K3_SEGMENT CTAs each select the k-1 best of one NT*PER slice as
// (key, index) pairs, and a K3_MERGE CTA selects the k-1 best of the concatenated lists.  The
// result is exact: a candidate with fewer than k-1 candidates ahead of it in the whole row
// has fewer than k-1 ahead of it in its own slice, and the concatenation keeps index order,
// so the tie rule carries over.  A STREAM instance (tiles of NT*PER re-read for every pass)
// serves rows whose merge lists would not fit in registers either.
#pragma once
#include <type_traits>

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
  // two-level selection of long rows (more candidates than one CTA holds in registers):
  uint32_t* pair_key;   // [G * rows, nseg * (k-1)] keys of each segment's local selection
  int32_t* pair_idx;    // [G * rows, nseg * (k-1)] their candidate indices (ascending per segment)
  int32_t* pair_cnt;    // [G * rows, nseg] entries each segment kept
  int32_t nseg;         // segments per row
  int32_t prefetch_ctas;  // a CTA warms L2 for the scores of CTA blockIdx.x + prefetch_ctas (0: off)
  // bound-filtered selection (K3_THRESHOLD, K3_SELECT; row r = g * rows + i):
  const uint32_t* keys_in;  // K3_THRESHOLD: group-maximum keys [G * rows, keys_ld], ceil(b_t / keys_gs) per row
  int32_t keys_gs;          // K3_THRESHOLD: candidates per group (8 or 16)
  int64_t keys_ld;
  uint32_t* thr_out;        // K3_THRESHOLD: bound per row (0: none)
  const uint32_t* smask;    // K3_SELECT: survivor bits [G * rows, ld32], one per candidate below b_t
  int64_t ld32;
  const uint32_t* skeys;    // K3_SELECT: the survivors' keys at their candidate index [G * rows, ld]
  int32_t cap;              // K3_SELECT: survivors a row may have (K3_SEL_CAP)
  int32_t n_mtiles;         // K3_SELECT: 128-row tiles per group of the launch
  int32_t* row_flag;        // K3_SELECT: set for a row whose survivors passed cap
  int32_t* tile_flag;       //   and for its (group, 128-row tile)
  const int32_t* only_flagged;  // K3_DIRECT / _SEGMENT / _MERGE: serve only rows whose flag is set
  int64_t pos[256];     // decode: absolute position of each row's query
};

// What a k3_topk launch reads and writes.
enum K3Mode : int {
  K3_DIRECT = 0,     // candidates = the row's scores; writes the final selection
  K3_SEGMENT = 1,    // candidates = one segment of the row's scores; writes (key, index) pairs
  K3_MERGE = 2,      // candidates = the row's segment pairs; writes the final selection
  K3_THRESHOLD = 3,  // candidates = the row's group maxima; writes the (k-1)-th largest (a bound)
  K3_SELECT = 4      // candidates = the row's survivors of that bound (mask bits and keys in
                     // place); writes the final selection
};
constexpr int K3_SEL_CAP = 4096;  // survivors a K3_SELECT row may hold (128 threads x 32)
constexpr int K3_SEL_MAX_WORDS = 131072 / 32;  // mask words of the longest K3_SELECT row


// Inclusive warp scan.
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
  const uint32_t lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= (uint32_t)o) v += t;
  }
  return v;
}

template <int NT>
__device__ __forceinline__ uint32_t k3_block_excl_scan(uint32_t v, uint32_t* warp_tot, uint32_t& total) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t incl = warp_incl_scan(v);
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t t = lane < NW ? warp_tot[lane] : 0u;
    t = warp_incl_scan(t);
    if (lane < NW) warp_tot[lane] = t;
  }
  __syncthreads();
  const uint32_t before = warp > 0 ? warp_tot[warp - 1] : 0u;
  total = warp_tot[NW - 1];
  __syncthreads();
  return before + incl - v;
}

template <int NT, int PER, bool STREAM, int MODE = K3_DIRECT>
__global__ void __launch_bounds__(NT, STREAM ? 1 : 1024 / NT) k3_topk(const __grid_constant__ K3Args a) {
  constexpr int NBINS = 2048;
  constexpr int BPT = NBINS / NT;  // bins per thread
  constexpr int NJ = PER / 4;      // groups of 4 consecutive keys per thread
  constexpr int NW = NT / 32;
  constexpr int TILE = NT * PER;
  __shared__ uint32_t hist2[2][NBINS];  // ping-pong: one is counted while the other is cleared
  __shared__ uint32_t warp_tot[NW];
  __shared__ uint32_t wsum[2][NW];
  __shared__ uint32_t jw_cnt[NJ * NW];  // counts per (group j, warp), then their exclusive scan
  __shared__ uint32_t sh_digit, sh_above, sh_eq;
  constexpr bool BITMAP = !STREAM && MODE != K3_THRESHOLD;
  __shared__ uint32_t bitmap[BITMAP ? NT * PER / 32 : 1];  // kept slots
  __shared__ uint32_t tiemap[BITMAP ? NT * PER / 32 : 1];  // slots equal to the threshold key
  __shared__ int32_t sel_list[MODE == K3_SELECT ? NT * PER : 1];  // K3_SELECT: survivor index of each slot

  constexpr int SEGLEN = NT * PER;  // candidates per segment (K3_SEGMENT)
  const int64_t r = MODE == K3_SEGMENT ? blockIdx.x / a.nseg : blockIdx.x;  // (group, row) of the launch
  const int seg = MODE == K3_SEGMENT ? (int)(blockIdx.x % a.nseg) : 0;
  const int64_t g = r / a.rows;
  const int64_t i = r % a.rows;
  const int64_t pos = a.use_pos ? a.pos[i] : a.pos0 + i;
  const int64_t bt = pos / a.B;
  const int need = a.k - 1;
  const int64_t pstride = (int64_t)a.nseg * need;  // pair slots per row
  int32_t* out = a.sel_idx + ((g * a.T_out) + a.out_row0 + i) * a.k;
  const float* row = a.scores + (g * a.rows + i) * a.ld;
  const int tid = threadIdx.x;
  const uint32_t lane = tid & 31, warp = tid >> 5;
  if (a.only_flagged && a.only_flagged[r] == 0) return;
  // Warm L2 for the scores of the CTA about two waves later (launched when a CTA of this
  // wave retires), one 128-byte line per thread, so that its row load hits L2.
  if ((MODE == K3_DIRECT || MODE == K3_SEGMENT) && !STREAM && a.prefetch_ctas > 0) {
    const int64_t cb = (int64_t)blockIdx.x + a.prefetch_ctas;
    const int64_t nseg2 = MODE == K3_SEGMENT ? a.nseg : 1;
    if (cb < (int64_t)a.G * a.rows * nseg2) {
      const int64_t r2 = cb / nseg2, seg2 = cb % nseg2;
      const int64_t i2 = r2 % a.rows;
      const int64_t bt2 = (a.use_pos ? a.pos[i2] : a.pos0 + i2) / a.B;
      const int64_t b2 = MODE == K3_SEGMENT ? seg2 * (NT * PER) : 0;
      int64_t n2 = bt2 - b2;
      n2 = n2 < (int64_t)NT * PER ? n2 : (int64_t)NT * PER;
      if ((int64_t)tid * 32 < n2) {
        const float* p2 = a.scores + ((r2 / a.rows) * a.rows + i2) * a.ld + b2 + (int64_t)tid * 32;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p2));
      }
    }
  }
  // n: candidate slots of this CTA; base: candidate index of slot 0 (K3_SEGMENT)
  int64_t n = bt, base = 0;
  if (MODE == K3_SEGMENT) {
    base = (int64_t)seg * SEGLEN;
    n = bt - base < SEGLEN ? bt - base : SEGLEN;
    if (n < 0) n = 0;
  } else if (MODE == K3_MERGE) {
    n = pstride;
  } else if (MODE == K3_THRESHOLD) {
    n = (bt + a.keys_gs - 1) / a.keys_gs;  // groups of keys_gs candidates below the own block
    if (n <= need) {   // fewer group maxima than blocks to keep: no bound
      if (tid == 0) a.thr_out[r] = 0u;
      return;
    }
  }

  if (need == 0) {  // k = 1: the own block alone (segmented launches are never made for k = 1)
    if (MODE != K3_SEGMENT && tid == 0) {
      out[0] = (int32_t)bt;
      a.sel_cnt[g * a.T_out + a.out_row0 + i] = 1;
    }
    return;
  }
  if (MODE == K3_SEGMENT) {
    uint32_t* pk = a.pair_key + r * pstride + (int64_t)seg * need;
    int32_t* pi = a.pair_idx + r * pstride + (int64_t)seg * need;
    if (n <= need) {  // the whole segment is kept; empty slots carry key 0 (below any score)
      for (int64_t j = tid; j < need; j += NT) {
        pk[j] = j < n ? score_key(__ldg(row + base + j)) : 0u;
        pi[j] = j < n ? (int32_t)(base + j) : -1;
      }
      if (tid == 0) a.pair_cnt[r * a.nseg + seg] = (int32_t)n;
      return;
    }
  } else if (MODE != K3_THRESHOLD && bt <= need) {  // every causal block is kept
    for (int64_t j = tid; j < a.k; j += NT) out[j] = j < bt ? (int32_t)j : (j == bt ? (int32_t)bt : -1);
    if (tid == 0) a.sel_cnt[g * a.T_out + a.out_row0 + i] = (int32_t)(bt + 1);
    return;
  }

  const int n_tiles = STREAM ? (int)((n + TILE - 1) / TILE) : 1;
  // candidate index of key e of group j in tile `tile`
  auto kidx = [&](int tile, int j, int e) -> int32_t { return tile * TILE + 4 * (j * NT + tid) + e; };
  uint32_t key[PER];
  const uint32_t* mkeys = MODE == K3_THRESHOLD ? a.keys_in + r * a.keys_ld : a.pair_key + r * pstride;
  if (MODE == K3_SELECT) {
    // The survivors' candidate indices, in index order, from the mask words: thread tid
    // takes words [tid WPT, tid WPT + WPT), all loaded before the first is used (their
    // latencies overlap), and one block scan places its survivors.
    constexpr int WPT = (K3_SEL_MAX_WORDS + NT - 1) / NT;
    const uint32_t* mrow = a.smask + r * a.ld32;
    const int64_t n_words = (bt + 31) / 32;  // <= K3_SEL_MAX_WORDS: rows of at most 131,072 candidates
    uint32_t words[MODE == K3_SELECT ? WPT : 1];
#pragma unroll
    for (int w = 0; w < WPT; ++w) {
      const int64_t wi = (int64_t)tid * WPT + w;
      words[MODE == K3_SELECT ? w : 0] = wi < n_words ? __ldg(mrow + wi) : 0u;
    }
    uint32_t c = 0;
#pragma unroll
    for (int w = 0; w < WPT; ++w) c += (uint32_t)__popc(words[MODE == K3_SELECT ? w : 0]);
    uint32_t total;
    uint32_t o = k3_block_excl_scan<NT>(c, warp_tot, total);
    if (total > (uint32_t)a.cap) {  // more survivors than one CTA holds: redone from the scores
      if (tid == 0) {
        a.row_flag[r] = 1;
        a.tile_flag[g * a.n_mtiles + i / 128] = 1;
      }
      return;
    }
#pragma unroll
    for (int w = 0; w < WPT; ++w) {
      const int64_t wi = (int64_t)tid * WPT + w;
      uint32_t bits = words[MODE == K3_SELECT ? w : 0];
      while (bits != 0u) {
        const uint32_t b = (uint32_t)__ffs(bits) - 1u;
        bits &= bits - 1u;
        sel_list[o++] = (int32_t)(wi * 32 + b);
      }
    }
    __syncthreads();
    n = total;
  }
  const uint32_t* srow = a.skeys + r * a.ld;  // K3_SELECT: keys at candidate indices
  auto load_tile = [&](int tile) {
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int32_t b = kidx(tile, j, 0);
      if (MODE == K3_MERGE || MODE == K3_THRESHOLD) {
#pragma unroll
        for (int e = 0; e < 4; ++e) key[4 * j + e] = (b + e < n) ? __ldg(mkeys + b + e) : 0u;
      } else if (MODE == K3_SELECT) {
#pragma unroll
        for (int e = 0; e < 4; ++e) key[4 * j + e] = b + e < n ? __ldg(srow + sel_list[b + e]) : 0u;
      } else if (b + 3 < n && ((base + b) & 3) == 0) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(row + base + b));
        key[4 * j] = score_key(f.x);
        key[4 * j + 1] = score_key(f.y);
        key[4 * j + 2] = score_key(f.z);
        key[4 * j + 3] = score_key(f.w);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) key[4 * j + e] = (b + e < n) ? score_key(__ldg(row + base + b + e)) : 0u;
      }
    }
  };
  if (tid == 0) {
    sh_digit = 0;
    sh_above = 0;
    sh_eq = 0;
  }
  if (MODE == K3_MERGE) {
    // rows whose candidates all fit in k-1 (short rows of a long launch): keep every real entry
    int64_t real = 0;
    for (int s2 = 0; s2 < a.nseg; ++s2) real += a.pair_cnt[r * a.nseg + s2];
    if (real <= need) {
      if (tid == 0) {
        int o = 0;
        for (int64_t j = 0; j < pstride; ++j)
          if (mkeys[j] != 0u) out[o++] = a.pair_idx[r * pstride + j];
        out[o] = (int32_t)bt;
        for (int j = o + 1; j < a.k; ++j) out[j] = -1;
        a.sel_cnt[g * a.T_out + a.out_row0 + i] = o + 1;
      }
      return;
    }
  }
  if (!STREAM) load_tile(0);

  // Slots past the last candidate hold key 0.  Every finite score maps to a key of at
  // least 0x007FFFFF (the key of -inf), so key 0 lies below every real candidate; the first
  // pass does not count it, and since there are more candidates than keys to keep, the
  // search never reaches it and no later pass needs an index test.
  for (int b = tid; b < NBINS; b += NT) {
    hist2[0][b] = 0;
    hist2[1][b] = 0;
  }
  if (BITMAP) {
    for (int w = tid; w < NT * PER / 32; w += NT) {
      bitmap[w] = 0;
      tiemap[w] = 0;
    }
  }
  __syncthreads();
  uint32_t prefix = 0, pmask = 0;
  uint32_t need_rem = (uint32_t)need, eq_count = 0;
#pragma unroll
  for (int p = 0; p < 3; ++p) {
    const int sh = p == 0 ? 21 : (p == 1 ? 10 : 0);
    const uint32_t wm = p == 2 ? 0x3FFu : 0x7FFu;
    uint32_t* hist = hist2[p & 1];
    for (int tile = 0; tile < n_tiles; ++tile) {
      if (STREAM) load_tile(tile);
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const uint32_t kk = key[q];
        // pass 0 skips the empty slots (key 0): they would all hit one bin
        if (p == 0 ? kk != 0u : (kk & pmask) == prefix) atomicAdd(&hist[(kk >> sh) & wm], 1u);
      }
    }
    __syncthreads();  // (1) histogram complete
    // digit holding the need_rem-th largest matching key: thread tid owns bins
    // [tid*BPT, tid*BPT + BPT); warp sums go to smem and every thread adds up the warps
    // above its own, so no second scan round is needed.
    uint32_t h[BPT];
    uint32_t loc = 0;
#pragma unroll
    for (int b = 0; b < BPT; ++b) {
      h[b] = hist[tid * BPT + b];
      loc += h[b];
    }
    // the other buffer is free: clear it for the next pass
    if (p < 2) {
#pragma unroll
      for (int b = 0; b < BPT; ++b) hist2[(p + 1) & 1][tid * BPT + b] = 0;
    }
    const uint32_t incl = warp_incl_scan(loc);
    const uint32_t wtot = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 31) wsum[p & 1][warp] = wtot;
    __syncthreads();  // (2) warp sums visible
    uint32_t above_warp = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w)
      if (w > (int)warp) above_warp += wsum[p & 1][w];
    uint32_t cum = above_warp + (wtot - incl);  // keys in bins above this thread's bins
#pragma unroll
    for (int b = BPT - 1; b >= 0; --b) {
      if (cum < need_rem && cum + h[b] >= need_rem) {
        sh_digit = (uint32_t)(tid * BPT + b);
        sh_above = cum;
        sh_eq = h[b];
      }
      cum += h[b];
    }
    __syncthreads();  // (3) digit visible
    const uint32_t d = sh_digit;
    need_rem -= sh_above;
    eq_count = sh_eq;
    prefix |= d << sh;
    pmask |= wm << sh;
    if (need_rem == eq_count) break;  // the whole bucket is kept: no tie to break
  }

  if (MODE == K3_THRESHOLD) {
    // The (k-1)-th largest maximum, or (the loop stopped at a bucket kept whole) the
    // bucket's lower end, which is at most that maximum: either is a bound.
    if (tid == 0) a.thr_out[r] = prefix;
    return;
  }

  // ---- compaction in ascending index order ----
  // A key is kept if its masked value exceeds the prefix, or equals it and its rank among
  // the equal keys (in index order) is at least `skip`.  Without ties to break (skip = 0,
  // the usual case) a key is kept iff its masked value is at least the prefix.
  const uint32_t skip = eq_count - need_rem;
  // Register-resident rows: the kept slots are marked in a bitmap and read out in
  // ascending order (one word per thread, one block scan of the counts).  With ties to
  // break, the keys equal to the threshold go to a second bitmap whose first `skip` set
  // bits (the smallest indices) are dropped before the two are merged.
  auto compact_bitmap = [&]() {
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      const uint32_t kh = key[q] & pmask;
      if (kh >= prefix) {
        const uint32_t slot = (uint32_t)kidx(0, q >> 2, q & 3);
        atomicOr(skip != 0u && kh == prefix ? &tiemap[slot >> 5] : &bitmap[slot >> 5], 1u << (slot & 31));
      }
    }
    __syncthreads();
    constexpr int NWORDS = NT * PER / 32;  // bitmap words; thread tid reads word tid
    uint32_t w = tid < NWORDS ? bitmap[tid] : 0u;
    if (skip != 0u) {  // block-uniform
      uint32_t wt = tid < NWORDS ? tiemap[tid] : 0u, ttot;
      uint32_t rank = k3_block_excl_scan<NT>((uint32_t)__popc(wt), warp_tot, ttot);  // ties before this word
      while (wt != 0u) {
        const uint32_t bit = wt & (0u - wt);
        wt ^= bit;
        if (rank >= skip) w |= bit;
        ++rank;
      }
    }
    uint32_t total;
    uint32_t o = k3_block_excl_scan<NT>((uint32_t)__popc(w), warp_tot, total);
    while (w != 0u) {
      const int32_t slot = (int32_t)(tid * 32 + (uint32_t)__ffs(w) - 1u);
      w &= w - 1u;
      if (o < (uint32_t)need) {  // exactly need bits are set
        if (MODE == K3_SEGMENT) {
          a.pair_key[r * pstride + (int64_t)seg * need + o] = score_key(__ldg(row + base + slot));
          a.pair_idx[r * pstride + (int64_t)seg * need + o] = (int32_t)(base + slot);
        } else if (MODE == K3_MERGE) {
          out[o] = __ldg(a.pair_idx + r * pstride + slot);
        } else if (MODE == K3_SELECT) {
          out[o] = sel_list[slot];
        } else {
          out[o] = slot;
        }
      }
      ++o;
    }
  };
  auto compact = [&](auto ties_tag) {
    constexpr bool TIES = decltype(ties_tag)::value;
    uint32_t out_base = 0, tie_base = 0;
    for (int tile = 0; tile < n_tiles; ++tile) {
      if (STREAM) load_tile(tile);
      // per (j, lane): counts of its 4 keys (TIES: packed greater << 16 | equal), scanned
      // per warp
      uint32_t wex[NJ];
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        uint32_t c = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t kh = key[4 * j + e] & pmask;
          if (TIES)
            c += kh > prefix ? (1u << 16) : (kh == prefix ? 1u : 0u);
          else
            c += kh >= prefix ? 1u : 0u;
        }
        const uint32_t inc = warp_incl_scan(c);
        wex[j] = inc - c;
        if (lane == 31) jw_cnt[j * NW + warp] = inc;
      }
      __syncthreads();
      // exclusive scan over the NJ*NW (group, warp) totals in index order (j major)
      if (warp == 0) {
        constexpr int PERL = (NJ * NW + 31) / 32;
        uint32_t v[PERL];
        uint32_t sum = 0;
#pragma unroll
        for (int q = 0; q < PERL; ++q) {
          const int idx = lane * PERL + q;
          v[q] = idx < NJ * NW ? jw_cnt[idx] : 0u;
          sum += v[q];
        }
        const uint32_t inc = warp_incl_scan(sum);
        uint32_t run = inc - sum;
#pragma unroll
        for (int q = 0; q < PERL; ++q) {
          const int idx = lane * PERL + q;
          if (idx < NJ * NW) jw_cnt[idx] = run;
          run += v[q];
        }
        if (lane == 31) warp_tot[0] = inc;  // tile total
      }
      __syncthreads();
      const uint32_t tile_tot = warp_tot[0];
      const uint32_t kept_prev = tie_base > skip ? tie_base - skip : 0u;  // ties kept by earlier tiles
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const uint32_t ex = jw_cnt[j * NW + warp] + wex[j];  // counts before this lane's group j
        uint32_t ties_before = 0, o;
        if (TIES) {
          ties_before = tie_base + (ex & 0xFFFFu);
          o = out_base + (ex >> 16) + (ties_before > skip ? ties_before - skip : 0u) - kept_prev;
        } else {
          o = out_base + ex;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int32_t slot = (int32_t)kidx(tile, j, e);
          const uint32_t kh = key[4 * j + e] & pmask;
          bool keep;
          if (TIES) {
            keep = kh > prefix;
            if (kh == prefix) {
              keep = ties_before >= skip;
              ++ties_before;
            }
          } else {
            keep = kh >= prefix;
          }
          if (keep) {
            if (MODE == K3_SEGMENT) {
              a.pair_key[r * pstride + (int64_t)seg * need + o] = key[4 * j + e];
              a.pair_idx[r * pstride + (int64_t)seg * need + o] = (int32_t)(base + slot);
            } else if (MODE == K3_MERGE) {
              out[o] = __ldg(a.pair_idx + r * pstride + slot);
            } else {
              out[o] = slot;
            }
            ++o;
          }
        }
      }
      if (TIES) {
        const uint32_t t_gt = tile_tot >> 16, t_eq = tile_tot & 0xFFFFu;
        out_base += t_gt + ((tie_base + t_eq > skip) ? (tie_base + t_eq - (tie_base > skip ? tie_base : skip)) : 0u);
        tie_base += t_eq;
      } else {
        out_base += tile_tot;
      }
      __syncthreads();  // jw_cnt / warp_tot are rewritten by the next tile
    }
  };
  // (the per-slice pass of the two-level top-k keeps one general path: registers are tight)
  if (!STREAM)
    compact_bitmap();
  else if (skip == 0 && MODE != K3_SEGMENT)
    compact(std::integral_constant<bool, false>{});
  else
    compact(std::integral_constant<bool, true>{});
  if (tid == 0) {
    if (MODE == K3_SEGMENT) {
      a.pair_cnt[r * a.nseg + seg] = need;
    } else {
      out[need] = (int32_t)bt;
      a.sel_cnt[g * a.T_out + a.out_row0 + i] = a.k;
    }
  }
}

}  // namespace sgqa
