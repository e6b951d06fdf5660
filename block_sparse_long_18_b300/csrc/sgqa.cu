// sgqa.cu -- the C ABI of the Sparse GQA layer (include/sgqa.h): argument checks,
// workspace carving, TMA tensor maps and the launch sequence of the four stages
// (block index -> indexer -> top-k -> gated sparse attention) and of decode.
//
// Single translation unit: the kernels live in the .cuh files included below.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/sgqa.h"
#include "ptx.cuh"
#include "k1_block_index.cuh"
#include "k2_indexer.cuh"
#include "k2d_decode_index.cuh"
#include "k3_topk.cuh"
#include "k4_attention.cuh"
#include "k4u_attention.cuh"
#include "k4r_route.cuh"

using namespace sgqa;

namespace {

uint64_t g_wait_ns = 1000000000ull;

constexpr int64_t kIndexChunkRows = 8192;  // preferred query rows per indexer/top-k pass
constexpr int kMaxBatch = 256;
constexpr int kK3Threads = 512;
constexpr int kK3Per = 32;
constexpr int64_t kK3RegRow = (int64_t)kK3Threads * kK3Per;  // rows up to this many candidates stay in registers

#define SGQA_CUDA_OK(expr)                       \
  do {                                           \
    if ((expr) != cudaSuccess) return SGQA_ERR_CUDA; \
  } while (0)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Parameters after defaults are resolved.
struct Prm {
  int G, Hg, H, D, P, B, k, gate_per_dim, attn_kernel;
  float scale;
};

sgqa_status check_params(const sgqa_params* p, Prm& o) {
  if (!p) return SGQA_ERR_INVALID_ARGUMENT;
  if (p->num_kv_groups < 1 || p->heads_per_group < 1 || p->head_dim < 1 || p->proxy_dim < 1 || p->block_size < 1 ||
      p->top_k_blocks < 1)
    return SGQA_ERR_INVALID_ARGUMENT;
  if (p->heads_per_group > 16 || p->head_dim != 192) return SGQA_ERR_UNSUPPORTED_SHAPE;
  if (p->proxy_dim % 64 != 0 || p->proxy_dim > 256) return SGQA_ERR_UNSUPPORTED_SHAPE;
  const int B = p->block_size;
  if (B != 1 && B != 2 && B != 4 && B != 8 && B != 16) return SGQA_ERR_UNSUPPORTED_SHAPE;
  if (p->gate_per_dim != 0 && p->gate_per_dim != 1) return SGQA_ERR_INVALID_ARGUMENT;
  if (p->attn_kernel != SGQA_ATTN_AUTO && p->attn_kernel != SGQA_ATTN_WARP && p->attn_kernel != SGQA_ATTN_TC_UNION &&
      p->attn_kernel != SGQA_ATTN_ROUTED && p->attn_kernel != SGQA_ATTN_GROUPED)
    return SGQA_ERR_INVALID_ARGUMENT;
  o.G = p->num_kv_groups;
  o.Hg = p->heads_per_group;
  o.H = o.G * o.Hg;
  o.D = p->head_dim;
  o.P = p->proxy_dim;
  o.B = B;
  o.k = p->top_k_blocks;
  o.gate_per_dim = p->gate_per_dim;
  o.attn_kernel = p->attn_kernel;
  o.scale = p->softmax_scale > 0.f ? p->softmax_scale : 1.0f / std::sqrt((float)o.D);
  return SGQA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D tiled tensor map with 128-byte swizzle.  dims/box innermost first; strides in bytes
// for dims 1 and 2.
bool make_map_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                 uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- per-device launch state ----
// The SM count and the kernels whose dynamic shared-memory limit has been raised, kept per
// device under one mutex: a process may drive several devices, from several threads.
constexpr int kMaxDevices = 64;
struct DevState {
  int sms = 0;
  uint32_t attr_done = 0;  // bit per AttrKernel
};
std::mutex g_dev_mu;
DevState g_dev[kMaxDevices];

int current_device() {
  int d = -1;
  return cudaGetDevice(&d) == cudaSuccess && d >= 0 && d < kMaxDevices ? d : -1;
}

int num_sms() {
  const int dev = current_device();
  if (dev < 0) return 148;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (g_dev[dev].sms == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    g_dev[dev].sms = n;
  }
  return g_dev[dev].sms;
}

enum AttrKernel { kAttrK2 = 0, kAttrK4Tma = 1, kAttrK4Cp = 2, kAttrK4U = 3 };

// Raises the dynamic shared-memory limit of `fn` to `bytes` once per device.
cudaError_t ensure_smem_attr(AttrKernel which, const void* fn, size_t bytes) {
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (g_dev[dev].attr_done & (1u << which)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) g_dev[dev].attr_done |= 1u << which;
  return e;
}

// ---- attention launch: 8 warps (units) per CTA, two stages each ----
constexpr int kK4Warps = 8;
size_t k4_smem(int nw, bool tma) {
  return (size_t)nw * 2 * k4_stage_bytes(tma) + (size_t)nw * 2 * 8 + (size_t)nw * K4_SEL_CACHE * 4 + 1024;
}

template <bool TMA>
cudaError_t launch_k4_t(const K4Args& a, const CUtensorMap& tk, const CUtensorMap& tv, int64_t n_units,
                        cudaStream_t st) {
  const size_t smem = k4_smem(kK4Warps, TMA);
  const cudaError_t e = ensure_smem_attr(TMA ? kAttrK4Tma : kAttrK4Cp,
                                         reinterpret_cast<const void*>(k4_sparse_attn<kK4Warps, TMA>), smem);
  if (e != cudaSuccess) return e;
  const int64_t grid = cdiv(n_units, kK4Warps);
  k4_sparse_attn<kK4Warps, TMA><<<(unsigned)grid, kK4Warps * 32, smem, st>>>(a, tk, tv);
  return cudaGetLastError();
}

cudaError_t launch_k4(const K4Args& a, const CUtensorMap& tk, const CUtensorMap& tv, int64_t n_units, bool tma,
                      cudaStream_t st) {
  return tma ? launch_k4_t<true>(a, tk, tv, n_units, st) : launch_k4_t<false>(a, tk, tv, n_units, st);
}

// K and V cache maps for the attention kernels: dims {64, tokens, 3 chunks} with strides
// {384 B, 128 B}; one copy of box {64, 8, 3} lands 8 tokens as three 1 KB swizzle atoms.
bool make_kv_map(CUtensorMap* m, const void* base, uint64_t tokens) {
  return make_map_3d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, 64, tokens, 3, 384, 128, 64, 8, 3);
}

cudaError_t launch_k2(const K2Args& a, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                      cudaStream_t st) {
  const cudaError_t e = ensure_smem_attr(kAttrK2, reinterpret_cast<const void*>(k2_indexer), K2_SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int64_t grid = std::min<int64_t>(a.n_items, num_sms());
  if (grid <= 0) return cudaSuccess;
  k2_indexer<<<(unsigned)grid, K2_THREADS, K2_SMEM_BYTES, st>>>(a, ta, tb, tc);
  return cudaGetLastError();
}

// Segments per row of the two-level top-k for rows of up to max_cand candidates: 0 when one
// CTA holds the row in registers (or k = 1), or when the merged lists would not fit either
// (the streaming instance then serves the row).
int64_t k3_segments(const Prm& p, int64_t max_cand) {
  if (max_cand <= kK3RegRow || p.k < 2) return 0;
  const int64_t nseg = cdiv(max_cand, kK3RegRow);
  return nseg * (p.k - 1) <= kK3RegRow ? nseg : 0;
}

// The bound-filtered top-k (indexer maxima -> bound -> survivors -> selection, the scores
// never written) can serve rows of up to 8 * kK3RegRow candidates (their group maxima fit
// one register-resident CTA), with k - 1 at most the survivor capacity; a row needs more
// than 8 (k - 1) candidates for a bound (fewer group maxima than blocks to keep give none).
// It runs the indexer's MMAs twice, which pays only for rows longer than one CTA's
// registers hold (kK3RegRow), where the plain top-k needs its segment + merge pair
// (measured on B300: the 1M chunk's indexer + top-k 15.6 -> 9.6 ms; rows of 16K
// candidates about break even).
#ifndef SGQA_K3_FILTER_MIN
#define SGQA_K3_FILTER_MIN 16384
#endif
int64_t filtered_min_cand(const Prm& p) { return std::max<int64_t>(8 * (int64_t)(p.k - 1), SGQA_K3_FILTER_MIN); }
bool filtered_topk_fits(const Prm& p, int64_t max_cand) {
  return p.k >= 2 && p.k - 1 <= K3_SEL_CAP && max_cand <= 8 * kK3RegRow && max_cand > filtered_min_cand(p);
}

// Layout of the top-k workspace for `rows` rows: fp32 scores [G, rows, ld], then (for
// segmented rows) pair keys and indices [G * rows, nseg * (k-1)] and counts [G * rows, nseg].
// With `filtered`: group maxima [G * rows, ld8], bounds [G * rows], survivor masks
// [G * rows, ld32], then the flags of rows with more survivors than K3_SEL_CAP [G * rows]
// and of their 128-row tiles [G, n_mtiles] (one memset clears them per pass).  The score
// buffer holds the survivors' keys in place, and the scores of flagged tiles.
struct IndexWs {
  int64_t ld, nseg, ld8, ld32, n_mtiles;
  bool filtered;
  size_t scores, pair_key, pair_idx, pair_cnt, maxima, thr, smask, flags, total;
};
IndexWs index_ws_layout(const Prm& p, int64_t rows, int64_t max_cand, bool filtered) {
  IndexWs w{};
  w.ld = std::max<int64_t>(4, (int64_t)align_up((size_t)max_cand, 4));
  w.nseg = k3_segments(p, max_cand);
  const size_t r = (size_t)p.G * rows;
  w.scores = 0;
  w.pair_key = align_up(r * w.ld * 4, 256);
  w.pair_idx = w.pair_key + align_up(r * w.nseg * (p.k - 1) * 4, 256);
  w.pair_cnt = w.pair_idx + align_up(r * w.nseg * (p.k - 1) * 4, 256);
  w.total = w.pair_cnt + align_up(r * w.nseg * 4, 256);
  if (filtered) {
    w.filtered = true;
    w.ld8 = 4 * cdiv(w.ld, 32);
    w.ld32 = cdiv(w.ld, 32);
    w.n_mtiles = cdiv(rows, 128);
    w.maxima = w.total;
    w.thr = w.maxima + align_up(r * w.ld8 * 4, 256);
    w.smask = w.thr + align_up(r * 4, 256);
    w.flags = w.smask + align_up(r * w.ld32 * 4, 256);
    w.total = w.flags + align_up(r * 4 + (size_t)p.G * w.n_mtiles * 4, 256);
  }
  return w;
}

// One CTA per row; the block is the smallest whose registers (32 keys per thread) hold
// the launch's longest row, so short rows do not pay for empty slots.  Longer rows go
// through the segment + merge pair when `wsl` gives them pair buffers inside `ws`.
// Register-resident top-k launch for rows of at most NT * PER candidates, PER the
// smallest multiple of 4 that holds max_cand (at least 8): short rows do not pay for
// empty slots.
template <int NT, int MODE = K3_DIRECT>
void launch_k3_regs(const K3Args& a, int64_t max_cand, int64_t grid, cudaStream_t st) {
  const int per = (int)std::max<int64_t>(8, cdiv(cdiv(max_cand, NT), 4) * 4);
  switch (per) {
    case 8: k3_topk<NT, 8, false, MODE><<<(unsigned)grid, NT, 0, st>>>(a); break;
    case 12: k3_topk<NT, 12, false, MODE><<<(unsigned)grid, NT, 0, st>>>(a); break;
    case 16: k3_topk<NT, 16, false, MODE><<<(unsigned)grid, NT, 0, st>>>(a); break;
    case 20: k3_topk<NT, 20, false, MODE><<<(unsigned)grid, NT, 0, st>>>(a); break;
    case 24: k3_topk<NT, 24, false, MODE><<<(unsigned)grid, NT, 0, st>>>(a); break;
    case 28: k3_topk<NT, 28, false, MODE><<<(unsigned)grid, NT, 0, st>>>(a); break;
    default: k3_topk<NT, 32, false, MODE><<<(unsigned)grid, NT, 0, st>>>(a); break;
  }
}
static_assert(K3_SEL_CAP == 128 * 32 && K3_SEL_CAP == kK3Threads * 8, "survivor selection: 128 x 32 or 512 x 8 keys");

// One CTA per row; the block is the smallest whose registers (up to 32 keys per thread)
// hold the launch's longest row.  Longer rows go through the segment + merge pair when
// `wsl` gives them pair buffers inside `ws`.
#ifndef SGQA_K3_PREFETCH_WAVES
#define SGQA_K3_PREFETCH_WAVES 1
#endif
cudaError_t launch_k3(K3Args a, int64_t max_cand, uint8_t* ws, const IndexWs& wsl, cudaStream_t st) {
  const int64_t grid = (int64_t)a.G * a.rows;
  if (grid <= 0) return cudaSuccess;
  // prefetch distance: resident CTAs (1,024 threads per SM) times the waves ahead (one
  // wave measured best on B300: 128K indexer + top-k 16.97 -> 16.46 ms; two 16.50, four 17.50)
  if (!a.only_flagged) {
    const int nt = max_cand <= 128 * kK3Per ? 128 : (max_cand <= 256 * kK3Per ? 256 : kK3Threads);
    a.prefetch_ctas = SGQA_K3_PREFETCH_WAVES * num_sms() * (1024 / nt);
  }
  if (max_cand <= 128 * kK3Per) {
    launch_k3_regs<128>(a, max_cand, grid, st);
  } else if (max_cand <= 256 * kK3Per) {
    launch_k3_regs<256>(a, max_cand, grid, st);
  } else if (max_cand <= kK3RegRow) {
    launch_k3_regs<kK3Threads>(a, max_cand, grid, st);
  } else if (wsl.nseg > 0 && cdiv(max_cand, kK3RegRow) <= wsl.nseg) {
    a.nseg = (int32_t)cdiv(max_cand, kK3RegRow);
    a.pair_key = reinterpret_cast<uint32_t*>(ws + wsl.pair_key);
    a.pair_idx = reinterpret_cast<int32_t*>(ws + wsl.pair_idx);
    a.pair_cnt = reinterpret_cast<int32_t*>(ws + wsl.pair_cnt);
    k3_topk<kK3Threads, kK3Per, false, K3_SEGMENT><<<(unsigned)(grid * a.nseg), kK3Threads, 0, st>>>(a);
    const int64_t slots = (int64_t)a.nseg * (a.k - 1);
    if (slots <= 128 * kK3Per)
      k3_topk<128, kK3Per, false, K3_MERGE><<<(unsigned)grid, 128, 0, st>>>(a);
    else if (slots <= 256 * kK3Per)
      k3_topk<256, kK3Per, false, K3_MERGE><<<(unsigned)grid, 256, 0, st>>>(a);
    else
      k3_topk<kK3Threads, kK3Per, false, K3_MERGE><<<(unsigned)grid, kK3Threads, 0, st>>>(a);
  } else {
    k3_topk<kK3Threads, kK3Per, true><<<(unsigned)grid, kK3Threads, 0, st>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_k1(const K1Args& a, cudaStream_t st, bool e4m3 = false) {
  const int64_t n_vec = (int64_t)a.G * a.n_blocks * (a.P / 8);
  if (n_vec <= 0) return cudaSuccess;
  const int64_t grid = std::min<int64_t>(cdiv(n_vec, 256), (int64_t)num_sms() * 16);
  if (e4m3)
    k1_block_index<true><<<(unsigned)grid, 256, 0, st>>>(a);
  else
    k1_block_index<false><<<(unsigned)grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

// Bytes of the indexer + top-k workspace for `rows` query rows whose largest candidate
// count is max_cand.
size_t index_ws_bytes(const Prm& p, int64_t rows, int64_t max_cand, bool filtered) {
  return index_ws_layout(p, rows, max_cand, filtered).total;
}
// what a prefill's indexer + top-k asks for: the filtered layout where it can serve
size_t index_ws_bytes(const Prm& p, int64_t rows, int64_t max_cand) {
  return index_ws_bytes(p, rows, max_cand, filtered_topk_fits(p, max_cand));
}

// ---- the indexer + top-k over rows [0, T) at positions q_start .. ----
sgqa_status run_index_topk(const Prm& p, const void* q_proxy, int64_t T, int64_t q_start, const void* k_blk,
                           int64_t nb_cap, int32_t* sel_idx, int32_t* sel_cnt, void* ws, size_t ws_bytes,
                           cudaStream_t st) {
  const int64_t max_cand = (q_start + T - 1) / p.B;  // candidates of the last row
  // rows per pass: as many as the workspace holds, preferring kIndexChunkRows; the
  // bound-filtered top-k when the workspace holds its buffers for kIndexChunkRows rows
  int64_t rows = std::min<int64_t>(T, kIndexChunkRows);
  const bool filtered = filtered_topk_fits(p, max_cand) && index_ws_bytes(p, rows, max_cand, true) <= ws_bytes;
  if (!filtered && index_ws_bytes(p, rows, max_cand, false) > ws_bytes) {
    int64_t lo = 0, hi = rows;  // largest row count that fits
    while (lo < hi) {
      const int64_t mid = (lo + hi + 1) / 2;
      if (index_ws_bytes(p, mid, max_cand, false) <= ws_bytes) lo = mid; else hi = mid - 1;
    }
    rows = lo >= 128 ? lo / 128 * 128 : lo;
    if (rows < std::min<int64_t>(T, 128)) return SGQA_ERR_WORKSPACE_TOO_SMALL;
  }
  if (!aligned16(ws)) return SGQA_ERR_INVALID_ARGUMENT;
  const IndexWs wsl = index_ws_layout(p, rows, max_cand, filtered);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const int64_t ld = wsl.ld;
  float* scores = static_cast<float*>(ws);

  CUtensorMap ta, tb;
  if (!make_map_3d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q_proxy, p.P, T, p.G, (uint64_t)p.P * 2,
                   (uint64_t)T * p.P * 2, 64, 128, 1))
    return SGQA_ERR_CUDA;
  if (!make_map_3d(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, k_blk, p.P, nb_cap, p.G, (uint64_t)p.P * 2,
                   (uint64_t)nb_cap * p.P * 2, 64, 128, 1))
    return SGQA_ERR_CUDA;

  for (int64_t r0 = 0; r0 < T; r0 += rows) {
    const int64_t rc = std::min<int64_t>(rows, T - r0);
    const int64_t cand_last = (q_start + r0 + rc - 1) / p.B;
    // the pass runs bound-filtered when every row has more than filtered_min_cand candidates
    const bool pass_filtered = wsl.filtered && (q_start + r0) / p.B > filtered_min_cand(p);
    CUtensorMap tc;
    if (cand_last > 0 && !make_map_3d(&tc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, scores, ld, rc, p.G, (uint64_t)ld * 4,
                                      (uint64_t)rc * ld * 4, 32, 32, 1))
      return SGQA_ERR_CUDA;
    K2Args a2{};
    a2.G = p.G;
    a2.P = p.P;
    a2.B = p.B;
    a2.kch = p.P / 64;
    a2.Tc = rc;
    a2.row_base = r0;
    a2.pos0 = q_start + r0;
    a2.n_mtiles = (int32_t)cdiv(rc, 128);
    a2.nti = 8;
    a2.items_per_m = (int32_t)cdiv(cdiv(cand_last, 128), a2.nti);
    a2.n_items = (int64_t)p.G * a2.n_mtiles * a2.items_per_m;
    a2.ld = ld;
    a2.wait_ns = g_wait_ns;
    a2.mode = K2_SCORES;
    K3Args a3{};
    a3.scores = scores;
    a3.ld = ld;
    a3.rows = rc;
    a3.pos0 = q_start + r0;
    a3.out_row0 = r0;
    a3.T_out = T;
    a3.G = p.G;
    a3.B = p.B;
    a3.k = p.k;
    a3.sel_idx = sel_idx;
    a3.sel_cnt = sel_cnt;
    a3.use_pos = 0;
    if (pass_filtered) {
      const int64_t rr = (int64_t)p.G * rc;
      uint32_t* maxima = reinterpret_cast<uint32_t*>(wsb + wsl.maxima);
      uint32_t* thr = reinterpret_cast<uint32_t*>(wsb + wsl.thr);
      uint32_t* smask = reinterpret_cast<uint32_t*>(wsb + wsl.smask);
      int32_t* row_flag = reinterpret_cast<int32_t*>(wsb + wsl.flags);  // [G * rc]
      int32_t* tile_flag = row_flag + rr;                                 // [G, n_mtiles of this pass]
      SGQA_CUDA_OK(cudaMemsetAsync(row_flag, 0, (size_t)(rr + (int64_t)p.G * a2.n_mtiles) * 4, st));
      // 1. group maxima of the scores (nothing else leaves the SM), over 16 candidates where
      // every row still has more than k - 1 groups and keeps few of its candidates (half the
      // bound's work; measured on B300: 1M chunk 15.2 -> 14.7 ms), else over 8 (with
      // k = 2,048 the coarser bound's extra survivors cost more: token-level 231 -> 238 ms)
      const int32_t gs = p.k - 1 <= 1024 && (q_start + r0) / p.B > 16 * (int64_t)(p.k - 1) ? 16 : 8;
      a2.mode = K2_MAXIMA;
      a2.maxima = maxima;
      a2.ld8 = wsl.ld8;
      a2.gs = gs;
      SGQA_CUDA_OK(launch_k2(a2, ta, tb, tc, st));
      // 2. each row's bound: the (k-1)-th largest of its group maxima
      {
        K3Args t = a3;
        t.keys_in = maxima;
        t.keys_ld = wsl.ld8;
        t.keys_gs = gs;
        t.thr_out = thr;
        const int64_t n_max = cdiv(cand_last, gs), grid = rr;
        if (n_max <= 128 * kK3Per)
          launch_k3_regs<128, K3_THRESHOLD>(t, n_max, grid, st);
        else if (n_max <= 256 * kK3Per)
          launch_k3_regs<256, K3_THRESHOLD>(t, n_max, grid, st);
        else
          launch_k3_regs<kK3Threads, K3_THRESHOLD>(t, n_max, grid, st);
        SGQA_CUDA_OK(cudaGetLastError());
      }
      // 3. the candidates that reach the bound: mask bits, keys in place
      a2.mode = K2_SURVIVORS;
      a2.thr = thr;
      a2.smask = smask;
      a2.ld32 = wsl.ld32;
      a2.skeys = reinterpret_cast<uint32_t*>(scores);
      SGQA_CUDA_OK(launch_k2(a2, ta, tb, tc, st));
      // 4. the exact selection over each row's survivors; a row past the capacity is flagged
      {
        K3Args t = a3;
        t.smask = smask;
        t.ld32 = wsl.ld32;
        t.skeys = reinterpret_cast<const uint32_t*>(scores);
        t.cap = K3_SEL_CAP;
        t.n_mtiles = a2.n_mtiles;
        t.row_flag = row_flag;
        t.tile_flag = tile_flag;
        // (128 x 32 keys for the usual k; large selections, where each row keeps thousands
        // of its survivors, spread over 512 x 8)
        if (p.k > 1024)
          k3_topk<kK3Threads, 8, false, K3_SELECT><<<(unsigned)rr, kK3Threads, 0, st>>>(t);
        else
          k3_topk<128, 32, false, K3_SELECT><<<(unsigned)rr, 128, 0, st>>>(t);
        SGQA_CUDA_OK(cudaGetLastError());
      }
      // 5. flagged rows (heavy ties) are redone from their scores: the indexer writes the
      // flagged tiles' scores, the top-k serves the flagged rows; other CTAs return at once
      a2.mode = K2_SCORES;
      a2.tile_flag = tile_flag;
      SGQA_CUDA_OK(launch_k2(a2, ta, tb, tc, st));
      a3.only_flagged = row_flag;
      k3_topk<128, kK3Per, true><<<(unsigned)rr, 128, 0, st>>>(a3);  // any row length
      SGQA_CUDA_OK(cudaGetLastError());
      continue;
    }
    if (cand_last > 0) SGQA_CUDA_OK(launch_k2(a2, ta, tb, tc, st));
    SGQA_CUDA_OK(launch_k3(a3, cand_last, wsb, wsl, st));
  }
  return SGQA_OK;
}

// The union kernel serves a prefill call when its shape holds: blocks of 8, 16 heads per
// group, at most 512 selected blocks per row (a unit's union fits its 4,096-entry table),
// block indices below K4U_MAX_BLOCKS, not dense mode.
bool union_fits(const Prm& p, int32_t dense, int64_t T, int64_t q_start) {
  return p.B == 8 && p.Hg == 16 && p.k <= 512 && !dense && T > 0 &&
         (q_start + T - 1) / 8 < (int64_t)K4U_MAX_BLOCKS;
}

// The attention kernel a call launches (SGQA_ATTN_WARP, _TC_UNION or _ROUTED), following
// sgqa_params.attn_kernel; -1 when the requested kernel cannot serve these arguments.
// ws_ok: the call's workspace holds the routed mode's buffers (attn_ws_layout).
int attn_choice(const Prm& p, int32_t dense, int64_t T, int64_t q_start, bool ws_ok) {
  const bool fits = union_fits(p, dense, T, q_start);
  switch (p.attn_kernel) {
    case SGQA_ATTN_AUTO:
      // (the routing rule sends no unit to the union kernel once every unit spans more
      // windows than kRoutePairCost * 8 / kRouteUnionCost: then the warp-level kernel alone)
      if (fits && (q_start / 8) / K4U_WIN + 1 > (int64_t)kRoutePairCost * 8 / kRouteUnionCost) return SGQA_ATTN_WARP;
      return fits ? (ws_ok ? SGQA_ATTN_GROUPED : SGQA_ATTN_TC_UNION) : SGQA_ATTN_WARP;
    case SGQA_ATTN_WARP: return SGQA_ATTN_WARP;
    case SGQA_ATTN_TC_UNION: return fits ? SGQA_ATTN_TC_UNION : -1;
    case SGQA_ATTN_ROUTED: return fits ? SGQA_ATTN_ROUTED : -1;
    case SGQA_ATTN_GROUPED: return fits ? SGQA_ATTN_GROUPED : -1;
  }
  return -1;
}

// Workspace of the routed and grouped attention modes for T query rows: the per-unit
// choice, the two unit lists and their lengths (units = G x ceil(T / 8)), and the grouped
// mode's row order [G, T] and sort keys [G, T].
struct AttnWs {
  size_t choice, union_units, warp_units, counts, perm, keys, total;
};
AttnWs attn_ws_layout(const Prm& p, int64_t T) {
  AttnWs w{};
  const size_t nu = (size_t)p.G * (size_t)cdiv(std::max<int64_t>(T, 0), 8);
  w.choice = 0;
  w.union_units = align_up(nu * 4, 256);
  w.warp_units = w.union_units + align_up(nu * 4, 256);
  w.counts = w.warp_units + align_up(nu * 4, 256);
  w.perm = w.counts + 256;
  w.keys = w.perm + align_up((size_t)p.G * (size_t)std::max<int64_t>(T, 0) * 4, 256);
  w.total = w.keys + align_up((size_t)p.G * (size_t)std::max<int64_t>(T, 0) * 8, 256);
  return w;
}

cudaError_t launch_k4u(const K4UArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
  const cudaError_t e = ensure_smem_attr(kAttrK4U, reinterpret_cast<const void*>(k4u_sparse_attn), K4U_SMEM);
  if (e != cudaSuccess) return e;
  const int64_t n_units = (int64_t)a.G * cdiv(a.rows, 8);
  const int64_t grid = std::min<int64_t>(n_units, num_sms());
  if (grid <= 0) return cudaSuccess;
  k4u_sparse_attn<<<(unsigned)grid, K4U_THREADS, K4U_SMEM, st>>>(a, tk, tv);
  return cudaGetLastError();
}

sgqa_status run_attention(const Prm& p, const void* q, const void* k, const void* v, int64_t ctx_cap, const void* gate,
                          const int32_t* sel_idx, const int32_t* sel_cnt, int64_t T, int64_t q_start, void* out,
                          float* lse, int32_t dense, void* ws, size_t ws_bytes, cudaStream_t st) {
  const AttnWs wl = attn_ws_layout(p, T);
  const bool ws_ok = ws && aligned16(ws) && ws_bytes >= wl.total;
  const int kernel = attn_choice(p, dense, T, q_start, ws_ok);
  if (kernel < 0) return SGQA_ERR_UNSUPPORTED_SHAPE;
  const bool routed = kernel == SGQA_ATTN_ROUTED || kernel == SGQA_ATTN_GROUPED;
  if (routed && !ws_ok) return SGQA_ERR_WORKSPACE_TOO_SMALL;
  const uint64_t kv_rows = (uint64_t)p.G * ctx_cap;
  uint8_t* w = static_cast<uint8_t*>(ws);
  const int32_t* union_units = nullptr;
  const int32_t* counts = nullptr;
  const int32_t* perm = nullptr;
  if (kernel == SGQA_ATTN_GROUPED) {
    // rows ordered by the MinHash signature of their selections within 1,024-row windows
    K4GroupArgs ga{};
    ga.sel_idx = sel_idx;
    ga.sel_cnt = sel_cnt;
    ga.perm = reinterpret_cast<int32_t*>(w + wl.perm);
    ga.keys = reinterpret_cast<uint64_t*>(w + wl.keys);
    ga.rows = T;
    ga.pos0 = q_start;
    ga.G = p.G;
    ga.kcap = p.k;
    k4g_signature<<<(unsigned)cdiv((int64_t)p.G * T, K4G_SIG_WARPS), K4G_SIG_WARPS * 32, 0, st>>>(ga);
    SGQA_CUDA_OK(cudaGetLastError());
    k4g_sort<<<(unsigned)(p.G * cdiv(T, K4G_WIN)), K4G_THREADS, 0, st>>>(ga);
    SGQA_CUDA_OK(cudaGetLastError());
    perm = ga.perm;
  }
  if (routed) {
    // each 8-row unit to the kernel that serves it more cheaply (k4r_route.cuh): the
    // warp-level kernel takes its list here, the union kernel below takes the other
    K4RouteArgs ra{};
    ra.sel_idx = sel_idx;
    ra.sel_cnt = sel_cnt;
    ra.perm = perm;
    ra.choice = reinterpret_cast<int32_t*>(w + wl.choice);
    ra.union_units = reinterpret_cast<int32_t*>(w + wl.union_units);
    ra.warp_units = reinterpret_cast<int32_t*>(w + wl.warp_units);
    ra.counts = reinterpret_cast<int32_t*>(w + wl.counts);
    ra.rows = T;
    ra.pos0 = q_start;
    ra.G = p.G;
    ra.kcap = p.k;
    const int64_t n_units = (int64_t)p.G * cdiv(T, 8);
    k4r_count<<<(unsigned)cdiv(n_units, K4R_WARPS), K4R_WARPS * 32, 0, st>>>(ra);
    SGQA_CUDA_OK(cudaGetLastError());
    k4r_compact<<<1, K4R_COMPACT_THREADS, 0, st>>>(ra);
    SGQA_CUDA_OK(cudaGetLastError());
    union_units = ra.union_units;
    counts = ra.counts;
    K4Args a{};
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.gate = static_cast<const __nv_bfloat16*>(gate);
    a.kc = static_cast<const __nv_bfloat16*>(k);
    a.vc = static_cast<const __nv_bfloat16*>(v);
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    a.sel_idx = sel_idx;
    a.sel_cnt = sel_cnt;
    a.rows = T;
    a.pos0 = q_start;
    a.ctx_cap = ctx_cap;
    a.G = p.G;
    a.Hg = p.Hg;
    a.H = p.H;
    a.B = p.B;
    a.kcap = p.k;
    a.scale_log2 = p.scale * 1.4426950408889634f;
    a.gate_per_dim = p.gate_per_dim;
    a.nsplit = 1;
    a.units = ra.warp_units;
    a.n_units_dev = ra.counts + 1;
    a.perm = perm;
    a.wait_ns = g_wait_ns;
    CUtensorMap tk, tv;
    if (!make_kv_map(&tk, k, kv_rows) || !make_kv_map(&tv, v, kv_rows)) return SGQA_ERR_CUDA;
    // one CTA of 8 warps per listed unit; CTAs past the list's length return at once
    SGQA_CUDA_OK(launch_k4(a, tk, tv, n_units * 8, true, st));
  }
  if (kernel == SGQA_ATTN_TC_UNION || routed) {
    K4UArgs a{};
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.gate = static_cast<const __nv_bfloat16*>(gate);
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    a.sel_idx = sel_idx;
    a.sel_cnt = sel_cnt;
    a.rows = T;
    a.pos0 = q_start;
    a.ctx_cap = ctx_cap;
    a.G = p.G;
    a.H = p.H;
    a.kcap = p.k;
    a.scale_log2 = p.scale * 1.4426950408889634f;
    a.gate_per_dim = p.gate_per_dim;
    a.wait_ns = g_wait_ns;
    a.units = union_units;
    a.n_units_dev = counts;
    a.perm = perm;
    CUtensorMap tk, tv;
    if (!make_kv_map(&tk, k, kv_rows) || !make_kv_map(&tv, v, kv_rows)) return SGQA_ERR_CUDA;
    SGQA_CUDA_OK(launch_k4u(a, tk, tv, st));
    return SGQA_OK;
  }
  K4Args a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.gate = static_cast<const __nv_bfloat16*>(gate);
  a.kc = static_cast<const __nv_bfloat16*>(k);
  a.vc = static_cast<const __nv_bfloat16*>(v);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.sel_idx = sel_idx;
  a.sel_cnt = sel_cnt;
  a.rows = T;
  a.pos0 = q_start;
  a.ctx_cap = ctx_cap;
  a.G = p.G;
  a.Hg = p.Hg;
  a.H = p.H;
  a.B = p.B;
  a.kcap = p.k;
  a.scale_log2 = p.scale * 1.4426950408889634f;
  a.dense = dense;
  a.gate_per_dim = p.gate_per_dim;
  a.nsplit = 1;
  a.use_pos = 0;
  a.wait_ns = g_wait_ns;
  const bool tma = p.B >= 8;
  CUtensorMap tk{}, tv{};
  if (tma) {
    const uint64_t rowsz = (uint64_t)p.G * ctx_cap;
    if (!make_kv_map(&tk, k, rowsz) || !make_kv_map(&tv, v, rowsz)) return SGQA_ERR_CUDA;
  }
  SGQA_CUDA_OK(launch_k4(a, tk, tv, (int64_t)p.G * T, tma, st));
  return SGQA_OK;
}

// Workspace the attention entries want for T rows ending at ctx_len: the routed mode's when
// the union kernel can serve the call (positions q_start = ctx_len - T onwards), else none.
size_t attn_ws_bytes(const Prm& p, int64_t T, int64_t ctx_len) {
  if (T <= 0 || !union_fits(p, 0, T, std::max<int64_t>(0, ctx_len - T))) return 0;
  return attn_ws_layout(p, T).total;
}

// ---- scratch for the allocation-free indexer entry ----
// A file-scope device array: every GPU that loads the library holds it until exit.  Host
// code must not pass the symbol itself to a kernel (in host code it names a host-side
// stand-in); its device address is looked up once per device with cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_noalloc_scratch[SGQA_NOALLOC_SCRATCH_BYTES];
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

sgqa_status noalloc_scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SGQA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SGQA_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return SGQA_OK;
}


// ---- end-to-end prefill from host memory: chunk layout and per-device copy streams ----
constexpr int64_t kHostChunkRows = 4096;  // default query rows per pipelined chunk
constexpr int kHostRing = 4;              // events per kind; chunk j uses slot j % kHostRing

// Rows per chunk: chunk_rows (default kHostChunkRows) rounded down to a multiple of B,
// at least B, at most T rounded up to B.
int64_t host_chunk_rows(const Prm& p, int64_t T, int64_t chunk_rows) {
  int64_t R = chunk_rows > 0 ? chunk_rows : kHostChunkRows;
  R = std::min<int64_t>(R, cdiv(std::max<int64_t>(T, 1), p.B) * p.B);
  return std::max<int64_t>(p.B, R / p.B * p.B);
}

// Workspace of sgqa_prefill_host: two q_proxy chunk buffers [G, R, P] (chunk j + 1 is
// copied in while chunk j is computed), the chunk's selection [G, R, k] and counts [G, R],
// then the indexer + top-k workspace of one chunk.
struct HostWs {
  size_t qp[2], sel, cnt, index, index_bytes, total;
};
HostWs host_ws_layout(const Prm& p, int64_t R, int64_t ctx_len) {
  HostWs w{};
  const size_t qp = align_up((size_t)p.G * R * p.P * 2, 256);
  w.qp[0] = 0;
  w.qp[1] = qp;
  w.sel = 2 * qp;
  w.cnt = w.sel + align_up((size_t)p.G * R * p.k * 4, 256);
  w.index = w.cnt + align_up((size_t)p.G * R * 4, 256);
  // one chunk's indexer + top-k scratch, reused by its attention (the routed mode's lists)
  w.index_bytes = std::max<size_t>({256, index_ws_bytes(p, R, (ctx_len - 1) / p.B), attn_ws_bytes(p, R, ctx_len)});
  w.total = w.index + w.index_bytes;
  return w;
}

// Two non-blocking copy streams (host to device, device to host) and the pipeline's events,
// created on a device's first sgqa_prefill_host call and kept until the process exits.
// The mutex is held while a call enqueues its work, so calls from several host threads
// do not interleave their use of the shared events.
struct HostPipe {
  bool ready = false;
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t begin = nullptr, end = nullptr, copied[kHostRing] = {}, done[kHostRing] = {};
  std::mutex mu;
};
HostPipe g_pipe[kMaxDevices];

sgqa_status host_pipe(HostPipe** out) {
  const int dev = current_device();
  if (dev < 0) return SGQA_ERR_CUDA;
  HostPipe& h = g_pipe[dev];
  {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (!h.ready) {
      const unsigned ef = cudaEventDisableTiming;
      bool ok = cudaStreamCreateWithFlags(&h.s_in, cudaStreamNonBlocking) == cudaSuccess &&
                cudaStreamCreateWithFlags(&h.s_out, cudaStreamNonBlocking) == cudaSuccess &&
                cudaEventCreateWithFlags(&h.begin, ef) == cudaSuccess &&
                cudaEventCreateWithFlags(&h.end, ef) == cudaSuccess;
      for (int i = 0; ok && i < kHostRing; ++i)
        ok = cudaEventCreateWithFlags(&h.copied[i], ef) == cudaSuccess &&
             cudaEventCreateWithFlags(&h.done[i], ef) == cudaSuccess;
      if (!ok) return SGQA_ERR_CUDA;  // partial objects stay allocated; the next call retries the rest
      h.ready = true;
    }
  }
  *out = &h;
  return SGQA_OK;
}

// Copies G rows of `bytes` each, `pitch_src` / `pitch_dst` apart (one strided copy).
cudaError_t copy_rows(void* dst, size_t pitch_dst, const void* src, size_t pitch_src, size_t bytes, size_t rows,
                      cudaMemcpyKind kind, cudaStream_t st) {
  if (bytes == 0 || rows == 0) return cudaSuccess;
  return cudaMemcpy2DAsync(dst, pitch_dst, src, pitch_src, bytes, rows, kind, st);
}

}  // namespace

extern "C" {

const char* sgqa_status_string(sgqa_status s) {
  switch (s) {
    case SGQA_OK: return "ok";
    case SGQA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case SGQA_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case SGQA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case SGQA_ERR_CUDA: return "CUDA runtime error";
    case SGQA_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case SGQA_ERR_DEVICE_BOUNDS: return "device-side index out of range";
  }
  return "unknown status";
}

int32_t sgqa_abi_version(void) { return SGQA_ABI_VERSION; }

int32_t sgqa_attention_kernel(const sgqa_params* prm, int64_t T, int64_t q_start, int32_t dense_mode) {
  Prm p;
  if (check_params(prm, p) != SGQA_OK || T < 0 || q_start < 0) return -1;
  return attn_choice(p, dense_mode ? 1 : 0, T, q_start, true);
}

sgqa_status sgqa_set_wait_timeout_ns(uint64_t ns) {
  g_wait_ns = ns;
  return SGQA_OK;
}

sgqa_status sgqa_get_device_error(sgqa_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return SGQA_ERR_CUDA;
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess) return SGQA_ERR_CUDA;
  if (v != 0 && cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero) != cudaSuccess) return SGQA_ERR_CUDA;
  return static_cast<sgqa_status>(v);
}

sgqa_status sgqa_selftest_wait_timeout(uint64_t limit_ns, sgqa_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  k_selftest_wait<<<1, 1, 0, st>>>(limit_ns, nullptr);
  return cudaGetLastError() == cudaSuccess ? SGQA_OK : SGQA_ERR_CUDA;
}

size_t sgqa_workspace_bytes(const sgqa_params* prm, int32_t op, int64_t T, int64_t ctx_len, int32_t batch) {
  Prm p;
  if (check_params(prm, p) != SGQA_OK || T < 0 || ctx_len < 1) return 0;
  const int64_t max_cand = (ctx_len - 1) / p.B;
  switch (op) {
    case SGQA_OP_INDEX_TOPK:
      return std::max<size_t>(256, index_ws_bytes(p, std::min<int64_t>(std::max<int64_t>(T, 1), kIndexChunkRows), max_cand));
    case SGQA_OP_PREFILL:  // the stages run one after another: they share the workspace
      return std::max<size_t>(
          {256, index_ws_bytes(p, std::min<int64_t>(std::max<int64_t>(T, 1), kIndexChunkRows), max_cand),
           attn_ws_bytes(p, T, ctx_len)});
    case SGQA_OP_ATTN:
      return std::max<size_t>(256, attn_ws_bytes(p, T, ctx_len));
    case SGQA_OP_PREFILL_HOST:
      return host_ws_layout(p, host_chunk_rows(p, T, batch), ctx_len).total;
    case SGQA_OP_DECODE: {
      if (batch < 1 || batch > kMaxBatch) return 0;
      const size_t sc = index_ws_bytes(p, batch, max_cand, false);
      const int nsplit = 32;
      const size_t po = align_up((size_t)p.G * batch * nsplit * 16 * 192 * 4, 256);
      const size_t pml = align_up((size_t)p.G * batch * nsplit * 16 * 2 * 4, 256);
      return sc + po + pml;
    }
  }
  return 0;
}

static sgqa_status build_block_index(const sgqa_params* prm, const void* k_proxy, int64_t ctx_cap, int64_t tok_begin,
                                     int64_t tok_end, void* k_blk, int64_t nb_cap, sgqa_stream_t stream, bool e4m3) {
  Prm p;
  sgqa_status s = check_params(prm, p);
  if (s != SGQA_OK) return s;
  if (!k_proxy || !k_blk || ctx_cap < 0 || tok_begin < 0 || tok_end < tok_begin || tok_end > ctx_cap)
    return SGQA_ERR_INVALID_ARGUMENT;
  if (!aligned16(k_proxy) || !aligned16(k_blk)) return SGQA_ERR_INVALID_ARGUMENT;
  if (tok_end == tok_begin) return SGQA_OK;
  const int64_t b0 = tok_begin / p.B, b1 = cdiv(tok_end, p.B);
  if (b1 > nb_cap) return SGQA_ERR_INVALID_ARGUMENT;
  K1Args a{};
  a.k_proxy = static_cast<const __nv_bfloat16*>(k_proxy);
  a.k_blk = k_blk;
  a.ctx_cap = ctx_cap;
  a.nb_cap = nb_cap;
  a.tok_end = tok_end;
  a.blk_begin = b0;
  a.n_blocks = b1 - b0;
  a.G = p.G;
  a.P = p.P;
  a.B = p.B;
  SGQA_CUDA_OK(launch_k1(a, reinterpret_cast<cudaStream_t>(stream), e4m3));
  return SGQA_OK;
}

sgqa_status sgqa_build_block_index(const sgqa_params* prm, const void* k_proxy, int64_t ctx_cap, int64_t tok_begin,
                                   int64_t tok_end, void* k_blk, int64_t nb_cap, sgqa_stream_t stream) {
  return build_block_index(prm, k_proxy, ctx_cap, tok_begin, tok_end, k_blk, nb_cap, stream, false);
}

sgqa_status sgqa_build_block_index_fp8(const sgqa_params* prm, const void* k_proxy, int64_t ctx_cap,
                                       int64_t tok_begin, int64_t tok_end, void* k_blk_e4m3, int64_t nb_cap,
                                       sgqa_stream_t stream) {
  return build_block_index(prm, k_proxy, ctx_cap, tok_begin, tok_end, k_blk_e4m3, nb_cap, stream, true);
}

sgqa_status sgqa_index_topk(const sgqa_params* prm, const void* q_proxy, int64_t T, int64_t q_start, const void* k_blk,
                            int64_t nb_cap, int32_t* sel_idx, int32_t* sel_cnt, void* ws, size_t ws_bytes,
                            sgqa_stream_t stream) {
  Prm p;
  sgqa_status s = check_params(prm, p);
  if (s != SGQA_OK) return s;
  if (!q_proxy || !k_blk || !sel_idx || !sel_cnt || T < 0 || q_start < 0) return SGQA_ERR_INVALID_ARGUMENT;
  if (T == 0) return SGQA_OK;
  if (!ws) return SGQA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(q_proxy) || !aligned16(k_blk)) return SGQA_ERR_INVALID_ARGUMENT;
  const int64_t max_cand = (q_start + T - 1) / p.B;
  if (max_cand > nb_cap || (q_start + T - 1) / p.B > (int64_t)INT32_MAX) return SGQA_ERR_INVALID_ARGUMENT;
  return run_index_topk(p, q_proxy, T, q_start, k_blk, nb_cap, sel_idx, sel_cnt, ws, ws_bytes,
                        reinterpret_cast<cudaStream_t>(stream));
}

sgqa_status sgqa_index_topk_noalloc(const sgqa_params* prm, const void* q_proxy, int64_t T, int64_t q_start,
                                    const void* k_blk, int64_t nb_cap, int32_t* sel_idx, int32_t* sel_cnt,
                                    sgqa_stream_t stream) {
  Prm p;
  sgqa_status s = check_params(prm, p);
  if (s != SGQA_OK) return s;
  if (!q_proxy || !k_blk || !sel_idx || !sel_cnt || T < 0 || q_start < 0) return SGQA_ERR_INVALID_ARGUMENT;
  if (T == 0) return SGQA_OK;
  if (!aligned16(q_proxy) || !aligned16(k_blk)) return SGQA_ERR_INVALID_ARGUMENT;
  const int64_t max_cand = (q_start + T - 1) / p.B;
  if (max_cand > nb_cap || max_cand > (int64_t)INT32_MAX) return SGQA_ERR_INVALID_ARGUMENT;
  // the smallest pass must fit in the fixed scratch array
  if (index_ws_bytes(p, std::min<int64_t>(T, 128), max_cand, false) > (size_t)SGQA_NOALLOC_SCRATCH_BYTES)
    return SGQA_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  s = noalloc_scratch_address(&ws);
  if (s != SGQA_OK) return s;
  return run_index_topk(p, q_proxy, T, q_start, k_blk, nb_cap, sel_idx, sel_cnt, ws, SGQA_NOALLOC_SCRATCH_BYTES,
                        reinterpret_cast<cudaStream_t>(stream));
}

sgqa_status sgqa_sparse_attn_fwd(const sgqa_params* prm, const void* q, const void* k, const void* v, int64_t ctx_cap,
                                 const void* gate, const int32_t* sel_idx, const int32_t* sel_cnt, int64_t T,
                                 int64_t q_start, void* out, float* lse, int32_t dense_mode, void* ws, size_t ws_bytes,
                                 sgqa_stream_t stream) {
  Prm p;
  sgqa_status s = check_params(prm, p);
  if (s != SGQA_OK) return s;
  if (!q || !k || !v || !gate || !out || T < 0 || q_start < 0 || ctx_cap < 1) return SGQA_ERR_INVALID_ARGUMENT;
  if (!dense_mode && (!sel_idx || !sel_cnt)) return SGQA_ERR_INVALID_ARGUMENT;
  if (q_start + T > ctx_cap) return SGQA_ERR_INVALID_ARGUMENT;
  if ((int64_t)p.G * ctx_cap > (int64_t)INT32_MAX) return SGQA_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || (p.gate_per_dim && !aligned16(gate)))
    return SGQA_ERR_INVALID_ARGUMENT;
  if (T == 0) return SGQA_OK;
  return run_attention(p, q, k, v, ctx_cap, gate, sel_idx, sel_cnt, T, q_start, out, lse, dense_mode ? 1 : 0, ws,
                       ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

sgqa_status sgqa_prefill(const sgqa_params* prm, const void* q, const void* k, const void* v, const void* gate,
                         const void* q_proxy, const void* k_proxy, int64_t ctx_cap, int64_t T, int64_t q_start,
                         void* k_blk, int64_t nb_cap, int32_t* sel_idx, int32_t* sel_cnt, void* out, float* lse,
                         void* ws, size_t ws_bytes, sgqa_stream_t stream) {
  Prm p;
  sgqa_status s = check_params(prm, p);
  if (s != SGQA_OK) return s;
  if (!q || !k || !v || !gate || !q_proxy || !k_proxy || !k_blk || !sel_idx || !sel_cnt || !out)
    return SGQA_ERR_INVALID_ARGUMENT;
  if (T < 0 || q_start < 0 || q_start + T > ctx_cap) return SGQA_ERR_INVALID_ARGUMENT;
  if (T == 0) return SGQA_OK;
  if (cdiv(q_start + T, p.B) > nb_cap) return SGQA_ERR_INVALID_ARGUMENT;
  if ((int64_t)p.G * ctx_cap > (int64_t)INT32_MAX) return SGQA_ERR_UNSUPPORTED_SHAPE;
  if (!ws) return SGQA_ERR_WORKSPACE_TOO_SMALL;
  // the attention stage's own checks, made before anything is enqueued
  const bool attn_ws_ok = aligned16(ws) && ws_bytes >= attn_ws_layout(p, T).total;
  const int kernel = attn_choice(p, 0, T, q_start, attn_ws_ok);
  if (kernel < 0) return SGQA_ERR_UNSUPPORTED_SHAPE;
  if ((kernel == SGQA_ATTN_ROUTED || kernel == SGQA_ATTN_GROUPED) && !attn_ws_ok) return SGQA_ERR_WORKSPACE_TOO_SMALL;
  s = sgqa_build_block_index(prm, k_proxy, ctx_cap, q_start, q_start + T, k_blk, nb_cap, stream);
  if (s != SGQA_OK) return s;
  s = sgqa_index_topk(prm, q_proxy, T, q_start, k_blk, nb_cap, sel_idx, sel_cnt, ws, ws_bytes, stream);
  if (s != SGQA_OK) return s;
  // the indexer's scratch is dead once the top-k has run: the attention reuses the workspace
  return sgqa_sparse_attn_fwd(prm, q, k, v, ctx_cap, gate, sel_idx, sel_cnt, T, q_start, out, lse, 0, ws, ws_bytes,
                              stream);
}

sgqa_status sgqa_prefill_host(const sgqa_params* prm, const sgqa_host_tensors* host, const sgqa_device_tensors* dev,
                              int64_t ctx_cap, int64_t T, int64_t q_start, int64_t chunk_rows, sgqa_stream_t stream) {
  Prm p;
  sgqa_status s = check_params(prm, p);
  if (s != SGQA_OK) return s;
  if (!host || !dev) return SGQA_ERR_INVALID_ARGUMENT;
  const sgqa_host_tensors& h = *host;
  const sgqa_device_tensors& d = *dev;
  if (!h.q || !h.k || !h.v || !h.gate || !h.q_proxy || !h.k_proxy || !h.out) return SGQA_ERR_INVALID_ARGUMENT;
  if (!d.q || !d.k || !d.v || !d.gate || !d.k_proxy || !d.k_blk || !d.out) return SGQA_ERR_INVALID_ARGUMENT;
  if (h.lse && !d.lse) return SGQA_ERR_INVALID_ARGUMENT;
  if (T < 0 || q_start < 0 || q_start + T > ctx_cap) return SGQA_ERR_INVALID_ARGUMENT;
  if (T == 0) return SGQA_OK;
  if (cdiv(q_start + T, p.B) > d.nb_cap) return SGQA_ERR_INVALID_ARGUMENT;
  if ((int64_t)p.G * ctx_cap > (int64_t)INT32_MAX) return SGQA_ERR_UNSUPPORTED_SHAPE;
  const int64_t R = host_chunk_rows(p, T, chunk_rows);
  const HostWs wl = host_ws_layout(p, R, q_start + T);
  if (!d.ws || d.ws_bytes < wl.total) return SGQA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(d.ws)) return SGQA_ERR_INVALID_ARGUMENT;
  // the same checks sgqa_prefill makes on every chunk, made once before anything is enqueued
  if (attn_choice(p, 0, std::min(T, R), q_start, true) < 0 ||
      attn_choice(p, 0, T - (T - 1) / R * R, q_start + (T - 1) / R * R, true) < 0)
    return SGQA_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(d.q) || !aligned16(d.k) || !aligned16(d.v) || !aligned16(d.out) || !aligned16(d.k_proxy) ||
      !aligned16(d.k_blk) || (p.gate_per_dim && !aligned16(d.gate)))
    return SGQA_ERR_INVALID_ARGUMENT;
  HostPipe* pp = nullptr;
  s = host_pipe(&pp);
  if (s != SGQA_OK) return s;
  std::lock_guard<std::mutex> lock(pp->mu);
  cudaStream_t comp = reinterpret_cast<cudaStream_t>(stream);
  const size_t D2 = (size_t)p.D * 2, P2 = (size_t)p.P * 2;
  const size_t row_q = (size_t)p.H * D2;                        // bytes of one query row of q / out
  const size_t row_g = p.gate_per_dim ? row_q : (size_t)p.H * 2;  // of gate
  uint8_t* ws = static_cast<uint8_t*>(d.ws);
  auto dq = static_cast<uint8_t*>(d.q);
  auto dg = static_cast<uint8_t*>(d.gate);
  auto dout = static_cast<uint8_t*>(d.out);
  auto hq = static_cast<const uint8_t*>(h.q);
  auto hg = static_cast<const uint8_t*>(h.gate);
  auto hqp = static_cast<const uint8_t*>(h.q_proxy);
  auto hout = static_cast<uint8_t*>(h.out);

  SGQA_CUDA_OK(cudaEventRecord(pp->begin, comp));
  SGQA_CUDA_OK(cudaStreamWaitEvent(pp->s_in, pp->begin, 0));
  SGQA_CUDA_OK(cudaStreamWaitEvent(pp->s_out, pp->begin, 0));
  int64_t ctx_done = 0;  // cache positions copied so far
  for (int64_t j = 0, a = 0; a < T; ++j, a += R) {
    const int64_t rows = std::min(R, T - a);
    const int slot = (int)(j % kHostRing);
    void* qp = ws + wl.qp[j & 1];
    // ---- copy-in (s_in): the cache up to the chunk's last position, then its query rows ----
    if (j >= 2) SGQA_CUDA_OK(cudaStreamWaitEvent(pp->s_in, pp->done[(j - 2) % kHostRing], 0));  // qp[j & 1] is free
    const int64_t hi = q_start + a + rows;
    const size_t c0 = (size_t)ctx_done, cl = (size_t)(hi - ctx_done);
    SGQA_CUDA_OK(copy_rows(static_cast<uint8_t*>(d.k) + c0 * D2, ctx_cap * D2, static_cast<const uint8_t*>(h.k) + c0 * D2,
                           ctx_cap * D2, cl * D2, p.G, cudaMemcpyHostToDevice, pp->s_in));
    SGQA_CUDA_OK(copy_rows(static_cast<uint8_t*>(d.v) + c0 * D2, ctx_cap * D2, static_cast<const uint8_t*>(h.v) + c0 * D2,
                           ctx_cap * D2, cl * D2, p.G, cudaMemcpyHostToDevice, pp->s_in));
    SGQA_CUDA_OK(copy_rows(static_cast<uint8_t*>(d.k_proxy) + c0 * P2, ctx_cap * P2,
                           static_cast<const uint8_t*>(h.k_proxy) + c0 * P2, ctx_cap * P2, cl * P2, p.G,
                           cudaMemcpyHostToDevice, pp->s_in));
    SGQA_CUDA_OK(cudaMemcpyAsync(dq + a * row_q, hq + a * row_q, rows * row_q, cudaMemcpyHostToDevice, pp->s_in));
    SGQA_CUDA_OK(cudaMemcpyAsync(dg + a * row_g, hg + a * row_g, rows * row_g, cudaMemcpyHostToDevice, pp->s_in));
    SGQA_CUDA_OK(copy_rows(qp, rows * P2, hqp + a * P2, T * P2, rows * P2, p.G, cudaMemcpyHostToDevice, pp->s_in));
    SGQA_CUDA_OK(cudaEventRecord(pp->copied[slot], pp->s_in));
    ctx_done = hi;
    // ---- compute (stream) ----
    SGQA_CUDA_OK(cudaStreamWaitEvent(comp, pp->copied[slot], 0));
    if (j == 0 && q_start > 0) {  // blocks of the cached prefix
      s = sgqa_build_block_index(prm, d.k_proxy, ctx_cap, 0, q_start, d.k_blk, d.nb_cap, stream);
      if (s != SGQA_OK) return s;
    }
    s = sgqa_prefill(prm, dq + a * row_q, d.k, d.v, dg + a * row_g, qp, d.k_proxy, ctx_cap, rows, q_start + a, d.k_blk,
                     d.nb_cap, reinterpret_cast<int32_t*>(ws + wl.sel), reinterpret_cast<int32_t*>(ws + wl.cnt),
                     dout + a * row_q, d.lse ? d.lse + a * p.H : nullptr, ws + wl.index, wl.index_bytes, stream);
    if (s != SGQA_OK) return s;
    SGQA_CUDA_OK(cudaEventRecord(pp->done[slot], comp));
    // ---- copy-out (s_out) ----
    SGQA_CUDA_OK(cudaStreamWaitEvent(pp->s_out, pp->done[slot], 0));
    SGQA_CUDA_OK(cudaMemcpyAsync(hout + a * row_q, dout + a * row_q, rows * row_q, cudaMemcpyDeviceToHost, pp->s_out));
    if (h.lse)
      SGQA_CUDA_OK(cudaMemcpyAsync(h.lse + a * p.H, d.lse + a * p.H, rows * p.H * sizeof(float), cudaMemcpyDeviceToHost,
                                   pp->s_out));
  }
  SGQA_CUDA_OK(cudaEventRecord(pp->end, pp->s_out));
  SGQA_CUDA_OK(cudaStreamWaitEvent(comp, pp->end, 0));
  return SGQA_OK;
}

static sgqa_status run_decode(const sgqa_params* prm, int32_t batch, const int64_t* ctx_len, const int64_t* kv_off,
                              const void* q, const void* q_proxy, const void* gate, const void* k_cache,
                              const void* v_cache, const void* k_proxy_cache, void* k_blk_cache, int64_t total,
                              int32_t* sel_idx, int32_t* sel_cnt, void* out, float* lse, void* ws, size_t ws_bytes,
                              sgqa_stream_t stream, bool e4m3) {
  Prm p;
  sgqa_status s = check_params(prm, p);
  if (s != SGQA_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (batch < 1 || batch > kMaxBatch || !ctx_len || !kv_off) return SGQA_ERR_INVALID_ARGUMENT;
  if (!q || !q_proxy || !gate || !k_cache || !v_cache || !k_blk_cache || !sel_idx || !sel_cnt || !out)
    return SGQA_ERR_INVALID_ARGUMENT;
  if (total < 1 || total % p.B != 0) return SGQA_ERR_INVALID_ARGUMENT;
  if ((int64_t)p.G * total > (int64_t)INT32_MAX) return SGQA_ERR_UNSUPPORTED_SHAPE;
  int64_t max_len = 0;
  for (int i = 0; i < batch; ++i) {
    if (ctx_len[i] < 1 || kv_off[i] < 0 || kv_off[i] % p.B != 0 || kv_off[i] + ctx_len[i] > total)
      return SGQA_ERR_INVALID_ARGUMENT;
    max_len = std::max(max_len, ctx_len[i]);
  }
  const size_t need = sgqa_workspace_bytes(prm, SGQA_OP_DECODE, 1, max_len, batch);
  if (!ws || ws_bytes < need) return SGQA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(ws) || !aligned16(q_proxy) || !aligned16(k_blk_cache) || !aligned16(q) || !aligned16(out) ||
      !aligned16(k_cache) || !aligned16(v_cache))
    return SGQA_ERR_INVALID_ARGUMENT;
  const int64_t nb_total = total / p.B;
  const int64_t max_cand = (max_len - 1) / p.B;
  const IndexWs wsl = index_ws_layout(p, batch, max_cand, false);
  const int64_t ld = wsl.ld;
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* scores = reinterpret_cast<float*>(w);
  w += wsl.total;
  const int nsplit = 32;
  float* part_o = reinterpret_cast<float*>(w);
  w += align_up((size_t)p.G * batch * nsplit * 16 * 192 * 4, 256);
  float* part_ml = reinterpret_cast<float*>(w);

  // 1. rebuild the block holding each new token
  if (k_proxy_cache) {
    if (!aligned16(k_proxy_cache)) return SGQA_ERR_INVALID_ARGUMENT;
    K1SeqArgs a1{};
    a1.k_proxy = static_cast<const __nv_bfloat16*>(k_proxy_cache);
    a1.k_blk = k_blk_cache;
    a1.total = total;
    a1.G = p.G;
    a1.P = p.P;
    a1.B = p.B;
    a1.batch = batch;
    for (int i = 0; i < batch; ++i) {
      a1.ctx_len[i] = ctx_len[i];
      a1.kv_off[i] = kv_off[i];
    }
    const int n_vec = p.G * batch * (p.P / 8);
    if (e4m3)
      k1_block_index_seq<true><<<(unsigned)cdiv(n_vec, 256), 256, 0, st>>>(a1);
    else
      k1_block_index_seq<false><<<(unsigned)cdiv(n_vec, 256), 256, 0, st>>>(a1);
    SGQA_CUDA_OK(cudaGetLastError());
  }
  // 2. indexer scores (matrix-vector per sequence and group)
  if (max_cand > 0) {
    K2dArgs a2{};
    a2.qp = static_cast<const __nv_bfloat16*>(q_proxy);
    a2.kblk = k_blk_cache;
    a2.scores = scores;
    a2.ld = ld;
    a2.nb_total = nb_total;
    a2.G = p.G;
    a2.P = p.P;
    a2.B = p.B;
    a2.batch = batch;
    a2.rows_per_cta = e4m3 ? 2048 : 1024;  // the same bytes per CTA with the 1-byte cache
    for (int i = 0; i < batch; ++i) {
      a2.ctx_len[i] = ctx_len[i];
      a2.kv_off[i] = kv_off[i];
    }
    dim3 grid((unsigned)cdiv(max_cand, a2.rows_per_cta), (unsigned)(p.G * batch));
    if (e4m3 && p.P == 192)
      k2d_decode_index_e4m3<true><<<grid, 256, 0, st>>>(a2);
    else if (e4m3)
      k2d_decode_index_e4m3<false><<<grid, 256, 0, st>>>(a2);
    else
      k2d_decode_index<<<grid, 256, 0, st>>>(a2);
    SGQA_CUDA_OK(cudaGetLastError());
  }
  // 3. top-k
  {
    K3Args a3{};
    a3.scores = scores;
    a3.ld = ld;
    a3.rows = batch;
    a3.pos0 = 0;
    a3.out_row0 = 0;
    a3.T_out = batch;
    a3.G = p.G;
    a3.B = p.B;
    a3.k = p.k;
    a3.sel_idx = sel_idx;
    a3.sel_cnt = sel_cnt;
    a3.use_pos = 1;
    for (int i = 0; i < batch; ++i) a3.pos[i] = ctx_len[i] - 1;
    SGQA_CUDA_OK(launch_k3(a3, max_cand, static_cast<uint8_t*>(ws), wsl, st));
  }
  // 4. split-K attention + combine
  {
    K4Args a{};
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.gate = static_cast<const __nv_bfloat16*>(gate);
    a.kc = static_cast<const __nv_bfloat16*>(k_cache);
    a.vc = static_cast<const __nv_bfloat16*>(v_cache);
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    a.sel_idx = sel_idx;
    a.sel_cnt = sel_cnt;
    a.part_o = part_o;
    a.part_ml = part_ml;
    a.rows = batch;
    a.pos0 = 0;
    a.ctx_cap = total;
    a.G = p.G;
    a.Hg = p.Hg;
    a.H = p.H;
    a.B = p.B;
    a.kcap = p.k;
    a.scale_log2 = p.scale * 1.4426950408889634f;
    a.dense = 0;
    a.gate_per_dim = p.gate_per_dim;
    a.nsplit = nsplit;
    a.use_pos = 1;
    a.wait_ns = g_wait_ns;
    for (int i = 0; i < batch; ++i) {
      a.pos[i] = ctx_len[i] - 1;
      a.kv_off[i] = kv_off[i];
    }
    const bool tma = p.B >= 8;
    CUtensorMap tk{}, tv{};
    if (tma) {
      const uint64_t rowsz = (uint64_t)p.G * total;
      if (!make_kv_map(&tk, k_cache, rowsz) || !make_kv_map(&tv, v_cache, rowsz)) return SGQA_ERR_CUDA;
    }
    SGQA_CUDA_OK(launch_k4(a, tk, tv, (int64_t)p.G * batch * nsplit, tma, st));
    K4CombineArgs c{};
    c.part_o = part_o;
    c.part_ml = part_ml;
    c.gate = a.gate;
    c.out = a.out;
    c.lse = lse;
    c.rows = batch;
    c.G = p.G;
    c.Hg = p.Hg;
    c.H = p.H;
    c.nsplit = nsplit;
    c.gate_per_dim = p.gate_per_dim;
    const int64_t warps = (int64_t)p.G * batch * p.Hg * K4C_SLICES;
    k4_combine<<<(unsigned)cdiv(warps * 32, 128), 128, 0, st>>>(c);  // 4 warps per CTA: spread over the SMs
    SGQA_CUDA_OK(cudaGetLastError());
  }
  return SGQA_OK;
}

sgqa_status sgqa_decode(const sgqa_params* prm, int32_t batch, const int64_t* ctx_len, const int64_t* kv_off,
                        const void* q, const void* q_proxy, const void* gate, const void* k_cache, const void* v_cache,
                        const void* k_proxy_cache, void* k_blk_cache, int64_t total, int32_t* sel_idx,
                        int32_t* sel_cnt, void* out, float* lse, void* ws, size_t ws_bytes, sgqa_stream_t stream) {
  return run_decode(prm, batch, ctx_len, kv_off, q, q_proxy, gate, k_cache, v_cache, k_proxy_cache, k_blk_cache,
                    total, sel_idx, sel_cnt, out, lse, ws, ws_bytes, stream, false);
}

sgqa_status sgqa_decode_fp8(const sgqa_params* prm, int32_t batch, const int64_t* ctx_len, const int64_t* kv_off,
                            const void* q, const void* q_proxy, const void* gate, const void* k_cache,
                            const void* v_cache, const void* k_proxy_cache, void* k_blk_cache_e4m3, int64_t total,
                            int32_t* sel_idx, int32_t* sel_cnt, void* out, float* lse, void* ws, size_t ws_bytes,
                            sgqa_stream_t stream) {
  return run_decode(prm, batch, ctx_len, kv_off, q, q_proxy, gate, k_cache, v_cache, k_proxy_cache,
                    k_blk_cache_e4m3, total, sel_idx, sel_cnt, out, lse, ws, ws_bytes, stream, true);
}

}  // extern "C"
