// Shared definitions of the CUDA side of the MoE layer: element access for
// the two storage types, the workspace layout and the device status word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/moe.h"

namespace moe {

constexpr int kRowPad = 256;      // the largest expert row padding (row_pad: 128 or 256)
constexpr int kTileRows = 128;    // rows of one tile-list entry
constexpr int kPermRounds = 16;   // 32-pair rounds per warp chunk in the counting sort
constexpr int kPermChunk = 32 * kPermRounds;
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 32;
constexpr int kLossBlocks = 2048;  // fixed partial count of the loss reduction
constexpr int kRouterBwdRanges = 608;  // max token ranges of the router-weight gradient partials
constexpr int kRouterBwdSmem = 200 * 1024;  // router backward: W_r^T + dW_r partial in shared memory
constexpr int kSimtMaxSplit = 8;  // most K chunks of a strict-float32 weight-gradient GEMM
// most (output tile x chunk) blocks of a chunked strict-float32 weight
// gradient: bounds its partials to this many 128 x 128 float tiles (256 MiB)
constexpr int kSimtChunkTiles = 4096;

// ---- element access ---------------------------------------------------------
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

__device__ __forceinline__ float sigmoidf_(float a) { return 1.0f / (1.0f + expf(-a)); }

// ---- routing selection ------------------------------------------------------
// The total order of the top-k selection: larger logit first, the lower
// expert index on equal logits (+0.0 == -0.0).
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// exp(sel - top) for float32 logits.  The gap sel - top is split exactly
// into its float rounding (head) and the rounding error (tail) with Knuth's
// TwoSum, so expf(head) * (1 + tail) is accurate to float even for large
// gaps, where a float32 difference alone would lose the tail (no float64
// arithmetic, which is slow on this part).
__device__ __forceinline__ float gate_exp(float sel, float top) {
  const float b = -top;
  const float head = sel + b;
  const float bv = head - sel;
  const float av = head - bv;
  const float tail = (sel - av) + (b - bv);
  return expf(head) * (1.f + tail);
}

// ---- device status word ---------------------------------------------------
// status[0] = first error code (moe_status), status[1] = detail word.
__device__ __forceinline__ void report_error(int* status, int code, int detail) {
  if (atomicCAS(status, 0, code) == 0) status[1] = detail;
}

// ---- workspace layout -------------------------------------------------------
struct Layout {
  size_t status, warp_counts, warp_base, counts, poff, rowpair, tiles, ntiles,
      loss_part, loss_tick, logits;
  size_t xs;       // expert-sorted copy of the token rows [padded rows, d]
  size_t pairrow;  // pair -> padded row [P]
  size_t osort;    // gate-weighted expert output per sorted row [padded rows, d]
  size_t rowgate;  // the gate of each sorted row's pair, 0 on padding [padded rows] (bf16 path)
  size_t ys;       // shared-expert output [T, d]
  size_t dg_part, dA, dxsort, dxs, dAs, dys, dsel, dwr_part;
  size_t rowdsel;  // the router logit gradient of each sorted row's pair [padded rows] (bf16 path)
  size_t gH, gHs;  // gate * H for the W_down gradients (float32 path only)
  size_t dl;      // dense router-logit gradient [T, E] (bf16 path)
  size_t wrt;     // W_r^T [E, d]
  size_t dwpart;  // per-split / per-chunk partials of the routed and router weight-gradient GEMMs
  size_t dwpart_sh;  // per-split partials of the shared expert's weight gradients (a region of
                     // its own: the shared expert's backward may run beside the routed one)
  size_t dw_tick;    // the routed weight gradients' per-tile chunk tickets [dw_tick_n]
  int64_t dw_tick_n;
  size_t total;
  int64_t P, PPcap, MTcap, NWc;
  int elem;  // bytes per storage element
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Column tile of a grouped GEMM with n output columns.
inline int pick_bn(int n) { return n % 256 == 0 ? 256 : n % 128 == 0 ? 128 : 64; }

// CTA pairs (tcgen05 cta_group::2, 256 x 256 tiles over two SMs) halve the
// B operand bytes each SM receives per FLOP.  They pay where the tensor
// cores bound the GEMM and the column tile is 256 wide:
//   a row GEMM with K-deep rows and N output columns moves a row of A in
//   and a row of D out per 2*K*N FLOPs, K*N/(K+N) FLOPs per byte; at 300 and
//   above it is past the ratio of the bf16 tensor peak to the HBM rate
//   (about 280 on GB300), below it is HBM-bound and pairs measured slower;
//   the weight-gradient GEMMs pair whenever BN = 256 and M splits into
//   256-row units.
inline bool row_gemm_pairs(int64_t K, int64_t N) {
  return pick_bn((int)N) == 256 && K * N >= 300 * (K + N);
}
// the down projection (K = h) and the input-gradient GEMM (K = 2h), N = d
inline bool down_pairs(int64_t h, int64_t dm) { return row_gemm_pairs(h, dm); }
inline bool dx_pairs(int64_t h, int64_t dm) { return row_gemm_pairs(2 * h, dm); }

// Expert row padding: 256 when a routed row GEMM runs as CTA pairs (a pair
// takes two 128-row tiles of one expert), else 128.
inline int row_pad(const moe_dims& d) {
  return d.dtype == MOE_BF16 && (down_pairs(d.d_hidden, d.d_model) ||
                                 dx_pairs(d.d_hidden, d.d_model))
             ? 256
             : 128;
}

inline int64_t padded_rows(const moe_dims& d) {
  const int pad = row_pad(d);
  int64_t P = d.tokens * (int64_t)d.top_k;
  int64_t cap = P + (int64_t)d.experts * (pad - 1);
  return (cap + pad - 1) / pad * pad;
}

// Most K splits a weight-gradient GEMM with `tiles` output tiles may use
// (a power of two; 1 when the tiles alone fill any GPU of <= 256 SMs).
inline int split_bound(int64_t tiles) {
  int s = 1;
  while (s < 16 && tiles * s < 256) s *= 2;
  return s;
}

// K splits of the router-weight gradient x^T dlogits, a d x E product over
// every token: enough splits that its few output tiles fill the GPU twice
// over (a power of two, at most 64).
inline int router_dw_split_bound(int64_t tiles) {
  int s = 1;
  while (s < 64 && tiles * s * 2 <= 512) s *= 2;
  return s;
}

inline Layout make_layout(const moe_dims& d, int mode) {
  Layout L{};
  L.elem = d.dtype == MOE_BF16 ? 2 : 4;
  L.P = d.tokens * (int64_t)d.top_k;
  L.PPcap = padded_rows(d);
  L.MTcap = L.PPcap / kTileRows;
  L.NWc = (L.P + kPermChunk - 1) / kPermChunk;
  const int64_t E = d.experts, T = d.tokens, h = d.d_hidden, dm = d.d_model,
                hs = d.shared_hidden;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + (bytes ? bytes : 1), 256);
    return at;
  };
  L.status = take(64);
  L.warp_counts = take(sizeof(int) * L.NWc * E);
  L.warp_base = take(sizeof(int) * L.NWc * E);
  L.counts = take(sizeof(int) * E);
  L.poff = take(sizeof(int) * (E + 1));
  L.rowpair = take(sizeof(int) * L.PPcap);
  L.tiles = take(sizeof(int4) * L.MTcap);
  L.ntiles = take(sizeof(int) * 4);
  L.loss_part = take(sizeof(float) * kLossBlocks);
  L.loss_tick = take(sizeof(int));  // the combine's blocks done (reset by its last block)
  L.logits = take(sizeof(float) * T * E);
  L.xs = take((size_t)L.elem * L.PPcap * dm);
  L.pairrow = take(sizeof(int) * L.P);
  L.osort = take((size_t)L.elem * L.PPcap * dm);
  L.rowgate = take(sizeof(float) * L.PPcap);
  L.ys = take((size_t)L.elem * (hs > 0 ? T : 0) * dm);
  if (mode == MOE_SAVE_FOR_BWD) {
    L.dg_part = take(sizeof(float) * L.P * 2 * (h / 64));
    L.dA = take((size_t)L.elem * L.PPcap * 2 * h);
    // the bf16 path's W_down gradients read the forward's saved H instead
    const bool gh = d.dtype != MOE_BF16;
    L.gH = take(gh ? (size_t)L.elem * L.PPcap * h : 0);
    L.dxsort = take((size_t)L.elem * L.PPcap * dm);
    L.dxs = take((size_t)L.elem * (hs > 0 ? T : 0) * dm);
    L.dAs = take((size_t)L.elem * T * 2 * hs);
    L.gHs = take(gh ? (size_t)L.elem * T * hs : 0);
    L.dys = take((size_t)L.elem * L.PPcap * dm);
    L.dsel = take(sizeof(float) * T * d.top_k);
    L.rowdsel = take(sizeof(float) * L.PPcap);
    L.dwr_part = take(sizeof(float) * kRouterBwdRanges * dm * E);
    L.dl = take((size_t)2 * T * E);
    L.wrt = take((size_t)L.elem * E * dm);
    // partials of the split weight-gradient GEMMs (one launch at a time)
    auto need = [&](int64_t experts, int64_t M, int64_t N, int bn, bool always) -> int64_t {
      const int64_t ldp = (N + bn - 1) / bn * bn;
      const int64_t tiles = experts * ((M + 127) / 128) * (ldp / bn);
      const int s = split_bound(tiles);
      return (s > 1 || always) ? s * experts * M * ldp : 0;
    };
    // routed weight gradients: per-chunk partials; the device-side schedule
    // takes at most E + grid / tiles_per_expert + 1 chunks (grid <= 256 SMs)
    auto chunked = [&](int64_t M, int64_t N, int bn) -> int64_t {
      const int64_t tpe = ((M + 127) / 128) * (N / bn);
      return (E + 256 / tpe + 1) * M * N;
    };
    int64_t pf = chunked(h, dm, pick_bn((int)dm));
    pf = std::max(pf, chunked(dm, 2 * h, pick_bn((int)h)));
    int64_t pfs = 0;
    if (hs > 0) {
      pfs = std::max(pfs, need(1, hs, dm, pick_bn((int)dm), false));
      pfs = std::max(pfs, need(1, dm, 2 * hs, pick_bn((int)hs), false));
    }
    pf = std::max(pf, (int64_t)router_dw_split_bound((dm + 127) / 128) * dm * 64);
    if (d.dtype != MOE_BF16) {
      // the strict-float32 weight gradients' K-chunk partials [chunk][E * M][N]
      // (chunks only where tiles x chunks <= kSimtChunkTiles)
      const int64_t cap = (int64_t)kSimtChunkTiles * 128 * 128;
      pf = std::max(pf, std::min(cap, (int64_t)kSimtMaxSplit * E * std::max(h * dm, dm * 2 * h)));
      if (hs > 0)
        pfs = std::max(pfs, std::min(cap, (int64_t)kSimtMaxSplit * std::max(hs * dm, dm * 2 * hs)));
    }
    L.dwpart = take(sizeof(float) * pf);
    L.dwpart_sh = take(sizeof(float) * pfs);
    L.dw_tick_n = std::max(E * ((h + 127) / 128) * (dm / pick_bn((int)dm)),
                           E * ((dm + 127) / 128) * (2 * h / pick_bn((int)h)));
    L.dw_tick = take(sizeof(int) * L.dw_tick_n);
  }
  L.total = o;
  return L;
}

template <typename T>
__host__ __device__ __forceinline__ T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(reinterpret_cast<char*>(base) + off);
}

// One 128-row tile of the expert-sorted (padded) rows.
// x = expert, y = first padded row, z = number of real rows (1..128), w = unused.
using TileEntry = int4;

}  // namespace moe
