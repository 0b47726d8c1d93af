// Backward launches of the tensor-core GEMMs (bf16 storage).  The upstream
// gradient rows are first copied into expert-sorted order, each scaled by
// its pair's gate (one HBM pass: row r of pair (t, j) holds g_tj dy_t); the
// forward's sorted copy of x and its saved H are reused.  Then
//   DZ  dH = (g dy_t) W_down[e]^T with the SwiGLU backward and the partials
//       of g dg = <dH, H> in the epilogue
//   DX  [dA_g | dA_u] [W_gate[e] | W_up[e]]^T per sorted row
//   DW  dW_down[e] = H^T (g dy_t) and dW_gate[e] | dW_up[e] = x_t^T [dA_g | dA_u]
//       with K the expert's own rows (ragged), split over CTAs when the
//       output has too few tiles to fill the GPU; splits write partials that
//       a second kernel sums in split order (deterministic)
// and the dense (shared-expert) instances of each, plus the router weight
// gradient dW_r = x^T dlogits as a dense DW GEMM.
#include "gemm_tc.cuh"

namespace moe {
using namespace tcg;

namespace {

template <int BN>
bool dz(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws, bool routed,
        cudaStream_t s) {
  const int dm = d.d_model;
  const int h = routed ? d.d_hidden : d.shared_hidden;
  const int64_t rows = routed ? L.PPcap : d.tokens;
  Maps mp;
  Params q;
  q.status = at<int>(ws, L.status);
  q.n_nt = h / BN;
  q.kb_total = dm / 64;
  q.ld_out = h;
  if (!make_map_sw64(&mp.o0, at<void>(ws, routed ? L.dA : L.dAs), rows, 2 * h)) return false;
  if (!make_map_sw64(&mp.i0, routed ? p.a_gate : p.as_gate, rows, h)) return false;
  if (!make_map_sw64(&mp.i1, routed ? p.a_up : p.as_up, rows, h)) return false;
  mp.o1 = mp.o2 = mp.o0;
  // single CTAs: this kernel is bound by its HBM traffic, which CTA pairs
  // do not reduce (their coupled epilogues measured slower)
  constexpr int BROWS = BN;
  if (routed) {
    if (!make_map(&mp.a, at<void>(ws, L.dys), L.PPcap, dm, 64, 128)) return false;
    if (!make_map(&mp.b0, p.w_down, (uint64_t)d.experts * h, dm, 64, BROWS)) return false;
    mp.b1 = mp.b0;
    q.tiles = at<int4>(ws, L.tiles);
    q.ntiles_dev = at<int>(ws, L.ntiles);
    q.rowpair = at<int32_t>(ws, L.rowpair);
    q.top_k = d.top_k;
    q.brow_stride = h;
    q.dg_part = at<float>(ws, L.dg_part);
    q.dg_ld = 2 * h / 64;
    q.dw_tick = at<int>(ws, L.dw_tick);  // zeroed here for the weight gradients
    q.dw_tick_n = (int)L.dw_tick_n;
    launch_tc<Cfg<A_K_TMA, B_K_TMA, E_DZ, BN, true>>(mp, q, L.MTcap * q.n_nt, "tc_dz", s);
  } else {
    if (!make_map(&mp.a, p.dy, d.tokens, dm, 64, 128)) return false;
    if (!make_map(&mp.b0, p.ws_down, h, dm, 64, BROWS)) return false;
    mp.b1 = mp.b0;
    q.rows = d.tokens;
    q.n_mt = (int)((d.tokens + 127) / 128);
    launch_tc<Cfg<A_K_TMA, B_K_TMA, E_DZ, BN, false>>(mp, q, (int64_t)q.n_mt * q.n_nt, "tc_dz_sh",
                                                       s);
  }
  return true;
}

template <int BN>
bool dx(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws, bool routed,
        cudaStream_t s) {
  const int dm = d.d_model;
  const int h = routed ? d.d_hidden : d.shared_hidden;
  Maps mp;
  Params q;
  q.status = at<int>(ws, L.status);
  q.n_nt = dm / BN;
  q.kb_total = 2 * h / 64;
  q.kb_split = h / 64;
  q.ld_out = dm;
  if (!make_map_sw64(&mp.o0, at<void>(ws, routed ? L.dxsort : L.dxs),
                     routed ? L.PPcap : d.tokens, dm))
    return false;
  // CTA pairs where the tensor cores bound this GEMM (the routed rows are
  // then padded to 256): BN / 2 rows of the K-major B per CTA
  const bool pr = BN == 256 && dx_pairs(h, dm);
  const int BROWS = pr ? BN / 2 : BN;
  if (routed) {
    if (!make_map(&mp.a, at<void>(ws, L.dA), L.PPcap, 2 * h, 64, 128)) return false;
    if (!make_map(&mp.b0, p.w_gate, (uint64_t)d.experts * dm, h, 64, BROWS)) return false;
    if (!make_map(&mp.b1, p.w_up, (uint64_t)d.experts * dm, h, 64, BROWS)) return false;
    q.tiles = at<int4>(ws, L.tiles);
    q.ntiles_dev = at<int>(ws, L.ntiles);
    q.rowpair = at<int32_t>(ws, L.rowpair);
    q.top_k = d.top_k;
    q.brow_stride = dm;
    // the router term: the logit gradient of each row's pair times W_r^T[e]
    q.gates = at<float>(ws, L.rowdsel);
    q.wrow = at<void>(ws, L.wrt);
    if constexpr (BN == 256) {
      if (pr) {
        launch_tc<Cfg<A_K_TMA, B_K_TMA, E_DX, BN, true, true>>(mp, q, L.MTcap / 2 * q.n_nt,
                                                               "tc_dx", s);
        return true;
      }
    }
    launch_tc<Cfg<A_K_TMA, B_K_TMA, E_DX, BN, true>>(mp, q, L.MTcap * q.n_nt, "tc_dx", s);
  } else {
    if (!make_map(&mp.a, at<void>(ws, L.dAs), d.tokens, 2 * h, 64, 128)) return false;
    if (!make_map(&mp.b0, p.ws_gate, dm, h, 64, BROWS)) return false;
    if (!make_map(&mp.b1, p.ws_up, dm, h, 64, BROWS)) return false;
    q.rows = d.tokens;
    q.n_mt = (int)((d.tokens + 127) / 128);
    if constexpr (BN == 256) {
      if (pr) {
        launch_tc<Cfg<A_K_TMA, B_K_TMA, E_DX, BN, false, true>>(
            mp, q, (int64_t)(q.n_mt + 1) / 2 * q.n_nt, "tc_dx_sh", s);
        return true;
      }
    }
    launch_tc<Cfg<A_K_TMA, B_K_TMA, E_DX, BN, false>>(mp, q, (int64_t)q.n_mt * q.n_nt,
                                                       "tc_dx_sh", s);
  }
  return true;
}

// K splits of a weight-gradient GEMM: split only while the tiles fill less
// than half of the GPU (a split costs a partial write and a reduction), at
// least four 64-row K blocks per split, never beyond the workspace's bound
int splits_for(int64_t tiles, int64_t kblocks_per_tile) {
  const int sms = sm_count();  // the device's (not the launch limit's): fixed results
  const int cap = split_bound(tiles);
  int s = 1;
  while (tiles * s * 2 <= sms && s < cap && kblocks_per_tile / (s * 2) >= 4) s *= 2;
  return s;
}

// Shared tail of the DW launches: partials when split, the fixed-order
// reduction afterwards.
// (the shared expert's weight gradients: partials in a region of their own)
void set_splits(Params& q, const Layout& L, void* ws, int64_t kblocks, bool always_partials) {
  q.splits = splits_for((int64_t)q.experts * q.n_mt * q.n_nt, kblocks);
  if (q.splits > 1 || always_partials) q.part = at<float>(ws, L.dwpart_sh);
}

void reduce_splits(const Params& q, float* out0, float* out1, cudaStream_t s) {
  if (!q.part) return;
  launch_split_reduce(q.part, q.splits, (int64_t)q.experts * q.M, q.ldp, q.N, q.hsplit, out0,
                      out1, s);
}

// Routed DW launches: K chunks per expert from the device-side schedule
// (balanced against the row counts; the last chunk of a tile to finish sums
// the chunks' partials); the work units are bounded by
// (E + grid / tiles_per_expert + 1) chunks.
// With CTA pairs (pair = true) a unit covers two row tiles and the grid
// holds half as many units.
int64_t set_chunks(Params& q, const Layout& L, void* ws, bool pair = false) {
  q.part = at<float>(ws, L.dwpart);
  q.dw_tick = at<int>(ws, L.dw_tick);
  const int64_t tpe = (int64_t)(pair ? q.n_mt / 2 : q.n_mt) * q.n_nt;
  const int64_t grid = pair ? sm_count() / 2 : sm_count();
  q.sched_units = (int)grid;  // the whole device's units, whatever the launch's SM limit
  return (q.experts + grid / tpe + 1) * tpe;
}

// Routed weight-gradient launches run as CTA pairs (256 output rows per
// unit) when the output rows split into 256-row units and BN = 256.

// A dense (shared-expert) weight-gradient launch with M output rows: CTA
// pairs when the rows split into 256-row units and BN = 256.
template <int BN>
void launch_dense_dw(const Maps& mp, const Params& q, int M, const char* name, cudaStream_t s) {
  if constexpr (BN == 256) {
    if (M % 256 == 0) {
      launch_tc<Cfg<A_MN_TMA, B_MN_TMA, E_DW, BN, false, true>>(
          mp, q, (int64_t)(q.n_mt / 2) * q.n_nt * q.splits, name, s);
      return;
    }
  }
  launch_tc<Cfg<A_MN_TMA, B_MN_TMA, E_DW, BN, false>>(mp, q, (int64_t)q.n_mt * q.n_nt * q.splits,
                                                      name, s);
}

// dW_down[e] = sum over the expert's rows of H_r^T (g dy)_r: A = the
// forward's saved H (MN-major: rows are K), B = the gate-scaled sorted dy
// (MN-major); the shared expert: Hs^T dy
template <int BN>
bool dw_down(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws, bool routed,
             cudaStream_t s) {
  const int dm = d.d_model;
  const int h = routed ? d.d_hidden : d.shared_hidden;
  const int E = routed ? d.experts : 1;
  Maps mp;
  Params q;
  q.status = at<int>(ws, L.status);
  q.M = h;
  q.N = dm;
  q.n_mt = (h + 127) / 128;
  q.n_nt = dm / BN;
  q.experts = E;
  q.ldp = dm;
  float* out = routed ? p.dw_down : p.dws_down;
  q.facc = out;
  if (routed) {
    if (!make_map(&mp.a, p.h_buf, L.PPcap, h, 64, 64)) return false;
    if (!make_map(&mp.b0, at<void>(ws, L.dys), L.PPcap, dm, 64, 64)) return false;
    mp.b1 = mp.b0;
    q.counts = at<int>(ws, L.counts);
    q.poff = at<int>(ws, L.poff);
    if constexpr (BN == 256) {
      if (h % 256 == 0) {
        launch_tc<Cfg<A_MN_TMA, B_MN_TMA, E_DW, BN, true, true>>(
            mp, q, set_chunks(q, L, ws, true), "tc_dw_down", s);
        return true;
      }
    }
    launch_tc<Cfg<A_MN_TMA, B_MN_TMA, E_DW, BN, true>>(mp, q, set_chunks(q, L, ws), "tc_dw_down", s);
    return true;
  } else {
    set_splits(q, L, ws, (d.tokens + 63) / 64, false);
    if (!make_map(&mp.a, p.hs_buf, d.tokens, h, 64, 64)) return false;
    if (!make_map(&mp.b0, p.dy, d.tokens, dm, 64, 64)) return false;
    mp.b1 = mp.b0;
    q.rows = d.tokens;
    launch_dense_dw<BN>(mp, q, h, "tc_dw_down_sh", s);
  }
  reduce_splits(q, out, nullptr, s);
  return true;
}

// dW_gate[e] | dW_up[e] = sum over the expert's rows of x_r^T [dA_g | dA_u]:
// A = sorted x (MN-major), B = dA (MN-major)
template <int BN>
bool dw_gateup(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws, bool routed,
               cudaStream_t s) {
  const int dm = d.d_model;
  const int h = routed ? d.d_hidden : d.shared_hidden;
  const int E = routed ? d.experts : 1;
  Maps mp;
  Params q;
  q.status = at<int>(ws, L.status);
  q.M = dm;
  q.N = 2 * h;
  q.hsplit = h;
  q.n_mt = (dm + 127) / 128;
  q.n_nt = 2 * h / BN;
  q.experts = E;
  q.ldp = 2 * h;
  float* g = routed ? p.dw_gate : p.dws_gate;
  float* u = routed ? p.dw_up : p.dws_up;
  q.facc = g;
  q.facc2 = u;
  if (routed) {
    if (!make_map(&mp.a, at<void>(ws, L.xs), L.PPcap, dm, 64, 64)) return false;
    if (!make_map(&mp.b0, at<void>(ws, L.dA), L.PPcap, 2 * h, 64, 64)) return false;
    mp.b1 = mp.b0;
    q.counts = at<int>(ws, L.counts);
    q.poff = at<int>(ws, L.poff);
    if constexpr (BN == 256) {
      if (dm % 256 == 0) {
        launch_tc<Cfg<A_MN_TMA, B_MN_TMA, E_DW, BN, true, true>>(
            mp, q, set_chunks(q, L, ws, true), "tc_dw_gateup", s);
        return true;
      }
    }
    launch_tc<Cfg<A_MN_TMA, B_MN_TMA, E_DW, BN, true>>(mp, q, set_chunks(q, L, ws), "tc_dw_gateup", s);
    return true;
  } else {
    set_splits(q, L, ws, (d.tokens + 63) / 64, false);
    if (!make_map(&mp.a, p.x, d.tokens, dm, 64, 64)) return false;
    if (!make_map(&mp.b0, at<void>(ws, L.dAs), d.tokens, 2 * h, 64, 64)) return false;
    mp.b1 = mp.b0;
    q.rows = d.tokens;
    launch_dense_dw<BN>(mp, q, dm, "tc_dw_gateup_sh", s);
  }
  reduce_splits(q, g, u, s);
  return true;
}

#define MOE_BN_DISPATCH(fn, n, ...)                         \
  ((n) % 256 == 0 ? fn<256>(__VA_ARGS__)                    \
                  : (n) % 128 == 0 ? fn<128>(__VA_ARGS__) : fn<64>(__VA_ARGS__))

// parts: 1 = dZ, 2 = dX and the weight gradients, 3 = both
bool backward_one(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws, bool routed,
                  cudaStream_t s, int parts = 3) {
  const int h = routed ? d.d_hidden : d.shared_hidden;
  const int dm = d.d_model;
  if ((parts & 1) && !MOE_BN_DISPATCH(dz, h, d, L, p, ws, routed, s)) return false;
  if (!(parts & 2)) return true;
  if (!MOE_BN_DISPATCH(dx, dm, d, L, p, ws, routed, s)) return false;
  if (!MOE_BN_DISPATCH(dw_down, dm, d, L, p, ws, routed, s)) return false;
  return MOE_BN_DISPATCH(dw_gateup, h, d, L, p, ws, routed, s);
}

}  // namespace

int tc_dz_bn(int h) { return pick_bn(h); }

bool tc_backward_routed_dz(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws,
                           cudaStream_t s) {
  launch_scatter_rows(d, L, p.dy, at<void>(ws, L.dys), ws, s, p.gates, nullptr);
  return backward_one(d, L, p, ws, true, s, 1);
}

bool tc_backward_routed_rest(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws,
                             cudaStream_t s) {
  return backward_one(d, L, p, ws, true, s, 2);
}

bool tc_backward_shared(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws,
                        cudaStream_t s) {
  return d.shared_hidden == 0 || backward_one(d, L, p, ws, false, s);
}

bool tc_router_dw_supported(const moe_dims& d) {
  return d.dtype == MOE_BF16 && d.experts % 8 == 0 && d.experts <= 64;
}

// dW_r [d, E] = x^T dl with dl the dense bf16 router-logit gradient [T, E]
// (zero off the selected experts): a dense DW GEMM, M = d, N = E (one
// 64-column tile, the columns past E read as zero), K = the tokens, split
// over CTAs into partials reduced in split order.
bool tc_router_dw(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws,
                  cudaStream_t s) {
  Maps mp;
  Params q;
  q.status = at<int>(ws, L.status);
  q.M = d.d_model;
  q.N = d.experts;
  q.n_mt = (d.d_model + 127) / 128;
  q.n_nt = 1;
  q.experts = 1;
  q.rows = d.tokens;
  // splits of at least four 64-row K blocks each
  const int64_t kblocks = (d.tokens + 63) / 64;
  q.splits = router_dw_split_bound(q.n_mt);
  while (q.splits > 1 && kblocks / q.splits < 4) q.splits /= 2;
  q.part = at<float>(ws, L.dwpart);
  q.ldp = 64;
  q.facc = p.dw_router;
  if (!make_map(&mp.a, p.x, d.tokens, d.d_model, 64, 64)) return false;
  if (!make_map(&mp.b0, at<void>(ws, L.dl), d.tokens, d.experts, 64, 64)) return false;
  mp.b1 = mp.b0;
  launch_tc<Cfg<A_MN_TMA, B_MN_TMA, E_DW, 64, false>>(mp, q, (int64_t)q.n_mt * q.splits,
                                                       "tc_router_dw", s);
  reduce_splits(q, p.dw_router, nullptr, s);
  return true;
}

}  // namespace moe
