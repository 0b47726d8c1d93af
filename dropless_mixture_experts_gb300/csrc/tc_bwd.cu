// Backward launches of the tensor-core GEMMs (bf16 storage).  The upstream
// gradient rows are first gathered into expert-sorted order (one HBM pass);
// the forward's sorted copy of x is reused.  Then
//   DZ  Z = dy_t W_down[e]^T with the SwiGLU backward and the gate-gradient
//       partials in the epilogue
//   DX  dx_acc[t] += [dA_g | dA_u] [W_gate[e] | W_up[e]]^T
//   DW  dW_down[e] = gH^T dy_t and dW_gate[e] | dW_up[e] = x_t^T [dA_g | dA_u]
//       with K the expert's own rows (ragged), split over CTAs when the
//       output has too few tiles to fill the GPU
// and the dense (shared-expert) instances of each.
#include "gemm_tc.cuh"

namespace moe {
using namespace tcg;

namespace {

int pick_bn(int n) { return n % 256 == 0 ? 256 : n % 128 == 0 ? 128 : 64; }

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
  if (!make_map_sw64(&mp.o1, at<void>(ws, routed ? L.gH : L.gHs), rows, h)) return false;
  if (!make_map_sw64(&mp.i0, routed ? p.a_gate : p.as_gate, rows, h)) return false;
  if (!make_map_sw64(&mp.i1, routed ? p.a_up : p.as_up, rows, h)) return false;
  mp.o2 = mp.o1;
  if (routed) {
    if (!make_map(&mp.a, at<void>(ws, L.dys), L.PPcap, dm, 64, 128)) return false;
    if (!make_map(&mp.b0, p.w_down, (uint64_t)d.experts * h, dm, 64, BN)) return false;
    mp.b1 = mp.b0;
    q.tiles = at<int4>(ws, L.tiles);
    q.ntiles_dev = at<int>(ws, L.ntiles);
    q.rowpair = at<int32_t>(ws, L.rowpair);
    q.top_k = d.top_k;
    q.brow_stride = h;
    q.gates = p.gates;
    q.dg_part = at<float>(ws, L.dg_part);
    q.dg_ld = 2 * h / 64;
    launch_tc<Cfg<A_K_TMA, B_K_TMA, E_DZ, BN, true>>(mp, q, L.MTcap * q.n_nt, "tc_dz", s);
  } else {
    if (!make_map(&mp.a, p.dy, d.tokens, dm, 64, 128)) return false;
    if (!make_map(&mp.b0, p.ws_down, h, dm, 64, BN)) return false;
    mp.b1 = mp.b0;
    q.rows = d.tokens;
    q.n_mt = (int)((d.tokens + 127) / 128);
    launch_tc<Cfg<A_K_TMA, B_K_TMA, E_DZ, BN, false>>(mp, q, (int64_t)q.n_mt * q.n_nt, "tc_dz",
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
  if (routed) {
    if (!make_map(&mp.a, at<void>(ws, L.dA), L.PPcap, 2 * h, 64, 128)) return false;
    if (!make_map(&mp.b0, p.w_gate, (uint64_t)d.experts * dm, h, 64, BN)) return false;
    if (!make_map(&mp.b1, p.w_up, (uint64_t)d.experts * dm, h, 64, BN)) return false;
    q.tiles = at<int4>(ws, L.tiles);
    q.ntiles_dev = at<int>(ws, L.ntiles);
    q.rowpair = at<int32_t>(ws, L.rowpair);
    q.top_k = d.top_k;
    q.brow_stride = dm;
    launch_tc<Cfg<A_K_TMA, B_K_TMA, E_DX, BN, true>>(mp, q, L.MTcap * q.n_nt, "tc_dx", s);
  } else {
    if (!make_map(&mp.a, at<void>(ws, L.dAs), d.tokens, 2 * h, 64, 128)) return false;
    if (!make_map(&mp.b0, p.ws_gate, dm, h, 64, BN)) return false;
    if (!make_map(&mp.b1, p.ws_up, dm, h, 64, BN)) return false;
    q.rows = d.tokens;
    q.n_mt = (int)((d.tokens + 127) / 128);
    launch_tc<Cfg<A_K_TMA, B_K_TMA, E_DX, BN, false>>(mp, q, (int64_t)q.n_mt * q.n_nt, "tc_dx",
                                                       s);
  }
  return true;
}

int splits_for(int64_t tiles, int64_t kblocks_per_tile) {
  const int sms = sm_count();
  int s = 1;
  while (tiles * s < sms && s < 16 && kblocks_per_tile / (s * 2) >= 4) s *= 2;
  return s;
}

// dW_down[e] = sum over the expert's rows of gH_r^T dy_r: A = gH (MN-major:
// rows are K), B = sorted dy (MN-major)
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
  const int64_t rows_per_e = routed ? L.P / E : d.tokens;
  q.splits = splits_for((int64_t)E * q.n_mt * q.n_nt, (rows_per_e + 63) / 64);
  float* out = routed ? p.dw_down : p.dws_down;
  if (q.splits > 1) zero_fill_f32(out, (int64_t)E * h * dm, s);
  q.facc = out;
  if (routed) {
    if (!make_map(&mp.a, at<void>(ws, L.gH), L.PPcap, h, 64, 64)) return false;
    if (!make_map(&mp.b0, at<void>(ws, L.dys), L.PPcap, dm, 64, 64)) return false;
    mp.b1 = mp.b0;
    q.counts = at<int>(ws, L.counts);
    q.poff = at<int>(ws, L.poff);
    launch_tc<Cfg<A_MN_TMA, B_MN_TMA, E_DW, BN, true>>(
        mp, q, (int64_t)E * q.n_mt * q.n_nt * q.splits, "tc_dw_down", s);
  } else {
    if (!make_map(&mp.a, at<void>(ws, L.gHs), d.tokens, h, 64, 64)) return false;
    if (!make_map(&mp.b0, p.dy, d.tokens, dm, 64, 64)) return false;
    mp.b1 = mp.b0;
    q.rows = d.tokens;
    launch_tc<Cfg<A_MN_TMA, B_MN_TMA, E_DW, BN, false>>(
        mp, q, (int64_t)q.n_mt * q.n_nt * q.splits, "tc_dw_down", s);
  }
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
  const int64_t rows_per_e = routed ? L.P / E : d.tokens;
  q.splits = splits_for((int64_t)E * q.n_mt * q.n_nt, (rows_per_e + 63) / 64);
  float* g = routed ? p.dw_gate : p.dws_gate;
  float* u = routed ? p.dw_up : p.dws_up;
  if (q.splits > 1) {
    zero_fill_f32(g, (int64_t)E * dm * h, s);
    zero_fill_f32(u, (int64_t)E * dm * h, s);
  }
  q.facc = g;
  q.facc2 = u;
  if (routed) {
    if (!make_map(&mp.a, at<void>(ws, L.xs), L.PPcap, dm, 64, 64)) return false;
    if (!make_map(&mp.b0, at<void>(ws, L.dA), L.PPcap, 2 * h, 64, 64)) return false;
    mp.b1 = mp.b0;
    q.counts = at<int>(ws, L.counts);
    q.poff = at<int>(ws, L.poff);
    launch_tc<Cfg<A_MN_TMA, B_MN_TMA, E_DW, BN, true>>(
        mp, q, (int64_t)E * q.n_mt * q.n_nt * q.splits, "tc_dw_gateup", s);
  } else {
    if (!make_map(&mp.a, p.x, d.tokens, dm, 64, 64)) return false;
    if (!make_map(&mp.b0, at<void>(ws, L.dAs), d.tokens, 2 * h, 64, 64)) return false;
    mp.b1 = mp.b0;
    q.rows = d.tokens;
    launch_tc<Cfg<A_MN_TMA, B_MN_TMA, E_DW, BN, false>>(
        mp, q, (int64_t)q.n_mt * q.n_nt * q.splits, "tc_dw_gateup", s);
  }
  return true;
}

#define MOE_BN_DISPATCH(fn, n, ...)                         \
  ((n) % 256 == 0 ? fn<256>(__VA_ARGS__)                    \
                  : (n) % 128 == 0 ? fn<128>(__VA_ARGS__) : fn<64>(__VA_ARGS__))

bool backward_one(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws, bool routed,
                  cudaStream_t s) {
  const int h = routed ? d.d_hidden : d.shared_hidden;
  const int dm = d.d_model;
  if (!MOE_BN_DISPATCH(dz, h, d, L, p, ws, routed, s)) return false;
  if (!MOE_BN_DISPATCH(dx, dm, d, L, p, ws, routed, s)) return false;
  if (!MOE_BN_DISPATCH(dw_down, dm, d, L, p, ws, routed, s)) return false;
  return MOE_BN_DISPATCH(dw_gateup, h, d, L, p, ws, routed, s);
}

}  // namespace

int tc_dz_bn(int h) { return pick_bn(h); }

bool tc_backward_gemms(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws,
                       cudaStream_t s) {
  launch_gather_rows(p.dy, at<int32_t>(ws, L.tokrow), at<int>(ws, L.ntiles) + 1,
                     at<void>(ws, L.dys), L.PPcap, (int64_t)d.d_model * 2, s);
  if (d.shared_hidden > 0 && !backward_one(d, L, p, ws, false, s)) return false;
  return backward_one(d, L, p, ws, true, s);
}

}  // namespace moe
