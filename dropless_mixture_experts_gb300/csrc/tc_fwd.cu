// Forward launches of the tensor-core GEMMs (bf16 storage; the down
// projection runs as CTA pairs of 256 rows where the tensor cores bound it,
// the store-heavy gate/up projection on single CTAs): the token rows
// are first gathered into expert-sorted order (one HBM pass), then
//   gate/up projection of the sorted rows with SwiGLU in the epilogue, and
//   the down projection with the gate-weighted combine in the epilogue;
// plus the dense shared expert.
#include "gemm_tc.cuh"

namespace moe {
using namespace tcg;

namespace {

template <int BN>
bool gateup(const moe_dims& d, const Layout& L, int mode, const LayerPtrs& p, void* ws,
            bool routed, cudaStream_t s) {
  const int dm = d.d_model;
  const int h = routed ? d.d_hidden : d.shared_hidden;
  const int64_t rows = routed ? L.PPcap : d.tokens;
  const bool save = mode == MOE_SAVE_FOR_BWD;
  Maps mp;
  Params q;
  q.status = at<int>(ws, L.status);
  q.n_nt = h / (BN / 2);
  q.kb_total = dm / 64;
  q.ld_out = h;
  q.save = save ? 1 : 0;
  void* H = routed ? p.h_buf : p.hs_buf;
  void* AG = routed ? p.a_gate : p.as_gate;
  void* AU = routed ? p.a_up : p.as_up;
  q.rows_out = rows;  // the epilogue's load/store-unit copies go straight to these
  q.dst0 = H;
  q.dst1 = AG;
  q.dst2 = AU;
  if (routed) {
    if (!make_map(&mp.a, at<void>(ws, L.xs), L.PPcap, dm, 64, 128)) return false;
    if (!make_map(&mp.b0, p.w_gate, (uint64_t)d.experts * dm, h, 64, 64)) return false;
    if (!make_map(&mp.b1, p.w_up, (uint64_t)d.experts * dm, h, 64, 64)) return false;
    q.tiles = at<int4>(ws, L.tiles);
    q.ntiles_dev = at<int>(ws, L.ntiles);
    q.rowpair = at<int32_t>(ws, L.rowpair);
    q.top_k = d.top_k;
    q.brow_stride = dm;
    launch_tc<Cfg<A_K_TMA, B_MN_TMA, E_GU, BN, true>>(mp, q, L.MTcap * q.n_nt, "tc_gateup", s);
  } else {
    if (!make_map(&mp.a, p.x, d.tokens, dm, 64, 128)) return false;
    if (!make_map(&mp.b0, p.ws_gate, dm, h, 64, 64)) return false;
    if (!make_map(&mp.b1, p.ws_up, dm, h, 64, 64)) return false;
    q.rows = d.tokens;
    q.n_mt = (int)((d.tokens + 127) / 128);
    launch_tc<Cfg<A_K_TMA, B_MN_TMA, E_GU, BN, false>>(mp, q, (int64_t)q.n_mt * q.n_nt,
                                                        "tc_gateup_sh", s);
  }
  return true;
}

template <int BN>
bool down(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws, bool routed,
          cudaStream_t s) {
  const int dm = d.d_model;
  const int h = routed ? d.d_hidden : d.shared_hidden;
  Maps mp;
  Params q;
  q.status = at<int>(ws, L.status);
  q.n_nt = dm / BN;
  q.kb_total = h / 64;
  q.ld_out = dm;
  if (!make_map_sw64(&mp.o0, at<void>(ws, routed ? L.osort : L.ys), routed ? L.PPcap : d.tokens,
                     dm))
    return false;
  if (routed) {
    if (!make_map(&mp.a, p.h_buf, L.PPcap, h, 64, 128)) return false;
    if (!make_map(&mp.b0, p.w_down, (uint64_t)d.experts * h, dm, 64, 64)) return false;
    mp.b1 = mp.b0;
    q.tiles = at<int4>(ws, L.tiles);
    q.ntiles_dev = at<int>(ws, L.ntiles);
    q.rowpair = at<int32_t>(ws, L.rowpair);
    q.top_k = d.top_k;
    q.brow_stride = h;
    q.gates = at<float>(ws, L.rowgate);
    if constexpr (BN == 256) {
      if (down_pairs(h, dm)) {  // the expert rows are then padded to 256
        launch_tc<Cfg<A_K_TMA, B_MN_TMA, E_DOWN, BN, true, true>>(mp, q, L.MTcap / 2 * q.n_nt,
                                                                  "tc_down", s);
        return true;
      }
    }
    launch_tc<Cfg<A_K_TMA, B_MN_TMA, E_DOWN, BN, true>>(mp, q, L.MTcap * q.n_nt, "tc_down", s);
  } else {
    if (!make_map(&mp.a, p.hs_buf, d.tokens, h, 64, 128)) return false;
    if (!make_map(&mp.b0, p.ws_down, h, dm, 64, 64)) return false;
    mp.b1 = mp.b0;
    q.rows = d.tokens;
    q.n_mt = (int)((d.tokens + 127) / 128);
    if constexpr (BN == 256) {
      if (down_pairs(h, dm)) {
        launch_tc<Cfg<A_K_TMA, B_MN_TMA, E_DOWN, BN, false, true>>(
            mp, q, (int64_t)(q.n_mt + 1) / 2 * q.n_nt, "tc_down_sh", s);
        return true;
      }
    }
    launch_tc<Cfg<A_K_TMA, B_MN_TMA, E_DOWN, BN, false>>(mp, q, (int64_t)q.n_mt * q.n_nt,
                                                          "tc_down_sh", s);
  }
  return true;
}

bool gateup_any(const moe_dims& d, const Layout& L, int mode, const LayerPtrs& p, void* ws,
                bool routed, cudaStream_t s) {
  const int h = routed ? d.d_hidden : d.shared_hidden;
  return h % 128 == 0 ? gateup<256>(d, L, mode, p, ws, routed, s)
                      : gateup<128>(d, L, mode, p, ws, routed, s);
}

bool down_any(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws, bool routed,
              cudaStream_t s) {
  const int n = d.d_model;
  if (n % 256 == 0) return down<256>(d, L, p, ws, routed, s);
  if (n % 128 == 0) return down<128>(d, L, p, ws, routed, s);
  return down<64>(d, L, p, ws, routed, s);
}

}  // namespace

bool tc_router_supported(const moe_dims& d) {
  return d.dtype == MOE_BF16 && d.experts % 8 == 0 && d.experts <= 64 && d.d_model % 64 == 0;
}

// logits = x W_r on the tensor cores (x: K-major rows; W_r [d, E]: MN-major
// tile of 64 columns, the columns past E read as zero), top-k and softmax in
// the epilogue
bool tc_router(const moe_dims& d, const Layout& L, const void* x, const void* w_router,
               const float* bias, float* logits_out, int32_t* idx, float* gates, void* ws,
               cudaStream_t s) {
  Maps mp;
  Params q;
  q.status = at<int>(ws, L.status);
  if (!make_map(&mp.a, x, d.tokens, d.d_model, 64, 128)) return false;
  if (!make_map(&mp.b0, w_router, d.d_model, d.experts, 64, 64)) return false;
  mp.b1 = mp.b0;
  q.rows = d.tokens;
  q.n_mt = (int)((d.tokens + 127) / 128);
  q.n_nt = 1;
  q.kb_total = d.d_model / 64;
  q.N = d.experts;
  q.top_k = d.top_k;
  q.out0 = idx;
  q.out1 = gates;
  q.facc = logits_out;
  q.gates = bias;  // the router's epilogue reads this as its logit offsets
  // narrow routers keep W_r resident in shared memory (one operand stream
  // per stage instead of two; measured faster at E = 8, not at E = 64,
  // whose epilogue's top-8 selection bounds it)
  if (d.experts <= 32 && d.d_model <= 64 * 10)
    launch_tc<Cfg<A_K_TMA, B_MN_RES, E_ROUTER, 64, false>>(mp, q, q.n_mt, "tc_router", s);
  else
    launch_tc<Cfg<A_K_TMA, B_MN_TMA, E_ROUTER, 64, false>>(mp, q, q.n_mt, "tc_router", s);
  return true;
}

bool tc_grouped_fwd(const moe_dims& d, const Layout& L, int mode, const LayerPtrs& p, void* ws,
                    cudaStream_t s) {
  launch_scatter_rows(d, L, p.x, at<void>(ws, L.xs), ws, s, p.gates, at<float>(ws, L.rowgate));
  if (!gateup_any(d, L, mode, p, ws, true, s)) return false;
  return down_any(d, L, p, ws, true, s);
}

bool tc_shared_fwd(const moe_dims& d, const Layout& L, int mode, const LayerPtrs& p, void* ws,
                   cudaStream_t s) {
  if (!gateup_any(d, L, mode, p, ws, false, s)) return false;
  return down_any(d, L, p, ws, false, s);
}

}  // namespace moe
