// The C ABI (include/moe.h): argument validation and the launch sequence of
// each call.  Nothing here computes; every step runs in the kernels.
#include <initializer_list>

#include "kernels.cuh"

using namespace moe;

namespace {

bool dims_ok(const moe_dims* d) {
  if (!d) return false;
  if (d->tokens < 0 || d->tokens > (int64_t(1) << 31) / 64) return false;
  if (d->experts < 1 || d->experts > kMaxExperts) return false;
  if (d->top_k < 1 || d->top_k > d->experts || d->top_k > kMaxTopK) return false;
  if (d->d_model < 64 || d->d_hidden < 64 || d->shared_hidden < 0) return false;
  if (d->dtype != MOE_F32 && d->dtype != MOE_BF16) return false;
  if (d->capacity < 0) return false;
  if (d->tokens * (int64_t)d->top_k + (int64_t)d->experts * kRowPad >= (int64_t(1) << 31))
    return false;
  return true;
}

moe_status shape_supported(const moe_dims* d) {
  if (d->d_model % 64 || d->d_hidden % 64 || d->shared_hidden % 64) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status check_ws(const moe_dims* d, int mode, const void* ws, size_t bytes) {
  if (!ws) return MOE_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) % 256) return MOE_ERR_WORKSPACE;
  if (bytes < make_layout(*d, mode).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

// Row data (activations, weights, their gradients) moves in 16-byte vectors
// and bulk copies: every such array must start on a 16-byte boundary.
bool aligned16(std::initializer_list<const void*> ptrs) {
  for (const void* q : ptrs)
    if (reinterpret_cast<uintptr_t>(q) % 16) return false;
  return true;
}

moe_status cuda_status() {
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

#define MOE_TRY(expr)                 \
  do {                                \
    moe_status _s = (expr);           \
    if (_s != MOE_OK) return _s;      \
  } while (0)

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MOE_ERR_CUDA: return "CUDA call failed";
    case MOE_ERR_TIMEOUT: return "device: a bounded wait ran out";
    case MOE_ERR_DEVICE_CHECK: return "device: an index check failed";
  }
  return "unknown status";
}

moe_status moe_workspace_bytes(const moe_dims* dims, int mode, size_t* bytes) {
  if (!dims_ok(dims) || !bytes) return MOE_ERR_INVALID_ARG;
  if (mode != MOE_FWD_ONLY && mode != MOE_SAVE_FOR_BWD) return MOE_ERR_INVALID_ARG;
  *bytes = make_layout(*dims, mode).total;
  return MOE_OK;
}

moe_status moe_padded_rows(const moe_dims* dims, int64_t* rows) {
  if (!dims_ok(dims) || !rows) return MOE_ERR_INVALID_ARG;
  *rows = padded_rows(*dims);
  return MOE_OK;
}

moe_status moe_route(const moe_dims* dims, const void* x, const void* w_router,
                     const float* router_bias, const float* logits_in, float* logits_out,
                     int32_t* topk_idx, float* gates, void* workspace, size_t workspace_bytes,
                     cudaStream_t stream) {
  if (!dims_ok(dims)) return MOE_ERR_INVALID_ARG;
  if (dims->tokens > 0) {
    if (!topk_idx || !gates) return MOE_ERR_INVALID_ARG;
    if (!logits_in && (!x || !w_router)) return MOE_ERR_INVALID_ARG;
  }
  if (!aligned16({x, w_router})) return MOE_ERR_INVALID_ARG;
  MOE_TRY(shape_supported(dims));
  MOE_TRY(check_ws(dims, MOE_FWD_ONLY, workspace, workspace_bytes));
  const Layout L = make_layout(*dims, MOE_FWD_ONLY);
  const int64_t T = dims->tokens;
  const int E = dims->experts;
  if (T == 0) return MOE_OK;
  const float* logits = logits_in;
  if (!logits_in) {
    if (tc_router_supported(*dims)) {
      if (!tc_router(*dims, L, x, w_router, router_bias, logits_out, topk_idx, gates, workspace,
                     stream))
        return MOE_ERR_CUDA;
      return cuda_status();
    }
    if (router_fused_supported(*dims)) {
      // router GEMM, selection and softmax in one pass over x
      launch_router_fused(*dims, x, w_router, router_bias, logits_out, topk_idx, gates, stream);
      return cuda_status();
    }
    float* dst = logits_out ? logits_out : at<float>(workspace, L.logits);
    LayerPtrs p;
    p.x = x;
    p.w_router = w_router;
    p.router_bias = router_bias;
    simt_router_logits(*dims, p, dst, stream);
    logits = dst;
  } else if (logits_out && logits_out != logits_in) {
    if (cudaMemcpyAsync(logits_out, logits_in, sizeof(float) * T * E, cudaMemcpyDeviceToDevice,
                        stream) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  launch_topk_softmax(logits, T, E, dims->top_k, topk_idx, gates, stream);
  return cuda_status();
}

moe_status moe_permute(const moe_dims* dims, const int32_t* topk_idx, int32_t* counts,
                       int32_t* offsets, int32_t* perm, int32_t* inv_perm, void* workspace,
                       size_t workspace_bytes, cudaStream_t stream) {
  if (!dims_ok(dims) || !counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (dims->tokens > 0 && (!topk_idx || !perm || !inv_perm)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(shape_supported(dims));
  MOE_TRY(check_ws(dims, MOE_FWD_ONLY, workspace, workspace_bytes));
  const Layout L = make_layout(*dims, MOE_FWD_ONLY);
  launch_permute(*dims, L, topk_idx, counts, offsets, perm, inv_perm, workspace, stream);
  return cuda_status();
}

moe_status moe_grouped_ffn_fwd(const moe_dims* dims, int mode, const void* x, const float* gates,
                               const void* w_gate, const void* w_up, const void* w_down,
                               void* h_buf, void* a_gate_saved, void* a_up_saved, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream) {
  if (!dims_ok(dims)) return MOE_ERR_INVALID_ARG;
  if (mode != MOE_FWD_ONLY && mode != MOE_SAVE_FOR_BWD) return MOE_ERR_INVALID_ARG;
  if (dims->tokens > 0) {
    if (!x || !gates || !w_gate || !w_up || !w_down || !h_buf) return MOE_ERR_INVALID_ARG;
    if (mode == MOE_SAVE_FOR_BWD && (!a_gate_saved || !a_up_saved)) return MOE_ERR_INVALID_ARG;
  }
  if (!aligned16({x, w_gate, w_up, w_down, h_buf, a_gate_saved, a_up_saved}))
    return MOE_ERR_INVALID_ARG;
  MOE_TRY(shape_supported(dims));
  MOE_TRY(check_ws(dims, MOE_FWD_ONLY, workspace, workspace_bytes));
  if (dims->tokens == 0) return MOE_OK;
  const Layout L = make_layout(*dims, MOE_FWD_ONLY);
  LayerPtrs p;
  p.x = x;
  p.gates = gates;
  p.w_gate = w_gate;
  p.w_up = w_up;
  p.w_down = w_down;
  p.h_buf = h_buf;
  p.a_gate = a_gate_saved;
  p.a_up = a_up_saved;
  if (dims->dtype == MOE_BF16) {
    if (!tc_grouped_fwd(*dims, L, mode, p, workspace, stream)) return MOE_ERR_CUDA;
  } else {
    simt_grouped_fwd(*dims, L, mode, p, workspace, stream);
  }
  return cuda_status();
}

moe_status moe_combine(const moe_dims* dims, int mode, const void* x, const void* ws_gate,
                       const void* ws_up, const void* ws_down, void* y,
                       void* hs_buf, void* as_gate_saved, void* as_up_saved, const void* upstream,
                       float* loss, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!dims_ok(dims)) return MOE_ERR_INVALID_ARG;
  // MOE_SHARED_READY: moe_shared_ffn_fwd already left the shared output
  const bool shared_ready = (mode & MOE_SHARED_READY) != 0;
  mode &= ~MOE_SHARED_READY;
  if (mode != MOE_FWD_ONLY && mode != MOE_SAVE_FOR_BWD) return MOE_ERR_INVALID_ARG;
  const bool shared = dims->shared_hidden > 0 && !shared_ready;
  if (dims->tokens > 0) {
    if (!y) return MOE_ERR_INVALID_ARG;
    if (shared && (!x || !ws_gate || !ws_up || !ws_down || !hs_buf)) return MOE_ERR_INVALID_ARG;
    if (shared && mode == MOE_SAVE_FOR_BWD && (!as_gate_saved || !as_up_saved))
      return MOE_ERR_INVALID_ARG;
  }
  if (upstream && !loss) return MOE_ERR_INVALID_ARG;
  if (!aligned16({x, ws_gate, ws_up, ws_down, y, hs_buf, as_gate_saved, as_up_saved, upstream}))
    return MOE_ERR_INVALID_ARG;
  MOE_TRY(shape_supported(dims));
  MOE_TRY(check_ws(dims, MOE_FWD_ONLY, workspace, workspace_bytes));
  const Layout L = make_layout(*dims, MOE_FWD_ONLY);
  if (shared && dims->tokens > 0) {
    LayerPtrs p;
    p.x = x;
    p.ws_gate = ws_gate;
    p.ws_up = ws_up;
    p.ws_down = ws_down;
    p.hs_buf = hs_buf;
    p.as_gate = as_gate_saved;
    p.as_up = as_up_saved;
    if (dims->dtype == MOE_BF16) {
      if (!tc_shared_fwd(*dims, L, mode, p, workspace, stream)) return MOE_ERR_CUDA;
    } else {
      simt_shared_fwd(*dims, L, mode, p, workspace, stream);
    }
  }
  launch_combine(*dims, L, y, upstream, loss, workspace, stream);
  return cuda_status();
}

moe_status moe_shared_ffn_fwd(const moe_dims* dims, int mode, const void* x, const void* ws_gate,
                              const void* ws_up, const void* ws_down, void* hs_buf,
                              void* as_gate_saved, void* as_up_saved, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
  if (!dims_ok(dims)) return MOE_ERR_INVALID_ARG;
  if (mode != MOE_FWD_ONLY && mode != MOE_SAVE_FOR_BWD) return MOE_ERR_INVALID_ARG;
  if (dims->shared_hidden == 0) return MOE_OK;
  if (dims->tokens > 0) {
    if (!x || !ws_gate || !ws_up || !ws_down || !hs_buf) return MOE_ERR_INVALID_ARG;
    if (mode == MOE_SAVE_FOR_BWD && (!as_gate_saved || !as_up_saved)) return MOE_ERR_INVALID_ARG;
  }
  if (!aligned16({x, ws_gate, ws_up, ws_down, hs_buf, as_gate_saved, as_up_saved}))
    return MOE_ERR_INVALID_ARG;
  MOE_TRY(shape_supported(dims));
  MOE_TRY(check_ws(dims, MOE_FWD_ONLY, workspace, workspace_bytes));
  if (dims->tokens == 0) return MOE_OK;
  const Layout L = make_layout(*dims, MOE_FWD_ONLY);
  LayerPtrs p;
  p.x = x;
  p.ws_gate = ws_gate;
  p.ws_up = ws_up;
  p.ws_down = ws_down;
  p.hs_buf = hs_buf;
  p.as_gate = as_gate_saved;
  p.as_up = as_up_saved;
  if (dims->dtype == MOE_BF16) {
    if (!tc_shared_fwd(*dims, L, mode, p, workspace, stream)) return MOE_ERR_CUDA;
  } else {
    simt_shared_fwd(*dims, L, mode, p, workspace, stream);
  }
  return cuda_status();
}

namespace {

// The backward's shared part (dws_*, and the shared expert's rows of dx in
// the workspace) and routed part (the routed experts' GEMMs and the router
// backward, which also forms dx); `parts`: 1 shared, 2 routed, 3 both.
moe_status backward_parts(int parts, const moe_dims* dims, const void* dy, const void* x,
                          const void* w_router, const void* w_gate, const void* w_up,
                          const void* w_down, const void* ws_gate, const void* ws_up,
                          const void* ws_down, const int32_t* topk_idx, const float* gates,
                          const void* a_gate_saved, const void* a_up_saved, const void* h_saved,
                          const void* as_gate_saved, const void* as_up_saved,
                          const void* hs_saved, void* dx, float* dw_router, float* dw_gate,
                          float* dw_up, float* dw_down, float* dws_gate, float* dws_up,
                          float* dws_down, cudaEvent_t shared_done, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
  if (!dims_ok(dims)) return MOE_ERR_INVALID_ARG;
  const bool routed = parts & 2;
  const bool shared = (parts & 1) && dims->shared_hidden > 0;
  if (routed && (!dw_router || !dw_gate || !dw_up || !dw_down || !w_router))
    return MOE_ERR_INVALID_ARG;
  if (shared && (!dws_gate || !dws_up || !dws_down || !ws_gate || !ws_up || !ws_down))
    return MOE_ERR_INVALID_ARG;
  if (dims->tokens > 0) {
    if (!dy || !x) return MOE_ERR_INVALID_ARG;
    if (routed && (!w_gate || !w_up || !w_down || !topk_idx || !gates || !a_gate_saved ||
                   !a_up_saved || !h_saved || !dx))
      return MOE_ERR_INVALID_ARG;
    if (shared && (!as_gate_saved || !as_up_saved || !hs_saved)) return MOE_ERR_INVALID_ARG;
  }
  if (!aligned16({dy, x, w_router, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, a_gate_saved,
                  a_up_saved, h_saved, as_gate_saved, as_up_saved, hs_saved, dx, dw_router,
                  dw_gate, dw_up, dw_down, dws_gate, dws_up, dws_down}))
    return MOE_ERR_INVALID_ARG;
  MOE_TRY(shape_supported(dims));
  // the router backward keeps W_r^T and one dW_r column block in shared memory
  if (routed && !router_backward_supported(*dims)) return MOE_ERR_UNSUPPORTED;
  MOE_TRY(check_ws(dims, MOE_SAVE_FOR_BWD, workspace, workspace_bytes));
  const Layout L = make_layout(*dims, MOE_SAVE_FOR_BWD);
  const int64_t E = dims->experts, dm = dims->d_model, h = dims->d_hidden,
                hs = dims->shared_hidden;
  if (dims->tokens == 0) {
    if (routed) {
      zero_fill_f32(dw_router, dm * E, stream);
      zero_fill_f32(dw_gate, E * dm * h, stream);
      zero_fill_f32(dw_up, E * dm * h, stream);
      zero_fill_f32(dw_down, E * h * dm, stream);
    }
    if (shared) {
      zero_fill_f32(dws_gate, dm * hs, stream);
      zero_fill_f32(dws_up, dm * hs, stream);
      zero_fill_f32(dws_down, hs * dm, stream);
    }
    return cuda_status();
  }
  LayerPtrs p;
  p.dy = dy;
  p.x = x;
  p.w_router = w_router;
  p.w_gate = w_gate;
  p.w_up = w_up;
  p.w_down = w_down;
  p.ws_gate = ws_gate;
  p.ws_up = ws_up;
  p.ws_down = ws_down;
  p.topk_idx = topk_idx;
  p.gates = gates;
  p.a_gate = const_cast<void*>(a_gate_saved);
  p.a_up = const_cast<void*>(a_up_saved);
  p.as_gate = const_cast<void*>(as_gate_saved);
  p.as_up = const_cast<void*>(as_up_saved);
  p.h_buf = const_cast<void*>(h_saved);
  p.hs_buf = const_cast<void*>(hs_saved);
  p.dx = dx;
  p.dw_router = dw_router;
  p.dw_gate = dw_gate;
  p.dw_up = dw_up;
  p.dw_down = dw_down;
  p.dws_gate = dws_gate;
  p.dws_up = dws_up;
  p.dws_down = dws_down;
  const bool bf = dims->dtype == MOE_BF16;
  if (shared) {
    if (bf) {
      if (!tc_backward_shared(*dims, L, p, workspace, stream)) return MOE_ERR_CUDA;
    } else {
      simt_backward_shared(*dims, L, p, workspace, stream);
    }
  }
  if (!routed) return cuda_status();
  // gate-gradient partials per pair: one per DZ column tile (and column
  // half of the tensor-core epilogue), pairs 2*h/64 apart
  const int dg_ld = (int)(2 * h / 64);
  int dg_n = (int)(h / 64);
  if (bf) {
    // dZ, the router logit gradients (dX adds each pair's router term to its
    // row), dX and the weight gradients, dW_r and dx
    if (!tc_backward_routed_dz(*dims, L, p, workspace, stream)) return MOE_ERR_CUDA;
    dg_n = (int)(2 * h / tc_dz_bn((int)h));
    launch_router_dsel(*dims, L, p, dg_n, dg_ld, workspace, stream, true);
    if (!tc_backward_routed_rest(*dims, L, p, workspace, stream)) return MOE_ERR_CUDA;
    launch_router_dw_dx(*dims, L, p, workspace, stream, shared_done, true);
  } else {
    simt_backward_routed(*dims, L, p, workspace, stream);
    dg_n = simt_dz_tiles((int)h);
    launch_router_backward(*dims, L, p, dg_n, dg_ld, workspace, stream, shared_done);
  }
  return cuda_status();
}

}  // namespace

moe_status moe_backward(const moe_dims* dims, const void* dy, const void* x, const void* w_router,
                        const void* w_gate, const void* w_up, const void* w_down,
                        const void* ws_gate, const void* ws_up, const void* ws_down,
                        const int32_t* topk_idx, const float* gates, const void* a_gate_saved,
                        const void* a_up_saved, const void* h_saved, const void* as_gate_saved,
                        const void* as_up_saved, const void* hs_saved, void* dx,
                        float* dw_router, float* dw_gate, float* dw_up, float* dw_down,
                        float* dws_gate, float* dws_up, float* dws_down, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
  return backward_parts(3, dims, dy, x, w_router, w_gate, w_up, w_down, ws_gate, ws_up, ws_down,
                        topk_idx, gates, a_gate_saved, a_up_saved, h_saved, as_gate_saved,
                        as_up_saved, hs_saved, dx, dw_router, dw_gate, dw_up, dw_down, dws_gate,
                        dws_up, dws_down, nullptr, workspace, workspace_bytes, stream);
}

moe_status moe_shared_backward(const moe_dims* dims, const void* dy, const void* x,
                               const void* ws_gate, const void* ws_up, const void* ws_down,
                               const void* as_gate_saved, const void* as_up_saved,
                               const void* hs_saved, float* dws_gate, float* dws_up,
                               float* dws_down, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
  if (dims && dims->shared_hidden == 0) return dims_ok(dims) ? MOE_OK : MOE_ERR_INVALID_ARG;
  return backward_parts(1, dims, dy, x, nullptr, nullptr, nullptr, nullptr, ws_gate, ws_up,
                        ws_down, nullptr, nullptr, nullptr, nullptr, nullptr, as_gate_saved,
                        as_up_saved, hs_saved, nullptr, nullptr, nullptr, nullptr, nullptr,
                        dws_gate, dws_up, dws_down, nullptr, workspace, workspace_bytes, stream);
}

moe_status moe_backward_routed(const moe_dims* dims, const void* dy, const void* x,
                               const void* w_router, const void* w_gate, const void* w_up,
                               const void* w_down, const int32_t* topk_idx, const float* gates,
                               const void* a_gate_saved, const void* a_up_saved,
                               const void* h_saved, void* dx, float* dw_router, float* dw_gate,
                               float* dw_up, float* dw_down, cudaEvent_t shared_done,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return backward_parts(2, dims, dy, x, w_router, w_gate, w_up, w_down, nullptr, nullptr, nullptr,
                        topk_idx, gates, a_gate_saved, a_up_saved, h_saved, nullptr, nullptr,
                        nullptr, dx, dw_router, dw_gate, dw_up, dw_down, nullptr, nullptr,
                        nullptr, shared_done, workspace, workspace_bytes, stream);
}

moe_status moe_set_sm_limit(int sms) {
  if (sms < 0) return MOE_ERR_INVALID_ARG;
  tcg::set_sm_limit(sms);
  return MOE_OK;
}

moe_status moe_read_device_status(void* workspace, size_t workspace_bytes, cudaStream_t stream,
                                  int32_t* detail) {
  if (!workspace || workspace_bytes < 64) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  int host[2] = {0, 0};
  if (cudaMemcpy(host, workspace, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (host[0] != 0) {
    const int zero[2] = {0, 0};
    if (cudaMemcpy(workspace, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (detail) *detail = host[1];
  return (moe_status)host[0];
}

}  // extern "C"
