// Launchers of the layer's kernels (host side), shared by the C ABI.
#pragma once

#include "common.cuh"

namespace moe {

// kernel timing records (profile.cu); MOE_LAUNCH brackets one launch
void prof_begin(const char* name, cudaStream_t s);
void prof_end(cudaStream_t s);
#define MOE_LAUNCH(name, stream, ...)   \
  do {                                  \
    ::moe::prof_begin(name, stream);    \
    __VA_ARGS__;                        \
    ::moe::prof_end(stream);            \
  } while (0)

// SMs the calling thread's launches may fill (tc_host.cu; moe_set_sm_limit)
namespace tcg {
int launch_sms();
void set_sm_limit(int n);
}  // namespace tcg
inline int tcg_launch_sms() { return tcg::launch_sms(); }

// utility kernels (misc.cu)
void zero_fill_i32(int32_t* p, int64_t n, cudaStream_t s);
void zero_fill_f32(float* p, int64_t n, cudaStream_t s);
// fixed-order sum of the K-split partials of a weight-gradient GEMM
void launch_split_reduce(const float* part, int S, int64_t EM, int ldp, int N, int hsplit,
                         float* out0, float* out1, cudaStream_t s);


// routing and permutation (route_permute.cu)
void launch_topk_softmax(const float* logits, int64_t T, int E, int k, int32_t* idx,
                         float* gates, cudaStream_t s);
bool router_fused_supported(const moe_dims& d);
void launch_router_fused(const moe_dims& d, const void* x, const void* w, const float* bias,
                         float* logits_out, int32_t* idx, float* gates, cudaStream_t s);
void launch_permute(const moe_dims& d, const Layout& L, const int32_t* idx, int32_t* counts,
                    int32_t* offsets, int32_t* perm, int32_t* inv_perm, void* ws,
                    cudaStream_t s);

// Operands and outputs of one layer invocation, as the grouped kernels see
// them.  Pointers are device pointers; storage type per dims.dtype.
struct LayerPtrs {
  const void* x = nullptr;
  const void* dy = nullptr;
  const void* w_router = nullptr;
  const float* router_bias = nullptr;  // [E] f32 routing offset, nullable
  const void* w_gate = nullptr;
  const void* w_up = nullptr;
  const void* w_down = nullptr;
  const void* ws_gate = nullptr;
  const void* ws_up = nullptr;
  const void* ws_down = nullptr;
  const float* gates = nullptr;
  const int32_t* topk_idx = nullptr;
  // forward outputs / saved activations
  void* h_buf = nullptr;
  void* a_gate = nullptr;
  void* a_up = nullptr;
  void* hs_buf = nullptr;
  void* as_gate = nullptr;
  void* as_up = nullptr;
  float* logits = nullptr;
  // backward outputs
  void* dx = nullptr;
  float* dw_router = nullptr;
  float* dw_gate = nullptr;
  float* dw_up = nullptr;
  float* dw_down = nullptr;
  float* dws_gate = nullptr;
  float* dws_up = nullptr;
  float* dws_down = nullptr;
};

// grouped expert GEMMs (gemm_simt.cu: float32 storage)
void simt_router_logits(const moe_dims& d, const LayerPtrs& p, float* logits, cudaStream_t s);
int simt_dz_tiles(int h);  // column tiles of the float32 dZ GEMM (its gate-gradient partials per row)
void simt_grouped_fwd(const moe_dims& d, const Layout& L, int mode, const LayerPtrs& p, void* ws,
                      cudaStream_t s);
void simt_shared_fwd(const moe_dims& d, const Layout& L, int mode, const LayerPtrs& p, void* ws,
                     cudaStream_t s);
void simt_backward_routed(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws,
                          cudaStream_t s);
void simt_backward_shared(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws,
                          cudaStream_t s);

// grouped expert GEMMs on the tensor cores (tc_fwd.cu, tc_bwd.cu: bfloat16
// storage); false when a tensor map could not be encoded
bool tc_grouped_fwd(const moe_dims& d, const Layout& L, int mode, const LayerPtrs& p, void* ws,
                    cudaStream_t s);
bool tc_shared_fwd(const moe_dims& d, const Layout& L, int mode, const LayerPtrs& p, void* ws,
                   cudaStream_t s);
// the routed backward in two parts: the row copy of g dy and dZ; then dX
// (with the router term from the logit gradients per sorted row) and the
// weight gradients
bool tc_backward_routed_dz(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws,
                           cudaStream_t s);
bool tc_backward_routed_rest(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws,
                             cudaStream_t s);
bool tc_backward_shared(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws,
                        cudaStream_t s);
int tc_dz_bn(int h);  // column tile of the DZ GEMM (its gate-gradient partials per row)
// router weight gradient x^T dlogits on the tensor cores (bf16, E a multiple of 8, <= 64)
bool tc_router_dw_supported(const moe_dims& d);
bool tc_router_dw(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws,
                  cudaStream_t s);
// router GEMM + top-k + softmax on the tensor cores (bf16, E a multiple of 8, <= 64)
bool tc_router_supported(const moe_dims& d);
bool tc_router(const moe_dims& d, const Layout& L, const void* x, const void* w_router,
               const float* bias, float* logits_out, int32_t* idx, float* gates, void* ws,
               cudaStream_t s);

// row streams (stream.cu)
// expert-sorted copy of token rows: out[pairrow[t*k + j]] = src[t] (with
// gates and no rowgate: g_tj src[t]), padding rows zeroed; with rowgate the
// rows are copied unscaled and rowgate[pairrow[t*k + j]] = g_tj (0 on padding)
void launch_scatter_rows(const moe_dims& d, const Layout& L, const void* src, void* out, void* ws,
                         cudaStream_t s, const float* gates, float* rowgate);
// y = shared + sum of each token's pair rows (from the workspace), and the
// value sum(y * upstream) when upstream is given
void launch_combine(const moe_dims& d, const Layout& L, void* y, const void* upstream, float* loss,
                    void* ws, cudaStream_t s);
// dx = shared + sum of each token's pair rows + dlogits W_r^T (wt = W_r^T [E, d]);
// term_in_rows: the pair rows already hold their dlogits W_r^T term (added
// here only for the slots without a row)
void launch_router_dx(const moe_dims& d, const Layout& L, const LayerPtrs& p, const float* dsel,
                      const void* wt, void* ws, cudaStream_t s, bool term_in_rows);

// router backward (router_bwd.cu)
bool router_backward_supported(const moe_dims& d);
// the input-gradient kernel (which adds the shared expert's dx rows) waits
// for `shared_done` when it is given
void launch_router_backward(const moe_dims& d, const Layout& L, const LayerPtrs& p, int dg_n,
                            int dg_ld, void* ws, cudaStream_t s, cudaEvent_t shared_done = nullptr);
// the same in two parts: the logit gradients (dsel; with rows, also per
// sorted row for the tensor-core input-gradient GEMM), then dW_r and dx
void launch_router_dsel(const moe_dims& d, const Layout& L, const LayerPtrs& p, int dg_n,
                        int dg_ld, void* ws, cudaStream_t s, bool rows);
void launch_router_dw_dx(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws,
                         cudaStream_t s, cudaEvent_t shared_done, bool term_in_rows);

}  // namespace moe
