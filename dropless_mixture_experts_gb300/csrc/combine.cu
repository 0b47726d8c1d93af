// Output cast with the train step's value, and the router backward.
//
// Value: L = sum(y * G) for the upstream gradient G (the train step of
// gpu_moe_h100.json is value_and_grad of the layer), reduced in a fixed
// order so repeated runs give the same bits.
//
// Router backward: the gates are a softmax over the k selected logits, so
// the logit gradient of slot j is g_j (dg_j - sum_i g_i dg_i), with dg_j the
// gradient of the gate (the row-dot <dy_t W_down[e]^T, H_r> produced by the
// grouped backward), and zero on the experts that were not selected.  Then
// dW_r = x^T dlogits and dx += dlogits W_r^T.
#include "kernels.cuh"

namespace moe {
namespace {

template <typename T>
__global__ void __launch_bounds__(256) finalize_y_kernel(const float* __restrict__ y_acc, T* y,
                                                         const T* __restrict__ G, int64_t n,
                                                         float* loss_part) {
  __shared__ float red[8];
  float acc = 0.f;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += stride) {
    const T v = from_f32<T>(y_acc[i]);
    y[i] = v;
    if (G) acc = fmaf(to_f32(v), to_f32(G[i]), acc);
  }
  if (!G) return;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < 8; ++w) s += red[w];
    loss_part[blockIdx.x] = s;
  }
}

__global__ void __launch_bounds__(32) loss_reduce_kernel(const float* __restrict__ part, int n,
                                                         float* loss) {
  // fixed-order reduction: lane l sums part[l], part[l+32], ...; then a
  // fixed butterfly
  float s = 0.f;
  for (int i = threadIdx.x; i < n; i += 32) s += part[i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (threadIdx.x == 0) *loss = s;
}

// One warp per token: dsel_j = g_j (dg_j - sum_i g_i dg_i), and
// dx[t] = dx_acc[t] + sum_j dsel_j W_r[:, e_j]  (W_r^T staged in shared memory).
template <typename T>
__global__ void __launch_bounds__(256) router_dl_dx_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ gates,
    const float* __restrict__ dg_part, int dg_ld, int dg_n, const int32_t* __restrict__ pad_inv,
    const T* __restrict__ w_router, const float* __restrict__ dx_acc, T* dx, float* dsel,
    int64_t Tn, int d, int E, int k) {
  extern __shared__ float s_wt[];  // [E][d]
  for (int i = threadIdx.x; i < d * E; i += blockDim.x) {
    const int r = i / E, e = i % E;  // coalesced read of W_r[r][e]
    s_wt[e * d + r] = to_f32(w_router[i]);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t t = warp; t < Tn; t += nwarps) {
    int e = 0;
    float g = 0.f, dg = 0.f;
    if (lane < k) {
      const int64_t p = t * k + lane;
      e = idx[p];
      g = gates[p];
      const float* row = dg_part + (int64_t)pad_inv[p] * dg_ld;
      for (int q = 0; q < dg_n; ++q) dg += row[q];
    }
    float sgd = g * dg;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sgd += __shfl_xor_sync(0xffffffffu, sgd, o);
    const float ds = g * (dg - sgd);
    if (lane < k) dsel[t * k + lane] = ds;
    for (int i = lane; i < d; i += 32) {
      float v = dx_acc[t * d + i];
      for (int j = 0; j < k; ++j) {
        const int ej = __shfl_sync(0xffffffffu, e, j);
        const float dj = __shfl_sync(0xffffffffu, ds, j);
        v = fmaf(dj, s_wt[ej * d + i], v);
      }
      dx[t * d + i] = from_f32<T>(v);
    }
  }
}

// dW_r partials: block (range, dim-slice) accumulates sum_t x[t, i] dsel[t, j]
// into column e_j, each thread owning one input dimension i (its column of
// the shared accumulator is private, so the order of the adds is fixed).
template <typename T>
__global__ void __launch_bounds__(256) router_dw_kernel(const T* __restrict__ x,
                                                        const int32_t* __restrict__ idx,
                                                        const float* __restrict__ dsel,
                                                        int64_t Tn, int d, int E, int k,
                                                        float* part) {
  extern __shared__ float s_acc[];  // [E][256]
  const int range = blockIdx.x;
  const int i = blockIdx.y * 256 + threadIdx.x;
  for (int e = 0; e < E; ++e) s_acc[e * 256 + threadIdx.x] = 0.f;
  const int64_t per = (Tn + gridDim.x - 1) / gridDim.x;
  const int64_t t0 = range * per;
  const int64_t t1 = t0 + per < Tn ? t0 + per : Tn;
  if (i < d) {
    for (int64_t t = t0; t < t1; ++t) {
      const float xv = to_f32(x[t * d + i]);
      for (int j = 0; j < k; ++j) {
        const int e = idx[t * k + j];
        s_acc[e * 256 + threadIdx.x] = fmaf(xv, dsel[t * k + j], s_acc[e * 256 + threadIdx.x]);
      }
    }
    for (int e = 0; e < E; ++e) part[((int64_t)range * d + i) * E + e] = s_acc[e * 256 + threadIdx.x];
  }
}

__global__ void __launch_bounds__(256) router_dw_reduce_kernel(const float* __restrict__ part,
                                                               int ranges, int64_t n, float* dw) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= n) return;
  float s = 0.f;
  for (int r = 0; r < ranges; ++r) s += part[(int64_t)r * n + i];
  dw[i] = s;
}

template <typename T>
void finalize_y_t(const moe_dims& d, const Layout& L, const float* y_acc, void* y,
                  const void* G, float* loss, void* ws, cudaStream_t s) {
  const int64_t n = d.tokens * (int64_t)d.d_model;
  float* part = at<float>(ws, L.loss_part);
  MOE_LAUNCH("finalize_y", s, finalize_y_kernel<T><<<kLossBlocks, 256, 0, s>>>(y_acc, reinterpret_cast<T*>(y),
                                                   reinterpret_cast<const T*>(G), n, part));
  if (G && loss) MOE_LAUNCH("loss_reduce", s, loss_reduce_kernel<<<1, 32, 0, s>>>(part, kLossBlocks, loss));
}

template <typename T>
void router_backward_t(const moe_dims& d, const Layout& L, const LayerPtrs& p, int dz_ntiles,
                       int dg_ld, void* ws, cudaStream_t s) {
  const int dm = d.d_model, E = d.experts, k = d.top_k;
  float* dsel = at<float>(ws, L.dsel);
  float* part = at<float>(ws, L.dwr_part);
  if (d.tokens > 0) {
    const size_t smem = sizeof(float) * dm * E;
    static bool attr_set = false;
    if (!attr_set) {
      cudaFuncSetAttribute(router_dl_dx_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           200 * 1024);
      cudaFuncSetAttribute(router_dw_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           200 * 1024);
      attr_set = true;
    }
    int64_t blocks = (d.tokens + 7) / 8;
    if (blocks > 152 * 2) blocks = 152 * 2;
    MOE_LAUNCH("router_dl_dx", s, router_dl_dx_kernel<T><<<(unsigned)blocks, 256, smem, s>>>(
        p.topk_idx, p.gates, at<float>(ws, L.dg_part), dg_ld, dz_ntiles, at<int32_t>(ws, L.pad_inv),
        reinterpret_cast<const T*>(p.w_router), at<float>(ws, L.dx_acc), reinterpret_cast<T*>(p.dx),
        dsel, d.tokens, dm, E, k));
    dim3 g(kRouterBwdRanges, (dm + 255) / 256);
    MOE_LAUNCH("router_dw", s, router_dw_kernel<T><<<g, 256, sizeof(float) * E * 256, s>>>(
        reinterpret_cast<const T*>(p.x), p.topk_idx, dsel, d.tokens, dm, E, k, part));
    const int64_t n = (int64_t)dm * E;
    MOE_LAUNCH("router_dw_reduce", s, router_dw_reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(part, kRouterBwdRanges, n,
                                                                       p.dw_router));
  } else {
    zero_fill_f32(p.dw_router, (int64_t)dm * E, s);
  }
}

}  // namespace

void launch_finalize_y(const moe_dims& d, const Layout& L, const float* y_acc, void* y,
                       const void* upstream, float* loss, void* ws, cudaStream_t s) {
  if (d.tokens == 0) {
    if (upstream && loss) zero_fill_f32(loss, 1, s);
    return;
  }
  if (d.dtype == MOE_BF16) finalize_y_t<__nv_bfloat16>(d, L, y_acc, y, upstream, loss, ws, s);
  else finalize_y_t<float>(d, L, y_acc, y, upstream, loss, ws, s);
}

void launch_router_backward(const moe_dims& d, const Layout& L, const LayerPtrs& p, int dz_ntiles,
                            int dg_ld, void* ws, cudaStream_t s) {
  if (d.dtype == MOE_BF16) router_backward_t<__nv_bfloat16>(d, L, p, dz_ntiles, dg_ld, ws, s);
  else router_backward_t<float>(d, L, p, dz_ntiles, dg_ld, ws, s);
}

}  // namespace moe
