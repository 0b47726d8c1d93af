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
// dW_r = x^T dlogits and dx = dx_acc + dlogits W_r^T.
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

// Router backward of a block's token range, in chunks of 256/k tokens:
//   phase A: thread i of the chunk takes pair i: its gate gradient (the sum
//            of the DZ partials), then dsel = g (dg - sum_j g_j dg_j)
//   phase B: thread i takes input dimensions i, i+256, ...: for every token
//            of the chunk dx = dx_acc + sum_j dsel_j W_r[i, e_j] and the
//            block's dW_r partial gains x[t, i] dsel_j in column e_j.  Each
//            thread owns its dimensions' accumulators, so the order of the
//            adds is fixed and the result deterministic.
template <typename T>
__global__ void __launch_bounds__(256) router_bwd_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ gates,
    const float* __restrict__ dg_part, int dg_ld, int dg_n, const T* __restrict__ w_router,
    const T* __restrict__ x, const float* __restrict__ dx_acc, T* __restrict__ dx,
    float* __restrict__ part, int64_t Tn, int d, int E, int k, int64_t per_block) {
  extern __shared__ __align__(16) float s_acc[];  // [E][d] f32, then W_r^T [E][d] (T)
  T* s_wt = reinterpret_cast<T*>(s_acc + (size_t)E * d);
  __shared__ int s_e[256];
  __shared__ float s_g[256], s_dg[256], s_ds[256];
  const int tid = threadIdx.x;
  for (int i = tid; i < E * d; i += blockDim.x) {
    s_acc[i] = 0.f;
    const int r = i / E, e = i % E;  // coalesced read of W_r[r][e]
    s_wt[e * d + r] = w_router[i];
  }
  const int64_t t0 = blockIdx.x * per_block;
  const int64_t t1 = t0 + per_block < Tn ? t0 + per_block : Tn;
  const int CH = 256 / k;
  for (int64_t tc = t0; tc < t1; tc += CH) {
    const int nt = (int)(t1 - tc < CH ? t1 - tc : CH);
    const int npair = nt * k;
    __syncthreads();
    if (tid < npair) {
      const int64_t p = tc * k + tid;
      s_e[tid] = idx[p];
      s_g[tid] = gates[p];
      float dg = 0.f;
      const float* row = dg_part + p * dg_ld;
      for (int q = 0; q < dg_n; ++q) dg += row[q];
      s_dg[tid] = dg;
    }
    __syncthreads();
    if (tid < npair) {
      const int base = (tid / k) * k;
      float sgd = 0.f;
      for (int j = 0; j < k; ++j) sgd = fmaf(s_g[base + j], s_dg[base + j], sgd);
      s_ds[tid] = s_g[tid] * (s_dg[tid] - sgd);
    }
    __syncthreads();
    for (int i = tid; i < d; i += blockDim.x) {
#pragma unroll 4
      for (int u = 0; u < nt; ++u) {
        const int64_t t = tc + u;
        float v = dx_acc[t * d + i];
        const float xv = to_f32(x[t * d + i]);
        for (int j = 0; j < k; ++j) {
          const int e = s_e[u * k + j];
          const float ds = s_ds[u * k + j];
          v = fmaf(ds, to_f32(s_wt[e * d + i]), v);
          s_acc[e * d + i] = fmaf(xv, ds, s_acc[e * d + i]);
        }
        dx[t * d + i] = from_f32<T>(v);
      }
    }
  }
  __syncthreads();
  float* out = part + (int64_t)blockIdx.x * d * E;
  for (int i = tid; i < E * d; i += blockDim.x) {
    const int r = i / E, e = i % E;
    out[i] = s_acc[e * d + r];
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
  MOE_LAUNCH("finalize_y", s,
             finalize_y_kernel<T><<<kLossBlocks, 256, 0, s>>>(
                 y_acc, reinterpret_cast<T*>(y), reinterpret_cast<const T*>(G), n, part));
  if (G && loss)
    MOE_LAUNCH("loss_reduce", s, loss_reduce_kernel<<<1, 32, 0, s>>>(part, kLossBlocks, loss));
}

template <typename T>
void router_backward_t(const moe_dims& d, const Layout& L, const LayerPtrs& p, int dg_n,
                       int dg_ld, void* ws, cudaStream_t s) {
  const int dm = d.d_model, E = d.experts, k = d.top_k;
  float* part = at<float>(ws, L.dwr_part);
  if (d.tokens == 0) {
    zero_fill_f32(p.dw_router, (int64_t)dm * E, s);
    return;
  }
  const size_t smem = (size_t)E * dm * (sizeof(float) + sizeof(T));
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(router_bwd_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kRouterBwdSmem);
    attr_set = true;
  }
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int CH = 256 / k;
  int64_t blocks = (d.tokens + CH - 1) / CH;
  const int64_t cap = sms < kRouterBwdRanges ? sms : kRouterBwdRanges;
  if (blocks > cap) blocks = cap;
  const int64_t per_block = (d.tokens + blocks - 1) / blocks;
  MOE_LAUNCH("router_bwd", s,
             router_bwd_kernel<T><<<(unsigned)blocks, 256, smem, s>>>(
                 p.topk_idx, p.gates, at<float>(ws, L.dg_part), dg_ld, dg_n,
                 reinterpret_cast<const T*>(p.w_router), reinterpret_cast<const T*>(p.x),
                 at<float>(ws, L.dx_acc), reinterpret_cast<T*>(p.dx), part, d.tokens, dm, E, k,
                 per_block));
  const int64_t n = (int64_t)dm * E;
  MOE_LAUNCH("router_dw_reduce", s,
             router_dw_reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(
                 part, (int)blocks, n, p.dw_router));
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

void launch_router_backward(const moe_dims& d, const Layout& L, const LayerPtrs& p, int dg_n,
                            int dg_ld, void* ws, cudaStream_t s) {
  if (d.dtype == MOE_BF16) router_backward_t<__nv_bfloat16>(d, L, p, dg_n, dg_ld, ws, s);
  else router_backward_t<float>(d, L, p, dg_n, dg_ld, ws, s);
}

bool router_backward_supported(const moe_dims& d) {
  const size_t elem = d.dtype == MOE_BF16 ? 2 : 4;
  return (size_t)d.experts * d.d_model * (4 + elem) <= (size_t)kRouterBwdSmem;
}

}  // namespace moe
