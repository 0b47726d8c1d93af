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

// dsel[t, j] = g_j (dg_j - sum_i g_i dg_i), one thread per token; dg_j is
// the sum of the grouped backward's per-column-tile partials of pair t*k+j.
__global__ void __launch_bounds__(256) router_dsel_kernel(const float* __restrict__ gates,
                                                          const float* __restrict__ dg_part,
                                                          int dg_ld, int dg_n, int64_t Tn, int k,
                                                          float* __restrict__ dsel) {
  const int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (t >= Tn) return;
  float sgd = 0.f;
  for (int j = 0; j < k; ++j) {
    const int64_t p = t * k + j;
    float dg = 0.f;
    for (int q = 0; q < dg_n; ++q) dg += dg_part[p * dg_ld + q];
    dsel[p] = dg;
    sgd = fmaf(gates[p], dg, sgd);
  }
  for (int j = 0; j < k; ++j) {
    const int64_t p = t * k + j;
    dsel[p] = gates[p] * (dsel[p] - sgd);
  }
}

// dx[t, :] = dx_acc[t, :] + sum_j dsel[t, j] W_r[:, e_j]: each thread takes
// four consecutive input dimensions of one token (W_r^T staged in shared
// memory), blocks loop over token groups.
template <typename T>
__global__ void __launch_bounds__(256) router_dx_kernel(const int32_t* __restrict__ idx,
                                                        const float* __restrict__ dsel,
                                                        const T* __restrict__ w_router,
                                                        const float* __restrict__ dx_acc,
                                                        T* __restrict__ dx, int64_t Tn, int d,
                                                        int E, int k) {
  extern __shared__ __align__(16) unsigned char s_raw[];
  T* s_wt = reinterpret_cast<T*>(s_raw);  // [E][d]
  for (int i = threadIdx.x; i < E * d; i += blockDim.x) {
    const int r = i / E, e = i % E;  // coalesced read of W_r[r][e]
    s_wt[e * d + r] = w_router[i];
  }
  __syncthreads();
  const int cpt = d / 4;                  // float4 chunks per token
  const int tpb = blockDim.x / cpt;       // tokens per block pass
  const int c = threadIdx.x % cpt, u = threadIdx.x / cpt;
  if (u >= tpb) return;
  for (int64_t t = (int64_t)blockIdx.x * tpb + u; t < Tn; t += (int64_t)gridDim.x * tpb) {
    float4 v = reinterpret_cast<const float4*>(dx_acc + t * d)[c];
    for (int j = 0; j < k; ++j) {
      const int e = __ldg(idx + t * k + j);
      const float ds = __ldg(dsel + t * k + j);
      const T* w = s_wt + e * d + 4 * c;
      v.x = fmaf(ds, to_f32(w[0]), v.x);
      v.y = fmaf(ds, to_f32(w[1]), v.y);
      v.z = fmaf(ds, to_f32(w[2]), v.z);
      v.w = fmaf(ds, to_f32(w[3]), v.w);
    }
    T* o = dx + t * d + 4 * c;
    o[0] = from_f32<T>(v.x);
    o[1] = from_f32<T>(v.y);
    o[2] = from_f32<T>(v.z);
    o[3] = from_f32<T>(v.w);
  }
}

// dW_r partial of one token range: thread i owns input dimension i and its
// column of the shared accumulator [E][256], so the order of the adds is
// fixed; the range's (expert, dsel) pairs are staged in shared memory.
template <typename T>
__global__ void __launch_bounds__(256) router_dw_kernel(const T* __restrict__ x,
                                                        const int32_t* __restrict__ idx,
                                                        const float* __restrict__ dsel,
                                                        int64_t Tn, int d, int E, int k,
                                                        int64_t per_range, float* part) {
  extern __shared__ __align__(16) float s_acc[];  // [E][256]
  __shared__ int s_e[256];
  __shared__ float s_ds[256];
  const int tid = threadIdx.x;
  const int i = blockIdx.y * 256 + tid;
  for (int e = 0; e < E; ++e) s_acc[e * 256 + tid] = 0.f;
  const int64_t t0 = blockIdx.x * per_range;
  const int64_t t1 = t0 + per_range < Tn ? t0 + per_range : Tn;
  const int CH = 256 / k;
  for (int64_t tc = t0; tc < t1; tc += CH) {
    const int nt = (int)(t1 - tc < CH ? t1 - tc : CH);
    __syncthreads();
    if (tid < nt * k) {
      s_e[tid] = idx[tc * k + tid];
      s_ds[tid] = dsel[tc * k + tid];
    }
    __syncthreads();
    if (i < d) {
      int u = 0;
      for (; u + 8 <= nt; u += 8) {
        float xv[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) xv[q] = to_f32(x[(tc + u + q) * d + i]);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          for (int j = 0; j < k; ++j) {
            const int e = s_e[(u + q) * k + j];
            s_acc[e * 256 + tid] = fmaf(xv[q], s_ds[(u + q) * k + j], s_acc[e * 256 + tid]);
          }
      }
      for (; u < nt; ++u) {
        const float xv = to_f32(x[(tc + u) * d + i]);
        for (int j = 0; j < k; ++j) {
          const int e = s_e[u * k + j];
          s_acc[e * 256 + tid] = fmaf(xv, s_ds[u * k + j], s_acc[e * 256 + tid]);
        }
      }
    }
  }
  if (i < d) {
    float* out = part + ((int64_t)blockIdx.x * d + i) * E;
    for (int e = 0; e < E; ++e) out[e] = s_acc[e * 256 + tid];
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
  if (d.tokens == 0) {
    zero_fill_f32(p.dw_router, (int64_t)dm * E, s);
    return;
  }
  float* dsel = at<float>(ws, L.dsel);
  float* part = at<float>(ws, L.dwr_part);
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(router_dx_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kRouterBwdSmem);
    cudaFuncSetAttribute(router_dw_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kRouterBwdSmem);
    attr_set = true;
  }
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);

  MOE_LAUNCH("router_dsel", s,
             router_dsel_kernel<<<(unsigned)((d.tokens + 255) / 256), 256, 0, s>>>(
                 p.gates, at<float>(ws, L.dg_part), dg_ld, dg_n, d.tokens, k, dsel));

  const int tpb = 256 / (dm / 4) > 0 ? 256 / (dm / 4) : 1;
  int64_t bx = (d.tokens + tpb - 1) / tpb;
  if (bx > (int64_t)sms * 4) bx = (int64_t)sms * 4;
  MOE_LAUNCH("router_dx", s,
             router_dx_kernel<T><<<(unsigned)bx, 256, sizeof(T) * E * dm, s>>>(
                 p.topk_idx, dsel, reinterpret_cast<const T*>(p.w_router), at<float>(ws, L.dx_acc),
                 reinterpret_cast<T*>(p.dx), d.tokens, dm, E, k));

  const int ny = (dm + 255) / 256;
  int64_t ranges = (int64_t)sms * 4 / ny;
  const int64_t by_tokens = (d.tokens + 63) / 64;
  if (ranges > by_tokens) ranges = by_tokens;
  if (ranges > kRouterBwdRanges) ranges = kRouterBwdRanges;
  if (ranges < 1) ranges = 1;
  const int64_t per_range = (d.tokens + ranges - 1) / ranges;
  MOE_LAUNCH("router_dw", s,
             router_dw_kernel<T><<<dim3((unsigned)ranges, ny), 256, sizeof(float) * E * 256, s>>>(
                 reinterpret_cast<const T*>(p.x), p.topk_idx, dsel, d.tokens, dm, E, k, per_range,
                 part));
  const int64_t n = (int64_t)dm * E;
  MOE_LAUNCH("router_dw_reduce", s,
             router_dw_reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(
                 part, (int)ranges, n, p.dw_router));
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
  return (size_t)d.experts * d.d_model * elem <= (size_t)kRouterBwdSmem &&
         (size_t)d.experts * 256 * 4 <= (size_t)kRouterBwdSmem && d.d_model % 4 == 0 &&
         d.d_model <= 1024;
}

}  // namespace moe
