// Combine (unpermute + gate-weighted sum) with the train step's value, and
// the router backward.
//
// Combine: the grouped down projection leaves, for every pair p = t*k + j,
// its gate-weighted expert output g_j O_{e_j}(x_t) as one row of the
// expert-sorted buffer; y[t] = shared(x_t) + sum_j row(pairrow[t*k + j]),
// summed in slot order (the unpermute_combine piece of kernel_gmm_gpu.json).
// The value of the train step (gpu_moe_h100.json: value_and_grad) is
// L = sum(y * G), reduced in a fixed order so repeated runs give the same
// bits.
//
// Router backward: the gates are a softmax over the k selected logits, so
// the logit gradient of slot j is g_j (dg_j - sum_i g_i dg_i), with dg_j the
// gradient of the gate (the row-dot <dy_t W_down[e]^T, H_r> produced by the
// grouped backward), and zero on the experts that were not selected.  Then
// dW_r = x^T dlogits and dx = (shared + sum of the pairs' rows) + dlogits W_r^T.
#include "kernels.cuh"

namespace moe {
namespace {

// 16-byte vector of storage elements as floats
template <typename T>
__device__ __forceinline__ void ld16(const T* p, float (&v)[16 / sizeof(T)]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  if constexpr (sizeof(T) == 2) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[j]));
      v[2 * j] = f.x;
      v[2 * j + 1] = f.y;
    }
  } else {
    v[0] = __uint_as_float(u.x);
    v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z);
    v[3] = __uint_as_float(u.w);
  }
}

template <typename T>
__device__ __forceinline__ void st16(T* p, const float (&v)[16 / sizeof(T)]) {
  if constexpr (sizeof(T) == 2) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
      w[j] = *reinterpret_cast<uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
}

// y[t] = ys[t] + sum_j osort[pairrow[t*k + j]] (16-byte chunks, one per
// thread), cast to the storage type, plus the block's share of sum(y * G).
template <typename T>
__global__ void __launch_bounds__(256) combine_kernel(const T* __restrict__ osort,
                                                      const int32_t* __restrict__ pairrow,
                                                      const T* __restrict__ ys, T* __restrict__ y,
                                                      const T* __restrict__ G, int64_t Tn, int d,
                                                      int k, float* loss_part) {
  constexpr int VE = 16 / sizeof(T);
  __shared__ float red[8];
  const int cpt = d / VE;
  const int64_t n = Tn * cpt;
  float lacc = 0.f;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += stride) {
    const int64_t t = i / cpt;
    const int c = (int)(i % cpt);
    float acc[VE];
    if (ys) {
      ld16(ys + t * d + c * VE, acc);
    } else {
#pragma unroll
      for (int q = 0; q < VE; ++q) acc[q] = 0.f;
    }
    // the token's rows in groups of four: all row indices, then all row
    // loads, then the adds (in slot order)
    for (int j0 = 0; j0 < k; j0 += 4) {
      int rows[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) rows[j] = j0 + j < k ? pairrow[t * k + j0 + j] : -1;
      float v[4][VE];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (rows[j] >= 0) ld16(osort + (int64_t)rows[j] * d + c * VE, v[j]);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (rows[j] >= 0)
#pragma unroll
          for (int q = 0; q < VE; ++q) acc[q] += v[j][q];
    }
    st16(y + t * d + c * VE, acc);
    if (G) {
      float g[VE];
      ld16(G + t * d + c * VE, g);
#pragma unroll
      for (int q = 0; q < VE; ++q) lacc = fmaf(to_f32(from_f32<T>(acc[q])), g[q], lacc);
    }
  }
  if (!G) return;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lacc += __shfl_xor_sync(0xffffffffu, lacc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = lacc;
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
                                                          float* __restrict__ dsel,
                                                          const int32_t* __restrict__ idx, int E,
                                                          __nv_bfloat16* __restrict__ dl) {
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
  if (dl) {  // dense bf16 row of the logit gradient (zero off the selection);
             // E is a multiple of 8 on this path: 16-byte stores
    uint4* row = reinterpret_cast<uint4*>(dl + t * E);
    for (int e8 = 0; e8 < E / 8; ++e8) row[e8] = make_uint4(0u, 0u, 0u, 0u);
  }
  for (int j = 0; j < k; ++j) {
    const int64_t p = t * k + j;
    const float v = gates[p] * (dsel[p] - sgd);
    dsel[p] = v;
    if (dl) dl[t * E + idx[p]] = __float2bfloat16_rn(v);
  }
}

// W_r^T [E, d] from W_r [d, E] (storage type unchanged)
template <typename T>
__global__ void __launch_bounds__(256) transpose_router_kernel(const T* __restrict__ w, int d,
                                                               int E, T* __restrict__ wt) {
  const int64_t n = (int64_t)d * E;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / E, e = i % E;
    wt[e * d + r] = w[i];
  }
}

// dx[t] = dxs[t] + sum_j dxsort[pairrow[t*k + j]] + sum_j dsel[t, j] W_r[:, e_j]:
// each thread takes one 16-byte chunk of one token; W_r^T [E, d] rows are
// read through the cache.
template <typename T>
__global__ void __launch_bounds__(256) router_dx_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ dsel, const T* __restrict__ s_wt,
    const T* __restrict__ dxsort, const int32_t* __restrict__ pairrow, const T* __restrict__ dxs,
    T* __restrict__ dx, int64_t Tn, int d, int E, int k) {
  constexpr int VE = 16 / sizeof(T);
  const int cpt = d / VE;
  const int64_t n = Tn * cpt;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / cpt;
    const int c = (int)(i % cpt);
    float acc[VE];
    if (dxs) {
      ld16(dxs + t * d + c * VE, acc);
    } else {
#pragma unroll
      for (int q = 0; q < VE; ++q) acc[q] = 0.f;
    }
    for (int j0 = 0; j0 < k; j0 += 4) {
      int rows[4], ex[4];
      float ds[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t p = t * k + j0 + j;
        const bool ok = j0 + j < k;
        rows[j] = ok ? pairrow[p] : -1;
        ex[j] = ok ? idx[p] : 0;
        ds[j] = ok ? dsel[p] : 0.f;
      }
      float v[4][VE];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (rows[j] >= 0) ld16(dxsort + (int64_t)rows[j] * d + c * VE, v[j]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (rows[j] < 0) continue;
        float w[VE];
        ld16(s_wt + ex[j] * d + c * VE, w);
#pragma unroll
        for (int q = 0; q < VE; ++q) acc[q] += fmaf(ds[j], w[q], v[j][q]);
      }
    }
    st16(dx + t * d + c * VE, acc);
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
#pragma unroll 8
  for (int r = 0; r < ranges; ++r) s += part[(int64_t)r * n + i];
  dw[i] = s;
}

template <typename T>
void combine_t(const moe_dims& d, const Layout& L, void* y, const void* G, float* loss, void* ws,
               cudaStream_t s) {
  float* part = at<float>(ws, L.loss_part);
  const T* ys = d.shared_hidden > 0 ? at<const T>(ws, L.ys) : nullptr;
  MOE_LAUNCH("combine", s,
             combine_kernel<T><<<kLossBlocks, 256, 0, s>>>(
                 at<const T>(ws, L.osort), at<const int32_t>(ws, L.pairrow), ys,
                 reinterpret_cast<T*>(y), reinterpret_cast<const T*>(G), d.tokens, d.d_model,
                 d.top_k, part));
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
    cudaFuncSetAttribute(router_dw_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kRouterBwdSmem);
    attr_set = true;
  }
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const bool tc_dw = tc_router_dw_supported(d);

  MOE_LAUNCH("router_dsel", s,
             router_dsel_kernel<<<(unsigned)((d.tokens + 255) / 256), 256, 0, s>>>(
                 p.gates, at<float>(ws, L.dg_part), dg_ld, dg_n, d.tokens, k, dsel, p.topk_idx, E,
                 tc_dw ? at<__nv_bfloat16>(ws, L.dl) : nullptr));

  T* wt = at<T>(ws, L.wrt);
  MOE_LAUNCH("router_transpose", s,
             transpose_router_kernel<T><<<(unsigned)((dm * E + 255) / 256), 256, 0, s>>>(
                 reinterpret_cast<const T*>(p.w_router), dm, E, wt));

  const int VE = 16 / sizeof(T);
  int64_t bx = (d.tokens * (dm / VE) + 255) / 256;
  if (bx > (int64_t)sms * 16) bx = (int64_t)sms * 16;
  const T* dxs = d.shared_hidden > 0 ? at<const T>(ws, L.dxs) : nullptr;
  MOE_LAUNCH("router_dx", s,
             router_dx_kernel<T><<<(unsigned)bx, 256, 0, s>>>(
                 p.topk_idx, dsel, wt, at<const T>(ws, L.dxsort), at<const int32_t>(ws, L.pairrow),
                 dxs, reinterpret_cast<T*>(p.dx), d.tokens, dm, E, k));

  if (tc_dw) {
    tc_router_dw(d, L, p, ws, s);
    return;
  }
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

void launch_combine(const moe_dims& d, const Layout& L, void* y, const void* upstream, float* loss,
                    void* ws, cudaStream_t s) {
  if (d.tokens == 0) {
    if (upstream && loss) zero_fill_f32(loss, 1, s);
    return;
  }
  if (d.dtype == MOE_BF16) combine_t<__nv_bfloat16>(d, L, y, upstream, loss, ws, s);
  else combine_t<float>(d, L, y, upstream, loss, ws, s);
}

void launch_router_backward(const moe_dims& d, const Layout& L, const LayerPtrs& p, int dg_n,
                            int dg_ld, void* ws, cudaStream_t s) {
  if (d.dtype == MOE_BF16) router_backward_t<__nv_bfloat16>(d, L, p, dg_n, dg_ld, ws, s);
  else router_backward_t<float>(d, L, p, dg_n, dg_ld, ws, s);
}

bool router_backward_supported(const moe_dims& d) {
  // the CUDA-core dW_r path keeps one [E][256] f32 accumulator per block
  return tc_router_dw_supported(d) || (size_t)d.experts * 256 * 4 <= (size_t)kRouterBwdSmem;
}

}  // namespace moe
