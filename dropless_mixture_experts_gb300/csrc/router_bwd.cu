// Router backward.  The gates are a softmax over the k selected logits, so
// the logit gradient of slot j is g_j (dg_j - sum_i g_i dg_i), with dg_j the
// gradient of the gate (the row-dot <dy_t W_down[e]^T, H_r>).  The grouped
// backward hands over q_j = g_j dg_j (its rows of dy come scaled by the
// gate), so the logit gradient is q_j - g_j sum_i q_i, with no division by
// a gate; zero on the experts that were not selected
// (gpu_moe_h100.json: value_and_grad through the router).  Then
// dW_r = x^T dlogits, and dx gains dlogits W_r^T (a row stream, stream.cu).
#include "kernels.cuh"

namespace moe {
namespace {

// dsel[t, j] = q_j - g_j sum_i q_i; q_j = g_j dg_j is the sum (in
// column-tile order) of the grouped backward's partials of pair t*k+j, and
// 0 for a pair without a row (capacity-dropped or a rejected index).  A group of G
// lanes (the power of two >= k) takes one token, lane j of the group its
// slot j.  With dl given, the token's dense bf16 row of the logit gradient
// (zero off the selection; E a multiple of 8) is written as well.
// With rowdsel given, the logit gradient of each pair with a sorted row is
// also stored at that row (the tensor-core input-gradient GEMM adds the
// router term to the pair's row).
// The blocks past the tokens' write W_r^T [E, d] from W_r [d, E] (storage
// type unchanged) for the router input gradient.
template <typename T>
__global__ void __launch_bounds__(256) router_dsel_kernel(const float* __restrict__ gates,
                                                          const float* __restrict__ dg_part,
                                                          int dg_ld, int dg_n, int64_t Tn, int k,
                                                          int G, float* __restrict__ dsel,
                                                          const int32_t* __restrict__ idx, int E,
                                                          const int32_t* __restrict__ pairrow,
                                                          __nv_bfloat16* __restrict__ dl,
                                                          unsigned dsel_blocks,
                                                          const T* __restrict__ w, int d,
                                                          T* __restrict__ wt,
                                                          float* __restrict__ rowdsel) {
  if (blockIdx.x >= dsel_blocks) {
    const int64_t n = (int64_t)d * E;
    const int64_t stride = (int64_t)(gridDim.x - dsel_blocks) * blockDim.x;
    for (int64_t i = (blockIdx.x - dsel_blocks) * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += stride)
      wt[(i % E) * d + i / E] = w[i];
    return;
  }
  const int j = threadIdx.x & (G - 1);
  const int64_t t = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) / G;
  const bool live = t < Tn;  // every lane stays for the shuffles
  const bool own = live && j < k;
  const int64_t p = t * k + j;
  float qj = 0.f, g = 0.f;
  int32_t prow = -1;
  if (own) {
    prow = pairrow[p];
    if (prow >= 0) {
      const float* src = dg_part + p * dg_ld;
      for (int q = 0; q < dg_n; ++q) qj += src[q];
    }
    g = gates[p];
  }
  float sq = qj;
  for (int o = G / 2; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  const float v = fmaf(-g, sq, qj);
  if (own) {
    dsel[p] = v;
    if (rowdsel && prow >= 0) rowdsel[prow] = v;
  }
  if (dl) {
    if (live) {
      uint4* row = reinterpret_cast<uint4*>(dl + t * E);
      for (int e8 = j; e8 < E / 8; e8 += G) row[e8] = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncwarp();  // the zeros land before the selected entries
    if (own) {
      const int e = idx[p];
      if (e >= 0 && e < E) dl[t * E + e] = __float2bfloat16_rn(v);  // a rejected index is skipped
    }
  }
}

// dW_r partial of one token range and one group of experts (blockIdx.z:
// experts [z * EG, z * EG + EG) of E): thread i owns input dimension i and
// its column of the shared accumulator [EG][256], so the order of the adds
// is fixed; the range's (expert, dsel) pairs are staged in shared memory.
template <typename T>
__global__ void __launch_bounds__(256) router_dw_kernel(const T* __restrict__ x,
                                                        const int32_t* __restrict__ idx,
                                                        const float* __restrict__ dsel,
                                                        int64_t Tn, int d, int E, int EG, int k,
                                                        int64_t per_range, float* part) {
  extern __shared__ __align__(16) float s_acc[];  // [EG][256]
  __shared__ int s_e[256];
  __shared__ float s_ds[256];
  const int tid = threadIdx.x;
  const int i = blockIdx.y * 256 + tid;
  const int e0 = blockIdx.z * EG;
  const int ne = E - e0 < EG ? E - e0 : EG;  // experts of this group
  for (int e = 0; e < ne; ++e) s_acc[e * 256 + tid] = 0.f;
  const int64_t t0 = blockIdx.x * per_range;
  const int64_t t1 = t0 + per_range < Tn ? t0 + per_range : Tn;
  const int CH = 256 / k;
  for (int64_t tc = t0; tc < t1; tc += CH) {
    const int nt = (int)(t1 - tc < CH ? t1 - tc : CH);
    __syncthreads();
    if (tid < nt * k) {
      // a rejected index, or an expert of another group, contributes nothing
      const int e = idx[tc * k + tid];
      const bool ok = e >= e0 && e < e0 + ne;
      s_e[tid] = ok ? e - e0 : 0;
      s_ds[tid] = ok ? dsel[tc * k + tid] : 0.f;
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
    float* out = part + ((int64_t)blockIdx.x * d + i) * E + e0;
    for (int e = 0; e < ne; ++e) out[e] = s_acc[e * 256 + tid];
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

int device_sms() {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

template <typename T>
void router_dsel_t(const moe_dims& d, const Layout& L, const LayerPtrs& p, int dg_n, int dg_ld,
                   void* ws, cudaStream_t s, bool rows) {
  const int dm = d.d_model, E = d.experts, k = d.top_k;
  const int sms = device_sms();
  int G = 1;
  while (G < k) G *= 2;
  const unsigned dsel_blocks = (unsigned)((d.tokens * G + 255) / 256);
  int64_t tr_blocks = ((int64_t)dm * E + 255) / 256;
  if (tr_blocks > sms) tr_blocks = sms;
  MOE_LAUNCH("router_dsel", s,
             router_dsel_kernel<T><<<dsel_blocks + (unsigned)tr_blocks, 256, 0, s>>>(
                 p.gates, at<float>(ws, L.dg_part), dg_ld, dg_n, d.tokens, k, G,
                 at<float>(ws, L.dsel), p.topk_idx, E, at<const int32_t>(ws, L.pairrow),
                 tc_router_dw_supported(d) ? at<__nv_bfloat16>(ws, L.dl) : nullptr, dsel_blocks,
                 reinterpret_cast<const T*>(p.w_router), dm, at<T>(ws, L.wrt),
                 rows ? at<float>(ws, L.rowdsel) : nullptr));
}

template <typename T>
void router_dw_dx_t(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws,
                    cudaStream_t s, cudaEvent_t shared_done, bool term_in_rows) {
  const int dm = d.d_model, E = d.experts, k = d.top_k;
  float* dsel = at<float>(ws, L.dsel);
  float* part = at<float>(ws, L.dwr_part);
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(router_dw_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kRouterBwdSmem);
    attr_set = true;
  }
  const int sms = device_sms();
  const bool tc_dw = tc_router_dw_supported(d);
  T* wt = at<T>(ws, L.wrt);

  // the router weight gradient first: the input gradient also needs the
  // shared expert's rows, which may come from another stream
  auto input_grad = [&] {
    if (shared_done) cudaStreamWaitEvent(s, shared_done, 0);
    launch_router_dx(d, L, p, dsel, wt, ws, s, term_in_rows);
  };
  if (tc_dw) {
    tc_router_dw(d, L, p, ws, s);
    input_grad();
    return;
  }
  const int ny = (dm + 255) / 256;
  int64_t ranges = (int64_t)sms * 4 / ny;
  const int64_t by_tokens = (d.tokens + 63) / 64;
  if (ranges > by_tokens) ranges = by_tokens;
  if (ranges > kRouterBwdRanges) ranges = kRouterBwdRanges;
  if (ranges < 1) ranges = 1;
  const int64_t per_range = (d.tokens + ranges - 1) / ranges;
  // experts in groups whose accumulators fit the shared-memory budget
  const int eg_max = (int)(kRouterBwdSmem / (sizeof(float) * 256));
  const int groups = (E + eg_max - 1) / eg_max;
  const int EG = (E + groups - 1) / groups;
  MOE_LAUNCH("router_dw", s,
             router_dw_kernel<T><<<dim3((unsigned)ranges, ny, groups), 256,
                                   sizeof(float) * EG * 256, s>>>(
                 reinterpret_cast<const T*>(p.x), p.topk_idx, dsel, d.tokens, dm, E, EG, k,
                 per_range, part));
  const int64_t n = (int64_t)dm * E;
  MOE_LAUNCH("router_dw_reduce", s,
             router_dw_reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(
                 part, (int)ranges, n, p.dw_router));
  input_grad();
}

}  // namespace

void launch_router_dsel(const moe_dims& d, const Layout& L, const LayerPtrs& p, int dg_n,
                        int dg_ld, void* ws, cudaStream_t s, bool rows) {
  if (d.tokens == 0) return;
  if (d.dtype == MOE_BF16) router_dsel_t<__nv_bfloat16>(d, L, p, dg_n, dg_ld, ws, s, rows);
  else router_dsel_t<float>(d, L, p, dg_n, dg_ld, ws, s, rows);
}

void launch_router_dw_dx(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws,
                         cudaStream_t s, cudaEvent_t shared_done, bool term_in_rows) {
  if (d.tokens == 0) {
    zero_fill_f32(p.dw_router, (int64_t)d.d_model * d.experts, s);
    if (shared_done) cudaStreamWaitEvent(s, shared_done, 0);
    return;
  }
  if (d.dtype == MOE_BF16)
    router_dw_dx_t<__nv_bfloat16>(d, L, p, ws, s, shared_done, term_in_rows);
  else
    router_dw_dx_t<float>(d, L, p, ws, s, shared_done, term_in_rows);
}

void launch_router_backward(const moe_dims& d, const Layout& L, const LayerPtrs& p, int dg_n,
                            int dg_ld, void* ws, cudaStream_t s, cudaEvent_t shared_done) {
  launch_router_dsel(d, L, p, dg_n, dg_ld, ws, s, false);
  launch_router_dw_dx(d, L, p, ws, s, shared_done, false);
}

bool router_backward_supported(const moe_dims& d) {
  // the CUDA-core dW_r path takes the experts in groups that fit its
  // shared-memory accumulator, so every E the layer takes
  return d.experts >= 1 && d.experts <= kMaxExperts;
}

}  // namespace moe
