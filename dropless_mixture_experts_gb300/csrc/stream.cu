// Row-streaming kernels of the layer: the expert-sorted copy of token rows
// (the permute piece of kernel_gmm_gpu.json), the combine of the pairs'
// gate-weighted expert outputs with the train step's value (unpermute_combine
// there; value_and_grad in gpu_moe_h100.json), and the input gradient of the
// router backward.  All three are HBM-bound moves of whole rows.
//
// One thread owns one 16-byte chunk of one token row per item (consecutive
// threads on consecutive chunks, so a warp moves 512 contiguous bytes of a
// row per access).  An item's row indices are loaded one item ahead, and
// every row load of an item is issued before the first use, so each thread
// keeps k+2 loads in flight and no load waits on an index load.
#include <mutex>

#include "kernels.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

// Resident blocks per SM of a kernel at kThreads threads (cached per kernel).
int resident_blocks(const void* kernel) {
  static std::mutex mu;
  static const void* keys[64];
  static int vals[64];
  static int n = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (keys[i] == kernel) return vals[i];
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, 0) != cudaSuccess ||
      occ < 1)
    occ = 1;
  if (n < 64) {
    keys[n] = kernel;
    vals[n++] = occ;
  }
  return occ;
}

// Grid of a grid-stride launch: `waves` whole waves of the kernel's resident
// blocks on the SMs the launch may fill, every thread looping over its items
// (no partial last wave; one wave measured fastest for the gathering sums,
// four for the row copy).  capped = false: per SM of the device, for a
// launch whose reduction order follows its grid and must not depend on the
// SM limit.
template <class K>
unsigned stream_grid(K kernel, int64_t items, int64_t cap, bool capped = true, int waves = 1) {
  int sms = tcg_launch_sms();
  if (!capped) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  }
  int64_t b = (items + kThreads - 1) / kThreads;
  const int64_t full =
      (int64_t)sms * resident_blocks(reinterpret_cast<const void*>(kernel)) * waves;
  if (b > full) b = full;
  if (b > cap) b = cap;
  if (b < 1) b = 1;
  return (unsigned)b;
}

// 16 bytes of storage elements as floats, and back
template <typename T>
__device__ __forceinline__ void cvt16(const uint4 u, float (&v)[16 / sizeof(T)]) {
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
__device__ __forceinline__ void st16(void* p, const float (&v)[16 / sizeof(T)]) {
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



__device__ __forceinline__ uint4 ldg16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// ---- expert-sorted row copy ---------------------------------------------------
// out[pairrow[t*k + j]] = src[t] for every slot j (with gates: the row
// scaled by the pair's gate, g_tj src[t], rounded to the storage type): each
// token row is read once and written to its k sorted rows (reading in sorted
// order instead would fetch a row k times once the rows outgrow the L2).
// The padding rows of each expert, [poff[e] + counts[e], poff[e+1]), are
// zeroed by the items past the tokens' (the grouped GEMMs read them; zero
// rows give zero contributions to every weight gradient).
// ROWGATE (unscaled copies): the first chunk's item of a row also stores the
// row's gate (0 for a padding row) into rowgate.
template <typename T, bool SCALE, bool ROWGATE = false>
__global__ void __launch_bounds__(kThreads)
    scatter_rows_kernel(const uint4* __restrict__ src, const int32_t* __restrict__ pairrow,
                        const float* __restrict__ gates, uint4* __restrict__ out, int64_t Tn,
                        int cpt, int k, const int32_t* __restrict__ poff,
                        const int32_t* __restrict__ counts, int E, int pad,
                        float* __restrict__ rowgate = nullptr) {
  const int64_t n = Tn * cpt;
  const int64_t per_e = (int64_t)(pad - 1) * cpt;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n + E * per_e;
       i += stride) {
    if (i < n) {
      const int64_t t = i / cpt;
      const int c = (int)(i % cpt);
      const uint4 v = __ldg(src + i);
      for (int j = 0; j < k; ++j) {
        const int64_t r = __ldg(pairrow + t * k + j);
        if (r < 0) continue;  // a pair without a row (a rejected index) is skipped
        if constexpr (SCALE) {
          constexpr int VE = 16 / sizeof(T);
          const float g = __ldg(gates + t * k + j);
          float f[VE];
          cvt16<T>(v, f);
#pragma unroll
          for (int q = 0; q < VE; ++q) f[q] *= g;
          st16<T>(out + r * cpt + c, f);
        } else {
          out[r * cpt + c] = v;
          if (ROWGATE && c == 0) rowgate[r] = __ldg(gates + t * k + j);
        }
      }
    } else {
      const int64_t q = i - n;
      const int e = (int)(q / per_e);
      const int64_t r = (int64_t)poff[e] + counts[e] + (q % per_e) / cpt;
      if (r < poff[e + 1]) {
        out[r * cpt + q % cpt] = make_uint4(0u, 0u, 0u, 0u);
        if (ROWGATE && q % cpt == 0) rowgate[r] = 0.f;
      }
    }
  }
}

// ---- combine ------------------------------------------------------------------
// y[t] = ys[t] + sum_j osort[pairrow[t*k + j]] in slot order, cast to the
// storage type, and the block's share of sum(y * G).  The first KM slots'
// rows are indexed one item ahead; slots past KM (k > 8) load inline.
template <typename T, int KM>
__global__ void __launch_bounds__(kThreads)
    combine_kernel(const T* __restrict__ osort, const int32_t* __restrict__ pairrow,
                   const T* __restrict__ ys, T* __restrict__ y, const T* __restrict__ G,
                   int64_t Tn, int d, int k, float* __restrict__ loss_part,
                   int* __restrict__ loss_tick, float* __restrict__ loss) {
  constexpr int VE = 16 / sizeof(T);
  __shared__ float red[kThreads / 32];
  const int cpt = d / VE;
  const int64_t n = Tn * cpt;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  float lacc = 0.f;
  int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  int nxt[KM];
  auto index_ahead = [&](int64_t ii) {
    const int32_t* pr = pairrow + (ii / cpt) * k;
#pragma unroll
    for (int j = 0; j < KM; ++j) nxt[j] = j < k ? __ldg(pr + j) : 0;
  };
  if (i < n) index_ahead(i);
  for (; i < n; i += stride) {
    const int64_t t = i / cpt;
    const int64_t col = (i % cpt) * VE;
    int rows[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j) rows[j] = nxt[j];
    const uint4 us = ys ? ldg16(ys + t * d + col) : make_uint4(0u, 0u, 0u, 0u);
    const uint4 ug = G ? ldg16(G + t * d + col) : make_uint4(0u, 0u, 0u, 0u);
    uint4 v[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j)
      if (j < k && rows[j] >= 0) v[j] = ldg16(osort + (int64_t)rows[j] * d + col);
    if (i + stride < n) index_ahead(i + stride);
    float acc[VE];
    if (ys) {
      cvt16<T>(us, acc);
    } else {
#pragma unroll
      for (int q = 0; q < VE; ++q) acc[q] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      if (j < k && rows[j] >= 0) {
        float f[VE];
        cvt16<T>(v[j], f);
#pragma unroll
        for (int q = 0; q < VE; ++q) acc[q] += f[q];
      }
    }
    for (int j0 = KM; j0 < k; j0 += KM) {  // k > KM: further slots, in order
#pragma unroll
      for (int j = 0; j < KM; ++j) {
        rows[j] = j0 + j < k ? __ldg(pairrow + t * k + j0 + j) : -1;
        if (rows[j] >= 0) v[j] = ldg16(osort + (int64_t)rows[j] * d + col);
      }
#pragma unroll
      for (int j = 0; j < KM; ++j) {
        if (rows[j] >= 0) {
          float f[VE];
          cvt16<T>(v[j], f);
#pragma unroll
          for (int q = 0; q < VE; ++q) acc[q] += f[q];
        }
      }
    }
    st16<T>(y + t * d + col, acc);
    if (G) {
      float g[VE];
      cvt16<T>(ug, g);
#pragma unroll
      for (int q = 0; q < VE; ++q) lacc = fmaf(to_f32(from_f32<T>(acc[q])), g[q], lacc);
    }
  }
  if (!G) return;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lacc += __shfl_xor_sync(0xffffffffu, lacc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = lacc;
  __syncthreads();
  __shared__ int last;
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) s += red[w];
    loss_part[blockIdx.x] = s;
    __threadfence();  // the partial before the ticket
    last = atomicAdd(loss_tick, 1) == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (!last || threadIdx.x >= 32 || !loss) return;
  // the last block: fixed-order reduction of the partials (lane l sums
  // part[l], part[l + 32], ...; then a fixed butterfly)
  __threadfence();
  float s = 0.f;
  for (int i = threadIdx.x; i < (int)gridDim.x; i += 32) s += __ldcg(loss_part + i);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (threadIdx.x == 0) {
    *loss = s;
    *loss_tick = 0;  // ready for the next call
  }
}

// ---- router backward: input gradient ------------------------------------------
// dx[t] = dxs[t] + sum_j (dxsort[pairrow[t*k + j]] + dsel[t, j] W_r[:, e_j]),
// the pair rows in slot order; W_r^T [E, d] rows come through the cache.
// A capacity-dropped slot has no row but keeps its router term (the softmax
// couples it to the kept slots); a rejected index (e outside [0, E)) has
// neither.  The first KM slots' indices and logit gradients are loaded one
// item ahead.  TERM_IN_ROWS: the pair rows already hold their router term
// (the tensor-core input-gradient GEMM adds it), which is then added here
// for the slots without a row only.
constexpr int kNoRow = 1 << 16;  // router_dx: the slot's pair has no row (E <= 256)

template <typename T, int KM, bool TERM_IN_ROWS>
__global__ void __launch_bounds__(kThreads)
    router_dx_kernel(const int32_t* __restrict__ idx, const float* __restrict__ dsel,
                     const T* __restrict__ wt, const T* __restrict__ dxsort,
                     const int32_t* __restrict__ pairrow, const T* __restrict__ dxs,
                     T* __restrict__ dx, int64_t Tn, int d, int k, int E) {
  constexpr int VE = 16 / sizeof(T);
  const int cpt = d / VE;
  const int64_t n = Tn * cpt;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  int nr[KM], ne[KM];
  float nd[KM];
  auto index_ahead = [&](int64_t ii) {
    const int64_t p0 = (ii / cpt) * k;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      const bool ok = j < k;
      nr[j] = ok ? __ldg(pairrow + p0 + j) : 0;
      ne[j] = ok ? __ldg(idx + p0 + j) : 0;
      nd[j] = ok ? __ldg(dsel + p0 + j) : 0.f;
    }
  };
  if (i < n) index_ahead(i);
  for (; i < n; i += stride) {
    const int64_t t = i / cpt;
    const int64_t col = (i % cpt) * VE;
    int ex[KM];
    float ds[KM];
    uint4 v[KM];  // zero for a slot without a row
    const uint4 us = dxs ? ldg16(dxs + t * d + col) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      // ex: the expert, with kNoRow set for a slot without a row; -1 for no
      // slot or a rejected index (nothing to add)
      ex[j] = j < k && (unsigned)ne[j] < (unsigned)E ? ne[j] | (nr[j] < 0 ? kNoRow : 0) : -1;
      ds[j] = nd[j];
      if (ex[j] >= 0 && !(ex[j] & kNoRow)) v[j] = ldg16(dxsort + (int64_t)nr[j] * d + col);
    }
    if (i + stride < n) index_ahead(i + stride);
    float acc[VE];
    if (dxs) {
      cvt16<T>(us, acc);
    } else {
#pragma unroll
      for (int q = 0; q < VE; ++q) acc[q] = 0.f;
    }
    // slot j adds its row (when it has one) and its router term
    auto add_slot = [&](int j) {
      if (ex[j] < 0) return;
      float fv[VE], fw[VE];
      if (TERM_IN_ROWS && !(ex[j] & kNoRow)) {
        cvt16<T>(v[j], fv);
#pragma unroll
        for (int q = 0; q < VE; ++q) acc[q] += fv[q];
        return;
      }
      if (ex[j] & kNoRow) {
#pragma unroll
        for (int q = 0; q < VE; ++q) fv[q] = 0.f;
      } else {
        cvt16<T>(v[j], fv);
      }
      cvt16<T>(ldg16(wt + (int64_t)(ex[j] & ~kNoRow) * d + col), fw);
#pragma unroll
      for (int q = 0; q < VE; ++q) acc[q] += fmaf(ds[j], fw[q], fv[q]);
    };
#pragma unroll
    for (int j = 0; j < KM; ++j) add_slot(j);
    for (int j0 = KM; j0 < k; j0 += KM) {  // k > KM: further slots, in order
#pragma unroll
      for (int j = 0; j < KM; ++j) {
        ex[j] = -1;
        if (j0 + j < k) {
          const int64_t p = t * k + j0 + j;
          const int e = __ldg(idx + p);
          const int64_t r = __ldg(pairrow + p);
          ex[j] = (unsigned)e < (unsigned)E ? e | (r < 0 ? kNoRow : 0) : -1;
          ds[j] = __ldg(dsel + p);
          if (r >= 0) v[j] = ldg16(dxsort + r * d + col);
        }
      }
#pragma unroll
      for (int j = 0; j < KM; ++j) add_slot(j);
    }
    st16<T>(dx + t * d + col, acc);
  }
}

// Slots whose indices are loaded ahead: the power of two >= k, at most 8.
int slots_ahead(int k) { return k <= 1 ? 1 : k <= 2 ? 2 : k <= 4 ? 4 : 8; }

template <typename T>
void combine_t(const moe_dims& d, const Layout& L, void* y, const void* G, float* loss, void* ws,
               cudaStream_t s) {
  float* part = G ? at<float>(ws, L.loss_part) : nullptr;
  const T* ys = d.shared_hidden > 0 ? at<const T>(ws, L.ys) : nullptr;
  const int64_t items = d.tokens * (d.d_model / (16 / (int)sizeof(T)));
  // the loss partials are summed in block order: the grid must not follow
  // the SM limit
  auto launch = [&](auto kernel) {
    const unsigned blocks = stream_grid(kernel, items, kLossBlocks, false);
    MOE_LAUNCH("combine", s,
               kernel<<<blocks, kThreads, 0, s>>>(
                   at<const T>(ws, L.osort), at<const int32_t>(ws, L.pairrow), ys,
                   reinterpret_cast<T*>(y), reinterpret_cast<const T*>(G), d.tokens, d.d_model,
                   d.top_k, part, at<int>(ws, L.loss_tick), loss));
  };
  switch (slots_ahead(d.top_k)) {
    case 1: launch(combine_kernel<T, 1>); break;
    case 2: launch(combine_kernel<T, 2>); break;
    case 4: launch(combine_kernel<T, 4>); break;
    default: launch(combine_kernel<T, 8>); break;
  }

}

template <typename T>
void router_dx_t(const moe_dims& d, const Layout& L, const LayerPtrs& p, const float* dsel,
                 const void* wt, void* ws, cudaStream_t s, bool term_in_rows) {
  const T* dxs = d.shared_hidden > 0 ? at<const T>(ws, L.dxs) : nullptr;
  const int64_t items = d.tokens * (d.d_model / (16 / (int)sizeof(T)));
  // the whole device's wave: this sum runs after the shared expert's part
  // (moe_backward_routed waits for it first), whatever the launch's SM limit
  auto launch = [&](auto kernel) {
    const unsigned blocks = stream_grid(kernel, items, INT32_MAX, false);
    MOE_LAUNCH("router_dx", s,
               kernel<<<blocks, kThreads, 0, s>>>(
                   p.topk_idx, dsel, reinterpret_cast<const T*>(wt), at<const T>(ws, L.dxsort),
                   at<const int32_t>(ws, L.pairrow), dxs, reinterpret_cast<T*>(p.dx), d.tokens,
                   d.d_model, d.top_k, d.experts));
  };
  switch (slots_ahead(d.top_k)) {
    case 1: term_in_rows ? launch(router_dx_kernel<T, 1, true>) : launch(router_dx_kernel<T, 1, false>); break;
    case 2: term_in_rows ? launch(router_dx_kernel<T, 2, true>) : launch(router_dx_kernel<T, 2, false>); break;
    case 4: term_in_rows ? launch(router_dx_kernel<T, 4, true>) : launch(router_dx_kernel<T, 4, false>); break;
    default: term_in_rows ? launch(router_dx_kernel<T, 8, true>) : launch(router_dx_kernel<T, 8, false>); break;
  }
}

}  // namespace

void launch_scatter_rows(const moe_dims& d, const Layout& L, const void* src, void* out, void* ws,
                         cudaStream_t s, const float* gates, float* rowgate) {
  if (d.tokens == 0) return;
  const int cpt = (int)((int64_t)d.d_model * L.elem / 16);
  const int pad = row_pad(d);
  const int64_t items = d.tokens * cpt + (int64_t)d.experts * (pad - 1) * cpt;
  auto launch = [&](auto kernel) {
    MOE_LAUNCH("scatter_rows", s,
               kernel<<<stream_grid(kernel, items, INT32_MAX, true, 4), kThreads, 0, s>>>(
                   reinterpret_cast<const uint4*>(src), at<const int32_t>(ws, L.pairrow), gates,
                   reinterpret_cast<uint4*>(out), d.tokens, cpt, d.top_k,
                   at<const int32_t>(ws, L.poff), at<const int32_t>(ws, L.counts), d.experts,
                   pad, rowgate));
  };
  if (rowgate) launch(scatter_rows_kernel<__nv_bfloat16, false, true>);
  else if (!gates) launch(scatter_rows_kernel<__nv_bfloat16, false>);
  else if (d.dtype == MOE_BF16) launch(scatter_rows_kernel<__nv_bfloat16, true>);
  else launch(scatter_rows_kernel<float, true>);
}

void launch_combine(const moe_dims& d, const Layout& L, void* y, const void* upstream, float* loss,
                    void* ws, cudaStream_t s) {
  if (d.tokens == 0) {
    if (upstream && loss) zero_fill_f32(loss, 1, s);
    return;
  }
  if (d.dtype == MOE_BF16) combine_t<__nv_bfloat16>(d, L, y, upstream, loss, ws, s);
  else combine_t<float>(d, L, y, upstream, loss, ws, s);
}

void launch_router_dx(const moe_dims& d, const Layout& L, const LayerPtrs& p, const float* dsel,
                      const void* wt, void* ws, cudaStream_t s, bool term_in_rows) {
  if (d.tokens == 0) return;
  if (d.dtype == MOE_BF16) router_dx_t<__nv_bfloat16>(d, L, p, dsel, wt, ws, s, term_in_rows);
  else router_dx_t<float>(d, L, p, dsel, wt, ws, s, term_in_rows);
}

}  // namespace moe
