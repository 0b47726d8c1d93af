// Routing (router GEMM, top-k selection, softmax over the selected logits)
// and the counting-sort permutation of token-expert pairs.
//
// Routing: benchmark page gpu_moe_h100.json (top_k field) and the layer
// structure fixed by gpu_nn.json's parameter count: per token the k largest
// router logits, ties to the lower expert index, slots in descending order,
// gates = softmax of the selected logits.
//
// Permutation: the `sort_permute` piece of kernel_gmm_gpu.json (dispatch
// `sorted`): pairs p = t*k + j ordered by expert, stable in p, plus an
// expert-padded copy of the order in which every expert's rows start on a
// multiple of 128, or of 256 where the grouped GEMMs run CTA pairs over
// 256-row units (tiles never straddle two experts), and the token of every
// padded row.
#include "kernels.cuh"

namespace moe {

constexpr int kMaxPerLane = kMaxExperts / 32;

// ---------------------------------------------------------------------------
// Top-k from a logits matrix (fed logits, or any expert count): one warp per
// token, lane l owns logits l, l+32, ...; k rounds of a butterfly arg-max.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) topk_softmax_kernel(const float* __restrict__ logits,
                                                           int64_t T, int E, int k,
                                                           int32_t* __restrict__ idx_out,
                                                           float* __restrict__ gates_out) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int per_lane = (E + 31) >> 5;
  for (int64_t t = warp; t < T; t += nwarps) {
    float v[kMaxPerLane];
    unsigned live = 0u;  // bit j: entry lane + 32*j not yet taken
#pragma unroll
    for (int j = 0; j < kMaxPerLane; ++j) {
      const int e = lane + 32 * j;
      const bool ok = (j < per_lane) && (e < E);
      if (ok) live |= 1u << j;
      v[j] = ok ? logits[t * E + e] : -INFINITY;
    }
    float my_sel = 0.f;
    int my_idx = 0;
    float top = 0.f;
    for (int r = 0; r < k; ++r) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < kMaxPerLane; ++j) {
        const int e = lane + 32 * j;
        if (((live >> j) & 1u) && (bi == 0x7fffffff || better(v[j], e, bv, bi))) {
          bv = v[j];
          bi = e;
        }
      }
      // the order is total, so every lane ends with the same winner
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, s);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, s);
        if (oi != 0x7fffffff && (bi == 0x7fffffff || better(ov, oi, bv, bi))) {
          bv = ov;
          bi = oi;
        }
      }
      if ((bi & 31) == lane) live &= ~(1u << (bi >> 5));
      if (r == 0) top = bv;
      if (lane == r) {
        my_sel = bv;
        my_idx = bi;
      }
    }
    const float z = lane < k ? gate_exp(my_sel, top) : 0.f;
    float sum = z;
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, s);
    if (lane < k) {
      idx_out[t * k + lane] = my_idx;
      gates_out[t * k + lane] = z / sum;
    }
  }
}

void launch_topk_softmax(const float* logits, int64_t T, int E, int k, int32_t* idx,
                         float* gates, cudaStream_t s) {
  if (T == 0) return;
  int64_t blocks = (T + 7) / 8;
  if (blocks > 152 * 16) blocks = 152 * 16;
  MOE_LAUNCH("topk_softmax", s,
             topk_softmax_kernel<<<(unsigned)blocks, 256, 0, s>>>(logits, T, E, k, idx, gates));
}

// ---------------------------------------------------------------------------
// Fused router: a group of G = 8 lanes per token computes its EN logits
// (float32 accumulate; lane g takes the model dimensions g, g + 8, ...,
// W_r staged in shared memory with rows padded to EN + 4 floats, so that
// the group's eight rows fall in distinct banks), sums the lanes' partials
// by a butterfly over the group, and the group's first lane selects the top
// k in registers and writes idx / gates (and the logits when asked).
// Persistent blocks loop over 16-token groups.
// ---------------------------------------------------------------------------
constexpr int kRouterLanes = 8;  // lanes per token

template <typename T, int EN>
__global__ void __launch_bounds__(128) router_fused_kernel(const T* __restrict__ x,
                                                           const T* __restrict__ w_router,
                                                           const float* __restrict__ bias,
                                                           int64_t Tn, int d, int k,
                                                           float* __restrict__ logits_out,
                                                           int32_t* __restrict__ idx_out,
                                                           float* __restrict__ gates_out) {
  constexpr int G = kRouterLanes, LD = EN + 4;
  extern __shared__ __align__(16) float s_w[];  // [d][EN + 4]
  // W_r in 16-byte (float) / 8-byte (bf16) pieces of four, loads unrolled
#pragma unroll 4
  for (int i = threadIdx.x; i < d * EN / 4; i += blockDim.x) {
    float4 v;
    if constexpr (sizeof(T) == 4) {
      v = __ldg(reinterpret_cast<const float4*>(w_router) + i);
    } else {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(w_router) + i);
      const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
      const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
      v = make_float4(lo.x, lo.y, hi.x, hi.y);
    }
    *reinterpret_cast<float4*>(s_w + (4 * i / EN) * LD + 4 * i % EN) = v;
  }
  __syncthreads();
  const int g = threadIdx.x % G;
  const int tpb = blockDim.x / G;  // tokens per block and pass
  // the loop bound is the same for every thread of the block, so every lane
  // of a warp takes part in each pass's shuffles
  for (int64_t t0 = (int64_t)blockIdx.x * tpb; t0 < Tn; t0 += (int64_t)gridDim.x * tpb) {
    const int64_t t = t0 + threadIdx.x / G;
    const bool valid = t < Tn;
    float acc[EN];
#pragma unroll
    for (int e = 0; e < EN; ++e) acc[e] = 0.f;
    if (valid) {
      const T* xr = x + t * d;
#pragma unroll 16
      for (int kk = g; kk < d; kk += G) {
        const float xv = to_f32(__ldg(xr + kk));
        const float4* wr = reinterpret_cast<const float4*>(s_w + kk * LD);
#pragma unroll
        for (int e4 = 0; e4 < EN / 4; ++e4) {
          const float4 w4 = wr[e4];
          acc[4 * e4 + 0] = fmaf(xv, w4.x, acc[4 * e4 + 0]);
          acc[4 * e4 + 1] = fmaf(xv, w4.y, acc[4 * e4 + 1]);
          acc[4 * e4 + 2] = fmaf(xv, w4.z, acc[4 * e4 + 2]);
          acc[4 * e4 + 3] = fmaf(xv, w4.w, acc[4 * e4 + 3]);
        }
      }
    }
#pragma unroll
    for (int o = 1; o < G; o <<= 1)
#pragma unroll
      for (int e = 0; e < EN; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
    if (!valid || g != 0) continue;
    if (bias) {
#pragma unroll
      for (int e = 0; e < EN; ++e) acc[e] += __ldg(bias + e);
    }
    if (logits_out) {
      float4* lo = reinterpret_cast<float4*>(logits_out + t * EN);
#pragma unroll
      for (int e4 = 0; e4 < EN / 4; ++e4)
        lo[e4] = make_float4(acc[4 * e4], acc[4 * e4 + 1], acc[4 * e4 + 2], acc[4 * e4 + 3]);
    }
    // selection: k passes over the EN logits in registers
    unsigned long long taken = 0ull;
    float top = 0.f, sum = 0.f;
    for (int r = 0; r < k; ++r) {
      float bv = 0.f;
      int bi = -1;
#pragma unroll
      for (int e = 0; e < EN; ++e) {
        if (!((taken >> e) & 1ull) && (bi < 0 || better(acc[e], e, bv, bi))) {
          bv = acc[e];
          bi = e;
        }
      }
      taken |= 1ull << bi;
      if (r == 0) top = bv;
      const float z = gate_exp(bv, top);
      sum += z;
      idx_out[t * k + r] = bi;
      gates_out[t * k + r] = z;
    }
    for (int r = 0; r < k; ++r) gates_out[t * k + r] = gates_out[t * k + r] / sum;
  }
}

template <typename T, int EN>
static void router_fused_t(const moe_dims& dm, const void* x, const void* w, const float* bias,
                           float* logits_out, int32_t* idx, float* gates, cudaStream_t s) {
  const size_t smem = sizeof(float) * dm.d_model * (EN + 4);
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(router_fused_kernel<T, EN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         160 * 1024);
    attr = true;
  }
  int64_t blocks = (dm.tokens + 128 / kRouterLanes - 1) / (128 / kRouterLanes);
  const int64_t cap = EN >= 32 ? 152 : 152 * 8;  // amortise the W_r staging for wide routers
  if (blocks > cap) blocks = cap;
  MOE_LAUNCH("router_fused", s,
             (router_fused_kernel<T, EN><<<(unsigned)blocks, 128, smem, s>>>(
                 reinterpret_cast<const T*>(x), reinterpret_cast<const T*>(w), bias, dm.tokens,
                 dm.d_model, dm.top_k, logits_out, idx, gates)));
}

bool router_fused_supported(const moe_dims& d) {
  const int E = d.experts;
  return (E == 8 || E == 16 || E == 32 || E == 64) &&
         (size_t)d.d_model * (E + 4) * sizeof(float) <= 160 * 1024;
}

void launch_router_fused(const moe_dims& d, const void* x, const void* w, const float* bias,
                         float* logits_out, int32_t* idx, float* gates, cudaStream_t s) {
  if (d.tokens == 0) return;
  const bool bf = d.dtype == MOE_BF16;
  switch (d.experts) {
    case 8:
      bf ? router_fused_t<__nv_bfloat16, 8>(d, x, w, bias, logits_out, idx, gates, s)
         : router_fused_t<float, 8>(d, x, w, bias, logits_out, idx, gates, s);
      break;
    case 16:
      bf ? router_fused_t<__nv_bfloat16, 16>(d, x, w, bias, logits_out, idx, gates, s)
         : router_fused_t<float, 16>(d, x, w, bias, logits_out, idx, gates, s);
      break;
    case 32:
      bf ? router_fused_t<__nv_bfloat16, 32>(d, x, w, bias, logits_out, idx, gates, s)
         : router_fused_t<float, 32>(d, x, w, bias, logits_out, idx, gates, s);
      break;
    default:
      bf ? router_fused_t<__nv_bfloat16, 64>(d, x, w, bias, logits_out, idx, gates, s)
         : router_fused_t<float, 64>(d, x, w, bias, logits_out, idx, gates, s);
      break;
  }
}

// ---------------------------------------------------------------------------
// Counting sort.  Warp w owns pairs [w*kPermChunk, (w+1)*kPermChunk) and
// walks them in rounds of 32; within a round, lanes holding the same expert
// find each other with __match_any_sync, so a pair's rank inside its warp
// chunk is (earlier rounds' count for its expert) + (lower lanes with the
// same expert).  Both passes run the same walk, so the ranks agree.
// ---------------------------------------------------------------------------
template <bool SCATTER>
__device__ __forceinline__ void walk_chunk(const int32_t* __restrict__ idx, int64_t P, int E,
                                           int k, int64_t chunk, int* hist, const int* base_e,
                                           const int* off_e, const int* poff_e, int32_t* perm,
                                           int32_t* inv_perm, int32_t* rowpair, int32_t* pairrow,
                                           int capacity, int* status) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  // every round's expert index is loaded before the walk starts
  int ev[kPermRounds];
#pragma unroll
  for (int r = 0; r < kPermRounds; ++r) {
    const int64_t p = chunk * kPermChunk + (int64_t)r * 32 + lane;
    ev[r] = p < P ? __ldg(idx + p) : -1;
  }
#pragma unroll
  for (int r = 0; r < kPermRounds; ++r) {
    const int64_t p = chunk * kPermChunk + (int64_t)r * 32 + lane;
    int e = -1;
    if (p < P) {
      e = ev[r];
      if (e < 0 || e >= E) {
        report_error(status, MOE_ERR_DEVICE_CHECK, 1);
        e = -1;
      }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int before = __popc(peers & lt);
    int rank = 0;
    if (e >= 0) rank = hist[e] + before;
    __syncwarp();
    if (e >= 0 && before == 0) hist[e] += __popc(peers);
    __syncwarp();
    // rank of the pair inside its expert, in increasing pair id
    const int within = SCATTER && e >= 0 ? base_e[e] + rank : 0;
    // a rejected index, or a pair past its expert's capacity: no sorted
    // position and no row (every consumer of the row map skips it)
    const bool dropped = e < 0 || (capacity > 0 && within >= capacity);
    if (SCATTER && p < P && dropped) {
      pairrow[p] = -1;
      inv_perm[p] = -1;
    }
    if (SCATTER && !dropped) {
      const int pos = off_e[e] + within;
      const int ppos = poff_e[e] + within;
      perm[pos] = (int32_t)p;
      inv_perm[p] = pos;
      rowpair[ppos] = (int32_t)p;
      pairrow[p] = ppos;
    }
  }
}

__global__ void __launch_bounds__(256) perm_hist_kernel(const int32_t* __restrict__ idx, int64_t P,
                                                        int E, int k, int64_t NW,
                                                        int* warp_counts, int* status) {
  __shared__ int hist[8][kMaxExperts];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t chunk = (int64_t)blockIdx.x * 8 + w;
  for (int e = lane; e < E; e += 32) hist[w][e] = 0;
  __syncwarp();
  if (chunk >= NW) return;
  walk_chunk<false>(idx, P, E, k, chunk, hist[w], nullptr, nullptr, nullptr, nullptr, nullptr,
                    nullptr, nullptr, 0, status);
  for (int e = lane; e < E; e += 32) warp_counts[chunk * E + e] = hist[w][e];
}

// Exclusive scan of column e of warp_counts (one block per expert).
__global__ void __launch_bounds__(1024) perm_colscan_kernel(const int* __restrict__ warp_counts,
                                                            int64_t NW, int E, int* warp_base,
                                                            int* counts_ws) {
  __shared__ int part[1024];
  const int e = blockIdx.x;
  const int tid = threadIdx.x;
  const int64_t per = (NW + 1023) / 1024;
  const int64_t lo = tid * per;
  const int64_t hi = lo + per < NW ? lo + per : NW;
  int s = 0;
  for (int64_t w = lo; w < hi; ++w) s += warp_counts[w * E + e];
  part[tid] = s;
  __syncthreads();
  // Hillis-Steele inclusive scan over 1024 partials
  for (int o = 1; o < 1024; o <<= 1) {
    int v = tid >= o ? part[tid - o] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  int run = tid ? part[tid - 1] : 0;
  for (int64_t w = lo; w < hi; ++w) {
    const int c = warp_counts[w * E + e];
    warp_base[w * E + e] = run;
    run += c;
  }
  if (tid == 1023) counts_ws[e] = part[1023];
}

// Offsets, padded offsets, the tile list and the padding rows (one block of
// 1024 threads).  With a capacity the counts become the kept counts (in the
// workspace too: the weight-gradient GEMMs take their K ranges from there),
// and perm past the kept rows reads -1.  It also starts the invocation's
// device status (an index the histogram pass rejected is rejected again by
// the scatter pass) and the combine's block ticket.  s_off / s_poff receive
// the offsets the scatter pass uses.
__device__ void finalize_block(int* __restrict__ counts_ws, int E, int capacity, int pad, int64_t P,
                               int32_t* counts_out, int32_t* offsets_out, int* poff, int4* tiles,
                               int* ntiles, int32_t* rowpair, int32_t* perm, int* status,
                               int* loss_tick, int* s_off, int* s_poff) {
  __shared__ int s_toff[kMaxExperts + 1];
  __shared__ int s_cnt[kMaxExperts];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int e = tid; e < E; e += blockDim.x) {
    const int c = counts_ws[e];
    s_cnt[e] = capacity > 0 && c > capacity ? capacity : c;
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scans of the counts, padded rows and tiles, 32 experts a round
    int o = 0, po = 0, to = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int c = e < E ? s_cnt[e] : 0;
      // padded to `pad` rows, listed as kTileRows-row tiles (the last
      // one of an expert may hold no rows when pad = 256)
      const int np = (c + pad - 1) / pad;
      const int nt = np * (pad / kTileRows);
      int ic = c, ip = np * pad, it = nt;  // inclusive scans over the lanes
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int vc = __shfl_up_sync(0xffffffffu, ic, d);
        const int vp = __shfl_up_sync(0xffffffffu, ip, d);
        const int vt = __shfl_up_sync(0xffffffffu, it, d);
        if (lane >= d) {
          ic += vc;
          ip += vp;
          it += vt;
        }
      }
      if (e < E) {
        s_off[e] = o + ic - c;
        s_poff[e] = po + ip - np * pad;
        s_toff[e] = to + it - nt;
      }
      o += __shfl_sync(0xffffffffu, ic, 31);
      po += __shfl_sync(0xffffffffu, ip, 31);
      to += __shfl_sync(0xffffffffu, it, 31);
    }
    if (lane == 0) {
      s_off[E] = o;
      s_poff[E] = po;
      s_toff[E] = to;
      ntiles[0] = to;
      ntiles[1] = po;
      status[0] = 0;
      status[1] = 0;
      *loss_tick = 0;
    }
  }
  __syncthreads();
  for (int e = tid; e <= E; e += blockDim.x) {
    offsets_out[e] = s_off[e];
    poff[e] = s_poff[e];
    if (e < E) {
      counts_out[e] = s_cnt[e];
      counts_ws[e] = s_cnt[e];
    }
  }
  for (int64_t r = s_off[E] + tid; r < P; r += blockDim.x) perm[r] = -1;  // past the kept rows
  // one warp per expert: its tiles, and the padding rows of its last tile
  for (int e = warp; e < E; e += blockDim.x >> 5) {
    const int c = s_cnt[e];
    const int nt = s_toff[e + 1] - s_toff[e];
    for (int j = lane; j < nt; j += 32) {
      const int valid = max(0, min(kTileRows, c - j * kTileRows));
      tiles[s_toff[e] + j] = make_int4(e, s_poff[e] + j * kTileRows, valid, 0);
    }
    for (int r = s_poff[e] + c + lane; r < s_poff[e + 1]; r += 32) rowpair[r] = -1;
  }
}

__global__ void __launch_bounds__(1024) perm_finalize_kernel(int* __restrict__ counts_ws, int E,
                                                             int capacity, int pad, int64_t P,
                                                             int32_t* counts_out,
                                                             int32_t* offsets_out, int* poff,
                                                             int4* tiles, int* ntiles,
                                                             int32_t* rowpair, int32_t* perm,
                                                             int* status, int* loss_tick) {
  __shared__ int s_off[kMaxExperts + 1], s_poff[kMaxExperts + 1];
  finalize_block(counts_ws, E, capacity, pad, P, counts_out, offsets_out, poff, tiles, ntiles, rowpair,
                 perm, status, loss_tick, s_off, s_poff);
}

__global__ void __launch_bounds__(256) perm_scatter_kernel(
    const int32_t* __restrict__ idx, int64_t P, int E, int k, int64_t NW,
    const int* __restrict__ warp_base, const int32_t* __restrict__ offsets,
    const int* __restrict__ poff, int32_t* perm, int32_t* inv_perm, int32_t* rowpair,
    int32_t* pairrow, int capacity, int* status) {
  __shared__ int hist[8][kMaxExperts];
  __shared__ int s_off[kMaxExperts], s_poff[kMaxExperts];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    s_off[e] = offsets[e];
    s_poff[e] = poff[e];
  }
  for (int e = lane; e < E; e += 32) hist[w][e] = 0;
  __syncthreads();
  const int64_t chunk = (int64_t)blockIdx.x * 8 + w;
  if (chunk >= NW) return;
  walk_chunk<true>(idx, P, E, k, chunk, hist[w], warp_base + chunk * E, s_off, s_poff, perm,
                   inv_perm, rowpair, pairrow, capacity, status);
}

void launch_permute(const moe_dims& d, const Layout& L, const int32_t* idx, int32_t* counts,
                    int32_t* offsets, int32_t* perm, int32_t* inv_perm, void* ws,
                    cudaStream_t s) {
  const int E = d.experts, k = d.top_k;
  int* status = at<int>(ws, L.status);
  int* warp_counts = at<int>(ws, L.warp_counts);
  int* warp_base = at<int>(ws, L.warp_base);
  int* counts_ws = at<int>(ws, L.counts);
  int* poff = at<int>(ws, L.poff);
  int32_t* rowpair = at<int32_t>(ws, L.rowpair);
  int4* tiles = at<int4>(ws, L.tiles);
  int* ntiles = at<int>(ws, L.ntiles);
  const int64_t NW = L.NWc;
  const unsigned blocks = (unsigned)((NW + 7) / 8);
  if (NW > 0) {
    MOE_LAUNCH("perm_hist", s,
               perm_hist_kernel<<<blocks, 256, 0, s>>>(idx, L.P, E, k, NW, warp_counts, status));
    MOE_LAUNCH("perm_colscan", s,
               perm_colscan_kernel<<<E, 1024, 0, s>>>(warp_counts, NW, E, warp_base, counts_ws));
  } else {
    zero_fill_i32(counts_ws, E, s);
  }
  MOE_LAUNCH("perm_finalize", s,
             perm_finalize_kernel<<<1, 1024, 0, s>>>(counts_ws, E, d.capacity, row_pad(d), L.P, counts,
                                                     offsets, poff, tiles, ntiles, rowpair,
                                                     perm, status, at<int>(ws, L.loss_tick)));
  if (NW > 0)
    MOE_LAUNCH("perm_scatter", s,
               perm_scatter_kernel<<<blocks, 256, 0, s>>>(idx, L.P, E, k, NW, warp_base, offsets,
                                                          poff, perm, inv_perm, rowpair,
                                                          at<int32_t>(ws, L.pairrow), d.capacity,
                                                          status));
}

}  // namespace moe
