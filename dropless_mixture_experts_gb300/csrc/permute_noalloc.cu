// moe_permute_noalloc: the counting sort of moe_permute (counts, offsets,
// perm, inv_perm) for callers that cannot allocate device memory.  Its
// scratch (per-warp-chunk expert histograms and their prefix sums) lives in
// one fixed-size array inside the library instead of a caller workspace.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it until the process exits, every call shares it, and each
// call overwrites what the previous one left (nothing in it has to start at
// zero: every entry a call reads was written earlier in that same call).
// Calls that overlap on the GPU (different streams, or different host
// threads without ordering) race on it.
//
// An expert index outside [0, E) gets what moe_permute gives it: no sorted
// position (inv_perm = -1), and perm reads -1 past offsets[E].  Unlike
// moe_permute, which records MOE_ERR_DEVICE_CHECK in its workspace, this
// entry has no status word a caller could read: the -1 entries are the
// only sign.
#include <mutex>

#include "kernels.cuh"

namespace moe {
namespace {

constexpr int kNaRounds = 16;              // 32-pair rounds per warp chunk
constexpr int kNaChunk = 32 * kNaRounds;   // pairs per warp chunk
constexpr int64_t kNaHist = int64_t(1) << 19;  // max (warp chunks) x (experts)
constexpr int kNaOff = 64;                 // ints [64, 64 + 257): expert offsets, then
                                           // the number of sorted pairs
constexpr int kNaHistAt = 64 + 320;        // ints: histograms, then their prefix sums
constexpr int64_t kNaInts = kNaHistAt + 2 * kNaHist;

// 4 MiB + 1.5 KiB of device memory per GPU that loads the library
static __device__ __align__(256) int g_noalloc_scratch[kNaInts];

// Rank of each pair inside its warp chunk among pairs of the same expert:
// earlier rounds' count plus the lower lanes of this round with that expert.
template <bool SCATTER>
__device__ __forceinline__ void na_walk(const int32_t* __restrict__ idx, int64_t P, int E,
                                        int64_t chunk, int* hist, const int* base_e,
                                        const int* off_e, int32_t* perm, int32_t* inv_perm) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  for (int r = 0; r < kNaRounds; ++r) {
    const int64_t p = chunk * kNaChunk + (int64_t)r * 32 + lane;
    int e = -1;
    if (p < P) {
      e = idx[p];
      if (e < 0 || e >= E) {
        e = -1;  // rejected: no sorted position
        if (SCATTER) inv_perm[p] = -1;
      }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int before = __popc(peers & lt);
    int rank = 0;
    if (e >= 0) rank = hist[e] + before;
    __syncwarp();
    if (e >= 0 && before == 0) hist[e] += __popc(peers);
    __syncwarp();
    if (SCATTER && e >= 0) {
      const int pos = off_e[e] + base_e[e] + rank;
      perm[pos] = (int32_t)p;
      inv_perm[p] = pos;
    }
  }
}

__global__ void __launch_bounds__(256) na_hist_kernel(const int32_t* __restrict__ idx, int64_t P,
                                                      int E, int64_t NW, int* scratch) {
  __shared__ int hist[8][kMaxExperts];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t chunk = (int64_t)blockIdx.x * 8 + w;
  for (int e = lane; e < E; e += 32) hist[w][e] = 0;
  __syncwarp();
  if (chunk >= NW) return;
  na_walk<false>(idx, P, E, chunk, hist[w], nullptr, nullptr, nullptr, nullptr);
  int* out = scratch + kNaHistAt;
  for (int e = lane; e < E; e += 32) out[chunk * E + e] = hist[w][e];
}

// Column e: exclusive prefix over the warp chunks, and the expert's total.
__global__ void __launch_bounds__(1024) na_scan_kernel(int64_t NW, int E, int* scratch,
                                                       int32_t* counts) {
  __shared__ int part[1024];
  const int* hist = scratch + kNaHistAt;
  int* base = scratch + kNaHistAt + kNaHist;
  const int e = blockIdx.x, tid = threadIdx.x;
  const int64_t per = (NW + 1023) / 1024;
  const int64_t lo = tid * per;
  const int64_t hi = lo + per < NW ? lo + per : NW;
  int s = 0;
  for (int64_t w = lo; w < hi; ++w) s += hist[w * E + e];
  part[tid] = s;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {
    const int v = tid >= o ? part[tid - o] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  int run = tid ? part[tid - 1] : 0;
  for (int64_t w = lo; w < hi; ++w) {
    base[w * E + e] = run;
    run += hist[w * E + e];
  }
  if (tid == 1023) counts[e] = part[1023];
}

__global__ void na_offsets_kernel(const int32_t* __restrict__ counts, int E, int* scratch,
                                  int32_t* offsets) {
  if (threadIdx.x != 0) return;
  int o = 0;
  for (int e = 0; e < E; ++e) {
    scratch[kNaOff + e] = o;
    offsets[e] = o;
    o += counts[e];
  }
  offsets[E] = o;
  scratch[kNaOff + E] = o;
}

__global__ void __launch_bounds__(256) na_scatter_kernel(const int32_t* __restrict__ idx,
                                                         int64_t P, int E, int64_t NW,
                                                         int* scratch, int32_t* perm,
                                                         int32_t* inv_perm) {
  __shared__ int hist[8][kMaxExperts];
  __shared__ int s_off[kMaxExperts];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_off[e] = scratch[kNaOff + e];
  for (int e = lane; e < E; e += 32) hist[w][e] = 0;
  __syncthreads();
  // sorted positions past the sorted pairs (pairs with a rejected index)
  const int64_t sorted = scratch[kNaOff + E];
  for (int64_t r = sorted + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < P;
       r += (int64_t)gridDim.x * blockDim.x)
    perm[r] = -1;
  const int64_t chunk = (int64_t)blockIdx.x * 8 + w;
  if (chunk >= NW) return;
  const int* base = scratch + kNaHistAt + kNaHist + chunk * E;
  na_walk<true>(idx, P, E, chunk, hist[w], base, s_off, perm, inv_perm);
}

std::mutex g_na_mu;
constexpr int kNaMaxDevices = 64;
int* g_na_addr[kNaMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (the array's name is only a host-side stand-in in host code).
moe_status na_scratch(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kNaMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_na_mu);
  if (!g_na_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return MOE_ERR_CUDA;
    g_na_addr[dev] = static_cast<int*>(ptr);
  }
  *out = g_na_addr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_permute_noalloc(const moe_dims* dims, const int32_t* topk_idx,
                                          int32_t* counts, int32_t* offsets, int32_t* perm,
                                          int32_t* inv_perm, cudaStream_t stream) {
  if (!dims || !counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (dims->tokens < 0 || dims->experts < 1 || dims->experts > kMaxExperts || dims->top_k < 1 ||
      dims->top_k > dims->experts)
    return MOE_ERR_INVALID_ARG;
  const int64_t P = dims->tokens * (int64_t)dims->top_k;
  if (P > 0 && (!topk_idx || !perm || !inv_perm)) return MOE_ERR_INVALID_ARG;
  const int E = dims->experts;
  const int64_t NW = (P + kNaChunk - 1) / kNaChunk;
  // the fixed scratch holds NW x E histogram entries at most
  if (P >= (int64_t(1) << 31) || NW * E > kNaHist) return MOE_ERR_UNSUPPORTED;
  if (dims->capacity != 0) return MOE_ERR_UNSUPPORTED;  // dropless sort only
  int* scratch = nullptr;
  const moe_status st = na_scratch(&scratch);
  if (st != MOE_OK) return st;
  const unsigned blocks = (unsigned)((NW + 7) / 8);
  if (NW > 0) na_hist_kernel<<<blocks, 256, 0, stream>>>(topk_idx, P, E, NW, scratch);
  na_scan_kernel<<<E, 1024, 0, stream>>>(NW, E, scratch, counts);
  na_offsets_kernel<<<1, 32, 0, stream>>>(counts, E, scratch, offsets);
  if (NW > 0)
    na_scatter_kernel<<<blocks, 256, 0, stream>>>(topk_idx, P, E, NW, scratch, perm, inv_perm);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
