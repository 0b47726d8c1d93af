// Small utility kernels: zero fills and the device status word.
#include "kernels.cuh"

namespace moe {

template <typename T>
__global__ void zero_kernel(T* __restrict__ p, int64_t n) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += stride) p[i] = T(0);
}

template <typename T>
static void zero_fill(T* p, int64_t n, cudaStream_t s) {
  if (n <= 0) return;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  MOE_LAUNCH("zero_fill", s, zero_kernel<T><<<(unsigned)blocks, 256, 0, s>>>(p, n));
}

// out[r, :] = src[tokrow[r], :] for the padded rows r < *used (a count the
// permutation wrote on the device): one warp per row, 16-byte copies.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ src,
                                                          const int32_t* __restrict__ tokrow,
                                                          const int* __restrict__ used,
                                                          uint4* __restrict__ out, int vecs,
                                                          int64_t cap) {
  const int lane = threadIdx.x & 31;
  const int64_t n = *used < cap ? *used : cap;
  const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  // four rows per warp per pass: every index and load is issued before the
  // stores, so each lane keeps several 16-byte loads in flight
  for (int64_t r0 = ((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5) * 4; r0 < n;
       r0 += warps * 4) {
    int64_t t[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) t[q] = r0 + q < n ? tokrow[r0 + q] : -1;
    for (int v0 = lane; v0 < vecs; v0 += 64) {
      uint4 buf[4][2];
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int v = v0 + 32 * u;
          if (t[q] >= 0 && v < vecs) buf[q][u] = __ldg(src + t[q] * vecs + v);
        }
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int v = v0 + 32 * u;
          if (t[q] >= 0 && v < vecs) out[(r0 + q) * vecs + v] = buf[q][u];
        }
    }
  }
}

void launch_gather_rows(const void* src, const int32_t* tokrow, const int* used, void* out,
                        int64_t cap_rows, int64_t row_bytes, cudaStream_t s) {
  if (cap_rows <= 0) return;
  int64_t blocks = (cap_rows + 31) / 32;  // 8 warps x 4 rows per block pass
  if (blocks > 152 * 8) blocks = 152 * 8;
  MOE_LAUNCH("gather_rows", s,
             gather_rows_kernel<<<(unsigned)blocks, 256, 0, s>>>(
                 reinterpret_cast<const uint4*>(src), tokrow, used, reinterpret_cast<uint4*>(out),
                 (int)(row_bytes / 16), cap_rows));
}

// out[em][n] = sum over s of part[s][em][n] in split order (n < N, row
// stride ldp in the partials); with hsplit > 0 columns n >= hsplit go to
// out1 (the up half of a gate|up gradient).
__global__ void __launch_bounds__(256) split_reduce_kernel(const float* __restrict__ part, int S,
                                                           int64_t EM, int ldp, int N, int hsplit,
                                                           float* out0, float* out1) {
  const int64_t n_all = EM * N;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_all; i += stride) {
    const int64_t em = i / N;
    const int n = (int)(i % N);
    float v = 0.f;
    for (int s = 0; s < S; ++s) v += part[((int64_t)s * EM + em) * ldp + n];
    if (hsplit > 0) {
      if (n < hsplit) out0[em * hsplit + n] = v;
      else out1[em * hsplit + (n - hsplit)] = v;
    } else {
      out0[em * N + n] = v;
    }
  }
}

void launch_split_reduce(const float* part, int S, int64_t EM, int ldp, int N, int hsplit,
                         float* out0, float* out1, cudaStream_t s) {
  const int64_t n = EM * N;
  if (n <= 0) return;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  MOE_LAUNCH("split_reduce", s,
             split_reduce_kernel<<<(unsigned)blocks, 256, 0, s>>>(part, S, EM, ldp, N, hsplit, out0,
                                                                  out1));
}

void zero_fill_i32(int32_t* p, int64_t n, cudaStream_t s) { zero_fill<int32_t>(p, n, s); }
void zero_fill_f32(float* p, int64_t n, cudaStream_t s) { zero_fill<float>(p, n, s); }
void clear_status(int* status, cudaStream_t s) { zero_fill<int>(status, 2, s); }

}  // namespace moe
