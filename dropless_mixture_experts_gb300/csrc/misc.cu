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
    // four partials loaded at a time, added in split order
    const float* src = part + em * ldp + n;
    const int64_t sstride = EM * ldp;
    float v = 0.f;
    int s = 0;
    for (; s + 4 <= S; s += 4) {
      const float a0 = src[(s + 0) * sstride], a1 = src[(s + 1) * sstride];
      const float a2 = src[(s + 2) * sstride], a3 = src[(s + 3) * sstride];
      v += a0;
      v += a1;
      v += a2;
      v += a3;
    }
    for (; s < S; ++s) v += src[s * sstride];
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


}  // namespace moe
