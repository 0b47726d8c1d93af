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

void zero_fill_i32(int32_t* p, int64_t n, cudaStream_t s) { zero_fill<int32_t>(p, n, s); }
void zero_fill_f32(float* p, int64_t n, cudaStream_t s) { zero_fill<float>(p, n, s); }
void clear_status(int* status, cudaStream_t s) { zero_fill<int>(status, 2, s); }

}  // namespace moe
