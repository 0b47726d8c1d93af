// Kernel timing records (a measurement aid): while enabled, each kernel
// launch of the library is bracketed by two CUDA events recorded on the
// launch stream.  Reading the records synchronises on the last event and
// aggregates launches and time per kernel name.
#include <mutex>
#include <string>
#include <vector>

#include "kernels.cuh"

namespace moe {
namespace {

struct Rec {
  const char* name;
  cudaEvent_t a, b;
};

std::mutex g_mu;
bool g_on = false;
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pool;
thread_local const char* t_open = nullptr;
thread_local cudaEvent_t t_start = nullptr;

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

}  // namespace

void prof_begin(const char* name, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on) return;
  t_open = name;
  t_start = take_event();
  cudaEventRecord(t_start, s);
}

void prof_end(cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on || !t_open) return;
  cudaEvent_t b = take_event();
  cudaEventRecord(b, s);
  g_recs.push_back({t_open, t_start, b});
  t_open = nullptr;
}

}  // namespace moe

extern "C" moe_status moe_profile_enable(int enable) {
  std::lock_guard<std::mutex> lk(moe::g_mu);
  for (auto& r : moe::g_recs) {
    moe::g_pool.push_back(r.a);
    moe::g_pool.push_back(r.b);
  }
  moe::g_recs.clear();
  moe::g_on = enable != 0;
  return MOE_OK;
}

extern "C" moe_status moe_profile_read(int max_entries, char* names, int64_t* launches,
                                       double* total_ms, int* n_entries) {
  if (max_entries < 0 || !n_entries) return MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(moe::g_mu);
  std::vector<std::string> keys;
  std::vector<int64_t> cnt;
  std::vector<double> ms;
  for (auto& r : moe::g_recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) return MOE_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return MOE_ERR_CUDA;
    size_t i = 0;
    while (i < keys.size() && keys[i] != r.name) ++i;
    if (i == keys.size()) {
      keys.emplace_back(r.name);
      cnt.push_back(0);
      ms.push_back(0.0);
    }
    cnt[i] += 1;
    ms[i] += t;
  }
  *n_entries = (int)keys.size();
  for (size_t i = 0; i < keys.size() && (int)i < max_entries; ++i) {
    if (names) {
      std::snprintf(names + 64 * i, 64, "%s", keys[i].c_str());
    }
    if (launches) launches[i] = cnt[i];
    if (total_ms) total_ms[i] = ms[i];
  }
  return MOE_OK;
}
