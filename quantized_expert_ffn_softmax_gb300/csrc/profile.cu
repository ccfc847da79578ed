// Per-kernel timing registry (see profile.cuh).
#include <string.h>

#include <mutex>
#include <string>
#include <vector>

#include "../../include/moe.h"
#include "profile.cuh"

namespace moe {
namespace prof {
namespace {

struct Pending {
  std::string name;
  cudaEvent_t a, b;
};
struct Total {
  std::string name;
  int count;
  double ms;
};

std::mutex g_mu;
bool g_on = false;
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_pool;
std::vector<Total> g_totals;

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return e;
}

void settle_locked() {
  for (Pending& p : g_pending) {
    float ms = 0.0f;
    if (p.a && p.b && cudaEventSynchronize(p.b) == cudaSuccess &&
        cudaEventElapsedTime(&ms, p.a, p.b) == cudaSuccess) {
      bool found = false;
      for (Total& t : g_totals)
        if (t.name == p.name) {
          t.count += 1;
          t.ms += ms;
          found = true;
          break;
        }
      if (!found) g_totals.push_back({p.name, 1, (double)ms});
    } else {
      cudaGetLastError();
    }
    if (p.a) g_pool.push_back(p.a);
    if (p.b) g_pool.push_back(p.b);
  }
  g_pending.clear();
}

}  // namespace

bool enabled() { return g_on; }

int begin(const char* name, cudaStream_t s) {
  if (!g_on) return -1;
  std::lock_guard<std::mutex> lk(g_mu);
  Pending p{name, take_event(), take_event()};
  if (p.a) cudaEventRecord(p.a, s);
  g_pending.push_back(p);
  return (int)g_pending.size() - 1;
}

void end(int token, cudaStream_t s) {
  if (token < 0) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (token < (int)g_pending.size() && g_pending[token].b) cudaEventRecord(g_pending[token].b, s);
}

}  // namespace prof
}  // namespace moe

extern "C" {

moe_status moe_profile_enable(int enable) {
  std::lock_guard<std::mutex> lk(moe::prof::g_mu);
  moe::prof::settle_locked();
  moe::prof::g_on = enable != 0;
  return MOE_OK;
}

int moe_profile_read(char* names, int name_len, int* counts, float* total_ms, int max_entries) {
  std::lock_guard<std::mutex> lk(moe::prof::g_mu);
  moe::prof::settle_locked();
  int n = 0;
  for (const auto& t : moe::prof::g_totals) {
    if (n >= max_entries) break;
    if (names && name_len > 0) {
      strncpy(names + (size_t)n * name_len, t.name.c_str(), (size_t)name_len - 1);
      names[(size_t)n * name_len + name_len - 1] = 0;
    }
    if (counts) counts[n] = t.count;
    if (total_ms) total_ms[n] = (float)t.ms;
    ++n;
  }
  moe::prof::g_totals.clear();
  return n;
}

}  // extern "C"
