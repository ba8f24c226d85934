// Optional per-kernel timing: when enabled, every kernel the library launches
// outside of stream capture is bracketed by a pair of CUDA events recorded on
// its own stream; ds4moe_profile_entry() resolves them into per-kernel totals.
#include <mutex>
#include <string>
#include <vector>

#include "internal.cuh"

namespace ds4 {
namespace {

struct Pending {
  const char *name;
  cudaEvent_t a, b;
};
struct Total {
  std::string name;
  double ms = 0;
  int64_t launches = 0;
};

std::mutex g_mu;
bool g_on = false;
std::vector<Pending> g_pending;
std::vector<Total> g_totals;
std::vector<cudaEvent_t> g_free;

cudaEvent_t get_event() {
  if (!g_free.empty()) {
    cudaEvent_t e = g_free.back();
    g_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

void resolve_locked() {
  for (auto &p : g_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(p.b) == cudaSuccess && cudaEventElapsedTime(&ms, p.a, p.b) == cudaSuccess) {
      Total *t = nullptr;
      for (auto &x : g_totals)
        if (x.name == p.name) t = &x;
      if (!t) {
        g_totals.push_back(Total{p.name});
        t = &g_totals.back();
      }
      t->ms += ms;
      t->launches += 1;
    }
    g_free.push_back(p.a);
    g_free.push_back(p.b);
  }
  g_pending.clear();
}

bool capturing(cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  return cudaStreamIsCapturing(s, &st) != cudaSuccess || st != cudaStreamCaptureStatusNone;
}

}  // namespace

ProfScope::ProfScope(const char *name, cudaStream_t s) : name_(name), s_(s) {
  if (!g_on || capturing(s)) return;
  std::lock_guard<std::mutex> lk(g_mu);
  a_ = get_event();
  b_ = get_event();
  if (a_ && b_) cudaEventRecord(a_, s);
}

ProfScope::~ProfScope() {
  if (!a_ || !b_) return;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEventRecord(b_, s_);
  g_pending.push_back(Pending{name_, a_, b_});
  if (g_pending.size() > 4096) resolve_locked();
}

}  // namespace ds4

using namespace ds4;

extern "C" {

ds4moe_status ds4moe_profile_enable(int32_t on) {
  std::lock_guard<std::mutex> lk(g_mu);
  resolve_locked();
  g_totals.clear();
  g_on = on != 0;
  return DS4MOE_OK;
}

int32_t ds4moe_profile_count(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  resolve_locked();
  return (int32_t)g_totals.size();
}

ds4moe_status ds4moe_profile_entry(int32_t i, const char **name, double *total_ms, int64_t *launches) {
  std::lock_guard<std::mutex> lk(g_mu);
  resolve_locked();
  if (i < 0 || i >= (int32_t)g_totals.size() || !name || !total_ms || !launches) return DS4MOE_EINVAL;
  *name = g_totals[i].name.c_str();
  *total_ms = g_totals[i].ms;
  *launches = g_totals[i].launches;
  return DS4MOE_OK;
}

}  // extern "C"
