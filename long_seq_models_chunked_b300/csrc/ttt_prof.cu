// Launch accounting and optional per-launch timing of the library's kernels.
//
// Every kernel launch of the library is counted per kernel class. When timing
// is enabled, a pair of CUDA events is recorded on the launching stream around
// each launch; the elapsed times are resolved when they are read.
#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/ttt_debug.h"
#include "ttt_internal.h"

namespace ttt {
namespace {

struct Rec {
  int kind;
  cudaEvent_t a, b;
};

std::atomic<long long> g_launches[TTT_KERNEL_COUNT];
std::atomic<int> g_enabled{0};
std::mutex g_mu;
std::vector<Rec> g_recs;          // recorded, not yet resolved
std::vector<cudaEvent_t> g_pool;  // reusable events
double g_ms[TTT_KERNEL_COUNT];
long long g_timed[TTT_KERNEL_COUNT];
thread_local cudaEvent_t t_pending = nullptr;

cudaEvent_t get_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

void resolve_locked() {
  for (Rec& r : g_recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) == cudaSuccess && cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
      g_ms[r.kind] += ms;
      g_timed[r.kind] += 1;
    }
    g_pool.push_back(r.a);
    g_pool.push_back(r.b);
  }
  g_recs.clear();
}

}  // namespace

void prof_before(int kind, cudaStream_t st) {
  g_launches[kind].fetch_add(1, std::memory_order_relaxed);
  if (!g_enabled.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_mu);
  t_pending = get_event();
  if (t_pending) cudaEventRecord(t_pending, st);
}

void prof_after(int kind, cudaStream_t st) {
  if (!g_enabled.load(std::memory_order_relaxed) || !t_pending) return;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEvent_t b = get_event();
  if (b && cudaEventRecord(b, st) == cudaSuccess) {
    g_recs.push_back({kind, t_pending, b});
  } else {
    g_pool.push_back(t_pending);
    if (b) g_pool.push_back(b);
  }
  t_pending = nullptr;
}

}  // namespace ttt

using namespace ttt;

extern "C" {

void ttt_prof_enable(int on) { g_enabled.store(on ? 1 : 0); }

void ttt_prof_reset(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  resolve_locked();
  for (int k = 0; k < TTT_KERNEL_COUNT; ++k) {
    g_launches[k].store(0);
    g_ms[k] = 0.0;
    g_timed[k] = 0;
  }
}

int ttt_prof_read(int kind, double* total_ms, long long* timed_launches, long long* launches) {
  if (kind < 0 || kind >= TTT_KERNEL_COUNT) return TTT_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  resolve_locked();
  if (total_ms) *total_ms = g_ms[kind];
  if (timed_launches) *timed_launches = g_timed[kind];
  if (launches) *launches = g_launches[kind].load();
  return TTT_OK;
}

long long ttt_launch_count(void) {
  long long n = 0;
  for (int k = 0; k < TTT_KERNEL_COUNT; ++k) n += g_launches[k].load();
  return n;
}

const char* ttt_kernel_name(int kind) {
  static const char* names[TTT_KERNEL_COUNT] = {
      "fwd_swiglu",  "apply_out", "grad_outer", "ns_gram",      "ns_poly", "ns_xupd",
      "update_norm", "aux",       "linear_chunk", "simt_layer", "ns_fused"};
  return (kind >= 0 && kind < TTT_KERNEL_COUNT) ? names[kind] : "unknown";
}

}  // extern "C"
