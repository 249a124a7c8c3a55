// Native tracing: a host-side count of every kernel launch the library issues, and optional
// CUDA-event timing (two events on the launching stream per launch) of the tcgen05 GEMM
// launches (kind 0, with their algorithmic flops) and of the rank-r passes (kind 1, with their
// algorithmic HBM bytes), so a benchmark can time them inside a long step without a profiler.
#include <atomic>
#include <mutex>
#include <vector>

#include "internal.h"

namespace lg {

static std::atomic<uint64_t> g_launches{0};

struct ProfRec {
  cudaEvent_t a, b;
  double work;   // flops (GEMM) or bytes (rank-r pass)
  int kind;
};
static std::mutex g_mu;
static bool g_prof_on = false;
static std::vector<ProfRec> g_recs;     // recorded since the last reset
static std::vector<cudaEvent_t> g_pool; // spare events

void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
uint64_t launch_count() { return g_launches.load(); }

static cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

bool prof_enabled() { return g_prof_on; }

void prof_set(bool on) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_prof_on = on;
}

// Bracket one launch: call with `start` = true before, false after (records nest one deep).
void prof_mark(cudaStream_t st, bool start, double work, int kind) {
  if (!g_prof_on) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (start) {
    ProfRec r{take_event(), take_event(), work, kind};
    if (r.a && r.b) {
      cudaEventRecord(r.a, st);
      g_recs.push_back(r);
    }
  } else if (!g_recs.empty()) {
    cudaEventRecord(g_recs.back().b, st);
  }
}

cudaError_t prof_collect(int kind, double* ms, int64_t* launches, double* work, bool reset) {
  std::lock_guard<std::mutex> lk(g_mu);
  double t = 0.0, f = 0.0;
  int64_t n = 0;
  for (auto& r : g_recs) {
    if (r.kind != kind) continue;
    cudaError_t e = cudaEventSynchronize(r.b);
    if (e != cudaSuccess) return e;
    float x = 0.f;
    e = cudaEventElapsedTime(&x, r.a, r.b);
    if (e != cudaSuccess) return e;
    t += x;
    f += r.work;
    ++n;
  }
  if (ms) *ms = t;
  if (launches) *launches = n;
  if (work) *work = f;
  if (reset) {
    std::vector<ProfRec> keep;
    for (auto& r : g_recs) {
      if (r.kind == kind) {
        g_pool.push_back(r.a);
        g_pool.push_back(r.b);
      } else {
        keep.push_back(r);
      }
    }
    g_recs.swap(keep);
  }
  return cudaSuccess;
}

}  // namespace lg
