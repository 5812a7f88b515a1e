// Launch tracing (see trace.h): event pairs per launch, summed per phase on read.
#include <atomic>
#include <mutex>
#include <vector>

#include "internal.h"
#include "trace.h"

namespace moe {
namespace {

const char* kPhaseNames[TP_COUNT] = {
    "router_gemm", "route_topk",  "permute_hist", "permute_scan", "permute_scatter",
    "gemm_fwd1",   "gemm_fwd2",   "combine",      "permute_rows", "gemm_bwd2t",
    "route_bwd",   "gemm_bwd1t",  "transpose",    "combine_bwd",  "gemm_dw2",
    "gemm_dw13",   "dwr",         "misc"};

struct Rec {
  int phase;
  cudaEvent_t a, b;
};

std::mutex g_mu;
std::atomic<bool> g_on{false};   // read without the lock by every launcher
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pool;
Rec g_open[TP_COUNT];
bool g_has_open[TP_COUNT];

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

bool trace_on() { return g_on.load(std::memory_order_relaxed); }

void trace_record(int phase, cudaStream_t st, bool begin) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on.load(std::memory_order_relaxed) || phase < 0 || phase >= TP_COUNT) return;
  if (begin) {
    Rec r{phase, take_event(), nullptr};
    cudaEventRecord(r.a, st);
    g_open[phase] = r;
    g_has_open[phase] = true;
  } else if (g_has_open[phase]) {
    Rec r = g_open[phase];
    r.b = take_event();
    cudaEventRecord(r.b, st);
    g_recs.push_back(r);
    g_has_open[phase] = false;
  }
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_trace_enable(int on) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (Rec& r : g_recs) {
    g_pool.push_back(r.a);
    g_pool.push_back(r.b);
  }
  g_recs.clear();
  for (int p = 0; p < TP_COUNT; ++p) g_has_open[p] = false;
  g_on.store(on != 0, std::memory_order_relaxed);
  return MOE_OK;
}

int moe_trace_read(moe_trace_entry* out, int max_entries, int* n_out) {
  if (out == nullptr || n_out == nullptr) return MOE_ERR_NULL_POINTER;
  std::lock_guard<std::mutex> lk(g_mu);
  double ms[TP_COUNT] = {};
  int64_t cnt[TP_COUNT] = {};
  for (const Rec& r : g_recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) return MOE_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return MOE_ERR_CUDA;
    ms[r.phase] += t;
    cnt[r.phase] += 1;
  }
  int n = 0;
  for (int p = 0; p < TP_COUNT && n < max_entries; ++p) {
    if (cnt[p] == 0) continue;
    out[n].name = kPhaseNames[p];
    out[n].launches = cnt[p];
    out[n].total_ms = ms[p];
    ++n;
  }
  *n_out = n;
  return MOE_OK;
}

}  // extern "C"
