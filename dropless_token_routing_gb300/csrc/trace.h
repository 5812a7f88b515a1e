// Launch tracing: when enabled, every kernel launch of the library is bracketed by a pair of
// CUDA events on its stream, grouped by phase; moe_trace_read sums the elapsed times.
#pragma once

#include <cuda_runtime.h>

namespace moe {

enum TracePhase : int {
  TP_ROUTER_GEMM = 0,
  TP_ROUTE_TOPK,
  TP_PERMUTE_HIST,
  TP_PERMUTE_SCAN,
  TP_PERMUTE_SCATTER,
  TP_GEMM_FWD1,
  TP_GEMM_FWD2,
  TP_COMBINE,
  TP_PERMUTE_ROWS,
  TP_GEMM_BWD2T,
  TP_ROUTE_BWD,
  TP_GEMM_BWD1T,
  TP_TRANSPOSE,
  TP_COMBINE_BWD,
  TP_GEMM_DW2,
  TP_GEMM_DW13,
  TP_DWR,
  TP_MISC,
  TP_COUNT
};

bool trace_on();
void trace_record(int phase, cudaStream_t st, bool begin);

struct TraceScope {
  int phase;
  cudaStream_t st;
  bool on;
  TraceScope(int p, cudaStream_t s) : phase(p), st(s), on(trace_on()) {
    if (on) trace_record(phase, st, true);
  }
  ~TraceScope() {
    if (on) trace_record(phase, st, false);
  }
};

}  // namespace moe
