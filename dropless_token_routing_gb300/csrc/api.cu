// C ABI of the MoE layer: argument validation, workspace layout and the order of launches.
// Nothing here synchronises with the device except moe_get_device_error.
#include <string.h>

#include <mutex>

#include "grouped.cuh"
#include "internal.h"

namespace moe {

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout ws_layout(const moe_dims& d) {
  WsLayout L;
  memset(&L, 0, sizeof(L));
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t r = o;
    o = align256(o + bytes);
    return r;
  };
  const size_t es = elt_bytes(d.dtype);
  const size_t T = (size_t)d.T, Tk = (size_t)d.T * d.k, E = d.E, D = d.d, f = d.f;
  const size_t R = (size_t)perm_rows(d);   // rows of the permuted buffers
  const size_t ST = (size_t)d.S * T, fs = d.f_s;
  L.n_chunks = (d.T + kChunk - 1) / kChunk;
  L.n_dgate_tiles = simt_dgate_tiles(d.f) > tc_dgate_tiles(d.f) ? simt_dgate_tiles(d.f)
                                                                 : tc_dgate_tiles(d.f);
  L.err = take(256);
  L.chunk_hist = take(4 * E * (size_t)L.n_chunks);
  L.chunk_base = take(4 * E * (size_t)L.n_chunks);
  L.local_rank = take(4 * Tk);
  L.dgate_part = take(4 * (size_t)L.n_dgate_tiles * R);
  L.dl_perm = take(4 * Tk);
  L.dl_tok = take(4 * Tk);
  L.dgate = take(4 * Tk);
  L.w_rT = take(4 * E * D);
  L.dwr_part = take(4 * (size_t)kDwrSplit * E * D);
  L.w_split = take(2 * 3 * E * D);
  L.router_part = take(4 * (size_t)kRouterSplit * T * ((E + 31) & ~size_t(31)));
  L.y_perm = take(es * R * D);
  L.y_sh = take(es * T * D);
  L.dy_perm = take(es * R * D);
  L.dz = take(es * R * 2 * f);
  L.dz_sh = take(es * ST * 2 * fs);
  L.hw = take(es * R * f);
  L.hw_sh = take(es * ST * fs);
  L.dx_sh = take(es * T * D);
  L.x_perm_tmp = take(es * R * D);      // selective recompute: x_perm not kept by the caller
  L.h_tmp = take(es * R * f);           // ... h (routed) not kept
  L.h_sh_tmp = take(es * ST * fs);      // ... h (shared) not kept
  const bool cap = d.capacity > 0;
  L.dest_full = take(cap ? 4 * Tk : 0);
  L.row_src_full = take(cap ? 4 * Tk : 0);
  L.offsets_full = take(cap ? 4 * (E + 1) : 0);
  L.scatter_rows = take(((d.rearrange & MOE_REARRANGE_SCATTER) && !cap) ? 4 * Tk : 0);
  L.total = o;
  return L;
}

namespace {

struct DevInfo {
  int sms = 0;
  int cc = 0;
};

DevInfo dev_info() {
  // per device, filled once under a lock (callers may be several host threads)
  static std::mutex mu;
  static DevInfo cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DevInfo();
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev].sms == 0) {
    int sms = 0, ma = 0, mi = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&ma, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&mi, cudaDevAttrComputeCapabilityMinor, dev);
    cache[dev].sms = sms;
    cache[dev].cc = ma * 10 + mi;
  }
  return cache[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// required pointer: non-null and 16-byte aligned
int req(const void* p) {
  if (p == nullptr) return MOE_ERR_NULL_POINTER;
  if (!aligned16(p)) return MOE_ERR_MISALIGNED;
  return MOE_OK;
}
// optional pointer: may be null; if not, 16-byte aligned
int opt(const void* p) { return (p == nullptr || aligned16(p)) ? MOE_OK : MOE_ERR_MISALIGNED; }
// pointer to a buffer whose size is proportional to T: may be null (empty) when T == 0
int reqT(const void* p, bool t0) { return t0 ? opt(p) : req(p); }

#define MOE_TRY(x)              \
  do {                          \
    const int _s = (x);         \
    if (_s != MOE_OK) return _s; \
  } while (0)
#define MOE_LAUNCH(x)                                   \
  do {                                                  \
    if ((x) != cudaSuccess) return MOE_ERR_LAUNCH;      \
  } while (0)

int check_dims(const moe_dims* d) {
  if (d == nullptr) return MOE_ERR_NULL_POINTER;
  if (d->dtype != MOE_F32 && d->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED_DTYPE;
  if (d->k < 1 || d->k > kMaxK || (d->E >= 1 && d->k > d->E)) return MOE_ERR_BAD_TOPK;
  if (d->T < 0 || d->T > (int64_t)0x7fffffff || d->E < 1 || d->E > kMaxE || d->d < 1 || d->f < 1 ||
      d->S < 0 || d->S > kMaxShared)
    return MOE_ERR_BAD_DIMS;
  if (d->S > 0 && d->f_s < 1) return MOE_ERR_BAD_DIMS;
  const int unit = d->dtype == MOE_BF16 ? 64 : 8;
  if (d->d % unit != 0 || d->f % unit != 0 || (d->S > 0 && d->f_s % unit != 0)) return MOE_ERR_BAD_DIMS;
  if (d->capacity < 0 || (int64_t)d->capacity * d->E >= (int64_t)0x7fffffff) return MOE_ERR_BAD_DIMS;
  if (d->rearrange < 0 || d->rearrange > (MOE_REARRANGE_GATHER | MOE_REARRANGE_SCATTER)) return MOE_ERR_BAD_DIMS;
  // T is below 2^31 here, so these products fit in 64 bits
  const int64_t rows = d->T * (int64_t)d->k + perm_rows(*d) + (int64_t)d->S * d->T;
  if (rows >= (int64_t)0x7fffffff) return MOE_ERR_BAD_DIMS;
  return MOE_OK;
}

int check_ws(const void* ws, size_t ws_bytes, const moe_dims* d) {
  if (ws == nullptr) return MOE_ERR_NULL_POINTER;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_MISALIGNED;
  if (ws_bytes < ws_layout(*d).total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return MOE_OK;
}

int check_gemm_device(const moe_dims* d) {
  const DevInfo di = dev_info();
  if (di.sms == 0) return MOE_ERR_CUDA;
  if (d->dtype == MOE_BF16 && di.cc != 103) return MOE_ERR_UNSUPPORTED_DEVICE;
  return MOE_OK;
}

GroupedArgs base_args(const moe_dims* d, const int32_t* offsets, int* err) {
  GroupedArgs a;
  memset(&a, 0, sizeof(a));
  a.T = d->T;
  a.Tk = perm_rows(*d);     // rows of the permuted buffers
  a.d = d->d;
  a.E = d->E;
  a.k = d->k;
  a.f = d->f;
  a.S = d->S;
  a.f_s = d->f_s;
  a.offsets = offsets;
  a.err = err;
  a.dgate_stride = a.Tk;
  return a;
}

int run_grouped(int mode, const GroupedArgs& a, const moe_dims* d, cudaStream_t st) {
  const DevInfo di = dev_info();
  if (d->dtype == MOE_F32) return launch_simt_grouped(mode, a, di.sms, st) == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
  return launch_tc_grouped(mode, a, di.sms, st);
}

// No token rows: every expert weight gradient is zero.
int zero_expert_grads(const moe_dims* dims, void* dw13, void* dw2, void* dws13, void* dws2,
                      cudaStream_t st) {
  const size_t es = elt_bytes(dims->dtype);
  const size_t n = (size_t)dims->E * 2 * dims->f * dims->d * es;
  if (cudaMemsetAsync(dw13, 0, n, st) != cudaSuccess || cudaMemsetAsync(dw2, 0, n / 2, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (dims->S > 0) {
    const size_t ns = (size_t)dims->S * 2 * dims->f_s * dims->d * es;
    if (cudaMemsetAsync(dws13, 0, ns, st) != cudaSuccess || cudaMemsetAsync(dws2, 0, ns / 2, st) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// Router scores: fp32 SIMT FMA for fp32 x; for bf16 x the tensor cores on the exact
// three-part bf16 split of W_r (products exact, fp32 accumulation).
int run_router(const void* x, const float* w_r, const moe_dims* d, float* logits, uint8_t* ws,
               const WsLayout& L, cudaStream_t st) {
  if (d->dtype == MOE_F32) return launch_router_logits(x, w_r, *d, logits, st) == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
  void* w_split = ws + L.w_split;
  if (launch_router_split(w_r, d->d, d->E, w_split, st) != cudaSuccess) return MOE_ERR_LAUNCH;
  GroupedArgs a = base_args(d, nullptr, reinterpret_cast<int*>(ws + L.err));
  a.x = x;
  a.w_split = w_split;
  float* part = reinterpret_cast<float*>(ws + L.router_part);
  a.logits_out = part;
  MOE_TRY(launch_tc_grouped(ROUTER, a, dev_info().sms, st));
  return launch_router_reduce(part, d->T, d->E, kRouterSplit, logits, st) == cudaSuccess ? MOE_OK
                                                                                        : MOE_ERR_LAUNCH;
}

// MOE_REARRANGE_GATHER on the bf16 dropless path fuses the rearrangement into the expert
// GEMMs: their routed token operands are gathered from x / dy by row_src (16-byte cp.async
// row copies in the tiles' swizzled layout), so x_perm and dy_perm are never materialised.
// fp32 (SIMT kernels) and drop-and-pad (zero padding rows) always keep the rearranged copies.
bool fused_gather(const moe_dims* d) {
  return (d->rearrange & MOE_REARRANGE_GATHER) && d->dtype == MOE_BF16 && d->capacity == 0;
}

// MOE_REARRANGE_SCATTER on the bf16 dropless path: the layer forward's second expert GEMM
// writes each output row at its token-major slot, and the combine reads each token's k rows
// as one block (no dest gather).
bool fused_scatter(const moe_dims* d) {
  return (d->rearrange & MOE_REARRANGE_SCATTER) && d->dtype == MOE_BF16 && d->capacity == 0;
}

int dgate_tiles(const moe_dims* d) {
  return d->dtype == MOE_F32 ? simt_dgate_tiles(d->f) : tc_dgate_tiles(d->f);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(int s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_NULL_POINTER: return "a required pointer is NULL";
    case MOE_ERR_MISALIGNED: return "a pointer is misaligned (16 bytes; workspace 256 bytes)";
    case MOE_ERR_BAD_DIMS: return "invalid dimensions";
    case MOE_ERR_BAD_TOPK: return "invalid top-k (need 1 <= k <= min(E, 32))";
    case MOE_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_LAUNCH: return "kernel launch failed";
    case MOE_ERR_CUDA: return "CUDA call failed";
    case MOE_ERR_UNSUPPORTED_DEVICE: return "bf16 grouped GEMM needs an sm_103 (GB300) device";
    case MOE_ERR_DEVICE_EXPERT_ID: return "device: expert id out of range or repeated in a row";
    case MOE_ERR_DEVICE_TIMEOUT: return "device: a bounded wait ran out";
    default: return "unknown status";
  }
}

size_t moe_workspace_bytes(const moe_dims* dims) {
  if (check_dims(dims) != MOE_OK) return 0;
  return ws_layout(*dims).total;
}

int moe_workspace_init(void* ws, size_t ws_bytes, const moe_dims* dims, moe_stream_t stream) {
  MOE_TRY(check_dims(dims));
  MOE_TRY(check_ws(ws, ws_bytes, dims));
  return cudaMemsetAsync(ws, 0, 256, (cudaStream_t)stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_get_device_error(void* ws, moe_stream_t stream, int* out) {
  if (ws == nullptr || out == nullptr) return MOE_ERR_NULL_POINTER;
  const cudaStream_t st = (cudaStream_t)stream;
  int v = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  *out = v;
  return MOE_OK;
}

int moe_router_logits(const void* x, const float* w_r, const moe_dims* dims, float* logits, void* ws,
                      size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_dims(dims));
  const bool t0 = dims->T == 0;
  MOE_TRY(check_ws(ws, ws_bytes, dims));
  MOE_TRY(reqT(x, t0));
  MOE_TRY(req(w_r));
  MOE_TRY(reqT(logits, t0));
  MOE_TRY(check_gemm_device(dims));
  if (dims->T == 0) return MOE_OK;
  const WsLayout L = ws_layout(*dims);
  return run_router(x, w_r, dims, logits, static_cast<uint8_t*>(ws), L, (cudaStream_t)stream);
}

int moe_route_topk(const float* logits, const float* bias, int64_t T, int32_t E, int32_t k,
                   int32_t* topk_idx, float* topk_w, int32_t* counts, void* ws, size_t ws_bytes,
                   moe_stream_t stream) {
  if (E < 1 || E > kMaxE || T < 0 || T > (int64_t)0x7fffffff) return MOE_ERR_BAD_DIMS;
  if (k < 1 || k > E || k > kMaxK) return MOE_ERR_BAD_TOPK;
  if (ws == nullptr) return MOE_ERR_NULL_POINTER;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_MISALIGNED;
  if (ws_bytes < 256) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const bool t0 = T == 0;
  MOE_TRY(reqT(logits, t0));
  MOE_TRY(opt(bias));
  MOE_TRY(reqT(topk_idx, t0));
  MOE_TRY(reqT(topk_w, t0));
  MOE_TRY(req(counts));
  const cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (T == 0) return MOE_OK;
  MOE_LAUNCH(launch_route_topk(logits, bias, T, E, k, topk_idx, topk_w, counts, dev_info().sms, st));
  return MOE_OK;
}

int moe_permute(const void* x, const int32_t* topk_idx, const float* topk_w, const moe_dims* dims,
                void* x_perm, int32_t* dest, int32_t* row_src, int32_t* offsets, float* w_perm,
                void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_dims(dims));
  const bool t0 = dims->T == 0;
  MOE_TRY(check_ws(ws, ws_bytes, dims));
  MOE_TRY(reqT(x, t0));
  MOE_TRY(reqT(topk_idx, t0));
  MOE_TRY(reqT(x_perm, t0));
  MOE_TRY(reqT(dest, t0));
  MOE_TRY(reqT(row_src, t0));
  MOE_TRY(req(offsets));
  MOE_TRY(opt(w_perm));
  if (w_perm != nullptr) MOE_TRY(reqT(topk_w, t0));
  const cudaStream_t st = (cudaStream_t)stream;
  if (dims->T == 0)
    return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (dims->E + 1), st) == cudaSuccess ? MOE_OK
                                                                                             : MOE_ERR_CUDA;
  const WsLayout L = ws_layout(*dims);
  uint8_t* w = static_cast<uint8_t*>(ws);
  MOE_LAUNCH(launch_permute(x, topk_idx, topk_w, *dims, x_perm, dest, row_src, offsets, w_perm, L, w,
                            reinterpret_cast<int*>(w + L.err), st));
  if (dims->capacity > 0)
    MOE_LAUNCH(launch_pad_rows(x_perm, dims->d, dims->dtype, reinterpret_cast<int32_t*>(w + L.offsets_full),
                               dims->E, dims->capacity, row_src, w_perm, st));
  return MOE_OK;
}

int moe_permute_rows(const void* x, const int32_t* dest, const moe_dims* dims, void* x_perm,
                     moe_stream_t stream) {
  MOE_TRY(check_dims(dims));
  const bool t0 = dims->T == 0;
  MOE_TRY(reqT(x, t0));
  MOE_TRY(reqT(dest, t0));
  MOE_TRY(reqT(x_perm, t0));
  if (dims->T == 0) return MOE_OK;
  MOE_LAUNCH(launch_permute_rows(x, dest, *dims, x_perm, (cudaStream_t)stream));
  return MOE_OK;
}

int moe_grouped_swiglu_fwd(const void* x_perm, const void* x, const void* w13, const void* w2,
                           const void* ws13, const void* ws2, const int32_t* offsets,
                           const moe_dims* dims, void* z, void* h, void* z_sh, void* h_sh,
                           void* y_perm, void* y_sh, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_dims(dims));
  const bool t0 = dims->T == 0;
  MOE_TRY(check_ws(ws, ws_bytes, dims));
  MOE_TRY(reqT(x_perm, t0));
  MOE_TRY(req(w13));
  MOE_TRY(req(w2));
  MOE_TRY(req(offsets));
  MOE_TRY(reqT(z, t0));
  MOE_TRY(reqT(h, t0));
  MOE_TRY(reqT(y_perm, t0));
  if (dims->S > 0) {
    MOE_TRY(reqT(x, t0));
    MOE_TRY(req(ws13));
    MOE_TRY(req(ws2));
    MOE_TRY(reqT(z_sh, t0));
    MOE_TRY(reqT(h_sh, t0));
    MOE_TRY(reqT(y_sh, t0));
  }
  MOE_TRY(check_gemm_device(dims));
  if (dims->T == 0) return MOE_OK;
  const cudaStream_t st = (cudaStream_t)stream;
  const WsLayout L = ws_layout(*dims);
  GroupedArgs a = base_args(dims, offsets, reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + L.err));
  a.x_perm = x_perm; a.x = x; a.w13 = w13; a.w2 = w2; a.ws13 = ws13; a.ws2 = ws2;
  a.z_out = z; a.h_out = h; a.z_sh_out = z_sh; a.h_sh_out = h_sh;
  MOE_TRY(run_grouped(FWD1, a, dims, st));
  a.h = h; a.h_sh = h_sh; a.y_perm = y_perm; a.y_sh = y_sh;
  MOE_TRY(run_grouped(FWD2, a, dims, st));
  return MOE_OK;
}

int moe_unpermute_combine(const void* y_perm, const int32_t* dest, const float* topk_w,
                          const void* y_sh, const moe_dims* dims, void* y, moe_stream_t stream) {
  MOE_TRY(check_dims(dims));
  const bool t0 = dims->T == 0;
  MOE_TRY(reqT(y_perm, t0));
  MOE_TRY(opt(dest));    // NULL: y_perm rows in token-major order
  if (dest == nullptr && dims->capacity > 0) return MOE_ERR_NULL_POINTER;
  MOE_TRY(opt(topk_w));
  MOE_TRY(opt(y_sh));
  MOE_TRY(reqT(y, t0));
  if (dims->T == 0) return MOE_OK;
  MOE_LAUNCH(launch_combine(y_perm, dest, topk_w, y_sh, nullptr, nullptr, nullptr, *dims, y,
                            (cudaStream_t)stream));
  return MOE_OK;
}

int moe_grouped_bwd_dx(const void* dy_perm, const void* dy, const void* z, const void* z_sh,
                       const void* w13, const void* w2, const void* ws13, const void* ws2,
                       const float* w_perm, const int32_t* offsets, const int32_t* dest,
                       const moe_dims* dims, void* dz, void* dz_sh, void* hw, void* hw_sh,
                       void* dx_perm, void* dx_sh, float* dgate, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
  MOE_TRY(check_dims(dims));
  const bool t0 = dims->T == 0;
  MOE_TRY(check_ws(ws, ws_bytes, dims));
  MOE_TRY(reqT(dy_perm, t0));
  MOE_TRY(reqT(z, t0));
  MOE_TRY(req(w13));
  MOE_TRY(req(w2));
  MOE_TRY(reqT(w_perm, t0));
  MOE_TRY(req(offsets));
  MOE_TRY(reqT(dest, t0));
  MOE_TRY(reqT(dz, t0));
  MOE_TRY(reqT(hw, t0));
  MOE_TRY(reqT(dx_perm, t0));
  MOE_TRY(reqT(dgate, t0));
  if (dims->S > 0) {
    MOE_TRY(reqT(dy, t0));
    MOE_TRY(reqT(z_sh, t0));
    MOE_TRY(req(ws13));
    MOE_TRY(req(ws2));
    MOE_TRY(reqT(dz_sh, t0));
    MOE_TRY(reqT(hw_sh, t0));
    MOE_TRY(reqT(dx_sh, t0));
  }
  MOE_TRY(check_gemm_device(dims));
  if (dims->T == 0) return MOE_OK;
  const cudaStream_t st = (cudaStream_t)stream;
  const WsLayout L = ws_layout(*dims);
  uint8_t* w = static_cast<uint8_t*>(ws);
  GroupedArgs a = base_args(dims, offsets, reinterpret_cast<int*>(w + L.err));
  a.dy_perm = dy_perm; a.dy = dy; a.z = z; a.z_sh = z_sh; a.w13 = w13; a.w2 = w2;
  a.ws13 = ws13; a.ws2 = ws2; a.w_perm = w_perm;
  a.dz_out = dz; a.dz_sh_out = dz_sh; a.hw_out = hw; a.hw_sh_out = hw_sh;
  a.dgate_part = reinterpret_cast<float*>(w + L.dgate_part);
  MOE_TRY(run_grouped(BWD2T, a, dims, st));
  MOE_LAUNCH(launch_route_bwd(nullptr, w_perm, nullptr, a.dgate_part, dgate_tiles(dims), a.Tk, dest,
                              nullptr, dims->T, dims->E, dims->k, dgate, nullptr, nullptr, nullptr, st));
  a.dz = dz; a.dz_sh = dz_sh; a.dx_perm = dx_perm; a.dx_sh = dx_sh;
  MOE_TRY(run_grouped(BWD1T, a, dims, st));
  return MOE_OK;
}

int moe_grouped_bwd_dw(const void* x_perm, const void* x, const void* hw, const void* hw_sh,
                       const void* dz, const void* dz_sh, const void* dy_perm, const void* dy,
                       const int32_t* offsets, const moe_dims* dims, void* dw13, void* dw2,
                       void* dws13, void* dws2, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_dims(dims));
  const bool t0 = dims->T == 0;
  MOE_TRY(check_ws(ws, ws_bytes, dims));
  MOE_TRY(reqT(x_perm, t0));
  MOE_TRY(reqT(hw, t0));
  MOE_TRY(reqT(dz, t0));
  MOE_TRY(reqT(dy_perm, t0));
  MOE_TRY(req(offsets));
  MOE_TRY(req(dw13));
  MOE_TRY(req(dw2));
  if (dims->S > 0) {
    MOE_TRY(reqT(x, t0));
    MOE_TRY(reqT(hw_sh, t0));
    MOE_TRY(reqT(dz_sh, t0));
    MOE_TRY(reqT(dy, t0));
    MOE_TRY(req(dws13));
    MOE_TRY(req(dws2));
  }
  MOE_TRY(check_gemm_device(dims));
  const cudaStream_t st = (cudaStream_t)stream;
  const WsLayout L = ws_layout(*dims);
  uint8_t* w = static_cast<uint8_t*>(ws);
  GroupedArgs a = base_args(dims, offsets, reinterpret_cast<int*>(w + L.err));
  a.x_perm = x_perm; a.x = x; a.hw = hw; a.hw_sh = hw_sh; a.dz = dz; a.dz_sh = dz_sh;
  a.dy_perm = dy_perm; a.dy = dy;
  a.dw13 = dw13; a.dw2 = dw2; a.dws13 = dws13; a.dws2 = dws2;
  if (dims->T == 0) return zero_expert_grads(dims, dw13, dw2, dws13, dws2, st);
  MOE_TRY(run_grouped(DW2, a, dims, st));
  MOE_TRY(run_grouped(DW13, a, dims, st));
  return MOE_OK;
}

int moe_route_balance(const float* logits, const float* bias, const int32_t* counts, int64_t T,
                      int32_t E, int32_t k, float alpha, float* prob_mean, float* aux_loss, void* ws,
                      size_t ws_bytes, moe_stream_t stream) {
  if (E < 1 || E > kMaxE || T < 1 || T > (int64_t)0x7fffffff) return MOE_ERR_BAD_DIMS;
  if (k < 1 || k > E || k > kMaxK) return MOE_ERR_BAD_TOPK;
  if (ws == nullptr) return MOE_ERR_NULL_POINTER;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_MISALIGNED;
  if (ws_bytes < 256 + sizeof(float) * ((size_t)balance_blocks(T) * E + balance_term_parts(E)))
    return MOE_ERR_WORKSPACE_TOO_SMALL;
  MOE_TRY(req(logits));
  MOE_TRY(opt(bias));
  MOE_TRY(req(counts));
  MOE_TRY(opt(prob_mean));
  MOE_TRY(req(aux_loss));
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + 256);
  MOE_LAUNCH(launch_balance(logits, bias, counts, T, E, k, alpha, part, prob_mean, aux_loss,
                            (cudaStream_t)stream));
  return MOE_OK;
}

int moe_route_topk_balance(const float* logits, const float* bias, int64_t T, int32_t E, int32_t k,
                           float alpha, int32_t* topk_idx, float* topk_w, int32_t* counts, float* prob_mean,
                           float* aux_loss, void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (E < 1 || E > kMaxE || T < 1 || T > (int64_t)0x7fffffff) return MOE_ERR_BAD_DIMS;
  if (k < 1 || k > E || k > kMaxK) return MOE_ERR_BAD_TOPK;
  if (ws == nullptr) return MOE_ERR_NULL_POINTER;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_MISALIGNED;
  if (ws_bytes < 256 + sizeof(float) * ((size_t)balance_blocks(T) * E + balance_term_parts(E)))
    return MOE_ERR_WORKSPACE_TOO_SMALL;
  MOE_TRY(req(logits));
  MOE_TRY(opt(bias));
  MOE_TRY(req(topk_idx));
  MOE_TRY(req(topk_w));
  MOE_TRY(req(counts));
  MOE_TRY(opt(prob_mean));
  MOE_TRY(req(aux_loss));
  const cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, st) != cudaSuccess) return MOE_ERR_CUDA;
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + 256);
  MOE_LAUNCH(launch_route_topk_balance(logits, bias, T, E, k, alpha, topk_idx, topk_w, counts, part, prob_mean,
                                       aux_loss, st));
  return MOE_OK;
}

int moe_route_balance_bwd(const float* logits, const float* bias, const int32_t* counts, int64_t T,
                          int32_t E, int32_t k, float alpha, float grad, float* dlogits,
                          moe_stream_t stream) {
  if (E < 1 || E > kMaxE || T < 0 || T > (int64_t)0x7fffffff) return MOE_ERR_BAD_DIMS;
  if (k < 1 || k > E || k > kMaxK) return MOE_ERR_BAD_TOPK;
  if (T == 0) return MOE_OK;
  MOE_TRY(req(logits));
  MOE_TRY(opt(bias));
  MOE_TRY(req(counts));
  MOE_TRY(req(dlogits));
  const double scale = (double)grad * alpha * E / ((double)T * (double)T * (double)k);
  MOE_LAUNCH(launch_balance_bwd(logits, bias, counts, T, E, T, (float)scale, dlogits, (cudaStream_t)stream));
  return MOE_OK;
}

int moe_route_balance_seq(const float* logits, const float* bias, const int32_t* topk_idx, int64_t T,
                          int32_t E, int32_t k, int64_t group_len, float alpha, float* prob_mean,
                          int32_t* counts, float* aux_loss, void* ws, size_t ws_bytes,
                          moe_stream_t stream) {
  if (E < 1 || E > kMaxE || T < 1 || T > (int64_t)0x7fffffff) return MOE_ERR_BAD_DIMS;
  if (k < 1 || k > E || k > kMaxK) return MOE_ERR_BAD_TOPK;
  if (group_len < 1 || T % group_len != 0 || T / group_len > 65535) return MOE_ERR_BAD_DIMS;
  if (ws == nullptr) return MOE_ERR_NULL_POINTER;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_MISALIGNED;
  const int64_t G = T / group_len;
  const size_t part_bytes = sizeof(float) * (size_t)G * balance_group_chunks(group_len) * E;
  if (ws_bytes < 256 + part_bytes + sizeof(float) * (size_t)G) return MOE_ERR_WORKSPACE_TOO_SMALL;
  MOE_TRY(req(logits));
  MOE_TRY(opt(bias));
  MOE_TRY(req(topk_idx));
  MOE_TRY(opt(prob_mean));
  MOE_TRY(req(counts));
  MOE_TRY(req(aux_loss));
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* part = reinterpret_cast<float*>(w + 256);
  float* gterm = reinterpret_cast<float*>(w + 256 + part_bytes);
  MOE_LAUNCH(launch_balance_groups(logits, bias, topk_idx, T, E, k, group_len, alpha, part, gterm, prob_mean,
                                   counts, aux_loss, (cudaStream_t)stream));
  return MOE_OK;
}

int moe_route_balance_seq_bwd(const float* logits, const float* bias, const int32_t* counts, int64_t T,
                              int32_t E, int32_t k, int64_t group_len, int64_t n_groups, float alpha,
                              float grad, float* dlogits, moe_stream_t stream) {
  if (E < 1 || E > kMaxE || T < 0 || T > (int64_t)0x7fffffff) return MOE_ERR_BAD_DIMS;
  if (k < 1 || k > E || k > kMaxK) return MOE_ERR_BAD_TOPK;
  if (group_len < 1 || n_groups < 1) return MOE_ERR_BAD_DIMS;
  if (T == 0) return MOE_OK;
  MOE_TRY(req(logits));
  MOE_TRY(opt(bias));
  MOE_TRY(req(counts));
  MOE_TRY(req(dlogits));
  const double scale =
      (double)grad * alpha * E / ((double)n_groups * (double)group_len * (double)group_len * (double)k);
  MOE_LAUNCH(launch_balance_bwd(logits, bias, counts, T, E, group_len, (float)scale, dlogits,
                                (cudaStream_t)stream));
  return MOE_OK;
}

int moe_route_topk_bwd(const int32_t* topk_idx, const float* topk_w, const float* dgate, int64_t T,
                       int32_t E, int32_t k, float* dlogits, moe_stream_t stream) {
  if (E < 1 || E > kMaxE || T < 0) return MOE_ERR_BAD_DIMS;
  if (k < 1 || k > E || k > kMaxK) return MOE_ERR_BAD_TOPK;
  if (T == 0) return MOE_OK;
  MOE_TRY(req(topk_idx));
  MOE_TRY(req(topk_w));
  MOE_TRY(req(dgate));
  MOE_TRY(req(dlogits));
  MOE_LAUNCH(launch_route_bwd(topk_idx, topk_w, dgate, nullptr, 0, 0, nullptr, nullptr, T, E, k,
                              nullptr, dlogits, nullptr, nullptr, (cudaStream_t)stream));
  return MOE_OK;
}

int moe_layer_fwd(const moe_layer_params* params, const void* x, const float* logits_in,
                  const moe_dims* dims, const moe_layer_saved* saved, void* y, void* ws,
                  size_t ws_bytes, moe_stream_t stream) {
  if (params == nullptr || saved == nullptr) return MOE_ERR_NULL_POINTER;
  MOE_TRY(check_dims(dims));
  const bool t0 = dims->T == 0;
  MOE_TRY(check_ws(ws, ws_bytes, dims));
  MOE_TRY(reqT(x, t0));
  MOE_TRY(reqT(y, t0));
  MOE_TRY(opt(logits_in));
  MOE_TRY(opt(params->bias));
  if (logits_in == nullptr) {
    MOE_TRY(req(params->w_r));
    MOE_TRY(reqT(saved->logits, t0));
  }
  MOE_TRY(reqT(saved->topk_idx, t0));
  MOE_TRY(reqT(saved->topk_w, t0));
  MOE_TRY(req(saved->counts));
  MOE_TRY(req(saved->offsets));
  MOE_TRY(reqT(saved->dest, t0));
  MOE_TRY(reqT(saved->row_src, t0));
  MOE_TRY(reqT(saved->w_perm, t0));
  MOE_TRY(opt(saved->x_perm));   // NULL: kept in the workspace, recomputed by the backward
  MOE_TRY(reqT(saved->z, t0));
  MOE_TRY(opt(saved->h));        // NULL: kept in the workspace (the backward recomputes h from z)
  MOE_TRY(req(params->w13));
  MOE_TRY(req(params->w2));
  if (dims->S > 0) {
    MOE_TRY(req(params->ws13));
    MOE_TRY(req(params->ws2));
    MOE_TRY(reqT(saved->z_sh, t0));
    MOE_TRY(opt(saved->h_sh));
  }
  MOE_TRY(check_gemm_device(dims));
  const cudaStream_t st = (cudaStream_t)stream;
  const WsLayout L = ws_layout(*dims);
  uint8_t* w = static_cast<uint8_t*>(ws);
  const bool gather = fused_gather(dims);
  // with the fused gather x_perm is written only when the caller keeps it
  void* x_perm = saved->x_perm != nullptr ? saved->x_perm : gather ? nullptr : (void*)(w + L.x_perm_tmp);
  void* h = saved->h != nullptr ? saved->h : (void*)(w + L.h_tmp);
  void* h_sh = dims->S == 0 ? nullptr : saved->h_sh != nullptr ? saved->h_sh : (void*)(w + L.h_sh_tmp);
  if (dims->T == 0) {
    if (cudaMemsetAsync(saved->counts, 0, sizeof(int32_t) * dims->E, st) != cudaSuccess ||
        cudaMemsetAsync(saved->offsets, 0, sizeof(int32_t) * (dims->E + 1), st) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  const float* scores = logits_in;
  if (scores == nullptr) {
    MOE_TRY(run_router(x, params->w_r, dims, saved->logits, w, L, st));
    scores = saved->logits;
  }
  if (cudaMemsetAsync(saved->counts, 0, sizeof(int32_t) * dims->E, st) != cudaSuccess) return MOE_ERR_CUDA;
  MOE_LAUNCH(launch_route_topk(scores, params->bias, dims->T, dims->E, dims->k, saved->topk_idx,
                               saved->topk_w, saved->counts, dev_info().sms, st));
  MOE_LAUNCH(launch_permute(x_perm != nullptr ? x : nullptr, saved->topk_idx, saved->topk_w, *dims, x_perm,
                            saved->dest, saved->row_src, saved->offsets, saved->w_perm, L, w,
                            reinterpret_cast<int*>(w + L.err), st));
  if (dims->capacity > 0)
    MOE_LAUNCH(launch_pad_rows(x_perm, dims->d, dims->dtype, reinterpret_cast<int32_t*>(w + L.offsets_full),
                               dims->E, dims->capacity, saved->row_src, saved->w_perm, st));
  GroupedArgs a = base_args(dims, saved->offsets, reinterpret_cast<int*>(w + L.err));
  a.x_perm = x_perm; a.x = x; a.w13 = params->w13; a.w2 = params->w2;
  a.gather_rows = gather ? saved->row_src : nullptr;
  a.ws13 = params->ws13; a.ws2 = params->ws2;
  a.z_out = saved->z; a.h_out = h; a.z_sh_out = saved->z_sh; a.h_sh_out = h_sh;
  MOE_TRY(run_grouped(FWD1, a, dims, st));
  void* y_perm = w + L.y_perm;
  void* y_sh = dims->S > 0 ? (void*)(w + L.y_sh) : nullptr;
  a.h = h; a.h_sh = h_sh; a.y_perm = y_perm; a.y_sh = y_sh;
  const bool scatter = fused_scatter(dims);
  if (scatter) {   // y_perm then holds the expert outputs in token-major order
    int32_t* srows = reinterpret_cast<int32_t*>(w + L.scatter_rows);
    MOE_LAUNCH(launch_scatter_rows(saved->dest, dims->T * (int64_t)dims->k, srows, st));
    a.scatter_rows = srows;
  }
  MOE_TRY(run_grouped(FWD2, a, dims, st));
  MOE_LAUNCH(launch_combine(y_perm, scatter ? nullptr : saved->dest, saved->topk_w, y_sh, nullptr, nullptr,
                            nullptr, *dims, y, st));
  return MOE_OK;
}

int moe_layer_bwd(const moe_layer_params* params, const moe_layer_saved* saved, const void* x,
                  const void* dy, const moe_dims* dims, const moe_layer_grads* grads, void* ws,
                  size_t ws_bytes, moe_stream_t stream) {
  if (params == nullptr || saved == nullptr || grads == nullptr) return MOE_ERR_NULL_POINTER;
  MOE_TRY(check_dims(dims));
  const bool t0 = dims->T == 0;
  MOE_TRY(check_ws(ws, ws_bytes, dims));
  MOE_TRY(reqT(x, t0));
  MOE_TRY(reqT(dy, t0));
  MOE_TRY(reqT(grads->dx, t0));
  MOE_TRY(req(grads->dw13));
  MOE_TRY(req(grads->dw2));
  MOE_TRY(opt(grads->dlogits));
  const bool router = params->w_r != nullptr;
  if (router) {
    MOE_TRY(req(params->w_r));
    MOE_TRY(req(grads->dw_r));
  } else {
    MOE_TRY(reqT(grads->dlogits, t0));
  }
  MOE_TRY(reqT(saved->topk_idx, t0));
  MOE_TRY(reqT(saved->topk_w, t0));
  MOE_TRY(req(saved->offsets));
  MOE_TRY(reqT(saved->dest, t0));
  MOE_TRY(reqT(saved->row_src, t0));
  MOE_TRY(reqT(saved->w_perm, t0));
  MOE_TRY(opt(saved->x_perm));   // NULL: re-permuted from x here
  MOE_TRY(reqT(saved->z, t0));
  MOE_TRY(req(params->w13));
  MOE_TRY(req(params->w2));
  if (dims->S > 0) {
    MOE_TRY(req(params->ws13));
    MOE_TRY(req(params->ws2));
    MOE_TRY(reqT(saved->z_sh, t0));
    MOE_TRY(req(grads->dws13));
    MOE_TRY(req(grads->dws2));
  }
  MOE_TRY(check_gemm_device(dims));
  const cudaStream_t st = (cudaStream_t)stream;
  const WsLayout L = ws_layout(*dims);
  uint8_t* w = static_cast<uint8_t*>(ws);
  int* err = reinterpret_cast<int*>(w + L.err);
  if (dims->T == 0) {
    if (router && cudaMemsetAsync(grads->dw_r, 0, sizeof(float) * dims->E * dims->d, st) != cudaSuccess)
      return MOE_ERR_CUDA;
    return zero_expert_grads(dims, grads->dw13, grads->dw2, grads->dws13, grads->dws2, st);
  }
  void* dy_perm = w + L.dy_perm;
  void* dz = w + L.dz;
  void* dz_sh = dims->S > 0 ? (void*)(w + L.dz_sh) : nullptr;
  void* hw = w + L.hw;
  void* hw_sh = dims->S > 0 ? (void*)(w + L.hw_sh) : nullptr;
  void* dx_perm = w + L.y_perm;  // the forward's y_perm is dead by now
  void* dx_sh = dims->S > 0 ? (void*)(w + L.dx_sh) : nullptr;
  float* dgate_part = reinterpret_cast<float*>(w + L.dgate_part);
  float* dl_tok = reinterpret_cast<float*>(w + L.dl_tok);
  float* dl_perm = reinterpret_cast<float*>(w + L.dl_perm);
  float* dgate = reinterpret_cast<float*>(w + L.dgate);

  // 0. drop-and-pad: the dropless positions of every copy (the router gradient reaches the
  //    dropped copies too) and the expert counts that locate the padding rows
  const bool cap = dims->capacity > 0;
  int32_t* dest_full = reinterpret_cast<int32_t*>(w + L.dest_full);
  int32_t* row_src_full = reinterpret_cast<int32_t*>(w + L.row_src_full);
  int32_t* offsets_full = reinterpret_cast<int32_t*>(w + L.offsets_full);
  if (cap) {
    moe_dims full = *dims;
    full.capacity = 0;
    MOE_LAUNCH(launch_permute(nullptr, saved->topk_idx, nullptr, full, nullptr, dest_full, row_src_full,
                              offsets_full, nullptr, L, w, err, st));
  }
  // 1. rearrange dY like x (fused into the GEMMs' operand loads on the bf16 dropless path)
  const bool gather = fused_gather(dims);
  if (!gather) {
    MOE_LAUNCH(launch_permute_rows(dy, saved->dest, *dims, dy_perm, st));
    if (cap)
      MOE_LAUNCH(launch_pad_rows(dy_perm, dims->d, dims->dtype, offsets_full, dims->E, dims->capacity,
                                 nullptr, nullptr, st));
  }
  // 2. expert dX chain, first half: D = dY W2, dgate partials, dz, hw
  GroupedArgs a = base_args(dims, saved->offsets, err);
  a.gather_rows = gather ? saved->row_src : nullptr;
  a.dy_perm = dy_perm; a.dy = dy; a.z = saved->z; a.z_sh = saved->z_sh;
  a.w13 = params->w13; a.w2 = params->w2; a.ws13 = params->ws13; a.ws2 = params->ws2;
  a.w_perm = saved->w_perm;
  a.dz_out = dz; a.dz_sh_out = dz_sh; a.hw_out = hw; a.hw_sh_out = hw_sh;
  a.dgate_part = dgate_part;
  MOE_TRY(run_grouped(BWD2T, a, dims, st));
  // 3. dgate -> score gradient (dlogits), in token and permuted order
  MOE_LAUNCH(launch_route_bwd(saved->topk_idx, saved->topk_w, nullptr, dgate_part, dgate_tiles(dims),
                              a.Tk, saved->dest, cap ? dest_full : saved->dest, dims->T, dims->E,
                              dims->k, dgate, grads->dlogits, dl_tok, dl_perm, st));
  // 4. expert dX chain, second half: dx_perm = dz W13. On the bf16 dropless path the router
  //    term dl W_r^T of each copy is added to its row here (every copy has a row); fp32 and
  //    drop-and-pad (dropped copies have no row) add it in the un-rearrangement instead.
  const float* w_rT = nullptr;
  if (router) {
    MOE_LAUNCH(launch_transpose_f32(params->w_r, dims->d, dims->E, reinterpret_cast<float*>(w + L.w_rT), st));
    w_rT = reinterpret_cast<const float*>(w + L.w_rT);
  }
  const bool fold_router = router && dims->dtype == MOE_BF16 && !cap;
  a.dz = dz; a.dz_sh = dz_sh; a.dx_perm = dx_perm; a.dx_sh = dx_sh;
  a.dl_perm = dl_perm;
  a.w_rT = fold_router ? w_rT : nullptr;
  MOE_TRY(run_grouped(BWD1T, a, dims, st));
  // 5. un-rearrange dX (+ shared dX, + the router term when not folded above)
  MOE_LAUNCH(launch_combine(dx_perm, saved->dest, nullptr, dx_sh, saved->topk_idx, dl_tok,
                            fold_router ? nullptr : w_rT, *dims, grads->dx, st));
  // 6. expert dW products (separate kernels from the dX chain)
  const void* x_perm = saved->x_perm;
  if (x_perm == nullptr && !gather) {  // selective recompute of the rearranged input
    MOE_LAUNCH(launch_permute_rows(x, saved->dest, *dims, w + L.x_perm_tmp, st));
    if (cap)
      MOE_LAUNCH(launch_pad_rows(w + L.x_perm_tmp, dims->d, dims->dtype, offsets_full, dims->E,
                                 dims->capacity, nullptr, nullptr, st));
    x_perm = w + L.x_perm_tmp;
  }
  a.x_perm = x_perm; a.x = x; a.hw = hw; a.hw_sh = hw_sh;
  a.dw13 = grads->dw13; a.dw2 = grads->dw2; a.dws13 = grads->dws13; a.dws2 = grads->dws2;
  MOE_TRY(run_grouped(DW2, a, dims, st));
  MOE_TRY(run_grouped(DW13, a, dims, st));
  // 7. router dW
  if (router)
    MOE_LAUNCH(launch_dwr(x, cap ? row_src_full : saved->row_src, dl_perm,
                          cap ? offsets_full : saved->offsets, *dims,
                          reinterpret_cast<float*>(w + L.dwr_part), grads->dw_r, st));
  return MOE_OK;
}

int moe_debug_timeout_probe(void* ws, size_t ws_bytes, uint64_t limit_ns, moe_stream_t stream) {
  if (ws == nullptr) return MOE_ERR_NULL_POINTER;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_MISALIGNED;
  if (ws_bytes < 256) return MOE_ERR_WORKSPACE_TOO_SMALL;
  MOE_LAUNCH(launch_timeout_probe(static_cast<int*>(ws), limit_ns, (cudaStream_t)stream));
  return MOE_OK;
}

}  // extern "C"
