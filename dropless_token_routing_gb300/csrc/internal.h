// Host-side internals of the MoE library: workspace layout and kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

struct GroupedArgs;

constexpr int kChunk = 64;        // tokens per permutation chunk (one 64-bit mask per expert)
constexpr int kDwrSplit = 8;      // fixed row split of the router dW reduction
constexpr int kMaxShared = 8;     // shared experts supported
constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
constexpr int kMaxDevices = 64;   // device ordinals the per-device host caches cover

inline size_t elt_bytes(int dtype) { return dtype == MOE_F32 ? 4 : 2; }

// Rows of the permuted buffers: T*k dropless, E*C in the drop-and-pad variant.
inline int64_t perm_rows(const moe_dims& d) {
  return d.capacity > 0 ? (int64_t)d.E * d.capacity : d.T * (int64_t)d.k;
}

// Byte offsets of the workspace regions (each 256-byte aligned).
struct WsLayout {
  size_t err;          // int error word (+ padding)
  size_t chunk_hist;   // [E][n_chunks] int32
  size_t chunk_base;   // [E][n_chunks] int32
  size_t local_rank;   // [T*k] int32
  size_t dgate_part;   // [n_dgate_tiles][T*k] fp32
  size_t dl_perm;      // [T*k] fp32  score gradient in permuted order
  size_t dl_tok;       // [T*k] fp32  score gradient in token order
  size_t dgate;        // [T*k] fp32
  size_t w_rT;         // [E][d] fp32
  size_t dwr_part;     // [kDwrSplit][E][d] fp32
  size_t w_split;      // [E][3d] bf16  exact 3-part split of W_r^T (bf16 router GEMM)
  size_t router_part;  // [kRouterSplit][T][round32(E)] fp32 K-slice partial scores
  size_t y_perm;       // [T*k, d]  (reused as dx_perm in the backward)
  size_t y_sh;         // [T, d]
  size_t dy_perm;      // [T*k, d]
  size_t dz;           // [T*k, 2f]
  size_t dz_sh;        // [S*T, 2f_s]
  size_t hw;           // [T*k, f]
  size_t hw_sh;        // [S*T, f_s]
  size_t dx_sh;        // [T, d]
  size_t x_perm_tmp;   // [T*k, d]   x_perm when the caller does not keep it
  size_t h_tmp;        // [T*k, f]   h when the caller does not keep it
  size_t h_sh_tmp;     // [S*T, f_s]
  size_t dest_full;    // [T*k] int32   drop-and-pad: dropless position of every copy
  size_t row_src_full; // [T*k] int32   ... and token of every dropless position
  size_t offsets_full; // [E+1] int32   ... dropless expert offsets
  size_t scatter_rows; // [T*k] int32   fused un-rearrangement: token-major slot of each row
  size_t total;
  int64_t n_chunks;
  int n_dgate_tiles;
};

WsLayout ws_layout(const moe_dims& d);

// launchers (return the launch's cudaError_t)
cudaError_t launch_router_logits(const void* x, const float* w_r, const moe_dims& dm, float* logits,
                                 cudaStream_t st);
cudaError_t launch_route_topk(const float* logits, const float* bias, int64_t T, int E, int k,
                              int32_t* idx, float* w, int32_t* counts, int num_sms, cudaStream_t st);
// dgate is gathered from dgate_part at dest (0 for a dropped copy); dl_perm is scattered
// at dest_dl (the dropless positions, also in the drop-and-pad variant).
cudaError_t launch_route_bwd(const int32_t* idx, const float* w, const float* dgate_in,
                             const float* dgate_part, int n_part, int64_t part_stride,
                             const int32_t* dest, const int32_t* dest_dl, int64_t T, int E, int k,
                             float* dgate_out, float* dlogits, float* dl_tok, float* dl_perm,
                             cudaStream_t st);
// With dm.capacity > 0 the permutation is the drop-and-pad one; it also writes the dropless
// index arrays (dest_full, row_src_full, offsets_full) into the workspace. x == nullptr
// builds the indices only (no row is moved).
cudaError_t launch_permute(const void* x, const int32_t* idx, const float* topk_w, const moe_dims& dm,
                           void* x_perm, int32_t* dest, int32_t* row_src, int32_t* offsets,
                           float* w_perm, const WsLayout& L, uint8_t* ws, int* err, cudaStream_t st);
// Drop-and-pad: zero the padding rows of a [E*C, width] buffer (row i of expert e = i / C is
// padding when i - e*C >= the expert's dropless count); row_src / w_perm, when given, get
// -1 / 0 there.
cudaError_t launch_pad_rows(void* buf, int width, int dtype, const int32_t* offsets_full, int E,
                            int C, int32_t* row_src, float* w_perm, cudaStream_t st);
cudaError_t launch_permute_rows(const void* x, const int32_t* dest, const moe_dims& dm, void* x_perm,
                                cudaStream_t st);
// Fused un-rearrangement: scatter_rows[dest[c]] = c for the n = T*k dropless copies.
cudaError_t launch_scatter_rows(const int32_t* dest, int64_t n, int32_t* scatter_rows, cudaStream_t st);
cudaError_t launch_combine(const void* y_perm, const int32_t* dest, const float* topk_w,
                           const void* y_sh, const int32_t* idx, const float* dl_tok,
                           const float* w_rT, const moe_dims& dm, void* y, cudaStream_t st);
cudaError_t launch_router_split(const float* w_r, int d, int E, void* w_split, cudaStream_t st);
cudaError_t launch_router_reduce(const float* part, int64_t T, int E, int nsplit, float* logits,
                                 cudaStream_t st);
int balance_blocks(int64_t T);
int balance_term_parts(int E);   // the loss shares after the partial rows (one per 32 experts)
cudaError_t launch_balance(const float* logits, const float* bias, const int32_t* counts, int64_t T,
                           int E, int k, float alpha, float* part, float* prob_mean, float* aux_loss,
                           cudaStream_t st);
// launch_route_topk with the balance statistics of launch_balance fused in (same results,
// bit for bit); part: [balance_blocks(T)][E] fp32, then balance_term_parts(E) fp32.
cudaError_t launch_route_topk_balance(const float* logits, const float* bias, int64_t T, int E, int k,
                                      float alpha, int32_t* idx, float* w, int32_t* counts, float* part,
                                      float* prob_mean, float* aux_loss, cudaStream_t st);
cudaError_t launch_balance_bwd(const float* logits, const float* bias, const int32_t* counts,
                               int64_t T, int E, int64_t group_len, float scale, float* dlogits,
                               cudaStream_t st);
int balance_group_chunks(int64_t group_len);
cudaError_t launch_balance_groups(const float* logits, const float* bias, const int32_t* idx, int64_t T,
                                  int E, int k, int64_t group_len, float alpha, float* part,
                                  float* gterm, float* prob_mean, int32_t* counts, float* aux_loss,
                                  cudaStream_t st);
cudaError_t launch_transpose_f32(const float* in, int rows, int cols, float* out, cudaStream_t st);
cudaError_t launch_dwr(const void* x, const int32_t* row_src, const float* dl_perm,
                       const int32_t* offsets, const moe_dims& dm, float* part, float* dw_r,
                       cudaStream_t st);
cudaError_t launch_timeout_probe(int* err, uint64_t limit_ns, cudaStream_t st);

int simt_dgate_tiles(int f);
int tc_dgate_tiles(int f);
cudaError_t launch_simt_grouped(int mode, const GroupedArgs& a, int num_sms, cudaStream_t st);
// Returns MOE_OK or a negative status (tensor-map encoding can fail on the host).
int launch_tc_grouped(int mode, const GroupedArgs& a, int num_sms, cudaStream_t st);
// dW2 / dW13 on CTA pairs (tcgen05.mma.cta_group::2)
int launch_tc_pair_dw(int mode, const GroupedArgs& a, int num_sms, cudaStream_t st);

}  // namespace moe
