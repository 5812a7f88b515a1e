// Router: fp32 scores (a0), fused softmax -> top-k -> gates -> counts (a1), and the router
// backward (score gradient of the renormalised softmax, router dW).
#include <float.h>

#include "common.cuh"
#include "internal.h"
#include "trace.h"

namespace moe {
namespace {

// ---------------------------------------------------------------- a0: L = x W_r (fp32 FMA)
constexpr int RBM = 64, RBN = 64, RBK = 16;

template <typename TX>
__global__ void __launch_bounds__(256) router_logits_kernel(const TX* __restrict__ x,
                                                            const float* __restrict__ w_r,
                                                            float* __restrict__ L, int64_t T,
                                                            int d, int E) {
  __shared__ float As[RBK][RBM + 4];
  __shared__ float Bs[RBK][RBN + 4];
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int64_t m0 = (int64_t)blockIdx.y * RBM;
  const int n0 = blockIdx.x * RBN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += RBK) {
    {  // A: 64 rows x 16 k, 4 consecutive k per thread (d is a multiple of 8)
      const int r = tid >> 2, kq = (tid & 3) * 4;
      const int64_t gm = m0 + r;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (gm < T && k0 + kq < d) {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = to_f32(x[gm * d + k0 + kq + i]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) As[kq + i][r] = v[i];
    }
    {  // B: 16 k x 64 experts
      const int kk = tid >> 4, nq = (tid & 15) * 4;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int n = n0 + nq + i;
        Bs[kk][nq + i] = (k0 + kk < d && n < E) ? w_r[(int64_t)(k0 + kk) * E + n] : 0.f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < RBK; ++kk) {
      const float4 a4 = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 b4 = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float av[4] = {a4.x, a4.y, a4.z, a4.w};
      const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t gm = m0 + ty * 4 + i;
    if (gm >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < E) L[gm * E + n] = acc[i][j];
    }
  }
}

// Order-preserving map of a float (not NaN) to uint32: a > b as floats iff key(a) > key(b);
// +0 and -0 get different keys, so callers pass x + 0.f (which is +0 for both zeros).
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// ---------------------------------------------------------------- a1: fused route
// One warp per token. Lane l holds the scores of experts l, l+32, ... (V per lane).
// k rounds of a warp arg-max under the order (score descending, index ascending).
// BAL: the balance statistics' softmax sums are taken from the same registers (the scores are
// read once): each lane keeps fp32 sums of the full softmax for its experts over the warp's
// tokens, and the block writes one partial row part[blockIdx.x][E], its warps summed in order.
// With the grid of balance_partial_kernel the partial rows are the same bits as that kernel's.
template <int V, bool BAL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits,
                                                         const float* __restrict__ bias, int64_t T,
                                                         int E, int k, int32_t* __restrict__ idx,
                                                         float* __restrict__ w,
                                                         int32_t* __restrict__ counts,
                                                         float* __restrict__ part) {
  extern __shared__ int hist[];   // [E] counts, then (BAL) [8][E] fp32 warp sums
  for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  float acc[BAL ? V : 1];
#pragma unroll
  for (int i = 0; i < (BAL ? V : 1); ++i) acc[i] = 0.f;
  // the next token's scores are loaded while this token's are ranked
  const int64_t stride = (int64_t)gridDim.x * nw;
  float nxt[V];
  auto load_row = [&](int64_t t) {
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int e = lane + 32 * i;
      nxt[i] = (t < T && e < E) ? __ldg(logits + t * E + e) : 0.f;
    }
  };
  load_row((int64_t)blockIdx.x * nw + warp);
  for (int64_t t = (int64_t)blockIdx.x * nw + warp; t < T; t += stride) {
    float v[V];
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        float s = nxt[i];
        if (bias != nullptr) s = s + __ldg(bias + e);   // one fp32 rounding
        v[i] = s;
      } else {
        v[i] = -FLT_MAX;
        taken |= 1u << i;
      }
    }
    load_row(t + stride);
    if constexpr (BAL) {
      // full softmax of the row, in the same operations as balance_partial_kernel
      float mx = -FLT_MAX;
#pragma unroll
      for (int i = 0; i < V; ++i)
        if (lane + 32 * i < E) mx = fmaxf(mx, v[i]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      float p[V];
      float z = 0.f;
#pragma unroll
      for (int i = 0; i < V; ++i) {
        p[i] = (lane + 32 * i < E) ? expf(v[i] - mx) : 0.f;
        z += p[i];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
      const float inv = 1.f / z;
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = fmaf(p[i], inv, acc[i]);
    }
    // selection on order-preserving integer keys of the scores (-0 taken as +0, so that the two
    // zeros tie as they do in a float comparison); a chosen or absent expert has key 0, below
    // every finite score. Round j: each lane's best key (its lowest expert on a tie), the
    // warp's maximum key, then the lowest expert index holding it: two warp reductions.
    uint32_t key[V];
#pragma unroll
    for (int i = 0; i < V; ++i) key[i] = ((taken >> i) & 1u) ? 0u : order_key(v[i] + 0.f);
    uint32_t my_key = 0;
    int my_i = 0;
    for (int j = 0; j < k; ++j) {
      uint32_t kb = 0;
      int ib = 0;
#pragma unroll
      for (int i = 0; i < V; ++i) {
        if (key[i] > kb) {
          kb = key[i];
          ib = i;
        }
      }
      const uint32_t wmax = __reduce_max_sync(0xffffffffu, kb);
      const uint32_t wi = __reduce_min_sync(0xffffffffu, kb == wmax ? (uint32_t)(lane + 32 * ib) : 0xffffffffu);
      if (lane == (int)(wi & 31u)) {
#pragma unroll
        for (int i = 0; i < V; ++i)
          if (i == (int)(wi >> 5)) key[i] = 0u;
      }
      if (lane == j) {
        my_key = wmax;
        my_i = (int)wi;
      }
    }
    const float my_v = key_value(my_key);
    const float m = __shfl_sync(0xffffffffu, my_v, 0);   // top-1 = row maximum
    const float ex = lane < k ? expf(my_v - m) : 0.f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane < k) {
      idx[t * k + lane] = my_i;
      w[t * k + lane] = ex / sum;
      atomicAdd(&hist[my_i], 1);
    }
  }
  if constexpr (BAL) {
    float* wsum = reinterpret_cast<float*>(hist + E);
#pragma unroll
    for (int i = 0; i < V; ++i)
      if (lane + 32 * i < E) wsum[warp * E + lane + 32 * i] = acc[i];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x)
    if (hist[i] != 0) atomicAdd(counts + i, hist[i]);
  if constexpr (BAL) {
    const float* wsum = reinterpret_cast<const float*>(hist + E);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      float s = 0.f;
      for (int w8 = 0; w8 < nw; ++w8) s += wsum[w8 * E + e];
      part[(int64_t)blockIdx.x * E + e] = s;
    }
  }
}

// ---------------------------------------------------------------- router backward
// dl_j = w_j (dgate_j - sum_i w_i dgate_i) on the top-k, 0 elsewhere. One warp per token.
// dgate comes either directly or as the sum of per-N-tile partials at row dest[q].
__global__ void __launch_bounds__(256) route_bwd_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ w, const float* __restrict__ dgate_in,
    const float* __restrict__ dgate_part, int n_part, int64_t part_stride,
    const int32_t* __restrict__ dest, const int32_t* __restrict__ dest_dl, int64_t T, int E, int k,
    float* __restrict__ dgate_out, float* __restrict__ dlogits, float* __restrict__ dl_tok,
    float* __restrict__ dl_perm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int64_t t = (int64_t)blockIdx.x * nw + warp; t < T; t += (int64_t)gridDim.x * nw) {
    const int64_t q = t * k + lane;
    float dg = 0.f, wj = 0.f;
    int dq = -1, e = -1, dl_at = -1;
    if (lane < k) {
      wj = w[q];
      e = idx[q];
      if (dest != nullptr) dq = dest[q];
      if (dest_dl != nullptr) dl_at = dest_dl[q];
      if (dgate_in != nullptr) {
        dg = dgate_in[q];
      } else if (dq >= 0) {
        for (int p = 0; p < n_part; ++p) dg += dgate_part[(int64_t)p * part_stride + dq];
      }
      if (dgate_out != nullptr) dgate_out[q] = dg;
    }
    float s = wj * dg;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float dl = wj * (dg - s);
    if (dlogits != nullptr) {
      for (int c = lane; c < E; c += 32) dlogits[t * E + c] = 0.f;
      __syncwarp();
      if (lane < k && e >= 0 && e < E) dlogits[t * E + e] = dl;
    }
    if (lane < k) {
      if (dl_tok != nullptr) dl_tok[q] = dl;
      if (dl_perm != nullptr && dl_at >= 0) dl_perm[dl_at] = dl;
    }
  }
}

// Exact split of the fp32 router weight into three bf16 parts, transposed to K-major:
// ws[e][j*d + c] = part j of W_r[c][e], with hi = bf16(w), mid = bf16(w - hi),
// lo = bf16(w - hi - mid).  Each bf16 holds 8 significant bits, every subtraction is exact and
// the residual shrinks by at least 2^8 per step, so hi + mid + lo == w exactly for every fp32 w
// of magnitude >= 2^-100 (where the residuals stay normal numbers).
__global__ void router_split_kernel(const float* __restrict__ w_r, int d, int E,
                                    __nv_bfloat16* __restrict__ ws) {
  __shared__ float tile[32][33];
  const int e0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int c = c0 + i, e = e0 + threadIdx.x;
    tile[i][threadIdx.x] = (c < d && e < E) ? w_r[(int64_t)c * E + e] : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int e = e0 + i, c = c0 + threadIdx.x;
    if (e >= E || c >= d) continue;
    const float v = tile[threadIdx.x][i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
    __nv_bfloat16* row = ws + (int64_t)e * 3 * d;
    row[c] = hi;
    row[d + c] = mid;
    row[2 * d + c] = lo;
  }
}

// logits[t][e] = sum over the K slices g (in order) of part[g][t][e]; part rows are padded
// to a multiple of 32 experts.
__global__ void router_reduce_kernel(const float* __restrict__ part, int64_t T, int E, int epad,
                                     int nsplit, float* __restrict__ logits) {
  const int64_t n = T * E;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / E;
    const int e = (int)(i - t * E);
    float s = 0.f;
    for (int g = 0; g < nsplit; ++g) s += part[((int64_t)g * T + t) * epad + e];
    logits[i] = s;
  }
}

// ---------------------------------------------------------------- load-balance statistics
// Mean full-softmax probability per expert. One warp per token (fixed token order per warp);
// each lane keeps fp32 sums for its experts, then the block sums its warps in order and writes
// one partial row per block; balance_final_kernel sums the block rows in order.
template <int V>
__global__ void __launch_bounds__(256) balance_partial_kernel(const float* __restrict__ logits,
                                                              const float* __restrict__ bias,
                                                              int64_t T, int E,
                                                              float* __restrict__ part) {
  __shared__ float wsum[8][kMaxE];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  // the next token's scores are loaded while this token's are summed
  const int64_t stride = (int64_t)gridDim.x * nw;
  float nxt[V];
  auto load_row = [&](int64_t t) {
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int e = lane + 32 * i;
      nxt[i] = (t < T && e < E) ? __ldg(logits + t * E + e) : 0.f;
    }
  };
  load_row((int64_t)blockIdx.x * nw + warp);
  for (int64_t t = (int64_t)blockIdx.x * nw + warp; t < T; t += stride) {
    float v[V];
    float m = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int e = lane + 32 * i;
      v[i] = -FLT_MAX;
      if (e < E) {
        float s = nxt[i];
        if (bias != nullptr) s = s + __ldg(bias + e);
        v[i] = s;
        m = fmaxf(m, s);
      }
    }
    load_row(t + stride);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      v[i] = (lane + 32 * i < E) ? expf(v[i] - m) : 0.f;
      z += v[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const float inv = 1.f / z;
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = fmaf(v[i], inv, acc[i]);
  }
#pragma unroll
  for (int i = 0; i < V; ++i)
    if (lane + 32 * i < E) wsum[warp][lane + 32 * i] = acc[i];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float s = 0.f;
    for (int w = 0; w < nw; ++w) s += wsum[w][e];
    part[(int64_t)blockIdx.x * E + e] = s;
  }
}

// P_e = (sum over block rows) / T;  L_aux = alpha * E / (T * k) * sum_e counts_e * P_e.
// Block b takes experts 32b .. 32b+31: thread (j, el) sums slice j of expert 32b + el (block
// rows j, j + 32, ..., ascending; a warp reads 32 consecutive experts of a row), warp 0 sums
// the 32 slices in order, writes P and the block's share of the loss sum (its experts in a
// fixed butterfly order). balance_loss_kernel adds the shares in block order.
__global__ void __launch_bounds__(1024) balance_final_kernel(const float* __restrict__ part,
                                                             int nblocks, const int32_t* __restrict__ counts,
                                                             int64_t T, int E,
                                                             float* __restrict__ prob_mean,
                                                             float* __restrict__ term_part) {
  __shared__ float slice[32][33];
  const int el = threadIdx.x & 31, j = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + el;
  float s = 0.f;
  if (e < E)
    for (int b = j; b < nblocks; b += 32) s += part[(int64_t)b * E + e];
  slice[j][el] = s;
  __syncthreads();
  if (j == 0) {
    float term = 0.f;
    if (e < E) {
      float tot = 0.f;
      for (int q = 0; q < 32; ++q) tot += slice[q][el];
      const float P = tot / (float)T;
      if (prob_mean != nullptr) prob_mean[e] = P;
      term = (float)counts[e] * P;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) term += __shfl_xor_sync(0xffffffffu, term, o);
    if (el == 0) term_part[blockIdx.x] = term;
  }
}

__global__ void balance_loss_kernel(const float* __restrict__ term_part, int nparts, int64_t T, int E, int k,
                                    float alpha, float* __restrict__ aux_loss) {
  if (threadIdx.x != 0 || aux_loss == nullptr) return;
  float s = 0.f;
  for (int i = 0; i < nparts; ++i) s += term_part[i];
  aux_loss[0] = alpha * (float)E / ((float)T * (float)k) * s;
}

// Sequence-level statistics: groups of group_len consecutive tokens. Block (c, g) sums the
// softmax probabilities of a fixed slice of group g's tokens (one warp per token, fixed order)
// into part[g][c][E] and counts the group's top-k choices (integer atomics: exact, so the
// result does not depend on their order).
template <int V>
__global__ void __launch_bounds__(256) balance_group_partial_kernel(
    const float* __restrict__ logits, const float* __restrict__ bias, const int32_t* __restrict__ idx,
    int E, int k, int64_t group_len, float* __restrict__ part, int32_t* __restrict__ counts) {
  __shared__ float wsum[8][kMaxE];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int64_t g = blockIdx.y, t0 = g * group_len;
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  for (int64_t u = (int64_t)blockIdx.x * nw + warp; u < group_len; u += (int64_t)gridDim.x * nw) {
    const int64_t t = t0 + u;
    float v[V];
    float m = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int e = lane + 32 * i;
      v[i] = -FLT_MAX;
      if (e < E) {
        float s = __ldg(logits + t * E + e);
        if (bias != nullptr) s = s + __ldg(bias + e);
        v[i] = s;
        m = fmaxf(m, s);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      v[i] = (lane + 32 * i < E) ? expf(v[i] - m) : 0.f;
      z += v[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const float inv = 1.f / z;
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = fmaf(v[i], inv, acc[i]);
    if (lane < k) {
      const int e = __ldg(idx + t * k + lane);
      if (e >= 0 && e < E) atomicAdd(counts + g * E + e, 1);
    }
  }
#pragma unroll
  for (int i = 0; i < V; ++i)
    if (lane + 32 * i < E) wsum[warp][lane + 32 * i] = acc[i];
  __syncthreads();
  float* out = part + ((int64_t)g * gridDim.x + blockIdx.x) * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float s = 0.f;
    for (int w = 0; w < nw; ++w) s += wsum[w][e];
    out[e] = s;
  }
}

// One block per group: P_ge = (sum of the group's block rows) / group_len and the group's
// term sum_e counts_ge * P_ge.
__global__ void __launch_bounds__(1024) balance_group_final_kernel(
    const float* __restrict__ part, int nchunks, const int32_t* __restrict__ counts, int E,
    int64_t group_len, float* __restrict__ prob_mean, float* __restrict__ gterm) {
  __shared__ float red[32];
  const int64_t g = blockIdx.x;
  const int e = threadIdx.x;
  float term = 0.f;
  if (e < E) {
    float s = 0.f;
    for (int c = 0; c < nchunks; ++c) s += part[(g * nchunks + c) * E + e];
    const float P = s / (float)group_len;
    if (prob_mean != nullptr) prob_mean[g * E + e] = P;
    term = (float)counts[g * E + e] * P;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) term += __shfl_xor_sync(0xffffffffu, term, o);
  if (lane == 0) red[warp] = term;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w];
    gterm[g] = s;
  }
}

// L_aux = alpha * E / (G * group_len * k) * sum_g term_g, summed in group order by one thread
// per 1024-group stripe and then a fixed shuffle tree.
__global__ void __launch_bounds__(1024) balance_group_loss_kernel(const float* __restrict__ gterm,
                                                                  int64_t G, float scale,
                                                                  float* __restrict__ aux_loss) {
  __shared__ float red[32];
  float s = 0.f;
  for (int64_t g = threadIdx.x; g < G; g += blockDim.x) s += gterm[g];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) red[warp] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
    aux_loss[0] = scale * t;
  }
}

// dlogits[t, e] += scale * p_te * (c_e - sum_e' c_e' p_te'), c = the counts of token t's group
// (group t / group_len), scale = grad * alpha * E / (n_groups * group_len^2 * k). One warp per
// token.
template <int V>
__global__ void __launch_bounds__(256) balance_bwd_kernel(const float* __restrict__ logits,
                                                          const float* __restrict__ bias,
                                                          const int32_t* __restrict__ counts_all,
                                                          int64_t T, int E, int64_t group_len,
                                                          float scale, float* __restrict__ dlogits) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int64_t t = (int64_t)blockIdx.x * nw + warp; t < T; t += (int64_t)gridDim.x * nw) {
    const int32_t* counts = counts_all + (t / group_len) * E;   // the token's group
    float v[V], c[V];
    float m = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int e = lane + 32 * i;
      v[i] = -FLT_MAX;
      c[i] = 0.f;
      if (e < E) {
        float s = __ldg(logits + t * E + e);
        if (bias != nullptr) s = s + __ldg(bias + e);
        v[i] = s;
        c[i] = (float)__ldg(counts + e);
        m = fmaxf(m, s);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      v[i] = (lane + 32 * i < E) ? expf(v[i] - m) : 0.f;
      z += v[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const float inv = 1.f / z;
    float cp = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      v[i] *= inv;
      cp = fmaf(c[i], v[i], cp);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cp += __shfl_xor_sync(0xffffffffu, cp, o);
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int e = lane + 32 * i;
      if (e < E) dlogits[t * E + e] += scale * v[i] * (c[i] - cp);
    }
  }
}

// out[c][r] = in[r][c] for an fp32 [rows][cols] matrix.
__global__ void transpose_f32_kernel(const float* __restrict__ in, int rows, int cols,
                                     float* __restrict__ out) {
  __shared__ float tile[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    tile[i][threadIdx.x] = (r < rows && c < cols) ? in[(int64_t)r * cols + c] : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (c < cols && r < rows) out[(int64_t)c * rows + r] = tile[threadIdx.x][i];
  }
}

// Router dW: dW_r[:, e] = sum over the copies routed to e of dl * x[token]. Deterministic:
// each expert's rows are cut into kDwrSplit fixed slices, each slice summed in row order,
// then the slices are summed in slice order.
// 16 bytes of x as fp32: 8 bf16 or 4 fp32 columns.
__device__ __forceinline__ void vec16_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ void vec16_to_f32(const uint4& u, float (&f)[4]) {
  f[0] = __uint_as_float(u.x);
  f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z);
  f[3] = __uint_as_float(u.w);
}

// Each thread owns 16 bytes of columns; the rows of its slice are fetched four at a time
// (indices, then the x vectors) and accumulated one by one in row order.
template <typename TX>
__global__ void __launch_bounds__(256) dwr_partial_kernel(const TX* __restrict__ x,
                                                          const int32_t* __restrict__ row_src,
                                                          const float* __restrict__ dl_perm,
                                                          const int32_t* __restrict__ offsets, int d,
                                                          int E, float* __restrict__ part) {
  constexpr int V = 16 / sizeof(TX);
  const int e = blockIdx.x / kDwrSplit, sl = blockIdx.x % kDwrSplit;
  const int64_t lo = offsets[e], n = offsets[e + 1] - lo;
  const int64_t r0 = lo + n * sl / kDwrSplit, r1 = lo + n * (sl + 1) / kDwrSplit;
  const int c = (blockIdx.y * blockDim.x + threadIdx.x) * V;
  if (c >= d) return;
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  int64_t r = r0;
  for (; r + 4 <= r1; r += 4) {
    int64_t t[4];
    float g[4];
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      t[j] = row_src[r + j];
      g[j] = dl_perm[r + j];
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = __ldg(reinterpret_cast<const uint4*>(x + t[j] * d + c));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float f[V];
      vec16_to_f32(v[j], f);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = fmaf(g[j], f[i], acc[i]);
    }
  }
  for (; r < r1; ++r) {
    float f[V];
    vec16_to_f32(__ldg(reinterpret_cast<const uint4*>(x + (int64_t)row_src[r] * d + c)), f);
    const float g = dl_perm[r];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = fmaf(g, f[i], acc[i]);
  }
  float4* out = reinterpret_cast<float4*>(part + ((int64_t)sl * E + e) * d + c);
#pragma unroll
  for (int i = 0; i < V / 4; ++i) out[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
}

// dw_r[c][e] = sum_sl part[sl][e][c] (slice order), through a 32x32 transpose tile.
__global__ void dwr_reduce_kernel(const float* __restrict__ part, int d, int E,
                                  float* __restrict__ dw_r) {
  __shared__ float tile[32][33];
  const int c0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int e = e0 + i, c = c0 + threadIdx.x;
    float s = 0.f;
    if (e < E && c < d)
      for (int sl = 0; sl < kDwrSplit; ++sl) s += part[((int64_t)sl * E + e) * d + c];
    tile[i][threadIdx.x] = s;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int c = c0 + i, e = e0 + threadIdx.x;
    if (c < d && e < E) dw_r[(int64_t)c * E + e] = tile[threadIdx.x][i];
  }
}

// A bounded wait on a barrier nothing completes: exercises the timeout path end to end.
__global__ void timeout_probe_kernel(int* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, err, limit_ns);
  __syncthreads();
}

}  // namespace

cudaError_t launch_router_logits(const void* x, const float* w_r, const moe_dims& dm, float* logits,
                                 cudaStream_t st) {
  const dim3 grid((dm.E + RBN - 1) / RBN, (unsigned)((dm.T + RBM - 1) / RBM)), block(256);
  TraceScope ts(TP_ROUTER_GEMM, st);
  if (dm.dtype == MOE_F32)
    router_logits_kernel<float><<<grid, block, 0, st>>>((const float*)x, w_r, logits, dm.T, dm.d, dm.E);
  else
    router_logits_kernel<__nv_bfloat16><<<grid, block, 0, st>>>((const __nv_bfloat16*)x, w_r, logits,
                                                                dm.T, dm.d, dm.E);
  return cudaGetLastError();
}

cudaError_t launch_route_topk(const float* logits, const float* bias, int64_t T, int E, int k,
                              int32_t* idx, float* w, int32_t* counts, int num_sms, cudaStream_t st) {
  const int threads = 256, wpb = threads / 32;
  int64_t blocks = (T + wpb - 1) / wpb;
  if (blocks > 4 * num_sms) blocks = 4 * num_sms;
  if (blocks < 1) blocks = 1;
  const size_t sm = sizeof(int) * E;
  const int V = (E + 31) / 32;
  TraceScope ts(TP_ROUTE_TOPK, st);
#define MOE_ROUTE_CASE(VV)                                                                          \
  route_topk_kernel<VV, false><<<(unsigned)blocks, threads, sm, st>>>(logits, bias, T, E, k, idx, w, \
                                                                      counts, nullptr);
  if (V <= 1) { MOE_ROUTE_CASE(1) }
  else if (V <= 2) { MOE_ROUTE_CASE(2) }
  else if (V <= 4) { MOE_ROUTE_CASE(4) }
  else if (V <= 8) { MOE_ROUTE_CASE(8) }
  else if (V <= 16) { MOE_ROUTE_CASE(16) }
  else { MOE_ROUTE_CASE(32) }
#undef MOE_ROUTE_CASE
  return cudaGetLastError();
}

cudaError_t launch_route_bwd(const int32_t* idx, const float* w, const float* dgate_in,
                             const float* dgate_part, int n_part, int64_t part_stride,
                             const int32_t* dest, const int32_t* dest_dl, int64_t T, int E, int k,
                             float* dgate_out, float* dlogits, float* dl_tok, float* dl_perm,
                             cudaStream_t st) {
  const int threads = 256, wpb = threads / 32;
  int64_t blocks = (T + wpb - 1) / wpb;
  if (blocks > 65535) blocks = 65535;
  TraceScope ts(TP_ROUTE_BWD, st);
  route_bwd_kernel<<<(unsigned)blocks, threads, 0, st>>>(idx, w, dgate_in, dgate_part, n_part,
                                                         part_stride, dest, dest_dl, T, E, k,
                                                         dgate_out, dlogits, dl_tok, dl_perm);
  return cudaGetLastError();
}

cudaError_t launch_router_split(const float* w_r, int d, int E, void* w_split, cudaStream_t st) {
  const dim3 grid((E + 31) / 32, (d + 31) / 32), block(32, 8);
  TraceScope ts(TP_TRANSPOSE, st);
  router_split_kernel<<<grid, block, 0, st>>>(w_r, d, E, static_cast<__nv_bfloat16*>(w_split));
  return cudaGetLastError();
}

cudaError_t launch_router_reduce(const float* part, int64_t T, int E, int nsplit, float* logits,
                                 cudaStream_t st) {
  int64_t blocks = (T * E + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  TraceScope ts(TP_ROUTER_GEMM, st);
  router_reduce_kernel<<<(unsigned)blocks, 256, 0, st>>>(part, T, E, (E + 31) & ~31, nsplit, logits);
  return cudaGetLastError();
}

int balance_term_parts(int E) { return (E + 31) / 32; }

int balance_blocks(int64_t T) {
  constexpr int64_t kMaxBlocks = 512;
  int64_t b = (T + 7) / 8;
  return (int)(b < kMaxBlocks ? (b < 1 ? 1 : b) : kMaxBlocks);
}

#define MOE_V_DISPATCH(E, CALL)            \
  do {                                     \
    const int V_ = ((E) + 31) / 32;        \
    if (V_ <= 1) { constexpr int VV = 1; CALL; } \
    else if (V_ <= 2) { constexpr int VV = 2; CALL; } \
    else if (V_ <= 4) { constexpr int VV = 4; CALL; } \
    else if (V_ <= 8) { constexpr int VV = 8; CALL; } \
    else if (V_ <= 16) { constexpr int VV = 16; CALL; } \
    else { constexpr int VV = 32; CALL; } \
  } while (0)

// part: nb rows of E partial sums, followed by room for balance_term_parts(E) floats.
static cudaError_t launch_balance_final(float* part, int nb, const int32_t* counts, int64_t T, int E, int k,
                                        float alpha, float* prob_mean, float* aux_loss, cudaStream_t st) {
  const int nt = balance_term_parts(E);
  float* term_part = part + (size_t)nb * E;
  TraceScope ts(TP_MISC, st);
  balance_final_kernel<<<nt, 1024, 0, st>>>(part, nb, counts, T, E, prob_mean, term_part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  balance_loss_kernel<<<1, 32, 0, st>>>(term_part, nt, T, E, k, alpha, aux_loss);
  return cudaGetLastError();
}

cudaError_t launch_balance(const float* logits, const float* bias, const int32_t* counts, int64_t T,
                           int E, int k, float alpha, float* part, float* prob_mean, float* aux_loss,
                           cudaStream_t st) {
  const int nb = balance_blocks(T);
  {
    TraceScope ts(TP_MISC, st);
    MOE_V_DISPATCH(E, (balance_partial_kernel<VV><<<nb, 256, 0, st>>>(logits, bias, T, E, part)));
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_balance_final(part, nb, counts, T, E, k, alpha, prob_mean, aux_loss, st);
}

cudaError_t launch_route_topk_balance(const float* logits, const float* bias, int64_t T, int E, int k,
                                      float alpha, int32_t* idx, float* w, int32_t* counts, float* part,
                                      float* prob_mean, float* aux_loss, cudaStream_t st) {
  // the grid of balance_partial_kernel, so that the partial rows (and everything after them)
  // are the same bits as the separate statistics call
  const int nb = balance_blocks(T);
  const size_t sm = sizeof(int) * E + sizeof(float) * 8 * E;
  {
    TraceScope ts(TP_ROUTE_TOPK, st);
    MOE_V_DISPATCH(E, (route_topk_kernel<VV, true><<<nb, 256, sm, st>>>(logits, bias, T, E, k, idx, w, counts,
                                                                         part)));
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_balance_final(part, nb, counts, T, E, k, alpha, prob_mean, aux_loss, st);
}

cudaError_t launch_balance_bwd(const float* logits, const float* bias, const int32_t* counts,
                               int64_t T, int E, int64_t group_len, float scale, float* dlogits,
                               cudaStream_t st) {
  int64_t blocks = (T + 7) / 8;
  if (blocks > 65535) blocks = 65535;
  TraceScope ts(TP_MISC, st);
  MOE_V_DISPATCH(E, (balance_bwd_kernel<VV><<<(unsigned)blocks, 256, 0, st>>>(logits, bias, counts, T, E,
                                                                               group_len, scale, dlogits)));
  return cudaGetLastError();
}

int balance_group_chunks(int64_t group_len) {
  int64_t c = (group_len + 63) / 64;
  return (int)(c < 32 ? (c < 1 ? 1 : c) : 32);
}

cudaError_t launch_balance_groups(const float* logits, const float* bias, const int32_t* idx, int64_t T,
                                  int E, int k, int64_t group_len, float alpha, float* part,
                                  float* gterm, float* prob_mean, int32_t* counts, float* aux_loss,
                                  cudaStream_t st) {
  const int64_t G = T / group_len;
  const int nc = balance_group_chunks(group_len);
  TraceScope ts(TP_MISC, st);
  if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * (size_t)G * E, st) != cudaSuccess) return cudaErrorUnknown;
  MOE_V_DISPATCH(E, (balance_group_partial_kernel<VV><<<dim3(nc, (unsigned)G), 256, 0, st>>>(
                        logits, bias, idx, E, k, group_len, part, counts)));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  balance_group_final_kernel<<<(unsigned)G, 1024, 0, st>>>(part, nc, counts, E, group_len, prob_mean, gterm);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const double scale = (double)alpha * E / ((double)G * (double)group_len * (double)k);
  balance_group_loss_kernel<<<1, 1024, 0, st>>>(gterm, G, (float)scale, aux_loss);
  return cudaGetLastError();
}

cudaError_t launch_transpose_f32(const float* in, int rows, int cols, float* out, cudaStream_t st) {
  const dim3 grid((cols + 31) / 32, (rows + 31) / 32), block(32, 8);
  TraceScope ts(TP_TRANSPOSE, st);
  transpose_f32_kernel<<<grid, block, 0, st>>>(in, rows, cols, out);
  return cudaGetLastError();
}

cudaError_t launch_dwr(const void* x, const int32_t* row_src, const float* dl_perm,
                       const int32_t* offsets, const moe_dims& dm, float* part, float* dw_r,
                       cudaStream_t st) {
  const int cols_per_block = 256 * (dm.dtype == MOE_F32 ? 4 : 8);
  const dim3 g1(dm.E * kDwrSplit, (dm.d + cols_per_block - 1) / cols_per_block), b1(256);
  {
  TraceScope ts(TP_DWR, st);
  if (dm.dtype == MOE_F32)
    dwr_partial_kernel<float><<<g1, b1, 0, st>>>((const float*)x, row_src, dl_perm, offsets, dm.d, dm.E, part);
  else
    dwr_partial_kernel<__nv_bfloat16><<<g1, b1, 0, st>>>((const __nv_bfloat16*)x, row_src, dl_perm,
                                                         offsets, dm.d, dm.E, part);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 g2((dm.d + 31) / 32, (dm.E + 31) / 32), b2(32, 8);
  TraceScope ts(TP_DWR, st);
  dwr_reduce_kernel<<<g2, b2, 0, st>>>(part, dm.d, dm.E, dw_r);
  return cudaGetLastError();
}

cudaError_t launch_timeout_probe(int* err, uint64_t limit_ns, cudaStream_t st) {
  TraceScope ts(TP_MISC, st);
  timeout_probe_kernel<<<1, 32, 0, st>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace moe
