// VectorSort rearrange / un-rearrange: the stable expert permutation of token copies built
// on the device (per-chunk expert bitmasks -> local ranks and chunk histograms -> scan ->
// scatter), the row moves in 16-byte vectors, and the gate-weighted combine.
#include "common.cuh"
#include "internal.h"
#include "trace.h"

namespace moe {
namespace {

// ---------------------------------------------------------------- P1: chunk masks
// One block per chunk of kChunk tokens, one thread per token. For every expert a 64-bit mask
// of the chunk's tokens routed to it; a copy's rank inside the chunk is the popcount of the
// mask below its token (tokens are distinct per expert, so this is the stable order).
__global__ void __launch_bounds__(kChunk) permute_hist_kernel(
    const int32_t* __restrict__ idx, int64_t T, int E, int k, int64_t n_chunks,
    int32_t* __restrict__ chunk_hist, int32_t* __restrict__ local_rank, int* err) {
  extern __shared__ uint32_t mask[];  // [E][2]
  const int64_t c = blockIdx.x;
  const int tid = threadIdx.x;
  for (int i = tid; i < 2 * E; i += kChunk) mask[i] = 0u;
  __syncthreads();
  const int64_t t = c * kChunk + tid;
  const bool tok = t < T;
  const int word = tid >> 5;
  const uint32_t bit = 1u << (tid & 31);
  if (tok) {
    for (int j = 0; j < k; ++j) {
      const int e = idx[t * k + j];
      bool ok = e >= 0 && e < E;
      for (int jj = 0; jj < j && ok; ++jj) ok = idx[t * k + jj] != e;
      if (ok) atomicOr(&mask[2 * e + word], bit);
      else record_error(err, MOE_ERR_DEVICE_EXPERT_ID);
    }
  }
  __syncthreads();
  if (tok) {
    const uint32_t below = bit - 1u;
    for (int j = 0; j < k; ++j) {
      const int e = idx[t * k + j];
      bool ok = e >= 0 && e < E;
      for (int jj = 0; jj < j && ok; ++jj) ok = idx[t * k + jj] != e;
      int r = -1;
      if (ok) r = (word ? __popc(mask[2 * e]) : 0) + __popc(mask[2 * e + word] & below);
      local_rank[t * k + j] = r;
    }
  }
  for (int e = tid; e < E; e += kChunk)
    chunk_hist[(int64_t)e * n_chunks + c] = __popc(mask[2 * e]) + __popc(mask[2 * e + 1]);
}

// ---------------------------------------------------------------- P2: scans
// One block of 1024 threads. Warp w scans the chunk histograms of experts w, w+32, ...;
// then the per-expert totals are scanned into offsets.
__global__ void __launch_bounds__(1024) permute_scan_kernel(const int32_t* __restrict__ chunk_hist,
                                                            int32_t* __restrict__ chunk_base,
                                                            int64_t n_chunks, int E, int capacity,
                                                            int32_t* __restrict__ offsets,
                                                            int32_t* __restrict__ offsets_full) {
  __shared__ int cnt[kMaxE];
  __shared__ int wsum[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = warp; e < E; e += 32) {
    int run = 0;
    const int32_t* hrow = chunk_hist + (int64_t)e * n_chunks;
    int32_t* brow = chunk_base + (int64_t)e * n_chunks;
    for (int64_t c0 = 0; c0 < n_chunks; c0 += 32) {
      const int64_t c = c0 + lane;
      const int v = c < n_chunks ? hrow[c] : 0;
      int inc = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
      }
      if (c < n_chunks) brow[c] = run + inc - v;
      run += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) cnt[e] = run;
  }
  __syncthreads();
  const int e = threadIdx.x;
  const int v = e < E ? cnt[e] : 0;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += u;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int s = wsum[lane];
    int si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, si, o);
      if (lane >= o) si += u;
    }
    wsum[lane] = si - s;
  }
  __syncthreads();
  const int excl = wsum[warp] + inc - v;
  if (capacity > 0) {  // drop-and-pad: uniform segments of C rows; the dropless scan kept aside
    if (e < E) {
      offsets[e] = e * capacity;
      offsets_full[e] = excl;
    }
    if (e == E - 1) {
      offsets[E] = E * capacity;
      offsets_full[E] = excl + v;
    }
  } else {
    if (e < E) offsets[e] = excl;
    if (e == E - 1) offsets[E] = excl + v;
  }
}

// ---------------------------------------------------------------- P3: scatter + row move
// One warp per token: lanes j < k compute dest of copy j, then the row x[t] is read once in
// 16-byte vectors and written to the k destination rows.
template <typename T, int U>
__device__ __forceinline__ void copy_row_to_dests(const T* __restrict__ src, T* __restrict__ dst,
                                                  int d, int k, int dq, int lane) {
  const int nvec = d / 8;
  // the loop is uniform across the warp (every lane takes part in every shuffle, also when
  // the row has fewer than 32 * U vectors left); loads and stores are predicated
  for (int base = 0; base < nvec; base += 32 * U) {
    Vec8<T> val[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = base + lane + 32 * u;
      if (v < nvec) val[u].load(src + (int64_t)v * 8);
    }
    for (int j = 0; j < k; ++j) {
      const int dj = __shfl_sync(0xffffffffu, dq, j);
      if (dj < 0) continue;
      T* drow = dst + (int64_t)dj * d;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = base + lane + 32 * u;
        if (v < nvec) val[u].store(drow + (int64_t)v * 8);
      }
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) permute_scatter_kernel(
    const T* __restrict__ x, const int32_t* __restrict__ idx, const float* __restrict__ topk_w,
    const int32_t* __restrict__ local_rank, const int32_t* __restrict__ chunk_base,
    const int32_t* __restrict__ offsets, int64_t Tn, int d, int k, int64_t n_chunks, int capacity,
    T* __restrict__ x_perm, int32_t* __restrict__ dest, int32_t* __restrict__ row_src,
    float* __restrict__ w_perm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int64_t t = (int64_t)blockIdx.x * nw + warp; t < Tn; t += (int64_t)gridDim.x * nw) {
    int dq = -1;
    if (lane < k) {
      const int64_t q = t * k + lane;
      const int r = local_rank[q];
      if (r >= 0) {
        const int e = idx[q];
        const int rank = chunk_base[(int64_t)e * n_chunks + t / kChunk] + r;  // within expert e
        // drop-and-pad keeps the first C copies of each expert
        if (capacity == 0 || rank < capacity) {
          dq = offsets[e] + rank;
          row_src[dq] = (int32_t)t;
          if (w_perm != nullptr) w_perm[dq] = topk_w[q];
        }
      }
      dest[q] = dq;
    }
    if (x != nullptr) copy_row_to_dests<T, 4>(x + t * d, x_perm, d, k, dq, lane);
  }
}

// Drop-and-pad: one warp per row of the [E*C, width] buffer; rows past the expert's dropless
// count are padding and become zero (row_src -1, w_perm 0).
template <typename T>
__global__ void __launch_bounds__(256) pad_rows_kernel(T* __restrict__ buf, int width,
                                                       const int32_t* __restrict__ offsets_full,
                                                       int E, int C, int32_t* __restrict__ row_src,
                                                       float* __restrict__ w_perm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int64_t rows = (int64_t)E * C;
  for (int64_t i = (int64_t)blockIdx.x * nw + warp; i < rows; i += (int64_t)gridDim.x * nw) {
    const int e = (int)(i / C), r = (int)(i - (int64_t)e * C);
    if (r < offsets_full[e + 1] - offsets_full[e]) continue;   // a kept copy
    if (buf != nullptr) {
      Vec8<T> z;
      const float zf[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      z.from_float(zf);
      T* row = buf + i * width;
      for (int v = lane; v < width / 8; v += 32) z.store(row + (int64_t)v * 8);
    }
    if (lane == 0) {
      if (row_src != nullptr) row_src[i] = -1;
      if (w_perm != nullptr) w_perm[i] = 0.f;
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) permute_rows_kernel(const T* __restrict__ x,
                                                           const int32_t* __restrict__ dest,
                                                           int64_t Tn, int d, int k,
                                                           T* __restrict__ x_perm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int64_t t = (int64_t)blockIdx.x * nw + warp; t < Tn; t += (int64_t)gridDim.x * nw) {
    const int dq = lane < k ? dest[t * k + lane] : -1;
    copy_row_to_dests<T, 4>(x + t * d, x_perm, d, k, dq, lane);
  }
}

// ---------------------------------------------------------------- fused un-rearrangement
// scatter_rows[dest[c]] = c: the token-major slot of every expert-order row (dropless).
__global__ void __launch_bounds__(256) scatter_rows_kernel(const int32_t* __restrict__ dest, int64_t n,
                                                          int32_t* __restrict__ scatter_rows) {
  for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < n; c += (int64_t)gridDim.x * blockDim.x) {
    const int32_t q = dest[c];
    if (q >= 0) scatter_rows[q] = (int32_t)c;
  }
}

// ---------------------------------------------------------------- a4: combine
// y[t] = sum_j w_j y_perm[dest_j] (+ y_sh[t]) (+ sum_j dl_j W_r^T[e_j]) in fp32, in that
// order, rounded once, 8 elements per lane per step. With k <= KMAX (no router term) the
// k rows' vectors of a step (and the shared expert's) are all requested before the sums
// start, so a warp keeps k + 1 loads in flight instead of one; the sums keep their order.
// dest == nullptr: the rows are already in token-major order (copy j of token t at row
// t*k + j, written there by the fused un-rearrangement), read as one contiguous block.
template <typename T, bool ROUTER, int KMAX>
__global__ void __launch_bounds__(256) combine_kernel(
    const T* __restrict__ y_perm, const int32_t* __restrict__ dest, const float* __restrict__ topk_w,
    const T* __restrict__ y_sh, const int32_t* __restrict__ idx, const float* __restrict__ dl_tok,
    const float* __restrict__ w_rT, int64_t Tn, int d, int k, T* __restrict__ y) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int nvec = d / 8;
  if constexpr (KMAX > 0) {
    // A warp's unit of work is one segment of up to kSegVec vectors of one token's row, so
    // that short rows still give every SM enough warps (and loads) in flight.
    constexpr int kSegVec = 128;
    const int nseg = (nvec + kSegVec - 1) / kSegVec;
    const int64_t items = Tn * nseg;
    for (int64_t it = (int64_t)blockIdx.x * nw + warp; it < items; it += (int64_t)gridDim.x * nw) {
      const int64_t t = it / nseg;
      const int seg = (int)(it - t * nseg);
      int dq = -1;
      float wq = 0.f;
      if (lane < k) {
        const int64_t q = t * k + lane;
        dq = dest != nullptr ? dest[q] : (int)q;
        wq = topk_w != nullptr ? topk_w[q] : 1.f;
      }
      // every lane holds every copy's row and weight (uniform across the warp)
      int dj[KMAX];
      float wj[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        dj[j] = __shfl_sync(0xffffffffu, dq, j);
        wj[j] = __shfl_sync(0xffffffffu, wq, j);
      }
      const int vend = min(nvec, (seg + 1) * kSegVec);
      for (int vb = seg * kSegVec; vb < vend; vb += 32) {
        const int v = vb + lane;
        if (v >= vend) break;        // no shuffles below: lanes may leave
        Vec8<T> val[KMAX], sh;
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < k && dj[j] >= 0) val[j].load(y_perm + (int64_t)dj[j] * d + (int64_t)v * 8);
        if (y_sh != nullptr) sh.load(y_sh + t * d + (int64_t)v * 8);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          if (j >= k || dj[j] < 0) continue;
          float f[8];
          val[j].to_float(f);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj[j], f[i], acc[i]);
        }
        if (y_sh != nullptr) {
          float f[8];
          sh.to_float(f);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] += f[i];
        }
        Vec8<T> out;
        out.from_float(acc);
        out.store(y + t * d + (int64_t)v * 8);
      }
    }
  } else {
    // general k (and the router term): one token per warp, one row at a time
    for (int64_t t = (int64_t)blockIdx.x * nw + warp; t < Tn; t += (int64_t)gridDim.x * nw) {
      int dq = -1, eq = 0;
      float wq = 0.f, gq = 0.f;
      if (lane < k) {
        const int64_t q = t * k + lane;
        dq = dest != nullptr ? dest[q] : (int)q;
        wq = topk_w != nullptr ? topk_w[q] : 1.f;
        if (ROUTER) {
          eq = idx[q];
          gq = dl_tok[q];
        }
      }
      // uniform across the warp: every lane takes part in every shuffle; accesses predicated
      for (int vb = 0; vb < nvec; vb += 32) {
        const int v = vb + lane;
        const bool on = v < nvec;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < k; ++j) {
          const int dj = __shfl_sync(0xffffffffu, dq, j);
          const float wj = __shfl_sync(0xffffffffu, wq, j);
          if (dj < 0 || !on) continue;
          Vec8<T> val;
          val.load(y_perm + (int64_t)dj * d + (int64_t)v * 8);
          float f[8];
          val.to_float(f);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, f[i], acc[i]);
        }
        if (y_sh != nullptr && on) {
          Vec8<T> val;
          val.load(y_sh + t * d + (int64_t)v * 8);
          float f[8];
          val.to_float(f);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] += f[i];
        }
        if (ROUTER) {
          for (int j = 0; j < k; ++j) {
            const int ej = __shfl_sync(0xffffffffu, eq, j);
            const float gj = __shfl_sync(0xffffffffu, gq, j);
            if (!on) continue;
            const float4* wr = reinterpret_cast<const float4*>(w_rT + (int64_t)ej * d + (int64_t)v * 8);
            const float4 p0 = __ldg(wr), p1 = __ldg(wr + 1);
            acc[0] = fmaf(gj, p0.x, acc[0]); acc[1] = fmaf(gj, p0.y, acc[1]);
            acc[2] = fmaf(gj, p0.z, acc[2]); acc[3] = fmaf(gj, p0.w, acc[3]);
            acc[4] = fmaf(gj, p1.x, acc[4]); acc[5] = fmaf(gj, p1.y, acc[5]);
            acc[6] = fmaf(gj, p1.z, acc[6]); acc[7] = fmaf(gj, p1.w, acc[7]);
          }
        }
        if (on) {
          Vec8<T> out;
          out.from_float(acc);
          out.store(y + t * d + (int64_t)v * 8);
        }
      }
    }
  }
}

int64_t token_blocks(int64_t T, int num_per_block, int64_t cap) {
  int64_t b = (T + num_per_block - 1) / num_per_block;
  if (b > cap) b = cap;
  return b < 1 ? 1 : b;
}

}  // namespace

cudaError_t launch_permute(const void* x, const int32_t* idx, const float* topk_w, const moe_dims& dm,
                           void* x_perm, int32_t* dest, int32_t* row_src, int32_t* offsets,
                           float* w_perm, const WsLayout& L, uint8_t* ws, int* err, cudaStream_t st) {
  int32_t* chunk_hist = reinterpret_cast<int32_t*>(ws + L.chunk_hist);
  int32_t* chunk_base = reinterpret_cast<int32_t*>(ws + L.chunk_base);
  int32_t* local_rank = reinterpret_cast<int32_t*>(ws + L.local_rank);
  {
    TraceScope ts(TP_PERMUTE_HIST, st);
    permute_hist_kernel<<<(unsigned)L.n_chunks, kChunk, sizeof(uint32_t) * 2 * dm.E, st>>>(
        idx, dm.T, dm.E, dm.k, L.n_chunks, chunk_hist, local_rank, err);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    TraceScope ts(TP_PERMUTE_SCAN, st);
    permute_scan_kernel<<<1, 1024, 0, st>>>(chunk_hist, chunk_base, L.n_chunks, dm.E, dm.capacity,
                                            offsets, reinterpret_cast<int32_t*>(ws + L.offsets_full));
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const unsigned blocks = (unsigned)token_blocks(dm.T, 8, 1 << 20);
  TraceScope ts(TP_PERMUTE_SCATTER, st);
  if (dm.dtype == MOE_F32)
    permute_scatter_kernel<float><<<blocks, 256, 0, st>>>(
        (const float*)x, idx, topk_w, local_rank, chunk_base, offsets, dm.T, dm.d, dm.k, L.n_chunks,
        dm.capacity, (float*)x_perm, dest, row_src, w_perm);
  else
    permute_scatter_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(
        (const __nv_bfloat16*)x, idx, topk_w, local_rank, chunk_base, offsets, dm.T, dm.d, dm.k,
        L.n_chunks, dm.capacity, (__nv_bfloat16*)x_perm, dest, row_src, w_perm);
  return cudaGetLastError();
}

cudaError_t launch_pad_rows(void* buf, int width, int dtype, const int32_t* offsets_full, int E,
                            int C, int32_t* row_src, float* w_perm, cudaStream_t st) {
  const unsigned blocks = (unsigned)token_blocks((int64_t)E * C, 8, 1 << 16);
  TraceScope ts(TP_MISC, st);
  if (dtype == MOE_F32)
    pad_rows_kernel<float><<<blocks, 256, 0, st>>>((float*)buf, width, offsets_full, E, C, row_src, w_perm);
  else
    pad_rows_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>((__nv_bfloat16*)buf, width, offsets_full, E, C,
                                                           row_src, w_perm);
  return cudaGetLastError();
}

cudaError_t launch_permute_rows(const void* x, const int32_t* dest, const moe_dims& dm, void* x_perm,
                                cudaStream_t st) {
  const unsigned blocks = (unsigned)token_blocks(dm.T, 8, 1 << 20);
  TraceScope ts(TP_PERMUTE_ROWS, st);
  if (dm.dtype == MOE_F32)
    permute_rows_kernel<float><<<blocks, 256, 0, st>>>((const float*)x, dest, dm.T, dm.d, dm.k,
                                                       (float*)x_perm);
  else
    permute_rows_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(
        (const __nv_bfloat16*)x, dest, dm.T, dm.d, dm.k, (__nv_bfloat16*)x_perm);
  return cudaGetLastError();
}

namespace {
template <typename T>
void combine_dispatch(const T* y_perm, const int32_t* dest, const float* topk_w, const T* y_sh,
                      const int32_t* idx, const float* dl_tok, const float* w_rT, const moe_dims& dm,
                      T* y, unsigned blocks, cudaStream_t st) {
  if (w_rT != nullptr)
    combine_kernel<T, true, 0><<<blocks, 256, 0, st>>>(y_perm, dest, topk_w, y_sh, idx, dl_tok, w_rT, dm.T,
                                                       dm.d, dm.k, y);
  else if (dm.k <= 8)
    combine_kernel<T, false, 8><<<blocks, 256, 0, st>>>(y_perm, dest, topk_w, y_sh, idx, dl_tok, w_rT, dm.T,
                                                        dm.d, dm.k, y);
  else
    combine_kernel<T, false, 0><<<blocks, 256, 0, st>>>(y_perm, dest, topk_w, y_sh, idx, dl_tok, w_rT, dm.T,
                                                        dm.d, dm.k, y);
}
}  // namespace

cudaError_t launch_scatter_rows(const int32_t* dest, int64_t n, int32_t* scatter_rows, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  TraceScope ts(TP_MISC, st);
  scatter_rows_kernel<<<blocks, 256, 0, st>>>(dest, n, scatter_rows);
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* y_perm, const int32_t* dest, const float* topk_w,
                           const void* y_sh, const int32_t* idx, const float* dl_tok,
                           const float* w_rT, const moe_dims& dm, void* y, cudaStream_t st) {
  // one warp per row segment of 128 vectors (general path: per token), eight warps a block
  const int64_t nseg = (dm.d / 8 + 127) / 128;
  const unsigned blocks = (unsigned)token_blocks(dm.T * nseg, 8, 1 << 20);
  TraceScope ts(topk_w != nullptr ? TP_COMBINE : TP_COMBINE_BWD, st);
  if (dm.dtype == MOE_F32)
    combine_dispatch<float>((const float*)y_perm, dest, topk_w, (const float*)y_sh, idx, dl_tok, w_rT, dm,
                            (float*)y, blocks, st);
  else
    combine_dispatch<__nv_bfloat16>((const __nv_bfloat16*)y_perm, dest, topk_w, (const __nv_bfloat16*)y_sh,
                                    idx, dl_tok, w_rT, dm, (__nv_bfloat16*)y, blocks, st);
  return cudaGetLastError();
}

}  // namespace moe
