// Grouped-GEMM problem description shared by the fp32 SIMT kernel and the bf16 tcgen05
// kernel: the six matmul shapes of the expert FFN (forward, dX chain, dW products), the
// groups they run over (routed experts with ragged row counts from `offsets`, then the
// shared experts), and the device-built tile schedule.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace moe {

// The six expert matmuls. Per group g (routed expert e, or shared expert s):
//   FWD1  Z  = X  W13^T  [rows, 2f]  K = d        epilogue: h = silu(a)*b, store Z and h
//   FWD2  Y  = h  W2^T   [rows, d]   K = f        (shared: one group, K = S*f_s concatenated)
//   BWD2T D  = dY W2     [rows, f]   K = d        epilogue: dgate, dz, hw = w*h
//   BWD1T dX = dz W13    [rows, d]   K = 2f       (shared: one group, K = S*2f_s concatenated)
//   DW2   dW2  = dY^T hw [d, f]      K = rows
//   DW13  dW13 = dz^T X  [2f, d]     K = rows
//   ROUTER L  = x Wsplit^T [T, E]     K = 3d       (bf16 x times the three bf16 parts of the
//                                                   fp32 router weight, fp32 accumulation; the
//                                                   groups are kRouterSplit K slices whose fp32
//                                                   partials are summed afterwards in order)
enum Mode : int { FWD1 = 0, FWD2 = 1, BWD2T = 2, BWD1T = 3, DW2 = 4, DW13 = 5, ROUTER = 6 };

struct GroupedArgs {
  int64_t T, Tk;
  int d, E, k, f, S, f_s;
  const int32_t* offsets;  // [E+1], device
  // inputs
  const void *x_perm, *x, *w13, *w2, *ws13, *ws2;
  const void *h, *h_sh, *z, *z_sh, *dy_perm, *dy, *dz, *dz_sh, *hw, *hw_sh;
  const float* w_perm;
  // outputs
  void *z_out, *z_sh_out, *h_out, *h_sh_out, *y_perm, *y_sh;
  void *dz_out, *dz_sh_out, *hw_out, *hw_sh_out, *dx_perm, *dx_sh;
  void *dw13, *dw2, *dws13, *dws2;
  const void* w_split;      // [E][3d] bf16: hi | mid | lo parts of W_r^T (ROUTER)
  float* logits_out;        // [T][E] fp32 (ROUTER)
  // Fused rearrangement: when set (routed groups of FWD1, BWD2T, DW2, DW13, bf16), the
  // permuted token rows are not read from x_perm / dy_perm but gathered from x / dy, row r
  // of the permuted order being token gather_rows[r] (the permutation's row_src).
  const int32_t* gather_rows;
  // Fused un-rearrangement: when set (FWD2, routed groups, bf16), output row r of the
  // permuted order is written at row scatter_rows[r] (its token-major slot t*k + j).
  const int32_t* scatter_rows;
  // BWD1T: when w_rT is set, routed row q also gets dl_perm[q] * w_rT[e] (the router term
  // of the x-gradient, so that the un-rearrangement need not add it)
  const float* dl_perm;     // [Tk] score gradient of each permuted row
  const float* w_rT;        // [E][d] fp32 router weight, transposed
  float* dgate_part;        // [n_tiles_f][Tk] per-N-tile partial sums of dgate (BWD2T)
  int64_t dgate_stride;     // = Tk
  int* err;
};

constexpr int kRouterSplit = 8;

__host__ __device__ __forceinline__ int num_groups(int mode, int E, int S) {
  if (mode == ROUTER) return kRouterSplit;
  if (mode == FWD2 || mode == BWD1T) return E + (S > 0 ? 1 : 0);
  return E + S;
}

struct GroupGeom {
  int64_t row0;   // first row of the group in the permuted/shared buffers
  int64_t rows;   // rows of the group (token copies)
  int M, N, K;    // matmul shape of the group
  int k0;         // first K element of the group (ROUTER K slices), else 0
  int e;          // routed expert index, or -1
  int s;          // shared expert index (>= 0 for per-shared-expert groups), or -1
  bool shared;
};

// `offs` is the expert offsets array [E+1] (a shared-memory copy inside the kernels).
__device__ __forceinline__ GroupGeom group_geom(const GroupedArgs& a, int mode, int g, const int* offs) {
  GroupGeom G;
  if (mode == ROUTER) {
    G.shared = false;
    G.row0 = 0;
    G.rows = a.T;
    G.e = 0;
    G.s = -1;
    G.M = (int)a.T;
    G.N = a.E;
    const int nkb = 3 * a.d / 64, per = (nkb + kRouterSplit - 1) / kRouterSplit;
    const int kb0 = min(g * per, nkb), kb1 = min(kb0 + per, nkb);
    G.k0 = kb0 * 64;
    G.K = (kb1 - kb0) * 64;
    return G;
  }
  G.k0 = 0;
  G.shared = g >= a.E;
  if (!G.shared) {
    const int lo = offs[g], hi = offs[g + 1];
    G.row0 = lo;
    G.rows = hi - lo;
    G.e = g;
    G.s = -1;
  } else {
    G.row0 = 0;
    G.rows = a.T;
    G.e = -1;
    G.s = (mode == FWD2 || mode == BWD1T) ? -1 : g - a.E;
  }
  const int fw = G.shared ? a.f_s : a.f;
  const int rows32 = (int)G.rows;
  switch (mode) {
    case FWD1: G.M = rows32; G.N = fw; G.K = a.d; break;                 // N counts gate cols
    case FWD2: G.M = rows32; G.N = a.d; G.K = G.shared ? a.S * a.f_s : a.f; break;
    case BWD2T: G.M = rows32; G.N = fw; G.K = a.d; break;
    case BWD1T: G.M = rows32; G.N = a.d; G.K = G.shared ? a.S * 2 * a.f_s : 2 * a.f; break;
    case DW2: G.M = a.d; G.N = fw; G.K = rows32; break;
    default: G.M = 2 * fw; G.N = a.d; G.K = rows32; break;             // DW13
  }
  return G;
}

constexpr int kMaxGroups = 1024 + 8;   // routed experts (at most 1024) plus the shared ones

// Groups with more rows than this reuse each weight tile over three or more 128-row M tiles
// (or, in the dW products, reduce over more than four 64-deep K blocks): at the sustained
// tensor rate against the HBM bandwidth their tiles are bound by the tensor cores, while
// the tiles of smaller groups are bound by streaming the group's weight (or writing its
// gradient). The schedule mixes the two kinds so that both units stay busy.
constexpr int64_t kHeavyRows = 256;

// Tile schedule of one grouped launch, built in shared memory by every CTA. The groups
// are split into two streams, 0 (at most kHeavyRows rows, or every group where the launch
// is not mixed) and 1 (more); start[s][g] is
// the first tile of group g within stream s (groups of the other stream hold no tiles
// there), start[s][ng] the stream's tile count.
struct TileSched {
  int start[2][kMaxGroups + 1];
};

// Exclusive block-wide scan of one int per thread; returns the thread's prefix.
// Every thread of the block must call it.
__device__ __forceinline__ int block_exclusive_scan(int local, int* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int nw = (blockDim.x + 31) >> 5;
    int v = lane < nw ? warp_sums[lane] : 0;
    int vi = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, vi, o);
      if (lane >= o) vi += u;
    }
    if (lane < nw) warp_sums[lane] = vi - v;
  }
  __syncthreads();
  const int r = warp_sums[warp] + inc - local;
  __syncthreads();   // warp_sums is reused by the next scan
  return r;
}

// Copies the expert offsets into s_off[0..E] and builds the tile schedule (both shared
// memory). Every thread of the block must call it.
// bn_eff = output columns one tile covers along N (for FWD1 this is gate columns: a tile
// holds bn_eff gate and bn_eff up columns).
__device__ __forceinline__ void build_tile_starts(const GroupedArgs& a, int mode, int bm,
                                                  int bn_eff, TileSched& ts, int* warp_sums,
                                                  int* s_off) {
  if (mode != ROUTER)
    for (int i = threadIdx.x; i <= a.E; i += blockDim.x) s_off[i] = __ldg(a.offsets + i);
  __syncthreads();
  const int ng = num_groups(mode, a.E, a.S);
  // measured per product: mixing shortens the products whose B operand is the expert
  // weight read along the full hidden size or width (FWD1, FWD2, BWD1T) and lengthens
  // BWD2T and the dW products, which keep the plain group order
  const bool mixed = mode == FWD1 || mode == FWD2 || mode == BWD1T;
  const int nt = blockDim.x;
  const int per = (ng + nt - 1) / nt;
  const int g0 = threadIdx.x * per;
  int local[2] = {0, 0};
  for (int i = 0; i < per; ++i) {
    const int g = g0 + i;
    if (g < ng) {
      const GroupGeom G = group_geom(a, mode, g, s_off);
      const int t = ((G.M + bm - 1) / bm) * ((G.N + bn_eff - 1) / bn_eff);
      const int s = (mixed && G.rows > kHeavyRows) ? 1 : 0;
      ts.start[s][g] = t;      // temporarily the count
      ts.start[s ^ 1][g] = 0;
      local[s] += t;
    }
  }
  int run[2];
  run[0] = block_exclusive_scan(local[0], warp_sums);
  run[1] = block_exclusive_scan(local[1], warp_sums);
  for (int i = 0; i < per; ++i) {
    const int g = g0 + i;
    if (g < ng) {
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const int t = ts.start[s][g];
        ts.start[s][g] = run[s];
        run[s] += t;
      }
    }
  }
  if (threadIdx.x == nt - 1) {
    ts.start[0][ng] = run[0];
    ts.start[1][ng] = run[1];
  }
  __syncthreads();
}

struct TileCoord {
  GroupGeom G;
  int g, mi, ni;
};

// Walks one CTA's (or CTA pair's) tiles, first, first + stride, ..., through the schedule.
// The two streams are merged in proportion: of the first i tiles, floor(i * n0 / (n0 + n1))
// come from stream 0, so every stretch of the launch holds both kinds of tile. Within a
// stream the groups keep their order, and the tiles of a group are ordered N-tile major,
// M-tile minor (optionally in panels of M tiles, see coord), so that CTAs working at the
// same time on one expert share its weight tile through L2. Each step costs a few integer operations: the merge position is carried as a
// quotient and remainder, and the group of each stream only moves forward. (The issuing
// threads of the short-K dW tiles cannot afford a search or a 64-bit division per tile.)
struct TileCursor {
  const int* st0;    // stream 0's group starts (shared memory)
  const int* st1;
  int ng, n0, stride;
  long long tot;
  int tile;
  int q;             // floor(tile * n0 / tot)
  long long r;       // tile * n0 - q * tot
  int dq;            // floor(stride * n0 / tot)
  long long dr;
  int g0 = 0, g1 = 0;  // current group of each stream
  int cached = -1;     // group whose geometry is in G
  GroupGeom G;

  __device__ __forceinline__ TileCursor(const TileSched& t, int ng_, int first, int stride_)
      : st0(t.start[0]), st1(t.start[1]), ng(ng_), n0(t.start[0][ng_]), stride(stride_),
        tot((long long)t.start[0][ng_] + t.start[1][ng_]), tile(first) {
    const long long d = tot > 0 ? tot : 1;
    q = (int)((long long)first * n0 / d);
    r = (long long)first * n0 - (long long)q * d;
    dq = (int)((long long)stride * n0 / d);
    dr = (long long)stride * n0 - (long long)dq * d;
  }
  __device__ __forceinline__ bool valid() const { return tile < tot; }
  __device__ __forceinline__ void advance() {
    tile += stride;
    q += dq;
    r += dr;
    if (r >= tot) { r -= tot; ++q; }
  }
  // panel > 0: a group of more than `panel` M tiles and K of at least 4096 is walked in panels
  // of `panel` M tiles, N-tile major inside each panel (bn = output columns of a tile along N)
  __device__ __forceinline__ TileCoord coord(const GroupedArgs& a, int mode, int bm, const int* s_off,
                                             int panel = 0, int bn = 256) {
    // tile is stream 0's iff floor((tile + 1) n0 / tot) > floor(tile n0 / tot)
    const bool s0 = r + n0 >= tot;
    const int j = s0 ? q : tile - q;
    const int* st = s0 ? st0 : st1;
    int gg = s0 ? g0 : g1;
    while (gg + 1 < ng && st[gg + 1] <= j) ++gg;
    if (s0) g0 = gg; else g1 = gg;
    if (gg != cached) {
      G = group_geom(a, mode, gg, s_off);
      cached = gg;
    }
    TileCoord c;
    c.g = gg;
    c.G = G;
    const int local = j - st[gg];
    const int mt = (G.M + bm - 1) / bm;
    // (a K below 4096 keeps a 128-row block of A under 1 MB: it stays in L2 without panels)
    if (panel <= 0 || mt <= panel || G.K < 4096) {
      c.ni = local / mt;
      c.mi = local - c.ni * mt;
    } else {
      const int nt = (G.N + bn - 1) / bn;
      const int p = local / (panel * nt);
      const int r0 = local - p * panel * nt;
      const int pm = min(panel, mt - p * panel);   // M tiles of this panel
      c.ni = r0 / pm;
      c.mi = p * panel + (r0 - c.ni * pm);
    }
    return c;
  }
};

}  // namespace moe
