// fp32 grouped expert GEMMs on CUDA cores (true fp32 FMA, no TF32), for the fp32 layer.
// Same six matmuls, groups and device-built tile schedule as the tcgen05 bf16 kernel; one
// 32 x 64 output tile per iteration of a grid-stride loop, K in slices of 32 through shared
// memory, the mode's epilogue fused.
#include "grouped.cuh"
#include "internal.h"
#include "trace.h"

namespace moe {
namespace {

constexpr int SBM = 32, SBN = 64, SBK = 32, STHREADS = 256;

template <int MODE> struct SimtOps {
  static constexpr bool a_mn = (MODE == DW2 || MODE == DW13);
  static constexpr bool b_mn = (MODE == BWD2T || MODE == BWD1T || MODE == DW2 || MODE == DW13);

  static __device__ __forceinline__ float A(const GroupedArgs& a, const GroupGeom& G, int m, int k) {
    const float* p;
    int64_t off;
    switch (MODE) {
      case FWD1:
        p = (const float*)(G.shared ? a.x : a.x_perm);
        off = (G.row0 + m) * (int64_t)a.d + k;
        break;
      case FWD2:
        if (!G.shared) { p = (const float*)a.h; off = (G.row0 + m) * (int64_t)a.f + k; }
        else { const int s = k / a.f_s; p = (const float*)a.h_sh;
               off = ((int64_t)s * a.T + m) * a.f_s + (k - s * a.f_s); }
        break;
      case BWD2T:
        p = (const float*)(G.shared ? a.dy : a.dy_perm);
        off = (G.row0 + m) * (int64_t)a.d + k;
        break;
      case BWD1T:
        if (!G.shared) { p = (const float*)a.dz; off = (G.row0 + m) * (int64_t)(2 * a.f) + k; }
        else { const int s = k / (2 * a.f_s); p = (const float*)a.dz_sh;
               off = ((int64_t)s * a.T + m) * (2 * a.f_s) + (k - s * 2 * a.f_s); }
        break;
      case DW2:
        p = (const float*)(G.shared ? a.dy : a.dy_perm);
        off = (G.row0 + k) * (int64_t)a.d + m;
        break;
      default:  // DW13
        if (!G.shared) { p = (const float*)a.dz; off = (G.row0 + k) * (int64_t)(2 * a.f) + m; }
        else { p = (const float*)a.dz_sh; off = ((int64_t)G.s * a.T + k) * (2 * a.f_s) + m; }
        break;
    }
    return __ldg(p + off);
  }

  // n is the global output column (FWD1: a row of W13 in [0, 2fw)).
  static __device__ __forceinline__ float B(const GroupedArgs& a, const GroupGeom& G, int n, int k) {
    const float* p;
    int64_t off;
    switch (MODE) {
      case FWD1:
        if (!G.shared) { p = (const float*)a.w13; off = ((int64_t)G.e * 2 * a.f + n) * a.d + k; }
        else { p = (const float*)a.ws13; off = ((int64_t)G.s * 2 * a.f_s + n) * a.d + k; }
        break;
      case FWD2:
        if (!G.shared) { p = (const float*)a.w2; off = ((int64_t)G.e * a.d + n) * a.f + k; }
        else { const int s = k / a.f_s; p = (const float*)a.ws2;
               off = ((int64_t)s * a.d + n) * a.f_s + (k - s * a.f_s); }
        break;
      case BWD2T:
        if (!G.shared) { p = (const float*)a.w2; off = ((int64_t)G.e * a.d + k) * a.f + n; }
        else { p = (const float*)a.ws2; off = ((int64_t)G.s * a.d + k) * a.f_s + n; }
        break;
      case BWD1T:
        if (!G.shared) { p = (const float*)a.w13; off = ((int64_t)G.e * 2 * a.f + k) * a.d + n; }
        else { const int s = k / (2 * a.f_s); p = (const float*)a.ws13;
               off = ((int64_t)s * 2 * a.f_s + (k - s * 2 * a.f_s)) * a.d + n; }
        break;
      case DW2:
        if (!G.shared) { p = (const float*)a.hw; off = (G.row0 + k) * (int64_t)a.f + n; }
        else { p = (const float*)a.hw_sh; off = ((int64_t)G.s * a.T + k) * a.f_s + n; }
        break;
      default:  // DW13
        p = (const float*)(G.shared ? a.x : a.x_perm);
        off = (G.row0 + k) * (int64_t)a.d + n;
        break;
    }
    return __ldg(p + off);
  }
};

template <int MODE>
__global__ void __launch_bounds__(STHREADS) simt_grouped_kernel(const GroupedArgs a) {
  using Ops = SimtOps<MODE>;
  __shared__ float As[SBK][SBM + 1];
  __shared__ float Bs[SBK][SBN + 1];
  __shared__ float red[SBM][SBN + 1];
  __shared__ TileSched sched;
  __shared__ int warp_sums[32];
  __shared__ int s_off[1024 + 1];

  const int bn_eff = (MODE == FWD1) ? SBN / 2 : SBN;
  build_tile_starts(a, MODE, SBM, bn_eff, sched, warp_sums, s_off);
  const int ng = num_groups(MODE, a.E, a.S);
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;

  for (TileCursor cur(sched, ng, blockIdx.x, gridDim.x); cur.valid(); cur.advance()) {
    const TileCoord tc = cur.coord(a, MODE, SBM, s_off);
    const GroupGeom& G = tc.G;
    const int m0 = tc.mi * SBM, n0 = tc.ni * bn_eff;
    const int fw = G.shared ? a.f_s : a.f;
    float acc[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < G.K; k0 += SBK) {
      // A tile [SBM x SBK]
#pragma unroll
      for (int i = 0; i < (SBM * SBK) / STHREADS; ++i) {
        const int idx = tid + i * STHREADS;
        int m, k;
        if (Ops::a_mn) { k = idx / SBM; m = idx % SBM; } else { m = idx / SBK; k = idx % SBK; }
        const int gm = m0 + m, gk = k0 + k;
        As[k][m] = (gm < G.M && gk < G.K) ? Ops::A(a, G, gm, gk) : 0.f;
      }
      // B tile [SBN x SBK]
#pragma unroll
      for (int i = 0; i < (SBN * SBK) / STHREADS; ++i) {
        const int idx = tid + i * STHREADS;
        int n, k;
        if (Ops::b_mn) { k = idx / SBN; n = idx % SBN; } else { n = idx / SBK; k = idx % SBK; }
        const int gk = k0 + k;
        int gn;
        bool ok;
        if (MODE == FWD1) {
          const int j = n0 + (n & 31);
          ok = j < fw;
          gn = (n < 32) ? j : fw + j;
        } else {
          gn = n0 + n;
          ok = gn < G.N;
        }
        Bs[k][n] = (ok && gk < G.K) ? Ops::B(a, G, gn, gk) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < SBK; ++kk) {
        const float a0 = As[kk][ty * 2], a1 = As[kk][ty * 2 + 1];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float b = Bs[kk][tx + 16 * j];
          acc[0][j] = fmaf(a0, b, acc[0][j]);
          acc[1][j] = fmaf(a1, b, acc[1][j]);
        }
      }
      __syncthreads();
    }

    // ---------------------------------------------------------------- epilogue
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int m = m0 + ty * 2 + i;
      const bool row_ok = m < G.M;
      if (MODE == FWD1) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int jc = n0 + tx + 16 * j;
          if (row_ok && jc < fw) {
            const float ga = acc[i][j], up = acc[i][j + 2];
            const float hv = silu_f(ga) * up;
            float *zr, *hr;
            if (!G.shared) {
              zr = (float*)a.z_out + (G.row0 + m) * (int64_t)(2 * a.f);
              hr = (float*)a.h_out + (G.row0 + m) * (int64_t)a.f;
            } else {
              zr = (float*)a.z_sh_out + ((int64_t)G.s * a.T + m) * (2 * a.f_s);
              hr = (float*)a.h_sh_out + ((int64_t)G.s * a.T + m) * a.f_s;
            }
            zr[jc] = ga;
            zr[fw + jc] = up;
            hr[jc] = hv;
          }
        }
      } else if (MODE == BWD2T) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = tx + 16 * j;
          const int n = n0 + c;
          float prod = 0.f;
          if (row_ok && n < fw) {
            const float D = acc[i][j];
            const float* zr;
            float *dzr, *hwr;
            float w = 1.f;
            if (!G.shared) {
              zr = (const float*)a.z + (G.row0 + m) * (int64_t)(2 * a.f);
              dzr = (float*)a.dz_out + (G.row0 + m) * (int64_t)(2 * a.f);
              hwr = (float*)a.hw_out + (G.row0 + m) * (int64_t)a.f;
              w = __ldg(a.w_perm + G.row0 + m);
            } else {
              zr = (const float*)a.z_sh + ((int64_t)G.s * a.T + m) * (2 * a.f_s);
              dzr = (float*)a.dz_sh_out + ((int64_t)G.s * a.T + m) * (2 * a.f_s);
              hwr = (float*)a.hw_sh_out + ((int64_t)G.s * a.T + m) * a.f_s;
            }
            const float av = zr[n], bv = zr[fw + n];
            const float sg = 1.f / (1.f + expf(-av));
            const float sl = av * sg;
            const float hv = sl * bv;
            prod = D * hv;
            dzr[n] = w * D * bv * (sg * (1.f + av * (1.f - sg)));
            dzr[fw + n] = w * D * sl;
            hwr[n] = w * hv;
          }
          red[ty * 2 + i][c] = prod;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int n = n0 + tx + 16 * j;
          if (!(row_ok && n < G.N)) continue;
          const float v = acc[i][j];
          float* out;
          switch (MODE) {
            case FWD2:
              out = G.shared ? (float*)a.y_sh + (int64_t)m * a.d
                             : (float*)a.y_perm + (G.row0 + m) * (int64_t)a.d;
              break;
            case BWD1T:
              out = G.shared ? (float*)a.dx_sh + (int64_t)m * a.d
                             : (float*)a.dx_perm + (G.row0 + m) * (int64_t)a.d;
              break;
            case DW2:
              out = G.shared ? (float*)a.dws2 + ((int64_t)G.s * a.d + m) * a.f_s
                             : (float*)a.dw2 + ((int64_t)G.e * a.d + m) * a.f;
              break;
            default:  // DW13
              out = G.shared ? (float*)a.dws13 + ((int64_t)G.s * 2 * a.f_s + m) * a.d
                             : (float*)a.dw13 + ((int64_t)G.e * 2 * a.f + m) * a.d;
              break;
          }
          out[n] = v;
        }
      }
    }
    if (MODE == BWD2T) {
      __syncthreads();
      if (!G.shared && tid < SBM && m0 + tid < G.M) {
        float s = 0.f;
        for (int c = 0; c < SBN; ++c) s += red[tid][c];   // fixed order: deterministic
        a.dgate_part[(int64_t)tc.ni * a.dgate_stride + G.row0 + m0 + tid] = s;
      }
      __syncthreads();
    }
  }
}

}  // namespace

int simt_dgate_tiles(int f) { return (f + SBN - 1) / SBN; }

cudaError_t launch_simt_grouped(int mode, const GroupedArgs& a, int num_sms, cudaStream_t st) {
  const dim3 grid(2 * num_sms), block(STHREADS);
  TraceScope ts(mode == FWD1 ? TP_GEMM_FWD1 : mode == FWD2 ? TP_GEMM_FWD2 : mode == BWD2T ? TP_GEMM_BWD2T :
                mode == BWD1T ? TP_GEMM_BWD1T : mode == DW2 ? TP_GEMM_DW2 : TP_GEMM_DW13, st);
  switch (mode) {
    case FWD1: simt_grouped_kernel<FWD1><<<grid, block, 0, st>>>(a); break;
    case FWD2: simt_grouped_kernel<FWD2><<<grid, block, 0, st>>>(a); break;
    case BWD2T: simt_grouped_kernel<BWD2T><<<grid, block, 0, st>>>(a); break;
    case BWD1T: simt_grouped_kernel<BWD1T><<<grid, block, 0, st>>>(a); break;
    case DW2: simt_grouped_kernel<DW2><<<grid, block, 0, st>>>(a); break;
    default: simt_grouped_kernel<DW13><<<grid, block, 0, st>>>(a); break;
  }
  return cudaGetLastError();
}

}  // namespace moe
