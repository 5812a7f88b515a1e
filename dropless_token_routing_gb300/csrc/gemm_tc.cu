// bf16 grouped expert GEMMs on the 5th-generation tensor cores (sm_103a).
//
// One persistent, warp-specialised kernel per matmul kind (the forward, dX-chain and router
// products of grouped.cuh; the dW products run on CTA pairs, gemm_tc_pair.cu):
//   warp 0      TMA producer: 4-stage ring of 128x64 A and 256x64 B tiles (128-byte swizzle)
//   warp 1      TMEM owner and single-thread tcgen05.mma issuer (M=128, N=256, K=16 steps,
//               fp32 accumulators in TMEM, two accumulator buffers of 256 columns)
//   warps 2..5  epilogue: tcgen05.ld -> fused math of the mode -> bf16 -> global memory
// The tile schedule (groups = routed experts with ragged row counts, then shared experts)
// is rebuilt by every CTA from the device-resident expert offsets, so nothing waits on the
// host. Tiles of one expert run N-tile major / M-tile minor (a heavy expert in panels of 16
// M tiles) so concurrently running CTAs share the expert's weight tile through L2.
// Ragged edges: M tails read neighbouring rows (or the TMA zero fill) and are not stored; a
// group's last M tile with at most 64 rows runs as an M=64 MMA on a 64-row A box.
// Every mbarrier wait is bounded (1 s); on expiry the CTA records MOE_ERR_DEVICE_TIMEOUT,
// drains its TMA loads and MMAs, frees its TMEM and exits.
#include <cuda.h>

#include <mutex>

#include "grouped.cuh"
#include "tc_common.cuh"
#include "internal.h"
#include "trace.h"

namespace moe {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;          // 16 KB
constexpr int B_BYTES = BN * BK * 2;          // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_STAGE_BYTES = 5120;        // per epilogue warp, a multiple of 1024
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 4 * EPI_STAGE_BYTES + 1024;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr int SLAB = 64 * 128;                // one 64-element-wide, 64-row swizzled slab
// A group of more than kPanelM M tiles is walked in panels of kPanelM M tiles (N-tile major
// inside a panel), so that a heavy expert's token rows are re-read from L2 by its N tiles
// rather than from HBM; a panel's weight tile is read once per panel.
constexpr int kPanelM = 16;

using namespace tc;

struct TcParams {
  CUtensorMap a0, a1, b0, b1;
  CUtensorMap h0, h1;   // A (routed / shared) in boxes of 64 rows, for the short last M tiles
  GroupedArgs g;
};

// A group's last M tile with at most 64 rows is multiplied as an M = 64 MMA on a 64-row A
// box (rows 0..63 of the tile sit in TMEM lanes 32 q + 0..15, q = row / 16), so that the
// ragged end of a segment does not pay for 128 rows. Gathered A tiles keep M = 128.
template <int MODE>
__device__ __forceinline__ bool short_tile(const GroupedArgs& a, const TileCoord& tc) {
  if (MODE == ROUTER) return false;
  if ((MODE == FWD1 || MODE == BWD2T) && a.gather_rows != nullptr && !tc.G.shared) return false;
  return tc.G.M - tc.mi * BM <= BM / 2;
}

// ------------------------------------------------------------------ tcgen05 (one CTA)
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t ad, uint64_t bd, uint32_t idesc,
                                     uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(ad), "l"(bd), "r"(idesc), "r"(accum)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}


__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16* src, float* v) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = __ldg(s4 + q);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
      v[8 * q + 2 * i] = t.x;
      v[8 * q + 2 * i + 1] = t.y;
    }
  }
}

// Fused rearrangement: the 128 x 64 A tile of K block kb, gathered from the token rows `tok`
// (lane L holds the tokens of tile rows 4i + L/8, i = 0..31) with 16-byte cp.async in the
// TMA's 128-byte swizzled layout (16-byte chunk c of row r at chunk c ^ (r & 7)). Each
// instruction of the warp copies four whole 128-byte row segments. The copies complete on
// `bar` (cp.async.mbarrier.arrive); the LSU path is not bound by the TMA unit's rate per
// instruction, which 512-byte tile::gather4 copies are (about 5 B/cycle per SM).
__device__ __forceinline__ void gather_a_tile(uint32_t a_s, const __nv_bfloat16* src, int d, int kb,
                                              const int (&tok)[32], int lane, uint32_t bar) {
  const int c = lane & 7;
  const __nv_bfloat16* s0 = src + kb * BK + 8 * c;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int r = 4 * i + (lane >> 3);
    cp_async16(a_s + r * 128 + ((c ^ (r & 7)) << 4), s0 + (int64_t)tok[i] * d);
  }
  cp_async_arrive(bar);
}

template <int MODE> struct ModeTraits {
  static constexpr bool b_mn = (MODE == BWD2T || MODE == BWD1T);
  static constexpr int bn_eff = (MODE == FWD1) ? BN / 2 : BN;
};

// The MMAs of one tile's K blocks (instruction descriptor IDESC), each after its stage has
// landed; the stage is released by a commit once they have read it. Returns false when a wait
// ran out.
template <int MODE, uint32_t IDESC>
__device__ __forceinline__ bool mma_kloop(uint32_t smem_base, uint32_t d_tmem, int nkb, int& stage,
                                          uint32_t& phase, uint64_t* full_bar, uint64_t* empty_bar,
                                          volatile int* abort_flag, int* err, bool gathered) {
  for (int kb = 0; kb < nkb; ++kb) {
    if (!mbar_wait_bounded(smem_u32(&full_bar[stage]), phase, abort_flag, err, kWaitLimitNs)) return false;
    if (gathered) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_after();
    const uint32_t a_s = smem_base + stage * STAGE_BYTES, b_s = a_s + A_BYTES;
#pragma unroll
    for (int kk = 0; kk < BK / 16; ++kk) {
      const uint64_t ad = sdesc(a_s + kk * 32, 16, 1024);
      const uint64_t bd = ModeTraits<MODE>::b_mn ? sdesc(b_s + kk * 2048, SLAB, 1024) : sdesc(b_s + kk * 32, 16, 1024);
      umma(d_tmem, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
    }
    umma_commit(smem_u32(&empty_bar[stage]));
    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
  }
  return true;
}

// ------------------------------------------------------------------ producer: TMA issue
// `gather`: the routed A tile is gathered row by row by the whole producer warp instead
// (gather_a_tile), so it is skipped here.
template <int MODE>
__device__ __forceinline__ void issue_tile_loads(const TcParams& p, const TileCoord& tc, int kb,
                                                 uint32_t a_s, uint32_t b_s, uint32_t bar, bool gather) {
  const GroupedArgs& a = p.g;
  const GroupGeom& G = tc.G;
  const int m0 = tc.mi * BM;
  const int k0 = kb * BK;
  const int row0 = (int)G.row0;
  const int T = (int)a.T;
  const bool sh_t = short_tile<MODE>(a, tc);
  const CUtensorMap* am0 = sh_t ? &p.h0 : &p.a0;
  const CUtensorMap* am1 = sh_t ? &p.h1 : &p.a1;
  if (MODE == ROUTER) {
    const int kk = G.k0 + k0;                 // K slice of this group
    tma2d(a_s, &p.a0, bar, kk % a.d, m0);     // x, read once per weight part
    tma2d(b_s, &p.b0, bar, kk, tc.ni * BN);
  } else if (MODE == FWD1) {
    const int j0 = tc.ni * (BN / 2);
    // the weight rows first: for a light expert they stream from HBM and land last
    if (!G.shared) {
      tma3d(b_s, &p.b0, bar, k0, j0, G.e);
      tma3d(b_s + B_BYTES / 2, &p.b0, bar, k0, a.f + j0, G.e);
      if (!gather) tma2d(a_s, am0, bar, k0, row0 + m0);
    } else {
      tma3d(b_s, &p.b1, bar, k0, j0, G.s);
      tma3d(b_s + B_BYTES / 2, &p.b1, bar, k0, a.f_s + j0, G.s);
      tma2d(a_s, am1, bar, k0, m0);
    }
  } else if (MODE == FWD2) {
    const int n0 = tc.ni * BN;
    if (!G.shared) {
      tma2d(a_s, am0, bar, k0, row0 + m0);
      // an expert of one M tile reads its W2 rows once: they leave L2 first (measured 2 %
      // faster here; the same policy on the MN-major weight slabs of BWD2T / BWD1T is slower)
      if (G.M <= BM) tma3d_hint(b_s, &p.b0, bar, k0, n0, G.e, l2_evict_first());
      else tma3d(b_s, &p.b0, bar, k0, n0, G.e);
    } else {
      const int kpb = a.f_s / BK, s = kb / kpb, kl = (kb - s * kpb) * BK;
      tma2d(a_s, am1, bar, kl, s * T + m0);
      tma3d(b_s, &p.b1, bar, kl, n0, s);
    }
  } else if (MODE == BWD2T) {
    // the weight operand's four 64-column slabs in one 4-D copy (map4d_slabs)
    const int n0 = tc.ni * BN;
    if (!G.shared) {
      if (!gather) tma2d(a_s, am0, bar, k0, row0 + m0);
      tma4d(b_s, &p.b0, bar, 0, k0, n0 / 64, G.e);
    } else {
      tma2d(a_s, am1, bar, k0, m0);
      tma4d(b_s, &p.b1, bar, 0, k0, n0 / 64, G.s);
    }
  } else if (MODE == BWD1T) {
    const int n0 = tc.ni * BN;
    if (!G.shared) {
      tma2d(a_s, am0, bar, k0, row0 + m0);
      tma4d(b_s, &p.b0, bar, 0, k0, n0 / 64, G.e);
    } else {
      const int kpb = 2 * a.f_s / BK, s = kb / kpb, kl = (kb - s * kpb) * BK;
      tma2d(a_s, am1, bar, kl, s * T + m0);
      tma4d(b_s, &p.b1, bar, 0, kl, n0 / 64, s);
    }
  }
}

// ------------------------------------------------------------------ epilogues
// Each epilogue warp owns 32 tile rows (its TMEM lane quarter). Results leave in chunks of
// 128 bytes per row (64 bf16 or 32 fp32 columns): every lane packs its row's chunk into the
// warp's staging buffer, then the warp re-reads it so that each store instruction writes
// four whole 128-byte lines. `dst` is this lane's row pointer at the chunk, or null when the
// row is not stored (ragged M tail).
constexpr int STAGE_PITCH = 144;                 // 128 B + 16 B pad: conflict-free both ways
static_assert(32 * STAGE_PITCH <= EPI_STAGE_BYTES, "staging buffer too small");

__device__ __forceinline__ void warp_store_chunk(uint8_t* stage, int lane, const uint4 (&v)[8],
                                                 void* dst) {
  uint4* srow = reinterpret_cast<uint4*>(stage + lane * STAGE_PITCH);
#pragma unroll
  for (int q = 0; q < 8; ++q) srow[q] = v[q];
  __syncwarp();
  const unsigned long long mine = reinterpret_cast<unsigned long long>(dst);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = i * 4 + (lane >> 3), q = lane & 7;
    const unsigned long long ptr = __shfl_sync(0xffffffffu, mine, row);
    const uint4 val = *reinterpret_cast<const uint4*>(stage + row * STAGE_PITCH + q * 16);
    if (ptr != 0ull) reinterpret_cast<uint4*>(ptr)[q] = val;
  }
  __syncwarp();
}


// 64 fp32 values -> 64 bf16 (RNE) packed in 8 x 16 bytes.
__device__ __forceinline__ void pack64(const float* f, uint4 (&v)[8]) {
#pragma unroll
  for (int q = 0; q < 8; ++q)
    v[q] = make_uint4(pack_bf16x2(f[8 * q], f[8 * q + 1]), pack_bf16x2(f[8 * q + 2], f[8 * q + 3]),
                      pack_bf16x2(f[8 * q + 4], f[8 * q + 5]), pack_bf16x2(f[8 * q + 6], f[8 * q + 7]));
}

// 64 consecutive fp32 accumulator columns of this lane's row.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* f) {
  uint32_t a[32], b[32];
  tmem_ld32(taddr, a);
  tmem_ld32(taddr + 32, b);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    f[i] = __uint_as_float(a[i]);
    f[32 + i] = __uint_as_float(b[i]);
  }
}

template <typename T>
__device__ __forceinline__ T* row_or_null(bool ok, T* p) { return ok ? p : nullptr; }

// Thread owns tile row r (TMEM lane); `acc` is the TMEM address of its lane, column 0.
template <int MODE>
__device__ __forceinline__ void epilogue_tile(const TcParams& p, const TileCoord& tc, int r,
                                              uint32_t acc, uint8_t* stage, int lane) {
  const GroupedArgs& a = p.g;
  const GroupGeom& G = tc.G;
  const int m0 = tc.mi * BM;
  const int m = m0 + r;
  const bool row_ok = m < G.M;
  const int fw = G.shared ? a.f_s : a.f;
  uint4 pk[8];

  if (MODE == ROUTER) {
    // fp32 partial scores of K slice g, rows padded to a multiple of 32 experts
    const int n0 = tc.ni * BN;
    const int epad = (a.E + 31) & ~31;
    float* out = a.logits_out + ((int64_t)tc.g * a.T + m) * epad;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      if (n0 + c >= epad) break;
      uint32_t u[32];
      if (G.K > 0) {
        tmem_ld32(acc + c, u);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) u[i] = 0u;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) pk[q] = make_uint4(u[4 * q], u[4 * q + 1], u[4 * q + 2], u[4 * q + 3]);
      warp_store_chunk(stage, lane, pk, row_or_null(row_ok, out + n0 + c));
    }
  } else if (MODE == FWD1) {
    const int j0 = tc.ni * (BN / 2);
    __nv_bfloat16 *zr, *hr;
    if (!G.shared) {
      zr = (__nv_bfloat16*)a.z_out + (G.row0 + m) * (int64_t)(2 * a.f);
      hr = (__nv_bfloat16*)a.h_out + (G.row0 + m) * (int64_t)a.f;
    } else {
      zr = (__nv_bfloat16*)a.z_sh_out + ((int64_t)G.s * a.T + m) * (2 * a.f_s);
      hr = (__nv_bfloat16*)a.h_sh_out + ((int64_t)G.s * a.T + m) * a.f_s;
    }
#pragma unroll 1
    for (int c = 0; c < BN / 2; c += 64) {
      if (j0 + c >= fw) break;  // uniform across the warp
      float g[64], u[64];
      tmem_ld64(acc + c, g);
      tmem_ld64(acc + BN / 2 + c, u);
      pack64(g, pk);
      warp_store_chunk(stage, lane, pk, row_or_null(row_ok, zr + j0 + c));
      pack64(u, pk);
      warp_store_chunk(stage, lane, pk, row_or_null(row_ok, zr + fw + j0 + c));
#pragma unroll
      for (int i = 0; i < 64; ++i) g[i] = silu_f(g[i]) * u[i];
      pack64(g, pk);
      warp_store_chunk(stage, lane, pk, row_or_null(row_ok, hr + j0 + c));
    }
  } else if (MODE == BWD2T) {
    const int n0 = tc.ni * BN;
    const __nv_bfloat16* zr;
    __nv_bfloat16 *dzr, *hwr;
    float w = 1.f;
    if (!G.shared) {
      zr = (const __nv_bfloat16*)a.z + (G.row0 + m) * (int64_t)(2 * a.f);
      dzr = (__nv_bfloat16*)a.dz_out + (G.row0 + m) * (int64_t)(2 * a.f);
      hwr = (__nv_bfloat16*)a.hw_out + (G.row0 + m) * (int64_t)a.f;
      if (row_ok) w = __ldg(a.w_perm + G.row0 + m);
    } else {
      zr = (const __nv_bfloat16*)a.z_sh + ((int64_t)G.s * a.T + m) * (2 * a.f_s);
      dzr = (__nv_bfloat16*)a.dz_sh_out + ((int64_t)G.s * a.T + m) * (2 * a.f_s);
      hwr = (__nv_bfloat16*)a.hw_sh_out + ((int64_t)G.s * a.T + m) * a.f_s;
    }
    float dg = 0.f;
#pragma unroll 1
    for (int c = 0; c < BN; c += 64) {
      if (n0 + c >= fw) break;
      uint4 pa[8], pb[8], ph[8];   // d(gate pre-act), d(up pre-act), gate-weighted h
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int cc = c + 32 * half;
        uint32_t u[32];
        float za[32], zb[32];
        tmem_ld32(acc + cc, u);
        tmem_ld_wait();
        if (row_ok) {
          load_bf16x32(zr + n0 + cc, za);
          load_bf16x32(zr + fw + n0 + cc, zb);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) za[i] = zb[i] = 0.f;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float va[8], vb[8], vh[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float D = __uint_as_float(u[8 * q + i]);
            const float av = za[8 * q + i], bv = zb[8 * q + i];
            // hardware exponential and reciprocal: a few ulp in fp32, far inside the bf16
            // rounding of the outputs, and a third of the instructions of the exact forms
            const float sg = __fdividef(1.f, 1.f + __expf(-av));
            const float sl = av * sg;
            const float hv = sl * bv;
            dg = fmaf(D, hv, dg);
            va[i] = w * D * bv * (sg * (1.f + av * (1.f - sg)));
            vb[i] = w * D * sl;
            vh[i] = w * hv;
          }
          pa[4 * half + q] = make_uint4(pack_bf16x2(va[0], va[1]), pack_bf16x2(va[2], va[3]),
                                        pack_bf16x2(va[4], va[5]), pack_bf16x2(va[6], va[7]));
          pb[4 * half + q] = make_uint4(pack_bf16x2(vb[0], vb[1]), pack_bf16x2(vb[2], vb[3]),
                                        pack_bf16x2(vb[4], vb[5]), pack_bf16x2(vb[6], vb[7]));
          ph[4 * half + q] = make_uint4(pack_bf16x2(vh[0], vh[1]), pack_bf16x2(vh[2], vh[3]),
                                        pack_bf16x2(vh[4], vh[5]), pack_bf16x2(vh[6], vh[7]));
        }
      }
      warp_store_chunk(stage, lane, pa, row_or_null(row_ok, dzr + n0 + c));
      warp_store_chunk(stage, lane, pb, row_or_null(row_ok, dzr + fw + n0 + c));
      warp_store_chunk(stage, lane, ph, row_or_null(row_ok, hwr + n0 + c));
    }
    if (!G.shared && row_ok) a.dgate_part[(int64_t)tc.ni * a.dgate_stride + G.row0 + m] = dg;
  } else {  // FWD2 / BWD1T: rows of ragged expert segments, stored row by row
    const int n0 = tc.ni * BN;
    __nv_bfloat16* out;
    if (MODE == FWD2) {
      // the fused un-rearrangement writes a routed row at its token-major slot
      const int64_t orow = G.row0 + m;
      const int64_t srow = a.scatter_rows != nullptr && row_ok ? __ldg(a.scatter_rows + orow) : orow;
      out = G.shared ? (__nv_bfloat16*)a.y_sh + (int64_t)m * a.d : (__nv_bfloat16*)a.y_perm + srow * a.d;
    }
    else
      out = G.shared ? (__nv_bfloat16*)a.dx_sh + (int64_t)m * a.d
                     : (__nv_bfloat16*)a.dx_perm + (G.row0 + m) * (int64_t)a.d;
    // router term of the x-gradient folded into the routed dx rows: row q of expert e gets
    // dl_q * W_r^T[e] (the segment shares one router row, read from L1)
    const bool router = MODE == BWD1T && a.w_rT != nullptr && !G.shared;
    const float dl = router && row_ok ? __ldg(a.dl_perm + G.row0 + m) : 0.f;
    const float* wr = router ? a.w_rT + (int64_t)G.e * a.d + n0 : nullptr;
#pragma unroll 1
    for (int c = 0; c < BN; c += 64) {
      if (n0 + c >= G.N) break;
      float v[64];
      tmem_ld64(acc + c, v);
      if (router) {
        const float4* w4 = reinterpret_cast<const float4*>(wr + c);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float4 t = __ldg(w4 + i);
          v[4 * i] = fmaf(dl, t.x, v[4 * i]);
          v[4 * i + 1] = fmaf(dl, t.y, v[4 * i + 1]);
          v[4 * i + 2] = fmaf(dl, t.z, v[4 * i + 2]);
          v[4 * i + 3] = fmaf(dl, t.w, v[4 * i + 3]);
        }
      }
      pack64(v, pk);
      warp_store_chunk(stage, lane, pk, row_or_null(row_ok, out + n0 + c));
    }
  }
}

// ------------------------------------------------------------------ the kernel
template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1) tc_grouped_kernel(const __grid_constant__ TcParams p) {
  using TR = ModeTraits<MODE>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[2], tempty_bar[2], final_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;
  __shared__ TileSched sched;
  __shared__ int warp_sums[32];
  __shared__ int s_off[1024 + 1];

  const GroupedArgs& a = p.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t smem_base = smem_u32(smem);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull_bar[b]), 1);
      mbar_init(smem_u32(&tempty_bar[b]), 4);
    }
    mbar_init(smem_u32(&final_bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_base_sh)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  build_tile_starts(a, MODE, BM, TR::bn_eff, sched, warp_sums, s_off);  // ends with __syncthreads
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;
  const int ng = num_groups(MODE, a.E, a.S);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t pending = 0;    // stages whose latest load may still be in flight
    uint32_t pend_par = 0;   // parity of the phase that load completes, per stage
    bool ok = true;
    for (TileCursor cur(sched, ng, blockIdx.x, gridDim.x); cur.valid() && ok; cur.advance()) {
      const TileCoord tc = cur.coord(a, MODE, BM, s_off, MODE == ROUTER ? 0 : kPanelM, TR::bn_eff);
      const int nkb = (tc.G.K + BK - 1) / BK;
      // fused rearrangement: lane L gathers chunk L % 8 of tile rows 4i + L / 8 (rows past the
      // segment repeat its first row; they are computed but never stored)
      const bool gather = (MODE == FWD1 || MODE == BWD2T) && a.gather_rows != nullptr && !tc.G.shared;
      int tok[32];
      if (gather) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int m = tc.mi * BM + 4 * i + (lane >> 3);
          tok[i] = __ldg(a.gather_rows + tc.G.row0 + (m < tc.G.M ? m : 0));
        }
      }
      for (int kb = 0; kb < nkb; ++kb) {
        const bool got = mbar_wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1u, &abort_flag,
                                           a.err, kWaitLimitNs);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        const uint32_t a_s = smem_base + stage * STAGE_BYTES, b_s = a_s + A_BYTES;
        const uint32_t bar = smem_u32(&full_bar[stage]);
        if (gather) {
          // the weight tile's TMA first; lane 0 arrives only after every lane's copies are
          // counted by the barrier
          if (lane == 0) {
            mbar_expect_tx(bar, B_BYTES);
            issue_tile_loads<MODE>(p, tc, kb, a_s, b_s, bar, true);
          }
          gather_a_tile(a_s, (const __nv_bfloat16*)(MODE == FWD1 ? a.x : a.dy), a.d, kb, tok, lane, bar);
          __syncwarp();
          if (lane == 0) mbar_arrive(bar);
        } else if (lane == 0) {
          mbar_arrive_expect_tx(bar, short_tile<MODE>(a, tc) ? STAGE_BYTES - A_BYTES / 2 : STAGE_BYTES);
          issue_tile_loads<MODE>(p, tc, kb, a_s, b_s, bar, false);
        }
        pending |= 1u << stage;
        pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    // drain: no TMA load may still be writing shared memory when the CTA exits
    for (int s = 0; s < STAGES; ++s)
      if ((pending >> s) & 1u)
        mbar_wait_bounded(smem_u32(&full_bar[s]), (pend_par >> s) & 1u, nullptr, a.err, kWaitLimitNs);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (one thread)
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(BM, BN, false, TR::b_mn);
      int stage = 0;
      uint32_t phase = 0;
      bool issued = false, ok = true;
      int it = 0;
      for (TileCursor cur(sched, ng, blockIdx.x, gridDim.x); cur.valid() && ok; cur.advance(), ++it) {
        const TileCoord tc = cur.coord(a, MODE, BM, s_off, MODE == ROUTER ? 0 : kPanelM, TR::bn_eff);
        const int nkb = (tc.G.K + BK - 1) / BK;
        const int b = it & 1;
        // a gathered A tile was written through the generic proxy (cp.async): order it before
        // the tensor core's reads
        const bool gathered = (MODE == FWD1 || MODE == BWD2T) && a.gather_rows != nullptr && !tc.G.shared;
        if (!mbar_wait_bounded(smem_u32(&tempty_bar[b]), ((it >> 1) & 1) ^ 1, &abort_flag, a.err,
                               kWaitLimitNs)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(b * BN);
        if (nkb > 0) issued = true;
        ok = short_tile<MODE>(a, tc)
                 ? mma_kloop<MODE, idesc_bf16(BM / 2, BN, false, TR::b_mn)>(smem_base, d_tmem, nkb, stage, phase,
                                                                            full_bar, empty_bar, &abort_flag, a.err,
                                                                            gathered)
                 : mma_kloop<MODE, idesc>(smem_base, d_tmem, nkb, stage, phase, full_bar, empty_bar, &abort_flag,
                                          a.err, gathered);
        if (!ok) break;
        if (nkb > 0) umma_commit(smem_u32(&tfull_bar[b]));
        else mbar_arrive(smem_u32(&tfull_bar[b]));
      }
      if (issued) {  // all MMAs retired before TMEM is released
        umma_commit(smem_u32(&final_bar));
        mbar_wait_bounded(smem_u32(&final_bar), 0, nullptr, a.err, kWaitLimitNs);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue warps 2..5
    const int lg = warp & 3;              // TMEM lane quarter this warp may access
    const int r = lg * 32 + lane;         // tile row
    uint8_t* stage = smem + STAGES * STAGE_BYTES + (warp - 2) * EPI_STAGE_BYTES;
    int it = 0;
    for (TileCursor cur(sched, ng, blockIdx.x, gridDim.x); cur.valid(); cur.advance(), ++it) {
      const TileCoord tc = cur.coord(a, MODE, BM, s_off, MODE == ROUTER ? 0 : kPanelM, TR::bn_eff);
      const int b = it & 1;
      const bool got = mbar_wait_bounded(smem_u32(&tfull_bar[b]), (it >> 1) & 1, &abort_flag,
                                         a.err, kWaitLimitNs);
      if (!__all_sync(0xffffffffu, got)) break;   // warp-uniform: tcgen05.ld is .sync.aligned
      tc_fence_after();
      const uint32_t acc = tmem_base + ((uint32_t)(lg * 32) << 16) + (uint32_t)(b * BN);
      // a short tile's rows 16 lg .. 16 lg + 15 are in lanes 0..15 of this warp's quarter; the
      // other lanes get a row past the tile's end (not stored)
      const int rr = short_tile<MODE>(a, tc) ? (lane < 16 ? lg * 16 + lane : BM / 2 + lane) : r;
      epilogue_tile<MODE>(p, tc, rr, acc, stage, lane);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[b]));
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host: tensor maps

constexpr int trace_phase_of(int mode) {
  return mode == FWD1 ? TP_GEMM_FWD1 : mode == FWD2 ? TP_GEMM_FWD2 : mode == BWD2T ? TP_GEMM_BWD2T
       : mode == BWD1T ? TP_GEMM_BWD1T
       : TP_ROUTER_GEMM;
}

template <int MODE>
int launch_mode(TcParams& p, int num_sms, cudaStream_t st) {
  // the shared-memory attribute is set once per device (under a lock: callers may be several
  // host threads, each with its own device)
  static std::mutex mu;
  static bool attr_set[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!attr_set[dev]) {
      if (cudaFuncSetAttribute(tc_grouped_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               SMEM_BYTES) != cudaSuccess)
        return MOE_ERR_CUDA;
      attr_set[dev] = true;
    }
  }
  TraceScope ts(trace_phase_of(MODE), st);
  tc_grouped_kernel<MODE><<<num_sms, NUM_THREADS, SMEM_BYTES, st>>>(p);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

}  // namespace

int tc_dgate_tiles(int f) { return (f + BN - 1) / BN; }

int launch_tc_grouped(int mode, const GroupedArgs& g, int num_sms, cudaStream_t st) {
  if (mode == DW2 || mode == DW13) return launch_tc_pair_dw(mode, g, num_sms, st);
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.g = g;
  const uint64_t Tk = (uint64_t)g.Tk, T = (uint64_t)g.T, ST = (uint64_t)g.S * g.T;
  const uint64_t d = g.d, f = g.f, fs = g.f_s, E = g.E, S = g.S;
  bool ok = true;
  const bool sh = g.S > 0;
  switch (mode) {
    case FWD1:
      ok = (g.gather_rows != nullptr || (map2d(&p.a0, g.x_perm, d, Tk, 64, 128) && map2d(&p.h0, g.x_perm, d, Tk, 64, 64))) &&
           map3d(&p.b0, g.w13, d, 2 * f, E, 64, 128);
      if (sh) ok = ok && map2d(&p.a1, g.x, d, T, 64, 128) && map2d(&p.h1, g.x, d, T, 64, 64) &&
                   map3d(&p.b1, g.ws13, d, 2 * fs, S, 64, 128);
      if (!ok) return MOE_ERR_CUDA;
      return launch_mode<FWD1>(p, num_sms, st);
    case FWD2:
      ok = map2d(&p.a0, g.h, f, Tk, 64, 128) && map2d(&p.h0, g.h, f, Tk, 64, 64) && map3d(&p.b0, g.w2, f, d, E, 64, 256);
      if (sh) ok = ok && map2d(&p.a1, g.h_sh, fs, ST, 64, 128) && map2d(&p.h1, g.h_sh, fs, ST, 64, 64) &&
                   map3d(&p.b1, g.ws2, fs, d, S, 64, 256);
      if (!ok) return MOE_ERR_CUDA;
      return launch_mode<FWD2>(p, num_sms, st);
    case BWD2T:
      ok = (g.gather_rows != nullptr || (map2d(&p.a0, g.dy_perm, d, Tk, 64, 128) && map2d(&p.h0, g.dy_perm, d, Tk, 64, 64))) &&
           map4d_slabs(&p.b0, g.w2, f, d, E, 4);
      if (sh) ok = ok && map2d(&p.a1, g.dy, d, T, 64, 128) && map2d(&p.h1, g.dy, d, T, 64, 64) &&
                   map4d_slabs(&p.b1, g.ws2, fs, d, S, 4);
      if (!ok) return MOE_ERR_CUDA;
      return launch_mode<BWD2T>(p, num_sms, st);
    case BWD1T:
      ok = map2d(&p.a0, g.dz, 2 * f, Tk, 64, 128) && map2d(&p.h0, g.dz, 2 * f, Tk, 64, 64) &&
           map4d_slabs(&p.b0, g.w13, d, 2 * f, E, 4);
      if (sh) ok = ok && map2d(&p.a1, g.dz_sh, 2 * fs, ST, 64, 128) && map2d(&p.h1, g.dz_sh, 2 * fs, ST, 64, 64) &&
                   map4d_slabs(&p.b1, g.ws13, d, 2 * fs, S, 4);
      if (!ok) return MOE_ERR_CUDA;
      return launch_mode<BWD1T>(p, num_sms, st);
    case ROUTER:
      ok = map2d(&p.a0, g.x, d, T, 64, 128) && map2d(&p.b0, g.w_split, 3 * d, E, 64, 256);
      if (!ok) return MOE_ERR_CUDA;
      return launch_mode<ROUTER>(p, num_sms, st);
    default:
      return MOE_ERR_BAD_DIMS;
  }
}

}  // namespace moe
