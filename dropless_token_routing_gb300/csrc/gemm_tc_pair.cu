// dW products of the expert FFN on CTA pairs (sm_103a):
//   dW2_e  = dY_e^T (w h)_e   [d, f]
//   dW13_e = dz_e^T x_e       [2f, d]
// (and the shared experts' dWs2 / dWs13 over all T rows). The reduction runs over each
// expert's token copies, a short and ragged K (about T*k/E rows).
//
// The two CTAs of a cluster compute one 256 x 256 output tile with tcgen05.mma.cta_group::2.
// Each CTA stages its own 128 output rows of A and its own 128 output columns of B for a
// 64-deep K block; one instruction, issued by the even CTA, multiplies the pair's operands
// into both CTAs' tensor memory (each CTA holds its 128 x 256 fp32 half of the tile). A CTA
// thus loads 32 KB per K block for the same 128 x 256 x 64 of MMA work that costs 48 KB
// with a single CTA per 128 x 256 tile: a third less L2->SM traffic per FLOP, and room for
// six pipeline stages instead of four.
//
// Roles in each CTA of the pair (3 + EW warps, EW = 4 or 8 epilogue warps):
//   warp 0      TMA producer: this CTA's A and B halves into the 6- (or 5-) stage ring; the
//               bytes complete on this CTA's land_bar
//   warp 1      TMEM owner (the pair allocates together); in the even CTA its lane-0
//               thread issues the MMAs of the even tiles (accumulator 0)
//   warps 2..   epilogue: TMEM -> bf16 -> 128-byte swizzled staging -> TMA tensor store
//   warp 2+EW   relay: waits until this CTA's K block has landed, zeroes the A rows past a
//               ragged expert segment, then arrives on the even CTA's full_bar of the
//               tile's issuer, which therefore completes once both halves are in place
//   warp 3+EW   in the even CTA, lane 0 issues the MMAs of the odd tiles (accumulator 1)
// The issuers' commits arrive on the stage and accumulator barriers of both CTAs
// (multicast); each epilogue warp of either CTA frees an accumulator buffer by arriving on
// the even CTA's tempty_bar (2 * EW arrivals).
// Every mbarrier wait is bounded (1 s). On expiry the CTA records MOE_ERR_DEVICE_TIMEOUT and
// winds down: its producer waits for its own loads, the issuers for their MMAs, and the two
// CTAs meet at a cluster barrier before they release the tensor memory.
#include <cuda.h>

#include <mutex>

#include "grouped.cuh"
#include "internal.h"
#include "tc_common.cuh"
#include "trace.h"

namespace moe {
namespace {

using namespace tc;

constexpr int PM = 256, HM = 128;       // pair tile rows, rows per CTA
constexpr int BN = 256, HN = 128;       // pair tile columns, B columns staged per CTA
constexpr int BK = 64;
constexpr int A_BYTES = HM * BK * 2;    // 16 KB
constexpr int B_BYTES = HN * BK * 2;    // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_BYTES = 32 * 128;     // per epilogue warp: 32 rows x 64 bf16
// EW epilogue warps (4: each owns a TMEM lane quarter and all 256 columns; 8: two per lane
// quarter, 128 columns each); the pipeline gets the stages that fit beside their staging.
template <int EW> struct PairCfg {
  static constexpr int STAGES = EW == 4 ? 6 : 5;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EW * EPI_BYTES + 1024;
  static constexpr int THREADS = 32 * (4 + EW);
  static constexpr int RELAY = 2 + EW;   // warp index of the relay
  static constexpr int MMA2 = 3 + EW;    // warp index of the second MMA issuer
};
constexpr uint32_t TMEM_COLS = 512;     // two accumulator buffers of 256 fp32 columns
constexpr int SLAB = 64 * 128;          // one 64-element-wide, 64-row swizzled slab

struct PairParams {
  CUtensorMap a0, a1, b0, b1;  // operands (routed / shared), box {64, 64}
  CUtensorMap o0, o1;          // dW outputs (routed / shared), box {64, 32, 1}
  GroupedArgs g;
};

// ------------------------------------------------------------------ cluster / pair PTX
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive on a barrier given by its cluster address (the peer's, or this CTA's own). The
// default semantics (release at CTA scope) suffice for every hand-off of this kernel; a
// cluster-scope release made each hand-off a full memory barrier and the kernel 1.9x slower.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void umma_pair(uint32_t d_tmem, uint64_t ad, uint64_t bd, uint32_t idesc,
                                          uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(ad), "l"(bd), "r"(idesc), "r"(accum)
      : "memory");
}
// Arrive on the mbarrier at the same offset in every CTA of `mask` once the MMAs issued so
// far by this thread have completed.
__device__ __forceinline__ void umma_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

// ------------------------------------------------------------------ producer: TMA issue
// This CTA's halves of K block kb: A = output rows [m0, m0+128), B = output columns
// [n0, n0+128), both MN-major (the token copies run along K). `gather`: the token operand
// (A = dY for dW2, B = x for dW13) is gathered by the whole producer warp instead
// (gather_token_half), so it is skipped here.
template <int MODE>
__device__ __forceinline__ void issue_half_loads(const PairParams& p, const TileCoord& tc, int kb,
                                                 uint32_t rank, uint32_t a_s, uint32_t b_s,
                                                 uint32_t bar, bool gather) {
  const GroupGeom& G = tc.G;
  const int T = (int)p.g.T;
  const int m0 = tc.mi * PM + HM * (int)rank;
  const int n0 = tc.ni * BN + HN * (int)rank;
  const int k0 = kb * BK;
  const int row0 = (int)G.row0;
  const int ka = G.shared ? ((MODE == DW13 ? G.s * T : 0) + k0) : row0 + k0;   // A rows
  const int kbr = G.shared ? ((MODE == DW2 ? G.s * T : 0) + k0) : row0 + k0;  // B rows
  const CUtensorMap* am = G.shared ? &p.a1 : &p.a0;
  const CUtensorMap* bm = G.shared ? &p.b1 : &p.b0;
  if (!(gather && MODE == DW2)) {
#pragma unroll
    for (int i = 0; i < 2; ++i) tma2d(a_s + i * SLAB, am, bar, m0 + 64 * i, ka);
  }
  if (!(gather && MODE == DW13)) {
#pragma unroll
    for (int i = 0; i < 2; ++i) tma2d(b_s + i * SLAB, bm, bar, n0 + 64 * i, kbr);
  }
}

// Fused rearrangement of the token operand of a routed group (dY for dW2, x for dW13): this
// CTA's 128 columns of the K block's 64 token rows are gathered from the token-order tensor
// with 16-byte cp.async (one 64-column slab = 128 bytes per row, in the TMA's 128-byte
// swizzled layout: chunk c of row k at chunk c ^ (k & 7)). Per instruction the warp copies
// two rows x 256 bytes; rows past the segment repeat its first row (the ragged K fix-up
// zeroes the matching A rows, so they add nothing), and columns past the tensor are zero
// filled. The copies complete on `bar`. (TMA tile::gather4 copies of 512 bytes are held to
// about 5 B/cycle per SM by the TMA unit's rate per instruction.)
template <int MODE>
__device__ __forceinline__ void gather_token_half(const PairParams& p, const TileCoord& tc, int kb,
                                                  uint32_t rank, uint32_t a_s, uint32_t b_s,
                                                  uint32_t bar, int lane) {
  const GroupGeom& G = tc.G;
  const int d = p.g.d;
  const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(MODE == DW13 ? p.g.x : p.g.dy);
  // this lane's token rows: lane and lane + 32 of the K block
  int tk[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int k = kb * BK + lane + 32 * h;
    tk[h] = __ldg(p.g.gather_rows + G.row0 + (k < G.K ? k : 0));
  }
  const int c0 = (MODE == DW13 ? tc.ni * BN + HN * (int)rank : tc.mi * PM + HM * (int)rank);
  const int sl = (lane >> 3) & 1, c = lane & 7;
  const int col = c0 + 64 * sl + 8 * c;                 // this lane's 8 columns
  const bool col_ok = col < d;                          // d is a multiple of 64
  const uint32_t dst0 = (MODE == DW13 ? b_s : a_s) + sl * SLAB;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int k = 2 * i + (lane >> 4);                  // K row of this copy
    const int t = __shfl_sync(0xffffffffu, i < 16 ? tk[0] : tk[1], k & 31);
    const __nv_bfloat16* g = src + (int64_t)t * d + (col_ok ? col : 0);
    cp_async16(dst0 + k * 128 + ((c ^ (k & 7)) << 4), g, col_ok ? 16u : 0u);
  }
  cp_async_arrive(bar);
}

// ------------------------------------------------------------------ epilogue
// Four epilogue warps (dW2): each warp's 256 columns do not fit in registers at once, so
// each 32 x 64 chunk is converted to bf16, staged in the 128-byte swizzled layout and
// written by one TMA tensor store, the TMEM load of the next chunk in flight meanwhile; the
// accumulator is freed after the last chunk. (Reading all 256 columns first, as the
// eight-warp epilogue below does with its 128, measured 4-5 % slower for dW2.)
template <int MODE>
__device__ __forceinline__ void epilogue_chunked(const PairParams& p, const TileCoord& tc, uint32_t rank,
                                              int lg, uint32_t acc, uint8_t* stage, int lane, int col0,
                                              int ncols, uint64_t store_policy) {
  const GroupGeom& G = tc.G;
  const int n0 = tc.ni * BN + col0;
  acc += (uint32_t)col0;
  const int rowc = tc.mi * PM + HM * (int)rank + lg * 32;   // first row of this warp's 32
  if (rowc >= G.M) return;
  const CUtensorMap* om = G.shared ? &p.o1 : &p.o0;
  const int zc = G.shared ? G.s : G.e;
  const bool empty = G.K == 0;                              // dW of an expert without rows
  if (n0 >= G.N) return;
  const int nch = (min(ncols, G.N - n0) + 63) / 64;
  uint4 pk[8];
  uint32_t u[64];
  if (!empty) {
    tmem_ld32(acc, *reinterpret_cast<uint32_t(*)[32]>(u));
    tmem_ld32(acc + 32, *reinterpret_cast<uint32_t(*)[32]>(u + 32));
  }
#pragma unroll 1
  for (int ch = 0; ch < nch; ++ch) {
    const int c = ch * 64;
    if (!empty) {
      tmem_ld_wait();
#pragma unroll
      for (int q = 0; q < 8; ++q)
        pk[q] = make_uint4(pack_bf16x2(__uint_as_float(u[8 * q]), __uint_as_float(u[8 * q + 1])),
                           pack_bf16x2(__uint_as_float(u[8 * q + 2]), __uint_as_float(u[8 * q + 3])),
                           pack_bf16x2(__uint_as_float(u[8 * q + 4]), __uint_as_float(u[8 * q + 5])),
                           pack_bf16x2(__uint_as_float(u[8 * q + 6]), __uint_as_float(u[8 * q + 7])));
      if (ch + 1 < nch) {
        tmem_ld32(acc + c + 64, *reinterpret_cast<uint32_t(*)[32]>(u));
        tmem_ld32(acc + c + 96, *reinterpret_cast<uint32_t(*)[32]>(u + 32));
      }
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) pk[q] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (lane == 0) bulk_wait_read0();      // the previous store has left the buffer
    __syncwarp();
    uint4* srow = reinterpret_cast<uint4*>(stage + lane * 128);
#pragma unroll
    for (int q = 0; q < 8; ++q) srow[q ^ (lane & 7)] = pk[q];
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      tma_store3d_hint(om, smem_u32(stage), n0 + c, rowc, zc, store_policy);
      bulk_commit();
    }
  }
}

// Eight epilogue warps (dW13): the warp owns 32 rows of this CTA's 128 x 256 half tile (its TMEM lane quarter) and NCH
// 64-column chunks of them. It first reads all its accumulator columns into registers as
// bf16 and frees the accumulator (so the pair's next MMAs into it need not wait for the
// stores), then stages each 32 x 64 chunk in the 128-byte swizzled layout and writes it with
// one TMA tensor store. `release` frees the accumulator (called exactly once). Freeing it
// before the stores: DeepSeek-shaped dW13 4.75 -> 4.40-4.51 ms, the Pangu shape unchanged.
template <int MODE, int NCH, typename Release>
__device__ __forceinline__ void epilogue_half(const PairParams& p, const TileCoord& tc, uint32_t rank,
                                              int lg, uint32_t acc, uint8_t* stage, int lane, int col0,
                                              uint64_t store_policy, Release release) {
  const GroupGeom& G = tc.G;
  const int n0 = tc.ni * BN + col0;
  acc += (uint32_t)col0;
  const int rowc = tc.mi * PM + HM * (int)rank + lg * 32;   // first row of this warp's 32
  const bool empty = G.K == 0;                              // dW of an expert without rows
  const int nch = (rowc >= G.M || n0 >= G.N) ? 0 : (min(NCH * 64, G.N - n0) + 63) / 64;
  uint32_t pk[NCH][32];   // bf16 pairs: chunk ch, 64 columns
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    if (ch < nch && !empty) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t u[32];
        tmem_ld32(acc + ch * 64 + hh * 32, u);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 16; ++q) pk[ch][hh * 16 + q] = pack_bf16x2(__uint_as_float(u[2 * q]), __uint_as_float(u[2 * q + 1]));
      }
    } else {
#pragma unroll
      for (int q = 0; q < 32; ++q) pk[ch][q] = 0u;
    }
  }
  release();
  if (nch == 0) return;
  const CUtensorMap* om = G.shared ? &p.o1 : &p.o0;
  const int zc = G.shared ? G.s : G.e;
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    if (ch >= nch) break;
    if (lane == 0) bulk_wait_read0();      // the previous store has left the buffer
    __syncwarp();
    uint4* srow = reinterpret_cast<uint4*>(stage + lane * 128);
#pragma unroll
    for (int q = 0; q < 8; ++q)
      srow[q ^ (lane & 7)] = make_uint4(pk[ch][4 * q], pk[ch][4 * q + 1], pk[ch][4 * q + 2], pk[ch][4 * q + 3]);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      tma_store3d_hint(om, smem_u32(stage), n0 + ch * 64, rowc, zc, store_policy);
      bulk_commit();
    }
  }
}

// ------------------------------------------------------------------ the kernel
template <int MODE, int EW>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairCfg<EW>::THREADS, 1)
    tc_pair_dw_kernel(const __grid_constant__ PairParams p) {
  constexpr int STAGES = PairCfg<EW>::STAGES;
  extern __shared__ uint8_t smem_raw[];
  // full_bar[w][s]: stage s holds a K block of a tile of MMA issuer w (one set per issuer,
  // so that neither issuer ever waits on a phase of the other's K blocks)
  __shared__ __align__(8) uint64_t land_bar[STAGES], full_bar[2][STAGES], empty_bar[STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[2], tempty_bar[2], final_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;
  __shared__ TileSched sched;
  __shared__ int warp_sums[32];
  __shared__ int s_off[1024 + 1];

  const GroupedArgs& a = p.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair = (int)cluster_id(), npairs = (int)cluster_count();
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t smem_base = smem_u32(smem);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&land_bar[s]), 1);
      mbar_init(smem_u32(&full_bar[0][s]), 2);  // the relays of both CTAs
      mbar_init(smem_u32(&full_bar[1][s]), 2);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull_bar[b]), 1);
      mbar_init(smem_u32(&tempty_bar[b]), 2 * EW);   // the epilogue warps of both CTAs
    }
    mbar_init(smem_u32(&final_bar), 2);        // one commit from each MMA issuer
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_base_sh)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  build_tile_starts(a, MODE, PM, BN, sched, warp_sums, s_off);  // ends with __syncthreads
  cluster_sync_all();   // the peer's barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;
  const int ng = num_groups(MODE, a.E, a.S);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    int stage = 0;
    uint32_t phase = 0, pending = 0, pend_par = 0;
    bool ok = true;
    for (TileCursor cur(sched, ng, pair, npairs); cur.valid() && ok; cur.advance()) {
      const TileCoord tc = cur.coord(a, MODE, PM, s_off);
      const int nkb = (tc.G.K + BK - 1) / BK;
      const bool gather = a.gather_rows != nullptr && !tc.G.shared;
      for (int kb = 0; kb < nkb; ++kb) {
        const bool got = mbar_wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1u, &abort_flag, a.err,
                                           kWaitLimitNs);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        const uint32_t a_s = smem_base + stage * STAGE_BYTES, b_s = a_s + A_BYTES;
        const uint32_t bar = smem_u32(&land_bar[stage]);
        if (gather) {
          // the tiled operand's TMA first; lane 0 arrives only after every lane's copies are
          // counted by the barrier
          if (lane == 0) {
            mbar_expect_tx(bar, STAGE_BYTES - (MODE == DW13 ? B_BYTES : A_BYTES));
            issue_half_loads<MODE>(p, tc, kb, rank, a_s, b_s, bar, true);
          }
          gather_token_half<MODE>(p, tc, kb, rank, a_s, b_s, bar, lane);
          __syncwarp();
          if (lane == 0) mbar_arrive(bar);
        } else if (lane == 0) {
          mbar_arrive_expect_tx(bar, STAGE_BYTES);
          issue_half_loads<MODE>(p, tc, kb, rank, a_s, b_s, bar, false);
        }
        pending |= 1u << stage;
        pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    // drain: no TMA load may still be writing shared memory when the CTA exits
    for (int s = 0; s < STAGES; ++s)
      if ((pending >> s) & 1u)
        mbar_wait_bounded(smem_u32(&land_bar[s]), (pend_par >> s) & 1u, nullptr, a.err, kWaitLimitNs);
  } else if (warp == PairCfg<EW>::RELAY) {
    // ------------------------------------------------------------ relay (both CTAs)
    int stage = 0, it = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (TileCursor cur(sched, ng, pair, npairs); cur.valid() && ok; cur.advance(), ++it) {
      const TileCoord tc = cur.coord(a, MODE, PM, s_off);
      const int nkb = (tc.G.K + BK - 1) / BK;
      const int w = it & 1;   // the issuer of this tile
      const bool gathered = a.gather_rows != nullptr && !tc.G.shared;
      for (int kb = 0; kb < nkb; ++kb) {
        const bool got = mbar_wait_bounded(smem_u32(&land_bar[stage]), phase, &abort_flag, a.err,
                                           kWaitLimitNs);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        const int rem = tc.G.K - kb * BK;
        if (rem < BK) {
          // zero K rows [rem, roundup16(rem)) of both 64-wide slabs of this CTA's A half;
          // the issuer stops at roundup16(rem), so rows past that are never read
          uint4* A4 = reinterpret_cast<uint4*>(smem + stage * STAGE_BYTES);
          const int per_slab = (((rem + 15) & ~15) - rem) * 8;  // 16-byte chunks
          for (int i = lane; i < 2 * per_slab; i += 32) {
            const int sl = i / per_slab, j = i - sl * per_slab;
            A4[sl * (SLAB / 16) + rem * 8 + j] = make_uint4(0u, 0u, 0u, 0u);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        } else if (gathered) {
          // the gathered half was written through the generic proxy (cp.async)
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(peer_addr(smem_u32(&full_bar[w][stage]), 0));
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (warp == 1 || warp == PairCfg<EW>::MMA2) {
    // ------------------------------------------------------------ MMA issuers (even CTA)
    // Two threads in different warps issue alternate tiles, issuer w the tiles that use
    // accumulator w, so that one thread's waits and bookkeeping between K blocks overlap
    // the other's MMAs (a single issuing thread leaves the tensor pipe idle there). Each
    // walks the whole tile sequence to keep its place in the stage ring; a commit covers
    // only the committing thread's own MMAs, which are the ones that read its stages.
    const int w = warp == 1 ? 0 : 1;
    if (leader && lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(PM, BN, true, true);
      int stage = 0;
      uint32_t fpar = 0;   // per stage: parity of this issuer's next wait on full_bar[w][stage]
      bool ok = true;
      int it = 0;
      for (TileCursor cur(sched, ng, pair, npairs); cur.valid() && ok; cur.advance(), ++it) {
        const TileCoord tc = cur.coord(a, MODE, PM, s_off);
        const int nkb = (tc.G.K + BK - 1) / BK;
        const int b = it & 1;
        if (b != w) {   // the other issuer's tile: step over its K blocks in the ring
          stage = (stage + nkb) % STAGES;
          continue;
        }
        if (!mbar_wait_bounded(smem_u32(&tempty_bar[b]), ((it >> 1) & 1) ^ 1, &abort_flag, a.err,
                               kWaitLimitNs)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(b * BN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full_bar[w][stage]), (fpar >> stage) & 1u, &abort_flag, a.err,
                                 kWaitLimitNs)) {
            ok = false;
            break;
          }
          fpar ^= 1u << stage;
          tc_fence_after();
          const uint32_t a_s = smem_base + stage * STAGE_BYTES, b_s = a_s + A_BYTES;
          // K=16 steps in this block: 4, or fewer in a ragged last block
          const int nks = min(BK, tc.G.K - kb * BK + 15) / 16;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            if (kk >= nks) break;
            umma_pair(d_tmem, sdesc(a_s + kk * 2048, SLAB, 1024), sdesc(b_s + kk * 2048, SLAB, 1024), idesc,
                      (kb | kk) != 0 ? 1u : 0u);
          }
          // the tile's last stage is released by the epilogue once the accumulator is full:
          // a commit straight after another one stalls the tensor pipe
          if (kb + 1 < nkb) umma_commit_mc(smem_u32(&empty_bar[stage]), 0x3);
          if (++stage == STAGES) stage = 0;
        }
        if (!ok) break;
        if (nkb > 0) {
          umma_commit_mc(smem_u32(&tfull_bar[b]), 0x3);
        } else {
          mbar_arrive(smem_u32(&tfull_bar[b]));
          mbar_arrive_remote(peer_addr(smem_u32(&tfull_bar[b]), 1));
        }
      }
      // every MMA of both issuers retired before the tensor memory is released (a commit
      // with no MMA before it arrives at once)
      umma_commit_mc(smem_u32(&final_bar), 0x1);
      mbar_wait_bounded(smem_u32(&final_bar), 0, nullptr, a.err, kWaitLimitNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue warps 2..5
    const int lg = warp & 3;              // TMEM lane quarter this warp may access
    const int col0 = EW == 4 ? 0 : ((warp - 2) >> 2) * (BN / 2), ncols = EW == 4 ? BN : BN / 2;
    uint8_t* stage = smem + STAGES * STAGE_BYTES + (warp - 2) * EPI_BYTES;
    // the gradient is written once and never read here: it leaves L2 first, so that the
    // token rows re-read by the expert's later tiles stay (dW13 4.93 -> 4.62-4.71 ms)
    const uint64_t store_policy = l2_evict_first();
    int it = 0, kblocks = 0;   // tiles and K blocks seen so far
    for (TileCursor cur(sched, ng, pair, npairs); cur.valid(); cur.advance(), ++it) {
      const TileCoord tc = cur.coord(a, MODE, PM, s_off);
      const int b = it & 1;
      const bool got = mbar_wait_bounded(smem_u32(&tfull_bar[b]), (it >> 1) & 1, &abort_flag, a.err,
                                         kWaitLimitNs);
      if (!__all_sync(0xffffffffu, got)) break;   // warp-uniform: tcgen05.ld is .sync.aligned
      // the accumulator is full, so every MMA of the tile has read its operands: release the
      // stage of the tile's last K block in this CTA (the issuer commits the others)
      const int nkb = (tc.G.K + BK - 1) / BK;
      if (warp == 2 && lane == 0 && nkb > 0) mbar_arrive(smem_u32(&empty_bar[(kblocks + nkb - 1) % STAGES]));
      kblocks += nkb;
      tc_fence_after();
      const uint32_t acc = tmem_base + ((uint32_t)(lg * 32) << 16) + (uint32_t)(b * BN);
      const uint32_t tempty_peer = peer_addr(smem_u32(&tempty_bar[b]), 0);
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(tempty_peer);
      };
      if constexpr (EW == 8) {
        epilogue_half<MODE, BN / 2 / 64>(p, tc, rank, lg, acc, stage, lane, col0, store_policy, release);
      } else {
        epilogue_chunked<MODE>(p, tc, rank, lg, acc, stage, lane, col0, ncols, store_policy);
        release();
      }
    }
    if (lane == 0) bulk_wait0();  // tensor stores fully written
  }
  __syncthreads();
  cluster_sync_all();   // neither CTA releases its tensor memory while the pair still uses it
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
}

template <int MODE, int EW>
int launch_pair_ew(PairParams& p, int num_sms, cudaStream_t st) {
  constexpr int SMEM_BYTES = PairCfg<EW>::SMEM_BYTES, THREADS = PairCfg<EW>::THREADS;
  // per device, once (under a lock: callers may be several host threads): the shared-memory
  // attribute and the pairs that can be resident at once
  static std::mutex mu;
  static int occ_dev[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  int occ;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (occ_dev[dev] == 0) {
      if (cudaFuncSetAttribute(tc_pair_dw_kernel<MODE, EW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               SMEM_BYTES) != cudaSuccess)
        return MOE_ERR_CUDA;
      cudaLaunchConfig_t cfg;
      memset(&cfg, 0, sizeof(cfg));
      cfg.gridDim = dim3((unsigned)(num_sms & ~1));
      cfg.blockDim = dim3(THREADS);
      cfg.dynamicSmemBytes = SMEM_BYTES;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, tc_pair_dw_kernel<MODE, EW>, &cfg) != cudaSuccess || n <= 0)
        return MOE_ERR_CUDA;
      occ_dev[dev] = n;
    }
    occ = occ_dev[dev];
  }
  const int nc = occ < num_sms / 2 ? occ : num_sms / 2;
  TraceScope ts(MODE == DW13 ? TP_GEMM_DW13 : TP_GEMM_DW2, st);
  tc_pair_dw_kernel<MODE, EW><<<2 * nc, THREADS, SMEM_BYTES, st>>>(p);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

// dW13 (2f = 4096 output rows, 5.0 vs 5.2 ms measured) takes eight epilogue warps and five
// stages; dW2 (2.57 vs 2.60 ms) four warps and six stages.
template <int MODE>
int launch_pair(PairParams& p, int num_sms, cudaStream_t st) {
  return MODE == DW13 ? launch_pair_ew<MODE, 8>(p, num_sms, st) : launch_pair_ew<MODE, 4>(p, num_sms, st);
}

}  // namespace

int launch_tc_pair_dw(int mode, const GroupedArgs& g, int num_sms, cudaStream_t st) {
  PairParams p;
  memset(&p, 0, sizeof(p));
  p.g = g;
  const uint64_t Tk = (uint64_t)g.Tk, T = (uint64_t)g.T, ST = (uint64_t)g.S * g.T;
  const uint64_t d = g.d, f = g.f, fs = g.f_s, E = g.E, S = g.S;
  const bool sh = g.S > 0;
  bool ok;
  const bool gather = g.gather_rows != nullptr;
  if (mode == DW2) {
    ok = (gather || map2d(&p.a0, g.dy_perm, d, Tk, 64, 64)) &&
         map2d(&p.b0, g.hw, f, Tk, 64, 64) && map3d(&p.o0, g.dw2, f, d, E, 64, 32);
    if (sh) ok = ok && map2d(&p.a1, g.dy, d, T, 64, 64) && map2d(&p.b1, g.hw_sh, fs, ST, 64, 64) &&
                 map3d(&p.o1, g.dws2, fs, d, S, 64, 32);
    if (!ok) return MOE_ERR_CUDA;
    return launch_pair<DW2>(p, num_sms, st);
  }
  ok = map2d(&p.a0, g.dz, 2 * f, Tk, 64, 64) &&
       (gather || map2d(&p.b0, g.x_perm, d, Tk, 64, 64)) &&
       map3d(&p.o0, g.dw13, d, 2 * f, E, 64, 32);
  if (sh) ok = ok && map2d(&p.a1, g.dz_sh, 2 * fs, ST, 64, 64) && map2d(&p.b1, g.x, d, T, 64, 64) &&
               map3d(&p.o1, g.dws13, d, 2 * fs, S, 64, 32);
  if (!ok) return MOE_ERR_CUDA;
  return launch_pair<DW13>(p, num_sms, st);
}

}  // namespace moe
