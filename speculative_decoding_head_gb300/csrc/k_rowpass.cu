// k_rowpass.cu -- row-oriented vocabulary passes on tcgen05: the training
// objective's two passes, the RNN head's per-step block masses, and the
// PCTree expansion's block masses and maxima.
//
// deepseek.csdn.net reading §6, eqs. (9)-(12): every teacher-forced position
// i = (b, k) has draft logits z_d = U[b, k] + W1[x*_{k-1}] W2 (x*_{-1} = the
// anchor) and target logits z_t = P[b, k]; the objective needs, per
// position, lse(z_d), lse(z_t), z_d at x*_k and sum_v |p_d(v) - p_t(v)|.
//
// Orientation: the positions are the MMA rows (M = 128 per row group) and a
// tile is 128 vocabulary entries (N), so a CTA reads each W2 tile once for
// its 128 positions (the column orientation of k_resid_tc.cu reads it once
// per 32). CTAs take row groups round-robin and, inside a group, contiguous
// ranges of 64-token blocks, as the Markov draft kernel does:
//   warp 0      TMA producer of W2 (64 K rows x 128 tokens per stage,
//               128-byte swizzle, L2 evict_last);
//   warp 10     TMA producer of U and P, [128 rows x 32] fp32 boxes, two per
//               64-token block (evict_first), into a ring of 32 KB stages;
//   warp 11     copier: each tile's U blocks into its accumulator and its P
//               blocks into a P buffer in tensor memory (tcgen05.cp), so an
//               epilogue thread reads z_d and z_t of its row from TMEM;
//   warp 1      allocates all 512 TMEM columns (two 128-column accumulators,
//               two 128-column P buffers; see below for the other modes) and
//               issues tcgen05.mma (M = 128, N = 128, K = r) onto the
//               accumulator that holds U: z_d;
//   warps 2-9   epilogue, two sets of four warps (blocks of even and odd
//               index), one thread per row: pass 0 keeps a running
//               (max, sum 2^(y - max)) of z_d and of z_t and picks z_d at x*;
//               pass 1 sums |2^(z_d - lse_d) - 2^(z_t - lse_t)| (log2 units).
// A row's two sets meet in shared memory at the end; the CTA writes one
// partial per position into slot cg (its index in the group) of the
// [n][G] partial arrays, and neutral values into the slots no CTA of the
// group owns, so the combine kernels read G slots as before.
//
// The same pass with requests as rows serves two more computations:
//   - one draft step of the RNN head (eq. (6), same reading §4.2): rows are
//     requests, A = o_k split into bf16 hi and lo images, which the cell
//     wrote in this operand's layout: the copier brings the lo image in by
//     one bulk copy and moves it to TMEM, then the hi image, which stays in
//     the A region as the shared-memory operand; per K step both MMAs
//     accumulate into the tile (hi from shared memory, lo from TMEM), and
//     TMEM holds three accumulators beside the lo image; U_k arrives by a 3-D
//     box; per row and 64-token block the log-mass log sum exp z goes to blk
//     [B][nblk] for the pick;
//   - one PCTree expansion (zdszero "spec_dspark", section "后续工作"): rows
//     are requests, A = W1[token of the node being expanded], and U of the
//     node's depth differs per row, so the epilogue adds it from global
//     memory (the accumulator starts at zero); four accumulators (no P
//     buffers); per block the log-mass and the maximum of z.
// The RNN and PCTree launches are dependent launches (programmatic stream
// serialization): only the epilogue (and, for RNN, the copier's image loads)
// waits for the kernel before, so the W2 and U streams start meanwhile.
// Every wait is bounded; a timeout sets DSPARK_ETIMEOUT and every role ends.
#include <cudaTypedefs.h>
#include <string.h>

#include "dspark_common.cuh"
#include "dspark_internal.h"
#include "tc_ptx.cuh"

namespace dspark {

namespace {

constexpr int kRpSets = 2;
constexpr int kRpEpi = kRpSets * 128;          // epilogue threads (warps 2 .. 9)
constexpr int kRpUWarp = 2 + 4 * kRpSets;      // U and P producer
constexpr int kRpCWarp = kRpUWarp + 1;         // copier
constexpr int kRpThreads = 32 * (kRpCWarp + 1);
constexpr int kRpRows = 128;                   // MMA M: positions of a row group
constexpr int kRpBlk = 64;                     // block = 64 tokens = one 64-column accumulator slice
constexpr int kRpTileBlocks = 2;               // MMA N = 128
constexpr int kRpKc = 64;                      // K rows of W2 per stage
constexpr int kRpW2Box = kRpKc * 128;          // 8 KB: 64 K rows x 64 tokens
constexpr int kRpW2Stage = kRpTileBlocks * kRpW2Box;  // 16 KB
constexpr int kRpNW = 4;                       // W2 ring (K chunks)
constexpr int kRpNU = 3;                       // U / P staging ring (blocks)
constexpr int kRpUStage = kRpRows * kRpBlk * 4;  // 32 KB: two 128 x 32 fp32 boxes
constexpr int kRpUBox = kRpRows * 32 * 4;        // 16 KB
constexpr int kRpAccCols = kRpTileBlocks * kRpBlk;  // 128
constexpr int kRpNAcc = 2;                     // accumulators (and as many P buffers)
constexpr int kRpNAccMax = 4;                  // RNN: three accumulators (o_k's hi image stays in shared memory); PCTree: four
constexpr int kRpTmemCols = 512;
constexpr int kRpMaxGroups = 64;               // n <= 8192 positions

// What a launch computes (template MODE)
constexpr int kRowLoss0 = 0;  // per position: (max, sum exp) of z_d and z_t, z_d at x*
constexpr int kRowLoss1 = 1;  // per position: sum |p_d - p_t|
constexpr int kRowRnn = 2;    // per request and block: log-mass of U_k + o_k W2 (o_k as bf16 hi + lo)
constexpr int kRowTree = 3;   // per request and block: log-mass and max of U[b, depth] + W1[token] W2

struct RpSmem {
  uint32_t a, w2, u, bars, misc, total;
  __host__ __device__ static RpSmem make(int r) {
    RpSmem s;
    s.a = 0;                                   // A = W1[x*_{k-1}] of the group's rows, K-major, swizzled
    s.w2 = s.a + kRpRows * r * 2;
    s.u = s.w2 + kRpNW * kRpW2Stage;
    s.bars = s.u + kRpNU * kRpUStage;
    // w2 full/empty, u full/empty, acc_u, t_full, t_empty, p_full, p_empty, a_full, drains,
    // a_cp_hi, a_cp_lo, a_ld
    s.misc = s.bars + 8 * (2 * kRpNW + 2 * kRpNU + 5 * kRpNAccMax + 6);
    // misc: TMEM address, abort word
    s.total = s.misc + 64;
    return s;
  }
};

struct RpParams {
  int n, g, V, r, nblk, nG, G;
  int step;            // RNN: draft step k (1-based)
  const float* ovec;   // RNN: [B][g][r] o_k
  const __nv_bfloat16* oimg;  // RNN: per row group, o_k's bf16 hi then lo image in the A operand's layout
  const float* U;      // PCTree: U [B][g][V], read by the epilogue
  const int32_t* tree_tok;   // PCTree: [B][N+1] nodes' tokens, depths; state[b].y = the node to expand
  const int32_t* tree_dep;
  const int4* tree_state;
  int tree_N;
  float* blk;          // RNN, PCTree: [B][nblk] block log-masses
  float* bmax;         // PCTree: [B][nblk] block maxima
  const int32_t* anchor;
  const int32_t* xstar;
  const void* W1;
  const float* lse_d;  // pass 1
  const float* lse_t;
  float4* lpart;       // pass 0: [n][G] (max_d, sum_d, max_t, sum_t), sums in 2^(y - max) form
  float* zx;           // pass 0: [n] z_d at x*
  float* l1part;       // pass 1: [n][G]
  int* status;
};

__device__ __forceinline__ int rp_group_ctas(int G, int nG, int g) { return (G - g + nG - 1) / nG; }

// Offset (bf16 elements) of the 16-byte piece ch of K-block kb of row m in the
// A operand: K-major, 128-byte swizzle, 8-row atoms of 1 KB, K-blocks of 64
// elements 16 KB apart.
__device__ __forceinline__ size_t rp_a_piece(int m, int kb, int ch) { return kmajor_sw128_piece(m, kb, ch, kRpRows); }

// (max, sum 2^(y log2e - max log2e)) of 32 values on fp32 pairs.
__device__ __forceinline__ void half_ms(const float (&y)[32], float& mb, float& sb) {
  float m4[4];
#pragma unroll
  for (int c4 = 0; c4 < 4; ++c4) {
    m4[c4] = tc::max3f(y[8 * c4], y[8 * c4 + 1], y[8 * c4 + 2]);
    m4[c4] = tc::max3f(m4[c4], y[8 * c4 + 3], y[8 * c4 + 4]);
    m4[c4] = tc::max3f(m4[c4], y[8 * c4 + 5], y[8 * c4 + 6]);
    m4[c4] = fmaxf(m4[c4], y[8 * c4 + 7]);
  }
  mb = fmaxf(tc::max3f(m4[0], m4[1], m4[2]), m4[3]);
  if (mb == -INFINITY) {
    sb = 0.f;
    return;
  }
  const unsigned long long l2e = tc::f2pack(tc::kLog2e, tc::kLog2e);
  const unsigned long long nml = tc::f2pack(-mb * tc::kLog2e, -mb * tc::kLog2e);
  unsigned long long acc[2];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float a0, a1;
    tc::f2unpack(tc::fma2(tc::f2pack(y[2 * i], y[2 * i + 1]), l2e, nml), a0, a1);
    const unsigned long long e2 = tc::f2pack(tc::ex2_ftz(a0), tc::ex2_ftz(a1));
    acc[i & 1] = i < 2 ? e2 : tc::add2(acc[i & 1], e2);
  }
  float sl, sh;
  tc::f2unpack(tc::add2(acc[0], acc[1]), sl, sh);
  sb = sl + sh;
}

// y[i] for a run-time i < 32 by a tree of selects on the bits of i (a
// register array indexed at run time would live in local memory)
__device__ __forceinline__ float pick32(const float (&y)[32], int i) {
  float t16[16], t8[8], t4[4], t2[2];
#pragma unroll
  for (int e = 0; e < 16; ++e) t16[e] = (i & 16) ? y[e + 16] : y[e];
#pragma unroll
  for (int e = 0; e < 8; ++e) t8[e] = (i & 8) ? t16[e + 8] : t16[e];
#pragma unroll
  for (int e = 0; e < 4; ++e) t4[e] = (i & 4) ? t8[e + 4] : t8[e];
#pragma unroll
  for (int e = 0; e < 2; ++e) t2[e] = (i & 2) ? t4[e + 2] : t4[e];
  return (i & 1) ? t2[1] : t2[0];
}

// merge (mb, sb) into the running (M, S): S = sum 2^((y - M) log2e)
__device__ __forceinline__ void ms_merge(float& M, float& S, float mb, float sb) {
  if (mb > M) {
    S = S * tc::ex2_ftz((M - mb) * tc::kLog2e) + sb;
    M = mb;
  } else if (mb > -INFINITY) {
    S += sb * tc::ex2_ftz((mb - M) * tc::kLog2e);
  }
}

template <int MODE>
__global__ void __launch_bounds__(kRpThreads, 1)
    k_rowpass(const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_u,
              const __grid_constant__ CUtensorMap tm_p, const RpParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const RpSmem L = RpSmem::make(p.r);
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t sA = sbase + L.a, sW2 = sbase + L.w2, sU = sbase + L.u;
  const uint32_t bars = sbase + L.bars;
  auto w2_full = [&](int i) { return bars + 8u * i; };
  auto w2_empty = [&](int i) { return bars + 8u * (kRpNW + i); };
  auto u_full = [&](int i) { return bars + 8u * (2 * kRpNW + i); };
  auto u_empty = [&](int i) { return bars + 8u * (2 * kRpNW + kRpNU + i); };
  const uint32_t b5 = bars + 8u * (2 * kRpNW + 2 * kRpNU);
  auto acc_u = [&](int i) { return b5 + 8u * i; };                 // the accumulator holds U
  auto t_full = [&](int i) { return b5 + 8u * (kRpNAccMax + i); };    // the MMAs of the tile are done
  auto t_empty = [&](int i) { return b5 + 8u * (2 * kRpNAccMax + i); };  // the epilogue read acc and P buffer
  auto p_full = [&](int i) { return b5 + 8u * (3 * kRpNAccMax + i); };   // the P buffer holds the tile's P
  auto p_empty = [&](int i) { return b5 + 8u * (4 * kRpNAccMax + i); };  // (unused slot: keeps the layout even)
  const uint32_t a_full = b5 + 8u * (5 * kRpNAccMax);
  const uint32_t drain = a_full + 8u, drain_c = a_full + 16u;
  // RNN: o_k's lo image is in TMEM (a_cp_lo), its hi image in the A region (a_cp_hi)
  const uint32_t a_cp_hi = a_full + 24u, a_cp_lo = a_full + 32u;
  const uint32_t a_ld = a_full + 40u;                              // RNN: an A image has landed in shared memory
  constexpr bool kLoss = MODE == kRowLoss0 || MODE == kRowLoss1;
  // TMEM: accumulators at columns 0 and 128, then the P buffers (loss); RNN:
  // accumulators at 0, 128 and 256, then o_k's lo image (r / 2 columns);
  // PCTree (no P, A in shared memory): four accumulators
  const int NACC = MODE == kRowRnn ? 3 : MODE == kRowTree ? 4 : kRpNAcc;
  const uint32_t tm_lo = (uint32_t)(NACC * kRpAccCols);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L.misc + 16);
  // [128] set 1's results per row, at the end: the A region is free once the
  // epilogue has read the last tile (every MMA has completed)
  float4* xchg = reinterpret_cast<float4*>(smem + L.a);
  (void)p_empty;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int grp = c % p.nG, cg = c / p.nG;
  const int Gg = rp_group_ctas(p.G, p.nG, grp);
  const int blo = (int)((long long)cg * p.nblk / Gg);
  const int nbc = (int)((long long)(cg + 1) * p.nblk / Gg) - blo;
  const int ntl = (nbc + kRpTileBlocks - 1) / kRpTileBlocks;
  const int nkc = p.r / kRpKc;
  auto tile_blocks = [&](int tj) { return min(kRpTileBlocks, nbc - tj * kRpTileBlocks); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRpNW; ++i) {
      tc::mbar_init(w2_full(i), 1);
      tc::mbar_init(w2_empty(i), 1);
    }
    for (int i = 0; i < kRpNU; ++i) {
      tc::mbar_init(u_full(i), 1);
      tc::mbar_init(u_empty(i), 1);
    }
    for (int i = 0; i < kRpNAccMax; ++i) {
      tc::mbar_init(acc_u(i), 1);
      tc::mbar_init(t_full(i), 1);
      tc::mbar_init(t_empty(i), kRpEpi / 32);
      tc::mbar_init(p_full(i), 1);
      tc::mbar_init(p_empty(i), 1);
    }
    tc::mbar_init(a_full, kRpEpi / 32);
    tc::mbar_init(drain, 1);
    tc::mbar_init(drain_c, 1);
    tc::mbar_init(a_cp_hi, 1);
    tc::mbar_init(a_cp_lo, 1);
    tc::mbar_init(a_ld, 1);
    *abort = 0;
    tc::fence_barrier_init();
    tc::prefetch_tmap(&tm_w2);
    tc::prefetch_tmap(&tm_u);
    tc::prefetch_tmap(&tm_p);
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(tmem_holder), kRpTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ W2 producer
    if (lane == 0) {
      const uint64_t keep = tc::policy_evict_last();
      int wiss = 0;
      bool ok = true;
      for (int tj = 0; tj < ntl && ok; ++tj) {
        const int nbt = tile_blocks(tj), v0 = (blo + tj * kRpTileBlocks) * kRpBlk;
        for (int ch = 0; ch < nkc && ok; ++ch) {
          const int wc = tj * nkc + ch, ws = wc % kRpNW;
          ok = tc::mbar_wait(w2_empty(ws), ((wc / kRpNW) & 1) ^ 1, abort);
          if (!ok) break;
          tc::mbar_arrive_expect_tx(w2_full(ws), (uint32_t)(nbt * kRpW2Box));
          for (int j = 0; j < nbt; ++j)
            tc::tma_load_2d(sW2 + ws * kRpW2Stage + j * kRpW2Box, &tm_w2, v0 + j * kRpBlk, ch * kRpKc, w2_full(ws),
                            keep);
          wiss = wc + 1;
        }
      }
      if (!ok) {
        if (!*abort) raise_status(p.status, DSPARK_ETIMEOUT);
        *abort = 1;
        volatile int never = 0;
        for (int wc = wiss - 1; wc >= 0 && wc >= wiss - kRpNW; --wc)
          tc::mbar_wait(w2_full(wc % kRpNW), (wc / kRpNW) & 1, &never);
      }
    }
  } else if (warp == kRpUWarp) {
    // ------------------------------------------------------------ U and P producer
    // per tile: its U blocks, then its P blocks, each one ring stage
    if (lane == 0 && MODE != kRowTree) {
      const uint64_t stream = tc::policy_evict_first();
      int iss = 0;
      bool ok = true;
      const int per_tile = kLoss ? 2 : 1;  // U blocks, then (loss) P blocks
      for (int tj = 0; tj < ntl && ok; ++tj) {
        const int nbt = tile_blocks(tj);
        for (int e = 0; e < per_tile * nbt && ok; ++e) {
          const int j = e % nbt, us = iss % kRpNU, v = (blo + tj * kRpTileBlocks + j) * kRpBlk;
          ok = tc::mbar_wait(u_empty(us), ((iss / kRpNU) & 1) ^ 1, abort);
          if (!ok) break;
          tc::mbar_arrive_expect_tx(u_full(us), kRpUStage);
          if constexpr (MODE == kRowRnn) {  // U_k of the group's requests: a 3-D box (V, g, B) at step k
            tc::tma_load_3d(sU + us * kRpUStage, &tm_u, v, p.step - 1, grp * kRpRows, u_full(us), stream);
            tc::tma_load_3d(sU + us * kRpUStage + kRpUBox, &tm_u, v + 32, p.step - 1, grp * kRpRows, u_full(us),
                            stream);
          } else {
            const CUtensorMap* tm = e < nbt ? &tm_u : &tm_p;
            tc::tma_load_2d(sU + us * kRpUStage, tm, v, grp * kRpRows, u_full(us), stream);
            tc::tma_load_2d(sU + us * kRpUStage + kRpUBox, tm, v + 32, grp * kRpRows, u_full(us), stream);
          }
          ++iss;
        }
      }
      if (!ok) {
        if (!*abort) raise_status(p.status, DSPARK_ETIMEOUT);
        *abort = 1;
        volatile int never = 0;
        for (int i = iss - 1; i >= 0 && i >= iss - kRpNU; --i)
          tc::mbar_wait(u_full(i % kRpNU), (i / kRpNU) & 1, &never);
      }
    }
  } else if (warp == kRpCWarp) {
    // ------------------------------------------------------------ copier
    // each tile's U blocks into its (free) accumulator, its P blocks into the
    // matching P buffer; a staging slot is free once its copies land
    if (lane == 0) {
      bool ok = true;
      int iss = 0;
      const int per_tile = MODE == kRowTree ? 0 : kLoss ? 2 : 1;
      auto copy_tile = [&](int tj) {
        const int nbt = tile_blocks(tj), ab = tj % NACC;
        bool okt = tc::mbar_wait(t_empty(ab), ((tj / NACC) & 1) ^ 1, abort);  // accumulator and P buffer free
        if (okt && per_tile == 0) tc::mma_commit(acc_u(ab));  // PCTree: the MMAs start from zero
        for (int e = 0; e < per_tile * nbt && okt; ++e) {
          const int j = e % nbt, us = iss % kRpNU;
          okt = tc::mbar_wait(u_full(us), (iss / kRpNU) & 1, abort);
          if (!okt) break;
          tc::tc_fence_after();
          const uint32_t d = tmem + (uint32_t)((e < nbt ? 0 : NACC * kRpAccCols) + ab * kRpAccCols + j * kRpBlk);
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
              tc::cp_128x256b(d + (uint32_t)(h * 32 + cc * 8),
                              tc::smem_desc(sU + us * kRpUStage + h * kRpUBox + cc * 32, 16, 1024));
          tc::mma_commit(u_empty(us));
          ++iss;
          if (e == nbt - 1) tc::mma_commit(acc_u(ab));
        }
        if (okt && kLoss) tc::mma_commit(p_full(ab));
        return okt;
      };
      if constexpr (MODE == kRowRnn) {
        // o_k's images, written by the cell in the operand's layout, each
        // come into the A region by one bulk copy: the lo image first, which
        // goes on to its TMEM columns (16 bf16 of K per 8 columns), then the
        // hi image, which stays there as the MMAs' shared-memory A operand
        // (a_cp_hi completes when it has landed). The first tiles' U goes
        // into the accumulators while the lo image is in flight.
        pdl_wait();  // the images are the cell's
        const uint32_t abytes = (uint32_t)(kRpRows * p.r * 2);
        const __nv_bfloat16* img = p.oimg + (size_t)grp * 2 * kRpRows * p.r;  // [hi | lo]
        bool hi_issued = false;
        tc::mbar_arrive_expect_tx(a_ld, abytes);
        tc::bulk_load(sA, img + (size_t)kRpRows * p.r, abytes, a_ld);
        const int pre = min(ntl, kRpNAcc);
        for (int tj = 0; tj < pre && ok; ++tj) ok = copy_tile(tj);
        if (ok) ok = tc::mbar_wait(a_ld, 0, abort);
        if (ok) {
          for (int ks = 0; ks < p.r / 16; ++ks)
            tc::cp_128x256b(tmem + tm_lo + (uint32_t)(ks * 8),
                            tc::smem_desc(sA + (ks >> 2) * (kRpRows * 128) + (ks & 3) * 32, 16, 1024));
          tc::mma_commit(a_cp_lo);
          ok = tc::mbar_wait(a_cp_lo, 0, abort);  // the copies have read the lo image: the region takes hi
        }
        if (ok) {
          tc::mbar_arrive_expect_tx(a_cp_hi, abytes);
          tc::bulk_load(sA, img, abytes, a_cp_hi);
          hi_issued = true;
        }
        if (!ok) {  // an image copy still in flight lands before the CTA ends
          volatile int never = 0;
          tc::mbar_wait(a_ld, 0, &never);
        }
        for (int tj = pre; tj < ntl && ok; ++tj) ok = copy_tile(tj);
        if (hi_issued) {  // the hi image has landed before the CTA ends (at once unless a wait gave up)
          volatile int never = 0;
          tc::mbar_wait(a_cp_hi, 0, &never);
        }
      } else {
        for (int tj = 0; tj < ntl && ok; ++tj) ok = copy_tile(tj);
      }
      if (!ok) {
        if (!*abort) raise_status(p.status, DSPARK_ETIMEOUT);
        *abort = 1;
      }
      tc::mma_commit(drain_c);
      volatile int never = 0;
      tc::mbar_wait(drain_c, 0, &never);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = MODE == kRowRnn ? (tc::mbar_wait(a_cp_hi, 0, abort) && tc::mbar_wait(a_cp_lo, 0, abort))
                                : tc::mbar_wait(a_full, 0, abort);
      if (ok) tc::tc_fence_after();
      for (int tj = 0; tj < ntl && ok; ++tj) {
        const int nbt = tile_blocks(tj), ab = tj % NACC;
        const uint32_t idesc = tc::idesc_bf16_f32(kRpRows, nbt * kRpBlk, true);
        const uint32_t d = tmem + (uint32_t)(ab * kRpAccCols);
        ok = tc::mbar_wait(acc_u(ab), (tj / NACC) & 1, abort);
        if (ok) tc::tc_fence_after();
        for (int ch = 0; ch < nkc && ok; ++ch) {
          const int wc = tj * nkc + ch, ws = wc % kRpNW;
          ok = tc::mbar_wait(w2_full(ws), (wc / kRpNW) & 1, abort);
          if (!ok) break;
          tc::tc_fence_after();
          for (int kk = 0; kk < kRpKc / 16; ++kk) {
            const int ks = ch * (kRpKc / 16) + kk;
            const uint64_t bd = tc::smem_desc(sW2 + ws * kRpW2Stage + kk * 2048, kRpW2Box, 1024);
            if constexpr (MODE == kRowRnn) {  // o_k hi (shared memory), then lo (TMEM), against the same W2 rows
              const uint64_t ah = tc::smem_desc(sA + (ks >> 2) * (kRpRows * 128) + (ks & 3) * 32, 16, 1024);
              tc::mma_bf16(d, ah, bd, idesc, 1u);
              tc::mma_bf16_ta(d, tmem + tm_lo + (uint32_t)(ks * 8), bd, idesc, 1u);
            } else {
              const uint64_t ad = tc::smem_desc(sA + (ks >> 2) * (kRpRows * 128) + (ks & 3) * 32, 16, 1024);
              // the accumulator starts as U (PCTree: from zero, U is added by the epilogue)
              tc::mma_bf16(d, ad, bd, idesc, (MODE != kRowTree || ks > 0) ? 1u : 0u);
            }
          }
          tc::mma_commit(w2_empty(ws));
        }
        if (ok) tc::mma_commit(t_full(ab));
      }
      if (!ok) {
        if (!*abort) raise_status(p.status, DSPARK_ETIMEOUT);
        *abort = 1;
      }
      tc::mma_commit(drain);
      volatile int never = 0;
      tc::mbar_wait(drain, 0, &never);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // (launched as a dependent kernel, only the epilogue waits for the kernel
    // before: the producers stream W2 and U, inputs, meanwhile; the pick
    // that follows launches when this grid ends, which measured faster than
    // an early trigger)
    pdl_wait();
    const int ew = warp - 2, set = ew >> 2, q = warp & 3, m = q * 32 + lane;
    const int row = grp * kRpRows + m;
    const bool valid = row < p.n;
    const __nv_bfloat16* W1 = reinterpret_cast<const __nv_bfloat16*>(p.W1);
    auto aborted = [&]() { return __any_sync(0xFFFFFFFFu, *abort != 0); };
    int xs = -1;  // x*_k of this row (pass 0)
    float ld2 = 0.f, lt2 = 0.f;  // lse_d, lse_t in log2 units (pass 1)
    bool live = valid;           // RNN, PCTree: the row's request has a node to expand / is drafted
    const float* urow = nullptr;  // PCTree: U of the expanded node's depth
    if constexpr (MODE == kRowRnn) {
      // ---- A = o_k's hi and lo images: the copier brings them ready-made
    } else {
      // ---- A = the rows' W1 row: W1[x*_{k-1}] (loss; the anchor at k = 0)
      // or W1[token of the node to expand] (PCTree)
      int x = 0;
      if constexpr (MODE == kRowTree) {
        if (valid) {
          const int4 st = p.tree_state[row];
          const int node = min(max(st.y, 0), p.tree_N);
          const size_t nb = (size_t)row * (p.tree_N + 1) + node;
          const int d = p.tree_dep[nb];
          live = st.w == 0 && d >= 0 && d < p.g;
          x = live ? p.tree_tok[nb] : 0;
          if (x < 0 || x >= p.V) {
            raise_status(p.status, DSPARK_ERANGE);
            x = 0;
            live = false;
          }
          if (live) urow = p.U + ((size_t)row * p.g + d) * p.V;
        }
      } else if (valid) {
        const int b = row / p.g, k = row - b * p.g;
        x = k == 0 ? p.anchor[b] : p.xstar[(size_t)b * p.g + k - 1];
        xs = p.xstar[row];
        if (x < 0 || x >= p.V || xs < 0 || xs >= p.V) {
          raise_status(p.status, DSPARK_ERANGE);
          x = 0;
          xs = -1;
        }
        if (MODE == kRowLoss1) {
          ld2 = p.lse_d[row] * tc::kLog2e;
          lt2 = p.lse_t[row] * tc::kLog2e;
        }
      }
      uint4 v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int rl = 2 * i + set;
        const int xr = __shfl_sync(0xFFFFFFFFu, x, rl);
        const bool vr = __shfl_sync(0xFFFFFFFFu, valid, rl);
        v[i] = (vr && lane < p.r / 8) ? __ldg(reinterpret_cast<const uint4*>(W1 + (size_t)xr * p.r) + lane)
                                      : make_uint4(0, 0, 0, 0);
      }
      if (lane < p.r / 8) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                           sA + 2u * (uint32_t)rp_a_piece(q * 32 + 2 * i + set, lane >> 3, lane & 7)),
                       "r"(v[i].x), "r"(v[i].y), "r"(v[i].z), "r"(v[i].w)
                       : "memory");
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(a_full);
    }
    float Md = -INFINITY, Sd = 0.f, Mt = -INFINITY, St = 0.f, zxv = 0.f, l1 = 0.f;
    bool have_zx = false;
    for (int tj = 0; tj < ntl && !aborted(); ++tj) {
      const int nbt = tile_blocks(tj), ab = tj % NACC;
      const int gb0 = tj * kRpTileBlocks;
      const int j0 = (set - gb0 % kRpSets + kRpSets) % kRpSets;
      bool ok = tc::mbar_wait(t_full(ab), (tj / NACC) & 1, abort) &&
                (!kLoss || tc::mbar_wait(p_full(ab), (tj / NACC) & 1, abort));
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) {
        if (lane == 0 && !*abort) {
          raise_status(p.status, DSPARK_ETIMEOUT);
          *abort = 1;
        }
        break;
      }
      tc::tc_fence_after();
      for (int j = j0; j < nbt; j += kRpSets) {
        const int t = blo + gb0 + j;
        const uint32_t lanes = (uint32_t)(q * 32) << 16;
        if constexpr (!kLoss) {
          // RNN, PCTree: the block's log-mass (and maximum), from two halves
          float mb = -INFINITY, sb = 0.f;
#pragma unroll 1
          for (int hh = 0; hh < 2; ++hh) {
            const int v0 = t * kRpBlk + hh * 32;
            float z[32];
            float4 u4[8];
            if (MODE == kRowTree && live) {  // U of the node's depth, this row's 32 entries
#pragma unroll
              for (int e = 0; e < 8; ++e)
                u4[e] = v0 + 4 * e + 3 < p.V ? __ldg(reinterpret_cast<const float4*>(urow + v0) + e)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            tc::tmem_ld32(tmem + lanes + (uint32_t)(ab * kRpAccCols + j * kRpBlk + hh * 32), z);
            tc::tmem_wait_ld();
            if (!live) continue;
            if constexpr (MODE == kRowTree) {
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                z[4 * e] += u4[e].x;
                z[4 * e + 1] += u4[e].y;
                z[4 * e + 2] += u4[e].z;
                z[4 * e + 3] += u4[e].w;
              }
            }
            if (v0 + 32 > p.V) {
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (v0 + e >= p.V) z[e] = -INFINITY;
            }
            float mh, sh;
            half_ms(z, mh, sh);
            ms_merge(mb, sb, mh, sh);
          }
          if (live && t * kRpBlk < p.V) {
            p.blk[(size_t)row * p.nblk + t] = mb > -INFINITY ? mb + logf(sb) : -INFINITY;
            if (MODE == kRowTree) p.bmax[(size_t)row * p.nblk + t] = mb;
          }
          continue;
        }
        // the block in two halves of 32 columns (z_d from the accumulator, z_t
        // from the P buffer), which keeps 64 values live instead of 128
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          const int v0 = t * kRpBlk + hh * 32;
          float z[32], y[32];
          tc::tmem_ld32(tmem + lanes + (uint32_t)(ab * kRpAccCols + j * kRpBlk + hh * 32), z);
          tc::tmem_ld32(tmem + lanes + (uint32_t)(NACC * kRpAccCols + ab * kRpAccCols + j * kRpBlk + hh * 32), y);
          tc::tmem_wait_ld();
          if (!valid) continue;
          if (v0 + 32 > p.V) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (v0 + e >= p.V) {
                z[e] = -INFINITY;
                y[e] = -INFINITY;
              }
          }
          if (MODE == kRowLoss0) {
            float mb, sb;
            half_ms(z, mb, sb);
            ms_merge(Md, Sd, mb, sb);
            half_ms(y, mb, sb);
            ms_merge(Mt, St, mb, sb);
            if (xs >= v0 && xs < v0 + 32) {
              zxv = pick32(z, xs - v0);
              have_zx = true;
            }
          } else {
            // |p_d - p_t| = |2^(z log2e - lse_d log2e) - 2^(y log2e - lse_t log2e)|
            const unsigned long long l2e = tc::f2pack(tc::kLog2e, tc::kLog2e);
            const unsigned long long nd = tc::f2pack(-ld2, -ld2), nt = tc::f2pack(-lt2, -lt2);
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float a0, a1, c0, c1;
              tc::f2unpack(tc::fma2(tc::f2pack(z[2 * i], z[2 * i + 1]), l2e, nd), a0, a1);
              tc::f2unpack(tc::fma2(tc::f2pack(y[2 * i], y[2 * i + 1]), l2e, nt), c0, c1);
              s += fabsf(tc::ex2_ftz(a0) - tc::ex2_ftz(c0)) + fabsf(tc::ex2_ftz(a1) - tc::ex2_ftz(c1));
            }
            l1 += s;
          }
        }
      }
      // the accumulator and P buffer are free once every epilogue warp read the tile
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(t_empty(ab));
    }
    // ---- the two sets of a row meet; set 0 writes the CTA's partial
    if constexpr (kLoss) {
    asm volatile("bar.sync 1, %0;" ::"n"(kRpEpi) : "memory");
    if (set == 1) xchg[m] = MODE == kRowLoss0 ? make_float4(Md, Sd, Mt, St) : make_float4(l1, 0.f, 0.f, 0.f);
    if (MODE == kRowLoss0 && valid && have_zx && !*abort) p.zx[row] = zxv;
    asm volatile("bar.sync 1, %0;" ::"n"(kRpEpi) : "memory");
    if (set == 0 && valid && !*abort) {
      const float4 o = xchg[m];
      float4 w;
      if (MODE == kRowLoss0) {
        ms_merge(Md, Sd, o.x, o.y);
        ms_merge(Mt, St, o.z, o.w);
        w = make_float4(Md, Sd, Mt, St);
      } else {
        w = make_float4(l1 + o.x, 0.f, 0.f, 0.f);
      }
      // slot cg holds this CTA's partial; the slots no CTA of the group owns get neutral values
      for (int s = cg; s < p.G; s += Gg) {
        if (MODE == kRowLoss0)
          p.lpart[(size_t)row * p.G + s] = s == cg ? w : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
        else
          p.l1part[(size_t)row * p.G + s] = s == cg ? w.x : 0.f;
      }
    }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kRpTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

}  // namespace

bool rowpass_supported(const dspark_ws* ws, int n) {
  const dspark_dims& d = ws->d;
  if (!ws->use_tc || d.wdtype != DSPARK_BF16) return false;
  if (d.r % 64 != 0 || d.r > 256 || d.V % 8 != 0 || n < 1) return false;
  const int nG = (n + kRpRows - 1) / kRpRows;
  if (nG > kRpMaxGroups || nG > ws->geo.num_sms) return false;
  if ((d.V + kRpBlk - 1) / kRpBlk < (ws->geo.num_sms + nG - 1) / nG) return false;  // a CTA per block at least
  return encode_fn() != nullptr;
}

namespace {

cudaError_t rowpass_configure() {
  static bool configured = false;
  if (configured) return cudaSuccess;
  const int mx = (int)(RpSmem::make(256).total + 1024);  // the largest operand (r = 256)
  cudaError_t e = cudaFuncSetAttribute(k_rowpass<kRowLoss0>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_rowpass<kRowLoss1>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_rowpass<kRowRnn>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_rowpass<kRowTree>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  if (e == cudaSuccess) configured = true;
  return e;
}

cudaError_t w2_map(const dspark_dims& d, const void* W2, CUtensorMap* tm) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)d.V, (cuuint64_t)d.r};
  const cuuint64_t strides[1] = {(cuuint64_t)d.V * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kRpBlk, (cuuint32_t)kRpKc};
  const cuuint32_t es[2] = {1, 1};
  if (enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W2), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

RpParams base_params(const dspark_ws* ws, int n) {
  RpParams p;
  memset(&p, 0, sizeof(p));
  p.n = n;
  p.g = ws->d.gamma;
  p.V = ws->d.V;
  p.r = ws->d.r;
  p.nblk = ws->geo.nblk;
  p.nG = (n + kRpRows - 1) / kRpRows;
  p.G = ws->geo.num_sms;
  p.status = ws->s.status;
  return p;
}

}  // namespace

cudaError_t launch_rnn_blocks_rowpass(const dspark_ws* ws, const float* U, const void* W2, const float* ovec,
                                      const __nv_bfloat16* oimg, int k, cudaStream_t st) {
  const dspark_dims& d = ws->d;
  cudaError_t e = rowpass_configure();
  CUtensorMap tm_w2, tm_u;
  if (e == cudaSuccess) e = w2_map(d, W2, &tm_w2);
  if (e != cudaSuccess) return e;
  {
    // U as (V, gamma, B): the rows of one step are a 3-D box
    const cuuint64_t dims[3] = {(cuuint64_t)d.V, (cuuint64_t)d.gamma, (cuuint64_t)d.B};
    const cuuint64_t strides[2] = {(cuuint64_t)d.V * 4, (cuuint64_t)d.gamma * d.V * 4};
    const cuuint32_t box[3] = {32, 1, (cuuint32_t)kRpRows};
    const cuuint32_t es[3] = {1, 1, 1};
    if (encode_fn()(&tm_u, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(U), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  RpParams p = base_params(ws, d.B);
  p.step = k;
  p.ovec = ovec;
  p.oimg = oimg;
  p.blk = ws->s.blk;
  const size_t smem = RpSmem::make(d.r).total + 1024;
  const cudaError_t el = launch_ex(k_rowpass<kRowRnn>, dim3(p.G), dim3(kRpThreads), smem, st, true, tm_w2, tm_u,
                                   tm_u, p);
  return el != cudaSuccess ? el : cudaGetLastError();
}

cudaError_t launch_tree_blocks_rowpass(const dspark_ws* ws, const float* U, const void* W1, const void* W2,
                                       const int32_t* tok, const int32_t* dep, const int4* state, int N, float* blk,
                                       float* bmax, cudaStream_t st) {
  const dspark_dims& d = ws->d;
  cudaError_t e = rowpass_configure();
  CUtensorMap tm_w2;
  if (e == cudaSuccess) e = w2_map(d, W2, &tm_w2);
  if (e != cudaSuccess) return e;
  RpParams p = base_params(ws, d.B);
  p.W1 = W1;
  p.U = U;
  p.tree_tok = tok;
  p.tree_dep = dep;
  p.tree_state = state;
  p.tree_N = N;
  p.blk = blk;
  p.bmax = bmax;
  const size_t smem = RpSmem::make(d.r).total + 1024;
  // a dependent launch: only the epilogue reads what the pick before wrote
  const cudaError_t el = launch_ex(k_rowpass<kRowTree>, dim3(p.G), dim3(kRpThreads), smem, st, true, tm_w2, tm_w2,
                                   tm_w2, p);
  if (el != cudaSuccess) return el;
  return cudaGetLastError();
}

cudaError_t launch_loss_rowpass(const dspark_ws* ws, const LossArgs& a, int pass, cudaStream_t st) {
  const dspark_dims& d = ws->d;
  const size_t smem = RpSmem::make(d.r).total + 1024;
  cudaError_t e0 = rowpass_configure();
  if (e0 != cudaSuccess) return e0;
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const int n = d.B * d.gamma;
  CUtensorMap tm_w2, tm_u, tm_p;
  e0 = w2_map(d, a.W2, &tm_w2);
  if (e0 != cudaSuccess) return e0;
  for (int w = 0; w < 2; ++w) {
    // U and P as [n positions][V] fp32
    const cuuint64_t dims[2] = {(cuuint64_t)d.V, (cuuint64_t)n};
    const cuuint64_t strides[1] = {(cuuint64_t)d.V * 4};
    const cuuint32_t box[2] = {32, (cuuint32_t)kRpRows};
    const cuuint32_t es[2] = {1, 1};
    if (enc(w == 0 ? &tm_u : &tm_p, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(w == 0 ? a.U : a.P),
            dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  RpParams p = base_params(ws, n);
  p.anchor = a.anchor;
  p.xstar = a.xstar;
  p.W1 = a.W1;
  p.lse_d = a.lse_d;
  p.lse_t = a.lse_t;
  p.lpart = a.lpart;
  p.zx = a.zx;
  p.l1part = a.l1part;
  if (pass == 0)
    k_rowpass<kRowLoss0><<<p.G, kRpThreads, smem, st>>>(tm_w2, tm_u, tm_p, p);
  else
    k_rowpass<kRowLoss1><<<p.G, kRpThreads, smem, st>>>(tm_w2, tm_u, tm_p, p);
  return cudaGetLastError();
}

}  // namespace dspark
