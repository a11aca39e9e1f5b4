// k_draft_tc.cu -- persistent tcgen05 Markov-head draft kernel (sm_103a).
//
// "DeepSeek-V4.1 模型结构（6）：解码，DSpark", eq. (4)/(5) and the sequential
// loop of section "Markov head": for k = 1..gamma,
//   z_k = U_k + W1[x_{k-1}] W2,  x_k ~ softmax(z_k),  x_0 = anchor,
// and eq. (7): c_k = sigma((w^T [h_k; W1[x_{k-1}]]) / T_k) (the temperature is
// the STS sigmoid(raw / T) of the zdszero.github.io "spec_dspark" page).
//
// One cooperative launch, k_draft_tc, runs all gamma steps. Each CTA (one per
// SM) owns a contiguous range of 64-token sampler blocks of one 128-row group,
// taken two at a time as MMA tiles:
//   warp 0      TMA producer of W2, in chunks of 64 K rows x 128 tokens (two
//               128-byte-swizzled boxes; L2 evict_last: W2 is reused by every
//               step), into a ring of 6 stages;
//   warp 10     TMA producer of U, one block [128 x 64] fp32 at a time
//               (evict_first: streamed once), into a ring of 2 stages (two
//               producers, so that neither stream waits behind the other);
//   warp 1      allocates all 512 TMEM columns and issues tcgen05.mma with
//               M = 128 rows, N = 64 x (blocks of the tile), K = r in steps of
//               16, into one of four 128-column accumulators, so the MMA can
//               run up to three tiles ahead; A = the rows W1[x_{k-1}] in shared
//               memory. Each accumulator starts as the tile's U blocks, copied
//               from shared memory by tcgen05.cp, so a U stage is free as soon
//               as that copy lands and z = U + A W2 comes out of TMEM. (The
//               tensor core takes about as long per instruction for N = 64 as
//               for N = 128, hence two blocks per tile.)
//   warps 2-9   epilogue, two sets of four warps (one per TMEM lane quarter);
//               set s takes the blocks gb with gb % 2 == s, one thread per row:
//               z = TMEM, the block's log-mass (max, sum exp), the block
//               draw key log mass + G_s, the row's online log-sum-exp, and a
//               register copy of z for the set's best block so far.
// Step boundary. The block draw is a grid-wide argmax of the block keys:
// per row, each CTA publishes its best (block key, block) with a 64-bit
// atomic max into the row's winner word, and the thread holding that block
// parks its z in shared memory; all CTAs meet at a grid barrier. Only then is
// the token inside the block drawn (the token level of the two-level sampler,
// argmax_v (z_v + G_v) over the block's 64 tokens with exact Gumbel keys), by
// the one CTA that owns the winning block, one warp per row it owns; it
// writes the token and its z beside the winner word, and a second grid
// barrier makes every token of the step final. (Drawing every CTA's
// candidate token before a single barrier costs each CTA the draw of all its
// rows, of which it wins about 1 in G.) In every CTA of the group the
// epilogue warps then read the 128 rows' tokens and gather W1[x_k] straight
// into the swizzled A operand in shared memory (the anchors' rows at step 1).
// The producers keep prefetching the next step's tiles meanwhile (they do not
// depend on the drafted token). Log-sum-exps, probabilities of the drawn
// tokens and confidences are off that chain: per-set partials (max, sum exp)
// are kept per step and combined after the last step, one warp per (row,
// step), which also forms the confidence logit w^T [h_k; W1[x_{k-1}]] from h
// and W1.
//
// Every wait is bounded (tc_ptx.cuh); a timeout sets DSPARK_ETIMEOUT, every
// role leaves its loop, in-flight copies and MMAs are drained, TMEM is freed.
#include <cudaTypedefs.h>
#include <stdio.h>
#include <string.h>

#include "dspark_common.cuh"
#include "dspark_internal.h"
#include "tc_ptx.cuh"

namespace dspark {

constexpr int kSets = 2;            // epilogue sets of four warps (one warp per TMEM lane quarter)
constexpr int kEpiThreads = kSets * 128;  // warps 2 .. 2 + 4 * kSets - 1
constexpr int kUWarp = 2 + 4 * kSets;     // U producer (TMA)
constexpr int kCWarp = kUWarp + 1;        // U copier (shared memory -> accumulator)
constexpr int kTcThreads = 32 * (kCWarp + 1);
constexpr int kTcRows = 128;        // MMA M: rows of one row group
constexpr int kBlk = 64;            // sampler block = one 64-column slice of the accumulator
constexpr int kTileBlocks = 2;      // MMA N = 64 x blocks of the tile
constexpr int kKc = 64;             // K rows of W2 per ring stage
constexpr int kW2Box = kKc * 128;   // 8 KB: 64 K rows x 64 tokens (128-byte rows)
constexpr int kW2Stage = kTileBlocks * kW2Box;  // 16 KB
constexpr int kNW = 6;              // W2 ring depth (K chunks): a tile and a half
constexpr int kNU = 2;              // U ring depth (blocks)
constexpr int kUStage = kTcRows * kBlk * 4;  // 32 KB: two 128 x 32 fp32 boxes
constexpr int kUBox = kTcRows * 32 * 4;      // 16 KB
constexpr int kAccCols = kTileBlocks * kBlk; // 128 columns per accumulator
constexpr int kNAcc = 4;                     // accumulators: the MMA runs up to three tiles ahead
// U blocks of step k + 1 the producer may load before the tokens of step k are
// final: more would keep HBM busy across the step boundary, but they queue
// ahead of the boundary's latency-bound traffic (barrier atomics, W1 rows).
constexpr int kUEarly = 6;
constexpr int kTmemCols = kNAcc * kAccCols;  // all of TMEM
constexpr int kMaxGroups = 8;       // B <= 1024
constexpr int kMaxPartLanes = 16;   // partials per lane in the finalize (kSets per CTA)
constexpr int kHChunk = 32 * 8;      // float4 of h per warp task of the hidden pass (eight per lane in flight)
// Winner words are kWinPad words apart (one 128-byte line per row), so that
// the CTAs' atomic maxima on different rows do not queue on shared lines.
constexpr int kWinPad = 16;

static_assert(kBlk == kBlockW, "an accumulator slice is one sampler block");
static_assert(kSets == 2, "the A gather splits a lane quarter's rows into even and odd");

struct TcSmem {  // byte offsets into dynamic shared memory (1024-aligned base)
  uint32_t a, w2, u, bars, misc, total;
  __host__ __device__ static TcSmem make(int r) {
    TcSmem s;
    s.a = 0;
    // the A operand; between the last tile of a step and the next gather it
    // holds every epilogue thread's best block of z (64 fp32 each)
    s.w2 = s.a + max(kTcRows * r * 2, kEpiThreads * kBlk * 4);
    s.u = s.w2 + kNW * kW2Stage;
    s.bars = s.u + kNU * kUStage;
    // w2 full/empty, u full, u empty, t full/empty, a_full, drain, acc_u
    // (accumulator holds U), the copier's drain, u_go
    s.misc = s.bars + 8 * (2 * kNW + 2 * kNU + 2 * kNAcc + 2 + kNAcc + 2);
    // misc: TMEM address and abort word (64 B), then the step-end exchange of
    // each set's best block per row: key [kSets][128] fp32, block [kSets][128] u16
    s.total = s.misc + 64 + kEpiThreads * 4 + kEpiThreads * 2;
    return s;
  }
};

struct TcParams {
  int B, g, V, r, H;
  int nblk, nG, G, Ggmax, P, rowsG;
  Rng rng;
  const int32_t* anchor;
  const void* W1;
  const float* w;
  const float* T;
  const float* h;           // [B*g][H] hidden states (the hidden half of each confidence logit)
  int32_t* tokens;
  float* pd_tok;
  float* lse;
  float* conf;
  float2* dpart;            // [g][rowsG][P]: (max, sum exp) of a row's blocks per CTA and set
  float* hpart;             // [B*g][nhc]: w_h . h over chunks of kHChunk float4 (H % 4 == 0)
  unsigned long long* win;  // [2][g][rowsG] x kWinPad: packed (block key, token), 0 = none
  unsigned* bar;            // [2] launches (parity of win and counters), [4 + parity] grid-barrier arrivals
  int* status;
};

__device__ __forceinline__ int group_ctas(int G, int nG, int g) { return (G - g + nG - 1) / nG; }

// (block key, block) as one unsigned 64-bit word whose unsigned order is:
// larger key first, then the smaller block. Never 0.
__device__ __forceinline__ unsigned long long pack_win(float key, int x) {
  uint32_t u = __float_as_uint(key);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)x);
}
__device__ __forceinline__ int win_block(unsigned long long w) {
  return (int)(0xFFFFFFFFu - (uint32_t)(w & 0xFFFFFFFFull));
}

// Offset (in bf16 elements) of the 16-byte piece ch of K-block kb of row m in
// the A operand: K-major, 128-byte swizzle, 8-row atoms of 1 KB, K-blocks of
// 64 elements 16 KB apart.
__device__ __forceinline__ size_t a_piece(int m, int kb, int ch) {
  return (size_t)kb * (kTcRows * 64) + (m >> 3) * 512 + (m & 7) * 64 + ((ch ^ (m & 7)) << 3);
}

// The set whose best block is this CTA's candidate for row m (larger key,
// then the smaller block), from the step-end exchange in shared memory.
__device__ __forceinline__ int cta_best_set(const float* keyx, const uint16_t* blkx, int m) {
  const float kA = keyx[m], kB = keyx[kTcRows + m];
  return (kB > kA || (kB == kA && blkx[kTcRows + m] < blkx[m])) ? 1 : 0;
}

// The token word beside a row's winner word: (z of the token) << 32 | token + 1,
// 0 while no token is written. Returns the token, -1 if none.
__device__ __forceinline__ int drawn_token(unsigned long long w) { return (int)(uint32_t)(w & 0xFFFFFFFFull) - 1; }

// Grid barrier among the epilogue warps (named barrier 1) of all CTAs: the
// leader of each CTA adds one to this launch's arrival counter (release) and
// waits (acquire) until it reaches `target` = G x (barriers so far). The
// counter only grows within a launch; the other launch parity's counter is
// cleared at the start of each launch. Returns false if the round is being
// abandoned.
__device__ bool grid_sync(const TcParams& p, unsigned* ctr, unsigned target, bool leader, volatile int* abort) {
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
  if (leader && !*abort) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
    const unsigned long long t0 = tc::globaltimer();
    while (tc::ld_acquire_gpu(ctr) < target) {
      if (*(volatile int*)p.status != 0) {
        *abort = 1;
        break;
      }
      if (tc::globaltimer() - t0 > tc::kWaitNs) {
        raise_status(p.status, DSPARK_ETIMEOUT);
        *abort = 1;
        break;
      }
    }
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
  return !*abort;
}

__global__ void __launch_bounds__(kTcThreads, 1)
    k_draft_tc(const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_u,
               const TcParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the runtime aligns dynamic shared memory to at least 16 B; round up to 1 KB
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const TcSmem L = TcSmem::make(p.r);
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t sA = sbase + L.a, sW2 = sbase + L.w2, sU = sbase + L.u;
  const uint32_t bars = sbase + L.bars;
  auto w2_full = [&](int i) { return bars + 8u * i; };
  auto w2_empty = [&](int i) { return bars + 8u * (kNW + i); };
  auto u_full = [&](int gb) { return bars + 8u * (2 * kNW + gb % kNU); };
  auto u_empty = [&](int i) { return bars + 8u * (2 * kNW + kNU + i); };
  auto t_full = [&](int i) { return bars + 8u * (2 * kNW + 2 * kNU + i); };
  auto t_empty = [&](int i) { return bars + 8u * (2 * kNW + 2 * kNU + kNAcc + i); };
  const uint32_t a_full = bars + 8u * (2 * kNW + 2 * kNU + 2 * kNAcc);
  const uint32_t drain = a_full + 8u;
  auto acc_u = [&](int i) { return a_full + 16u + 8u * i; };
  const uint32_t drain_c = a_full + 16u + 8u * kNAcc;
  const uint32_t u_go = drain_c + 8u;  // completes once per step: that step's tokens are final
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L.misc + 16);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int grp = c % p.nG, cg = c / p.nG;  // row group, index within the group
  const int Gg = group_ctas(p.G, p.nG, grp);
  // this CTA's sampler blocks [blo, blo + nbc), in MMA tiles of up to four
  const int blo = (int)((long long)cg * p.nblk / Gg);
  const int nbc = (int)((long long)(cg + 1) * p.nblk / Gg) - blo;
  const int ntl = (nbc + kTileBlocks - 1) / kTileBlocks;
  const int nkc = p.r / kKc;  // W2 chunks per tile
  auto tile_blocks = [&](int tj) { return min(kTileBlocks, nbc - tj * kTileBlocks); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNW; ++i) {
      tc::mbar_init(w2_full(i), 1);
      tc::mbar_init(w2_empty(i), 1);
    }
    for (int i = 0; i < kNU; ++i) {
      tc::mbar_init(u_full(i), 1);
      tc::mbar_init(u_empty(i), 1);
    }
    for (int i = 0; i < kNAcc; ++i) {
      tc::mbar_init(t_full(i), 1);
      tc::mbar_init(t_empty(i), kEpiThreads / 32);
    }
    tc::mbar_init(a_full, kEpiThreads / 32);
    tc::mbar_init(drain, 1);
    for (int i = 0; i < kNAcc; ++i) tc::mbar_init(acc_u(i), 1);
    tc::mbar_init(drain_c, 1);
    tc::mbar_init(u_go, 1);
    *abort = 0;
    tc::fence_barrier_init();
    tc::prefetch_tmap(&tm_w2);
    tc::prefetch_tmap(&tm_u);
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(tmem_holder), kTmemCols);
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
      int wiss = 0;  // chunks issued
      bool ok = true;
      for (int k = 1; k <= p.g && ok; ++k) {
        for (int tj = 0; tj < ntl && ok; ++tj) {
          const int it = (k - 1) * ntl + tj, nbt = tile_blocks(tj);
          const int v0 = (blo + tj * kTileBlocks) * kBlk;
          for (int ch = 0; ch < nkc && ok; ++ch) {
            const int wc = it * nkc + ch, ws = wc % kNW;
            ok = tc::mbar_wait(w2_empty(ws), ((wc / kNW) & 1) ^ 1, abort);
            if (!ok) break;
            tc::mbar_arrive_expect_tx(w2_full(ws), (uint32_t)(nbt * kW2Box));
            for (int j = 0; j < nbt; ++j)
              tc::tma_load_2d(sW2 + ws * kW2Stage + j * kW2Box, &tm_w2, v0 + j * kBlk, ch * kKc, w2_full(ws), keep);
            wiss = wc + 1;
          }
        }
      }
      if (!ok) {
        if (!*abort) raise_status(p.status, DSPARK_ETIMEOUT);
        *abort = 1;
        volatile int never = 0;  // let the copies already issued land before the CTA can exit
        for (int wc = wiss - 1; wc >= 0 && wc >= wiss - kNW; --wc)
          tc::mbar_wait(w2_full(wc % kNW), (wc / kNW) & 1, &never);
      }
    }
  } else if (warp == kUWarp) {
    // ------------------------------------------------------------ U producer
    if (lane == 0) {
      const uint64_t stream = tc::policy_evict_first();
      int uiss = 0;  // blocks issued
      bool ok = true;
      for (int k = 1; k <= p.g && ok; ++k) {
        for (int i = 0; i < nbc && ok; ++i) {
          const int gb = (k - 1) * nbc + i, us = gb % kNU, v = (blo + i) * kBlk;
          if (k > 1 && i == kUEarly) ok = tc::mbar_wait(u_go, (k - 2) & 1, abort);
          if (!ok) break;
          ok = tc::mbar_wait(u_empty(us), ((gb / kNU) & 1) ^ 1, abort);
          if (!ok) break;
          tc::mbar_arrive_expect_tx(u_full(gb), kUStage);
          tc::tma_load_3d(sU + us * kUStage, &tm_u, v, k - 1, grp * kTcRows, u_full(gb), stream);
          tc::tma_load_3d(sU + us * kUStage + kUBox, &tm_u, v + 32, k - 1, grp * kTcRows, u_full(gb), stream);
          uiss = gb + 1;
        }
      }
      if (!ok) {
        if (!*abort) raise_status(p.status, DSPARK_ETIMEOUT);
        *abort = 1;
        volatile int never = 0;
        for (int gb = uiss - 1; gb >= 0 && gb >= uiss - kNU; --gb)
          tc::mbar_wait(u_full(gb), (gb / kNU) & 1, &never);
      }
    }
  } else if (warp == kCWarp) {
    // ------------------------------------------------------------ U copier
    // Each accumulator starts as the tile's U blocks ([128 x 64] fp32, two
    // 128-byte-swizzled boxes of 32 columns each), copied into its columns by
    // tcgen05.cp once the epilogue has released it. The copier's commits track
    // only its own copies, so a U stage is free as soon as they land, not
    // when the MMA queue drains.
    if (lane == 0) {
      bool ok = true;
      for (int k = 1; k <= p.g && ok; ++k) {
        for (int tj = 0; tj < ntl && ok; ++tj) {
          const int it = (k - 1) * ntl + tj, ab = it % kNAcc, nbt = tile_blocks(tj);
          const uint32_t d = tmem + (uint32_t)(ab * kAccCols);
          ok = tc::mbar_wait(t_empty(ab), ((it / kNAcc) & 1) ^ 1, abort);
          for (int j = 0; j < nbt && ok; ++j) {
            const int gb = (k - 1) * nbc + tj * kTileBlocks + j, us = gb % kNU;
            ok = tc::mbar_wait(u_full(gb), (gb / kNU) & 1, abort);
            if (!ok) break;
            tc::tc_fence_after();
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int cc = 0; cc < 4; ++cc)
                tc::cp_128x256b(d + (uint32_t)(j * kBlk + h * 32 + cc * 8),
                                tc::smem_desc(sU + us * kUStage + h * kUBox + cc * 32, 16, 1024));
            tc::mma_commit(u_empty(us));
          }
          if (ok) tc::mma_commit(acc_u(ab));
        }
      }
      if (!ok) {
        if (!*abort) raise_status(p.status, DSPARK_ETIMEOUT);
        *abort = 1;
      }
      // every copy this thread issued completes before TMEM is freed
      tc::mma_commit(drain_c);
      volatile int never = 0;
      tc::mbar_wait(drain_c, 0, &never);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      for (int k = 1; k <= p.g && ok; ++k) {
        ok = tc::mbar_wait(a_full, (k - 1) & 1, abort);
        if (!ok) break;
        tc::tc_fence_after();
        for (int tj = 0; tj < ntl && ok; ++tj) {
          const int it = (k - 1) * ntl + tj, ab = it % kNAcc, nbt = tile_blocks(tj);
          const uint32_t idesc = tc::idesc_bf16_f32(kTcRows, nbt * kBlk, true);
          const uint32_t d = tmem + (uint32_t)(ab * kAccCols);
          // the copier has filled the (free) accumulator with the tile's U
          ok = tc::mbar_wait(acc_u(ab), (it / kNAcc) & 1, abort);
          if (ok) tc::tc_fence_after();
          for (int ch = 0; ch < nkc && ok; ++ch) {
            const int wc = it * nkc + ch, ws = wc % kNW;
            ok = tc::mbar_wait(w2_full(ws), (wc / kNW) & 1, abort);
            if (!ok) break;
            tc::tc_fence_after();
            for (int kk = 0; kk < kKc / 16; ++kk) {
              // A: K-major, 128-byte swizzle; K-block ks / 4 is [128 rows x
              // 128 B], the 16-wide K step moves 32 B inside the swizzled row.
              const int ks = ch * (kKc / 16) + kk;
              const uint64_t ad = tc::smem_desc(sA + (ks >> 2) * (kTcRows * 128) + (ks & 3) * 32, 16, 1024);
              // B: N-major (W2 rows are contiguous in N), 128-byte swizzle;
              // 8 K rows of 128 B form a 1 KB atom, 16 K rows per step, the
              // 64-token boxes of the chunk are 4 KB apart.
              const uint64_t bd = tc::smem_desc(sW2 + ws * kW2Stage + kk * 2048, kW2Box, 1024);
              tc::mma_bf16(d, ad, bd, idesc, 1u);
            }
            tc::mma_commit(w2_empty(ws));
          }
          if (ok) tc::mma_commit(t_full(ab));
        }
      }
      if (!ok) {
        if (!*abort) raise_status(p.status, DSPARK_ETIMEOUT);
        *abort = 1;
      }
      // every MMA this thread issued completes before TMEM is freed
      tc::mma_commit(drain);
      volatile int never = 0;
      tc::mbar_wait(drain, 0, &never);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Every epilogue warp runs all gamma steps and every grid barrier even
    // after an abort (the named barrier inside grid_sync has no timeout, so no
    // warp may skip one); an abort only skips the work.
    const int ew = warp - 2;     // 0 .. 4 * kSets - 1
    const int set = ew >> 2;     // this warp takes the blocks gb with gb % kSets == set
    const int q = warp & 3;      // TMEM lane quarter this warp may access
    const int m = q * 32 + lane;
    const int b = grp * kTcRows + m;
    const bool valid = b < p.B;
    const bool leader = warp == 2 && lane == 0;
    const __nv_bfloat16* W1 = reinterpret_cast<const __nv_bfloat16*>(p.W1);
    // warp-uniform view of the abort word (the loops below hold warp collectives)
    auto aborted = [&]() { return __any_sync(0xFFFFFFFFu, *abort != 0); };
    // this launch's half of the winner and flag slots; the other half, last
    // used by the previous launch, is cleared for the next one
    const int par = (int)(__ldcg(p.bar + 2) & 1u);
    unsigned* gctr = p.bar + 4 + par;
    const size_t half = (size_t)p.g * p.rowsG;
    unsigned long long* win = p.win + par * half * kWinPad;
    {
      const int et = threadIdx.x - 64;
      if (c == 0 && et == 0) p.bar[4 + (par ^ 1)] = 0u;
      for (size_t i = (size_t)c * kEpiThreads + et; i < half; i += (size_t)p.G * kEpiThreads) {
        p.win[((par ^ 1) * half + i) * kWinPad] = 0ull;
        p.win[((par ^ 1) * half + i) * kWinPad + 1] = 0ull;
      }
    }
    for (int k = 1; k <= p.g; ++k) {
      // ---- A = W1[x_{k-1}], gathered by the epilogue warps into the swizzled
      // operand. x_0 is the anchor; x_{k-1} is the token of the row's winning
      // word of step k-1, final since that step's grid barrier. Every MMA of
      // step k-1 has completed (this warp waited for all of its tiles), so the
      // operand is free.
      if (!aborted()) {
        int x = 0;
        if (valid) {
          if (k == 1) {
            x = p.anchor[b];
          } else {
            x = drawn_token(__ldcg(win + ((size_t)(k - 2) * p.rowsG + b) * kWinPad + 1));
          }
          if (x < 0 || x >= p.V) {
            if (k == 1) {
              raise_status(p.status, DSPARK_ERANGE);  // reported; the row drafts from token 0
            } else {
              raise_status(p.status, DSPARK_ENUMERIC);  // no block with finite mass
              *abort = 1;
            }
            x = 0;
          }
        }
        // coalesced: the warp copies one row at a time (lane l takes the
        // 16-byte piece l of the row); the two sets' warps of a lane quarter
        // take its even and odd rows
        uint4 v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int rl = 2 * i + set;  // row (lane) within the quarter
          const int xr = __shfl_sync(0xFFFFFFFFu, x, rl);
          const bool vr = __shfl_sync(0xFFFFFFFFu, valid, rl);
          v[i] = (vr && lane < p.r / 8) ? __ldg(reinterpret_cast<const uint4*>(W1 + (size_t)xr * p.r) + lane)
                                        : make_uint4(0, 0, 0, 0);
        }
        if (lane < p.r / 8) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                             sA + 2u * (uint32_t)a_piece(q * 32 + 2 * i + set, lane >> 3, lane & 7)),
                         "r"(v[i].x), "r"(v[i].y), "r"(v[i].z), "r"(v[i].w)
                         : "memory");
        }
        tc::fence_proxy_async_smem();  // read by tcgen05.mma
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(a_full);
      }

      // ---- this CTA's tiles; set s takes the blocks whose running index gb
      // has gb % kSets == s (so the sets share the tiles and the U ring evenly)
      float M = -INFINITY, S = 0.f, bk = -INFINITY;
      int bs = kNoIdx;
      float zb[kBlk];  // z of this set's best block so far
#pragma unroll
      for (int e = 0; e < kBlk; ++e) zb[e] = 0.f;
      // G_s of the set's next block, drawn one block ahead so that the Philox
      // rounds and logarithms interleave with the current block's exponentials
      const int tlast = blo + nbc - 1;
      float g_next = gumbel(p.rng.word(kDraftBlock, b, k, min(blo + (set - ((k - 1) * nbc) % kSets + kSets) % kSets, tlast)));
      for (int tj = 0; tj < ntl && !aborted(); ++tj) {
        const int it = (k - 1) * ntl + tj, ab = it % kNAcc, nbt = tile_blocks(tj);
        const int gb0 = (k - 1) * nbc + tj * kTileBlocks;
        const int j0 = (set - gb0 % kSets + kSets) % kSets;  // first block of this set in the tile
        const int jl = j0 + (nbt - 1 - j0) / kSets * kSets;  // last one (j0 >= nbt: none)
        bool ok = tc::mbar_wait(t_full(ab), (it / kNAcc) & 1, abort);
        ok = __all_sync(0xFFFFFFFFu, ok);  // tcgen05.ld below is warp-collective
        if (!ok) {
          if (lane == 0 && !*abort) {
            raise_status(p.status, DSPARK_ETIMEOUT);
            *abort = 1;
          }
          break;
        }
        tc::tc_fence_after();
        if (j0 >= nbt) {  // no block of this set in the tile
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(t_empty(ab));
          continue;
        }
        for (int j = j0; j < nbt; j += kSets) {
          const int t = blo + tj * kTileBlocks + j;
          float z[kBlk];  // U + W1[x_{k-1}] W2: the accumulator started as U
          const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(ab * kAccCols + j * kBlk);
          tc::tmem_ld32(ta, z);
          tc::tmem_ld32(ta + 32, z + 32);
          tc::tmem_wait_ld();
          if (j == jl) {  // the accumulator is free once the last slice of this set is read
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(t_empty(ab));
          }
          const float g_cur = g_next;
          g_next = gumbel(p.rng.word(kDraftBlock, b, k, min(t + kSets, tlast)));
          if (valid) {
            const int v0 = t * kBlk;
            if (v0 + kBlk > p.V) {
#pragma unroll
              for (int e = 0; e < kBlk; ++e)
                if (v0 + e >= p.V) z[e] = -INFINITY;
            }
            // block max (three-input max, 8 chains) and sum of exponentials
            // e^(z - mb) = 2^(z log2e - mb log2e) on fp32 pairs (FFMA2, MUFU
            // ex2, FADD2 into 4 pair accumulators)
            float m8[8];
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
              m8[c8] = tc::max3f(z[8 * c8], z[8 * c8 + 1], z[8 * c8 + 2]);
              m8[c8] = tc::max3f(m8[c8], z[8 * c8 + 3], z[8 * c8 + 4]);
              m8[c8] = tc::max3f(m8[c8], z[8 * c8 + 5], z[8 * c8 + 6]);
              m8[c8] = fmaxf(m8[c8], z[8 * c8 + 7]);
            }
            const float mb = tc::max3f(tc::max3f(m8[0], m8[1], m8[2]), tc::max3f(m8[3], m8[4], m8[5]),
                                       fmaxf(m8[6], m8[7]));
            const unsigned long long l2e = tc::f2pack(tc::kLog2e, tc::kLog2e);
            const unsigned long long nml = tc::f2pack(-mb * tc::kLog2e, -mb * tc::kLog2e);
            unsigned long long acc[2];
#pragma unroll
            for (int i = 0; i < kBlk / 2; ++i) {
              float a0, a1;
              tc::f2unpack(tc::fma2(tc::f2pack(z[2 * i], z[2 * i + 1]), l2e, nml), a0, a1);
              const unsigned long long e2 = tc::f2pack(tc::ex2_ftz(a0), tc::ex2_ftz(a1));
              acc[i & 1] = i < 2 ? e2 : tc::add2(acc[i & 1], e2);
            }
            float sl, sh;
            tc::f2unpack(tc::add2(acc[0], acc[1]), sl, sh);
            const float sb = sl + sh;
            const float lm = mb + logf(sb);
            if (mb > M) {
              S = S * __expf(M - mb) + sb;
              M = mb;
            } else {
              S += sb * __expf(mb - M);
            }
            const float key = lm + g_cur;
            if (key > bk) {  // this set sees its blocks in increasing order: ties keep the first
              bk = key;
              bs = t;
#pragma unroll
              for (int e = 0; e < kBlk; ++e) zb[e] = z[e];
            }
          }
        }
      }

      // ---- step end. Every MMA of this step has completed once both sets
      // are here (each waited for all of its tiles), so the A operand is free
      // until the next gather.
      // (1) Per row, this CTA's candidate is the better of the two sets' best
      // blocks (larger key, then the smaller block). Its (block key, block)
      // goes into the row's winner word by atomic max, and the thread that
      // holds it parks the block's z in the A region.
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
      const bool cand = valid && bs != kNoIdx && !*abort;
      float* keyx = reinterpret_cast<float*>(smem + L.misc + 64);
      uint16_t* blkx = reinterpret_cast<uint16_t*>(smem + L.misc + 64 + kEpiThreads * 4);
      unsigned* own = reinterpret_cast<unsigned*>(smem + L.misc + 32);  // [4] rows whose token this CTA draws
      keyx[set * kTcRows + m] = cand ? bk : -INFINITY;
      blkx[set * kTcRows + m] = (uint16_t)(cand ? bs : 0xFFFF);
      if (ew == 0 && lane < kTcRows / 32) own[lane] = 0u;
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
      const bool mine = cand && set == cta_best_set(keyx, blkx, m);
      if (mine) {
        unsigned long long* wrow = win + ((size_t)(k - 1) * p.rowsG + b) * kWinPad;
        float4* zs = reinterpret_cast<float4*>(smem + L.a) + (size_t)m * (kBlk / 4);
#pragma unroll
        for (int c4 = 0; c4 < kBlk / 4; ++c4)  // chunk swizzle: a quarter-warp's stores hit distinct banks
          zs[c4 ^ (m & 7)] = make_float4(zb[4 * c4], zb[4 * c4 + 1], zb[4 * c4 + 2], zb[4 * c4 + 3]);
        atomicMax(wrow, pack_win(bk, bs));
      }
      // every set writes its slot every step (a set without blocks writes the
      // neutral partial), so no entry of an earlier launch is combined
      if (valid && !*abort)
        p.dpart[((size_t)(k - 1) * p.rowsG + b) * p.P + kSets * cg + set] = make_float2(M, S);
      // (2) the winner words of step k are final once every CTA has passed here
      grid_sync(p, gctr, (unsigned)(p.G * (2 * k - 1)), leader, abort);
      if (mine && !*abort && win_block(__ldcg(win + ((size_t)(k - 1) * p.rowsG + b) * kWinPad)) == bs)
        atomicOr(own + (m >> 5), 1u << (m & 31));
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
      // (3) the token inside the winning block, drawn by the CTA that owns the
      // block: one warp per owned row, two tokens per lane, exact keys
      // z_v + G_v with G_v from the draft-token stream at (b, k, v); the token
      // and its z go into the second word of the row's winner line
      if (!aborted()) {
        for (int rr = ew; rr < kTcRows; rr += 4 * kSets) {
          if (!((own[rr >> 5] >> (rr & 31)) & 1u)) continue;  // the same smem word for the whole warp
          const int br = grp * kTcRows + rr;
          const int v0 = (int)blkx[cta_best_set(keyx, blkx, rr) * kTcRows + rr] * kBlk;
          const float4 zz = reinterpret_cast<const float4*>(smem + L.a)[(size_t)rr * (kBlk / 4) + ((lane >> 1) ^ (rr & 7))];
          const int i0 = 2 * lane;  // tokens i0 and i0 + 1 of the block: half of chunk lane / 2
          const float za = (lane & 1) ? zz.z : zz.x, zb1 = (lane & 1) ? zz.w : zz.y;
          const uint4 o = p.rng.block4(kDraftToken, br, k, v0 + i0);
          const uint32_t ua = (lane & 1) ? o.z : o.x, ub = (lane & 1) ? o.w : o.y;
          KeyIdx kb = better(KeyIdx{za + gumbel(ua), i0}, KeyIdx{zb1 + gumbel(ub), i0 + 1});
          kb = warp_best(kb);
          const int src = kb.idx >> 1;
          const float zsel = __shfl_sync(0xFFFFFFFFu, (kb.idx & 1) ? zb1 : za, src);
          if (lane == 0) {
            if (!(kb.key > -INFINITY)) {
              raise_status(p.status, DSPARK_ENUMERIC);  // no finite logit in the block
              *abort = 1;
            } else {
              const int x = v0 + kb.idx;
              __stcg(win + ((size_t)(k - 1) * p.rowsG + br) * kWinPad + 1,
                     ((unsigned long long)__float_as_uint(zsel) << 32) | (unsigned long long)(uint32_t)(x + 1));
              // every CTA gathers this row after the next barrier: bring it into L2 now
              const char* w1row = reinterpret_cast<const char*>(W1 + (size_t)x * p.r);
              tc::bulk_prefetch_l2(w1row, (uint32_t)(p.r * 2));
            }
          }
        }
      }
      // the hidden halves of the confidence logits, w_h . h_k for every row
      // and step, do not depend on the draws: before the last barrier every
      // warp sums whole chunks of h (eight 16-byte loads per lane in flight)
      // into per-chunk partials, which the combine below adds in order
      if (k == p.g && (p.H & 3) == 0 && p.H > 0 && !aborted()) {
        const int nq = p.H / 4, nhc = (nq + kHChunk - 1) / kHChunk;
        const int ntask = p.B * p.g * nhc, nw = p.G * (kEpiThreads / 32);
        const float4* w4 = reinterpret_cast<const float4*>(p.w);
        for (int ti = c * (kEpiThreads / 32) + ew; ti < ntask; ti += nw) {
          const int it = ti / nhc, ch = ti - it * nhc;
          const float4* h4 = reinterpret_cast<const float4*>(p.h + (size_t)it * p.H);
          float4 a[8], b4[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int i = ch * kHChunk + 32 * u + lane;
            a[u] = i < nq ? __ldcs(h4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);  // h is read once
            b4[u] = i < nq ? __ldg(w4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
          float hs = 0.f;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            hs = fmaf(a[u].x, b4[u].x, hs);
            hs = fmaf(a[u].y, b4[u].y, hs);
            hs = fmaf(a[u].z, b4[u].z, hs);
            hs = fmaf(a[u].w, b4[u].w, hs);
          }
          hs = warp_sum(hs);
          if (lane == 0) p.hpart[ti] = hs;
        }
      }
      // (4) the step's tokens are final once every CTA has passed here
      grid_sync(p, gctr, (unsigned)(p.G * 2 * k), leader, abort);
      if (leader) tc::mbar_arrive(u_go);  // the U producer may run ahead into step k + 1
    }

    // ---- after the last step: per (row, step), one warp combines the
    // partials into the log-sum-exp, the drawn token's probability, and the
    // confidence c_k from W1[x_{k-1}]
    pdl_trigger();  // the planner may be scheduled while this tail runs
    if (!aborted()) {
      const int nw = p.G * (kEpiThreads / 32);
      for (int pi = c * (kEpiThreads / 32) + ew; pi < p.B * p.g; pi += nw) {
        const int br = pi / p.g, kk = pi - br * p.g;  // step kk + 1
        const int Pr = kSets * group_ctas(p.G, p.nG, br / kTcRows);
        const float Tk = __ldg(p.T + kk);
        const unsigned long long tw = __ldcg(win + ((size_t)kk * p.rowsG + br) * kWinPad + 1);
        int xp = kk == 0 ? p.anchor[br] : drawn_token(__ldcg(win + ((size_t)(kk - 1) * p.rowsG + br) * kWinPad + 1));
        const int x = drawn_token(tw);
        if (x < 0 || x >= p.V) {
          if (lane == 0) raise_status(p.status, DSPARK_ENUMERIC);
          continue;
        }
        const float zx = __uint_as_float((uint32_t)(tw >> 32));
        if (xp < 0 || xp >= p.V) xp = 0;  // an anchor out of range was reported at the step-1 gather
        const float2* pr = p.dpart + ((size_t)kk * p.rowsG + br) * p.P;
        float2 dd[kMaxPartLanes];
#pragma unroll
        for (int u = 0; u < kMaxPartLanes; ++u) {
          const int i = lane + 32 * u;
          dd[u] = i < Pr ? __ldcg(pr + i) : make_float2(-INFINITY, 0.f);
        }
        // w^T [h_k; W1[x_{k-1}]]: the hidden half from the chunk partials
        // (lane j holds chunk j, chunks beyond 32 folded in order) or, when
        // H % 4 != 0, from h directly; then the W1 half
        float cd = 0.f;
        const float* hr = p.h + ((size_t)br * p.g + kk) * p.H;
        if ((p.H & 3) == 0) {
          const int nhc = (p.H / 4 + kHChunk - 1) / kHChunk;
          for (int j = lane; j < nhc; j += 32) cd += __ldcg(p.hpart + (size_t)pi * nhc + j);
        } else {
          for (int i = lane; i < p.H; i += 32) cd = fmaf(__ldcs(hr + i), __ldg(p.w + i), cd);
        }
        for (int ci = lane; ci < p.r / 8; ci += 32) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(W1 + (size_t)xp * p.r) + ci);
          const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v);
          const float* wr = p.w + p.H + ci * 8;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h2[e]);
            cd = fmaf(f.x, wr[2 * e], cd);
            cd = fmaf(f.y, wr[2 * e + 1], cd);
          }
        }
        // this lane's partials: the largest max first, then the scaled sums
        // (independent exponentials rather than a chain of pairwise combines)
        float mx = -INFINITY;
#pragma unroll
        for (int u = 0; u < kMaxPartLanes; ++u) mx = fmaxf(mx, dd[u].x);
        float sx = 0.f;
        if (mx > -INFINITY) {
#pragma unroll
          for (int u = 0; u < kMaxPartLanes; ++u)
            if (dd[u].x > -INFINITY) sx += dd[u].y * __expf(dd[u].x - mx);
        }
        MS ms = warp_ms(MS{mx, sx});
        cd = warp_sum(cd);
        if (lane == 0) {
          const size_t o = (size_t)br * p.g + kk;
          const float L2 = ms_log(ms);
          p.tokens[o] = x;
          p.pd_tok[o] = expf(zx - L2);
          p.lse[o] = L2;
          const float cf = 1.f / (1.f + expf(-cd / Tk));
          if (!isfinite(cf)) raise_status(p.status, DSPARK_ENUMERIC);
          p.conf[o] = cf;
        }
      }
    }
    // the launch count picks the slots' half; every CTA read it before the
    // first grid barrier
    if (leader && c == 0) atomicAdd(p.bar + 2, 1u);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
namespace {

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

int draft_tc_supported(const dspark_dims& d) {
  if (d.wdtype != DSPARK_BF16) return 0;
  if (d.r % 64 != 0 || d.r > 256) return 0;
  if (d.V % 8 != 0) return 0;
  if (d.B > kTcRows * kMaxGroups) return 0;
  if ((d.V + kBlk - 1) / kBlk > 65535) return 0;  // block indices are exchanged as 16-bit words
  return 1;
}

cudaError_t draft_tc_configure(dspark_ws* ws) {
  const dspark_dims& d = ws->d;
  const TcSmem L = TcSmem::make(d.r);
  const size_t smem = L.total + 1024;
  cudaError_t e = cudaFuncSetAttribute(k_draft_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_draft_tc, kTcThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  int coop = 0;
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, ws->device);
  if (!coop || !encode_fn()) return cudaErrorNotSupported;
  ws->geo.tc_groups = (d.B + kTcRows - 1) / kTcRows;
  ws->geo.tc_grid = ws->geo.num_sms;  // one CTA per SM, all co-resident
  if (ws->geo.tc_grid < ws->geo.tc_groups) return cudaErrorInvalidConfiguration;
  // the finalize holds a row's partials (two per CTA of its group) in registers
  const int Ggmax = (ws->geo.tc_grid + ws->geo.tc_groups - 1) / ws->geo.tc_groups;
  if (kSets * Ggmax > 32 * kMaxPartLanes) return cudaErrorInvalidConfiguration;
  return cudaSuccess;
}

size_t draft_tc_partials(const dspark_dims& d, int grid) {
  const int nG = (d.B + kTcRows - 1) / kTcRows;
  const int Ggmax = (grid + nG - 1) / nG;
  return (size_t)d.gamma * nG * kTcRows * kSets * Ggmax;
}

size_t draft_tc_hidden_partials(const dspark_dims& d) {
  const int nq = d.H / 4;
  return (size_t)d.B * d.gamma * (size_t)((nq + kHChunk - 1) / kHChunk + 1);
}

size_t draft_tc_winners(const dspark_dims& d) {
  const int nG = (d.B + kTcRows - 1) / kTcRows;
  return (size_t)2 * d.gamma * nG * kTcRows * kWinPad;
}

cudaError_t launch_draft_tc(const dspark_ws* ws, const DraftArgs& a, cudaStream_t st, int* launches) {
  const dspark_dims& d = ws->d;
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap tm_w2, tm_u;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)d.V, (cuuint64_t)d.r};
    const cuuint64_t strides[1] = {(cuuint64_t)d.V * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBlk, (cuuint32_t)kKc};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&tm_w2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.W2), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)d.V, (cuuint64_t)d.gamma, (cuuint64_t)d.B};
    const cuuint64_t strides[2] = {(cuuint64_t)d.V * 4, (cuuint64_t)d.gamma * d.V * 4};
    const cuuint32_t box[3] = {32, 1, (cuuint32_t)kTcRows};
    const cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tm_u, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(a.U), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.B = d.B;
  p.g = d.gamma;
  p.V = d.V;
  p.r = d.r;
  p.H = d.H;
  p.nblk = ws->geo.nblk;
  p.nG = ws->geo.tc_groups;
  p.G = ws->geo.tc_grid;
  p.Ggmax = (p.G + p.nG - 1) / p.nG;
  p.P = kSets * p.Ggmax;
  p.rowsG = p.nG * kTcRows;
  p.rng = Rng::make(a.seed, a.round, (uint32_t)ws->b0);
  p.anchor = a.anchor;
  p.W1 = a.W1;
  p.w = a.w;
  p.T = a.T;
  p.h = a.h;
  p.tokens = a.tokens;
  p.pd_tok = a.pd_tok;
  p.lse = a.lse;
  p.conf = a.conf;
  p.dpart = ws->s.dpart;
  p.hpart = ws->s.hpart;
  p.win = ws->s.dwin;
  p.bar = ws->s.barrier;
  p.status = ws->s.status;

  const TcSmem L = TcSmem::make(d.r);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = L.total + 1024;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k_draft_tc, tm_w2, tm_u, p);
  ++*launches;
  return e;
}

}  // namespace dspark
