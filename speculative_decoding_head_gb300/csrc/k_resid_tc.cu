// k_resid_tc.cu -- residual block draw on tcgen05 (sm_103a).
//
// After the first rejection n of request b, the next anchor is drawn from
// norm(max(0, p_t - p_d)) ("DeepSeek-V4.1 模型结构（6）：解码，DSpark",
// derivation box; "DSpark：不让大模型更聪明，而让它「吐字更快」" §02), with
//   p_t(v) = exp(P[row, v] - lse_t)   (row = the rejected target row),
//   p_d(v) = exp(U[b, n, v] + W1[x_n] . W2[:, v] - lse_d)   (draft position n+1),
// recomputed rather than stored. This kernel makes the block draw of the
// two-level sampler: for each 64-token block s the residual mass
// W_s = sum_v max(0, p_t(v) - p_d(v)) and the key log W_s + G_s; the token
// draw inside the winning block is k_resid_pick's.
//
// Orientation: D[v, i] = sum_k W2[k, v] W1[x_i, k] with M = 128 vocabulary
// entries (A = W2 tile, N-major in memory, 128-byte swizzle, two 64-wide
// boxes) and N = 32 rejected requests (B = gathered W1 rows, K-major). A
// producer warp stages, per tile, each request's 512-byte slices of U and P in
// shared memory with bulk copies (a three-stage ring), so each epilogue thread
// owns one vocabulary entry and reads U and P of every request from shared
// memory; a block's mass is a sum over two warps' lanes (a 31-shuffle
// transpose-reduce per 32 requests, then shared memory). Requests are taken in
// groups of 32 (the list of rejected requests is compacted in each CTA from
// the verify flags); more groups re-read W2, which the draft left in L2.
// Persistent, one CTA per SM over 128-wide vocabulary tiles; W2 is read with
// the L2 evict_last policy (the draft kept it there), in K-halves through a
// three-stage ring; U and P with plain bulk copies. Every wait is bounded.
//
// The same vocabulary pass serves three other computations (template MODE),
// each with every position or request as an MMA column:
//   - the draft head's teacher-forced training objective (eqs. (9)-(12) of the
//     deepseek.csdn.net reading, §6): pass kModeLossStats keeps per thread a
//     running (max, sum 2^(y - max)) of z_d and of z_t per column and reduces
//     it once per column group; pass kModeLossL1 sums |p_d - p_t|. A group's
//     U and P rows are consecutive, so they arrive as two TMA boxes; the tiles
//     are walked in alternating directions per group so that W2 is reused
//     from L2;
//   - one draft step of the RNN head (eq. (6), same reading §4.2),
//     kModeDraft: z = U_k + o_k W2 with o_k split into bf16 hi and lo
//     operands that both accumulate into the tile, and the log-mass of every
//     64-token block for the SIMT pick;
//   - the residual block draw of a round drafted by the RNN head,
//     kModeResidRnn: kModeResid with p_d from U + o_{n+1} W2, the head vector
//     of the rejected position as the hi and lo operands of kModeDraft (its
//     U/P ring is two tiles deep so that both operands fit beside it).
#include <cudaTypedefs.h>
#include <string.h>

#include "dspark_common.cuh"
#include "dspark_internal.h"
#include "tc_ptx.cuh"

namespace dspark {

namespace {

constexpr int kRThreads = 352;   // warp 0 W2 TMA, warp 1 MMA, warps 2-9 epilogue, warp 10 U/P bulk copies
constexpr int kREpi = 8;
constexpr int kRUPWarp = 10;
constexpr int kRM = 128;          // vocabulary entries per tile (MMA M)
constexpr int kRN = 32;           // requests per group (MMA N)
constexpr int kRNW = 3;           // W2 ring depth in K-halves of a tile (1.5 tiles)
constexpr int kRUP = 3;           // U/P ring depth (tiles)
constexpr int kRUPStage = kRN * 2 * kRM * 4;  // 32 KB: per request a 512-byte slice of U and of P
constexpr int kRTmemCols = 64;    // two 32-column accumulators
static_assert(kRN == 32, "one 32-request chunk per tile, 16 requests for each warp of a TMEM lane quarter");
constexpr int kRGMax = 16;        // block Gumbels of a group kept in shared memory (blocks per CTA)
constexpr int kRMaxB = 1024;
constexpr int kRGather = kRN * (256 / 8) / (32 * 8);  // 16-byte W1 chunks per epilogue thread (r <= 256)

// What a launch computes over its columns (MMA N): the residual block draw of
// the rejected requests, or one of the two passes of the draft head's
// teacher-forced training objective over every position (b, k).
constexpr int kModeResid = 0;      // per block: residual mass and Gumbel key; the best block per CTA
constexpr int kModeLossStats = 1;  // per column: (max, sum exp) of z_d and of z_t over the CTA's tiles, z_d at x*
constexpr int kModeLossL1 = 2;     // per column: sum |p_d - p_t| over the CTA's tiles
constexpr int kModeDraft = 3;      // per column (request) and 64-token block: log sum exp z of one draft step
                                   // of the RNN head, z = U_k + o_k W2 with o_k split into bf16 hi + lo parts
constexpr int kModeTree = 4;       // per column (request) and 64-token block: log sum exp z and max z of the
                                   // expansion of a PCTree node, z = U[b, depth] + W1[token] W2
constexpr int kModeResidRnn = 5;   // kModeResid with the RNN head's o_{n+1} (hi + lo) in place of W1[x_n]

// the residual block draw (either head); B as bf16 hi + lo parts of an fp32
// vector; U/P ring depth
__host__ __device__ constexpr bool mode_resid(int m) { return m == kModeResid || m == kModeResidRnn; }
__host__ __device__ constexpr bool mode_hilo(int m) { return m == kModeDraft || m == kModeResidRnn; }
__host__ __device__ constexpr int mode_up(int m) { return m == kModeResidRnn ? 2 : kRUP; }

struct RSmem {
  uint32_t bop, w2, up, stage, col, part, best, gum, list, bars, misc, total;
  __host__ __device__ static RSmem make(int r, int mode) {
    RSmem s;
    s.bop = 0;                              // [32 columns x r] bf16, K-major swizzled (hi + lo modes: hi, then lo)
    s.w2 = s.bop + (mode_hilo(mode) ? 2 : 1) * kRN * r * 2;  // kRNW x (two boxes of [r/2 x 64] bf16: a K-half)
    s.up = s.w2 + kRNW * r * 128;           // mode_up x [request][U slice | P slice] fp32 (draft: U rows only)
    s.stage = mode == kModeDraft ? kRN * kRM * 4 : kRUPStage;
    s.col = s.up + mode_up(mode) * s.stage;  // per-request: b, n, row, x (int), lse_d, lse_t (float)
    s.part = s.col + 6 * 4 * kRN;           // [4 quarters][32 columns] partials (float4 for the loss statistics)
    s.best = s.part + 4 * 16 * kRN;         // [128] best key, [128] best block
    s.gum = s.best + 2 * 4 * kRN;           // [kRN][kRGMax] block Gumbels of this CTA's blocks
    s.list = s.gum + 4 * kRN * kRGMax;      // [kRMaxB] rejected requests
    s.bars = s.list + 4 * kRMaxB;
    s.misc = s.bars + 8 * (2 * kRNW + 4 + 2 + 2 * kRUP);
    s.total = s.misc + 64;
    return s;
  }
};

struct RParams {
  int B, g, V, r;
  int ntiles, G;
  Rng rng;
  const float* P;
  const float* U;
  const void* W1;
  const int32_t* anchor;
  const int32_t* tokens;
  const float* lse;
  const int* vflag;
  const int32_t* n_acc;
  const int* vrow;
  const float* vlset;
  float2* rpart;  // [B][G] (key, block) of each CTA
  int* status;
  // the training objective's passes: column i = b * g + k (teacher-forced)
  const int32_t* xstar;  // [B][g] the reference tokens x*
  float4* lpart;         // [B*g][G] (max, sum exp) of z_d, then of z_t, over the CTA's tiles
  float* zx;             // [B*g] z_d at x*
  float* l1part;         // [B*g][G] sum |p_d - p_t| over the CTA's tiles
  const float* lse_d;    // [B*g]
  const float* lse_t;    // [B*g]
  // one draft step of the RNN head: column b takes o_k of request b
  const float* ovec;     // [B][g][r] fp32
  int step;              // k (1-based)
  float* blk;            // [B][nblk] block log-masses
  int nblk;
  // one expansion step of PCTree: column b expands node state[b].y of its tree
  const int32_t* tree_tok;  // [B][N+1] node tokens
  const int32_t* tree_dep;  // [B][N+1] node depths
  const int4* tree_state;   // [B] (nodes admitted, node to expand, frontier size, done)
  int tree_N;
  float* bmax;              // [B][nblk] block maxima of z
};

// Sum over the 32 lanes of 16 per-lane values: afterwards lane L holds the
// sum of every lane's a[L & 15]. Each step keeps the half whose index bit
// matches the lane's bit and adds the partner's other half (four steps over
// the lanes that share bit 4), then the two half-warps are added.
__device__ __forceinline__ float transpose_sum16(float (&a)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int k = 0; k < o; ++k) {
      const float send = upper ? a[k] : a[k + o];
      const float keep = upper ? a[k + o] : a[k];
      a[k] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
    }
  }
  return a[0] + __shfl_xor_sync(0xFFFFFFFFu, a[0], 16);
}

// The same transpose over 32 lanes with a maximum instead of a sum.
__device__ __forceinline__ float transpose_max16(float (&a)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int k = 0; k < o; ++k) {
      const float send = upper ? a[k] : a[k + o];
      const float keep = upper ? a[k + o] : a[k];
      a[k] = fmaxf(keep, __shfl_xor_sync(0xFFFFFFFFu, send, o));
    }
  }
  return fmaxf(a[0], __shfl_xor_sync(0xFFFFFFFFu, a[0], 16));
}

constexpr float kNegBig = -1e30f;  // "no entry yet" of a running maximum (finite: no inf - inf)
constexpr float kLn2 = 0.693147180559945309f;

// y joins a running (m, s = sum 2^(y_i - m)) pair: one ex2 per entry.
__device__ __forceinline__ void online_add(float& m, float& s, float y) {
  const float d = y - m;
  const float e = tc::ex2_ftz(-fabsf(d));
  s = d > 0.f ? fmaf(s, e, 1.f) : s + e;
  m = fmaxf(m, y);
}

// Two (m, s) pairs in base 2 combined.
__device__ __forceinline__ float2 ms2_combine(float2 a, float2 b) {
  const float m = fmaxf(a.x, b.x);
  return make_float2(m, fmaf(a.y, tc::ex2_ftz(a.x - m), b.y * tc::ex2_ftz(b.x - m)));
}

// The transpose of transpose_sum16 over (m, s) pairs: afterwards lane L holds
// the combination of every lane's pair L & 15.
__device__ __forceinline__ float2 transpose_ms16(float (&m)[16], float (&s)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int k = 0; k < o; ++k) {
      const float sm = upper ? m[k] : m[k + o], ss = upper ? s[k] : s[k + o];
      const float km = upper ? m[k + o] : m[k], ks = upper ? s[k + o] : s[k];
      const float2 r = ms2_combine(make_float2(km, ks), make_float2(__shfl_xor_sync(0xFFFFFFFFu, sm, o),
                                                                   __shfl_xor_sync(0xFFFFFFFFu, ss, o)));
      m[k] = r.x;
      s[k] = r.y;
    }
  }
  return ms2_combine(make_float2(m[0], s[0]),
                     make_float2(__shfl_xor_sync(0xFFFFFFFFu, m[0], 16), __shfl_xor_sync(0xFFFFFFFFu, s[0], 16)));
}

template <int MODE>
__global__ void __launch_bounds__(kRThreads, 1)
    k_resid_tc(const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_u,
               const __grid_constant__ CUtensorMap tm_p, const RParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr bool kRes = mode_resid(MODE);
  constexpr int kUP = mode_up(MODE);
  const RSmem L = RSmem::make(p.r, MODE);
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t sB = sbase + L.bop, sW2 = sbase + L.w2;
  int* col_b = reinterpret_cast<int*>(smem + L.col);
  int* col_n = col_b + kRN;
  int* col_row = col_n + kRN;
  int* col_x = col_row + kRN;                                 // the row of W1 gathered into B
  float* col_nld = reinterpret_cast<float*>(col_x + kRN);    // -lse_d log2(e)
  float* col_nlt = col_nld + kRN;                              // -lse_t log2(e)
  float* part = reinterpret_cast<float*>(smem + L.part);   // [4][128]
  float* best_key = reinterpret_cast<float*>(smem + L.best);
  int* best_blk = reinterpret_cast<int*>(best_key + kRN);
  int* list = reinterpret_cast<int*>(smem + L.list);
  float* gsm = reinterpret_cast<float*>(smem + L.gum);
  const uint32_t bars = sbase + L.bars;
  auto w2_full = [&](int i) { return bars + 8u * i; };
  auto w2_empty = [&](int i) { return bars + 8u * (kRNW + i); };
  auto t_full = [&](int i) { return bars + 8u * (2 * kRNW + i); };
  auto t_empty = [&](int i) { return bars + 8u * (2 * kRNW + 2 + i); };
  const uint32_t a_full = bars + 8u * (2 * kRNW + 4);
  const uint32_t drain = a_full + 8u;
  auto up_full = [&](int i) { return drain + 8u * (1 + i); };
  auto up_empty = [&](int i) { return drain + 8u * (1 + kRUP + i); };
  const uint32_t sUP = sbase + L.up;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L.misc + 16);
  int* s_nrej = reinterpret_cast<int*>(smem + L.misc + 32);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int tile_lo = (int)((long long)c * p.ntiles / p.G);
  const int tile_hi = (int)((long long)(c + 1) * p.ntiles / p.G);
  const int nt = tile_hi - tile_lo;
  // The loss modes walk the CTA's tiles forwards in even groups and backwards
  // in odd ones, so the W2 tiles used last are the first reused (from L2).
  auto tile_of = [&](int gq, int i) { return tile_lo + ((!kRes && (gq & 1)) ? nt - 1 - i : i); };
  const uint32_t box_bytes = (uint32_t)p.r * 64u;  // one [r/2 x 64] bf16 box
  const uint32_t w2_bytes = 2u * box_bytes;         // one K-half of a tile

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRNW; ++i) {
      tc::mbar_init(w2_full(i), 1);
      tc::mbar_init(w2_empty(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(t_full(i), 1);
      tc::mbar_init(t_empty(i), kREpi);
    }
    tc::mbar_init(a_full, kREpi);
    tc::mbar_init(drain, 1);
    for (int i = 0; i < kUP; ++i) {
      tc::mbar_init(up_full(i), 1);
      tc::mbar_init(up_empty(i), kREpi);  // every epilogue warp reads the stage
    }
    *abort = 0;
    tc::fence_barrier_init();
    tc::prefetch_tmap(&tm_w2);
    if constexpr (!kRes) {
      tc::prefetch_tmap(&tm_u);
      tc::prefetch_tmap(&tm_p);
    }
  }
  // W2 is an input: the first ring stages of the first group's tiles are
  // filled before the wait on the previous kernel (thread 0, which initialised
  // the barriers, is the W2 producer)
  const int npre = min(kRNW, 2 * nt);
  if (threadIdx.x == 0) {
    const uint64_t keep = tc::policy_evict_last();
    for (int hs = 0; hs < npre; ++hs) {
      const int t = tile_of(0, hs >> 1), h = hs & 1;
      tc::mbar_arrive_expect_tx(w2_full(hs), w2_bytes);
      tc::tma_load_2d(sW2 + hs * w2_bytes, &tm_w2, t * kRM, h * (p.r / 2), w2_full(hs), keep);
      tc::tma_load_2d(sW2 + hs * w2_bytes + box_bytes, &tm_w2, t * kRM + 64, h * (p.r / 2), w2_full(hs), keep);
    }
  }
  // the rejected requests, in request order (every CTA builds the same list).
  // The flags, positions and rows are this round's only if every stage so far
  // left the status clear: an error leaves the list empty.
  pdl_wait();  // the verify flags are the sweep's
  if (warp == 2) {
    if constexpr (kRes) {
      const bool clear = __shfl_sync(0xFFFFFFFFu, *(volatile int*)p.status, 0) == 0;
      int base = 0;
      for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int b = b0 + lane;
        const bool f = clear && b < p.B && p.vflag[b] != 0;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, f);
        if (f) list[base + __popc(m & ((1u << lane) - 1u))] = b;
        base += __popc(m);
      }
      if (lane == 0) *s_nrej = base;
    } else if constexpr (MODE == kModeDraft || MODE == kModeTree) {
      if (lane == 0) *s_nrej = p.B;  // every request is a column
    } else {
      if (lane == 0) *s_nrej = p.B * p.g;  // every position is a column
    }
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(tmem_holder), kRTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int nrej = *s_nrej;
  const int ngroups = (nrej + kRN - 1) / kRN;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (W2 tiles)
    if (lane == 0 && ngroups == 0) {  // nothing to do: the stages filled before the wait land first
      for (int hs = 0; hs < npre; ++hs) {
        volatile int never = 0;
        tc::mbar_wait(w2_full(hs), 0, &never);
      }
    }
    if (lane == 0 && ngroups > 0) {
      const uint64_t keep = tc::policy_evict_last();
      int issued = npre;
      bool ok = true;
      for (int gq = 0; gq < ngroups && ok; ++gq) {
        for (int i = 0; i < nt && ok; ++i) {
          const int t = tile_of(gq, i);
          for (int h = 0; h < 2 && ok; ++h) {
            const int hs = 2 * (gq * nt + i) + h, ws = hs % kRNW;
            if (hs < npre) continue;  // filled before the wait
            ok = tc::mbar_wait(w2_empty(ws), ((hs / kRNW) & 1) ^ 1, abort);
            if (!ok) break;
            tc::mbar_arrive_expect_tx(w2_full(ws), w2_bytes);
            tc::tma_load_2d(sW2 + ws * w2_bytes, &tm_w2, t * kRM, h * (p.r / 2), w2_full(ws), keep);
            tc::tma_load_2d(sW2 + ws * w2_bytes + box_bytes, &tm_w2, t * kRM + 64, h * (p.r / 2), w2_full(ws), keep);
            issued = hs + 1;
          }
        }
      }
      if (!ok) {
        if (!*abort) raise_status(p.status, DSPARK_ETIMEOUT);
        *abort = 1;
        for (int it = issued - 1; it >= 0 && it >= issued - kRNW; --it) {
          volatile int never = 0;
          tc::mbar_wait(w2_full(it % kRNW), (it / kRNW) & 1, &never);
        }
      }
    }
  } else if (warp == kRUPWarp) {
    // ------------------------------------------------------------ U/P producer
    // per tile, lane i copies request i's 512-byte slices of U (row n, the
    // draft position that was rejected) and of P (its target row) with two
    // bulk copies, so the epilogue reads them from shared memory
    bool ok = true;
    int issued = 0;
    const uint64_t stream_pol = tc::policy_evict_first();
    for (int gq = 0; gq < ngroups && ok; ++gq) {
      const int ncols = min(kRN, nrej - gq * kRN);
      const float* urow = p.U;
      const float* prow = p.P;
      if (lane < ncols) {
        if constexpr (kRes) {
          const int b = list[gq * kRN + lane];
          urow = p.U + ((size_t)b * p.g + min(max(p.n_acc[b], 0), p.g - 1)) * p.V;
          prow = p.P + (size_t)min(max(p.vrow[b], 0), p.B * (p.g + 1) - 1) * p.V;
        } else if constexpr (MODE == kModeTree) {  // U of the expanded node's depth
          const int b = gq * kRN + lane;
          const int node = min(max(p.tree_state[b].y, 0), p.tree_N);
          const int d = min(max(p.tree_dep[(size_t)b * (p.tree_N + 1) + node], 0), p.g - 1);
          urow = p.U + ((size_t)b * p.g + d) * p.V;
        } else {  // position i of the objective: U row i, target logits row i
          urow = p.U + (size_t)(gq * kRN + lane) * p.V;
          prow = p.P + (size_t)(gq * kRN + lane) * p.V;
        }
      }
      for (int i = 0; i < nt && ok; ++i) {
        const int it = gq * nt + i, us = it % kUP, v0 = tile_of(gq, i) * kRM;
        const uint32_t bytes = (uint32_t)min(kRM, p.V - v0) * 4u;  // a multiple of 32 (V % 8 == 0)
        int got = 1;
        if (lane == 0) got = tc::mbar_wait(up_empty(us), ((it / kUP) & 1) ^ 1, abort) ? 1 : 0;
        ok = __shfl_sync(0xFFFFFFFFu, got, 0) != 0;
        if (!ok) break;
        if constexpr (kRes) {
          if (lane == 0) tc::mbar_arrive_expect_tx(up_full(us), 2u * bytes * (uint32_t)ncols);
          __syncwarp();
          if (lane < ncols) {
            const uint32_t dst = sUP + us * L.stage + lane * (2 * kRM * 4);
            tc::bulk_load(dst, urow + v0, bytes, up_full(us));
            tc::bulk_load(dst + kRM * 4, prow + v0, bytes, up_full(us));
          }
        } else if constexpr (MODE == kModeTree) {  // the residual's layout, U slices only
          if (lane == 0) tc::mbar_arrive_expect_tx(up_full(us), bytes * (uint32_t)ncols);
          __syncwarp();
          if (lane < ncols) tc::bulk_load(sUP + us * L.stage + lane * (2 * kRM * 4), urow + v0, bytes, up_full(us));
        } else if (MODE == kModeDraft && lane == 0) {
          // U_k of the group's 32 requests: one [32 x 128] box of the
          // tensor map whose rows are the requests (stride gamma V)
          tc::mbar_arrive_expect_tx(up_full(us), (uint32_t)(kRN * kRM * 4));
          tc::tma_load_2d(sUP + us * L.stage, &tm_u, v0, gq * kRN, up_full(us), stream_pol);
        } else if (MODE != kModeDraft && lane == 0) {
          // the group's 32 consecutive rows of U and of P: one [32 x 128] box
          // each (rows past B*gamma and entries past V read as zeros)
          tc::mbar_arrive_expect_tx(up_full(us), (uint32_t)kRUPStage);
          const uint32_t dst = sUP + us * L.stage;
          tc::tma_load_2d(dst, &tm_u, v0, gq * kRN, up_full(us), stream_pol);
          tc::tma_load_2d(dst + kRN * kRM * 4, &tm_p, v0, gq * kRN, up_full(us), stream_pol);
        }
        issued = it + 1;
      }
    }
    if (!ok && lane == 0) {
      if (!*abort) raise_status(p.status, DSPARK_ETIMEOUT);
      *abort = 1;
      volatile int never = 0;  // let the copies already issued land before the CTA can exit
      for (int it = issued - 1; it >= 0 && it >= issued - kUP; --it)
        tc::mbar_wait(up_full(it % kUP), (it / kUP) & 1, &never);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && ngroups > 0) {
      // A = W2 tile, M-major (vocabulary contiguous); B = W1 rows, K-major
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | ((uint32_t)(kRN >> 3) << 17) |
                             ((uint32_t)(kRM >> 4) << 24);
      bool ok = true;
      for (int gq = 0; gq < ngroups && ok; ++gq) {
        ok = tc::mbar_wait(a_full, gq & 1, abort);
        if (!ok) break;
        tc::tc_fence_after();
        for (int i = 0; i < nt && ok; ++i) {
          const int it = gq * nt + i, ab = it & 1;
          ok = tc::mbar_wait(t_empty(ab), ((it >> 1) & 1) ^ 1, abort);
          const uint32_t d = tmem + (uint32_t)(ab * kRN);
          for (int h = 0; h < 2 && ok; ++h) {
            const int hs = 2 * it + h, ws = hs % kRNW;
            ok = tc::mbar_wait(w2_full(ws), (hs / kRNW) & 1, abort);
            if (!ok) break;
            tc::tc_fence_after();
            const uint32_t astage = sW2 + ws * w2_bytes;
            for (int kh = 0; kh < p.r / 32; ++kh) {
              const int ks = h * (p.r / 32) + kh;
              // A: two 64-wide M atoms (LBO apart), 8 K rows per 1 KB atom (SBO)
              const uint64_t ad = tc::smem_desc(astage + kh * 2048, box_bytes, 1024);
              const uint32_t boff = (ks >> 2) * (kRN * 128) + (ks & 3) * 32;
              tc::mma_bf16(d, ad, tc::smem_desc(sB + boff, 16, 1024), idesc, ks > 0 ? 1u : 0u);
              if constexpr (mode_hilo(MODE))  // the lo part of o_k against the same W2 rows
                tc::mma_bf16(d, ad, tc::smem_desc(sB + kRN * p.r * 2 + boff, 16, 1024), idesc, 1u);
            }
            tc::mma_commit(w2_empty(ws));
          }
          if (!ok) break;
          tc::mma_commit(t_full(ab));
        }
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
    // All eight warps run every group and every named barrier of every tile;
    // an abort only skips work. Warps w and w + 4 share a TMEM lane quarter and
    // split its 32-request chunks between them.
    const int q = warp & 3;         // TMEM lane quarter = vocabulary entries 32q..32q+31
    const int half = (warp - 2) >> 2;
    const int et = threadIdx.x - 64;  // 0..255
    auto aborted = [&]() { return __any_sync(0xFFFFFFFFu, *abort != 0); };
    const __nv_bfloat16* W1 = reinterpret_cast<const __nv_bfloat16*>(p.W1);
    for (int gq = 0; gq < ngroups; ++gq) {
      // ---- gather B = W1[x_n] of this group's requests; per-request constants
      if (!aborted()) {
        const int i = gq * kRN + et;
        int x = 0;
        const bool valid = et < kRN && i < nrej;
        if (valid) {
          if constexpr (kRes) {
            const int b = list[i];
            const int n = min(max(p.n_acc[b], 0), p.g - 1);  // a rejection leaves n <= gamma - 1
            if constexpr (MODE == kModeResid)
              x = n == 0 ? p.anchor[b] : p.tokens[(size_t)b * p.g + (n - 1)];
            else
              x = b * p.g + n;  // the row of o_{n+1}, the head vector of draft position n + 1
            col_b[et] = b;
            col_n[et] = n;
            col_row[et] = p.vrow[b];
            col_nld[et] = -p.lse[(size_t)b * p.g + n] * tc::kLog2e;
            col_nlt[et] = -p.vlset[b] * tc::kLog2e;
          } else if constexpr (MODE == kModeDraft) {
            col_b[et] = i;  // request i; its B row is o_k, not a W1 row
            x = i;
          } else if constexpr (MODE == kModeTree) {  // request i expands its node state.y
            const int node = min(max(p.tree_state[i].y, 0), p.tree_N);
            x = p.tree_tok[(size_t)i * (p.tree_N + 1) + node];
            col_b[et] = i;
          } else {  // teacher forcing: position k drafts from x*_{k-1} (the anchor at k = 0)
            const int b = i / p.g, k = i - b * p.g;
            x = k == 0 ? p.anchor[b] : p.xstar[i - 1];
            col_b[et] = i;
            col_n[et] = k;
            int xt = p.xstar[i];
            if (xt < 0 || xt >= p.V) {
              raise_status(p.status, DSPARK_ERANGE);
              xt = 0;
            }
            col_row[et] = xt;  // the reference token, whose z_d the cross entropy needs
            if constexpr (MODE == kModeLossL1) {
              col_nld[et] = -p.lse_d[i] * tc::kLog2e;
              col_nlt[et] = -p.lse_t[i] * tc::kLog2e;
            }
          }
          if (!mode_hilo(MODE) && (x < 0 || x >= p.V)) {
            raise_status(p.status, DSPARK_ERANGE);
            x = 0;
          }
        }
        if (et < kRN) {
          best_key[et] = -INFINITY;
          best_blk[et] = kNoIdx;
          col_x[et] = valid ? x : -1;
        }
      }
      asm volatile("bar.sync 2, 256;" ::: "memory");  // column constants visible to all epilogue warps
      if (!aborted()) {
        // B = the columns' W1 rows, K-major with the 128-byte swizzle: every
        // epilogue thread loads up to kRGather 16-byte chunks (consecutive
        // threads take consecutive chunks of a row), all in flight at once
        const int cpr = p.r / 8;  // 16-byte chunks per row
        if constexpr (mode_hilo(MODE)) {
          // o_k rows in fp32 -> hi = bf16(o), lo = bf16(o - hi), eight values per chunk
          float4 f[kRGather][2];
#pragma unroll
          for (int j = 0; j < kRGather; ++j) {
            const int idx = et + j * 32 * kREpi;
            f[j][0] = f[j][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (idx < kRN * cpr) {
              const int m = idx / cpr, b = col_x[m];
              if (b >= 0) {
                const size_t orow = MODE == kModeDraft ? (size_t)b * p.g + (p.step - 1) : (size_t)b;
                const float4* src =
                    reinterpret_cast<const float4*>(p.ovec + orow * p.r + (size_t)(idx - m * cpr) * 8);
                f[j][0] = __ldg(src);
                f[j][1] = __ldg(src + 1);
              }
            }
          }
#pragma unroll
          for (int j = 0; j < kRGather; ++j) {
            const int idx = et + j * 32 * kREpi;
            if (idx < kRN * cpr) {
              const int m = idx / cpr, cc = idx - m * cpr, kb = cc >> 3, ch = cc & 7;
              const float x8[8] = {f[j][0].x, f[j][0].y, f[j][0].z, f[j][0].w,
                                   f[j][1].x, f[j][1].y, f[j][1].z, f[j][1].w};
              uint32_t hi[4], lo[4];
#pragma unroll
              for (int t2 = 0; t2 < 4; ++t2) {
                const __nv_bfloat16 h0 = __float2bfloat16_rn(x8[2 * t2]), h1 = __float2bfloat16_rn(x8[2 * t2 + 1]);
                const __nv_bfloat16 l0 = __float2bfloat16_rn(x8[2 * t2] - __bfloat162float(h0));
                const __nv_bfloat16 l1 = __float2bfloat16_rn(x8[2 * t2 + 1] - __bfloat162float(h1));
                hi[t2] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
                lo[t2] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
              }
              const uint32_t dst = sB + kb * (kRN * 128) + (m >> 3) * 1024 + (m & 7) * 128 +
                                   ((uint32_t)(ch ^ (m & 7)) << 4);
              asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(hi[0]), "r"(hi[1]),
                           "r"(hi[2]), "r"(hi[3])
                           : "memory");
              asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst + kRN * p.r * 2), "r"(lo[0]),
                           "r"(lo[1]), "r"(lo[2]), "r"(lo[3])
                           : "memory");
            }
          }
        } else {
        uint4 v[kRGather];
#pragma unroll
        for (int j = 0; j < kRGather; ++j) {
          const int idx = et + j * 32 * kREpi;
          v[j] = make_uint4(0, 0, 0, 0);
          if (idx < kRN * cpr) {
            const int m = idx / cpr, x = col_x[m];
            if (x >= 0) v[j] = __ldg(reinterpret_cast<const uint4*>(W1 + (size_t)x * p.r) + (idx - m * cpr));
          }
        }
#pragma unroll
        for (int j = 0; j < kRGather; ++j) {
          const int idx = et + j * 32 * kREpi;
          if (idx < kRN * cpr) {
            const int m = idx / cpr, cc = idx - m * cpr, kb = cc >> 3, ch = cc & 7;
            const uint32_t dst = sB + kb * (kRN * 128) + (m >> 3) * 1024 + (m & 7) * 128 +
                                 ((uint32_t)(ch ^ (m & 7)) << 4);
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v[j].x), "r"(v[j].y),
                         "r"(v[j].z), "r"(v[j].w)
                         : "memory");
          }
        }
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(a_full);
      }
      const int ncols = min(kRN, nrej - gq * kRN);
      // the block draw's Gumbel noise of every (request, block) of this CTA,
      // computed once up front (visible to the combining warp after the first
      // tile's barrier) instead of on the per-tile critical path
      const int nbl = 2 * nt;
      const bool gpre = kRes && nbl <= kRGMax;
      if (gpre)
        for (int idx = et; idx < ncols * nbl; idx += 32 * kREpi) {
          const int col = idx / nbl, lb = idx - col * nbl;
          gsm[col * kRGMax + lb] = gumbel(p.rng.word(kResidBlock, col_b[col], col_n[col], 2 * tile_lo + lb));
        }
      // the loss modes' running values of this thread's entries, per column of
      // its half: (max, sum) of z_d and of z_t in base 2, or sum |p_d - p_t|
      float ra[16], rb[16], rc[16], rd[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        ra[j] = MODE == kModeLossStats ? kNegBig : 0.f;
        rb[j] = 0.f;
        rc[j] = kNegBig;
        rd[j] = 0.f;
      }
      for (int i = 0; i < nt; ++i) {
        const int it = gq * nt + i, t = tile_of(gq, i), ab = it & 1, us = it % kUP;
        bool live = !aborted();
        if (live) {
          bool ok = tc::mbar_wait(t_full(ab), (it >> 1) & 1, abort);
          ok = ok && tc::mbar_wait(up_full(us), (it / kUP) & 1, abort);
          ok = __all_sync(0xFFFFFFFFu, ok);
          if (!ok) {
            if (lane == 0 && !*abort) {
              raise_status(p.status, DSPARK_ETIMEOUT);
              *abort = 1;
            }
            live = false;
          }
        }
        const int v = t * kRM + q * 32 + lane;
        if (live) {
          tc::tc_fence_after();
          {
            // the two warps of a lane quarter take requests 16 half .. 16 half + 15
            float a[16];
            tc::tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(ab * kRN + half * 16), a);
            tc::tmem_wait_ld();
            // U and P of request j at this entry, from the staged slices
            // (consecutive lanes read consecutive words)
            float uu[16], pp[16];
            // stage layout: per request [U slice | P slice] (residual), or
            // [32 rows of U][32 rows of P] (the loss modes' two boxes)
            constexpr uint32_t kRow = (kRes || MODE == kModeTree) ? 2 * kRM * 4 : kRM * 4;
            constexpr uint32_t kPOff = kRes ? kRM * 4 : kRN * kRM * 4;
            const uint32_t su = sUP + us * L.stage + (uint32_t)(half * 16) * kRow + (uint32_t)(q * 32 + lane) * 4u;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              asm volatile("ld.shared.f32 %0, [%1];" : "=f"(uu[j]) : "r"(su + j * kRow));
              if constexpr (MODE != kModeDraft && MODE != kModeTree)
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(pp[j]) : "r"(su + j * kRow + kPOff));
            }
            if constexpr (MODE == kModeLossStats) {
              // running (max, sum 2^(y - max)) of y = z log2(e) per column,
              // for z_d = D + U and z_t = P; the entry of x* records z_d
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int col = half * 16 + j;
                const bool ok = col < ncols && v < p.V;
                const float zd = a[j] + uu[j];
                if (ok && v == col_row[col]) p.zx[col_b[col]] = zd;  // z_d at x*: one entry of the grid
                online_add(ra[j], rb[j], ok ? zd * tc::kLog2e : -INFINITY);
                online_add(rc[j], rd[j], ok ? pp[j] * tc::kLog2e : -INFINITY);
              }
            } else if constexpr (MODE == kModeDraft || MODE == kModeTree) {
              // per column, over this warp's 32 entries (half of a 64-token
              // block): max and sum exp of z = D + U (a transpose-max, the
              // columns' maxima broadcast, then a transpose-sum)
              float zd[16], e[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int col = half * 16 + j;
                zd[j] = (col < ncols && v < p.V) ? a[j] + uu[j] : -INFINITY;
                e[j] = zd[j];
              }
              const float mx = transpose_max16(e);  // lane l: column 16 half + (l & 15)
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float mj = __shfl_sync(0xFFFFFFFFu, mx, j);
                e[j] = zd[j] == -INFINITY ? 0.f : tc::ex2_ftz((zd[j] - mj) * tc::kLog2e);
              }
              const float sm = transpose_sum16(e);
              if (lane < 16) reinterpret_cast<float2*>(part)[q * kRN + half * 16 + lane] = make_float2(mx, sm);
            } else if constexpr (MODE == kModeLossL1) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int col = half * 16 + j;
                const float d = tc::ex2_ftz(fmaf(pp[j], tc::kLog2e, col_nlt[col])) -
                                tc::ex2_ftz(fmaf(a[j] + uu[j], tc::kLog2e, col_nld[col]));
                ra[j] += (col < ncols && v < p.V) ? fabsf(d) : 0.f;
              }
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int col = half * 16 + j;
                const int cl = min(col, ncols - 1);
                // p_t - p_d = 2^(P log2e - lse_t log2e) - 2^(z_d log2e - lse_d log2e), z_d = D + U
                const float w = fmaxf(0.f, tc::ex2_ftz(fmaf(pp[j], tc::kLog2e, col_nlt[cl])) -
                                               tc::ex2_ftz(fmaf(a[j] + uu[j], tc::kLog2e, col_nld[cl])));
                a[j] = (col < ncols && v < p.V) ? w : 0.f;
              }
              const float s = transpose_sum16(a);  // this warp's 32 entries, request 16 half + (lane & 15)
              if (lane < 16) part[q * kRN + half * 16 + lane] = s;
            }
          }
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(up_empty(us));
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(t_empty(ab));
        }
        if constexpr (MODE == kModeDraft || MODE == kModeTree) {
          asm volatile("bar.sync 2, 256;" ::: "memory");
          // block 2t from quarters 0, 1 and block 2t + 1 from quarters 2, 3
          if (live && et < 2 * ncols) {
            const int col = et >> 1, hh = et & 1, sblk = 2 * t + hh;
            if (sblk * 64 < p.V) {
              const float2 p0 = reinterpret_cast<const float2*>(part)[(2 * hh) * kRN + col];
              const float2 p1 = reinterpret_cast<const float2*>(part)[(2 * hh + 1) * kRN + col];
              const float m = fmaxf(p0.x, p1.x);
              float lm = -INFINITY;
              if (m > -INFINITY) lm = m + logf(p0.y * __expf(p0.x - m) + p1.y * __expf(p1.x - m));
              p.blk[(size_t)col_b[col] * p.nblk + sblk] = lm;
              if constexpr (MODE == kModeTree) p.bmax[(size_t)col_b[col] * p.nblk + sblk] = m;
            }
          }
          asm volatile("bar.sync 2, 256;" ::: "memory");  // part[] is rewritten by the next tile
        }
        if constexpr (kRes) {
          asm volatile("bar.sync 2, 256;" ::: "memory");
          if (live && warp == 4) {
            // blocks 2t (entries 0..63: quarters 0, 1) and 2t+1 (quarters 2, 3)
            for (int col = lane; col < ncols; col += 32) {
              const int b = col_b[col], n = col_n[col];
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int s = 2 * t + h;
                if (s * 64 >= p.V) continue;
                const float W = part[(2 * h) * kRN + col] + part[(2 * h + 1) * kRN + col];
                if (!(W > 0.f)) continue;
                const float key =
                    logf(W) + (gpre ? gsm[col * kRGMax + 2 * i + h] : gumbel(p.rng.word(kResidBlock, b, n, s)));
                if (key > best_key[col]) {  // blocks arrive in increasing order: ties keep the first
                  best_key[col] = key;
                  best_blk[col] = s;
                }
              }
            }
          }
          asm volatile("bar.sync 2, 256;" ::: "memory");  // part[] is rewritten by the next tile
        }
      }
      // the group's per-CTA results: the loss modes reduce each thread's
      // running values over the lanes and the four lane quarters once here
      if constexpr (MODE == kModeLossStats) {
        float2 d2 = transpose_ms16(ra, rb), t2 = transpose_ms16(rc, rd);  // lane l: column 16 half + (l & 15)
        if (lane < 16)
          reinterpret_cast<float4*>(part)[q * kRN + half * 16 + lane] = make_float4(d2.x, d2.y, t2.x, t2.y);
        asm volatile("bar.sync 2, 256;" ::: "memory");
        if (warp == 4 && !aborted())
          for (int col = lane; col < ncols; col += 32) {
            float4 r = reinterpret_cast<const float4*>(part)[col];
#pragma unroll
            for (int qq = 1; qq < 4; ++qq) {
              const float4 o = reinterpret_cast<const float4*>(part)[qq * kRN + col];
              const float2 x = ms2_combine(make_float2(r.x, r.y), make_float2(o.x, o.y));
              const float2 y = ms2_combine(make_float2(r.z, r.w), make_float2(o.z, o.w));
              r = make_float4(x.x, x.y, y.x, y.y);
            }
            // back to natural-log units; a column with no finite entry is (-inf, 0)
            p.lpart[(size_t)col_b[col] * p.G + c] =
                make_float4(r.y > 0.f ? r.x * kLn2 : -INFINITY, r.y, r.w > 0.f ? r.z * kLn2 : -INFINITY, r.w);
          }
      } else if constexpr (MODE == kModeLossL1) {
        const float s = transpose_sum16(ra);
        if (lane < 16) part[q * kRN + half * 16 + lane] = s;
        asm volatile("bar.sync 2, 256;" ::: "memory");
        if (warp == 4 && !aborted())
          for (int col = lane; col < ncols; col += 32)
            p.l1part[(size_t)col_b[col] * p.G + c] =
                (part[col] + part[kRN + col]) + (part[2 * kRN + col] + part[3 * kRN + col]);
      } else if constexpr (kRes) {
        if (warp == 4 && !aborted())
          for (int col = lane; col < ncols; col += 32)
            p.rpart[(size_t)col_b[col] * p.G + c] = make_float2(best_key[col], __int_as_float(best_blk[col]));
      }
      asm volatile("bar.sync 2, 256;" ::: "memory");  // constants are rewritten by the next group
    }
  }
  pdl_trigger();  // the token pick may be scheduled while this CTA finishes
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kRTmemCols);
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

int resid_tc_supported(const dspark_dims& d) {
  return d.wdtype == DSPARK_BF16 && d.r % 64 == 0 && d.r <= 256 && d.V % 8 == 0 && d.B <= kRMaxB;
}

cudaError_t resid_tc_configure(dspark_ws* ws) {
  const RSmem L = RSmem::make(ws->d.r, kModeResid);
  const size_t smem = L.total + 1024;
  cudaError_t e = cudaFuncSetAttribute(k_resid_tc<kModeResid>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_resid_tc<kModeLossStats>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_resid_tc<kModeLossL1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_resid_tc<kModeDraft>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(RSmem::make(ws->d.r, kModeDraft).total + 1024));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_resid_tc<kModeResidRnn>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(RSmem::make(ws->d.r, kModeResidRnn).total + 1024));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_resid_tc<kModeTree>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_resid_tc<kModeResid>, kRThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1 || !encode_fn()) return cudaErrorNotSupported;
  return cudaSuccess;
}

// The residual block draw for the requests verify flagged; writes
// rpart[b * grid + cta]. Grid = one CTA per SM (no grid-wide barrier, so no
// co-residency requirement).
namespace {

// W2 as [r rows x V] bf16, boxes of [r/2 x 64] (a K-half of a tile) with the
// 128-byte swizzle.
cudaError_t w2_tensor_map(const dspark_dims& d, const void* W2, CUtensorMap* tm) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)d.V, (cuuint64_t)d.r};
  const cuuint64_t strides[1] = {(cuuint64_t)d.V * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)d.r / 2};
  const cuuint32_t es[2] = {1, 1};
  if (enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W2), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

// A [rows x V] fp32 matrix (rows `stride` floats apart) as boxes of
// [32 rows x 128 entries], no swizzle.
cudaError_t rows_tensor_map(const float* X, int rows, int V, size_t stride, CUtensorMap* tm) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)V, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)stride * 4};
  const cuuint32_t box[2] = {(cuuint32_t)kRM, (cuuint32_t)kRN};
  const cuuint32_t es[2] = {1, 1};
  if (enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(X), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

RParams base_params(const dspark_ws* ws, int grid) {
  const dspark_dims& d = ws->d;
  RParams p;
  memset(&p, 0, sizeof(p));
  p.B = d.B;
  p.g = d.gamma;
  p.V = d.V;
  p.r = d.r;
  p.ntiles = (d.V + kRM - 1) / kRM;
  p.G = grid;
  p.status = ws->s.status;
  return p;
}

}  // namespace

cudaError_t launch_resid_tc(const dspark_ws* ws, const VerifyArgs& a, float2* rpart, int grid, cudaStream_t st,
                            bool pdl) {
  const dspark_dims& d = ws->d;
  CUtensorMap tm;
  cudaError_t e = w2_tensor_map(d, a.W2, &tm);
  if (e != cudaSuccess) return e;
  RParams p = base_params(ws, grid);
  p.rng = Rng::make(a.seed, a.round, (uint32_t)ws->b0);
  p.P = a.P;
  p.U = a.U;
  p.W1 = a.W1;
  p.anchor = a.anchor;
  p.tokens = a.tokens;
  p.lse = a.lse;
  p.vflag = ws->s.vflag;
  p.n_acc = a.n_acc;
  p.vrow = ws->s.vrow;
  p.vlset = ws->s.vlset;
  p.rpart = rpart;
  p.ovec = a.ovec;
  if (a.ovec)  // the RNN head: B = o_{n+1} as bf16 hi + lo
    return launch_ex(k_resid_tc<kModeResidRnn>, dim3(grid), dim3(kRThreads),
                     RSmem::make(d.r, kModeResidRnn).total + 1024, st, pdl, tm, tm, tm, p);
  return launch_ex(k_resid_tc<kModeResid>, dim3(grid), dim3(kRThreads), RSmem::make(d.r, kModeResid).total + 1024,
                   st, pdl, tm, tm, tm, p);
}

cudaError_t launch_loss_tc(const dspark_ws* ws, const LossArgs& a, int pass, cudaStream_t st) {
  const dspark_dims& d = ws->d;
  CUtensorMap tm;
  cudaError_t e = w2_tensor_map(d, a.W2, &tm);
  if (e != cudaSuccess) return e;
  CUtensorMap tu, tp;
  const int rows = d.B * d.gamma;
  e = rows_tensor_map(a.U, rows, d.V, (size_t)d.V, &tu);
  if (e == cudaSuccess) e = rows_tensor_map(a.P, rows, d.V, (size_t)d.V, &tp);
  if (e != cudaSuccess) return e;
  RParams p = base_params(ws, ws->geo.num_sms);
  p.P = a.P;
  p.U = a.U;
  p.W1 = a.W1;
  p.anchor = a.anchor;
  p.xstar = a.xstar;
  p.lpart = a.lpart;
  p.zx = a.zx;
  p.l1part = a.l1part;
  p.lse_d = a.lse_d;
  p.lse_t = a.lse_t;
  const RSmem L = RSmem::make(d.r, kModeResid);
  if (pass == 0)
    k_resid_tc<kModeLossStats><<<p.G, kRThreads, L.total + 1024, st>>>(tm, tu, tp, p);
  else
    k_resid_tc<kModeLossL1><<<p.G, kRThreads, L.total + 1024, st>>>(tm, tu, tp, p);
  return cudaGetLastError();
}

// One draft step k of the RNN head: blk[b][s] = log sum_{v in block s} exp z_v
// with z = U_k + o_k W2 for every request. Grid = one CTA per SM.
cudaError_t launch_rnn_blocks_tc(const dspark_ws* ws, const float* U, const void* W2, const float* ovec, int k,
                                 cudaStream_t st) {
  const dspark_dims& d = ws->d;
  CUtensorMap tm, tu;
  cudaError_t e = w2_tensor_map(d, W2, &tm);
  if (e == cudaSuccess) e = rows_tensor_map(U + (size_t)(k - 1) * d.V, d.B, d.V, (size_t)d.gamma * d.V, &tu);
  if (e != cudaSuccess) return e;
  RParams p = base_params(ws, ws->geo.num_sms);
  p.ovec = ovec;
  p.step = k;
  p.blk = ws->s.blk;
  p.nblk = ws->geo.nblk;
  const RSmem L = RSmem::make(d.r, kModeDraft);
  k_resid_tc<kModeDraft><<<p.G, kRThreads, L.total + 1024, st>>>(tm, tu, tu, p);
  return cudaGetLastError();
}

// One expansion step of PCTree: for every request b, blk[b][s] and bmax[b][s]
// are the log-mass and the maximum of z = U[b, depth] + W1[token] W2 over
// 64-token block s, (token, depth) those of node state[b].y. Grid = one CTA
// per SM.
cudaError_t launch_tree_blocks_tc(const dspark_ws* ws, const float* U, const void* W1, const void* W2,
                                  const int32_t* tok, const int32_t* dep, const int4* state, int N, float* blk,
                                  float* bmax, cudaStream_t st) {
  const dspark_dims& d = ws->d;
  CUtensorMap tm;
  cudaError_t e = w2_tensor_map(d, W2, &tm);
  if (e != cudaSuccess) return e;
  RParams p = base_params(ws, ws->geo.num_sms);
  p.U = U;
  p.W1 = W1;
  p.tree_tok = tok;
  p.tree_dep = dep;
  p.tree_state = state;
  p.tree_N = N;
  p.blk = blk;
  p.bmax = bmax;
  p.nblk = ws->geo.nblk;
  const RSmem L = RSmem::make(d.r, kModeResid);
  k_resid_tc<kModeTree><<<p.G, kRThreads, L.total + 1024, st>>>(tm, tm, tm, p);
  return cudaGetLastError();
}

}  // namespace dspark
