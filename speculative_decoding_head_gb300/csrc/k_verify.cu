// k_verify.cu -- lossless ragged rejection-sampling verify.
//
// "DeepSeek-V4.1 模型结构（6）：解码，DSpark", section "投机解码" and the
// derivation box; "DSpark：不让大模型更聪明，而让它「吐字更快」" §02;
// deepseek.csdn.net close reading §2.1:
//   * row j of request b (packed row row_off[b] + j) is the target
//     distribution p_t after x_j; for j < l_b - 1 it tests draft x_{j+1}:
//     accept with probability min(1, p_t(x_{j+1}) / p_d(x_{j+1})), written as
//     u * p_d < p_t with u from the stream (purpose "accept", v = 0);
//   * checking runs left to right and stops at the first rejection n;
//   * after a rejection the next anchor is drawn from
//     norm(max(0, p_t,n - p_d,n+1)), where p_d,n+1 is recomputed from
//     (U row n, W1[x_n], W2, lse_n+1) rather than stored;
//   * if all l_b - 1 drafts pass, the next anchor is the bonus token drawn
//     from p_t of row l_b - 1.
// Every draw is the library's two-level Gumbel-max (64-token blocks).
//
// Kernels (all launched with grids that do not depend on device-side sizes):
//   k_verify_sweep_dyn  V % 64 == 0 and at least 128 blocks a row: the packed
//                       rows' blocks in 32 KB chunks taken from a counter;
//                       per block its log-sum-exp, per 32 blocks each row's
//                       (max, sum).
//   k_verify_fin_dyn    after it, one CTA per request: the accept tests, the
//                       first rejection, the bonus block and token draws.
//   k_verify_sweep_bulk V % 64 == 0 and fewer blocks: equal contiguous ranges
//                       of blocks, one per CTA, with the finalize of each
//                       request in the CTA that completes its partials.
//   k_verify_sweep      otherwise: equal ranges, then k_verify_finalize (one
//                       warp per request, one lane per row).
//   k_resid_blocks      grid (chunks, B): residual block masses and block draw
//                       on CUDA cores (k_resid_tc.cu: the tcgen05 version).
//   k_resid_pick        grid (B): residual token draw inside the drawn block.
#include "dspark_common.cuh"
#include "dspark_internal.h"
#include "tc_ptx.cuh"

namespace dspark {

constexpr int kSweepThreads = 256;
constexpr int kPickThreads = 1024;  // k_resid_pick: 16 groups of K rows x 64 tokens

__device__ __forceinline__ int request_of_row(const int32_t* __restrict__ row_off, int B, int q) {
  int lo = 0, hi = B - 1;  // largest b with row_off[b] <= q
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (row_off[mid] <= q) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// The verified rows, flattened into 64-token block units u = q * nblk + s
// (row q, block s), are split into gridDim.x contiguous ranges of (almost)
// equal length, one per CTA: every CTA streams the same number of bytes.
// A range touches a few consecutive rows; for each it writes one partial
// (max, sum exp, best block key, best block) to part[cta * SL + row - first].
__device__ __forceinline__ long long unit_lo(int c, long long T, int G) { return (long long)c * T / G; }
// the CTA whose range holds unit u
__device__ __forceinline__ int unit_owner(long long u, long long T, int G) {
  return (int)(((u + 1) * (long long)G - 1) / T);
}

constexpr int kSweepUnroll = 4;

__global__ void __launch_bounds__(kSweepThreads)
    k_verify_sweep(const float* __restrict__ P, const int32_t* __restrict__ row_off,
                   const int32_t* __restrict__ lengths, int B, int V, int nblk, int Rmax, int SL, Rng rng,
                   float4* __restrict__ part) {
  __shared__ MS red_ms[kSweepThreads / 32];
  __shared__ KeyIdx red_k[kSweepThreads / 32];
  const int R = min(max(row_off[B], 0), Rmax);  // finalize reports an inconsistent row_off
  const long long T = (long long)R * nblk;
  if (T == 0) return;
  const int G = gridDim.x, c = blockIdx.x;
  const long long lo = unit_lo(c, T, G), hi = unit_lo(c + 1, T, G);
  if (lo >= hi) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int half = lane >> 4, l16 = lane & 15;
  const bool vec = (V & 3) == 0;
  const int q0 = (int)(lo / nblk);
  for (int q = q0; (long long)q * nblk < hi; ++q) {
    const int s0 = (int)max(lo - (long long)q * nblk, 0ll);
    const int s1 = (int)min(hi - (long long)q * nblk, (long long)nblk);
    const int b = request_of_row(row_off, B, q);
    const int j = q - row_off[b];
    const bool bonus = j == lengths[b] - 1;
    const float* row = P + (size_t)q * V;
    MS ms{-INFINITY, 0.f};
    KeyIdx kb = key_none();
    // a half-warp takes one 64-token block: 16 lanes x 4 tokens
    for (int sb = s0 + 2 * warp; sb < s1; sb += 2 * nw * kSweepUnroll) {
      float x[kSweepUnroll][4];
#pragma unroll
      for (int u = 0; u < kSweepUnroll; ++u) {
        const int s = sb + half + 2 * nw * u;
        const int v = s * kBlockW + 4 * l16;
        if (s < s1 && v < V) {
          if (vec) {
            const float4 f = __ldcs(reinterpret_cast<const float4*>(row + v));
            x[u][0] = f.x; x[u][1] = f.y; x[u][2] = f.z; x[u][3] = f.w;
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) x[u][e] = v + e < V ? __ldcs(row + v + e) : -INFINITY;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) x[u][e] = -INFINITY;
        }
      }
#pragma unroll
      for (int u = 0; u < kSweepUnroll; ++u) {
        const float m4 = fmaxf(fmaxf(x[u][0], x[u][1]), fmaxf(x[u][2], x[u][3]));
        if (bonus) {
          float m = m4;
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
          float t = 0.f;
          if (m != -INFINITY)
            t = __expf(x[u][0] - m) + __expf(x[u][1] - m) + __expf(x[u][2] - m) + __expf(x[u][3] - m);
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
          const int s = sb + half + 2 * nw * u;
          if (l16 == 0 && s < s1 && m != -INFINITY) {
            ms = ms_combine(ms, MS{m, t});
            kb = better(kb, KeyIdx{m + logf(t) + gumbel(rng.word(kBonusBlock, b, j, s)), s});
          }
        } else if (m4 != -INFINITY) {
          const float m = fmaxf(m4, ms.m);
          float t = ms.m == -INFINITY ? 0.f : ms.s * __expf(ms.m - m);
          t += __expf(x[u][0] - m) + __expf(x[u][1] - m) + __expf(x[u][2] - m) + __expf(x[u][3] - m);
          ms = MS{m, t};
        }
      }
    }
    ms = warp_ms(ms);
    kb = warp_best(kb);
    if (lane == 0) {
      red_ms[warp] = ms;
      red_k[warp] = kb;
    }
    __syncthreads();
    if (warp == 0) {
      MS m2 = lane < nw ? red_ms[lane] : MS{-INFINITY, 0.f};
      KeyIdx k2 = lane < nw ? red_k[lane] : key_none();
      m2 = warp_ms(m2);
      k2 = warp_best(k2);
      if (lane == 0 && q - q0 < SL) part[(size_t)c * SL + (q - q0)] = make_float4(m2.m, m2.s, k2.key, __int_as_float(k2.idx));
    }
    __syncthreads();
  }
}

// What the accept tests and the bonus draw read, and what they write.
struct FinArgs {
  const float* P;
  const int32_t* row_off;
  const int32_t* lengths;
  const int32_t* anchor;
  const int32_t* tokens;
  const float* pd_tok;
  int B, g, V, nblk, SL, Gs;
  Rng rng;
  const float4* part;
  int32_t* n_acc;
  int32_t* next_anchor;
  int* vflag;
  int* vrow;
  float* vlset;
  int* status;
  float* px;  // [rows] P at each row's draft token, stored by the bulk sweep (nullptr: read P)
  const float4* rowstat;  // non-null: (max, sum, bonus key, block) of each of the request's rows, from row_off[b]
};

// Request b, by one whole warp. Lane j handles target row j: its
// log-sum-exp from the sweep partials, p_t of draft x_{j+1} and the accept
// test; the first rejection is the lowest failing lane. Then the bonus token
// draw inside its block, or the hand-over to the residual pass.
// ell = lengths[b], base = row_off[b], R = row_off[B] (clamped to the row
// capacity), as the caller read them.
struct FinIn {  // lane j's draft token x_{j+1}, its draft probability and P at it (rows 0 .. ell-2)
  int x;
  float pdx, Px;
};
__device__ __forceinline__ FinIn finalize_inputs(int b, const FinArgs& f, int ell, int base, int R) {
  const int lane = threadIdx.x & 31;
  FinIn in{0, 0.f, 0.f};
  if (ell < 1 || ell > f.g + 1 || base < 0 || base + ell > R || lane >= ell - 1) return in;
  in.x = f.tokens[(size_t)b * f.g + lane];
  in.pdx = f.pd_tok[(size_t)b * f.g + lane];
  if (in.x >= 0 && in.x < f.V) in.Px = f.px ? __ldcg(f.px + base + lane) : f.P[(size_t)(base + lane) * f.V + in.x];
  return in;
}
__device__ void finalize_core(int b, const FinArgs& f, int ell, int base, int R, const FinIn& in) {
  const int lane = threadIdx.x & 31;
  const float* __restrict__ P = f.P;
  const int g = f.g, V = f.V, nblk = f.nblk, SL = f.SL, Gs = f.Gs;
  const Rng rng = f.rng;
  const float4* __restrict__ part = f.part;
  int32_t* __restrict__ n_acc = f.n_acc;
  int32_t* __restrict__ next_anchor = f.next_anchor;
  int* __restrict__ vflag = f.vflag;
  int* __restrict__ vrow = f.vrow;
  float* __restrict__ vlset = f.vlset;
  int* __restrict__ status = f.status;
  if (lane == 0) vflag[b] = 0;  // no residual pass unless a rejection is found below
  if (ell < 1 || ell > g + 1 || base < 0 || base + ell > R) {
    if (lane == 0) raise_status(status, DSPARK_ERANGE);
    return;
  }
  const long long T = (long long)R * nblk;
  // partials of row q: the CTAs whose unit ranges meet [q nblk, (q+1) nblk),
  // or the row's statistics already combined by the caller
  auto row_partials = [&](int q, MS* ms_out, KeyIdx* kb_out) {
    if (f.rowstat) {
      const float4 d = f.rowstat[q - base];
      *ms_out = MS{d.x, d.y};
      *kb_out = KeyIdx{d.z, __float_as_int(d.w)};
      return;
    }
    const long long u0 = (long long)q * nblk, u1 = u0 + nblk - 1;
    MS ms{-INFINITY, 0.f};
    KeyIdx kb = key_none();
    const int c0 = unit_owner(u0, T, Gs), c1 = unit_owner(u1, T, Gs);
    for (int cb = c0; cb <= c1; cb += 4) {  // four partials' loads in flight at a time
      float4 d[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = cb + e;
        d[e] = make_float4(-INFINITY, 0.f, -INFINITY, __int_as_float(kNoIdx));
        if (c > c1) continue;
        const long long clo = unit_lo(c, T, Gs);
        if (clo >= unit_lo(c + 1, T, Gs)) continue;  // an empty range wrote nothing
        const int first = (int)(clo / nblk);
        if (q - first >= SL) continue;
        d[e] = __ldcg(part + (size_t)c * SL + (q - first));
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        ms = ms_combine(ms, MS{d[e].x, d[e].y});
        kb = better(kb, KeyIdx{d[e].z, __float_as_int(d[e].w)});
      }
    }
    *ms_out = ms;
    *kb_out = kb;
  };
  // ---- one lane per verified row: accept tests of rows 0 .. ell-2, and the
  // bonus block key of row ell-1; the draft token's target logit is loaded
  // alongside the row's partials
  bool acc = true, bad = false;
  float Lt = 0.f;
  KeyIdx kbonus = key_none();
  const bool arow = lane < ell - 1;
  const int x = in.x;
  const float Px = in.Px, pdx = in.pdx;
  if (lane < ell) {
    MS ms;
    KeyIdx kb;
    row_partials(base + lane, &ms, &kb);
    Lt = ms_log(ms);
    kbonus = kb;
  }
  if (arow) {
    if (!isfinite(Lt) || x < 0 || x >= V) {
      bad = true;
    } else {
      const float pt = expf(Px - Lt);
      const float u = u01(rng.word(kAccept, b, lane, 0));
      acc = u * pdx < pt;
    }
  }
  const unsigned badm = __ballot_sync(0xFFFFFFFFu, bad);
  if (badm) {
    if (lane == 0) raise_status(status, DSPARK_ERANGE);
    return;
  }
  const unsigned rej = __ballot_sync(0xFFFFFFFFu, !acc);
  if (rej) {
    const int n = __ffs(rej) - 1;
    const float lset = __shfl_sync(0xFFFFFFFFu, Lt, n);
    if (lane == 0) {
      n_acc[b] = n;
      vflag[b] = 1;
      vrow[b] = base + n;
      vlset[b] = lset;
    }
    return;
  }
  // ---- every verified draft accepted: bonus token from row ell - 1
  const int n = ell - 1;
  const size_t q = (size_t)base + n;
  KeyIdx kb = kbonus;
  if (n >= 32) {  // gamma = 32: the bonus row has no lane of its own
    MS unused;
    if (lane == 0) row_partials((int)q, &unused, &kb);
  }
  kb.key = __shfl_sync(0xFFFFFFFFu, kb.key, n < 32 ? n : 0);
  kb.idx = __shfl_sync(0xFFFFFFFFu, kb.idx, n < 32 ? n : 0);
  if (kb.idx == kNoIdx) {
    if (lane == 0) raise_status(status, DSPARK_ENUMERIC);
    return;
  }
  KeyIdx kt = key_none();
  {  // lane: tokens v and v + 1 of the block, which share one counter draw
    const int v = kb.idx * kBlockW + 2 * lane;
    const uint4 w = rng.block4(kBonusToken, b, n, v);
    const uint32_t w0 = (v & 3) ? w.z : w.x, w1 = (v & 3) ? w.w : w.y;
    if (v < V) kt = better(kt, KeyIdx{P[q * V + v] + gumbel(w0), v});
    if (v + 1 < V) kt = better(kt, KeyIdx{P[q * V + v + 1] + gumbel(w1), v + 1});
  }
  kt = warp_best(kt);
  if (lane == 0) {
    n_acc[b] = n;
    next_anchor[b] = kt.idx;
  }
}

__device__ __forceinline__ void finalize_core(int b, const FinArgs& f, int ell, int base, int R) {
  finalize_core(b, f, ell, base, R, finalize_inputs(b, f, ell, base, R));
}

// log of the residual weight max(0, p_t - p_d) of one token, written as
// log p_t + log(-expm1(log p_d - log p_t)) so that near-equal p_t and p_d keep
// their relative precision; -inf when p_t <= p_d.
__device__ __forceinline__ float resid_logw(float lpt, float lpd) {
  if (!(lpt > lpd)) return -INFINITY;
  return lpt + logf(-expm1f(lpd - lpt));
}

// One warp per request, after the register sweep.
__global__ void __launch_bounds__(128) k_verify_finalize(const FinArgs f) {
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (b >= f.B) return;
  const int R = min(max(f.row_off[f.B], 0), f.B * (f.g + 1));
  if (f.anchor[b] < 0 || f.anchor[b] >= f.V) {
    if ((threadIdx.x & 31) == 0) raise_status(f.status, DSPARK_ERANGE);
    return;
  }
  finalize_core(b, f, f.lengths[b], f.row_off[b], R);
}

// Bulk-copy sweep for V % 64 == 0: unit u is then tokens [64u, 64u + 64) of
// the packed rows, so a CTA's range is one contiguous byte range of P. It is
// streamed through a 3-deep ring of 32 KB stages by cp.async.bulk and
// consumed from shared memory one 64-token block per thread: the thread reads
// its block's 16 float4 in a rotated order (conflict-free across the warp;
// the order does not matter for a max and a sum), forms the block's
// (max, sum exp) with 64 independent exponentials, folds it into the row and,
// on the last verified row of a request, draws the bonus block key. Rows
// change only at block boundaries; a thread flushes a finished row into its
// per-row slot.
constexpr int kBulkThreads = 128;
constexpr int kBulkStages = 3;
constexpr int kBulkUnits = kBulkThreads;             // one block per thread per stage
constexpr int kBulkFloats = kBulkUnits * kBlockW;   // 8192 fp32 = 32 KB
constexpr int kBulkMaxSlots = 32;  // rows one CTA range may touch (per-row partials of every thread)

int sweep_bulk_max_slots() { return kBulkMaxSlots; }

// ring stages, then SL rows of per-thread partials, the ring barriers, and
// the rows' (request, position, ...) and (length, offset)
size_t sweep_bulk_smem_bytes(int SL) {
  return (size_t)kBulkStages * kBulkFloats * 4 + (size_t)SL * kBulkThreads * 16 + 64 + (size_t)SL * (16 + 8);
}

__global__ void __launch_bounds__(kBulkThreads)
    k_verify_sweep_bulk(const float* __restrict__ P, const int32_t* __restrict__ row_off,
                        const int32_t* __restrict__ lengths, int B, int nblk, int Rmax, int SL, Rng rng,
                        float4* __restrict__ part, int* __restrict__ status, const FinArgs fin,
                        int* __restrict__ vdone, const int4* __restrict__ rowtab) {
  extern __shared__ __align__(128) unsigned char smem[];
  pdl_wait();  // row offsets and lengths are the planner's
  float* stage = reinterpret_cast<float*>(smem);
  float4* slot = reinterpret_cast<float4*>(smem + (size_t)kBulkStages * kBulkFloats * 4);  // [SL][threads]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kBulkStages * kBulkFloats * 4 +
                                               (size_t)SL * kBulkThreads * 16);
  int4* rowinfo = reinterpret_cast<int4*>(bars + 8);  // [SL] (b, j, last row?, tested token)
  int2* rowlen = reinterpret_cast<int2*>(rowinfo + SL);  // [SL] (lengths[b], row_off[b])
  // The finalize of a request whose rows no range covers never runs, so the
  // lengths, offsets and anchors of all requests are checked by one CTA.
  auto check_requests = [&]() {
    if (threadIdx.x == 0 && row_off[0] != 0) raise_status(status, DSPARK_ERANGE);
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
      const int ell = lengths[b], base = row_off[b];
      if (ell < 1 || ell > fin.g + 1 || base < 0 || row_off[b + 1] != base + ell || base + ell > Rmax ||
          fin.anchor[b] < 0 || fin.anchor[b] >= fin.V)
        raise_status(status, DSPARK_ERANGE);
    }
  };
  const int R = min(max(row_off[B], 0), Rmax);
  const long long T = (long long)R * nblk;
  if (T == 0) {  // no rows at all
    if (blockIdx.x == gridDim.x - 1) check_requests();
    return;
  }
  const int G = gridDim.x, c = blockIdx.x, tid = threadIdx.x;
  const long long lo = unit_lo(c, T, G), hi = unit_lo(c + 1, T, G);
  if (lo >= hi) return;
  const int q0 = (int)(lo / nblk);
  const int nslots = (int)((hi - 1) / nblk) - q0 + 1;
  if (nslots > SL || nslots > kBulkMaxSlots) {  // a range never spans this many rows
    if (tid == 0) raise_status(status, DSPARK_ERANGE);
    return;
  }
  const int nchunks = (int)((hi - lo + kBulkUnits - 1) / kBulkUnits);
  const uint32_t bar0 = tc::smem_u32(bars);
  const uint32_t st0 = tc::smem_u32(stage);
  // P is read once: evict it first, so that W2 (kept with evict_last by the
  // draft and the residual pass) stays in L2 across the sweep
  const uint64_t pol = tc::policy_evict_first();
  auto issue = [&](int ch) {
    const long long u = lo + (long long)ch * kBulkUnits;
    const int units = (int)min((long long)kBulkUnits, hi - u);
    const uint32_t bytes = (uint32_t)units * kBlockW * 4u;
    const int sidx = ch % kBulkStages;
    tc::mbar_arrive_expect_tx(bar0 + 8u * sidx, bytes);
    tc::bulk_load_hint(st0 + (uint32_t)sidx * kBulkFloats * 4u, P + u * kBlockW, bytes, bar0 + 8u * sidx, pol);
  };
  int issued = 0;  // chunks issued (thread 0's count)
  if (tid == 0) {  // the first copies fly while the row table is built
    for (int i = 0; i < kBulkStages; ++i) tc::mbar_init(bar0 + 8u * i, 1);
    tc::fence_barrier_init();
    for (; issued < kBulkStages && issued < nchunks; ++issued) issue(issued);
  }
  // request, position and bonus flag of each row the range touches: from the
  // planner's row table when it wrote one for this round; else warp 1 finds
  // the requests by 32-way sampling of row_off (each round of loads narrows
  // the request of row q0 to a 32nd of its interval) instead of a binary
  // search's log2(B) dependent loads; the range's rows then belong to the
  // next few requests, read in one more round.
  if (rowtab && tid >= 32 && tid < 32 + nslots) {
    const int4 t4 = rowtab[q0 + tid - 32];
    const int b = min(max(t4.x, 0), B - 1), j = t4.y, ell = t4.z;
    const bool tested = j >= 0 && j < min(ell, fin.g + 1) - 1;
    const int xt = tested ? fin.tokens[(size_t)b * fin.g + j] : -1;
    rowinfo[tid - 32] = make_int4(b, j, j == ell - 1 ? 1 : 0, xt >= 0 && xt < fin.V ? xt : -1);
    rowlen[tid - 32] = make_int2(ell, t4.w);
  } else if (!rowtab && tid >= 32 && tid < 64) {
    const int lane = tid - 32;
    int lo = 0, hi = B;  // the request of row q0 lies in [lo, hi)
    while (hi - lo > 16) {
      const int stride = (hi - lo + 31) / 32;
      const int sidx = lo + lane * stride;
      const int v = sidx < hi ? row_off[sidx] : INT_MAX;
      const unsigned m = __ballot_sync(0xFFFFFFFFu, v <= q0);
      const int L = m ? 31 - __clz((int)m) : 0;  // offsets that do not add up are reported by the last CTA
      lo += L * stride;
      hi = min(hi, lo + stride);
    }
    const int sidx = lo + lane;
    const int v = sidx < B ? row_off[sidx] : INT_MAX;
    int my_b = lo, my_ro = 0;
    for (int i = 0; i < nslots; ++i) {
      const unsigned m = __ballot_sync(0xFFFFFFFFu, v <= q0 + i);
      const int b = lo + (m ? 31 - __clz((int)m) : 0);
      const int ro = __shfl_sync(0xFFFFFFFFu, v, b - lo);
      if (lane == i) {
        my_b = b;
        my_ro = ro;
      }
    }
    if (lane < nslots) {
      const int b = min(max(my_b, 0), B - 1);
      const int j = q0 + lane - my_ro;
      // the draft token the row tests (-1 on the last verified row; offsets
      // and lengths are checked by the last CTA meanwhile, so stay in bounds here)
      const int ell = lengths[b];
      const bool tested = j >= 0 && j < min(ell, fin.g + 1) - 1;
      const int xt = tested ? fin.tokens[(size_t)b * fin.g + j] : -1;
      rowinfo[lane] = make_int4(b, j, j == ell - 1 ? 1 : 0, xt >= 0 && xt < fin.V ? xt : -1);
      rowlen[lane] = make_int2(ell, my_ro);
    }
  }
  for (int i = tid; i < nslots * kBulkThreads; i += kBulkThreads)
    slot[i] = make_float4(-INFINITY, 0.f, -INFINITY, __int_as_float(kNoIdx));
  __syncthreads();
  volatile int never = 0;
  int q_cur = -1, bcur = 0, jcur = 0;
  bool bonus = false;
  MS ms{-INFINITY, 0.f};
  KeyIdx kb = key_none();
  auto flush = [&]() {
    if (q_cur >= 0) {
      float4& sl = slot[(q_cur - q0) * kBulkThreads + tid];
      const MS mm = ms_combine(MS{sl.x, sl.y}, ms);
      const KeyIdx kk = better(KeyIdx{sl.z, __float_as_int(sl.w)}, kb);
      sl = make_float4(mm.m, mm.s, kk.key, __int_as_float(kk.idx));
    }
    ms = MS{-INFINITY, 0.f};
    kb = key_none();
  };
  bool failed = false;
  for (int ch = 0; ch < nchunks; ++ch) {
    const int sidx = ch % kBulkStages;
    bool ok = tc::mbar_wait(bar0 + 8u * sidx, (ch / kBulkStages) & 1, &never);
    if (__syncthreads_or(!ok)) {  // the same answer in every thread
      if (tid == 0) raise_status(status, DSPARK_ETIMEOUT);
      failed = true;
      break;
    }
    const long long u = lo + (long long)ch * kBulkUnits + tid;
    if (u < hi) {
      const float4* blk4 = reinterpret_cast<const float4*>(stage + (size_t)sidx * kBulkFloats) + tid * 16;
      float4 x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = blk4[(i + tid) & 15];  // rotated: conflict-free
      // block max (three-input max, 4 chains) and sum of e^(x - m) =
      // 2^(x log2e - m log2e) on fp32 pairs (FFMA2, MUFU ex2, FADD2)
      float m4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) m4[i] = tc::max3f(x[i].x, x[i].y, tc::max3f(x[i].z, x[i].w, -INFINITY));
#pragma unroll
      for (int i = 4; i < 16; ++i) m4[i & 3] = tc::max3f(tc::max3f(m4[i & 3], x[i].x, x[i].y), x[i].z, x[i].w);
      const float m = tc::max3f(fmaxf(m4[0], m4[1]), m4[2], m4[3]);
      float t = 0.f;
      if (m != -INFINITY) {
        const unsigned long long l2e = tc::f2pack(tc::kLog2e, tc::kLog2e);
        const unsigned long long nml = tc::f2pack(-m * tc::kLog2e, -m * tc::kLog2e);
        unsigned long long acc0 = 0ull, acc1 = 0ull;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float a0, a1, a2, a3;
          tc::f2unpack(tc::fma2(tc::f2pack(x[i].x, x[i].y), l2e, nml), a0, a1);
          tc::f2unpack(tc::fma2(tc::f2pack(x[i].z, x[i].w), l2e, nml), a2, a3);
          const unsigned long long e01 = tc::f2pack(tc::ex2_ftz(a0), tc::ex2_ftz(a1));
          const unsigned long long e23 = tc::f2pack(tc::ex2_ftz(a2), tc::ex2_ftz(a3));
          acc0 = i == 0 ? e01 : tc::add2(acc0, e01);
          acc1 = i == 0 ? e23 : tc::add2(acc1, e23);
        }
        float s0, s1;
        tc::f2unpack(tc::add2(acc0, acc1), s0, s1);
        t = s0 + s1;
        const int q = (int)(u / nblk), sblk = (int)(u - (long long)q * nblk);
        if (q != q_cur) {
          flush();
          q_cur = q;
          const int4 ri = rowinfo[q - q0];
          bcur = ri.x;
          jcur = ri.y;
          bonus = ri.z != 0;
        }
        ms = ms_combine(ms, MS{m, t});
        if (bonus) kb = better(kb, KeyIdx{m + logf(t) + gumbel(rng.word(kBonusBlock, bcur, jcur, sblk)), sblk});
        const int xt = rowinfo[q - q0].w;  // the accept test's target logit, while the block is staged
        if (xt >= 0 && (xt >> 6) == sblk) fin.px[q] = stage[(size_t)sidx * kBulkFloats + tid * kBlockW + (xt & 63)];
      }
    }
    __syncthreads();  // every thread is done with this stage
    if (tid == 0 && issued < nchunks) issue(issued++);
  }
  if (failed) {
    if (tid == 0)  // let the copies already issued land before the CTA exits
      for (int ch = max(0, issued - kBulkStages); ch < issued; ++ch) {
        volatile int nv = 0;
        tc::mbar_wait(bar0 + 8u * (ch % kBulkStages), (ch / kBulkStages) & 1, &nv);
      }
    return;
  }
  flush();
  pdl_trigger();  // the residual pass may be scheduled while this tail runs
  __syncthreads();
  // reduce each row slot over the CTA's threads: warp w takes slots w, w + 4, ...
  const int warp = tid >> 5, lane = tid & 31;
  for (int sl = warp; sl < nslots; sl += kBulkThreads / 32) {
    MS m2{-INFINITY, 0.f};
    KeyIdx k2 = key_none();
    for (int i = lane; i < kBulkThreads; i += 32) {
      const float4 d = slot[sl * kBulkThreads + i];
      m2 = ms_combine(m2, MS{d.x, d.y});
      k2 = better(k2, KeyIdx{d.z, __float_as_int(d.w)});
    }
    m2 = warp_ms(m2);
    k2 = warp_best(k2);
    if (lane == 0) part[(size_t)c * SL + sl] = make_float4(m2.m, m2.s, k2.key, __int_as_float(k2.idx));
  }
  // the last CTA checks the requests after its own range, so that the check
  // does not delay the stream
  if (blockIdx.x == gridDim.x - 1) check_requests();
  // ---- the accept tests and the bonus draw of a request run in the CTA that
  // completes its last partial: each CTA counts itself in for every request
  // its range touched (release), and the CTA whose count completes the
  // request's set of covering ranges (acquire) finalizes it with one warp
  __threadfence();
  __syncthreads();
  for (int i = warp; i < nslots; i += kBulkThreads / 32) {
    const int4 ri = rowinfo[i];
    if (i > 0 && rowinfo[i - 1].x == ri.x) continue;  // counted once per request
    int last = 0;
    if (lane == 0) {
      const int b = ri.x;
      const long long r0 = min(max(row_off[b], 0), R), r1 = min(max((long long)row_off[b] + lengths[b], r0), (long long)R);
      // the CTA ranges [c T / G, (c + 1) T / G) that cover the request's
      // units: with T >= G every range holds at least one unit, so they are
      // the owners of its first through its last unit; with T < G a range
      // holds at most one, so there is one per unit
      int ncov = 0;  // 0 (never finalized here) when the request has no rows; CTA 0 reports it
      if (r1 > r0)
        ncov = T >= G ? unit_owner(r1 * nblk - 1, T, G) - unit_owner(r0 * nblk, T, G) + 1
                      : (int)((r1 - r0) * nblk);
      last = atomicAdd(vdone + b, 1) == ncov - 1;
      if (last) {
        __threadfence();
        vdone[b] = 0;  // the last user: ready for the next launch
      }
    }
    if (__shfl_sync(0xFFFFFFFFu, last, 0)) finalize_core(ri.x, fin, rowlen[i].x, rowlen[i].y, R);
  }
}

// Dynamic bulk sweep (V % 64 == 0 and at least 128 blocks per row): the
// packed rows' units are cut into chunks of kBulkUnits (32 KB of P) that the
// CTAs take from a global counter, so a CTA that starts late or streams
// slowly takes fewer chunks and every CTA ends within about a chunk of the
// others. Warp 4 is the producer: it refills a stage as soon as the four
// consumer warps have its data in registers, with the chunk its previous
// take returned (one take ahead, so the counter's round trip hides behind
// the ring). The consumer warps never wait for one another: per chunk each
// thread reduces one block, stores the block's log-sum-exp at its unit
// index (vlse, [rows][nblk] in packed-row order) and each warp writes, for
// its 32 blocks (a "group", g = unit / 32), the per-row (max, sum) to
// part[2 g + slot]. No fence, no random draw and no per-row counting sits
// on the stream, and the stream needs no row table: the bonus row's Gumbel
// keys and the accept tests run in the next kernel (k_verify_fin_dyn), one
// CTA per request, which also clears the counter for the next launch.
constexpr int kDynStages = kBulkStages;
constexpr int kDynConsumers = kBulkThreads / 32;
constexpr int kDynThreads = kBulkThreads + 32;
constexpr int kDynGroup = 32;  // units per partial
constexpr int kFinWarps = 16;  // warps per request in k_verify_fin_dyn
constexpr int kFinRows = 33;   // verified rows a request can have (gamma <= 32, checked when a workspace is made)

size_t sweep_dyn_smem_bytes() { return (size_t)kDynStages * (kBulkFloats * 4 + 2 * 8); }

// (max, sum of exp(x - max)) of one row over the warp: the maximum first,
// then every lane's sum rescaled to it and added (one exponential per lane
// rather than two per combining step).
__device__ __forceinline__ MS warp_ms_maxfirst(MS x) {
  float M = x.m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
  float t = x.m == -INFINITY ? 0.f : x.s * __expf(x.m - M);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
  return MS{M, M == -INFINITY ? 0.f : t};
}

__global__ void __launch_bounds__(kDynThreads)
    k_verify_sweep_dyn(const float* __restrict__ P, const int32_t* __restrict__ row_off, int B, int nblk, int Rmax,
                       float2* __restrict__ part, float* __restrict__ vlse, int* __restrict__ status,
                       int* __restrict__ sched, int pre_nc) {
  extern __shared__ __align__(128) unsigned char smem[];
  float* stage = reinterpret_cast<float*>(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kDynStages * kBulkFloats * 4);  // full[S], empty[S]
  __shared__ int s_chunk[kDynStages];  // chunk in each stage, -1: none (the consumers stop there)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t full0 = tc::smem_u32(bars), empty0 = full0 + 8u * kDynStages, st0 = tc::smem_u32(stage);
  if (tid == 0) {
    for (int i = 0; i < kDynStages; ++i) {
      tc::mbar_init(full0 + 8u * i, 1);
      tc::mbar_init(empty0 + 8u * i, kDynConsumers);
    }
    tc::fence_barrier_init();
  }
  __syncthreads();
  const bool prod = warp == kDynConsumers && lane == 0;
  const uint64_t pol = tc::policy_evict_first();  // P is read once: W2 stays in L2 for the residual pass
  // ---- before the wait: inside a round (pre_nc > 0) the producer takes its
  // first chunks and starts the copies of those below pre_nc, blocks that
  // exist whatever the plan (the planner gives every request a row)
  int first = 0, pending = 0, npre = 0;
  if (prod && pre_nc > 0) {
    first = atomicAdd(sched, kDynStages);  // the first stages' chunks in one take
    pending = atomicAdd(sched, 1);
    for (; npre < kDynStages && first + npre < pre_nc; ++npre) {
      const uint32_t fb = full0 + 8u * npre;
      s_chunk[npre] = first + npre;
      tc::mbar_arrive_expect_tx(fb, (uint32_t)kBulkFloats * 4u);
      tc::bulk_load_hint(st0 + (uint32_t)npre * kBulkFloats * 4u, P + (size_t)(first + npre) * kBulkFloats,
                         (uint32_t)kBulkFloats * 4u, fb, pol);
    }
  }
  pdl_wait();     // the row offsets may be the planner's
  pdl_trigger();  // the finalize's CTAs may become resident and wait for this grid's end
  volatile int never = 0;
  const int R = min(max(row_off[B], 0), Rmax);
  const long long T = (long long)R * nblk;
  const int NC = (int)((T + kBulkUnits - 1) / kBulkUnits);
  if (warp == kDynConsumers) {  // ---- producer
    if (lane != 0) return;
    if (pre_nc <= 0) {
      first = atomicAdd(sched, kDynStages);
      pending = atomicAdd(sched, 1);
    }
    int it = npre;  // stage fills so far
    // (a chunk taken before the wait at or past the end: the consumers stop
    // there, so nothing more is filled)
    const bool stop = npre > 0 && first + npre - 1 >= NC;
    for (; !stop; ++it) {
      const int sidx = it % kDynStages;
      const uint32_t fb = full0 + 8u * sidx;
      if (it >= kDynStages && !tc::mbar_wait(empty0 + 8u * sidx, (it / kDynStages - 1) & 1, &never)) {
        raise_status(status, DSPARK_ETIMEOUT);
        break;
      }
      int c = first + it;
      if (it >= kDynStages) {
        c = pending;
        pending = atomicAdd(sched, 1);
      }
      if (c >= NC) {  // no work left: the consumers stop at this stage
        s_chunk[sidx] = -1;
        tc::mbar_arrive(fb);
        ++it;
        break;
      }
      s_chunk[sidx] = c;
      const long long u = (long long)c * kBulkUnits;
      const int units = (int)min((long long)kBulkUnits, T - u);
      const uint32_t bytes = (uint32_t)units * kBlockW * 4u;
      tc::mbar_arrive_expect_tx(fb, bytes);
      tc::bulk_load_hint(st0 + (uint32_t)sidx * kBulkFloats * 4u, P + u * kBlockW, bytes, fb, pol);
    }
    // the copies of the last fill of each stage have landed before the CTA
    // exits (at once when the consumers took them)
    volatile int nv = 0;
    for (int i = max(it - kDynStages, 0); i < it; ++i)
      tc::mbar_wait(full0 + 8u * (i % kDynStages), (i / kDynStages) & 1, &nv);
    return;
  }
  if (T == 0) return;  // no rows
  // ---- consumers: each warp on its own
  for (int it = 0;; ++it) {
    const int sidx = it % kDynStages;
    if (!tc::mbar_wait(full0 + 8u * sidx, (it / kDynStages) & 1, &never)) {
      if (lane == 0) raise_status(status, DSPARK_ETIMEOUT);
      break;  // this warp releases no more stages: the producer gives up too
    }
    const int c = s_chunk[sidx];
    if (c < 0 || c >= NC) break;  // (a chunk taken before the wait may lie past the end)
    const long long uw = (long long)c * kBulkUnits + (warp << 5), u = uw + lane;  // the warp's group, the lane's unit
    if (uw >= T) {  // the ragged last chunk: a group past the end
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(empty0 + 8u * sidx);
      continue;
    }
    const bool live = u < T;
    const int qa = (int)(uw / nblk);  // the group's first row
    MS ms{-INFINITY, 0.f};
    int slot = 0;
    float4 x[16];
    if (live) {
      const float4* blk4 = reinterpret_cast<const float4*>(stage + (size_t)sidx * kBulkFloats) + tid * 16;
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = blk4[(i + tid) & 15];  // rotated: conflict-free
      slot = (int)(u / nblk) - qa;
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(empty0 + 8u * sidx);  // this warp is done with the stage
    if (live) {
      float m4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) m4[i] = tc::max3f(x[i].x, x[i].y, tc::max3f(x[i].z, x[i].w, -INFINITY));
#pragma unroll
      for (int i = 4; i < 16; ++i) m4[i & 3] = tc::max3f(tc::max3f(m4[i & 3], x[i].x, x[i].y), x[i].z, x[i].w);
      const float m = tc::max3f(fmaxf(m4[0], m4[1]), m4[2], m4[3]);
      if (m != -INFINITY) {
        const unsigned long long l2e = tc::f2pack(tc::kLog2e, tc::kLog2e);
        const unsigned long long nml = tc::f2pack(-m * tc::kLog2e, -m * tc::kLog2e);
        unsigned long long acc0 = 0ull, acc1 = 0ull;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float a0, a1, a2, a3;
          tc::f2unpack(tc::fma2(tc::f2pack(x[i].x, x[i].y), l2e, nml), a0, a1);
          tc::f2unpack(tc::fma2(tc::f2pack(x[i].z, x[i].w), l2e, nml), a2, a3);
          const unsigned long long e01 = tc::f2pack(tc::ex2_ftz(a0), tc::ex2_ftz(a1));
          const unsigned long long e23 = tc::f2pack(tc::ex2_ftz(a2), tc::ex2_ftz(a3));
          acc0 = i == 0 ? e01 : tc::add2(acc0, e01);
          acc1 = i == 0 ? e23 : tc::add2(acc1, e23);
        }
        float s0, s1;
        tc::f2unpack(tc::add2(acc0, acc1), s0, s1);
        const float t = s0 + s1;
        ms = MS{m, t};
      }
      vlse[u] = ms.m == -INFINITY ? -INFINITY : ms.m + logf(ms.s);  // the block's log-sum-exp
    }
    // the group's rows (one, or two where a row ends inside the group)
    const int nslot = (int)(min(uw + 31, T - 1) / nblk) - qa + 1;
    for (int rr = 0; rr < nslot; ++rr) {
      const MS mr = warp_ms_maxfirst(slot == rr ? ms : MS{-INFINITY, 0.f});
      if (lane == 0) part[(size_t)(uw / kDynGroup) * 2 + rr] = make_float2(mr.m, mr.s);
    }
  }
}

// After the dynamic sweep: one CTA per request. The row layout, the draft
// tokens and P at them were final before the sweep began (the sweep waited
// for the kernel before it), so they are read before the wait, while the
// sweep still streams. Then the warps combine the
// group partials of the accept rows 0 .. ell-2 (row j by warp j mod 16) and,
// together, draw the bonus row's block: every block's key is its
// log-sum-exp from the sweep plus its Gumbel draw. Warp 0 runs the accept
// tests and the bonus token draw on these. Block 0 also checks the row
// layout's start and clears the sweep's chunk counter for the next launch.
__global__ void __launch_bounds__(kFinWarps * 32)
    k_verify_fin_dyn(const FinArgs f, int Rmax, int* __restrict__ sched, const float* __restrict__ vlse) {
  __shared__ float4 s_stat[kFinRows];
  __shared__ KeyIdx s_key[kFinWarps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, b = blockIdx.x;
  const int R = min(max(f.row_off[f.B], 0), Rmax);
  const int ell = f.lengths[b], base = f.row_off[b];
  const bool bad = f.anchor[b] < 0 || f.anchor[b] >= f.V || f.row_off[b + 1] != base + ell || ell < 1 ||
                   ell > f.g + 1 || base < 0 || base + ell > R;  // the same for every thread
  FinIn in{0, 0.f, 0.f};
  if (!bad && warp == 0) in = finalize_inputs(b, f, ell, base, R);
  pdl_wait();  // the sweep's partials and block log-sum-exps
  pdl_trigger();
  if (b == 0 && tid == 0) {
    sched[0] = 0;
    if (f.row_off[0] != 0) raise_status(f.status, DSPARK_ERANGE);
  }
  if (bad) {
    if (tid == 0) {
      f.vflag[b] = 0;
      raise_status(f.status, DSPARK_ERANGE);
    }
    return;
  }
  const long long nb = f.nblk;
  const float2* __restrict__ part = reinterpret_cast<const float2*>(f.part);
  for (int j = warp; j < ell - 1; j += kFinWarps) {
    const long long q = base + j;
    const long long g0 = q * nb / kDynGroup, g1 = (q * nb + nb - 1) / kDynGroup;
    MS ms{-INFINITY, 0.f};
    for (long long gb = g0 + lane; gb <= g1; gb += 4 * 32) {  // four partials' loads in flight per lane
      float2 d[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const long long gi = gb + 32 * e;
        d[e] = make_float2(-INFINITY, 0.f);
        if (gi <= g1) d[e] = __ldcg(part + (size_t)gi * 2 + (size_t)(q - gi * kDynGroup / nb));
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) ms = ms_combine(ms, MS{d[e].x, d[e].y});
    }
    ms = warp_ms(ms);
    if (lane == 0) s_stat[j] = make_float4(ms.m, ms.s, -INFINITY, __int_as_float(kNoIdx));
  }
  KeyIdx kb = key_none();
  const float* __restrict__ L = vlse + (size_t)(base + ell - 1) * nb;  // the bonus row's blocks
  for (int k4 = tid; 4 * k4 < (int)nb; k4 += kFinWarps * 32) {  // four blocks per counter draw
    float l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) l[e] = 4 * k4 + e < (int)nb ? __ldcg(L + 4 * k4 + e) : -INFINITY;
    const uint4 w = f.rng.block4(kBonusBlock, b, ell - 1, 4 * k4);
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (l[e] > -INFINITY) kb = better(kb, KeyIdx{l[e] + gumbel(wv[e]), 4 * k4 + e});
  }
  kb = warp_best(kb);
  if (lane == 0) s_key[warp] = kb;
  __syncthreads();
  if (warp == 0) {
    if (lane == 0) {
      KeyIdx best = key_none();
#pragma unroll
      for (int w = 0; w < kFinWarps; ++w) best = better(best, s_key[w]);
      s_stat[ell - 1] = make_float4(-INFINITY, 0.f, best.key, __int_as_float(best.idx));
    }
    __syncwarp();
    FinArgs fr = f;
    fr.rowstat = s_stat;
    finalize_core(b, fr, ell, base, R, in);
  }
}

template <int BF16>
__global__ void __launch_bounds__(256)
    k_resid_blocks(const float* __restrict__ P, const float* __restrict__ U, const void* __restrict__ W1,
                   const void* __restrict__ W2, const int32_t* __restrict__ anchor,
                   const int32_t* __restrict__ tokens, const float* __restrict__ lse, int g, int V, int r,
                   int nblk, const int* __restrict__ vflag, const int32_t* __restrict__ n_acc,
                   const int* __restrict__ vrow, const float* __restrict__ vlset, const float* __restrict__ ovec,
                   Rng rng, float2* __restrict__ rpart, const int* __restrict__ status) {
  extern __shared__ float e[];  // W1[x_n] (Markov head) or o_{n+1} (RNN head), [r]
  __shared__ KeyIdx red_k[8];
  const int b = blockIdx.y, c = blockIdx.x;
  // this round's flags only if every stage so far left the status clear (no
  // kernel running now writes the status, so every thread reads the same)
  if (!vflag[b] || *(volatile const int*)status != 0) return;
  const int n = min(max(n_acc[b], 0), g - 1);
  const int x = n == 0 ? anchor[b] : tokens[(size_t)b * g + (n - 1)];
  for (int i = threadIdx.x; i < r; i += blockDim.x)
    e[i] = ovec ? ovec[((size_t)b * g + n) * r + i] : ld_w(W1, BF16, (size_t)x * r + i);
  __syncthreads();
  const float Ld = lse[(size_t)b * g + n];  // draft position n + 1
  const float Lt = vlset[b];
  const float* Urow = U + ((size_t)b * g + n) * V;
  const float* Prow = P + (size_t)vrow[b] * V;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int per = (nblk + gridDim.x - 1) / gridDim.x;
  KeyIdx kb = key_none();
  for (int s = c * per + warp; s < min(nblk, (c + 1) * per); s += nw) {
    float lw[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int v = s * kBlockW + lane + 32 * h;
      lw[h] = -INFINITY;
      if (v < V) {
        float acc = 0.f;
        for (int i = 0; i < r; ++i) acc = fmaf(e[i], ld_w(W2, BF16, (size_t)i * V + v), acc);
        lw[h] = resid_logw(Prow[v] - Lt, Urow[v] + acc - Ld);
      }
    }
    const float m = warp_max(fmaxf(lw[0], lw[1]));
    if (m == -INFINITY) continue;
    float t = (lw[0] > -INFINITY ? __expf(lw[0] - m) : 0.f) + (lw[1] > -INFINITY ? __expf(lw[1] - m) : 0.f);
    t = warp_sum(t);
    if (lane == 0) kb = better(kb, KeyIdx{m + logf(t) + gumbel(rng.word(kResidBlock, b, n, s)), s});
  }
  kb = warp_best(kb);
  if (lane == 0) red_k[warp] = kb;
  __syncthreads();
  if (threadIdx.x == 0) {
    KeyIdx k2 = red_k[0];
    for (int i = 1; i < nw; ++i) k2 = better(k2, red_k[i]);
    rpart[(size_t)b * gridDim.x + c] = make_float2(k2.key, __int_as_float(k2.idx));
  }
}

template <int BF16>
__global__ void __launch_bounds__(kPickThreads)
    k_resid_pick(const float* __restrict__ P, const float* __restrict__ U, const void* __restrict__ W1,
                 const void* __restrict__ W2, const int32_t* __restrict__ anchor,
                 const int32_t* __restrict__ tokens, const float* __restrict__ lse, int g, int V, int r,
                 int nblk, int nchunk, const int* __restrict__ vflag, const int32_t* __restrict__ n_acc,
                 const int* __restrict__ vrow, const float* __restrict__ vlset, const float* __restrict__ ovec,
                 Rng rng, const float2* __restrict__ rpart, int32_t* __restrict__ next_anchor,
                 const int* __restrict__ status) {
  extern __shared__ float e[];  // [r]
  __shared__ KeyIdx red_k[kPickThreads / 32];
  __shared__ float zpart[kPickThreads / kBlockW][kBlockW];
  __shared__ int s_blk;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
  // the flag, the first rejection and its row are the finalize's, which ended
  // before the block pass began (the block pass waited for it), so they and
  // W1[x_n] (the previous token's row, which does not depend on the drawn
  // block) load before the wait on the block pass
  const int flag = vflag[b];
  const int n = min(max(n_acc[b], 0), g - 1);
  const float* Prow = P + (size_t)min(max(vrow[b], 0), (int)gridDim.x * (g + 1) - 1) * V;
  if (flag) {
    const int x = n == 0 ? anchor[b] : tokens[(size_t)b * g + (n - 1)];
    for (int i = tid; i < r; i += blockDim.x)
      e[i] = ovec ? ovec[((size_t)b * g + n) * r + i] : ld_w(W1, BF16, (size_t)x * r + i);
  }
  pdl_wait();  // the residual block keys are the previous kernel's
  // this round's flags only if every stage so far left the status clear (no
  // kernel running now writes the status, so every thread reads the same)
  if (!flag || *(volatile const int*)status != 0) return;
  if (warp == 0) {
    KeyIdx k2 = key_none();
    for (int i = lane; i < nchunk; i += 32) {
      const float2 p = rpart[(size_t)b * nchunk + i];
      k2 = better(k2, KeyIdx{p.x, __float_as_int(p.y)});
    }
    k2 = warp_best(k2);
    if (lane == 0) s_blk = k2.idx;
  }
  __syncthreads();
  const int sb = s_blk;
  if (sb == kNoIdx) {
    // no positive residual mass (p_t <= p_d everywhere after rounding):
    // draw from p_t of this row itself, with the bonus stream of row n
    KeyIdx kb = key_none();
    for (int s = warp; s < nblk; s += nw) {
      const int v0 = s * kBlockW + lane, v1 = v0 + 32;
      const float x0 = v0 < V ? Prow[v0] : -INFINITY, x1 = v1 < V ? Prow[v1] : -INFINITY;
      const float m = warp_max(fmaxf(x0, x1));
      float t = (v0 < V ? __expf(x0 - m) : 0.f) + (v1 < V ? __expf(x1 - m) : 0.f);
      t = warp_sum(t);
      if (lane == 0) kb = better(kb, KeyIdx{m + logf(t) + gumbel(rng.word(kBonusBlock, b, n, s)), s});
    }
    kb = warp_best(kb);
    if (lane == 0) red_k[warp] = kb;
    __syncthreads();
    if (tid == 0) {
      KeyIdx k2 = red_k[0];
      for (int i = 1; i < nw; ++i) k2 = better(k2, red_k[i]);
      s_blk = k2.idx;
    }
    __syncthreads();
    const int s2 = s_blk;
    if (s2 == kNoIdx) return;  // the row itself has no finite logit
    if (warp == 0) {
      KeyIdx kt = key_none();
      for (int v = s2 * kBlockW + lane; v < min(V, (s2 + 1) * kBlockW); v += 32)
        kt = better(kt, KeyIdx{Prow[v] + gumbel(rng.word(kBonusToken, b, n, v)), v});
      kt = warp_best(kt);
      if (lane == 0) next_anchor[b] = kt.idx;
    }
    return;
  }
  float uz = 0.f, pz = 0.f;
  if (tid < kBlockW && sb * kBlockW + tid < V) {  // issued ahead of the W2 columns, used after the barrier
    uz = U[((size_t)b * g + n) * V + sb * kBlockW + tid];
    pz = Prow[sb * kBlockW + tid];
  }
  {
    // z_v - U = sum_i e_i W2[i, v] for the 64 tokens of the block: 16 groups
    // of K rows, each thread's loads (r / 16 of them) all in flight together
    constexpr int kQ = kPickThreads / kBlockW;
    const int vl = tid & (kBlockW - 1), q = tid >> 6;
    const int v = sb * kBlockW + vl;
    float acc = 0.f;
    if (v < V) {
#pragma unroll 16
      for (int i = q; i < r; i += kQ) acc = fmaf(e[i], ld_w(W2, BF16, (size_t)i * V + v), acc);
    }
    zpart[q][vl] = acc;
  }
  __syncthreads();
  if (tid < kBlockW) {
    const int v = sb * kBlockW + tid;
    KeyIdx kt = key_none();
    if (v < V) {
      float zs = 0.f;
#pragma unroll
      for (int q = 0; q < kPickThreads / kBlockW; ++q) zs += zpart[q][tid];
      const float z = uz + zs;
      const float lw = resid_logw(pz - vlset[b], z - lse[(size_t)b * g + n]);
      if (lw > -INFINITY) kt = KeyIdx{lw + gumbel(rng.word(kResidToken, b, n, v)), v};
    }
    kt = warp_best(kt);
    if (lane == 0) red_k[warp] = kt;
  }
  __syncthreads();
  if (tid == 0) {
    const KeyIdx kt = better(red_k[0], red_k[1]);
    // the block had positive mass when its draw was made; a token from it
    // must exist unless rounding differs between the two passes
    next_anchor[b] = kt.idx == kNoIdx ? sb * kBlockW : kt.idx;
  }
}

template <int BF16>
static cudaError_t verify_impl(const dspark_ws* ws, const VerifyArgs& a, cudaStream_t st, int* launches) {
  const dspark_dims& d = ws->d;
  const Geometry& geo = ws->geo;
  const Rng rng = Rng::make(a.seed, a.round, (uint32_t)ws->b0);
  const bool pdl = ws->pdl != 0;
  const bool dyn = geo.sweep_dyn != 0;
  const FinArgs fin{a.P, a.row_off, a.lengths, a.anchor, a.tokens, a.pd_tok, d.B, d.gamma, d.V, geo.nblk,
                    geo.SL, geo.sweep_grid, rng, ws->s.vpart, a.n_acc, a.next_anchor, ws->s.vflag, ws->s.vrow,
                    ws->s.vlset, ws->s.status, (geo.sweep_bulk && !dyn) ? ws->s.vpx : nullptr, nullptr};
  if (dyn) {  // chunks taken from a counter; the accept tests in a kernel of their own
    cudaError_t e = launch_ex(k_verify_sweep_dyn, dim3(2 * geo.num_sms), dim3(kDynThreads), sweep_dyn_smem_bytes(),
                              st, pdl, a.P, a.row_off, d.B, geo.nblk, d.B * (d.gamma + 1),
                              reinterpret_cast<float2*>(ws->s.vpart), ws->s.vlse, ws->s.status, ws->s.vsched,
                              a.rowtab ? (int)((long long)d.B * geo.nblk / kBulkUnits) : 0);
    if (e != cudaSuccess) return e;
    e = launch_ex(k_verify_fin_dyn, dim3(d.B), dim3(kFinWarps * 32), 0, st, pdl, fin, d.B * (d.gamma + 1),
                  ws->s.vsched, ws->s.vlse);
    if (e != cudaSuccess) return e;
  } else if (geo.sweep_bulk) {  // the finalize runs in the sweep's CTAs
    const cudaError_t e = launch_ex(k_verify_sweep_bulk, dim3(geo.sweep_grid), dim3(kBulkThreads),
                                    sweep_bulk_smem_bytes(geo.SL), st, pdl, a.P, a.row_off, a.lengths, d.B, geo.nblk,
                                    d.B * (d.gamma + 1), geo.SL, rng, ws->s.vpart, ws->s.status, fin, ws->s.vdone,
                                    a.rowtab);
    if (e != cudaSuccess) return e;
    *launches -= 1;
  } else {  // ordinary launches (these kernels do not wait in-kernel)
    k_verify_sweep<<<geo.sweep_grid, kSweepThreads, 0, st>>>(a.P, a.row_off, a.lengths, d.B, d.V, geo.nblk,
                                                            d.B * (d.gamma + 1), geo.SL, rng, ws->s.vpart);
    k_verify_finalize<<<(d.B + 3) / 4, 128, 0, st>>>(fin);
  }
  const bool pdl_resid = pdl && (geo.sweep_bulk || dyn);  // the residual kernels follow a bulk sweep
  const size_t smem = sizeof(float) * d.r;
  int nchunk = kResidChunks;
  if (BF16 && ws->use_tc && geo.resid_tc_ok) {
    // residual block draw on tensor cores (either head): one CTA per SM
    nchunk = geo.num_sms;
    cudaError_t e = launch_resid_tc(ws, a, ws->s.rpart, nchunk, st, pdl_resid);
    if (e != cudaSuccess) return e;
  } else {
    k_resid_blocks<BF16><<<dim3(kResidChunks, d.B), 256, smem, st>>>(
        a.P, a.U, a.W1, a.W2, a.anchor, a.tokens, a.lse, d.gamma, d.V, d.r, geo.nblk, ws->s.vflag, a.n_acc,
        ws->s.vrow, ws->s.vlset, a.ovec, rng, ws->s.rpart, ws->s.status);
  }
  // after the SIMT block pass (an ordinary launch) the pick may still start
  // early: it waits in-kernel
  const cudaError_t e = launch_ex(k_resid_pick<BF16>, dim3(d.B), dim3(kPickThreads), smem, st, pdl_resid, a.P, a.U,
                                  a.W1, a.W2, a.anchor, a.tokens, a.lse, d.gamma, d.V, d.r, geo.nblk, nchunk,
                                  ws->s.vflag, a.n_acc, ws->s.vrow, ws->s.vlset, a.ovec, rng, ws->s.rpart,
                                  a.next_anchor, ws->s.status);
  *launches += 4;
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_verify(const dspark_ws* ws, const VerifyArgs& a, cudaStream_t st, int* launches) {
  if (ws->d.wdtype == DSPARK_BF16) return verify_impl<1>(ws, a, st, launches);
  return verify_impl<0>(ws, a, st, launches);
}

}  // namespace dspark

namespace dspark {
int sweep_dyn_min_blocks() { return kBulkUnits; }
size_t sweep_dyn_parts(long long units) { return (size_t)((units + kDynGroup - 1) / kDynGroup); }
cudaError_t sweep_dyn_configure() {
  return cudaFuncSetAttribute(k_verify_sweep_dyn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sweep_dyn_smem_bytes());
}
cudaError_t sweep_bulk_configure() {
  return cudaFuncSetAttribute(k_verify_sweep_bulk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sweep_bulk_smem_bytes(kBulkMaxSlots));
}
}  // namespace dspark
