// k_plan.cu -- confidence-scheduled planner (one CTA, fp64).
//
// "DeepSeek-V4.1 模型结构（6）：解码，DSpark", sections "目标函数" and
// "贪心就能解"; deepseek.csdn.net close reading §5.3 (Algorithm 1):
//   a_{b,j} = prod_{i<=j} c_{b,i}                      (prefix survival)
//   B_tot = sum_b (1 + l_b),  tau = sum_b (1 + sum_{j<=l_b} a_{b,j})
//   Theta = tau * SPS(B_tot)
// Candidates (b, j) are taken in decreasing a (ties: smaller j, then smaller
// b) and admitted one at a time while Theta strictly rises; because a is
// non-increasing in j, the admitted set is a prefix of every request. The
// rise test (tau + a) SPS(n+1) > tau SPS(n) is evaluated in its threshold
// form a SPS(n+1) > tau (SPS(n) - SPS(n+1)) (section "阈值随负载变化").
// The asynchronous planner of the close reading's §8 takes the capacity
// K = argmax_m Theta_m over the whole path (no early stop; first maximum) on
// the confidences of round t - lag, then admits the K best current
// candidates. "spec_dspark" (section "在 SGLang 里"): lengths lie in
// [1, gamma+1] because the anchor is always verified.
//
// Layout: a candidate is its survival value's 64-bit pattern (non-negative
// doubles order like their bit patterns) and the id (j-1)*B + b, which
// carries the tie order. Each request's candidates are already in admission
// order (a is non-increasing in j, ties go to the smaller j), so the sort is a
// merge sort that starts from B sorted runs of gamma: each round merges pairs
// of runs, every element finding its place in the partner run by binary
// search (log2(B) rounds in shared memory, one barrier each). Afterwards
// thread t holds ranks e * 1024 + t, so the prefix sums of the admission path
// are one block scan per slot, and each thread tests its own ranks.
//
// Lagged mode: the capacity of round t is the first maximum of Theta over the
// confidences of round t - lag. It is computed at round t - lag from that
// round's own sort and kept in a ring of lag + 1 capacities, so that every
// round sorts once.
#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace dspark {

constexpr int kPlanThreads = 1024;  // B * gamma <= 8192: up to 8 candidates per thread

__host__ __device__ inline int plan_mp(int M) {
  int p = kPlanThreads;
  while (p < M) p <<= 1;
  return p;
}

// Shared memory of a compact plan: two buffers of M (64-bit value, 32-bit
// id), 64 words of block-reduction scratch, then the per-request counts
// (static mode: the counts only).
__host__ __device__ inline size_t plan_red_offset(int M) {  // in 8-byte words
  return ((size_t)M * 24 + 7) / 8;
}
__host__ __device__ inline size_t plan_cnt_offset(int M) {  // in bytes
  return (plan_red_offset(M) + 64) * 8;
}

size_t plan_smem_bytes(const dspark_dims& d) {
  const size_t cnt = sizeof(int) * (size_t)(d.B + 1);
  if (d.mode == DSPARK_STATIC) return cnt;
  return plan_cnt_offset(d.B * d.gamma) + cnt;
}

// "x goes before y": larger a first, then smaller id
__device__ __forceinline__ bool before(unsigned long long ka, unsigned ia, unsigned long long kb, unsigned ib) {
  return ka > kb || (ka == kb && ia < ib);
}

// Sort the M candidates of confidences c [B, g] into admission order and
// load ranks e * 1024 + t into (k, id). (k0, i0), (k1, i1): two buffers of M
// (value, id).
template <int E>
__device__ __forceinline__ void sort_candidates(const float* __restrict__ c, int B, int g, unsigned long long* k0,
                                                unsigned* i0, unsigned long long* k1, unsigned* i1,
                                                unsigned long long (&k)[E], unsigned (&id)[E], int* status) {
  const int M = B * g, t = threadIdx.x;
  // runs: request b's survival values at positions b * g .. b * g + g - 1;
  // the confidences are staged (coalesced) in the second buffer
  float* stage = reinterpret_cast<float*>(k1);
  for (int i = t; i < M; i += kPlanThreads) stage[i] = c[i];
  __syncthreads();
  for (int b = t; b < B; b += kPlanThreads) {
    double s = 1.0;
    for (int j = 1; j <= g; ++j) {
      const float cf = stage[(size_t)b * g + (j - 1)];
      if (!(cf >= 0.f && cf <= 1.f)) raise_status(status, DSPARK_ENUMERIC);  // also catches NaN
      s = __dmul_rn(s, (double)cf);
      k0[(size_t)b * g + (j - 1)] = (unsigned long long)__double_as_longlong(s);
      i0[(size_t)b * g + (j - 1)] = (unsigned)((j - 1) * B + b);
    }
  }
  __syncthreads();
  // merge rounds: runs of length L = g 2^r at [R L, R L + L) (the last one
  // shorter); thread t keeps position p = t + 1024 u in every round, so its
  // run index at L = g is computed once
  int pr[E];
#pragma unroll
  for (int u = 0; u < E; ++u) pr[u] = (u * kPlanThreads + t) / g;
  unsigned long long* sk = k0;
  unsigned* si = i0;
  unsigned long long* dk = k1;
  unsigned* di = i1;
  int rl = 0;
#pragma unroll 1
  for (int L = g; L < M; L <<= 1, ++rl) {
    int top = 1;  // the largest power of two <= L
    while ((top << 1) <= L) top <<= 1;
#pragma unroll
    for (int u = 0; u < E; ++u) {
      const int p = u * kPlanThreads + t;
      if (p < M) {
        const int R = pr[u] >> rl, i = p - R * L;
        const int s2 = (R ^ 1) * L;
        const int n2 = max(0, min(L, M - s2));
        const unsigned long long mk = sk[p];
        const unsigned mi = si[p];
        // count of the partner run's elements that go before this one
        // (the run is in admission order): a branchless binary search
        int q = 0;
        for (int step = top; step > 0; step >>= 1)
          if (q + step <= n2 && before(sk[s2 + q + step - 1], si[s2 + q + step - 1], mk, mi)) q += step;
        dk[(R & ~1) * L + i + q] = mk;
        di[(R & ~1) * L + i + q] = mi;
      }
    }
    __syncthreads();
    unsigned long long* tk = sk;
    sk = dk;
    dk = tk;
    unsigned* ti = si;
    si = di;
    di = ti;
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int r = e * kPlanThreads + t;
    k[e] = r < M ? sk[r] : 0ull;
    id[e] = r < M ? si[r] : 0xFFFFFFFFu;
  }
  __syncthreads();  // the buffers are free for the caller
}

// The fp64 pipe of this part is narrow, so the fixed-point conversions below
// are integer arithmetic on the bit patterns.
// a in [0, 1] (its fp64 bit pattern) times 2^50, rounded to the nearest
// integer (ties to even): a = m 2^(E - 1075) with the 53-bit significand m,
// so a 2^50 = m / 2^(1025 - E).
__device__ __forceinline__ unsigned long long fixed50_of(unsigned long long bits) {
  const int E = (int)(bits >> 52);
  const int s = 1025 - E;  // >= 2 for a <= 1
  if (E == 0 || s >= 54) return 0ull;  // below 2^-51: rounds to 0
  const unsigned long long m = (bits & ((1ull << 52) - 1)) | (1ull << 52);
  const unsigned long long q = m >> s, r = m & ((1ull << s) - 1), half = 1ull << (s - 1);
  return q + ((r > half || (r == half && (q & 1ull))) ? 1ull : 0ull);
}

// x 2^-50 for an integer x < 2^64, rounded to the nearest double (ties to
// even).
__device__ __forceinline__ double double_of_fixed50(unsigned long long x) {
  if (x == 0ull) return 0.0;
  const int nb = 64 - __clzll((long long)x);  // bits in x
  unsigned long long m;
  int e;  // x 2^-50 = m 2^e with m < 2^53
  if (nb <= 53) {
    m = x;
    e = -50;
  } else {
    const int s = nb - 53;
    const unsigned long long q = x >> s, r = x & ((1ull << s) - 1), half = 1ull << (s - 1);
    m = q + ((r > half || (r == half && (q & 1ull))) ? 1ull : 0ull);  // may reach 2^53: still exact
    e = s - 50;
  }
  // m 2^e: normalise m to [2^52, 2^53] and build the pattern
  const int lz = __clzll((long long)m) - 11;  // shift that puts the leading one at bit 52
  if (lz >= 0) {
    m <<= lz;
    e -= lz;
  } else {  // m = 2^53 after rounding
    m >>= 1;
    e += 1;
  }
  const unsigned long long bits = ((unsigned long long)(e + 52 + 1023) << 52) | (m & ((1ull << 52) - 1));
  return __longlong_as_double((long long)bits);
}

// Exclusive prefix sums of the sorted survival values in rank order, in
// 2^-50 fixed point: each a in [0, 1] is rounded to a multiple of 2^-50
// (error <= 2^-51 each) and the integers are summed exactly (total < 2^63 for
// up to 8192 candidates), so the sums do not depend on the order of the adds;
// the absolute error of a prefix is below m 2^-51 < 4e-12, relative to
// tau = B + prefix >= 1. Returns the total through *total (every thread).
template <int E>
__device__ __forceinline__ void prefix_fixed(const unsigned long long (&k)[E], unsigned long long (&pre)[E], unsigned long long* red,
                             unsigned long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long carry = 0ull;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const unsigned long long x = fixed50_of(k[e]);
    unsigned long long incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) red[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const unsigned long long w = red[lane];
      unsigned long long wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, wi, o);
        if (lane >= o) wi += y;
      }
      red[lane] = wi - w;  // exclusive over warps
      if (lane == 31) red[32] = wi;
    }
    __syncthreads();
    pre[e] = carry + red[warp] + (incl - x);
    carry += red[32];
    __syncthreads();  // red is reused by the next slot
  }
  *total = carry;
}

// tau = B + (a prefix in 2^-50 fixed point), formed exactly in fixed point
// (B 2^50 + prefix < 2^62 + 2^63) and rounded once
__device__ __forceinline__ double tau_of(int B, unsigned long long pre) {
  return double_of_fixed50(((unsigned long long)B << 50) + pre);
}

// Block-wide first maximum of (v, m): larger v, then smaller m.
__device__ __forceinline__ int block_argmax_first(double v, int m, double* rv, int* rm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double ov = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int om = __shfl_xor_sync(0xFFFFFFFFu, m, o);
    if (ov > v || (ov == v && om < m)) {
      v = ov;
      m = om;
    }
  }
  if (lane == 0) {
    rv[warp] = v;
    rm[warp] = m;
  }
  __syncthreads();
  if (warp == 0) {
    v = rv[lane];
    m = rm[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const double ov = __shfl_xor_sync(0xFFFFFFFFu, v, o);
      const int om = __shfl_xor_sync(0xFFFFFFFFu, m, o);
      if (ov > v || (ov == v && om < m)) {
        v = ov;
        m = om;
      }
    }
    if (lane == 0) rm[32] = m;
  }
  __syncthreads();
  const int r = rm[32];
  __syncthreads();
  return r;
}

__device__ __forceinline__ int block_min(int x, int* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = min(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
  if (lane == 0) red[warp] = x;
  __syncthreads();
  if (warp == 0) {
    x = red[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = min(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
    if (lane == 0) red[32] = x;
  }
  __syncthreads();
  const int r = red[32];
  __syncthreads();
  return r;
}

// SPS(B + m) and SPS(B + m + 1) of rank m (1.0 where the path does not reach)
__device__ __forceinline__ void sps_of(const double* __restrict__ sps, int B, int M, int m, double& a0, double& a1) {
  a0 = m <= M ? __ldg(sps + B + m) : 1.0;
  a1 = m < M ? __ldg(sps + B + m + 1) : 1.0;
}

template <int E>
__device__ __forceinline__ void plan_compact(const float* __restrict__ conf, const double* __restrict__ sps, int B,
                                             int g, int mode, int lag, int32_t* __restrict__ kring,
                                             uint32_t* __restrict__ plan_round, int* cnt, unsigned char* smem,
                                             int* __restrict__ status) {
  const int M = B * g, t = threadIdx.x;
  unsigned long long* k0 = reinterpret_cast<unsigned long long*>(smem);
  unsigned long long* k1 = k0 + M;
  unsigned* i0 = reinterpret_cast<unsigned*>(k1 + M);
  unsigned* i1 = i0 + M;
  unsigned long long* red = reinterpret_cast<unsigned long long*>(smem) + plan_red_offset(M);  // 64 words
  // the SPS entries of this thread's ranks m = e * 1024 + t, SPS(B + m) and
  // SPS(B + m + 1): fixed by the layout, so with up to two candidates per
  // thread they load while the candidates are sorted (more would spill
  // registers; those load after the sort); every entry the search can reach
  // is checked
  constexpr bool kEarly = E <= 2;
  double s0[kEarly ? E : 1], s1[kEarly ? E : 1];
  if constexpr (kEarly) {
#pragma unroll
    for (int e = 0; e < E; ++e) sps_of(sps, B, M, e * kPlanThreads + t, s0[e], s1[e]);
  }
  for (int n = 1 + t; n <= B + M; n += kPlanThreads)
    if (!(sps[n] > 0.0) || !isfinite(sps[n])) raise_status(status, DSPARK_ENUMERIC);
  const double sB = t == 0 ? __ldg(sps + B + M) : 0.0;  // Theta at m = M uses SPS(B + M)
  pdl_wait();  // the confidences are the draft's

  const uint32_t rt = *plan_round;
  const bool lagged = mode == DSPARK_COMPACT_LAGGED;
  unsigned long long k[E];
  unsigned id[E];
  unsigned long long pre[E];
  sort_candidates<E>(conf, B, g, k0, i0, k1, i1, k, id, status);
  unsigned long long tot;
  prefix_fixed<E>(k, pre, red, &tot);
  int cut = M;
  if (lagged) {
    // this round's capacity was taken lag rounds ago (the first lag rounds
    // after a reset plan synchronously); the capacity of round rt + lag is the
    // first maximum of Theta_m over m = 0..M on this round's candidates
    const int depth = lag + 1;
    double bv = -1.0;
    int bm = 0x7FFFFFFF;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int m = e * kPlanThreads + t;
      if (m < M) {
        double a0, a1;
        if constexpr (kEarly) {
          a0 = s0[e];
        } else {
          sps_of(sps, B, M, m, a0, a1);
        }
        const double th = __dmul_rn(tau_of(B, pre[e]), a0);
        if (th > bv) {
          bv = th;
          bm = m;
        }
      }
    }
    if (t == 0) {  // m = M: every candidate admitted
      const double th = __dmul_rn(tau_of(B, tot), sB);
      if (th > bv || (th == bv && M < bm)) {
        bv = th;
        bm = M;
      }
    }
    const int K = block_argmax_first(bv, bm, reinterpret_cast<double*>(red), reinterpret_cast<int*>(red + 33));
    if (rt >= (uint32_t)lag) cut = kring[(rt - lag) % depth];  // written lag launches ago
    if (t == 0) kring[rt % depth] = K;
  }
  if (!lagged || rt < (uint32_t)lag) {
    // Algorithm 1: stop at the first m whose admission does not raise Theta,
    // tested in the threshold form a SPS(n+1) > tau (SPS(n) - SPS(n+1)) (same
    // blog, "阈值随负载变化"), which does not absorb a tiny a into tau
    int first = M;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int m = e * kPlanThreads + t;
      if (m < M) {
        double a0, a1;
        if constexpr (kEarly) {
          a0 = s0[e];
          a1 = s1[e];
        } else {
          sps_of(sps, B, M, m, a0, a1);
        }
        const double a = __longlong_as_double((long long)k[e]);
        const double tau = tau_of(B, pre[e]);
        const double gain = __dmul_rn(a, a1);
        const double cost = __dmul_rn(tau, a0 - a1);
        if (!(gain > cost)) first = min(first, m);
      }
    }
    cut = block_min(first, reinterpret_cast<int*>(red));
  }
  cut = min(max(cut, 0), M);
  // admitted: ranks below the cut; each adds one verified draft to its request
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (e * kPlanThreads + t < cut) atomicAdd(&cnt[id[e] % B], 1);
  if (t == 0) *plan_round = rt + 1;
  __syncthreads();
}

__global__ void __launch_bounds__(kPlanThreads)
    k_plan(const float* __restrict__ conf, const double* __restrict__ sps, int B, int g, int mode, int lag,
           int32_t* __restrict__ kring, uint32_t* __restrict__ plan_round, int32_t* __restrict__ lengths,
           int32_t* __restrict__ row_off, int4* __restrict__ rowtab, int* __restrict__ status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int warp_int[32];
  const int M = B * g;
  const bool compact = mode != DSPARK_STATIC;
  // the layout of plan_smem_bytes
  int* cnt = reinterpret_cast<int*>(smem_raw + (compact ? plan_cnt_offset(M) : 0));
  for (int b = threadIdx.x; b < B; b += blockDim.x) cnt[b] = 0;
  __syncthreads();
  if (!compact) pdl_wait();  // lengths are written below
  if (compact) {
    switch (plan_mp(M) / kPlanThreads) {
      case 1: plan_compact<1>(conf, sps, B, g, mode, lag, kring, plan_round, cnt, smem_raw, status); break;
      case 2: plan_compact<2>(conf, sps, B, g, mode, lag, kring, plan_round, cnt, smem_raw, status); break;
      case 4: plan_compact<4>(conf, sps, B, g, mode, lag, kring, plan_round, cnt, smem_raw, status); break;
      default: plan_compact<8>(conf, sps, B, g, mode, lag, kring, plan_round, cnt, smem_raw, status); break;
    }
  }
  // lengths and their exclusive scan row_off
  pdl_trigger();  // the sweep may be scheduled while this tail runs
  {
    const int T = blockDim.x, per = (B + T - 1) / T, lo = threadIdx.x * per;
    int loc = 0;
    for (int b = lo; b < lo + per && b < B; ++b) {
      const int l = mode == DSPARK_STATIC ? g + 1 : 1 + cnt[b];
      lengths[b] = l;
      loc += l;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_int[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int nw = T >> 5;
      const int x = lane < nw ? warp_int[lane] : 0;
      int inc = x;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += y;
      }
      if (lane < nw) warp_int[lane] = inc - x;
      if (lane == nw - 1) row_off[B] = inc;
    }
    __syncthreads();
    int run = warp_int[warp] + (incl - loc);
    for (int b = lo; b < lo + per && b < B; ++b) {
      const int l = mode == DSPARK_STATIC ? g + 1 : 1 + cnt[b];
      row_off[b] = run;
      if (rowtab)
        for (int j = 0; j < l; ++j) rowtab[run + j] = make_int4(b, j, l, run);
      run += l;
    }
  }
}

cudaError_t plan_configure() {
  return cudaFuncSetAttribute(k_plan, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
}

cudaError_t launch_plan(const dspark_ws* ws, const float* conf, const double* sps, int32_t* lengths,
                        int32_t* row_off, int4* rowtab, cudaStream_t st, int* launches) {
  const dspark_dims& d = ws->d;
  const cudaError_t e = launch_ex(k_plan, dim3(1), dim3(kPlanThreads), plan_smem_bytes(d), st, ws->pdl != 0, conf,
                                  sps, d.B, d.gamma, (int)d.mode, d.lag, ws->s.kring, ws->s.plan_round, lengths,
                                  row_off, rowtab, ws->s.status);
  ++*launches;
  return e;
}

__global__ void k_plan_slice(const int32_t* __restrict__ lengths, const int32_t* __restrict__ row_off, int b_begin,
                             int n, int32_t* __restrict__ lengths_l, int32_t* __restrict__ row_off_l) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i > n) return;
  const int32_t base = row_off[b_begin];
  row_off_l[i] = row_off[b_begin + i] - base;
  if (i < n) lengths_l[i] = lengths[b_begin + i];
}

cudaError_t launch_plan_slice(const int32_t* lengths, const int32_t* row_off, int b_begin, int n, int32_t* lengths_l,
                              int32_t* row_off_l, cudaStream_t st, int* launches) {
  k_plan_slice<<<(n + 1 + 255) / 256, 256, 0, st>>>(lengths, row_off, b_begin, n, lengths_l, row_off_l);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace dspark
