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
// Layout: survival values are sorted as 64-bit patterns of non-negative
// doubles (their integer order is their numeric order) with a 32-bit id
// (j-1)*B + b that carries the tie order.
#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace dspark {

constexpr int kPlanThreads = 1024;

constexpr int kRankMaxChunks = 16;  // up to this many 64-element chunks: rank merge, else bitonic

// Padded candidate count: whole 64-element chunks; a power of two when the
// bitonic network sorts them (more than kRankMaxChunks chunks).
__host__ __device__ inline int plan_mp(int M) {
  const int c = (M + 63) / 64 * 64;
  if (c <= 64 * kRankMaxChunks) return c < 64 ? 64 : c;
  int p = 64;
  while (p < M) p <<= 1;
  return p;
}

size_t plan_smem_bytes(const dspark_dims& d) {
  const int Mp = d.mode == DSPARK_STATIC ? 0 : plan_mp(d.B * d.gamma);  // static: counts only
  return (size_t)Mp * (sizeof(unsigned long long) + sizeof(unsigned) + sizeof(double)) +
         sizeof(int) * (size_t)(d.B + 1) + 64;
}

struct PlanSmem {
  unsigned long long* key;  // [Mp] bits of a
  unsigned* id;             // [Mp]
  double* pre;              // [Mp] exclusive prefix sums of sorted a
  int* cnt;                 // [B]
};

// "x goes before y": larger a first, then smaller id
__device__ __forceinline__ bool before(unsigned long long ka, unsigned ia, unsigned long long kb, unsigned ib) {
  return ka > kb || (ka == kb && ia < ib);
}

// Fill and sort the candidates of confidences `c` [B, g]. Returns via smem.
__device__ void sort_candidates(const float* c, int B, int g, int Mp, PlanSmem sm, int* status) {
  const int M = B * g;
  for (int i = threadIdx.x; i < Mp; i += blockDim.x) {
    sm.key[i] = 0ull;
    sm.id[i] = (unsigned)i;  // padding (i >= M) sorts after every candidate, ids stay distinct
  }
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    double a = 1.0;
    for (int j = 1; j <= g; ++j) {
      const float cf = c[(size_t)b * g + (j - 1)];
      if (!(cf >= 0.f && cf <= 1.f)) raise_status(status, DSPARK_ENUMERIC);  // also catches NaN
      a = __dmul_rn(a, (double)cf);
      const int i = (j - 1) * B + b;
      sm.key[i] = (unsigned long long)__double_as_longlong(a);
      sm.id[i] = (unsigned)i;
    }
  }
  __syncthreads();
  (void)M;
  // Bitonic sort into "before" order. A warp keeps a 64-element chunk in
  // registers (lane l: elements 64c + l and 64c + 32 + l), so every stage of
  // stride <= 32 is an in-lane swap or a shuffle with no block barrier; only
  // strides >= 64 go through shared memory, one barrier each.
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  // flat: the 64-wide stage leaves every chunk in "before" order (for the rank
  // merge) instead of alternating directions (for the next bitonic stage)
  auto reg_stages = [&](int size_lo, int size_hi, int s_hi, bool flat) {
    for (int c = warp; c < Mp / 64; c += nwarps) {
      const int e0 = 64 * c + lane, e1 = e0 + 32;
      unsigned long long k0 = sm.key[e0], k1 = sm.key[e1];
      unsigned i0 = sm.id[e0], i1 = sm.id[e1];
      for (int size = size_lo; size <= size_hi; size <<= 1) {
        for (int st = min(size >> 1, s_hi); st > 0; st >>= 1) {
          if (st == 32) {  // e0 and e1 pair up inside the lane; e0 is the lower index
            const bool up = (e0 & size) == 0 || (flat && size == 64);
            if (before(k0, i0, k1, i1) != up) {
              const unsigned long long tk = k0;
              k0 = k1;
              k1 = tk;
              const unsigned ti = i0;
              i0 = i1;
              i1 = ti;
            }
          } else {
            const unsigned long long p0 = __shfl_xor_sync(0xFFFFFFFFu, k0, st), p1 = __shfl_xor_sync(0xFFFFFFFFu, k1, st);
            const unsigned q0 = __shfl_xor_sync(0xFFFFFFFFu, i0, st), q1 = __shfl_xor_sync(0xFFFFFFFFu, i1, st);
            // keep the element that goes first iff (this index is the lower one) == up
            const bool up0 = (e0 & size) == 0 || (flat && size == 64);
            const bool up1 = (e1 & size) == 0 || (flat && size == 64);
            const bool keep0 = ((e0 & st) == 0) == up0;
            const bool keep1 = ((e1 & st) == 0) == up1;
            if (before(k0, i0, p0, q0) != keep0) {
              k0 = p0;
              i0 = q0;
            }
            if (before(k1, i1, p1, q1) != keep1) {
              k1 = p1;
              i1 = q1;
            }
          }
        }
      }
      sm.key[e0] = k0;
      sm.key[e1] = k1;
      sm.id[e0] = i0;
      sm.id[e1] = i1;
    }
    __syncthreads();
  };
  const int nch = Mp / 64;
  reg_stages(2, 64, 32, nch <= kRankMaxChunks);
  if (nch <= kRankMaxChunks) {
    // Every element's place in the sorted whole: its index in its own sorted
    // chunk plus, for every other chunk, how many of that chunk's elements go
    // before it (a branchless binary search over the 64 sorted entries). The
    // order is strict (ids are distinct), so the places are a permutation.
    constexpr int kPer = 64 * kRankMaxChunks / kPlanThreads;
    unsigned long long kx[kPer];
    unsigned ix[kPer];
    int rk[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = threadIdx.x + u * blockDim.x;
      rk[u] = -1;
      if (e < Mp) {
        kx[u] = sm.key[e];
        ix[u] = sm.id[e];
        int r = e & 63;
#pragma unroll 4
        for (int c2 = 0; c2 < nch; ++c2) {
          const unsigned long long* ck = sm.key + 64 * c2;
          const unsigned* ci = sm.id + 64 * c2;
          int q = 0;
#pragma unroll
          for (int st = 32; st > 0; st >>= 1)
            if (before(ck[q + st - 1], ci[q + st - 1], kx[u], ix[u])) q += st;
          if (q == 63 && before(ck[63], ci[63], kx[u], ix[u])) q = 64;
          r += c2 == (e >> 6) ? 0 : q;  // own chunk: e & 63 above
        }
        rk[u] = r;
      }
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kPer; ++u)
      if (rk[u] >= 0) {
        sm.key[rk[u]] = kx[u];
        sm.id[rk[u]] = ix[u];
      }
    __syncthreads();
    return;
  }
  for (int size = 128; size <= Mp; size <<= 1) {
    for (int stride = size >> 1; stride >= 64; stride >>= 1) {
      for (int t = threadIdx.x; t < Mp / 2; t += blockDim.x) {
        const int lo = 2 * t - (t & (stride - 1));
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;  // this half ends in "before" order
        const unsigned long long kl = sm.key[lo], kh = sm.key[hi];
        const unsigned il = sm.id[lo], ih = sm.id[hi];
        const bool swap = up ? before(kh, ih, kl, il) : before(kl, il, kh, ih);
        if (swap) {
          sm.key[lo] = kh;
          sm.key[hi] = kl;
          sm.id[lo] = ih;
          sm.id[hi] = il;
        }
      }
      __syncthreads();
    }
    reg_stages(size, size, 32, false);
  }
}

// pre[m] = sum_{i<m} a_(i) for m = 0..Mp-1 (padding contributes 0). fp64
// adds are scarce on this part, so the sum runs in 64-bit fixed point: each
// a in [0, 1] is rounded to a multiple of 2^-50 (error <= 2^-51 each), the
// integers are summed exactly (total < 2^63 for up to 8192 candidates), and
// each prefix goes back to fp64. The absolute error of pre[m] is below
// m 2^-51 < 4e-12, relative to tau = B + pre >= 1.
__device__ void prefix_sums(int Mp, PlanSmem sm) {
  unsigned long long* fx = reinterpret_cast<unsigned long long*>(sm.pre);
  for (int i = threadIdx.x; i < Mp; i += blockDim.x)
    fx[i] = __double2ull_rn(__longlong_as_double((long long)sm.key[i]) * 0x1p50);
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (Mp + 31) / 32, lo = lane * per, hi = min(lo + per, Mp);
    unsigned long long loc = 0ull;
    for (int i = lo; i < hi; ++i) loc += fx[i];
    unsigned long long incl = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    unsigned long long run = incl - loc;
    for (int i = lo; i < hi; ++i) {
      const unsigned long long v = fx[i];
      fx[i] = run;
      run += v;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < Mp; i += blockDim.x) sm.pre[i] = __ull2double_rn(fx[i]) * 0x1p-50;
  __syncthreads();
}

__device__ __forceinline__ double theta_at(const double* sps, int B, double pre_m, int m) {
  return ((double)B + pre_m) * sps[B + m];
}

__global__ void __launch_bounds__(kPlanThreads)
    k_plan(const float* __restrict__ conf, const double* __restrict__ sps, int B, int g, int mode, int lag,
           float* __restrict__ ring, uint32_t* __restrict__ plan_round, int32_t* __restrict__ lengths,
           int32_t* __restrict__ row_off, int* __restrict__ status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ double warp_bv[32];
  __shared__ int warp_bm[32];
  __shared__ int warp_int[32];
  __shared__ int s_cut;
  __shared__ int s_bestm;
  const int M = B * g;
  const int Mp = mode == DSPARK_STATIC ? 0 : plan_mp(M);  // the layout of plan_smem_bytes
  PlanSmem sm;
  sm.key = reinterpret_cast<unsigned long long*>(smem_raw);
  sm.pre = reinterpret_cast<double*>(sm.key + Mp);
  sm.id = reinterpret_cast<unsigned*>(sm.pre + Mp);
  sm.cnt = reinterpret_cast<int*>(sm.id + Mp);

  for (int b = threadIdx.x; b < B; b += blockDim.x) sm.cnt[b] = 0;
  int cut = 0;
  if (mode != DSPARK_STATIC) {
    // validate the SPS entries the search can reach
    for (int n = 1 + threadIdx.x; n <= B + M; n += blockDim.x)
      if (!(sps[n] > 0.0) || !isfinite(sps[n])) raise_status(status, DSPARK_ENUMERIC);
    const uint32_t t = *plan_round;
    const float* cnow = conf;
    bool lagged = false;
    if (mode == DSPARK_COMPACT_LAGGED) {
      const int depth = lag + 1;
      float* slot = ring + (size_t)(t % depth) * M;
      for (int i = threadIdx.x; i < M; i += blockDim.x) slot[i] = conf[i];
      lagged = t >= (uint32_t)lag;
      __syncthreads();
      if (lagged) {
        // capacity from the confidences of round t - lag: full-path argmax
        const float* clag = ring + (size_t)((t - lag) % depth) * M;
        sort_candidates(clag, B, g, Mp, sm, status);
        prefix_sums(Mp, sm);
        // first maximum of Theta_m, m = 0..M
        double bv = -1.0;
        int bm = 0x7FFFFFFF;
        for (int m = threadIdx.x; m <= M; m += blockDim.x) {
          const double pm = m < Mp ? sm.pre[m] : sm.pre[Mp - 1] + __longlong_as_double((long long)sm.key[Mp - 1]);
          const double th = theta_at(sps, B, pm, m);
          if (th > bv) {
            bv = th;
            bm = m;
          }
        }
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const double ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
          const int om = __shfl_xor_sync(0xFFFFFFFFu, bm, o);
          if (ov > bv || (ov == bv && om < bm)) {
            bv = ov;
            bm = om;
          }
        }
        if (lane == 0) {
          warp_bv[warp] = bv;
          warp_bm[warp] = bm;
        }
        __syncthreads();
        if (warp == 0) {
          const int nw = blockDim.x >> 5;
          bv = lane < nw ? warp_bv[lane] : -1.0;
          bm = lane < nw ? warp_bm[lane] : 0x7FFFFFFF;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const double ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
            const int om = __shfl_xor_sync(0xFFFFFFFFu, bm, o);
            if (ov > bv || (ov == bv && om < bm)) {
              bv = ov;
              bm = om;
            }
          }
          if (lane == 0) s_bestm = bm;
        }
        __syncthreads();
        cut = s_bestm;
        __syncthreads();
      }
    }
    // current candidates in admission order
    sort_candidates(cnow, B, g, Mp, sm, status);
    if (!lagged) {
      prefix_sums(Mp, sm);
      if (threadIdx.x == 0) s_cut = M;
      __syncthreads();
      // Algorithm 1: stop at the first m whose admission does not raise
      // Theta, tested in the threshold form a SPS(n+1) > tau (SPS(n) - SPS(n+1))
      // (same blog, "阈值随负载变化"), which does not absorb a tiny a into tau.
      for (int m = threadIdx.x; m < M; m += blockDim.x) {
        const double a = __longlong_as_double((long long)sm.key[m]);
        const double tau = (double)B + sm.pre[m];
        const double gain = __dmul_rn(a, sps[B + m + 1]);
        const double cost = __dmul_rn(tau, sps[B + m] - sps[B + m + 1]);
        if (!(gain > cost)) atomicMin(&s_cut, m);
      }
      __syncthreads();
      cut = s_cut;
    }
    for (int i = threadIdx.x; i < cut; i += blockDim.x) atomicAdd(&sm.cnt[sm.id[i] % B], 1);
    __syncthreads();
    if (threadIdx.x == 0) *plan_round = t + 1;
  }
  // lengths and their exclusive scan row_off
  __syncthreads();
  {
    const int T = blockDim.x, per = (B + T - 1) / T, lo = threadIdx.x * per;
    int loc = 0;
    for (int b = lo; b < lo + per && b < B; ++b) {
      const int l = mode == DSPARK_STATIC ? g + 1 : 1 + sm.cnt[b];
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
      row_off[b] = run;
      run += mode == DSPARK_STATIC ? g + 1 : 1 + sm.cnt[b];
    }
  }
}

cudaError_t plan_configure() {
  return cudaFuncSetAttribute(k_plan, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
}

cudaError_t launch_plan(const dspark_ws* ws, const float* conf, const double* sps, int32_t* lengths,
                        int32_t* row_off, cudaStream_t st, int* launches) {
  const dspark_dims& d = ws->d;
  k_plan<<<1, kPlanThreads, plan_smem_bytes(d), st>>>(conf, sps, d.B, d.gamma, (int)d.mode, d.lag,
                                                     ws->s.ring, ws->s.plan_round, lengths, row_off,
                                                     ws->s.status);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace dspark
