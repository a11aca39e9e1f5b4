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
//   k_verify_sweep     persistent grid-stride over (row, chunk) items: online
//                      log-sum-exp of P; for the last verified row of a
//                      request also the block draw of the bonus token.
//   k_verify_finalize  one warp per request: accept tests, first rejection,
//                      bonus token draw inside its block.
//   k_resid_blocks     grid (chunks, B): residual block masses and block draw.
//   k_resid_pick       grid (B): residual token draw inside the drawn block.
#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace dspark {

constexpr int kSweepThreads = 256;

__device__ __forceinline__ int request_of_row(const int32_t* __restrict__ row_off, int B, int q) {
  int lo = 0, hi = B - 1;  // largest b with row_off[b] <= q
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (row_off[mid] <= q) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kSweepThreads)
    k_verify_sweep(const float* __restrict__ P, const int32_t* __restrict__ row_off,
                   const int32_t* __restrict__ lengths, int B, int V, int S, int chunk, int Rmax, Rng rng,
                   float4* __restrict__ part) {
  __shared__ MS red_ms[kSweepThreads / 32];
  __shared__ KeyIdx red_k[kSweepThreads / 32];
  const int R = min(max(row_off[B], 0), Rmax);  // finalize reports an inconsistent row_off
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int item = blockIdx.x; item < R * S; item += gridDim.x) {
    const int q = item / S, sp = item - q * S;
    const int b = request_of_row(row_off, B, q);
    const int j = q - row_off[b];
    const bool bonus = j == lengths[b] - 1;
    const int lo = sp * chunk, hi = min(V, lo + chunk);
    const float* row = P + (size_t)q * V;
    MS ms{-INFINITY, 0.f};
    KeyIdx kb = key_none();
    // each warp takes whole 64-token blocks: lanes read v and v + 32
    for (int s0 = lo / kBlockW + warp; s0 * kBlockW < hi; s0 += nw) {
      const int v0 = s0 * kBlockW + lane, v1 = v0 + 32;
      const float x0 = v0 < hi ? __ldcs(row + v0) : -INFINITY;
      const float x1 = v1 < hi ? __ldcs(row + v1) : -INFINITY;
      if (bonus) {
        const float m = warp_max(fmaxf(x0, x1));
        if (m == -INFINITY) continue;  // a fully masked block has no mass
        float t = (v0 < hi ? __expf(x0 - m) : 0.f) + (v1 < hi ? __expf(x1 - m) : 0.f);
        t = warp_sum(t);
        const MS blk{m, t};
        if (lane == 0) {
          ms = ms_combine(ms, blk);
          kb = better(kb, KeyIdx{m + logf(t) + gumbel(rng.word(kBonusBlock, b, j, s0)), s0});
        }
      } else {
        const float m = fmaxf(fmaxf(x0, x1), ms.m);
        if (m == -INFINITY) continue;
        float t = ms.m == -INFINITY ? 0.f : ms.s * __expf(ms.m - m);
        if (v0 < hi) t += __expf(x0 - m);
        if (v1 < hi) t += __expf(x1 - m);
        ms = MS{m, t};
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
      if (lane == 0) part[item] = make_float4(m2.m, m2.s, k2.key, __int_as_float(k2.idx));
    }
    __syncthreads();
  }
}

// Vectorised sweep for V % 4 == 0 (rows 16-byte aligned): each thread streams
// float4 values, four loads in flight per thread; a half-warp holds one
// 64-token block per load, so the bonus row's block masses need only
// 16-lane shuffles.
constexpr int kSweepUnroll = 4;

__global__ void __launch_bounds__(kSweepThreads)
    k_verify_sweep4(const float* __restrict__ P, const int32_t* __restrict__ row_off,
                    const int32_t* __restrict__ lengths, int B, int V, int S, int chunk, int Rmax, Rng rng,
                    float4* __restrict__ part) {
  __shared__ MS red_ms[kSweepThreads / 32];
  __shared__ KeyIdx red_k[kSweepThreads / 32];
  const int R = min(max(row_off[B], 0), Rmax);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int V4 = V >> 2;
  for (int item = blockIdx.x; item < R * S; item += gridDim.x) {
    const int q = item / S, sp = item - q * S;
    const int b = request_of_row(row_off, B, q);
    const int j = q - row_off[b];
    const bool bonus = j == lengths[b] - 1;
    const int lo4 = (sp * chunk) >> 2, hi4 = min(V4, lo4 + (chunk >> 2));
    const float4* row = reinterpret_cast<const float4*>(P + (size_t)q * V);
    MS ms{-INFINITY, 0.f};
    KeyIdx kb = key_none();
    // uniform trip count across the CTA: the bonus branch shuffles over full warps
    for (int base = lo4; base < hi4; base += kSweepUnroll * kSweepThreads) {
      const int f0 = base + threadIdx.x;
      float4 x[kSweepUnroll];
#pragma unroll
      for (int u = 0; u < kSweepUnroll; ++u) {
        const int f = f0 + u * kSweepThreads;
        x[u] = f < hi4 ? __ldcs(row + f) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int u = 0; u < kSweepUnroll; ++u) {
        const float m4 = fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w));
        if (bonus) {
          // this half-warp's 16 float4 are one 64-token block
          float m = m4;
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
          float t = 0.f;
          if (m != -INFINITY)
            t = __expf(x[u].x - m) + __expf(x[u].y - m) + __expf(x[u].z - m) + __expf(x[u].w - m);
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
          const int f = f0 + u * kSweepThreads;
          if ((lane & 15) == 0 && f < hi4 && m != -INFINITY) {
            const int s0 = f >> 4;  // 16 float4 per block
            ms = ms_combine(ms, MS{m, t});
            kb = better(kb, KeyIdx{m + logf(t) + gumbel(rng.word(kBonusBlock, b, j, s0)), s0});
          }
        } else if (m4 != -INFINITY) {
          const float m = fmaxf(m4, ms.m);
          float t = ms.m == -INFINITY ? 0.f : ms.s * __expf(ms.m - m);
          t += __expf(x[u].x - m) + __expf(x[u].y - m) + __expf(x[u].z - m) + __expf(x[u].w - m);
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
      if (lane == 0) part[item] = make_float4(m2.m, m2.s, k2.key, __int_as_float(k2.idx));
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(128)
    k_verify_finalize(const float* __restrict__ P, const int32_t* __restrict__ row_off,
                      const int32_t* __restrict__ lengths, const int32_t* __restrict__ anchor,
                      const int32_t* __restrict__ tokens,
                      const float* __restrict__ pd_tok, int B, int g, int V, int S, Rng rng,
                      const float4* __restrict__ part, int32_t* __restrict__ n_acc,
                      int32_t* __restrict__ next_anchor, int* __restrict__ vflag, int* __restrict__ vrow,
                      float* __restrict__ vlset, int* __restrict__ status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * (blockDim.x >> 5) + warp;
  if (b >= B) return;
  if (lane == 0) vflag[b] = 0;  // no residual pass unless a rejection is found below
  const int ell = lengths[b], base = row_off[b];
  const int Rmax = B * (g + 1);
  if (ell < 1 || ell > g + 1 || base < 0 || base + ell > Rmax || base + ell > row_off[B] ||
      anchor[b] < 0 || anchor[b] >= V) {
    if (lane == 0) raise_status(status, DSPARK_ERANGE);
    return;
  }
  int n = ell - 1;
  bool rejected = false;
  float lset = 0.f;
  for (int j = 0; j < ell - 1; ++j) {
    const size_t q = (size_t)base + j;
    MS ms{-INFINITY, 0.f};
    for (int i = lane; i < S; i += 32) {
      const float4 p = part[q * S + i];
      ms = ms_combine(ms, MS{p.x, p.y});
    }
    ms = warp_ms(ms);
    const float Lt = ms_log(ms);
    if (!isfinite(Lt)) {
      if (lane == 0) raise_status(status, DSPARK_ENUMERIC);
      return;
    }
    const int x = tokens[(size_t)b * g + j];
    if (x < 0 || x >= V) {
      if (lane == 0) raise_status(status, DSPARK_ERANGE);
      return;
    }
    const float pt = expf(P[q * V + x] - Lt);
    const float u = u01(rng.word(kAccept, b, j, 0));
    if (!(u * pd_tok[(size_t)b * g + j] < pt)) {
      n = j;
      rejected = true;
      lset = Lt;
      break;
    }
  }
  if (rejected) {
    if (lane == 0) {
      n_acc[b] = n;
      vflag[b] = 1;
      vrow[b] = base + n;
      vlset[b] = lset;
    }
    return;
  }
  // bonus token from row ell - 1: the block draw was made by the sweep
  const size_t q = (size_t)base + n;
  KeyIdx kb = key_none();
  for (int i = lane; i < S; i += 32) {
    const float4 p = part[q * S + i];
    kb = better(kb, KeyIdx{p.z, __float_as_int(p.w)});
  }
  kb = warp_best(kb);
  if (kb.idx == kNoIdx) {
    if (lane == 0) raise_status(status, DSPARK_ENUMERIC);
    return;
  }
  KeyIdx kt = key_none();
  for (int v = kb.idx * kBlockW + lane; v < min(V, (kb.idx + 1) * kBlockW); v += 32)
    kt = better(kt, KeyIdx{P[q * V + v] + gumbel(rng.word(kBonusToken, b, n, v)), v});
  kt = warp_best(kt);
  if (lane == 0) {
    n_acc[b] = n;
    next_anchor[b] = kt.idx;
    vflag[b] = 0;
  }
}

// log of the residual weight max(0, p_t - p_d) of one token, written as
// log p_t + log(-expm1(log p_d - log p_t)) so that near-equal p_t and p_d keep
// their relative precision; -inf when p_t <= p_d.
__device__ __forceinline__ float resid_logw(float lpt, float lpd) {
  if (!(lpt > lpd)) return -INFINITY;
  return lpt + logf(-expm1f(lpd - lpt));
}

template <int BF16>
__global__ void __launch_bounds__(256)
    k_resid_blocks(const float* __restrict__ P, const float* __restrict__ U, const void* __restrict__ W1,
                   const void* __restrict__ W2, const int32_t* __restrict__ anchor,
                   const int32_t* __restrict__ tokens, const float* __restrict__ lse, int g, int V, int r,
                   int nblk, const int* __restrict__ vflag, const int32_t* __restrict__ n_acc,
                   const int* __restrict__ vrow, const float* __restrict__ vlset, Rng rng,
                   float2* __restrict__ rpart) {
  extern __shared__ float e[];  // W1[x_n], [r]
  __shared__ KeyIdx red_k[8];
  const int b = blockIdx.y, c = blockIdx.x;
  if (!vflag[b]) return;
  const int n = n_acc[b];
  const int x = n == 0 ? anchor[b] : tokens[(size_t)b * g + (n - 1)];
  for (int i = threadIdx.x; i < r; i += blockDim.x) e[i] = ld_w(W1, BF16, (size_t)x * r + i);
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
__global__ void __launch_bounds__(256)
    k_resid_pick(const float* __restrict__ P, const float* __restrict__ U, const void* __restrict__ W1,
                 const void* __restrict__ W2, const int32_t* __restrict__ anchor,
                 const int32_t* __restrict__ tokens, const float* __restrict__ lse, int g, int V, int r,
                 int nblk, int nchunk, const int* __restrict__ vflag, const int32_t* __restrict__ n_acc,
                 const int* __restrict__ vrow, const float* __restrict__ vlset, Rng rng,
                 const float2* __restrict__ rpart, int32_t* __restrict__ next_anchor) {
  extern __shared__ float e[];  // [r]
  __shared__ KeyIdx red_k[8];
  __shared__ float zpart[4][kBlockW];
  __shared__ int s_blk;
  const int b = blockIdx.x;
  if (!vflag[b]) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
  const int n = n_acc[b];
  const float* Prow = P + (size_t)vrow[b] * V;
  if (tid == 0) {
    KeyIdx k2 = key_none();
    for (int i = 0; i < nchunk; ++i) {
      const float2 p = rpart[(size_t)b * nchunk + i];
      k2 = better(k2, KeyIdx{p.x, __float_as_int(p.y)});
    }
    s_blk = k2.idx;
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
  const int x = n == 0 ? anchor[b] : tokens[(size_t)b * g + (n - 1)];
  for (int i = tid; i < r; i += blockDim.x) e[i] = ld_w(W1, BF16, (size_t)x * r + i);
  __syncthreads();
  {
    const int vl = tid & (kBlockW - 1), q = tid >> 6;
    const int v = sb * kBlockW + vl;
    if (q < 4) {
      float acc = 0.f;
      if (v < V)
        for (int i = q; i < r; i += 4) acc = fmaf(e[i], ld_w(W2, BF16, (size_t)i * V + v), acc);
      zpart[q][vl] = acc;
    }
  }
  __syncthreads();
  if (tid < kBlockW) {
    const int v = sb * kBlockW + tid;
    KeyIdx kt = key_none();
    if (v < V) {
      const float z = U[((size_t)b * g + n) * V + v] + ((zpart[0][tid] + zpart[1][tid]) + (zpart[2][tid] + zpart[3][tid]));
      const float lw = resid_logw(Prow[v] - vlset[b], z - lse[(size_t)b * g + n]);
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
  const Rng rng = Rng::make(a.seed, a.round);
  const int grid = geo.num_sms * 8;
  if ((d.V & 3) == 0)
    k_verify_sweep4<<<grid, kSweepThreads, 0, st>>>(a.P, a.row_off, a.lengths, d.B, d.V, geo.S, geo.chunk,
                                                    d.B * (d.gamma + 1), rng, ws->s.vpart);
  else
    k_verify_sweep<<<grid, kSweepThreads, 0, st>>>(a.P, a.row_off, a.lengths, d.B, d.V, geo.S, geo.chunk,
                                                   d.B * (d.gamma + 1), rng, ws->s.vpart);
  k_verify_finalize<<<(d.B + 3) / 4, 128, 0, st>>>(a.P, a.row_off, a.lengths, a.anchor, a.tokens, a.pd_tok, d.B, d.gamma,
                                                   d.V, geo.S, rng, ws->s.vpart, a.n_acc, a.next_anchor,
                                                   ws->s.vflag, ws->s.vrow, ws->s.vlset, ws->s.status);
  const size_t smem = sizeof(float) * d.r;
  int nchunk = kResidChunks;
  if (BF16 && ws->use_tc && geo.resid_tc_ok) {
    // residual block draw on tensor cores: one CTA per SM
    nchunk = geo.num_sms;
    cudaError_t e = launch_resid_tc(ws, a, ws->s.rpart, nchunk, st);
    if (e != cudaSuccess) return e;
  } else {
    k_resid_blocks<BF16><<<dim3(kResidChunks, d.B), 256, smem, st>>>(
        a.P, a.U, a.W1, a.W2, a.anchor, a.tokens, a.lse, d.gamma, d.V, d.r, geo.nblk, ws->s.vflag, a.n_acc,
        ws->s.vrow, ws->s.vlset, rng, ws->s.rpart);
  }
  k_resid_pick<BF16><<<d.B, 256, smem, st>>>(a.P, a.U, a.W1, a.W2, a.anchor, a.tokens, a.lse, d.gamma, d.V,
                                             d.r, geo.nblk, nchunk, ws->s.vflag, a.n_acc, ws->s.vrow,
                                             ws->s.vlset, rng, ws->s.rpart, a.next_anchor);
  *launches += 4;
  return cudaGetLastError();
}

cudaError_t launch_verify(const dspark_ws* ws, const VerifyArgs& a, cudaStream_t st, int* launches) {
  if (ws->d.wdtype == DSPARK_BF16) return verify_impl<1>(ws, a, st, launches);
  return verify_impl<0>(ws, a, st, launches);
}

}  // namespace dspark
