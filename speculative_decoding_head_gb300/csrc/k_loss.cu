// k_loss.cu -- the draft head's teacher-forced training objective.
//
// "DeepSeek-V4.1 模型结构（6）：解码，DSpark", section on training (optimise the
// acceptance rate directly); deepseek.csdn.net reading §6, eqs. (9)-(12);
// "DSpark：不让大模型更聪明，而让它「吐字更快」" §07. Teacher forcing makes
// every position (b, k) independent: position k drafts from x*_{k-1} (the
// anchor at k = 0), so with z_d = U[b, k] + W1[x_prev] W2, p_d = softmax(z_d)
// and p_t = softmax(P[b, k]):
//   ce  = lse(z_d) - z_d[x*_k]                                   (9)
//   l1  = sum_v |p_d(v) - p_t(v)|                                 (10)
//   c*  = 1 - l1 / 2, bce = -(c* log c + (1 - c*) log(1 - c))     (11)
//   loss = (1/B) sum_{b,k} exp(-k / tau) (0.1 ce + 0.9 l1 + bce)  (12)
//
// Five launches. The two vocabulary passes are the tcgen05 kernel of
// k_resid_tc.cu with every position as an MMA column: pass 0 leaves per CTA
// the (max, sum exp) of z_d and of z_t over its vocabulary tiles and z_d at
// x*; k_loss_lse combines them into lse_d and lse_t; pass 1 leaves per CTA
// sum |p_d - p_t|; k_loss_pos forms ce, l1, bce and the weighted term of each
// position; k_loss_sum adds the terms in a fixed order (fp64).
#include <stdio.h>

#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace dspark {

namespace {

constexpr int kLossWarps = 8;  // positions per CTA of the per-position kernels

// One warp per position: lse of z_d and of z_t from the G per-CTA pairs.
__global__ void __launch_bounds__(32 * kLossWarps)
    k_loss_lse(const float4* __restrict__ lpart, int n, int G, float* __restrict__ lse_d,
               float* __restrict__ lse_t) {
  const int i = blockIdx.x * kLossWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (i >= n) return;
  MS md{-INFINITY, 0.f}, mt{-INFINITY, 0.f};
  for (int c = lane; c < G; c += 32) {
    const float4 q = lpart[(size_t)i * G + c];
    md = ms_combine(md, MS{q.x, q.y});
    mt = ms_combine(mt, MS{q.z, q.w});
  }
  md = warp_ms(md);
  mt = warp_ms(mt);
  if (lane == 0) {
    lse_d[i] = ms_log(md);
    lse_t[i] = ms_log(mt);
  }
}

// One warp per position: l1 from the G per-CTA sums, then ce, c*, bce and the
// position's weighted term. A confidence outside (0, 1) makes bce infinite or
// NaN, as the formula does, and raises DSPARK_ENUMERIC.
__global__ void __launch_bounds__(32 * kLossWarps)
    k_loss_pos(const float* __restrict__ l1part, const float* __restrict__ zx, const float* __restrict__ lse_d,
               const float* __restrict__ conf, int n, int g, int G, double tau, float* __restrict__ ce,
               float* __restrict__ l1, float* __restrict__ bce, double* __restrict__ term, int* status) {
  const int i = blockIdx.x * kLossWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (i >= n) return;
  float s = 0.f;
  for (int c = lane; c < G; c += 32) s += l1part[(size_t)i * G + c];
  s = warp_sum(s);
  if (lane == 0) {
    const double cd = (double)lse_d[i] - (double)zx[i];
    const double cs = 1.0 - 0.5 * (double)s;
    const double c = (double)conf[i];
    if (!(c > 0.0 && c < 1.0)) raise_status(status, DSPARK_ENUMERIC);
    const double b = -(cs * log(c) + (1.0 - cs) * log(1.0 - c));
    const int k = i % g;
    ce[i] = (float)cd;
    l1[i] = s;
    bce[i] = (float)b;
    term[i] = exp(-(double)k / tau) * (0.1 * cd + 0.9 * (double)s + 1.0 * b);
  }
}

// loss = (1/B) sum of the terms: each thread a strided partial, then a tree
// over the threads; the order depends only on n.
__global__ void __launch_bounds__(1024) k_loss_sum(const double* __restrict__ term, int n, int B, double* loss) {
  __shared__ double red[1024];
  double s = 0.0;
  for (int i = threadIdx.x; i < n; i += 1024) s += term[i];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int o = 512; o > 0; o >>= 1) {
    if ((int)threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) *loss = red[0] / (double)B;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Scratch layout: lpart [n][G] float4, l1part [n][G], zx, lse_d, lse_t [n]
// fp32, term [n] fp64, each section 256-byte aligned.
struct LossScratch {
  size_t lpart, l1part, zx, lse_d, lse_t, term, total;
  static LossScratch make(size_t n, size_t G) {
    LossScratch s;
    size_t off = 0;
    auto carve = [&](size_t bytes) {
      const size_t o = off;
      off += round_up(bytes > 0 ? bytes : 1, 256);
      return o;
    };
    s.lpart = carve(16 * n * G);
    s.l1part = carve(4 * n * G);
    s.zx = carve(4 * n);
    s.lse_d = carve(4 * n);
    s.lse_t = carve(4 * n);
    s.term = carve(8 * n);
    s.total = off;
    return s;
  }
};

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_train_loss_scratch_bytes(const dspark_ws* ws) {
  if (!ws) return 0;
  return LossScratch::make((size_t)ws->d.B * ws->d.gamma, (size_t)ws->geo.num_sms).total;
}

extern "C" dspark_status dspark_train_loss(dspark_ws* ws, const float* U, const void* W1, const void* W2,
                                           const int32_t* anchor, const int32_t* xstar, const float* P,
                                           const float* conf, double tau, float* ce, float* l1, float* bce,
                                           double* loss, void* scratch, dspark_stream_t stream) {
  if (!ws) return DSPARK_EINVAL;
  if (!aligned16(U) || !aligned16(W1) || !aligned16(W2) || !aligned16(anchor) || !aligned16(xstar) ||
      !aligned16(P) || !aligned16(conf) || !aligned16(ce) || !aligned16(l1) || !aligned16(bce) || !loss ||
      (reinterpret_cast<uintptr_t>(loss) & 7u) != 0 || !aligned16(scratch) ||
      (reinterpret_cast<uintptr_t>(scratch) & 255u) != 0)
    return DSPARK_EINVAL;
  if (!(tau > 0.0) || !(tau < INFINITY)) return DSPARK_EINVAL;
  const bool rows = rowpass_supported(ws, ws->d.B * ws->d.gamma);
  if (!rows && !ws->geo.resid_tc_ok) return DSPARK_EUNSUPPORTED;
  const dspark_dims& d = ws->d;
  const int n = d.B * d.gamma, G = ws->geo.num_sms;
  const LossScratch L = LossScratch::make((size_t)n, (size_t)G);
  char* base = static_cast<char*>(scratch);
  LossArgs a{U, W1, W2, anchor, xstar, P, conf, tau, ce, l1, bce, loss,
             reinterpret_cast<float4*>(base + L.lpart), reinterpret_cast<float*>(base + L.l1part),
             reinterpret_cast<float*>(base + L.zx), reinterpret_cast<float*>(base + L.lse_d),
             reinterpret_cast<float*>(base + L.lse_t), reinterpret_cast<double*>(base + L.term)};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int blocks = (n + kLossWarps - 1) / kLossWarps;
  auto pass = [&](int ps) { return rows ? launch_loss_rowpass(ws, a, ps, st) : launch_loss_tc(ws, a, ps, st); };
  cudaError_t e = pass(0);
  if (e == cudaSuccess) {
    k_loss_lse<<<blocks, 32 * kLossWarps, 0, st>>>(a.lpart, n, G, a.lse_d, a.lse_t);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = pass(1);
  if (e == cudaSuccess) {
    k_loss_pos<<<blocks, 32 * kLossWarps, 0, st>>>(a.l1part, a.zx, a.lse_d, conf, n, d.gamma, G, tau, ce, l1, bce,
                                                   a.term, ws->s.status);
    k_loss_sum<<<1, 1024, 0, st>>>(a.term, n, d.B, loss);
    e = cudaGetLastError();
  }
  ws->last_launches = 5;
  if (e == cudaSuccess) return DSPARK_OK;
  fprintf(stderr, "dspark: CUDA error %s\n", cudaGetErrorString(e));
  return DSPARK_ECUDA;
}
