// k_sts.cu -- sequential temperature scaling (STS) of the confidence head.
//
// "DeepSeek-V4.1 模型结构（6）：解码，DSpark", section "confidence head": a
// temperature per position, fitted on held-out data so that the survival
// products a_j match measured acceptance; zdszero.github.io "spec_dspark"
// ("STS 校准"), "DSpark：不让大模型更聪明，而让它「吐字更快」" §05 and the
// deepseek.csdn.net reading §5.2: left to right, a one-dimensional grid search
// per position that minimises the expected calibration error (ECE) of the
// cumulative product, the positions already calibrated kept fixed.
//
// For held-out blocks n < N and positions k: c_k(n) = sigma(raw[n][k] / T_k),
// a_k(n) = prod_{i<=k} c_i(n), the label y_k(n) = prod_{i<=k} cstar[n][i] (the
// prefix's joint acceptance factorises into its positions' acceptance
// probabilities), and with M equal-width bins of [0, 1]
//   ECE_k(T) = (1/N) sum_m | sum_{n: a_k(n) in bin m} (a_k(n) - y_k(n)) |.
// T_k = the first grid value with the smallest ECE_k.
//
// Per position two launches: k_sts_ece, one CTA per (grid temperature, slice
// of the samples), each thread keeping its own bin sums in shared memory as
// 64-bit fixed point (2^-40 units: exact and independent of the summation
// order) and the CTA writing its bins' sums, then k_sts_pick, one CTA: the
// ECE of every temperature from the slices' sums and the argmin. The running
// products of the positions already calibrated advance inside k_sts_ece: each
// CTA forms a_{k-1} from the stored a_{k-2} and the chosen T_{k-1}, and the
// CTAs of grid value 0 store it for the next position (two buffers).
#include <stdio.h>

#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace dspark {

constexpr int kStsThreads = 256;
constexpr int kStsMaxBins = 32;
constexpr int kStsSlices = 8;  // sample slices per temperature (CTAs per grid value)
constexpr float kStsFix = 1099511627776.0f;  // 2^40

__device__ __forceinline__ float sts_sigmoid(float raw, float T) { return 1.f / (1.f + expf(-raw / T)); }

__device__ __forceinline__ int sts_bin(float a, int M) {
  int m = (int)floorf(a * (float)M);
  return m < 0 ? 0 : (m > M - 1 ? M - 1 : m);
}

// bsum[(gi * kStsSlices + slice) * M + m]: the fixed-point sum of a - y over
// the slice's samples in bin m, for grid temperature gi at position k.
// a_in / y_in hold the products of positions 1..k-2 (k >= 2); with T_out[k-1]
// they give the products up to k-1, which grid value 0 stores in a_out / y_out.
__global__ void __launch_bounds__(kStsThreads)
    k_sts_ece(const float* __restrict__ raw, const float* __restrict__ cstar, int N, int g, int k,
              const float* __restrict__ a_in, const float* __restrict__ y_in, float* __restrict__ a_out,
              float* __restrict__ y_out, const float* __restrict__ T_out, const float* __restrict__ Tgrid, int M,
              long long* __restrict__ bsum, int* __restrict__ status) {
  extern __shared__ long long bins[];  // [M][kStsThreads], one column per thread
  const int tid = threadIdx.x;
  const int gi = blockIdx.x, sl = blockIdx.y;
  long long* out = bsum + ((size_t)gi * kStsSlices + sl) * M;
  const float T = Tgrid[gi];
  if (!(T > 0.f) || !isfinite(T)) {
    if (tid == 0) raise_status(status, DSPARK_ERANGE);
    if (tid < M) out[tid] = 0;
    return;
  }
  const int n0 = (int)((long long)N * sl / kStsSlices), n1 = (int)((long long)N * (sl + 1) / kStsSlices);
  for (int m = 0; m < M; ++m) bins[m * kStsThreads + tid] = 0;
  const float Tp = k > 0 ? T_out[k - 1] : 1.f;  // the previous position's chosen temperature
  for (int n = n0 + tid; n < n1; n += kStsThreads) {
    const float r = raw[(size_t)n * g + k], cs = cstar[(size_t)n * g + k];
    float ap = 1.f, yp = 1.f;  // products up to position k-1
    if (k > 0) {
      ap = (k > 1 ? a_in[n] : 1.f) * sts_sigmoid(raw[(size_t)n * g + k - 1], Tp);
      yp = (k > 1 ? y_in[n] : 1.f) * cstar[(size_t)n * g + k - 1];
      if (gi == 0) {
        a_out[n] = ap;
        y_out[n] = yp;
      }
    }
    const float a = ap * sts_sigmoid(r, T);
    const float y = yp * cs;
    bins[sts_bin(a, M) * kStsThreads + tid] += __float2ll_rn((a - y) * kStsFix);
  }
  __syncthreads();
  // the slice's sum of each bin: warp w reduces bins w, w + 8, ...
  const int warp = tid >> 5, lane = tid & 31;
  for (int m = warp; m < M; m += kStsThreads / 32) {
    long long s = 0;
    for (int i = lane; i < kStsThreads; i += 32) s += bins[m * kStsThreads + i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    if (lane == 0) out[m] = s;
  }
}

// ECE_k(T) for every grid value from the slices' bin sums; the first grid
// temperature with the smallest ECE: T_out[k], ece_out[k].
__global__ void __launch_bounds__(1024)
    k_sts_pick(int N, int k, const float* __restrict__ Tgrid, int G, int M, const long long* __restrict__ bsum,
               double* __restrict__ ece, float* __restrict__ T_out, double* __restrict__ ece_out) {
  __shared__ double bv[32];
  __shared__ int bi[32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < G; i += blockDim.x) {
    const float T = Tgrid[i];
    double e = 0.0;
    for (int m = 0; m < M; ++m) {
      long long s = 0;
      for (int sl = 0; sl < kStsSlices; ++sl) s += bsum[((size_t)i * kStsSlices + sl) * M + m];
      e += (double)(s < 0 ? -s : s);
    }
    ece[i] = (T > 0.f && isfinite(T)) ? e / (double)kStsFix / (double)N : INFINITY;
  }
  __syncthreads();
  double v = INFINITY;
  int idx = 0x7FFFFFFF;
  for (int i = tid; i < G; i += blockDim.x) {
    const double x = ece[i];
    if (x < v || (x == v && i < idx)) {
      v = x;
      idx = i;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double ov = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int oi = __shfl_xor_sync(0xFFFFFFFFu, idx, o);
    if (ov < v || (ov == v && oi < idx)) {
      v = ov;
      idx = oi;
    }
  }
  if (lane == 0) {
    bv[warp] = v;
    bi[warp] = idx;
  }
  __syncthreads();
  if (tid == 0) {
    double b = INFINITY;
    int ib = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w)
      if (bv[w] < b || (bv[w] == b && bi[w] < ib)) {
        b = bv[w];
        ib = bi[w];
      }
    if (ib < 0 || ib >= G) ib = 0;  // every ECE infinite: an invalid grid, already reported
    T_out[k] = Tgrid[ib];
    ece_out[k] = b;
  }
}

}  // namespace dspark

using namespace dspark;

namespace {
dspark_status sts_fail(cudaError_t e) {
  if (e == cudaSuccess) return DSPARK_OK;
  fprintf(stderr, "dspark: CUDA error %s\n", cudaGetErrorString(e));
  return DSPARK_ECUDA;
}
}  // namespace

extern "C" dspark_status dspark_sts_fit(const float* raw, const float* cstar, int N, int gamma,
                                        const float* Tgrid, int G, int M, float* T_out, double* ece_out,
                                        void* scratch, int32_t* device_status, dspark_stream_t stream) {
  if (!raw || !cstar || !Tgrid || !T_out || !ece_out || !scratch || !device_status) return DSPARK_EINVAL;
  if (N < 1 || gamma < 1 || gamma > 1024 || G < 1 || G > 65535 || M < 1 || M > kStsMaxBins) return DSPARK_EINVAL;
  if ((size_t)N * (size_t)gamma >= ((size_t)1 << 34)) return DSPARK_EUNSUPPORTED;
  if (N >= (1 << 23)) return DSPARK_EUNSUPPORTED;  // the 2^-40 fixed-point bin sums stay below 2^63
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // scratch: the slices' bin sums [G][slices][M] int64, ece [G] fp64, then
  // two buffers of the running products a and y, [N] fp32 each
  long long* bsum = static_cast<long long*>(scratch);
  double* ece = reinterpret_cast<double*>(bsum + (size_t)G * kStsSlices * kStsMaxBins);
  float* abuf[2] = {reinterpret_cast<float*>(ece + G), reinterpret_cast<float*>(ece + G) + N};
  float* ybuf[2] = {abuf[1] + N, abuf[1] + 2 * (size_t)N};
  const size_t smem = sizeof(long long) * (size_t)M * kStsThreads;
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(k_sts_ece, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(sizeof(long long) * kStsMaxBins * kStsThreads)) != cudaSuccess)
      return sts_fail(cudaGetLastError());
    configured = true;
  }
  cudaError_t e = cudaMemsetAsync(device_status, 0, sizeof(int32_t), st);
  for (int k = 0; k < gamma && e == cudaSuccess; ++k) {
    // position k reads the products up to k-2 from buffer k % 2 and stores
    // those up to k-1 in the other one
    k_sts_ece<<<dim3(G, kStsSlices), kStsThreads, smem, st>>>(raw, cstar, N, gamma, k, abuf[k & 1], ybuf[k & 1],
                                                              abuf[(k + 1) & 1], ybuf[(k + 1) & 1], T_out, Tgrid,
                                                              M, bsum, device_status);
    k_sts_pick<<<1, 1024, 0, st>>>(N, k, Tgrid, G, M, bsum, ece, T_out, ece_out);
    e = cudaGetLastError();
  }
  return sts_fail(e);
}

extern "C" size_t dspark_sts_scratch_bytes(int N, int G) {
  const size_t g = (size_t)(G > 0 ? G : 0);
  return sizeof(long long) * g * kStsSlices * kStsMaxBins + sizeof(double) * g +
         4 * sizeof(float) * (size_t)(N > 0 ? N : 0);
}
