// k_rnn.cu -- the RNN head's recurrent cell (eq. (6)).
//
// "DeepSeek-V4.1 模型结构（6）：解码，DSpark", section on the Markov head (the
// paper also tried a small RNN whose bias depends on the longer prefix);
// "DSpark：不让大模型更聪明，而让它「吐字更快」" (RNN head, optional);
// deepseek.csdn.net reading §4.2, eq. (6). A state s_k in R^r summarises the
// block's prefix: with z_k = [s_{k-1}; W1[x_{k-1}]; h_k] (length 2r + H),
//   s_k = sigma(W_g z_k) * s_{k-1} + (1 - sigma(W_g z_k)) * tanh(W_c z_k),
//   B_k = W2^T tanh(W_o z_k),
// s_0 = 0 and x_0 = the anchor. The weights are stacked as Wr [3][r][2r + H]
// (W_g, W_c, W_o) in the dtype of W1 and W2. The draft tail then takes
// o_k = tanh(W_o z_k) in place of W1[x_{k-1}]: the vocabulary pass on tcgen05
// (k_rowpass.cu, o_k as bf16 hi + lo operands that the cell writes in its
// operand layout; k_resid_tc.cu for other shapes) or on CUDA cores, then the
// SIMT pick (k_draft_simt.cu).
//
// Two kernels: k_rnn_hproj, once per round, the h_k part of all three
// projections for every position (a [B*gamma x H] x [H x 3r] product, the
// bulk of the cell's arithmetic, which does not depend on drafted tokens; on
// tcgen05 in k_rnn_tc.cu where the shape allows); k_rnn_cell, before each
// draft step, one CTA per 8 state entries and 16 requests: the [s; W1[x]]
// part, then the gate, the state update and o_k.
#include <stdio.h>

#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace dspark {

namespace {

constexpr int kHpTile = 128;    // output tile of k_rnn_hproj (rows x columns)
constexpr int kHpK = 16;        // K step
constexpr int kHpSplit = kRnnHpSlices;  // K is split over 10 CTAs (two per SM at prod); each writes its own partial product
constexpr int kCellThreads = 256;
constexpr int kCellJ = 8;   // state entries per CTA of k_rnn_cell: one per warp
constexpr int kCellB = 16;  // requests per CTA of k_rnn_cell
static_assert(kCellJ * kCellB <= kCellThreads, "one (entry, request) per thread in the update");
static_assert(kCellJ == kCellThreads / 32, "one warp per state entry");

// Sum over the 32 lanes of 16 per-lane values: afterwards lane L holds the
// sum of every lane's a[L & 15] (each step keeps the half whose index bit
// matches the lane's bit and adds the partner's other half).
__device__ __forceinline__ float transpose_sum16(float (&a)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int q = 0; q < o; ++q) {
      const float send = upper ? a[q] : a[q + o];
      const float keep = upper ? a[q + o] : a[q];
      a[q] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
    }
  }
  return a[0] + __shfl_xor_sync(0xFFFFFFFFu, a[0], 16);
}

// Hp[p][m][n] = sum_{i in slice p of H} h[m][i] Wr[n][2r + i] for m < M =
// B*gamma, n < 3r and the kHpSplit slices p of the H inputs (the cell adds the
// slices in order): 128 x 128 output tiles, 256 threads with 8 x 8 outputs
// each (two 4-wide strips per dimension, read as float4 from shared memory),
// K in steps of 16 staged in shared memory (fp32 accumulation), the next
// step's operands loaded into registers while one step computes.
template <int BF16>
__global__ void __launch_bounds__(256, 2)
    k_rnn_hproj(const float* __restrict__ h, const void* __restrict__ Wr, int M, int H, int r,
                float* __restrict__ Hp) {
  __shared__ __align__(16) float As[kHpK][kHpTile];
  __shared__ __align__(16) float Bs[kHpK][kHpTile];
  const int N = 3 * r, Z = 2 * r + H;
  const int m0 = blockIdx.y * kHpTile, n0 = blockIdx.x * kHpTile;
  const int ksl = (H + kHpSplit - 1) / kHpSplit;
  const int kbeg = blockIdx.z * ksl, kend = min(H, kbeg + ksl);
  Hp += (size_t)blockIdx.z * M * N;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  float acc[8][8] = {};
  constexpr int kPer = (kHpTile * kHpK) / 256;  // 8 elements of each operand per thread
  float ra[kPer], rw[kPer];
  auto gload = [&](int k0) {
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int idx = tid + q * 256, row = idx / kHpK, kg = k0 + idx % kHpK;
      ra[q] = (m0 + row < M && kg < kend) ? h[(size_t)(m0 + row) * H + kg] : 0.f;
      rw[q] = (n0 + row < N && kg < kend) ? ld_w(Wr, BF16, (size_t)(n0 + row) * Z + 2 * r + kg) : 0.f;
    }
  };
  gload(kbeg);
  for (int k0 = kbeg; k0 < kend; k0 += kHpK) {
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int idx = tid + q * 256, row = idx / kHpK, kk = idx % kHpK;
      As[kk][row] = ra[q];
      Bs[kk][row] = rw[q];
    }
    __syncthreads();
    if (k0 + kHpK < kend) gload(k0 + kHpK);
#pragma unroll
    for (int kk = 0; kk < kHpK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[kk][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[kk][64 + tx * 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j2 = 0; j2 < 8; ++j2) acc[i][j2] = fmaf(a[i], b[j2], acc[i][j2]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j2 = 0; j2 < 8; ++j2) {
      const int m = m0 + (i >> 2) * 64 + ty * 4 + (i & 3), n = n0 + (j2 >> 2) * 64 + tx * 4 + (j2 & 3);
      if (m < M && n < N) Hp[(size_t)m * N + n] = acc[i][j2];
    }
}

// Step k for requests b0 .. b0 + 15 and state entries j0 .. j0 + 7 (one CTA):
// pre = W_{g,c,o}[:, :2r] [s_{k-1}; W1[x_{k-1}]] + Hp. Warp w takes entry
// j0 + w: it runs the three rows (g, c, o) over the 2r inputs with the 16
// requests' inputs from shared memory, lane l on inputs 2l + 64 i and the next
// one, then one transpose-reduce per row. The gate, the state update and o_k
// follow per (entry, request). The state is double-buffered by step parity
// (every CTA reads the whole s_{k-1} of its requests).
// Before its wait on the previous kernel (programmatic dependent launch) the
// CTA loads what does not depend on the previous step: the three weight rows
// of each warp (bf16 pairs in registers, for 2r <= 512) and the h
// projection's sums of its (entry, request) pairs. After it, the state rows
// go out while the tokens come back, and all staging loads are 16 bytes wide
// and in flight together.
constexpr int kCellWp = 8;  // bf16 pairs of a weight row per lane (2r <= 64 * kCellWp)

template <int BF16>
__global__ void __launch_bounds__(kCellThreads)
    k_rnn_cell(const void* __restrict__ W1, const void* __restrict__ Wr, const int32_t* __restrict__ anchor,
               const int32_t* __restrict__ tokens, const float* __restrict__ Hp, const float* __restrict__ S_in,
               float* __restrict__ S_out, float* __restrict__ ovec, __nv_bfloat16* __restrict__ oimg, int B, int g,
               int V, int r, int H, int k, int* __restrict__ status) {
  extern __shared__ __align__(16) float zin[];  // [kCellB][2r]: s_{k-1}, W1[x_{k-1}] of each request
  __shared__ float pre[3][kCellJ][kCellB];
  __shared__ int xs[kCellB];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j0 = blockIdx.x * kCellJ, b0 = blockIdx.y * kCellB;
  const int r2 = 2 * r, Z = r2 + H;
  const int jw = j0 + warp;  // this warp's state entry
  // ---- before the wait
  const bool wreg = BF16 && r2 <= 64 * kCellWp && (Z & 1) == 0;  // the same for every thread
  uint32_t wv[3][kCellWp];
  if (wreg) {
    const __nv_bfloat16* wr = reinterpret_cast<const __nv_bfloat16*>(Wr);
#pragma unroll
    for (int q = 0; q < 3; ++q)
#pragma unroll
      for (int t = 0; t < kCellWp; ++t) {
        const int i = 2 * lane + 64 * t;
        wv[q][t] = jw < r && i < r2 ? __ldg(reinterpret_cast<const uint32_t*>(wr + (size_t)(q * r + jw) * Z + i)) : 0u;
      }
  }
  const int ejj = tid % kCellJ, erb = tid / kCellJ, ej = j0 + ejj, eb = b0 + erb;  // the update's (entry, request)
  const bool eact = tid < kCellJ * kCellB && ej < r && eb < B;
  float hq[3] = {0.f, 0.f, 0.f};
  if (eact) {
    const size_t row = (size_t)eb * g + (k - 1);
    const size_t slice = (size_t)B * g * 3 * r;  // the h projection's K slices, added in order
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const float* hp = Hp + row * 3 * r + q * r + ej;
      float t = hp[0];
#pragma unroll
      for (int sl = 1; sl < kHpSplit; ++sl) t += hp[sl * slice];
      hq[q] = t;
    }
  }
  // ---- the previous step's pick (tokens) and cell (state). No early
  // trigger: the row pass launched during the cell slowed the step down
  pdl_wait();
  int x = 0;
  if (tid < kCellB && b0 + tid < B) x = k == 1 ? anchor[b0 + tid] : tokens[(size_t)(b0 + tid) * g + (k - 2)];
  const bool v16 = (r & 7) == 0;  // rows in 16-byte pieces
  if (v16) {  // s_{k-1}: kCellB rows of r/4 float4, four a thread in flight
    const int r4 = r >> 2, n4 = kCellB * r4;
    for (int e0 = tid; e0 < n4; e0 += 4 * kCellThreads) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * kCellThreads, rb = e / r4, b = b0 + rb;
        v[u] = e < n4 && b < B ? __ldg(reinterpret_cast<const float4*>(S_in + (size_t)b * r) + (e - rb * r4))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * kCellThreads, rb = e / r4;
        if (e < n4) *reinterpret_cast<float4*>(zin + rb * r2 + 4 * (e - rb * r4)) = v[u];
      }
    }
  } else {
    for (int e = tid; e < kCellB * r; e += kCellThreads) {
      const int rb = e / r, i = e - rb * r, b = b0 + rb;
      zin[rb * r2 + i] = b < B ? S_in[(size_t)b * r + i] : 0.f;
    }
  }
  if (tid < kCellB) {
    if (x < 0 || x >= V) {
      raise_status(status, DSPARK_ERANGE);
      x = 0;
    }
    xs[tid] = x;
  }
  __syncthreads();
  if (v16) {  // W1[x_{k-1}]: kCellB rows of 16-byte pieces (8 bf16 or 4 fp32), four a thread in flight
    constexpr int per = BF16 ? 8 : 4;
    const int rp = r / per, np = kCellB * rp;
    for (int e0 = tid; e0 < np; e0 += 4 * kCellThreads) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * kCellThreads, rb = e / rp, b = b0 + rb;
        const char* wrow = reinterpret_cast<const char*>(W1) + (size_t)xs[rb < kCellB ? rb : 0] * r * (BF16 ? 2 : 4);
        v[u] = e < np && b < B ? __ldg(reinterpret_cast<const uint4*>(wrow) + (e - rb * rp)) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * kCellThreads, rb = e / rp;
        if (e >= np) continue;
        float* dst = zin + rb * r2 + r + per * (e - rb * rp);
        if (BF16) {
          const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v[u]);
          float2 f[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) f[t] = __bfloat1622float2(h2[t]);
          reinterpret_cast<float4*>(dst)[0] = make_float4(f[0].x, f[0].y, f[1].x, f[1].y);
          reinterpret_cast<float4*>(dst)[1] = make_float4(f[2].x, f[2].y, f[3].x, f[3].y);
        } else {
          *reinterpret_cast<uint4*>(dst) = v[u];
        }
      }
    }
  } else {
    for (int e = tid; e < kCellB * r; e += kCellThreads) {
      const int rb = e / r, i = e - rb * r, b = b0 + rb;
      zin[rb * r2 + r + i] = b < B ? ld_w(W1, BF16, (size_t)xs[rb] * r + i) : 0.f;
    }
  }
  __syncthreads();
  if (jw < r) {  // warp-uniform
    float acc[3][kCellB];
#pragma unroll
    for (int q = 0; q < 3; ++q)
#pragma unroll
      for (int rb = 0; rb < kCellB; ++rb) acc[q][rb] = 0.f;
    if (wreg) {
#pragma unroll
      for (int t = 0; t < kCellWp; ++t) {
        const int i = 2 * lane + 64 * t;
        if (i >= r2) break;
        float2 w2[3];
#pragma unroll
        for (int q = 0; q < 3; ++q) w2[q] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[q][t]));
#pragma unroll
        for (int rb = 0; rb < kCellB; ++rb) {
          const float2 zv = *reinterpret_cast<const float2*>(zin + rb * r2 + i);
#pragma unroll
          for (int q = 0; q < 3; ++q) acc[q][rb] = fmaf(w2[q].y, zv.y, fmaf(w2[q].x, zv.x, acc[q][rb]));
        }
      }
    } else {
#pragma unroll 8
      for (int i = lane; i < r2; i += 32) {
        const float wg = ld_w(Wr, BF16, (size_t)jw * Z + i);
        const float wc = ld_w(Wr, BF16, (size_t)(r + jw) * Z + i);
        const float wo = ld_w(Wr, BF16, (size_t)(2 * r + jw) * Z + i);
#pragma unroll
        for (int rb = 0; rb < kCellB; ++rb) {
          const float zv = zin[rb * r2 + i];
          acc[0][rb] = fmaf(wg, zv, acc[0][rb]);
          acc[1][rb] = fmaf(wc, zv, acc[1][rb]);
          acc[2][rb] = fmaf(wo, zv, acc[2][rb]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const float sum = transpose_sum16(acc[q]);  // lane l: request l & 15
      if (lane < kCellB) pre[q][warp][lane] = sum;
    }
  }
  __syncthreads();
  if (eact) {
    const size_t row = (size_t)eb * g + (k - 1);
    const float gk = 1.f / (1.f + expf(-(pre[0][ejj][erb] + hq[0])));
    S_out[(size_t)eb * r + ej] = gk * zin[erb * r2 + ej] + (1.f - gk) * tanhf(pre[1][ejj][erb] + hq[1]);
    const float o = tanhf(pre[2][ejj][erb] + hq[2]);
    ovec[row * r + ej] = o;
    if (oimg) {  // o_k as bf16 hi and lo, each in the layout of the row pass's A operand (128 rows a group)
      const __nv_bfloat16 hi = __float2bfloat16_rn(o), lo = __float2bfloat16_rn(o - __bfloat162float(hi));
      __nv_bfloat16* im = oimg + (size_t)(eb >> 7) * 2 * 128 * r;
      const size_t off = kmajor_sw128_piece(eb & 127, ej >> 6, (ej >> 3) & 7, 128) + (ej & 7);
      im[off] = hi;
      im[(size_t)128 * r + off] = lo;
    }
  }
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Scratch: Hp [10][B*gamma][3r] fp32 (the h projection's K slices), then the
// state S [2][B][r] fp32 (two buffers alternating by step parity; 256-byte
// aligned).
size_t hp_bytes(const dspark_dims& d) {
  return round_up(sizeof(float) * kHpSplit * (size_t)d.B * d.gamma * 3 * d.r, 256);
}
size_t state_bytes(const dspark_dims& d) { return round_up(2 * sizeof(float) * (size_t)d.B * d.r, 256); }
// o_k's bf16 hi and lo images for the row pass, per group of 128 requests
size_t oimg_bytes(const dspark_dims& d) {
  return round_up(sizeof(__nv_bfloat16) * 2 * 128 * (size_t)((d.B + 127) / 128) * d.r, 256);
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

cudaError_t launch_rnn_hproj(const dspark_ws* ws, const float* h, const void* Wr, float* Hp, cudaStream_t st,
                             int* launches) {
  const dspark_dims& d = ws->d;
  const int M = d.B * d.gamma, N = 3 * d.r;
  if (d.H == 0) return cudaMemsetAsync(Hp, 0, sizeof(float) * kHpSplit * (size_t)M * N, st);
  const dim3 grid((N + kHpTile - 1) / kHpTile, (M + kHpTile - 1) / kHpTile, kHpSplit);
  if (d.wdtype == DSPARK_BF16)
    k_rnn_hproj<1><<<grid, 256, 0, st>>>(h, Wr, M, d.H, d.r, Hp);
  else
    k_rnn_hproj<0><<<grid, 256, 0, st>>>(h, Wr, M, d.H, d.r, Hp);
  ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_rnn_cell(const dspark_ws* ws, const DraftArgs& a, const void* Wr, const float* Hp, float* S,
                            float* ovec, __nv_bfloat16* oimg, int k, cudaStream_t st, int* launches) {
  const dspark_dims& d = ws->d;
  const size_t smem = sizeof(float) * kCellB * 2 * (size_t)d.r;  // 128 KB at r = 1024
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k_rnn_cell<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(sizeof(float) * kCellB * 2 * 1024));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_rnn_cell<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)(sizeof(float) * kCellB * 2 * 1024));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  // step k reads the state of step k - 1 from buffer (k - 1) % 2, writes buffer k % 2
  const size_t BR = (size_t)d.B * d.r;
  const float* S_in = S + ((k - 1) & 1) * BR;
  float* S_out = S + (k & 1) * BR;
  const dim3 grid((d.r + kCellJ - 1) / kCellJ, (d.B + kCellB - 1) / kCellB);
  // programmatic dependent launch: the step's kernels wait in-kernel for the one before
  const cudaError_t e =
      d.wdtype == DSPARK_BF16
          ? launch_ex(k_rnn_cell<1>, grid, dim3(kCellThreads), smem, st, true, a.W1, Wr, a.anchor, a.tokens, Hp,
                      S_in, S_out, ovec, oimg, d.B, d.gamma, d.V, d.r, d.H, k, ws->s.status)
          : launch_ex(k_rnn_cell<0>, grid, dim3(kCellThreads), smem, st, true, a.W1, Wr, a.anchor, a.tokens, Hp,
                      S_in, S_out, ovec, oimg, d.B, d.gamma, d.V, d.r, d.H, k, ws->s.status);
  ++*launches;
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_rnn_draft_scratch_bytes(const dspark_ws* ws) {
  if (!ws) return 0;
  // the hi | lo copy of h for the tcgen05 h projection, wherever the shape allows it
  // (whichever compute path the workspace is set to when the call runs)
  return hp_bytes(ws->d) + state_bytes(ws->d) + oimg_bytes(ws->d) +
         (rnn_hproj_tc_shape(ws->d) ? rnn_hsplit_bytes(ws->d) : 0);
}

extern "C" dspark_status dspark_rnn_draft(dspark_ws* ws, const float* U, const void* W1, const void* W2,
                                          const void* Wr, const int32_t* anchor, const float* h, const float* w,
                                          const float* T, uint64_t seed, uint64_t round, int32_t* tokens,
                                          float* pd_tok, float* lse, float* conf, float* ovec, void* scratch,
                                          dspark_stream_t stream) {
  if (!ws) return DSPARK_EINVAL;
  const dspark_dims& d = ws->d;
  if (!aligned16(U) || !aligned16(W1) || !aligned16(W2) || !aligned16(Wr) || !aligned16(anchor) || !aligned16(w) ||
      !aligned16(T) || !aligned16(tokens) || !aligned16(pd_tok) || !aligned16(lse) || !aligned16(conf) ||
      !aligned16(ovec) || !scratch || (reinterpret_cast<uintptr_t>(scratch) & 255u) != 0)
    return DSPARK_EINVAL;
  if (d.H > 0 && !aligned16(h)) return DSPARK_EINVAL;
  char* base = static_cast<char*>(scratch);
  float* Hp = reinterpret_cast<float*>(base);
  float* S = reinterpret_cast<float*>(base + hp_bytes(d));
  __nv_bfloat16* oimg = reinterpret_cast<__nv_bfloat16*>(base + hp_bytes(d) + state_bytes(d));
  void* hl = rnn_hproj_tc_shape(d) ? static_cast<void*>(base + hp_bytes(d) + state_bytes(d) + oimg_bytes(d)) : nullptr;
  DraftArgs a{U, W1, W2, anchor, h, w, T, seed, round, tokens, pd_tok, lse, conf};
  int launches = 0;
  const cudaError_t e =
      launch_rnn_draft(ws, a, Wr, Hp, S, ovec, hl, oimg, oimg_bytes(d), reinterpret_cast<cudaStream_t>(stream),
                       &launches);
  ws->last_launches = launches;
  if (e == cudaSuccess) return DSPARK_OK;
  fprintf(stderr, "dspark: CUDA error %s\n", cudaGetErrorString(e));
  return DSPARK_ECUDA;
}
