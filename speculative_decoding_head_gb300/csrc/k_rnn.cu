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
// (W_g, W_c, W_o) in the dtype of W1 and W2. The draft tail then runs the
// Markov draft's SIMT kernels with o_k = tanh(W_o z_k) in place of W1[x_{k-1}]
// (k_draft_simt.cu).
//
// Two kernels: k_rnn_hproj, once per round, the h_k part of all three
// projections for every position (a [B*gamma x H] x [H x 3r] product, the
// bulk of the cell's arithmetic, which does not depend on drafted tokens);
// k_rnn_cell, before each draft step, one CTA per request: the [s; W1[x]]
// part (a warp per output row), then the gate, the state update and o_k.
#include <stdio.h>

#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace dspark {

namespace {

constexpr int kHpTile = 64;     // output tile of k_rnn_hproj (rows x columns)
constexpr int kHpK = 32;        // K step
constexpr int kCellThreads = 256;

// Hp[m][n] = sum_{i<H} h[m][i] Wr[n][2r + i] for m < M = B*gamma, n < 3r:
// 64 x 64 output tiles, 256 threads with 4 x 4 outputs each, K in steps of 32
// staged in shared memory (fp32 accumulation).
template <int BF16>
__global__ void __launch_bounds__(256)
    k_rnn_hproj(const float* __restrict__ h, const void* __restrict__ Wr, int M, int H, int r,
                float* __restrict__ Hp) {
  __shared__ float As[kHpK][kHpTile + 4];
  __shared__ float Bs[kHpK][kHpTile + 4];
  const int N = 3 * r, Z = 2 * r + H;
  const int m0 = blockIdx.y * kHpTile, n0 = blockIdx.x * kHpTile;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < H; k0 += kHpK) {
#pragma unroll
    for (int q = 0; q < (kHpTile * kHpK) / 256; ++q) {
      const int idx = tid + q * 256, row = idx / kHpK, kk = idx % kHpK;
      const int kg = k0 + kk;
      As[kk][row] = (m0 + row < M && kg < H) ? h[(size_t)(m0 + row) * H + kg] : 0.f;
      Bs[kk][row] = (n0 + row < N && kg < H) ? ld_w(Wr, BF16, (size_t)(n0 + row) * Z + 2 * r + kg) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kHpK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
      if (m < M && n < N) Hp[(size_t)m * N + n] = acc[i][j];
    }
}

// Step k of request b = blockIdx.x: pre = W_{g,c,o}[:, :2r] [s_{k-1}; W1[x_{k-1}]]
// + Hp (a warp per output row, lanes across the 2r inputs), then the gate, the
// state update (S in place: this CTA alone owns row b) and o_k.
template <int BF16>
__global__ void __launch_bounds__(kCellThreads)
    k_rnn_cell(const void* __restrict__ W1, const void* __restrict__ Wr, const int32_t* __restrict__ anchor,
               const int32_t* __restrict__ tokens, const float* __restrict__ Hp, float* __restrict__ S,
               float* __restrict__ ovec, int g, int V, int r, int H, int k, int* __restrict__ status) {
  extern __shared__ float sm[];
  float* zin = sm;          // [2r]: s_{k-1}, W1[x_{k-1}]
  float* pre = sm + 2 * r;  // [3r]: the three pre-activations
  const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int x = k == 1 ? anchor[b] : tokens[(size_t)b * g + (k - 2)];
  if (x < 0 || x >= V) {
    if (tid == 0) raise_status(status, DSPARK_ERANGE);
    return;
  }
  for (int i = tid; i < r; i += kCellThreads) {
    zin[i] = S[(size_t)b * r + i];
    zin[r + i] = ld_w(W1, BF16, (size_t)x * r + i);
  }
  __syncthreads();
  const int Z = 2 * r + H;
  const size_t row = (size_t)b * g + (k - 1);
  for (int n = warp; n < 3 * r; n += kCellThreads / 32) {
    float acc = 0.f;
    for (int i = lane; i < 2 * r; i += 32) acc = fmaf(ld_w(Wr, BF16, (size_t)n * Z + i), zin[i], acc);
    acc = warp_sum(acc);
    if (lane == 0) pre[n] = acc + Hp[row * 3 * r + n];
  }
  __syncthreads();
  for (int j = tid; j < r; j += kCellThreads) {
    const float gk = 1.f / (1.f + expf(-pre[j]));
    S[(size_t)b * r + j] = gk * zin[j] + (1.f - gk) * tanhf(pre[r + j]);
    ovec[row * r + j] = tanhf(pre[2 * r + j]);
  }
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Scratch: Hp [B*gamma][3r] fp32, then S [B][r] fp32 (256-byte aligned).
size_t hp_bytes(const dspark_dims& d) { return round_up(sizeof(float) * (size_t)d.B * d.gamma * 3 * d.r, 256); }
size_t state_bytes(const dspark_dims& d) { return round_up(sizeof(float) * (size_t)d.B * d.r, 256); }

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

cudaError_t launch_rnn_hproj(const dspark_ws* ws, const float* h, const void* Wr, float* Hp, cudaStream_t st,
                             int* launches) {
  const dspark_dims& d = ws->d;
  const int M = d.B * d.gamma, N = 3 * d.r;
  if (d.H == 0) return cudaMemsetAsync(Hp, 0, sizeof(float) * (size_t)M * N, st);
  const dim3 grid((N + kHpTile - 1) / kHpTile, (M + kHpTile - 1) / kHpTile);
  if (d.wdtype == DSPARK_BF16)
    k_rnn_hproj<1><<<grid, 256, 0, st>>>(h, Wr, M, d.H, d.r, Hp);
  else
    k_rnn_hproj<0><<<grid, 256, 0, st>>>(h, Wr, M, d.H, d.r, Hp);
  ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_rnn_cell(const dspark_ws* ws, const DraftArgs& a, const void* Wr, const float* Hp, float* S,
                            float* ovec, int k, cudaStream_t st, int* launches) {
  const dspark_dims& d = ws->d;
  const size_t smem = sizeof(float) * 5 * (size_t)d.r;
  if (d.wdtype == DSPARK_BF16)
    k_rnn_cell<1><<<d.B, kCellThreads, smem, st>>>(a.W1, Wr, a.anchor, a.tokens, Hp, S, ovec, d.gamma, d.V, d.r,
                                                   d.H, k, ws->s.status);
  else
    k_rnn_cell<0><<<d.B, kCellThreads, smem, st>>>(a.W1, Wr, a.anchor, a.tokens, Hp, S, ovec, d.gamma, d.V, d.r,
                                                   d.H, k, ws->s.status);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_rnn_draft_scratch_bytes(const dspark_ws* ws) {
  if (!ws) return 0;
  return hp_bytes(ws->d) + state_bytes(ws->d);
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
  if (5 * (size_t)d.r * sizeof(float) > 48 * 1024) return DSPARK_EUNSUPPORTED;  // the cell's shared memory
  char* base = static_cast<char*>(scratch);
  float* Hp = reinterpret_cast<float*>(base);
  float* S = reinterpret_cast<float*>(base + hp_bytes(d));
  DraftArgs a{U, W1, W2, anchor, h, w, T, seed, round, tokens, pd_tok, lse, conf};
  int launches = 0;
  const cudaError_t e = launch_rnn_draft(ws, a, Wr, Hp, S, ovec, reinterpret_cast<cudaStream_t>(stream), &launches);
  ws->last_launches = launches;
  if (e == cudaSuccess) return DSPARK_OK;
  fprintf(stderr, "dspark: CUDA error %s\n", cudaGetErrorString(e));
  return DSPARK_ECUDA;
}
