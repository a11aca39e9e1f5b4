// k_draft_simt.cu -- Markov-head draft tail on CUDA cores (fp32 FMA).
//
// "DeepSeek-V4.1 模型结构（6）：解码，DSpark", eq. (4)/(5) and the sequential
// loop of section "Markov head": for k = 1..gamma the logits of position k
// are z = U_k + W1[x_{k-1}] W2 (x_0 = anchor) and x_k ~ softmax(z); eq. (7)
// gives c_k = sigma((w^T [h_k; W1[x_{k-1}]]) / T_k).
//
// This path serves every weight dtype and rank (the tiny fp32 workload, and
// as a plain baseline of the tensor-core path). Per step two kernels run:
//   k_draft_blocks  grid (chunks, B): z for every token, folded into the
//                   log-mass of each 64-token vocabulary block;
//   k_draft_pick    grid (B): log-sum-exp over blocks, the block draw
//                   argmax_s(log mass_s + G_s), then z of the 64 tokens of the
//                   drawn block recomputed and the token inside it drawn by
//                   argmax_v (z_v + G_v); also c_k.
// With the RNN head (eq. (6)) the r-vector that multiplies W2 is the head's
// o_k, which k_rnn_cell writes before each step (ovec); the confidence still
// takes W1[x_{k-1}].
#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace dspark {

constexpr int kSimtThreads = 256;
constexpr int kPickThreadsS = 1024;             // k_draft_pick: 16 K slices of the 64-token recompute
constexpr int kPickKs = kPickThreadsS / kBlockW;

// s_h[row] = sum_{i<H} w[i] h[row, i]: the part of the confidence logit that
// does not depend on drafted tokens (one CTA of 128 threads per row of h, all
// of a thread's float4 loads in flight together).
__global__ void __launch_bounds__(128) k_conf_hidden(const float* __restrict__ h,
                                                     const float* __restrict__ w, int H,
                                                     float* __restrict__ s_h) {
  __shared__ float red[4];
  const int row = blockIdx.x;
  const float d = hidden_dot128(h + (size_t)row * H, w, H, red);
  if (threadIdx.x == 0) s_h[row] = d;
}

__device__ __forceinline__ int prev_token(const int32_t* anchor, const int32_t* tokens, int b, int g,
                                          int k) {
  return k == 1 ? anchor[b] : tokens[(size_t)b * g + (k - 2)];
}

// z_v - U_k(v) = sum_i e_i W2[i, v] for one token (fp32 FMA in i order)
template <int BF16>
__device__ __forceinline__ float markov_dot(const float* __restrict__ e, const void* __restrict__ W2,
                                            int r, int V, int v) {
  float acc = 0.f;
  for (int i = 0; i < r; ++i) acc = fmaf(e[i], ld_w(W2, BF16, (size_t)i * V + v), acc);
  return acc;
}

template <int BF16>
__global__ void __launch_bounds__(kSimtThreads)
    k_draft_blocks(const float* __restrict__ U, const void* __restrict__ W1, const void* __restrict__ W2,
                   const int32_t* __restrict__ anchor, const int32_t* __restrict__ tokens,
                   const float* __restrict__ ovec, int g, int V, int r, int k, int nblk, float* __restrict__ blk,
                   int* __restrict__ status) {
  extern __shared__ float e[];  // W1[x_{k-1}] (Markov head) or o_k (RNN head) as fp32, [r]
  pdl_wait();  // the previous step's pick (launched as a dependent kernel)
  const int b = blockIdx.y;
  const int x = prev_token(anchor, tokens, b, g, k);
  if (x < 0 || x >= V) {
    if (threadIdx.x == 0) raise_status(status, DSPARK_ERANGE);
    return;
  }
  for (int i = threadIdx.x; i < r; i += blockDim.x)
    e[i] = ovec ? ovec[((size_t)b * g + (k - 1)) * r + i] : ld_w(W1, BF16, (size_t)x * r + i);
  __syncthreads();
  const float* Urow = U + ((size_t)b * g + (k - 1)) * V;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wpc = blockDim.x >> 5;
  for (int s = blockIdx.x * wpc + warp; s < nblk; s += gridDim.x * wpc) {
    const int v0 = s * kBlockW + lane, v1 = v0 + 32;
    float z0 = -INFINITY, z1 = -INFINITY;
    if (v0 < V) z0 = Urow[v0] + markov_dot<BF16>(e, W2, r, V, v0);
    if (v1 < V) z1 = Urow[v1] + markov_dot<BF16>(e, W2, r, V, v1);
    const float m = warp_max(fmaxf(z0, z1));
    float t = (v0 < V ? expf(z0 - m) : 0.f) + (v1 < V ? expf(z1 - m) : 0.f);
    t = warp_sum(t);
    if (lane == 0) blk[(size_t)b * nblk + s] = m + logf(t);
  }
}

template <int BF16>
__global__ void __launch_bounds__(kPickThreadsS)
    k_draft_pick(const float* __restrict__ U, const void* __restrict__ W1, const void* __restrict__ W2,
                 const int32_t* __restrict__ anchor, const float* __restrict__ w,
                 const float* __restrict__ T, const float* __restrict__ s_h, const float* __restrict__ ovec, int g,
                 int V, int r, int H, int k, int nblk, const float* __restrict__ blk, Rng rng,
                 int32_t* __restrict__ tokens,
                 float* __restrict__ pd_tok, float* __restrict__ lse_out, float* __restrict__ conf,
                 int* __restrict__ status) {
  extern __shared__ float e[];  // [r]
  __shared__ float red_f[32];
  __shared__ MS red_ms[32];
  __shared__ KeyIdx red_k[32];
  __shared__ float zpart[kPickKs][kBlockW];
  __shared__ float zblk[kBlockW];
  pdl_wait();  // the block pass (and the previous step's pick) of this step
  pdl_trigger();
  const int b = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
  const size_t o = (size_t)b * g + (k - 1);
  // the loads that do not depend on the previous token go out with it
  const int x = prev_token(anchor, tokens, b, g, k);
  if (ovec)
    for (int i = tid; i < r; i += blockDim.x) e[i] = ovec[o * r + i];
  // the block log-masses, four consecutive blocks a thread (one counter draw
  // serves four blocks): the thread's (max, sum) and its best block key
  MS ms{-INFINITY, 0.f};
  KeyIdx kb = key_none();
  for (int s4 = 4 * tid; s4 < nblk; s4 += 4 * blockDim.x) {
    float lm[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) lm[u] = s4 + u < nblk ? blk[(size_t)b * nblk + s4 + u] : -INFINITY;
    const uint4 wq = rng.block4(kDraftBlock, b, k, s4);
    const uint32_t wv[4] = {wq.x, wq.y, wq.z, wq.w};
    const float m4 = fmaxf(fmaxf(lm[0], lm[1]), fmaxf(lm[2], lm[3]));
    if (m4 > -INFINITY) {
      float t4 = 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) t4 += __expf(lm[u] - m4);
      ms = ms_combine(ms, MS{m4, t4});
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (lm[u] > -INFINITY) kb = better(kb, KeyIdx{lm[u] + gumbel(wv[u]), s4 + u});
  }
  if (x < 0 || x >= V) {
    if (tid == 0) raise_status(status, DSPARK_ERANGE);
    return;
  }
  if (!ovec)
    for (int i = tid; i < r; i += blockDim.x) e[i] = ld_w(W1, BF16, (size_t)x * r + i);
  __syncthreads();

  // eq. (7): c_k = sigma((s_h + w_r . W1[x_{k-1}]) / T_k)
  float cr = 0.f;
  for (int i = tid; i < r; i += blockDim.x)
    cr = fmaf(w[H + i], ovec ? ld_w(W1, BF16, (size_t)x * r + i) : e[i], cr);
  cr = warp_sum(cr);
  if (lane == 0) red_f[warp] = cr;
  // log-sum-exp over the block log-masses: the warp's maximum first, then the
  // rescaled sums (one exponential a lane)
  {
    float M = ms.m;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
    float t = ms.m == -INFINITY ? 0.f : ms.s * __expf(ms.m - M);
    t = warp_sum(t);
    if (lane == 0) red_ms[warp] = MS{M, M == -INFINITY ? 0.f : t};
  }
  // block draw: argmax_s (log mass_s + G_s)
  kb = warp_best(kb);
  if (lane == 0) red_k[warp] = kb;
  __syncthreads();
  if (warp == 0) {
    float c = lane < nw ? red_f[lane] : 0.f;
    c = warp_sum(c);
    MS m2 = lane < nw ? red_ms[lane] : MS{-INFINITY, 0.f};
    m2 = warp_ms(m2);
    KeyIdx k2 = lane < nw ? red_k[lane] : key_none();
    k2 = warp_best(k2);
    if (lane == 0) {
      const float raw = s_h[o] + c;
      const float cf = 1.f / (1.f + expf(-raw / T[k - 1]));
      if (!isfinite(cf)) raise_status(status, DSPARK_ENUMERIC);
      conf[o] = cf;
      red_f[0] = ms_log(m2);
      red_k[0] = k2;
    }
  }
  __syncthreads();
  const float L = red_f[0];
  const int sb = red_k[0].idx;
  if (sb == kNoIdx) {
    if (tid == 0) raise_status(status, DSPARK_ENUMERIC);
    return;
  }
  // U of the block's tokens, loaded beside the W2 columns below
  float ublk = 0.f;
  if (tid < kBlockW && sb * kBlockW + tid < V) ublk = U[o * V + sb * kBlockW + tid];
  // token draw inside block sb: recompute z for its 64 tokens, each over
  // 16 K slices (a thread's slice of rows i = q, q + 16, ... with all of its
  // W2 loads in flight), the slices added in a fixed order
  {
    const int vl = tid & (kBlockW - 1), q = tid / kBlockW;
    const int v = sb * kBlockW + vl;
    float acc = 0.f;
    if (v < V)
#pragma unroll 16
      for (int i = q; i < r; i += kPickKs) acc = fmaf(e[i], ld_w(W2, BF16, (size_t)i * V + v), acc);
    zpart[q][vl] = acc;
  }
  __syncthreads();
  // token draw inside block sb: argmax_v (z_v + G_v) over its 64 tokens, one
  // thread per token, then across the two warps
  if (tid < kBlockW) {
    const int v = sb * kBlockW + tid;
    float z = -INFINITY;
    if (v < V) {
      float zs = 0.f;
#pragma unroll
      for (int q = 0; q < kPickKs; ++q) zs += zpart[q][tid];
      z = ublk + zs;
    }
    zblk[tid] = z;
    KeyIdx kt = key_none();
    if (z > -INFINITY) kt = KeyIdx{z + gumbel(rng.word(kDraftToken, b, k, v)), tid};
    kt = warp_best(kt);
    if (lane == 0) red_k[warp] = kt;
  }
  __syncthreads();
  if (tid == 0) {
    const KeyIdx kt = better(red_k[0], red_k[1]);
    int xl = kt.idx;
    if (xl == kNoIdx) {  // only non-finite logits get here
      raise_status(status, DSPARK_ENUMERIC);
      xl = 0;
    }
    tokens[o] = sb * kBlockW + xl;
    pd_tok[o] = expf(zblk[xl] - L);
    lse_out[o] = L;
  }
}

cudaError_t launch_conf_hidden(const dspark_ws* ws, const float* h, const float* w, cudaStream_t st,
                               int* launches) {
  const int rows = ws->d.B * ws->d.gamma;
  if (ws->d.H == 0) return cudaMemsetAsync(ws->s.s_h, 0, sizeof(float) * rows, st);
  k_conf_hidden<<<rows, 128, 0, st>>>(h, w, ws->d.H, ws->s.s_h);
  ++*launches;
  return cudaGetLastError();
}

// rnn: the RNN head's cell runs before each step (Hp, S, ovec: its scratch
// and output); null for the Markov head.
struct RnnStep {
  const void* Wr;
  float* Hp;
  float* S;
  float* ovec;
  bool tc;              // block pass on tcgen05
  __nv_bfloat16* oimg;  // o_k's images for the row pass (when it runs the block pass)
};

template <int BF16>
static cudaError_t draft_simt_impl(const dspark_ws* ws, const DraftArgs& a, cudaStream_t st,
                                   int* launches, const RnnStep* rnn = nullptr) {
  const dspark_dims& d = ws->d;
  const int nblk = ws->geo.nblk;
  const size_t smem = sizeof(float) * d.r;
  const int wpc = kSimtThreads / 32;
  int chunks = (nblk + 4 * wpc - 1) / (4 * wpc);  // about 4 blocks per warp
  if (chunks < 1) chunks = 1;
  const Rng rng = Rng::make(a.seed, a.round, (uint32_t)ws->b0);
  const float* ovec = rnn ? rnn->ovec : nullptr;
  for (int k = 1; k <= d.gamma; ++k) {
    if (rnn) {
      const bool rowpass = rnn->tc && rowpass_supported(ws, d.B);
      const cudaError_t e =
          launch_rnn_cell(ws, a, rnn->Wr, rnn->Hp, rnn->S, rnn->ovec, rowpass ? rnn->oimg : nullptr, k, st, launches);
      if (e != cudaSuccess) return e;
    }
    if (rnn && rnn->tc) {  // the block pass on tcgen05 (requests as MMA rows where the shape allows)
      const cudaError_t e = rowpass_supported(ws, d.B)
                                ? launch_rnn_blocks_rowpass(ws, a.U, a.W2, ovec, rnn->oimg, k, st)
                                : launch_rnn_blocks_tc(ws, a.U, a.W2, ovec, k, st);
      if (e != cudaSuccess) return e;
    } else {
      const cudaError_t e =
          launch_ex(k_draft_blocks<BF16>, dim3(chunks, d.B), dim3(kSimtThreads), smem, st, true, a.U, a.W1, a.W2,
                    a.anchor, a.tokens, ovec, d.gamma, d.V, d.r, k, nblk, ws->s.blk, ws->s.status);
      if (e != cudaSuccess) return e;
    }
    // the steps are chained by programmatic dependent launch (the block
    // pass, the cell and the pick wait in-kernel for the kernel before)
    const cudaError_t e = launch_ex(k_draft_pick<BF16>, dim3(d.B), dim3(kPickThreadsS), smem, st, true,
                                    a.U, a.W1, a.W2, a.anchor, a.w, a.T, ws->s.s_h, ovec, d.gamma, d.V, d.r, d.H, k,
                                    nblk, ws->s.blk, rng, a.tokens, a.pd_tok, a.lse, a.conf, ws->s.status);
    if (e != cudaSuccess) return e;
    *launches += 2;
  }
  return cudaGetLastError();
}

cudaError_t launch_draft_simt(const dspark_ws* ws, const DraftArgs& a, cudaStream_t st, int* launches) {
  if (ws->d.wdtype == DSPARK_BF16) return draft_simt_impl<1>(ws, a, st, launches);
  return draft_simt_impl<0>(ws, a, st, launches);
}

cudaError_t launch_rnn_draft(const dspark_ws* ws, const DraftArgs& a, const void* Wr, float* Hp, float* S,
                             float* ovec, void* hl, __nv_bfloat16* oimg, size_t oimg_len, cudaStream_t st,
                             int* launches) {
  cudaError_t e = launch_conf_hidden(ws, a.h, a.w, st, launches);
  if (e == cudaSuccess) {
    if (hl && rnn_hproj_tc_supported(ws))
      e = launch_rnn_hproj_tc(ws, a.h, Wr, Hp, hl, st, launches);
    else
      e = launch_rnn_hproj(ws, a.h, Wr, Hp, st, launches);
  }
  if (e == cudaSuccess) e = cudaMemsetAsync(S, 0, sizeof(float) * (size_t)ws->d.B * ws->d.r, st);  // s_0 = 0 (buffer 0)
  // the images' rows past the last request stay zero (the cell writes the others every step)
  if (e == cudaSuccess && ws->d.B % 128 != 0) e = cudaMemsetAsync(oimg, 0, oimg_len, st);
  if (e != cudaSuccess) return e;
  const RnnStep rnn{Wr, Hp, S, ovec, ws->use_tc && ws->geo.resid_tc_ok && ws->d.r <= 256, oimg};
  if (ws->d.wdtype == DSPARK_BF16) return draft_simt_impl<1>(ws, a, st, launches, &rnn);
  return draft_simt_impl<0>(ws, a, st, launches, &rnn);
}

}  // namespace dspark
