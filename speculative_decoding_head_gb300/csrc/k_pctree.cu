// k_pctree.cu -- PCTree: the Markov head's draft made a tree (sm_103a).
//
// "DeepSeek-V4.1 模型结构（6）：解码，DSpark", follow-up note ("后续工作"): the
// Markov head already scores every child token under a parent token, so the
// chain becomes a tree -- candidate children per parent, the most probable
// paths kept within a fixed verify budget, no retraining and no extra
// backbone pass. The build below is best first: node 0 is the anchor (depth
// 0, log-probability 0); expanding a node x at depth k < gamma proposes its c
// most probable children under p_d(. | x) = softmax(U[b, k] + W1[x] W2), each
// with its parent's path log-probability plus log p_d(child); the best
// frontier candidate (higher log-probability, then smaller depth, parent,
// token) is admitted as the next node and expanded in turn, until N nodes
// besides the root are in. The verify is lossless: at a node with target
// p = softmax(P[node]), its children are tried in admission order, child i
// accepted with its current renormalised probability p(t_i) / (1 - the
// probability of the children already rejected); an accepted child becomes
// the node; otherwise the next anchor is drawn from p with the rejected
// children removed (the two-level sampler, purposes 9 and 10 at j = node).
//
// Kernels, per expansion step (N steps; a request whose frontier runs dry is
// done and its later steps do nothing):
//   k_resid_tc<kModeTree> (k_resid_tc.cu) or k_tree_blocks (CUDA cores):
//                      per request and 64-token block, the log-mass and the
//                      maximum of z = U[b, depth] + W1[token] W2 of the node
//                      being expanded;
//   k_tree_pick        grid (B): log-sum-exp over the blocks; the c blocks with
//                      the largest maxima hold the c largest z (a block holding
//                      one of them has its maximum above every other token
//                      outside them), so z is recomputed for those tokens
//                      only and the top c become children; then the frontier's
//                      best candidate is admitted.
// The verify: k_tree_verify, one CTA per request walking down its tree, each
// visited node's target row streamed once through a ring of bulk copies.
#include <stdio.h>

#include "dspark_common.cuh"
#include "dspark_internal.h"
#include "tc_ptx.cuh"

namespace dspark {

constexpr int kTreeMaxC = kTreeMaxChildren;  // children per expanded node
constexpr int kPickT = 1024;   // k_tree_pick threads
constexpr int kPickKG = kPickT / kBlockW;  // K slices of the z recompute (16)

struct TreeScratch {
  int4* state;       // [B] (nodes admitted n, node to expand, frontier size, done)
  float4* frontier;  // [B][N c] (log-probability, depth, parent, token) candidates
  float* bmax;       // [B][nblk] block maxima of the expansion's z
};

__host__ __device__ inline size_t tree_align(size_t x) { return (x + 255) / 256 * 256; }

size_t tree_scratch_bytes(const dspark_dims& d, int nblk, int c, int N) {
  return tree_align(sizeof(int4) * (size_t)d.B) + tree_align(sizeof(float4) * (size_t)d.B * N * c) +
         tree_align(sizeof(float) * (size_t)d.B * nblk);
}

static TreeScratch tree_scratch(void* base, const dspark_dims& d, int c, int N) {
  char* p = static_cast<char*>(base);
  TreeScratch t;
  t.state = reinterpret_cast<int4*>(p);
  p += tree_align(sizeof(int4) * (size_t)d.B);
  t.frontier = reinterpret_cast<float4*>(p);
  p += tree_align(sizeof(float4) * (size_t)d.B * N * c);
  t.bmax = reinterpret_cast<float*>(p);
  return t;
}

// "a goes before b" for frontier candidates: higher log-probability, then
// smaller depth, parent, token
__device__ __forceinline__ bool cand_before(float4 a, float4 b) {
  if (a.x != b.x) return a.x > b.x;
  if (a.y != b.y) return a.y < b.y;
  if (a.z != b.z) return a.z < b.z;
  return a.w < b.w;
}

// (value, index) with the larger value first, ties to the smaller index
__device__ __forceinline__ bool vi_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// every node empty but the root (the anchor); every request starts active
__global__ void k_tree_init(const int32_t* __restrict__ anchor, int B, int N, int V, int32_t* __restrict__ tok,
                            int32_t* __restrict__ par, int32_t* __restrict__ dep, float* __restrict__ lp,
                            int4* __restrict__ state, int* __restrict__ status) {
  const int b = blockIdx.x;
  for (int i = threadIdx.x; i <= N; i += blockDim.x) {
    const size_t o = (size_t)b * (N + 1) + i;
    int t = -1;
    if (i == 0) {
      t = anchor[b];
      if (t < 0 || t >= V) {
        raise_status(status, DSPARK_ERANGE);
        t = 0;
      }
    }
    tok[o] = t;
    par[o] = -1;
    dep[o] = i == 0 ? 0 : -1;
    lp[o] = i == 0 ? 0.f : -INFINITY;
  }
  if (threadIdx.x == 0) state[b] = make_int4(0, 0, 0, 0);
}

// The expansion pass on CUDA cores (shapes the tcgen05 pass does not take):
// grid (chunks, B), a warp per 64-token block.
template <int BF16>
__global__ void __launch_bounds__(256)
    k_tree_blocks(const float* __restrict__ U, const void* __restrict__ W1, const void* __restrict__ W2,
                  const int32_t* __restrict__ tok, const int32_t* __restrict__ dep, const int4* __restrict__ state,
                  int N, int g, int V, int r, int nblk, float* __restrict__ blk, float* __restrict__ bmax) {
  extern __shared__ float e[];  // W1[token], [r]
  const int b = blockIdx.y;
  const int4 st = state[b];
  if (st.w) return;
  const int node = min(max(st.y, 0), N);
  const int x = min(max(tok[(size_t)b * (N + 1) + node], 0), V - 1);
  const int d = min(max(dep[(size_t)b * (N + 1) + node], 0), g - 1);
  for (int i = threadIdx.x; i < r; i += blockDim.x) e[i] = ld_w(W1, BF16, (size_t)x * r + i);
  __syncthreads();
  const float* Urow = U + ((size_t)b * g + d) * V;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, wpc = blockDim.x >> 5;
  for (int s = blockIdx.x * wpc + warp; s < nblk; s += gridDim.x * wpc) {
    const int v0 = s * kBlockW + lane, v1 = v0 + 32;
    float z0 = -INFINITY, z1 = -INFINITY;
    if (v0 < V) {
      float acc = 0.f;
      for (int i = 0; i < r; ++i) acc = fmaf(e[i], ld_w(W2, BF16, (size_t)i * V + v0), acc);
      z0 = Urow[v0] + acc;
    }
    if (v1 < V) {
      float acc = 0.f;
      for (int i = 0; i < r; ++i) acc = fmaf(e[i], ld_w(W2, BF16, (size_t)i * V + v1), acc);
      z1 = Urow[v1] + acc;
    }
    const float m = warp_max(fmaxf(z0, z1));
    float t = (v0 < V ? expf(z0 - m) : 0.f) + (v1 < V ? expf(z1 - m) : 0.f);
    t = warp_sum(t);
    if (lane == 0) {
      blk[(size_t)b * nblk + s] = m == -INFINITY ? -INFINITY : m + logf(t);
      bmax[(size_t)b * nblk + s] = m;
    }
  }
}

// Insert (v, i) into a lane's list of the kTreeMaxC best (value, index)
// pairs, best first (empty entries have index -1 and sit at the end): the
// carried pair sinks past every entry it goes before.
__device__ __forceinline__ void list_insert(float (&lv)[kTreeMaxC], int (&li)[kTreeMaxC], float v, int i) {
#pragma unroll
  for (int j = 0; j < kTreeMaxC; ++j) {
    if (i >= 0 && (li[j] < 0 || vi_before(v, i, lv[j], li[j]))) {
      const float tv = lv[j];
      const int ti = li[j];
      lv[j] = v;
      li[j] = i;
      v = tv;
      i = ti;
    }
  }
}

// The warp's k best of the lanes' lists (indices distinct across lanes): each
// round takes the best head and its lane drops it. out_* hold the k best in
// order in every lane; missing entries are (-inf, -1).
__device__ __forceinline__ void warp_merge_top(float (&lv)[kTreeMaxC], int (&li)[kTreeMaxC], int k,
                                               float (&out_v)[kTreeMaxC], int (&out_i)[kTreeMaxC]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < kTreeMaxC; ++t) {
    out_v[t] = -INFINITY;
    out_i[t] = -1;
    if (t >= k) continue;
    float v = lv[0];
    int i = li[0], src = lane;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, v, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, i, o);
      const int os = __shfl_xor_sync(0xFFFFFFFFu, src, o);
      const bool take = oi >= 0 && (i < 0 || vi_before(ov, oi, v, i) || (oi == i && os < src));
      if (take) {
        v = ov;
        i = oi;
        src = os;
      }
    }
    out_v[t] = v;
    out_i[t] = i;
    if (lane == src && i >= 0) {
#pragma unroll
      for (int j = 0; j + 1 < kTreeMaxC; ++j) {
        lv[j] = lv[j + 1];
        li[j] = li[j + 1];
      }
      lv[kTreeMaxC - 1] = -INFINITY;
      li[kTreeMaxC - 1] = -1;
    }
  }
}

// One expansion step and one admission for request b (one CTA).
template <int BF16>
__global__ void __launch_bounds__(kPickT)
    k_tree_pick(const float* __restrict__ U, const void* __restrict__ W1, const void* __restrict__ W2, int g,
                int V, int r, int nblk, int c, int N, const float* __restrict__ blk, const float* __restrict__ bmax,
                int32_t* __restrict__ tok, int32_t* __restrict__ par, int32_t* __restrict__ dep,
                float* __restrict__ lp, int4* __restrict__ state, float4* __restrict__ frontier,
                int* __restrict__ status) {
  extern __shared__ float e[];  // W1[token] [r]
  __shared__ MS red_ms[kPickT / 32];
  __shared__ int s_blk[kTreeMaxC];
  __shared__ float cz[kTreeMaxC * kBlockW];  // z of the candidate tokens
  __shared__ int cv[kTreeMaxC * kBlockW];
  __shared__ float zp[kPickKG][kTreeMaxC * kBlockW];  // K-slice partial sums of the recompute
  __shared__ float wl_v[kPickT / 32][kTreeMaxC];        // each warp's best blocks
  __shared__ int wl_i[kPickT / 32][kTreeMaxC];
  __shared__ float4 red_c[kPickT / 32];
  __shared__ int red_i[kPickT / 32];
  __shared__ float s_L;
  pdl_wait();  // the expansion's block masses (launched as a dependent kernel)
  pdl_trigger();
  const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int4 st = state[b];
  if (st.w) return;
  int n = st.x, nf = st.z;
  const int last = min(max(st.y, 0), N);
  const size_t nb = (size_t)b * (N + 1);
  const int d = dep[nb + last];
  const int x = min(max(tok[nb + last], 0), V - 1);
  float4* fr = frontier + (size_t)b * N * c;
  if (d >= 0 && d < g && c > 0) {
    for (int i = tid; i < r; i += kPickT) e[i] = ld_w(W1, BF16, (size_t)x * r + i);
    // log-sum-exp of z over the blocks' log-masses
    MS ms{-INFINITY, 0.f};
    for (int s = tid; s < nblk; s += kPickT) ms = ms_combine(ms, MS{blk[(size_t)b * nblk + s], 1.f});
    ms = warp_ms(ms);
    if (lane == 0) red_ms[warp] = ms;
    // the c blocks with the largest maxima: every warp its own best c, then
    // warp 0 merges the warps' lists (each lane one warp's)
    {
      float lv[kTreeMaxC];
      int li[kTreeMaxC];
#pragma unroll
      for (int j = 0; j < kTreeMaxC; ++j) {
        lv[j] = -INFINITY;
        li[j] = -1;
      }
      for (int s = tid; s < nblk; s += kPickT) {
        const float m = bmax[(size_t)b * nblk + s];
        if (m > -INFINITY) list_insert(lv, li, m, s);
      }
      float ov[kTreeMaxC];
      int oi[kTreeMaxC];
      warp_merge_top(lv, li, c, ov, oi);
      if (lane == 0)
#pragma unroll
        for (int t = 0; t < kTreeMaxC; ++t) {
          wl_v[warp][t] = ov[t];
          wl_i[warp][t] = oi[t];
        }
    }
    __syncthreads();
    if (warp == 0) {
      float lv[kTreeMaxC];
      int li[kTreeMaxC];
#pragma unroll
      for (int t = 0; t < kTreeMaxC; ++t) {
        lv[t] = wl_v[lane][t];
        li[t] = wl_i[lane][t];
      }
      float ov[kTreeMaxC];
      int oi[kTreeMaxC];
      warp_merge_top(lv, li, c, ov, oi);
      if (lane < kTreeMaxC) {
        int pick = -1;
#pragma unroll
        for (int t = 0; t < kTreeMaxC; ++t)
          if (t == lane) pick = oi[t];
        s_blk[lane] = pick;
      }
      if (lane == 0) {
        MS m2 = red_ms[0];
        for (int i = 1; i < kPickT / 32; ++i) m2 = ms_combine(m2, red_ms[i]);
        s_L = ms_log(m2);
      }
    }
    __syncthreads();
    // z of the chosen blocks' tokens, recomputed in fp32: thread t takes token
    // t % 64 of every chosen block over K rows t / 64, t / 64 + 16, ... (all
    // of its W2 loads in flight), then the slices are added in a fixed order
    const int vl = tid & (kBlockW - 1), kg = tid / kBlockW;
    for (int j = 0; j < c; ++j) {
      const int sb = s_blk[j];
      const int v = sb * kBlockW + vl;
      float acc = 0.f;
      if (sb >= 0 && v < V) {
#pragma unroll 16
        for (int i = kg; i < r; i += kPickKG) acc = fmaf(e[i], ld_w(W2, BF16, (size_t)i * V + v), acc);
      }
      zp[kg][j * kBlockW + vl] = acc;
    }
    __syncthreads();
    const float* Urow = U + ((size_t)b * g + d) * V;
    if (tid < c * kBlockW) {
      const int sb = s_blk[tid / kBlockW];
      const int v = sb * kBlockW + vl;
      float z = -INFINITY;
      if (sb >= 0 && v < V) {
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < kPickKG; ++q) sum += zp[q][tid];
        z = Urow[v] + sum;
      }
      cz[tid] = z;
      cv[tid] = (sb >= 0 && v < V) ? v : -1;
    }
    __syncthreads();
    // the c largest z among them (warp 0), children in decreasing z
    if (warp == 0) {
      float lv[kTreeMaxC];
      int li[kTreeMaxC];
#pragma unroll
      for (int j = 0; j < kTreeMaxC; ++j) {
        lv[j] = -INFINITY;
        li[j] = -1;
      }
      for (int q = lane; q < c * kBlockW; q += 32)
        if (cv[q] >= 0 && cz[q] > -INFINITY) list_insert(lv, li, cz[q], cv[q]);
      float ov[kTreeMaxC];
      int oi[kTreeMaxC];
      warp_merge_top(lv, li, c, ov, oi);
      const float L = s_L, base = lp[nb + last];
      if (lane == 0) {
#pragma unroll
        for (int t = 0; t < kTreeMaxC; ++t)
          if (t < c && oi[t] >= 0 && nf < N * c)
            fr[nf++] = make_float4(base + (ov[t] - L), (float)(d + 1), (float)last, (float)oi[t]);
      }
      nf = __shfl_sync(0xFFFFFFFFu, nf, 0);
    }
    __syncthreads();
    if (tid == 0) red_i[0] = nf;
    __syncthreads();
    nf = red_i[0];
    __syncthreads();
  }
  // ---- admit the frontier's best candidate
  if (n < N && nf > 0) {
    float4 best = make_float4(-INFINITY, 1e30f, 1e30f, 1e30f);
    int bi = -1;
    for (int i = tid; i < nf; i += kPickT) {
      const float4 f4 = fr[i];
      if (bi < 0 || cand_before(f4, best)) {
        best = f4;
        bi = i;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float4 ob;
      ob.x = __shfl_xor_sync(0xFFFFFFFFu, best.x, o);
      ob.y = __shfl_xor_sync(0xFFFFFFFFu, best.y, o);
      ob.z = __shfl_xor_sync(0xFFFFFFFFu, best.z, o);
      ob.w = __shfl_xor_sync(0xFFFFFFFFu, best.w, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
      if (oi >= 0 && (bi < 0 || cand_before(ob, best))) {
        best = ob;
        bi = oi;
      }
    }
    if (lane == 0) {
      red_c[warp] = best;
      red_i[warp] = bi;
    }
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < kPickT / 32; ++w)
        if (red_i[w] >= 0 && (bi < 0 || cand_before(red_c[w], best))) {
          best = red_c[w];
          bi = red_i[w];
        }
      ++n;
      tok[nb + n] = (int)best.w;
      par[nb + n] = (int)best.z;
      dep[nb + n] = (int)best.y;
      lp[nb + n] = best.x;
      fr[bi] = fr[nf - 1];  // the last candidate takes its place
      state[b] = make_int4(n, n, nf - 1, 0);
    }
  } else if (tid == 0) {
    state[b] = make_int4(n, last, nf, 1);  // no more nodes: done
  }
}

// ---------------------------------------------------------------- verify
constexpr int kTvThreads = 512;
constexpr int kTvStages = 4;
constexpr int kTvChunk = 128 * kBlockW;  // floats per stage (32 KB): 128 blocks, four threads each

size_t tree_verify_smem_bytes(int nblk) {
  return (size_t)kTvStages * kTvChunk * 4 + (size_t)nblk * 4 + 64;
}

// One CTA per request: the walk down its tree.
__global__ void __launch_bounds__(kTvThreads)
    k_tree_verify(const float* __restrict__ P, const int32_t* __restrict__ tok, const int32_t* __restrict__ par,
                  int N, int g, int V, int nblk, Rng rng, int32_t* __restrict__ path, int32_t* __restrict__ n_acc,
                  int32_t* __restrict__ next_anchor, int* __restrict__ status) {
  extern __shared__ __align__(128) unsigned char smem[];
  float* stage = reinterpret_cast<float*>(smem);
  float* blkm = stage + (size_t)kTvStages * kTvChunk;  // [nblk] block log-mass without the removed children
  uint64_t* bars = reinterpret_cast<uint64_t*>(blkm + nblk + (nblk & 1));
  __shared__ int ch_node[kTreeMaxC];  // children of the current node, in admission order
  __shared__ int ch_tok[kTreeMaxC];
  __shared__ float ch_logit[kTreeMaxC];     // their target logits in the node's row
  __shared__ int t_tok[kTreeMaxNodes + 1];  // the request's tree
  __shared__ int t_par[kTreeMaxNodes + 1];
  __shared__ int s_nch, s_next;
  __shared__ MS red_ms[kTvThreads / 32];
  __shared__ KeyIdx red_k[kTvThreads / 32];
  const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t nb = (size_t)b * (N + 1);
  const uint32_t bar0 = tc::smem_u32(bars), st0 = tc::smem_u32(stage);
  if (tid == 0) {
    for (int i = 0; i < kTvStages; ++i) tc::mbar_init(bar0 + 8u * i, 1);
    tc::fence_barrier_init();
  }
  for (int i = tid; i <= g; i += kTvThreads) path[(size_t)b * (g + 1) + i] = i == 0 ? 0 : -1;
  for (int i = tid; i <= N; i += kTvThreads) {
    t_tok[i] = tok[nb + i];
    t_par[i] = par[nb + i];
  }
  __syncthreads();
  const int nchunks = (V + kTvChunk - 1) / kTvChunk;
  volatile int never = 0;
  int node = 0, n = 0, phase_base = 0;  // chunks consumed so far (ring phase)
  for (int level = 0; level <= g; ++level) {
    // the node's children (nodes after it whose parent it is, until the
    // first empty slot), in admission order
    if (tid == 0) {
      int k = 0;
      for (int ch = node + 1; ch <= N && t_tok[ch] >= 0; ++ch)
        if (t_par[ch] == node && k < kTreeMaxC) {
          ch_node[k] = ch;
          ch_tok[k] = t_tok[ch];
          ++k;
        }
      s_nch = k;
    }
    __syncthreads();
    const int nch = s_nch;
    const float* row = P + (nb + node) * (size_t)V;
    if (tid < nch) {  // the children's target logits, loaded while the row streams
      const int t = ch_tok[tid];
      ch_logit[tid] = (t >= 0 && t < V) ? row[t] : -INFINITY;
    }
    // stream the row: thread t takes block t of each chunk; per block the
    // log-mass without the children's tokens, and the running total of all
    auto issue = [&](int ch) {
      const int v0 = ch * kTvChunk;
      const uint32_t bytes = (uint32_t)min(kTvChunk, V - v0) * 4u;  // V % 4 == 0
      const int gi = phase_base + ch, sidx = gi % kTvStages;
      tc::mbar_arrive_expect_tx(bar0 + 8u * sidx, bytes);
      tc::bulk_load(st0 + (uint32_t)sidx * kTvChunk * 4u, row + v0, bytes, bar0 + 8u * sidx);
    };
    int issued = 0;
    if (tid == 0)
      for (; issued < kTvStages && issued < nchunks; ++issued) issue(issued);
    MS tot{-INFINITY, 0.f};
    bool failed = false;
    for (int ch = 0; ch < nchunks; ++ch) {
      const int gi = phase_base + ch, sidx = gi % kTvStages;
      const bool ok = tc::mbar_wait(bar0 + 8u * sidx, (gi / kTvStages) & 1, &never);
      if (__syncthreads_or(!ok)) {
        if (tid == 0) {
          raise_status(status, DSPARK_ETIMEOUT);
          // let the copies already issued land before the CTA exits
          for (int c2 = ch; c2 < issued; ++c2) {
            volatile int nv = 0;
            const int g2 = phase_base + c2;
            tc::mbar_wait(bar0 + 8u * (g2 % kTvStages), (g2 / kTvStages) & 1, &nv);
          }
        }
        failed = true;
        break;
      }
      // four threads per 64-token block (a quarter of 16 tokens each); the
      // quarters' 16-byte pieces are read in a rotated order (fewer bank
      // conflicts across the warp); the children's tokens are masked
      const int qb = tid >> 2, qq = tid & 3;
      const int s = ch * (kTvChunk / kBlockW) + qb;
      {
        const float4* xb4 = reinterpret_cast<const float4*>(stage + (size_t)sidx * kTvChunk + qb * kBlockW + qq * 16);
        unsigned rem = 0u;  // the quarter's 16 tokens
        for (int k = 0; k < nch; ++k) {
          const int t = ch_tok[k] - s * kBlockW - qq * 16;
          if (t >= 0 && t < 16) rem |= 1u << t;
        }
        const int vlim = V - s * kBlockW - qq * 16;  // tokens of the quarter inside the vocabulary
        float4 x4[4];
        int jj[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          jj[i] = (i + qb) & 3;
          x4[i] = xb4[jj[i]];
        }
        float mall = -INFINITY, m = -INFINITY;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float xv[4] = {x4[i].x, x4[i].y, x4[i].z, x4[i].w};
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const int e = 4 * jj[i] + c4;
            const float val = (s < nblk && e < vlim) ? xv[c4] : -INFINITY;
            mall = fmaxf(mall, val);
            if (!((rem >> e) & 1u)) m = fmaxf(m, val);
          }
        }
        // the block's maxima over its four quarters (consecutive lanes)
        mall = fmaxf(mall, __shfl_xor_sync(0xFFFFFFFFu, mall, 1));
        mall = fmaxf(mall, __shfl_xor_sync(0xFFFFFFFFu, mall, 2));
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
        float sall = 0.f, sm = 0.f;
        if (mall > -INFINITY) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float xv[4] = {x4[i].x, x4[i].y, x4[i].z, x4[i].w};
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              const int e = 4 * jj[i] + c4;
              const float ev = (s < nblk && e < vlim && xv[c4] > -INFINITY) ? __expf(xv[c4] - mall) : 0.f;
              sall += ev;
              if (!((rem >> e) & 1u)) sm += ev;
            }
          }
        }
        sall += __shfl_xor_sync(0xFFFFFFFFu, sall, 1);
        sall += __shfl_xor_sync(0xFFFFFFFFu, sall, 2);
        sm += __shfl_xor_sync(0xFFFFFFFFu, sm, 1);
        sm += __shfl_xor_sync(0xFFFFFFFFu, sm, 2);
        if (s < nblk && qq == 0) {
          blkm[s] = (m > -INFINITY && sm > 0.f) ? mall + logf(sm) : -INFINITY;
          tot = ms_combine(tot, MS{mall, sall});
        }
      }
      __syncthreads();  // the stage is consumed
      if (tid == 0 && issued < nchunks) issue(issued++);
    }
    if (failed) return;
    phase_base += nchunks;
    tot = warp_ms(tot);
    if (lane == 0) red_ms[warp] = tot;
    __syncthreads();
    // accept tests, in admission order (thread 0)
    if (tid == 0) {
      MS t2 = red_ms[0];
      for (int i = 1; i < kTvThreads / 32; ++i) t2 = ms_combine(t2, red_ms[i]);
      const float L = ms_log(t2);
      int next = -1;
      float gone = 0.f;  // probability of the children rejected so far
      for (int k = 0; k < nch; ++k) {
        const float pt = expf(ch_logit[k] - L);
        const float q = pt / (1.f - gone);
        const float u = u01(rng.word(kTreeAccept, b, node, k));
        if (u < q) {
          next = ch_node[k];
          break;
        }
        gone += pt;
      }
      s_next = next;
    }
    __syncthreads();
    const int next = s_next;
    if (next >= 0 && n < g) {
      node = next;
      ++n;
      if (tid == 0) path[(size_t)b * (g + 1) + n] = node;
      __syncthreads();
      continue;
    }
    // ---- no child accepted: the next anchor from the row without them
    KeyIdx kb = key_none();
    for (int s = tid; s < nblk; s += kTvThreads) {
      const float lm = blkm[s];
      if (lm > -INFINITY) kb = better(kb, KeyIdx{lm + gumbel(rng.word(kTreeBlock, b, node, s)), s});
    }
    kb = warp_best(kb);
    if (lane == 0) red_k[warp] = kb;
    __syncthreads();
    if (warp == 0) {
      KeyIdx k2 = lane < kTvThreads / 32 ? red_k[lane] : key_none();
      k2 = warp_best(k2);
      const int sb = k2.idx;
      KeyIdx kt = key_none();
      if (sb != kNoIdx)
        for (int v = sb * kBlockW + lane; v < min(V, (sb + 1) * kBlockW); v += 32) {
          bool removed = false;
          for (int k = 0; k < nch; ++k) removed |= ch_tok[k] == v;
          if (!removed) kt = better(kt, KeyIdx{row[v] + gumbel(rng.word(kTreeToken, b, node, v)), v});
        }
      kt = warp_best(kt);
      if (lane == 0) {
        if (kt.idx == kNoIdx) raise_status(status, DSPARK_ENUMERIC);
        n_acc[b] = n;
        next_anchor[b] = kt.idx == kNoIdx ? 0 : kt.idx;
      }
    }
    return;
  }
}

__global__ void k_tree_count(const int4* __restrict__ state, int B, int32_t* __restrict__ n_nodes) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) n_nodes[b] = state[b].x;
}

// ---------------------------------------------------------------- host side
cudaError_t launch_pctree_verify(const dspark_ws* ws, const float* P, const int32_t* tok, const int32_t* par, int N,
                                 uint64_t seed, uint64_t round, int32_t* path, int32_t* n_acc, int32_t* next_anchor,
                                 cudaStream_t st, int* launches) {
  const dspark_dims& d = ws->d;
  const size_t smem = tree_verify_smem_bytes(ws->geo.nblk);
  cudaError_t e = cudaFuncSetAttribute(k_tree_verify, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_tree_verify<<<d.B, kTvThreads, smem, st>>>(P, tok, par, N, d.gamma, d.V, ws->geo.nblk, Rng::make(seed, round, (uint32_t)ws->b0),
                                               path, n_acc, next_anchor, ws->s.status);
  ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_pctree_build(const dspark_ws* ws, const float* U, const void* W1, const void* W2,
                                const int32_t* anchor, int c, int N, int32_t* tok, int32_t* par, int32_t* dep,
                                float* lp, int32_t* n_nodes, void* scratch, cudaStream_t st, int* launches) {
  const dspark_dims& d = ws->d;
  const int nblk = ws->geo.nblk;
  TreeScratch ts = tree_scratch(scratch, d, c, N);
  k_tree_init<<<d.B, 128, 0, st>>>(anchor, d.B, N, d.V, tok, par, dep, lp, ts.state, ws->s.status);
  ++*launches;
  const bool tc = ws->use_tc && ws->geo.resid_tc_ok && d.wdtype == DSPARK_BF16;
  const size_t esm = sizeof(float) * d.r;
  for (int step = 0; step < N; ++step) {
    if (tc) {
      const cudaError_t e = rowpass_supported(ws, d.B)
                                ? launch_tree_blocks_rowpass(ws, U, W1, W2, tok, dep, ts.state, N, ws->s.blk, ts.bmax, st)
                                : launch_tree_blocks_tc(ws, U, W1, W2, tok, dep, ts.state, N, ws->s.blk, ts.bmax, st);
      if (e != cudaSuccess) return e;
    } else {
      const int chunks = max(1, (nblk + 31) / 32);
      if (d.wdtype == DSPARK_BF16)
        k_tree_blocks<1><<<dim3(chunks, d.B), 256, esm, st>>>(U, W1, W2, tok, dep, ts.state, N, d.gamma, d.V, d.r,
                                                              nblk, ws->s.blk, ts.bmax);
      else
        k_tree_blocks<0><<<dim3(chunks, d.B), 256, esm, st>>>(U, W1, W2, tok, dep, ts.state, N, d.gamma, d.V, d.r,
                                                              nblk, ws->s.blk, ts.bmax);
    }
    // the expansion and the pick are chained by programmatic dependent launch
    // (each waits in-kernel for the one before)
    const cudaError_t ep =
        d.wdtype == DSPARK_BF16
            ? launch_ex(k_tree_pick<1>, dim3(d.B), dim3(kPickT), esm, st, true, U, W1, W2, d.gamma, d.V, d.r, nblk, c,
                        N, ws->s.blk, ts.bmax, tok, par, dep, lp, ts.state, ts.frontier, ws->s.status)
            : launch_ex(k_tree_pick<0>, dim3(d.B), dim3(kPickT), esm, st, true, U, W1, W2, d.gamma, d.V, d.r, nblk, c,
                        N, ws->s.blk, ts.bmax, tok, par, dep, lp, ts.state, ts.frontier, ws->s.status);
    if (ep != cudaSuccess) return ep;
    *launches += 2;
  }
  k_tree_count<<<(d.B + 127) / 128, 128, 0, st>>>(ts.state, d.B, n_nodes);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace dspark

// ---------------------------------------------------------------- C-ABI
namespace {
bool aligned_to(const void* p, uintptr_t a) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool tree_shape_ok(const dspark_dims& d, int c, int N) {
  return c >= 1 && c <= dspark::kTreeMaxChildren && N >= 1 && N <= dspark::kTreeMaxNodes && d.V < (1 << 24) &&
         c <= d.V;
}
dspark_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return DSPARK_OK;
  fprintf(stderr, "dspark: CUDA error %s\n", cudaGetErrorString(e));
  return DSPARK_ECUDA;
}
}  // namespace

extern "C" size_t dspark_pctree_scratch_bytes(const dspark_ws* ws, int c, int N) {
  if (!ws || !tree_shape_ok(ws->d, c, N)) return 0;
  return dspark::tree_scratch_bytes(ws->d, ws->geo.nblk, c, N);
}

extern "C" dspark_status dspark_pctree_build(dspark_ws* ws, const float* U, const void* W1, const void* W2,
                                             const int32_t* anchor, int c, int N, int32_t* tok, int32_t* par,
                                             int32_t* dep, float* lp, int32_t* n_nodes, void* scratch,
                                             dspark_stream_t stream) {
  if (!ws) return DSPARK_EINVAL;
  if (!tree_shape_ok(ws->d, c, N)) return DSPARK_EUNSUPPORTED;
  if (!aligned_to(U, 16) || !aligned_to(W1, 16) || !aligned_to(W2, 16) || !aligned_to(anchor, 4) ||
      !aligned_to(tok, 4) || !aligned_to(par, 4) || !aligned_to(dep, 4) || !aligned_to(lp, 4) ||
      !aligned_to(n_nodes, 4) || !aligned_to(scratch, 256))
    return DSPARK_EINVAL;
  int launches = 0;
  const cudaError_t e = dspark::launch_pctree_build(ws, U, W1, W2, anchor, c, N, tok, par, dep, lp, n_nodes, scratch,
                                                    reinterpret_cast<cudaStream_t>(stream), &launches);
  ws->last_launches = launches;
  return cuda_status(e);
}

extern "C" dspark_status dspark_pctree_verify(dspark_ws* ws, const float* P, const int32_t* tok, const int32_t* par,
                                              int N, uint64_t seed, uint64_t round, int32_t* path,
                                              int32_t* n_accepted, int32_t* next_anchor, dspark_stream_t stream) {
  if (!ws) return DSPARK_EINVAL;
  if (N < 1 || N > dspark::kTreeMaxNodes || ws->d.V % 4 != 0) return DSPARK_EUNSUPPORTED;
  if (dspark::tree_verify_smem_bytes(ws->geo.nblk) > 227 * 1024) return DSPARK_EUNSUPPORTED;
  if (!aligned_to(P, 16) || !aligned_to(tok, 4) || !aligned_to(par, 4) || !aligned_to(path, 4) ||
      !aligned_to(n_accepted, 4) || !aligned_to(next_anchor, 4))
    return DSPARK_EINVAL;
  int launches = 0;
  const cudaError_t e = dspark::launch_pctree_verify(ws, P, tok, par, N, seed, round, path, n_accepted, next_anchor,
                                                     reinterpret_cast<cudaStream_t>(stream), &launches);
  ws->last_launches = launches;
  return cuda_status(e);
}
