// dspark_common.cuh -- device helpers shared by the DSpark kernels.
//
// Random stream: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies
// (0xD2511F53 on word 0, 0xCD9E8D57 on word 2) with the key bumped by the Weyl
// constants 0x9E3779B9 / 0xBB67AE85 between rounds. Counter layout of this
// library: (v >> 2, b, j, purpose << 24 | round mod 2^24), key = seed, output
// word v & 3. Uniforms live on the odd grid u = (2m + 1) 2^-24 (never 0 or 1,
// exact in fp32); Gumbel noise is -log(-log u).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "dspark.h"

namespace dspark {

// Stream purposes (counter word 3, bits 24..31).
enum : uint32_t {
  kDraftBlock = 1,
  kDraftToken = 2,
  kAccept = 3,
  kBonusBlock = 4,
  kBonusToken = 5,
  kResidBlock = 6,
  kResidToken = 7,
  kTreeAccept = 8,  // PCTree: accept test of child i at a node (j = node, v = i)
  kTreeBlock = 9,   // PCTree: the next anchor's block and token draws (j = node)
  kTreeToken = 10,
};

// Width of the vocabulary blocks of the two-level sampler: a block is drawn
// by argmax_s (log mass_s + G_s), then a token inside it by
// argmax_v (log weight_v + G_v) over the block's tokens; together an exact
// draw from the softmax. Every draw of the library (draft, bonus, residual)
// takes this form.
constexpr int kBlockW = 64;

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    if (i > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// The counter's request word is the request's index in the whole batch: a
// workspace that holds requests b0 .. b0 + B - 1 of a batch split across
// devices passes b0, so every request draws the same numbers wherever it runs.
struct Rng {
  uint32_t k0, k1, tag;  // tag = purpose << 24 | round mod 2^24 (without purpose)
  uint32_t b0;           // batch index of the workspace's request 0
  __host__ __device__ static Rng make(uint64_t seed, uint64_t round, uint32_t b0 = 0) {
    Rng r;
    r.k0 = (uint32_t)(seed & 0xFFFFFFFFull);
    r.k1 = (uint32_t)(seed >> 32);
    r.tag = (uint32_t)(round & 0xFFFFFFull);
    r.b0 = b0;
    return r;
  }
  // all four words of the counter block that holds token v (b: index in the workspace)
  __device__ __forceinline__ uint4 block4(uint32_t purpose, uint32_t b, uint32_t j, uint32_t v) const {
    return philox4x32_10(make_uint4(v >> 2, b0 + b, j, (purpose << 24) | tag), k0, k1);
  }
  __device__ __forceinline__ uint32_t word(uint32_t purpose, uint32_t b, uint32_t j, uint32_t v) const {
    const uint4 o = block4(purpose, b, j, v);
    const uint32_t s = v & 3u;
    return s == 0 ? o.x : (s == 1 ? o.y : (s == 2 ? o.z : o.w));
  }
};

__device__ __forceinline__ float u01(uint32_t x) {
  return (float)(2u * (x >> 9) + 1u) * 0x1p-24f;  // exact: 2m+1 < 2^24
}

__device__ __forceinline__ float gumbel(uint32_t x) { return -logf(-logf(u01(x))); }

__device__ __forceinline__ float ld_w(const void* W, int bf16, size_t i) {
  if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(W)[i]);
  return reinterpret_cast<const float*>(W)[i];
}

// Offset (bf16 elements) of the 16-byte piece ch of K-block kb of row m in a
// K-major MMA operand of `rows` rows with the 128-byte swizzle: 8-row atoms
// of 1 KB, K-blocks of 64 elements rows x 128 bytes apart.
__device__ __forceinline__ size_t kmajor_sw128_piece(int m, int kb, int ch, int rows) {
  return (size_t)kb * (rows * 64) + (m >> 3) * 512 + (m & 7) * 64 + ((ch ^ (m & 7)) << 3);
}

// Largest key wins; equal keys go to the smaller index (the first maximum).
// "Nothing yet" is {-inf, kNoIdx}.
constexpr int kNoIdx = 0x7FFFFFFF;
struct KeyIdx {
  float key;
  int idx;
};
__device__ __forceinline__ KeyIdx key_none() { return KeyIdx{-INFINITY, kNoIdx}; }
__device__ __forceinline__ KeyIdx better(KeyIdx a, KeyIdx b) {
  return (b.key > a.key || (b.key == a.key && b.idx < a.idx)) ? b : a;
}
__device__ __forceinline__ KeyIdx warp_best(KeyIdx x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    KeyIdx y;
    y.key = __shfl_xor_sync(0xFFFFFFFFu, x.key, o);
    y.idx = __shfl_xor_sync(0xFFFFFFFFu, x.idx, o);
    x = better(x, y);
  }
  return x;
}

// (max, sum of exp(x - max)) pair combination for online log-sum-exp.
struct MS {
  float m, s;
};
__device__ __forceinline__ MS ms_combine(MS a, MS b) {
  if (a.m == -INFINITY) return b;
  if (b.m == -INFINITY) return a;
  const float m = fmaxf(a.m, b.m);
  return MS{m, a.s * __expf(a.m - m) + b.s * __expf(b.m - m)};
}
__device__ __forceinline__ MS warp_ms(MS x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    MS y;
    y.m = __shfl_xor_sync(0xFFFFFFFFu, x.m, o);
    y.s = __shfl_xor_sync(0xFFFFFFFFu, x.s, o);
    x = ms_combine(x, y);
  }
  return x;
}
__device__ __forceinline__ float ms_log(MS a) { return a.m == -INFINITY ? -INFINITY : a.m + logf(a.s); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
  return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
  return x;
}

// sum_{i<H} w[i] hr[i] by a CTA of 128 threads; the result is valid in
// every thread. `red` is a 4-float shared array of the caller.
__device__ __forceinline__ float hidden_dot128(const float* __restrict__ hr, const float* __restrict__ w, int H,
                                               float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float acc = 0.f;
  if ((H & 3) == 0) {
    const float4* h4 = reinterpret_cast<const float4*>(hr);
    const float4* w4 = reinterpret_cast<const float4*>(w);
    // up to 16 of a thread's float4 pairs loaded before any is used (H = 5120
    // is one round), then accumulated in index order
    for (int i0 = threadIdx.x; i0 < H / 4; i0 += 16 * 128) {
      float4 a[16], c[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int i = i0 + u * 128;
        a[u] = i < H / 4 ? __ldcs(h4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);  // h is streamed once
        c[u] = i < H / 4 ? __ldg(w4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        if (i0 + u * 128 >= H / 4) break;
        acc = fmaf(a[u].x, c[u].x, acc);
        acc = fmaf(a[u].y, c[u].y, acc);
        acc = fmaf(a[u].z, c[u].z, acc);
        acc = fmaf(a[u].w, c[u].w, acc);
      }
    }
  } else {
    for (int i = threadIdx.x; i < H; i += 128) acc = fmaf(hr[i], w[i], acc);
  }
  acc = warp_sum(acc);
  if (lane == 0) red[warp] = acc;
  __syncthreads();
  return (red[0] + red[1]) + (red[2] + red[3]);
}

// Programmatic dependent launch. Inside dspark_round the planner, the sweep
// and the residual kernels are launched so that each may start while the
// kernel before it drains (CUDA's programmatic stream serialization); such a
// kernel calls pdl_wait() before it touches anything an earlier kernel of the
// round writes, which returns once those kernels have completed and their
// writes are visible. Launched without that attribute, pdl_wait() returns at
// once. pdl_trigger() lets the next kernel of the round be scheduled as soon
// as every CTA of this one has issued it.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// First error wins; kernels poll it to stop early.
__device__ __forceinline__ void raise_status(int* st, int code) { atomicCAS(st, 0, code); }

}  // namespace dspark
