// k_rnn_tc.cu -- the RNN head's h projection on tcgen05 (sm_103a).
//
// The RNN head of deepseek.csdn.net's reading, §4.2, eq. (6), feeds
// z_k = [s_{k-1}; W1[x_{k-1}]; h_k] to three r x (2r + H) matrices. The h_k
// part, Hp[m][n] = sum_i h[m][i] Wr[n][2r + i] for every position m = (b, k)
// and n < 3r (W_g, W_c, W_o stacked), does not depend on drafted tokens, so it
// is one [B*gamma x H] x [H x 3r] product per round, ahead of the step loop.
//
// h is fp32 and the tensor cores take bf16, so h is split first into
// hi = bf16(h) and lo = bf16(h - hi) (k_hsplit; h is then carried to about 16
// mantissa bits, the way the head vectors o_k enter the vocabulary pass) and
// the product runs over K' = 2H: [hi | lo] x [Wr_h | Wr_h]. k_hproj_tc takes a
// 128 x N output tile (N = 3r split into tiles of at most 256) over one of
// ten slices of K', so that 5 x 3 x 10 = 150 CTAs cover the prod shape;
// it writes its fp32 partial product to Hp[slice], and the cell adds the
// slices in order (the layout of the CUDA-core k_rnn_hproj).
//
//   warp 0      TMA producer: per 64-wide K block an A box [128 x 64] of
//               [hi | lo] and a B box [N x 64] of Wr's h columns (both
//               K-major, 128-byte swizzle) into a 4-stage ring;
//   warp 1      allocates 256 TMEM columns, issues tcgen05.mma (M = 128,
//               N, K = 16, bf16 -> fp32) and commits;
//   warps 2-5   epilogue: one TMEM lane quarter each, 32 columns at a time,
//               to Hp.
// Every wait is bounded; a timeout sets DSPARK_ETIMEOUT and every role ends.
#include <cudaTypedefs.h>
#include <string.h>

#include "dspark_common.cuh"
#include "dspark_internal.h"
#include "tc_ptx.cuh"

namespace dspark {

namespace {

constexpr int kHtM = 128;        // output rows per tile (MMA M)
constexpr int kHtKb = 64;        // K elements per stage (one 128-byte swizzled row)
constexpr int kHtStages = 4;
constexpr int kHtThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kHtNMax = 256;
constexpr int kHtASize = kHtM * kHtKb * 2;      // 16 KB
constexpr int kHtBSize = kHtNMax * kHtKb * 2;   // 32 KB
constexpr int kHtStage = kHtASize + kHtBSize;   // 48 KB
constexpr int kHtSplit = kRnnHpSlices;          // K' slices (the cell adds the partial products in order)
constexpr size_t kHtSmem = (size_t)kHtStages * kHtStage + 1024 + 256;

// h [M][H] fp32 -> hl [M][2H] bf16: hi in columns [0, H), lo in [H, 2H).
__global__ void k_hsplit(const float* __restrict__ h, int M, int H, __nv_bfloat16* __restrict__ hl) {
  const size_t q = (size_t)blockIdx.x * blockDim.x + threadIdx.x;  // 4 floats per thread (H % 4 == 0)
  const size_t n4 = (size_t)M * H / 4;
  if (q >= n4) return;
  const size_t m = q * 4 / H, i = q * 4 - m * H;
  const float4 x = __ldcs(reinterpret_cast<const float4*>(h) + q);
  const float xs[4] = {x.x, x.y, x.z, x.w};
  __nv_bfloat16 hi[4], lo[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    hi[e] = __float2bfloat16_rn(xs[e]);
    lo[e] = __float2bfloat16_rn(xs[e] - __bfloat162float(hi[e]));
  }
  __nv_bfloat16* row = hl + m * 2 * (size_t)H;
  *reinterpret_cast<uint2*>(row + i) = *reinterpret_cast<const uint2*>(hi);
  *reinterpret_cast<uint2*>(row + H + i) = *reinterpret_cast<const uint2*>(lo);
}

__global__ void __launch_bounds__(kHtThreads, 1)
    k_hproj_tc(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, int M, int H,
               int N3, int NT, float* __restrict__ Hp, int* __restrict__ status) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t bars = sbase + kHtStages * kHtStage;
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (kHtStages + s); };
  const uint32_t tfull = bars + 8u * (2 * kHtStages);
  const uint32_t drain = tfull + 8u;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kHtStages * kHtStage + 128);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + kHtStages * kHtStage + 144);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * NT, m0 = blockIdx.y * kHtM, sl = blockIdx.z;
  const int N = min(NT, N3 - n0);
  const int nkb = 2 * H / kHtKb;  // K' blocks
  const int per = (nkb + kHtSplit - 1) / kHtSplit;
  const int kb0 = min(nkb, sl * per), kb1 = min(nkb, kb0 + per);
  float* out = Hp + (size_t)sl * M * N3;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kHtStages; ++s) {
      tc::mbar_init(full(s), 1);
      tc::mbar_init(empty(s), 1);
    }
    tc::mbar_init(tfull, 1);
    tc::mbar_init(drain, 1);
    *abort = 0;
    tc::fence_barrier_init();
    tc::prefetch_tmap(&tm_a);
    tc::prefetch_tmap(&tm_b);
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(tmem_holder), kHtNMax);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    if (lane == 0 && kb1 > kb0) {
      const uint64_t pol_a = tc::policy_evict_first();  // [hi | lo] is read by three N tiles, then dropped
      const uint64_t pol_b = tc::policy_evict_last();   // Wr's h columns by every M tile
      int iss = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1 && ok; ++kb, ++iss) {
        const int s = iss % kHtStages;
        ok = tc::mbar_wait(empty(s), ((iss / kHtStages) & 1) ^ 1, abort);
        if (!ok) break;
        const int kp = kb * kHtKb;  // K' coordinate; B's is the same column of Wr_h for hi and lo
        tc::mbar_arrive_expect_tx(full(s), (uint32_t)(kHtASize + N * kHtKb * 2));
        tc::tma_load_2d(sbase + s * kHtStage, &tm_a, kp, m0, full(s), pol_a);
        tc::tma_load_2d(sbase + s * kHtStage + kHtASize, &tm_b, kp < H ? kp : kp - H, n0, full(s), pol_b);
      }
      if (!ok) {
        if (!*abort) raise_status(status, DSPARK_ETIMEOUT);
        *abort = 1;
        volatile int never = 0;  // the copies already issued land before the CTA can exit
        for (int i = max(0, iss - kHtStages); i < iss; ++i)
          tc::mbar_wait(full(i % kHtStages), (i / kHtStages) & 1, &never);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && kb1 > kb0) {
      const uint32_t idesc = tc::idesc_bf16_f32(kHtM, N, false);
      bool ok = true;
      int it = 0;
      for (int kb = kb0; kb < kb1 && ok; ++kb, ++it) {
        const int s = it % kHtStages;
        ok = tc::mbar_wait(full(s), (it / kHtStages) & 1, abort);
        if (!ok) break;
        tc::tc_fence_after();
        const uint32_t sa = sbase + s * kHtStage, sb = sa + kHtASize;
#pragma unroll
        for (int kk = 0; kk < kHtKb / 16; ++kk)
          tc::mma_bf16(tmem, tc::smem_desc(sa + kk * 32, 16, 1024), tc::smem_desc(sb + kk * 32, 16, 1024), idesc,
                       (it > 0 || kk > 0) ? 1u : 0u);
        tc::mma_commit(empty(s));
      }
      if (ok) {
        tc::mma_commit(tfull);
      } else {
        if (!*abort) raise_status(status, DSPARK_ETIMEOUT);
        *abort = 1;
      }
      tc::mma_commit(drain);  // every MMA issued completes before TMEM is freed
      volatile int never = 0;
      tc::mbar_wait(drain, 0, &never);
    }
  } else {
    // epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 (output rows)
    const int q = warp & 3, m = m0 + q * 32 + lane;
    bool ok = true;
    if (kb1 > kb0) {
      ok = tc::mbar_wait(tfull, 0, abort);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (ok) tc::tc_fence_after();
    }
    if (ok) {
      for (int c = 0; c < N; c += 32) {
        float v[32];
        if (kb1 > kb0) {
          tc::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c, v);
          tc::tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0.f;  // an empty slice adds nothing
        }
        if (m < M) {
          float4* dst = reinterpret_cast<float4*>(out + (size_t)m * N3 + n0 + c);
#pragma unroll
          for (int e = 0; e < 8; ++e) dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
        }
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kHtNMax);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// N tile: 3r in equal tiles of at most 256 columns, each a multiple of 32
int hproj_ntile(int r) {
  const int N3 = 3 * r, nt = (N3 + kHtNMax - 1) / kHtNMax;
  return N3 / nt;
}

}  // namespace

bool rnn_hproj_tc_shape(const dspark_dims& d) {
  if (d.wdtype != DSPARK_BF16 || d.H < kHtKb || d.H % kHtKb != 0) return false;
  if (d.r % 64 != 0 || d.r > 256) return false;
  const int nt = hproj_ntile(d.r);
  return nt % 32 == 0 && (3 * d.r) % nt == 0;
}

bool rnn_hproj_tc_supported(const dspark_ws* ws) {
  return ws->use_tc && rnn_hproj_tc_shape(ws->d) && encode_fn() != nullptr;
}

size_t rnn_hsplit_bytes(const dspark_dims& d) {
  const size_t b = sizeof(__nv_bfloat16) * 2 * (size_t)d.B * d.gamma * d.H;
  return (b + 255) / 256 * 256;
}

cudaError_t launch_rnn_hproj_tc(const dspark_ws* ws, const float* h, const void* Wr, float* Hp, void* hl_scratch,
                                cudaStream_t st, int* launches) {
  const dspark_dims& d = ws->d;
  const int M = d.B * d.gamma, H = d.H, r = d.r, N3 = 3 * r, NT = hproj_ntile(r);
  static bool configured = false;
  if (!configured) {
    const cudaError_t e = cudaFuncSetAttribute(k_hproj_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kHtSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  __nv_bfloat16* hl = static_cast<__nv_bfloat16*>(hl_scratch);
  const size_t n4 = (size_t)M * H / 4;
  k_hsplit<<<(unsigned)((n4 + 255) / 256), 256, 0, st>>>(h, M, H, hl);
  ++*launches;
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  CUtensorMap tm_a, tm_b;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)(2 * H), (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)(2 * H) * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kHtKb, (cuuint32_t)kHtM};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&tm_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, hl, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // Wr's h columns: rows n < 3r of Wr [3r][2r + H], columns 2r .. 2r + H - 1
    const __nv_bfloat16* wb = static_cast<const __nv_bfloat16*>(Wr) + 2 * r;
    const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)N3};
    const cuuint64_t strides[1] = {(cuuint64_t)(2 * r + H) * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kHtKb, (cuuint32_t)NT};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&tm_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16*>(wb), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const dim3 grid((unsigned)(N3 / NT), (unsigned)((M + kHtM - 1) / kHtM), kHtSplit);
  k_hproj_tc<<<grid, kHtThreads, kHtSmem, st>>>(tm_a, tm_b, M, H, N3, NT, Hp, ws->s.status);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace dspark
