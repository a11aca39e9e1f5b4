// k_draft_tc.cu -- persistent tcgen05 Markov-head draft kernel (sm_103a).
//
// "DeepSeek-V4.1 模型结构（6）：解码，DSpark", eq. (4)/(5) and the sequential
// loop of section "Markov head": for k = 1..gamma,
//   z_k = U_k + W1[x_{k-1}] W2,  x_k ~ softmax(z_k),  x_0 = anchor,
// and eq. (7): c_k = sigma((w^T [h_k; W1[x_{k-1}]]) / T_k) (the temperature is
// the STS sigmoid(raw / T) of the zdszero.github.io "spec_dspark" page).
//
// One cooperative launch runs all gamma steps. Each CTA (one per SM) owns a
// contiguous range of 64-token vocabulary tiles of one 128-row group:
//   warp 0      TMA producer: W2 tile [r x 64] bf16 (128-byte swizzle, L2
//               evict_last: W2 is reused by every step) and U tile [128 x 64]
//               fp32 (evict_first: streamed once), into rings of 2 and 3 stages;
//   warp 1      allocates 128 TMEM columns and issues tcgen05.mma
//               (M = 128 rows, N = 64, K = r in steps of 16) into one of two
//               TMEM accumulators; A = gathered rows W1[x_{k-1}] in shared memory;
//   warps 2-5   epilogue, one thread per row: z = TMEM + U, the block's
//               log-mass (max, sum exp), the block draw key log mass + G_s,
//               the row's online log-sum-exp, and a copy of z for the row's
//               best block so far (to global scratch).
// Between steps the epilogue warps of all CTAs meet at a grid barrier, reduce
// each row's per-CTA partials (one warp per row: log-sum-exp, winning block,
// token draw argmax_v (z_v + G_v) inside it), meet again, and gather the next
// A. The producer keeps prefetching the next step's tiles meanwhile (they do
// not depend on the drafted token).
//
// Every wait is bounded (tc_ptx.cuh); a timeout sets DSPARK_ETIMEOUT, every
// role leaves its loop, in-flight copies and MMAs are drained, TMEM is freed.
#include <cudaTypedefs.h>
#include <stdio.h>
#include <string.h>

#include "dspark_common.cuh"
#include "dspark_internal.h"
#include "tc_ptx.cuh"

namespace dspark {

constexpr int kTcThreads = 192;
constexpr int kTcRows = 128;        // MMA M: rows of one row group
constexpr int kTcN = 64;            // vocabulary tile = one sampler block
constexpr int kNW = 2;              // W2 ring depth
constexpr int kNU = 3;              // U ring depth
constexpr int kUStage = kTcRows * kTcN * 4;  // 32 KB: two 128 x 32 fp32 boxes
constexpr int kUBox = kTcRows * 32 * 4;      // 16 KB
constexpr int kTmemCols = 128;      // two 64-column fp32 accumulators
constexpr int kMaxGroups = 8;       // B <= 1024
constexpr int kMaxPartLanes = 8;    // partials per lane in the row reduction (grid <= 256)

static_assert(kTcN == kBlockW, "a vocabulary tile is one sampler block");

struct TcSmem {  // byte offsets into dynamic shared memory (1024-aligned base)
  uint32_t a, w2, u, bars, misc, total;
  __host__ __device__ static TcSmem make(int r) {
    TcSmem s;
    s.a = 0;
    s.w2 = s.a + kTcRows * r * 2;
    s.u = s.w2 + kNW * r * 128;
    s.bars = s.u + kNU * kUStage;
    s.misc = s.bars + 8 * (2 * kNW + 2 * kNU + 4 + 3);
    s.total = s.misc + 64;
    return s;
  }
};

struct TcParams {
  int B, g, V, r, H;
  int ntiles, nG, G, Ggmax;
  Rng rng;
  const int32_t* anchor;
  const void* W1;
  const float* w;
  const float* T;
  const float* s_h;
  int32_t* tokens;
  float* pd_tok;
  float* lse;
  float* conf;
  int32_t* xbuf;
  float4* dpart;  // [nG * 128][Ggmax]
  float* drec;    // [G][128][64]
  __nv_bfloat16* aimg;  // [nG][128 x r] next A operand, already in its swizzled shared layout
  unsigned* bar;  // [0] arrivals, [1] generation
  int* status;
};

__device__ __forceinline__ int group_ctas(int G, int nG, int g) { return (G - g + nG - 1) / nG; }

// Grid barrier among the epilogue warps (128 threads, named barrier 1) of all
// CTAs. Self-resetting: the last arriver zeroes the count and bumps the
// generation. Returns false if the round is being abandoned.
__device__ bool grid_sync(const TcParams& p, bool leader, volatile int* abort) {
  asm volatile("bar.sync 1, 128;" ::: "memory");
  if (leader && !*abort) {
    const unsigned g0 = tc::ld_acquire_gpu(p.bar + 1);
    __threadfence();
    const unsigned arrived = atomicAdd(p.bar, 1u);
    if (arrived == (unsigned)p.G - 1) {
      atomicExch(p.bar, 0u);
      __threadfence();
      atomicAdd(p.bar + 1, 1u);
    } else {
      const unsigned long long t0 = tc::globaltimer();
      while (tc::ld_acquire_gpu(p.bar + 1) == g0) {
        if (*(volatile int*)p.status != 0) {
          *abort = 1;
          break;
        }
        if (tc::globaltimer() - t0 > tc::kWaitNs) {
          raise_status(p.status, DSPARK_ETIMEOUT);
          *abort = 1;
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
  }
  asm volatile("bar.sync 1, 128;" ::: "memory");
  return !*abort;
}

__global__ void __launch_bounds__(kTcThreads, 1)
    k_draft_tc(const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_u,
               const TcParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the runtime aligns dynamic shared memory to at least 16 B; round up to 1 KB
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const TcSmem L = TcSmem::make(p.r);
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t sA = sbase + L.a, sW2 = sbase + L.w2, sU = sbase + L.u;
  const uint32_t bars = sbase + L.bars;
  auto w2_full = [&](int i) { return bars + 8u * i; };
  auto w2_empty = [&](int i) { return bars + 8u * (kNW + i); };
  auto u_full = [&](int i) { return bars + 8u * (2 * kNW + i); };
  auto u_empty = [&](int i) { return bars + 8u * (2 * kNW + kNU + i); };
  auto t_full = [&](int i) { return bars + 8u * (2 * kNW + 2 * kNU + i); };
  auto t_empty = [&](int i) { return bars + 8u * (2 * kNW + 2 * kNU + 2 + i); };
  const uint32_t a_full = bars + 8u * (2 * kNW + 2 * kNU + 4);
  const uint32_t drain = a_full + 8u;
  const uint32_t a_img = a_full + 16u;  // the bulk copy of the next A image
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L.misc + 16);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int grp = c % p.nG, cg = c / p.nG;  // row group, index within the group
  const int Gg = group_ctas(p.G, p.nG, grp);
  const int tile_lo = (int)((long long)cg * p.ntiles / Gg);
  const int tile_hi = (int)((long long)(cg + 1) * p.ntiles / Gg);
  const int nt = tile_hi - tile_lo;
  const uint32_t w2_bytes = (uint32_t)p.r * 128u;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNW; ++i) {
      tc::mbar_init(w2_full(i), 1);
      tc::mbar_init(w2_empty(i), 1);
    }
    for (int i = 0; i < kNU; ++i) {
      tc::mbar_init(u_full(i), 1);
      tc::mbar_init(u_empty(i), 4);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(t_full(i), 1);
      tc::mbar_init(t_empty(i), 4);
    }
    tc::mbar_init(a_full, 4);
    tc::mbar_init(drain, 1);
    tc::mbar_init(a_img, 1);
    *abort = 0;
    tc::fence_barrier_init();
    tc::prefetch_tmap(&tm_w2);
    tc::prefetch_tmap(&tm_u);
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(tmem_holder), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t keep = tc::policy_evict_last(), stream = tc::policy_evict_first();
      int issued = 0;
      bool ok = true;
      for (int k = 1; k <= p.g && ok; ++k) {
        for (int i = 0; i < nt && ok; ++i) {
          const int it = (k - 1) * nt + i, t = tile_lo + i;
          const int ws = it % kNW, us = it % kNU;
          ok = tc::mbar_wait(w2_empty(ws), ((it / kNW) & 1) ^ 1, abort);
          if (!ok) break;
          tc::mbar_arrive_expect_tx(w2_full(ws), w2_bytes);
          tc::tma_load_2d(sW2 + ws * w2_bytes, &tm_w2, t * kTcN, 0, w2_full(ws), keep);
          ok = tc::mbar_wait(u_empty(us), ((it / kNU) & 1) ^ 1, abort);
          if (!ok) break;
          tc::mbar_arrive_expect_tx(u_full(us), kUStage);
          tc::tma_load_3d(sU + us * kUStage, &tm_u, t * kTcN, k - 1, grp * kTcRows, u_full(us), stream);
          tc::tma_load_3d(sU + us * kUStage + kUBox, &tm_u, t * kTcN + 32, k - 1, grp * kTcRows, u_full(us),
                          stream);
          issued = it + 1;
        }
      }
      if (!ok) {
        if (!*abort) raise_status(p.status, DSPARK_ETIMEOUT);
        *abort = 1;
        // let the copies already issued land before the CTA can exit
        for (int it = issued - 1; it >= 0 && it >= issued - kNU; --it) {
          volatile int never = 0;
          tc::mbar_wait(u_full(it % kNU), (it / kNU) & 1, &never);
          if (it >= issued - kNW) tc::mbar_wait(w2_full(it % kNW), (it / kNW) & 1, &never);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(kTcRows, kTcN, true);
      bool ok = true;
      for (int k = 1; k <= p.g && ok; ++k) {
        ok = tc::mbar_wait(a_full, (k - 1) & 1, abort);
        if (!ok) break;
        tc::tc_fence_after();
        for (int i = 0; i < nt && ok; ++i) {
          const int it = (k - 1) * nt + i;
          const int ws = it % kNW, ab = it & 1;
          ok = tc::mbar_wait(w2_full(ws), (it / kNW) & 1, abort) &&
               tc::mbar_wait(t_empty(ab), ((it >> 1) & 1) ^ 1, abort);
          if (!ok) break;
          tc::tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(ab * kTcN);
          const uint32_t bstage = sW2 + ws * w2_bytes;
          for (int ks = 0; ks < p.r / 16; ++ks) {
            // A: K-major, 128-byte swizzle; K-block of 64 is [128 rows x 128 B],
            // the 16-wide K step moves 32 B inside the swizzled row.
            const uint64_t ad = tc::smem_desc(sA + (ks >> 2) * (kTcRows * 128) + (ks & 3) * 32, 16, 1024);
            // B: N-major (W2 rows are contiguous in N), 128-byte swizzle; each
            // K row is 128 B, 8 rows form a 1 KB atom, 16 rows per K step.
            const uint64_t bd = tc::smem_desc(bstage + ks * 2048, w2_bytes, 1024);
            tc::mma_bf16(d, ad, bd, idesc, ks > 0 ? 1u : 0u);
          }
          tc::mma_commit(w2_empty(ws));
          tc::mma_commit(t_full(ab));
        }
      }
      if (!ok) {
        if (!*abort) raise_status(p.status, DSPARK_ETIMEOUT);
        *abort = 1;
      }
      // every MMA this thread issued completes before TMEM is freed
      tc::mma_commit(drain);
      volatile int never = 0;
      tc::mbar_wait(drain, 0, &never);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Every epilogue warp runs all gamma steps and both grid barriers of each
    // step even after an abort (the named barrier inside grid_sync has no
    // timeout, so no warp may skip one); an abort only skips the work.
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int m = q * 32 + lane;
    const int b = grp * kTcRows + m;
    const bool valid = b < p.B;
    const bool leader = warp == 2 && lane == 0;
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
    const __nv_bfloat16* W1 = reinterpret_cast<const __nv_bfloat16*>(p.W1);
    // warp-uniform view of the abort word (the loops below hold warp collectives)
    auto aborted = [&]() { return __any_sync(0xFFFFFFFFu, *abort != 0); };
    float* rec = p.drec + ((size_t)c * kTcRows + m) * kTcN;
    for (int k = 1; k <= p.g; ++k) {
      // ---- gather A = W1[x_{k-1}] rows (K-major, 128-byte swizzle) and c_k
      if (!aborted() && k > 1) {
        // the reducers of the last step wrote this group's A (rows W1[x_{k-1}]
        // in the swizzled layout) as one contiguous image: one bulk copy
        if (leader) {
          tc::fence_proxy_async_global();
          const uint32_t bytes = (uint32_t)kTcRows * p.r * 2u;
          tc::mbar_arrive_expect_tx(a_img, bytes);
          tc::bulk_load(sA, p.aimg + (size_t)grp * kTcRows * p.r, bytes, a_img);
        }
        bool ok = tc::mbar_wait(a_img, (k - 2) & 1, abort);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) {
          if (lane == 0 && !*abort) {
            raise_status(p.status, DSPARK_ETIMEOUT);
            *abort = 1;
          }
        } else {
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(a_full);
        }
      } else if (!aborted()) {
        int x = 0;
        if (valid) {
          x = p.anchor[b];
          if (x < 0 || x >= p.V) {
            raise_status(p.status, DSPARK_ERANGE);
            x = 0;
          }
        }
        // every 16-byte piece of the row in flight at once (cp.async), written
        // straight into its 128-byte-swizzled position
        const uint4* src = reinterpret_cast<const uint4*>(W1 + (size_t)x * p.r);
        for (int kb = 0; kb < p.r / 64; ++kb) {
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint32_t dst = sA + kb * (kTcRows * 128) + (m >> 3) * 1024 + (m & 7) * 128 +
                                 ((uint32_t)(ch ^ (m & 7)) << 4);
            if (valid) {
              tc::cp_async16(dst, src + kb * 8 + ch);
            } else {
              asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0u) : "memory");
            }
          }
        }
        tc::cp_async_wait_all();
        float cdot = 0.f;
        if (cg == 0 && valid) {
          for (int kb = 0; kb < p.r / 64; ++kb) {
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              uint4 v;
              const uint32_t a = sA + kb * (kTcRows * 128) + (m >> 3) * 1024 + (m & 7) * 128 +
                                 ((uint32_t)(ch ^ (m & 7)) << 4);
              asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
              const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v);
              const float* wr = p.w + p.H + kb * 64 + ch * 8;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(h2[e]);
                cdot = fmaf(f.x, wr[2 * e], cdot);
                cdot = fmaf(f.y, wr[2 * e + 1], cdot);
              }
            }
          }
        }
        if (cg == 0 && valid) {
          const size_t o = (size_t)b * p.g + (k - 1);
          const float raw = p.s_h[o] + cdot;
          const float cf = 1.f / (1.f + expf(-raw / p.T[k - 1]));
          if (!isfinite(cf)) raise_status(p.status, DSPARK_ENUMERIC);
          p.conf[o] = cf;
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(a_full);
      }

      // ---- vocabulary tiles of this CTA
      float M = -INFINITY, S = 0.f, bk = -INFINITY;
      int bs = kNoIdx;
      for (int i = 0; i < nt && !aborted(); ++i) {
        const int it = (k - 1) * nt + i, t = tile_lo + i;
        const int ab = it & 1, us = it % kNU;
        bool ok = tc::mbar_wait(t_full(ab), (it >> 1) & 1, abort) && tc::mbar_wait(u_full(us), (it / kNU) & 1, abort);
        ok = __all_sync(0xFFFFFFFFu, ok);  // tcgen05.ld below is warp-collective
        if (!ok) {
          if (lane == 0 && !*abort) {
            raise_status(p.status, DSPARK_ETIMEOUT);
            *abort = 1;
          }
          break;
        }
        tc::tc_fence_after();
        float z[kTcN];
        tc::tmem_ld32(trow + (uint32_t)(ab * kTcN), z);
        tc::tmem_ld32(trow + (uint32_t)(ab * kTcN + 32), z + 32);
        tc::tmem_wait_ld();
        const uint32_t ub = sU + us * kUStage + m * 128;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            float4 u;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(u.x), "=f"(u.y), "=f"(u.z), "=f"(u.w)
                         : "r"(ub + h * kUBox + ((uint32_t)(cc ^ (m & 7)) << 4)));
            z[h * 32 + cc * 4 + 0] += u.x;
            z[h * 32 + cc * 4 + 1] += u.y;
            z[h * 32 + cc * 4 + 2] += u.z;
            z[h * 32 + cc * 4 + 3] += u.w;
          }
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(t_empty(ab));
          tc::mbar_arrive(u_empty(us));
        }
        if (valid) {
          const int v0 = t * kTcN;
          if (v0 + kTcN > p.V) {
#pragma unroll
            for (int j = 0; j < kTcN; ++j)
              if (v0 + j >= p.V) z[j] = -INFINITY;
          }
          float mb = z[0];
#pragma unroll
          for (int j = 1; j < kTcN; ++j) mb = fmaxf(mb, z[j]);
          float sb = 0.f;
#pragma unroll
          for (int j = 0; j < kTcN; ++j) sb += __expf(z[j] - mb);
          const float lm = mb + logf(sb);
          if (mb > M) {
            S = S * __expf(M - mb) + sb;
            M = mb;
          } else {
            S += sb * __expf(mb - M);
          }
          const float key = lm + gumbel(p.rng.word(kDraftBlock, b, k, t));
          if (key > bk) {  // ties keep the smaller block (processed first)
            bk = key;
            bs = t;
            float4* r4 = reinterpret_cast<float4*>(rec);
#pragma unroll
            for (int j = 0; j < kTcN / 4; ++j) r4[j] = make_float4(z[4 * j], z[4 * j + 1], z[4 * j + 2], z[4 * j + 3]);
          }
        }
      }
      if (valid && !*abort) p.dpart[(size_t)b * p.Ggmax + cg] = make_float4(M, S, bk, __int_as_float(bs));
      grid_sync(p, leader, abort);

      // ---- per-row reduction and the token draw inside the winning block
      const int ew = warp - 2;
      for (int jr = ew; !aborted(); jr += 4) {
        const int br = c + jr * p.G;
        if (br >= p.B) break;
        const int g2 = br / kTcRows, m2 = br % kTcRows;
        const int Gg2 = group_ctas(p.G, p.nG, g2);
        MS ms{-INFINITY, 0.f};
        KeyIdx kb = key_none();
        int owner = -1;
        {
          // every partial of the row in flight at once (written by other CTAs)
          float4 dd[kMaxPartLanes];
#pragma unroll
          for (int u = 0; u < kMaxPartLanes; ++u) {
            const int i = lane + 32 * u;
            dd[u] = i < Gg2 ? __ldcg(p.dpart + (size_t)br * p.Ggmax + i) : make_float4(-INFINITY, 0.f, -INFINITY, __int_as_float(kNoIdx));
          }
#pragma unroll
          for (int u = 0; u < kMaxPartLanes; ++u) {
            const float4 d = dd[u];
            ms = ms_combine(ms, MS{d.x, d.y});
            const KeyIdx nb = better(kb, KeyIdx{d.z, __float_as_int(d.w)});
            if (nb.idx != kb.idx || nb.key != kb.key) owner = lane + 32 * u;
            kb = nb;
          }
        }
        ms = warp_ms(ms);
        const KeyIdx best = warp_best(kb);
        const unsigned own_mask =
            __ballot_sync(0xFFFFFFFFu, owner >= 0 && kb.idx == best.idx && kb.key == best.key);
        const int own_cg = own_mask ? __shfl_sync(0xFFFFFFFFu, owner, __ffs(own_mask) - 1) : -1;
        if (best.idx == kNoIdx || own_cg < 0) {
          if (lane == 0) raise_status(p.status, DSPARK_ENUMERIC);
          continue;
        }
        const int own_c = g2 + p.nG * own_cg;
        const float* r2 = p.drec + ((size_t)own_c * kTcRows + m2) * kTcN;
        const int v0 = best.idx * kTcN + lane, v1 = v0 + 32;
        const float z0 = __ldcg(r2 + lane), z1 = __ldcg(r2 + lane + 32);
        KeyIdx kt = key_none();
        if (v0 < p.V) kt = KeyIdx{z0 + gumbel(p.rng.word(kDraftToken, br, k, v0)), v0};
        if (v1 < p.V) kt = better(kt, KeyIdx{z1 + gumbel(p.rng.word(kDraftToken, br, k, v1)), v1});
        kt = warp_best(kt);
        if (kt.idx == kNoIdx) {
          if (lane == 0) raise_status(p.status, DSPARK_ENUMERIC);
          continue;
        }
        const int jx = kt.idx - best.idx * kTcN;  // 0..63
        const float zx = __shfl_sync(0xFFFFFFFFu, jx < 32 ? z0 : z1, jx & 31);
        if (lane == 0) {
          const float L2 = ms_log(ms);
          const size_t o = (size_t)br * p.g + (k - 1);
          p.tokens[o] = kt.idx;
          p.pd_tok[o] = expf(zx - L2);
          p.lse[o] = L2;
          p.xbuf[br] = kt.idx;
        }
        if (k < p.g) {
          // the next step's A row W1[x_k] into the group's image, and
          // c_{k+1} = sigma((s_h + w_r . W1[x_k]) / T_{k+1}) while the row is at hand
          const uint4* src = reinterpret_cast<const uint4*>(W1 + (size_t)kt.idx * p.r);
          __nv_bfloat16* img = p.aimg + (size_t)g2 * kTcRows * p.r;
          float cd = 0.f;
          for (int ci = lane; ci < p.r / 8; ci += 32) {
            const int kb2 = ci >> 3, ch = ci & 7;
            const uint4 v = __ldg(src + ci);
            *reinterpret_cast<uint4*>(img + kb2 * (kTcRows * 64) + (m2 >> 3) * 512 + (m2 & 7) * 64 +
                                      ((ch ^ (m2 & 7)) << 3)) = v;
            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v);
            const float* wr = p.w + p.H + ci * 8;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __bfloat1622float2(h2[e]);
              cd = fmaf(f.x, wr[2 * e], cd);
              cd = fmaf(f.y, wr[2 * e + 1], cd);
            }
          }
          tc::fence_proxy_async_global();  // the image is read by bulk copies
          cd = warp_sum(cd);
          if (lane == 0) {
            const size_t o2 = (size_t)br * p.g + k;
            const float cf = 1.f / (1.f + expf(-(p.s_h[o2] + cd) / p.T[k]));
            if (!isfinite(cf)) raise_status(p.status, DSPARK_ENUMERIC);
            p.conf[o2] = cf;
          }
        }
      }
      grid_sync(p, leader, abort);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
namespace {

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

}  // namespace

int draft_tc_supported(const dspark_dims& d) {
  if (d.wdtype != DSPARK_BF16) return 0;
  if (d.r % 64 != 0 || d.r > 256) return 0;
  if (d.V % 8 != 0) return 0;
  if (d.B > kTcRows * kMaxGroups) return 0;
  return 1;
}

cudaError_t draft_tc_configure(dspark_ws* ws) {
  const dspark_dims& d = ws->d;
  const TcSmem L = TcSmem::make(d.r);
  const size_t smem = L.total + 1024;
  cudaError_t e = cudaFuncSetAttribute(k_draft_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_draft_tc, kTcThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  int coop = 0;
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, ws->device);
  if (!coop || !encode_fn()) return cudaErrorNotSupported;
  ws->geo.tc_groups = (d.B + kTcRows - 1) / kTcRows;
  ws->geo.tc_grid = ws->geo.num_sms;  // one CTA per SM, all co-resident
  if (ws->geo.tc_grid < ws->geo.tc_groups) return cudaErrorInvalidConfiguration;
  return cudaSuccess;
}

size_t draft_tc_scratch_rows(const dspark_dims& d, int grid) {
  const int nG = (d.B + kTcRows - 1) / kTcRows;
  const int Ggmax = (grid + nG - 1) / nG;
  const size_t a = (size_t)nG * kTcRows * Ggmax;
  const size_t b = (size_t)grid * kTcRows;
  return a > b ? a : b;
}

cudaError_t launch_draft_tc(const dspark_ws* ws, const DraftArgs& a, cudaStream_t st, int* launches) {
  const dspark_dims& d = ws->d;
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap tm_w2, tm_u;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)d.V, (cuuint64_t)d.r};
    const cuuint64_t strides[1] = {(cuuint64_t)d.V * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kTcN, (cuuint32_t)d.r};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&tm_w2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.W2), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)d.V, (cuuint64_t)d.gamma, (cuuint64_t)d.B};
    const cuuint64_t strides[2] = {(cuuint64_t)d.V * 4, (cuuint64_t)d.gamma * d.V * 4};
    const cuuint32_t box[3] = {32, 1, (cuuint32_t)kTcRows};
    const cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tm_u, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(a.U), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.B = d.B;
  p.g = d.gamma;
  p.V = d.V;
  p.r = d.r;
  p.H = d.H;
  p.ntiles = ws->geo.nblk;
  p.nG = ws->geo.tc_groups;
  p.G = ws->geo.tc_grid;
  p.Ggmax = (p.G + p.nG - 1) / p.nG;
  p.rng = Rng::make(a.seed, a.round);
  p.anchor = a.anchor;
  p.W1 = a.W1;
  p.w = a.w;
  p.T = a.T;
  p.s_h = ws->s.s_h;
  p.tokens = a.tokens;
  p.pd_tok = a.pd_tok;
  p.lse = a.lse;
  p.conf = a.conf;
  p.xbuf = ws->s.xbuf;
  p.dpart = ws->s.dpart;
  p.drec = ws->s.drec;
  p.aimg = reinterpret_cast<__nv_bfloat16*>(ws->s.aimg);
  p.bar = ws->s.barrier;
  p.status = ws->s.status;

  const TcSmem L = TcSmem::make(d.r);
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = L.total + 1024;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_draft_tc, tm_w2, tm_u, p);
  ++*launches;
  return e;
}

}  // namespace dspark
