// dspark_noalloc.cu -- the draft entry point for callers that cannot allocate.
//
// Some callers cannot call cudaMalloc: a serving engine whose device memory is
// all handed out up front by its own pool, which forbids any other
// allocation; a plug-in loaded into a host process that must not change the
// device's memory footprint once it runs; code under a hard memory budget
// where an allocation may fail in the middle of a request. For them,
// dspark_markov_draft_noalloc runs the CUDA-core draft kernels of
// dspark_markov_draft with their scratch (the hidden-state half of each
// confidence logit and the per-block log-masses of one draft step) taken from
// a fixed array compiled into this library instead of a workspace.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (4 MiB) until the process exits. Host code may not pass
// the array's name to a kernel (that name is only a host-side stand-in): the
// device address is fetched with cudaGetSymbolAddress, once per device and
// context, with that device current, by the first call made there, so make
// that first call before any stream capture begins. The address is cached
// with the context it belongs to: after the device's primary context is
// destroyed and recreated (cudaDeviceReset), the module is loaded again and
// the next call fetches the new address. All calls share the array and it
// keeps the last call's contents: two calls whose kernels overlap on the GPU
// race on it, so never issue calls on concurrent streams.
#include <cudaTypedefs.h>
#include <mutex>
#include <stdio.h>
#include <string.h>

#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace {

constexpr size_t kNoAllocFloats = (size_t)1 << 20;  // 4 MiB of fp32 scratch
constexpr int kMaxDevices = 64;

__device__ __align__(256) float g_noalloc_scratch[kNoAllocFloats];

std::mutex g_mu;
float* g_scratch_addr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

// cuCtxGetCurrent through the runtime's driver entry point (the library links
// only the runtime)
PFN_cuCtxGetCurrent_v4000 ctx_get_current_fn() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
  }
  return fn;
}

float* scratch_for_current_device(int* dev_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  *dev_out = dev;
  PFN_cuCtxGetCurrent_v4000 get_ctx = ctx_get_current_fn();
  if (!get_ctx) return nullptr;
  CUcontext ctx = nullptr;  // null while this thread has no current context yet
  if (get_ctx(&ctx) != CUDA_SUCCESS) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (ctx == nullptr || !g_scratch_addr[dev] || g_scratch_ctx[dev] != ctx) {
    // the lookup also makes the device's primary context current
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      g_scratch_addr[dev] = nullptr;
      return nullptr;
    }
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return nullptr;
    g_scratch_addr[dev] = static_cast<float*>(p);
    g_scratch_ctx[dev] = ctx;
  }
  return g_scratch_addr[dev];
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" dspark_status dspark_markov_draft_noalloc(const dspark_dims* dims, const float* U, const void* W1,
                                                     const void* W2, const int32_t* anchor, const float* h,
                                                     const float* w, const float* T, uint64_t seed,
                                                     uint64_t round, int32_t* tokens, float* pd_tok, float* lse,
                                                     float* conf, int32_t* device_status,
                                                     dspark_stream_t stream) {
  using namespace dspark;
  if (!dims) return DSPARK_EINVAL;
  const dspark_dims d = *dims;
  if (d.B < 1 || d.B > 4096 || d.gamma < 1 || d.gamma > 32 || d.V < 1 || d.V > (1 << 28) || d.r < 1 ||
      d.r > 1024 || d.H < 0 || d.H > (1 << 20) || (d.wdtype != DSPARK_F32 && d.wdtype != DSPARK_BF16))
    return DSPARK_EINVAL;
  if (!aligned16(U) || !aligned16(W1) || !aligned16(W2) || !aligned16(anchor) || !aligned16(w) ||
      !aligned16(T) || !aligned16(tokens) || !aligned16(pd_tok) || !aligned16(lse) || !aligned16(conf) ||
      !aligned16(device_status) || (d.H > 0 && !aligned16(h)))
    return DSPARK_EINVAL;
  const size_t nblk = ((size_t)d.V + kBlockW - 1) / kBlockW;
  const size_t sh_floats = ((size_t)d.B * d.gamma + 63) / 64 * 64;  // keeps the block part 256-B aligned
  const size_t need = sh_floats + (size_t)d.B * nblk;
  if (need > kNoAllocFloats) {
    fprintf(stderr,
            "dspark_markov_draft_noalloc: B*gamma + B*ceil(V/64) = %zu floats exceeds the static scratch of "
            "%zu floats\n",
            need, kNoAllocFloats);
    return DSPARK_EUNSUPPORTED;
  }
  int dev = -1;
  float* scratch = scratch_for_current_device(&dev);
  if (!scratch) return DSPARK_ECUDA;

  // A workspace view over the static scratch; nothing here allocates.
  dspark_ws view;
  memset(&view, 0, sizeof(view));
  view.d = d;
  view.device = dev;
  view.geo.nblk = (int)nblk;
  view.s.s_h = scratch;
  view.s.blk = scratch + sh_floats;
  view.s.status = device_status;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the status word must start at zero; the scratch is fully overwritten by
  // each call before it is read, so it needs no clearing
  cudaError_t e = cudaMemsetAsync(device_status, 0, sizeof(int32_t), st);
  int launches = 0;
  DraftArgs a{U, W1, W2, anchor, h, w, T, seed, round, tokens, pd_tok, lse, conf};
  if (e == cudaSuccess) e = launch_conf_hidden(&view, h, w, st, &launches);
  if (e == cudaSuccess) e = launch_draft_simt(&view, a, st, &launches);
  if (e != cudaSuccess) {
    fprintf(stderr, "dspark_markov_draft_noalloc: CUDA error %s\n", cudaGetErrorString(e));
    return DSPARK_ECUDA;
  }
  return DSPARK_OK;
}
