// dspark_api.cu -- the C-ABI of libdspark.so: argument checks, the workspace
// arena and the order of the launches of one round. Every arithmetic step of
// the round runs in the kernels of the other translation units.
#include <stdio.h>
#include <string.h>

#include <algorithm>

#include "dspark_common.cuh"
#include "dspark_internal.h"

using namespace dspark;

namespace {

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

dspark_status check_dims(const dspark_dims& d) {
  if (d.B < 1 || d.B > 4096 || d.gamma < 1 || d.gamma > 32 || d.V < 1 || d.V > (1 << 28) || d.r < 1 ||
      d.r > 1024 || d.H < 0 || d.H > (1 << 20))
    return DSPARK_EINVAL;
  if (d.wdtype != DSPARK_F32 && d.wdtype != DSPARK_BF16) return DSPARK_EINVAL;
  if (d.mode != DSPARK_STATIC && d.mode != DSPARK_COMPACT && d.mode != DSPARK_COMPACT_LAGGED)
    return DSPARK_EINVAL;
  if (d.mode == DSPARK_COMPACT_LAGGED && (d.lag < 1 || d.lag > 8)) return DSPARK_EINVAL;
  if (d.wdtype == DSPARK_BF16 && (d.V % 8) != 0) return DSPARK_EINVAL;
  if (d.mode != DSPARK_STATIC && d.B * d.gamma > 8192) return DSPARK_EUNSUPPORTED;
  if ((size_t)d.B * (d.gamma + 1) * (size_t)d.V >= ((size_t)1 << 40)) return DSPARK_EUNSUPPORTED;
  return DSPARK_OK;
}

dspark_status cuda_fail(cudaError_t e) {
  if (e == cudaSuccess) return DSPARK_OK;
  fprintf(stderr, "dspark: CUDA error %s\n", cudaGetErrorString(e));
  return DSPARK_ECUDA;
}

}  // namespace

extern "C" {

const char* dspark_status_string(int status) {
  switch (status) {
    case DSPARK_OK: return "ok";
    case DSPARK_EINVAL: return "invalid argument";
    case DSPARK_ECUDA: return "CUDA runtime error";
    case DSPARK_ETIMEOUT: return "grid barrier timed out";
    case DSPARK_ENUMERIC: return "non-finite or non-positive confidence or SPS entry";
    case DSPARK_EUNSUPPORTED: return "unsupported shape or mode";
    case DSPARK_ERANGE: return "token id or length out of range";
    default: return "unknown status";
  }
}

dspark_status dspark_ws_create(const dspark_dims* dims, dspark_ws** out) {
  if (!dims || !out) return DSPARK_EINVAL;
  *out = nullptr;
  const dspark_dims d = *dims;
  dspark_status st = check_dims(d);
  if (st != DSPARK_OK) return st;

  dspark_ws* ws = new dspark_ws();
  memset(ws, 0, sizeof(*ws));
  ws->d = d;
  if (cudaGetDevice(&ws->device) != cudaSuccess) {
    delete ws;
    return DSPARK_ECUDA;
  }
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, ws->device);
  Geometry& geo = ws->geo;
  geo.num_sms = sms > 0 ? sms : 1;
  geo.nblk = (d.V + kBlockW - 1) / kBlockW;
  geo.sweep_bulk = (d.V % kBlockW) == 0 && sweep_bulk_configure() == cudaSuccess;
  cudaGetLastError();
  // The bulk sweep keeps per-thread partials of every row its range touches
  // (a range of ceil(R nblk / grid) blocks touches at most ceil(R / grid) + 1
  // rows). Two CTAs per SM (a 96 KB ring each) while that is at most 8 rows;
  // else one CTA per SM with up to 32 rows; beyond, the register sweep.
  const int Rmax = d.B * (d.gamma + 1);
  // no more CTAs than ranges of 32 blocks of the row capacity (a small round
  // would leave most CTAs idle, and every working CTA counts itself in for
  // each request it touches), nor so few that a range spans more than 6 rows
  const long long units_max = (long long)Rmax * geo.nblk;
  auto capped = [&](int grid) {
    return (int)std::min<long long>(grid, std::max<long long>((units_max + 31) / 32, (Rmax + 5) / 6));
  };
  if (geo.sweep_bulk && (Rmax + 2 * geo.num_sms - 1) / (2 * geo.num_sms) + 2 <= 8) {
    geo.sweep_grid = capped(2 * geo.num_sms);
  } else if (geo.sweep_bulk && (Rmax + geo.num_sms - 1) / geo.num_sms + 2 <= sweep_bulk_max_slots()) {
    geo.sweep_grid = capped(geo.num_sms);
  } else {
    geo.sweep_bulk = 0;
    geo.sweep_grid = 4 * geo.num_sms;
  }
  geo.SL = (Rmax + geo.sweep_grid - 1) / geo.sweep_grid + 2;
  geo.sweep_dyn = (d.V % kBlockW) == 0 && geo.nblk >= sweep_dyn_min_blocks() && sweep_dyn_configure() == cudaSuccess;
  cudaGetLastError();
  geo.tc_ok = draft_tc_supported(d);

  const size_t BG = (size_t)d.B * d.gamma;
  size_t off = 0;
  auto carve = [&](size_t bytes) {
    const size_t o = off;
    off += round_up(bytes > 0 ? bytes : 1, 256);
    return o;
  };
  const size_t o_status = carve(sizeof(int));
  const size_t o_round = carve(sizeof(uint32_t));
  const size_t o_bar = carve(8 * sizeof(unsigned));
  const size_t o_sh = carve(sizeof(float) * BG);
  const size_t o_blk = carve(sizeof(float) * (size_t)d.B * geo.nblk);
  const size_t o_ring = carve(d.mode == DSPARK_COMPACT_LAGGED ? sizeof(int32_t) * (d.lag + 1) : 0);
  const size_t vparts = geo.sweep_dyn ? sweep_dyn_parts((long long)Rmax * geo.nblk) : 0;
  const size_t o_vpart = carve(sizeof(float4) * std::max((size_t)geo.sweep_grid * geo.SL, vparts));
  const size_t o_vsched = carve(sizeof(int));
  const size_t o_vlse = carve(geo.sweep_dyn ? sizeof(float) * (size_t)Rmax * geo.nblk : 0);
  const size_t o_vflag = carve(sizeof(int) * d.B);
  const size_t o_vrow = carve(sizeof(int) * d.B);
  const size_t o_vlset = carve(sizeof(float) * d.B);
  const size_t o_vdone = carve(sizeof(int) * d.B);
  const size_t o_vpx = carve(sizeof(float) * (size_t)d.B * (d.gamma + 1));
  const size_t o_rowtab = carve(sizeof(int4) * (size_t)d.B * (d.gamma + 1));
  geo.resid_tc_ok = resid_tc_supported(d);
  if (geo.resid_tc_ok && resid_tc_configure(ws) != cudaSuccess) geo.resid_tc_ok = 0;
  cudaGetLastError();
  geo.rchunks = geo.num_sms > kResidChunks ? geo.num_sms : kResidChunks;
  const size_t o_rpart = carve(sizeof(float2) * (size_t)d.B * geo.rchunks);
  size_t o_dpart = 0, o_dwin = 0, o_hpart = 0;
  if (geo.tc_ok) {
    if (draft_tc_configure(ws) != cudaSuccess) geo.tc_ok = 0;
  }
  if (geo.tc_ok) {
    o_dpart = carve(sizeof(float2) * draft_tc_partials(d, geo.tc_grid));
    o_dwin = carve(sizeof(unsigned long long) * draft_tc_winners(d));
    o_hpart = carve(sizeof(float) * draft_tc_hidden_partials(d));
  }
  if (plan_configure() != cudaSuccess) {
    delete ws;
    return DSPARK_ECUDA;
  }
  cudaGetLastError();
  ws->arena_bytes = off;
  if (cudaMalloc(&ws->arena, off) != cudaSuccess) {
    cudaGetLastError();
    delete ws;
    return DSPARK_ECUDA;
  }
  char* base = static_cast<char*>(ws->arena);
  Scratch& s = ws->s;
  s.status = reinterpret_cast<int*>(base + o_status);
  s.plan_round = reinterpret_cast<uint32_t*>(base + o_round);
  s.barrier = reinterpret_cast<unsigned*>(base + o_bar);
  s.s_h = reinterpret_cast<float*>(base + o_sh);
  s.blk = reinterpret_cast<float*>(base + o_blk);
  s.kring = reinterpret_cast<int32_t*>(base + o_ring);
  s.vpart = reinterpret_cast<float4*>(base + o_vpart);
  s.vflag = reinterpret_cast<int*>(base + o_vflag);
  s.vrow = reinterpret_cast<int*>(base + o_vrow);
  s.vlset = reinterpret_cast<float*>(base + o_vlset);
  s.vdone = reinterpret_cast<int*>(base + o_vdone);
  s.vpx = reinterpret_cast<float*>(base + o_vpx);
  s.rowtab = reinterpret_cast<int4*>(base + o_rowtab);
  s.vsched = reinterpret_cast<int*>(base + o_vsched);
  s.vlse = geo.sweep_dyn ? reinterpret_cast<float*>(base + o_vlse) : nullptr;
  s.rpart = reinterpret_cast<float2*>(base + o_rpart);
  s.dpart = geo.tc_ok ? reinterpret_cast<float2*>(base + o_dpart) : nullptr;
  s.dwin = geo.tc_ok ? reinterpret_cast<unsigned long long*>(base + o_dwin) : nullptr;
  s.hpart = geo.tc_ok ? reinterpret_cast<float*>(base + o_hpart) : nullptr;
  ws->use_tc = geo.tc_ok;
  if (cudaMemset(ws->arena, 0, off) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    cudaFree(ws->arena);
    delete ws;
    return DSPARK_ECUDA;
  }
  *out = ws;
  return DSPARK_OK;
}

void dspark_ws_destroy(dspark_ws* ws) {
  if (!ws) return;
  cudaDeviceSynchronize();
  cudaFree(ws->arena);
  delete ws;
}

dspark_status dspark_ws_reset(dspark_ws* ws, dspark_stream_t stream) {
  if (!ws) return DSPARK_EINVAL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws->s.status, 0, sizeof(int), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws->s.plan_round, 0, sizeof(uint32_t), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws->s.barrier, 0, 8 * sizeof(unsigned), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws->s.vdone, 0, sizeof(int) * ws->d.B, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws->s.vsched, 0, sizeof(int), st);
  if (e == cudaSuccess && ws->s.dwin)
    e = cudaMemsetAsync(ws->s.dwin, 0, sizeof(unsigned long long) * draft_tc_winners(ws->d), st);
  return cuda_fail(e);
}

dspark_status dspark_last_error(dspark_ws* ws, int* device_status) {
  if (!ws || !device_status) return DSPARK_EINVAL;
  return cuda_fail(cudaMemcpy(device_status, ws->s.status, sizeof(int), cudaMemcpyDeviceToHost));
}

int dspark_last_launch_count(dspark_ws* ws) { return ws ? ws->last_launches : -1; }

const char* dspark_path(dspark_ws* ws) {
  if (!ws) return "none";
  return ws->use_tc ? "tcgen05" : "simt";
}

dspark_status dspark_ws_set_path(dspark_ws* ws, const char* path) {
  if (!ws || !path) return DSPARK_EINVAL;
  if (strcmp(path, "simt") == 0) {
    ws->use_tc = 0;
    return DSPARK_OK;
  }
  if (strcmp(path, "tcgen05") == 0) {
    if (!ws->geo.tc_ok) return DSPARK_EUNSUPPORTED;
    ws->use_tc = 1;
    return DSPARK_OK;
  }
  return DSPARK_EINVAL;
}

dspark_status dspark_markov_draft(dspark_ws* ws, const float* U, const void* W1, const void* W2,
                                  const int32_t* anchor, const float* h, const float* w, const float* T,
                                  uint64_t seed, uint64_t round, int32_t* tokens, float* pd_tok, float* lse,
                                  float* conf, dspark_stream_t stream) {
  if (!ws) return DSPARK_EINVAL;
  const dspark_dims& d = ws->d;
  if (!aligned16(U) || !aligned16(W1) || !aligned16(W2) || !aligned16(anchor) || !aligned16(w) ||
      !aligned16(T) || !aligned16(tokens) || !aligned16(pd_tok) || !aligned16(lse) || !aligned16(conf))
    return DSPARK_EINVAL;
  if (d.H > 0 && !aligned16(h)) return DSPARK_EINVAL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int launches = 0;
  DraftArgs a{U, W1, W2, anchor, h, w, T, seed, round, tokens, pd_tok, lse, conf};
  cudaError_t e;
  if (ws->use_tc && ws->geo.tc_ok) {
    e = launch_draft_tc(ws, a, st, &launches);  // one launch; it forms c_k from h itself
  } else {
    e = launch_conf_hidden(ws, h, w, st, &launches);
    if (e == cudaSuccess) e = launch_draft_simt(ws, a, st, &launches);
  }
  ws->last_launches = launches;
  return cuda_fail(e);
}

namespace {

dspark_status plan_call(dspark_ws* ws, const float* conf, const double* sps, int32_t* lengths, int32_t* row_off,
                        int4* rowtab, dspark_stream_t stream) {
  if (!ws) return DSPARK_EINVAL;
  if (!aligned16(lengths) || !aligned16(row_off)) return DSPARK_EINVAL;
  if (ws->d.mode != DSPARK_STATIC && (!aligned16(conf) || !aligned16(sps))) return DSPARK_EINVAL;
  int launches = 0;
  cudaError_t e =
      launch_plan(ws, conf, sps, lengths, row_off, rowtab, reinterpret_cast<cudaStream_t>(stream), &launches);
  ws->last_launches = launches;
  return cuda_fail(e);
}

dspark_status verify_call(dspark_ws* ws, const float* P, const int32_t* row_off, const int32_t* lengths,
                          const int32_t* anchor, const int32_t* tokens, const float* pd_tok, const float* lse,
                          const float* U, const void* W1, const void* W2, uint64_t seed, uint64_t round,
                          int32_t* n_accepted, int32_t* next_anchor, const int4* rowtab, dspark_stream_t stream) {
  if (!ws) return DSPARK_EINVAL;
  if (!aligned16(P) || !aligned16(row_off) || !aligned16(lengths) || !aligned16(anchor) || !aligned16(tokens) ||
      !aligned16(pd_tok) || !aligned16(lse) || !aligned16(U) || !aligned16(W1) || !aligned16(W2) ||
      !aligned16(n_accepted) || !aligned16(next_anchor))
    return DSPARK_EINVAL;
  VerifyArgs a{P, row_off, lengths, anchor, tokens, pd_tok, lse, U, W1, W2, seed, round, n_accepted, next_anchor,
               nullptr, rowtab};
  int launches = 0;
  cudaError_t e = launch_verify(ws, a, reinterpret_cast<cudaStream_t>(stream), &launches);
  ws->last_launches = launches;
  return cuda_fail(e);
}

}  // namespace

dspark_status dspark_plan(dspark_ws* ws, const float* conf, const double* sps, int32_t* lengths,
                          int32_t* row_off, dspark_stream_t stream) {
  return plan_call(ws, conf, sps, lengths, row_off, nullptr, stream);
}

dspark_status dspark_ws_set_shard(dspark_ws* ws, int b_offset) {
  if (!ws || b_offset < 0 || (long long)b_offset + ws->d.B > 0x7FFFFFFFLL) return DSPARK_EINVAL;
  ws->b0 = b_offset;
  return DSPARK_OK;
}

dspark_status dspark_plan_shard(dspark_ws* ws, const float* conf, const double* sps, int b_begin, int b_count,
                                int32_t* lengths, int32_t* row_off, int32_t* lengths_local, int32_t* row_off_local,
                                dspark_stream_t stream) {
  if (!ws || b_begin < 0 || b_count < 1 || b_count > ws->d.B - b_begin) return DSPARK_EINVAL;
  if (!aligned16(lengths_local) || !aligned16(row_off_local)) return DSPARK_EINVAL;
  const dspark_status s = plan_call(ws, conf, sps, lengths, row_off, nullptr, stream);
  if (s != DSPARK_OK) return s;
  int launches = ws->last_launches;
  cudaError_t e = launch_plan_slice(lengths, row_off, b_begin, b_count, lengths_local, row_off_local,
                                    reinterpret_cast<cudaStream_t>(stream), &launches);
  ws->last_launches = launches;
  return cuda_fail(e);
}

dspark_status dspark_verify(dspark_ws* ws, const float* P, const int32_t* row_off, const int32_t* lengths,
                            const int32_t* anchor, const int32_t* tokens, const float* pd_tok, const float* lse,
                            const float* U, const void* W1, const void* W2, uint64_t seed, uint64_t round,
                            int32_t* n_accepted, int32_t* next_anchor, dspark_stream_t stream) {
  return verify_call(ws, P, row_off, lengths, anchor, tokens, pd_tok, lse, U, W1, W2, seed, round, n_accepted,
                     next_anchor, nullptr, stream);
}

dspark_status dspark_verify_rnn(dspark_ws* ws, const float* P, const int32_t* row_off, const int32_t* lengths,
                                const int32_t* anchor, const int32_t* tokens, const float* pd_tok, const float* lse,
                                const float* U, const float* ovec, const void* W2, uint64_t seed, uint64_t round,
                                int32_t* n_accepted, int32_t* next_anchor, dspark_stream_t stream) {
  if (!ws) return DSPARK_EINVAL;
  if (!aligned16(P) || !aligned16(row_off) || !aligned16(lengths) || !aligned16(anchor) || !aligned16(tokens) ||
      !aligned16(pd_tok) || !aligned16(lse) || !aligned16(U) || !aligned16(ovec) || !aligned16(W2) ||
      !aligned16(n_accepted) || !aligned16(next_anchor))
    return DSPARK_EINVAL;
  VerifyArgs a{P, row_off, lengths, anchor, tokens, pd_tok, lse, U, nullptr, W2, seed, round, n_accepted,
               next_anchor, ovec, nullptr};
  int launches = 0;
  cudaError_t e = launch_verify(ws, a, reinterpret_cast<cudaStream_t>(stream), &launches);
  ws->last_launches = launches;
  return cuda_fail(e);
}

dspark_status dspark_round(dspark_ws* ws, const float* U, const void* W1, const void* W2, const int32_t* anchor,
                           const float* h, const float* w, const float* T, const double* sps, const float* P,
                           uint64_t seed, uint64_t round, int32_t* tokens, float* pd_tok, float* lse, float* conf,
                           int32_t* lengths, int32_t* row_off, int32_t* n_accepted, int32_t* next_anchor,
                           dspark_stream_t stream) {
  dspark_status s =
      dspark_markov_draft(ws, U, W1, W2, anchor, h, w, T, seed, round, tokens, pd_tok, lse, conf, stream);
  if (s != DSPARK_OK) return s;
  const int l1 = ws->last_launches;
  // within the round each kernel after the draft may start while the one
  // before it drains: every input it reads before its in-kernel wait was
  // written before the draft began
  ws->pdl = 1;
  // the planner also writes each packed row's request and position, so the
  // sweep reads them instead of searching the offsets
  s = plan_call(ws, conf, sps, lengths, row_off, ws->s.rowtab, stream);
  const int l2 = ws->last_launches;
  if (s == DSPARK_OK)
    s = verify_call(ws, P, row_off, lengths, anchor, tokens, pd_tok, lse, U, W1, W2, seed, round, n_accepted,
                    next_anchor, ws->s.rowtab, stream);
  ws->pdl = 0;
  ws->last_launches += l1 + l2;
  return s;
}

}  // extern "C"
