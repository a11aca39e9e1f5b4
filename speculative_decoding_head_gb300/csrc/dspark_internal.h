// dspark_internal.h -- workspace layout and kernel launchers shared by the
// translation units of libdspark.so (not part of the public C-ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dspark.h"

namespace dspark {

// Tunables of the launch shapes (none of them changes a result).
constexpr int kResidChunks = 32;    // CTAs per rejected request in the SIMT residual pass
constexpr int kRnnHpSlices = 10;    // K slices of the RNN head's h projection (partial products the cell adds)

struct DraftArgs {
  const float* U;
  const void* W1;
  const void* W2;
  const int32_t* anchor;
  const float* h;
  const float* w;
  const float* T;
  uint64_t seed, round;
  int32_t* tokens;
  float* pd_tok;
  float* lse;
  float* conf;
};

struct VerifyArgs {
  const float* P;
  const int32_t* row_off;
  const int32_t* lengths;
  const int32_t* anchor;
  const int32_t* tokens;
  const float* pd_tok;
  const float* lse;
  const float* U;
  const void* W1;
  const void* W2;
  uint64_t seed, round;
  int32_t* n_acc;
  int32_t* next_anchor;
  const float* ovec;  // [B][gamma][r] the RNN head's o_k (p_d from U + o W2), or null (Markov head)
  const int4* rowtab;  // [rows] (b, j, lengths[b], row_off[b]) per packed row, written by this
                       // round's planner (dspark_round), or null: the sweep looks the rows up
};

// The draft head's teacher-forced training objective: inputs, outputs and the
// caller's scratch (column i = b * gamma + k, G = ws->geo.num_sms partials).
struct LossArgs {
  const float* U;
  const void* W1;
  const void* W2;
  const int32_t* anchor;
  const int32_t* xstar;
  const float* P;
  const float* conf;
  double tau;
  float* ce;
  float* l1;
  float* bce;
  double* loss;
  float4* lpart;   // [B*gamma][G] (max, sum exp) of z_d and of z_t per CTA
  float* l1part;   // [B*gamma][G] sum |p_d - p_t| per CTA
  float* zx;       // [B*gamma] z_d at x*
  float* lse_d;    // [B*gamma]
  float* lse_t;    // [B*gamma]
  double* term;    // [B*gamma] w_k (0.1 ce + 0.9 l1 + bce)
};

// Device scratch carved out of one arena by dspark_ws_create.
struct Scratch {
  int* status;            // [1] first device error, 0 = none
  float* s_h;             // [B*gamma] hidden half of the confidence logit
  float* blk;             // [B*nblk] block log-masses of one draft step (SIMT path)
  int32_t* kring;         // [lag+1] capacities of the lagged planner, by round mod (lag+1)
  uint32_t* plan_round;   // [1] rounds planned since the last reset
  float4* vpart;          // [sweep_grid*SL] verify-sweep partials (m, s, key, block)
  int* vflag;             // [B] 1 = next anchor comes from the residual
  int* vrow;              // [B] packed row of the first rejection
  float* vlset;           // [B] target log-sum-exp of that row
  int* vdone;             // [B] sweep ranges done per request (back to 0 by the finalizing CTA)
  float* vpx;             // [B*(gamma+1)] P at each verified row's draft token (bulk sweep)
  int4* rowtab;           // [B*(gamma+1)] (b, j, lengths[b], row_off[b]) per packed row (dspark_round)
  int* vsched;            // [1] the dynamic sweep's chunk counter (cleared by its finalize kernel)
  float* vlse;            // [B*(gamma+1)*nblk] block log-sum-exps of the packed rows (dynamic sweep)
  float2* rpart;          // [B*kResidChunks] residual (key, block) per CTA
  // persistent tcgen05 draft kernel
  float2* dpart;          // [gamma][groups*128][sets*ceil(grid/groups)] per-CTA, per-epilogue-set
                          // (max, sum exp) of a row's blocks
  unsigned long long* dwin;  // [2][gamma][groups*128] lines of 16 words: word 0 the packed (block key,
                             // block) winner, word 1 the token drawn in it; the two halves alternate
                             // between launches
  float* hpart;           // [B*gamma][ceil(H/1024)] partial sums of w_h . h_k over 1024-float chunks
  unsigned* barrier;      // [8] draft kernel words: [2] launch count, [4 + launch parity] barrier arrivals
};

struct Geometry {
  int nblk;        // ceil(V / 64)
  int sweep_grid;  // CTAs of the verify sweep
  int sweep_bulk;  // bulk-copy sweep (V % 64 == 0)
  int sweep_dyn;   // the bulk sweep with chunks taken from a counter (at least 128 blocks a row)
  int SL;          // sweep partial slots per CTA (rows one range can touch)
  int num_sms;
  // persistent draft kernel
  int tc_ok;        // tcgen05 path usable for these dims
  int tc_grid;      // CTAs of the persistent draft kernel
  int tc_groups;    // 128-row groups
  int resid_tc_ok;  // tcgen05 residual kernel usable for these dims
  int rchunks;      // residual partials per request (CTAs of the residual pass)
};

}  // namespace dspark

struct dspark_ws {
  dspark_dims d;
  int device;
  void* arena;
  size_t arena_bytes;
  dspark::Scratch s;
  dspark::Geometry geo;
  int use_tc;  // tensor-core draft and residual where geo.tc_ok / geo.resid_tc_ok hold
  int last_launches;
  int pdl;     // set by dspark_round: the plan and verify kernels wait on the previous kernel in-kernel
  int b0;      // batch index of request 0 (dspark_ws_set_shard): the request word of every random draw
};

namespace dspark {

// Launch with programmatic stream serialization when `pdl` is set (the kernel
// must call pdl_wait() before it reads what earlier kernels write).
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                      Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Launchers: return cudaGetLastError() of their launches; add their launch
// count to *launches.
cudaError_t launch_conf_hidden(const dspark_ws* ws, const float* h, const float* w, cudaStream_t st,
                               int* launches);
cudaError_t launch_draft_simt(const dspark_ws* ws, const DraftArgs& a, cudaStream_t st, int* launches);
cudaError_t launch_draft_tc(const dspark_ws* ws, const DraftArgs& a, cudaStream_t st, int* launches);
// The RNN head (eq. (6)): Hp[row][3r] = the h_k part of W_g, W_c, W_o z_k for
// every position; the cell of step k (S [B][r] the state, updated in place;
// ovec [B*gamma][r] receives o_k); the whole draft tail on the SIMT path.
cudaError_t launch_rnn_hproj(const dspark_ws* ws, const float* h, const void* Wr, float* Hp, cudaStream_t st,
                             int* launches);
// oimg: o_k's bf16 hi and lo images in the row pass's operand layout (null: not written)
cudaError_t launch_rnn_cell(const dspark_ws* ws, const DraftArgs& a, const void* Wr, const float* Hp, float* S,
                            float* ovec, __nv_bfloat16* oimg, int k, cudaStream_t st, int* launches);
// hl: scratch for h split into bf16 hi | lo (rnn_hsplit_bytes), or null: the
// h projection then runs on CUDA cores; oimg: scratch of oimg_len bytes for
// o_k's images, which the cell writes when the row pass runs the block pass
cudaError_t launch_rnn_draft(const dspark_ws* ws, const DraftArgs& a, const void* Wr, float* Hp, float* S,
                             float* ovec, void* hl, __nv_bfloat16* oimg, size_t oimg_len, cudaStream_t st,
                             int* launches);
// The h projection on tcgen05 (k_rnn_tc.cu): shapes it takes (bf16 weights,
// H % 64 == 0, r % 64 == 0, r <= 256), whether this workspace runs it, the
// bytes of its hi | lo copy of h, and its launch (same Hp layout as
// launch_rnn_hproj).
bool rnn_hproj_tc_shape(const dspark_dims& d);
bool rnn_hproj_tc_supported(const dspark_ws* ws);
size_t rnn_hsplit_bytes(const dspark_dims& d);
cudaError_t launch_rnn_hproj_tc(const dspark_ws* ws, const float* h, const void* Wr, float* Hp, void* hl_scratch,
                                cudaStream_t st, int* launches);
// rowtab (may be null): also write each packed row's (b, j, lengths[b], row_off[b])
cudaError_t launch_plan(const dspark_ws* ws, const float* conf, const double* sps, int32_t* lengths,
                        int32_t* row_off, int4* rowtab, cudaStream_t st, int* launches);
cudaError_t launch_verify(const dspark_ws* ws, const VerifyArgs& a, cudaStream_t st, int* launches);

// Whether the tcgen05 draft kernel supports these dims, and its launch shape.
int draft_tc_supported(const dspark_dims& d);
cudaError_t draft_tc_configure(dspark_ws* ws);
size_t draft_tc_partials(const dspark_dims& d, int grid);  // float2 entries of Scratch::dpart
size_t draft_tc_winners(const dspark_dims& d);             // entries of Scratch::dwin
size_t draft_tc_hidden_partials(const dspark_dims& d);     // floats of Scratch::hpart

int resid_tc_supported(const dspark_dims& d);
cudaError_t resid_tc_configure(dspark_ws* ws);
cudaError_t launch_resid_tc(const dspark_ws* ws, const VerifyArgs& a, float2* rpart, int grid, cudaStream_t st,
                            bool pdl);
// pass 0: per-CTA (max, sum exp) of z_d and z_t and z_d at x*; pass 1: per-CTA
// sum |p_d - p_t| (needs lse_d, lse_t). Grid = ws->geo.num_sms.
cudaError_t launch_loss_tc(const dspark_ws* ws, const LossArgs& a, int pass, cudaStream_t st);
// The same two passes with the positions as MMA rows (k_rowpass.cu), where
// rowpass_supported: the same partial layout ([n][num_sms], neutral values in
// the slots no CTA fills).
// n: the rows (positions for the loss, requests for the RNN and PCTree passes).
bool rowpass_supported(const dspark_ws* ws, int n);
cudaError_t launch_loss_rowpass(const dspark_ws* ws, const LossArgs& a, int pass, cudaStream_t st);
// One RNN draft step's block log-masses into Scratch::blk (as launch_rnn_blocks_tc),
// and one PCTree expansion's block log-masses and maxima (as launch_tree_blocks_tc).
cudaError_t launch_rnn_blocks_rowpass(const dspark_ws* ws, const float* U, const void* W2, const float* ovec,
                                      const __nv_bfloat16* oimg, int k, cudaStream_t st);
cudaError_t launch_tree_blocks_rowpass(const dspark_ws* ws, const float* U, const void* W1, const void* W2,
                                       const int32_t* tok, const int32_t* dep, const int4* state, int N, float* blk,
                                       float* bmax, cudaStream_t st);
// One draft step of the RNN head on tcgen05: Scratch::blk = the block
// log-masses of z = U_k + o_k W2 (o_k from ovec, split into bf16 hi + lo).
cudaError_t launch_rnn_blocks_tc(const dspark_ws* ws, const float* U, const void* W2, const float* ovec, int k,
                                 cudaStream_t st);

// PCTree (k_pctree.cu): the best-first draft tree of N nodes with c children
// per expansion, and its lossless verify.
constexpr int kTreeMaxChildren = 8;
constexpr int kTreeMaxNodes = 64;
size_t tree_scratch_bytes(const dspark_dims& d, int nblk, int c, int N);
size_t tree_verify_smem_bytes(int nblk);
cudaError_t launch_pctree_build(const dspark_ws* ws, const float* U, const void* W1, const void* W2,
                                const int32_t* anchor, int c, int N, int32_t* tok, int32_t* par, int32_t* dep,
                                float* lp, int32_t* n_nodes, void* scratch, cudaStream_t st, int* launches);
cudaError_t launch_pctree_verify(const dspark_ws* ws, const float* P, const int32_t* tok, const int32_t* par, int N,
                                 uint64_t seed, uint64_t round, int32_t* path, int32_t* n_acc, int32_t* next_anchor,
                                 cudaStream_t st, int* launches);
cudaError_t launch_tree_blocks_tc(const dspark_ws* ws, const float* U, const void* W1, const void* W2,
                                  const int32_t* tok, const int32_t* dep, const int4* state, int N, float* blk,
                                  float* bmax, cudaStream_t st);

size_t plan_smem_bytes(const dspark_dims& d);
// lengths_l[i] = lengths[b_begin + i] and row_off_l[i] = row_off[b_begin + i] - row_off[b_begin]
// (i <= n for row_off_l): one device's share of a plan made for the whole batch.
cudaError_t launch_plan_slice(const int32_t* lengths, const int32_t* row_off, int b_begin, int n, int32_t* lengths_l,
                              int32_t* row_off_l, cudaStream_t st, int* launches);
cudaError_t sweep_bulk_configure();
int sweep_bulk_max_slots();  // rows one CTA range of the bulk sweep may span
size_t sweep_bulk_smem_bytes(int SL);
// The dynamic sweep: rows of at least sweep_dyn_min_blocks() blocks, the
// partial count for a number of units (two float2, one float4, per group of 32), its configuration.
int sweep_dyn_min_blocks();
size_t sweep_dyn_parts(long long units);
cudaError_t sweep_dyn_configure();
cudaError_t plan_configure();

}  // namespace dspark
