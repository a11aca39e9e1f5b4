/*
 * dspark.h -- C-ABI of the GB300 DSpark round library (libdspark.so).
 *
 * One DSpark round over a batch of B requests, in three calls:
 *
 *   dspark_markov_draft  Markov-head draft tail + confidence head.
 *       "DeepSeek-V4.1 模型结构（6）：解码，DSpark", eq. (4) and (5):
 *       p_k(v) = softmax_v(U_k(v) + W1[x_{k-1}] . W2[:, v]), x_0 = anchor,
 *       sampled left to right for k = 1..gamma (section "Markov head", the
 *       sequential loop); eq. (7) with the STS temperature of the
 *       zdszero.github.io "spec_dspark" page (section "在 SGLang 里",
 *       sigmoid(raw / T)): c_k = sigma((w^T [h_k; W1[x_{k-1}]]) / T_k).
 *   dspark_plan          confidence-scheduled planner.
 *       Same blog, sections "目标函数" and "贪心就能解"; deepseek.csdn.net
 *       close reading §5.3 (Algorithm 1): survival a_{b,j} = prod_{i<=j} c_{b,i};
 *       candidates are admitted in decreasing a while Theta = tau * SPS(B_tot)
 *       rises. COMPACT_LAGGED is the asynchronous planner of the same
 *       close reading §8: capacity K = argmax Theta over the full path on the
 *       confidences of round t - lag, then the top-K current candidates.
 *       lengths[b] in [1, gamma+1] counts the anchor ("spec_dspark", SGLang
 *       section: the anchor is always verified).
 *   dspark_verify        lossless ragged rejection-sampling verify.
 *       Same blog, section "投机解码" and the derivation box;
 *       "DSpark：不让大模型更聪明，而让它「吐字更快」" §02: accept x_{j+1} with
 *       probability min(1, p_t(x_{j+1}) / p_d(x_{j+1})); at the first rejection
 *       draw from norm(max(0, p_t - p_d)); if every verified draft passes, draw
 *       the bonus token from the last verified target row.
 *
 * Conventions
 *   - Every data pointer is a DEVICE pointer owned by the caller. The library
 *     reads inputs and writes outputs during the call's stream work and keeps
 *     no pointer past it. Inputs are const and must not alias outputs.
 *   - Layouts are dense row-major: U [B, gamma, V] fp32; W1 [V, r] and
 *     W2 [r, V] in the workspace's weight dtype (fp32 or bf16); h [B, gamma, H]
 *     fp32; w [H + r] fp32 (hidden part first); T [gamma] fp32; per-position
 *     outputs [B, gamma] with column k-1 for draft position k; P packed
 *     [row_off[B], V] fp32 where rows row_off[b] + j, j < lengths[b], are the
 *     target logits for the token after x_j (x_0 = anchor).
 *   - Base pointers must be 16-byte aligned; V % 8 == 0 for bf16 weights.
 *   - Every call is asynchronous on `stream` (NULL = the legacy default
 *     stream) and returns at once. Host-detectable errors (null pointer,
 *     misalignment, bad dims) return a status and enqueue nothing.
 *     Device-detected errors (non-finite confidence or SPS entry, token id out
 *     of range, a grid-barrier timeout) set the workspace status word, the
 *     kernels stop early and the outputs of that round are undefined; read it
 *     with dspark_last_error after synchronising the stream.
 *   - Random numbers come from Philox4x32-10 (Salmon et al., SC'11) with key
 *     = seed and counter = (v >> 2, b, j, purpose << 24 | round mod 2^24);
 *     the same (seed, round, inputs) always give the same outputs, whatever
 *     the GPU's SM count.
 *   - The workspace holds per-round scratch and the planner's confidence
 *     ring; calls that share a workspace must be ordered on one stream.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so that callers need no CUDA header. */
typedef struct CUstream_st* dspark_stream_t;

typedef enum {
    DSPARK_OK = 0,
    DSPARK_EINVAL = 1,        /* bad argument: null, misaligned, bad dims */
    DSPARK_ECUDA = 2,         /* a CUDA runtime call failed */
    DSPARK_ETIMEOUT = 3,      /* a grid barrier did not complete in time (device) */
    DSPARK_ENUMERIC = 4,      /* non-finite or non-positive confidence/SPS (device) */
    DSPARK_EUNSUPPORTED = 5,  /* valid but unsupported shape or mode */
    DSPARK_ERANGE = 6         /* token id or length out of range (device) */
} dspark_status;

typedef enum { DSPARK_F32 = 0, DSPARK_BF16 = 1 } dspark_wdtype;

typedef enum {
    DSPARK_STATIC = 0,          /* no planner: every request verifies gamma + 1 rows */
    DSPARK_COMPACT = 1,         /* Algorithm 1 with early stop */
    DSPARK_COMPACT_LAGGED = 2   /* capacity from confidences `lag` rounds old, top-K now */
} dspark_mode;

typedef struct {
    int B;                  /* requests, 1 .. 4096 */
    int gamma;              /* draft positions, 1 .. 32 */
    int V;                  /* vocabulary size */
    int r;                  /* Markov rank, 1 .. 1024 */
    int H;                  /* confidence-head hidden size, >= 0 */
    dspark_wdtype wdtype;   /* storage type of W1 and W2 */
    dspark_mode mode;
    int lag;                /* lag depth for DSPARK_COMPACT_LAGGED, 1 .. 8 */
} dspark_dims;

typedef struct dspark_ws dspark_ws;

/* Create a workspace for `dims` on the current CUDA device. This is the only
 * call that allocates device memory (one arena: scratch, barrier words, the
 * confidence ring, the status word). Returns EINVAL/EUNSUPPORTED/ECUDA. */
dspark_status dspark_ws_create(const dspark_dims* dims, dspark_ws** out);

/* Free the workspace (synchronises the device first). NULL is a no-op. */
void dspark_ws_destroy(dspark_ws* ws);

/* Clear the device status word, the lagged planner's round counter, the
 * draft kernel's grid-barrier words and winner slots, and the verify sweeps'
 * counters (per-request completion counts, the chunk counter), on `stream`.
 * Call it after any call that left a non-zero device status. */
dspark_status dspark_ws_reset(dspark_ws* ws, dspark_stream_t stream);

/* Copy the device status word into *device_status (a synchronous 4-byte copy;
 * synchronise the work's stream first). Returns the host status of the copy. */
dspark_status dspark_last_error(dspark_ws* ws, int* device_status);

/* Static text for a status code. */
const char* dspark_status_string(int status);

/* Kernels launched by the last call on this workspace (for accounting). */
int dspark_last_launch_count(dspark_ws* ws);

/* Name of the compute path the workspace uses ("tcgen05" or "simt"). */
const char* dspark_path(dspark_ws* ws);

/* Choose the compute path of the two stages that contract with W2 (the draft
 * and the residual recompute of verify): "tcgen05" (tensor-core kernels; bf16
 * weights, r % 64 == 0, r <= 256, B <= 1024) or "simt" (CUDA-core kernels, any
 * shape). Both compute the same draws; the default is "tcgen05" where it
 * applies. Returns EUNSUPPORTED if the tcgen05 path does not apply. */
dspark_status dspark_ws_set_path(dspark_ws* ws, const char* path);

/*
 * Draft x_1..x_gamma for every request. Outputs, each [B, gamma]:
 *   tokens  int32   x_k
 *   pd_tok  fp32    p_k(x_k), the draft probability of the drafted token
 *   lse     fp32    log sum_v exp(U_k(v) + W1[x_{k-1}] . W2[:, v])
 *   conf    fp32    c_k
 * anchor [B] int32 in [0, V). Sampling, temperature 1: a two-level Gumbel-max
 * over vocabulary blocks of 64 tokens, the block s by argmax (log mass_s + G)
 * and the token inside it by argmax (z_v + G), each G = -log(-log u) with u
 * from Philox4x32-10 (key = seed, counter (index >> 2, b, k, purpose << 24 |
 * round mod 2^24), word index & 3; purpose 1 for blocks, 2 for tokens).
 */
dspark_status dspark_markov_draft(dspark_ws* ws, const float* U, const void* W1, const void* W2,
                                  const int32_t* anchor, const float* h, const float* w,
                                  const float* T, uint64_t seed, uint64_t round,
                                  int32_t* tokens, float* pd_tok, float* lse, float* conf,
                                  dspark_stream_t stream);

/*
 * Verify lengths from the confidences conf [B, gamma] and the SPS table
 * sps [1 + B * (gamma + 1)] (fp64; sps[n] = engine steps per second at n
 * verify tokens; entry 0 unused). Outputs lengths [B] int32 in [1, gamma+1]
 * and row_off [B + 1] int32, the exclusive scan of lengths (row_off[B] =
 * total verify rows). STATIC mode ignores conf and sps. COMPACT_LAGGED pushes
 * conf into the workspace ring; its first `lag` calls after a reset plan
 * synchronously (Algorithm 1).
 */
dspark_status dspark_plan(dspark_ws* ws, const float* conf, const double* sps,
                          int32_t* lengths, int32_t* row_off, dspark_stream_t stream);

/*
 * A batch split by request across devices. The planner's objective
 * Theta = tau * SPS(B_tot) ("spec_dspark", section "目标函数": the SPS table
 * is a property of the target engine's whole verify batch) couples every
 * request of the batch, while draft and verify are independent per request.
 * So each device drafts and verifies its own contiguous range of requests
 * with a workspace of that range's size, every device plans the whole batch
 * from the confidences of all devices (the caller all-gathers them: B * gamma
 * fp32), and each keeps its own range's lengths.
 *
 * dspark_ws_set_shard: the workspace holds requests b_offset .. b_offset +
 * B - 1 of the batch. The request word b of every Philox counter becomes
 * b_offset + b, so each request draws the same numbers as in an unsplit
 * batch. Default 0. EINVAL if b_offset < 0 or b_offset + B > 2^31 - 1.
 *
 * dspark_plan_shard: dspark_plan on a workspace made for the WHOLE batch
 * (dims.B = every device's requests; conf [B, gamma] gathered in batch
 * order; lengths [B], row_off [B + 1] as dspark_plan writes them), then
 * lengths_local[i] = lengths[b_begin + i] for i < b_count and
 * row_off_local[i] = row_off[b_begin + i] - row_off[b_begin] for i <= b_count:
 * the range's lengths and its own packed-row offsets, ready for that device's
 * dspark_verify. All buffers are the caller's device memory, 16-byte aligned.
 * EINVAL unless 0 <= b_begin, 1 <= b_count and b_begin + b_count <= B. Every
 * device that runs it on the same gathered confidences (and, for
 * COMPACT_LAGGED, the same history) gets the same whole-batch plan.
 */
dspark_status dspark_ws_set_shard(dspark_ws* ws, int b_offset);
dspark_status dspark_plan_shard(dspark_ws* ws, const float* conf, const double* sps, int b_begin, int b_count,
                                int32_t* lengths, int32_t* row_off, int32_t* lengths_local,
                                int32_t* row_off_local, dspark_stream_t stream);

/*
 * Verify. P packed [row_off[B], V] fp32 target logits; row_off and lengths as
 * written by dspark_plan; anchor [B]; tokens, pd_tok, lse [B, gamma] as written
 * by dspark_markov_draft; U, W1, W2 as given to it (the draft distribution at
 * a rejected position is recomputed from them). Outputs n_accepted [B] (drafts
 * accepted, 0 .. lengths[b]-1) and next_anchor [B] (residual or bonus token).
 */
dspark_status dspark_verify(dspark_ws* ws, const float* P, const int32_t* row_off,
                            const int32_t* lengths, const int32_t* anchor, const int32_t* tokens,
                            const float* pd_tok, const float* lse, const float* U,
                            const void* W1, const void* W2, uint64_t seed, uint64_t round,
                            int32_t* n_accepted, int32_t* next_anchor, dspark_stream_t stream);

/*
 * A whole round: draft, plan, then verify on P, which the caller has packed
 * for the lengths this round produces (benchmark use: with fixed inputs and
 * round the lengths are deterministic), so P holds at least B rows (every
 * request verifies at least one); the verify may start reading those first B
 * rows before the planner has finished. Same arguments as the three calls.
 */
dspark_status dspark_round(dspark_ws* ws, const float* U, const void* W1, const void* W2,
                           const int32_t* anchor, const float* h, const float* w, const float* T,
                           const double* sps, const float* P, uint64_t seed, uint64_t round,
                           int32_t* tokens, float* pd_tok, float* lse, float* conf,
                           int32_t* lengths, int32_t* row_off, int32_t* n_accepted,
                           int32_t* next_anchor, dspark_stream_t stream);

/*
 * Draft without a workspace and without allocating anything, for callers that
 * cannot call cudaMalloc (an engine whose memory pool owns all device memory,
 * a plug-in that must not grow the process's device footprint, code under a
 * hard memory budget). The pages describe no such call; it exists only for
 * those callers.
 *
 * Same inputs and outputs as dspark_markov_draft, computed by the same
 * CUDA-core draft kernels (the "simt" path), plus device_status: a caller-owned
 * device int32 that the call zeroes and the kernels set to a dspark_status code
 * on a device error (read it after synchronising `stream`). Scratch comes from
 * a 4 MiB array built into the library (2^20 floats): calls whose
 * B*gamma (rounded up to 64) + B*ceil(V/64) exceeds 2^20 return
 * DSPARK_EUNSUPPORTED and enqueue nothing. The first call on a device looks up
 * the array's device address, so make it before any stream capture. Every
 * call shares the array: calls whose work overlaps on the GPU race, so issue
 * them on one stream. No cudaMalloc, cudaFree or allocating routine is called.
 */
dspark_status dspark_markov_draft_noalloc(const dspark_dims* dims, const float* U, const void* W1,
                                          const void* W2, const int32_t* anchor, const float* h,
                                          const float* w, const float* T, uint64_t seed, uint64_t round,
                                          int32_t* tokens, float* pd_tok, float* lse, float* conf,
                                          int32_t* device_status, dspark_stream_t stream);

/*
 * Sequential temperature scaling (STS) of the confidence head
 * ("DeepSeek-V4.1 模型结构（6）：解码，DSpark", section "confidence head";
 * zdszero "spec_dspark", "STS 校准"; deepseek.csdn.net §5.2). For N held-out
 * blocks of gamma positions, raw [N, gamma] fp32 holds the confidence logits
 * w^T [h_k; W1[x_{k-1}]] before the temperature and cstar [N, gamma] fp32 the
 * soft labels (each position's acceptance probability 1 - ||p_d - p_t||_1 / 2).
 * Left to right, T_out[k] becomes the first value of Tgrid [G] fp32 (> 0) that
 * minimises the expected calibration error, over M equal-width bins of [0, 1],
 * of a_k = prod_{i<=k} sigmoid(raw_i / T_i) against y_k = prod_{i<=k} cstar_i,
 * the earlier positions' temperatures kept; ece_out [gamma] fp64 receives that
 * ECE. All pointers are device pointers owned by the caller; scratch holds
 * dspark_sts_scratch_bytes(N, G) bytes (8-byte aligned) and device_status one
 * int32 that the call zeroes and a kernel sets to DSPARK_ERANGE for a grid
 * value that is not positive and finite. 1 <= M <= 32, N < 2^23, G <= 65535. Returns
 * EINVAL/EUNSUPPORTED/ECUDA on the host; asynchronous on `stream`.
 */
dspark_status dspark_sts_fit(const float* raw, const float* cstar, int N, int gamma, const float* Tgrid,
                             int G, int M, float* T_out, double* ece_out, void* scratch,
                             int32_t* device_status, dspark_stream_t stream);
size_t dspark_sts_scratch_bytes(int N, int G);

/*
 * The draft head's teacher-forced training objective
 * ("DeepSeek-V4.1 模型结构（6）：解码，DSpark", section on training the head for
 * the acceptance rate; deepseek.csdn.net §6, eqs. (9)-(12)). Position k of
 * request b drafts from x_prev = anchor[b] (k = 0) or xstar[b][k-1]; with
 * z_d = U[b][k] + W1[x_prev] W2, p_d = softmax(z_d), p_t = softmax(P[b][k]):
 *   ce[b][k]  = logsumexp(z_d) - z_d[xstar[b][k]]
 *   l1[b][k]  = sum_v |p_d(v) - p_t(v)|
 *   bce[b][k] = -(c* log c + (1 - c*) log(1 - c)),  c* = 1 - l1 / 2, c = conf[b][k]
 *   *loss     = (1/B) sum_{b,k} exp(-k / tau) (0.1 ce + 0.9 l1 + bce)
 * The workspace's dims give B, gamma, V, r; the call needs bf16 weights,
 * r a multiple of 64 up to 256, V % 8 == 0 and B <= 1024 (else
 * DSPARK_EUNSUPPORTED). U and P are [B][gamma][V] fp32 (P: the target's logits
 * at the teacher-forced positions), W1 [V][r] and W2 [r][V] bf16, anchor [B]
 * and xstar [B][gamma] int32, conf [B][gamma] fp32 in (0, 1); ce, l1, bce
 * [B][gamma] fp32 and loss [1] fp64 receive the results. Every pointer is a
 * 16-byte aligned device pointer owned by the caller (loss: 8-byte);
 * scratch holds dspark_train_loss_scratch_bytes(ws) bytes, 256-byte aligned.
 * tau must be positive and finite (else DSPARK_EINVAL). A token id out of
 * [0, V) raises DSPARK_ERANGE and a confidence outside (0, 1) DSPARK_ENUMERIC
 * in the workspace's device status (dspark_last_error). Five launches,
 * asynchronous on `stream`; W2 is read through the L2 by every 32 positions.
 */
dspark_status dspark_train_loss(dspark_ws* ws, const float* U, const void* W1, const void* W2,
                                const int32_t* anchor, const int32_t* xstar, const float* P, const float* conf,
                                double tau, float* ce, float* l1, float* bce, double* loss, void* scratch,
                                dspark_stream_t stream);
size_t dspark_train_loss_scratch_bytes(const dspark_ws* ws);

/*
 * The draft tail with the RNN head instead of the Markov head
 * ("DeepSeek-V4.1 模型结构（6）：解码，DSpark", section on the Markov head, the
 * RNN variant; deepseek.csdn.net §4.2, eq. (6)). With s_0 = 0, x_0 = anchor[b]
 * and z_k = [s_{k-1}; W1[x_{k-1}]; h_k] (length 2r + H):
 *   s_k = sigma(W_g z_k) * s_{k-1} + (1 - sigma(W_g z_k)) * tanh(W_c z_k),
 *   o_k = tanh(W_o z_k),  logits_k = U_k + o_k W2,
 * and x_k, pd_tok, lse and conf exactly as dspark_markov_draft (the
 * confidence takes W1[x_{k-1}], eq. (7)). Wr is [3][r][2r + H] (W_g, W_c, W_o,
 * row-major, no bias) in the workspace's weight dtype; ovec [B][gamma][r] fp32
 * receives o_k. The other arguments are those of dspark_markov_draft. Every
 * pointer is a 16-byte aligned device pointer owned by the caller; scratch
 * holds dspark_rnn_draft_scratch_bytes(ws) bytes, 256-byte aligned. With
 * bf16 weights and r a multiple of 64 up to 256, each step's vocabulary pass
 * runs on tcgen05, and so does the h projection when H is a multiple of 64;
 * otherwise they run on CUDA cores. 2 or 3 launches, then 3 per draft step.
 * Asynchronous on `stream`; device errors go to the workspace's status word.
 */
dspark_status dspark_rnn_draft(dspark_ws* ws, const float* U, const void* W1, const void* W2, const void* Wr,
                               const int32_t* anchor, const float* h, const float* w, const float* T,
                               uint64_t seed, uint64_t round, int32_t* tokens, float* pd_tok, float* lse,
                               float* conf, float* ovec, void* scratch, dspark_stream_t stream);
size_t dspark_rnn_draft_scratch_bytes(const dspark_ws* ws);

/*
 * The verify of drafts made with the RNN head: as dspark_verify, but the draft
 * distribution of a rejected position n+1 is recomputed from ovec[b][n] (the
 * head vector o_{n+1} that dspark_rnn_draft wrote, fp32 [B][gamma][r]) as
 * softmax(U_{n+1} + o_{n+1} W2) instead of from W1[x_n]; W1 is not read. On
 * the tcgen05 path (bf16 weights, r a multiple of 64 up to 256, V % 8 == 0)
 * the residual block pass takes o_{n+1} as bf16 hi + lo operands (about 16
 * significant bits of o); otherwise it runs on CUDA cores in fp32. Same
 * pointer rules, outputs and errors as dspark_verify.
 */
dspark_status dspark_verify_rnn(dspark_ws* ws, const float* P, const int32_t* row_off, const int32_t* lengths,
                                const int32_t* anchor, const int32_t* tokens, const float* pd_tok, const float* lse,
                                const float* U, const float* ovec, const void* W2, uint64_t seed, uint64_t round,
                                int32_t* n_accepted, int32_t* next_anchor, dspark_stream_t stream);

/*
 * PCTree: the Markov head's draft made a tree ("DeepSeek-V4.1 模型结构（6）：
 * 解码，DSpark", follow-up note "后续工作": the Markov head scores every child
 * token under a parent, so candidate children are proposed per parent node
 * and the most probable paths are kept within a fixed verify budget, with no
 * retraining and no extra backbone pass).
 *
 * dspark_pctree_build grows, for every request b, a tree of N nodes besides
 * the root best first: node 0 is anchor[b] (depth 0, log-probability 0);
 * expanding a node with token x at depth k < gamma proposes its c most
 * probable children under softmax(U[b, k] + W1[x] W2) (ties to the smaller
 * token); the next node admitted is the best candidate so far (the higher path
 * log-probability, then the smaller depth, parent index, token), and it is
 * expanded in turn, until N nodes are in or no candidate is left. Outputs,
 * each [B][N+1] with node i in admission order: tok int32, par int32 (parent
 * node index, -1 for the root), dep int32, lp fp32 (path log-probability:
 * the sum of log p_d along the path); slots past the last node hold -1 (lp:
 * -inf). n_nodes [B] int32. 1 <= c <= 8, 1 <= N <= 64, V < 2^24, c <= V.
 * scratch holds dspark_pctree_scratch_bytes(ws, c, N) bytes, 256-byte aligned
 * (0 means unsupported dims). An anchor out of range sets DSPARK_ERANGE.
 *
 * dspark_pctree_verify walks each request's tree: P [B][N+1][V] fp32 holds
 * the target's logits after each node's path (row i for node i). At a node,
 * its children (par == node, in index order) are tried in turn, child i
 * accepted when u < p(t_i) / (1 - the target probability of the children
 * rejected before it), u uniform from the stream (purpose 8, j = node, index
 * i); an accepted child becomes the node. With no child accepted the next
 * anchor is drawn from the target with the tried children removed: the
 * two-level Gumbel-max (purposes 9 and 10, j = node). Outputs: path
 * [B][gamma+1] int32 (the accepted nodes, root first, -1 after the last),
 * n_accepted [B] (accepted draft tokens), next_anchor [B]. V % 4 == 0 and
 * ceil(V/64) * 4 + 128 KiB of shared memory must fit one CTA, else
 * EUNSUPPORTED. Both calls are asynchronous on `stream`; all pointers are
 * device pointers owned by the caller.
 */
size_t dspark_pctree_scratch_bytes(const dspark_ws* ws, int c, int N);
dspark_status dspark_pctree_build(dspark_ws* ws, const float* U, const void* W1, const void* W2,
                                  const int32_t* anchor, int c, int N, int32_t* tok, int32_t* par, int32_t* dep,
                                  float* lp, int32_t* n_nodes, void* scratch, dspark_stream_t stream);
dspark_status dspark_pctree_verify(dspark_ws* ws, const float* P, const int32_t* tok, const int32_t* par, int N,
                                   uint64_t seed, uint64_t round, int32_t* path, int32_t* n_accepted,
                                   int32_t* next_anchor, dspark_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* DSPARK_H */
