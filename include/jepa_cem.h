/*
 * jepa_cem.h -- C ABI of the GB300 (sm_103a) CEM planner over an action-conditioned
 * JEPA world-model predictor.
 *
 * What it computes follows "Real-time inference for JEPA world-model architectures
 * with Ray", section "Where the sixteen seconds actually goes": in each of R rounds a
 * planning step samples N action sequences from a Gaussian, predicts with the world
 * model where each one leads, measures how far each predicted embedding lies from the
 * goal embedding and refits the Gaussian to the K closest; the caller receives only
 * the first action of the closest sequence of the last round. Section "Measured on 8x A100" adds that the
 * predictor attends only to current and earlier frames (so keys and values cached between
 * rollout steps stay exact), that it
 * runs in bf16 with flash attention, and that the same seed gives the same plan
 * however the candidates are batched.
 *
 * Conventions for every entry point:
 *   - Tensors are dense, row-major, float32 unless stated. Shapes use
 *     B problems, N candidates, H horizon steps, A action dim, S state dim,
 *     P patch tokens per frame, E embedding dim.
 *   - Pointers marked "dev" are device pointers on the context's device. Pointers
 *     marked "dev|host" may be device memory or host memory (pinned or pageable);
 *     the library copies them with cudaMemcpyAsync(cudaMemcpyDefault).
 *   - The caller owns every buffer it passes; the context owns weights, workspaces
 *     and captured CUDA graphs. Nothing passed in is retained after the call returns
 *     except through the stream's pending work.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Work is enqueued
 *     asynchronously; outputs are valid once the stream has been synchronised.
 *   - Every call returns a jepa_status and never aborts the process. After an error
 *     the output contents are unspecified; the context stays usable and
 *     jepa_last_error() describes the failure. A context must not be used from two
 *     host threads at once.
 */
#ifndef JEPA_CEM_H_
#define JEPA_CEM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  JEPA_OK = 0,
  JEPA_ERR_INVALID_ARG = 1,  /* NULL pointer, non-positive size, K > N, ... */
  JEPA_ERR_SHAPE = 2,        /* shape outside what the context was created for */
  JEPA_ERR_NOT_LOADED = 3,   /* weights not loaded yet */
  JEPA_ERR_OOM = 4,          /* device allocation failed */
  JEPA_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed */
  JEPA_ERR_TIMEOUT = 6,      /* a bounded device-side wait gave up (kernel returned early) */
  JEPA_ERR_UNSUPPORTED = 7   /* device is not sm_103 / feature not built */
} jepa_status;

/* FP8: the bf16 path with the GEMMs fed by a LayerNorm (QKV, MLP up, projection to E) on
 * fp8 e4m3 operands (kind::f8f6f4): weights with one scale per output channel, the
 * LayerNorm output with one scale per row; everything else as in BF16. (The planning
 * page's "Further Optimization", D, and the Realtime-VLA notes, 9.1, name 8-bit
 * quantisation of the predictor as the way to shrink its compute.) */
typedef enum { JEPA_FP32 = 0, JEPA_BF16 = 1, JEPA_FP8 = 2 } jepa_precision;

/* MLP of each layer. GELU: u = GELU(W_1 h + b_1). GATED (the Realtime-VLA notes, section 4.2
 * "Fusing Gated Linear Layers": FC1(x, w1) * GELU(FC2(x, w2))): u = (W_1 h + b_1) *
 * GELU(W_g h + b_g), computed by one GEMM over the two weight matrices' rows interleaved in
 * blocks of 32, whose epilogue writes only the product. */
typedef enum { JEPA_MLP_GELU = 0, JEPA_MLP_GATED = 1 } jepa_mlp_kind;

/* Predictor shape. Pre-LN transformer, block-causal over frame blocks of
 * T = patch_tokens + 2 tokens ([action, state, P patches]). */
typedef struct {
  int32_t layers;        /* L */
  int32_t width;         /* d, multiple of 32 (bf16: multiple of 64) */
  int32_t heads;         /* h; head dim d/h = 64 in bf16 mode, <= 128 in fp32 mode */
  int32_t mlp;           /* m, hidden width of the MLP (bf16 gated: multiple of 128) */
  int32_t patch_tokens;  /* P */
  int32_t embed_dim;     /* E, multiple of 32 (bf16: multiple of 64) */
  int32_t action_dim;    /* A (7 in the planning workloads) */
  int32_t state_dim;     /* S (7) */
  int32_t max_horizon;   /* largest H any call will use; sizes the KV cache */
  int32_t precision;     /* jepa_precision: FP32 = SIMT fp32 path, BF16 = tensor-core path,
                            FP8 = tensor-core path with fp8 LayerNorm-fed GEMMs */
  float ln_eps;          /* LayerNorm epsilon (1e-5) */
  int32_t max_chunk;     /* candidates per predictor pass (0 = library default); bounds workspace */
  int32_t mlp_kind;      /* jepa_mlp_kind */
} jepa_config;

typedef struct jepa_ctx jepa_ctx;

/* Optional per-round record of a plan. All device pointers; each may be NULL. */
typedef struct {
  float* mu;        /* [R+1, B, H, A]  mu_0 .. mu_R */
  float* sigma;     /* [R+1, B, H, A]  sigma_0 .. sigma_R */
  float* actions;   /* [R, B, N, H, A] clipped candidates of each round */
  float* energy;    /* [R, B, N]       energies of each round */
  int32_t* elites;  /* [R, B, K]       elite indices, ascending (energy, index) */
  int32_t* winner;  /* [B]             winner of the final round */
} jepa_cem_trace;

/* Create a context on CUDA device `device` for predictor shape *cfg.
 * Fails with JEPA_ERR_UNSUPPORTED unless the device is compute capability 10.3. */
jepa_status jepa_create(const jepa_config* cfg, int device, jepa_ctx** out);

/* Free the context and everything it owns. Synchronises the device first. NULL is a no-op. */
void jepa_destroy(jepa_ctx* ctx);

/* Text of the last error on this context ("" if none). Valid until the next call on ctx. */
const char* jepa_last_error(const jepa_ctx* ctx);

/* Static name of a status code. */
const char* jepa_status_string(jepa_status s);

/* Size in bytes of the weight blob for *cfg: a 64-byte header (int32 magic 0x4150454A,
 * version 1, layers, width, heads, mlp, patch_tokens, embed_dim, action_dim, state_dim,
 * mlp_kind, then zeros) followed by float32 tensors in this order, each row-major [out, in]:
 * W_in[d,E] b_in[d] W_a[d,A] b_a[d] W_s[d,S] b_s[d] pos[T,d], per layer
 * {ln1_g[d] ln1_b[d] W_qkv[3d,d] b_qkv[3d] W_o[d,d] b_o[d] ln2_g[d] ln2_b[d]
 *  W_1[m,d] b_1[m] (gated only: W_g[m,d] b_g[m]) W_2[d,m] b_2[d]},
 * lnf_g[d] lnf_b[d] W_out[E,d] b_out[E]. */
size_t jepa_weight_blob_bytes(const jepa_config* cfg);

/* Upload predictor weights from a host blob (format above). Validates the header
 * against the context's config (JEPA_ERR_SHAPE on mismatch), converts the GEMM
 * matrices to bf16 in bf16 mode, and blocks until the upload is done. On error the
 * previously loaded weights (if any) stay in place. */
jepa_status jepa_load_weights(jepa_ctx* ctx, const void* host_blob, size_t bytes);

/* Candidate sampler (the planning page, "Where the sixteen seconds actually goes": each
 * round's candidate action sequences are drawn from a Gaussian around the current guess).
 *   mu, sigma [B,H,A] dev; actions [B,N,H,A] dev (output).
 * eps[b,n,h,j] comes from Philox4x32-10 with key (seed lo, seed hi) and counter
 * (n, b, round*Q + q, 0), Q = ceil(H*A/4), q = (h*A+j)/4, word (h*A+j)%4, turned into
 * normals by Box-Muller on u = ((x>>9)+0.5)*2^-23 (cos for words 0/2, sin for 1/3);
 * actions = clip(mu + sigma*eps, -1, 1). Draws depend only on (seed, b, n, round, h, j). */
jepa_status jepa_sample_actions(jepa_ctx* ctx, const float* mu, const float* sigma, int B, int N,
                                int H, int round, uint64_t seed, float* actions, void* stream);

/* The sampler's generator alone: out[i] = Philox4x32-10(counter[i], key = (seed lo, seed hi)),
 * the four 32-bit output words of counter words counters[4i .. 4i+3] (uint32, dev; n >= 1).
 * Exposed so that integer outputs can be compared bit for bit. */
jepa_status jepa_philox4x32_10(jepa_ctx* ctx, const uint32_t* counters, uint64_t seed, int n,
                               uint32_t* out, void* stream);

/* Predictor rollout and L1 energy (the step of the same section that rolls every candidate
 * through the predictor and scores the outcome against the goal embedding; frame-causal
 * with a KV cache).
 *   z_ctx [B,P,E] dev   encoded context frame of each problem
 *   state0 [B,S] dev    state of each problem (s_k = s_{k-1} + a_{k-1})
 *   actions [B,N,H,A] dev
 *   goal [B,P,E] dev or NULL
 *   z_pred [B,N,P,E] dev or NULL   output: the last predicted frame z_H
 *   energy [B,N] dev or NULL       output: mean |z_H - goal| (needs goal)
 * 1 <= H <= cfg.max_horizon. */
jepa_status jepa_predictor_forward(jepa_ctx* ctx, const float* z_ctx, const float* state0,
                                   const float* actions, int B, int N, int H, const float* goal,
                                   float* z_pred, float* energy, void* stream);

/* Elite selection and Gaussian refit (the same section: the best K candidates are kept and
 * the Gaussian is moved onto them): per problem, the K lowest energies ordered by
 * (energy, index), NaN last; then
 * mu' = elite mean and sigma' = elite population std per (h, j).
 *   energy [B,N] dev; actions [B,N,H,A] dev; mu_out, sigma_out [B,H,A] dev (outputs);
 *   elites_out [B,K] int32 dev or NULL. 1 <= K <= N <= 8192. */
jepa_status jepa_cem_select_refit(jepa_ctx* ctx, const float* energy, const float* actions, int B,
                                  int N, int H, int K, float* mu_out, float* sigma_out,
                                  int32_t* elites_out, void* stream);

/* One full planning step: R rounds of sample -> predictor -> energy -> select/refit with
 * no host round-trip between rounds (one captured CUDA graph per (B,H,N,K,R), cached in
 * the context), then action_out[b] = first action of problem b's lowest-energy
 * candidate in the final round.
 *   z0, goal [B,P,E], state0 [B,S], mu0, sigma0 [B,H,A]: dev|host inputs
 *   action_out [B,A]: dev|host output
 *   trace: NULL or per-round record (device pointers, see jepa_cem_trace)
 * The first call for a new (B,H,N,K,R) allocates workspace and captures the graph. */
jepa_status jepa_cem_plan(jepa_ctx* ctx, const float* z0, const float* state0, const float* goal,
                          const float* mu0, const float* sigma0, int B, int H, int N, int K,
                          int rounds, uint64_t seed, float* action_out,
                          const jepa_cem_trace* trace, void* stream);

/* Warm start of the next planning step under receding-horizon control (planning page,
 * section "Further Optimization", B "Warm-started CEM": only the first action of a plan is
 * executed, and the rest of it may seed the next step instead of a fresh Gaussian).
 *   mu_prev [B,H,A] dev        the previous plan's last-round mean (the slice
 *                              trace->mu + rounds*B*H*A of jepa_cem_plan's trace)
 *   mu_prior, sigma_prior [B,H,A] dev   the fresh Gaussian
 *   mu_out, sigma_out [B,H,A] dev       outputs; mu_out may equal mu_prev and sigma_out may
 *                                       equal sigma_prior (no other overlap)
 * mu_out[b,h] = mu_prev[b,h+1] for h < H-1, mu_out[b,H-1] = mu_prior[b,H-1];
 * sigma_out = sigma_prior. With H = 1 this is the prior itself. */
jepa_status jepa_cem_warm_start(jepa_ctx* ctx, const float* mu_prev, const float* mu_prior,
                                const float* sigma_prior, int B, int H, float* mu_out,
                                float* sigma_out, void* stream);

/* One step of the world model playing the robot, as in that section's closed-loop
 * experiments: the executed action goes through the predictor with horizon 1.
 *   z [B,P,E], state [B,S], action [B,A]: dev inputs
 *   z_next [B,P,E] dev   output: the predicted next frame (must not overlap z)
 *   state_next [B,S] dev output: state + action (may equal state)
 *   goal [B,P,E] dev or NULL; distance [B] dev or NULL: mean |z_next - goal| (needs goal) */
jepa_status jepa_world_model_step(jepa_ctx* ctx, const float* z, const float* state,
                                  const float* action, int B, const float* goal, float* z_next,
                                  float* state_next, float* distance, void* stream);

/* Closed-loop episode: `steps` times (plan with jepa_cem_plan, execute the winner's first
 * action with jepa_world_model_step, replan from the predicted frame), all enqueued on
 * `stream` with no host synchronisation between steps. Step t plans with seed + t and
 * starts from the prior (warm = 0) or, for t >= 1, from jepa_cem_warm_start of step t-1's
 * last-round mean (warm = 1).
 *   z0, goal [B,P,E], state0 [B,S], mu_prior, sigma_prior [B,H,A]: dev|host inputs
 *   actions_out [steps,B,A]: dev|host output, the executed actions
 *   distance_out [steps,B]: dev|host output, mean |z_{t+1} - goal| after each action
 * Workspace for the episode is kept in the context and grows on demand (the first call
 * with larger sizes synchronises the device). */
jepa_status jepa_cem_closed_loop(jepa_ctx* ctx, const float* z0, const float* state0,
                                 const float* goal, const float* mu_prior,
                                 const float* sigma_prior, int B, int H, int N, int K, int rounds,
                                 int steps, int warm, uint64_t seed, float* actions_out,
                                 float* distance_out, void* stream);

/* Number of kernel launches one jepa_cem_plan call with these sizes makes (captures
 * the graph if needed). */
jepa_status jepa_plan_kernel_count(jepa_ctx* ctx, int B, int H, int N, int K, int rounds,
                                   int64_t* count);

/* Dense linear layer on the tensor-core GEMM used by the predictor (bf16 in, fp32
 * accumulate): out[M,N] = act(A[M,K] * W[N,K]^T + bias[N]).
 *   A, W: bf16 bit patterns (uint16) dev; bias [N] dev or NULL; out [M,N] float32 dev.
 *   gelu: 0 = identity, 1 = erf GELU, 2 = gated: W's rows are FC1 and gate blocks of 32
 *   interleaved (rows 64p..64p+31 = FC1 rows 32p.., rows 64p+32..64p+63 = gate rows 32p..),
 *   bias interleaved the same way (required), N a multiple of 256, and
 *   out[M,N/2][32p + c] = (acc[64p + c] + bias) * GELU(acc[64p + 32 + c] + bias).
 * K a multiple of 8. Needs a bf16 context. */
jepa_status jepa_linear_bf16(jepa_ctx* ctx, const uint16_t* A, const uint16_t* W,
                             const float* bias, int M, int N, int K, int gelu, float* out,
                             void* stream);

/* The residual GEMM of the predictor on caller data (the attention out-projection and the
 * MLP down-projection of a pre-LN block, "Real-time inference for JEPA world-model
 * architectures with Ray", the predictor of section "Measured on 8x A100"):
 *   x[M,N] += A[M,K] * W[N,K]^T + bias[N], fp32 accumulation, x fp32 updated in place.
 *   A, W: bf16 bit patterns dev, 16-byte aligned; bias [N] dev or NULL; x [M,N] fp32 dev.
 *   K a multiple of 8, N a multiple of 4. Needs a bf16 context. */
jepa_status jepa_linear_resid_bf16(jepa_ctx* ctx, const uint16_t* A, const uint16_t* W,
                                   const float* bias, int M, int N, int K, float* x,
                                   void* stream);

/* The QKV GEMM of the predictor on caller data, writing one rollout step's rows into the
 * candidates' K/V caches (KV cache across rollout steps, the planning page, "Measured on
 * 8x A100"): acc = A[M,K] * W[3d,K]^T + bias[3d] (fp32), rounded to bf16, and for each
 * row r < M, with candidate c = r / T and t = r % T,
 *   q[r, 0:d] = acc[r, 0:d],   kv[c][frame*T + t][0:2d] = acc[r, d:3d].
 * Other rows of kv are not written.
 *   A, W: bf16 bit patterns dev, 16-byte aligned; bias [3d] dev or NULL;
 *   q [M, d] and kv [ceil(M/T)][kv_rows][2d]: bf16 bit patterns dev.
 *   d a multiple of 32, K a multiple of 8, T >= 1, 0 <= frame, (frame + 1) * T <= kv_rows.
 * Needs a bf16 context. */
jepa_status jepa_linear_qkv_bf16(jepa_ctx* ctx, const uint16_t* A, const uint16_t* W,
                                 const float* bias, int M, int d, int K, int T, int kv_rows,
                                 int frame, uint16_t* q, uint16_t* kv, void* stream);

/* The fp8 GEMM of the FP8 mode on caller data: out[M,N] = act((A[M,K] * W[N,K]^T) *
 * a_scale[M] (rows) * w_scale[N] (columns) + bias[N]), A and W e4m3 codes (one byte each,
 * OCP E4M3: bias 7, no infinities, largest 448), fp32 accumulation, fp32 output.
 *   gelu: 0 identity, 1 erf GELU, 2 gated (as jepa_linear_bf16; out [M, N/2]).
 *   K a multiple of 16; A, W 16-byte aligned dev; scales and bias dev. Needs a BF16 or FP8
 *   context. */
jepa_status jepa_linear_fp8(jepa_ctx* ctx, const uint8_t* A, const float* a_scale,
                            const uint8_t* W, const float* w_scale, const float* bias, int M,
                            int N, int K, int gelu, float* out, void* stream);

/* Row-wise fp8 quantisation, the rule of the FP8 mode: per row r, scales[r] = max|x[r,:]| /
 * 448 (1 for an all-zero row) and codes[r,c] = e4m3(x[r,c] * (448 / max|x[r,:]|)), rounded to
 * nearest even and saturated (fp32 arithmetic: the division and the product each rounded).
 *   x [rows, cols] float32 dev; codes [rows, cols] uint8 dev; scales [rows] float32 dev. */
jepa_status jepa_quantize_rows_fp8(jepa_ctx* ctx, const float* x, int rows, int cols,
                                   uint8_t* codes, float* scales, void* stream);

/* Block-causal attention of one rollout step as the predictor runs it (bf16 mode): for each
 * candidate c and head h, queries q[c*T + t, h*64 : h*64+64] attend to cached key / value
 * rows [0, Lk) of kv[c] (keys at columns [h*64, h*64+64), values at [d + h*64, ...)) with
 * scale 1/8: out[c*T + t, h*64 + j] = sum_i softmax_i(q . k_i / 8) v_i[j]. (Frame-causal
 * predictor with a KV cache, the planning page, "Measured on 8x A100".)
 *   q [ncand*T, d], kv [ncand][kv_rows][2d], out [ncand*T, d]: bf16 bit patterns, dev.
 *   1 <= Lk <= kv_rows; d = heads * 64; rows of kv past Lk must hold finite values.
 * Runs the predictor's tcgen05 attention kernel. Needs a bf16 context. */
jepa_status jepa_attention_bf16(jepa_ctx* ctx, const uint16_t* q, const uint16_t* kv, uint16_t* out,
                                int ncand, int T, int Lk, int kv_rows, int heads, int d,
                                void* stream);

/* enable = 0: jepa_cem_plan launches the kernels of its captured graph one by one on the
 * stream instead of replaying the graph (same kernels, same results; for measuring what the
 * graph saves). enable != 0 (the default): graph replay. */
jepa_status jepa_set_use_graphs(jepa_ctx* ctx, int enable);

/* Kernel-level timing of the predictor GEMMs inside plan graphs. enable != 0 makes graphs
 * captured afterwards record a CUDA event pair around every GEMM launch (graphs captured
 * before keep their state). jepa_profile_read (after the stream is synchronised) returns
 * the summed event time, summed algorithmic FLOPs (2*M*N*K) and launch count of the
 * GEMMs in the most recent plan call, and resets nothing. */
jepa_status jepa_profile_enable(jepa_ctx* ctx, int enable);
jepa_status jepa_profile_read(jepa_ctx* ctx, double* gemm_ms, double* gemm_flops,
                              int64_t* gemm_launches);

/* L1 energy of already-predicted frames, for callers that cannot allocate device memory
 * (the planning pages have no counterpart: this is a deployment variant of the energy
 * step). Typical callers: a process running under a fixed device-memory budget owned by
 * a host framework, or a real-time control loop that must not pay for, or risk failure
 * of, an allocation in the middle of an episode. No context is needed and nothing is
 * allocated: the per-candidate partial sums go to one fixed device array inside this
 * library, 2^20 floats (4 MiB), which every GPU that loads the library keeps until the
 * process exits.
 *   z_pred [B,N,P,E] dev   predicted frames (e.g. the z_pred output of jepa_predictor_forward)
 *   goal   [B,P,E]   dev
 *   energy [B,N]     dev   output: mean |z_pred - goal| per candidate
 *   err, err_len           optional caller buffer for a text description of a failure
 * Limits: B*N*ceil(P/32) <= 2^20, otherwise JEPA_ERR_SHAPE (split the candidates over
 * several calls). Runs on the current CUDA device. The first call in a device's CUDA context
 * looks up the array's device address and caches it for that context (a device reset makes a
 * new context, and the next call looks the address up again), so make that first call before
 * any stream capture. All calls share the array: calls that can overlap on the GPU (on streams with
 * no ordering between them) race and can return wrong energies; calls ordered on one
 * stream are safe. */
jepa_status jepa_energy_l1_noalloc(const float* z_pred, const float* goal, int B, int N, int P,
                                   int E, float* energy, void* stream, char* err, size_t err_len);

/* Failure-detection self-test: launches one thread that waits, through the bounded mbarrier
 * wait every pipelined kernel of this library uses, on a barrier nothing will arrive on.
 * After the wait's limit (2 s) it gives up, raises this context's error flag and returns;
 * the next jepa_sync_check then reports JEPA_ERR_TIMEOUT (and clears the flag). Nothing
 * faults or hangs; the context stays usable. */
jepa_status jepa_selftest_bounded_wait(jepa_ctx* ctx, void* stream);

/* Synchronise `stream`, then report JEPA_ERR_TIMEOUT if a bounded device-side wait in
 * any kernel of this context gave up since the last check (the flag is then cleared). */
jepa_status jepa_sync_check(jepa_ctx* ctx, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* JEPA_CEM_H_ */
