// Host runtime behind the C ABI (jepa_cem.h): context, weights, workspace, the chunked
// predictor pass, and the CUDA-graph-captured CEM round loop.
//
// One planning step ("Real-time inference for JEPA world-model architectures with Ray",
// section "Where the sixteen seconds actually goes") is captured once per
// (B, H, N, K, R) as a single CUDA graph: rounds follow each other on the device with
// mu/sigma kept in device memory, so the host is not involved between rounds (the pages
// point out that rounds which must run one after another bound the latency from below).
#include "jepa_cem.h"
#include "common.cuh"

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <string>
#include <tuple>
#include <vector>

using namespace jepa;

namespace {

constexpr int32_t kMagic = 0x4150454A;  // "JEPA"
constexpr int kHeaderBytes = 64;
constexpr int kDefaultChunk = 1024;
constexpr int kMaxSelectN = 8192;

struct LayerW {
  const float *ln1_g, *ln1_b, *b_qkv, *b_o, *ln2_g, *ln2_b, *b_1, *b_2;
  const void *W_qkv, *W_o, *W_1, *W_2;  // bf16 (bf16 mode) or fp32
  // gated MLP: W_1 and b_1 above point at the interleaved [FC1 | gate] pair (2m rows)
  const uint8_t *W_qkv8 = nullptr, *W_18 = nullptr;   // fp8 mode: e4m3 codes
  const float *s_qkv = nullptr, *s_1 = nullptr;        // and their channel scales
};

struct Weights {
  float* f32 = nullptr;   // device copy of every tensor (blob minus header)
  bf16* mats = nullptr;   // bf16 copies of the GEMM matrices (bf16 mode)
  uint8_t* q8 = nullptr;  // fp8 mode: e4m3 codes of W_qkv, W_1 (or the gated pair), W_out
  float* q8s = nullptr;   // fp8 mode: their per-output-channel scales
  const uint8_t* W_out8 = nullptr;
  const float* s_out = nullptr;
  void* gmat = nullptr;   // gated MLP: per layer W_1 / W_g rows interleaved in blocks of 32
  float* gbias = nullptr; // gated MLP: per layer b_1 / b_g interleaved the same way
  const float *b_in, *W_a, *b_a, *W_s, *b_s, *pos, *lnf_g, *lnf_b, *b_out;
  const void *W_in, *W_out;
  std::vector<LayerW> layers;
};

struct PlanGraph {
  int B = 0, H = 0, N = 0, K = 0, R = 0;
  bool profiled = false;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int64_t kernels = 0;
  std::vector<void*> allocs;
  float *z0 = nullptr, *goal = nullptr, *state0 = nullptr, *mu = nullptr, *sigma = nullptr;
  float *actions = nullptr, *energy = nullptr, *action_out = nullptr, *base = nullptr;
  void* z0_act = nullptr;
  // layer 0's q / kv of the frame-0 patch rows per problem (and the LayerNorm output they
  // come from): shared by every candidate of the problem
  void *q_base = nullptr, *kv_base = nullptr, *xn_base = nullptr;
  float* xs_base = nullptr;
  int *elites = nullptr, *winner = nullptr;
  unsigned int* select_counter = nullptr;   // per problem, for the fused energy + selection
  uint64_t* seed = nullptr;
  std::vector<cudaEvent_t> ev_start, ev_end;
  std::vector<double> ev_flops;
};

}  // namespace

struct jepa_ctx {
  jepa_config cfg;
  int device = 0;
  int num_sms = 148;
  std::string err;
  bool loaded = false;
  Weights w;
  // workspace for predictor passes
  int ws_chunk = 0, ws_H = 0;
  std::vector<void*> ws_allocs;
  float* x = nullptr;
  void *xn = nullptr, *q = nullptr, *kv = nullptr, *o = nullptr, *hbuf = nullptr, *zhat = nullptr;
  float* partial = nullptr;
  float* xs = nullptr;   // fp8 mode: row scales of the LayerNorm output in xn
  int ntiles = 0;
  // scratch for jepa_predictor_forward (base + converted context + layer-0 patch q / kv)
  std::vector<void*> fw_allocs;
  float* fw_base = nullptr;
  void* fw_z = nullptr;
  void *fw_qb = nullptr, *fw_kvb = nullptr, *fw_xnb = nullptr;
  float* fw_xsb = nullptr;
  size_t fw_cap = 0;  // problems
  int* dev_err = nullptr;
  cudaStream_t cap_stream = nullptr;
  bool profile = false;
  bool use_graphs = true;   // false: jepa_cem_plan launches the graph's kernels on the stream
  PlanGraph* last_plan = nullptr;
  // closed-loop episode state (grow-only; see jepa_cem_closed_loop)
  std::vector<void*> ep_allocs;
  int ep_B = 0, ep_H = 0, ep_R = 0;
  float *ep_z[2] = {nullptr, nullptr}, *ep_s[2] = {nullptr, nullptr}, *ep_goal = nullptr;
  float *ep_mu_prior = nullptr, *ep_sg_prior = nullptr, *ep_mu0 = nullptr, *ep_sg0 = nullptr;
  float *ep_mu_trace = nullptr, *ep_a = nullptr, *ep_dist = nullptr;
  std::map<std::tuple<int, int, int, int, int, bool>, PlanGraph*> graphs;
};

namespace {

jepa_status fail(jepa_ctx* c, jepa_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (c) c->err = buf;
  return s;
}

#define CK(call)                                                                          \
  do {                                                                                    \
    cudaError_t e_ = (call);                                                              \
    if (e_ != cudaSuccess)                                                                \
      return fail(ctx, e_ == cudaErrorMemoryAllocation ? JEPA_ERR_OOM : JEPA_ERR_CUDA,    \
                  "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__, __LINE__); \
  } while (0)

// bf16 activations and tensor-core path (the fp8 mode is the bf16 path with its
// LayerNorm-fed GEMMs on e4m3 operands)
inline bool bf16_mode(const jepa_ctx* c) { return c->cfg.precision != JEPA_FP32; }
inline bool fp8_mode(const jepa_ctx* c) { return c->cfg.precision == JEPA_FP8; }
inline int tokens(const jepa_ctx* c) { return c->cfg.patch_tokens + 2; }
inline size_t act_bytes(const jepa_ctx* c) { return bf16_mode(c) ? 2 : 4; }

size_t blob_floats(const jepa_config* c) {
  const size_t d = c->width, m = c->mlp, E = c->embed_dim, A = c->action_dim, S = c->state_dim,
               T = c->patch_tokens + 2;
  size_t n = d * E + d + d * A + d + d * S + d + T * d;
  n += (size_t)c->layers * (2 * d + 3 * d * d + 3 * d + d * d + d + 2 * d + m * d + m + d * m + d);
  if (c->mlp_kind == JEPA_MLP_GATED) n += (size_t)c->layers * (m * d + m);
  n += 2 * d + E * d + E;
  return n;
}

jepa_status validate_config(const jepa_config* c) {
  if (!c) return JEPA_ERR_INVALID_ARG;
  if (c->layers < 1 || c->width < 32 || c->heads < 1 || c->mlp < 32 || c->patch_tokens < 1 ||
      c->embed_dim < 32 || c->action_dim < 1 || c->action_dim > 32 || c->state_dim != c->action_dim ||
      c->max_horizon < 1 || c->max_horizon > 16 || c->width % c->heads != 0 || c->width % 32 ||
      c->embed_dim % 32 || c->mlp % 32 || c->width > 2048 || !(c->ln_eps >= 0.f) ||
      c->max_chunk < 0 || c->max_chunk > 65535 ||
      (c->mlp_kind != JEPA_MLP_GELU && c->mlp_kind != JEPA_MLP_GATED))
    return JEPA_ERR_SHAPE;
  const int hd = c->width / c->heads;
  if (c->precision == JEPA_BF16 || c->precision == JEPA_FP8) {
    if (hd != 64 || c->width % 64 || c->embed_dim % 64 || c->mlp % 64) return JEPA_ERR_SHAPE;
    if (c->mlp_kind == JEPA_MLP_GATED && c->mlp % 128) return JEPA_ERR_SHAPE;
  } else if (c->precision == JEPA_FP32) {
    if (hd % 32 || hd > 128) return JEPA_ERR_SHAPE;
  } else {
    return JEPA_ERR_INVALID_ARG;
  }
  return JEPA_OK;
}

template <typename T>
jepa_status dalloc(jepa_ctx* ctx, std::vector<void*>& list, T** p, size_t bytes) {
  void* q = nullptr;
  bytes = (bytes + 255) & ~(size_t)255;
  if (bytes == 0) bytes = 256;
  cudaError_t e = cudaMalloc(&q, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(ctx, JEPA_ERR_OOM, "cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
  }
  list.push_back(q);
  *p = (T*)q;
  return JEPA_OK;
}

void free_list(std::vector<void*>& l) {
  for (void* p : l) cudaFree(p);
  l.clear();
}

void free_plan(PlanGraph* g) {
  if (!g) return;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  for (auto e : g->ev_start) cudaEventDestroy(e);
  for (auto e : g->ev_end) cudaEventDestroy(e);
  free_list(g->allocs);
  delete g;
}

void drop_graphs(jepa_ctx* c) {
  cudaDeviceSynchronize();
  for (auto& kv : c->graphs) free_plan(kv.second);
  c->graphs.clear();
  c->last_plan = nullptr;
}

// Workspace for passes over `chunk` candidates with horizon up to H.
jepa_status ensure_workspace(jepa_ctx* ctx, int chunk, int H) {
  if (chunk <= ctx->ws_chunk && H <= ctx->ws_H) return JEPA_OK;
  drop_graphs(ctx);
  free_list(ctx->ws_allocs);
  ctx->ws_chunk = ctx->ws_H = 0;
  const jepa_config& c = ctx->cfg;
  const size_t T = tokens(ctx), d = c.width, m = c.mlp, P = c.patch_tokens, E = c.embed_dim;
  const size_t rows = (size_t)chunk * T, ab = act_bytes(ctx);
  const size_t kv_slots = H > 1 ? (size_t)c.layers : 1;
  ctx->ntiles = bf16_mode(ctx) ? gemm_tc_partials((int)E) : gemm_simt_partials((int)E);
  jepa_status s;
  if ((s = dalloc(ctx, ctx->ws_allocs, &ctx->x, rows * d * 4)) ||
      (s = dalloc(ctx, ctx->ws_allocs, &ctx->xn, rows * d * ab)) ||
      (s = dalloc(ctx, ctx->ws_allocs, &ctx->q, rows * d * ab)) ||
      (s = dalloc(ctx, ctx->ws_allocs, &ctx->kv, kv_slots * chunk * (size_t)H * T * 2 * d * ab)) ||
      (s = dalloc(ctx, ctx->ws_allocs, &ctx->o, rows * d * ab)) ||
      (s = dalloc(ctx, ctx->ws_allocs, &ctx->hbuf, rows * m * ab)) ||
      (s = dalloc(ctx, ctx->ws_allocs, &ctx->zhat, (size_t)chunk * P * E * ab)) ||
      (s = dalloc(ctx, ctx->ws_allocs, &ctx->partial, (size_t)chunk * P * ctx->ntiles * 4)) ||
      (s = dalloc(ctx, ctx->ws_allocs, &ctx->xs, fp8_mode(ctx) ? rows * 4 : 256))) {
    free_list(ctx->ws_allocs);
    return s;
  }
  // cache rows past the current key bound are read (and masked) by the attention kernels:
  // keep them finite
  const cudaError_t me = cudaMemset(ctx->kv, 0, kv_slots * chunk * (size_t)H * T * 2 * d * ab);
  if (me != cudaSuccess) {
    free_list(ctx->ws_allocs);
    return fail(ctx, JEPA_ERR_CUDA, "workspace init: %s", cudaGetErrorString(me));
  }
  ctx->ws_chunk = chunk;
  ctx->ws_H = H;
  return JEPA_OK;
}

int chunk_for(const jepa_ctx* c, long long total) {
  const int cap = c->cfg.max_chunk > 0 ? c->cfg.max_chunk : kDefaultChunk;
  return (int)(total < cap ? total : cap);
}

Epilogue epi_base(const jepa_ctx* c, int mode) {
  Epilogue e;
  memset(&e, 0, sizeof e);
  e.mode = mode;
  e.act_bf16 = bf16_mode(c) ? 1 : 0;
  e.map0 = identity_map();
  e.map1 = identity_map();
  e.split = 1 << 30;
  return e;
}

// out = epilogue(A * W^T) on the path of the context's precision; optionally bracketed by
// profiling events (graph capture).
jepa_status gemm(jepa_ctx* ctx, const void* A, const void* W, int M, int N, int K,
                 const Epilogue& e, cudaStream_t s, PlanGraph* prof, bool fp8 = false) {
  if (M <= 0) return JEPA_OK;
  if (prof) {
    cudaEvent_t a, b;
    CK(cudaEventCreate(&a));
    CK(cudaEventCreate(&b));
    prof->ev_start.push_back(a);
    prof->ev_end.push_back(b);
    prof->ev_flops.push_back(2.0 * M * N * (double)K);
    CK(cudaEventRecordWithFlags(a, s, cudaEventRecordExternal));
  }
  if (fp8) {
    CK(gemm_tc_fp8((const uint8_t*)A, (const uint8_t*)W, M, N, K, e, ctx->dev_err, ctx->num_sms, s));
  } else if (bf16_mode(ctx)) {
    CK(gemm_tc_bf16((const bf16*)A, (const bf16*)W, M, N, K, e, ctx->dev_err, ctx->num_sms, s));
  } else {
    CK(gemm_simt_f32((const float*)A, (const float*)W, M, N, K, e, s));
  }
  if (prof) CK(cudaEventRecordWithFlags(prof->ev_end.back(), s, cudaEventRecordExternal));
  return JEPA_OK;
}

// base[b, p, :] = W_in z[b, p, :] + b_in + pos[2 + p]  (candidate-independent patch tokens
// of frame 0, computed once per problem).
jepa_status context_projection(jepa_ctx* ctx, const float* z, void* z_act, float* base, int B,
                               cudaStream_t s, PlanGraph* prof) {
  const jepa_config& c = ctx->cfg;
  const int P = c.patch_tokens, E = c.embed_dim, d = c.width;
  const void* A = z;
  if (bf16_mode(ctx)) {
    CK(convert_f32_bf16(z, (bf16*)z_act, (long long)B * P * E, s));
    A = z_act;
  }
  Epilogue e = epi_base(ctx, EPI_INPROJ);
  e.bias = ctx->w.b_in;
  e.out0 = base;
  e.ld0 = d;
  e.map0 = RowMap{P, (long long)P, 0};
  e.pos = ctx->w.pos;
  e.pos_off = 2;
  return gemm(ctx, A, ctx->w.W_in, B * P, d, E, e, s, prof);
}

// Predictor rollout + energy for all B*N candidates (chunked). base holds the frame-0
// patch tokens per problem. Writes z_pred (last frame, fp32) and/or energy when non-null.
// LayerNorm 1 and the QKV product of layer 0 over the frame-0 patch rows base [B*P, d]: the
// same for every candidate of a problem (only the action and state tokens differ before the
// first attention). q_base [B*P, d] and kv_base [B*P, 2d] in the activation type; xn_base
// and xs_base hold the LayerNorm output (and its fp8 row scales).
jepa_status base_qkv(jepa_ctx* ctx, const float* base, int B, void* xn_base, float* xs_base,
                     void* q_base, void* kv_base, cudaStream_t s, PlanGraph* prof) {
  const jepa_config& c = ctx->cfg;
  const int P = c.patch_tokens, d = c.width;
  const LayerW& lw = ctx->w.layers[0];
  const bool f8 = fp8_mode(ctx);
  CK(layernorm(base, identity_map(), xn_base, f8 ? 2 : bf16_mode(ctx) ? 1 : 0, lw.ln1_g, lw.ln1_b,
               B * P, d, c.ln_eps, s, xs_base));
  Epilogue e = epi_base(ctx, EPI_STORE);
  e.bias = lw.b_qkv;
  e.out0 = q_base;
  e.ld0 = d;
  e.split = d;
  e.out1 = kv_base;
  e.ld1 = 2 * d;
  if (f8) {
    e.row_scale = xs_base;
    e.col_scale = lw.s_qkv;
  }
  return gemm(ctx, xn_base, f8 ? (const void*)lw.W_qkv8 : lw.W_qkv, B * P, 3 * d, d, e, s, prof, f8);
}

// Predictor rollout + energy for all B*N candidates (chunked). base holds the frame-0 patch
// tokens per problem; q_base / kv_base (or null) their layer-0 queries, keys and values
// (base_qkv), which frame 0 then takes instead of recomputing them per candidate. Writes
// z_pred (last frame, fp32) and/or energy when non-null.
jepa_status predictor_pass(jepa_ctx* ctx, const float* base, const void* q_base,
                           const void* kv_base, const float* state0, const float* actions, int B,
                           int N, int H, const float* goal, float* z_pred, float* energy,
                           cudaStream_t s, PlanGraph* prof) {
  const jepa_config& c = ctx->cfg;
  const int T = tokens(ctx), P = c.patch_tokens, E = c.embed_dim, d = c.width, m = c.mlp;
  const int A = c.action_dim, S = c.state_dim, L = c.layers, heads = c.heads;
  const long long total = (long long)B * N;
  const int chunk = ctx->ws_chunk;
  const long long kv_stride = (long long)ctx->ws_H * T;              // rows per candidate
  const size_t ab = act_bytes(ctx);
  const size_t kv_slot_elems = (size_t)chunk * kv_stride * 2 * d;
  // LayerNorm output: fp32, bf16, or (fp8 mode) e4m3 codes with row scales in xs
  const bool f8 = fp8_mode(ctx);
  const int ln_out = f8 ? 2 : bf16_mode(ctx) ? 1 : 0;
  jepa_status st;
  for (long long c0 = 0; c0 < total; c0 += chunk) {
    const int nc = (int)((total - c0) < chunk ? (total - c0) : chunk);
    const int rows = nc * T;
    for (int k = 0; k < H; ++k) {
      if (k > 0) {
        Epilogue e = epi_base(ctx, EPI_INPROJ);
        e.bias = ctx->w.b_in;
        e.out0 = ctx->x;
        e.ld0 = d;
        e.map0 = RowMap{P, (long long)T, 2};
        e.pos = ctx->w.pos;
        e.pos_off = 2;
        if ((st = gemm(ctx, ctx->zhat, ctx->w.W_in, nc * P, d, E, e, s, prof))) return st;
      }
      // frame 0 with shared patch rows: layer 0 computes LayerNorm 1 and QKV for the action
      // and state rows only; the patch rows' q / kv are broadcast from q_base / kv_base
      const bool shared0 = k == 0 && q_base != nullptr;
      BaseRows br;
      if (shared0) {
        br.q_base = (const uint8_t*)q_base;
        br.kv_base = (const uint8_t*)kv_base;
        br.q = (uint8_t*)ctx->q;
        br.kv = (uint8_t*)ctx->kv;   // layer 0's slot
        br.kv_stride = kv_stride;
        br.ab = (int)ab;
      }
      CK(assemble_block(actions, state0, ctx->w.W_a, ctx->w.b_a, ctx->w.W_s, ctx->w.b_s,
                        ctx->w.pos, k == 0 ? base : nullptr, ctx->x, (int)c0, nc, N, H, k, A, S,
                        P, d, br, s));
      for (int l = 0; l < L; ++l) {
        const LayerW& lw = ctx->w.layers[l];
        uint8_t* kv_slot = (uint8_t*)ctx->kv + (H > 1 ? (size_t)l * kv_slot_elems * ab : 0);
        const bool two_rows = shared0 && l == 0;   // rows 0 and 1 of every candidate only
        const int qkv_rows = two_rows ? nc * 2 : rows;
        CK(layernorm(ctx->x, two_rows ? RowMap{2, (long long)T, 0} : identity_map(), ctx->xn, ln_out,
                     lw.ln1_g, lw.ln1_b, qkv_rows, d, c.ln_eps, s, ctx->xs));
        {
          Epilogue e = epi_base(ctx, EPI_STORE);
          e.bias = lw.b_qkv;
          e.out0 = ctx->q;
          e.ld0 = d;
          e.split = d;
          e.out1 = kv_slot;
          e.ld1 = 2 * d;
          e.map0 = two_rows ? RowMap{2, (long long)T, 0} : identity_map();
          e.map1 = two_rows ? RowMap{2, kv_stride, 0} : RowMap{T, kv_stride, (long long)k * T};
          if (f8) {
            e.row_scale = ctx->xs;
            e.col_scale = lw.s_qkv;
          }
          if ((st = gemm(ctx, ctx->xn, f8 ? (const void*)lw.W_qkv8 : lw.W_qkv, qkv_rows, 3 * d, d, e,
                         s, prof, f8)))
            return st;
        }
        if (bf16_mode(ctx)) {
          CK(attention_tc_bf16((const bf16*)ctx->q, (const bf16*)kv_slot, (bf16*)ctx->o, nc, T,
                               (k + 1) * T, kv_stride, heads, d, ctx->dev_err, s));
        } else {
          CK(attention_f32((const float*)ctx->q, (const float*)kv_slot, (float*)ctx->o, nc, T,
                           (k + 1) * T, kv_stride, heads, d, s));
        }
        {
          Epilogue e = epi_base(ctx, EPI_RESID);
          e.bias = lw.b_o;
          e.out0 = ctx->x;
          e.ld0 = d;
          if ((st = gemm(ctx, ctx->o, lw.W_o, rows, d, d, e, s, prof))) return st;
        }
        CK(layernorm(ctx->x, identity_map(), ctx->xn, ln_out, lw.ln2_g, lw.ln2_b, rows, d,
                     c.ln_eps, s, ctx->xs));
        {
          const bool gated = c.mlp_kind == JEPA_MLP_GATED;
          Epilogue e = epi_base(ctx, gated ? EPI_GATED : EPI_GELU);
          e.bias = lw.b_1;
          e.out0 = ctx->hbuf;
          e.ld0 = m;
          if (f8) {
            e.row_scale = ctx->xs;
            e.col_scale = lw.s_1;
          }
          if ((st = gemm(ctx, ctx->xn, f8 ? (const void*)lw.W_18 : lw.W_1, rows, gated ? 2 * m : m, d,
                         e, s, prof, f8)))
            return st;
        }
        {
          Epilogue e = epi_base(ctx, EPI_RESID);
          e.bias = lw.b_2;
          e.out0 = ctx->x;
          e.ld0 = d;
          if ((st = gemm(ctx, ctx->hbuf, lw.W_2, rows, d, m, e, s, prof))) return st;
        }
      }
      // final LayerNorm on the patch rows of this block, then the out-projection to E
      CK(layernorm(ctx->x, RowMap{P, (long long)T, 2}, ctx->xn, ln_out, ctx->w.lnf_g,
                   ctx->w.lnf_b, nc * P, d, c.ln_eps, s, ctx->xs));
      {
        const bool last = (k == H - 1);
        Epilogue e = epi_base(ctx, EPI_OUTPROJ);
        e.bias = ctx->w.b_out;
        e.zpred = (last && z_pred) ? z_pred + c0 * P * (long long)E : nullptr;
        e.zhat = last ? nullptr : ctx->zhat;
        e.goal = (last && goal) ? goal : nullptr;
        e.P = P;
        e.cand0 = (int)c0;
        e.cands_per_problem = N;
        e.partial = ctx->partial;
        e.ntiles = ctx->ntiles;
        if (f8) {
          e.row_scale = ctx->xs;
          e.col_scale = ctx->w.s_out;
        }
        if ((st = gemm(ctx, ctx->xn, f8 ? (const void*)ctx->w.W_out8 : ctx->w.W_out, nc * P, E, d, e,
                       s, prof, f8)))
          return st;
      }
    }
    if (goal && energy)
      CK(energy_finalize(ctx->partial, P, ctx->ntiles, nc, 1.0f / ((float)P * E), energy + c0, s));
  }
  return JEPA_OK;
}

jepa_status check_ready(jepa_ctx* ctx) {
  if (!ctx) return JEPA_ERR_INVALID_ARG;
  if (!ctx->loaded) return fail(ctx, JEPA_ERR_NOT_LOADED, "weights not loaded");
  CK(cudaSetDevice(ctx->device));
  return JEPA_OK;
}

// The kernels of one planning step (all rounds), enqueued on s: captured once into the
// plan's graph, or launched directly when graphs are switched off.
jepa_status plan_body(jepa_ctx* ctx, PlanGraph* g, cudaStream_t s, PlanGraph* prof) {
  const int B = g->B, H = g->H, N = g->N, K = g->K, R = g->R;
  const int A = ctx->cfg.action_dim, HA = H * A;
  const size_t BN = (size_t)B * N;
  jepa_status s2;
  if ((s2 = context_projection(ctx, g->z0, g->z0_act, g->base, B, s, prof))) return s2;
  const bool shared = N > 1;
  if (shared && (s2 = base_qkv(ctx, g->base, B, g->xn_base, g->xs_base, g->q_base, g->kv_base, s,
                               prof)))
    return s2;
  // When one pass covers every candidate, its energy partials are all still in place when
  // the pass ends: one kernel then finalises the energies, selects and refits (the pass's
  // own finalisation is skipped).
  const bool fused = BN <= (size_t)ctx->ws_chunk;
  const jepa_config& c = ctx->cfg;
  for (int r = 0; r < R; ++r) {
    float* act_r = g->actions + (size_t)r * BN * HA;
    float* en_r = g->energy + (size_t)r * BN;
    CK(sample_actions(g->mu + (size_t)r * B * HA, g->sigma + (size_t)r * B * HA, B, N, H, A, r,
                      g->seed, 0, act_r, s));
    if ((s2 = predictor_pass(ctx, g->base, shared ? g->q_base : nullptr,
                             shared ? g->kv_base : nullptr, g->state0, act_r, B, N, H, g->goal,
                             nullptr, fused ? nullptr : en_r, s, prof)))
      return s2;
    if (fused) {
      CK(energy_select(ctx->partial, c.patch_tokens, ctx->ntiles, B, N,
                       1.0f / ((float)c.patch_tokens * c.embed_dim), en_r, act_r, HA, K,
                       g->mu + (size_t)(r + 1) * B * HA, g->sigma + (size_t)(r + 1) * B * HA,
                       g->elites + (size_t)r * B * K, g->winner, g->select_counter, s));
    } else {
      CK(select_refit(en_r, act_r, B, N, HA, K, g->mu + (size_t)(r + 1) * B * HA,
                      g->sigma + (size_t)(r + 1) * B * HA, g->elites + (size_t)r * B * K,
                      g->winner, s));
    }
  }
  CK(winner_action(g->actions + (size_t)(R - 1) * BN * HA, g->winner, B, N, HA, A,
                   g->action_out, s));
  return JEPA_OK;
}

jepa_status build_plan(jepa_ctx* ctx, int B, int H, int N, int K, int R, PlanGraph** out) {
  const auto key = std::make_tuple(B, H, N, K, R, ctx->profile);
  auto it = ctx->graphs.find(key);
  if (it != ctx->graphs.end()) {
    *out = it->second;
    return JEPA_OK;
  }
  const jepa_config& c = ctx->cfg;
  const int P = c.patch_tokens, E = c.embed_dim, A = c.action_dim, S = c.state_dim, d = c.width;
  const int HA = H * A;
  jepa_status st = ensure_workspace(ctx, chunk_for(ctx, (long long)B * N), H);
  if (st) return st;
  PlanGraph* g = new PlanGraph();
  g->B = B; g->H = H; g->N = N; g->K = K; g->R = R; g->profiled = ctx->profile;
  const size_t BN = (size_t)B * N;
  if ((st = dalloc(ctx, g->allocs, &g->z0, (size_t)B * P * E * 4)) ||
      (st = dalloc(ctx, g->allocs, &g->goal, (size_t)B * P * E * 4)) ||
      (st = dalloc(ctx, g->allocs, &g->state0, (size_t)B * S * 4)) ||
      (st = dalloc(ctx, g->allocs, &g->mu, (size_t)(R + 1) * B * HA * 4)) ||
      (st = dalloc(ctx, g->allocs, &g->sigma, (size_t)(R + 1) * B * HA * 4)) ||
      (st = dalloc(ctx, g->allocs, &g->actions, (size_t)R * BN * HA * 4)) ||
      (st = dalloc(ctx, g->allocs, &g->energy, (size_t)R * BN * 4)) ||
      (st = dalloc(ctx, g->allocs, &g->action_out, (size_t)B * A * 4)) ||
      (st = dalloc(ctx, g->allocs, &g->base, (size_t)B * P * d * 4)) ||
      (st = dalloc(ctx, g->allocs, &g->z0_act, (size_t)B * P * E * act_bytes(ctx))) ||
      (st = dalloc(ctx, g->allocs, &g->q_base, (size_t)B * P * d * act_bytes(ctx))) ||
      (st = dalloc(ctx, g->allocs, &g->kv_base, (size_t)B * P * 2 * d * act_bytes(ctx))) ||
      (st = dalloc(ctx, g->allocs, &g->xn_base, (size_t)B * P * d * act_bytes(ctx))) ||
      (st = dalloc(ctx, g->allocs, &g->xs_base, (size_t)B * P * 4)) ||
      (st = dalloc(ctx, g->allocs, &g->elites, (size_t)R * B * K * 4)) ||
      (st = dalloc(ctx, g->allocs, &g->winner, (size_t)B * 4)) ||
      (st = dalloc(ctx, g->allocs, &g->select_counter, (size_t)B * 4)) ||
      (st = dalloc(ctx, g->allocs, &g->seed, 8))) {
    free_plan(g);
    return st;
  }
  if (cudaMemset(g->select_counter, 0, (size_t)B * 4) != cudaSuccess) {
    free_plan(g);
    return fail(ctx, JEPA_ERR_CUDA, "plan: counter init failed");
  }
  PlanGraph* prof = ctx->profile ? g : nullptr;
  cudaStream_t s = ctx->cap_stream;
  cudaError_t ce = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
  auto body = [&]() { return plan_body(ctx, g, s, prof); };
  if (ce != cudaSuccess) {
    free_plan(g);
    return fail(ctx, JEPA_ERR_CUDA, "begin capture: %s", cudaGetErrorString(ce));
  }
  st = body();
  cudaGraph_t graph = nullptr;
  ce = cudaStreamEndCapture(s, &graph);
  if (st || ce != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();
    free_plan(g);
    if (st) return st;
    return fail(ctx, JEPA_ERR_CUDA, "end capture: %s", cudaGetErrorString(ce));
  }
  g->graph = graph;
  ce = cudaGraphInstantiate(&g->exec, graph, 0);
  if (ce != cudaSuccess) {
    free_plan(g);
    return fail(ctx, JEPA_ERR_CUDA, "graph instantiate: %s", cudaGetErrorString(ce));
  }
  size_t nn = 0;
  cudaGraphGetNodes(graph, nullptr, &nn);
  std::vector<cudaGraphNode_t> nodes(nn);
  cudaGraphGetNodes(graph, nodes.data(), &nn);
  for (auto n : nodes) {
    cudaGraphNodeType t;
    if (cudaGraphNodeGetType(n, &t) == cudaSuccess && t == cudaGraphNodeTypeKernel) g->kernels++;
  }
  ctx->graphs[key] = g;
  *out = g;
  return JEPA_OK;
}

bool bad_ptr(const void* p) { return p == nullptr; }

}  // namespace

// =====================================================================================
extern "C" {

const char* jepa_status_string(jepa_status s) {
  switch (s) {
    case JEPA_OK: return "ok";
    case JEPA_ERR_INVALID_ARG: return "invalid argument";
    case JEPA_ERR_SHAPE: return "shape not supported by this context";
    case JEPA_ERR_NOT_LOADED: return "weights not loaded";
    case JEPA_ERR_OOM: return "device out of memory";
    case JEPA_ERR_CUDA: return "CUDA error";
    case JEPA_ERR_TIMEOUT: return "device wait timed out";
    case JEPA_ERR_UNSUPPORTED: return "unsupported device";
  }
  return "unknown status";
}

size_t jepa_weight_blob_bytes(const jepa_config* cfg) {
  if (validate_config(cfg) != JEPA_OK) return 0;
  return kHeaderBytes + blob_floats(cfg) * sizeof(float);
}

jepa_status jepa_create(const jepa_config* cfg, int device, jepa_ctx** out) {
  if (!out) return JEPA_ERR_INVALID_ARG;
  *out = nullptr;
  jepa_status vs = validate_config(cfg);
  if (vs) return vs;
  jepa_ctx* ctx = new jepa_ctx();
  ctx->cfg = *cfg;
  ctx->device = device;
  cudaDeviceProp prop;
  cudaError_t e = cudaGetDeviceProperties(&prop, device);
  if (e != cudaSuccess) {
    cudaGetLastError();
    delete ctx;
    return JEPA_ERR_CUDA;
  }
  if (!(prop.major == 10 && prop.minor == 3)) {
    delete ctx;
    return JEPA_ERR_UNSUPPORTED;
  }
  ctx->num_sms = prop.multiProcessorCount;
  if (cudaSetDevice(device) != cudaSuccess ||
      cudaStreamCreateWithFlags(&ctx->cap_stream, cudaStreamNonBlocking) != cudaSuccess ||
      cudaMalloc(&ctx->dev_err, sizeof(int)) != cudaSuccess ||
      cudaMemset(ctx->dev_err, 0, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    jepa_destroy(ctx);
    return JEPA_ERR_CUDA;
  }
  *out = ctx;
  return JEPA_OK;
}

void jepa_destroy(jepa_ctx* ctx) {
  if (!ctx) return;
  cudaSetDevice(ctx->device);
  drop_graphs(ctx);
  free_list(ctx->ws_allocs);
  free_list(ctx->ep_allocs);
  if (ctx->w.f32) cudaFree(ctx->w.f32);
  if (ctx->w.mats) cudaFree(ctx->w.mats);
  if (ctx->w.gmat) cudaFree(ctx->w.gmat);
  if (ctx->w.gbias) cudaFree(ctx->w.gbias);
  if (ctx->w.q8) cudaFree(ctx->w.q8);
  if (ctx->w.q8s) cudaFree(ctx->w.q8s);
  free_list(ctx->fw_allocs);
  if (ctx->dev_err) cudaFree(ctx->dev_err);
  if (ctx->cap_stream) cudaStreamDestroy(ctx->cap_stream);
  delete ctx;
}

const char* jepa_last_error(const jepa_ctx* ctx) { return ctx ? ctx->err.c_str() : ""; }

jepa_status jepa_load_weights(jepa_ctx* ctx, const void* host_blob, size_t bytes) {
  if (!ctx || !host_blob) return fail(ctx, JEPA_ERR_INVALID_ARG, "null argument");
  CK(cudaSetDevice(ctx->device));
  const jepa_config& c = ctx->cfg;
  const size_t nf = blob_floats(&c);
  if (bytes != kHeaderBytes + nf * 4)
    return fail(ctx, JEPA_ERR_SHAPE, "blob has %zu bytes, config needs %zu", bytes,
                kHeaderBytes + nf * 4);
  int32_t hdr[16];
  memcpy(hdr, host_blob, sizeof hdr);
  const int32_t want[11] = {kMagic, 1, c.layers, c.width, c.heads, c.mlp, c.patch_tokens,
                            c.embed_dim, c.action_dim, c.state_dim, c.mlp_kind};
  for (int i = 0; i < 11; ++i)
    if (hdr[i] != want[i])
      return fail(ctx, JEPA_ERR_SHAPE, "blob header field %d is %d, expected %d", i, hdr[i], want[i]);
  const float* src = (const float*)((const uint8_t*)host_blob + kHeaderBytes);
  Weights w;
  float* f32 = nullptr;
  CK(cudaMalloc(&f32, nf * 4));
  cudaError_t e = cudaMemcpy(f32, src, nf * 4, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(f32);
    return fail(ctx, JEPA_ERR_CUDA, "weight upload: %s", cudaGetErrorString(e));
  }
  w.f32 = f32;
  const size_t d = c.width, m = c.mlp, E = c.embed_dim, A = c.action_dim, S = c.state_dim,
               T = c.patch_tokens + 2;
  // walk the canonical order; record fp32 offsets of the matrices for bf16 conversion
  size_t off = 0;
  std::vector<std::pair<size_t, size_t>> mats;  // (offset, count)
  auto take = [&](size_t n) {
    const float* p = f32 + off;
    off += n;
    return p;
  };
  auto take_mat = [&](size_t n) {
    mats.push_back({off, n});
    return take(n);
  };
  const float* W_in = take_mat(d * E);
  w.b_in = take(d);
  w.W_a = take(d * A);
  w.b_a = take(d);
  w.W_s = take(d * S);
  w.b_s = take(d);
  w.pos = take(T * d);
  const bool gated = c.mlp_kind == JEPA_MLP_GATED;
  std::vector<const float*> lm;  // per layer: W_qkv, W_o, W_1, W_2 (fp32)
  std::vector<const float*> g_w1, g_b1, g_wg, g_bg;  // gated: the two branches, fp32
  for (int l = 0; l < c.layers; ++l) {
    LayerW L;
    L.ln1_g = take(d);
    L.ln1_b = take(d);
    lm.push_back(take_mat(3 * d * d));
    L.b_qkv = take(3 * d);
    lm.push_back(take_mat(d * d));
    L.b_o = take(d);
    L.ln2_g = take(d);
    L.ln2_b = take(d);
    if (gated) {
      lm.push_back(take(m * d));
      L.b_1 = take(m);
      g_w1.push_back(lm.back());
      g_b1.push_back(L.b_1);
      g_wg.push_back(take(m * d));
      g_bg.push_back(take(m));
    } else {
      lm.push_back(take_mat(m * d));
      L.b_1 = take(m);
    }
    lm.push_back(take_mat(d * m));
    L.b_2 = take(d);
    w.layers.push_back(L);
  }
  w.lnf_g = take(d);
  w.lnf_b = take(d);
  const float* W_out = take_mat(E * d);
  w.b_out = take(E);
  if (bf16_mode(ctx)) {
    size_t total = 0;
    for (auto& p : mats) total += p.second;
    bf16* mb = nullptr;
    e = cudaMalloc(&mb, total * 2);
    if (e != cudaSuccess) {
      cudaFree(f32);
      cudaGetLastError();
      return fail(ctx, JEPA_ERR_OOM, "bf16 weights: %s", cudaGetErrorString(e));
    }
    w.mats = mb;
    std::map<size_t, const bf16*> conv;
    size_t moff = 0;
    for (auto& p : mats) {
      e = convert_f32_bf16(f32 + p.first, mb + moff, (long long)p.second, 0);
      conv[p.first] = mb + moff;
      moff += p.second;
      if (e != cudaSuccess) break;
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
      cudaFree(f32);
      cudaFree(mb);
      return fail(ctx, JEPA_ERR_CUDA, "bf16 conversion: %s", cudaGetErrorString(e));
    }
    w.W_in = conv[(size_t)(W_in - f32)];
    w.W_out = conv[(size_t)(W_out - f32)];
    for (int l = 0; l < c.layers; ++l) {
      w.layers[l].W_qkv = conv[(size_t)(lm[4 * l] - f32)];
      w.layers[l].W_o = conv[(size_t)(lm[4 * l + 1] - f32)];
      if (!gated) w.layers[l].W_1 = conv[(size_t)(lm[4 * l + 2] - f32)];
      w.layers[l].W_2 = conv[(size_t)(lm[4 * l + 3] - f32)];
    }
  } else {
    w.W_in = W_in;
    w.W_out = W_out;
    for (int l = 0; l < c.layers; ++l) {
      w.layers[l].W_qkv = lm[4 * l];
      w.layers[l].W_o = lm[4 * l + 1];
      w.layers[l].W_1 = lm[4 * l + 2];
      w.layers[l].W_2 = lm[4 * l + 3];
    }
  }
  // fp8 mode: e4m3 codes with per-output-channel scales for the LayerNorm-fed GEMMs, per
  // layer [W_qkv | W_1 (or the interleaved gated pair)], then W_out
  const size_t mrows = gated ? 2 * m : m;
  const size_t q8_layer = (3 * d + mrows) * d, q8s_layer = 3 * d + mrows;
  if (fp8_mode(ctx)) {
    e = cudaMalloc(&w.q8, c.layers * q8_layer + E * d);
    if (e == cudaSuccess) e = cudaMalloc(&w.q8s, (c.layers * q8s_layer + E) * 4);
    for (int l = 0; l < c.layers && e == cudaSuccess; ++l) {
      uint8_t* q = w.q8 + l * q8_layer;
      float* qs = w.q8s + l * q8s_layer;
      e = quantize_rows_fp8(lm[4 * l], 3 * d, (int)d, q, qs, 0);
      if (e == cudaSuccess && !gated) e = quantize_rows_fp8(lm[4 * l + 2], m, (int)d, q + 3 * d * d, qs + 3 * d, 0);
      w.layers[l].W_qkv8 = q;
      w.layers[l].s_qkv = qs;
      w.layers[l].W_18 = q + 3 * d * d;
      w.layers[l].s_1 = qs + 3 * d;
    }
    if (e == cudaSuccess)
      e = quantize_rows_fp8(W_out, E, (int)d, w.q8 + c.layers * q8_layer, w.q8s + c.layers * q8s_layer, 0);
    w.W_out8 = w.q8 + c.layers * q8_layer;
    w.s_out = w.q8s + c.layers * q8s_layer;
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
      cudaGetLastError();
      cudaFree(f32);
      if (w.mats) cudaFree(w.mats);
      if (w.q8) cudaFree(w.q8);
      if (w.q8s) cudaFree(w.q8s);
      return fail(ctx, JEPA_ERR_CUDA, "fp8 weights: %s", cudaGetErrorString(e));
    }
  }
  if (gated) {
    // one up-projection GEMM per layer over [FC1 | gate] rows interleaved in blocks of 32
    // (2-D copies on the device), converted to bf16 in bf16 mode
    const size_t nmat = 2 * m * d, nb = 2 * m;
    float* tmp = nullptr;
    e = cudaMalloc(&w.gbias, c.layers * nb * 4);
    if (e == cudaSuccess) e = cudaMalloc(&w.gmat, c.layers * nmat * (bf16_mode(ctx) ? 2 : 4));
    if (e == cudaSuccess && bf16_mode(ctx)) e = cudaMalloc(&tmp, nmat * 4);
    for (int l = 0; l < c.layers && e == cudaSuccess; ++l) {
      float* dm = bf16_mode(ctx) ? tmp : (float*)w.gmat + l * nmat;
      float* db = w.gbias + l * nb;
      const size_t row = d * 4;
      e = cudaMemcpy2D(dm, 64 * row, g_w1[l], 32 * row, 32 * row, m / 32, cudaMemcpyDeviceToDevice);
      if (e == cudaSuccess)
        e = cudaMemcpy2D(dm + 32 * d, 64 * row, g_wg[l], 32 * row, 32 * row, m / 32,
                         cudaMemcpyDeviceToDevice);
      if (e == cudaSuccess)
        e = cudaMemcpy2D(db, 64 * 4, g_b1[l], 32 * 4, 32 * 4, m / 32, cudaMemcpyDeviceToDevice);
      if (e == cudaSuccess)
        e = cudaMemcpy2D(db + 32, 64 * 4, g_bg[l], 32 * 4, 32 * 4, m / 32,
                         cudaMemcpyDeviceToDevice);
      if (e == cudaSuccess && bf16_mode(ctx))
        e = convert_f32_bf16(tmp, (bf16*)w.gmat + l * nmat, (long long)nmat, 0);
      if (e == cudaSuccess && fp8_mode(ctx))
        e = quantize_rows_fp8(tmp, 2 * m, (int)d, w.q8 + l * q8_layer + 3 * d * d,
                              w.q8s + l * q8s_layer + 3 * d, 0);
      if (e == cudaSuccess && bf16_mode(ctx)) e = cudaDeviceSynchronize();  // tmp is reused
      if (e == cudaSuccess) {
        w.layers[l].W_1 = bf16_mode(ctx) ? (const void*)((bf16*)w.gmat + l * nmat)
                                         : (const void*)((float*)w.gmat + l * nmat);
        w.layers[l].b_1 = db;
      }
    }
    if (tmp) cudaFree(tmp);
    if (e != cudaSuccess) {
      cudaGetLastError();
      cudaFree(f32);
      if (w.mats) cudaFree(w.mats);
      if (w.gmat) cudaFree(w.gmat);
      if (w.gbias) cudaFree(w.gbias);
      if (w.q8) cudaFree(w.q8);
      if (w.q8s) cudaFree(w.q8s);
      return fail(ctx, JEPA_ERR_CUDA, "gated MLP weights: %s", cudaGetErrorString(e));
    }
  }
  drop_graphs(ctx);  // captured graphs hold the old weight pointers
  if (ctx->w.f32) cudaFree(ctx->w.f32);
  if (ctx->w.mats) cudaFree(ctx->w.mats);
  if (ctx->w.gmat) cudaFree(ctx->w.gmat);
  if (ctx->w.gbias) cudaFree(ctx->w.gbias);
  if (ctx->w.q8) cudaFree(ctx->w.q8);
  if (ctx->w.q8s) cudaFree(ctx->w.q8s);
  ctx->w = w;
  ctx->loaded = true;
  return JEPA_OK;
}

jepa_status jepa_sample_actions(jepa_ctx* ctx, const float* mu, const float* sigma, int B, int N,
                                int H, int round, uint64_t seed, float* actions, void* stream) {
  if (!ctx) return JEPA_ERR_INVALID_ARG;
  if (bad_ptr(mu) || bad_ptr(sigma) || bad_ptr(actions) || B < 1 || N < 1 || H < 1 || round < 0 ||
      H > ctx->cfg.max_horizon)
    return fail(ctx, JEPA_ERR_INVALID_ARG, "sample_actions: bad argument");
  CK(cudaSetDevice(ctx->device));
  CK(sample_actions(mu, sigma, B, N, H, ctx->cfg.action_dim, round, nullptr, seed, actions,
                    (cudaStream_t)stream));
  return JEPA_OK;
}

jepa_status jepa_philox4x32_10(jepa_ctx* ctx, const uint32_t* counters, uint64_t seed, int n,
                               uint32_t* out, void* stream) {
  if (!ctx) return JEPA_ERR_INVALID_ARG;
  if (bad_ptr(counters) || bad_ptr(out) || n < 1 || (((uintptr_t)counters) & 15) ||
      (((uintptr_t)out) & 15))
    return fail(ctx, JEPA_ERR_INVALID_ARG, "philox: bad argument (pointers must be 16-byte aligned)");
  CK(cudaSetDevice(ctx->device));
  CK(philox_raw(counters, seed, n, out, (cudaStream_t)stream));
  return JEPA_OK;
}

jepa_status jepa_predictor_forward(jepa_ctx* ctx, const float* z_ctx, const float* state0,
                                   const float* actions, int B, int N, int H, const float* goal,
                                   float* z_pred, float* energy, void* stream) {
  jepa_status st = check_ready(ctx);
  if (st) return st;
  if (bad_ptr(z_ctx) || bad_ptr(state0) || bad_ptr(actions) || B < 1 || N < 1 || H < 1 ||
      (energy && !goal) || (!z_pred && !energy))
    return fail(ctx, JEPA_ERR_INVALID_ARG, "predictor_forward: bad argument");
  if (H > ctx->cfg.max_horizon) return fail(ctx, JEPA_ERR_SHAPE, "H > max_horizon");
  if ((long long)B * N > (1LL << 30)) return fail(ctx, JEPA_ERR_SHAPE, "too many candidates");
  const jepa_config& c = ctx->cfg;
  if ((st = ensure_workspace(ctx, chunk_for(ctx, (long long)B * N), H))) return st;
  if ((size_t)B > ctx->fw_cap) {
    CK(cudaDeviceSynchronize());
    free_list(ctx->fw_allocs);
    ctx->fw_cap = 0;
    const size_t BP = (size_t)B * c.patch_tokens, d = c.width, ab = act_bytes(ctx);
    if ((st = dalloc(ctx, ctx->fw_allocs, &ctx->fw_base, BP * d * 4)) ||
        (st = dalloc(ctx, ctx->fw_allocs, &ctx->fw_z, BP * c.embed_dim * ab)) ||
        (st = dalloc(ctx, ctx->fw_allocs, &ctx->fw_qb, BP * d * ab)) ||
        (st = dalloc(ctx, ctx->fw_allocs, &ctx->fw_kvb, BP * 2 * d * ab)) ||
        (st = dalloc(ctx, ctx->fw_allocs, &ctx->fw_xnb, BP * d * ab)) ||
        (st = dalloc(ctx, ctx->fw_allocs, &ctx->fw_xsb, BP * 4))) {
      free_list(ctx->fw_allocs);
      return st;
    }
    ctx->fw_cap = B;
  }
  cudaStream_t s = (cudaStream_t)stream;
  if ((st = context_projection(ctx, z_ctx, ctx->fw_z, ctx->fw_base, B, s, nullptr))) return st;
  // with a single candidate per problem nothing is shared: the plain pass does the same work
  const bool shared = N > 1;
  if (shared && (st = base_qkv(ctx, ctx->fw_base, B, ctx->fw_xnb, ctx->fw_xsb, ctx->fw_qb,
                               ctx->fw_kvb, s, nullptr)))
    return st;
  return predictor_pass(ctx, ctx->fw_base, shared ? ctx->fw_qb : nullptr,
                        shared ? ctx->fw_kvb : nullptr, state0, actions, B, N, H, goal, z_pred,
                        energy, s, nullptr);
}

jepa_status jepa_cem_select_refit(jepa_ctx* ctx, const float* energy, const float* actions, int B,
                                  int N, int H, int K, float* mu_out, float* sigma_out,
                                  int32_t* elites_out, void* stream) {
  if (!ctx) return JEPA_ERR_INVALID_ARG;
  if (bad_ptr(energy) || bad_ptr(actions) || bad_ptr(mu_out) || bad_ptr(sigma_out) || B < 1 ||
      N < 1 || H < 1 || K < 1 || K > N)
    return fail(ctx, JEPA_ERR_INVALID_ARG, "select_refit: bad argument");
  if (N > kMaxSelectN) return fail(ctx, JEPA_ERR_SHAPE, "N > %d", kMaxSelectN);
  CK(cudaSetDevice(ctx->device));
  CK(select_refit(energy, actions, B, N, H * ctx->cfg.action_dim, K, mu_out, sigma_out,
                  (int*)elites_out, nullptr, (cudaStream_t)stream));
  return JEPA_OK;
}

static jepa_status plan_args(jepa_ctx* ctx, int B, int H, int N, int K, int rounds) {
  if (B < 1 || N < 1 || H < 1 || K < 1 || K > N || rounds < 1)
    return fail(ctx, JEPA_ERR_INVALID_ARG, "plan: need B,N,H,rounds >= 1 and 1 <= K <= N");
  if (H > ctx->cfg.max_horizon) return fail(ctx, JEPA_ERR_SHAPE, "H > max_horizon");
  if (N > kMaxSelectN) return fail(ctx, JEPA_ERR_SHAPE, "N > %d", kMaxSelectN);
  if ((long long)B * N > (1LL << 30)) return fail(ctx, JEPA_ERR_SHAPE, "too many candidates");
  return JEPA_OK;
}

jepa_status jepa_cem_plan(jepa_ctx* ctx, const float* z0, const float* state0, const float* goal,
                          const float* mu0, const float* sigma0, int B, int H, int N, int K,
                          int rounds, uint64_t seed, float* action_out,
                          const jepa_cem_trace* trace, void* stream) {
  jepa_status st = check_ready(ctx);
  if (st) return st;
  if (bad_ptr(z0) || bad_ptr(state0) || bad_ptr(goal) || bad_ptr(mu0) || bad_ptr(sigma0) ||
      bad_ptr(action_out))
    return fail(ctx, JEPA_ERR_INVALID_ARG, "plan: null pointer");
  if ((st = plan_args(ctx, B, H, N, K, rounds))) return st;
  PlanGraph* g = nullptr;
  if ((st = build_plan(ctx, B, H, N, K, rounds, &g))) return st;
  const jepa_config& c = ctx->cfg;
  const size_t PE = (size_t)c.patch_tokens * c.embed_dim, HA = (size_t)H * c.action_dim;
  cudaStream_t s = (cudaStream_t)stream;
  CK(cudaMemcpyAsync(g->z0, z0, B * PE * 4, cudaMemcpyDefault, s));
  CK(cudaMemcpyAsync(g->goal, goal, B * PE * 4, cudaMemcpyDefault, s));
  CK(cudaMemcpyAsync(g->state0, state0, (size_t)B * c.state_dim * 4, cudaMemcpyDefault, s));
  CK(cudaMemcpyAsync(g->mu, mu0, B * HA * 4, cudaMemcpyDefault, s));
  CK(cudaMemcpyAsync(g->sigma, sigma0, B * HA * 4, cudaMemcpyDefault, s));
  CK(set_u64(g->seed, seed, s));
  if (ctx->use_graphs) {
    CK(cudaGraphLaunch(g->exec, s));
  } else if ((st = plan_body(ctx, g, s, nullptr))) {
    return st;
  }
  CK(cudaMemcpyAsync(action_out, g->action_out, (size_t)B * c.action_dim * 4, cudaMemcpyDefault, s));
  if (trace) {
    const size_t BN = (size_t)B * N, R = rounds;
    if (trace->mu)
      CK(cudaMemcpyAsync(trace->mu, g->mu, (R + 1) * B * HA * 4, cudaMemcpyDefault, s));
    if (trace->sigma)
      CK(cudaMemcpyAsync(trace->sigma, g->sigma, (R + 1) * B * HA * 4, cudaMemcpyDefault, s));
    if (trace->actions)
      CK(cudaMemcpyAsync(trace->actions, g->actions, R * BN * HA * 4, cudaMemcpyDefault, s));
    if (trace->energy)
      CK(cudaMemcpyAsync(trace->energy, g->energy, R * BN * 4, cudaMemcpyDefault, s));
    if (trace->elites)
      CK(cudaMemcpyAsync(trace->elites, g->elites, R * B * (size_t)K * 4, cudaMemcpyDefault, s));
    if (trace->winner)
      CK(cudaMemcpyAsync(trace->winner, g->winner, (size_t)B * 4, cudaMemcpyDefault, s));
  }
  ctx->last_plan = g;
  return JEPA_OK;
}

jepa_status jepa_cem_warm_start(jepa_ctx* ctx, const float* mu_prev, const float* mu_prior,
                                const float* sigma_prior, int B, int H, float* mu_out,
                                float* sigma_out, void* stream) {
  if (!ctx) return JEPA_ERR_INVALID_ARG;
  if (bad_ptr(mu_prev) || bad_ptr(mu_prior) || bad_ptr(sigma_prior) || bad_ptr(mu_out) ||
      bad_ptr(sigma_out) || B < 1 || H < 1)
    return fail(ctx, JEPA_ERR_INVALID_ARG, "warm_start: bad argument");
  if ((long long)B * H * ctx->cfg.action_dim > (1LL << 30))
    return fail(ctx, JEPA_ERR_SHAPE, "warm_start: too large");
  CK(cudaSetDevice(ctx->device));
  CK(warm_start(mu_prev, mu_prior, sigma_prior, B, H, ctx->cfg.action_dim, mu_out, sigma_out,
                (cudaStream_t)stream));
  return JEPA_OK;
}

jepa_status jepa_world_model_step(jepa_ctx* ctx, const float* z, const float* state,
                                  const float* action, int B, const float* goal, float* z_next,
                                  float* state_next, float* distance, void* stream) {
  jepa_status st = check_ready(ctx);
  if (st) return st;
  if (bad_ptr(z) || bad_ptr(state) || bad_ptr(action) || bad_ptr(z_next) || bad_ptr(state_next) ||
      B < 1 || (distance && !goal) || z_next == z)
    return fail(ctx, JEPA_ERR_INVALID_ARG, "world_model_step: bad argument");
  // the predicted frame first: it reads `state`, which state_next may overwrite
  if ((st = jepa_predictor_forward(ctx, z, state, action, B, 1, 1, goal, z_next, distance,
                                   stream)))
    return st;
  CK(state_step(state, action, B * ctx->cfg.state_dim, state_next, (cudaStream_t)stream));
  return JEPA_OK;
}

jepa_status jepa_cem_closed_loop(jepa_ctx* ctx, const float* z0, const float* state0,
                                 const float* goal, const float* mu_prior,
                                 const float* sigma_prior, int B, int H, int N, int K, int rounds,
                                 int steps, int warm, uint64_t seed, float* actions_out,
                                 float* distance_out, void* stream) {
  jepa_status st = check_ready(ctx);
  if (st) return st;
  if (bad_ptr(z0) || bad_ptr(state0) || bad_ptr(goal) || bad_ptr(mu_prior) ||
      bad_ptr(sigma_prior) || bad_ptr(actions_out) || bad_ptr(distance_out) || steps < 1 ||
      (warm != 0 && warm != 1))
    return fail(ctx, JEPA_ERR_INVALID_ARG, "closed_loop: bad argument");
  if ((st = plan_args(ctx, B, H, N, K, rounds))) return st;
  const jepa_config& c = ctx->cfg;
  const size_t PE = (size_t)c.patch_tokens * c.embed_dim, A = c.action_dim, S = c.state_dim;
  const size_t HA = (size_t)H * A;
  if (B > ctx->ep_B || H > ctx->ep_H || rounds > ctx->ep_R) {
    const int nB = B > ctx->ep_B ? B : ctx->ep_B, nH = H > ctx->ep_H ? H : ctx->ep_H;
    const int nR = rounds > ctx->ep_R ? rounds : ctx->ep_R;
    CK(cudaDeviceSynchronize());
    free_list(ctx->ep_allocs);
    ctx->ep_B = ctx->ep_H = ctx->ep_R = 0;
    const size_t nHA = (size_t)nH * A;
    if ((st = dalloc(ctx, ctx->ep_allocs, &ctx->ep_z[0], nB * PE * 4)) ||
        (st = dalloc(ctx, ctx->ep_allocs, &ctx->ep_z[1], nB * PE * 4)) ||
        (st = dalloc(ctx, ctx->ep_allocs, &ctx->ep_s[0], nB * S * 4)) ||
        (st = dalloc(ctx, ctx->ep_allocs, &ctx->ep_s[1], nB * S * 4)) ||
        (st = dalloc(ctx, ctx->ep_allocs, &ctx->ep_goal, nB * PE * 4)) ||
        (st = dalloc(ctx, ctx->ep_allocs, &ctx->ep_mu_prior, nB * nHA * 4)) ||
        (st = dalloc(ctx, ctx->ep_allocs, &ctx->ep_sg_prior, nB * nHA * 4)) ||
        (st = dalloc(ctx, ctx->ep_allocs, &ctx->ep_mu0, nB * nHA * 4)) ||
        (st = dalloc(ctx, ctx->ep_allocs, &ctx->ep_sg0, nB * nHA * 4)) ||
        (st = dalloc(ctx, ctx->ep_allocs, &ctx->ep_mu_trace, (nR + 1) * nB * nHA * 4)) ||
        (st = dalloc(ctx, ctx->ep_allocs, &ctx->ep_a, nB * A * 4)) ||
        (st = dalloc(ctx, ctx->ep_allocs, &ctx->ep_dist, nB * 4))) {
      free_list(ctx->ep_allocs);
      return st;
    }
    ctx->ep_B = nB;
    ctx->ep_H = nH;
    ctx->ep_R = nR;
  }
  cudaStream_t s = (cudaStream_t)stream;
  CK(cudaMemcpyAsync(ctx->ep_z[0], z0, B * PE * 4, cudaMemcpyDefault, s));
  CK(cudaMemcpyAsync(ctx->ep_s[0], state0, B * S * 4, cudaMemcpyDefault, s));
  CK(cudaMemcpyAsync(ctx->ep_goal, goal, B * PE * 4, cudaMemcpyDefault, s));
  CK(cudaMemcpyAsync(ctx->ep_mu_prior, mu_prior, B * HA * 4, cudaMemcpyDefault, s));
  CK(cudaMemcpyAsync(ctx->ep_sg_prior, sigma_prior, B * HA * 4, cudaMemcpyDefault, s));
  jepa_cem_trace tr;
  memset(&tr, 0, sizeof tr);
  tr.mu = ctx->ep_mu_trace;
  for (int t = 0; t < steps; ++t) {
    const int cur = t & 1, nxt = cur ^ 1;
    const bool from_prior = t == 0 || !warm;
    if (!from_prior)
      CK(warm_start(ctx->ep_mu_trace + (size_t)rounds * B * HA, ctx->ep_mu_prior,
                    ctx->ep_sg_prior, B, H, (int)A, ctx->ep_mu0, ctx->ep_sg0, s));
    if ((st = jepa_cem_plan(ctx, ctx->ep_z[cur], ctx->ep_s[cur], ctx->ep_goal,
                            from_prior ? ctx->ep_mu_prior : ctx->ep_mu0,
                            from_prior ? ctx->ep_sg_prior : ctx->ep_sg0, B, H, N, K, rounds,
                            seed + (uint64_t)t, ctx->ep_a, &tr, stream)))
      return st;
    if ((st = jepa_world_model_step(ctx, ctx->ep_z[cur], ctx->ep_s[cur], ctx->ep_a, B,
                                    ctx->ep_goal, ctx->ep_z[nxt], ctx->ep_s[nxt], ctx->ep_dist,
                                    stream)))
      return st;
    CK(cudaMemcpyAsync(actions_out + (size_t)t * B * A, ctx->ep_a, B * A * 4, cudaMemcpyDefault,
                       s));
    CK(cudaMemcpyAsync(distance_out + (size_t)t * B, ctx->ep_dist, (size_t)B * 4,
                       cudaMemcpyDefault, s));
  }
  return JEPA_OK;
}

jepa_status jepa_plan_kernel_count(jepa_ctx* ctx, int B, int H, int N, int K, int rounds,
                                   int64_t* count) {
  jepa_status st = check_ready(ctx);
  if (st) return st;
  if (!count) return fail(ctx, JEPA_ERR_INVALID_ARG, "null count");
  if ((st = plan_args(ctx, B, H, N, K, rounds))) return st;
  PlanGraph* g = nullptr;
  if ((st = build_plan(ctx, B, H, N, K, rounds, &g))) return st;
  *count = g->kernels + 1;  // + the seed-setting kernel launched before the graph
  return JEPA_OK;
}

jepa_status jepa_linear_bf16(jepa_ctx* ctx, const uint16_t* A, const uint16_t* W,
                             const float* bias, int M, int N, int K, int gelu, float* out,
                             void* stream) {
  if (!ctx) return JEPA_ERR_INVALID_ARG;
  if (!bf16_mode(ctx)) return fail(ctx, JEPA_ERR_UNSUPPORTED, "linear_bf16 needs a bf16 context");
  if (bad_ptr(A) || bad_ptr(W) || bad_ptr(out) || M < 1 || N < 1 || K < 8 || K % 8)
    return fail(ctx, JEPA_ERR_INVALID_ARG, "linear_bf16: bad argument");
  if ((((uintptr_t)A) & 15) || (((uintptr_t)W) & 15))
    return fail(ctx, JEPA_ERR_INVALID_ARG, "linear_bf16: A and W must be 16-byte aligned");
  if (gelu < 0 || gelu > 2 || (gelu == 2 && (N % 256 != 0 || !bias)))
    return fail(ctx, JEPA_ERR_INVALID_ARG, "linear_bf16: gated mode needs N %% 256 == 0 and a bias");
  CK(cudaSetDevice(ctx->device));
  Epilogue e = epi_base(ctx, gelu == 2 ? EPI_GATED : gelu ? EPI_GELU : EPI_STORE);
  e.act_bf16 = 0;
  e.bias = bias;
  e.out0 = out;
  e.ld0 = gelu == 2 ? N / 2 : N;
  CK(gemm_tc_bf16((const bf16*)A, (const bf16*)W, M, N, K, e, ctx->dev_err, ctx->num_sms,
                  (cudaStream_t)stream));
  return JEPA_OK;
}

jepa_status jepa_linear_resid_bf16(jepa_ctx* ctx, const uint16_t* A, const uint16_t* W,
                                   const float* bias, int M, int N, int K, float* x,
                                   void* stream) {
  if (!ctx) return JEPA_ERR_INVALID_ARG;
  if (!bf16_mode(ctx)) return fail(ctx, JEPA_ERR_UNSUPPORTED, "linear_resid_bf16 needs a bf16 context");
  if (bad_ptr(A) || bad_ptr(W) || bad_ptr(x) || M < 1 || N < 4 || N % 4 || K < 8 || K % 8)
    return fail(ctx, JEPA_ERR_INVALID_ARG, "linear_resid_bf16: bad argument");
  if ((((uintptr_t)A) & 15) || (((uintptr_t)W) & 15) || (((uintptr_t)x) & 15))
    return fail(ctx, JEPA_ERR_INVALID_ARG, "linear_resid_bf16: A, W and x must be 16-byte aligned");
  CK(cudaSetDevice(ctx->device));
  Epilogue e = epi_base(ctx, EPI_RESID);
  e.bias = bias;
  e.out0 = x;
  e.ld0 = N;
  CK(gemm_tc_bf16((const bf16*)A, (const bf16*)W, M, N, K, e, ctx->dev_err, ctx->num_sms,
                  (cudaStream_t)stream));
  return JEPA_OK;
}

jepa_status jepa_linear_qkv_bf16(jepa_ctx* ctx, const uint16_t* A, const uint16_t* W,
                                 const float* bias, int M, int d, int K, int T, int kv_rows,
                                 int frame, uint16_t* q, uint16_t* kv, void* stream) {
  if (!ctx) return JEPA_ERR_INVALID_ARG;
  if (!bf16_mode(ctx)) return fail(ctx, JEPA_ERR_UNSUPPORTED, "linear_qkv_bf16 needs a bf16 context");
  if (bad_ptr(A) || bad_ptr(W) || bad_ptr(q) || bad_ptr(kv) || M < 1 || d < 32 || d % 32 ||
      K < 8 || K % 8 || T < 1 || frame < 0 || (long long)(frame + 1) * T > kv_rows)
    return fail(ctx, JEPA_ERR_INVALID_ARG, "linear_qkv_bf16: bad argument");
  if ((((uintptr_t)A) & 15) || (((uintptr_t)W) & 15))
    return fail(ctx, JEPA_ERR_INVALID_ARG, "linear_qkv_bf16: A and W must be 16-byte aligned");
  CK(cudaSetDevice(ctx->device));
  Epilogue e = epi_base(ctx, EPI_STORE);
  e.bias = bias;
  e.out0 = q;
  e.ld0 = d;
  e.split = d;
  e.out1 = kv;
  e.ld1 = 2 * d;
  e.map1 = RowMap{T, (long long)kv_rows, (long long)frame * T};
  CK(gemm_tc_bf16((const bf16*)A, (const bf16*)W, M, 3 * d, K, e, ctx->dev_err, ctx->num_sms,
                  (cudaStream_t)stream));
  return JEPA_OK;
}

jepa_status jepa_linear_fp8(jepa_ctx* ctx, const uint8_t* A, const float* a_scale,
                            const uint8_t* W, const float* w_scale, const float* bias, int M,
                            int N, int K, int gelu, float* out, void* stream) {
  if (!ctx) return JEPA_ERR_INVALID_ARG;
  if (!bf16_mode(ctx)) return fail(ctx, JEPA_ERR_UNSUPPORTED, "linear_fp8 needs a bf16 or fp8 context");
  if (bad_ptr(A) || bad_ptr(a_scale) || bad_ptr(W) || bad_ptr(w_scale) || bad_ptr(out) || M < 1 ||
      N < 1 || K < 16 || K % 16 || N % 4 || gelu < 0 || gelu > 2 ||
      (gelu == 2 && (N % 256 != 0 || !bias)))
    return fail(ctx, JEPA_ERR_INVALID_ARG, "linear_fp8: bad argument");
  if ((((uintptr_t)A) & 15) || (((uintptr_t)W) & 15))
    return fail(ctx, JEPA_ERR_INVALID_ARG, "linear_fp8: A and W must be 16-byte aligned");
  CK(cudaSetDevice(ctx->device));
  Epilogue e = epi_base(ctx, gelu == 2 ? EPI_GATED : gelu ? EPI_GELU : EPI_STORE);
  e.act_bf16 = 0;
  e.bias = bias;
  e.out0 = out;
  e.ld0 = gelu == 2 ? N / 2 : N;
  e.row_scale = a_scale;
  e.col_scale = w_scale;
  CK(gemm_tc_fp8(A, W, M, N, K, e, ctx->dev_err, ctx->num_sms, (cudaStream_t)stream));
  return JEPA_OK;
}

jepa_status jepa_quantize_rows_fp8(jepa_ctx* ctx, const float* x, int rows, int cols,
                                   uint8_t* codes, float* scales, void* stream) {
  if (!ctx) return JEPA_ERR_INVALID_ARG;
  if (bad_ptr(x) || bad_ptr(codes) || bad_ptr(scales) || rows < 1 || cols < 1)
    return fail(ctx, JEPA_ERR_INVALID_ARG, "quantize_rows_fp8: bad argument");
  CK(cudaSetDevice(ctx->device));
  CK(quantize_rows_fp8(x, rows, cols, codes, scales, (cudaStream_t)stream));
  return JEPA_OK;
}

jepa_status jepa_attention_bf16(jepa_ctx* ctx, const uint16_t* q, const uint16_t* kv, uint16_t* out,
                                int ncand, int T, int Lk, int kv_rows, int heads, int d,
                                void* stream) {
  if (!ctx) return JEPA_ERR_INVALID_ARG;
  if (!bf16_mode(ctx)) return fail(ctx, JEPA_ERR_UNSUPPORTED, "attention_bf16 needs a bf16 context");
  if (bad_ptr(q) || bad_ptr(kv) || bad_ptr(out) || ncand < 1 || ncand > 65535 || T < 1 || Lk < 1 ||
      Lk > kv_rows || heads < 1 || d != heads * 64)
    return fail(ctx, JEPA_ERR_INVALID_ARG, "attention_bf16: bad argument");
  if ((((uintptr_t)q) & 15) || (((uintptr_t)kv) & 15) || (((uintptr_t)out) & 15))
    return fail(ctx, JEPA_ERR_INVALID_ARG, "attention_bf16: buffers must be 16-byte aligned");
  CK(cudaSetDevice(ctx->device));
  cudaStream_t s = (cudaStream_t)stream;
  CK(attention_tc_bf16((const bf16*)q, (const bf16*)kv, (bf16*)out, ncand, T, Lk, kv_rows, heads, d,
                       ctx->dev_err, s));
  return JEPA_OK;
}

jepa_status jepa_set_use_graphs(jepa_ctx* ctx, int enable) {
  if (!ctx) return JEPA_ERR_INVALID_ARG;
  ctx->use_graphs = enable != 0;
  return JEPA_OK;
}

jepa_status jepa_profile_enable(jepa_ctx* ctx, int enable) {
  if (!ctx) return JEPA_ERR_INVALID_ARG;
  ctx->profile = enable != 0;
  return JEPA_OK;
}

jepa_status jepa_profile_read(jepa_ctx* ctx, double* gemm_ms, double* gemm_flops,
                              int64_t* gemm_launches) {
  if (!ctx || !gemm_ms || !gemm_flops || !gemm_launches) return JEPA_ERR_INVALID_ARG;
  *gemm_ms = 0;
  *gemm_flops = 0;
  *gemm_launches = 0;
  PlanGraph* g = ctx->last_plan;
  if (!g || !g->profiled) return fail(ctx, JEPA_ERR_INVALID_ARG, "last plan was not profiled");
  for (size_t i = 0; i < g->ev_start.size(); ++i) {
    float ms = 0.f;
    CK(cudaEventElapsedTime(&ms, g->ev_start[i], g->ev_end[i]));
    *gemm_ms += ms;
    *gemm_flops += g->ev_flops[i];
  }
  *gemm_launches = (int64_t)g->ev_start.size();
  return JEPA_OK;
}

jepa_status jepa_selftest_bounded_wait(jepa_ctx* ctx, void* stream) {
  if (!ctx) return JEPA_ERR_INVALID_ARG;
  CK(cudaSetDevice(ctx->device));
  CK(wait_selftest(ctx->dev_err, (cudaStream_t)stream));
  return JEPA_OK;
}

jepa_status jepa_sync_check(jepa_ctx* ctx, void* stream) {
  if (!ctx) return JEPA_ERR_INVALID_ARG;
  CK(cudaSetDevice(ctx->device));
  CK(cudaStreamSynchronize((cudaStream_t)stream));
  int flag = 0;
  CK(cudaMemcpy(&flag, ctx->dev_err, sizeof(int), cudaMemcpyDeviceToHost));
  if (flag) {
    CK(cudaMemset(ctx->dev_err, 0, sizeof(int)));
    return fail(ctx, JEPA_ERR_TIMEOUT, "a bounded device wait expired (kernel returned early)");
  }
  return JEPA_OK;
}

}  // extern "C"
