// Internal declarations shared by the CUDA translation units of the planner library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace jepa {

typedef __nv_bfloat16 bf16;

// Row remap used by epilogues and row-gathering kernels:
//   r -> (r / rpg) * gstride + goff + (r % rpg)
// e.g. patch row (cand, p) of a [cand*P] matrix -> token row cand*T + 2 + p.
struct RowMap {
  int rpg;
  long long gstride;
  long long goff;
};
__host__ __device__ __forceinline__ long long map_row(const RowMap& m, int r) {
  return (long long)(r / m.rpg) * m.gstride + m.goff + (r % m.rpg);
}
static inline RowMap identity_map() { return RowMap{1 << 30, 0, 0}; }

enum EpiMode : int {
  EPI_STORE = 0,    // out = acc + bias                      (QKV: split into q and the KV cache)
  EPI_GELU = 1,     // out = gelu(acc + bias)                (MLP up)
  EPI_RESID = 2,    // x  += acc + bias   (fp32 residual)    (attention out-proj, MLP down)
  EPI_INPROJ = 3,   // x   = acc + bias + pos[token]         (patch in-projection)
  EPI_OUTPROJ = 4,  // z = acc + bias; optional z outputs; optional L1 energy partials
};

// What a GEMM does with its fp32 accumulators. One struct serves every mode; unused
// fields are ignored. Element types of out0/out1/zhat follow `act_bf16`.
struct Epilogue {
  int mode;
  int act_bf16;          // 1: bf16 activations (out0/out1/zhat), 0: fp32
  const float* bias;     // [N] or null
  void* out0;            // columns [0, split)
  int ld0;
  RowMap map0;
  int split;             // columns >= split go to out1 (column - split)
  void* out1;
  int ld1;
  RowMap map1;
  const float* pos;      // EPI_INPROJ: pos[(r % map0.rpg + pos_off) * N + c]
  int pos_off;
  float* zpred;          // EPI_OUTPROJ: fp32 [M, N] or null
  void* zhat;            // EPI_OUTPROJ: activation-typed [M, N] or null (next frame input)
  const float* goal;     // EPI_OUTPROJ: [B, P, N] or null
  int P;                 // rows per candidate
  int cand0;             // global candidate index of local candidate 0
  int cands_per_problem; // N of the plan (candidate -> problem)
  float* partial;        // [M, ntiles] per-tile sums of |z - goal|
  int ntiles;
};

__device__ __forceinline__ float gelu_erf(float x) {
  return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
}

// Apply the epilogue to `n` consecutive accumulators v[0..n) of row r starting at
// column c (c, n multiples of 4 except at the matrix edge; the run never crosses
// `split`). Returns this run's sum of |z - goal| for EPI_OUTPROJ (0 otherwise).
template <int RUN>
__device__ __forceinline__ float epilogue_run(const Epilogue& e, int r, int c, float* v, int n,
                                              int N) {
  if (e.bias) {
#pragma unroll
    for (int i = 0; i < RUN; ++i)
      if (i < n) v[i] += __ldg(e.bias + c + i);
  }
  const bool full = (n == RUN);
  if (e.mode == EPI_GELU) {
#pragma unroll
    for (int i = 0; i < RUN; ++i) v[i] = gelu_erf(v[i]);
  }
  if (e.mode == EPI_STORE || e.mode == EPI_GELU) {
    void* base;
    long long row;
    int col, ld;
    if (c >= e.split) {
      base = e.out1; row = map_row(e.map1, r); col = c - e.split; ld = e.ld1;
    } else {
      base = e.out0; row = map_row(e.map0, r); col = c; ld = e.ld0;
    }
    if (e.act_bf16) {
      bf16* o = reinterpret_cast<bf16*>(base) + row * ld + col;
      if (full && (RUN % 8 == 0) && ((((uintptr_t)o) & 15) == 0)) {
#pragma unroll
        for (int i = 0; i < RUN; i += 8) {
          __nv_bfloat162 p0 = __floats2bfloat162_rn(v[i], v[i + 1]);
          __nv_bfloat162 p1 = __floats2bfloat162_rn(v[i + 2], v[i + 3]);
          __nv_bfloat162 p2 = __floats2bfloat162_rn(v[i + 4], v[i + 5]);
          __nv_bfloat162 p3 = __floats2bfloat162_rn(v[i + 6], v[i + 7]);
          uint4 u;
          u.x = *reinterpret_cast<uint32_t*>(&p0);
          u.y = *reinterpret_cast<uint32_t*>(&p1);
          u.z = *reinterpret_cast<uint32_t*>(&p2);
          u.w = *reinterpret_cast<uint32_t*>(&p3);
          *reinterpret_cast<uint4*>(o + i) = u;
        }
      } else {
#pragma unroll
        for (int i = 0; i < RUN; ++i)
          if (i < n) o[i] = __float2bfloat16_rn(v[i]);
      }
    } else {
      float* o = reinterpret_cast<float*>(base) + row * ld + col;
#pragma unroll
      for (int i = 0; i < RUN; ++i)
        if (i < n) o[i] = v[i];
    }
    return 0.f;
  }
  if (e.mode == EPI_RESID || e.mode == EPI_INPROJ) {
    float* o = reinterpret_cast<float*>(e.out0) + map_row(e.map0, r) * e.ld0 + c;
    if (e.mode == EPI_INPROJ) {
      const float* pr = e.pos + (long long)(r % e.map0.rpg + e.pos_off) * N + c;
#pragma unroll
      for (int i = 0; i < RUN; ++i)
        if (i < n) v[i] += __ldg(pr + i);
    }
    if (full && (RUN % 4 == 0) && ((((uintptr_t)o) & 15) == 0)) {
#pragma unroll
      for (int i = 0; i < RUN; i += 4) {
        float4 x = *reinterpret_cast<float4*>(o + i);
        if (e.mode == EPI_RESID) {
          x.x += v[i]; x.y += v[i + 1]; x.z += v[i + 2]; x.w += v[i + 3];
        } else {
          x = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        }
        *reinterpret_cast<float4*>(o + i) = x;
      }
    } else {
#pragma unroll
      for (int i = 0; i < RUN; ++i)
        if (i < n) o[i] = (e.mode == EPI_RESID) ? o[i] + v[i] : v[i];
    }
    return 0.f;
  }
  // EPI_OUTPROJ
  const long long off = (long long)r * N + c;
  if (e.zpred) {
#pragma unroll
    for (int i = 0; i < RUN; ++i)
      if (i < n) e.zpred[off + i] = v[i];
  }
  if (e.zhat) {
    if (e.act_bf16) {
      bf16* o = reinterpret_cast<bf16*>(e.zhat) + off;
#pragma unroll
      for (int i = 0; i < RUN; ++i)
        if (i < n) o[i] = __float2bfloat16_rn(v[i]);
    } else {
      float* o = reinterpret_cast<float*>(e.zhat) + off;
#pragma unroll
      for (int i = 0; i < RUN; ++i)
        if (i < n) o[i] = v[i];
    }
  }
  float s = 0.f;
  if (e.goal) {
    const int cand = e.cand0 + r / e.P;
    const int b = cand / e.cands_per_problem;
    const float* g = e.goal + ((long long)b * e.P + (r % e.P)) * N + c;
#pragma unroll
    for (int i = 0; i < RUN; ++i)
      if (i < n) s += fabsf(v[i] - __ldg(g + i));
  }
  return s;
}

// ---- kernel launchers (each returns cudaGetLastError() of its launch) ----

// tcgen05 / TMA GEMM: out = epilogue(A[M,K] * W[N,K]^T), bf16 in, fp32 accumulate.
cudaError_t gemm_tc_bf16(const bf16* A, const bf16* W, int M, int N, int K, const Epilogue& epi,
                         int* err_flag, int num_sms, cudaStream_t s);
// Tile width the tensor-core GEMM uses for N (sizes the energy partial buffer).
int gemm_tc_tile_n(int N);

// SIMT fp32 GEMM with the same epilogue (fp32 mode).
cudaError_t gemm_simt_f32(const float* A, const float* W, int M, int N, int K, const Epilogue& epi,
                          cudaStream_t s);
int gemm_simt_tile_n();

// Flash-style attention, bf16 (head dim 64) and fp32 (head dim <= 128, multiple of 32).
// q [ncand*T, d]; kv [ncand][kv_stride_rows][2d] (K at columns [0,d), V at [d,2d));
// queries of the current block attend to key rows [0, Lk) of their candidate.
cudaError_t attention_bf16(const bf16* q, const bf16* kv, bf16* o, int ncand, int T, int Lk,
                           long long kv_cand_stride_rows, int heads, int d, cudaStream_t s);
cudaError_t attention_f32(const float* q, const float* kv, float* o, int ncand, int T, int Lk,
                          long long kv_cand_stride_rows, int heads, int d, cudaStream_t s);

// LayerNorm of fp32 rows (gathered through in_map) into bf16 or fp32 rows.
cudaError_t layernorm(const float* x, RowMap in_map, void* y, int y_bf16, const float* g,
                      const float* b, int rows, int d, float eps, cudaStream_t s);

// Philox4x32-10 + Box-Muller candidate sampler (seed from *seed_dev if non-null).
cudaError_t sample_actions(const float* mu, const float* sigma, int B, int N, int H, int A,
                           int round, const uint64_t* seed_dev, uint64_t seed, float* actions,
                           cudaStream_t s);

// Raw generator words for counters[4i..4i+3] (test surface of the sampler's generator).
cudaError_t philox_raw(const uint32_t* counters, uint64_t seed, int n, uint32_t* out, cudaStream_t s);

// Frame-block token assembly for candidates [cand0, cand0+ncand) at rollout step k:
// action and state tokens always; patch tokens copied from base[b] when base != null.
cudaError_t assemble_block(const float* actions, const float* state0, const float* W_a,
                           const float* b_a, const float* W_s, const float* b_s, const float* pos,
                           const float* base, float* x, int cand0, int ncand, int N, int H, int k,
                           int A, int S, int P, int d, cudaStream_t s);

// energy[c] = sum of partial rows of candidate c / (P * E), fixed summation order.
cudaError_t energy_finalize(const float* partial, int P, int ntiles, int ncand, float inv_count,
                            float* energy, cudaStream_t s);

// Per problem: sort (energy, index), elites = first K, refit mean / population std.
cudaError_t select_refit(const float* energy, const float* actions, int B, int N, int HA, int K,
                         float* mu, float* sigma, int* elites, int* winner, cudaStream_t s);

// out[b, :] = actions[b, winner[b], 0, :]
cudaError_t winner_action(const float* actions, const int* winner, int B, int N, int HA, int A,
                          float* out, cudaStream_t s);

// *p = v (one thread; lets a captured graph read a per-call value)
cudaError_t set_u64(uint64_t* p, uint64_t v, cudaStream_t s);

// fp32 -> bf16 (round to nearest even)
cudaError_t convert_f32_bf16(const float* x, bf16* y, long long n, cudaStream_t s);

}  // namespace jepa
