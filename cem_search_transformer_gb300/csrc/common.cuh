// Internal declarations shared by the CUDA translation units of the planner library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace jepa {

typedef __nv_bfloat16 bf16;

// cudaFuncSetAttribute acts on the current device only. Each kernel that needs more than
// 48 KB of dynamic shared memory keeps a mask of the devices (ordinals 0..63) it has been
// configured on; a device outside the mask range is configured on every call.
inline cudaError_t set_max_dynamic_smem(const void* func, int bytes,
                                        std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

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
  EPI_GATED = 5,    // gated MLP up: W rows hold FC1 and gate blocks of 32 interleaved
                    // (block 2p = FC1 rows 32p.., block 2p+1 = gate rows 32p..); output
                    // column 32p + c = (acc[64p + c] + bias) * gelu(acc[64p + 32 + c] + bias)
                    // of width N / 2, written to out0 (row stride ld0)
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
  float* partial;        // [M, ntiles] per-tile (and per column half) sums of |z - goal|
  int ntiles;            // partial sums per row (energy finalisation adds all of them)
  // fp8 operands only: accumulator (r, c) is multiplied by row_scale[r] * col_scale[c]
  // (activation row scale, weight output-channel scale) before the bias
  const float* row_scale;
  const float* col_scale;
  // set by the GEMM launchers only (callers leave it 0): which epilogue data move by TMA
  // through the kernel's extra tensor maps. CTA pairs: bit 0 = bf16 out0 rows (identity row
  // map) by TMA stores, bit 1 = out1 K/V cache rows by TMA stores (3-D map of row blocks).
  // Single CTAs: bit 2 = the projection's goal rows by TMA loads (energies only).
  int tma_out;
};

// GELU with the Gaussian CDF written through erf: x * (1 + erf(x / sqrt 2)) / 2.
// erf by Abramowitz & Stegun, Handbook of Mathematical Functions, eq. 7.1.26:
// erf(|u|) = 1 - t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-u^2), t = 1 / (1 + p |u|),
// |error| <= 1.5e-7, odd in u; here u = x / sqrt 2 and exp(-u^2) = 2^-(x^2 log2(e) / 2),
// evaluated with the fast reciprocal and base-2 exponential (max GELU error ~5e-7 abs).
__device__ __forceinline__ float gelu_erf(float x) {
  const float au = fabsf(x) * 0.70710678118654752f;
  const float t = __fdividef(1.0f, fmaf(0.3275911f, au, 1.0f));
  float p = fmaf(1.061405429f, t, -1.453152027f);
  p = fmaf(p, t, 1.421413741f);
  p = fmaf(p, t, -0.284496736f);
  p = fmaf(p, t, 0.254829592f);
  float e;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-0.72134752044448170f * x * x));
  const float erf_abs = fmaf(-p * t, e, 1.0f);
  const float hx = 0.5f * x;
  return fmaf(hx, copysignf(erf_abs, x), hx);
}

// Packed fp32 pairs (sm_100-family f32x2 arithmetic): two lanes of math per instruction.
__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(unsigned long long r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Two GELUs at once for the tensor-core epilogues, X = (x0, x1) in packed f32x2 arithmetic.
// erf by Abramowitz & Stegun eq. 7.1.28: erf(u) = 1 - (1 + a1 u + ... + a6 u^6)^-16 for
// u >= 0, |error| <= 3e-7, here with u = |x| / sqrt(2) folded into the coefficients
// (b_i = a_i 2^(-i/2), rounded to fp32; the folded polynomial keeps |error| <= 2.7e-7).
// With E = erf(|x| / sqrt(2)), GELU(x) = x (1 + erf(x / sqrt(2))) / 2 = (x + |x| E) / 2,
// which needs no sign selection: T = |x| - |x| R with R = (1 + ...)^-16, GELU = x / 2 + T / 2.
// One reciprocal per element and no exponential; everything else is packed. In fp32 the
// GELU stays within 7e-7 of the exact one over [-8, 8] (relative to max(1, |GELU|)).
__device__ __forceinline__ unsigned long long gelu2x(unsigned long long X) {
  unsigned long long AX, NAX;   // |x| and -|x| (sign bits cleared / set)
  asm("and.b64 %0, %1, 0x7fffffff7fffffff;" : "=l"(AX) : "l"(X));
  asm("or.b64 %0, %1, 0x8000000080000000;" : "=l"(NAX) : "l"(X));
  unsigned long long p = f2_fma(f2_pack(5.382974905e-06f, 5.382974905e-06f), AX,
                                f2_pack(4.889063712e-05f, 4.889063712e-05f));
  p = f2_fma(p, AX, f2_pack(3.800357445e-05f, 3.800357445e-05f));
  p = f2_fma(p, AX, f2_pack(3.277626354e-03f, 3.277626354e-03f));
  p = f2_fma(p, AX, f2_pack(2.114100568e-02f, 2.114100568e-02f));
  p = f2_fma(p, AX, f2_pack(4.986734688e-02f, 4.986734688e-02f));
  p = f2_fma(p, AX, f2_pack(1.0f, 1.0f));
  p = f2_mul(p, p);   // ^2
  p = f2_mul(p, p);   // ^4
  p = f2_mul(p, p);   // ^8
  p = f2_mul(p, p);   // ^16 (overflows to inf for large |x|: R = 0, erf = 1)
  const float2 q = f2_unpack(p);
  float r0, r1;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(q.x));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r1) : "f"(q.y));
  const unsigned long long T = f2_fma(NAX, f2_pack(r0, r1), AX);   // |x| (1 - R) = |x| E
  const unsigned long long H = f2_pack(0.5f, 0.5f);
  return f2_fma(T, H, f2_mul(X, H));
}

__device__ __forceinline__ float2 gelu2(float x0, float x1) {
  return f2_unpack(gelu2x(f2_pack(x0, x1)));
}

__device__ __forceinline__ float4 gelu4(float4 v) {
  const float2 a = gelu2(v.x, v.y), b = gelu2(v.z, v.w);
  return make_float4(a.x, a.y, b.x, b.y);
}

// Per-row addressing, computed once per output row. Meaning by mode (a < 0: row >= M):
//   STORE/GELU: a = out0 row offset, b = out1 row offset (elements)
//   RESID:      a = x row offset
//   INPROJ:     a = x row offset,   b = pos row offset
//   OUTPROJ:    a = r * N (zpred / zhat row), b = goal row offset
struct EpiRow {
  long long a, b;
};

__device__ __forceinline__ EpiRow epi_row(const Epilogue& e, int r, int M, int N) {
  EpiRow w;
  w.a = -1;
  w.b = 0;
  if (r >= M) return w;
  if (e.mode == EPI_STORE || e.mode == EPI_GELU) {
    w.a = map_row(e.map0, r) * e.ld0;
    if (e.out1) w.b = map_row(e.map1, r) * e.ld1;
  } else if (e.mode == EPI_RESID) {
    w.a = map_row(e.map0, r) * e.ld0;
  } else if (e.mode == EPI_INPROJ) {
    w.a = map_row(e.map0, r) * e.ld0;
    w.b = (long long)(r % e.map0.rpg + e.pos_off) * N;
  } else {
    w.a = (long long)r * N;
    if (e.goal) {
      const int cand = e.cand0 + r / e.P;
      const int b = cand / e.cands_per_problem;
      w.b = ((long long)b * e.P + (r % e.P)) * N;
    }
  }
  return w;
}

__device__ __forceinline__ void store4(void* base, long long off, int bf, float4 v) {
  if (bf) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(reinterpret_cast<bf16*>(base) + off) = u;
  } else {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + off) = v;
  }
}

// The per-element global operand of a mode (residual x, position row or goal row) for
// columns c..c+3, loaded separately so callers can issue it ahead of the accumulator.
__device__ __forceinline__ float4 epi_load4(const Epilogue& e, const EpiRow& w, int c) {
  if (w.a >= 0) {
    if (e.mode == EPI_RESID)
      return *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(e.out0) + w.a + c);
    if (e.mode == EPI_INPROJ) return __ldg(reinterpret_cast<const float4*>(e.pos + w.b + c));
    if (e.mode == EPI_OUTPROJ && e.goal)
      return __ldg(reinterpret_cast<const float4*>(e.goal + w.b + c));
  }
  return make_float4(0.f, 0.f, 0.f, 0.f);
}

__device__ __forceinline__ float4 epi_bias4(const Epilogue& e, int c) {
  return e.bias ? __ldg(reinterpret_cast<const float4*>(e.bias + c)) : make_float4(0.f, 0.f, 0.f, 0.f);
}

// Apply the epilogue to the 4 accumulators of columns c..c+3 (c % 4 == 0, c + 3 < N) of the
// row described by w, given that row's bias and operand from epi_bias4 / epi_load4.
// Requires N, ld0, ld1 and split to be multiples of 4 and 16-byte aligned buffers. Returns
// |z - goal| summed over the 4 columns (EPI_OUTPROJ with goal).
__device__ __forceinline__ float epi_apply4(const Epilogue& e, const EpiRow& w, int c, float4 v,
                                            float4 bb, float4 op) {
  v.x += bb.x; v.y += bb.y; v.z += bb.z; v.w += bb.w;
  if (e.mode == EPI_STORE || e.mode == EPI_GELU) {
    if (e.mode == EPI_GELU) v = gelu4(v);
    if (c >= e.split)
      store4(e.out1, w.b + (c - e.split), e.act_bf16, v);
    else
      store4(e.out0, w.a + c, e.act_bf16, v);
    return 0.f;
  }
  if (e.mode == EPI_RESID || e.mode == EPI_INPROJ) {
    // residual: x + (acc + bias); in-projection: (acc + bias) + pos
    v.x += op.x; v.y += op.y; v.z += op.z; v.w += op.w;
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(e.out0) + w.a + c) = v;
    return 0.f;
  }
  // EPI_OUTPROJ
  const long long off = w.a + c;
  if (e.zpred) *reinterpret_cast<float4*>(e.zpred + off) = v;
  if (e.zhat) store4(e.zhat, off, e.act_bf16, v);
  if (e.goal)
    return ((fabsf(v.x - op.x) + fabsf(v.y - op.y)) + fabsf(v.z - op.z)) + fabsf(v.w - op.w);
  return 0.f;
}

// Convenience form that loads its own bias and operand.
__device__ __forceinline__ float epi_apply4(const Epilogue& e, const EpiRow& w, int c, float4 v) {
  return epi_apply4(e, w, c, v, epi_bias4(e, c), epi_load4(e, w, c));
}

// ---- kernel launchers (each returns cudaGetLastError() of its launch) ----

// tcgen05 / TMA GEMM: out = epilogue(A[M,K] * W[N,K]^T), bf16 in, fp32 accumulate.
cudaError_t gemm_tc_bf16(const bf16* A, const bf16* W, int M, int N, int K, const Epilogue& epi,
                         int* err_flag, int num_sms, cudaStream_t s);
// fp8 e4m3 operands (codes), scales in epi.row_scale / epi.col_scale; K a multiple of 16
cudaError_t gemm_tc_fp8(const uint8_t* A, const uint8_t* W, int M, int N, int K,
                        const Epilogue& epi, int* err_flag, int num_sms, cudaStream_t s);
// Energy partial sums per row that the tensor-core GEMM writes for an output width N.
int gemm_tc_partials(int N);

// SIMT fp32 GEMM with the same epilogue (fp32 mode).
cudaError_t gemm_simt_f32(const float* A, const float* W, int M, int N, int K, const Epilogue& epi,
                          cudaStream_t s);
int gemm_simt_partials(int N);

// Flash-style attention, bf16 on the tensor cores (head dim 64) and fp32 (head dim <= 128,
// multiple of 32). q [ncand*T, d]; kv [ncand][kv_stride_rows][2d] (K at columns [0,d), V at
// [d,2d)); queries of the current block attend to key rows [0, Lk) of their candidate.
cudaError_t attention_tc_bf16(const bf16* q, const bf16* kv, bf16* o, int ncand, int T, int Lk,
                              long long kv_cand_stride_rows, int heads, int d, int* err_flag,
                              cudaStream_t s);
cudaError_t attention_f32(const float* q, const float* kv, float* o, int ncand, int T, int Lk,
                          long long kv_cand_stride_rows, int heads, int d, cudaStream_t s);

// LayerNorm of fp32 rows (gathered through in_map) into bf16 or fp32 rows.
// out_kind: 0 fp32, 1 bf16, 2 fp8 e4m3 codes (row scales to yscale)
cudaError_t layernorm(const float* x, RowMap in_map, void* y, int out_kind, const float* g,
                      const float* b, int rows, int d, float eps, cudaStream_t s,
                      float* yscale = nullptr);
cudaError_t quantize_rows_fp8(const float* src, long long rows, int cols, uint8_t* codes,
                              float* scales, cudaStream_t s);

// Philox4x32-10 + Box-Muller candidate sampler (seed from *seed_dev if non-null).
cudaError_t sample_actions(const float* mu, const float* sigma, int B, int N, int H, int A,
                           int round, const uint64_t* seed_dev, uint64_t seed, float* actions,
                           cudaStream_t s);

// Raw generator words for counters[4i..4i+3] (test surface of the sampler's generator).
cudaError_t philox_raw(const uint32_t* counters, uint64_t seed, int n, uint32_t* out, cudaStream_t s);

// Layer-0 queries / keys / values of the frame-0 patch rows, which every candidate of a
// problem shares (computed once per problem) and where to broadcast them. q_base [B*P, d] and
// kv_base [B*P, 2d] in the activation type (ab bytes per element); q [ncand*T, d] and kv
// (the layer-0 cache slot, kv_stride rows per candidate, 2d columns). q_base == nullptr: off.
struct BaseRows {
  const uint8_t* q_base = nullptr;
  const uint8_t* kv_base = nullptr;
  uint8_t* q = nullptr;
  uint8_t* kv = nullptr;
  long long kv_stride = 0;
  int ab = 0;
};

// Frame-block token assembly for candidates [cand0, cand0+ncand) at rollout step k:
// action and state tokens always; patch tokens copied from base[b] when base != null; the
// layer-0 patch rows of q and the cache broadcast from br when br.q_base != null.
cudaError_t assemble_block(const float* actions, const float* state0, const float* W_a,
                           const float* b_a, const float* W_s, const float* b_s, const float* pos,
                           const float* base, float* x, int cand0, int ncand, int N, int H, int k,
                           int A, int S, int P, int d, const BaseRows& br, cudaStream_t s);

// energy[c] = sum of partial rows of candidate c / (P * E), fixed summation order.
cudaError_t energy_finalize(const float* partial, int P, int ntiles, int ncand, float inv_count,
                            float* energy, cudaStream_t s);

// Per problem: sort (energy, index), elites = first K, refit mean / population std.
cudaError_t select_refit(const float* energy, const float* actions, int B, int N, int HA, int K,
                         float* mu, float* sigma, int* elites, int* winner, cudaStream_t s);
// Energy finalisation of a single-chunk pass (partials of all B*N candidates in `partial`),
// then selection and refit per problem, in one launch. counter: B zero-initialised unsigned
// ints, left at zero again.
cudaError_t energy_select(const float* partial, int P, int ntiles, int B, int N, float inv_count,
                          float* energy, const float* actions, int HA, int K, float* mu,
                          float* sigma, int* elites, int* winner, unsigned int* counter,
                          cudaStream_t s);

// out[b, :] = actions[b, winner[b], 0, :]
cudaError_t winner_action(const float* actions, const int* winner, int B, int N, int HA, int A,
                          float* out, cudaStream_t s);

// *p = v (one thread; lets a captured graph read a per-call value)
cudaError_t set_u64(uint64_t* p, uint64_t v, cudaStream_t s);
cudaError_t warm_start(const float* mu_prev, const float* mu_prior, const float* sigma_prior, int B,
                       int H, int A, float* mu_out, float* sigma_out, cudaStream_t s);
cudaError_t state_step(const float* st, const float* a, int n, float* s_out, cudaStream_t s);
cudaError_t wait_selftest(int* err_flag, cudaStream_t s);

// fp32 -> bf16 (round to nearest even)
cudaError_t convert_f32_bf16(const float* x, bf16* y, long long n, cudaStream_t s);

}  // namespace jepa
