// Sampler, token assembly, LayerNorm, energy, elite selection / refit, and the fp32
// (SIMT) GEMM and attention used by the fp32 precision mode.
//
// Method: "Real-time inference for JEPA world-model architectures with Ray", section
// "Where the sixteen seconds actually goes" (sample from a Gaussian, measure each
// sample's distance to the goal, refit the Gaussian to the K closest).
#include "common.cuh"
#include "tc_common.cuh"

#include <float.h>

namespace jepa {

// ---------------------------------------------------------------------------------
// Candidate sampler: Philox4x32-10 (Salmon et al., SC'11) + Box-Muller.
// Counter (n, b, round*Q + q, 0), key (seed lo, seed hi); word w of quad q feeds
// element 4q + w of the candidate's H*A draws. Transform in fp64, stored as fp32.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t hi0 = __umulhi(M0, c.x), lo0 = M0 * c.x;
    const uint32_t hi1 = __umulhi(M1, c.z), lo1 = M1 * c.z;
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
    k.x += W0;
    k.y += W1;
  }
  return c;
}

__device__ __forceinline__ double uniform_open01(uint32_t x) {
  return ((double)(x >> 9) + 0.5) * (1.0 / 8388608.0);
}

__global__ void k_sample(const float* __restrict__ mu, const float* __restrict__ sigma, int B,
                         int N, int H, int A, int round, const uint64_t* __restrict__ seed_dev,
                         uint64_t seed_val, float* __restrict__ actions) {
  const int HA = H * A, Q = (HA + 3) / 4;
  const long long total = (long long)B * N * Q;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int q = (int)(i % Q);
  const long long bn = i / Q;
  const int n = (int)(bn % N), b = (int)(bn / N);
  const uint64_t seed = seed_dev ? *seed_dev : seed_val;
  const uint4 w = philox4x32_10(make_uint4((uint32_t)n, (uint32_t)b, (uint32_t)(round * Q + q), 0u),
                                make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
  double z[4];
  {
    const double r0 = sqrt(-2.0 * log(uniform_open01(w.x)));
    double s, c;
    sincospi(2.0 * uniform_open01(w.y), &s, &c);
    z[0] = r0 * c;
    z[1] = r0 * s;
    const double r1 = sqrt(-2.0 * log(uniform_open01(w.z)));
    sincospi(2.0 * uniform_open01(w.w), &s, &c);
    z[2] = r1 * c;
    z[3] = r1 * s;
  }
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int e = 4 * q + t;
    if (e < HA) {
      const double m = (double)mu[(long long)b * HA + e];
      const double sg = (double)sigma[(long long)b * HA + e];
      double a = m + sg * z[t];
      a = fmin(1.0, fmax(-1.0, a));
      actions[bn * HA + e] = (float)a;
    }
  }
}

cudaError_t sample_actions(const float* mu, const float* sigma, int B, int N, int H, int A,
                           int round, const uint64_t* seed_dev, uint64_t seed, float* actions,
                           cudaStream_t s) {
  const int Q = (H * A + 3) / 4;
  const long long total = (long long)B * N * Q;
  const int threads = 256;
  k_sample<<<(unsigned)((total + threads - 1) / threads), threads, 0, s>>>(
      mu, sigma, B, N, H, A, round, seed_dev, seed, actions);
  return cudaGetLastError();
}

__global__ void k_philox_raw(const uint4* __restrict__ ctr, uint64_t seed, int n,
                             uint4* __restrict__ out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = philox4x32_10(ctr[i], make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
}

cudaError_t philox_raw(const uint32_t* counters, uint64_t seed, int n, uint32_t* out,
                       cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  k_philox_raw<<<(n + 255) / 256, 256, 0, s>>>(reinterpret_cast<const uint4*>(counters), seed, n,
                                               reinterpret_cast<uint4*>(out));
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------
// Token assembly for frame block k: [action a_k, state s_k, P patches].
// s_k = state0[b] + sum_{j<k} a_j. Patch rows are copied from base (W_in z0 + b_in + pos,
// computed once per problem) for k == 0; for k >= 1 the in-projection GEMM writes them.
// ---------------------------------------------------------------------------------
// 16-byte copy of n16 vectors, block-strided, four loads in flight per thread.
__device__ __forceinline__ void copy16(void* __restrict__ dst, const void* __restrict__ src,
                                       long long n16) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  const long long step = blockDim.x;
  long long i = threadIdx.x;
  for (; i + 3 * step < n16; i += 4 * step) {
    const uint4 a = s4[i], b = s4[i + step], c = s4[i + 2 * step], e = s4[i + 3 * step];
    d4[i] = a;
    d4[i + step] = b;
    d4[i + 2 * step] = c;
    d4[i + 3 * step] = e;
  }
  for (; i < n16; i += step) d4[i] = s4[i];
}

__global__ void k_assemble(const float* __restrict__ actions, const float* __restrict__ state0,
                           const float* __restrict__ W_a, const float* __restrict__ b_a,
                           const float* __restrict__ W_s, const float* __restrict__ b_s,
                           const float* __restrict__ pos, const float* __restrict__ base,
                           float* __restrict__ x, int cand0, int N, int H, int k, int A, int S,
                           int P, int d, BaseRows br) {
  __shared__ float a_s[32], s_s[32];
  const int lc = blockIdx.x;               // local candidate
  const int cand = cand0 + lc;
  const int b = cand / N;
  const int T = P + 2;
  // blockIdx.y: 0 = action and state tokens and the patch rows of x; 1 = the shared patch rows
  // of q; 2, 3 = the two halves of the shared patch rows of the layer-0 cache slot
  if (blockIdx.y > 0) {
    const long long qrow = (long long)d * br.ab, kvrow = 2 * qrow;
    if (blockIdx.y == 1) {
      copy16(br.q + ((long long)lc * T + 2) * qrow, br.q_base + (long long)b * P * qrow,
             (long long)P * qrow / 16);
    } else {
      const long long half = (long long)P * kvrow / 32;   // 16-byte vectors per half
      const long long off = (blockIdx.y - 2) * half * 16;
      copy16(br.kv + ((long long)lc * br.kv_stride + 2) * kvrow + off,
             br.kv_base + (long long)b * P * kvrow + off, half);
    }
    return;
  }
  const float* act = actions + (long long)cand * H * A;
  if (threadIdx.x < A) a_s[threadIdx.x] = act[k * A + threadIdx.x];
  if (threadIdx.x < S) {
    float sv = state0[(long long)b * S + threadIdx.x];
    for (int j = 0; j < k; ++j) sv += act[j * A + threadIdx.x];   // S == A (checked on the host)
    s_s[threadIdx.x] = sv;
  }
  __syncthreads();
  float* xr = x + (long long)lc * T * d;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    float va = b_a[c] + pos[c], vs = b_s[c] + pos[d + c];
    for (int j = 0; j < A; ++j) va += W_a[(long long)c * A + j] * a_s[j];
    for (int j = 0; j < S; ++j) vs += W_s[(long long)c * S + j] * s_s[j];
    xr[c] = va;
    xr[d + c] = vs;
  }
  if (base) copy16(xr + 2 * (long long)d, base + (long long)b * P * d, (long long)P * d / 4);
}

cudaError_t assemble_block(const float* actions, const float* state0, const float* W_a,
                           const float* b_a, const float* W_s, const float* b_s, const float* pos,
                           const float* base, float* x, int cand0, int ncand, int N, int H, int k,
                           int A, int S, int P, int d, const BaseRows& br, cudaStream_t s) {
  if (ncand <= 0) return cudaSuccess;
  if (br.q_base && ((((uintptr_t)br.q | (uintptr_t)br.kv | (uintptr_t)br.q_base |
                      (uintptr_t)br.kv_base) & 15) || ((long long)P * d * br.ab) % 32))
    return cudaErrorInvalidValue;
  // layer 0's queries, keys and values of the frame-0 patch rows, computed once for the
  // problem, go to rows 2 .. T-1 of every candidate's q block and cache slot (blocks y >= 1)
  const dim3 grid(ncand, br.q_base ? 4 : 1);
  k_assemble<<<grid, 256, 0, s>>>(actions, state0, W_a, b_a, W_s, b_s, pos, base, x, cand0, N, H,
                                  k, A, S, P, d, br);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------
// LayerNorm: one warp per row, fp32 statistics (two passes over registers).
// ---------------------------------------------------------------------------------
// e4m3 code of x (round to nearest even, saturating to +-448): the low byte of a converted
// pair whose two inputs are both x.
__device__ __forceinline__ uint8_t e4m3_code(float x) {
  uint16_t p;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(p) : "f"(x));
  return (uint8_t)(p & 0xFF);
}

// Output kinds of the LayerNorm: 0 fp32, 1 bf16, 2 fp8 e4m3 codes with one scale per row
// (scale = max |row| / 448, codes = e4m3(row * (448 / max |row|)); a zero row has scale 1).
template <int VPL, int OUT>
__global__ void k_layernorm(const float* __restrict__ x, RowMap in_map, void* __restrict__ y,
                            float* __restrict__ yscale, const float* __restrict__ g,
                            const float* __restrict__ bta, int rows, int d, float eps) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= rows) return;
  const float* xr = x + map_row(in_map, warp) * d;
  float v[VPL];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int c = lane + 32 * i;
    v[i] = (c < d) ? xr[c] : 0.f;
    s += v[i];
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float mean = s / d;
  float q = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int c = lane + 32 * i;
    const float t = (c < d) ? v[i] - mean : 0.f;
    q += t * t;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
  const float rstd = rsqrtf(q / d + eps);
  if constexpr (OUT == 2) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int c = lane + 32 * i;
      if (c < d) {
        v[i] = (v[i] - mean) * rstd * g[c] + bta[c];
        amax = fmaxf(amax, fabsf(v[i]));
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float inv = amax > 0.f ? 448.f / amax : 1.f;
    if (lane == 0) yscale[warp] = amax > 0.f ? amax / 448.f : 1.f;
    uint8_t* yr = reinterpret_cast<uint8_t*>(y) + (long long)warp * d;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int c = lane + 32 * i;
      if (c < d) yr[c] = e4m3_code(v[i] * inv);
    }
  } else {
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int c = lane + 32 * i;
      if (c < d) {
        const float t = (v[i] - mean) * rstd * g[c] + bta[c];
        if (OUT == 1)
          reinterpret_cast<bf16*>(y)[(long long)warp * d + c] = __float2bfloat16_rn(t);
        else
          reinterpret_cast<float*>(y)[(long long)warp * d + c] = t;
      }
    }
  }
}

// The same LayerNorm for widths that are a multiple of 128: lane l holds columns
// 128 i + 4 l .. + 3 (i < G = d / 128), so every load is a 16-byte vector and every warp
// instruction moves 512 contiguous bytes.
template <int G, int OUT>
__global__ void k_layernorm_v4(const float* __restrict__ x, RowMap in_map, void* __restrict__ y,
                               float* __restrict__ yscale, const float* __restrict__ g,
                               const float* __restrict__ bta, int rows, float eps) {
  constexpr int D = 128 * G;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= rows) return;
  const float4* xr = reinterpret_cast<const float4*>(x + map_row(in_map, warp) * D) + lane;
  float4 v[G];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < G; ++i) {
    v[i] = __ldcs(xr + 32 * i);
    s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float mean = s * (1.0f / D);
  float q = 0.f;
#pragma unroll
  for (int i = 0; i < G; ++i) {
    const float a = v[i].x - mean, b = v[i].y - mean, c = v[i].z - mean, e = v[i].w - mean;
    q += (a * a + b * b) + (c * c + e * e);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
  const float rstd = rsqrtf(q * (1.0f / D) + eps);
  const float4* g4 = reinterpret_cast<const float4*>(g) + lane;
  const float4* b4 = reinterpret_cast<const float4*>(bta) + lane;
#pragma unroll
  for (int i = 0; i < G; ++i) {
    const float4 gg = __ldg(g4 + 32 * i), bb = __ldg(b4 + 32 * i);
    v[i] = make_float4((v[i].x - mean) * rstd * gg.x + bb.x, (v[i].y - mean) * rstd * gg.y + bb.y,
                       (v[i].z - mean) * rstd * gg.z + bb.z, (v[i].w - mean) * rstd * gg.w + bb.w);
  }
  const long long base = (long long)warp * D + 4 * lane;
  if constexpr (OUT == 2) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < G; ++i)
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float inv = amax > 0.f ? 448.f / amax : 1.f;
    if (lane == 0) yscale[warp] = amax > 0.f ? amax / 448.f : 1.f;
#pragma unroll
    for (int i = 0; i < G; ++i) {
      const uint32_t w = (uint32_t)e4m3_code(v[i].x * inv) | ((uint32_t)e4m3_code(v[i].y * inv) << 8) |
                         ((uint32_t)e4m3_code(v[i].z * inv) << 16) | ((uint32_t)e4m3_code(v[i].w * inv) << 24);
      *reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(y) + base + 128 * i) = w;
    }
  } else if constexpr (OUT == 1) {
#pragma unroll
    for (int i = 0; i < G; ++i) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(v[i].x, v[i].y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(v[i].z, v[i].w);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&lo);
      u.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(reinterpret_cast<bf16*>(y) + base + 128 * i) = u;
    }
  } else {
#pragma unroll
    for (int i = 0; i < G; ++i)
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(y) + base + 128 * i) = v[i];
  }
}

// Per-row fp8 quantisation of fp32 rows (weights at load time, and the C ABI): one warp per
// row, the same scale rule and rounding as the LayerNorm's fp8 output.
__global__ void k_quantize_rows(const float* __restrict__ src, long long rows, int cols,
                                uint8_t* __restrict__ codes, float* __restrict__ scales) {
  const long long r = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const float* xr = src + r * cols;
  float amax = 0.f;
  for (int c = lane; c < cols; c += 32) amax = fmaxf(amax, fabsf(xr[c]));
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float inv = amax > 0.f ? 448.f / amax : 1.f;
  if (lane == 0) scales[r] = amax > 0.f ? amax / 448.f : 1.f;
  uint8_t* cr = codes + r * cols;
  for (int c = lane; c < cols; c += 32) cr[c] = e4m3_code(xr[c] * inv);
}

cudaError_t quantize_rows_fp8(const float* src, long long rows, int cols, uint8_t* codes,
                              float* scales, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const int threads = 256;
  const unsigned blocks = (unsigned)((rows * 32 + threads - 1) / threads);
  k_quantize_rows<<<blocks, threads, 0, s>>>(src, rows, cols, codes, scales);
  return cudaGetLastError();
}

template <int VPL>
static cudaError_t launch_ln(const float* x, RowMap m, void* y, float* yscale, int out_kind,
                             const float* g, const float* b, int rows, int d, float eps,
                             cudaStream_t s) {
  const int threads = 256;
  const unsigned blocks = (unsigned)(((long long)rows * 32 + threads - 1) / threads);
  if (out_kind == 2)
    k_layernorm<VPL, 2><<<blocks, threads, 0, s>>>(x, m, y, yscale, g, b, rows, d, eps);
  else if (out_kind == 1)
    k_layernorm<VPL, 1><<<blocks, threads, 0, s>>>(x, m, y, yscale, g, b, rows, d, eps);
  else
    k_layernorm<VPL, 0><<<blocks, threads, 0, s>>>(x, m, y, yscale, g, b, rows, d, eps);
  return cudaGetLastError();
}

template <int G>
static cudaError_t launch_ln4(const float* x, RowMap m, void* y, float* yscale, int out_kind,
                              const float* g, const float* b, int rows, float eps, cudaStream_t s) {
  const int threads = 256;
  const unsigned blocks = (unsigned)(((long long)rows * 32 + threads - 1) / threads);
  if (out_kind == 2)
    k_layernorm_v4<G, 2><<<blocks, threads, 0, s>>>(x, m, y, yscale, g, b, rows, eps);
  else if (out_kind == 1)
    k_layernorm_v4<G, 1><<<blocks, threads, 0, s>>>(x, m, y, yscale, g, b, rows, eps);
  else
    k_layernorm_v4<G, 0><<<blocks, threads, 0, s>>>(x, m, y, yscale, g, b, rows, eps);
  return cudaGetLastError();
}

cudaError_t layernorm(const float* x, RowMap in_map, void* y, int out_kind, const float* g,
                      const float* b, int rows, int d, float eps, cudaStream_t s,
                      float* yscale) {
  if (rows <= 0) return cudaSuccess;
  if (out_kind == 2 && !yscale) return cudaErrorInvalidValue;
  switch (d) {   // widths of the predictor configurations: 16-byte vector path
    case 128: return launch_ln4<1>(x, in_map, y, yscale, out_kind, g, b, rows, eps, s);
    case 384: return launch_ln4<3>(x, in_map, y, yscale, out_kind, g, b, rows, eps, s);
    case 512: return launch_ln4<4>(x, in_map, y, yscale, out_kind, g, b, rows, eps, s);
    case 768: return launch_ln4<6>(x, in_map, y, yscale, out_kind, g, b, rows, eps, s);
    case 1024: return launch_ln4<8>(x, in_map, y, yscale, out_kind, g, b, rows, eps, s);
    case 2048: return launch_ln4<16>(x, in_map, y, yscale, out_kind, g, b, rows, eps, s);
    default: break;
  }
  if (d <= 128) return launch_ln<4>(x, in_map, y, yscale, out_kind, g, b, rows, d, eps, s);
  if (d <= 512) return launch_ln<16>(x, in_map, y, yscale, out_kind, g, b, rows, d, eps, s);
  if (d <= 1024) return launch_ln<32>(x, in_map, y, yscale, out_kind, g, b, rows, d, eps, s);
  if (d <= 2048) return launch_ln<64>(x, in_map, y, yscale, out_kind, g, b, rows, d, eps, s);
  return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------------
// Energy: E[c] = (1 / (P*E)) * sum over the candidate's P rows and ntiles partials.
// One warp per candidate; lane-strided sums then a fixed xor tree (order independent of
// how candidates are chunked).
// ---------------------------------------------------------------------------------
__global__ void k_energy_finalize(const float* __restrict__ partial, int P, int ntiles, int ncand,
                                  float inv_count, float* __restrict__ energy) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= ncand) return;
  const float* p = partial + (long long)warp * P * ntiles;
  const int n = P * ntiles;
  float s = 0.f;
  for (int i = lane; i < n; i += 32) s += p[i];
#pragma unroll
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) energy[warp] = s * inv_count;
}

cudaError_t energy_finalize(const float* partial, int P, int ntiles, int ncand, float inv_count,
                            float* energy, cudaStream_t s) {
  if (ncand <= 0) return cudaSuccess;
  const int threads = 256;
  k_energy_finalize<<<(ncand * 32 + threads - 1) / threads, threads, 0, s>>>(
      partial, P, ntiles, ncand, inv_count, energy);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------
// Elite selection + refit: one CTA per problem. Keys (orderable energy bits << 32 | index)
// are bitonic-sorted in shared memory, so ties go to the lower index and NaN sorts last.
// Refit in fp64: mean and population std of the elites per (h, j).
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t orderable(float e) {
  if (isnan(e)) return 0xFFFFFFFFu;
  const uint32_t u = (e == 0.0f) ? 0u : __float_as_uint(e);   // -0 and +0 are the same energy
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Selection and refit of problem b by one block: keys (orderable energy bits << 32 | index)
// bitonic-sorted in shared memory, elites = the first K, refit of the elites in fp64. The
// energies are read through L2 (they may have been written by other blocks of the same
// kernel, which the caller has ordered with a fence).
__device__ void select_refit_block(const float* e, const float* __restrict__ ab, int N, int HA, int K,
                                   int npow2, float* __restrict__ mu, float* __restrict__ sigma,
                                   int* __restrict__ elites, int* __restrict__ winner, int b,
                                   unsigned long long* keys) {
  for (int i = threadIdx.x; i < npow2; i += blockDim.x)
    keys[i] = (i < N) ? (((unsigned long long)orderable(__ldcg(e + i)) << 32) | (unsigned)i)
                      : 0xFFFFFFFFFFFFFFFFull;
  __syncthreads();
  for (int size = 2; size <= npow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < npow2 / 2; i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool up = ((lo & size) == 0);
        const unsigned long long a = keys[lo], c = keys[hi];
        if ((a > c) == up) {
          keys[lo] = c;
          keys[hi] = a;
        }
      }
      __syncthreads();
    }
  }
  if (elites)
    for (int i = threadIdx.x; i < K; i += blockDim.x)
      elites[(long long)b * K + i] = (int)(keys[i] & 0xFFFFFFFFu);
  if (threadIdx.x == 0 && winner) winner[b] = (int)(keys[0] & 0xFFFFFFFFu);
  // refit: one warp per (h, j) element
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int el = warp; el < HA; el += nw) {
    double s = 0.0;
    for (int i = lane; i < K; i += 32) s += (double)ab[(long long)(keys[i] & 0xFFFFFFFFu) * HA + el];
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const double m = s / K;
    double q = 0.0;
    for (int i = lane; i < K; i += 32) {
      const double t = (double)ab[(long long)(keys[i] & 0xFFFFFFFFu) * HA + el] - m;
      q += t * t;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
    if (lane == 0) {
      mu[(long long)b * HA + el] = (float)m;
      sigma[(long long)b * HA + el] = (float)sqrt(q / K);
    }
  }
}

__global__ void k_select_refit(const float* __restrict__ energy, const float* __restrict__ actions,
                               int N, int HA, int K, int npow2, float* __restrict__ mu,
                               float* __restrict__ sigma, int* __restrict__ elites,
                               int* __restrict__ winner) {
  extern __shared__ unsigned long long keys[];
  const int b = blockIdx.x;
  select_refit_block(energy + (long long)b * N, actions + (long long)b * N * HA, N, HA, K, npow2, mu,
                     sigma, elites, winner, b, keys);
}

cudaError_t select_refit(const float* energy, const float* actions, int B, int N, int HA, int K,
                         float* mu, float* sigma, int* elites, int* winner, cudaStream_t s) {
  int npow2 = 1;
  while (npow2 < N) npow2 <<= 1;
  const size_t smem = (size_t)npow2 * sizeof(unsigned long long);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_select_refit, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  k_select_refit<<<B, 1024, smem, s>>>(energy, actions, N, HA, K, npow2, mu, sigma, elites, winner);
  return cudaGetLastError();
}

// Energy finalisation, elite selection and refit in one launch: blocks (x, b) each finalise
// 32 candidates of problem b (one warp per candidate, the same fixed summation order as
// k_energy_finalize), then the last block of problem b to finish, told by a per-problem
// arrival counter, selects and refits that problem and resets its counter for the next use.
__global__ void k_energy_select(const float* __restrict__ partial, int P, int ntiles, int N,
                                float inv_count, float* energy, const float* __restrict__ actions,
                                int HA, int K, int npow2, float* __restrict__ mu,
                                float* __restrict__ sigma, int* __restrict__ elites,
                                int* __restrict__ winner, unsigned int* __restrict__ counter) {
  extern __shared__ unsigned long long keys[];
  __shared__ bool last;
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * (blockDim.x >> 5) + warp;
  if (n < N) {
    const long long c = (long long)b * N + n;
    const float* p = partial + c * P * ntiles;
    const int cnt = P * ntiles;
    float s = 0.f;
    for (int i = lane; i < cnt; i += 32) s += p[i];
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) energy[c] = s * inv_count;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(counter + b, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  select_refit_block(energy + (long long)b * N, actions + (long long)b * N * HA, N, HA, K, npow2, mu,
                     sigma, elites, winner, b, keys);
  if (threadIdx.x == 0) counter[b] = 0u;
}

cudaError_t energy_select(const float* partial, int P, int ntiles, int B, int N, float inv_count,
                          float* energy, const float* actions, int HA, int K, float* mu,
                          float* sigma, int* elites, int* winner, unsigned int* counter,
                          cudaStream_t s) {
  int npow2 = 1;
  while (npow2 < N) npow2 <<= 1;
  const size_t smem = (size_t)npow2 * sizeof(unsigned long long);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_energy_select, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid((N + 31) / 32, B);
  k_energy_select<<<grid, 1024, smem, s>>>(partial, P, ntiles, N, inv_count, energy, actions, HA, K,
                                           npow2, mu, sigma, elites, winner, counter);
  return cudaGetLastError();
}

__global__ void k_winner_action(const float* __restrict__ actions, const int* __restrict__ winner,
                                int N, int HA, int A, float* __restrict__ out) {
  const int b = blockIdx.x;
  const int w = winner[b];
  for (int j = threadIdx.x; j < A; j += blockDim.x)
    out[(long long)b * A + j] = actions[((long long)b * N + w) * HA + j];
}

cudaError_t winner_action(const float* actions, const int* winner, int B, int N, int HA, int A,
                          float* out, cudaStream_t s) {
  k_winner_action<<<B, 32, 0, s>>>(actions, winner, N, HA, A, out);
  return cudaGetLastError();
}

// Receding-horizon warm start ("Further Optimization", B. Warm-started CEM): the last
// round's mean loses its executed first step, steps 1..H-1 move to 0..H-2, the new last
// step and every width come from the prior. One thread per (problem, action dim) walks h
// upwards, so mu_out may alias mu_prev (step h reads h+1 before anything writes it) and
// sigma_out may alias sigma_prior.
__global__ void k_warm_start(const float* mu_prev, const float* mu_prior, const float* sigma_prior,
                             int B, int H, int A, float* mu_out, float* sigma_out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= B * A) return;
  const int b = i / A, j = i % A;
  const long long base = (long long)b * H * A + j;
  for (int h = 0; h + 1 < H; ++h) mu_out[base + (long long)h * A] = mu_prev[base + (long long)(h + 1) * A];
  mu_out[base + (long long)(H - 1) * A] = mu_prior[base + (long long)(H - 1) * A];
  for (int h = 0; h < H; ++h) sigma_out[base + (long long)h * A] = sigma_prior[base + (long long)h * A];
}

cudaError_t warm_start(const float* mu_prev, const float* mu_prior, const float* sigma_prior, int B,
                       int H, int A, float* mu_out, float* sigma_out, cudaStream_t s) {
  const int n = B * A;
  k_warm_start<<<(n + 127) / 128, 128, 0, s>>>(mu_prev, mu_prior, sigma_prior, B, H, A, mu_out,
                                               sigma_out);
  return cudaGetLastError();
}

// State of the next control step, s' = s + a (the same integration the rollout uses
// between frame blocks). s_out may alias s.
__global__ void k_state_step(const float* st, const float* a, int n, float* s_out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) s_out[i] = st[i] + a[i];
}

cudaError_t state_step(const float* st, const float* a, int n, float* s_out, cudaStream_t s) {
  k_state_step<<<(n + 127) / 128, 128, 0, s>>>(st, a, n, s_out);
  return cudaGetLastError();
}

__global__ void k_set_u64(uint64_t* p, uint64_t v) { *p = v; }

cudaError_t set_u64(uint64_t* p, uint64_t v, cudaStream_t s) {
  k_set_u64<<<1, 1, 0, s>>>(p, v);
  return cudaGetLastError();
}

__global__ void k_convert(const float* __restrict__ x, bf16* __restrict__ y, long long n) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    y[i] = __float2bfloat16_rn(x[i]);
}

cudaError_t convert_f32_bf16(const float* x, bf16* y, long long n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  long long blocks = (n + 255) / 256;
  if (blocks > 65535LL * 16) blocks = 65535LL * 16;
  k_convert<<<(unsigned)blocks, 256, 0, s>>>(x, y, n);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------
// fp32 SIMT GEMM (fp32 precision mode): C = A[M,K] * W[N,K]^T, 64x64 tiles, 4x4 per thread.
// The energy partial of a row is the fixed-order sum over the tile's 64 columns.
// ---------------------------------------------------------------------------------
constexpr int SG_BM = 64, SG_BN = 64, SG_BK = 16;

__global__ void __launch_bounds__(256) k_gemm_simt(const float* __restrict__ A,
                                                   const float* __restrict__ W, int M, int N,
                                                   int K, Epilogue epi) {
  __shared__ float As[SG_BK][SG_BM + 4];
  __shared__ float Ws[SG_BK][SG_BN + 4];
  __shared__ float red[SG_BM][SG_BN / 2 + 1];   // energy partials; gated: gelu(gate) tile
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * SG_BM, n0 = blockIdx.x * SG_BN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += SG_BK) {
    for (int i = threadIdx.x; i < SG_BM * SG_BK; i += 256) {
      const int r = i / SG_BK, kk = i % SG_BK;
      const int gr = m0 + r, gk = k0 + kk;
      As[kk][r] = (gr < M && gk < K) ? A[(long long)gr * K + gk] : 0.f;
      const int gn = n0 + r;
      Ws[kk][r] = (gn < N && gk < K) ? W[(long long)gn * K + gk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SG_BK; ++kk) {
      float a[4], w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = Ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
    }
    __syncthreads();
  }
  if (epi.mode == EPI_GATED) {
    // a 64-column tile is one FC1 block (threads tx < 8) and its gate block (tx >= 8):
    // the gate threads publish gelu(gate + b), the FC1 threads multiply and store
    float (*gate)[SG_BN / 2 + 1] = red;
    if (tx >= 8) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int col = n0 + tx * 4 + j;
          gate[ty * 4 + i][(tx - 8) * 4 + j] = col < N ? gelu_erf(acc[i][j] + epi.bias[col]) : 0.f;
        }
    }
    __syncthreads();
    if (tx < 8) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = m0 + ty * 4 + i;
        if (r >= M) continue;
        const long long off = map_row(epi.map0, r) * epi.ld0 + (n0 >> 1) + tx * 4;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int col = n0 + tx * 4 + j;
          if (col >= N) continue;
          const float h = (acc[i][j] + epi.bias[col]) * gate[ty * 4 + i][tx * 4 + j];
          if (epi.act_bf16)
            reinterpret_cast<bf16*>(epi.out0)[off + j] = __float2bfloat16_rn(h);
          else
            reinterpret_cast<float*>(epi.out0)[off + j] = h;
        }
      }
    }
    return;
  }
  const int c = n0 + tx * 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = m0 + ty * 4 + i;
    float s = 0.f;
    const EpiRow w = epi_row(epi, r, M, N);
    if (w.a >= 0 && c < N)
      s = epi_apply4(epi, w, c, make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]));
    red[ty * 4 + i][tx] = s;
  }
  if (epi.mode == EPI_OUTPROJ && epi.goal) {
    __syncthreads();
    if (threadIdx.x < SG_BM) {
      const int r = m0 + threadIdx.x;
      float s = 0.f;
      for (int j = 0; j < 16; ++j) s += red[threadIdx.x][j];
      if (r < M) epi.partial[(long long)r * epi.ntiles + blockIdx.x] = s;
    }
  }
}

int gemm_simt_partials(int N) { return (N + SG_BN - 1) / SG_BN; }

cudaError_t gemm_simt_f32(const float* A, const float* W, int M, int N, int K, const Epilogue& epi,
                          cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  if (epi.mode == EPI_GATED && (N % SG_BN != 0 || !epi.bias)) return cudaErrorInvalidValue;
  dim3 grid((N + SG_BN - 1) / SG_BN, (M + SG_BM - 1) / SG_BM);
  k_gemm_simt<<<grid, 256, 0, s>>>(A, W, M, N, K, epi);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------
// fp32 attention (fp32 mode): one warp per query row; scores in shared memory,
// max-subtracted softmax, then P*V with each lane owning head_dim/32 output columns.
// ---------------------------------------------------------------------------------
constexpr int FA32_WARPS = 8;

__global__ void __launch_bounds__(FA32_WARPS * 32) k_attention_f32(
    const float* __restrict__ q, const float* __restrict__ kv, float* __restrict__ o, int T, int Lk,
    long long kv_stride, int heads, int d, float scale) {
  extern __shared__ float sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * FA32_WARPS + warp;
  const int h = blockIdx.y, cand = blockIdx.z;
  const int hd = d / heads;
  if (t >= T) return;
  float* sc = sm + warp * Lk;
  const float* qr = q + ((long long)cand * T + t) * d + h * hd;
  const float* kb = kv + (long long)cand * kv_stride * 2 * d + h * hd;
  const float* vb = kb + d;
  float mx = -FLT_MAX;
  for (int j = lane; j < Lk; j += 32) {
    const float* kr = kb + (long long)j * 2 * d;
    float s = 0.f;
    for (int c = 0; c < hd; ++c) s = fmaf(qr[c], kr[c], s);
    s *= scale;
    sc[j] = s;
    mx = fmaxf(mx, s);
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  float sum = 0.f;
  for (int j = lane; j < Lk; j += 32) {
    const float p = expf(sc[j] - mx);
    sc[j] = p;
    sum += p;
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  __syncwarp();
  const float inv = 1.f / sum;
  for (int c = lane; c < hd; c += 32) {
    float acc = 0.f;
    for (int j = 0; j < Lk; ++j) acc = fmaf(sc[j], vb[(long long)j * 2 * d + c], acc);
    o[((long long)cand * T + t) * d + h * hd + c] = acc * inv;
  }
}

cudaError_t attention_f32(const float* q, const float* kv, float* o, int ncand, int T, int Lk,
                          long long kv_cand_stride_rows, int heads, int d, cudaStream_t s) {
  if (ncand <= 0) return cudaSuccess;
  const size_t smem = (size_t)FA32_WARPS * Lk * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_attention_f32,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid((T + FA32_WARPS - 1) / FA32_WARPS, heads, ncand);
  const float scale = 1.0f / sqrtf((float)(d / heads));
  k_attention_f32<<<grid, FA32_WARPS * 32, smem, s>>>(q, kv, o, T, Lk, kv_cand_stride_rows, heads, d,
                                                       scale);
  return cudaGetLastError();
}

// Failure-detection self-test: one thread waits on an mbarrier that nothing arrives on,
// through the same bounded wait every pipelined kernel uses; after its limit the wait gives
// up, raises the context's error flag and the kernel returns (no fault, no hang).
__global__ void k_wait_selftest(int* err_flag) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = tc::smem_u32(&bar);
  tc::mbar_init(b, 1);
  abort_flag = 0;
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  tc::mbar_wait(b, 0, &abort_flag, err_flag);
}

cudaError_t wait_selftest(int* err_flag, cudaStream_t s) {
  k_wait_selftest<<<1, 1, 0, s>>>(err_flag);
  return cudaGetLastError();
}

}  // namespace jepa
