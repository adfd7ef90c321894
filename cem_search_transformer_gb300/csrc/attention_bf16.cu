// Block-causal flash-style attention over the per-candidate KV cache, bf16, head dim 64.
//
// The predictor is frame-causal ("Real-time inference for JEPA world-model architectures
// with Ray", section "Measured on 8x A100": KV cache across rollout steps, bf16 with
// FlashAttention). Rollout step k only computes the queries of frame block k; they see
// every key of blocks 0..k, which the cache holds as rows [0, (k+1)*T). So the block-causal
// mask reduces to a key-length bound Lk, and no per-element mask is needed.
//
// One CTA = 4 warps = 64 query rows of one (candidate, head); each warp owns 16 rows.
// K/V tiles of 64 keys are double-buffered with cp.async; S = Q K^T and O += P V use
// mma.sync m16n8k16 (bf16 in, fp32 accumulate) with an online (running-max) softmax.
#include "common.cuh"

namespace jepa {

namespace {

constexpr int BQ = 64, BKV = 64, HD = 64, LD = HD + 8;  // smem row stride (elements) avoids bank conflicts

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                            const void* p) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(s));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3, const void* p) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(s));
}
__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// 2^x on the special-function unit (flush-to-zero; relative error ~2^-22)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

}  // namespace

__global__ void __launch_bounds__(128) k_attention_bf16(const bf16* __restrict__ q,
                                                        const bf16* __restrict__ kv,
                                                        bf16* __restrict__ o, int T, int Lk,
                                                        long long kv_stride_rows, int d,
                                                        float scale_log2) {
  __shared__ __align__(128) bf16 Qs[BQ * LD];
  __shared__ __align__(128) bf16 Ks[2][BKV * LD];
  __shared__ __align__(128) bf16 Vs[2][BKV * LD];
  const int qt = blockIdx.x, h = blockIdx.y, cand = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bf16* qb = q + (long long)cand * T * d + h * HD;
  const bf16* kb = kv + (long long)cand * kv_stride_rows * 2 * d + h * HD;
  const bf16* vb = kb + d;
  const uint4 zero = make_uint4(0, 0, 0, 0);

  for (int i = threadIdx.x; i < BQ * (HD / 8); i += blockDim.x) {
    const int r = i >> 3, ch = i & 7;
    const int t = qt * BQ + r;
    bf16* dst = Qs + r * LD + ch * 8;
    if (t < T)
      cp_async16(dst, qb + (long long)t * d + ch * 8);
    else
      *reinterpret_cast<uint4*>(dst) = zero;
  }
  // each thread copies 16-byte chunk (tid & 7) of key rows (tid >> 3) + 16 s, s = 0..3
  const int ld_row = threadIdx.x >> 3, ld_ch = threadIdx.x & 7;
  const bf16* kg = kb + (long long)ld_row * 2 * d + ld_ch * 8;
  const long long key_step = 16LL * 2 * d;    // 16 key rows
  const int sm_off = ld_row * LD + ld_ch * 8;
  auto load_kv = [&](int j, int st) {
    const bf16* g0 = kg + (long long)j * BKV * 2 * d;
    const int key0 = j * BKV + ld_row;
#pragma unroll
    for (int s2 = 0; s2 < BKV / 16; ++s2) {
      bf16* dk = Ks[st] + sm_off + s2 * 16 * LD;
      bf16* dv = Vs[st] + sm_off + s2 * 16 * LD;
      if (key0 + 16 * s2 < Lk) {
        const bf16* gk = g0 + s2 * key_step;
        cp_async16(dk, gk);
        cp_async16(dv, gk + d);
      } else {
        *reinterpret_cast<uint4*>(dk) = zero;
        *reinterpret_cast<uint4*>(dv) = zero;
      }
    }
  };
  load_kv(0, 0);
  cp_async_commit();

  const int nkv = (Lk + BKV - 1) / BKV;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  uint32_t qf[4][4];
  const int g = lane >> 2, tq = lane & 3;

  // warps whose 16 query rows all lie past T only help with the loads
  const bool active = (qt * BQ + warp * 16) < T;
  for (int j = 0; j < nkv; ++j) {
    if (j + 1 < nkv) {
      load_kv(j + 1, (j + 1) & 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (!active) {
      __syncthreads();
      continue;
    }
    // key blocks of 8 (S) and 16 (P V) that hold at least one valid key of this tile; the
    // skipped ones would contribute exp(-inf) = 0 exactly
    const int kv_left = Lk - j * BKV;
    const int nbv = kv_left >= BKV ? 8 : (kv_left + 7) / 8;
    const int kcv = kv_left >= BKV ? 4 : (kv_left + 15) / 16;
    if (j == 0) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        ldmatrix_x4(qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3],
                    Qs + (warp * 16 + (lane & 15)) * LD + kk * 16 + ((lane >> 4) << 3));
    }
    const bf16* Kst = Ks[j & 1];
    const bf16* Vst = Vs[j & 1];
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int nb = 0; nb < 8; nb += 2) {
        if (nb >= nbv) continue;
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(b0, b1, b2, b3,
                    Kst + (nb * 8 + ((lane >> 4) << 3) + (lane & 7)) * LD + kk * 16 +
                        (((lane >> 3) & 1) << 3));
        mma_bf16(s[nb], qf[kk], b0, b1);
        mma_bf16(s[nb + 1], qf[kk], b2, b3);
      }
    }
    if (kv_left < BKV) {
      // only the tile that crosses Lk needs masking
#pragma unroll
      for (int nb = 0; nb < 8; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (j * BKV + nb * 8 + 2 * tq + (e & 1) >= Lk) s[nb][e] = -INFINITY;
    }
    // running max on raw scores (the positive scale does not change the order); the scale
    // is folded into one FFMA per element below
    float mx[2] = {m_run[0], m_run[1]};
#pragma unroll
    for (int nb = 0; nb < 8; ++nb) {
      mx[0] = fmaxf(mx[0], fmaxf(s[nb][0], s[nb][1]));
      mx[1] = fmaxf(mx[1], fmaxf(s[nb][2], s[nb][3]));
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    }
    const float alpha0 = ex2((m_run[0] - mx[0]) * scale_log2);
    const float alpha1 = ex2((m_run[1] - mx[1]) * scale_log2);
    m_run[0] = mx[0];
    m_run[1] = mx[1];
    const float ms0 = mx[0] * scale_log2, ms1 = mx[1] * scale_log2;
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int nb = 0; nb < 8; ++nb) {
      s[nb][0] = ex2(fmaf(s[nb][0], scale_log2, -ms0));
      s[nb][1] = ex2(fmaf(s[nb][1], scale_log2, -ms0));
      s[nb][2] = ex2(fmaf(s[nb][2], scale_log2, -ms1));
      s[nb][3] = ex2(fmaf(s[nb][3], scale_log2, -ms1));
      rs0 += s[nb][0] + s[nb][1];
      rs1 += s[nb][2] + s[nb][3];
    }
    l_run[0] = l_run[0] * alpha0 + rs0;
    l_run[1] = l_run[1] * alpha1 + rs1;
#pragma unroll
    for (int db = 0; db < 8; ++db) {
      acc[db][0] *= alpha0;
      acc[db][1] *= alpha0;
      acc[db][2] *= alpha1;
      acc[db][3] *= alpha1;
    }
#pragma unroll
    for (int kc = 0; kc < 4; ++kc) {
      if (kc >= kcv) continue;
      uint32_t a[4];
      a[0] = pack_bf16(s[2 * kc][0], s[2 * kc][1]);
      a[1] = pack_bf16(s[2 * kc][2], s[2 * kc][3]);
      a[2] = pack_bf16(s[2 * kc + 1][0], s[2 * kc + 1][1]);
      a[3] = pack_bf16(s[2 * kc + 1][2], s[2 * kc + 1][3]);
#pragma unroll
      for (int db = 0; db < 8; db += 2) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(b0, b1, b2, b3,
                          Vst + (kc * 16 + (((lane >> 3) & 1) << 3) + (lane & 7)) * LD + db * 8 +
                              ((lane >> 4) << 3));
        mma_bf16(acc[db], a, b0, b1);
        mma_bf16(acc[db + 1], a, b2, b3);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
    l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
  }
  if (!active) return;
  const float inv0 = 1.f / l_run[0], inv1 = 1.f / l_run[1];
  const int t0 = qt * BQ + warp * 16 + g, t1 = t0 + 8;
  bf16* ob = o + (long long)cand * T * d + h * HD;
#pragma unroll
  for (int db = 0; db < 8; ++db) {
    const int c = db * 8 + 2 * tq;
    if (t0 < T)
      *reinterpret_cast<__nv_bfloat162*>(ob + (long long)t0 * d + c) =
          __floats2bfloat162_rn(acc[db][0] * inv0, acc[db][1] * inv0);
    if (t1 < T)
      *reinterpret_cast<__nv_bfloat162*>(ob + (long long)t1 * d + c) =
          __floats2bfloat162_rn(acc[db][2] * inv1, acc[db][3] * inv1);
  }
}

cudaError_t attention_bf16(const bf16* q, const bf16* kv, bf16* o, int ncand, int T, int Lk,
                           long long kv_cand_stride_rows, int heads, int d, cudaStream_t s) {
  if (ncand <= 0) return cudaSuccess;
  if (d != heads * HD) return cudaErrorInvalidValue;
  dim3 grid((T + BQ - 1) / BQ, heads, ncand);
  const float scale_log2 = (1.0f / 8.0f) * 1.4426950408889634f;  // 1/sqrt(64) * log2(e)
  k_attention_bf16<<<grid, 128, 0, s>>>(q, kv, o, T, Lk, kv_cand_stride_rows, d, scale_log2);
  return cudaGetLastError();
}

}  // namespace jepa
