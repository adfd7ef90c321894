// Block-causal flash attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA), head
// dim 64, over the query rows of one frame block (tiles of 128; the last may be partial).
//
// The predictor is frame-causal ("Real-time inference for JEPA world-model architectures
// with Ray", section "Measured on 8x A100": KV cache across rollout steps, bf16 with
// FlashAttention). Rollout step k computes the queries of frame block k only; they attend
// to every cached key row [0, Lk = (k+1) T) of their candidate, so the block-causal mask
// reduces to the key bound Lk.
//
// Persistent: each CTA walks work items (128-query tile, head, candidate), tile fastest so
// that the CTAs working on one candidate's K/V at the same time share it in L2. 6 warps:
//   warp 0      TMA producer: for each item its Q tile (double-buffered) and its 64-key K and
//               V chunks through a 4-stage ring. It runs ahead across item boundaries, so
//               the next item's loads hide behind the current item's math;
//   warp 1      TMEM allocator and single-thread MMA issuer:
//                 S = Q K^T   (M 128, N 64, K 64; both operands K-major, 128B-swizzled)
//                 O += P V    (M 128, N 64, K 64; P read from TMEM, V read MN-major
//                              straight from its TMA tile)
//               Chunk g's scores go to S buffer g % 2; the scores of chunk g + 2 are issued
//               right after P V of chunk g, which has consumed that buffer. This thread
//               bounds the kernel (it issues eight short MMAs per 64 keys), so it does
//               nothing else: it commits only S and P V completion;
//   warps 2-5   softmax, one query row per thread: read S from TMEM, online max / sum,
//               write P (bf16, two per column) over the first 32 columns of the same S
//               buffer, rescale O in TMEM, and at the end of an item normalise O and store it.
//               The exponentials of chunk g overlap P V of chunk g - 1: only the O rescale
//               (rare, see below) and the hand-over of P wait for it. Warp 2, having seen a
//               chunk's P V complete, also hands its K/V stage (and an item's Q tile after
//               its last chunk) back to the producer.
// TMEM: S / P buffers in columns [0, 64) and [192, 256), O of even items in [64, 128), of
// odd items in [128, 192). An item's output is read out (normalised, stored) right after
// the next item's first P hand-over, so the read-out overlaps that chunk's P V instead of
// delaying it; the P hand-over and P V completion barriers alternate by chunk parity, which
// keeps every warp within one phase of each barrier while it postpones that wait.
// In a partial last tile the rows of inactive warps keep stale words in P; their O rows
// are computed from them but never read. Keys past Lk are masked to
// -inf (their P is 0; the K/V rows loaded there are finite: cache rows are zero-initialised
// or belong to a neighbouring candidate, and rows past the tensor read as zero). In the last
// tile of a block whose T is not a multiple of 128, warps whose rows all lie past T skip the
// math. All mbarrier waits are bounded (error flag + early exit, as in the GEMM).
#include "common.cuh"
#include "tc_common.cuh"

namespace jepa {

namespace {

using namespace tc;

constexpr int AQ = 128;    // query rows per item (MMA M)
constexpr int AK = 64;     // keys per chunk
constexpr int AHD = 64;    // head dim
constexpr int A_THREADS = 192;
constexpr int KV_STAGES = 4;
constexpr int Q_BYTES = AQ * AHD * 2;     // 16 KB
constexpr int KV_BYTES = AK * AHD * 2;    // 8 KB (K or V chunk)
constexpr int OFF_Q = 0;                  // two Q buffers
constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
constexpr int OFF_V = OFF_K + KV_STAGES * KV_BYTES;
constexpr int OFF_BAR = OFF_V + KV_STAGES * KV_BYTES;
// q_full[2], q_empty[2], kv_full[S], kv_empty[S], s_full[2], p_full[2], o_full[2],
// o_free[2], teardown
constexpr int NUM_BARS = 4 + 2 * KV_STAGES + 2 + 2 + 2 + 2 + 1;
constexpr int A_SMEM = OFF_BAR + NUM_BARS * 8 + 16 + 1024;
constexpr uint32_t TMEM_COLS = 256;
constexpr int CTAS_PER_SM = 2;

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// max of three (sm_100-family three-input max.f32)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

}  // namespace

__global__ void __launch_bounds__(A_THREADS, CTAS_PER_SM)
    k_attention_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKV,
                   bf16* __restrict__ o, int T, int Lk, long long kv_stride_rows, int d,
                   float scale_log2, int nq, int heads, int ncand, int* err_flag) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar = sb + OFF_BAR;
  auto q_full = [&](int b) { return bar + 8u * b; };
  auto q_empty = [&](int b) { return bar + 8u * (2 + b); };
  auto kv_full = [&](int s) { return bar + 8u * (4 + s); };
  auto kv_empty = [&](int s) { return bar + 8u * (4 + KV_STAGES + s); };
  const uint32_t s_full0 = bar + 8u * (4 + 2 * KV_STAGES);
  auto s_full = [&](int b) { return s_full0 + 8u * b; };
  // chunk g's P hand-over and P V completion use barrier g % 2 of each pair: a warp is then
  // never more than one phase ahead on either, so it may postpone a wait on o_full
  auto p_full = [&](int b) { return s_full0 + 16 + 8u * b; };
  auto o_full = [&](int b) { return s_full0 + 32 + 8u * b; };
  auto o_free = [&](int b) { return s_full0 + 48 + 8u * b; };
  const uint32_t teardown = s_full0 + 64;
  uint32_t* tmem_slot = (uint32_t*)(smem + OFF_BAR + NUM_BARS * 8);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nch = (Lk + AK - 1) / AK;                 // key chunks per item
  const int items = nq * heads * ncand;
  // items of this CTA: it = blockIdx.x + i * gridDim.x, i = 0, 1, ...
  const int my_items = blockIdx.x < items ? (items - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  auto item_coords = [&](int i, int& qt, int& h, int& cand) {
    const int it = (int)blockIdx.x + i * (int)gridDim.x;
    qt = it % nq;
    h = (it / nq) % heads;
    cand = it / (nq * heads);
  };

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(q_full(b), 1);
      mbar_init(q_empty(b), 1);
      mbar_init(o_free(b), 4);
    }
    for (int s = 0; s < KV_STAGES; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
    }
    mbar_init(s_full(0), 1);
    mbar_init(s_full(1), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(p_full(b), 4);
      mbar_init(o_full(b), 1);
    }
    mbar_init(teardown, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto tS = [&](int g) { return tmem + ((g & 1) ? 192u : 0u); };   // S / P buffer of chunk g
  auto tO = [&](int i) { return tmem + 64u + 64u * (uint32_t)(i & 1); };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int g = 0;   // global chunk counter of this CTA
      bool ok = true;
      for (int i = 0; i < my_items && ok; ++i) {
        int qt, h, cand;
        item_coords(i, qt, h, cand);
        const int qb = i & 1;
        if (i >= 2 && !mbar_wait(q_empty(qb), ((i >> 1) - 1) & 1, abort_flag, err_flag)) break;
        mbar_expect_tx(q_full(qb), Q_BYTES);
        tma_load_2d(sb + OFF_Q + qb * Q_BYTES, &tmQ, h * AHD, cand * T + qt * AQ, q_full(qb));
        for (int j = 0; j < nch; ++j, ++g) {
          const int st = g % KV_STAGES;
          if (g >= KV_STAGES &&
              !mbar_wait(kv_empty(st), ((g / KV_STAGES) - 1) & 1, abort_flag, err_flag)) {
            ok = false;
            break;
          }
          const int ky = (int)(cand * kv_stride_rows + (long long)j * AK);
          mbar_expect_tx(kv_full(st), 2 * KV_BYTES);
          tma_load_2d(sb + OFF_K + st * KV_BYTES, &tmKV, h * AHD, ky, kv_full(st));
          tma_load_2d(sb + OFF_V + st * KV_BYTES, &tmKV, d + h * AHD, ky, kv_full(st));
        }
      }
      if (*abort_flag) {
        // give copies still in flight into this CTA's shared memory time to land
        const unsigned long long t0 = globaltimer();
        while (globaltimer() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t idS = idesc_bf16(AQ, AK, false);
      constexpr uint32_t idO = idesc_bf16(AQ, AHD, true);
      const int total = my_items * nch;
      // (item, chunk within the item) of the chunk being multiplied by V and of the next
      // chunk whose scores are issued, advanced by counting (no divisions on this thread,
      // which bounds the kernel)
      auto advance = [&](int& it, int& jj) {
        if (++jj == nch) {
          jj = 0;
          ++it;
        }
      };
      auto issue_s = [&](int gg, int it) {   // chunk gg of item it, whose Q sits in buffer it & 1
        const uint64_t qdesc = desc_sw128(sb + OFF_Q + (it & 1) * Q_BYTES);
        const uint64_t kdesc = desc_sw128(sb + OFF_K + (gg % KV_STAGES) * KV_BYTES);
#pragma unroll
        for (int kk = 0; kk < AHD / 16; ++kk)
          mma_bf16_ss(tS(gg), qdesc + 2 * kk, kdesc + 2 * kk, idS, kk > 0);
        mma_commit(s_full(gg & 1));
      };
      auto ready_s = [&](int gg, int it, int jj) {   // operands of S for chunk gg in shared memory
        if (jj == 0 && !mbar_wait(q_full(it & 1), (it >> 1) & 1, abort_flag, err_flag)) return false;
        return mbar_wait(kv_full(gg % KV_STAGES), (gg / KV_STAGES) & 1, abort_flag, err_flag);
      };
      bool ok = true;
      int si = 0, sj = 0;   // next chunk whose scores are issued
      for (int gg = 0; gg < 2 && gg < total && ok; ++gg) {
        ok = ready_s(gg, si, sj);
        if (ok) {
          tc_fence_after();
          issue_s(gg, si);
          advance(si, sj);
        }
      }
      int ii = 0, j = 0;
      for (int gg = 0; gg < total && ok; ++gg, advance(ii, j)) {
        if (!mbar_wait(p_full(gg & 1), (gg >> 1) & 1, abort_flag, err_flag)) break;
        // the O buffer of this item was last read out for item ii - 2
        if (j == 0 && ii >= 2 && !mbar_wait(o_free(ii & 1), ((ii >> 1) - 1) & 1, abort_flag, err_flag))
          break;
        tc_fence_after();
        const uint64_t vdesc = desc_sw128_mn(sb + OFF_V + (gg % KV_STAGES) * KV_BYTES);
#pragma unroll
        for (int kk = 0; kk < AK / 16; ++kk)  // 16 keys: 8 TMEM columns of P, 16 rows x 128 B of V
          mma_bf16_ts(tO(ii), tS(gg) + 8u * kk, vdesc + (uint64_t)(kk * (2048 >> 4)), idO,
                      (j > 0) || (kk > 0));
        mma_commit(o_full(gg & 1));
        // the K/V stage and (after an item's last chunk) the Q buffer are released by softmax
        // warp 2 once it has seen this P V complete, which keeps those commits off this thread
        // tensor-core operations of this thread run in issue order, so the scores of chunk
        // gg + 2 overwrite this S / P buffer only after the P V above has read it
        if (gg + 2 < total) {
          if (!ready_s(gg + 2, si, sj)) break;
          tc_fence_after();
          issue_s(gg + 2, si);
          advance(si, sj);
        }
      }
      mma_commit(teardown);
      const unsigned long long t0 = globaltimer();
      while (!mbar_try_wait(teardown, 0) && globaltimer() - t0 < WAIT_LIMIT_NS) {
      }
    }
  } else {
    // ---------------- softmax warps 2..5 (thread = query row) ----------------
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    auto po_wait = [&](int gc) {   // P V of chunk gc complete
      return mbar_wait(o_full(gc & 1), (gc >> 1) & 1, abort_flag, err_flag);
    };
    // An item's output is read out after the next item's first P hand-over, so that the
    // read-out overlaps that chunk's P V instead of delaying it.
    struct Pending {
      int i, qt, h, cand, glast;
      bool active;
      float l;
    } pend = {-1, 0, 0, 0, 0, false, 0.f};
    auto finish_item = [&](const Pending& it) {
      if (!po_wait(it.glast)) return false;
      tc_fence_after();
      if (warp == 2 && lane == 0) {
        mbar_arrive(kv_empty(it.glast % KV_STAGES));   // the item's last K/V stage
        mbar_arrive(q_empty(it.i & 1));                 // and its Q tile
      }
      if (it.active) {
        const float inv = 1.f / it.l;
        const int t = it.qt * AQ + row;
        bf16* orow = o + ((long long)it.cand * T + t) * d + it.h * AHD;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t ov[32];
          tmem_ld32_async(tO(it.i) + lane_off + 32 * hf, ov);
          tmem_wait(ov);
          if (t < T) {
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
              uint4 u;
              __nv_bfloat162 p0 = __floats2bfloat162_rn(__uint_as_float(ov[c]) * inv, __uint_as_float(ov[c + 1]) * inv);
              __nv_bfloat162 p1 = __floats2bfloat162_rn(__uint_as_float(ov[c + 2]) * inv, __uint_as_float(ov[c + 3]) * inv);
              __nv_bfloat162 p2 = __floats2bfloat162_rn(__uint_as_float(ov[c + 4]) * inv, __uint_as_float(ov[c + 5]) * inv);
              __nv_bfloat162 p3 = __floats2bfloat162_rn(__uint_as_float(ov[c + 6]) * inv, __uint_as_float(ov[c + 7]) * inv);
              u.x = *reinterpret_cast<uint32_t*>(&p0);
              u.y = *reinterpret_cast<uint32_t*>(&p1);
              u.z = *reinterpret_cast<uint32_t*>(&p2);
              u.w = *reinterpret_cast<uint32_t*>(&p3);
              *reinterpret_cast<uint4*>(orow + 32 * hf + c) = u;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free(it.i & 1));
      return true;
    };
    bool ok = true;
    int g = 0;
    for (int i = 0; i < my_items && ok; ++i) {
      int qt, h, cand;
      item_coords(i, qt, h, cand);
      // a warp whose 32 query rows all lie past T (last, partial tile) skips the math but
      // keeps the same barrier sequence, so its arrivals never count toward another phase
      const bool active = (qt * AQ + quarter * 32) < T;
      const uint32_t tOi = tO(i);
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nch; ++j, ++g) {
        const uint32_t tSg = tS(g);
        if (!mbar_wait(s_full(g & 1), (g >> 1) & 1, abort_flag, err_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (!active) {
          if (j > 0) {
            if (!po_wait(g - 1)) {
              ok = false;
              break;
            }
            if (warp == 2 && lane == 0) mbar_arrive(kv_empty((g - 1) % KV_STAGES));
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(p_full(g & 1));
          if (j == 0 && pend.i >= 0) {
            if (!finish_item(pend)) {
              ok = false;
              break;
            }
            pend.i = -1;
          }
          continue;
        }
        uint32_t sa[32], sc[32];
        tmem_ld32_async(tSg + lane_off, sa);
        tmem_ld32_async(tSg + lane_off + 32, sc);
        tmem_wait(sa);
        tmem_wait(sc);
        float s[64];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          s[c] = __uint_as_float(sa[c]);
          s[32 + c] = __uint_as_float(sc[c]);
        }
        const int kv_left = Lk - j * AK;
        if (kv_left < AK) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c >= kv_left) s[c] = -INFINITY;
        }
        // row max as a tree of three-input maxima (8 independent chains, then combine)
        float part[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          part[q] = fmax3(fmax3(s[8 * q], s[8 * q + 1], s[8 * q + 2]),
                          fmax3(s[8 * q + 3], s[8 * q + 4], s[8 * q + 5]), fmaxf(s[8 * q + 6], s[8 * q + 7]));
        const float cmax = fmax3(fmax3(part[0], part[1], part[2]), fmax3(part[3], part[4], part[5]),
                                 fmaxf(part[6], part[7]));
        // The exponent reference m only moves when the row max grows by more than 8 (log2
        // units): until then P = 2^(s c - m c) stays <= 256, and since the same m scales the
        // numerator (O) and the denominator (l), the result is unchanged. Most chunks then
        // skip the O rescale in TMEM.
        const bool bump = (m == -INFINITY) || ((cmax - m) * scale_log2 > 8.0f);
        const float mnew = bump ? fmaxf(m, cmax) : m;
        const float alpha = ex2f((m - mnew) * scale_log2);   // 1 when m is kept, 0 at j = 0
        const float ms = mnew * scale_log2;
        // exponentiate and sum, packing P as bf16 pairs (key 2c in the low half of column c);
        // the exponent arguments and the row sum in packed f32x2 arithmetic
        uint32_t pk[32];
        unsigned long long rsp[8];
        const unsigned long long sc2 = f2_pack(scale_log2, scale_log2), nms2 = f2_pack(-ms, -ms);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          float e[8];
          if (8 * cc >= kv_left) {
            // every key of this group lies past Lk: P is exactly 0
#pragma unroll
            for (int t = 0; t < 8; ++t) e[t] = 0.f;
          } else {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const float2 a = f2_unpack(f2_fma(f2_pack(s[8 * cc + 2 * t], s[8 * cc + 2 * t + 1]), sc2, nms2));
              e[2 * t] = ex2f(a.x);
              e[2 * t + 1] = ex2f(a.y);
            }
          }
          rsp[cc] = f2_add(f2_add(f2_pack(e[0], e[1]), f2_pack(e[2], e[3])),
                           f2_add(f2_pack(e[4], e[5]), f2_pack(e[6], e[7])));
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            __nv_bfloat162 pp = __floats2bfloat162_rn(e[2 * t], e[2 * t + 1]);
            pk[4 * cc + t] = *reinterpret_cast<uint32_t*>(&pp);
          }
        }
        // S of this chunk is in registers: P takes its first 32 columns
        tmem_st32(tSg + lane_off, pk);
        const float2 rs2 = f2_unpack(f2_add(f2_add(f2_add(rsp[0], rsp[1]), f2_add(rsp[2], rsp[3])),
                                            f2_add(f2_add(rsp[4], rsp[5]), f2_add(rsp[6], rsp[7]))));
        const float rs = rs2.x + rs2.y;
        l = l * alpha + rs;
        m = mnew;
        // P V of the previous chunk must be complete before O is rescaled and P handed over;
        // its K/V stage is then free for the producer
        if (j > 0) {
          if (!po_wait(g - 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (warp == 2 && lane == 0) mbar_arrive(kv_empty((g - 1) % KV_STAGES));
        }
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
          uint32_t ov[32], ow[32];
          tmem_ld32_async(tOi + lane_off, ov);
          tmem_ld32_async(tOi + lane_off + 32, ow);
          tmem_wait(ov);
          tmem_wait(ow);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
            ow[c] = __float_as_uint(__uint_as_float(ow[c]) * alpha);
          }
          tmem_st32(tOi + lane_off, ov);
          tmem_st32(tOi + lane_off + 32, ow);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full(g & 1));
        if (j == 0 && pend.i >= 0) {
          if (!finish_item(pend)) {
            ok = false;
            break;
          }
          pend.i = -1;
        }
      }
      if (!ok) break;
      pend = Pending{i, qt, h, cand, g - 1, active, l};
    }
    if (ok && pend.i >= 0) finish_item(pend);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    __syncwarp();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

cudaError_t attention_tc_bf16(const bf16* q, const bf16* kv, bf16* o, int ncand, int T, int Lk,
                              long long kv_cand_stride_rows, int heads, int d, int* err_flag,
                              cudaStream_t s) {
  if (ncand <= 0) return cudaSuccess;
  const int nq = (T + AQ - 1) / AQ;
  if (d != heads * AHD || d % 8) return cudaErrorInvalidValue;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = set_max_dynamic_smem((const void*)k_attention_tc, A_SMEM, attr_done);
  if (e != cudaSuccess) return e;
  static std::atomic<int> sms_of_device[64];   // SM count per device ordinal, 0 = not read yet
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  int num_sms = (dev >= 0 && dev < 64) ? sms_of_device[dev].load(std::memory_order_relaxed) : 0;
  if (num_sms <= 0) {
    if ((e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    if (dev >= 0 && dev < 64) sms_of_device[dev].store(num_sms, std::memory_order_relaxed);
  }
  CUtensorMap mq, mkv;
  if (!make_map(&mq, q, ncand * T, d, AQ, AHD) ||
      !make_map(&mkv, kv, (int)(ncand * kv_cand_stride_rows), 2 * d, AK, AHD))
    return cudaErrorInvalidValue;
  const long long items = (long long)nq * heads * ncand;
  const long long slots = (long long)num_sms * CTAS_PER_SM;
  const int grid = (int)(items < slots ? items : slots);
  const float scale_log2 = (1.0f / 8.0f) * 1.4426950408889634f;  // 1/sqrt(64) * log2(e)
  k_attention_tc<<<grid, A_THREADS, A_SMEM, s>>>(mq, mkv, o, T, Lk, kv_cand_stride_rows, d,
                                                  scale_log2, nq, heads, ncand, err_flag);
  return cudaGetLastError();
}

}  // namespace jepa
