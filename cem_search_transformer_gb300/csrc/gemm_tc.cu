// Tensor-core GEMM for the predictor's linear layers on sm_103a:
//   out = epilogue(A[M,K] * W[N,K]^T), A and W bf16 (K-major), fp32 accumulation in TMEM.
//
// Design (GB300-first; the planning pages only say "bf16"):
//   - persistent CTAs (one per SM) walk 128 x BN output tiles, m-major so the CTAs that run
//     at the same time share A row blocks in L2 (W is at most a few MB and stays in L2);
//   - warp 0: TMA producer (128B-swizzled 128x64 A and BNx64 W boxes into a STAGES-deep ring);
//   - warp 1: TMEM allocator and single-thread tcgen05.mma issuer (M=128, N=BN, K=16 per
//     instruction), committing to "smem empty" barriers and to a per-accumulator "full" barrier;
//   - warps 2..: epilogue, EW warps in all (8, or 16 for the GELU and gated layers whose
//     erf is the expensive part), EW/4 warps per TMEM lane quarter, each taking a 4/EW
//     share of the tile's columns. A warp reads 32 rows x 32 columns with tcgen05.ld
//     32x32b.x32 (thread = row) and releases the accumulator with a relaxed arrive once its
//     last TMEM load has landed. The GELU and gated epilogues (and, on CTA pairs, the QKV
//     store) apply bias and activation in that layout and stage only bf16 results, in the
//     64-byte swizzle of a 32 x 32 TMA box: on CTA pairs a TMA store writes each chunk
//     (K/V cache rows through a 3-D map of the cache's per-candidate blocks). The residual
//     epilogue of CTA pairs loads each 32 x 32 chunk of x by TMA into a 128-byte-swizzled
//     buffer, adds accumulator and bias per lane in place and stores it back by TMA. The
//     single-CTA kernel's other epilogues transpose fp32 accumulators through a swizzled
//     4 KB shared-memory buffer so that each global access covers contiguous columns of a
//     row, and apply bias / residual / position / L1 energy (see common.cuh) four columns
//     at a time. The next chunk's TMEM load is in flight while the current chunk is
//     processed.
//   - two TMEM accumulators (2 x BN columns) so the epilogue of tile i overlaps the MMAs of
//     tile i+1;
//   - QKV, the MLP up-projection and the residual projections run on CTA pairs
//     (k_gemm_tc2: 256 x 256 tiles with tcgen05.mma.cta_group::2, A loaded with an L2
//     evict_last policy so that the pairs sharing a row block find it in L2), the
//     projections to and from the embedding space and small or ragged shapes on single
//     CTAs (k_gemm_tc).
// Every mbarrier wait is bounded by a wall-clock limit; on expiry the kernel records an
// error flag, stops issuing work, waits (bounded) for its own copies and MMAs, frees TMEM
// and returns.
#include "common.cuh"
#include "tc_common.cuh"

namespace jepa {

namespace {

using namespace tc;

constexpr int BM = 128, BK = 64;
constexpr int STG_FLOATS = 32 * 32;                     // per-warp transpose buffer

// Epilogue warps per CTA for an epilogue mode, and the CTA size (producer + MMA warps too).
__host__ __device__ constexpr int epi_warps(int mode) {
  return (mode == EPI_GELU || mode == EPI_GATED) ? 16 : 8;
}
__host__ __device__ constexpr int cta_threads(int mode) { return 64 + 32 * epi_warps(mode); }
// Per-warp staging floats: the GELU and gated epilogues transpose bf16 results (32 rows x
// 64 B), the others fp32 accumulators (32 x 32 x 4 B).
__host__ __device__ constexpr int stg_floats(int mode) {
  return (mode == EPI_GELU || mode == EPI_GATED) ? 512 : STG_FLOATS;
}

template <int BN, int MODE>
struct Cfg {
  static constexpr int EW = epi_warps(MODE);
  // the projection to E stages goal chunks (two 32 x 32 fp32 TMA boxes per warp) in the
  // transpose buffer's place when it computes energies only
  static constexpr int STG = MODE == EPI_OUTPROJ ? 2 * STG_FLOATS : stg_floats(MODE);
  static constexpr int XBARS = MODE == EPI_OUTPROJ ? 2 * EW : 0;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // as many ring stages (up to 6) as the shared memory left by the staging buffers holds
  static constexpr int FIT =
      (232448 - 1024 - 16 - (5 + XBARS) * 8 - EW * STG * 4) / (STAGE_BYTES + 16);
  static constexpr int STAGES = FIT < 6 ? FIT : 6;
  static constexpr int TMEM_COLS = 2 * BN;   // two accumulators; 256 or 512 (power of 2)
  // ring, epilogue transpose buffers, barriers (full/empty per stage, tfull/tempty per
  // accumulator, teardown), TMEM address slot + abort flag, 1024 B alignment slack
  static constexpr int STG_OFF = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFF = STG_OFF + EW * STG * 4;
  static constexpr int SMEM = BAR_OFF + (2 * STAGES + 5 + XBARS) * 8 + 16 + 1024;
  static_assert(STAGES >= 3 && SMEM <= 232448, "shared memory budget");
};

// Residual tiles of the CTA-pair residual epilogue: 32 rows x 32 fp32 columns (4 KB, one
// TMA box) per buffer, RES_BUFS buffers per epilogue warp.
constexpr int RES_BUFS = 2;
constexpr int RES_FLOATS = 32 * 32;

// 2-SM tiles: a CTA pair computes 256 x 256 (each CTA 128 rows, all 256 columns in its TMEM);
// each CTA stages its own 128 rows of A and its own 128-row half of W per K step. The
// residual mode stages x through TMA buffers instead of a transpose buffer, with one
// mbarrier per buffer.
template <int MODE>
struct Cfg2 {
  static constexpr int EW = epi_warps(MODE);
  static constexpr int STG = MODE == EPI_RESID ? RES_BUFS * RES_FLOATS
                             : MODE == EPI_STORE ? 512   // bf16 rows, as GELU
                                                 : stg_floats(MODE);
  static constexpr int XBARS = MODE == EPI_RESID ? EW * RES_BUFS : 0;
  static constexpr int A_BYTES = BM * BK * 2;   // 16 KB
  static constexpr int B_BYTES = 128 * BK * 2;  // 16 KB: this CTA's half of the 256 columns
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int FIT =
      (232448 - 1024 - 16 - (5 + XBARS) * 8 - EW * STG * 4) / (STAGE_BYTES + 16);
  static constexpr int STAGES = FIT < 6 ? FIT : 6;
  static constexpr int TMEM_COLS = 512;         // two 256-column accumulators
  static constexpr int STG_OFF = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFF = STG_OFF + EW * STG * 4;
  static constexpr int SMEM = BAR_OFF + (2 * STAGES + 5 + XBARS) * 8 + 16 + 1024;
  static_assert(SMEM <= 232448, "shared memory budget");
};

}  // namespace

// Epilogue of one accumulator tile held in TMEM (rows m0 .. m0+127 of this CTA, columns of
// tile n_blk), executed by every epilogue warp. Waits for `tfull` (parity), releases the
// accumulator through `release(tempty)` as soon as its last TMEM load has landed, then
// finishes the global stores. Returns false if a bounded wait expired.

// Stores 32 consecutive output columns [c0, c0 + 32) of rows row_base .. row_base + 31,
// lane i holding row row_base + i in v[0..31]. bf16 output goes through the warp's staging
// buffer (32 rows x 64 B, 16-byte pieces swizzled by row) so that the global stores are
// row-contiguous; fp32 output (the C-ABI linear layer) is stored row by row.
// With a 2-D output map (tmO) the staged chunk leaves by one TMA store. With a 3-D map of the
// K/V cache (tmC: columns, row within a block of map.rpg rows, block), the rows that lie in
// the first row's block leave by one TMA store (clipped at the block end) and the rest, which
// belong to the next candidate, by per-lane stores.
__device__ __forceinline__ bool store_rows32(void* out, long long ld, const RowMap& map,
                                             int act_bf16, int M, int N, int row_base, int c0,
                                             const float (&v)[32], float* stg_f, int lane,
                                             const CUtensorMap* tmO, bool drain,
                                             const CUtensorMap* tmC = nullptr) {
  const int row = row_base + lane;
  if (!act_bf16) {
    if (row < M) {
      float* orow = reinterpret_cast<float*>(out) + map_row(map, row) * ld;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (c0 + 4 * k < N)
          *reinterpret_cast<float4*>(orow + c0 + 4 * k) =
              make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
    }
    return true;
  }
  uint8_t* stg = reinterpret_cast<uint8_t*>(stg_f);
  if (drain) {
    // the buffer is rewritten once an earlier chunk's TMA store has read it
    if (lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
  }
  // row `lane`, 16-byte piece q (8 columns) at byte lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4),
  // which is the 64-byte swizzle of a 32 x 32 bf16 TMA box
  const int swz = (lane >> 1) & 3;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    __nv_bfloat162 h0 = __floats2bfloat162_rn(v[8 * q], v[8 * q + 1]);
    __nv_bfloat162 h1 = __floats2bfloat162_rn(v[8 * q + 2], v[8 * q + 3]);
    __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * q + 4], v[8 * q + 5]);
    __nv_bfloat162 h3 = __floats2bfloat162_rn(v[8 * q + 6], v[8 * q + 7]);
    u.x = *reinterpret_cast<uint32_t*>(&h0);
    u.y = *reinterpret_cast<uint32_t*>(&h1);
    u.z = *reinterpret_cast<uint32_t*>(&h2);
    u.w = *reinterpret_cast<uint32_t*>(&h3);
    *reinterpret_cast<uint4*>(stg + lane * 64 + ((q ^ swz) << 4)) = u;
  }
  if (tmO) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && row_base < M) {
      tma_store_2d(tmO, smem_u32(stg), c0, row_base);
      bulk_commit_group();
    }
    return true;
  }
  int lsu_from = 0;   // first staged row written by per-lane stores
  if (tmC && row_base + 32 <= M) {
    const int blk_row = row_base % map.rpg;
    lsu_from = map.rpg - blk_row < 32 ? map.rpg - blk_row : 32;
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      const long long blk = (long long)(row_base / map.rpg) * (map.gstride / map.rpg) + map.goff / map.rpg;
      tma_store_3d(tmC, smem_u32(stg), c0, blk_row, (int)blk);
      bulk_commit_group();
    }
    if (lsu_from == 32) return true;
  }
  __syncwarp();
  // 128 pieces of 16 bytes; lane takes pieces lane + 32 i: rows (lane >> 2) + 8 i, piece lane & 3
  const int q = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int rr = (lane >> 2) + 8 * i;
    const uint4 u = *reinterpret_cast<const uint4*>(stg + rr * 64 + ((q ^ ((rr >> 1) & 3)) << 4));
    const int grow = row_base + rr;
    const int col = c0 + 8 * q;
    if (rr >= lsu_from && grow < M && col < N) {
      bf16* dst = reinterpret_cast<bf16*>(out) + map_row(map, grow) * ld + col;
      if (col + 8 <= N) {
        *reinterpret_cast<uint4*>(dst) = u;
      } else {                                // N % 8 == 4: the last 4 columns
        *reinterpret_cast<uint2*>(dst) = make_uint2(u.x, u.y);
      }
    }
  }
  __syncwarp();
  return true;
}

// Gated-MLP epilogue (EPI_GATED, 256-column tiles, 16 epilogue warps): each warp owns a
// 32-row quarter and 64 accumulator columns, i.e. exactly one FC1 block and the gate block
// that follows it in the interleaved weight. Per half of 16 columns the lane loads its row's
// FC1 and gate values from TMEM and forms (fc1 + b) * gelu(gate + b); the row's 32 outputs
// then leave like the GELU epilogue's (bf16 staging, row-contiguous stores).
template <int EW, int OP, typename Release>
__device__ __forceinline__ bool epilogue_tile_gated(const Epilogue& epi, int M, int N, int m0,
                                                    int n_blk, uint32_t tmem_acc, uint32_t tfull,
                                                    uint32_t tfull_parity, uint32_t tempty,
                                                    Release release, float* stg_f, int ew,
                                                    int warp, int lane, volatile int* abort_flag,
                                                    int* err_flag, const CUtensorMap* tmO) {
  static_assert(EW == 16, "one FC1/gate block pair per epilogue warp");
  const int quarter = warp & 3;
  const int part = ew >> 2;                  // block pair within the 256-column tile
  const int cbase = n_blk * 256 + part * 64; // FC1 block; the gate block is cbase + 32
  const int ocol = (cbase >> 1);             // first output column of this pair
  const bool active = cbase < N;
  if (!mbar_wait(tfull, tfull_parity, abort_flag, err_flag)) return false;
  tc_fence_after();
  const uint32_t tbase = tmem_acc + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(part * 64);
  float rs = 1.f;                            // fp8: this lane's row scale
  if constexpr (OP) rs = (m0 + quarter * 32 + lane < M) ? epi.row_scale[m0 + quarter * 32 + lane] : 0.f;
  uint32_t r[32];
  float v[32];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    if (active) {
      tmem_ld16_async(tbase + 16u * half, r);
      tmem_ld16_async(tbase + 32u + 16u * half, r + 16);
    }
    tmem_wait(r);
    if (half == 1) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) release(tempty);
    }
    if (!active) continue;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int c = cbase + 16 * half + 4 * k;
      const float4 b1 = __ldg(reinterpret_cast<const float4*>(epi.bias + c));
      const float4 bg = __ldg(reinterpret_cast<const float4*>(epi.bias + c + 32));
      float4 f = make_float4(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1]),
                             __uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3]));
      float4 q = make_float4(__uint_as_float(r[16 + 4 * k]), __uint_as_float(r[16 + 4 * k + 1]),
                             __uint_as_float(r[16 + 4 * k + 2]), __uint_as_float(r[16 + 4 * k + 3]));
      if constexpr (OP) {
        const float4 c1 = __ldg(reinterpret_cast<const float4*>(epi.col_scale + c));
        const float4 cg = __ldg(reinterpret_cast<const float4*>(epi.col_scale + c + 32));
        f.x *= rs * c1.x; f.y *= rs * c1.y; f.z *= rs * c1.z; f.w *= rs * c1.w;
        q.x *= rs * cg.x; q.y *= rs * cg.y; q.z *= rs * cg.z; q.w *= rs * cg.w;
      }
      const unsigned long long g01 = gelu2x(f2_add(f2_pack(q.x, q.y), f2_pack(bg.x, bg.y)));
      const unsigned long long g23 = gelu2x(f2_add(f2_pack(q.z, q.w), f2_pack(bg.z, bg.w)));
      const float2 o01 = f2_unpack(f2_mul(f2_add(f2_pack(f.x, f.y), f2_pack(b1.x, b1.y)), g01));
      const float2 o23 = f2_unpack(f2_mul(f2_add(f2_pack(f.z, f.w), f2_pack(b1.z, b1.w)), g23));
      float* o = v + 16 * half + 4 * k;
      o[0] = o01.x;
      o[1] = o01.y;
      o[2] = o23.x;
      o[3] = o23.y;
    }
  }
  if (!active) return true;
  return store_rows32(epi.out0, epi.ld0, epi.map0, epi.act_bf16, M, N, m0 + quarter * 32, ocol, v,
                      stg_f, lane, tmO, tmO != nullptr);
}

// Row-per-lane epilogue (EPI_GELU; EPI_STORE in the CTA-pair kernel): each lane owns one
// accumulator row. Bias (and GELU) are applied in that layout straight from TMEM (the bias is
// the same for every lane: broadcast loads), and only the bf16 results go through the warp's
// staging buffer (32 rows x 64 B, 16-byte pieces swizzled by row), from which a TMA store
// (out0 with identity rows, when the launcher made its tensor map) or row-contiguous
// global stores write them. Staging bf16 instead of fp32 halves the buffer, which leaves
// room for one more stage of the operand ring. With fp32 output (the C-ABI linear layer)
// rows are stored directly. A STORE chunk goes to out0 or out1 by its columns (split).
template <int BN, int EW, int OP, bool GELU, typename Release>
__device__ __forceinline__ bool epilogue_tile_rows(const Epilogue& epi, int M, int N, int m0,
                                                   int n_blk, uint32_t tmem_acc, uint32_t tfull,
                                                   uint32_t tfull_parity, uint32_t tempty,
                                                   Release release, float* stg_f, int ew, int warp,
                                                   int lane, volatile int* abort_flag,
                                                   int* err_flag, const CUtensorMap* tmO,
                                                   const CUtensorMap* tmC) {
  const int quarter = warp & 3;
  const int part = ew >> 2;
  constexpr int SPAN = BN * 4 / EW;          // columns per epilogue warp
  const int cbase = n_blk * BN + part * SPAN;
  int nvalid = 0;
  while (nvalid < SPAN / 32 && cbase + 32 * nvalid < N) ++nvalid;
  if (!mbar_wait(tfull, tfull_parity, abort_flag, err_flag)) return false;
  tc_fence_after();
  const uint32_t tbase = tmem_acc + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(part * SPAN);
  const int row_base = m0 + quarter * 32;
  float rs = 1.f;                            // fp8: this lane's row scale
  if constexpr (OP) rs = (row_base + lane < M) ? epi.row_scale[row_base + lane] : 0.f;
  uint32_t r[32];
  if (nvalid > 0) tmem_ld32_async(tbase, r);
#pragma unroll
  for (int j = 0; j < SPAN / 32; ++j) {
    if (j >= nvalid) break;
    tmem_wait(r);
    if (j == nvalid - 1) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) release(tempty);
    }
    const int c0 = cbase + 32 * j;
    float v[32];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = c0 + 4 * k;
      const float4 b = (epi.bias && c < N) ? __ldg(reinterpret_cast<const float4*>(epi.bias + c))
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
      float4 a = make_float4(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1]),
                             __uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3]));
      if constexpr (OP) {
        const float4 cs = c < N ? __ldg(reinterpret_cast<const float4*>(epi.col_scale + c))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        a.x *= rs * cs.x; a.y *= rs * cs.y; a.z *= rs * cs.z; a.w *= rs * cs.w;
      }
      unsigned long long x01 = f2_add(f2_pack(a.x, a.y), f2_pack(b.x, b.y));
      unsigned long long x23 = f2_add(f2_pack(a.z, a.w), f2_pack(b.z, b.w));
      if constexpr (GELU) {
        x01 = gelu2x(x01);
        x23 = gelu2x(x23);
      }
      const float2 g01 = f2_unpack(x01), g23 = f2_unpack(x23);
      v[4 * k] = g01.x;
      v[4 * k + 1] = g01.y;
      v[4 * k + 2] = g23.x;
      v[4 * k + 3] = g23.y;
    }
    if (j + 1 < nvalid) tmem_ld32_async(tbase + 32u * (j + 1), r);   // r is free again
    // a chunk goes wholly to out0 or to out1 (split is a multiple of 32); only out0 may have
    // an output tensor map
    if (c0 >= epi.split)
      store_rows32(epi.out1, epi.ld1, epi.map1, epi.act_bf16, M, N - epi.split, row_base,
                   c0 - epi.split, v, stg_f, lane, nullptr, tmO != nullptr || tmC != nullptr, tmC);
    else
      store_rows32(epi.out0, epi.ld0, epi.map0, epi.act_bf16, M, N, row_base, c0, v, stg_f, lane,
                   tmO, tmO != nullptr || tmC != nullptr);
  }
  if (nvalid == 0) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) release(tempty);
  }
  return true;
}

template <int BN, int MODE, int EW, int OP, bool PAIR, typename Release>
__device__ __forceinline__ bool epilogue_tile(const Epilogue& epi, int M, int N, int m0, int n_blk,
                                              uint32_t tmem_acc, uint32_t tfull,
                                              uint32_t tfull_parity, uint32_t tempty,
                                              Release release, float* stg, int ew, int warp,
                                              int lane, volatile int* abort_flag, int* err_flag,
                                              const CUtensorMap* tmO = nullptr,
                                              const CUtensorMap* tmC = nullptr) {
  if constexpr (MODE == EPI_GATED) {
    static_assert(BN == 256, "gated tiles hold four FC1/gate block pairs");
    return epilogue_tile_gated<EW, OP>(epi, M, N, m0, n_blk, tmem_acc, tfull, tfull_parity,
                                       tempty, release, stg, ew, warp, lane, abort_flag, err_flag,
                                       tmO);
  } else if constexpr (MODE == EPI_GELU) {
    return epilogue_tile_rows<BN, EW, OP, true>(epi, M, N, m0, n_blk, tmem_acc, tfull, tfull_parity,
                                                 tempty, release, stg, ew, warp, lane, abort_flag,
                                                 err_flag, tmO, nullptr);
  } else if constexpr (MODE == EPI_STORE && PAIR) {
    return epilogue_tile_rows<BN, EW, OP, false>(epi, M, N, m0, n_blk, tmem_acc, tfull, tfull_parity,
                                                  tempty, release, stg, ew, warp, lane, abort_flag,
                                                  err_flag, tmO, tmC);
  } else {
  const int quarter = warp & 3;              // TMEM lanes quarter*32 .. +31
  const int part = ew >> 2;                  // which share of the tile's columns
  constexpr int SPAN = BN * 4 / EW;          // columns per epilogue warp
  const int cg = lane & 7;                   // column group (4 columns) in the transposed phase
  const int rsub = lane >> 3;                // rows rsub + 4 i, i = 0..7
  constexpr bool kStore = (MODE == EPI_STORE || MODE == EPI_GELU);
  constexpr bool kResid = (MODE == EPI_RESID);
  constexpr bool kGeneric = !kStore && !kResid;
  const bool has_operand = kResid || MODE == EPI_INPROJ || (MODE == EPI_OUTPROJ && epi.goal != nullptr);
  // row addressing and the first chunk's global operands are prepared before the
  // accumulator is ready, so their latency hides behind this tile's MMAs
  const int cbase = n_blk * BN + part * SPAN;
  const int row0 = m0 + quarter * 32 + rsub;
  // per-row element offsets: a = destination (out0 / x), b = out1 (STORE) or generic use
  long long ra[8], rb[8];
  uint32_t vmask = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = row0 + 4 * i;
    if (r < M) vmask |= 1u << i;
    if constexpr (kStore) {
      ra[i] = map_row(epi.map0, r) * epi.ld0;
      rb[i] = epi.out1 ? map_row(epi.map1, r) * epi.ld1 : 0;
    } else if constexpr (kResid) {
      ra[i] = map_row(epi.map0, r) * epi.ld0;
      rb[i] = 0;
    } else {
      const EpiRow w = epi_row(epi, r, M, N);
      ra[i] = w.a;
      rb[i] = w.b;
    }
  }
  float esum[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) esum[i] = 0.f;
  // fp8 operands: per-row (activation) and per-column (weight) scales of the accumulators;
  // the row scales are read where they are used (L1-resident), not held in registers
  int nvalid = 0;
  while (nvalid < SPAN / 32 && cbase + 32 * nvalid < N) ++nvalid;
  float4 nxt[8], nbias = make_float4(0.f, 0.f, 0.f, 0.f), ncs = make_float4(0.f, 0.f, 0.f, 0.f);
  auto fetch = [&](int c) {
    const bool ok = c < N;
    nbias = ok ? epi_bias4(epi, c) : make_float4(0.f, 0.f, 0.f, 0.f);
    if constexpr (OP)
      ncs = ok ? __ldg(reinterpret_cast<const float4*>(epi.col_scale + c)) : make_float4(0.f, 0.f, 0.f, 0.f);
    if constexpr (kResid) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        nxt[i] = (ok && ((vmask >> i) & 1))
                     ? *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(epi.out0) + ra[i] + c)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    } else if constexpr (kGeneric) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        EpiRow w;
        w.a = ((vmask >> i) & 1) ? ra[i] : -1;
        w.b = rb[i];
        nxt[i] = (ok && has_operand) ? epi_load4(epi, w, c) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  };
  if (nvalid > 0) fetch(cbase + 4 * cg);
  if (!mbar_wait(tfull, tfull_parity, abort_flag, err_flag)) return false;
  tc_fence_after();
  const uint32_t tbase =
      tmem_acc + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(part * SPAN);
  uint32_t r[32];
  if (nvalid > 0) tmem_ld32_async(tbase, r);
#pragma unroll
  for (int j = 0; j < SPAN / 32; ++j) {
    if (j >= nvalid) break;
    tmem_wait(r);
    if (j == nvalid - 1) {
      // accumulator fully read: hand it back to the MMA warp before finishing the stores
      tc_fence_before();
      __syncwarp();
      if (lane == 0) release(tempty);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k)
      *reinterpret_cast<float4*>(stg + lane * 32 + ((k ^ (lane & 7)) << 2)) =
          make_float4(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1]),
                      __uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3]));
    __syncwarp();
    if (j + 1 < nvalid) tmem_ld32_async(tbase + 32u * (j + 1), r);
    const int cchunk = cbase + 32 * j;
    const int c = cchunk + 4 * cg;
    const bool col_ok = c < N;
    float4 cur[8];
    const float4 bb = nbias;
    const float4 cs = ncs;
    if constexpr (!kStore) {
#pragma unroll
      for (int i = 0; i < 8; ++i) cur[i] = nxt[i];
    }
    if (j + 1 < nvalid) fetch(c + 32);   // next chunk's operands while this one is processed
    // the whole 32-column chunk goes to one destination (split is a multiple of 32)
    const bool second = kStore && cchunk >= epi.split;
    const int col = second ? c - epi.split : c;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = rsub + 4 * i;
      float4 v = *reinterpret_cast<const float4*>(stg + rr * 32 + ((cg ^ (rr & 7)) << 2));
      if (!(((vmask >> i) & 1) && col_ok)) continue;
      if constexpr (OP) {
        const float rsi = __ldg(epi.row_scale + row0 + 4 * i);
        v.x *= rsi * cs.x; v.y *= rsi * cs.y; v.z *= rsi * cs.z; v.w *= rsi * cs.w;
      }
      v.x += bb.x; v.y += bb.y; v.z += bb.z; v.w += bb.w;
      if constexpr (kStore) {
        if (MODE == EPI_GELU) v = gelu4(v);
        const long long off = (second ? rb[i] : ra[i]) + col;
        if (epi.act_bf16) {
          __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
          __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
          uint2 u;
          u.x = *reinterpret_cast<uint32_t*>(&lo);
          u.y = *reinterpret_cast<uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(reinterpret_cast<bf16*>(second ? epi.out1 : epi.out0) + off) = u;
        } else {
          *reinterpret_cast<float4*>(reinterpret_cast<float*>(second ? epi.out1 : epi.out0) + off) = v;
        }
      } else if constexpr (kResid) {
        float4 x = cur[i];
        x.x += v.x; x.y += v.y; x.z += v.z; x.w += v.w;
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(epi.out0) + ra[i] + c) = x;
      } else {
        EpiRow w;
        w.a = ra[i];
        w.b = rb[i];
        esum[i] += epi_apply4(epi, w, c, v, make_float4(0.f, 0.f, 0.f, 0.f), cur[i]);
      }
    }
    __syncwarp();
  }
  if (nvalid == 0) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) release(tempty);
  }
  if constexpr (MODE == EPI_OUTPROJ) {
    if (epi.goal) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float sum = esum[i];
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        const int row = row0 + 4 * i;
        if (cg == 0 && row < M)
          epi.partial[(long long)row * epi.ntiles + (EW / 4) * n_blk + part] = sum;
      }
    }
  }
  return true;
  }
}

// Energy-only epilogue of the projection to E (EPI_OUTPROJ with a goal and no z outputs) in
// the single-CTA kernel, run by each epilogue warp over all of its tiles. Per 32 x 32 chunk
// the goal rows of the chunk's candidate (32 consecutive goal rows, as P is a multiple of
// 32) arrive by TMA in one of two 128-byte-swizzled buffers, loaded two chunks ahead across
// tile boundaries; each lane takes its accumulator row from TMEM (thread = row), forms
// z = acc (* scales) + bias and sums |z - goal| over the warp's columns of the tile in
// column order, and writes that sum as the row's partial for the tile and column share.
// Reading the goal per element through L1 limited the projection (883 us per full-size
// launch, 629 without the goal reads).
template <int BN, int EW, int OP, typename Release>
__device__ __forceinline__ bool epilogue_energy_tma(const CUtensorMap* tmG, const Epilogue& epi,
                                                    int M, int N, int num_n, int total,
                                                    uint32_t tmem_base, const uint32_t (&tfull)[2],
                                                    const uint32_t (&tempty)[2], Release release,
                                                    float* bufs, uint32_t gbar0, int ew, int warp,
                                                    int lane, volatile int* abort_flag,
                                                    int* err_flag) {
  constexpr int SPAN = BN * 4 / EW;          // columns per epilogue warp and tile
  constexpr int NCH = SPAN / 32;             // 32-column chunks per tile
  constexpr int NB = 2;                      // goal buffers per warp
  const int quarter = warp & 3, part = ew >> 2;
  const int bid = blockIdx.x, nblk = gridDim.x;
  const int my_tiles = bid < total ? (total - 1 - bid) / nblk + 1 : 0;
  const int nchunks = my_tiles * NCH;
  const uint32_t buf0 = smem_u32(bufs);
  auto chunk_rc = [&](int g, int& row_base, int& c0) {
    const int t = bid + (g / NCH) * nblk;
    row_base = (t / num_n) * BM + quarter * 32;
    c0 = (t % num_n) * BN + part * SPAN + 32 * (g % NCH);
  };
  auto issue_goal = [&](int g) {   // lane 0 only
    if (g >= nchunks) return;
    const uint32_t bar = gbar0 + 8u * (g % NB);
    int row_base, c0;
    chunk_rc(g, row_base, c0);
    if (row_base < M && c0 < N) {
      const int cand = epi.cand0 + row_base / epi.P;
      const int grow = (cand / epi.cands_per_problem) * epi.P + row_base % epi.P;
      mbar_expect_tx(bar, STG_FLOATS * 4);
      tma_load_2d(buf0 + (g % NB) * STG_FLOATS * 4, tmG, c0, grow, bar);
    } else {
      mbar_arrive(bar);   // nothing of this chunk is used
    }
  };
  if (lane == 0)
    for (int g = 0; g < NB; ++g) issue_goal(g);
  bool ok = true;
  int acc = 0;
  uint32_t acc_phase = 0;
  for (int i = 0; i < my_tiles && ok; ++i) {
    const int t = bid + i * nblk;
    const int row = (t / num_n) * BM + quarter * 32 + lane;
    const int n_blk = t % num_n;
    const uint32_t tbase =
        tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(part * SPAN);
    if (!mbar_wait(tfull[acc], acc_phase, abort_flag, err_flag)) {
      ok = false;
      break;
    }
    tc_fence_after();
    float rs = 1.f;                          // fp8: this lane's row scale
    if constexpr (OP) rs = row < M ? epi.row_scale[row] : 0.f;
    uint32_t r[32];
    tmem_ld32_async(tbase, r);
    float esum = 0.f;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int g = i * NCH + j;
      tmem_wait(r);
      if (j == NCH - 1) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release(tempty[acc]);
      }
      if (!mbar_wait(gbar0 + 8u * (g % NB), (uint32_t)(g / NB) & 1u, abort_flag, err_flag)) {
        ok = false;
        break;
      }
      int row_base, c0;
      chunk_rc(g, row_base, c0);
      // row `lane` of the goal box: 16-byte piece k at k ^ (lane & 7) (128-byte swizzle)
      const float* grow_s = bufs + (g % NB) * STG_FLOATS + lane * 32;
      float4 gv[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) gv[k] = *reinterpret_cast<const float4*>(grow_s + ((k ^ (lane & 7)) << 2));
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) issue_goal(g + NB);     // the buffer has been read by every lane
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int c = c0 + 4 * k;
        if (c >= N) break;
        float4 v = make_float4(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1]),
                               __uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3]));
        if constexpr (OP) {
          const float4 cs = __ldg(reinterpret_cast<const float4*>(epi.col_scale + c));
          v.x *= rs * cs.x; v.y *= rs * cs.y; v.z *= rs * cs.z; v.w *= rs * cs.w;
        }
        const float4 bb = epi_bias4(epi, c);
        v.x += bb.x; v.y += bb.y; v.z += bb.z; v.w += bb.w;
        esum += ((fabsf(v.x - gv[k].x) + fabsf(v.y - gv[k].y)) + fabsf(v.z - gv[k].z)) +
                fabsf(v.w - gv[k].w);
      }
      if (j + 1 < NCH) tmem_ld32_async(tbase + 32u * (j + 1), r);   // r is free again
    }
    if (!ok) break;
    if (row < M) epi.partial[(long long)row * epi.ntiles + (EW / 4) * n_blk + part] = esum;
    if (++acc == 2) acc = 0, acc_phase ^= 1u;
  }
  if (!ok && lane == 0) {
    // goal loads may still be in flight into this CTA's shared memory: let them land
    const unsigned long long t0 = globaltimer();
    while (globaltimer() - t0 < 2000000ull) {
    }
  }
  __syncwarp();
  return ok;
}

// Residual epilogue of the CTA-pair kernel (EPI_RESID: x[r, c] += acc + bias; x fp32 with
// the identity row map and row stride N), run by each epilogue warp over all of its tiles.
// Global loads through L1 limit the bytes a warp can keep in flight, and x is read and
// written once per element, so each warp moves its 32-row x 32-column chunks of x with TMA
// instead: the chunk lands in one of RES_BUFS swizzled shared-memory buffers (loads run
// RES_BUFS - 1 chunks ahead, across tile boundaries), each lane adds its accumulator row
// (tcgen05.ld, thread = row) and the bias to its row of the buffer in place, and the buffer
// leaves by a TMA store. Lane 0 issues the copies; rows past M read as zero and are not
// stored. Returns false if a bounded wait expired.
template <int EW, typename Release>
__device__ __forceinline__ bool epilogue_resid_tma(const CUtensorMap* tmX, const Epilogue& epi,
                                                   int M, int rank, int cid, int ncl, int num_n,
                                                   int total, uint32_t tmem_base,
                                                   const uint32_t (&tfull)[2],
                                                   const uint32_t (&tempty)[2], Release release,
                                                   float* bufs, uint32_t xbar0, int ew, int warp,
                                                   int lane, volatile int* abort_flag,
                                                   int* err_flag) {
  constexpr int BN = 256;
  constexpr int SPAN = BN * 4 / EW;          // columns per epilogue warp and tile
  constexpr int NCH = SPAN / 32;             // 32-column chunks per tile
  const int quarter = warp & 3, part = ew >> 2;
  const int my_tiles = cid < total ? (total - 1 - cid) / ncl + 1 : 0;
  const int nchunks = my_tiles * NCH;
  const uint32_t buf0 = smem_u32(bufs);
  // chunk g of this warp: tile cid + (g / NCH) ncl, columns 32 (g % NCH) of the warp's share
  auto chunk_xy = [&](int g, int& x, int& y) {
    const int t = cid + (g / NCH) * ncl;
    y = (t / num_n) * 2 * BM + rank * BM + quarter * 32;
    x = (t % num_n) * BN + part * SPAN + 32 * (g % NCH);
  };
  auto issue_load = [&](int g) {   // lane 0 only
    if (g >= nchunks) return;
    const int b = g % RES_BUFS;
    int x, y;
    chunk_xy(g, x, y);
    if (y < M) {
      mbar_expect_tx(xbar0 + 8u * b, RES_FLOATS * 4);
      tma_load_2d(buf0 + b * RES_FLOATS * 4, tmX, x, y, xbar0 + 8u * b);
    } else {
      mbar_arrive(xbar0 + 8u * b);   // all 32 rows past M: nothing to load or store
    }
  };
  if (lane == 0)
    for (int g = 0; g < RES_BUFS; ++g) issue_load(g);
  bool ok = true;
  int acc = 0;
  uint32_t acc_phase = 0;
  for (int i = 0; i < my_tiles && ok; ++i) {
    const uint32_t tbase =
        tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(part * SPAN);
    if (!mbar_wait(tfull[acc], acc_phase, abort_flag, err_flag)) {
      ok = false;
      break;
    }
    tc_fence_after();
    uint32_t r[32];
    tmem_ld32_async(tbase, r);
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int g = i * NCH + j;
      const int b = g % RES_BUFS;
      tmem_wait(r);
      if (j == NCH - 1) {
        // accumulator fully read: hand it back to the MMA warp before finishing the stores
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release(tempty[acc]);
      }
      if (!mbar_wait(xbar0 + 8u * b, (uint32_t)(g / RES_BUFS) & 1u, abort_flag, err_flag)) {
        ok = false;
        break;
      }
      int x, y;
      chunk_xy(g, x, y);
      // row `lane` of the buffer: 16-byte piece k at k ^ (lane & 7) (128-byte swizzle)
      float* row = bufs + b * RES_FLOATS + lane * 32;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float4* pp = reinterpret_cast<float4*>(row + ((k ^ (lane & 7)) << 2));
        const float4 bb = epi_bias4(epi, x + 4 * k);
        float4 xv = *pp;
        xv.x += __uint_as_float(r[4 * k]) + bb.x;
        xv.y += __uint_as_float(r[4 * k + 1]) + bb.y;
        xv.z += __uint_as_float(r[4 * k + 2]) + bb.z;
        xv.w += __uint_as_float(r[4 * k + 3]) + bb.w;
        *pp = xv;
      }
      if (j + 1 < NCH) tmem_ld32_async(tbase + 32u * (j + 1), r);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (y < M) {
          tma_store_2d(tmX, buf0 + b * RES_FLOATS * 4, x, y);
          bulk_commit_group();
        }
        // the buffer is refilled once the store has read it
        bulk_wait_group_read<0>();
        issue_load(g + RES_BUFS);
      }
      __syncwarp();
    }
    if (++acc == 2) acc = 0, acc_phase ^= 1u;
  }
  if (lane == 0) {
    bulk_wait_group_all();
    if (!ok) {
      // loads may still be in flight into this CTA's shared memory: let them land
      const unsigned long long t0 = globaltimer();
      while (globaltimer() - t0 < 2000000ull) {
      }
    }
  }
  __syncwarp();
  return ok;
}

// OP 0: bf16 operands (kind::f16, 64 elements of K per 128-byte row); OP 1: fp8 e4m3
// operands (kind::f8f6f4, 128 elements per row) with per-row / per-column scales applied in
// the epilogue. Stages hold the same bytes either way.
template <int BN, int MODE, int OP>
__global__ void __launch_bounds__(cta_threads(MODE), 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmX, int M, int N, int K, Epilogue epi,
              int* err_flag) {
  constexpr int EW = epi_warps(MODE);
  using C = Cfg<BN, MODE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::BAR_OFF;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + 2 + a); };
  const uint32_t teardown_bar = bar0 + 8u * (2 * C::STAGES + 4);
  const uint32_t xbar0 = bar0 + 8u * (2 * C::STAGES + 5);   // goal buffers (EPI_OUTPROJ)
  uint32_t* tmem_slot = (uint32_t*)(smem + C::BAR_OFF + (2 * C::STAGES + 5 + C::XBARS) * 8);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_n = (N + BN - 1) / BN;
  const int num_m = (M + BM - 1) / BM;
  const int total = num_m * num_n;
  constexpr int BKE = OP ? 2 * BK : BK;        // K elements per stage (128 bytes per row)
  const int num_k = (K + BKE - 1) / BKE;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), EW);   // one arrival per epilogue warp
    }
    mbar_init(teardown_bar, 1);
    for (int b = 0; b < C::XBARS; ++b) mbar_init(xbar0 + 8u * b, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"((uint32_t)C::TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase[8];
      bool issued[8];
      for (int s = 0; s < 8; ++s) issued[s] = false, issued_phase[s] = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const int m0 = (t / num_n) * BM, n0 = (t % num_n) * BN;
        for (int kb = 0; kb < num_k; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, err_flag)) {
            ok = false;
            break;
          }
          const uint32_t sa = sbase + stage * C::STAGE_BYTES;
          mbar_expect_tx(full_bar(stage), C::STAGE_BYTES);
          tma_load_2d(sa, &tmA, kb * BKE, m0, full_bar(stage));
          tma_load_2d(sa + C::A_BYTES, &tmB, kb * BKE, n0, full_bar(stage));
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == C::STAGES) stage = 0, phase ^= 1u;
        }
      }
      if (!ok) {
        // drain: wait (bounded) until every copy this thread started has landed
        for (int s = 0; s < C::STAGES; ++s) {
          if (!issued[s]) continue;
          const unsigned long long t0 = globaltimer();
          while (!mbar_try_wait(full_bar(s), issued_phase[s]) &&
                 globaltimer() - t0 < WAIT_LIMIT_NS) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t idesc = OP ? idesc_e4m3(BM, BN) : idesc_bf16(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, err_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < num_k; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag, err_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = sbase + stage * C::STAGE_BYTES;
          const uint64_t adesc = desc_sw128(sa);
          const uint64_t bdesc = desc_sw128(sa + C::A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // advance 32 bytes along K inside the swizzle atom (+2 in 16-byte units): 16 bf16
            // or 32 e4m3 elements per MMA
            if constexpr (OP)
              mma_e4m3_ss(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb | kk) != 0);
            else
              mma_bf16_ss(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb | kk) != 0);
          }
          mma_commit(empty_bar(stage));
          if (++stage == C::STAGES) stage = 0, phase ^= 1u;
        }
        if (!ok) break;
        mma_commit(tfull_bar(acc));
        if (++acc == 2) acc = 0, acc_phase ^= 1u;
      }
      // all MMAs issued by this thread complete before TMEM is released
      mma_commit(teardown_bar);
      const unsigned long long t0 = globaltimer();
      while (!mbar_try_wait(teardown_bar, 0) && globaltimer() - t0 < WAIT_LIMIT_NS) {
      }
    }
  } else {
    // ---------------- epilogue (warps 2..) ----------------
    const int ew = warp - 2;
    float* stg = reinterpret_cast<float*>(smem + C::STG_OFF) + ew * C::STG;
    int acc = 0;
    uint32_t acc_phase = 0;
    auto release = [](uint32_t bar) { mbar_arrive_relaxed(bar); };
    bool streamed = false;   // all tiles done by the energy epilogue
    if constexpr (MODE == EPI_OUTPROJ) {
      if (epi.tma_out & 4) {
        const uint32_t tf[2] = {tfull_bar(0), tfull_bar(1)};
        const uint32_t te[2] = {tempty_bar(0), tempty_bar(1)};
        epilogue_energy_tma<BN, EW, OP>(&tmX, epi, M, N, num_n, total, tmem_base, tf, te, release,
                                        stg, xbar0 + 8u * (ew * 2), ew, warp, lane, abort_flag,
                                        err_flag);
        streamed = true;
      }
    }
    for (int t = blockIdx.x; t < total && !streamed; t += gridDim.x) {
      const int m0 = (t / num_n) * BM, n_blk = t % num_n;
      if (!epilogue_tile<BN, MODE, EW, OP, false>(epi, M, N, m0, n_blk, tmem_base + (uint32_t)(acc * BN),
                                       tfull_bar(acc), acc_phase, tempty_bar(acc), release, stg, ew,
                                       warp, lane, abort_flag, err_flag))
        break;
      if (++acc == 2) acc = 0, acc_phase ^= 1u;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"((uint32_t)C::TMEM_COLS));
  }
}

// 2-SM GEMM: clusters of 2 CTAs walk 256 x 256 output tiles. Both CTAs stage their halves;
// the leader (cluster rank 0) issues tcgen05.mma.cta_group::2 (M 256, N 256, K 16) and commits
// to the "smem empty" and "accumulator full" barriers of both CTAs; each CTA's epilogue drains
// its own 128 rows and releases the accumulator on the leader's barrier. Halving the operand
// bytes each SM stages per MMA keeps shared-memory traffic within its bandwidth.
template <int MODE, int OP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(cta_threads(MODE), 1)
    k_gemm_tc2(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
               int M, int N, int K, Epilogue epi, int* err_flag) {
  constexpr int EW = epi_warps(MODE);
  constexpr int BN = 256;
  using C = Cfg2<MODE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::BAR_OFF;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + 2 + a); };
  const uint32_t teardown_bar = bar0 + 8u * (2 * C::STAGES + 4);
  const uint32_t xbar0 = bar0 + 8u * (2 * C::STAGES + 5);   // residual buffers (EPI_RESID)
  uint32_t* tmem_slot = (uint32_t*)(smem + C::BAR_OFF + (2 * C::STAGES + 5 + C::XBARS) * 8);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  const int num_n = (N + BN - 1) / BN;
  const int num_m = (M + 2 * BM - 1) / (2 * BM);
  const int total = num_m * num_n;
  constexpr int BKE = OP ? 2 * BK : BK;        // K elements per stage (128 bytes per row)
  const int num_k = (K + BKE - 1) / BKE;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), 1);     // the leader's arrive + both CTAs' transaction bytes
      mbar_init(empty_bar(s), 1);    // the leader's MMA commit (multicast)
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 2 * EW);   // epilogue warps of both CTAs (used in the leader)
    }
    mbar_init(teardown_bar, 1);
    for (int b = 0; b < C::XBARS; ++b) mbar_init(xbar0 + 8u * b, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), (uint32_t)C::TMEM_COLS);
  tc_fence_before();
  cluster_sync();   // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs) ----------------
      int stage = 0;
      uint32_t phase = 0;
      bool issued_any = false;
      // A rows are read by the num_n CTA pairs that share a row block, at times that drift
      // apart over a long K loop: keep them in L2 ahead of the streaming epilogue traffic
      const uint64_t a_policy = l2_policy_evict_last();
      for (int t = cid; t < total; t += ncl) {
        const int m0 = (t / num_n) * 2 * BM + (int)rank * BM, n0 = (t % num_n) * BN + (int)rank * 128;
        bool ok = true;
        for (int kb = 0; kb < num_k; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, err_flag)) {
            ok = false;
            break;
          }
          const uint32_t sa = sbase + stage * C::STAGE_BYTES;
          const uint32_t lfull = map_to_rank(full_bar(stage), 0);
          if (rank == 0) mbar_expect_tx(full_bar(stage), 2 * C::STAGE_BYTES);
          tma_load_2d_pair_hint(sa, &tmA, kb * BKE, m0, lfull, a_policy);
          tma_load_2d_pair(sa + C::A_BYTES, &tmB, kb * BKE, n0, lfull);
          issued_any = true;
          if (++stage == C::STAGES) stage = 0, phase ^= 1u;
        }
        if (!ok) break;
      }
      if (*abort_flag && issued_any) {
        // let copies still in flight into this CTA's shared memory land before exiting
        const unsigned long long t0 = globaltimer();
        while (globaltimer() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (leader only) ----------------
      constexpr uint32_t idesc = OP ? idesc_e4m3(2 * BM, BN) : idesc_bf16(2 * BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = cid; t < total && ok; t += ncl) {
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, err_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < num_k; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag, err_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = sbase + stage * C::STAGE_BYTES;
          const uint64_t adesc = desc_sw128(sa);
          const uint64_t bdesc = desc_sw128(sa + C::A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            if constexpr (OP)
              mma_e4m3_pair(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb | kk) != 0);
            else
              mma_bf16_pair(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb | kk) != 0);
          }
          mma_commit_pair_both(empty_bar(stage));
          if (++stage == C::STAGES) stage = 0, phase ^= 1u;
        }
        if (!ok) break;
        mma_commit_pair_both(tfull_bar(acc));
        if (++acc == 2) acc = 0, acc_phase ^= 1u;
      }
      mma_commit_pair_local(teardown_bar);
      const unsigned long long t0 = globaltimer();
      while (!mbar_try_wait(teardown_bar, 0) && globaltimer() - t0 < WAIT_LIMIT_NS) {
      }
    }
  } else {
    // ---------------- epilogue (warps 2.., both CTAs) ----------------
    const int ew = warp - 2;
    float* stg = reinterpret_cast<float*>(smem + C::STG_OFF) + ew * C::STG;
    int acc = 0;
    uint32_t acc_phase = 0;
    auto release = [](uint32_t bar) { mbar_arrive_cluster_relaxed(bar); };
    if constexpr (MODE == EPI_RESID) {
      const uint32_t tf[2] = {tfull_bar(0), tfull_bar(1)};
      const uint32_t te[2] = {map_to_rank(tempty_bar(0), 0), map_to_rank(tempty_bar(1), 0)};
      epilogue_resid_tma<EW>(&tmX, epi, M, (int)rank, cid, ncl, num_n, total, tmem_base, tf, te,
                             release, stg, xbar0 + 8u * (ew * RES_BUFS), ew, warp, lane,
                             abort_flag, err_flag);
    } else {
      const CUtensorMap* tmO = (epi.tma_out & 1) ? &tmX : nullptr;
      const CUtensorMap* tmC = (epi.tma_out & 2) ? &tmY : nullptr;
      for (int t = cid; t < total; t += ncl) {
        const int m0 = (t / num_n) * 2 * BM + (int)rank * BM, n_blk = t % num_n;
        if (!epilogue_tile<BN, MODE, EW, OP, true>(epi, M, N, m0, n_blk, tmem_base + (uint32_t)(acc * BN),
                                             tfull_bar(acc), acc_phase, map_to_rank(tempty_bar(acc), 0),
                                             release, stg, ew, warp, lane, abort_flag, err_flag, tmO,
                                             tmC))
          break;
        if (++acc == 2) acc = 0, acc_phase ^= 1u;
      }
      if ((tmO || tmC) && lane == 0) bulk_wait_group_all();   // TMA stores done before exit
    }
  }
  tc_fence_before();
  cluster_sync();   // both CTAs done with TMEM and with each other's barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, (uint32_t)C::TMEM_COLS);
  }
}

// ------------------------------- host side -------------------------------------------

static int tile_n(int N) { return (N % 256 == 0 || N > 2048) ? 256 : 128; }

// energy partials per row written by the out-projection mode: one per epilogue warp share
int gemm_tc_partials(int N) {
  return (epi_warps(EPI_OUTPROJ) / 4) * ((N + tile_n(N) - 1) / tile_n(N));
}

template <int OP>
static bool operand_map(CUtensorMap* m, const void* p, int rows, int cols, int box_rows) {
  return OP ? make_map_u8(m, p, rows, cols, box_rows) : make_map(m, p, rows, cols, box_rows);
}

template <int BN, int MODE, int OP>
static cudaError_t launch_tc(const void* A, const void* W, int M, int N, int K, const Epilogue& epi,
                             int* err_flag, int num_sms, cudaStream_t s) {
  using C = Cfg<BN, MODE>;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = set_max_dynamic_smem((const void*)k_gemm_tc<BN, MODE, OP>, C::SMEM, attr_done);
  if (e != cudaSuccess) return e;
  CUtensorMap ma, mb, mx;
  if (!operand_map<OP>(&ma, A, M, K, BM) || !operand_map<OP>(&mb, W, N, K, BN))
    return cudaErrorInvalidValue;
  Epilogue ek = epi;
  ek.tma_out = 0;
  mx = ma;   // unused unless the goal map below is made
  // energies only: the goal rows arrive by TMA (32-row chunks stay within one candidate)
  if (MODE == EPI_OUTPROJ && epi.goal && !epi.zpred && !epi.zhat && epi.P % 32 == 0 &&
      (((uintptr_t)epi.goal) & 15) == 0) {
    const int problems = (epi.cand0 + (M - 1) / epi.P) / epi.cands_per_problem + 1;
    if (make_map_f32(&mx, epi.goal, problems * epi.P, N, 32)) ek.tma_out = 4;
    else mx = ma;
  }
  const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const int grid = tiles < num_sms ? tiles : num_sms;
  k_gemm_tc<BN, MODE, OP><<<grid, cta_threads(MODE), C::SMEM, s>>>(ma, mb, mx, M, N, K, ek, err_flag);
  return cudaGetLastError();
}

template <int BN, int OP>
static cudaError_t launch_mode(const void* A, const void* W, int M, int N, int K,
                               const Epilogue& epi, int* err_flag, int num_sms, cudaStream_t s) {
  switch (epi.mode) {
    case EPI_STORE: return launch_tc<BN, EPI_STORE, OP>(A, W, M, N, K, epi, err_flag, num_sms, s);
    case EPI_GELU: return launch_tc<BN, EPI_GELU, OP>(A, W, M, N, K, epi, err_flag, num_sms, s);
    case EPI_OUTPROJ: return launch_tc<BN, EPI_OUTPROJ, OP>(A, W, M, N, K, epi, err_flag, num_sms, s);
    case EPI_GATED:
      if constexpr (BN == 256) return launch_tc<256, EPI_GATED, OP>(A, W, M, N, K, epi, err_flag, num_sms, s);
      return cudaErrorInvalidValue;
    default: break;
  }
  if constexpr (OP == 0) {   // the residual and in-projection GEMMs have bf16 operands only
    switch (epi.mode) {
      case EPI_RESID: return launch_tc<BN, EPI_RESID, 0>(A, W, M, N, K, epi, err_flag, num_sms, s);
      case EPI_INPROJ: return launch_tc<BN, EPI_INPROJ, 0>(A, W, M, N, K, epi, err_flag, num_sms, s);
      default: break;
    }
  }
  return cudaErrorInvalidValue;
}

template <int MODE, int OP>
static cudaError_t launch_tc2(const void* A, const void* W, int M, int N, int K, const Epilogue& epi,
                              int* err_flag, int num_sms, cudaStream_t s) {
  using C = Cfg2<MODE>;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = set_max_dynamic_smem((const void*)k_gemm_tc2<MODE, OP>, C::SMEM, attr_done);
  if (e != cudaSuccess) return e;
  CUtensorMap ma, mb, mx, my;
  if (!operand_map<OP>(&ma, A, M, K, BM) || !operand_map<OP>(&mb, W, N, K, 128))
    return cudaErrorInvalidValue;
  Epilogue ek = epi;
  ek.tma_out = 0;
  if (MODE == EPI_RESID) {
    if (!make_map_f32(&mx, epi.out0, M, N, 32)) return cudaErrorInvalidValue;
  } else if ((MODE == EPI_GELU || MODE == EPI_GATED || MODE == EPI_STORE) && epi.act_bf16 &&
             epi.map0.goff == 0 && epi.map0.rpg >= M && (((uintptr_t)epi.out0) & 15) == 0 &&
             (epi.ld0 % 8) == 0) {
    // bf16 out0 rows leave by TMA stores (the staging buffer is the box's 64-byte swizzle);
    // the columns of out0 are [0, split) in the store mode, N / 2 in the gated one
    const int cols = MODE == EPI_GATED ? N / 2 : (MODE == EPI_STORE && epi.split < N ? epi.split : N);
    if (!make_map_bf16_out(&mx, epi.out0, M, cols, epi.ld0)) return cudaErrorInvalidValue;
    ek.tma_out = 1;
  } else {
    mx = ma;   // unused
  }
  my = ma;   // unused unless the K/V cache map below is made
  // the store mode's out1 (the K/V cache: blocks of rpg rows, gstride rows per group) by TMA
  // through a 3-D map when its blocks tile the cache exactly
  if (MODE == EPI_STORE && epi.act_bf16 && epi.split < N && epi.out1 && epi.map1.rpg >= 32 &&
      epi.map1.gstride % epi.map1.rpg == 0 && epi.map1.goff % epi.map1.rpg == 0 &&
      (((uintptr_t)epi.out1) & 15) == 0 && (epi.ld1 % 8) == 0) {
    const RowMap& m1 = epi.map1;
    // an identity map (one block of at least M rows) is encoded as a single block of M rows
    const int rpg_dim = m1.rpg >= M ? M : m1.rpg;
    const long long nblocks =
        (long long)((M - 1) / m1.rpg) * (m1.gstride / m1.rpg) + m1.goff / m1.rpg + 1;
    if (make_map_bf16_blocks(&my, epi.out1, N - epi.split, rpg_dim, nblocks, epi.ld1))
      ek.tma_out |= 2;   // else the rows leave by per-lane stores
    else
      my = ma;
  }
  const int tiles = ((M + 2 * BM - 1) / (2 * BM)) * ((N + 255) / 256);
  const int pairs = num_sms / 2;
  const int grid = 2 * (tiles < pairs ? tiles : pairs);
  k_gemm_tc2<MODE, OP><<<grid, cta_threads(MODE), C::SMEM, s>>>(ma, mb, mx, my, M, N, K, ek, err_flag);
  return cudaGetLastError();
}

template <int OP>
static cudaError_t gemm_tc(const void* A, const void* W, int M, int N, int K, const Epilogue& epi,
                           int* err_flag, int num_sms, cudaStream_t s) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  // TMA: 16-byte aligned bases and row strides
  if (K <= 0 || K % (OP ? 16 : 8) != 0 || N % 4 != 0 || (((uintptr_t)A) & 15) ||
      (((uintptr_t)W) & 15))
    return cudaErrorInvalidValue;
  if (epi.mode == EPI_STORE && (epi.split % 32) != 0) return cudaErrorInvalidValue;
  if (epi.mode == EPI_GATED && (N % 256 != 0 || !epi.bias)) return cudaErrorInvalidValue;
  if (OP && (!epi.row_scale || !epi.col_scale)) return cudaErrorInvalidValue;
  // QKV, the MLP up-projection (GELU or gated) and the residual projections (N a multiple
  // of 256, many row tiles) run on CTA pairs. Measured at the full shape (M = 206,400,
  // K = 1024, bf16 out): GELU N = 4096 1232 -> 1204 us, gated N = 8192 2112 -> 2010 us
  // against single CTAs.
  if (N % 256 == 0 && M >= 4 * BM && num_sms >= 2) {
    if (epi.mode == EPI_STORE) return launch_tc2<EPI_STORE, OP>(A, W, M, N, K, epi, err_flag, num_sms, s);
    if (epi.mode == EPI_GELU) return launch_tc2<EPI_GELU, OP>(A, W, M, N, K, epi, err_flag, num_sms, s);
    if (epi.mode == EPI_GATED) return launch_tc2<EPI_GATED, OP>(A, W, M, N, K, epi, err_flag, num_sms, s);
    // the residual epilogue moves x with TMA: identity row map, row stride N, 16-byte base
    if constexpr (OP == 0)
      if (epi.mode == EPI_RESID && epi.ld0 == N && epi.map0.goff == 0 && epi.map0.rpg >= M &&
          (((uintptr_t)epi.out0) & 15) == 0)
        return launch_tc2<EPI_RESID, 0>(A, W, M, N, K, epi, err_flag, num_sms, s);
  }
  if (tile_n(N) == 256) return launch_mode<256, OP>(A, W, M, N, K, epi, err_flag, num_sms, s);
  return launch_mode<128, OP>(A, W, M, N, K, epi, err_flag, num_sms, s);
}

cudaError_t gemm_tc_bf16(const bf16* A, const bf16* W, int M, int N, int K, const Epilogue& epi,
                         int* err_flag, int num_sms, cudaStream_t s) {
  return gemm_tc<0>(A, W, M, N, K, epi, err_flag, num_sms, s);
}

cudaError_t gemm_tc_fp8(const uint8_t* A, const uint8_t* W, int M, int N, int K,
                        const Epilogue& epi, int* err_flag, int num_sms, cudaStream_t s) {
  return gemm_tc<1>(A, W, M, N, K, epi, err_flag, num_sms, s);
}

}  // namespace jepa
