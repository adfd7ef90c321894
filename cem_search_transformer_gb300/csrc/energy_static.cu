// L1 energy of predicted frames against the goal, using no device allocation at all.
//
// For callers that cannot allocate device memory: processes that run under a fixed
// memory budget handed out by a host framework, real-time control loops that must not
// pay cudaMalloc's latency or risk its failure mid-episode, and code that runs where
// allocation calls are not permitted. The per-candidate partial sums that the regular
// energy path keeps in context workspace live here in one file-scope device array of
// fixed size instead.
//
// The array is shared by every call in the process: calls whose work overlaps on the GPU
// (different streams, no ordering between them) race on it and may return wrong energies.
// Calls ordered on one stream are safe. Every partial that a call reads is first written by
// the same call, so nothing has to be cleared between calls.
#include "jepa_cem.h"
#include "common.cuh"

#include <cuda.h>

#include <cstdio>
#include <mutex>

namespace {

constexpr int kRowsPerPartial = 32;                 // patch rows summed by one block
constexpr long long kMaxPartials = 1LL << 20;       // 4 MiB of fp32 scratch
static __device__ __align__(256) float g_energy_partials[kMaxPartials];

constexpr int kMaxDevices = 64;
// Device address of the array per device, with the id of the CUDA context it was taken in:
// after a device reset the module is loaded again in a new context, possibly elsewhere, so
// an address taken in an earlier context is looked up afresh.
struct ScratchAddr {
  unsigned long long ctx_id = 0;
  float* ptr = nullptr;
};
ScratchAddr g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

// Block (candidate c, row block rb): sum of |z - goal| over rows [32 rb, 32 rb + 32) x E.
// Fixed summation order: thread-strided, then a shuffle tree, then warps in order.
__global__ void k_energy_partials_static(const float* __restrict__ z, const float* __restrict__ goal,
                                         int N, int P, int E, int nblk,
                                         float* __restrict__ partials) {
  __shared__ float warp_sums[32];
  const int c = blockIdx.x / nblk, rb = blockIdx.x % nblk;
  const int b = c / N;
  const int r0 = rb * kRowsPerPartial;
  const int r1 = min(P, r0 + kRowsPerPartial);
  const float* zc = z + ((long long)c * P + r0) * E;
  const float* gc = goal + ((long long)b * P + r0) * E;
  const long long n = (long long)(r1 - r0) * E;
  float s = 0.f;
  for (long long i = threadIdx.x; i < n; i += blockDim.x) s += fabsf(zc[i] - gc[i]);
#pragma unroll
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) warp_sums[warp] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += warp_sums[w];
    partials[blockIdx.x] = t;
  }
}

// energy[c] = (sum of the candidate's nblk partials) / (P * E), summed in index order.
__global__ void k_energy_reduce_static(const float* __restrict__ partials, int nblk, int ncand,
                                       float inv_count, float* __restrict__ energy) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= ncand) return;
  float s = 0.f;
  for (int i = 0; i < nblk; ++i) s += partials[(long long)c * nblk + i];
  energy[c] = s * inv_count;
}

void set_msg(char* buf, size_t len, const char* msg) {
  if (buf && len) snprintf(buf, len, "%s", msg);
}

// Driver entry points for the current context and its process-unique id (CUDA 12.0+),
// resolved once through the runtime.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

cudaError_t current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_current || !get_id) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorDeviceUninitialized;
  return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

// Device address of the scratch array in the current device's context: looked up on the
// first call in a context (cudaGetSymbolAddress, which also makes the runtime bind the
// device's primary context) and cached until the context changes.
cudaError_t scratch_for_current_device(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  unsigned long long id = 0;
  if (current_context_id(&id) == cudaSuccess && g_scratch[dev].ptr && g_scratch[dev].ctx_id == id) {
    *out = g_scratch[dev].ptr;
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_energy_partials);
  if (e != cudaSuccess) return e;
  if ((e = current_context_id(&id)) != cudaSuccess) return e;
  g_scratch[dev].ctx_id = id;
  g_scratch[dev].ptr = static_cast<float*>(p);
  *out = g_scratch[dev].ptr;
  return cudaSuccess;
}

}  // namespace

extern "C" jepa_status jepa_energy_l1_noalloc(const float* z_pred, const float* goal, int B, int N,
                                              int P, int E, float* energy, void* stream,
                                              char* err, size_t err_len) {
  set_msg(err, err_len, "");
  if (!z_pred || !goal || !energy || B < 1 || N < 1 || P < 1 || E < 1) {
    set_msg(err, err_len, "energy_l1_noalloc: null pointer or non-positive size");
    return JEPA_ERR_INVALID_ARG;
  }
  const long long nblk = (P + kRowsPerPartial - 1) / kRowsPerPartial;
  const long long ncand = (long long)B * N;
  if (ncand > (1LL << 30) || ncand * nblk > kMaxPartials) {
    char msg[200];
    snprintf(msg, sizeof msg,
             "energy_l1_noalloc: B*N*ceil(P/32) = %lld partial sums exceed the fixed scratch of "
             "%lld; split the candidates into smaller calls",
             ncand * nblk, kMaxPartials);
    set_msg(err, err_len, msg);
    return JEPA_ERR_SHAPE;
  }
  float* scratch = nullptr;
  cudaError_t e = scratch_for_current_device(&scratch);
  if (e != cudaSuccess) {
    set_msg(err, err_len, cudaGetErrorString(e));
    return JEPA_ERR_CUDA;
  }
  cudaStream_t s = (cudaStream_t)stream;
  k_energy_partials_static<<<(unsigned)(ncand * nblk), 256, 0, s>>>(z_pred, goal, N, P, E, (int)nblk,
                                                                     scratch);
  e = cudaGetLastError();
  if (e == cudaSuccess) {
    k_energy_reduce_static<<<(unsigned)((ncand + 255) / 256), 256, 0, s>>>(
        scratch, (int)nblk, (int)ncand, 1.0f / ((float)P * (float)E), energy);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    set_msg(err, err_len, cudaGetErrorString(e));
    return JEPA_ERR_CUDA;
  }
  return JEPA_OK;
}
