// Device helpers shared by the q2 kernels.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include <algorithm>

#include "q2_internal.h"

namespace q2 {

// ---------------------------------------------------------------- launch state
struct DevInfo {
  int sms;
};
DevInfo dev_info();                       // cached per device (q2_launch.cu)
int set_smem(const void* fn, int bytes);  // raise the dynamic smem cap once per device

// ------------------------------------------------------------------ loads
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  // weight stream: read once, keep it out of L1
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// acc += f16 * f16 in fp32 (mixed-precision FMA, sm_100+ PTX)
__device__ __forceinline__ float fma_h(unsigned short a, unsigned short b, float c) {
  float d;
  asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
  return d;
}

__device__ __forceinline__ unsigned short lo16(uint32_t v) { return (unsigned short)(v & 0xffffu); }
__device__ __forceinline__ unsigned short hi16(uint32_t v) { return (unsigned short)(v >> 16); }

// ------------------------------------------------------- subset-sum tables
// For one 256-column slice of x, T[v][b] = sum of x[8b + i] over the set bits
// i of the byte v (b = 0..31), stored twice per v (columns b and b + 32) so a
// lane at rotated position P reads column P + lane without a modulo:
// address = v*256 + lane*4 + P*4 bytes.  Built in two phases: 64 threads
// each load four x values and write the 16 subset sums of that nibble
// (lo[n][b] for bits 0..3 of byte b, hi[n][b] for bits 4..7); then
// T[v][b] = lo[v & 15][b] + hi[v >> 4][b].  Also returns the slice sum of x
// in *gsum.  Layout in shared memory: T (64 KiB) | lo[16][32] | hi[16][32].
constexpr int kTableBytes = 256 * 64 * 4;
constexpr int kBuildBytes = kTableBytes + 2 * 16 * 32 * 4 + 256 * 4 + 16;

template <int NT>
__device__ __forceinline__ void build_table(const __half* __restrict__ xg, int ncols, float* T,
                                            float* gsum) {
  float* lo = T + 256 * 64;
  float* hi = lo + 16 * 32;
  const int t = threadIdx.x;
  if (t < 64) {
    const int b = t & 31, half = t >> 5;
    const int c0 = 8 * b + 4 * half;
    float x4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) x4[i] = (c0 + i < ncols) ? __half2float(xg[c0 + i]) : 0.f;
    float* dst = (half ? hi : lo) + b;
    float s[16];
    s[0] = 0.f;
#pragma unroll
    for (int n = 1; n < 16; ++n) {
      const int low = n & -n;                       // lowest set bit
      const int i = (low == 1) ? 0 : (low == 2) ? 1 : (low == 4) ? 2 : 3;
      s[n] = s[n ^ low] + x4[i];
    }
#pragma unroll
    for (int n = 0; n < 16; ++n) dst[n * 32] = s[n];
  }
  __syncthreads();
  // 256 v x 8 quads of b: thread -> (quad, vlo), loops over vhi
  for (int e = t; e < 16 * 16 * 8; e += NT) {
    const int q = e & 7, vlo = (e >> 3) & 15, vhi = e >> 7;
    const float4 a = *reinterpret_cast<const float4*>(lo + vlo * 32 + 4 * q);
    const float4 bq = *reinterpret_cast<const float4*>(hi + vhi * 32 + 4 * q);
    float4 s;
    s.x = a.x + bq.x;
    s.y = a.y + bq.y;
    s.z = a.z + bq.z;
    s.w = a.w + bq.w;
    float* row = T + (vhi * 16 + vlo) * 64;
    *reinterpret_cast<float4*>(row + 4 * q) = s;
    *reinterpret_cast<float4*>(row + 32 + 4 * q) = s;
  }
  if (t >= NT - 32) {                                // last warp: slice sum of x
    const int b = t & 31;
    float v = lo[15 * 32 + b] + hi[15 * 32 + b];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (b == 0) *gsum = v;
  }
  __syncthreads();
}

// ---------------------------------------------------- split-K reduction
// Each (slice, 32-row block) item writes fp32 partials for its rows with
// plain stores.  A second kernel (q2_reduce.cu), chained by programmatic
// dependent launch, sums the partials of every output in slice order, so the
// result does not depend on scheduling.
struct Reduce {
  float* partial;      // [ntok][nslice][Rpad]
  int nslice;
  int Rpad;
};

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch with programmatic stream serialization allowed (PDL): the kernel
// may start while the previous kernel on the stream drains; it must call
// pdl_wait() before reading anything that kernel writes.
template <typename A>
int launch_pdl(void (*kernel)(A), const A& args, int grid, int threads, int smem, void* stream) {
  if (set_smem(reinterpret_cast<const void*>(kernel), smem)) return Q2_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, args) != cudaSuccess) {
    (void)cudaGetLastError();
    return Q2_ECUDA;
  }
  return cudaGetLastError() == cudaSuccess ? Q2_OK : Q2_ECUDA;
}

// Contiguous share of n items for this CTA.
__device__ __forceinline__ void cta_range(int n, int& i0, int& i1) {
  const int g = gridDim.x, b = blockIdx.x;
  const int per = n / g, rem = n % g;
  i0 = b * per + min(b, rem);
  i1 = i0 + per + (b < rem ? 1 : 0);
}

}  // namespace q2
