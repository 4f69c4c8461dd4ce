// Device helpers shared by the q2 kernels.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

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
// address = v*256 + lane*4 + P*4 bytes.  Built from two 16-entry nibble
// tables.  Also returns the slice sum of x in *gsum.
// Layout in shared memory: T (64 KiB) | lo[16][32] | hi[16][32] | xs[256].
constexpr int kTableBytes = 256 * 64 * 4;
constexpr int kBuildBytes = kTableBytes + 2 * 16 * 32 * 4 + 256 * 4 + 16;

template <int NT>
__device__ __forceinline__ void build_table(const __half* __restrict__ xg, int ncols, float* T,
                                            float* gsum) {
  float* lo = T + 256 * 64;
  float* hi = lo + 16 * 32;
  float* xs = hi + 16 * 32;
  const int t = threadIdx.x;
  for (int c = t; c < 256; c += NT) xs[c] = (c < ncols) ? __half2float(xg[c]) : 0.f;
  __syncthreads();
  for (int e = t; e < 1024; e += NT) {
    const int which = e >> 9, n = (e >> 5) & 15, b = e & 31;
    const float* src = xs + 8 * b + 4 * which;
    float v = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) v += ((n >> i) & 1) ? src[i] : 0.f;
    (which ? hi : lo)[n * 32 + b] = v;
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
  if (t < 32) {
    float v = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) v += xs[8 * t + i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (t == 0) *gsum = v;
  }
  __syncthreads();
}

// ---------------------------------------------------- split-K reduction
// Each (slice, 32-row block) item writes fp32 partials for its rows; the
// last warp to finish a row block (atomic counter) sums the partials of all
// slices in slice order, so the result does not depend on scheduling, and
// resets the counter to zero for the next call.  No thread waits.
struct Reduce {
  float* partial;      // [ntok][nslice][Rpad]
  unsigned* counter;   // [nrb]
  int nslice;
  int Rpad;
};

// Returns true in every lane of the warp that must finish row block rb.
__device__ __forceinline__ bool arrive(const Reduce& rd, int rb) {
  __threadfence();
  __syncwarp();
  unsigned old = 0;
  if ((threadIdx.x & 31) == 0) old = atomicAdd(rd.counter + rb, 1u);
  old = __shfl_sync(0xffffffffu, old, 0);
  const bool last = (old == (unsigned)rd.nslice - 1u);
  if (last) {
    __threadfence();
    if ((threadIdx.x & 31) == 0) rd.counter[rb] = 0u;
  }
  return last;
}

__device__ __forceinline__ float gather(const Reduce& rd, int tok, int row) {
  const float* p = rd.partial + (size_t)tok * rd.nslice * rd.Rpad + row;
  float acc = 0.f;
  for (int s = 0; s < rd.nslice; ++s) acc += __ldcg(p + (size_t)s * rd.Rpad);
  return acc;
}

// Contiguous share of n items for this CTA.
__device__ __forceinline__ void cta_range(int n, int& i0, int& i1) {
  const int g = gridDim.x, b = blockIdx.x;
  const int per = n / g, rem = n % g;
  i0 = b * per + min(b, rem);
  i1 = i0 + per + (b < rem ? 1 : 0);
}

}  // namespace q2
