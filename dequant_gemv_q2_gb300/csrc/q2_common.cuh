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

// Bulk prefetch of [p, p + bytes) into L2 (16-byte aligned, multiple of 16),
// issued by one thread in 64 KiB pieces; no registers or shared memory are
// held while the bytes arrive.
__device__ __forceinline__ void prefetch_l2(const void* p, size_t bytes) {
  const char* c = static_cast<const char*>(p);
  for (size_t off = 0; off < bytes; off += 65536) {
    const uint32_t n = (uint32_t)((bytes - off) < 65536 ? (bytes - off) : 65536);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c + off), "r"(n) : "memory");
  }
}

// acc += f16 * f16 in fp32 (mixed-precision FMA, sm_100+ PTX)
__device__ __forceinline__ float fma_h(unsigned short a, unsigned short b, float c) {
  float d;
  asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
  return d;
}

__device__ __forceinline__ unsigned short lo16(uint32_t v) { return (unsigned short)(v & 0xffffu); }
__device__ __forceinline__ unsigned short hi16(uint32_t v) { return (unsigned short)(v >> 16); }

// -------------------------------------------------------------- mbarriers
constexpr long long kSpinLimit = 1ll << 24;   // bounded mbarrier waits

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Wait for the phase with the given parity to complete, for at most `limit`
// polls; false on timeout.  With `abort` (a shared-memory flag other roles of
// the CTA set when they give up), also false as soon as the flag is seen.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, long long limit = kSpinLimit,
                                          const volatile int* abort = nullptr) {
  if (limit < kSpinLimit) {                    // a shortened (test) limit: non-blocking probes
    for (long long i = 0; i < limit; ++i) {
      uint32_t done;
      asm volatile(
          "{\n\t.reg .pred p;\n\t"
          "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
          "selp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(done)
          : "r"(bar), "r"(parity)
          : "memory");
      if (done) return true;
    }
    return false;
  }
  for (long long i = 0; i < limit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    if (abort && (i & 63) == 63 && *abort) return false;
  }
  return false;
}

// ------------------------------------------------------- subset-sum tables
// For one 256-column slice of x, T[v][b] = sum of x[8b + i] over the set bits
// i of the byte v (b = 0..31), stored twice per v (columns b and b + 32) so a
// lane at rotated position P reads column P + lane without a modulo:
// address = v*256 + lane*4 + P*4 bytes.  Each of 512 (column-byte b, high
// nibble h) tasks loads the 8 x values of byte b, forms the 16 sums of its
// low nibble by doubling, adds the sum selected by h, and writes the 16
// entries T[16h + l][b] (consecutive b across a warp: conflict-free stores).
// Also returns the slice sum of x in *gsum.  The caller synchronises the
// building threads before any of them reads T.
constexpr int kTableBytes = 256 * 64 * 4;
constexpr int kBuildBytes = kTableBytes + 16;

template <int NT>
__device__ __forceinline__ void build_table(const __half* __restrict__ xg, int ncols, float* T,
                                            float* gsum) {
  for (int e = threadIdx.x; e < 512; e += NT) {
    const int b = e & 31, h = e >> 5;
    const int c0 = 8 * b;
    float x8[8];
    if (c0 + 8 <= ncols) {
      const uint4 raw = *reinterpret_cast<const uint4*>(xg + c0);
      const __half2* hv = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __half22float2(hv[k]);
        x8[2 * k] = f.x;
        x8[2 * k + 1] = f.y;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) x8[i] = (c0 + i < ncols) ? __half2float(xg[c0 + i]) : 0.f;
    }
    // sum selected by the high nibble h (bits 4..7)
    float hs = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) hs += ((h >> i) & 1) ? x8[4 + i] : 0.f;
    float s[16];
    s[0] = hs;
#pragma unroll
    for (int n = 1; n < 16; ++n) {
      const int low = n & -n;
      const int i = (low == 1) ? 0 : (low == 2) ? 1 : (low == 4) ? 2 : 3;
      s[n] = s[n ^ low] + x8[i];
    }
    float* col = T + (h * 16) * 64 + b;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      col[n * 64] = s[n];
      col[n * 64 + 32] = s[n];
    }
    if (h == 15) {                               // this warp holds all 32 bytes' full sums
      float v = s[15];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (b == 0) *gsum = v;
    }
  }
}

// ------------------------------------------- programmatic dependent launch
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------- fixed-point accumulation
// Accumulator word: bits 56..63 count the terms added so far; bit 55 is a
// sticky flag set by any non-finite term; bits 0..54 hold the sum of
// (q + 2^46) over the finite terms, q = round(partial * 2^F), where the
// launcher picks F so that |partial| * 2^F < 2^45 for every fp16 x (the
// clamp below only ever bites on absurd inputs).  At most Q2_MAX_SPLIT
// (255) terms of less than 2^47 each sum below 255 * 2^47 < 2^55: the value
// never reaches the flag or the count.  The batch-1 kernels add one term
// per 256-column slice, the tensor-core kernel one per K split.
//
// One inf or NaN in x makes the IEEE result non-finite, but an integer sum
// cannot carry it.  A lane whose partial is not finite therefore sets the
// flag with an atomic OR and then adds its count with an atomic add, both
// on the same word: later atomics on a word see earlier ones, so whichever
// lane completes the count finds the flag in its add's result and writes
// NaN (IEEE would give inf or NaN: non-finite either way).
constexpr unsigned long long kBias = 1ull << 46;
constexpr unsigned long long kCountOne = 1ull << 56;
constexpr unsigned long long kNonFinite = 1ull << 55;
constexpr unsigned long long kValueMask = kNonFinite - 1;

__device__ __forceinline__ unsigned long long fx_term(float p, float fscale) {
  long long q = __float2ll_rn(p * fscale);
  q = max(min(q, (long long)kBias - 1), -(long long)kBias + 1);
  return kCountOne + (unsigned long long)(q + (long long)kBias);
}

// The term to add for partial p to *word.  A non-finite p sets the flag on
// the word first (the OR is ordered before the caller's add on the same
// word) and adds only the count.  The caller adds the returned term with
// atomicAdd and may look at the result later (its round trip overlaps work).
__device__ __forceinline__ unsigned long long fx_prepare(unsigned long long* word, float p, float fscale) {
  if (isfinite(p)) return fx_term(p, fscale);
  atomicOr(word, kNonFinite);
  return kCountOne;
}

// The value of a completed word (all n terms added): NaN when a term was not
// finite, else the fixed-point sum scaled back by finv = 2^-F.
__device__ __forceinline__ float fx_value(unsigned long long w, int n, float finv) {
  if (w & kNonFinite) return __int_as_float(0x7fc00000);
  const long long v = (long long)(w & kValueMask) - (long long)n * (long long)kBias;
  return (float)v * finv;
}

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
