// Dense fp16 control GEMV ("Unfolding the Leech Lattice", section 7: the
// byte bound is the fp16 control's measured bandwidth).  A warp owns one
// row at a time; each lane streams 16-byte chunks of the row and accumulates
// in fp32 with mixed-precision FMAs; a shuffle reduction finishes the row.
#include <cuda_fp16.h>

#include "q2_common.cuh"

extern __shared__ __align__(1024) unsigned char q2_smem[];

namespace q2 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

struct DenseArgs {
  const __half* w;
  const __half* x;
  __half* y;
  int R, C, ntok;
};

__device__ __forceinline__ float dot8(const uint4& w, const uint4& x, float acc) {
  acc = fma_h(lo16(w.x), lo16(x.x), acc);
  acc = fma_h(hi16(w.x), hi16(x.x), acc);
  acc = fma_h(lo16(w.y), lo16(x.y), acc);
  acc = fma_h(hi16(w.y), hi16(x.y), acc);
  acc = fma_h(lo16(w.z), lo16(x.z), acc);
  acc = fma_h(hi16(w.z), hi16(x.z), acc);
  acc = fma_h(lo16(w.w), lo16(x.w), acc);
  acc = fma_h(hi16(w.w), hi16(x.w), acc);
  return acc;
}

__global__ void __launch_bounds__(kThreads) k_fp16_b1(DenseArgs a) {
  uint4* xs = reinterpret_cast<uint4*>(q2_smem);
  const int nch = a.C / 8;
  const uint4* xg = reinterpret_cast<const uint4*>(a.x);
  for (int i = threadIdx.x; i < nch; i += kThreads) xs[i] = xg[i];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5), nw = gridDim.x * kWarps;
  for (int r = gw; r < a.R; r += nw) {
    const uint4* wr = reinterpret_cast<const uint4*>(a.w + (size_t)r * a.C);
    float acc0 = 0.f, acc1 = 0.f;
    int c = lane;
    for (; c + 96 < nch; c += 128) {
      const uint4 w0 = ldg_stream(wr + c), w1 = ldg_stream(wr + c + 32), w2 = ldg_stream(wr + c + 64),
                  w3 = ldg_stream(wr + c + 96);
      acc0 = dot8(w0, xs[c], acc0);
      acc1 = dot8(w1, xs[c + 32], acc1);
      acc0 = dot8(w2, xs[c + 64], acc0);
      acc1 = dot8(w3, xs[c + 96], acc1);
    }
    for (; c < nch; c += 32) acc0 = dot8(ldg_stream(wr + c), xs[c], acc0);
    float acc = acc0 + acc1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) a.y[r] = __float2half_rn(acc);
  }
}

template <int NT>
__global__ void __launch_bounds__(kThreads) k_fp16_mt(DenseArgs a) {
  const int lane = threadIdx.x & 31;
  const int nch = a.C / 8;
  const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5), nw = gridDim.x * kWarps;
  for (int r = gw; r < a.R; r += nw) {
    const uint4* wr = reinterpret_cast<const uint4*>(a.w + (size_t)r * a.C);
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.f;
    for (int c = lane; c < nch; c += 32) {
      const uint4 w = ldg_stream(wr + c);
#pragma unroll
      for (int t = 0; t < NT; ++t)
        if (t < a.ntok) acc[t] = dot8(w, __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)t * a.C) + c), acc[t]);
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t >= a.ntok) break;
      float v = acc[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) a.y[(size_t)t * a.R + r] = __float2half_rn(v);
    }
  }
}

}  // namespace
}  // namespace q2

using namespace q2;

extern "C" int q2_launch_fp16(const q2_handle* h, const void* x, void* y, int ntok, void* stream, const q2_pf*) {
  const q2_blob_header& d = h->hdr;
  DenseArgs a;
  a.w = reinterpret_cast<const __half*>(h->dev + d.off[SEC_FP16_W]);
  a.x = static_cast<const __half*>(x);
  a.y = static_cast<__half*>(y);
  a.R = d.R;
  a.C = d.C;
  a.ntok = ntok;
  const DevInfo di = dev_info();
  const int grid = max(1, min((d.R + kWarps - 1) / kWarps, 8 * di.sms));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (ntok == 1) {
    const int smem = d.C * 2;
    if (set_smem(reinterpret_cast<const void*>(k_fp16_b1), smem)) return Q2_ECUDA;
    k_fp16_b1<<<grid, kThreads, smem, st>>>(a);
  } else if (ntok <= 4) {
    k_fp16_mt<4><<<grid, kThreads, 0, st>>>(a);
  } else if (ntok <= 16) {
    k_fp16_mt<16><<<grid, kThreads, 0, st>>>(a);
  } else {
    k_fp16_mt<64><<<grid, kThreads, 0, st>>>(a);
  }
  return cudaGetLastError() == cudaSuccess ? Q2_OK : Q2_ECUDA;
}
