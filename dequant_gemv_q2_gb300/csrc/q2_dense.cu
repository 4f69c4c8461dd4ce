// Dense fp16 control GEMV ("Unfolding the Leech Lattice", section 7: the
// byte bound is the fp16 control's measured bandwidth), one token.  A warp
// owns one row at a time; each lane streams 16-byte chunks of the row and
// accumulates in fp32 with mixed-precision FMAs; a shuffle reduction
// finishes the row.  More tokens run on the tensor cores (q2_tc.cu).
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
  int R, C;
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

}  // namespace
}  // namespace q2

using namespace q2;

extern "C" int q2_tc_fp16(const q2_handle* h, const void* x, void* y, int ntok, void* stream);

// One token on CUDA cores; 2..64 through the tensor-core kernel (q2_tc.cu),
// whose weight stage is a plain row load for this format.
extern "C" int q2_launch_fp16(const q2_handle* h, const void* x, void* y, int ntok, void* stream, const q2_pf*) {
  if (ntok > 1) return q2_tc_fp16(h, x, y, ntok, stream);
  const q2_blob_header& d = h->hdr;
  DenseArgs a;
  a.w = reinterpret_cast<const __half*>(h->dev + d.off[SEC_FP16_W]);
  a.x = static_cast<const __half*>(x);
  a.y = static_cast<__half*>(y);
  a.R = d.R;
  a.C = d.C;
  const DevInfo di = dev_info();
  const int grid = max(1, min((d.R + kWarps - 1) / kWarps, 8 * di.sms));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int smem = d.C * 2;
  if (set_smem(reinterpret_cast<const void*>(k_fp16_b1), smem)) return Q2_ECUDA;
  k_fp16_b1<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? Q2_OK : Q2_ECUDA;
}
