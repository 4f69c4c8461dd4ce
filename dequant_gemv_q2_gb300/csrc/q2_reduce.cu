// Split-K reduction and epilogue of the tensor-core path: y[t][r] =
// epilogue(sum over K splits s, in order, of partial[t][s][r]).  Runs as the
// second launch of a GEMV, chained to the main kernel by programmatic
// dependent launch: its CTAs may start
// while the main kernel drains and wait (griddepcontrol.wait) until every
// partial is visible.  One thread per output, consecutive threads on
// consecutive rows, so every slice's partials are read as coalesced lines.
//
// Epilogues: BPDQ and the no-weights control, none; trellis, x scale_r;
// Leech, + 16 x[col] for each v = +8 exception, x scale_r / sqrt(8), + the
// fp16 tail dot product ("Tetra", section 5.1: row scale after the block
// dot product, then the unquantised tail).
#include <cuda_fp16.h>

#include "q2_common.cuh"

namespace q2 {
namespace {

constexpr int kThreads = 128;   // small CTAs: they co-reside with two GEMV CTAs on an SM

struct RedArgs {
  const float* partial;      // [ntok][nslice][Rpad]
  int nslice, Rpad, R, ntok, C;
  const __half* scale;       // [R] or null
  float post;                // factor applied with the scale
  const __half* tail;        // [Rpad][tailpad] or null
  int tail_n, tailpad, tail_col0;
  const uint32_t* excptr;    // [Rpad + 1] or null
  const uint32_t* exccol;
  const __half* x;
  __half* y;
};

__global__ void __launch_bounds__(kThreads) k_reduce(RedArgs a) {
  pdl_trigger();
  pdl_wait();
  const size_t n = (size_t)a.ntok * a.R;
  const size_t st = (size_t)a.Rpad;
  for (size_t idx = blockIdx.x * (size_t)kThreads + threadIdx.x; idx < n; idx += (size_t)gridDim.x * kThreads) {
    const int t = (int)(idx / a.R), row = (int)(idx % a.R);
    const float* p = a.partial + (size_t)t * a.nslice * st + row;
    float v = 0.f;
    int s = 0;
    for (; s + 16 <= a.nslice; s += 16) {
      float b[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) b[k] = __ldcg(p + (size_t)(s + k) * st);
#pragma unroll
      for (int k = 0; k < 16; ++k) v += b[k];
    }
    if (s < a.nslice) {
      float b[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) b[k] = (s + k < a.nslice) ? __ldcg(p + (size_t)(s + k) * st) : 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (s + k < a.nslice) v += b[k];
    }
    const __half* xt = a.x + (size_t)t * a.C;
    if (a.excptr)
      for (uint32_t e = a.excptr[row]; e < a.excptr[row + 1]; ++e) v = fmaf(16.f, __half2float(xt[a.exccol[e]]), v);
    if (a.scale) v *= __half2float(a.scale[row]) * a.post;
    for (int j = 0; j < a.tail_n; ++j)
      v = fmaf(__half2float(a.tail[(size_t)row * a.tailpad + j]), __half2float(xt[a.tail_col0 + j]), v);
    a.y[(size_t)t * a.R + row] = __float2half_rn(v);
  }
}

}  // namespace
}  // namespace q2

using namespace q2;

// Second launch of a split-K GEMV whose partials are [ntok][nsplit][Rpad].
extern "C" int q2_launch_reduce_n(const q2_handle* h, const void* x, void* y, int ntok, int nsplit, void* stream) {
  const q2_blob_header& d = h->hdr;
  RedArgs a = {};
  a.partial = reinterpret_cast<const float*>(static_cast<const unsigned char*>(h->ws) + Q2_WS_PARTIAL_OFFSET);
  a.nslice = nsplit;
  a.Rpad = d.Rpad;
  a.R = d.R;
  a.ntok = ntok;
  a.C = d.C;
  a.post = 1.f;
  a.x = static_cast<const __half*>(x);
  a.y = static_cast<__half*>(y);
  if (d.fmt == Q2_TRELLIS) {
    a.scale = reinterpret_cast<const __half*>(h->dev + d.off[SEC_TRL_SCALE]);
  } else if (d.fmt == Q2_LEECH) {
    a.scale = reinterpret_cast<const __half*>(h->dev + d.off[SEC_LEECH_SCALE]);
    a.post = d.inv_sqrt8;
    a.tail = reinterpret_cast<const __half*>(h->dev + d.off[SEC_LEECH_TAIL]);
    a.tail_n = d.tail;
    a.tailpad = d.tailpad;
    a.tail_col0 = d.nblock * 24;
    a.excptr = reinterpret_cast<const uint32_t*>(h->dev + d.off[SEC_LEECH_EXCPTR]);
    a.exccol = reinterpret_cast<const uint32_t*>(h->dev + d.off[SEC_LEECH_EXCCOL]);
  }
  const DevInfo di = dev_info();
  const size_t n = (size_t)ntok * d.R;
  const int grid = (int)std::min<size_t>((n + kThreads - 1) / kThreads, (size_t)4 * di.sms);
  return launch_pdl(k_reduce, a, max(grid, 1), kThreads, 0, stream);
}

