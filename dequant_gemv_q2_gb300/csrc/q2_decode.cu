// Debug decode of a bound blob back to the canonical form, read straight
// from the device layouts (used to check the packers and the layouts bit for
// bit against the oracle's decode).
#include <cuda_fp16.h>

#include "q2_common.cuh"

namespace q2 {
namespace {

constexpr int kThreads = 256;

__global__ void k_dec_fp16(const uint16_t* w, uint16_t* out, size_t n) {
  for (size_t i = blockIdx.x * (size_t)kThreads + threadIdx.x; i < n; i += (size_t)gridDim.x * kThreads)
    out[i] = w[i];
}

// BPDQ: one thread per (row, column-byte); 8 fp16 weights from the value table.
__global__ void k_dec_bpdq(const unsigned char* bits, const uint16_t* vtab, uint16_t* out, int R, int C,
                           int Rpad) {
  const int nby = C / 8;
  const size_t n = (size_t)R * nby;
  for (size_t e = blockIdx.x * (size_t)kThreads + threadIdx.x; e < n; e += (size_t)gridDim.x * kThreads) {
    const int r = (int)(e / nby), cb = (int)(e % nby);
    const int g = cb / 32, beta = cb % 32, l = r % 32, rb = r / 32;
    const int P = (beta - l + 32) & 31;
    const size_t item = (size_t)g * (Rpad / 32) + rb;
    const unsigned char* it = bits + item * Q2_ITEM_BYTES_BPDQ + l * 16 + (P & 15);
    const int k = P >> 4;
    const uint32_t b0 = it[k * 512], b1 = it[(2 + k) * 512];
    const uint16_t* vt = vtab + ((size_t)g * Rpad + r) * 4;
    for (int i = 0; i < 8; ++i) {
      const int code = ((b0 >> i) & 1) | (((b1 >> i) & 1) << 1);
      out[(size_t)r * C + cb * 8 + i] = vt[code];
    }
  }
}

// Trellis: one thread per (row, segment, step).
__global__ void k_dec_trellis(const unsigned char* stream, const uint32_t* table, const __half* scale,
                              float* out, int R, int C, int Rpad) {
  const int S = C / 256;
  const size_t n = (size_t)R * S * 128;
  for (size_t e = blockIdx.x * (size_t)kThreads + threadIdx.x; e < n; e += (size_t)gridDim.x * kThreads) {
    const int k = (int)(e % 128);
    const int s = (int)((e / 128) % S);
    const int r = (int)(e / (128 * (size_t)S));
    const int l = r % 32, rb = r / 32;
    const unsigned char* it = stream + ((size_t)s * (Rpad / 32) + rb) * Q2_ITEM_BYTES_TRL + l * 16;
    uint32_t W[16];
    for (int w = 0; w < 16; ++w) W[w] = *reinterpret_cast<const uint32_t*>(it + (w >> 2) * 512 + (w & 3) * 4);
    const int nn = 127 - k;
    const uint32_t f = __funnelshift_r(W[nn >> 3], W[((nn >> 3) + 1) & 15], 4 * (nn & 7));
    const uint32_t s16 = f & 0xffffu;
    const uint32_t idx = ((s16 * 0x9E37u) & 0xffffu) >> 4;
    uint32_t v = table[idx];
    if (s16 & 1u) v ^= 0x80008000u;
    const float sc = __half2float(scale[r]);
    out[(size_t)r * C + s * 256 + 2 * k] = sc * __half2float(__ushort_as_half(lo16(v)));
    out[(size_t)r * C + s * 256 + 2 * k + 1] = sc * __half2float(__ushort_as_half(hi16(v)));
  }
}

// Leech: one thread per (row, block); rebuilds v from parity, planes and the
// exception list.
__global__ void k_dec_leech(const unsigned char* planes, const uint16_t* parity, const uint32_t* excptr,
                            const uint32_t* exccol, int8_t* out, int R, int Rpad, int nblock, int off4) {
  const size_t n = (size_t)R * nblock;
  for (size_t e = blockIdx.x * (size_t)kThreads + threadIdx.x; e < n; e += (size_t)gridDim.x * kThreads) {
    const int r = (int)(e / nblock), b = (int)(e % nblock);
    const int l = r % 32, rb = r / 32;
    const int c0 = b * 24;
    const int sb = c0 / 256;
    const int first = (sb * 256 + 23) / 24;
    const int p = (parity[(size_t)sb * Rpad + r] >> (b - first)) & 1;
    for (int i = 0; i < 24; ++i) {
      const int c = c0 + i;
      const int s = c / 256, cc = c % 256, beta = cc / 8, bit = cc % 8;
      const int P = (beta - l + 32) & 31;
      const size_t item = off4 ? Q2_ITEM_BYTES_LEECH4 : Q2_ITEM_BYTES_LEECH;
      const unsigned char* it = planes + ((size_t)s * (Rpad / 32) + rb) * item + l * 16 + (P & 15);
      const int k = P >> 4;
      const int b0 = (it[k * 512] >> bit) & 1, b1 = (it[(2 + k) * 512] >> bit) & 1,
                b2 = (it[(4 + k) * 512] >> bit) & 1;
      // two's-complement u = (v - p)/2, or the offset-binary code (v - p)/2 + 4
      int v = off4 ? p - 8 + 2 * b0 + 4 * b1 + 8 * b2 + 16 * ((it[(6 + k) * 512] >> bit) & 1)
                   : p + 2 * b0 + 4 * b1 - 8 * b2;
      for (uint32_t x = excptr[r]; x < excptr[r + 1]; ++x)
        if (exccol[x] == (uint32_t)c) v = 8;
      out[(size_t)r * nblock * 24 + c] = (int8_t)v;
    }
  }
}

__global__ void k_dec_tail(const uint16_t* tail, uint16_t* out, int R, int TL, int TLp) {
  const size_t n = (size_t)R * TL;
  for (size_t e = blockIdx.x * (size_t)kThreads + threadIdx.x; e < n; e += (size_t)gridDim.x * kThreads) {
    const int r = (int)(e / TL), j = (int)(e % TL);
    out[e] = tail[(size_t)r * TLp + j];
  }
}

int grid_for(size_t n) {
  size_t g = (n + kThreads - 1) / kThreads;
  return (int)(g < 4096 ? (g ? g : 1) : 4096);
}

}  // namespace
}  // namespace q2

using namespace q2;

extern "C" int q2_launch_decode(const q2_handle* h, void* out, void* stream) {
  const q2_blob_header& d = h->hdr;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (d.fmt) {
    case Q2_FP16: {
      const size_t n = (size_t)d.R * d.C;
      k_dec_fp16<<<grid_for(n), kThreads, 0, st>>>(reinterpret_cast<const uint16_t*>(h->dev + d.off[SEC_FP16_W]),
                                                   static_cast<uint16_t*>(out), n);
      break;
    }
    case Q2_BPDQ:
      k_dec_bpdq<<<grid_for((size_t)d.R * d.C / 8), kThreads, 0, st>>>(
          h->dev + d.off[SEC_BPDQ_BITS], reinterpret_cast<const uint16_t*>(h->dev + d.off[SEC_BPDQ_VTAB]),
          static_cast<uint16_t*>(out), d.R, d.C, d.Rpad);
      break;
    case Q2_TRELLIS:
      k_dec_trellis<<<grid_for((size_t)d.R * d.C / 2), kThreads, 0, st>>>(
          h->dev + d.off[SEC_TRL_STREAM], reinterpret_cast<const uint32_t*>(h->dev + d.off[SEC_TRL_TABLE]),
          reinterpret_cast<const __half*>(h->dev + d.off[SEC_TRL_SCALE]), static_cast<float*>(out), d.R, d.C,
          d.Rpad);
      break;
    case Q2_LEECH: {
      k_dec_leech<<<grid_for((size_t)d.R * d.nblock), kThreads, 0, st>>>(
          h->dev + d.off[SEC_LEECH_PLANES], reinterpret_cast<const uint16_t*>(h->dev + d.off[SEC_LEECH_PARITY]),
          reinterpret_cast<const uint32_t*>(h->dev + d.off[SEC_LEECH_EXCPTR]),
          reinterpret_cast<const uint32_t*>(h->dev + d.off[SEC_LEECH_EXCCOL]), static_cast<int8_t*>(out), d.R,
          d.Rpad, d.nblock, d.layout == Q2_LEECH_OFFSET4 ? 1 : 0);
      if (d.tail) {
        size_t body = (size_t)d.R * d.nblock * 24;
        body = (body + 15) / 16 * 16;
        k_dec_tail<<<grid_for((size_t)d.R * d.tail), kThreads, 0, st>>>(
            reinterpret_cast<const uint16_t*>(h->dev + d.off[SEC_LEECH_TAIL]),
            reinterpret_cast<uint16_t*>(static_cast<unsigned char*>(out) + body), d.R, d.tail, d.tailpad);
      }
      break;
    }
    default:
      return Q2_EFMT;
  }
  return cudaGetLastError() == cudaSuccess ? Q2_OK : Q2_ECUDA;
}
