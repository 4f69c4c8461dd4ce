// Multi-token kernels (2 <= ntok <= 64) on CUDA cores: each lane decodes the
// weights of its row to fp32 eight at a time and accumulates every token.
// Same items, CTA ranges and fixed-order split-K reduction as the batch-1
// kernels.  BPDQ decodes through the per-(group, row) 4-entry value table
// (one rounding of c0*b0 + c1*b1 + off, as the packer stores it); the
// trellis through the shared 4096 x 2 table; Leech through the
// two's-complement planes plus the per-block parity term.
#include <cuda_fp16.h>

#include "q2_common.cuh"

extern __shared__ __align__(1024) unsigned char q2_smem[];

extern "C" int q2_launch_reduce(const q2_handle* h, const void* x, void* y, int ntok, void* stream);

namespace q2 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

// x of one 256-column slice for ntok tokens as fp32 [tok][i][b] with column
// 8b + i, so lanes that visit different column-bytes b read different banks.
__device__ __forceinline__ void stage_x_bi(const __half* x, int C, int col0, int ncols, int ntok,
                                           float* xs) {
  for (int e = threadIdx.x; e < ntok * 256; e += kThreads) {
    const int t = e >> 8, c = e & 255;
    const float v = (c < ncols) ? __half2float(x[(size_t)t * C + col0 + c]) : 0.f;
    xs[t * 256 + (c & 7) * 32 + (c >> 3)] = v;
  }
}

struct MtArgs {
  const unsigned char* bits;     // item stream
  const uint2* vtab;             // BPDQ: 4 halves per (g, row)
  const uint16_t* parity;        // Leech
  const __half* scale;           // trellis / Leech
  const __half* tail;            // Leech
  const uint32_t* excptr;
  const uint32_t* exccol;
  const uint32_t* table;         // trellis
  const __half* x;
  __half* y;
  Reduce rd;
  int R, C, nrb, ntok, nblock, tail_n, tailpad;
  float inv_sqrt8;
};

template <int NT>
__global__ void __launch_bounds__(kThreads) k_bpdq_mt(MtArgs a) {
  float* xs = reinterpret_cast<float*>(q2_smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int i0, i1;
  cta_range(a.rd.nslice * a.nrb, i0, i1);
  pdl_wait();
  pdl_trigger();
  for (int s0 = i0; s0 < i1;) {
    const int g = s0 / a.nrb;
    const int s1 = min(i1, (g + 1) * a.nrb);
    __syncthreads();
    stage_x_bi(a.x, a.C, g * Q2_SLICE, Q2_SLICE, a.ntok, xs);
    __syncthreads();
    for (int it = s0 + warp; it < s1; it += kWarps) {
      const int rb = it - g * a.nrb, row = rb * 32 + lane;
      const unsigned char* p = a.bits + (size_t)it * Q2_ITEM_BYTES_BPDQ + lane * 16;
      const uint4 w0 = ldg_stream(p), w1 = ldg_stream(p + 512), w2 = ldg_stream(p + 1024),
                  w3 = ldg_stream(p + 1536);
      const uint2 vt = a.vtab[(size_t)g * a.rd.Rpad + row];
      const float v[4] = {__half2float(__ushort_as_half(lo16(vt.x))), __half2float(__ushort_as_half(hi16(vt.x))),
                          __half2float(__ushort_as_half(lo16(vt.y))), __half2float(__ushort_as_half(hi16(vt.y)))};
      const uint32_t b0w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      const uint32_t b1w[8] = {w2.x, w2.y, w2.z, w2.w, w3.x, w3.y, w3.z, w3.w};
      float acc[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[t] = 0.f;
#pragma unroll 4
      for (int P = 0; P < 32; ++P) {
        const int beta = (P + lane) & 31;
        const uint32_t by0 = (b0w[P >> 2] >> (8 * (P & 3))) & 0xffu;
        const uint32_t by1 = (b1w[P >> 2] >> (8 * (P & 3))) & 0xffu;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const bool b0 = (by0 >> i) & 1, b1 = (by1 >> i) & 1;
          const float w = b1 ? (b0 ? v[3] : v[2]) : (b0 ? v[1] : v[0]);
#pragma unroll
          for (int t = 0; t < NT; ++t)
            if (t < a.ntok) acc[t] = fmaf(w, xs[t * 256 + i * 32 + beta], acc[t]);
        }
      }
#pragma unroll
      for (int t = 0; t < NT; ++t)
        if (t < a.ntok) a.rd.partial[((size_t)t * a.rd.nslice + g) * a.rd.Rpad + row] = acc[t];
    }
    s0 = s1;
  }
}

template <int NT>
__global__ void __launch_bounds__(kThreads) k_leech_mt(MtArgs a) {
  float* xs = reinterpret_cast<float*>(q2_smem);
  float* xb = xs + 64 * 256;            // [11][ntok] block sums
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int i0, i1;
  cta_range(a.rd.nslice * a.nrb, i0, i1);
  pdl_wait();
  pdl_trigger();
  for (int s0 = i0; s0 < i1;) {
    const int sl = s0 / a.nrb;
    const int s1 = min(i1, (sl + 1) * a.nrb);
    const int bfirst = (sl * Q2_SLICE + 23) / 24;
    const int blast = min(a.nblock - 1, (sl * Q2_SLICE + Q2_SLICE + 23) / 24 - 1);
    const int nbk = max(0, blast - bfirst + 1);
    __syncthreads();
    stage_x_bi(a.x, a.C, sl * Q2_SLICE, min(Q2_SLICE, a.C - sl * Q2_SLICE), a.ntok, xs);
    for (int e = threadIdx.x; e < nbk * a.ntok; e += kThreads) {
      const int j = e / a.ntok, t = e % a.ntok;
      const __half* xp = a.x + (size_t)t * a.C + (size_t)(bfirst + j) * 24;
      float v = 0.f;
      for (int i = 0; i < 24; ++i) v += __half2float(xp[i]);
      xb[j * 64 + t] = v;
    }
    __syncthreads();
    for (int it = s0 + warp; it < s1; it += kWarps) {
      const int rb = it - sl * a.nrb, row = rb * 32 + lane;
      const unsigned char* p = a.bits + (size_t)it * Q2_ITEM_BYTES_LEECH + lane * 16;
      uint32_t pw[3][8];
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        const uint4 c0 = ldg_stream(p + (2 * q) * 512), c1 = ldg_stream(p + (2 * q + 1) * 512);
        pw[q][0] = c0.x; pw[q][1] = c0.y; pw[q][2] = c0.z; pw[q][3] = c0.w;
        pw[q][4] = c1.x; pw[q][5] = c1.y; pw[q][6] = c1.z; pw[q][7] = c1.w;
      }
      float acc[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[t] = 0.f;
#pragma unroll 2
      for (int P = 0; P < 32; ++P) {
        const int beta = (P + lane) & 31;
        const uint32_t by0 = (pw[0][P >> 2] >> (8 * (P & 3))) & 0xffu;
        const uint32_t by1 = (pw[1][P >> 2] >> (8 * (P & 3))) & 0xffu;
        const uint32_t by2 = (pw[2][P >> 2] >> (8 * (P & 3))) & 0xffu;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          // 2u = 2*b0 + 4*b1 - 8*b2 (the parity part is added per block below)
          const float w = (float)(2 * (int)((by0 >> i) & 1) + 4 * (int)((by1 >> i) & 1) - 8 * (int)((by2 >> i) & 1));
#pragma unroll
          for (int t = 0; t < NT; ++t)
            if (t < a.ntok) acc[t] = fmaf(w, xs[t * 256 + i * 32 + beta], acc[t]);
        }
      }
      const uint32_t par = a.parity[(size_t)sl * a.rd.Rpad + row];
      for (int j = 0; j < nbk; ++j)
        if ((par >> j) & 1u) {
#pragma unroll
          for (int t = 0; t < NT; ++t)
            if (t < a.ntok) acc[t] += xb[j * 64 + t];
        }
#pragma unroll
      for (int t = 0; t < NT; ++t)
        if (t < a.ntok) a.rd.partial[((size_t)t * a.rd.nslice + sl) * a.rd.Rpad + row] = acc[t];
    }
    s0 = s1;
  }
}

constexpr uint32_t kHashHi = 0x9E37u << 16;

template <int NT>
__global__ void __launch_bounds__(kThreads) k_trellis_mt(MtArgs a) {
  uint32_t* tab = reinterpret_cast<uint32_t*>(q2_smem);              // 16 KiB
  float* xs = reinterpret_cast<float*>(q2_smem + 4096 * 4);          // [tok][256]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 4096; i += kThreads) tab[i] = a.table[i];
  int i0, i1;
  cta_range(a.rd.nslice * a.nrb, i0, i1);
  pdl_wait();
  pdl_trigger();
  for (int s0 = i0; s0 < i1;) {
    const int sg = s0 / a.nrb;
    const int s1 = min(i1, (sg + 1) * a.nrb);
    __syncthreads();
    for (int e = threadIdx.x; e < a.ntok * 256; e += kThreads) {
      const int t = e >> 8, c = e & 255;
      xs[e] = __half2float(a.x[(size_t)t * a.C + sg * 256 + c]);
    }
    __syncthreads();
    for (int it = s0 + warp; it < s1; it += kWarps) {
      const int rb = it - sg * a.nrb, row = rb * 32 + lane;
      const unsigned char* p = a.bits + (size_t)it * Q2_ITEM_BYTES_TRL + lane * 16;
      const uint4 w0 = ldg_stream(p), w1 = ldg_stream(p + 512), w2 = ldg_stream(p + 1024),
                  w3 = ldg_stream(p + 1536);
      const uint32_t W[16] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w,
                              w2.x, w2.y, w2.z, w2.w, w3.x, w3.y, w3.z, w3.w};
      float acc[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[t] = 0.f;
#pragma unroll 8
      for (int k = 0; k < 128; ++k) {
        const int n = 127 - k;
        const uint32_t f = __funnelshift_r(W[n >> 3], W[((n >> 3) + 1) & 15], 4 * (n & 7));
        uint32_t e = tab[(f * kHashHi) >> 20];
        e ^= (f & 1u) ? 0x80008000u : 0u;
        const float u0 = __half2float(__ushort_as_half(lo16(e)));
        const float u1 = __half2float(__ushort_as_half(hi16(e)));
#pragma unroll
        for (int t = 0; t < NT; ++t)
          if (t < a.ntok) {
            const float2 xx = *reinterpret_cast<const float2*>(xs + t * 256 + 2 * k);
            acc[t] = fmaf(u0, xx.x, fmaf(u1, xx.y, acc[t]));
          }
      }
#pragma unroll
      for (int t = 0; t < NT; ++t)
        if (t < a.ntok) a.rd.partial[((size_t)t * a.rd.nslice + sg) * a.rd.Rpad + row] = acc[t];
    }
    s0 = s1;
  }
}

Reduce make_reduce(const q2_handle* h) {
  Reduce r;
  r.partial = static_cast<float*>(h->ws);
  r.nslice = h->hdr.nslice;
  r.Rpad = h->hdr.Rpad;
  return r;
}

template <int NT>
int launch_nt(int fmt, const MtArgs& a, int items, void* stream) {
  const int grid = max(1, min(items, 2 * dev_info().sms));
  if (fmt == Q2_BPDQ) return launch_pdl(k_bpdq_mt<NT>, a, grid, kThreads, NT * 256 * 4, stream);
  if (fmt == Q2_LEECH) return launch_pdl(k_leech_mt<NT>, a, grid, kThreads, 64 * 256 * 4 + 11 * 64 * 4, stream);
  return launch_pdl(k_trellis_mt<NT>, a, grid, kThreads, 4096 * 4 + NT * 256 * 4, stream);
}

}  // namespace
}  // namespace q2

using namespace q2;

extern "C" int q2_mt_launch(const q2_handle* h, const void* x, void* y, int ntok, void* stream) {
  const q2_blob_header& d = h->hdr;
  MtArgs a = {};
  a.x = static_cast<const __half*>(x);
  a.y = static_cast<__half*>(y);
  a.rd = make_reduce(h);
  a.R = d.R;
  a.C = d.C;
  a.nrb = q2_nrb(d);
  a.ntok = ntok;
  switch (d.fmt) {
    case Q2_BPDQ:
      a.bits = h->dev + d.off[SEC_BPDQ_BITS];
      a.vtab = reinterpret_cast<const uint2*>(h->dev + d.off[SEC_BPDQ_VTAB]);
      break;
    case Q2_TRELLIS:
      a.bits = h->dev + d.off[SEC_TRL_STREAM];
      a.table = reinterpret_cast<const uint32_t*>(h->dev + d.off[SEC_TRL_TABLE]);
      a.scale = reinterpret_cast<const __half*>(h->dev + d.off[SEC_TRL_SCALE]);
      break;
    case Q2_LEECH:
      a.bits = h->dev + d.off[SEC_LEECH_PLANES];
      a.parity = reinterpret_cast<const uint16_t*>(h->dev + d.off[SEC_LEECH_PARITY]);
      a.scale = reinterpret_cast<const __half*>(h->dev + d.off[SEC_LEECH_SCALE]);
      a.tail = reinterpret_cast<const __half*>(h->dev + d.off[SEC_LEECH_TAIL]);
      a.excptr = reinterpret_cast<const uint32_t*>(h->dev + d.off[SEC_LEECH_EXCPTR]);
      a.exccol = reinterpret_cast<const uint32_t*>(h->dev + d.off[SEC_LEECH_EXCCOL]);
      a.nblock = d.nblock;
      a.tail_n = d.tail;
      a.tailpad = d.tailpad;
      a.inv_sqrt8 = d.inv_sqrt8;
      break;
    default:
      return Q2_EFMT;
  }
  const int items = d.nslice * a.nrb;
  int st;
  if (ntok <= 4) st = launch_nt<4>(d.fmt, a, items, stream);
  else if (ntok <= 8) st = launch_nt<8>(d.fmt, a, items, stream);
  else if (ntok <= 16) st = launch_nt<16>(d.fmt, a, items, stream);
  else if (ntok <= 32) st = launch_nt<32>(d.fmt, a, items, stream);
  else st = launch_nt<64>(d.fmt, a, items, stream);
  return st ? st : q2_launch_reduce(h, x, y, ntok, stream);
}
