// Batch-1 kernels (ntok == 1) for the packed formats and the no-weights
// control.  One lane owns one output row; a warp owns 32 rows of one
// 256-column slice (an "item").  CTAs take contiguous, equal shares of the
// items in slice-major order and keep the x-dependent tables of the current
// slice in shared memory.  Per-slice partial sums go to the workspace with
// plain stores; a second launch (q2_reduce.cu) sums them in slice order
// (deterministic) and writes y.
//
// BPDQ and Leech use subset-sum tables in place of a per-weight decode: for
// each 8-column byte of a bit-plane the table holds the sum of the x values
// the byte selects, so one shared-memory load covers 8 weights of a plane.
// This is the "multiply without dequantising" formulation of
// "Qwen3-8B -- 2-bit BPDQ (packed)", Kernels (c0*S0 + c1*S1 + off*sum(x)
// per 256-column group), laid out for 32 banks: each lane visits the 32
// column-bytes of its row in an order rotated by its lane index, so the 32
// lanes of a load always hit 32 different banks.
//
// One CTA of 16 warps per SM (grid = SM count; each CTA asks for more than
// half of the SM's shared memory so no SM ever holds two).  Launches use
// programmatic dependent launch: a CTA prefetches its weights into L2 and
// its first items into registers, then waits for the previous kernel on the
// stream (griddepcontrol) before it touches x or the workspace, and lets the
// dependent reduction and the next GEMV's CTAs get scheduled while it runs.
#include <cuda_fp16.h>

#include <mutex>
#include <vector>

#include "q2_common.cuh"

extern __shared__ __align__(1024) unsigned char q2_smem[];

extern "C" int q2_launch_reduce(const q2_handle* h, const void* x, void* y, int ntok, void* stream);

namespace q2 {
namespace {


// T lookup for byte b of word at rotated position P (see build_table).
__device__ __forceinline__ float tl(uint32_t lane4, uint32_t word, int b, int P) {
  const uint32_t a = __byte_perm(word, lane4, 0x5504u | ((uint32_t)b << 4));
  return *reinterpret_cast<const float*>(q2_smem + a + P * 4);
}

// Sum of the table entries selected by 32 rotated bytes (two uint4 chunks).
__device__ __forceinline__ float plane_sum(uint32_t lane4, const uint4& c0, const uint4& c1) {
  const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int P = 0; P < 32; ++P) s[P & 3] += tl(lane4, w[P >> 2], P & 3, P);
  return (s[0] + s[1]) + (s[2] + s[3]);
}

struct BpdqArgs {
  const unsigned char* bits;
  const __half2* c01;
  const __half* off;
  const __half* x;
  __half* y;
  Reduce rd;
  int R, C, nrb;
  int ntok;            // tokens (the multi-token kernel; 1 elsewhere)
};

__device__ __forceinline__ void ld_item4(const unsigned char* base, int it, int lane, uint4 (&w)[4]) {
  const unsigned char* p = base + (size_t)it * Q2_ITEM_BYTES_BPDQ + lane * 16;
#pragma unroll
  for (int k = 0; k < 4; ++k) w[k] = ldg_stream(p + k * 512);
}

// The CTA's items are contiguous in the bit stream, and the coefficients of a
// slice's row blocks are contiguous too: thread 0 prefetches all of them
// into L2 before waiting on the previous kernel, so the weight stream of
// this GEMV overlaps the tail of the previous one.
__device__ __forceinline__ void prefetch_items(const unsigned char* base, int item_bytes, int i0, int i1) {
  if (i1 > i0) prefetch_l2(base + (size_t)i0 * item_bytes, (size_t)(i1 - i0) * item_bytes);
}

__device__ __forceinline__ void prefetch_rows(const void* base, int elem_bytes, int nrb, int Rpad, int i0, int i1) {
  // rows of items i0..i1-1 in [slice][Rpad] arrays: one contiguous run per slice
  for (int s0 = i0; s0 < i1;) {
    const int g = s0 / nrb, s1 = min(i1, (g + 1) * nrb);
    const size_t first = (size_t)g * Rpad + (size_t)(s0 - g * nrb) * 32;
    const size_t n = (size_t)(s1 - s0) * 32 * elem_bytes;
    const size_t a0 = (first * elem_bytes) & ~(size_t)15;
    const size_t a1 = (first * elem_bytes + n + 15) & ~(size_t)15;
    prefetch_l2(static_cast<const char*>(base) + a0, a1 - a0);
    s0 = s1;
  }
}

// ------------------------------------------------------- pipelined items
// run_items drives every subset-sum kernel.  The CTA walks its contiguous
// item range one slice at a time: item it of a slice goes to warp
// (it - first item) mod W, and each warp keeps AHEAD items beyond the one
// it is summing in flight in registers (F::load), so a CTA has
// (AHEAD + 1) x W items of weights outstanding.  The first AHEAD loads of a
// slice are issued before the CTA waits on the previous kernel (weights do
// not depend on it); F::slice then builds the slice's x tables, F::ready
// reads what every item of the slice shares, and F::compute sums one item
// and stores its partials.
template <int W, int AHEAD, class F>
__device__ __forceinline__ void run_items(F& f, int nrb, int i0, int i1) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  bool waited = false;
  for (int s0 = i0; s0 < i1;) {
    const int g = s0 / nrb;
    const int s1 = min(i1, (g + 1) * nrb);
    typename F::Item buf[AHEAD + 1];
    const int it0 = s0 + warp;
#pragma unroll
    for (int d = 0; d < AHEAD; ++d)
      if (it0 + d * W < s1) f.load(it0 + d * W, g, lane, buf[d]);
    if (!waited) {
      pdl_wait();
      pdl_trigger();
      waited = true;
    }
    __syncthreads();                              // every warp is done with the previous tables
    f.slice(g);
    __syncthreads();
    f.ready();
    // the AHEAD + 1 buffers are indexed statically: AHEAD + 1 items per trip
    for (int base = it0; base < s1; base += (AHEAD + 1) * W) {
#pragma unroll
      for (int u = 0; u <= AHEAD; ++u) {
        const int it = base + u * W;
        if (it < s1) {
          const int nx = it + AHEAD * W;
          if (nx < s1) f.load(nx, g, lane, buf[(u + AHEAD) % (AHEAD + 1)]);
          f.compute(it, g, lane, buf[u]);
        }
      }
    }
    s0 = s1;
  }
}

// Launch shapes, measured on GB300: BPDQ 16 warps with 2 items ahead (the
// 8B stack); Leech, whose items are 1.5x larger, 8 warps with 3 ahead (the
// 14B layers).
constexpr int kBpdqWarps = 16, kBpdqAhead = 2;
constexpr int kLeechWarps = 8, kLeechAhead = 3;

// ------------------------------------------------------------------- BPDQ
template <int NT>
struct BpdqF {
  struct Item {
    uint4 w[4];          // 64 bytes of planes: two uint4 per plane
    uint32_t c01;        // c0 | c1 << 16 (fp16)
    unsigned short off;  // fp16
  };
  const BpdqArgs& a;
  float* T;
  float* gsum;
  float xs = 0.f;        // sum of x over the slice
  __device__ void load(int it, int g, int lane, Item& b) const {
    ld_item4(a.bits, it, lane, b.w);
    const size_t r = (size_t)g * a.rd.Rpad + (size_t)(it - g * a.nrb) * 32 + lane;
    b.c01 = __ldg(reinterpret_cast<const unsigned int*>(a.c01) + r);
    b.off = __ldg(reinterpret_cast<const unsigned short*>(a.off) + r);
  }
  __device__ void slice(int g) {
    build_table<NT>(a.x + (size_t)g * Q2_SLICE, Q2_SLICE, T, gsum);
  }
  __device__ void ready() { xs = *gsum; }
  __device__ void compute(int it, int g, int lane, const Item& b) {
    const uint32_t lane4 = lane * 4u;
    const float S0 = plane_sum(lane4, b.w[0], b.w[1]);
    const float S1 = plane_sum(lane4, b.w[2], b.w[3]);
    const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&b.c01));
    const float of = __half2float(__ushort_as_half(b.off));
    const int row = (it - g * a.nrb) * 32 + lane;
    a.rd.partial[(size_t)g * a.rd.Rpad + row] = fmaf(c.x, S0, fmaf(c.y, S1, of * xs));
  }
};

template <int W, int AHEAD>
__global__ void __launch_bounds__(W * 32, 1) k_bpdq_b1(BpdqArgs a) {
  int i0, i1;
  cta_range(a.rd.nslice * a.nrb, i0, i1);
  if (threadIdx.x == 0) {
    prefetch_items(a.bits, Q2_ITEM_BYTES_BPDQ, i0, i1);
    prefetch_rows(a.c01, 4, a.nrb, a.rd.Rpad, i0, i1);
    prefetch_rows(a.off, 2, a.nrb, a.rd.Rpad, i0, i1);
  }
  float* T = reinterpret_cast<float*>(q2_smem);
  BpdqF<W * 32> f{a, T, T + (kBuildBytes - 16) / 4};
  run_items<W, AHEAD>(f, a.nrb, i0, i1);
}

// ------------------------------------------------------------------ Leech
struct LeechArgs {
  const unsigned char* planes;
  const uint16_t* parity;     // [nslice][Rpad]
  const __half* scale;        // [Rpad]
  const __half* tail;         // [Rpad][tailpad]
  const uint32_t* excptr;     // [Rpad + 1]
  const uint32_t* exccol;
  const __half* x;
  __half* y;
  Reduce rd;
  int R, C, nrb, nblock, tail_n, tailpad;
  float inv_sqrt8;
};

__device__ __forceinline__ void ld_item6(const unsigned char* base, int it, int lane, uint4 (&w)[6]) {
  const unsigned char* p = base + (size_t)it * Q2_ITEM_BYTES_LEECH + lane * 16;
#pragma unroll
  for (int k = 0; k < 6; ++k) w[k] = ldg_stream(p + k * 512);
}

// The three planes hold the two's-complement bits of u = (v - p)/2 per
// weight (p = the block's parity bit), so v = p + 2*b0 + 4*b1 - 8*b2: three
// subset sums plus, per 24-column block of the slice, the block sum of x
// when the row's parity bit for the block is set.
template <int NT>
struct LeechF {
  struct Item {
    uint4 w[6];
    uint32_t pw;         // parity bits of the slice's blocks for this row
  };
  const LeechArgs& a;
  float* T;
  float* gsum;
  float* xb;             // block sums of x in the slice, <= 11
  int nbk;
  __device__ void load(int it, int g, int lane, Item& b) const {
    ld_item6(a.planes, it, lane, b.w);
    b.pw = __ldg(a.parity + (size_t)g * a.rd.Rpad + (size_t)(it - g * a.nrb) * 32 + lane);
  }
  __device__ void slice(int g) {
    const int bfirst = (g * Q2_SLICE + 23) / 24;
    const int blast = min(a.nblock - 1, (g * Q2_SLICE + Q2_SLICE + 23) / 24 - 1);
    nbk = max(0, blast - bfirst + 1);
    if ((int)threadIdx.x < nbk) {
      const __half* xp = a.x + (size_t)(bfirst + threadIdx.x) * 24;
      float v = 0.f;
      for (int i = 0; i < 24; ++i) v += __half2float(xp[i]);
      xb[threadIdx.x] = v;
    }
    build_table<NT>(a.x + (size_t)g * Q2_SLICE, min(Q2_SLICE, a.C - g * Q2_SLICE), T, gsum);
  }
  __device__ void ready() {}
  __device__ void compute(int it, int g, int lane, const Item& b) {
    const uint32_t lane4 = lane * 4u;
    const float P0 = plane_sum(lane4, b.w[0], b.w[1]);
    const float P1 = plane_sum(lane4, b.w[2], b.w[3]);
    const float P2 = plane_sum(lane4, b.w[4], b.w[5]);
    float pacc = 0.f;
    for (int j = 0; j < nbk; ++j) pacc += ((b.pw >> j) & 1u) ? xb[j] : 0.f;
    const int row = (it - g * a.nrb) * 32 + lane;
    a.rd.partial[(size_t)g * a.rd.Rpad + row] = fmaf(2.f, P0, fmaf(4.f, P1, fmaf(-8.f, P2, pacc)));
  }
};

template <int W, int AHEAD>
__global__ void __launch_bounds__(W * 32, 1) k_leech_b1(LeechArgs a) {
  int i0, i1;
  cta_range(a.rd.nslice * a.nrb, i0, i1);
  if (threadIdx.x == 0) {
    prefetch_items(a.planes, Q2_ITEM_BYTES_LEECH, i0, i1);
    prefetch_rows(a.parity, 2, a.nrb, a.rd.Rpad, i0, i1);
  }
  float* T = reinterpret_cast<float*>(q2_smem);
  LeechF<W * 32> f{a, T, T + (kBuildBytes - 16) / 4, reinterpret_cast<float*>(q2_smem + kBuildBytes), 0};
  run_items<W, AHEAD>(f, a.nrb, i0, i1);
}

// ------------------------------------------------------- no-weights control
// Same grid, PDL, table build, per-lane lookups and reduction as k_bpdq_b1;
// the "weight" words are derived from the lane and item index instead of
// being loaded, so the kernel reads x and writes the workspace and y only.
template <int NT>
struct NoWeightsF {
  struct Item {
    uint32_t h;
  };
  const BpdqArgs& a;
  float* T;
  float* gsum;
  __device__ void load(int it, int, int lane, Item& b) const { b.h = (uint32_t)it * 0x9E3779B9u ^ (lane * 0x85EBCA6Bu); }
  float xs = 0.f;
  __device__ void slice(int g) { build_table<NT>(a.x + (size_t)g * Q2_SLICE, Q2_SLICE, T, gsum); }
  __device__ void ready() { xs = *gsum; }
  __device__ void compute(int it, int g, int lane, const Item& b) {
    const uint32_t h = b.h, lane4 = lane * 4u;
    const uint4 w0 = make_uint4(h, h ^ 0x5bd1e995u, h * 3u, h * 5u);
    const uint4 w1 = make_uint4(h * 7u, h ^ 0x27d4eb2fu, h * 11u, h * 13u);
    const float S0 = plane_sum(lane4, w0, w1);
    const float S1 = plane_sum(lane4, w1, w0);
    const int row = (it - g * a.nrb) * 32 + lane;
    a.rd.partial[(size_t)g * a.rd.Rpad + row] = fmaf(0.02f, S0, fmaf(0.01f, S1, 0.01f * xs));
  }
};

template <int W>
__global__ void __launch_bounds__(W * 32, 1) k_noweights_b1(BpdqArgs a) {
  int i0, i1;
  cta_range(a.rd.nslice * a.nrb, i0, i1);
  float* T = reinterpret_cast<float*>(q2_smem);
  NoWeightsF<W * 32> f{a, T, T + (kBuildBytes - 16) / 4};
  run_items<W, 1>(f, a.nrb, i0, i1);
}

// ------------------------------------------------- BPDQ, 2 to 6 tokens
// The subset-sum method for several tokens at once.  For the token pair
// (2p, 2p+1) the slice's table holds float2 entries
//   E_p[v][b] = (sum of x_2p over the set bits of byte v at column-byte b,
//                the same for x_2p+1)
// at byte offset p*64 KiB + v*256 + b*8, with no duplicated columns: a lane
// at rotated position P reads column-byte b = (P + lane) mod 32, whose
// address byte b*8 it keeps in one of 11 lane-constant registers (three
// positions each), so one byte permute still forms v*256 + b*8.  Each
// lookup is then one 8-byte shared load and one packed fp32 add per token
// pair; a half-warp's 16 lanes read 16 different column-bytes (conflict-free).
constexpr int kMtMaxTok = 6;
constexpr int kPairBytes = 256 * 32 * 8;                   // 64 KiB per token pair

template <int NT, int NP>
__device__ __forceinline__ void build_pairs(const __half* __restrict__ x, int ntok, int ldx, int col0, float* T,
                                            float* gsum) {
  for (int e = threadIdx.x; e < 512 * NP; e += NT) {
    const int p = e >> 9, h = (e >> 5) & 15, b = e & 31;
    float xa[8], xb[8];
    {
      const uint4 raw = *reinterpret_cast<const uint4*>(x + (size_t)(2 * p) * ldx + col0 + 8 * b);
      const __half2* hv = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __half22float2(hv[k]);
        xa[2 * k] = f.x;
        xa[2 * k + 1] = f.y;
      }
    }
    if (2 * p + 1 < ntok) {                            // an odd count leaves the last pair half empty
      const uint4 raw = *reinterpret_cast<const uint4*>(x + (size_t)(2 * p + 1) * ldx + col0 + 8 * b);
      const __half2* hv = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __half22float2(hv[k]);
        xb[2 * k] = f.x;
        xb[2 * k + 1] = f.y;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) xb[i] = 0.f;
    }
    float2 hs = make_float2(0.f, 0.f);                  // sums selected by the high nibble h
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if ((h >> i) & 1) {
        hs.x += xa[4 + i];
        hs.y += xb[4 + i];
      }
    float2 sv[16];
    sv[0] = hs;
#pragma unroll
    for (int n = 1; n < 16; ++n) {
      const int low = n & -n;
      const int i = (low == 1) ? 0 : (low == 2) ? 1 : (low == 4) ? 2 : 3;
      sv[n] = make_float2(sv[n ^ low].x + xa[i], sv[n ^ low].y + xb[i]);
    }
    float2* col = reinterpret_cast<float2*>(reinterpret_cast<char*>(T) + p * kPairBytes) + (h * 16) * 32 + b;
#pragma unroll
    for (int n = 0; n < 16; ++n) col[n * 32] = sv[n];
    if (h == 15) {                                      // this warp holds the 32 bytes' full sums
      float va = sv[15].x, vb = sv[15].y;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        va += __shfl_xor_sync(0xffffffffu, va, o);
        vb += __shfl_xor_sync(0xffffffffu, vb, o);
      }
      if (b == 0) {
        gsum[2 * p] = va;
        gsum[2 * p + 1] = vb;
      }
    }
  }
}

template <int NT, int NP>
struct BpdqMtF {
  struct Item {
    uint4 w[4];
    uint32_t c01;
    unsigned short off;
  };
  const BpdqArgs& a;
  float* T;
  float* gsum;
  uint32_t rot[11];      // byte j of rot[k]: ((3k + j + lane) mod 32) * 8; byte 3 = 0
  float xs[2 * NP];      // per-token sums of x over the slice
  __device__ void init(int lane) {
#pragma unroll
    for (int k = 0; k < 11; ++k) {
      uint32_t r = 0;
#pragma unroll
      for (int j = 0; j < 3; ++j) r |= (uint32_t)(((3 * k + j + lane) & 31) * 8) << (8 * j);
      rot[k] = r;
    }
  }
  __device__ void load(int it, int g, int lane, Item& b) const {
    ld_item4(a.bits, it, lane, b.w);
    const size_t r = (size_t)g * a.rd.Rpad + (size_t)(it - g * a.nrb) * 32 + lane;
    b.c01 = __ldg(reinterpret_cast<const unsigned int*>(a.c01) + r);
    b.off = __ldg(reinterpret_cast<const unsigned short*>(a.off) + r);
  }
  __device__ void slice(int g) { build_pairs<NT, NP>(a.x, a.ntok, a.C, g * Q2_SLICE, T, gsum); }
  __device__ void ready() {
#pragma unroll
    for (int t = 0; t < 2 * NP; ++t) xs[t] = gsum[t];
  }
  __device__ void plane(const uint4& c0, const uint4& c1, float2 (&S)[NP]) const {
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const char* base = reinterpret_cast<const char*>(T);
#pragma unroll
    for (int P = 0; P < 32; ++P) {
      const uint32_t sel = (4u + (uint32_t)(P % 3)) | ((uint32_t)(P & 3) << 4) | 0x7700u;
      const uint32_t ad = __byte_perm(w[P >> 2], rot[P / 3], sel);
#pragma unroll
      for (int p = 0; p < NP; ++p) S[p] = __fadd2_rn(S[p], *reinterpret_cast<const float2*>(base + p * kPairBytes + ad));
    }
  }
  __device__ void compute(int it, int g, int lane, const Item& b) {
    float2 S0[NP], S1[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) S0[p] = S1[p] = make_float2(0.f, 0.f);
    plane(b.w[0], b.w[1], S0);
    plane(b.w[2], b.w[3], S1);
    const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&b.c01));
    const float of = __half2float(__ushort_as_half(b.off));
    const int row = (it - g * a.nrb) * 32 + lane;
    float* out = a.rd.partial + (size_t)g * a.rd.Rpad + row;
    const size_t tstride = (size_t)a.rd.nslice * a.rd.Rpad;
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      out[(2 * p) * tstride] = fmaf(c.x, S0[p].x, fmaf(c.y, S1[p].x, of * xs[2 * p]));
      if (2 * p + 1 < a.ntok) out[(2 * p + 1) * tstride] = fmaf(c.x, S0[p].y, fmaf(c.y, S1[p].y, of * xs[2 * p + 1]));
    }
  }
};

template <int W, int AHEAD, int NP>
__global__ void __launch_bounds__(W * 32, 1) k_bpdq_mt(BpdqArgs a) {
  int i0, i1;
  cta_range(a.rd.nslice * a.nrb, i0, i1);
  if (threadIdx.x == 0) {
    prefetch_items(a.bits, Q2_ITEM_BYTES_BPDQ, i0, i1);
    prefetch_rows(a.c01, 4, a.nrb, a.rd.Rpad, i0, i1);
    prefetch_rows(a.off, 2, a.nrb, a.rd.Rpad, i0, i1);
  }
  float* T = reinterpret_cast<float*>(q2_smem);
  BpdqMtF<W * 32, NP> f{a, T, reinterpret_cast<float*>(q2_smem + NP * kPairBytes)};
  f.init(threadIdx.x & 31);
  run_items<W, AHEAD>(f, a.nrb, i0, i1);
}

// ---------------------------------------------------------------- trellis
// Lane = row, item = (segment, 32 rows).  The 16 KiB table and all of x sit
// in shared memory for the whole kernel.  Step k of a segment reads the
// 16-bit state at bit offset 4*(127 - k) of the lane's 512-bit packet (a
// funnel shift of two words), hashes it, loads one fp16 pair, flips both
// signs by state bit 0 and accumulates two fp32 FMAs.
struct TrellisArgs {
  const unsigned char* stream;
  const uint32_t* table;     // 4096 half2
  const __half* scale;
  const __half* x;
  __half* y;
  Reduce rd;
  int R, C, nrb;
};

constexpr uint32_t kHashHi = 0x9E37u << 16;   // (s*0x9E37 mod 2^16) lands in bits 16..31

__device__ __forceinline__ void ld_trl(const unsigned char* base, int it, int lane, uint4 (&w)[4]) {
  const unsigned char* p = base + (size_t)it * Q2_ITEM_BYTES_TRL + lane * 16;
#pragma unroll
  for (int k = 0; k < 4; ++k) w[k] = ldg_stream(p + k * 512);
}

// Items of every segment in one pass: x and the table stay in shared memory
// for the whole kernel, so the "slice" step of run_items only copies x.
template <int NT>
struct TrellisF {
  struct Item {
    uint4 w[4];
  };
  const TrellisArgs& a;
  const uint32_t* tab;
  uint32_t* xs;
  __device__ void load(int it, int, int lane, Item& b) const { ld_trl(a.stream, it, lane, b.w); }
  __device__ void slice(int) {
    const uint32_t* xg = reinterpret_cast<const uint32_t*>(a.x);
    for (int i = threadIdx.x; i < a.C / 2; i += NT) xs[i] = xg[i];
  }
  __device__ void ready() {}
  __device__ void compute(int it, int, int lane, const Item& b) {
    const int sg = it / a.nrb, rb = it - sg * a.nrb;
    const uint32_t W[16] = {b.w[0].x, b.w[0].y, b.w[0].z, b.w[0].w, b.w[1].x, b.w[1].y, b.w[1].z, b.w[1].w,
                            b.w[2].x, b.w[2].y, b.w[2].z, b.w[2].w, b.w[3].x, b.w[3].y, b.w[3].z, b.w[3].w};
    const uint4* xv = reinterpret_cast<const uint4*>(xs + sg * 128);
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int k4 = 0; k4 < 32; ++k4) {
      const uint4 x4 = xv[k4];
      const uint32_t xx[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int k = k4 * 4 + kk;
        const int n = 127 - k;
        const uint32_t f = __funnelshift_r(W[n >> 3], W[((n >> 3) + 1) & 15], 4 * (n & 7));
        const uint32_t h = f * kHashHi;
        uint32_t e = tab[h >> 20];
        e ^= (f & 1u) ? 0x80008000u : 0u;
        if (kk & 1) {
          acc1 = fma_h(lo16(e), lo16(xx[kk]), acc1);
          acc1 = fma_h(hi16(e), hi16(xx[kk]), acc1);
        } else {
          acc0 = fma_h(lo16(e), lo16(xx[kk]), acc0);
          acc0 = fma_h(hi16(e), hi16(xx[kk]), acc0);
        }
      }
    }
    a.rd.partial[(size_t)sg * a.rd.Rpad + rb * 32 + lane] = acc0 + acc1;
  }
};

constexpr int kTrellisWarps = 16, kTrellisAhead = 1;

template <int W, int AHEAD>
__global__ void __launch_bounds__(W * 32, 1) k_trellis_b1(TrellisArgs a) {
  uint32_t* tab = reinterpret_cast<uint32_t*>(q2_smem);                 // 16 KiB
  uint32_t* xs = reinterpret_cast<uint32_t*>(q2_smem + 4096 * 4);      // x as half2, C/2 words
  int i0, i1;
  cta_range(a.rd.nslice * a.nrb, i0, i1);
  if (threadIdx.x == 0) prefetch_items(a.stream, Q2_ITEM_BYTES_TRL, i0, i1);
  for (int i = threadIdx.x; i < 4096; i += W * 32) tab[i] = a.table[i];
  TrellisF<W * 32> f{a, tab, xs};
  run_items<W, AHEAD>(f, 1 << 30, i0, i1);         // one pass over all segments
}

// Batch-1 kernels ask for more than half of an SM's shared memory, so an SM
// never holds two CTAs of them.  Under programmatic dependent launch the
// next GEMV's CTAs are placed while the current GEMV drains; an SM whose
// CTA has already left could otherwise take two CTAs of the same grid (and
// another SM none), and those two would set the GEMV's end.
constexpr int kOneCtaSmem = 116 * 1024;
static_assert(kBuildBytes + 64 <= kOneCtaSmem, "batch-1 tables fit the one-CTA footprint");

template <typename A>
int launch(const q2_handle* h, void (*kernel)(A), const A& args, int smem, int items, const void* x, void* y,
           void* stream, int threads, int ntok = 1) {
  const int grid = max(1, min(items, dev_info().sms));
  const int st = launch_pdl(kernel, args, grid, threads, smem, stream);
  return st ? st : q2_launch_reduce(h, x, y, ntok, stream);
}

Reduce make_reduce(const q2_handle* h) {
  Reduce r;
  r.partial = static_cast<float*>(h->ws);
  r.nslice = h->hdr.nslice;
  r.Rpad = h->hdr.Rpad;
  return r;
}

}  // namespace
}  // namespace q2

using namespace q2;

extern "C" int q2_b1_bpdq(const q2_handle* h, const void* x, void* y, void* stream) {
  const q2_blob_header& d = h->hdr;
  BpdqArgs a;
  a.bits = h->dev + d.off[SEC_BPDQ_BITS];
  a.c01 = reinterpret_cast<const __half2*>(h->dev + d.off[SEC_BPDQ_C01]);
  a.off = reinterpret_cast<const __half*>(h->dev + d.off[SEC_BPDQ_OFF]);
  a.x = static_cast<const __half*>(x);
  a.y = static_cast<__half*>(y);
  a.rd = make_reduce(h);
  a.R = d.R;
  a.C = d.C;
  a.nrb = q2_nrb(d);
  a.ntok = 1;
  return launch(h, k_bpdq_b1<kBpdqWarps, kBpdqAhead>, a, kOneCtaSmem, d.nslice * a.nrb, x, y, stream,
                kBpdqWarps * 32);
}

// BPDQ at 2..6 tokens on CUDA cores (x is [ntok][C]; partials [ntok][nslice][Rpad]).
extern "C" int q2_mt_bpdq(const q2_handle* h, const void* x, void* y, int ntok, void* stream) {
  const q2_blob_header& d = h->hdr;
  BpdqArgs a;
  a.bits = h->dev + d.off[SEC_BPDQ_BITS];
  a.c01 = reinterpret_cast<const __half2*>(h->dev + d.off[SEC_BPDQ_C01]);
  a.off = reinterpret_cast<const __half*>(h->dev + d.off[SEC_BPDQ_OFF]);
  a.x = static_cast<const __half*>(x);
  a.y = static_cast<__half*>(y);
  a.rd = make_reduce(h);
  a.R = d.R;
  a.C = d.C;
  a.nrb = q2_nrb(d);
  a.ntok = ntok;
  if (ntok < 2 || ntok > kMtMaxTok) return Q2_ENTOK;
  const int items = d.nslice * a.nrb;
  constexpr int W = 16;
  const int np = (ntok + 1) / 2;
  const int smem = std::max(kOneCtaSmem, np * kPairBytes + 64);
  switch (np) {
    case 1: return launch(h, k_bpdq_mt<W, 2, 1>, a, smem, items, x, y, stream, W * 32, ntok);
    case 2: return launch(h, k_bpdq_mt<W, 1, 2>, a, smem, items, x, y, stream, W * 32, ntok);
    case 3: return launch(h, k_bpdq_mt<W, 1, 3>, a, smem, items, x, y, stream, W * 32, ntok);
    default: return Q2_ENTOK;
  }
}

extern "C" int q2_b1_noweights(const q2_handle* h, const void* x, void* y, void* stream) {
  const q2_blob_header& d = h->hdr;
  BpdqArgs a = {};
  a.x = static_cast<const __half*>(x);
  a.y = static_cast<__half*>(y);
  a.rd = make_reduce(h);
  a.R = d.R;
  a.C = d.C;
  a.nrb = q2_nrb(d);
  a.ntok = 1;
  return launch(h, k_noweights_b1<kBpdqWarps>, a, kOneCtaSmem, d.nslice * a.nrb, x, y, stream, kBpdqWarps * 32);
}

extern "C" int q2_b1_leech(const q2_handle* h, const void* x, void* y, void* stream) {
  const q2_blob_header& d = h->hdr;
  LeechArgs a;
  a.planes = h->dev + d.off[SEC_LEECH_PLANES];
  a.parity = reinterpret_cast<const uint16_t*>(h->dev + d.off[SEC_LEECH_PARITY]);
  a.scale = reinterpret_cast<const __half*>(h->dev + d.off[SEC_LEECH_SCALE]);
  a.tail = reinterpret_cast<const __half*>(h->dev + d.off[SEC_LEECH_TAIL]);
  a.excptr = reinterpret_cast<const uint32_t*>(h->dev + d.off[SEC_LEECH_EXCPTR]);
  a.exccol = reinterpret_cast<const uint32_t*>(h->dev + d.off[SEC_LEECH_EXCCOL]);
  a.x = static_cast<const __half*>(x);
  a.y = static_cast<__half*>(y);
  a.rd = make_reduce(h);
  a.R = d.R;
  a.C = d.C;
  a.nrb = q2_nrb(d);
  a.nblock = d.nblock;
  a.tail_n = d.tail;
  a.tailpad = d.tailpad;
  a.inv_sqrt8 = d.inv_sqrt8;
  return launch(h, k_leech_b1<kLeechWarps, kLeechAhead>, a, kOneCtaSmem, d.nslice * a.nrb, x, y, stream,
                kLeechWarps * 32);
}

extern "C" int q2_b1_trellis(const q2_handle* h, const void* x, void* y, void* stream) {
  const q2_blob_header& d = h->hdr;
  TrellisArgs a;
  a.stream = h->dev + d.off[SEC_TRL_STREAM];
  a.table = reinterpret_cast<const uint32_t*>(h->dev + d.off[SEC_TRL_TABLE]);
  a.scale = reinterpret_cast<const __half*>(h->dev + d.off[SEC_TRL_SCALE]);
  a.x = static_cast<const __half*>(x);
  a.y = static_cast<__half*>(y);
  a.rd = make_reduce(h);
  a.R = d.R;
  a.C = d.C;
  a.nrb = q2_nrb(d);
  const int smem = std::max(4096 * 4 + d.C * 2, kOneCtaSmem);
  return launch(h, k_trellis_b1<kTrellisWarps, kTrellisAhead>, a, smem, d.nslice * a.nrb, x, y, stream,
                kTrellisWarps * 32);
}

// ---------------------------------------------------------------------------
// Allocation-free batch-1 BPDQ entry point.
//
// Some callers cannot allocate device memory when they call the GEMV: code
// that runs while a CUDA stream is being captured into a graph (cudaMalloc
// is not permitted there), plugins whose host framework owns all device
// memory and offers them no allocator, and real-time decode loops that must
// not touch the allocator after start-up.  q2_gemv_bpdq_noalloc serves them:
// the split-K partial sums that q2_gemv keeps in a caller-bound workspace go
// to a scratch array that belongs to this library instead, so the caller
// passes only the handle, x, y and a stream.  Every GPU that loads the
// library holds the array (Q2_NOALLOC_SCRATCH_BYTES) until the process exits.

namespace {

// Device memory for the partial sums; host code must never hand this symbol
// to a kernel (on the host it only stands in for the device address).
static __device__ __align__(256) unsigned char q2_noalloc_scratch[Q2_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
std::vector<void*> g_noalloc_ptr;   // device address of the scratch, per device

// The device address of the scratch on the current device, looked up once
// per device (cudaGetSymbolAddress with that device current).
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return Q2_ECUDA;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if ((int)g_noalloc_ptr.size() <= dev) g_noalloc_ptr.resize(dev + 1, nullptr);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, q2_noalloc_scratch) != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return Q2_ECUDA;
    }
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return Q2_OK;
}

}  // namespace

extern "C" int q2_gemv_bpdq_noalloc(const q2_handle* h, const void* x, void* y, q2_stream stream) {
  if (!h || !x || !y) return Q2_EINVAL;
  if (h->hdr.fmt != Q2_BPDQ) return Q2_EFMT;
  if (reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(y) % 16) return Q2_EALIGN;
  const size_t need = (size_t)h->hdr.nslice * h->hdr.Rpad * 4;
  if (need > (size_t)Q2_NOALLOC_SCRATCH_BYTES) return Q2_ESCRATCH;
  void* scratch = nullptr;
  const int st = noalloc_scratch(&scratch);
  if (st) return st;
  // the same two launches as q2_gemv at ntok = 1, with the scratch in place
  // of the caller's workspace; nothing in the scratch needs to start at zero
  q2_handle view = *h;
  view.ws = scratch;
  view.ws_bytes = Q2_NOALLOC_SCRATCH_BYTES;
  return q2_b1_bpdq(&view, x, y, static_cast<void*>(stream));
}
