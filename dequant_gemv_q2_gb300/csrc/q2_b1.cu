// Batch-1 kernels (ntok == 1) for the packed formats and the no-weights
// control, and BPDQ at 2..6 tokens.  One lane owns one output row; a warp
// owns 32 rows of one 256-column slice (an "item").  CTAs take contiguous,
// equal shares of the items in slice-major order, so a CTA touches one or a
// few slices; it builds the x-dependent table of each slice in shared
// memory and streams the slice's items.
//
// The split-K reduction happens inside the launch and needs no fence and no
// second pass: each lane adds its fp32 slice partial, converted to a 48-bit
// fixed-point integer (scale 2^F, F chosen per matrix so that no partial of
// any fp16 x can overflow), together with an arrival count of one, to the
// 64-bit accumulator word of its (token, row) with a single atomic.
// Integer addition is associative, so the sum is the same whatever order
// the slices arrive in (deterministic); the lane whose addition brings the
// count to the number of slices holds the complete sum in the atomic's
// return value, converts it back, applies the format's epilogue, writes y
// and resets the word to zero.  Nothing ever waits on another CTA.
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
// One 16-warp CTA per SM (grid = SM count; each CTA asks for more than half
// of the SM's shared memory).  Launches use programmatic dependent launch: a
// CTA loads its first items into registers, then waits for the previous
// kernel on the stream (griddepcontrol.wait) before it touches x, y or the
// workspace, and triggers its own dependents right after.  Measured on
// GB300: bulk L2 prefetches of the CTA's weights (or of the next GEMV's)
// issued before the wait made every shape slower, so there are none.
#include <cuda_fp16.h>

#include <cmath>
#include <mutex>
#include <vector>

#include "q2_common.cuh"

extern __shared__ __align__(1024) unsigned char q2_smem[];

namespace q2 {
namespace {

// ------------------------------------------------------------ shared state
struct B1 {
  const __half* x;              // [ntok][C]
  __half* y;                    // [ntok][R]
  unsigned long long* acc;      // [ntok][Rpad] accumulator words (zero between calls)
  float fscale, finv;           // 2^F and 2^-F of the fixed-point partials
  int R, C, Rpad, nrb, nslice, ntok;
  q2_pf pf;                     // weights of later launches to fetch into L2 (zero lengths: none)
};

// Shared memory of the single-token table kernels: a small tail at the
// start of dynamic shared memory (slice sums of x, Leech block sums, staged
// x: up to kStageBytes / (512 * ntok) slices at once), then the table of the
// current slice at the fixed shared-window address kTabAddr, so that a
// lookup's address is the byte permute's result plus an immediate offset.
constexpr int kTab = 64 * 1024;        // one slice's table (duplicated columns)
constexpr uint32_t kTabAddr = 0x2000;  // shared-window address of the table
constexpr int kTabSmem = kTabAddr + kTab;   // dynamic smem reaching kTabAddr + kTab from any window base
constexpr int kTailGsum = 0;           // float [8]
constexpr int kTailXb = 128;           // float [kStageMax][12], Leech block sums
constexpr int kTailX = 512;            // fp16 staged x [slice][tok][256]
constexpr int kStageBytes = 4096;
constexpr int kStageMax = kStageBytes / 512;
constexpr int kTailFixed = kTailX + kStageBytes;

// x of slices [g0, g0 + nt) for tokens 0..ntok-1 into smem, as fp16
// [t][tok][256] (columns past C read as zero); one 16-byte load per thread.
template <int NT>
__device__ __forceinline__ void stage_x(const B1& c, int g0, int nt, __half* xs) {
  const int per_slice = c.ntok * 32;
  for (int i = threadIdx.x; i < nt * per_slice; i += NT) {
    const int t = i / per_slice, r = i - t * per_slice;
    const int tok = r >> 5;
    const int col = (g0 + t) * Q2_SLICE + (r & 31) * 8;
    const __half* src = c.x + (size_t)tok * c.C + col;
    uint4 v;
    if (col + 8 <= c.C) {
      v = *reinterpret_cast<const uint4*>(src);
    } else {
      __half hv[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) hv[k] = (col + k < c.C) ? src[k] : __float2half_rn(0.f);
      v = *reinterpret_cast<const uint4*>(hv);
    }
    reinterpret_cast<uint4*>(xs)[i] = v;
  }
}

// Subset-sum table of one staged slice.  T[v][b] = sum of x[8b + i] over
// the set bits i of the byte v (b = 0..31), stored twice per v (columns b
// and b + 32) so a lane at rotated position P reads column P + lane without
// a modulo: byte address v*256 + lane*4 + P*4.  Each of 512 (column-byte b,
// high nibble h) tasks forms the 16 sums of its low nibble by doubling, adds
// the sum selected by h, and writes the 16 entries T[16h + l][b]
// (consecutive b across a warp: conflict-free stores).  The h = 15 warp also
// reduces the slice sum of x into *gsum.
template <int NT>
__device__ __forceinline__ void build_table(const __half* xs, float* T, float* gsum) {
  for (int e = threadIdx.x; e < 512; e += NT) {
    const int h = e >> 5, b = e & 31;
    const uint4 raw = *reinterpret_cast<const uint4*>(xs + 8 * b);
    const __half2* hv = reinterpret_cast<const __half2*>(&raw);
    float x8[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __half22float2(hv[k]);
      x8[2 * k] = f.x;
      x8[2 * k + 1] = f.y;
    }
    float hs = 0.f;                              // sum selected by the high nibble h (bits 4..7)
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

// The table of the single-token kernels, at shared address kTabAddr (the
// dynamic shared memory starts below it: the window's reserved bytes plus
// the tail).
__device__ __forceinline__ float* tab1() {
  return reinterpret_cast<float*>(q2_smem + (kTabAddr - (uint32_t)__cvta_generic_to_shared(q2_smem)));
}

// Table lookup for the byte at rotated position P (byte P & 3 of `word`).
// lane4 = lane*4, so the permute gives v*256 + lane*4 and the load adds
// kTabAddr + P*4 as its immediate offset.
template <int P>
__device__ __forceinline__ float tl(uint32_t lane4, uint32_t word) {
  const uint32_t a = __byte_perm(word, lane4, 0x5504u | ((uint32_t)(P & 3) << 4));
  float v;
  asm volatile("ld.shared.f32 %0, [%1+%2];" : "=f"(v) : "r"(a), "n"(kTabAddr + P * 4));
  return v;
}
constexpr uint32_t kLane4Hi = 0;          // nothing to OR into lane*4

// Lookup P into accumulator P mod 4, then the rest.
template <int P>
__device__ __forceinline__ void plane_steps(uint32_t lane4, const uint32_t (&w)[8], float (&s)[4]) {
  if constexpr (P < 32) {
    s[P & 3] += tl<P>(lane4, w[P >> 2]);
    plane_steps<P + 1>(lane4, w, s);
  }
}

// Sum of the table entries selected by 32 rotated bytes (two uint4 chunks),
// in four independent fp32 accumulators.
__device__ __forceinline__ float plane_sum(uint32_t lane4, const uint4& c0, const uint4& c1) {
  const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  float s[4] = {0.f, 0.f, 0.f, 0.f};
  plane_steps<0>(lane4, w, s);
  return (s[0] + s[1]) + (s[2] + s[3]);
}

// Lookup P of both planes into pair accumulator P mod 4, then the rest.
template <int P>
__device__ __forceinline__ void pair_steps(uint32_t lane4, const uint32_t (&w0)[8], const uint32_t (&w1)[8],
                                           float2 (&s)[4]) {
  if constexpr (P < 32) {
    s[P & 3] = __fadd2_rn(s[P & 3], make_float2(tl<P>(lane4, w0[P >> 2]), tl<P>(lane4, w1[P >> 2])));
    pair_steps<P + 1>(lane4, w0, w1, s);
  }
}

// (sum of plane 0's 32 lookups, sum of plane 1's)
__device__ __forceinline__ float2 planes_sum(uint32_t lane4, const uint4& a0, const uint4& a1, const uint4& b0,
                                             const uint4& b1) {
  const uint32_t w0[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  const uint32_t w1[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
  float2 s[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  pair_steps<0>(lane4, w0, w1, s);
  return __fadd2_rn(__fadd2_rn(s[0], s[1]), __fadd2_rn(s[2], s[3]));
}

// Atomics a lane has issued for one item (NT tokens), settled one item later
// so the atomic's round trip overlaps the next item's work.
template <int NT>
struct Pending {
  unsigned long long old[NT], add[NT];
  int row = -1;
};

template <int NT>
__device__ __forceinline__ void acc_issue(Pending<NT>& pd, const B1& c, int row, const float (&p)[NT]) {
#pragma unroll
  for (int t = 0; t < NT; ++t)
    if (t < c.ntok) {
      unsigned long long* word = c.acc + (size_t)t * c.Rpad + row;
      pd.add[t] = fx_prepare(word, p[t], c.fscale);
      pd.old[t] = atomicAdd(word, pd.add[t]);
    }
  pd.row = row;
}

template <int NT, class F>
__device__ __forceinline__ void acc_settle(Pending<NT>& pd, const B1& c, const F& f) {
  if (pd.row < 0) return;
#pragma unroll
  for (int t = 0; t < NT; ++t)
    if (t < c.ntok) {
      const unsigned long long w = pd.old[t] + pd.add[t];
      if ((int)(w >> 56) == c.nslice) {                // this lane completed the row
        if (pd.row < c.R) f.finish(t, pd.row, fx_value(w, c.nslice, c.finv));   // NaN stays NaN
        c.acc[(size_t)t * c.Rpad + pd.row] = 0ull;
      }
    }
  pd.row = -1;
}

// ------------------------------------------------------- work split
// The CTA's contiguous range [i0, i1) of items in slice-major order: equal
// shares of all items (the Leech and trellis kernels).  A share that crosses
// a slice boundary builds a second table; their items are heavy enough that
// balancing the counts pays more (measured on GB300).  The BPDQ kernels
// split by slice instead (make_lean).
__device__ __forceinline__ void b1_range(const B1& c, int& i0, int& i1) {
  cta_range(c.nslice * c.nrb, i0, i1);
}

// This CTA's 1/grid share of each range in c.pf, fetched into L2 by one
// thread with bulk prefetches: the weights of the launches that follow
// stream from HBM while this launch and its successors run their
// latency-bound prologues and reductions.
__device__ __forceinline__ void prefetch_next(const q2_pf& pf) {
  const unsigned long long G = gridDim.x, b = blockIdx.x;
#pragma unroll
  for (int r = 0; r < Q2_PF_SLOTS; ++r) {
    const unsigned long long n16 = pf.len[r] >> 4;        // whole 16-byte units
    if (!n16) continue;
    const unsigned long long u0 = n16 * b / G, u1 = n16 * (b + 1) / G;
    if (u1 > u0) prefetch_l2(pf.ptr[r] + u0 * 16, (size_t)(u1 - u0) * 16);
  }
}

// ------------------------------------------------------- pipelined items
// run_b1 drives every split-K kernel.  The CTA's item range (b1_range) is
// cut into groups: one slice per group for the table kernels (F::kGroup ==
// 1), one group for everything in the trellis kernel.  x is staged into
// shared memory for up to kStageMax / ntok slices at a time (F::kStaged);
// per group the CTA builds the slice's table (F::tables) and streams the
// group's items: item j0 + warp + k*W goes to warp `warp`, which keeps AHEAD
// items beyond the one it is summing in flight in registers (F::load).  The
// first group's loads are issued before the CTA waits on the previous
// kernel (weights do not depend on it).  F::compute sums one item into a
// partial per token, which the lane adds to the row's accumulator word.
template <int W, int AHEAD, class F>
__device__ __forceinline__ void run_b1(F& f, const B1& c, unsigned char* tail) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int i0, i1;
  b1_range(c, i0, i1);
  const int glast = (i1 - 1) / c.nrb;
  __half* xs = reinterpret_cast<__half*>(tail + kTailX);
  const int stage_n = max(1, kStageMax / c.ntok);
  int sg0 = 0, sgn = 0;                          // staged slices [sg0, sg0 + sgn)
  bool waited = false;
  Pending<F::kTok> pd;
  for (int j0 = i0; j0 < i1;) {
    const int gA = j0 / c.nrb;
    const int gB = min(glast, gA + F::kGroup - 1);
    const int j1 = min(i1, (gB + 1) * c.nrb);
    typename F::Item buf[AHEAD + 1];
    const int it0 = j0 + warp;
    // the slice of an item: gA for one-slice groups, else a division
    auto slice_of = [&](int it) { return F::kGroup == 1 ? gA : it / c.nrb; };
#pragma unroll
    for (int d = 0; d < AHEAD; ++d)
      if (it0 + d * W < j1) f.load(it0 + d * W, slice_of(it0 + d * W), lane, buf[d]);
    if (!waited) {
      if (threadIdx.x == 0) prefetch_next(c.pf);
      pdl_wait();
      pdl_trigger();
      waited = true;
    } else {
      __syncthreads();                           // the previous group's table is no longer read
    }
    if (F::kStaged && gA >= sg0 + sgn) {
      sg0 = gA;
      sgn = min(stage_n, glast - gA + 1);
      stage_x<W * 32>(c, sg0, sgn, xs);
      f.stage_extra(sg0, sgn, tail);
      __syncthreads();
    }
    f.tables(gA, xs + (size_t)(gA - sg0) * c.ntok * Q2_SLICE, tail);
    __syncthreads();
    // the AHEAD + 1 buffers are indexed statically: AHEAD + 1 items per trip
    for (int base = it0; base < j1; base += (AHEAD + 1) * W) {
#pragma unroll
      for (int u = 0; u <= AHEAD; ++u) {
        const int it = base + u * W;
        if (it < j1) {
          const int nx = it + AHEAD * W;
          if (nx < j1) f.load(nx, slice_of(nx), lane, buf[(u + AHEAD) % (AHEAD + 1)]);
          const int g = slice_of(it);
          float p[F::kTok];
          f.compute(it, g, lane, buf[u], p);
          acc_settle(pd, c, f);
          acc_issue(pd, c, (it - g * c.nrb) * 32 + lane, p);
        }
      }
    }
    j0 = j1;
  }
  if (!waited) {
    if (threadIdx.x == 0) prefetch_next(c.pf);
    pdl_wait();
    pdl_trigger();
  }
  acc_settle(pd, c, f);
}

__device__ __forceinline__ void ld_item(const unsigned char* base, int item_bytes, int it, int lane, uint4* w,
                                        int n) {
  const unsigned char* p = base + (size_t)it * item_bytes + lane * 16;
  for (int k = 0; k < n; ++k) w[k] = ldg_stream(p + k * 512);
}

// Launch shape of the generic (run_b1) kernels, Leech and trellis: one CTA
// per SM (16 warps for Leech, 24 for the trellis), one item ahead per warp
// in registers (measured: 2 ahead is slower).
constexpr int kMinBlocks = 1;
#ifndef Q2_LEECH_AHEAD
#define Q2_LEECH_AHEAD 1
#endif
constexpr int kLeechAhead = Q2_LEECH_AHEAD;   // items a warp holds in registers beyond the one it sums
#ifndef Q2_LEECH_W
#define Q2_LEECH_W 16
#endif
constexpr int kLeechWarps = Q2_LEECH_W;   // warps per CTA of the Leech kernel

// ------------------------------------------------------------------ Leech
struct LeechArgs {
  B1 c;
  const unsigned char* planes;
  const uint16_t* parity;     // [nslice][Rpad]
  const __half* scale;        // [Rpad]
  const __half* tail;         // [Rpad][tailpad]
  const uint32_t* excptr;     // [Rpad + 1]
  const uint32_t* exccol;
  int nblock, tail_n, tailpad;
  float inv_sqrt8;
};

// Blocks of 24 columns whose first column lies in slice g.
__device__ __forceinline__ void leech_blocks(int g, int nblock, int& bfirst, int& nbk) {
  bfirst = (g * Q2_SLICE + 23) / 24;
  const int blast = min(nblock - 1, (g * Q2_SLICE + Q2_SLICE + 23) / 24 - 1);
  nbk = max(0, blast - bfirst + 1);
}

// Two layouts (q2_pack_leech).  NP = 3: the planes hold the two's-complement
// bits of u = (v - p)/2 per weight (p = the block's parity bit), so
// v = p + 2*b0 + 4*b1 - 8*b2: three subset sums plus, per 24-column block
// starting in the slice, the block sum of x when the row's parity bit for
// the block is set; the epilogue adds 16 x[col] for each v = +8 exception.
// NP = 4: the planes hold the offset-binary code c = (v - p)/2 + 4, so
// v = p - 8 + 2*b0 + 4*b1 + 8*b2 + 16*b3 (and every column outside the
// blocks holds c = 4): four subset sums, the parity term and -8 times the
// slice's sum of x (no exceptions); plane 3 is set only
// where v = +8, so its lookups are skipped when no lane of the warp has a
// bit in it.  Then x scale_r / sqrt(8) and the fp16 tail ("Tetra", section
// 5.1: the row scale after the block dot product, then the unquantised
// tail).
template <int NT, int NP>
struct LeechF {
  struct Item {
    uint4 w[2 * NP];
    uint32_t pw;         // parity bits of the slice's blocks for this row
  };
  static constexpr bool kStaged = true;
  static constexpr int kGroup = 1;
  static constexpr int kTok = 1;
  static constexpr int kItemBytes = NP == 4 ? Q2_ITEM_BYTES_LEECH4 : Q2_ITEM_BYTES_LEECH;
  const LeechArgs& a;
  int sg0 = 0;           // first staged slice (block sums in the tail are per staged slice)
  __device__ void load(int it, int g, int lane, Item& b) const {
    ld_item(a.planes, kItemBytes, it, lane, b.w, 2 * NP);
    b.pw = __ldg(a.parity + (size_t)g * a.c.Rpad + (size_t)(it - g * a.c.nrb) * 32 + lane);
  }
  // block sums of x for the blocks that start in each staged slice (<= 11
  // each; a block may run into the next slice, so they are read from x)
  __device__ void stage_extra(int s0, int sn, unsigned char* tail) {
    sg0 = s0;
    float* xb = reinterpret_cast<float*>(tail + kTailXb);
    for (int i = threadIdx.x; i < sn * 12; i += NT) {
      const int t = i / 12, j = i - t * 12;
      int bfirst, nbk;
      leech_blocks(s0 + t, a.nblock, bfirst, nbk);
      if (j < nbk) {
        const __half* xp = a.c.x + (size_t)(bfirst + j) * 24;
        float v = 0.f;
#pragma unroll
        for (int k = 0; k < 24; ++k) v += __half2float(xp[k]);
        xb[i] = v;
      }
    }
  }
  __device__ void tables(int, const __half* xs, unsigned char* tail) const {
    build_table<NT>(xs, tab1(), reinterpret_cast<float*>(tail + kTailGsum));
  }
  __device__ void compute(int, int g, int lane, const Item& b, float (&p)[1]) const {
    const uint32_t lane4 = (uint32_t)lane * 4u | kLane4Hi;
    const float2 P01 = planes_sum(lane4, b.w[0], b.w[1], b.w[2], b.w[3]);   // same sums as plane_sum, paired
    const float P0 = P01.x, P1 = P01.y;
    const float P2 = plane_sum(lane4, b.w[4], b.w[5]);
    int bfirst, nbk;
    leech_blocks(g, a.nblock, bfirst, nbk);
    const float* xb = reinterpret_cast<const float*>(q2_smem + kTailXb) + (g - sg0) * 12;
    float pacc = 0.f;
    for (int j = 0; j < nbk; ++j) pacc += ((b.pw >> j) & 1u) ? xb[j] : 0.f;
    // + 0 x (sum of the slice's x): the subset sums skip zero weights, but in
    // IEEE arithmetic 0 x inf is NaN, so an inf or NaN anywhere in the slice
    // must still make the partial non-finite
    const float gs = *reinterpret_cast<const float*>(q2_smem + kTailGsum);
    if constexpr (NP == 3) {
      p[0] = fmaf(0.f, gs, fmaf(2.f, P0, fmaf(4.f, P1, fmaf(-8.f, P2, pacc))));
    } else {
      const uint4 h0 = b.w[6], h1 = b.w[7];
      const bool any3 = __any_sync(0xffffffffu, (h0.x | h0.y | h0.z | h0.w | h1.x | h1.y | h1.z | h1.w) != 0u);
      const float P3 = any3 ? plane_sum(lane4, h0, h1) : 0.f;
      // every column of the slice carries the -8 offset (columns outside the
      // blocks hold code 4, so theirs cancels): -8 x (the slice's sum of x)
      p[0] = fmaf(2.f, P0, fmaf(4.f, P1, fmaf(8.f, P2, fmaf(16.f, P3, fmaf(-8.f, gs, pacc)))));
    }
  }
  __device__ void finish(int tok, int row, float v) const {
    const __half* xt = a.c.x + (size_t)tok * a.c.C;
    for (uint32_t e = a.excptr[row]; e < a.excptr[row + 1]; ++e) v = fmaf(16.f, __half2float(xt[a.exccol[e]]), v);
    v *= __half2float(a.scale[row]) * a.inv_sqrt8;
    const int col0 = a.nblock * 24;
    for (int j = 0; j < a.tail_n; ++j)
      v = fmaf(__half2float(a.tail[(size_t)row * a.tailpad + j]), __half2float(xt[col0 + j]), v);
    a.c.y[(size_t)tok * a.c.R + row] = __float2half_rn(v);
  }
};

// The tail sits at the start of dynamic shared memory for every
// single-token table kernel.
__device__ __forceinline__ unsigned char* tail1() { return q2_smem; }

template <int W, int AHEAD, int NP>
__global__ void __launch_bounds__(W * 32, 1) k_leech_b1(LeechArgs a) {
  if ((uint32_t)__cvta_generic_to_shared(q2_smem) + kTailFixed > kTabAddr) return;   // layout needs a low window base
  LeechF<W * 32, NP> f{a};
  run_b1<W, AHEAD>(f, a.c, tail1());
}

// ------------------------------------------------ BPDQ, one token (lean)
// The single-token BPDQ GEMV and its no-weights control.  Same work unit,
// tables and reduction as run_b1, but written for the fewest instructions
// per item, because at one token the item loop is bound by issue and
// shared-memory throughput rather than by HBM (measured on GB300: a
// 24576x4096 GEMV whose weights are all in L2 is no faster than one
// reading them from HBM):
//   - the CTA's item range comes from the host in the parameter block
//     (a slice-aligned split, make_lean), so no warp spends its prologue on
//     integer divisions;
//   - each warp walks its items with pointers advanced by a constant
//     stride instead of recomputing 64-bit addresses per item;
//   - the lookups of plane 0 and plane 1 at the same rotated position are
//     added as one packed fp32 pair, into four pair accumulators (lookup P
//     into accumulator P mod 4, then (s0 + s1) + (s2 + s3)): per plane the
//     same operations in the same order as plane_sum, so the result is
//     bit-identical to run_b1's and to the token-pair kernel's;
//   - x is read straight from global memory by the table build (16 tasks
//     share each 16-byte load), without a staging pass.
constexpr int kLeanMaxGrid = 192;
// Launch shape (build-time tunables): 24 warps in one CTA per SM, 80
// registers.  Measured on the Qwen3-8B stack (us per step): 16 warps 698,
// 20 warps 689, 24 warps 659, 28 warps 740, 32 warps 781 (spills); two CTAs
// per SM, so that the next GEMV's CTAs are resident early: 8 warps 921,
// 12 warps 808, 16 warps 898 (fewer registers, less in flight).
#ifndef Q2_LEAN_W
#define Q2_LEAN_W 24
#endif
#ifndef Q2_LEAN_MB
#define Q2_LEAN_MB 1
#endif
constexpr int kLeanW = Q2_LEAN_W;        // warps per CTA
constexpr int kLeanMinBlocks = Q2_LEAN_MB;

struct LeanArgs {
  const __half* x;              // [C]
  __half* y;                    // [R]
  unsigned long long* acc;      // [Rpad] accumulator words (zero between calls)
  const uint4* bits;            // item-major planes (see q2_layout.h)
  const uint32_t* c01;          // [nslice][Rpad] c0 | c1 << 16 (fp16)
  const unsigned short* off;    // [nslice][Rpad] fp16
  float fscale, finv;
  int R, C, Rpad, nrb, nslice;
  q2_pf pf;
  uint32_t pfq, pfr;            // slot 0 of pf in 16-byte units over grid x W warps: quotient, remainder
  uint32_t start[kLeanMaxGrid + 1];   // CTA b owns items [start[b], start[b+1])
};

struct LeanItem {
  uint4 w[4];            // plane 0: w[0], w[1]; plane 1: w[2], w[3]
  uint32_t c01;
  unsigned short off;
};

template <bool kWeights>
__device__ __forceinline__ void lean_load(const uint32_t* c01, const unsigned short* off, const uint4* wp, size_t ci,
                                          int it, int lane, LeanItem& b) {
  if constexpr (kWeights) {
#pragma unroll
    for (int k = 0; k < 4; ++k) b.w[k] = ldg_stream(wp + k * 32);
    b.c01 = __ldg(c01 + ci);
    b.off = __ldg(off + ci);
  } else {
    // the no-weights control: "weights" derived from the item and lane
    const uint32_t h = (uint32_t)it * 0x9E3779B9u ^ ((uint32_t)lane * 0x85EBCA6Bu);
    b.w[0] = make_uint4(h, h ^ 0x5bd1e995u, h * 3u, h * 5u);
    b.w[1] = make_uint4(h * 7u, h ^ 0x27d4eb2fu, h * 11u, h * 13u);
    b.w[2] = b.w[1];
    b.w[3] = b.w[0];
    b.c01 = 0x211F251Fu;      // fp16 (0.02, 0.01)
    b.off = 0x211Fu;          // fp16 0.01
  }
}

__device__ __forceinline__ float lean_partial(uint32_t lane4, const LeanItem& b, float gs) {
  const float2 S = planes_sum(lane4, b.w[0], b.w[1], b.w[2], b.w[3]);
  const float2 cf = __half22float2(*reinterpret_cast<const __half2*>(&b.c01));
  const float of = __half2float(__ushort_as_half(b.off));
  return fmaf(cf.x, S.x, fmaf(cf.y, S.y, of * gs));
}

// The weights of a later GEMV (c.pf slot 0), fetched into L2 a piece per
// item: warp w of CTA b owns 1/(grid*W) of the range and issues it in as
// many pieces as it has items, one after each item's own loads, so the
// extra HBM traffic is spread over the GEMV instead of queueing ahead of
// its loads in one burst (a burst at launch start made every GEMV of a
// stack slower on GB300).  Other slots, and warps without items, issue
// their share at once.
struct PacedPf {
  const unsigned char* cur;
  uint32_t left, piece;
  __device__ __forceinline__ void step(int lane) {
    if (left) {
      const uint32_t n = left < piece ? left : piece;
      if (lane == 0) asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(cur), "r"(n) : "memory");
      cur += n;
      left -= n;
    }
  }
};

// Warp k = b*W + w of the grid gets 16-byte units [k*q + min(k, r), ...) of
// slot 0, q and r being the quotient and remainder of its units over all
// warps (computed on the host).
__device__ __forceinline__ PacedPf paced_share(const q2_pf& pf, uint32_t q, uint32_t r, int warp, int W, int nitems) {
  PacedPf p;
  const uint32_t k = blockIdx.x * (uint32_t)W + (uint32_t)warp;
  const uint32_t u0 = k * q + min(k, r), n = q + (k < r ? 1u : 0u);
  p.cur = pf.ptr[0] + (size_t)u0 * 16;
  p.left = n * 16;
  const uint32_t m = nitems > 0 ? (uint32_t)nitems : 1u;
  p.piece = p.left ? min(65536u, ((p.left + m - 1) / m + 15) / 16 * 16) : 0u;
  return p;
}

struct LeanPending {
  unsigned long long old, add;
  unsigned long long* p;
  int row;               // -1: nothing pending
};

__device__ __forceinline__ void lean_settle(LeanPending& pd, const LeanArgs& a) {
  if (pd.row < 0) return;
  const unsigned long long w = pd.old + pd.add;
  if ((int)(w >> 56) == a.nslice) {                   // this lane completed the row
    if (pd.row < a.R) a.y[pd.row] = __float2half_rn(fx_value(w, a.nslice, a.finv));
    *pd.p = 0ull;
  }
  pd.row = -1;
}

template <int W, bool kWeights, bool kPaced>
__global__ void __launch_bounds__(W * 32, kLeanMinBlocks) k_bpdq1(const __grid_constant__ LeanArgs a) {
  if ((uint32_t)__cvta_generic_to_shared(q2_smem) + kTailFixed > kTabAddr) return;   // layout needs a low window base
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t lane4 = (uint32_t)lane * 4u;
  const int i0 = (int)a.start[blockIdx.x], i1 = (int)a.start[blockIdx.x + 1];
  float* gsum = reinterpret_cast<float*>(q2_smem + kTailGsum);
  LeanPending pd;
  pd.row = -1;
  bool waited = false;
  PacedPf pp;
  pp.left = 0;
  if constexpr (kPaced) pp = paced_share(a.pf, a.pfq, a.pfr, warp, W, (i1 - i0 - warp + W - 1) / W);
  int g = i0 / a.nrb;
  for (int j0 = i0; j0 < i1; ++g) {
    const int j1 = min(i1, (g + 1) * a.nrb);
    int it = j0 + warp;
    const int rb = it - g * a.nrb;
    const uint4* wp = a.bits + (size_t)it * (Q2_ITEM_BYTES_BPDQ / 16) + lane;
    size_t ci = (size_t)g * a.Rpad + (size_t)rb * 32 + lane;
    unsigned long long* ap = a.acc + (size_t)rb * 32 + lane;
    int row = rb * 32 + lane;
    LeanItem b0, b1;
    if (it < j1) lean_load<kWeights>(a.c01, a.off, wp, ci, it, lane, b0);
    if (!waited) {
      if (threadIdx.x == 0) {                           // slots past the first: at once
        q2_pf rest = a.pf;
        rest.len[0] = 0;
        prefetch_next(rest);
      }
      if (kPaced && it >= j1) pp.step(lane);            // no items: the whole share now
      pdl_wait();
      pdl_trigger();
      waited = true;
    } else {
      __syncthreads();                                  // the previous slice's table is no longer read
    }
    q2::build_table<W * 32>(a.x + (size_t)g * Q2_SLICE, a.C - g * Q2_SLICE, tab1(), gsum);
    __syncthreads();
    const float gs = *gsum;
    constexpr int kStrideW = W * (Q2_ITEM_BYTES_BPDQ / 16);
    // two items per trip so the two buffers are named statically
    for (; it < j1; it += 2 * W) {
      const bool m1 = it + W < j1;
      if (m1) lean_load<kWeights>(a.c01, a.off, wp + kStrideW, ci + W * 32, it + W, lane, b1);
      if constexpr (kPaced) pp.step(lane);
      float p = lean_partial(lane4, b0, gs);
      lean_settle(pd, a);
      pd.add = fx_prepare(ap, p, a.fscale);
      pd.old = atomicAdd(ap, pd.add);
      pd.p = ap;
      pd.row = row;
      if (!m1) break;
      const bool m2 = it + 2 * W < j1;
      if (m2) lean_load<kWeights>(a.c01, a.off, wp + 2 * kStrideW, ci + 2 * W * 32, it + 2 * W, lane, b0);
      if constexpr (kPaced) pp.step(lane);
      p = lean_partial(lane4, b1, gs);
      lean_settle(pd, a);
      pd.add = fx_prepare(ap + W * 32, p, a.fscale);
      pd.old = atomicAdd(ap + W * 32, pd.add);
      pd.p = ap + W * 32;
      pd.row = row + W * 32;
      wp += 2 * kStrideW;
      ci += 2 * W * 32;
      ap += 2 * W * 32;
      row += 2 * W * 32;
    }
    j0 = j1;
  }
  if (!waited) {
    if (threadIdx.x == 0) prefetch_next(a.pf);
    pdl_wait();
    pdl_trigger();
  }
  pp.left = 0;
  lean_settle(pd, a);
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
// The CTA holds one slice's tables at a time (groups of one slice).
constexpr int kMtMaxTok = 6;
constexpr int kPairBytes = 256 * 32 * 8;                   // 64 KiB per token pair

// ------------------------------------------------ BPDQ, token pairs (lean)
// NP token-pair tables per slice (64 KiB each): for the pair (2p, 2p+1)
//   E_p[v][b] = (sum of x_2p over the set bits of byte v at column-byte b,
//                the same for x_2p+1)
// at byte offset p*64 KiB + v*256 + b*8, with no duplicated columns: a lane
// at rotated position P reads column-byte b = (P + lane) mod 32, whose
// address byte b*8 it keeps in one of 11 lane-constant registers (three
// positions each), so one byte permute still forms v*256 + b*8; each lookup
// is one 8-byte load and one packed fp32 add per pair, and a half-warp's 16
// lanes read 16 different column-bytes (conflict-free).  The item loop is
// k_bpdq1's (host-computed CTA ranges, pointer-walked items, atomics settled
// one item later).  Per token the lookups, sums and epilogue are those of
// k_bpdq1 in the same order (lookup P into accumulator P mod 4, then
// (s0 + s1) + (s2 + s3)), so every token's output is bit-identical to the
// same token run alone (batch invariance).
struct LeanMArgs {
  const __half* x;              // [ntok][C]
  __half* y;                    // [ntok][R]
  unsigned long long* acc;      // [ntok][Rpad] accumulator words (zero between calls)
  const uint4* bits;
  const uint32_t* c01;
  const unsigned short* off;
  float fscale, finv;
  int R, C, Rpad, nrb, nslice, ntok;
  q2_pf pf;
  uint32_t start[kLeanMaxGrid + 1];
};

// The pair tables of slice g straight from global x (16 tasks share each
// 16-byte load); per token the same sums in the same order as build_table.
template <int NT, int NP>
__device__ __forceinline__ void build_pairs_g(const __half* __restrict__ x, int C, int ntok, int g, float* T,
                                              float* gsum) {
  for (int e = threadIdx.x; e < 512 * NP; e += NT) {
    const int p = e >> 9, h = (e >> 5) & 15, b = e & 31;
    const size_t col = (size_t)g * Q2_SLICE + 8 * b;
    float xa[8], xb[8];
    {
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(2 * p) * C + col));
      const __half2* hv = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __half22float2(hv[k]);
        xa[2 * k] = f.x;
        xa[2 * k + 1] = f.y;
      }
    }
    if (2 * p + 1 < ntok) {                            // an odd count leaves the last pair half empty
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(2 * p + 1) * C + col));
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
    float2 hs = make_float2(0.f, 0.f);
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
    float2* colp = reinterpret_cast<float2*>(reinterpret_cast<char*>(T) + p * kPairBytes) + (h * 16) * 32 + b;
#pragma unroll
    for (int n = 0; n < 16; ++n) colp[n * 32] = sv[n];
    if (h == 15) {
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

template <int NP>
__device__ __forceinline__ void pair_plane(const uint32_t (&rot)[11], const uint4& c0, const uint4& c1,
                                           float2 (&S)[NP]) {
  const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const char* base = reinterpret_cast<const char*>(q2_smem);
  float2 acc[NP][4];
#pragma unroll
  for (int p = 0; p < NP; ++p)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[p][k] = make_float2(0.f, 0.f);
#pragma unroll
  for (int P = 0; P < 32; ++P) {
    const uint32_t sel = (4u + (uint32_t)(P % 3)) | ((uint32_t)(P & 3) << 4) | 0x7700u;
    const uint32_t ad = __byte_perm(w[P >> 2], rot[P / 3], sel);
#pragma unroll
    for (int p = 0; p < NP; ++p)
      acc[p][P & 3] = __fadd2_rn(acc[p][P & 3], *reinterpret_cast<const float2*>(base + p * kPairBytes + ad));
  }
#pragma unroll
  for (int p = 0; p < NP; ++p) S[p] = __fadd2_rn(__fadd2_rn(acc[p][0], acc[p][1]), __fadd2_rn(acc[p][2], acc[p][3]));
}

template <int NP>
struct LeanMPending {
  unsigned long long old[2 * NP], add[2 * NP];
  unsigned long long* p;    // token 0's word of the row
  int row;                  // -1: nothing pending
};

template <int NP>
__device__ __forceinline__ void leanm_settle(LeanMPending<NP>& pd, const LeanMArgs& a) {
  if (pd.row < 0) return;
#pragma unroll
  for (int t = 0; t < 2 * NP; ++t)
    if (t < a.ntok) {
      const unsigned long long w = pd.old[t] + pd.add[t];
      if ((int)(w >> 56) == a.nslice) {
        if (pd.row < a.R) a.y[(size_t)t * a.R + pd.row] = __float2half_rn(fx_value(w, a.nslice, a.finv));
        pd.p[(size_t)t * a.Rpad] = 0ull;
      }
    }
  pd.row = -1;
}

template <int NP>
__device__ __forceinline__ void leanm_issue(LeanMPending<NP>& pd, const LeanMArgs& a, unsigned long long* ap, int row,
                                            const float (&p)[2 * NP]) {
#pragma unroll
  for (int t = 0; t < 2 * NP; ++t)
    if (t < a.ntok) {
      unsigned long long* word = ap + (size_t)t * a.Rpad;
      pd.add[t] = fx_prepare(word, p[t], a.fscale);
      pd.old[t] = atomicAdd(word, pd.add[t]);
    }
  pd.p = ap;
  pd.row = row;
}

template <int NP>
__device__ __forceinline__ void leanm_partials(const uint32_t (&rot)[11], const LeanItem& b, const float* gsum,
                                               float (&p)[2 * NP]) {
  float2 S0[NP], S1[NP];
  pair_plane<NP>(rot, b.w[0], b.w[1], S0);
  pair_plane<NP>(rot, b.w[2], b.w[3], S1);
  const float2 cf = __half22float2(*reinterpret_cast<const __half2*>(&b.c01));
  const float of = __half2float(__ushort_as_half(b.off));
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    p[2 * q] = fmaf(cf.x, S0[q].x, fmaf(cf.y, S1[q].x, of * gsum[2 * q]));
    p[2 * q + 1] = fmaf(cf.x, S0[q].y, fmaf(cf.y, S1[q].y, of * gsum[2 * q + 1]));
  }
}

template <int W, int NP>
__global__ void __launch_bounds__(W * 32, 1) k_bpdqm(const __grid_constant__ LeanMArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t rot[11];      // byte j of rot[k]: ((3k + j + lane) mod 32) * 8; byte 3 = 0
#pragma unroll
  for (int k = 0; k < 11; ++k) {
    uint32_t r = 0;
#pragma unroll
    for (int j = 0; j < 3; ++j) r |= (uint32_t)(((3 * k + j + lane) & 31) * 8) << (8 * j);
    rot[k] = r;
  }
  const int i0 = (int)a.start[blockIdx.x], i1 = (int)a.start[blockIdx.x + 1];
  float* gsum = reinterpret_cast<float*>(q2_smem + (size_t)NP * kPairBytes + kTailGsum);
  LeanMPending<NP> pd;
  pd.row = -1;
  bool waited = false;
  int g = i0 / a.nrb;
  for (int j0 = i0; j0 < i1; ++g) {
    const int j1 = min(i1, (g + 1) * a.nrb);
    int it = j0 + warp;
    const int rb = it - g * a.nrb;
    const uint4* wp = a.bits + (size_t)it * (Q2_ITEM_BYTES_BPDQ / 16) + lane;
    size_t ci = (size_t)g * a.Rpad + (size_t)rb * 32 + lane;
    unsigned long long* ap = a.acc + (size_t)rb * 32 + lane;
    int row = rb * 32 + lane;
    LeanItem b0, b1;
    if (it < j1) lean_load<true>(a.c01, a.off, wp, ci, it, lane, b0);
    if (!waited) {
      if (threadIdx.x == 0) prefetch_next(a.pf);
      pdl_wait();
      pdl_trigger();
      waited = true;
    } else {
      __syncthreads();                                  // the previous slice's tables are no longer read
    }
    build_pairs_g<W * 32, NP>(a.x, a.C, a.ntok, g, reinterpret_cast<float*>(q2_smem), gsum);
    __syncthreads();
    float gs[2 * NP];
#pragma unroll
    for (int t = 0; t < 2 * NP; ++t) gs[t] = gsum[t];
    constexpr int kStrideW = W * (Q2_ITEM_BYTES_BPDQ / 16);
    for (; it < j1; it += 2 * W) {
      const bool m1 = it + W < j1;
      if (m1) lean_load<true>(a.c01, a.off, wp + kStrideW, ci + W * 32, it + W, lane, b1);
      float p[2 * NP];
      leanm_partials<NP>(rot, b0, gs, p);
      leanm_settle<NP>(pd, a);
      leanm_issue<NP>(pd, a, ap, row, p);
      if (!m1) break;
      const bool m2 = it + 2 * W < j1;
      if (m2) lean_load<true>(a.c01, a.off, wp + 2 * kStrideW, ci + 2 * W * 32, it + 2 * W,
                              lane, b0);
      leanm_partials<NP>(rot, b1, gs, p);
      leanm_settle<NP>(pd, a);
      leanm_issue<NP>(pd, a, ap + W * 32, row + W * 32, p);
      wp += 2 * kStrideW;
      ci += 2 * W * 32;
      ap += 2 * W * 32;
      row += 2 * W * 32;
    }
    j0 = j1;
  }
  if (!waited) {
    if (threadIdx.x == 0) prefetch_next(a.pf);
    pdl_wait();
    pdl_trigger();
  }
  leanm_settle<NP>(pd, a);
}

// ---------------------------------------------------------------- trellis
// Lane = row, item = (segment, 32 rows).  The codebook and all of x sit in
// shared memory for the whole kernel (one group spanning every segment).
// Step k of a segment reads the 16-bit state at bit offset 4*(127 - k) of
// the lane's 512-bit packet (a funnel shift of two words), hashes it, loads
// one fp16 pair, flips both signs by state bit 0 and accumulates two fp32
// FMAs.  The epilogue multiplies by the row scale.
//
// The codebook row of a step is effectively random per lane, so 32 lanes
// loading one word each from a single 16 KiB table land about 3.5 to a bank
// at worst (the expected maximum of 32 uniform draws over 32 banks), and the
// warp's load replays that often.  The table is therefore stored K times,
// interleaved: copy c of entry i is word i*K + c, so copy c lives in banks
// c, c + K, c + 2K, ..., and lane l reads copy l % K.  A warp's 32 loads then
// split into K independent groups of 32/K lanes over 32/K banks each: the
// expected worst bank load is 2.1 at K = 8 (four lanes over four banks), 2.5
// at K = 4, against 3.5 at K = 1.  The byte address of entry i is
// i * 4K + 4c: a shift and a masked OR of the hashed state, as cheap as the
// single table's.
struct TrellisArgs {
  B1 c;
  const unsigned char* stream;
  const uint32_t* table;     // 4096 half2
  const __half* scale;
};

constexpr uint32_t kHashHi = 0x9E37u << 16;   // (s*0x9E37 mod 2^16) lands in bits 16..31

template <int K>
constexpr int trl_table_bytes() { return 4096 * 4 * K; }

template <int NT, int K>
struct TrellisF {
  struct Item {
    uint4 w[4];
  };
  static constexpr bool kStaged = false;
  static constexpr int kGroup = 1 << 30;   // one group: x and the table stay for every segment
  static constexpr int kTok = 1;
  static constexpr int kLog4K = K == 8 ? 5 : K == 4 ? 4 : 2;   // log2(4K)
  const TrellisArgs& a;
  const unsigned char* tab;   // K interleaved copies of the codebook
  uint32_t* xs;
  uint32_t c4;                // 4 * (this lane's copy)
  __device__ void load(int it, int, int lane, Item& b) const { ld_item(a.stream, Q2_ITEM_BYTES_TRL, it, lane, b.w, 4); }
  __device__ void stage_extra(int, int, unsigned char*) {}
  __device__ void tables(int, const __half*, unsigned char*) const {
    const uint32_t* xg = reinterpret_cast<const uint32_t*>(a.c.x);
    for (int i = threadIdx.x; i < a.c.C / 2; i += NT) xs[i] = xg[i];
  }
  __device__ void compute(int, int sg, int, const Item& b, float (&p)[1]) const {
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
        // byte address of copy c4/4 of entry h >> 20: (h >> 20) * 4K + c4
        const uint32_t off = ((h >> (20 - kLog4K)) & (0xFFFu << kLog4K)) | c4;
        uint32_t e = *reinterpret_cast<const uint32_t*>(tab + off);
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
    p[0] = acc0 + acc1;
  }
  __device__ void finish(int tok, int row, float v) const {
    a.c.y[(size_t)tok * a.c.R + row] = __float2half_rn(v * __half2float(a.scale[row]));
  }
};

#ifndef Q2_TRL_W
#define Q2_TRL_W 24                   // 16: 13.8 us, 24: 13.2, 32: 13.8 per 12288x4096 GEMV (GB300)
#endif
#ifndef Q2_TRL_AHEAD
#define Q2_TRL_AHEAD 1
#endif
constexpr int kTrellisAhead = Q2_TRL_AHEAD;
constexpr int kTrlWarps = Q2_TRL_W;   // warps per CTA of the trellis kernel

template <int W, int AHEAD, int K>
__global__ void __launch_bounds__(W * 32, kMinBlocks) k_trellis_b1(TrellisArgs a) {
  uint32_t* tab = reinterpret_cast<uint32_t*>(q2_smem);                                  // K copies
  uint32_t* xs = reinterpret_cast<uint32_t*>(q2_smem + trl_table_bytes<K>());           // x as half2, C/2 words
  // K copies of each entry, written as K consecutive words (16-byte stores for K >= 4)
  for (int i = threadIdx.x; i < 4096; i += W * 32) {
    const uint32_t v = __ldg(a.table + i);
    if constexpr (K >= 4) {
#pragma unroll
      for (int c = 0; c < K; c += 4) *reinterpret_cast<uint4*>(tab + i * K + c) = make_uint4(v, v, v, v);
    } else {
      tab[i] = v;
    }
  }
  TrellisF<W * 32, K> f{a, reinterpret_cast<const unsigned char*>(tab), xs, (uint32_t)((threadIdx.x & 31) % K) * 4u};
  unsigned char* tail = q2_smem + trl_table_bytes<K>() + ((a.c.C * 2 + 15) / 16) * 16;
  run_b1<W, AHEAD>(f, a.c, tail);                  // one group over all segments
}

// ------------------------------------------------------------ host side
// The generic kernels ask for more than half of an SM's shared memory, so an
// SM holds one of their CTAs.
constexpr int kOneCtaSmem = 116 * 1024;
constexpr int kMaxDynSmem = 227 * 1024;   // opt-in dynamic shared memory per CTA
constexpr int kTwoCtaSmem = kMinBlocks == 2 ? 80 * 1024 : kOneCtaSmem;

struct Geo {
  int grid;      // CTAs
};

Geo geometry(const q2_blob_header& d) {
  const int items = d.nslice * q2_nrb(d);
  Geo g;
  g.grid = std::max(1, std::min(items, dev_info().sms));
  return g;
}

// The accumulator words hold at most Q2_MAX_SPLIT slices per row, and the
// workspace at most Q2_MAX_ROWS rows per token.
bool b1_shape_ok(const q2_blob_header& d) { return d.nslice >= 1 && d.nslice <= Q2_MAX_SPLIT && d.Rpad <= Q2_MAX_ROWS; }

B1 make_b1(const q2_handle* h, const void* x, void* y, int ntok, const q2_pf* pf = nullptr) {
  const q2_blob_header& d = h->hdr;
  B1 c;
  if (pf) c.pf = *pf;
  else c.pf = q2_pf{};
  c.x = static_cast<const __half*>(x);
  c.y = static_cast<__half*>(y);
  c.acc = static_cast<unsigned long long*>(h->ws);
  // fixed-point scale 2^F with |partial| * 2^F < 2^45 for every fp16 x
  int e = 0;
  if (h->pbound > 0.0) std::frexp(h->pbound, &e);    // pbound < 2^e
  const int F = std::max(-100, std::min(100, 45 - e));
  c.fscale = std::ldexp(1.0f, F);
  c.finv = std::ldexp(1.0f, -F);
  c.R = d.R;
  c.C = d.C;
  c.Rpad = d.Rpad;
  c.nrb = q2_nrb(d);
  c.nslice = d.nslice;
  c.ntok = ntok;
  return c;
}

template <typename A>
int launch1(void (*kernel)(A), const A& args, const Geo& g, int threads, int table_bytes, void* stream,
            int min_smem = kTwoCtaSmem) {
  const int smem = std::max(min_smem, table_bytes + kTailFixed);
  return launch_pdl(kernel, args, g.grid, threads, smem, stream);
}

// The lean single-token kernel's arguments: the pointers and scalars of
// make_b1, and each CTA's item range.  The split is slice-aligned, so no CTA
// builds a second table (BPDQ items are cheap enough that a second table
// costs more than the few extra items this leaves on some CTAs).  With at
// least as many CTAs as slices, slice g gets CTAs [floor(g*G/ns),
// floor((g+1)*G/ns)), floor(G/ns) or ceil(G/ns) of them, which split its nrb
// row blocks evenly; the last slice gets the larger count, so the CTAs with
// the highest indices, which start last (the previous launch frees their
// SMs last), get the fewer items (Qwen3-8B stack on GB300: 651.4 against
// 655.3 us per step with the larger counts first).  With fewer CTAs than
// slices, each CTA takes whole slices [floor(b*ns/G), floor((b+1)*ns/G)).
LeanArgs make_lean(const q2_handle* h, const void* x, void* y, const q2_pf* pf, int grid) {
  const q2_blob_header& d = h->hdr;
  const B1 c = make_b1(h, x, y, 1, pf);
  LeanArgs a;
  a.x = c.x;
  a.y = c.y;
  a.acc = c.acc;
  a.bits = reinterpret_cast<const uint4*>(h->dev + d.off[SEC_BPDQ_BITS]);
  a.c01 = reinterpret_cast<const uint32_t*>(h->dev + d.off[SEC_BPDQ_C01]);
  a.off = reinterpret_cast<const unsigned short*>(h->dev + d.off[SEC_BPDQ_OFF]);
  a.fscale = c.fscale;
  a.finv = c.finv;
  a.R = c.R;
  a.C = c.C;
  a.Rpad = c.Rpad;
  a.nrb = c.nrb;
  a.nslice = c.nslice;
  a.pf = c.pf;
  const unsigned long long units = a.pf.len[0] >> 4, parts = (unsigned long long)grid * kLeanW;
  a.pfq = (uint32_t)(units / parts);
  a.pfr = (uint32_t)(units % parts);
  const int ns = c.nslice, nrb = c.nrb, G = grid;
  if (ns <= G) {
    for (int g = 0; g < ns; ++g) {
      const int f0 = g * G / ns, f1 = (g + 1) * G / ns, n = f1 - f0;
      for (int k = 0; k < n; ++k) a.start[f0 + k] = (uint32_t)(g * nrb + k * nrb / n);
    }
  } else {
    for (int b = 0; b < G; ++b) a.start[b] = (uint32_t)(b * ns / G * nrb);
  }
  a.start[G] = (uint32_t)(ns * nrb);
  return a;
}

int lean_grid(const q2_blob_header& d) { return std::min(geometry(d).grid, kLeanMaxGrid); }

// The lean multi-token kernel's arguments: those of make_lean plus ntok.
LeanMArgs make_leanm(const q2_handle* h, const void* x, void* y, int ntok, const q2_pf* pf, int grid) {
  const LeanArgs l = make_lean(h, x, y, pf, grid);
  LeanMArgs a;
  a.x = l.x;
  a.y = l.y;
  a.acc = l.acc;
  a.bits = l.bits;
  a.c01 = l.c01;
  a.off = l.off;
  a.fscale = l.fscale;
  a.finv = l.finv;
  a.R = l.R;
  a.C = l.C;
  a.Rpad = l.Rpad;
  a.nrb = l.nrb;
  a.nslice = l.nslice;
  a.ntok = ntok;
  a.pf = l.pf;
  for (int b = 0; b <= grid; ++b) a.start[b] = l.start[b];
  return a;
}

// Warps per CTA of the one-pair kernel (127 registers).
constexpr int kMWarps = 16;

}  // namespace
}  // namespace q2

using namespace q2;

extern "C" int q2_b1_bpdq(const q2_handle* h, const void* x, void* y, void* stream, const q2_pf* pf) {
  const q2_blob_header& d = h->hdr;
  if (!b1_shape_ok(d)) return Q2_ESHAPE;
  const int G = lean_grid(d);
  const LeanArgs a = make_lean(h, x, y, pf, G);
  if (a.pf.len[0]) return launch_pdl(k_bpdq1<kLeanW, true, true>, a, G, kLeanW * 32, kTabSmem, stream);
  return launch_pdl(k_bpdq1<kLeanW, true, false>, a, G, kLeanW * 32, kTabSmem, stream);
}

// BPDQ at 2..6 tokens on CUDA cores.  Each token pair runs through the lean
// one-pair kernel and an odd last token through the single-token kernel,
// stream-ordered (x is [ntok][C], y [ntok][R]); each launch uses the first
// 2 x Rpad accumulator words and leaves them zero for the next.  Measured on
// the Qwen3-8B stack (ms per step at 2/3/4/5/6 tokens): one launch with
// ceil(ntok/2) pair tables (12 warps for two pairs, 8 for three, by
// registers) ran 0.92/1.81/2.01/3.17/3.42, the pair launches 0.92 at two
// tokens and less at more, since the lookups are bound by shared-memory
// bandwidth and more warps hide it better.  Every token's result is
// bit-identical to the same token run alone through q2_b1_bpdq.
extern "C" int q2_mt_bpdq(const q2_handle* h, const void* x, void* y, int ntok, void* stream, const q2_pf* pf) {
  const q2_blob_header& d = h->hdr;
  if (ntok < 2 || ntok > kMtMaxTok) return Q2_ENTOK;
  if (!b1_shape_ok(d)) return Q2_ESHAPE;
  const int G = lean_grid(d);
  const __half* xh = static_cast<const __half*>(x);
  __half* yh = static_cast<__half*>(y);
  for (int t = 0; t < ntok; t += 2) {
    const q2_pf* p = t == 0 ? pf : nullptr;
    int st;
    if (t + 1 < ntok) {
      const LeanMArgs a = make_leanm(h, xh + (size_t)t * d.C, yh + (size_t)t * d.R, 2, p, G);
      st = launch_pdl(k_bpdqm<kMWarps, 1>, a, G, kMWarps * 32, kPairBytes + 256, stream);
    } else {
      st = q2_b1_bpdq(h, xh + (size_t)t * d.C, yh + (size_t)t * d.R, stream, p);
    }
    if (st) return st;
  }
  return Q2_OK;
}

extern "C" int q2_b1_noweights(const q2_handle* h, const void* x, void* y, void* stream, const q2_pf* pf) {
  if (!b1_shape_ok(h->hdr)) return Q2_ESHAPE;
  const int G = lean_grid(h->hdr);
  const LeanArgs a = make_lean(h, x, y, pf, G);
  if (a.pf.len[0]) return launch_pdl(k_bpdq1<kLeanW, false, true>, a, G, kLeanW * 32, kTabSmem, stream);
  return launch_pdl(k_bpdq1<kLeanW, false, false>, a, G, kLeanW * 32, kTabSmem, stream);
}

extern "C" int q2_b1_leech(const q2_handle* h, const void* x, void* y, void* stream, const q2_pf* pf) {
  const q2_blob_header& d = h->hdr;
  if (!b1_shape_ok(d)) return Q2_ESHAPE;
  LeechArgs a;
  a.c = make_b1(h, x, y, 1, pf);
  a.planes = h->dev + d.off[SEC_LEECH_PLANES];
  a.parity = reinterpret_cast<const uint16_t*>(h->dev + d.off[SEC_LEECH_PARITY]);
  a.scale = reinterpret_cast<const __half*>(h->dev + d.off[SEC_LEECH_SCALE]);
  a.tail = reinterpret_cast<const __half*>(h->dev + d.off[SEC_LEECH_TAIL]);
  a.excptr = reinterpret_cast<const uint32_t*>(h->dev + d.off[SEC_LEECH_EXCPTR]);
  a.exccol = reinterpret_cast<const uint32_t*>(h->dev + d.off[SEC_LEECH_EXCCOL]);
  a.nblock = d.nblock;
  a.tail_n = d.tail;
  a.tailpad = d.tailpad;
  a.inv_sqrt8 = d.inv_sqrt8;
  if (d.layout == Q2_LEECH_OFFSET4)
    return launch1(k_leech_b1<kLeechWarps, kLeechAhead, 4>, a, geometry(d), kLeechWarps * 32, kTabSmem, stream);
  return launch1(k_leech_b1<kLeechWarps, kLeechAhead, 3>, a, geometry(d), kLeechWarps * 32, kTabSmem, stream);
}

extern "C" int q2_b1_trellis(const q2_handle* h, const void* x, void* y, void* stream, const q2_pf* pf) {
  const q2_blob_header& d = h->hdr;
  if (!b1_shape_ok(d)) return Q2_ESHAPE;
  TrellisArgs a;
  a.c = make_b1(h, x, y, 1, pf);
  a.stream = h->dev + d.off[SEC_TRL_STREAM];
  a.table = reinterpret_cast<const uint32_t*>(h->dev + d.off[SEC_TRL_TABLE]);
  a.scale = reinterpret_cast<const __half*>(h->dev + d.off[SEC_TRL_SCALE]);
  // as many codebook copies as fit beside x and the tail in one CTA's shared memory
  const int xbytes = (d.C * 2 + 15) / 16 * 16;
  auto fits = [&](int tb) { return tb + xbytes + kTailFixed <= kMaxDynSmem; };
  if (fits(trl_table_bytes<8>()))
    return launch1(k_trellis_b1<kTrlWarps, kTrellisAhead, 8>, a, geometry(d), kTrlWarps * 32, trl_table_bytes<8>() + xbytes,
                   stream);
  if (fits(trl_table_bytes<4>()))
    return launch1(k_trellis_b1<kTrlWarps, kTrellisAhead, 4>, a, geometry(d), kTrlWarps * 32, trl_table_bytes<4>() + xbytes,
                   stream);
  return launch1(k_trellis_b1<kTrlWarps, kTrellisAhead, 1>, a, geometry(d), kTrlWarps * 32, trl_table_bytes<1>() + xbytes,
                 stream);
}

// ---------------------------------------------------------------------------
// Allocation-free batch-1 BPDQ entry point.
//
// Some callers cannot allocate device memory when they call the GEMV: code
// that runs while a CUDA stream is being captured into a graph (cudaMalloc
// is not permitted there), plugins whose host framework owns all device
// memory and offers them no allocator, and real-time decode loops that must
// not touch the allocator after start-up.  q2_gemv_bpdq_noalloc serves them:
// the split-K accumulator words that q2_gemv keeps in a caller-bound
// workspace go to a scratch array that belongs to this library instead, so
// the caller passes only the handle, x, y and a stream.  Every
// GPU that loads the library holds the array (Q2_NOALLOC_SCRATCH_BYTES)
// until the process exits.

namespace {

// Device memory for the accumulator words; host code must never hand this
// symbol to a kernel (on the host it only stands in for the device
// address).  Zero-initialised when the module loads; every completed call
// leaves the words it used at zero again.
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
  const size_t need = (size_t)h->hdr.Rpad * 8;           // one accumulator word per row
  if (need > (size_t)Q2_NOALLOC_SCRATCH_BYTES) return Q2_ESCRATCH;
  void* scratch = nullptr;
  const int st = noalloc_scratch(&scratch);
  if (st) return st;
  // the same launch as q2_gemv at ntok = 1, with the scratch in place of the
  // caller's workspace
  q2_handle view = *h;
  view.ws = scratch;
  view.ws_bytes = Q2_NOALLOC_SCRATCH_BYTES;
  return q2_b1_bpdq(&view, x, y, static_cast<void*>(stream), nullptr);
}
