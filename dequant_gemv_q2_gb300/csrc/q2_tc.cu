// Skinny-GEMM path on the 5th-generation tensor cores (tcgen05) for
// 16 <= padded ntok <= 64: decode once per tile, multiply for every token.
//
// A CTA owns 128 output rows (four 32-row blocks) and a range of 256-column
// slices.  For each slice, its 8 warps decode the packed weights of the
// 128 x 256 tile into fp16 in shared memory (the canonical decoded weights:
// BPDQ through the per-(group, row) 4-entry value table, one byte permute
// per two or four weights), the x tile of all tokens is staged next to it,
// and one thread issues sixteen tcgen05.mma.kind::f16 (M = 128, N = padded
// ntok, K = 16) that accumulate in a TMEM fp32 tile.  A and B tiles are
// double-buffered; an mbarrier per buffer, armed by tcgen05.commit, tells
// the decoders when the tensor core has finished reading a buffer.  At the
// end each warp reads its 32 TMEM lanes (its 32 rows) and writes fp32
// partial sums for the split-K reduction kernel, or y directly.
//
// Operand layout in shared memory: K-major, no swizzle, core matrices of
// 8 rows x 16 bytes; the byte offset of element (row m, k) is
// (m / 8) * 4096 + (k / 8) * 128 + (m % 8) * 16 + (k % 8) * 2, i.e. leading
// (K) byte offset 128 and stride (M/N) byte offset 4096.
//
// Every wait is bounded: a wait that runs out records an error code in
// q2_tc_error (read back with q2_device_errors) and the kernel skips the
// rest of its work, then frees its TMEM columns.
#include <cuda_fp16.h>

#include "q2_common.cuh"

extern __shared__ __align__(1024) unsigned char q2_smem[];
extern "C" int q2_launch_reduce_n(const q2_handle* h, const void* x, void* y, int ntok, int nsplit, void* stream);

__device__ unsigned int q2_tc_error = 0;

namespace q2 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kParts = kWarps / 4;            // warps per 32-row block, each decoding 256/kParts columns
constexpr int kPartBytes = 32 / kParts;       // rotated column-bytes of one plane per lane and part
constexpr int kRows = 128;                    // M of the MMA
constexpr int kTileA = kRows * 256 * 2;       // 64 KiB per A buffer
constexpr uint32_t kLBO = 128, kSBO = 4096;   // core-matrix strides (bytes)

// Shared-memory matrix descriptor (tcgen05): start >> 4 in bits 0-13,
// leading byte offset >> 4 in 16-29, stride byte offset >> 4 in 32-45,
// descriptor version 1 in 46-47, no swizzle (61-63 = 0).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)((kLBO >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((kSBO >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B fp16
// (7-9, 10-12 = 0), both K-major (15, 16 = 0), N >> 3 in 17-22, M >> 4 in 24-28.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t dtmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dtmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// 16 fp32 columns of this warp's 32 TMEM lanes (one row per lane).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Decode of 4 column-bytes (32 columns) of one row.  w0, w1: the 4 plane-0
// and plane-1 bytes.  The 2-bit code of column 8q + i is b0_i | b1_i << 1;
// E / O hold the codes of the even / odd columns of every byte (code of
// column 2j of a byte at bits 2j..2j+1 of that byte); masks by 0x33 split
// each into the codes of columns {0,4} and {2,6} (or {1,5}, {3,7}).  One byte
// permute per byte then forms a selector with four codes in its nibbles, and
// two permutes of the row's value table (low bytes, high bytes of v0..v3)
// give the fp16 weights; two more put them back in column order.
struct Codes4 {
  uint32_t ea, eb, oa, ob;
};

__device__ __forceinline__ Codes4 codes4(uint32_t w0, uint32_t w1) {
  const uint32_t e = (w0 & 0x55555555u) | ((w1 << 1) & 0xAAAAAAAAu);
  const uint32_t o = ((w0 >> 1) & 0x55555555u) | (w1 & 0xAAAAAAAAu);
  Codes4 c;
  c.ea = e & 0x33333333u;          // cols 0,4 of each byte
  c.eb = (e >> 2) & 0x33333333u;   // cols 2,6
  c.oa = o & 0x33333333u;          // cols 1,5
  c.ob = (o >> 2) & 0x33333333u;   // cols 3,7
  return c;
}

// 8 fp16 weights of byte q (0..3) of a Codes4, in column order.
template <int Q>
__device__ __forceinline__ uint4 decode_q(const Codes4& c, uint32_t tlo, uint32_t thi) {
  constexpr uint32_t sel = (uint32_t)Q | ((4u + Q) << 4);
  const uint32_t s0 = __byte_perm(c.ea, c.oa, sel);   // nibbles: codes of cols 0,4,1,5
  const uint32_t s1 = __byte_perm(c.eb, c.ob, sel);   // cols 2,6,3,7
  const uint32_t lo0 = __byte_perm(tlo, 0u, s0), hi0 = __byte_perm(thi, 0u, s0);
  const uint32_t lo1 = __byte_perm(tlo, 0u, s1), hi1 = __byte_perm(thi, 0u, s1);
  uint4 r;
  r.x = __byte_perm(lo0, hi0, 0x6240u);     // cols 0,1
  r.y = __byte_perm(lo1, hi1, 0x6240u);     // cols 2,3
  r.z = __byte_perm(lo0, hi0, 0x7351u);     // cols 4,5
  r.w = __byte_perm(lo1, hi1, 0x7351u);     // cols 6,7
  return r;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

struct TcArgs {
  const unsigned char* bits;   // item stream (BPDQ bits, trellis symbols, Leech planes)
  const uint2* vtab;           // BPDQ: [G][Rpad] 4 halves
  const uint32_t* table;       // trellis: 4096 half2
  const uint16_t* parity;      // Leech: [S][Rpad]
  const __half* x;             // [ntok][C]
  __half* y;                   // [ntok][R]  (nsplit == 1, BPDQ only)
  float* partial;              // [ntok][nsplit][Rpad]
  int R, C, Rpad, nrb, S, ntok, N, nsplit, ntile, nblock;
};

constexpr uint32_t kHashHi = 0x9E37u << 16;     // trellis: (s*0x9E37 mod 2^16) in bits 16..31

// Per-format shape of a slice's K range: 32 chunks of 8 columns, plus, for
// Leech, 4 chunks carrying the parity term (A = parity bit of the blocks
// starting in the slice, B = their block sums of x split into fp16 hi + lo).
template <int FMT>
struct TcShape {
  static constexpr int kch = FMT == Q2_LEECH ? 36 : 32;
  static constexpr uint32_t sbo = kch * 128;
  static constexpr int tileA = kRows * kch * 16;
  static constexpr int table = FMT == Q2_TRELLIS ? 4096 * 4 : 0;
  static constexpr int item = FMT == Q2_BPDQ ? Q2_ITEM_BYTES_BPDQ : FMT == Q2_TRELLIS ? Q2_ITEM_BYTES_TRL
                                                                                     : Q2_ITEM_BYTES_LEECH;
};

__device__ __forceinline__ uint64_t sdesc_s(uint32_t addr, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)((kLBO >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// Leech: 3-bit codes b0 | b1 << 1 | b2 << 2 of the columns of 4 column-bytes
// in nibble fields (the BPDQ split of codes4, with bit 2 from plane 2).
__device__ __forceinline__ Codes4 codes4x3(uint32_t w0, uint32_t w1, uint32_t w2) {
  Codes4 c = codes4(w0, w1);
  c.ea |= (w2 << 2) & 0x44444444u;   // cols 0,4: b2 bits 0,4 -> 2,6
  c.eb |= w2 & 0x44444444u;          // cols 2,6: bits 2,6
  c.oa |= (w2 << 1) & 0x44444444u;   // cols 1,5: bits 1,5 -> 2,6
  c.ob |= (w2 >> 1) & 0x44444444u;   // cols 3,7: bits 3,7 -> 2,6
  return c;
}

// 2u = 2*(b0 + 2*b1 - 4*b2) in fp16 for the 8 columns of byte Q; the low
// byte of every such fp16 value is 0, so only high bytes are looked up.
template <int Q>
__device__ __forceinline__ uint4 decode_leech_q(const Codes4& c) {
  // fp16 high bytes of 0, 2, 4, 6, -8, -6, -4, -2 (code 0..7)
  constexpr uint32_t HA = 0x46444000u, HB = 0xC0C4C6C8u;
  constexpr uint32_t sel = (uint32_t)Q | ((4u + Q) << 4);
  const uint32_t s0 = __byte_perm(c.ea, c.oa, sel);   // codes of cols 0,4,1,5
  const uint32_t s1 = __byte_perm(c.eb, c.ob, sel);   // cols 2,6,3,7
  const uint32_t h0 = __byte_perm(HA, HB, s0), h1 = __byte_perm(HA, HB, s1);
  uint4 r;
  r.x = __byte_perm(h0, 0u, 0x2404u);       // cols 0,1: [0, h(c0), 0, h(c1)]
  r.y = __byte_perm(h1, 0u, 0x2404u);       // cols 2,3
  r.z = __byte_perm(h0, 0u, 0x3414u);       // cols 4,5
  r.w = __byte_perm(h1, 0u, 0x3414u);       // cols 6,7
  return r;
}

// Trellis: steps (128/kParts)*H .. of a segment -> columns (256/kParts)*H ..
// of the A row (column-byte = step / 4); H is a template parameter so every
// window index is static.
template <int H>
__device__ __forceinline__ void trellis_part(const uint32_t (&W)[16], const uint32_t* tab, unsigned char* arow) {
#pragma unroll
  for (int cb = 0; cb < kPartBytes; ++cb) {
    uint32_t e4[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int k = H * kPartBytes * 4 + cb * 4 + t;
      const int n = 127 - k;
      const uint32_t f = __funnelshift_r(W[n >> 3], W[((n >> 3) + 1) & 15], 4 * (n & 7));
      const uint32_t e = tab[(f * kHashHi) >> 20];
      e4[t] = e ^ ((f & 1u) ? 0x80008000u : 0u);
    }
    *reinterpret_cast<uint4*>(arow + (H * kPartBytes + cb) * kLBO) = make_uint4(e4[0], e4[1], e4[2], e4[3]);
  }
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1) k_tc(TcArgs a) {
  using Sh = TcShape<FMT>;
  uint32_t* tab = reinterpret_cast<uint32_t*>(q2_smem);            // trellis table
  unsigned char* A0 = q2_smem + Sh::table;
  unsigned char* B0 = A0 + 2 * Sh::tileA;
  const int bbytes = (a.N / 8) * (int)Sh::sbo;
  uint64_t* bars = reinterpret_cast<uint64_t*>(B0 + 2 * bbytes);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rbl = warp & 3, part = warp >> 2;        // row block in tile, part of the slice
  const int tile = blockIdx.x % a.ntile, split = blockIdx.x / a.ntile;
  const int sA = split * a.S / a.nsplit, sB = (split + 1) * a.S / a.nsplit;
  const int rb = tile * 4 + rbl;
  const bool valid = rb < a.nrb;                     // the last tile may be ragged
  const int row = rb * 32 + lane;
  const int m = rbl * 32 + lane;                     // row inside the tile
  const uint32_t ncols = a.N <= 32 ? 32u : 64u;
  const int tile_rbs = min(4, a.nrb - tile * 4);

  if (threadIdx.x == 0) {
    for (int s = sA; s < sB; ++s)
      prefetch_l2(a.bits + ((size_t)s * a.nrb + tile * 4) * Sh::item, (size_t)tile_rbs * Sh::item);
    mbar_init(saddr(&bars[0]), 1);
    mbar_init(saddr(&bars[1]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tslot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (FMT == Q2_TRELLIS)
    for (int i = threadIdx.x; i < 4096; i += kThreads) tab[i] = a.table[i];
  // zero both B buffers once (padding tokens, unused parity columns)
  for (int i = threadIdx.x; i < 2 * bbytes / 16; i += kThreads) reinterpret_cast<uint4*>(B0)[i] = make_uint4(0, 0, 0, 0);

  // per-lane payload of one slice: BPDQ/Leech the part's kPartBytes rotated
  // bytes of each plane (rotated positions part*kPartBytes ..), trellis the
  // whole 64-byte packet; plus BPDQ's value table / Leech's parity
  constexpr int NP = FMT == Q2_BPDQ ? 2 : FMT == Q2_LEECH ? 3 : 4;
  uint4 pl[NP];
  uint2 vt = make_uint2(0, 0);
  uint32_t par = 0;
  auto load = [&](int s, uint4 (&d)[NP], uint2& v, uint32_t& pw) {
    const unsigned char* ip = a.bits + ((size_t)s * a.nrb + rb) * Sh::item + lane * 16;
    if (FMT == Q2_TRELLIS) {
#pragma unroll
      for (int k = 0; k < NP; ++k) d[k] = __ldg(reinterpret_cast<const uint4*>(ip + k * 512));
    } else if (kParts == 2) {
#pragma unroll
      for (int k = 0; k < NP; ++k) d[k] = ldg_stream(ip + (2 * k + part) * 512);
    } else {                                  // kParts == 4: 8 bytes of a chunk
#pragma unroll
      for (int k = 0; k < NP; ++k) {
        const uint2 h = __ldg(reinterpret_cast<const uint2*>(ip + (2 * k + (part >> 1)) * 512 + (part & 1) * 8));
        d[k] = make_uint4(h.x, h.y, 0u, 0u);
      }
    }
    if (FMT == Q2_BPDQ) v = a.vtab[(size_t)s * a.Rpad + row];
    if (FMT == Q2_LEECH) pw = a.parity[(size_t)s * a.Rpad + row];
  };
#pragma unroll
  for (int k = 0; k < NP; ++k) pl[k] = make_uint4(0, 0, 0, 0);
  if (valid && sA < sB) load(sA, pl, vt, par);
  pdl_wait();
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t idesc = idesc_f16(kRows, a.N);
  bool ok = true;

  // x tile (and Leech parity columns) of slice s into B buffer Bb: cp.async
  // copies, waited for before the slice's MMAs are issued
  auto stage_x = [&](int s, unsigned char* Bb) {
    const int ncols_s = min(256, a.C - s * 256);     // Leech: the last slice may be short
    const __half* xs = a.x + (size_t)s * 256;
    const uint32_t bb0 = saddr(Bb);
    for (int e = threadIdx.x; e < a.ntok * 32; e += kThreads) {
      const int n = e >> 5, kc = e & 31;
      const uint32_t dst = bb0 + (n >> 3) * Sh::sbo + kc * kLBO + (n & 7) * 16;
      if (kc * 8 + 8 <= ncols_s) {
        cp_async16(dst, xs + (size_t)n * a.C + kc * 8);
      } else {
        uint4 v = make_uint4(0, 0, 0, 0);
        __half* hv = reinterpret_cast<__half*>(&v);
        for (int i = 0; i < 8; ++i)
          if (kc * 8 + i < ncols_s) hv[i] = xs[(size_t)n * a.C + kc * 8 + i];
        *reinterpret_cast<uint4*>(Bb + (n >> 3) * Sh::sbo + kc * kLBO + (n & 7) * 16) = v;
      }
    }
    if (FMT == Q2_LEECH) {
      // parity columns: block sums of x for the blocks starting in this slice,
      // hi part in chunks 32-33, lo part (x - hi) in chunks 34-35
      const int bfirst = (s * 256 + 23) / 24;
      const int blast = min(a.nblock - 1, (s * 256 + 256 + 23) / 24 - 1);
      const int nbk = max(0, blast - bfirst + 1);
      for (int e = threadIdx.x; e < a.ntok * 16; e += kThreads) {
        const int n = e >> 4, jb = e & 15;
        float xsum = 0.f;
        if (jb < nbk) {
          const __half* xp = a.x + (size_t)n * a.C + (size_t)(bfirst + jb) * 24;
          for (int i = 0; i < 24; ++i) xsum += __half2float(xp[i]);
        }
        const __half hi = __float2half_rn(xsum);
        const __half lo = __float2half_rn(xsum - __half2float(hi));
        unsigned char* bn = Bb + (n >> 3) * Sh::sbo + (n & 7) * 16;
        reinterpret_cast<__half*>(bn + (32 + (jb >> 3)) * kLBO)[jb & 7] = hi;
        reinterpret_cast<__half*>(bn + (34 + (jb >> 3)) * kLBO)[jb & 7] = lo;
      }
    }
  };
  if (sA < sB) stage_x(sA, B0);

  // Slice s: decode the weights into A[buf] while x(s) lands in B[buf], then
  // one thread issues the MMAs.  Right after, once the MMAs of slice s - 1
  // have released the other buffers, x(s + 1) is staged into them, so its
  // L2 round trip overlaps the decode of slice s + 1.
  for (int s = sA; s < sB && ok; ++s) {
    const int buf = (s - sA) & 1;
    unsigned char* Ab = A0 + buf * Sh::tileA;
    unsigned char* Bb = B0 + buf * bbytes;
    uint4 nx[NP];
    uint2 nvt = vt;
    uint32_t npar = par;
#pragma unroll
    for (int k = 0; k < NP; ++k) nx[k] = pl[k];
    if (valid && s + 1 < sB) load(s + 1, nx, nvt, npar);
    if (ok) {
      unsigned char* arow = Ab + (m >> 3) * Sh::sbo + (m & 7) * 16;
      if (FMT == Q2_TRELLIS) {
        const uint32_t W[16] = {pl[0].x, pl[0].y, pl[0].z, pl[0].w, pl[1].x, pl[1].y, pl[1].z, pl[1].w,
                                pl[2].x, pl[2].y, pl[2].z, pl[2].w, pl[3].x, pl[3].y, pl[3].z, pl[3].w};
        if (part == 0) trellis_part<0>(W, tab, arow);
        else if (part == 1) trellis_part<1>(W, tab, arow);
        else if (kParts > 2 && part == 2) trellis_part<(kParts > 2 ? 2 : 0)>(W, tab, arow);
        else if (kParts > 2) trellis_part<(kParts > 2 ? 3 : 0)>(W, tab, arow);
      } else {
        const uint32_t rot = (uint32_t)(part * kPartBytes + lane) * kLBO;
        constexpr int NW = kPartBytes / 4;      // 32-bit words of a plane per lane and part
        if (FMT == Q2_BPDQ) {
          const uint32_t tlo = __byte_perm(vt.x, vt.y, 0x6420u);
          const uint32_t thi = __byte_perm(vt.x, vt.y, 0x7531u);
          const uint32_t w0[4] = {pl[0].x, pl[0].y, pl[0].z, pl[0].w};
          const uint32_t w1[4] = {pl[1].x, pl[1].y, pl[1].z, pl[1].w};
#pragma unroll
          for (int j = 0; j < NW; ++j) {
            const Codes4 c = codes4(w0[j], w1[j]);
            *reinterpret_cast<uint4*>(arow + ((rot + (4 * j + 0) * kLBO) & 4095u)) = decode_q<0>(c, tlo, thi);
            *reinterpret_cast<uint4*>(arow + ((rot + (4 * j + 1) * kLBO) & 4095u)) = decode_q<1>(c, tlo, thi);
            *reinterpret_cast<uint4*>(arow + ((rot + (4 * j + 2) * kLBO) & 4095u)) = decode_q<2>(c, tlo, thi);
            *reinterpret_cast<uint4*>(arow + ((rot + (4 * j + 3) * kLBO) & 4095u)) = decode_q<3>(c, tlo, thi);
          }
        } else {
          const uint32_t w0[4] = {pl[0].x, pl[0].y, pl[0].z, pl[0].w};
          const uint32_t w1[4] = {pl[1].x, pl[1].y, pl[1].z, pl[1].w};
          const uint32_t w2[4] = {pl[2].x, pl[2].y, pl[2].z, pl[2].w};
#pragma unroll
          for (int j = 0; j < NW; ++j) {
            const Codes4 c = codes4x3(w0[j], w1[j], w2[j]);
            *reinterpret_cast<uint4*>(arow + ((rot + (4 * j + 0) * kLBO) & 4095u)) = decode_leech_q<0>(c);
            *reinterpret_cast<uint4*>(arow + ((rot + (4 * j + 1) * kLBO) & 4095u)) = decode_leech_q<1>(c);
            *reinterpret_cast<uint4*>(arow + ((rot + (4 * j + 2) * kLBO) & 4095u)) = decode_leech_q<2>(c);
            *reinterpret_cast<uint4*>(arow + ((rot + (4 * j + 3) * kLBO) & 4095u)) = decode_leech_q<3>(c);
          }
          if (part == 0) {
            // parity columns: A = 1.0 where the block starting in this slice is odd
            uint32_t pv[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uint32_t lo = ((par >> (2 * q)) & 1u) ? 0x3C00u : 0u;
              const uint32_t hi = ((par >> (2 * q + 1)) & 1u) ? 0x3C000000u : 0u;
              pv[q] = lo | hi;
            }
            const uint4 p0 = make_uint4(pv[0], pv[1], pv[2], pv[3]), p1 = make_uint4(pv[4], pv[5], pv[6], pv[7]);
            *reinterpret_cast<uint4*>(arow + 32 * kLBO) = p0;
            *reinterpret_cast<uint4*>(arow + 33 * kLBO) = p1;
            *reinterpret_cast<uint4*>(arow + 34 * kLBO) = p0;
            *reinterpret_cast<uint4*>(arow + 35 * kLBO) = p1;
          }
        }
      }
    }
    cp_async_wait_all();
    fence_async_smem();
    tc_fence_before();
    ok = __syncthreads_and(ok);
    tc_fence_after();
    if (threadIdx.x == 0 && ok) {
      const uint32_t aa = saddr(Ab), bb = saddr(Bb);
#pragma unroll
      for (int k = 0; k < Sh::kch / 2; ++k)
        mma_f16(tmem, sdesc_s(aa + k * 2 * kLBO, Sh::sbo), sdesc_s(bb + k * 2 * kLBO, Sh::sbo), idesc,
                (s > sA || k > 0) ? 1u : 0u);
      mma_commit(saddr(&bars[buf]));
    }
    if (ok && s + 1 < sB) {
      const int nb = buf ^ 1;
      if (s > sA && !mbar_wait(saddr(&bars[nb]), (uint32_t)((s - 1 - sA) >> 1) & 1u)) {
        ok = false;
        if (threadIdx.x == 0) atomicExch(&q2_tc_error, 1u);
      }
      if (ok) stage_x(s + 1, B0 + nb * bbytes);
    }
#pragma unroll
    for (int k = 0; k < NP; ++k) pl[k] = nx[k];
    vt = nvt;
    par = npar;
  }
  const int used = sB - sA;
  if (ok && used > 0) {
    const int last = used - 1;
    if (!mbar_wait(saddr(&bars[last & 1]), (uint32_t)(last >> 1) & 1u)) ok = false;
    if (ok && used > 1 && !mbar_wait(saddr(&bars[(last - 1) & 1]), (uint32_t)((last - 1) >> 1) & 1u)) ok = false;
    if (!ok && threadIdx.x == 0) atomicExch(&q2_tc_error, 2u);
  }
  ok = __syncthreads_and(ok);
  tc_fence_after();
  if (warp < 4 && ok) {
    const int orow = (tile * 4 + warp) * 32 + lane;
    for (int c0 = 0; c0 < a.N; c0 += 16) {
      float v[16];
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int t = c0 + i;
        if (t < a.ntok) {
          if (a.nsplit == 1 && FMT == Q2_BPDQ) {
            if (orow < a.R) a.y[(size_t)t * a.R + orow] = __float2half_rn(v[i]);
          } else if (orow < a.Rpad) {
            a.partial[((size_t)t * a.nsplit + split) * a.Rpad + orow] = v[i];
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
}

// Packed formats at 2..64 tokens on the tensor cores (tokens padded to a
// multiple of 16).  Split-K partials (and every trellis / Leech result, whose
// epilogue needs the row scale, exceptions and tail) go through the reduce
// kernel.
template <int FMT>
int launch_tc(const q2_handle* h, const void* x, void* y, int ntok, void* stream) {
  using Sh = TcShape<FMT>;
  const q2_blob_header& d = h->hdr;
  TcArgs a = {};
  if (FMT == Q2_BPDQ) {
    a.bits = h->dev + d.off[SEC_BPDQ_BITS];
    a.vtab = reinterpret_cast<const uint2*>(h->dev + d.off[SEC_BPDQ_VTAB]);
  } else if (FMT == Q2_TRELLIS) {
    a.bits = h->dev + d.off[SEC_TRL_STREAM];
    a.table = reinterpret_cast<const uint32_t*>(h->dev + d.off[SEC_TRL_TABLE]);
  } else {
    a.bits = h->dev + d.off[SEC_LEECH_PLANES];
    a.parity = reinterpret_cast<const uint16_t*>(h->dev + d.off[SEC_LEECH_PARITY]);
    a.nblock = d.nblock;
  }
  a.x = static_cast<const __half*>(x);
  a.y = static_cast<__half*>(y);
  a.partial = reinterpret_cast<float*>(static_cast<unsigned char*>(h->ws) + Q2_WS_PARTIAL_OFFSET);
  a.R = d.R;
  a.C = d.C;
  a.Rpad = d.Rpad;
  a.nrb = q2_nrb(d);
  a.S = d.nslice;
  a.ntok = ntok;
  a.N = (ntok + 15) / 16 * 16;
  a.ntile = (d.Rpad + kRows - 1) / kRows;
  const int sms = dev_info().sms;
  // K split: one CTA per SM at a time, so the makespan is (waves of CTAs) x
  // (slices per CTA + about one slice of prologue and epilogue)
  long best = -1;
  for (int ns = 1; ns <= a.S; ++ns) {
    const long ctas = (long)a.ntile * ns;
    const long waves = (ctas + sms - 1) / sms;
    const long cost = waves * ((a.S + ns - 1) / ns + 1);
    if (best < 0 || cost < best) {
      best = cost;
      a.nsplit = ns;
    }
  }
  const int smem = Sh::table + 2 * Sh::tileA + 2 * (a.N / 8) * (int)Sh::sbo + 64;
  int st = launch_pdl(k_tc<FMT>, a, a.ntile * a.nsplit, kThreads, smem, stream);
  if (st) return st;
  if (a.nsplit == 1 && FMT == Q2_BPDQ) return Q2_OK;
  return q2_launch_reduce_n(h, x, y, ntok, a.nsplit, stream);
}

}  // namespace
}  // namespace q2

extern "C" int q2_tc_bpdq(const q2_handle* h, const void* x, void* y, int ntok, void* stream) {
  return q2::launch_tc<Q2_BPDQ>(h, x, y, ntok, stream);
}
extern "C" int q2_tc_trellis(const q2_handle* h, const void* x, void* y, int ntok, void* stream) {
  return q2::launch_tc<Q2_TRELLIS>(h, x, y, ntok, stream);
}
extern "C" int q2_tc_leech(const q2_handle* h, const void* x, void* y, int ntok, void* stream) {
  return q2::launch_tc<Q2_LEECH>(h, x, y, ntok, stream);
}

// Device-side error word of the tensor-core kernels since the last call
// (then cleared): 0 in normal operation, else the code of a bounded wait
// that ran out.  Synchronous (reads device memory).
extern "C" int q2_device_errors(unsigned int* out) {
  if (!out) return Q2_EINVAL;
  unsigned int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, q2_tc_error, sizeof(v)) != cudaSuccess) return Q2_ECUDA;
  if (cudaMemcpyToSymbol(q2_tc_error, &z, sizeof(z)) != cudaSuccess) return Q2_ECUDA;
  *out = v;
  return Q2_OK;
}
