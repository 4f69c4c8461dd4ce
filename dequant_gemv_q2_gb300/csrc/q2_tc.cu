// Skinny-GEMM path on the 5th-generation tensor cores (tcgen05) for
// 2..64 tokens (padded to N = 16, 32, 48 or 64): decode once per tile,
// multiply for every token.
//
// A CTA owns 128 output rows (four 32-row blocks) and a range of 256-column
// slices, and runs them through a ring of kStages stages with three roles:
//   - 8 decoder warps turn the packed weights of the 128 x 256 tile into
//     fp16 in registers (BPDQ through the per-(group, row) 4-entry value
//     table, one byte permute per two or four weights) and store them into
//     tensor memory with tcgen05.st, one TMEM lane per row (the stage's A);
//   - one producer lane of the ninth warp loads the x tile of all tokens into
//     shared memory with four 2D TMA copies (the stage's B);
//   - the same lane, once a stage's A and B are both complete (one mbarrier
//     per stage: 8 decoder arrivals plus the TMA bytes), issues sixteen
//     tcgen05.mma.kind::f16 (M = 128, N, K = 16) reading A from TMEM and B
//     from shared memory into one fp32 accumulator in TMEM, and commits them
//     to the stage's "empty" mbarrier, which frees the stage for refilling.
// No role waits for another except through these barriers, so the decode of
// slice s + 1, the x copy of slice s + 2 and the MMAs of slice s overlap.
// At the end the decoder warps read the accumulator (each its 32 TMEM
// lanes) and write fp32 partial sums for the split-K reduction kernel, or y
// directly.
//
// TMEM columns (all 512 are allocated; one CTA per SM): D at 0 .. N - 1,
// A of stage st at kAcol0 + st * (4 x K chunks); A column j of a lane holds
// the fp16 weights k = 2j (low half) and 2j + 1 (high half) of its row.
//
// B in shared memory: K-major with the 128-byte swizzle, as the TMA writes
// it: the slice's K range in atoms of 64 columns, atom a at a * N * 128
// bytes; inside it token n's 128-byte row at n * 128 with 16-byte chunk c
// stored at chunk c ^ (n % 8).  The MMA descriptor gives stride 1024 bytes
// between 8-row groups and steps 32 bytes per K = 16 inside an atom.
//
// The BPDQ and Leech planes are stored lane-rotated for the batch-1 kernels
// (byte j of lane l's 32-byte plane row holds column-byte (j + l) mod 32).
// Every lane loads its whole rows and undoes the rotation in registers
// before decoding, because a TMEM store writes the same columns in every
// lane.
//
// Every wait is bounded: a wait that runs out records an error code in
// q2_tc_error (read back with q2_device_errors) and the kernel skips the
// rest of its work; the producer lane waits for its outstanding copies and
// MMAs before the CTA frees its TMEM columns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "q2_common.cuh"

extern __shared__ __align__(1024) unsigned char q2_smem[];
extern "C" int q2_launch_reduce_n(const q2_handle* h, const void* x, void* y, int ntok, int nsplit, void* stream);

__device__ unsigned int q2_tc_error = 0;

namespace q2 {
namespace {

constexpr int kDecWarps = 8;                  // decoder warps; one more warp copies x and issues MMAs
constexpr int kThreads = (kDecWarps + 1) * 32;
constexpr int kStages = 3;                    // slices in flight (A in TMEM, B in shared memory)
constexpr int kParts = kDecWarps / 4;         // warps per 32-row block, each decoding 256/kParts columns
constexpr int kPartBytes = 32 / kParts;       // column-bytes of one plane per lane and part
static_assert(kParts == 2, "the decode splits a row's 32 column-bytes between two warps");
constexpr int kRows = 128;                    // M of the MMA
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcol0 = 64;               // D takes TMEM columns 0..63
constexpr int kOneCtaSmem = 116 * 1024;       // two CTAs never share an SM (each holds all of TMEM)

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B fp16
// (7-9, 10-12 = 0), both K-major (15, 16 = 0), N >> 3 in 17-22, M >> 4 in 24-28.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[tmem] x B[smem descriptor]
__device__ __forceinline__ void mma_f16_ta(uint32_t dtmem, uint32_t atmem, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(dtmem),
      "r"(atmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane (the warp's 32 lanes).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, uint4 a, uint4 b, uint4 c, uint4 d) {
  const uint32_t r[16] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
  tmem_st16(taddr, r);
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Canonical words 4P .. 4P + 3 (column-bytes 16P .. 16P + 15) of one plane
// row from its 8 lane-rotated words R (rotated byte j = column-byte
// (j + lane) mod 32).  With lane = 4a + r, canonical word c starts at
// rotated byte 4(c - a) - r: the word rotation by a runs as three
// conditional rotations by 1, 2 and 4 words, the byte offset r as a funnel
// shift (clamped: r = 0 takes the high word whole).
template <int P>
__device__ __forceinline__ void unrotate_half(const uint32_t (&R)[8], int lane, uint32_t (&cw)[4]) {
  const int a = lane >> 2;
  const uint32_t sh = 32u - 8u * (uint32_t)(lane & 3);
  uint32_t t[8], u[8], v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) t[i] = (a & 1) ? R[(i + 7) & 7] : R[i];
#pragma unroll
  for (int i = 0; i < 8; ++i) u[i] = (a & 2) ? t[(i + 6) & 7] : t[i];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = (a & 4) ? u[(i + 4) & 7] : u[i];
#pragma unroll
  for (int c = 0; c < 4; ++c) cw[c] = __funnelshift_rc(v[(4 * P + c + 7) & 7], v[4 * P + c], sh);
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

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// one arrival that also expects `bytes` of asynchronous copies
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// 2D TMA tile load of box (x, y) of the tensor map into shared memory; the
// bytes are reported to the mbarrier.  x * 2 bytes is a multiple of 128.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void sleep_us(int us) {
  for (int k = 0; k < us; ++k) __nanosleep(1000);
}

struct TcArgs {
  CUtensorMap xmap;            // x [ntok][C] fp16: box 64 columns x N tokens, 128-byte swizzle (use_tma)
  const unsigned char* bits;   // item stream (BPDQ bits, trellis symbols, Leech planes)
  const uint2* vtab;           // BPDQ: [G][Rpad] 4 halves
  const uint32_t* table;       // trellis: 4096 half2
  const uint16_t* parity;      // Leech: [S][Rpad]
  const __half* x;             // [ntok][C]
  __half* y;                   // [ntok][R]  (nsplit == 1, BPDQ only)
  float* partial;              // [ntok][nsplit][Rpad]
  int R, C, Rpad, nrb, S, ntok, N, nsplit, ntile, nblock;
  int use_tma;                 // 0: x rows not 16-byte aligned, staged with element loads
};

constexpr uint32_t kHashHi = 0x9E37u << 16;     // trellis: (s*0x9E37 mod 2^16) in bits 16..31

// Per-format shape of a slice's K range: 32 chunks of 8 columns, plus, for
// Leech, 4 chunks carrying the parity term (A = parity bit of the blocks
// starting in the slice, B = their block sums of x split into fp16 hi + lo).
template <int FMT>
struct TcShape {
  static constexpr int kch = FMT == Q2_LEECH ? 36 : 32;
  static constexpr int kmma = kch / 2;                  // K = 16 steps per slice
  static constexpr int atoms = (kch + 7) / 8;           // 64-column swizzle atoms of B
  static constexpr uint32_t acols = kch * 4;            // TMEM columns of one A stage
  static constexpr int table = FMT == Q2_TRELLIS ? 4096 * 4 : 0;
  static constexpr int item = FMT == Q2_BPDQ ? Q2_ITEM_BYTES_BPDQ : FMT == Q2_TRELLIS ? Q2_ITEM_BYTES_TRL
                                                                                     : Q2_ITEM_BYTES_LEECH;
};
static_assert(kAcol0 + kStages * TcShape<Q2_LEECH>::acols <= kTmemCols, "A stages exceed TMEM");

// Shared-memory matrix descriptor (tcgen05) of a K-major operand with the
// 128-byte swizzle: start >> 4 in bits 0-13, leading byte offset field 1
// (not used by swizzled K-major layouts), stride byte offset 1024 >> 4 in
// 32-45 (8 rows x 128 bytes), version 1 in 46-47, base offset 0, swizzle
// mode 2 (128-byte) in 61-63.  A K step inside an atom adds its byte offset
// to the start address.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
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
// of the A row (column-byte = step / 4, four TMEM columns per column-byte);
// H is a template parameter so every window index is static.
template <int H>
__device__ __forceinline__ void trellis_part(const uint32_t (&W)[16], const uint32_t* tab, uint32_t ta) {
#pragma unroll
  for (int g = 0; g < kPartBytes / 4; ++g) {
    uint32_t e[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const int k = H * kPartBytes * 4 + g * 16 + t;
      const int n = 127 - k;
      const uint32_t f = __funnelshift_r(W[n >> 3], W[((n >> 3) + 1) & 15], 4 * (n & 7));
      e[t] = tab[(f * kHashHi) >> 20] ^ ((f & 1u) ? 0x80008000u : 0u);
    }
    tmem_st16(ta + (uint32_t)(H * kPartBytes + g * 4) * 4u, e);
  }
}

// BPDQ: column-bytes 16P .. 16P + 15 of one row (planes R0, R1 as loaded,
// lane-rotated) into TMEM columns 64P .. 64P + 63 at ta.
template <int P>
__device__ __forceinline__ void bpdq_part(const uint32_t (&R0)[8], const uint32_t (&R1)[8], int lane, uint32_t tlo,
                                          uint32_t thi, uint32_t ta) {
  uint32_t c0[4], c1[4];
  unrotate_half<P>(R0, lane, c0);
  unrotate_half<P>(R1, lane, c1);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const Codes4 c = codes4(c0[j], c1[j]);
    tmem_st16(ta + (uint32_t)(64 * P + 16 * j), decode_q<0>(c, tlo, thi), decode_q<1>(c, tlo, thi),
              decode_q<2>(c, tlo, thi), decode_q<3>(c, tlo, thi));
  }
}

// Leech: the same for the three sign/magnitude planes (values 2u).
template <int P>
__device__ __forceinline__ void leech_part(const uint32_t (&R0)[8], const uint32_t (&R1)[8], const uint32_t (&R2)[8],
                                           int lane, uint32_t ta) {
  uint32_t c0[4], c1[4], c2[4];
  unrotate_half<P>(R0, lane, c0);
  unrotate_half<P>(R1, lane, c1);
  unrotate_half<P>(R2, lane, c2);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const Codes4 c = codes4x3(c0[j], c1[j], c2[j]);
    tmem_st16(ta + (uint32_t)(64 * P + 16 * j), decode_leech_q<0>(c), decode_leech_q<1>(c), decode_leech_q<2>(c),
              decode_leech_q<3>(c));
  }
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1) k_tc(const __grid_constant__ TcArgs a) {
  using Sh = TcShape<FMT>;
  uint32_t* tab = reinterpret_cast<uint32_t*>(q2_smem);            // trellis table
  // kStages B buffers from the first 1024-byte boundary after the table
  const uint32_t sbase = saddr(q2_smem);
  unsigned char* B0 = q2_smem + (((sbase + Sh::table + 1023u) & ~1023u) - sbase);
  const int atom_bytes = a.N * 128;
  const int bbytes = Sh::atoms * atom_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(B0 + kStages * bbytes);
  uint64_t* empty = full + kStages;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(empty + kStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool producer = warp == kDecWarps;
  const int rbl = warp & 3, part = (warp >> 2) & 1;  // row block in tile (= TMEM lane quarter), half of the slice
  const int tile = blockIdx.x % a.ntile, split = blockIdx.x / a.ntile;
  const int sA = split * a.S / a.nsplit, sB = (split + 1) * a.S / a.nsplit;
  const int used = sB - sA;
  const int rb = tile * 4 + rbl;
  const bool valid = !producer && rb < a.nrb;        // the last tile may be ragged
  const int row = rb * 32 + lane;
  const int tile_rbs = min(4, a.nrb - tile * 4);

  if (threadIdx.x == 0) {
    for (int s = sA; s < sB; ++s)
      prefetch_l2(a.bits + ((size_t)s * a.nrb + tile * 4) * Sh::item, (size_t)tile_rbs * Sh::item);
    for (int st = 0; st < kStages; ++st) {
      mbar_init(saddr(&full[st]), kDecWarps + 1);
      mbar_init(saddr(&empty[st]), 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tslot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (FMT == Q2_TRELLIS)
    for (int i = threadIdx.x; i < 4096; i += kThreads) tab[i] = a.table[i];
  // zero the B buffers once: token rows past ntok of the Leech parity atom
  // (and of every atom when x is staged without TMA) stay zero
  for (int i = threadIdx.x; i < kStages * bbytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(B0)[i] = make_uint4(0, 0, 0, 0);
  fence_async_smem();

  // per-lane payload of one slice: the whole 512-byte chunks of the item at
  // this lane (BPDQ / Leech: chunk 2p + h = half h of plane p, lane-rotated;
  // trellis: the 64-byte packet); plus BPDQ's value table / Leech's parity
  constexpr int NP = FMT == Q2_LEECH ? 6 : 4;
  uint4 pl[NP], n1[NP];
  uint2 vt = make_uint2(0, 0), v1 = make_uint2(0, 0);
  uint32_t par = 0, p1 = 0;
  auto load = [&](int s, uint4 (&d)[NP], uint2& v, uint32_t& pw) {
    const unsigned char* ip = a.bits + ((size_t)s * a.nrb + rb) * Sh::item + lane * 16;
#pragma unroll
    for (int k = 0; k < NP; ++k) d[k] = __ldg(reinterpret_cast<const uint4*>(ip + k * 512));
    if (FMT == Q2_BPDQ) v = a.vtab[(size_t)s * a.Rpad + row];
    if (FMT == Q2_LEECH) pw = a.parity[(size_t)s * a.Rpad + row];
  };
#pragma unroll
  for (int k = 0; k < NP; ++k) pl[k] = n1[k] = make_uint4(0, 0, 0, 0);
  if (valid && used > 0) load(sA, pl, vt, par);
  if (valid && used > 1) load(sA + 1, n1, v1, p1);
  pdl_wait();
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tlane = tmem + ((uint32_t)(rbl * 32) << 16);     // this warp's lane quarter
  bool ok = true;

  if (producer) {
    // ---- x copies and MMAs (the MMAs and TMA copies are issued by lane 0)
    const uint32_t idesc = idesc_f16(kRows, a.N);
    auto produce = [&](int i) {                      // x of slice sA + i into stage i % kStages
      const int st = i % kStages, s = sA + i;
      const uint32_t fb = saddr(&full[st]);
      unsigned char* Bs = B0 + st * bbytes;
      if (a.use_tma) {
        if (lane == 0) {
          mbar_expect_tx(fb, 4u * (uint32_t)atom_bytes);
#pragma unroll
          for (int at = 0; at < 4; ++at) tma_load_2d(saddr(Bs + at * atom_bytes), &a.xmap, s * 256 + 64 * at, 0, fb);
        }
      } else {
        // x rows not 16-byte aligned: element loads by the warp's 32 lanes
        for (int e = lane; e < a.ntok * 32; e += 32) {
          const int n = e >> 5, kc = e & 31, c0 = s * 256 + kc * 8;
          uint4 v = make_uint4(0, 0, 0, 0);
          __half* hv = reinterpret_cast<__half*>(&v);
          for (int k = 0; k < 8; ++k)
            if (c0 + k < a.C) hv[k] = a.x[(size_t)n * a.C + c0 + k];
          *reinterpret_cast<uint4*>(Bs + (kc >> 3) * atom_bytes + n * 128 + (((kc & 7) ^ (n & 7)) << 4)) = v;
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(fb);
      }
    };
    for (int i = 0; i < min(kStages, used); ++i) produce(i);
    int issued = 0;
    for (int i = 0; i < used; ++i) {
      const int st = i % kStages;
      if (!__all_sync(~0u, mbar_wait(saddr(&full[st]), (uint32_t)(i / kStages) & 1u))) {
        ok = false;
        if (lane == 0) atomicExch(&q2_tc_error, 3u);
        break;
      }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t bs = saddr(B0 + st * bbytes);
        const uint32_t at = tmem + kAcol0 + (uint32_t)st * Sh::acols;
#pragma unroll
        for (int k = 0; k < Sh::kmma; ++k)
          mma_f16_ta(tmem, at + (uint32_t)(k * 8), sdesc_sw128(bs + (k >> 2) * atom_bytes + (k & 3) * 32), idesc,
                     (i > 0 || k > 0) ? 1u : 0u);
        mma_commit(saddr(&empty[st]));
      }
      __syncwarp();
      issued = i + 1;
      // refill the stage of slice i - 1 (its MMAs precede slice i's) with slice i - 1 + kStages
      const int j = i - 1 + kStages;
      if (i >= 1 && j < used) {
        if (!__all_sync(~0u, mbar_wait(saddr(&empty[(i - 1) % kStages]), (uint32_t)((i - 1) / kStages) & 1u))) {
          ok = false;
          if (lane == 0) atomicExch(&q2_tc_error, 4u);
          break;
        }
        produce(j);
      }
    }
    // the last commit covers every MMA issued; on an error, also give the
    // copies in flight time to land before the CTA exits
    if (issued > 0 && !mbar_wait(saddr(&empty[(issued - 1) % kStages]), (uint32_t)((issued - 1) / kStages) & 1u)) {
      ok = false;
      if (lane == 0) atomicExch(&q2_tc_error, 5u);
    }
    if (!ok) sleep_us(50);
  } else {
    // ---- decode into TMEM
    for (int i = 0; i < used; ++i) {
      const int s = sA + i, st = i % kStages;
      uint4 n2[NP];
      uint2 v2 = make_uint2(0, 0);
      uint32_t p2 = 0;
#pragma unroll
      for (int k = 0; k < NP; ++k) n2[k] = make_uint4(0, 0, 0, 0);
      if (valid && i + 2 < used) load(s + 2, n2, v2, p2);
      // stage st is free once the MMAs of slice i - kStages have completed
      if (i >= kStages && !__all_sync(~0u, mbar_wait(saddr(&empty[st]), (uint32_t)(i / kStages - 1) & 1u))) {
        ok = false;
        if (lane == 0) atomicExch(&q2_tc_error, 6u);
        break;
      }
      tc_fence_after();
      const uint32_t ta = tlane + kAcol0 + (uint32_t)st * Sh::acols;
      if (FMT == Q2_TRELLIS) {
        const uint32_t W[16] = {pl[0].x, pl[0].y, pl[0].z, pl[0].w, pl[1].x, pl[1].y, pl[1].z, pl[1].w,
                                pl[2].x, pl[2].y, pl[2].z, pl[2].w, pl[3].x, pl[3].y, pl[3].z, pl[3].w};
        if (part == 0) trellis_part<0>(W, tab, ta);
        else trellis_part<1>(W, tab, ta);
      } else if (FMT == Q2_BPDQ) {
        const uint32_t tlo = __byte_perm(vt.x, vt.y, 0x6420u);
        const uint32_t thi = __byte_perm(vt.x, vt.y, 0x7531u);
        const uint32_t R0[8] = {pl[0].x, pl[0].y, pl[0].z, pl[0].w, pl[1].x, pl[1].y, pl[1].z, pl[1].w};
        const uint32_t R1[8] = {pl[2].x, pl[2].y, pl[2].z, pl[2].w, pl[3].x, pl[3].y, pl[3].z, pl[3].w};
        if (part == 0) bpdq_part<0>(R0, R1, lane, tlo, thi, ta);
        else bpdq_part<1>(R0, R1, lane, tlo, thi, ta);
      } else {
        const uint32_t R0[8] = {pl[0].x, pl[0].y, pl[0].z, pl[0].w, pl[1].x, pl[1].y, pl[1].z, pl[1].w};
        const uint32_t R1[8] = {pl[2].x, pl[2].y, pl[2].z, pl[2].w, pl[3].x, pl[3].y, pl[3].z, pl[3].w};
        const uint32_t R2[8] = {pl[4].x, pl[4].y, pl[4].z, pl[4].w, pl[5].x, pl[5].y, pl[5].z, pl[5].w};
        if (part == 0) {
          leech_part<0>(R0, R1, R2, lane, ta);
          // parity columns (K 256..287, TMEM columns 128..143): A = 1.0 where
          // the block starting in this slice is odd, once for the hi and
          // once for the lo part of the block sums
          uint32_t pv[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t lo = ((par >> (2 * q)) & 1u) ? 0x3C00u : 0u;
            const uint32_t hi = ((par >> (2 * q + 1)) & 1u) ? 0x3C000000u : 0u;
            pv[q] = lo | hi;
          }
          const uint4 q0 = make_uint4(pv[0], pv[1], pv[2], pv[3]), q1 = make_uint4(pv[4], pv[5], pv[6], pv[7]);
          tmem_st16(ta + 128u, q0, q1, q0, q1);
        } else {
          leech_part<1>(R0, R1, R2, lane, ta);
        }
        // B side of the parity columns (atom 4): block sums of x for the
        // blocks starting in this slice, hi part at K 256 + jb, lo part
        // (sum - hi) at K 272 + jb
        const int bfirst = (s * 256 + 23) / 24;
        const int blast = min(a.nblock - 1, (s * 256 + 256 + 23) / 24 - 1);
        const int nbk = max(0, blast - bfirst + 1);
        unsigned char* Bp = B0 + st * bbytes + 4 * atom_bytes;
        for (int e = threadIdx.x; e < a.ntok * 16; e += kDecWarps * 32) {
          const int n = e >> 4, jb = e & 15;
          float xsum = 0.f;
          if (jb < nbk) {
            const __half* xp = a.x + (size_t)n * a.C + (size_t)(bfirst + jb) * 24;
            if (a.use_tma) {                         // 48-byte blocks of 16-byte aligned rows
              const uint4* xv = reinterpret_cast<const uint4*>(xp);
#pragma unroll
              for (int k = 0; k < 3; ++k) {
                const uint4 r = __ldg(xv + k);
                const __half2* h2 = reinterpret_cast<const __half2*>(&r);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                  const float2 f = __half22float2(h2[m]);
                  xsum += f.x + f.y;
                }
              }
            } else {
              for (int k = 0; k < 24; ++k) xsum += __half2float(xp[k]);
            }
          }
          const __half hi = __float2half_rn(xsum);
          const __half lo = __float2half_rn(xsum - __half2float(hi));
          unsigned char* rp = Bp + n * 128 + (jb & 7) * 2;
          *reinterpret_cast<__half*>(rp + ((((jb >> 3) + 0) ^ (n & 7)) << 4)) = hi;
          *reinterpret_cast<__half*>(rp + ((((jb >> 3) + 2) ^ (n & 7)) << 4)) = lo;
        }
        fence_async_smem();
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(saddr(&full[st]));
#pragma unroll
      for (int k = 0; k < NP; ++k) {
        pl[k] = n1[k];
        n1[k] = n2[k];
      }
      vt = v1;
      v1 = v2;
      par = p1;
      p1 = p2;
    }
    // the accumulator is final once the last slice's commit has arrived
    if (ok && warp < 4 && used > 0 &&
        !__all_sync(~0u, mbar_wait(saddr(&empty[(used - 1) % kStages]), (uint32_t)((used - 1) / kStages) & 1u))) {
      ok = false;
      if (lane == 0) atomicExch(&q2_tc_error, 2u);
    }
  }
  ok = __syncthreads_and(ok);
  tc_fence_after();
  if (warp < 4 && ok) {
    const int orow = (tile * 4 + warp) * 32 + lane;
    for (int c0 = 0; c0 < a.N; c0 += 16) {
      float v[16];
      tmem_ld16(tlane + (uint32_t)c0, v);
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
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

// cuTensorMapEncodeTiled from the driver, looked up once (null if absent).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      (void)cudaGetLastError();
      p = nullptr;
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// Tensor map of x [ntok][C] fp16 for the B tiles: box of 64 columns (128
// bytes, the swizzle span) x N token rows, rows past ntok and columns past C
// read as zero.  False when the rows are not 16-byte aligned or the driver
// refuses the map; the kernel then stages x with element loads.
bool encode_x_map(CUtensorMap* map, const void* x, int C, int ntok, int N) {
  if (C % 8 || (reinterpret_cast<uintptr_t>(x) & 15)) return false;
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)ntok};
  const cuuint64_t strides[1] = {(cuuint64_t)C * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)N};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
  a.use_tma = encode_x_map(&a.xmap, x, d.C, ntok, a.N) ? 1 : 0;
  // table, 1024-byte alignment slack, kStages B buffers, 2 x kStages mbarriers, TMEM slot
  const int smem = max(kOneCtaSmem, Sh::table + 1024 + kStages * Sh::atoms * a.N * 128 + 2 * kStages * 8 + 16);
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
