// Skinny-GEMM path on the 5th-generation tensor cores (tcgen05) for
// 2..64 tokens (padded to N = 16, 32, 48 or 64): decode once per tile,
// multiply for every token.  The dense fp16 control runs through the same
// kernel with plain row loads in place of a decode.
//
// A CTA owns 128 output rows (four 32-row blocks) and a range of 256-column
// slices, and runs them through rings of stages with three roles:
//   - 16 decoder warps (four per 32-row block, each a quarter of the slice's
//     columns) turn the packed weights into fp16 in registers (BPDQ through
//     the per-(group, row) 4-entry value table, one byte permute per two or
//     four weights) and store them into tensor memory with tcgen05.st, one
//     TMEM lane per row: the slice's A, in one of kStagesA TMEM stages;
//   - a helper warp copies the x tile of all tokens into one of kStagesB
//     shared-memory stages with four 2D TMA copies (the slice's B), waits
//     until a slice's A and B are complete, and hands the slice to
//   - the MMA warp, whose lane 0 issues sixteen tcgen05.mma.kind::f16
//     (M = 128, N, K = 16) reading A from TMEM and B from shared memory into
//     one fp32 accumulator in TMEM, and commits them to the stages' "empty"
//     mbarriers, which free the stages for refilling.
// The handoff is a named barrier with a flag reduction, not a memory
// access: any memory access by the issuing thread waits for its queue of
// MMAs to drain and leaves the tensor core idle (about 350 cycles per
// access on GB300), so the MMA lane touches no memory at all.
// At the end the decoder warps copy the accumulator (fp32, 128 rows x N)
// into shared memory.  A tile split over K runs as one thread-block cluster
// of its nsplit CTAs: each sums a share of the tile's rows over the
// cluster's partials through distributed shared memory, in split order, so
// the result does not depend on which CTA finished first; no global
// atomics, no workspace and no second launch.  The same pass applies the
// format's row epilogue (trellis: x scale; Leech: exceptions, scale, tail)
// and writes y.
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
// A TMEM store writes the same columns in every lane, so each lane undoes
// its rotation: the word part through per-lane load addresses, the byte
// part with a funnel shift.
//
// Every wait is bounded: a wait that runs out records an error code in
// q2_tc_error (read back with q2_device_errors) and the kernel skips the
// rest of its work; the helper warp waits for the outstanding copies and
// MMAs before the CTA frees its TMEM columns.
#include <cuda.h>
#include <cmath>
#include <algorithm>
#include <mutex>
#include <vector>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "q2_common.cuh"

extern __shared__ __align__(1024) unsigned char q2_smem[];

__device__ unsigned int q2_tc_error = 0;
// Poll limit of the helper warp's stage waits (decoded A and x tile of a
// slice ready), 0 = the normal bound.  Set only by q2_debug_wait_limit, so
// that a test can make these waits run out and check the error path.
__device__ long long q2_tc_stage_wait_limit = 0;

namespace q2 {
namespace {

constexpr int kDecWarps = 16;                 // decoder warps
constexpr int kMmaWarp = kDecWarps;           // lane 0 issues the MMAs
constexpr int kHelperWarp = kDecWarps + 1;    // waits on the stage barriers, issues the x copies
constexpr int kThreads = (kDecWarps + 2) * 32;
constexpr int kStagesA = 3;                   // slices in flight in TMEM (decoded A)
constexpr int kStagesB = 4;                   // slices in flight in shared memory (x tiles)
constexpr int kGroup = 2;                     // slices per handoff to the MMA warp
static_assert(kStagesB % kGroup == 0 && kStagesB / kGroup == 2, "B stages are freed a group at a time");
constexpr int kParts = kDecWarps / 4;         // warps per 32-row block, each decoding 256/kParts columns
constexpr int kPartBytes = 32 / kParts;       // column-bytes of one plane per lane and part
constexpr int kPartWords = kPartBytes / 4;    // canonical 32-bit words of one plane per lane and part
constexpr int kRows = 128;                    // M of the MMA
constexpr int kMaxSplit = 8;                  // K splits of a tile at most: the portable cluster size
constexpr int kPf16Ahead = 3;                 // fp16 control: slices of rows fetched into L2 ahead
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

// Lane un-rotation.  Lane l = 4a + r stores its 32-byte plane row rotated:
// rotated byte j holds column-byte (j + l) mod 32, so canonical word c
// starts at rotated byte 4(c - a) - r.  A lane decoding canonical words
// c0 .. c0 + n - 1 loads the n + 1 rotated words L[t] = R[(c0 - 1 + t - a)
// mod 8] (the word rotation is in the load addresses, see rot_word_offset)
// and joins neighbours with a funnel shift by 32 - 8r (clamped: r = 0 takes
// the high word whole).
__device__ __forceinline__ uint32_t unrot(uint32_t lo, uint32_t hi, uint32_t sh) { return __funnelshift_rc(lo, hi, sh); }

// Byte offset, inside the lane's part of an item (after lane * 16), of
// rotated word w of plane q: half w / 4 of the plane is chunk 2q + w / 4.
__device__ __forceinline__ int rot_word_offset(int q, int w) { return (2 * q + (w >> 2)) * 512 + (w & 3) * 4; }

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
  const __half* w16;           // fp16 control: [R][C]
  const uint16_t* parity;      // Leech: [S][Rpad]
  const __half* x;             // [ntok][C]
  __half* y;                   // [ntok][R]
  int R, C, Rpad, nrb, S, ntok, N, nsplit, ntile, nblock;
  int use_tma;                 // 0: x rows not 16-byte aligned, staged with element loads
  // Per-row finish after the K sum (the reduction kernel's epilogue before):
  // trellis x scale_r; Leech + 16 x[col] for each v = +8 exception, x scale_r
  // * post (1/sqrt(8)), + the fp16 tail dot product ("Tetra", section 5.1:
  // the row scale after the block dot product, then the unquantised tail)
  const __half* scale;         // [R] or null
  float post;
  const __half* tail;          // Leech [Rpad][tailpad]
  int tail_n, tailpad, tail_col0;
  const uint32_t* excptr;      // Leech [Rpad + 1] (empty lists for the offset-binary layout)
  const uint32_t* exccol;
};

// Distributed shared memory: this CTA's shared address in CTA `rank` of the
// cluster, and a 16-byte load from it (ordered against writes by the
// cluster barriers around the reads).
__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t saddr_local, uint32_t rank) {
  uint32_t remote;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(saddr_local), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(remote));
  return v;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t saddr_local, uint32_t rank) {
  uint32_t remote;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(saddr_local), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote));
  return v;
}
// Every thread of every CTA of the cluster: writes before it are visible to
// reads after it, cluster-wide.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

constexpr uint32_t kHashHi = 0x9E37u << 16;     // trellis: (s*0x9E37 mod 2^16) in bits 16..31

// Per-format shape of a slice's K range: 32 chunks of 8 columns.  OFF4: the
// Leech offset-binary layout (four planes).
template <int FMT, bool OFF4 = false>
struct TcShape {
  static constexpr int kch = 32;
  static constexpr int kmma = kch / 2;                  // K = 16 steps per slice
  static constexpr int atoms = (kch + 7) / 8;           // 64-column swizzle atoms of B
  static constexpr uint32_t acols = kch * 4;            // TMEM columns of one A stage
  // trellis: the codebook; fp16 control: each decoder warp's 4 KB transpose tile
  static constexpr int table = FMT == Q2_TRELLIS ? 4096 * 4 : FMT == Q2_FP16 ? kDecWarps * 4096 : 0;
  static constexpr int item = FMT == Q2_BPDQ ? Q2_ITEM_BYTES_BPDQ : FMT == Q2_TRELLIS ? Q2_ITEM_BYTES_TRL
                              : FMT == Q2_FP16 ? 0 : OFF4 ? Q2_ITEM_BYTES_LEECH4 : Q2_ITEM_BYTES_LEECH;
  static constexpr int planes = FMT == Q2_BPDQ ? 2 : FMT == Q2_LEECH ? (OFF4 ? 4 : 3) : 0;
};
static_assert(kAcol0 + kStagesA * TcShape<Q2_LEECH>::acols <= kTmemCols, "A stages exceed TMEM");

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

// v = p + 2u = p + 2*(b0 + 2*b1 - 4*b2) in fp16 for the 8 columns of byte
// Q, p being the parity bit of the block the byte lies in (a block is three
// column-bytes, so a byte never straddles two).  Every value in -8..7 has a
// zero low byte in fp16, so only high bytes are looked up, from the table
// of the byte's parity.
template <int Q>
__device__ __forceinline__ uint4 decode_leech_q(const Codes4& c, uint32_t p) {
  // fp16 high bytes of p + (0, 2, 4, 6, -8, -6, -4, -2) (code 0..7)
  const uint32_t HA = p ? 0x4745423Cu : 0x46444000u, HB = p ? 0xBCC2C5C7u : 0xC0C4C6C8u;
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

// Offset-binary Leech (four planes): v = p + 2c - 8 for the code
// c = b0 + 2 b1 + 4 b2 + 8 b3 in 0..8 and the byte's block parity p.  The
// low three bits index the fp16 high bytes of p + (-8, -6, ..., 6); c = 8
// (v = +8, rare, p = 0) has low bits 0, so its -8 is turned into +8 by
// flipping the sign bit of each column whose plane-3 bit is set (byte q3 of
// plane 3 for these 8 columns).
template <int Q>
__device__ __forceinline__ uint4 decode_leech4_q(const Codes4& c, uint32_t q3, uint32_t p) {
  // fp16 high bytes of p + (-8, -6, -4, -2, 0, 2, 4, 6) (code 0..7)
  const uint32_t HA = p ? 0xBCC2C5C7u : 0xC0C4C6C8u, HB = p ? 0x4745423Cu : 0x46444000u;
  constexpr uint32_t sel = (uint32_t)Q | ((4u + Q) << 4);
  const uint32_t s0 = __byte_perm(c.ea, c.oa, sel);   // codes of cols 0,4,1,5
  const uint32_t s1 = __byte_perm(c.eb, c.ob, sel);   // cols 2,6,3,7
  const uint32_t h0 = __byte_perm(HA, HB, s0), h1 = __byte_perm(HA, HB, s1);
  uint4 r;
  r.x = __byte_perm(h0, 0u, 0x2404u);       // cols 0,1: [0, h(c0), 0, h(c1)]
  r.y = __byte_perm(h1, 0u, 0x2404u);       // cols 2,3
  r.z = __byte_perm(h0, 0u, 0x3414u);       // cols 4,5
  r.w = __byte_perm(h1, 0u, 0x3414u);       // cols 6,7
  if (q3) {                                 // column i's sign bit: bit 15 (even i) or 31 (odd i) of word i / 2
    r.x ^= ((q3 & 0x01u) << 15) | ((q3 & 0x02u) << 30);
    r.y ^= ((q3 & 0x04u) << 13) | ((q3 & 0x08u) << 28);
    r.z ^= ((q3 & 0x10u) << 11) | ((q3 & 0x20u) << 26);
    r.w ^= ((q3 & 0x40u) << 9) | ((q3 & 0x80u) << 24);
  }
  return r;
}

// Trellis: the 32 steps of one part of a segment (column-bytes 8H .. 8H + 7
// of the A row, four TMEM columns per column-byte).  Lw holds the part's
// window of the lane's 16 symbol words, Lw[t] = W[(12 - 4H + t) mod 16]:
// step 32H + kk reads words ((127 - kk) >> 3) - 12 and the next one of Lw,
// indices that do not depend on H.
__device__ __forceinline__ void trellis_part(const uint32_t (&Lw)[5], const uint32_t* tab, uint32_t ta) {
#pragma unroll
  for (int g = 0; g < kPartBytes / 4; ++g) {
    uint32_t e[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const int kk = g * 16 + t;
      const int n = 127 - kk;
      const uint32_t f = __funnelshift_r(Lw[(n >> 3) - 12], Lw[(n >> 3) - 11], 4 * (n & 7));
      e[t] = tab[(f * kHashHi) >> 20] ^ ((f & 1u) ? 0x80008000u : 0u);
    }
    tmem_st16(ta + (uint32_t)(g * 16), e);
  }
}

// BPDQ: the part's kPartBytes column-bytes of one row from the loaded
// rotated words of planes 0 and 1, into TMEM columns from ta.
__device__ __forceinline__ void bpdq_part(const uint32_t (&L0)[kPartWords + 1], const uint32_t (&L1)[kPartWords + 1],
                                          uint32_t sh, uint32_t tlo, uint32_t thi, uint32_t ta) {
#pragma unroll
  for (int j = 0; j < kPartWords; ++j) {
    const Codes4 c = codes4(unrot(L0[j], L0[j + 1], sh), unrot(L1[j], L1[j + 1], sh));
    tmem_st16(ta + (uint32_t)(16 * j), decode_q<0>(c, tlo, thi), decode_q<1>(c, tlo, thi), decode_q<2>(c, tlo, thi),
              decode_q<3>(c, tlo, thi));
  }
}

// Leech: the same for the three sign/magnitude planes (values p + 2u); bit
// k of pm is the parity of the part's column-byte k.
__device__ __forceinline__ void leech_part(const uint32_t (&L0)[kPartWords + 1], const uint32_t (&L1)[kPartWords + 1],
                                           const uint32_t (&L2)[kPartWords + 1], uint32_t sh, uint32_t ta,
                                           uint32_t pm) {
#pragma unroll
  for (int j = 0; j < kPartWords; ++j) {
    const Codes4 c = codes4x3(unrot(L0[j], L0[j + 1], sh), unrot(L1[j], L1[j + 1], sh), unrot(L2[j], L2[j + 1], sh));
    const uint32_t pb = pm >> (4 * j);
    tmem_st16(ta + (uint32_t)(16 * j), decode_leech_q<0>(c, pb & 1u), decode_leech_q<1>(c, pb & 2u),
              decode_leech_q<2>(c, pb & 4u), decode_leech_q<3>(c, pb & 8u));
  }
}

// Offset-binary Leech: the part from its four planes (values p + 2c - 8).
__device__ __forceinline__ void leech4_part(const uint32_t (&L0)[kPartWords + 1], const uint32_t (&L1)[kPartWords + 1],
                                            const uint32_t (&L2)[kPartWords + 1], const uint32_t (&L3)[kPartWords + 1],
                                            uint32_t sh, uint32_t ta, uint32_t pm) {
#pragma unroll
  for (int j = 0; j < kPartWords; ++j) {
    const Codes4 c = codes4x3(unrot(L0[j], L0[j + 1], sh), unrot(L1[j], L1[j + 1], sh), unrot(L2[j], L2[j + 1], sh));
    const uint32_t w3 = unrot(L3[j], L3[j + 1], sh);
    const uint32_t pb = pm >> (4 * j);
    tmem_st16(ta + (uint32_t)(16 * j), decode_leech4_q<0>(c, w3 & 0xFFu, pb & 1u),
              decode_leech4_q<1>(c, (w3 >> 8) & 0xFFu, pb & 2u), decode_leech4_q<2>(c, (w3 >> 16) & 0xFFu, pb & 4u),
              decode_leech4_q<3>(c, w3 >> 24, pb & 8u));
  }
}

// Named barrier 1 between the MMA warp and the helper warp, with an AND of a
// flag: no memory access, so the MMA lane's queue of tensor-core
// instructions is not drained by the handoff.
__device__ __forceinline__ bool handoff(bool in) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, 1, 64, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(in ? 1u : 0u)
      : "memory");
  return r != 0;
}

template <int FMT, bool OFF4>
__global__ void __launch_bounds__(kThreads, 1) k_tc(const __grid_constant__ TcArgs a) {
  using Sh = TcShape<FMT, OFF4>;
  uint32_t* tab = reinterpret_cast<uint32_t*>(q2_smem);            // trellis table
  // kStagesB B buffers from the first 1024-byte boundary after the table
  const uint32_t sbase = saddr(q2_smem);
  unsigned char* B0 = q2_smem + (((sbase + Sh::table + 1023u) & ~1023u) - sbase);
  const int atom_bytes = a.N * 128;
  const int bbytes = Sh::atoms * atom_bytes;
  uint64_t* fullA = reinterpret_cast<uint64_t*>(B0 + kStagesB * bbytes);   // decoder arrivals
  uint64_t* emptyA = fullA + kStagesA;                                      // MMA commits
  uint64_t* fullB = emptyA + kStagesA;                                      // TMA bytes
  uint64_t* emptyG = fullB + kStagesB;        // MMA commits per group: the group's B stages are free
  uint32_t* tslot = reinterpret_cast<uint32_t*>(emptyG + 2);
  // set by the first role whose wait runs out: the others stop waiting on
  // each other (the drains of copies and MMAs in flight keep their full bound)
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool decoder = warp < kDecWarps;
  const int rbl = warp & 3, part = (warp >> 2) & (kParts - 1);   // row block in tile (= TMEM lane quarter), part of the slice
  // the K splits of a tile are consecutive CTAs, one thread-block cluster
  // (split = the CTA's rank in it)
  const int tile = blockIdx.x / a.nsplit, split = blockIdx.x % a.nsplit;
  const int sA = split * a.S / a.nsplit, sB = (split + 1) * a.S / a.nsplit;
  const int used = sB - sA;
  const int rb = tile * 4 + rbl;
  const bool valid = decoder && rb < a.nrb;          // the last tile may be ragged
  const int row = rb * 32 + lane;
  const int tile_rbs = min(4, a.nrb - tile * 4);

  if (threadIdx.x == 0) {
    if (Sh::item)        // the packed formats: the CTA's whole range (a few KB per slice)
      for (int s = sA; s < sB; ++s)
        prefetch_l2(a.bits + ((size_t)s * a.nrb + tile * 4) * Sh::item, (size_t)tile_rbs * Sh::item);
    for (int st = 0; st < kStagesA; ++st) {
      mbar_init(saddr(&fullA[st]), kDecWarps);
      mbar_init(saddr(&emptyA[st]), 1);
    }
    for (int st = 0; st < kStagesB; ++st) mbar_init(saddr(&fullB[st]), 1);
    for (int st = 0; st < 2; ++st) mbar_init(saddr(&emptyG[st]), 1);
    *abort_flag = 0;
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
  // zero the B stages when x is staged without TMA (token rows past ntok
  // stay zero); the TMA fills whole boxes itself
  if (!a.use_tma)
    for (int st = 0; st < kStagesB; ++st)
      for (int i = threadIdx.x * 16; i < bbytes; i += kThreads * 16)
        *reinterpret_cast<uint4*>(B0 + st * bbytes + i) = make_uint4(0, 0, 0, 0);
  fence_async_smem();

  // Decoder payload of one slice: the rotated words this lane's part needs
  // (BPDQ / Leech: kPartWords + 1 per plane; trellis: a 5-word window of the
  // 64-byte symbol packet), at per-lane offsets fixed for the whole kernel;
  // plus BPDQ's value table / Leech's parity words.
  constexpr int NPL = Sh::planes;
  // (fp16 control: nothing is held ahead; the rows are read when the slice is stored)
  constexpr int NW = FMT == Q2_TRELLIS ? 5 : FMT == Q2_FP16 ? 1 : NPL * (kPartWords + 1);
  int off[NW];
  {
    const int aa = lane >> 2;
    if (FMT == Q2_TRELLIS) {
#pragma unroll
      for (int t = 0; t < 5; ++t) {
        const int w = (12 - 4 * part + t) & 15;
        off[t] = (w >> 2) * 512 + (w & 3) * 4;
      }
    } else {
#pragma unroll
      for (int q = 0; q < NPL; ++q)
#pragma unroll
        for (int t = 0; t <= kPartWords; ++t)
          off[q * (kPartWords + 1) + t] = rot_word_offset(q, (kPartWords * part - 1 + t - aa) & 7);
    }
  }
  uint32_t pl[NW], n1[NW];
  uint2 vt = make_uint2(0, 0), v1 = make_uint2(0, 0);
  uint32_t par = 0, p1 = 0;
  // fp16 control: the warp's 32 rows x the part's 64 columns of slice s,
  // read as whole 128-byte row segments (load k: rows 4k .. 4k + 3 of the
  // block, lane l the 16-byte chunk l % 8 of row 4k + l / 8; zeros past R
  // and C, C being a multiple of 8), one slice held ahead of the one being
  // stored.  A load touching 32 rows (one per lane) keeps 32 lines in flight
  // per instruction and was measured at 0.4 of HBM; these keep 4.
  uint4 fcur[FMT == Q2_FP16 ? 8 : 1], fnext[FMT == Q2_FP16 ? 8 : 1];
  auto load16 = [&](int s, uint4* w) {
    const int c = s * 256 + part * 64 + (lane & 7) * 8;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int r = rb * 32 + 4 * k + (lane >> 3);
      w[k] = (valid && r < a.R && c < a.C) ? ldg_stream(a.w16 + (size_t)r * a.C + c) : make_uint4(0, 0, 0, 0);
    }
  };
  // ... and the rows' 512-byte segments of slice s fetched into L2 ahead of
  // the register loads (by the part-0 warps, one lane per row), kPf16Ahead
  // slices ahead of the slice being stored, so the register loads hit L2
  auto prefetch16 = [&](int s) {
    if (part == 0 && valid && row < a.R && s * 256 < a.C)
      prefetch_l2(a.w16 + (size_t)row * a.C + (size_t)s * 256, (size_t)min(256, a.C - s * 256) * 2);
  };
  if constexpr (FMT == Q2_FP16) {
    for (int j = 1; j <= kPf16Ahead && j < used; ++j) prefetch16(sA + j);
    if (used > 0) load16(sA, fcur);
  }
  auto load = [&](int s, uint32_t (&d)[NW], uint2& v, uint32_t& pw) {
    if (FMT == Q2_FP16) return;
    const unsigned char* ip = a.bits + ((size_t)s * a.nrb + rb) * Sh::item + lane * 16;
#pragma unroll
    for (int t = 0; t < NW; ++t) d[t] = __ldg(reinterpret_cast<const uint32_t*>(ip + off[t]));
    if (FMT == Q2_BPDQ) v = a.vtab[(size_t)s * a.Rpad + row];
    // Leech: the parity bits of the blocks starting in slice s, and in the
    // high half those of slice s - 1 (its last block may reach into slice s)
    if (FMT == Q2_LEECH)
      pw = (uint32_t)a.parity[(size_t)s * a.Rpad + row] |
           (s > 0 ? (uint32_t)a.parity[(size_t)(s - 1) * a.Rpad + row] << 16 : 0u);
  };
#pragma unroll
  for (int t = 0; t < NW; ++t) pl[t] = n1[t] = 0;
  if (valid && used > 0) load(sA, pl, vt, par);
  if (valid && used > 1) load(sA + 1, n1, v1, p1);
  // Programmatic dependent launch: only x and y depend on the kernel before
  // this one on the stream, so the helper waits for it (griddepcontrol.wait)
  // just before it first copies x, and every thread before the epilogue
  // writes y.  The weights are decoded into TMEM meanwhile: a CTA
  // that lands on an SM freed early has its first slices decoded when the
  // previous kernel completes.
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tlane = tmem + ((uint32_t)(rbl * 32) << 16);     // this warp's lane quarter
  bool ok = true;

  if (warp == kMmaWarp) {
    // ---- MMAs: one handoff per group of kGroup slices, then lane 0 issues
    // and commits (per slice for its A stage, per group for its B stages)
    const uint32_t idesc = idesc_f16(kRows, a.N);
    for (int g = 0; g * kGroup < used; ++g) {
      ok = handoff(ok);
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
          const int i = g * kGroup + u;
          if (i < used) {
            const int sa = i % kStagesA, sb = i % kStagesB;
            const uint32_t bs = saddr(B0 + sb * bbytes);
            const uint32_t at = tmem + kAcol0 + (uint32_t)sa * Sh::acols;
#pragma unroll
            for (int k = 0; k < Sh::kmma; ++k)
              mma_f16_ta(tmem, at + (uint32_t)(k * 8), sdesc_sw128(bs + (k >> 2) * atom_bytes + (k & 3) * 32), idesc,
                         (i > 0 || k > 0) ? 1u : 0u);
            mma_commit(saddr(&emptyA[sa]));
          }
        }
        mma_commit(saddr(&emptyG[g & 1]));
      }
      __syncwarp();
    }
  } else if (warp == kHelperWarp) {
    // ---- stage barriers and x copies (TMA issued by lane 0)
    auto produce = [&](int i) {                      // x of slice sA + i into B stage i % kStagesB
      const int sb = i % kStagesB, s = sA + i;
      const uint32_t fb = saddr(&fullB[sb]);
      unsigned char* Bs = B0 + sb * bbytes;
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
    const long long stage_limit = q2_tc_stage_wait_limit > 0 ? q2_tc_stage_wait_limit : kSpinLimit;
    pdl_wait();                                      // x is the previous kernel's output
    int produced = min(kStagesB, used), waitedB = 0;   // slices whose x copy was issued / seen complete
    for (int i = 0; i < produced; ++i) produce(i);
    int handed = 0;
    for (int g = 0; g * kGroup < used; ++g) {
      bool ready = true;
#pragma unroll
      for (int u = 0; u < kGroup; ++u) {
        const int i = g * kGroup + u;
        if (ready && i < used) {
          ready = mbar_wait(saddr(&fullA[i % kStagesA]), (uint32_t)(i / kStagesA) & 1u, stage_limit);
          ready = ready && mbar_wait(saddr(&fullB[i % kStagesB]), (uint32_t)(i / kStagesB) & 1u, stage_limit);
          if (__all_sync(~0u, ready)) waitedB = i + 1;
        }
      }
      if (!__all_sync(~0u, ready)) {
        ok = false;
        if (lane == 0) {
          atomicExch(&q2_tc_error, 3u);
          *abort_flag = 1;
        }
      }
      tc_fence_before();
      ok = handoff(ok);
      if (!ok) break;
      handed = min(used, (g + 1) * kGroup);
      // refill the B stages of group g - 1 (its MMAs precede group g's) with the slices kStagesB later
      const int j0 = (g - 1) * kGroup + kStagesB;
      if (g >= 1 && j0 < used) {
        if (!__all_sync(~0u, mbar_wait(saddr(&emptyG[(g - 1) & 1]), (uint32_t)((g - 1) >> 1) & 1u, kSpinLimit,
                                       abort_flag))) {
          ok = false;
          if (lane == 0) {
            atomicExch(&q2_tc_error, 4u);
            *abort_flag = 1;
          }
        }
        if (ok)
          for (int u = 0; u < kGroup && j0 + u < used; ++u) {
            produce(j0 + u);
            produced = j0 + u + 1;
          }
      }
    }
    // on an error, wait (with the full bound) for every x copy still in
    // flight, so that none lands in shared memory after the CTA has exited
    if (!ok)
      for (int i = waitedB; i < produced; ++i)
        (void)mbar_wait(saddr(&fullB[i % kStagesB]), (uint32_t)(i / kStagesB) & 1u);
    // the last commit covers every MMA issued; on an error, also give the
    // copies in flight time to land before the CTA exits
    if (handed > 0 &&
        !mbar_wait(saddr(&emptyA[(handed - 1) % kStagesA]), (uint32_t)((handed - 1) / kStagesA) & 1u)) {
      ok = false;
      if (lane == 0) atomicExch(&q2_tc_error, 5u);
    }
    if (!ok) sleep_us(50);
  } else {
    // ---- decoders: slice i into A stage i % kStagesA
    const uint32_t sh = 32u - 8u * (uint32_t)(lane & 3);
    for (int i = 0; i < used; ++i) {
      const int s = sA + i, sa = i % kStagesA;
      uint32_t n2[NW];
      uint2 v2 = make_uint2(0, 0);
      uint32_t p2 = 0;
#pragma unroll
      for (int t = 0; t < NW; ++t) n2[t] = 0;
      if (valid && i + 2 < used) load(s + 2, n2, v2, p2);
      if constexpr (FMT == Q2_FP16) {
        if (i + 1 + kPf16Ahead < used) prefetch16(s + 1 + kPf16Ahead);
        if (i + 1 < used) load16(s + 1, fnext);
      }
      // the stage is free once the MMAs of slice i - kStagesA have completed
      if (i >= kStagesA &&
          !__all_sync(~0u, mbar_wait(saddr(&emptyA[sa]), (uint32_t)(i / kStagesA - 1) & 1u, kSpinLimit, abort_flag))) {
        ok = false;
        if (lane == 0) {
          atomicExch(&q2_tc_error, 6u);
          *abort_flag = 1;
        }
        break;
      }
      tc_fence_after();
      const uint32_t ta = tlane + kAcol0 + (uint32_t)sa * Sh::acols + (uint32_t)(32 * part);
      if (FMT == Q2_FP16) {
        // transpose through the warp's shared-memory tile (row r at 128 r,
        // chunk c at 16 (c ^ r % 8): conflict-free both ways) so that lane r
        // holds row r's 64 columns, then store them as they are
        unsigned char* tt = q2_smem + warp * 4096;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int r = 4 * k + (lane >> 3), c = lane & 7;
          *reinterpret_cast<uint4*>(tt + r * 128 + ((c ^ (r & 7)) << 4)) = fcur[k];
        }
        __syncwarp();
        uint4 w[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) w[c] = *reinterpret_cast<const uint4*>(tt + lane * 128 + ((c ^ (lane & 7)) << 4));
        __syncwarp();
        tmem_st16(ta, w[0], w[1], w[2], w[3]);
        tmem_st16(ta + 16u, w[4], w[5], w[6], w[7]);
#pragma unroll
        for (int k = 0; k < 8; ++k) fcur[k] = fnext[k];
      } else if (FMT == Q2_TRELLIS) {
        const uint32_t Lw[5] = {pl[0], pl[1], pl[2], pl[3], pl[4]};
        trellis_part(Lw, tab, ta);
      } else if (FMT == Q2_BPDQ) {
        const uint32_t tlo = __byte_perm(vt.x, vt.y, 0x6420u);
        const uint32_t thi = __byte_perm(vt.x, vt.y, 0x7531u);
        uint32_t L0[kPartWords + 1], L1[kPartWords + 1];
#pragma unroll
        for (int t = 0; t <= kPartWords; ++t) {
          L0[t] = pl[t];
          L1[t] = pl[kPartWords + 1 + t];
        }
        bpdq_part(L0, L1, sh, tlo, thi, ta);
      } else {
        uint32_t L0[kPartWords + 1], L1[kPartWords + 1], L2[kPartWords + 1];
#pragma unroll
        for (int t = 0; t <= kPartWords; ++t) {
          L0[t] = pl[t];
          L1[t] = pl[kPartWords + 1 + t];
          L2[t] = pl[2 * (kPartWords + 1) + t];
        }
        // The parity of each of the part's 8 column-bytes.  Byte GB of the
        // row lies in block GB / 3; blocks from bf on start in slice s (low
        // half of par), block bf - 1 in slice s - 1 (high half).  With
        // P = (bit of block bf - 1) | (slice s's bits << 1), the part's
        // first byte q lies in block q / 3 and its 8 bytes in blocks
        // q / 3 .. q / 3 + 3: take those 4 bits, widen each to the 3 bytes
        // of its block and drop the q % 3 bytes before q.
        const int q = s * 32 + part * kPartBytes, bf = (s * 32 + 2) / 3;
        const int bfp = s > 0 ? ((s - 1) * 32 + 2) / 3 : 0;
        const uint32_t P = ((par >> (16 + bf - 1 - bfp)) & 1u) | ((par & 0xFFFFu) << 1);
        const uint32_t B = (P >> (q / 3 - bf + 1)) & 0xFu;
        const uint32_t E = (B & 1u) * 7u | (B & 2u) * 28u | (B & 4u) * 112u | (B & 8u) * 448u;
        const uint32_t pm = (E >> (q % 3)) & 0xFFu;
        if constexpr (OFF4) {
          uint32_t L3[kPartWords + 1];
#pragma unroll
          for (int t = 0; t <= kPartWords; ++t) L3[t] = pl[(NPL - 1) * (kPartWords + 1) + t];
          leech4_part(L0, L1, L2, L3, sh, ta, pm);
        } else {
          leech_part(L0, L1, L2, sh, ta, pm);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(saddr(&fullA[sa]));
#pragma unroll
      for (int t = 0; t < NW; ++t) {
        pl[t] = n1[t];
        n1[t] = n2[t];
      }
      vt = v1;
      v1 = v2;
      par = p1;
      p1 = p2;
    }
    // the accumulator is final once the last slice's commit has arrived
    if (ok && warp < 4 && used > 0 &&
        !__all_sync(~0u, mbar_wait(saddr(&emptyA[(used - 1) % kStagesA]), (uint32_t)((used - 1) / kStagesA) & 1u,
                                   kSpinLimit, abort_flag))) {
      ok = false;
      if (lane == 0) {
        atomicExch(&q2_tc_error, 2u);
        *abort_flag = 1;
      }
    }
  }
  pdl_wait();                                        // before anything writes y (returns at once if done)
  ok = __syncthreads_and(ok);
  tc_fence_after();
  // ---- epilogue.  (1) The accumulator, or NaN where a bounded wait ran out,
  // into this CTA's partial P [token][128 rows] fp32, over the B stages (all
  // MMAs have completed): warp w reads TMEM lane quarter w % 4 (the lanes a
  // warp may access) and token columns 16 (w / 4) + 64 j.
  float* P = reinterpret_cast<float*>(B0);
  if (decoder)
    for (int c0 = 16 * (warp >> 2); c0 < a.N; c0 += 16 * (kDecWarps / 4)) {
      float v[16];
      if (ok && used > 0) {
        tmem_ld16(tlane + (uint32_t)c0, v);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(0x7FC00000u);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) P[(c0 + i) * kRows + rbl * 32 + lane] = v[i];
    }
  __syncthreads();
  // (2) With a K split, the tile's CTAs form a cluster: after a cluster
  // barrier CTA `split` sums its share of the rows over the cluster's
  // partials through distributed shared memory, in split order (the result
  // does not depend on which CTA finished first), finishes and writes y; a
  // second barrier keeps every partial readable until all shares are done.
  // Without a split the CTA finishes all 128 rows from its own partial.
  const int CS = a.nsplit;
  if (CS > 1) cluster_sync();
  if constexpr (FMT == Q2_LEECH) {
    // Leech: one row per element (its finish, exceptions and the tail dot
    // product, is a chain of loads per row); CTA `split` takes rows
    // [split * 128 / CS, (split + 1) * 128 / CS)
    const int r0 = split * kRows / CS, nr = (split + 1) * kRows / CS - r0;
    const uint32_t pbase = saddr(P);
    for (int e = threadIdx.x; e < nr * a.ntok; e += kThreads) {
      const int t = e / nr, rl = r0 + (e - t * nr);
      const int row = tile * kRows + rl;
      if (row >= a.R) continue;
      float v;
      if (CS == 1) {
        v = P[t * kRows + rl];
      } else {
        // every partial's load in flight, then the sum in split order
        float pv[kMaxSplit];
        const uint32_t off = pbase + (uint32_t)(t * kRows + rl) * 4u;
#pragma unroll
        for (int q = 0; q < kMaxSplit; ++q)
          if (q < CS) pv[q] = ld_cluster_f32(off, (uint32_t)q);
        v = pv[0];
#pragma unroll
        for (int q = 1; q < kMaxSplit; ++q)
          if (q < CS) v += pv[q];
      }
      const __half* xt = a.x + (size_t)t * a.C;
      for (uint32_t k = a.excptr[row]; k < a.excptr[row + 1]; ++k) v = fmaf(16.f, __half2float(xt[a.exccol[k]]), v);
      v *= __half2float(a.scale[row]) * a.post;
      for (int c = 0; c < a.tail_n; ++c)
        v = fmaf(__half2float(a.tail[(size_t)row * a.tailpad + c]), __half2float(xt[a.tail_col0 + c]), v);
      a.y[(size_t)t * a.R + row] = __float2half_rn(v);
    }
  } else {
    // rows in groups of 4 (one float4 of every partial per token); CTA
    // `split` takes groups [split * 32 / CS, (split + 1) * 32 / CS)
    const int g0 = split * (kRows / 4) / CS, ng = (split + 1) * (kRows / 4) / CS - g0;
    const uint32_t pbase = saddr(P);
    for (int e = threadIdx.x; e < ng * a.ntok; e += kThreads) {
      const int t = e / ng, rl = 4 * (g0 + (e - t * ng));
      const int row0 = tile * kRows + rl;
      if (row0 >= a.R) continue;
      float4 v;
      if (CS == 1) {
        v = *reinterpret_cast<const float4*>(P + t * kRows + rl);
      } else {
        float4 pv[kMaxSplit];
        const uint32_t off = pbase + (uint32_t)(t * kRows + rl) * 4u;
#pragma unroll
        for (int q = 0; q < kMaxSplit; ++q)
          if (q < CS) pv[q] = ld_cluster_f32x4(off, (uint32_t)q);
        v = pv[0];
#pragma unroll
        for (int q = 1; q < kMaxSplit; ++q)
          if (q < CS) {
            v.x += pv[q].x;
            v.y += pv[q].y;
            v.z += pv[q].z;
            v.w += pv[q].w;
          }
      }
      float f[4] = {v.x, v.y, v.z, v.w};
      if (FMT == Q2_TRELLIS) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (row0 + j < a.R) f[j] *= __half2float(a.scale[row0 + j]);
      }
      __half* yp = a.y + (size_t)t * a.R + row0;
      if ((a.R & 3) == 0) {                      // 8-byte aligned, all four rows inside R
        const __half2 lo = __floats2half2_rn(f[0], f[1]), hi = __floats2half2_rn(f[2], f[3]);
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t*>(&lo);
        u.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(yp) = u;
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (row0 + j < a.R) yp[j] = __float2half_rn(f[j]);
      }
    }
  }
  if (CS > 1) cluster_sync();
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

// The K split of the tensor-core launch.  One CTA per SM at a time, so the
// makespan is (waves of tiles) x (slices per CTA + the CTA's fixed cost in
// slice times): about 1 us from the previous kernel's end to the wait
// release, 2 us until the first pair of slices is decoded and handed to the
// MMA warp, and about 1 us of drain and epilogue, against about 1 us per
// slice (globaltimer traces on GB300), so kSplitOverhead = 4.  A split tile's
// CTAs run as one cluster, so a wave holds as many tiles as clusters of that
// size fit on the device at once (cudaOccupancyMaxActiveClusters: clusters
// live inside one GPC).  At most kMaxSplit = 8 splits, the portable cluster
// size.
constexpr int kSplitOverhead = 4;

// 256-column slices of the tensor-core launch (the fp16 control's last one
// may be partial)
int tc_slices(const q2_blob_header& d) { return d.fmt == Q2_FP16 ? (d.C + Q2_SLICE - 1) / Q2_SLICE : d.nslice; }

std::mutex g_cl_mu;
struct ClusterFit {
  int dev;
  const void* fn;
  int smem, cs, n;
};
std::vector<ClusterFit> g_cl;

// Clusters of `cs` CTAs of `fn` (kThreads threads, `smem` bytes each) that
// fit on the current device at once (cached).
int max_clusters(const void* fn, int smem, int cs) {
  if (cs == 1) return dev_info().sms;
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lk(g_cl_mu);
    for (const ClusterFit& c : g_cl)
      if (c.dev == dev && c.fn == fn && c.smem == smem && c.cs == cs) return c.n;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  std::lock_guard<std::mutex> lk(g_cl_mu);
  g_cl.push_back({dev, fn, smem, cs, n});
  return n;
}

int tc_nsplit(const q2_blob_header& d, const void* fn, int smem) {
  const int ntile = (d.Rpad + kRows - 1) / kRows, S = tc_slices(d);
  long best = -1;
  int nsplit = 1;
  for (int ns = 1; ns <= std::min(S, kMaxSplit); ++ns) {
    const int per_wave = max_clusters(fn, smem, ns);
    if (per_wave < 1) continue;
    const long waves = (ntile + per_wave - 1) / per_wave;
    const long cost = waves * ((S + ns - 1) / ns + kSplitOverhead);
    if (best < 0 || cost < best) {
      best = cost;
      nsplit = ns;
    }
  }
  return nsplit;
}

// Packed formats and the fp16 control at 2..64 tokens on the tensor cores
// (tokens padded to a multiple of 16), one launch: the K split is summed
// inside it and every format's epilogue applied there.
template <int FMT, bool OFF4 = false>
int launch_tc(const q2_handle* h, const void* x, void* y, int ntok, void* stream) {
  using Sh = TcShape<FMT, OFF4>;
  const q2_blob_header& d = h->hdr;
  TcArgs a = {};
  a.post = 1.f;
  if (FMT == Q2_FP16) {
    a.w16 = reinterpret_cast<const __half*>(h->dev + d.off[SEC_FP16_W]);
  } else if (FMT == Q2_BPDQ) {
    a.bits = h->dev + d.off[SEC_BPDQ_BITS];
    a.vtab = reinterpret_cast<const uint2*>(h->dev + d.off[SEC_BPDQ_VTAB]);
  } else if (FMT == Q2_TRELLIS) {
    a.bits = h->dev + d.off[SEC_TRL_STREAM];
    a.table = reinterpret_cast<const uint32_t*>(h->dev + d.off[SEC_TRL_TABLE]);
    a.scale = reinterpret_cast<const __half*>(h->dev + d.off[SEC_TRL_SCALE]);
  } else {
    a.bits = h->dev + d.off[SEC_LEECH_PLANES];
    a.parity = reinterpret_cast<const uint16_t*>(h->dev + d.off[SEC_LEECH_PARITY]);
    a.nblock = d.nblock;
    a.scale = reinterpret_cast<const __half*>(h->dev + d.off[SEC_LEECH_SCALE]);
    a.post = d.inv_sqrt8;
    a.tail = reinterpret_cast<const __half*>(h->dev + d.off[SEC_LEECH_TAIL]);
    a.tail_n = d.tail;
    a.tailpad = d.tailpad;
    a.tail_col0 = d.nblock * 24;
    a.excptr = reinterpret_cast<const uint32_t*>(h->dev + d.off[SEC_LEECH_EXCPTR]);
    a.exccol = reinterpret_cast<const uint32_t*>(h->dev + d.off[SEC_LEECH_EXCCOL]);
  }
  a.x = static_cast<const __half*>(x);
  a.y = static_cast<__half*>(y);
  a.R = d.R;
  a.C = d.C;
  a.Rpad = d.Rpad;
  a.nrb = q2_nrb(d);
  a.S = tc_slices(d);
  a.ntok = ntok;
  a.N = (ntok + 15) / 16 * 16;
  a.ntile = (d.Rpad + kRows - 1) / kRows;
  a.use_tma = encode_x_map(&a.xmap, x, d.C, ntok, a.N) ? 1 : 0;
  // table (or transpose tiles), 1024-byte alignment slack, B buffers (the
  // partial sums reuse them), the mbarriers, TMEM slot and abort flag
  const int smem =
      max(kOneCtaSmem, Sh::table + 1024 + kStagesB * Sh::atoms * a.N * 128 + (2 * kStagesA + kStagesB + 2) * 8 + 16);
  const void* fn = reinterpret_cast<const void*>(k_tc<FMT, OFF4>);
  if (set_smem(fn, smem)) return Q2_ECUDA;
  a.nsplit = tc_nsplit(d, fn, smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.ntile * a.nsplit);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = a.nsplit;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.nsplit > 1 ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, k_tc<FMT, OFF4>, a) != cudaSuccess) {
    (void)cudaGetLastError();
    return Q2_ECUDA;
  }
  return cudaGetLastError() == cudaSuccess ? Q2_OK : Q2_ECUDA;
}

}  // namespace
}  // namespace q2

// Workspace bytes of a tensor-core launch: none (the K split is summed in
// distributed shared memory).
extern "C" size_t q2_tc_workspace_bytes(const q2_handle*, int) { return 0; }

extern "C" int q2_tc_fp16(const q2_handle* h, const void* x, void* y, int ntok, void* stream) {
  return q2::launch_tc<Q2_FP16>(h, x, y, ntok, stream);
}
extern "C" int q2_tc_bpdq(const q2_handle* h, const void* x, void* y, int ntok, void* stream) {
  return q2::launch_tc<Q2_BPDQ>(h, x, y, ntok, stream);
}
extern "C" int q2_tc_trellis(const q2_handle* h, const void* x, void* y, int ntok, void* stream) {
  return q2::launch_tc<Q2_TRELLIS>(h, x, y, ntok, stream);
}
extern "C" int q2_tc_leech(const q2_handle* h, const void* x, void* y, int ntok, void* stream) {
  if (h->hdr.layout == Q2_LEECH_OFFSET4) return q2::launch_tc<Q2_LEECH, true>(h, x, y, ntok, stream);
  return q2::launch_tc<Q2_LEECH, false>(h, x, y, ntok, stream);
}

// Test hook: the poll limit of the tensor-core kernel's stage waits (0 = the
// normal bound), on the current device.
extern "C" int q2_debug_wait_limit(long long polls) {
  if (polls < 0) return Q2_EINVAL;
  return cudaMemcpyToSymbol(q2_tc_stage_wait_limit, &polls, sizeof(polls)) == cudaSuccess ? Q2_OK : Q2_ECUDA;
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
