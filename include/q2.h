/*
 * q2.h -- C ABI of the fused dequantize-plus-matvec library for packed
 * ~2-bit weights on GB300 (sm_103a).
 *
 * The operation is y = W x for a packed weight matrix W with R output rows
 * and C input columns, called once per projection ("Unfolding the Leech
 * Lattice", introduction: a fused dequantize-plus-matvec, decode-phase GEMV
 * at batch 1; "Qwen3-8B -- 2-bit BPDQ (packed)", Kernels: one kernel per
 * matmul, tile shape picked per batch size).  x holds ntok token vectors,
 * fp16 row-major [ntok][C]; y is fp16 row-major [ntok][R]; accumulation is
 * fp32.  The weights stay packed and are never expanded to dense fp16.
 *
 * Formats:
 *   Q2_FP16      dense fp16 control.
 *   Q2_BPDQ      two bit-planes, w = c0*b0 + c1*b1 + off per (256-column
 *                group, row) ("Qwen3-8B -- 2-bit BPDQ (packed)", Format).
 *   Q2_TRELLIS   bitshift trellis, L=16, T=4, V=2, 4096x2 fp16 table
 *                codebook, fp16 row scale, restart every 256 columns
 *                ("Qwen3.8-27B on a 12 GB card", "A trellis is a codebook
 *                you walk").
 *   Q2_LEECH     Leech-lattice blocks of 24 weights, w = scale_r * v / sqrt(8),
 *                fp16 tail for the last C % 24 columns ("Unfolding the Leech
 *                Lattice", introduction and section 2; "Tetra", section 5.1).
 *   Q2_NOWEIGHTS launch-geometry control: same grid, table build and
 *                reduction as the BPDQ kernel, reads no weight bytes
 *                ("Unfolding the Leech Lattice", contribution C4).
 *
 * Conventions (all entry points):
 *   - Return Q2_OK (0) or a negative Q2_E* status; nothing aborts, nothing
 *     throws across the ABI.  q2_strerror() names a status.
 *   - Host pointers are read during the call only.  Device pointers stay
 *     owned by the caller; the library allocates no device memory.
 *   - Packers are two-phase: call with out == NULL to get *out_bytes, then
 *     with a buffer of that size.
 */
#ifndef Q2_H
#define Q2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  Q2_FP16 = 0,
  Q2_BPDQ = 1,
  Q2_TRELLIS = 2,
  Q2_LEECH = 3,
  Q2_NOWEIGHTS = 4
} q2_fmt;

enum {
  Q2_OK = 0,
  Q2_EINVAL = -1,      /* null pointer or bad scalar argument            */
  Q2_ESHAPE = -2,      /* R, C outside what the format accepts            */
  Q2_EALIGN = -3,      /* x, y or the device blob not 16-byte aligned     */
  Q2_EFMT = -4,        /* fmt does not match the handle                    */
  Q2_ENTOK = -5,       /* ntok outside 1..64                               */
  Q2_EBLOB = -6,       /* blob header corrupt or wrong version            */
  Q2_EWORKSPACE = -7,  /* no workspace bound, or smaller than needed       */
  Q2_ECUDA = -8,       /* a CUDA call or kernel launch failed              */
  Q2_ENOMEM = -9,      /* host allocation failed                           */
  Q2_ESIZE = -10,      /* caller's buffer smaller than required            */
  Q2_ESCRATCH = -11    /* problem too large for the built-in scratch       */
};

typedef struct q2_handle q2_handle;   /* opaque; owns no device memory */
typedef struct CUstream_st* q2_stream; /* a cudaStream_t; NULL = legacy default stream */

#define Q2_MAX_NTOK 64

/* ------------------------------------------------------------------ packers
 * Offline packers: canonical host arrays in, self-describing host blob out
 * (header + sections, each 256-byte aligned).  The blob can be written to a
 * file and bound later; its device copy must be byte-identical.
 */

/* Dense fp16 control.  w: fp16 bits [R][C] row-major.  C % 8 == 0. */
int q2_pack_fp16(const uint16_t* w, int R, int C, void* out, size_t* out_bytes);

/* BPDQ ("Qwen3-8B -- 2-bit BPDQ (packed)", Format: w[r,c] = sum_i
 * coeffs[g(c),r,i] * bit_i(r,c) + coeffs[g(c),r,msbits], group 256).
 * plane0, plane1: [R][C/8] bytes, bit i (LSB first) of byte j = column 8j+i.
 * coef: fp16 bits [C/256][R][3] = (c0, c1, off).  C % 256 == 0, R >= 1.
 * The 2-bit code of a weight is b0 | b1 << 1. */
int q2_pack_bpdq(const uint8_t* plane0, const uint8_t* plane1, const uint16_t* coef,
                 int R, int C, void* out, size_t* out_bytes);

/* Bitshift trellis ("Qwen3.8-27B on a 12 GB card": state = last L bits;
 * each step shifts T bits in and emits V weights).  stream: [R][C/256][64]
 * bytes, byte i of a segment = symbol 2i (low nibble) and 2i+1 (high
 * nibble).  table: fp16 bits [4096][2].  scale: fp16 bits [R].  The state of
 * step k is t[k-3]<<12 | t[k-2]<<8 | t[k-1]<<4 | t[k] (indices modulo 128
 * inside the segment); its row is ((s*0x9E37) & 0xFFFF) >> 4; bit 0 of the
 * state negates both weights.  C % 256 == 0. */
int q2_pack_trellis(const uint8_t* stream, const uint16_t* table, const uint16_t* scale,
                    int R, int C, void* out, size_t* out_bytes);

/* Leech lattice ("Unfolding the Leech Lattice": blocks of 24 weights, each a
 * lattice point; unfolded offline into a bit-plane layout whose bits per
 * weight read from memory are a design axis, section 3 and contribution
 * C2).  v: int8 [R][C/24][24] lattice points, |v_i| <= 8 with all
 * coordinates of a block of one parity; tail: fp16 bits [R][C%24]; scale:
 * fp16 bits [R].  Any C with C >= 24 is accepted; inv_sqrt8 is the fp32
 * factor applied with the row scale (the caller passes 1/sqrt(8) rounded to
 * fp32).  Layouts, both with a parity bit p per block:
 *   Q2_LEECH_PLANES3: three two's-complement planes of u = (v - p)/2, so
 *     v = p + 2 b0 + 4 b1 - 8 b2; v = +8 (rare at shells 2..6) is stored as
 *     -8 and listed in an exception side channel.  About 3.07 bpw read.
 *   Q2_LEECH_OFFSET4: four planes of the offset-binary code c = (v - p)/2 + 4
 *     (0..8), v = p - 8 + 2 b0 + 4 b1 + 8 b2 + 16 b3; no exceptions.  About
 *     4.07 bpw read.
 * Anything else returns Q2_EINVAL. */
#define Q2_LEECH_PLANES3 0
#define Q2_LEECH_OFFSET4 1
int q2_pack_leech(const int8_t* v, const uint16_t* tail, const uint16_t* scale,
                  int R, int C, float inv_sqrt8, int layout, void* out, size_t* out_bytes);

/* No-weights control: a header only. */
int q2_pack_noweights(int R, int C, void* out, size_t* out_bytes);

/* ------------------------------------------------------------------ binding
 * blob_host: the packed blob (read now); blob_dev: its device copy, 256-byte
 * aligned, kept alive by the caller while the handle is used.  Returns a
 * handle that holds pointers into blob_dev only. */
int q2_bind(const void* blob_host, const void* blob_dev, q2_handle** h);
void q2_unbind(q2_handle* h);

/* Split-K workspace: device memory owned by the caller, 256-byte aligned.
 * The CUDA-core paths (BPDQ at 1..6 tokens, trellis and Leech at 1 token)
 * use its first ntok x Rpad 64-bit words as split-K accumulators: each
 * 256-column slice's partial sum of a row is added as a fixed-point integer
 * together with an arrival count, in one atomic, and the addition that
 * completes the count writes y and resets the word.  These words must be
 * zero when the workspace is first used (allocate it zero-filled); every
 * completed call leaves them at zero again (a call whose x holds an inf or
 * NaN too: its outputs are NaN).  The tensor-core path (2..64 tokens) uses
 * no workspace: a K split's CTAs run as one thread-block cluster and sum
 * their fp32 partials in distributed shared memory.  One workspace may serve
 * many handles whose calls are ordered on one stream; calls that overlap on
 * the GPU must use different workspaces.  Limits: R <= 524288 rows; on the
 * CUDA-core paths C <= 255 x 256 columns.  The size depends on the path a
 * token count takes, so it is not monotone in ntok: a workspace for every
 * call up to N tokens is the largest q2_workspace_bytes over ntok = 1..N. */
int q2_workspace_bytes(const q2_handle* h, int ntok, size_t* bytes);
int q2_set_workspace(q2_handle* h, void* ws_dev, size_t ws_bytes);

/* Format, shape and algorithmic bytes read from HBM per call at ntok tokens
 * (weights and side data; x and y not included). */
int q2_info(const q2_handle* h, int* fmt, int* R, int* C);
int q2_bytes(const q2_handle* h, int ntok, size_t* weight_bytes_read_per_call);

/* ------------------------------------------------------------------ compute
 * y = W x ("Unfolding the Leech Lattice", introduction).  x: device fp16
 * [ntok][C]; y: device fp16 [ntok][R]; both 16-byte aligned; 1 <= ntok <= 64.
 * Asynchronous and ordered on `stream`; never synchronises.  Needs the
 * workspace of q2_workspace_bytes(h, ntok) bound first (0 bytes for fp16 at
 * one token).  The dense fp16 control runs one token on CUDA cores and
 * 2..64 tokens through the tensor-core kernel, loading its rows as they are.
 * The packed formats at 1 token, and BPDQ at 2..6 tokens, run on CUDA cores
 * in launches that reduce their split-K partial sums themselves, through the
 * workspace's fixed-point accumulator words (integer sums: the result does
 * not depend on the order in which slices arrive).  BPDQ at 3..6 tokens runs
 * its tokens in pairs plus a single-token launch, stream-ordered; every
 * token's BPDQ result at 1..6 tokens is bit-identical whatever the batch.
 * Leech at 2 tokens runs two single-token launches when C and R are
 * multiples of 8.  The tensor-core path (7..64 tokens, or 2..64 for trellis
 * and the other Leech cases) is one launch: a tile's K splits (at most 8,
 * one thread-block cluster) add their fp32 partials in split order, so the
 * result does not depend on which finished first, and the same pass applies
 * the format's row epilogue (trellis: scale; Leech: exceptions, scale,
 * tail).  The fixed-point scale 2^F of the CUDA-core paths is chosen per
 * matrix from its largest weight magnitude so that no fp16 x can overflow
 * it; each term then carries an absolute rounding error of at most
 * 2^-(F+1), about 2e-8 per 256-column slice for weights of magnitude
 * 0.05.  An inf or NaN in a token's x makes that token's outputs NaN (the
 * IEEE result is non-finite for every row; the fixed-point sums carry a
 * sticky flag for it).  Launches use programmatic dependent launch: weights are
 * fetched before the previous kernel on the stream has finished; x, y and
 * the workspace are touched only after it has.  Returns Q2_ECUDA if a
 * launch fails. */
int q2_gemv(q2_fmt fmt, const q2_handle* h, const void* x, void* y, int ntok, q2_stream stream);

/* A decode step's chain of GEMVs: for i = 0..n-1, y[i] = W_i x[i] with W_i
 * the packed matrix of h[i] (format fmt[i]), all at ntok tokens, launched in
 * order on `stream` exactly as n q2_gemv calls would be (each launch reads
 * x[i] only after the launch before it has finished, so x[i+1] may be
 * computed from y[i] by the caller's own kernels in between, or be y[i]).
 * The difference is the weight stream: on the CUDA-core paths (BPDQ at
 * 1..6 tokens, trellis and Leech at 1 token) launch i also fetches the
 * weights of GEMV i + lookahead (launch 0: GEMVs 1..lookahead; lookahead
 * 0..4) from HBM into L2, each of its CTAs a 1/grid share, so that every
 * GEMV's weights are requested once, `lookahead` launches before its own,
 * and those bytes arrive while the
 * launches before them run their latency-bound parts (the wait for the
 * previous launch, staging x, building the slice tables, the split-K
 * atomics).  This is the cross-matmul prefetch of "Qwen3-8B -- 2-bit BPDQ
 * (packed)", Kernels (at up to 8 tokens a second stream loads each weight
 * matrix into L2 two matmuls ahead of its use, paced by a progress flag);
 * here the launch order itself paces it, so nothing waits on a flag.
 * Results are bit-identical to the same q2_gemv calls.  Every handle needs
 * its workspace as for q2_gemv (handles may share one workspace: the calls
 * are ordered).  All handles and pointers are checked before anything is
 * launched; a launch failure returns its status with the launches before
 * it already enqueued.  lookahead == 0 is exactly n q2_gemv calls. */
int q2_gemv_chain(int n, const q2_fmt* fmt, q2_handle* const* h, const void* const* x, void* const* y, int ntok,
                  int lookahead, q2_stream stream);

/* Allocation-free y = W x for a BPDQ handle at one token (no counterpart on
 * the source pages; an addition of this library).  For callers that cannot
 * allocate device memory when they run the GEMV: code running under CUDA
 * stream capture, plugins whose host framework owns the device memory, and
 * real-time loops that must not call the allocator.  It does what q2_gemv
 * does at ntok == 1, but keeps the split-K accumulator words in a scratch
 * array
 * that the library owns (a file-scope __device__ array of
 * Q2_NOALLOC_SCRATCH_BYTES = 1 MiB, held on every GPU that loads the
 * library until the process exits) instead of a workspace bound with
 * q2_set_workspace.  It calls no cudaMalloc or cudaFree.
 *   - x: device fp16 [C]; y: device fp16 [R]; both 16-byte aligned.
 *   - Needs Rpad * 8 bytes (one word per row, R rounded up to 32), so R up
 *     to 131072; larger problems return Q2_ESCRATCH.  Every Qwen3-8B and
 *     -14B linear fits.
 *   - The first call on a device looks up the scratch's device address
 *     (cudaGetSymbolAddress, once per device); make that first call before
 *     any stream capture.
 *   - All calls in a process share the one scratch array of a GPU: two
 *     calls that can run at the same time on that GPU (streams with no
 *     ordering between them) race and corrupt each other's results, so
 *     order them on one stream.  The words are zero when the library loads
 *     and every completed call leaves them at zero. */
#define Q2_NOALLOC_SCRATCH_BYTES (1024 * 1024)
int q2_gemv_bpdq_noalloc(const q2_handle* h, const void* x, void* y, q2_stream stream);

/* Debug decode to the canonical form (all formats but Q2_NOWEIGHTS):
 *   fp16:    fp16 [R][C]
 *   BPDQ:    fp16 [R][C], one round-to-nearest-even of c0*b0 + c1*b1 + off
 *   trellis: fp32 [R][C], float(scale_r) * float(sign * table value)
 *   Leech:   int8 [R][24*(C/24)] lattice coordinates, then fp16 [R][C%24]
 *            tail at byte offset R*24*(C/24) rounded up to 16.
 * out: device buffer of q2_decode_bytes() bytes. */
int q2_decode_bytes(const q2_handle* h, size_t* bytes);
int q2_decode(const q2_handle* h, void* out_dev, q2_stream stream);

/* ------------------------------------------------------------------ rotation
 * Activation rotation ahead of the GEMV ("Qwen3.8-27B on a 12 GB card",
 * section "What the kernel does per token"): weights stored in a rotated
 * basis need their input rotated at run time, per token,
 *     x_rot = (H (x) Q)(S x),   C = nh * nq,
 * with S the column signs, Q an nq x nq orthogonal matrix acting on every
 * run of nq consecutive columns, and H the orthonormal Sylvester
 * Walsh-Hadamard transform, H[i][j] = (-1)^popcount(i & j) / sqrt(nh),
 * acting across the runs: entry (i*nq + a, j*nq + b) of H (x) Q is
 * H[i][j] * Q[a][b].  Computed in fp32, rounded once to fp16.
 *   - x, x_rot: device fp16 [ntok][C], distinct buffers; 1 <= ntok <= 64.
 *   - nh a power of two, C a multiple of nh, nq = C / nh <= 32,
 *     C <= Q2_ROT_MAX_C; otherwise Q2_ESHAPE.
 *   - signs: device uint8 [ceil(C/8)]; bit c % 8 of byte c / 8 set means
 *     column c is negated.
 *   - q: device fp32 [nq][nq] row-major; may be NULL only when nq == 1
 *     (Q = [1]).
 *   - Asynchronous on `stream`, launched like q2_gemv (x is read only after
 *     the previous kernel on the stream has finished).  One CTA per token.
 * q2_rotate_split gives the split the page's examples follow: nh = 2048
 * when 2048 divides C, else 1024 (5120 = 5 x 1024, 6144 = 3 x 2048,
 * 17408 = 17 x 1024); Q2_ESHAPE if C is not a multiple of it. */
#define Q2_ROT_MAX_C 49152
int q2_rotate(const void* x, void* x_rot, int ntok, int C, int nh, const void* signs, const float* q,
              q2_stream stream);
int q2_rotate_split(int C, int* nh, int* nq);

/* Device-side error word of the tensor-core (multi-token) kernels, then
 * cleared: 0 in normal operation; nonzero means a bounded wait on the
 * tensor core ran out and the kernel skipped its work (the rows of the tiles
 * concerned are NaN).  Before such a kernel's CTA exits it waits, with the
 * full bound, for its copies and MMAs in flight, and it still meets the
 * other CTAs of its cluster at both of their barriers.  Synchronous: reads
 * device memory of the current device. */
int q2_device_errors(unsigned int* out);

/* Test hook, not for production use: limits the tensor-core kernel's stage
 * waits (the helper warp's wait for a slice's decoded weights and x tile) to
 * `polls` polls on the current device (0 restores the normal bound), so a
 * test can make them run out and check the error path above without
 * faulting or hanging the GPU.  Synchronous.  Q2_EINVAL for polls < 0. */
int q2_debug_wait_limit(long long polls);

const char* q2_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* Q2_H */
