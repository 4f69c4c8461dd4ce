// Blob header and device layouts shared by the host packers and the kernels.
#pragma once
#include <stdint.h>
#include <stddef.h>

#define Q2_MAGIC 0x31423251u   // "Q2B1"
#define Q2_VERSION 2u
#define Q2_ROWS 32             // rows per lane-group (one warp, one row per lane)
#define Q2_SLICE 256           // columns per group / segment / slice
#define Q2_ITEM_BYTES_BPDQ 2048   // 32 lanes x (2 planes x 32 bytes)
#define Q2_ITEM_BYTES_TRL 2048    // 32 lanes x 64 bytes of symbols
#define Q2_ITEM_BYTES_LEECH 3072  // 32 lanes x (3 planes x 32 bytes)
#define Q2_ITEM_BYTES_LEECH4 4096 // 32 lanes x (4 planes x 32 bytes): offset-binary layout
#define Q2_MAX_SECTIONS 8

// Workspace layout.  The CUDA-core paths (1..6 tokens) keep one 64-bit
// accumulator per (token, row) at offset 0: [ntok][Rpad] words, zero between
// calls (see q2_b1.cu).  The tensor-core path (2..64 tokens) needs none: it
// sums its K splits in distributed shared memory.
#define Q2_MAX_ROWS 524288
#define Q2_MAX_ACC_TOK 6
#define Q2_MAX_SPLIT 255          // count field of the accumulator word

// Section indices per format.
enum { SEC_FP16_W = 0 };
enum { SEC_BPDQ_BITS = 0, SEC_BPDQ_C01 = 1, SEC_BPDQ_OFF = 2, SEC_BPDQ_VTAB = 3 };
enum { SEC_TRL_STREAM = 0, SEC_TRL_TABLE = 1, SEC_TRL_SCALE = 2 };
enum { SEC_LEECH_PLANES = 0, SEC_LEECH_PARITY = 1, SEC_LEECH_SCALE = 2, SEC_LEECH_TAIL = 3,
       SEC_LEECH_EXCPTR = 4, SEC_LEECH_EXCCOL = 5 };

struct q2_blob_header {
  uint32_t magic;
  uint32_t version;
  int32_t fmt;
  int32_t R;          // output rows
  int32_t C;          // input columns
  int32_t Rpad;       // R rounded up to 32
  int32_t nslice;     // 256-column groups / segments / slices
  int32_t nblock;     // Leech: whole 24-column blocks per row
  int32_t tail;       // Leech: C % 24
  int32_t tailpad;    // Leech: tail columns stored per row (multiple of 8)
  uint32_t nexc;      // Leech: exception count
  float inv_sqrt8;    // Leech: fp32 factor applied with the row scale
  uint64_t total_bytes;
  uint64_t off[Q2_MAX_SECTIONS];
  uint64_t len[Q2_MAX_SECTIONS];
  int32_t layout;     // Leech: Q2_LEECH_PLANES3 or Q2_LEECH_OFFSET4; 0 otherwise
  int32_t reserved;
};

// Byte layout of one item (slice s, row block rb), item index it = s*nrb + rb:
//   chunk k of 512 bytes at it*ITEM + k*512; lane l's 16 bytes at +l*16.
// BPDQ:   chunks 0,1 = plane 0, chunks 2,3 = plane 1.  Leech: chunks 2p, 2p+1
//         = plane p (p = 0,1,2, and 3 in the offset-binary layout).  Byte q of chunk k is rotated position
//         P = (k&1)*16 + q, which holds the canonical column-byte
//         (P + lane) mod 32 of the slice for row rb*32 + lane.
// Trellis: 16 little-endian words per lane; nibble n (0..127) of the lane's
//         64 bytes holds symbol 127 - n of the segment, so the state of step
//         k is the 16 bits at bit offset 4*(127 - k), wrapping modulo 512.
