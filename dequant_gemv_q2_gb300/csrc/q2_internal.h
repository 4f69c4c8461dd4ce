// Internal declarations shared by the host code and the CUDA sources.
#pragma once
#include "q2_layout.h"
#include "../../include/q2.h"

struct q2_handle {
  q2_blob_header hdr;
  const unsigned char* dev;  // device copy of the blob (caller-owned)
  void* ws;                  // split-K workspace (caller-owned), may be null
  size_t ws_bytes;
  double pbound;             // |partial of one 256-column slice| <= pbound for any fp16 x
};

static inline int q2_nrb(const q2_blob_header& h) { return h.Rpad / Q2_ROWS; }

// Device byte ranges a launch prefetches into L2 for the launches after it
// (q2_gemv_chain); each CTA issues its 1/grid share of every range.  Ranges
// start 16-byte aligned; a zero length is an unused slot.
#define Q2_PF_SLOTS 4
struct q2_pf {
  const unsigned char* ptr[Q2_PF_SLOTS];
  unsigned long long len[Q2_PF_SLOTS];
};


#ifdef __cplusplus
extern "C" {
#endif
// Launchers (CUDA side).  Each returns a q2 status.
// pf: ranges to prefetch into L2 (batch-1 launches only), or NULL.
int q2_launch_fp16(const q2_handle* h, const void* x, void* y, int ntok, void* stream, const q2_pf* pf);
int q2_launch_bpdq(const q2_handle* h, const void* x, void* y, int ntok, void* stream, const q2_pf* pf);
int q2_launch_trellis(const q2_handle* h, const void* x, void* y, int ntok, void* stream, const q2_pf* pf);
int q2_launch_leech(const q2_handle* h, const void* x, void* y, int ntok, void* stream, const q2_pf* pf);
int q2_launch_noweights(const q2_handle* h, const void* x, void* y, int ntok, void* stream, const q2_pf* pf);
int q2_launch_decode(const q2_handle* h, void* out, void* stream);
#ifdef __cplusplus
}
#endif
