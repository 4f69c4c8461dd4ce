// Launch-side state (SM count, shared-memory opt-in) and the per-format
// launchers that pick the batch-1 CUDA-core or the tensor-core kernel.
#include <cuda_runtime.h>

#include <mutex>
#include <utility>
#include <vector>

#include "q2_common.cuh"

extern "C" int q2_b1_bpdq(const q2_handle* h, const void* x, void* y, void* stream, const q2_pf* pf);
extern "C" int q2_b1_noweights(const q2_handle* h, const void* x, void* y, void* stream, const q2_pf* pf);
extern "C" int q2_b1_leech(const q2_handle* h, const void* x, void* y, void* stream, const q2_pf* pf);
extern "C" int q2_b1_trellis(const q2_handle* h, const void* x, void* y, void* stream, const q2_pf* pf);
extern "C" int q2_mt_bpdq(const q2_handle* h, const void* x, void* y, int ntok, void* stream, const q2_pf* pf);
extern "C" int q2_tc_bpdq(const q2_handle* h, const void* x, void* y, int ntok, void* stream);
extern "C" int q2_tc_trellis(const q2_handle* h, const void* x, void* y, int ntok, void* stream);
extern "C" int q2_tc_leech(const q2_handle* h, const void* x, void* y, int ntok, void* stream);

namespace q2 {

namespace {
std::mutex g_mu;
std::vector<int> g_sms;                                  // per device
std::vector<std::pair<std::pair<int, const void*>, int>> g_smem;  // (dev, fn) -> bytes set
}  // namespace

DevInfo dev_info() {
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if ((int)g_sms.size() <= dev) g_sms.resize(dev + 1, 0);
  if (!g_sms[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = n > 0 ? n : 1;
  }
  return DevInfo{g_sms[dev]};
}

int set_smem(const void* fn, int bytes) {
  if (bytes <= 48 * 1024) return 0;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& e : g_smem)
    if (e.first.first == dev && e.first.second == fn) {
      if (e.second >= bytes) return 0;
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return 1;
      e.second = bytes;
      return 0;
    }
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return 1;
  g_smem.push_back({{dev, fn}, bytes});
  return 0;
}

}  // namespace q2

extern "C" {

// BPDQ: batch 1 and 2..6 tokens on CUDA cores (subset-sum tables), 7..64 on
// the tensor cores.
int q2_launch_bpdq(const q2_handle* h, const void* x, void* y, int ntok, void* stream, const q2_pf* pf) {
  if (ntok == 1) return q2_b1_bpdq(h, x, y, stream, pf);
  if (ntok <= 6) return q2_mt_bpdq(h, x, y, ntok, stream, pf);
  return q2_tc_bpdq(h, x, y, ntok, stream);
}

int q2_launch_trellis(const q2_handle* h, const void* x, void* y, int ntok, void* stream, const q2_pf* pf) {
  return ntok == 1 ? q2_b1_trellis(h, x, y, stream, pf) : q2_tc_trellis(h, x, y, ntok, stream);
}

int q2_launch_leech(const q2_handle* h, const void* x, void* y, int ntok, void* stream, const q2_pf* pf) {
  if (ntok == 1) return q2_b1_leech(h, x, y, stream, pf);
  // Two tokens: one single-token launch each, measured faster than the
  // tensor-core path padded to 16 tokens, when every token's x and y rows
  // start 16-byte aligned (the single-token kernel loads x in 16-byte pieces).
  if (ntok == 2 && h->hdr.C % 8 == 0 && h->hdr.R % 8 == 0) {
    for (int t = 0; t < 2; ++t) {
      const int st = q2_b1_leech(h, static_cast<const char*>(x) + (size_t)t * h->hdr.C * 2,
                                 static_cast<char*>(y) + (size_t)t * h->hdr.R * 2, stream, t == 1 ? pf : nullptr);
      if (st) return st;
    }
    return Q2_OK;
  }
  return q2_tc_leech(h, x, y, ntok, stream);
}

int q2_launch_noweights(const q2_handle* h, const void* x, void* y, int ntok, void* stream, const q2_pf* pf) {
  if (ntok != 1) return Q2_ENTOK;
  return q2_b1_noweights(h, x, y, stream, pf);
}

}  // extern "C"
