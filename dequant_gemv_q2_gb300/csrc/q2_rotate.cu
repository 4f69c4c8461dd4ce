// Activation rotation ahead of the GEMV ("Qwen3.8-27B on a 12 GB card",
// section "What the kernel does per token"): the weights are stored in a
// rotated basis, so each token's input is rotated at run time,
//
//   x_rot = (H (x) Q)(S x),   C = nh * nq,
//
// S the column signs, Q an nq x nq orthogonal matrix acting on every run of
// nq consecutive columns, H the orthonormal Sylvester Walsh-Hadamard
// transform of nh points acting across the runs (entry (i*nq + a, j*nq + b)
// of H (x) Q is H[i][j] Q[a][b]).
//
// One CTA of 512 threads per token holds the token's C values in shared
// memory as fp32 (index e stored at e + e / 32, which spreads the strided
// accesses below over the banks):
//   1. z = S x, loaded from fp16 eight columns (and their sign byte) at a
//      time, several loads in flight per thread;
//   2. each thread takes whole runs j and replaces z[j*nq .. j*nq + nq - 1]
//      by Q times it, from registers (nq <= 32);
//   3. the Walsh-Hadamard transform over j, for every a, in passes of up to
//      five butterfly stages: a task loads the 2^w values whose j differ
//      only in the pass's w bits, runs the w radix-2 stages in registers
//      and stores them back; one barrier per pass;
//   4. x_rot = fp16(u / sqrt(nh)), round to nearest.
// The whole transform is fp32; the only rounding to fp16 is the last step.
#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include <mutex>
#include <utility>
#include <vector>

#include "q2_common.cuh"

namespace cg = cooperative_groups;

namespace q2 {
namespace {

constexpr int kRotThreads = 512;
constexpr int kMaxNq = 32;

struct RotArgs {
  const __half* x;          // [ntok][C]
  __half* y;                // [ntok][C]
  const uint8_t* signs;     // [ceil(C/8)]
  const float* q;           // [nq][nq] or null (nq == 1)
  int C, nh, nq, lognh;
  float inv_sqrt_nh;
  int vec;                  // x and y 16-byte aligned and every CTA's first column a multiple of 8:
                            // 8 columns per load and store
};

constexpr int kInFlight = 4;   // 16-byte loads a thread issues before it uses the first

__host__ __device__ __forceinline__ int pad(int e) { return e + (e >> 5); }

// One pass of W radix-2 stages over bits [p, p + W) of the run index j, for
// nrun runs of nq columns held in u (padded indices).
template <int W>
__device__ __forceinline__ void wht_pass(float* u, int nrun, int nq, int p) {
  constexpr int n = 1 << W;
  const int rest = nrun >> W;                      // index values of the other bits of j
  const int tasks = rest * nq;
  const int lowmask = (1 << p) - 1;
  for (int task = threadIdx.x; task < tasks; task += kRotThreads) {
    const int col = task % nq, r = task / nq;      // lanes take consecutive columns a first
    const int jb = (r & lowmask) | ((r >> p) << (p + W));
    float v[n];
#pragma unroll
    for (int t = 0; t < n; ++t) v[t] = u[pad((jb + (t << p)) * nq + col)];
#pragma unroll
    for (int h = 1; h < n; h <<= 1)
#pragma unroll
      for (int t = 0; t < n; ++t)
        if (!(t & h)) {
          const float s = v[t], d = v[t + h];
          v[t] = s + d;
          v[t + h] = s - d;
        }
#pragma unroll
    for (int t = 0; t < n; ++t) u[pad((jb + (t << p)) * nq + col)] = v[t];
  }
}

// The full transform over bits [0, lognrun) of the run index, one barrier per pass.
__device__ __forceinline__ void wht_runs(float* u, int nrun, int nq, int lognrun) {
  for (int p = 0; p < lognrun; p += 5) {
    switch (min(5, lognrun - p)) {
      case 5: wht_pass<5>(u, nrun, nq, p); break;
      case 4: wht_pass<4>(u, nrun, nq, p); break;
      case 3: wht_pass<3>(u, nrun, nq, p); break;
      case 2: wht_pass<2>(u, nrun, nq, p); break;
      default: wht_pass<1>(u, nrun, nq, p); break;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kRotThreads, 1) k_rotate(RotArgs a) {
  extern __shared__ __align__(16) unsigned char q2_rot_smem[];
  float* qs = reinterpret_cast<float*>(q2_rot_smem);           // Q, nq * nq
  float* u = qs + kMaxNq * kMaxNq;                              // padded token vector
  const __half* xt = a.x + (size_t)blockIdx.x * a.C;
  __half* yt = a.y + (size_t)blockIdx.x * a.C;
  if (a.q)
    for (int i = threadIdx.x; i < a.nq * a.nq; i += kRotThreads) qs[i] = a.q[i];
  pdl_wait();                                                   // x may come from the previous kernel
  pdl_trigger();
  // 1. z = S x, with kInFlight loads in flight per thread
  if (a.vec) {
    const int nv = a.C >> 3;
    const uint4* x4 = reinterpret_cast<const uint4*>(xt);
    for (int v0 = threadIdx.x; v0 < nv; v0 += kInFlight * kRotThreads) {
      uint4 r[kInFlight];
      uint32_t sg[kInFlight];
#pragma unroll
      for (int k = 0; k < kInFlight; ++k) {
        const int v = v0 + k * kRotThreads;
        if (v < nv) {
          r[k] = x4[v];
          sg[k] = a.signs[v];
        }
      }
#pragma unroll
      for (int k = 0; k < kInFlight; ++k) {
        const int v = v0 + k * kRotThreads;
        if (v < nv) {
          const __half2* h2 = reinterpret_cast<const __half2*>(&r[k]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(h2[i]);
            u[pad(8 * v + 2 * i)] = ((sg[k] >> (2 * i)) & 1) ? -f.x : f.x;
            u[pad(8 * v + 2 * i + 1)] = ((sg[k] >> (2 * i + 1)) & 1) ? -f.y : f.y;
          }
        }
      }
    }
  } else {
    for (int e0 = threadIdx.x; e0 < a.C; e0 += kInFlight * kRotThreads) {
      float f[kInFlight];
      uint32_t sg[kInFlight];
#pragma unroll
      for (int k = 0; k < kInFlight; ++k) {
        const int e = e0 + k * kRotThreads;
        if (e < a.C) {
          f[k] = __half2float(xt[e]);
          sg[k] = a.signs[e >> 3];
        }
      }
#pragma unroll
      for (int k = 0; k < kInFlight; ++k) {
        const int e = e0 + k * kRotThreads;
        if (e < a.C) u[pad(e)] = ((sg[k] >> (e & 7)) & 1) ? -f[k] : f[k];
      }
    }
  }
  __syncthreads();
  // 2. Q on every run of nq columns
  if (a.q) {
    for (int j = threadIdx.x; j < a.nh; j += kRotThreads) {
      float z[kMaxNq];
#pragma unroll
      for (int b = 0; b < kMaxNq; ++b) z[b] = b < a.nq ? u[pad(j * a.nq + b)] : 0.f;
      for (int r = 0; r < a.nq; ++r) {
        float acc = 0.f;
#pragma unroll
        for (int b = 0; b < kMaxNq; ++b)
          if (b < a.nq) acc = fmaf(qs[r * a.nq + b], z[b], acc);
        u[pad(j * a.nq + r)] = acc;
      }
    }
    __syncthreads();
  }
  // 3. Walsh-Hadamard transform across the runs
  wht_runs(u, a.nh, a.nq, a.lognh);
  // 4. normalise, round to fp16
  if (a.vec) {
    uint4* y4 = reinterpret_cast<uint4*>(yt);
    for (int v = threadIdx.x; v < (a.C >> 3); v += kRotThreads) {
      uint4 o;
      uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 h = __floats2half2_rn(u[pad(8 * v + 2 * i)] * a.inv_sqrt_nh, u[pad(8 * v + 2 * i + 1)] * a.inv_sqrt_nh);
        ow[i] = *reinterpret_cast<const uint32_t*>(&h);
      }
      y4[v] = o;
    }
  } else {
    for (int e = threadIdx.x; e < a.C; e += kRotThreads) yt[e] = __float2half_rn(u[pad(e)] * a.inv_sqrt_nh);
  }
}

// The same transform spread over a cluster of G CTAs per token (G = 8, 4 or
// 2, when G^2 divides nh).  Sylvester's H over nh = G * J points factors as
// H_G (x) H_J on the run index j = g * J + jl, so CTA g owns the
// J runs (J * nq consecutive columns) with high bits g:
//   1. z = S x of its columns; 2. Q on each of its runs;
//   3. the Walsh-Hadamard transform over the low log2(J) bits locally;
//   4. after a cluster barrier, the G-point transform over the high bits:
//      CTA g takes 1/G of the local positions and, for each, reads the value
//      at that position in every CTA's shared memory (distributed shared
//      memory), transforms the G values and writes them, normalised and
//      rounded to fp16, straight to their columns of x_rot;
//   5. a split cluster barrier (arrive after the peer reads, wait before
//      exit) keeps every CTA's shared memory alive until its peers are done.
template <int G>
__global__ void __launch_bounds__(kRotThreads, 1) k_rotate_cluster(RotArgs a) {
  extern __shared__ __align__(16) unsigned char q2_rot_smem[];
  cg::cluster_group cluster = cg::this_cluster();
  const int g = (int)cluster.block_rank();
  const int J = a.nh / G, Cl = J * a.nq;                        // runs and columns of this CTA
  float* qs = reinterpret_cast<float*>(q2_rot_smem);            // Q, nq * nq
  float* z = qs + kMaxNq * kMaxNq;                              // S x, padded
  float* u = z + pad(Cl) + 1;                                   // Q z, then the transform, padded
  const size_t col0 = (size_t)(blockIdx.x / G) * a.C + (size_t)g * Cl;
  const __half* xt = a.x + col0;
  const int gcol = g * Cl;                                      // first column of this CTA in the token
  if (a.q)
    for (int i = threadIdx.x; i < a.nq * a.nq; i += kRotThreads) qs[i] = a.q[i];
  pdl_wait();
  pdl_trigger();
  // 1. z = S x
  if (a.vec) {
    const int nv = Cl >> 3;
    const uint4* x4 = reinterpret_cast<const uint4*>(xt);
    for (int v0 = threadIdx.x; v0 < nv; v0 += kInFlight * kRotThreads) {
      uint4 r[kInFlight];
      uint32_t sg[kInFlight];
#pragma unroll
      for (int k = 0; k < kInFlight; ++k) {
        const int v = v0 + k * kRotThreads;
        if (v < nv) {
          r[k] = x4[v];
          sg[k] = a.signs[(gcol >> 3) + v];
        }
      }
#pragma unroll
      for (int k = 0; k < kInFlight; ++k) {
        const int v = v0 + k * kRotThreads;
        if (v < nv) {
          const __half2* h2 = reinterpret_cast<const __half2*>(&r[k]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(h2[i]);
            z[pad(8 * v + 2 * i)] = ((sg[k] >> (2 * i)) & 1) ? -f.x : f.x;
            z[pad(8 * v + 2 * i + 1)] = ((sg[k] >> (2 * i + 1)) & 1) ? -f.y : f.y;
          }
        }
      }
    }
  } else {
    for (int e = threadIdx.x; e < Cl; e += kRotThreads) {
      const float f = __half2float(xt[e]);
      z[pad(e)] = ((a.signs[(gcol + e) >> 3] >> ((gcol + e) & 7)) & 1) ? -f : f;
    }
  }
  __syncthreads();
  // 2. u = Q z on each run: one (run, output column) per task
  for (int task = threadIdx.x; task < Cl; task += kRotThreads) {
    const int j = task / a.nq, r = task - j * a.nq;
    float acc;
    if (a.q) {
      acc = 0.f;
      for (int b = 0; b < a.nq; ++b) acc = fmaf(qs[r * a.nq + b], z[pad(j * a.nq + b)], acc);
    } else {
      acc = z[pad(task)];
    }
    u[pad(task)] = acc;
  }
  __syncthreads();
  // 3. local transform over the low bits of the run index
  wht_runs(u, J, a.nq, a.lognh - (G == 8 ? 3 : G == 4 ? 2 : 1));
  cluster.sync();
  // 4. G-point transform over the high bits, through distributed shared
  // memory, written straight to x_rot: position pos of chunk k is column
  // k * Cl + pos of the token
  {
    const int P = Cl / G;
    __half* ytok = a.y + (size_t)(blockIdx.x / G) * a.C;
    const float* peer[G];
#pragma unroll
    for (int k = 0; k < G; ++k) peer[k] = cluster.map_shared_rank(u, k);
    for (int pos = g * P + threadIdx.x; pos < (g + 1) * P; pos += kRotThreads) {
      const int pp = pad(pos);
      float v[G];
#pragma unroll
      for (int k = 0; k < G; ++k) v[k] = peer[k][pp];
#pragma unroll
      for (int h = 1; h < G; h <<= 1)
#pragma unroll
        for (int t = 0; t < G; ++t)
          if (!(t & h)) {
            const float s0 = v[t], d0 = v[t + h];
            v[t] = s0 + d0;
            v[t + h] = s0 - d0;
          }
#pragma unroll
      for (int k = 0; k < G; ++k) ytok[k * Cl + pos] = __float2half_rn(v[k] * a.inv_sqrt_nh);
    }
  }
  // 5. no CTA leaves while a peer may still read its shared memory
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int G>
int cluster_smem(int C) { return (kMaxNq * kMaxNq + 2 * (pad(C / G) + 1)) * (int)sizeof(float); }

// How many clusters of G CTAs (smem bytes each) the device runs at once,
// from the occupancy calculator, cached per (device, G, smem); 0 if unknown.
template <int G>
int clusters_in_flight(int smem) {
  static std::mutex mu;
  static std::vector<std::pair<std::pair<int, int>, int>> cache;   // ((device, smem), clusters)
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(mu);
  for (const auto& e : cache)
    if (e.first.first == dev && e.first.second == smem) return e.second;
  int n = 0;
  if (!set_smem(reinterpret_cast<const void*>(k_rotate_cluster<G>), smem)) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(kRotThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, k_rotate_cluster<G>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
  }
  cache.push_back({{dev, smem}, n});
  return n;
}

// Cluster launch with programmatic stream serialization allowed.
template <int G>
int launch_rotate_cluster(const RotArgs& a, int ntok, void* stream) {
  const int smem = cluster_smem<G>(a.C);
  if (set_smem(reinterpret_cast<const void*>(k_rotate_cluster<G>), smem)) return Q2_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ntok * G);
  cfg.blockDim = dim3(kRotThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = G;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, k_rotate_cluster<G>, a) != cudaSuccess) {
    (void)cudaGetLastError();
    return Q2_ECUDA;
  }
  return cudaGetLastError() == cudaSuccess ? Q2_OK : Q2_ECUDA;
}

}  // namespace
}  // namespace q2

extern "C" int q2_rotate_split(int C, int* nh, int* nq) {
  if (!nh || !nq) return Q2_EINVAL;
  const int h = (C > 0 && C % 2048 == 0) ? 2048 : 1024;
  if (C <= 0 || C % h) return Q2_ESHAPE;
  *nh = h;
  *nq = C / h;
  return Q2_OK;
}

extern "C" int q2_rotate(const void* x, void* x_rot, int ntok, int C, int nh, const void* signs, const float* q,
                         q2_stream stream) {
  using namespace q2;
  if (!x || !x_rot || !signs) return Q2_EINVAL;
  if (ntok < 1 || ntok > Q2_MAX_NTOK) return Q2_ENTOK;
  if (nh < 1 || (nh & (nh - 1)) || C < 1 || C > Q2_ROT_MAX_C || C % nh) return Q2_ESHAPE;
  const int nq = C / nh;
  if (nq > kMaxNq || (nq > 1 && !q)) return nq > kMaxNq ? Q2_ESHAPE : Q2_EINVAL;
  if (x == x_rot) return Q2_EINVAL;
  RotArgs a = {};
  a.x = static_cast<const __half*>(x);
  a.y = static_cast<__half*>(x_rot);
  a.signs = static_cast<const uint8_t*>(signs);
  a.q = q;
  a.C = C;
  a.nh = nh;
  a.nq = nq;
  int lg = 0;
  while ((1 << lg) < nh) ++lg;
  a.lognh = lg;
  a.inv_sqrt_nh = (float)(1.0 / sqrt((double)nh));
  a.vec = (C % 8 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0 && (reinterpret_cast<uintptr_t>(x_rot) & 15) == 0) ? 1 : 0;
  // cluster of G CTAs per token: the largest of 8, 4, 2 that splits the
  // transform evenly (G^2 divides nh) and runs all ntok clusters in one wave
  auto fits = [&](int g) {
    if (nh % (g * g)) return false;
    const int n = g == 8 ? clusters_in_flight<8>(cluster_smem<8>(C))
                : g == 4 ? clusters_in_flight<4>(cluster_smem<4>(C))
                         : clusters_in_flight<2>(cluster_smem<2>(C));
    return ntok <= n;
  };
  int G = 8;
  while (G > 1 && !fits(G)) G >>= 1;
  // 16-byte loads and stores start at each CTA's first column: C / G % 8 == 0
  if (C % (8 * G)) a.vec = 0;
  if (G == 8) return launch_rotate_cluster<8>(a, ntok, stream);
  if (G == 4) return launch_rotate_cluster<4>(a, ntok, stream);
  if (G == 2) return launch_rotate_cluster<2>(a, ntok, stream);
  const int smem = (kMaxNq * kMaxNq + pad(C) + 1) * (int)sizeof(float);
  return launch_pdl(k_rotate, a, ntok, kRotThreads, smem, stream);
}
