// pack.cu -- moving per-token tensors between the replicated and the packed
// layout, so that the token reduction of shared-prompt packing reaches the
// layers around attention (DualKV paper, abstract: with the prompt stored
// once, every per-token layer, not only attention, works on fewer rows).
//
//   replicated: sequence n = prompt rows 0..P-1 then its R_n response rows,
//               sequences laid end to end; sequence n starts at n*P + off[n]
//   packed:     prompt rows, then the response rows of segments 0..N-1
//
// pack   (replicated -> packed): a prompt row is taken from replica 0
// unpack (packed -> replicated): a prompt row is copied into every replica
// fold   (replicated -> packed): the adjoint of unpack (the gradient of the
//        packed rows): a prompt row sums its N replica rows in replica order
//        in fp32 and rounds once to bf16; a response row is copied.
//
// A row is `row_elems` bf16 values moved as 16-byte vectors.  A group of G
// lanes (G = 32, or the next power of two above a shorter row) works on one
// unit at a time -- a whole row, or for the prompt rows of unpack and fold a
// chunk of G vectors of one row -- so the index mapping is computed once per
// unit; groups stride over the units.  Unpack reads each packed row once.
// All three kernels are bound by HBM bandwidth.
#include <cuda_bf16.h>

#include "kernels.h"

namespace dkv {

namespace {

constexpr int kPackThreads = 256;

// Segment holding response row r: the largest n with off[n] <= r.  Empty
// segments share their offset with the next one, so the largest such n is the
// one whose range [off[n], off[n+1]) contains r.
__device__ __forceinline__ int seg_of_response(const int32_t* off, int N, int r) {
  int lo = 0, hi = N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(off + mid) <= r) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

struct RowGroup {
  int64_t first, stride;
  int lane, G;
};

__device__ __forceinline__ RowGroup row_group(int G) {
  const int64_t g = (int64_t)blockIdx.x * kPackThreads + threadIdx.x;
  return RowGroup{g / G, (int64_t)gridDim.x * kPackThreads / G, (int)(g % G), G};
}

__global__ void __launch_bounds__(kPackThreads) pack_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                            const int32_t* __restrict__ off, int P, int N,
                                                            int64_t T, int vpr, int G) {
  const RowGroup rg = row_group(G);
  for (int64_t t = rg.first; t < T; t += rg.stride) {
    int64_t x = t;  // prompt rows come from replica 0
    if (t >= P) {
      const int r = (int)(t - P);
      // n*P + off[n] + P + (r - off[n])
      x = (int64_t)(seg_of_response(off, N, r) + 1) * P + r;
    }
    const uint4* s = src + x * vpr;
    uint4* d = dst + t * vpr;
#pragma unroll 4
    for (int c = rg.lane; c < vpr; c += G) d[c] = s[c];
  }
}

// Work units of unpack and fold: P * nch prompt units (a prompt row's chunk of
// G consecutive vectors, one per lane), then one unit per response row.  A
// prompt unit touches N replicated rows, so those heavy units come first and
// spread over all groups before the light response rows.
struct Units {
  int64_t prompt, total;
  int nch;
};
__device__ __forceinline__ Units make_units(int P, int64_t T, int vpr, int G) {
  const int nch = (vpr + G - 1) / G;
  return Units{(int64_t)P * nch, (int64_t)P * nch + (T - P), nch};
}

__global__ void __launch_bounds__(kPackThreads) unpack_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                              const int32_t* __restrict__ off, int P, int N,
                                                              int64_t T, int vpr, int G) {
  const RowGroup rg = row_group(G);
  const Units U = make_units(P, T, vpr, G);
  for (int64_t u = rg.first; u < U.total; u += rg.stride) {
    if (u < U.prompt) {
      // prompt row t, vector c: read once, written into every replica
      const int64_t t = u / U.nch;
      const int c = (int)(u % U.nch) * G + rg.lane;
      if (c >= vpr) continue;
      const uint4 v = src[t * vpr + c];
#pragma unroll 4
      for (int n = 0; n < N; ++n) dst[((int64_t)n * P + __ldg(off + n) + t) * vpr + c] = v;
      continue;
    }
    const int r = (int)(u - U.prompt);
    // response row r of segment n sits at n*P + off[n] + P + (r - off[n])
    const int64_t x = (int64_t)(seg_of_response(off, N, r) + 1) * P + r;
    const uint4* s = src + ((int64_t)P + r) * vpr;
    uint4* d = dst + x * vpr;
#pragma unroll 4
    for (int c = rg.lane; c < vpr; c += G) d[c] = s[c];
  }
}

__global__ void __launch_bounds__(kPackThreads) fold_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                            const int32_t* __restrict__ off, int P, int N,
                                                            int64_t T, int vpr, int G) {
  const RowGroup rg = row_group(G);
  const Units U = make_units(P, T, vpr, G);
  for (int64_t u = rg.first; u < U.total; u += rg.stride) {
    if (u < U.prompt) {
      const int64_t t = u / U.nch;
      const int c = (int)(u % U.nch) * G + rg.lane;
      if (c >= vpr) continue;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
      for (int n = 0; n < N; ++n) {
        const uint4 v = src[((int64_t)n * P + __ldg(off + n) + t) * vpr + c];
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(h[e]);
          acc[2 * e] += f.x;
          acc[2 * e + 1] += f.y;
        }
      }
      uint4 o;
      __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int e = 0; e < 4; ++e) oh[e] = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
      dst[t * vpr + c] = o;
      continue;
    }
    const int r = (int)(u - U.prompt);
    const uint4* s = src + ((int64_t)(seg_of_response(off, N, r) + 1) * P + r) * vpr;
    uint4* d = dst + ((int64_t)P + r) * vpr;
#pragma unroll 4
    for (int c = rg.lane; c < vpr; c += G) d[c] = s[c];
  }
}

}  // namespace

int pack_group_lanes(int row_elems) {
  const int vpr = row_elems / 8;
  int G = 1;
  while (G < 32 && G < vpr) G <<= 1;
  return G;
}

cudaError_t launch_pack(int kind, const void* src, void* dst, const int32_t* d_off, int P, int N, int64_t T,
                        int row_elems, int num_sms, cudaStream_t st) {
  const int vpr = row_elems / 8;
  const int G = pack_group_lanes(row_elems);
  const int64_t units = kind == 0 ? T : (int64_t)P * ((vpr + G - 1) / G) + (T - P);
  // one resident wave: 2048 threads per SM
  const int64_t full = (int64_t)num_sms * (2048 / kPackThreads);
  const int64_t need = (units * G + kPackThreads - 1) / kPackThreads;
  const unsigned grid = (unsigned)(need < full ? (need > 0 ? need : 1) : full);
  const uint4* s = static_cast<const uint4*>(src);
  uint4* d = static_cast<uint4*>(dst);
  switch (kind) {
    case 0:
      pack_kernel<<<grid, kPackThreads, 0, st>>>(s, d, d_off, P, N, T, vpr, G);
      break;
    case 1:
      unpack_kernel<<<grid, kPackThreads, 0, st>>>(s, d, d_off, P, N, T, vpr, G);
      break;
    case 2:
      fold_kernel<<<grid, kPackThreads, 0, st>>>(s, d, d_off, P, N, T, vpr, G);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace dkv
