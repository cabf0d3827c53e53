// noalloc.cu -- dualkv_bwd_noalloc: the backward pass without any device
// allocation, for callers that cannot call cudaMalloc (see include/dualkv.h).
//
// Everything the backward needs besides the caller's inputs and outputs --
// the work lists, Delta, the log2-scaled LSE, the split dK/dV partials and a
// status word -- lives in one fixed array in device memory, g_scratch.  In
// host code `g_scratch` names a host-side stand-in, not the device array, so
// its device address is looked up once per device with cudaGetSymbolAddress
// and only that address is handed to the kernels.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <map>
#include <mutex>
#include <vector>

#include "../../include/dualkv.h"
#include "kernels.h"
#include "plan.h"

using namespace dkv;

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // DUALKV_NOALLOC_SCRATCH_BYTES
static_assert(kScratchBytes == (size_t)DUALKV_NOALLOC_SCRATCH_BYTES, "header and library disagree");

// Shared by every call on a device; it keeps the last call's contents.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// dK/dV key tiles whose query walk exceeds this many blocks are split (same value as dualkv_bwd)
constexpr int kMaxDkvIters = 512;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_na_mu;
EncodeTiledFn g_na_encode = nullptr;
std::map<int, unsigned char*> g_na_base;  // device -> device address of g_scratch

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Set-up, once per device with that device current: the device address of g_scratch.
int scratch_base(int device, unsigned char** out) {
  auto it = g_na_base.find(device);
  if (it != g_na_base.end()) {
    *out = it->second;
    return DUALKV_OK;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return DUALKV_ERR_CUDA;
  if (!g_na_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return DUALKV_ERR_CUDA;
    g_na_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  g_na_base[device] = static_cast<unsigned char*>(p);
  *out = static_cast<unsigned char*>(p);
  return DUALKV_OK;
}

int tmap(CUtensorMap* m, const void* base, int64_t T, int H, int D, int box_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_na_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DUALKV_OK : DUALKV_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename T>
cudaError_t put(unsigned char* dst, const std::vector<T>& v, cudaStream_t st) {
  if (v.empty()) return cudaSuccess;
  return cudaMemcpyAsync(dst, v.data(), sizeof(T) * v.size(), cudaMemcpyHostToDevice, st);
}

}  // namespace

extern "C" int dualkv_bwd_noalloc(const void* q, const void* k, const void* v, const void* out, const float* lse,
                                  const void* dout, int P, int N, const int32_t* R_offsets, int Hq, int Hkv, int D,
                                  float scale, int window, void* dq, void* dk, void* dv, void* stream) {
  if (validate_layout(P, N, R_offsets, Hq, Hkv, D)) return DUALKV_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return DUALKV_ERR_INVALID;
  if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv) return DUALKV_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return DUALKV_ERR_ALIGN;
  if (D != 64 && D != 128) return DUALKV_ERR_UNSUPPORTED;
  const int W = window <= 0 ? 0 : window;
  const int64_t T = (int64_t)P + R_offsets[N];
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  // host-side plan and the scratch layout: status | work lists | Delta | lse2 | partials
  Layout L{P, N, std::vector<int32_t>(R_offsets, R_offsets + N + 1), Hq, Hkv, D, W};
  const std::vector<QTileItem> dq_items = plan_qtiles(L, dq_query_tile(D), dq_key_tile(D));
  const KVPlan kv = plan_kvtiles(L, dkv_key_tile(D), dkv_query_block(D), kMaxDkvIters);
  size_t off = 256;  // status word
  const size_t o_dq = off;
  off = up256(off + sizeof(QTileItem) * dq_items.size());
  const size_t o_kv = off;
  off = up256(off + sizeof(KVTileItem) * kv.items.size());
  const size_t o_qb = off;
  off = up256(off + sizeof(QBlock) * kv.qblocks.size());
  const size_t o_red = off;
  off = up256(off + sizeof(ReduceItem) * kv.reduces.size());
  const size_t o_delta = off;
  off = up256(off + sizeof(float) * (size_t)Hq * T);
  const size_t o_lse2 = off;
  off = up256(off + sizeof(float) * (size_t)Hq * T);
  const size_t o_part = off;
  off += sizeof(float) * (size_t)kv.nslots * 2 * dkv_key_tile(D) * D;
  if (off > kScratchBytes) return DUALKV_ERR_WORKSPACE;  // layout needs more than the fixed scratch

  std::lock_guard<std::mutex> lock(g_na_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DUALKV_ERR_CUDA;
  unsigned char* base = nullptr;
  int rc = scratch_base(dev, &base);
  if (rc) return rc;
  uint32_t* status = reinterpret_cast<uint32_t*>(base);

  // From the first queued operation on, every exit waits for the work already on
  // `stream`: the next call may come from another stream once the lock is released,
  // and must not overlap copies or kernels of this one that still use the scratch.
  auto fail = [&](int code) {
    cudaStreamSynchronize(st);
    return code;
  };
  // the status word must start at zero; every other region is fully written before it is read
  if (cudaMemsetAsync(status, 0, sizeof(uint32_t), st) != cudaSuccess) return fail(DUALKV_ERR_CUDA);
  if (put(base + o_dq, dq_items, st) != cudaSuccess || put(base + o_kv, kv.items, st) != cudaSuccess ||
      put(base + o_qb, kv.qblocks, st) != cudaSuccess || put(base + o_red, kv.reduces, st) != cudaSuccess)
    return fail(DUALKV_ERR_CUDA);
  float* delta = reinterpret_cast<float*>(base + o_delta);
  float* lse2 = reinterpret_cast<float*>(base + o_lse2);
  float* partial = reinterpret_cast<float*>(base + o_part);
  const float sl2 = scale * 1.4426950408889634f;

  PrepArgs pa{static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), lse, delta, lse2, T, Hq, D};
  pa.check_items = reinterpret_cast<QTileItem*>(base + o_dq);  // checked before the dQ kernel reads it
  pa.n_check = (int)dq_items.size();
  pa.check_tile = dq_query_tile(D);
  pa.status = status;
  if (launch_prep(pa, st) != cudaSuccess) return fail(DUALKV_ERR_CUDA);
  CUtensorMap tq, tk, tv, tdo;
  if (tmap(&tq, q, T, Hq, D, dkv_query_block(D)) || tmap(&tk, k, T, Hkv, D, dkv_key_tile(D)) ||
      tmap(&tv, v, T, Hkv, D, dkv_key_tile(D)) || tmap(&tdo, dout, T, Hq, D, dkv_query_block(D)))
    return fail(DUALKV_ERR_CUDA);
  DkvArgs ka{reinterpret_cast<const KVTileItem*>(base + o_kv), reinterpret_cast<const QBlock*>(base + o_qb), delta,
             lse2, static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv), partial, (int)T, Hq, Hkv, W, sl2,
             scale, status, kv.nslots};
  if (launch_dkv(D, tq, tk, tv, tdo, ka, (int)kv.items.size(), st) != cudaSuccess) return fail(DUALKV_ERR_CUDA);
  if (!kv.reduces.empty()) {
    ReduceArgs ra{reinterpret_cast<const ReduceItem*>(base + o_red), partial, static_cast<__nv_bfloat16*>(dk),
                  static_cast<__nv_bfloat16*>(dv), Hkv, D, dkv_key_tile(D), T, kv.nslots, status};
    if (launch_reduce(ra, (int)kv.reduces.size(), st) != cudaSuccess) return fail(DUALKV_ERR_CUDA);
  }
  CUtensorMap tq2, tk2, tv2, tdo2;
  if (tmap(&tq2, q, T, Hq, D, dq_query_tile(D)) || tmap(&tk2, k, T, Hkv, D, dq_key_tile(D)) ||
      tmap(&tv2, v, T, Hkv, D, dq_key_tile(D)) || tmap(&tdo2, dout, T, Hq, D, dq_query_tile(D)))
    return fail(DUALKV_ERR_CUDA);
  DqArgs qa{reinterpret_cast<const QTileItem*>(base + o_dq), delta, lse2, static_cast<__nv_bfloat16*>(dq), (int)T, Hq,
            Hkv, W, sl2, scale, status};
  if (launch_dq(D, tq2, tk2, tv2, tdo2, qa, (int)dq_items.size(), st) != cudaSuccess) return fail(DUALKV_ERR_CUDA);

  // device-side failures land in the scratch's status word: read it once the pass is done
  uint32_t h = 0;
  if (cudaMemcpyAsync(&h, status, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess) return fail(DUALKV_ERR_CUDA);
  if (cudaStreamSynchronize(st) != cudaSuccess) return DUALKV_ERR_CUDA;
  return h ? DUALKV_ERR_DEVICE : DUALKV_OK;
}
