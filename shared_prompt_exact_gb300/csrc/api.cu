// api.cu -- the C ABI of libdualkv.so (declared in include/dualkv.h): argument
// validation, the per-layout plan cache, TMA tensor maps, the per-device status
// word and the launch sequence of the forward and backward passes.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/dualkv.h"
#include "kernels.h"
#include "plan.h"

using namespace dkv;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;
std::map<int, uint32_t*> g_status;  // device -> status word

// dK/dV key tiles whose query walk is longer than this many query blocks are
// split into contiguous chunks reduced in a fixed order.
constexpr int kMaxDkvIters = 512;

struct DevPlan {
  int device = -1;
  bool fwd_ready = false, bwd_ready = false;
  QTileItem* fwd_items = nullptr;
  int n_fwd = 0;
  QTileItem* dq_items = nullptr;
  int n_dq = 0;
  KVTileItem* kv_items = nullptr;
  int n_kv = 0;
  QBlock* qblocks = nullptr;
  ReduceItem* reduces = nullptr;
  int n_reduce = 0;
  int nslots = 0;
  // head dimension 512
  int32_t* block_base = nullptr;
  int64_t n_blocks = 0;
  XTItem* xt_items = nullptr;
  int n_xt = 0;
  XTEntry* xt_entries = nullptr;
  ~DevPlan() {
    cudaFree(block_base);
    cudaFree(xt_items);
    cudaFree(xt_entries);
    cudaFree(fwd_items);
    cudaFree(dq_items);
    cudaFree(kv_items);
    cudaFree(qblocks);
    cudaFree(reduces);
  }
};
std::map<std::string, std::unique_ptr<DevPlan>> g_plans;

struct DevOffsets {
  int32_t* d = nullptr;
  int num_sms = 0;
  ~DevOffsets() { cudaFree(d); }
};
std::map<std::string, std::unique_ptr<DevOffsets>> g_offsets;  // (device, P, N, R_offsets) -> device copy

std::string plan_key(int device, int P, int N, const int32_t* off, int Hq, int Hkv, int D, int window, int kv_lo = 0,
                     int kv_hi = 0) {
  std::string k;
  k.reserve(64 + 4 * (N + 1));
  int32_t hdr[9] = {device, P, N, Hq, Hkv, D, window <= 0 ? 0 : window, kv_lo, kv_hi};
  k.append(reinterpret_cast<const char*>(hdr), sizeof(hdr));
  k.append(reinterpret_cast<const char*>(off), sizeof(int32_t) * (N + 1));
  return k;
}

template <typename T>
cudaError_t upload(T** dst, const std::vector<T>& v) {
  *dst = nullptr;
  if (v.empty()) return cudaSuccess;
  cudaError_t e = cudaMalloc(dst, sizeof(T) * v.size());
  if (e != cudaSuccess) return e;
  return cudaMemcpy(*dst, v.data(), sizeof(T) * v.size(), cudaMemcpyHostToDevice);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int ensure_encode() {
  if (g_encode) return DUALKV_OK;
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return DUALKV_ERR_CUDA;
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  return DUALKV_OK;
}

int status_word(int device, uint32_t** out) {
  auto it = g_status.find(device);
  if (it != g_status.end()) {
    *out = it->second;
    return DUALKV_OK;
  }
  uint32_t* p = nullptr;
  if (cudaMalloc(&p, 256) != cudaSuccess) return DUALKV_ERR_CUDA;
  if (cudaMemset(p, 0, 256) != cudaSuccess) return DUALKV_ERR_CUDA;
  g_status[device] = p;
  *out = p;
  return DUALKV_OK;
}

// [T, H, D] bf16 rows, box of 64 head-dim columns x 1 head x box_rows rows, 128-byte swizzle.
int make_tmap(CUtensorMap* m, const void* base, int64_t T, int H, int D, int box_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DUALKV_OK : DUALKV_ERR_CUDA;
}

// Looks up (or builds) the plan of a layout restricted to kv-heads [kv_lo, kv_hi);
// caller holds g_mu.
int get_plan(int P, int N, const int32_t* off, int Hq, int Hkv, int D, int window, int kv_lo, int kv_hi,
             bool need_bwd, DevPlan** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DUALKV_ERR_CUDA;
  const std::string key = plan_key(dev, P, N, off, Hq, Hkv, D, window, kv_lo, kv_hi);
  auto& slot = g_plans[key];
  if (!slot) {
    slot.reset(new DevPlan());
    slot->device = dev;
  }
  DevPlan* pl = slot.get();
  Layout L{P, N, std::vector<int32_t>(off, off + N + 1), Hq, Hkv, D, window <= 0 ? 0 : window, kv_lo, kv_hi};
  if (!pl->fwd_ready) {
    auto items = plan_qtiles(L, fwd_query_tile(D), fwd_key_tile(D));
    if (upload(&pl->fwd_items, items) != cudaSuccess) return DUALKV_ERR_CUDA;
    pl->n_fwd = (int)items.size();
    pl->fwd_ready = true;
  }
  if (need_bwd && !pl->bwd_ready && D == 512) {
    auto dq = plan_qtiles(L, 128, 128);
    if (upload(&pl->dq_items, dq) != cudaSuccess) return DUALKV_ERR_CUDA;
    pl->n_dq = (int)dq.size();
    Plan512 p5 = plan_512(L, dq, kMaxDkvIters);
    if (upload(&pl->block_base, p5.block_base) != cudaSuccess) return DUALKV_ERR_CUDA;
    if (upload(&pl->xt_items, p5.items) != cudaSuccess) return DUALKV_ERR_CUDA;
    if (upload(&pl->xt_entries, p5.entries) != cudaSuccess) return DUALKV_ERR_CUDA;
    if (upload(&pl->reduces, p5.reduces) != cudaSuccess) return DUALKV_ERR_CUDA;
    pl->n_blocks = p5.n_blocks;
    pl->n_xt = (int)p5.items.size();
    pl->n_reduce = (int)p5.reduces.size();
    pl->nslots = p5.nslots;
    pl->bwd_ready = true;
  }
  if (need_bwd && !pl->bwd_ready) {
    auto dq = plan_qtiles(L, dq_query_tile(D), dq_key_tile(D));
    if (upload(&pl->dq_items, dq) != cudaSuccess) return DUALKV_ERR_CUDA;
    pl->n_dq = (int)dq.size();
    KVPlan kv = plan_kvtiles(L, dkv_key_tile(D), dkv_query_block(D), kMaxDkvIters);
    if (upload(&pl->kv_items, kv.items) != cudaSuccess) return DUALKV_ERR_CUDA;
    if (upload(&pl->qblocks, kv.qblocks) != cudaSuccess) return DUALKV_ERR_CUDA;
    if (upload(&pl->reduces, kv.reduces) != cudaSuccess) return DUALKV_ERR_CUDA;
    pl->n_kv = (int)kv.items.size();
    pl->n_reduce = (int)kv.reduces.size();
    pl->nslots = kv.nslots;
    pl->bwd_ready = true;
  }
  *out = pl;
  return DUALKV_OK;
}

// ---------------------------------------------------------------- kernel timing
struct TimedLaunch {
  int kind;
  cudaEvent_t start, stop;
};
bool g_profile = false;
std::vector<TimedLaunch> g_timed;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Runs `launch` on stream `st`, bracketed by events when timing is enabled.
template <typename F>
cudaError_t timed(int kind, cudaStream_t st, F&& launch) {
  if (!g_profile) return launch();
  TimedLaunch t{kind, take_event(), take_event()};
  if (!t.start || !t.stop) return cudaErrorMemoryAllocation;
  cudaEventRecord(t.start, st);
  cudaError_t e = launch();
  cudaEventRecord(t.stop, st);
  g_timed.push_back(t);
  return e;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t delta, lse2, partial, pblk, dsblk, total;
};
// Delta | lse2 | fp32 split partials | (D = 512) P blocks | dS blocks
WsLayout ws_layout(int64_t T, int Hq, int D, int nslots, int64_t n_blocks) {
  WsLayout w;
  w.delta = 0;
  w.lse2 = align256(sizeof(float) * (size_t)Hq * T);
  w.partial = w.lse2 + align256(sizeof(float) * (size_t)Hq * T);
  const int key_tile = D == 512 ? 128 : dkv_key_tile(D);
  w.pblk = align256(w.partial + sizeof(float) * (size_t)nslots * 2 * key_tile * D);
  w.dsblk = w.pblk + (size_t)n_blocks * 128 * 128 * 2;
  w.total = w.dsblk + (size_t)n_blocks * 128 * 128 * 2;
  return w;
}

// [n_blocks, 128, 128] bf16 blocks, box 64 columns x box_rows rows x 1 block, 128-byte swizzle.
int make_block_tmap(CUtensorMap* m, const void* base, int64_t n_blocks, int box_rows) {
  cuuint64_t dims[3] = {128, 128, (cuuint64_t)n_blocks};
  cuuint64_t strides[2] = {256, 128 * 256};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DUALKV_OK : DUALKV_ERR_CUDA;
}

// Device copy of R_offsets and the SM count for the pack kernels; caller holds g_mu.
int get_offsets(int P, int N, const int32_t* off, DevOffsets** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DUALKV_ERR_CUDA;
  auto& slot = g_offsets[plan_key(dev, P, N, off, 0, 0, 0, 0)];
  if (!slot) {
    std::unique_ptr<DevOffsets> o(new DevOffsets());
    if (cudaDeviceGetAttribute(&o->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return DUALKV_ERR_CUDA;
    if (upload(&o->d, std::vector<int32_t>(off, off + N + 1)) != cudaSuccess) return DUALKV_ERR_CUDA;
    slot = std::move(o);
  }
  *out = slot.get();
  return DUALKV_OK;
}

// Shared checks and launch of dualkv_pack / dualkv_unpack / dualkv_fold.
int pack_call(int kind, const void* src, void* dst, int P, int N, const int32_t* off, int row_elems, void* stream) {
  if (P < 0 || N < 1 || !off || off[0] != 0) return DUALKV_ERR_INVALID;
  for (int n = 0; n < N; ++n)
    if (off[n + 1] < off[n]) return DUALKV_ERR_INVALID;
  const int64_t T = (int64_t)P + off[N];
  const int64_t T_rep = (int64_t)N * P + off[N];
  if (T < 1 || T_rep > INT32_MAX) return DUALKV_ERR_INVALID;
  if (row_elems < 8 || row_elems % 8) return DUALKV_ERR_INVALID;
  if (!src || !dst) return DUALKV_ERR_INVALID;
  if (!aligned16(src) || !aligned16(dst)) return DUALKV_ERR_ALIGN;
  const uint64_t row_bytes = (uint64_t)row_elems * 2;
  const uint64_t src_bytes = row_bytes * (uint64_t)(kind == 1 ? T : T_rep);
  const uint64_t dst_bytes = row_bytes * (uint64_t)(kind == 1 ? T_rep : T);
  const uint64_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
  if (s0 < d0 + dst_bytes && d0 < s0 + src_bytes) return DUALKV_ERR_INVALID;  // overlapping buffers
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_mu);
  DevOffsets* o = nullptr;
  int rc = get_offsets(P, N, off, &o);
  if (rc) return rc;
  if (timed(DUALKV_KERNEL_PACK, st, [&] {
        return launch_pack(kind, src, dst, o->d, P, N, T, row_elems, o->num_sms, st);
      }) != cudaSuccess)
    return DUALKV_ERR_CUDA;
  return DUALKV_OK;
}

bool supported_d(int D) { return D == 64 || D == 128 || D == 512; }  // backward
bool supported_fwd_d(int D) { return D == 64 || D == 128 || D == 512; }

int fwd_impl(const void* q, const void* k, const void* v, int P, int N, const int32_t* R_offsets, int Hq, int Hkv,
             int D, float scale, int window, int kv_lo, int kv_hi, void* out, float* lse, void* stream) {
  if (validate_layout(P, N, R_offsets, Hq, Hkv, D)) return DUALKV_ERR_INVALID;
  if (kv_lo < 0 || kv_hi > Hkv || kv_lo >= kv_hi) return DUALKV_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return DUALKV_ERR_INVALID;
  if (!q || !k || !v || !out || !lse) return DUALKV_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse)) return DUALKV_ERR_ALIGN;
  if (!supported_fwd_d(D)) return DUALKV_ERR_UNSUPPORTED;
  const int64_t T = (int64_t)P + R_offsets[N];
  std::lock_guard<std::mutex> lock(g_mu);
  int rc = ensure_encode();
  if (rc) return rc;
  DevPlan* pl = nullptr;
  if ((rc = get_plan(P, N, R_offsets, Hq, Hkv, D, window, kv_lo, kv_hi, false, &pl))) return rc;
  uint32_t* status = nullptr;
  if ((rc = status_word(pl->device, &status))) return rc;
  CUtensorMap tq, tk, tv;
  if (make_tmap(&tq, q, T, Hq, D, fwd_query_tile(D)) || make_tmap(&tk, k, T, Hkv, D, fwd_key_tile(D)) ||
      make_tmap(&tv, v, T, Hkv, D, fwd_key_tile(D)))
    return DUALKV_ERR_CUDA;
  FwdArgs a{pl->fwd_items, static_cast<__nv_bfloat16*>(out), lse, (int)T, Hq, Hkv, window <= 0 ? 0 : window,
            scale * 1.4426950408889634f, status};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (timed(DUALKV_KERNEL_FWD, st, [&] { return launch_fwd(D, tq, tk, tv, a, pl->n_fwd, st); }) != cudaSuccess)
    return DUALKV_ERR_CUDA;
  return DUALKV_OK;
}

int bwd_impl(const void* q, const void* k, const void* v, const void* out, const float* lse, const void* dout, int P,
             int N, const int32_t* R_offsets, int Hq, int Hkv, int D, float scale, int window, int kv_lo, int kv_hi,
             void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, void* stream) {
  if (validate_layout(P, N, R_offsets, Hq, Hkv, D)) return DUALKV_ERR_INVALID;
  if (kv_lo < 0 || kv_hi > Hkv || kv_lo >= kv_hi) return DUALKV_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return DUALKV_ERR_INVALID;
  if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv) return DUALKV_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return DUALKV_ERR_ALIGN;
  if (!supported_d(D)) return DUALKV_ERR_UNSUPPORTED;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return DUALKV_ERR_WORKSPACE;
  const int64_t T = (int64_t)P + R_offsets[N];
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_mu);
  int rc = ensure_encode();
  if (rc) return rc;
  DevPlan* pl = nullptr;
  if ((rc = get_plan(P, N, R_offsets, Hq, Hkv, D, window, kv_lo, kv_hi, true, &pl))) return rc;
  const WsLayout ws = ws_layout(T, Hq, D, pl->nslots, D == 512 ? pl->n_blocks : 0);
  if (workspace_bytes < ws.total) return DUALKV_ERR_WORKSPACE;
  uint32_t* status = nullptr;
  if ((rc = status_word(pl->device, &status))) return rc;
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  float* delta = reinterpret_cast<float*>(wsb + ws.delta);
  float* lse2 = reinterpret_cast<float*>(wsb + ws.lse2);
  float* partial = reinterpret_cast<float*>(wsb + ws.partial);
  const int W = window <= 0 ? 0 : window;
  const float sl2 = scale * 1.4426950408889634f;

  const int gs = Hq / Hkv;
  PrepArgs pa{static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), lse, delta, lse2, T, Hq, D,
              kv_lo * gs, kv_hi * gs};
  if (timed(DUALKV_KERNEL_PREP, st, [&] { return launch_prep(pa, st); }) != cudaSuccess) return DUALKV_ERR_CUDA;

  if (D == 512) {
    __nv_bfloat16* pblk = reinterpret_cast<__nv_bfloat16*>(wsb + ws.pblk);
    __nv_bfloat16* dsblk = reinterpret_cast<__nv_bfloat16*>(wsb + ws.dsblk);
    CUtensorMap tq, tk, tv, tdo, tq64, tdo64, tk64, tP64, tDS64, tDS128;
    if (make_tmap(&tq, q, T, Hq, D, 128) || make_tmap(&tk, k, T, Hkv, D, 128) || make_tmap(&tv, v, T, Hkv, D, 128) ||
        make_tmap(&tdo, dout, T, Hq, D, 128) || make_tmap(&tq64, q, T, Hq, D, 64) ||
        make_tmap(&tdo64, dout, T, Hq, D, 64) || make_tmap(&tk64, k, T, Hkv, D, 64) ||
        make_block_tmap(&tP64, pblk, pl->n_blocks, 64) || make_block_tmap(&tDS64, dsblk, pl->n_blocks, 64) ||
        make_block_tmap(&tDS128, dsblk, pl->n_blocks, 128))
      return DUALKV_ERR_CUDA;
    PdsArgs p0{pl->dq_items, pl->block_base, lse2, delta, nullptr, pblk, (int)T, Hq, Hkv, W, sl2, status};
    PdsArgs p1{pl->dq_items, pl->block_base, lse2, delta, pblk, dsblk, (int)T, Hq, Hkv, W, sl2, status};
    XtgArgs xv{pl->xt_items, pl->xt_entries, static_cast<__nv_bfloat16*>(dv), partial, 1, (int)T, Hq, Hkv, 1.f, status};
    XtgArgs xk{pl->xt_items, pl->xt_entries, static_cast<__nv_bfloat16*>(dk), partial, 0, (int)T, Hq, Hkv, scale, status};
    Dq512Args qa{pl->dq_items, pl->block_base, static_cast<__nv_bfloat16*>(dq), (int)T, Hq, Hkv, scale, status};
    if (timed(DUALKV_KERNEL_DKV, st, [&] {
          cudaError_t e = launch_pds(0, tq, tk, p0, pl->n_dq, st);
          if (e == cudaSuccess) e = launch_pds(1, tdo, tv, p1, pl->n_dq, st);
          if (e == cudaSuccess) e = launch_xtg(tP64, tdo64, xv, pl->n_xt, st);
          if (e == cudaSuccess) e = launch_xtg(tDS64, tq64, xk, pl->n_xt, st);
          return e;
        }) != cudaSuccess)
      return DUALKV_ERR_CUDA;
    if (pl->n_reduce > 0) {
      ReduceArgs ra{pl->reduces, partial, static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv), Hkv, D, 128};
      if (timed(DUALKV_KERNEL_REDUCE, st, [&] { return launch_reduce(ra, pl->n_reduce, st); }) != cudaSuccess)
        return DUALKV_ERR_CUDA;
    }
    if (timed(DUALKV_KERNEL_DQ, st, [&] { return launch_dq512(tDS128, tk64, qa, pl->n_dq, st); }) != cudaSuccess)
      return DUALKV_ERR_CUDA;
    return DUALKV_OK;
  }

  CUtensorMap tq, tk, tv, tdo;
  if (make_tmap(&tq, q, T, Hq, D, dkv_query_block(D)) || make_tmap(&tk, k, T, Hkv, D, dkv_key_tile(D)) ||
      make_tmap(&tv, v, T, Hkv, D, dkv_key_tile(D)) || make_tmap(&tdo, dout, T, Hq, D, dkv_query_block(D)))
    return DUALKV_ERR_CUDA;
  DkvArgs ka{pl->kv_items, pl->qblocks, delta, lse2, static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv),
             partial, (int)T, Hq, Hkv, W, sl2, scale, status};
  if (timed(DUALKV_KERNEL_DKV, st, [&] { return launch_dkv(D, tq, tk, tv, tdo, ka, pl->n_kv, st); }) != cudaSuccess)
    return DUALKV_ERR_CUDA;
  if (pl->n_reduce > 0) {
    ReduceArgs ra{pl->reduces, partial, static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv), Hkv, D,
                  dkv_key_tile(D)};
    if (timed(DUALKV_KERNEL_REDUCE, st, [&] { return launch_reduce(ra, pl->n_reduce, st); }) != cudaSuccess)
      return DUALKV_ERR_CUDA;
  }

  CUtensorMap tq2, tk2, tv2, tdo2;
  if (make_tmap(&tq2, q, T, Hq, D, dq_query_tile(D)) || make_tmap(&tk2, k, T, Hkv, D, dq_key_tile(D)) ||
      make_tmap(&tv2, v, T, Hkv, D, dq_key_tile(D)) || make_tmap(&tdo2, dout, T, Hq, D, dq_query_tile(D)))
    return DUALKV_ERR_CUDA;
  DqArgs qa{pl->dq_items, delta, lse2, static_cast<__nv_bfloat16*>(dq), (int)T, Hq, Hkv, W, sl2, scale, status};
  if (timed(DUALKV_KERNEL_DQ, st, [&] { return launch_dq(D, tq2, tk2, tv2, tdo2, qa, pl->n_dq, st); }) != cudaSuccess)
    return DUALKV_ERR_CUDA;
  return DUALKV_OK;
}

}  // namespace

extern "C" {

int dualkv_fwd(const void* q, const void* k, const void* v, int P, int N, const int32_t* R_offsets, int Hq, int Hkv,
               int D, float scale, int window, void* out, float* lse, void* stream) {
  return fwd_impl(q, k, v, P, N, R_offsets, Hq, Hkv, D, scale, window, 0, Hkv, out, lse, stream);
}

int dualkv_fwd_heads(const void* q, const void* k, const void* v, int P, int N, const int32_t* R_offsets, int Hq,
                     int Hkv, int D, float scale, int window, int kv_head_begin, int kv_head_end, void* out,
                     float* lse, void* stream) {
  return fwd_impl(q, k, v, P, N, R_offsets, Hq, Hkv, D, scale, window, kv_head_begin, kv_head_end, out, lse, stream);
}


size_t dualkv_bwd_workspace_bytes(int P, int N, const int32_t* R_offsets, int Hq, int Hkv, int D, int window) {
  if (validate_layout(P, N, R_offsets, Hq, Hkv, D) || !supported_d(D)) return 0;
  Layout L{P, N, std::vector<int32_t>(R_offsets, R_offsets + N + 1), Hq, Hkv, D, window <= 0 ? 0 : window};
  if (D == 512) {
    Plan512 p5 = plan_512(L, plan_qtiles(L, 128, 128), kMaxDkvIters);
    return ws_layout(L.T(), Hq, D, p5.nslots, p5.n_blocks).total;
  }
  KVPlan kv = plan_kvtiles(L, dkv_key_tile(D), dkv_query_block(D), kMaxDkvIters);
  return ws_layout(L.T(), Hq, D, kv.nslots, 0).total;
}

int dualkv_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse, const void* dout, int P,
               int N, const int32_t* R_offsets, int Hq, int Hkv, int D, float scale, int window, void* dq, void* dk,
               void* dv, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, out, lse, dout, P, N, R_offsets, Hq, Hkv, D, scale, window, 0, Hkv, dq, dk, dv, workspace,
                  workspace_bytes, stream);
}

int dualkv_bwd_heads(const void* q, const void* k, const void* v, const void* out, const float* lse, const void* dout,
                     int P, int N, const int32_t* R_offsets, int Hq, int Hkv, int D, float scale, int window,
                     int kv_head_begin, int kv_head_end, void* dq, void* dk, void* dv, void* workspace,
                     size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, out, lse, dout, P, N, R_offsets, Hq, Hkv, D, scale, window, kv_head_begin, kv_head_end,
                  dq, dk, dv, workspace, workspace_bytes, stream);
}


size_t dualkv_bwd_layers_workspace_bytes(int n_layers, const int32_t* window, int P, int N, const int32_t* R_offsets,
                                         int Hq, int Hkv, int D) {
  if (n_layers < 1 || !window) return 0;
  size_t need = 0;
  for (int l = 0; l < n_layers; ++l) {
    const size_t b = dualkv_bwd_workspace_bytes(P, N, R_offsets, Hq, Hkv, D, window[l]);
    if (b == 0) return 0;
    need = b > need ? b : need;
  }
  return need;
}

int dualkv_fwd_layers(int n_layers, const void* const* q, const void* const* k, const void* const* v,
                      const int32_t* window, int P, int N, const int32_t* R_offsets, int Hq, int Hkv, int D,
                      float scale, void* const* out, float* const* lse, void* stream) {
  if (n_layers < 1 || !q || !k || !v || !window || !out || !lse) return DUALKV_ERR_INVALID;
  if (validate_layout(P, N, R_offsets, Hq, Hkv, D) || !supported_fwd_d(D)) return DUALKV_ERR_INVALID;
  // check every layer before the first launch
  for (int l = 0; l < n_layers; ++l) {
    if (!q[l] || !k[l] || !v[l] || !out[l] || !lse[l]) return DUALKV_ERR_INVALID;
    if (!aligned16(q[l]) || !aligned16(k[l]) || !aligned16(v[l]) || !aligned16(out[l]) || !aligned16(lse[l]))
      return DUALKV_ERR_ALIGN;
  }
  for (int l = 0; l < n_layers; ++l) {
    const int rc = fwd_impl(q[l], k[l], v[l], P, N, R_offsets, Hq, Hkv, D, scale, window[l], 0, Hkv, out[l], lse[l],
                            stream);
    if (rc) return rc;
  }
  return DUALKV_OK;
}

int dualkv_bwd_layers(int n_layers, const void* const* q, const void* const* k, const void* const* v,
                      const void* const* out, const float* const* lse, const void* const* dout, const int32_t* window,
                      int P, int N, const int32_t* R_offsets, int Hq, int Hkv, int D, float scale, void* const* dq,
                      void* const* dk, void* const* dv, void* workspace, size_t workspace_bytes, void* stream) {
  if (n_layers < 1 || !q || !k || !v || !out || !lse || !dout || !window || !dq || !dk || !dv)
    return DUALKV_ERR_INVALID;
  if (validate_layout(P, N, R_offsets, Hq, Hkv, D) || !supported_d(D)) return DUALKV_ERR_INVALID;
  for (int l = 0; l < n_layers; ++l) {
    const void* ptrs[9] = {q[l], k[l], v[l], out[l], lse[l], dout[l], dq[l], dk[l], dv[l]};
    for (const void* p : ptrs) {
      if (!p) return DUALKV_ERR_INVALID;
      if (!aligned16(p)) return DUALKV_ERR_ALIGN;
    }
  }
  const size_t need = dualkv_bwd_layers_workspace_bytes(n_layers, window, P, N, R_offsets, Hq, Hkv, D);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || need == 0 || workspace_bytes < need)
    return DUALKV_ERR_WORKSPACE;
  for (int l = 0; l < n_layers; ++l) {
    const int rc = bwd_impl(q[l], k[l], v[l], out[l], lse[l], dout[l], P, N, R_offsets, Hq, Hkv, D, scale, window[l],
                            0, Hkv, dq[l], dk[l], dv[l], workspace, workspace_bytes, stream);
    if (rc) return rc;
  }
  return DUALKV_OK;
}

int dualkv_build_index(int P, int N, const int32_t* R_offsets, int32_t* seg_id, int32_t* pos_id,
                       int32_t* cu_seqlens_rep, int32_t* rep2pack) {
  if (P < 0 || N < 1 || !R_offsets || R_offsets[0] != 0) return DUALKV_ERR_INVALID;
  for (int n = 0; n < N; ++n)
    if (R_offsets[n + 1] < R_offsets[n]) return DUALKV_ERR_INVALID;
  if ((int64_t)N * P + R_offsets[N] > INT32_MAX) return DUALKV_ERR_INVALID;
  build_index(P, N, R_offsets, seg_id, pos_id, cu_seqlens_rep, rep2pack);
  return DUALKV_OK;
}

double dualkv_rho(int P, int N, const int32_t* R_offsets) {
  if (P < 0 || N < 1 || !R_offsets || R_offsets[0] != 0) return -1.0;
  for (int n = 0; n < N; ++n)
    if (R_offsets[n + 1] < R_offsets[n]) return -1.0;
  const double packed = (double)P + R_offsets[N];
  if (packed <= 0) return -1.0;
  return ((double)N * P + R_offsets[N]) / packed;
}

int64_t dualkv_pairs(int P, int N, const int32_t* R_offsets, int window) {
  if (P < 0 || N < 1 || !R_offsets || R_offsets[0] != 0) return -1;
  for (int n = 0; n < N; ++n)
    if (R_offsets[n + 1] < R_offsets[n]) return -1;
  // keys attended by the query at position p: p + 1, or min(p + 1, window)
  auto upto = [window](int64_t len) -> int64_t {  // sum over positions 0..len-1
    if (window <= 0 || window >= len) return len * (len + 1) / 2;
    const int64_t w = window;
    return w * (w + 1) / 2 + (len - w) * w;
  };
  int64_t total = upto(P);
  for (int n = 0; n < N; ++n) {
    const int64_t R = R_offsets[n + 1] - R_offsets[n];
    total += upto((int64_t)P + R) - upto(P);
  }
  return total;
}

int dualkv_pack(const void* x_rep, void* x_packed, int P, int N, const int32_t* R_offsets, int row_elems,
                void* stream) {
  return pack_call(0, x_rep, x_packed, P, N, R_offsets, row_elems, stream);
}

int dualkv_unpack(const void* x_packed, void* x_rep, int P, int N, const int32_t* R_offsets, int row_elems,
                  void* stream) {
  return pack_call(1, x_packed, x_rep, P, N, R_offsets, row_elems, stream);
}

int dualkv_fold(const void* g_rep, void* g_packed, int P, int N, const int32_t* R_offsets, int row_elems,
                void* stream) {
  return pack_call(2, g_rep, g_packed, P, N, R_offsets, row_elems, stream);
}

int dualkv_check_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DUALKV_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DUALKV_ERR_CUDA;
  uint32_t* st = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (status_word(dev, &st)) return DUALKV_ERR_CUDA;
  }
  uint32_t h = 0;
  if (cudaMemcpy(&h, st, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return DUALKV_ERR_CUDA;
  if (h) {
    cudaMemset(st, 0, sizeof(uint32_t));
    return DUALKV_ERR_DEVICE;
  }
  return DUALKV_OK;
}

const char* dualkv_error_string(int code) {
  switch (code) {
    case DUALKV_OK:
      return "ok";
    case DUALKV_ERR_INVALID:
      return "invalid argument (sizes, offsets, head counts, head dimension or scale)";
    case DUALKV_ERR_ALIGN:
      return "a device pointer is not 16-byte aligned";
    case DUALKV_ERR_WORKSPACE:
      return "workspace missing, misaligned or too small";
    case DUALKV_ERR_CUDA:
      return "a CUDA runtime call or kernel launch failed";
    case DUALKV_ERR_DEVICE:
      return "a kernel reported a timed-out wait or an index out of range";
    case DUALKV_ERR_UNSUPPORTED:
      return "valid arguments outside what this library supports";
    default:
      return "unknown error code";
  }
}

int dualkv_selftest_timeout(uint64_t limit_ns, void* stream) {
  if (limit_ns < 1000000ull || limit_ns > 10000000000ull) return DUALKV_ERR_INVALID;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DUALKV_ERR_CUDA;
  uint32_t* status = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (status_word(dev, &status)) return DUALKV_ERR_CUDA;
  }
  if (launch_selftest_timeout(limit_ns, status, static_cast<cudaStream_t>(stream)) != cudaSuccess) return DUALKV_ERR_CUDA;
  return DUALKV_OK;
}

int dualkv_profile_enable(int on) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_profile = on != 0;
  return DUALKV_OK;
}

int dualkv_profile_read(double* ms, int64_t* launches) {
  std::lock_guard<std::mutex> lock(g_mu);
  int rc = DUALKV_OK;
  for (const TimedLaunch& t : g_timed) {
    float e = 0.f;
    if (cudaEventSynchronize(t.stop) != cudaSuccess || cudaEventElapsedTime(&e, t.start, t.stop) != cudaSuccess) {
      rc = DUALKV_ERR_CUDA;
    } else if (t.kind >= 0 && t.kind < DUALKV_KERNEL_KINDS) {
      if (ms) ms[t.kind] += e;
      if (launches) launches[t.kind] += 1;
    }
    g_event_pool.push_back(t.start);
    g_event_pool.push_back(t.stop);
  }
  g_timed.clear();
  return rc;
}

void dualkv_release(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (const TimedLaunch& t : g_timed) {
    g_event_pool.push_back(t.start);
    g_event_pool.push_back(t.stop);
  }
  g_timed.clear();
  for (cudaEvent_t e : g_event_pool) cudaEventDestroy(e);
  g_event_pool.clear();
  g_plans.clear();
  g_offsets.clear();
  for (auto& kv : g_status) cudaFree(kv.second);
  g_status.clear();
}

}  // extern "C"
