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
#include "plan_cache.h"

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

// ---------------------------------------------------------------- plan cache
// Device memory of the plans comes from "blobs": one device buffer plus one
// pinned host buffer of the same capacity.  A plan's arrays are serialised
// into the host buffer and uploaded with a single cudaMemcpyAsync on the
// caller's stream (no synchronisation); an event recorded after the copy
// (`ready`) lets calls on other streams wait for it, and an event recorded
// after the last launch that read the plan (`last_use`) tells when its blob may
// be reused.  Evicted plans return their blobs to a small per-process pool, so
// a loop whose layout changes every call reuses the same few buffers instead
// of allocating.
struct Blob {
  int device = -1;
  void* d = nullptr;  // device
  void* h = nullptr;  // pinned host
  size_t cap = 0;
};

constexpr size_t kPlanCacheCapacity = 32;   // layouts whose plans stay resident
constexpr size_t kFreeBlobsKept = 16;       // released blobs kept for reuse

std::vector<Blob> g_free_blobs;
size_t g_blob_bytes = 0;  // device bytes held by all blobs (in use or pooled)

void free_blob(Blob& b) {
  if (b.d) cudaFree(b.d);
  if (b.h) cudaFreeHost(b.h);
  g_blob_bytes -= b.cap;
  b = Blob{};
}

// A blob of at least `bytes` on `device`: the smallest pooled one that fits, else a new one.
int acquire_blob(int device, size_t bytes, Blob* out) {
  size_t best = g_free_blobs.size();
  for (size_t i = 0; i < g_free_blobs.size(); ++i)
    if (g_free_blobs[i].device == device && g_free_blobs[i].cap >= bytes &&
        (best == g_free_blobs.size() || g_free_blobs[i].cap < g_free_blobs[best].cap))
      best = i;
  if (best < g_free_blobs.size()) {
    *out = g_free_blobs[best];
    g_free_blobs.erase(g_free_blobs.begin() + best);
    return DUALKV_OK;
  }
  Blob b;
  b.device = device;
  b.cap = ((bytes + bytes / 4) + 65535) & ~size_t(65535);  // headroom so later layouts fit
  if (cudaMalloc(&b.d, b.cap) != cudaSuccess) return DUALKV_ERR_CUDA;
  if (cudaMallocHost(&b.h, b.cap) != cudaSuccess) {
    cudaFree(b.d);
    return DUALKV_ERR_CUDA;
  }
  g_blob_bytes += b.cap;
  *out = b;
  return DUALKV_OK;
}

// Returns a blob whose last reader has finished to the pool; beyond kFreeBlobsKept
// the smallest pooled blobs are freed (large ones fit any later plan).
void release_blob(Blob& b) {
  if (!b.d) return;
  g_free_blobs.push_back(b);
  b = Blob{};
  while (g_free_blobs.size() > kFreeBlobsKept) {
    size_t small = 0;
    for (size_t i = 1; i < g_free_blobs.size(); ++i)
      if (g_free_blobs[i].cap < g_free_blobs[small].cap) small = i;
    free_blob(g_free_blobs[small]);
    g_free_blobs.erase(g_free_blobs.begin() + small);
  }
}

// Host-side serialisation of several arrays into one blob (16-byte aligned parts).
struct Packer {
  std::vector<uint8_t> bytes;
  template <typename T>
  size_t add(const std::vector<T>& v) {
    const size_t off = (bytes.size() + 15) & ~size_t(15);
    bytes.resize(off + sizeof(T) * v.size());
    if (!v.empty()) std::memcpy(bytes.data() + off, v.data(), sizeof(T) * v.size());
    return off;
  }
};

// One plan part (forward, or backward) in device memory.
struct PlanPart {
  Blob blob;
  cudaEvent_t ready = nullptr;  // recorded after the upload
  bool built = false;
};

struct DevPlan {
  int device = -1;
  cudaEvent_t last_use = nullptr;  // recorded after the last launch that read the plan
  PlanPart fwd, bwd;
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
  int64_t n_xt_entries = 0;
};

// Waits until no launch reads the plan any more, then returns its memory to the pool.
void retire_plan(DevPlan& pl) {
  for (PlanPart* part : {&pl.fwd, &pl.bwd}) {
    if (part->ready) {
      cudaEventSynchronize(part->ready);
      cudaEventDestroy(part->ready);
      part->ready = nullptr;
    }
  }
  if (pl.last_use) {
    cudaEventSynchronize(pl.last_use);
    cudaEventDestroy(pl.last_use);
    pl.last_use = nullptr;
  }
  release_blob(pl.fwd.blob);
  release_blob(pl.bwd.blob);
}

LruCache<DevPlan> g_plans(kPlanCacheCapacity);

struct DevOffsets {
  int32_t* d = nullptr;
  int num_sms = 0;
  PlanPart part;
  cudaEvent_t last_use = nullptr;
};
LruCache<DevOffsets> g_offsets(kPlanCacheCapacity);  // (device, P, N, R_offsets) -> device copy

void retire_offsets(DevOffsets& o) {
  if (o.part.ready) {
    cudaEventSynchronize(o.part.ready);
    cudaEventDestroy(o.part.ready);
    o.part.ready = nullptr;
  }
  if (o.last_use) {
    cudaEventSynchronize(o.last_use);
    cudaEventDestroy(o.last_use);
    o.last_use = nullptr;
  }
  release_blob(o.part.blob);
}

std::string plan_key(int device, int P, int N, const int32_t* off, int Hq, int Hkv, int D, int window, int kv_lo = 0,
                     int kv_hi = 0) {
  std::string k;
  k.reserve(64 + 4 * (N + 1));
  int32_t hdr[9] = {device, P, N, Hq, Hkv, D, window <= 0 ? 0 : window, kv_lo, kv_hi};
  k.append(reinterpret_cast<const char*>(hdr), sizeof(hdr));
  k.append(reinterpret_cast<const char*>(off), sizeof(int32_t) * (N + 1));
  return k;
}

// Serialised part -> pinned host buffer -> one asynchronous copy on `st`; records `ready`.
int upload_part(int device, const Packer& pk, cudaStream_t st, PlanPart* part) {
  const size_t bytes = pk.bytes.empty() ? 16 : pk.bytes.size();
  int rc = acquire_blob(device, bytes, &part->blob);
  if (rc) return rc;
  if (!pk.bytes.empty()) {
    std::memcpy(part->blob.h, pk.bytes.data(), pk.bytes.size());
    if (cudaMemcpyAsync(part->blob.d, part->blob.h, pk.bytes.size(), cudaMemcpyHostToDevice, st) != cudaSuccess) {
      cudaStreamSynchronize(st);  // the blob goes back to the pool: nothing may still copy into it
      release_blob(part->blob);
      return DUALKV_ERR_CUDA;
    }
  }
  if (!part->ready && cudaEventCreateWithFlags(&part->ready, cudaEventDisableTiming) != cudaSuccess)
    return DUALKV_ERR_CUDA;
  if (cudaEventRecord(part->ready, st) != cudaSuccess) return DUALKV_ERR_CUDA;
  part->built = true;
  return DUALKV_OK;
}

template <typename T>
T* at(const PlanPart& part, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(part.blob.d) + off);
}

// Orders `st` after the part's upload (a no-op once the copy has completed).
int wait_part(const PlanPart& part, cudaStream_t st) {
  if (part.ready && cudaStreamWaitEvent(st, part.ready, 0) != cudaSuccess) return DUALKV_ERR_CUDA;
  return DUALKV_OK;
}

// Marks the end of the launches that read the plan on `st`.
int mark_use(cudaEvent_t* ev, cudaStream_t st) {
  if (!*ev && cudaEventCreateWithFlags(ev, cudaEventDisableTiming) != cudaSuccess) return DUALKV_ERR_CUDA;
  return cudaEventRecord(*ev, st) == cudaSuccess ? DUALKV_OK : DUALKV_ERR_CUDA;
}

template <class V, class Retire>
void insert_retiring(LruCache<V>& cache, const std::string& key, std::unique_ptr<V> v, Retire retire) {
  std::vector<std::unique_ptr<V>> evicted;
  cache.insert(key, std::move(v), &evicted);
  for (auto& e : evicted) retire(*e);
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

// Looks up (or builds and uploads on `st`) the plan of a layout restricted to kv-heads
// [kv_lo, kv_hi), and orders `st` after its uploads; caller holds g_mu.
int get_plan(int P, int N, const int32_t* off, int Hq, int Hkv, int D, int window, int kv_lo, int kv_hi,
             bool need_bwd, cudaStream_t st, DevPlan** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DUALKV_ERR_CUDA;
  const std::string key = plan_key(dev, P, N, off, Hq, Hkv, D, window, kv_lo, kv_hi);
  DevPlan* pl = g_plans.find(key);
  if (!pl) {
    std::unique_ptr<DevPlan> fresh(new DevPlan());
    fresh->device = dev;
    pl = fresh.get();
    insert_retiring(g_plans, key, std::move(fresh), retire_plan);
  }
  Layout L{P, N, std::vector<int32_t>(off, off + N + 1), Hq, Hkv, D, window <= 0 ? 0 : window, kv_lo, kv_hi};
  int rc;
  if (!pl->fwd.built) {
    Packer pk;
    auto items = plan_qtiles(L, fwd_query_tile(D), fwd_key_tile(D));
    const size_t o_items = pk.add(items);
    if ((rc = upload_part(dev, pk, st, &pl->fwd))) return rc;
    pl->fwd_items = at<QTileItem>(pl->fwd, o_items);
    pl->n_fwd = (int)items.size();
  }
  if (need_bwd && !pl->bwd.built) {
    Packer pk;
    if (D == 512) {
      auto dq = plan_qtiles(L, 128, 128);
      Plan512 p5 = plan_512(L, dq, kMaxDkvIters);
      const size_t o_dq = pk.add(dq), o_bb = pk.add(p5.block_base), o_xi = pk.add(p5.items),
                   o_xe = pk.add(p5.entries), o_red = pk.add(p5.reduces);
      if ((rc = upload_part(dev, pk, st, &pl->bwd))) return rc;
      pl->dq_items = at<QTileItem>(pl->bwd, o_dq);
      pl->n_dq = (int)dq.size();
      pl->block_base = at<int32_t>(pl->bwd, o_bb);
      pl->xt_items = at<XTItem>(pl->bwd, o_xi);
      pl->xt_entries = at<XTEntry>(pl->bwd, o_xe);
      pl->reduces = at<ReduceItem>(pl->bwd, o_red);
      pl->n_blocks = p5.n_blocks;
      pl->n_xt_entries = (int64_t)p5.entries.size();
      pl->n_xt = (int)p5.items.size();
      pl->n_reduce = (int)p5.reduces.size();
      pl->nslots = p5.nslots;
    } else {
      auto dq = plan_qtiles(L, dq_query_tile(D), dq_key_tile(D));
      KVPlan kv = plan_kvtiles(L, dkv_key_tile(D), dkv_query_block(D), kMaxDkvIters);
      const size_t o_dq = pk.add(dq), o_kv = pk.add(kv.items), o_qb = pk.add(kv.qblocks), o_red = pk.add(kv.reduces);
      if ((rc = upload_part(dev, pk, st, &pl->bwd))) return rc;
      pl->dq_items = at<QTileItem>(pl->bwd, o_dq);
      pl->n_dq = (int)dq.size();
      pl->kv_items = at<KVTileItem>(pl->bwd, o_kv);
      pl->qblocks = at<QBlock>(pl->bwd, o_qb);
      pl->reduces = at<ReduceItem>(pl->bwd, o_red);
      pl->n_kv = (int)kv.items.size();
      pl->n_reduce = (int)kv.reduces.size();
      pl->nslots = kv.nslots;
    }
  }
  if ((rc = wait_part(pl->fwd, st))) return rc;
  if (need_bwd && (rc = wait_part(pl->bwd, st))) return rc;
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
// A P / dS block is 16 column groups x 128 rows x 8 keys; seen here as
// [block][group][row quarter][32 rows x 8 keys].  box_rows = 64: 64 rows, all 16
// groups (a transposed-GEMM stage); box_rows = 128: all rows, 8 groups (a dQ stage).
int make_block_tmap(CUtensorMap* m, const void* base, int64_t n_blocks, int box_rows) {
  cuuint64_t dims[4] = {256, 4, 16, (cuuint64_t)n_blocks};
  cuuint64_t strides[3] = {512, 2048, 32768};
  cuuint32_t box[4] = {256, (cuuint32_t)(box_rows / 32), box_rows == 64 ? 16u : 8u, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DUALKV_OK : DUALKV_ERR_CUDA;
}

// Device copy of R_offsets and the SM count for the pack kernels, ordered on `st`
// after its upload; caller holds g_mu.
int get_offsets(int P, int N, const int32_t* off, cudaStream_t st, DevOffsets** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DUALKV_ERR_CUDA;
  const std::string key = plan_key(dev, P, N, off, 0, 0, 0, 0);
  DevOffsets* o = g_offsets.find(key);
  if (!o) {
    std::unique_ptr<DevOffsets> fresh(new DevOffsets());
    if (cudaDeviceGetAttribute(&fresh->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return DUALKV_ERR_CUDA;
    Packer pk;
    const size_t o_off = pk.add(std::vector<int32_t>(off, off + N + 1));
    const int rc = upload_part(dev, pk, st, &fresh->part);
    if (rc) {
      retire_offsets(*fresh);
      return rc;
    }
    fresh->d = at<int32_t>(fresh->part, o_off);
    o = fresh.get();
    insert_retiring(g_offsets, key, std::move(fresh), retire_offsets);
  }
  const int rc = wait_part(o->part, st);
  if (rc) return rc;
  *out = o;
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
  int rc = get_offsets(P, N, off, st, &o);
  if (rc) return rc;
  if (timed(DUALKV_KERNEL_PACK, st, [&] {
        return launch_pack(kind, src, dst, o->d, P, N, T, row_elems, o->num_sms, st);
      }) != cudaSuccess)
    return DUALKV_ERR_CUDA;
  return mark_use(&o->last_use, st);
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
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_mu);
  int rc = ensure_encode();
  if (rc) return rc;
  DevPlan* pl = nullptr;
  if ((rc = get_plan(P, N, R_offsets, Hq, Hkv, D, window, kv_lo, kv_hi, false, st, &pl))) return rc;
  uint32_t* status = nullptr;
  if ((rc = status_word(pl->device, &status))) return rc;
  CUtensorMap tq, tk, tv;
  if (make_tmap(&tq, q, T, Hq, D, fwd_query_tile(D)) || make_tmap(&tk, k, T, Hkv, D, fwd_key_tile(D)) ||
      make_tmap(&tv, v, T, Hkv, D, fwd_key_tile(D)))
    return DUALKV_ERR_CUDA;
  FwdArgs a{pl->fwd_items, static_cast<__nv_bfloat16*>(out), lse, (int)T, Hq, Hkv, window <= 0 ? 0 : window,
            scale * 1.4426950408889634f, status};
  if (timed(DUALKV_KERNEL_FWD, st, [&] { return launch_fwd(D, tq, tk, tv, a, pl->n_fwd, st); }) != cudaSuccess)
    return DUALKV_ERR_CUDA;
  return mark_use(&pl->last_use, st);
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
  if ((rc = get_plan(P, N, R_offsets, Hq, Hkv, D, window, kv_lo, kv_hi, true, st, &pl))) return rc;
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
  if (D != 512) {  // the dQ kernel's work list is checked by the preprocess
    pa.check_items = pl->dq_items;
    pa.n_check = pl->n_dq;
    pa.check_tile = dq_query_tile(D);
    pa.status = status;
  }
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
    PdsArgs pa5{pl->dq_items, pl->block_base, lse2, delta, pblk, dsblk, (int)T, Hq, Hkv, W, sl2, status,
                pl->n_blocks};
    XtgArgs xv{pl->xt_items, pl->xt_entries, static_cast<__nv_bfloat16*>(dv), partial, 1, (int)T, Hq, Hkv, 1.f, status,
               pl->n_xt_entries, pl->n_blocks, pl->nslots};
    XtgArgs xk{pl->xt_items, pl->xt_entries, static_cast<__nv_bfloat16*>(dk), partial, 0, (int)T, Hq, Hkv, scale, status,
               pl->n_xt_entries, pl->n_blocks, pl->nslots};
    Dq512Args qa{pl->dq_items, pl->block_base, static_cast<__nv_bfloat16*>(dq), (int)T, Hq, Hkv, scale, status,
                 pl->n_blocks};
    if (timed(DUALKV_KERNEL_DKV, st, [&] {
          cudaError_t e = launch_pds_fused(tq, tdo, tk, tv, pa5, pl->n_dq, st);
          if (e == cudaSuccess) e = launch_xtg(tP64, tdo64, xv, pl->n_xt, st);
          if (e == cudaSuccess) e = launch_xtg(tDS64, tq64, xk, pl->n_xt, st);
          return e;
        }) != cudaSuccess)
      return DUALKV_ERR_CUDA;
    if (pl->n_reduce > 0) {
      ReduceArgs ra{pl->reduces, partial, static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv), Hkv, D, 128,
                    T, pl->nslots, status};
      if (timed(DUALKV_KERNEL_REDUCE, st, [&] { return launch_reduce(ra, pl->n_reduce, st); }) != cudaSuccess)
        return DUALKV_ERR_CUDA;
    }
    if (timed(DUALKV_KERNEL_DQ, st, [&] { return launch_dq512(tDS128, tk64, qa, pl->n_dq, st); }) != cudaSuccess)
      return DUALKV_ERR_CUDA;
    return mark_use(&pl->last_use, st);
  }

  CUtensorMap tq, tk, tv, tdo;
  if (make_tmap(&tq, q, T, Hq, D, dkv_query_block(D)) || make_tmap(&tk, k, T, Hkv, D, dkv_key_tile(D)) ||
      make_tmap(&tv, v, T, Hkv, D, dkv_key_tile(D)) || make_tmap(&tdo, dout, T, Hq, D, dkv_query_block(D)))
    return DUALKV_ERR_CUDA;
  DkvArgs ka{pl->kv_items, pl->qblocks, delta, lse2, static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv),
             partial, (int)T, Hq, Hkv, W, sl2, scale, status, pl->nslots};
  if (timed(DUALKV_KERNEL_DKV, st, [&] { return launch_dkv(D, tq, tk, tv, tdo, ka, pl->n_kv, st); }) != cudaSuccess)
    return DUALKV_ERR_CUDA;
  if (pl->n_reduce > 0) {
    ReduceArgs ra{pl->reduces, partial, static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv), Hkv, D,
                  dkv_key_tile(D), T, pl->nslots, status};
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
  return mark_use(&pl->last_use, st);
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

int dualkv_plan_cache_info(int* n_plans, int64_t* device_bytes) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (n_plans) *n_plans = (int)g_plans.size();
  if (device_bytes) *device_bytes = (int64_t)g_blob_bytes;
  return DUALKV_OK;
}

// The head-dimension-512 P / dS pass on a tiny layout (zero inputs, P = 128, two
// responses of 128, one head) whose first K/V ring unit is never loaded.
static int selftest_pds512(uint64_t limit_ns, cudaStream_t st, uint32_t* status) {
  constexpr int P = 128, N = 2, Hq = 1, Hkv = 1, D = 512;
  const int32_t off[N + 1] = {0, 128, 256};
  constexpr int64_t T = P + 256;
  DevPlan* pl = nullptr;
  int rc = get_plan(P, N, off, Hq, Hkv, D, 0, 0, Hkv, true, st, &pl);
  if (rc) return rc;
  const size_t tensor_bytes = (size_t)T * Hq * D * 2;
  const WsLayout ws = ws_layout(T, Hq, D, pl->nslots, pl->n_blocks);
  const size_t o_lse = 5 * tensor_bytes, o_ws = align256(o_lse + sizeof(float) * Hq * T),
               total = o_ws + align256(ws.total);
  uint8_t* mem = nullptr;
  if (cudaMalloc(&mem, total) != cudaSuccess) return DUALKV_ERR_CUDA;
  auto done = [&](int code) {
    cudaStreamSynchronize(st);
    cudaFree(mem);
    return code;
  };
  if (cudaMemsetAsync(mem, 0, total, st) != cudaSuccess) return done(DUALKV_ERR_CUDA);
  void *q = mem, *k = mem + tensor_bytes, *v = mem + 2 * tensor_bytes, *out = mem + 3 * tensor_bytes,
       *dout = mem + 4 * tensor_bytes;
  float* lse = reinterpret_cast<float*>(mem + o_lse);
  uint8_t* wsb = mem + o_ws;
  float* delta = reinterpret_cast<float*>(wsb + ws.delta);
  float* lse2 = reinterpret_cast<float*>(wsb + ws.lse2);
  PrepArgs pa{static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), lse, delta, lse2, T, Hq, D};
  if (launch_prep(pa, st) != cudaSuccess) return done(DUALKV_ERR_CUDA);
  CUtensorMap tq, tk, tv, tdo;
  if (make_tmap(&tq, q, T, Hq, D, 128) || make_tmap(&tk, k, T, Hkv, D, 128) || make_tmap(&tv, v, T, Hkv, D, 128) ||
      make_tmap(&tdo, dout, T, Hq, D, 128))
    return done(DUALKV_ERR_CUDA);
  PdsArgs a{pl->dq_items, pl->block_base, lse2, delta,
            reinterpret_cast<__nv_bfloat16*>(wsb + ws.pblk), reinterpret_cast<__nv_bfloat16*>(wsb + ws.dsblk),
            (int)T, Hq, Hkv, 0, 0.04419417382415922f * 1.4426950408889634f, status, pl->n_blocks};
  a.wait_limit_ns = limit_ns;
  a.test_skip_unit = 0;
  if (launch_pds_fused(tq, tdo, tk, tv, a, pl->n_dq, st) != cudaSuccess) return done(DUALKV_ERR_CUDA);
  return done(mark_use(&pl->last_use, st));
}

int dualkv_selftest_kernel(int which, uint64_t limit_ns, void* stream) {
  if (which < 0 || which > 4) return DUALKV_ERR_INVALID;
  if (limit_ns < 1000000ull || limit_ns > 10000000000ull) return DUALKV_ERR_INVALID;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_mu);
  int rc = ensure_encode();
  if (rc) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DUALKV_ERR_CUDA;
  uint32_t* status = nullptr;
  if ((rc = status_word(dev, &status))) return rc;
  if (which == 4) return selftest_pds512(limit_ns, st, status);
  // a tiny layout with zero inputs: P = 128 and two responses of 128, one head, D = 128
  constexpr int P = 128, N = 2, Hq = 1, Hkv = 1, D = 128;
  const int32_t off[N + 1] = {0, 128, 256};
  constexpr int64_t T = P + 256;
  const float scale = 0.08838834764831845f;
  DevPlan* pl = nullptr;
  if ((rc = get_plan(P, N, off, Hq, Hkv, D, 0, 0, Hkv, which == 1 || which == 3, st, &pl))) return rc;
  const size_t tensor_bytes = (size_t)T * Hq * D * 2;
  const WsLayout ws = ws_layout(T, Hq, D, pl->nslots, 0);
  uint8_t* mem = nullptr;
  const size_t o_lse = 7 * tensor_bytes, o_ws = align256(o_lse + sizeof(float) * Hq * T),
               o_items = o_ws + align256(ws.total),
               total = o_items + align256(sizeof(QTileItem) * (pl->n_fwd > pl->n_dq ? pl->n_fwd : pl->n_dq));
  if (cudaMalloc(&mem, total) != cudaSuccess) return DUALKV_ERR_CUDA;
  auto done = [&](int code) {
    cudaStreamSynchronize(st);
    cudaFree(mem);
    return code;
  };
  if (cudaMemsetAsync(mem, 0, total, st) != cudaSuccess) return done(DUALKV_ERR_CUDA);
  void *q = mem, *k = mem + tensor_bytes, *v = mem + 2 * tensor_bytes, *out = mem + 3 * tensor_bytes,
       *dout = mem + 4 * tensor_bytes, *dk = mem + 5 * tensor_bytes, *dv = mem + 6 * tensor_bytes;
  float* lse = reinterpret_cast<float*>(mem + o_lse);
  uint8_t* wsb = mem + o_ws;
  CUtensorMap tq, tk, tv, tdo;
  if (which == 3) {
    // dQ: its work list's first entry moved past the last row; the preprocess, which
    // checks the list before the dQ kernel reads it, empties the entry
    Layout L{P, N, std::vector<int32_t>(off, off + N + 1), Hq, Hkv, D, 0};
    std::vector<QTileItem> bad = plan_qtiles(L, dq_query_tile(D), dq_key_tile(D));
    bad[0].q_row0 = (int32_t)T + 64;
    QTileItem* d_items = reinterpret_cast<QTileItem*>(mem + o_items);
    if (cudaMemcpyAsync(d_items, bad.data(), sizeof(QTileItem) * bad.size(), cudaMemcpyHostToDevice, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return done(DUALKV_ERR_CUDA);
    float* delta = reinterpret_cast<float*>(wsb + ws.delta);
    float* lse2 = reinterpret_cast<float*>(wsb + ws.lse2);
    PrepArgs pa{static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), lse, delta, lse2, T,
                Hq, D};
    pa.check_items = d_items;
    pa.n_check = (int)bad.size();
    pa.check_tile = dq_query_tile(D);
    pa.status = status;
    if (launch_prep(pa, st) != cudaSuccess) return done(DUALKV_ERR_CUDA);
    if (make_tmap(&tq, q, T, Hq, D, dq_query_tile(D)) || make_tmap(&tk, k, T, Hkv, D, dq_key_tile(D)) ||
        make_tmap(&tv, v, T, Hkv, D, dq_key_tile(D)) || make_tmap(&tdo, dout, T, Hq, D, dq_query_tile(D)))
      return done(DUALKV_ERR_CUDA);
    DqArgs qa{d_items, delta, lse2, static_cast<__nv_bfloat16*>(dk), (int)T, Hq, Hkv, 0,
              scale * 1.4426950408889634f, scale, status};
    if (launch_dq(D, tq, tk, tv, tdo, qa, (int)bad.size(), st) != cudaSuccess) return done(DUALKV_ERR_CUDA);
    return done(mark_use(&pl->last_use, st));
  }
  if (which != 1) {
    // forward: every CTA waits for K/V unit 0, which is never loaded (which = 0), or the
    // first work item is moved past the last row (which = 2)
    const QTileItem* items = pl->fwd_items;
    if (which == 2) {
      Layout L{P, N, std::vector<int32_t>(off, off + N + 1), Hq, Hkv, D, 0};
      std::vector<QTileItem> bad = plan_qtiles(L, fwd_query_tile(D), fwd_key_tile(D));
      bad[0].q_row0 = (int32_t)T + 64;
      QTileItem* d_items = reinterpret_cast<QTileItem*>(mem + o_items);
      if (cudaMemcpyAsync(d_items, bad.data(), sizeof(QTileItem) * bad.size(), cudaMemcpyHostToDevice, st) !=
              cudaSuccess ||
          cudaStreamSynchronize(st) != cudaSuccess)
        return done(DUALKV_ERR_CUDA);
      items = d_items;
    }
    if (make_tmap(&tq, q, T, Hq, D, fwd_query_tile(D)) || make_tmap(&tk, k, T, Hkv, D, fwd_key_tile(D)) ||
        make_tmap(&tv, v, T, Hkv, D, fwd_key_tile(D)))
      return done(DUALKV_ERR_CUDA);
    FwdArgs a{items, static_cast<__nv_bfloat16*>(out), lse, (int)T, Hq, Hkv, 0, scale * 1.4426950408889634f, status};
    a.wait_limit_ns = limit_ns;
    if (which == 0) a.test_skip_unit = 0;
    if (launch_fwd(D, tq, tk, tv, a, pl->n_fwd, st) != cudaSuccess) return done(DUALKV_ERR_CUDA);
    return done(mark_use(&pl->last_use, st));
  }
  // dK/dV: the first work item's first Q/dO block gets one arrival too few
  float* delta = reinterpret_cast<float*>(wsb + ws.delta);
  float* lse2 = reinterpret_cast<float*>(wsb + ws.lse2);
  PrepArgs pa{static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), lse, delta, lse2, T, Hq, D};
  if (launch_prep(pa, st) != cudaSuccess) return done(DUALKV_ERR_CUDA);
  if (make_tmap(&tq, q, T, Hq, D, dkv_query_block(D)) || make_tmap(&tk, k, T, Hkv, D, dkv_key_tile(D)) ||
      make_tmap(&tv, v, T, Hkv, D, dkv_key_tile(D)) || make_tmap(&tdo, dout, T, Hq, D, dkv_query_block(D)))
    return done(DUALKV_ERR_CUDA);
  DkvArgs ka{pl->kv_items, pl->qblocks, delta, lse2, static_cast<__nv_bfloat16*>(dk),
             static_cast<__nv_bfloat16*>(dv), reinterpret_cast<float*>(wsb + ws.partial), (int)T, Hq, Hkv, 0,
             scale * 1.4426950408889634f, scale, status, pl->nslots};
  ka.wait_limit_ns = limit_ns;
  ka.test_skip_iter = 0;
  if (launch_dkv(D, tq, tk, tv, tdo, ka, pl->n_kv, st) != cudaSuccess) return done(DUALKV_ERR_CUDA);
  return done(mark_use(&pl->last_use, st));
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
  {
    std::vector<std::unique_ptr<DevPlan>> plans;
    g_plans.clear(&plans);
    for (auto& p : plans) retire_plan(*p);
    std::vector<std::unique_ptr<DevOffsets>> offs;
    g_offsets.clear(&offs);
    for (auto& o : offs) retire_offsets(*o);
    for (Blob& b : g_free_blobs) free_blob(b);
    g_free_blobs.clear();
  }
  for (auto& kv : g_status) cudaFree(kv.second);
  g_status.clear();
}

}  // extern "C"
