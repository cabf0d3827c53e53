// kernels.h -- launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "plan.h"

namespace dkv {

// Limit of every bounded wait in a normal launch (a healthy wait ends in microseconds).
constexpr uint64_t kLaunchWaitLimitNs = 2000000000ull;

struct FwdArgs {
  const QTileItem* items;
  __nv_bfloat16* out;
  float* lse;
  int T, Hq, Hkv, window;
  float scale_log2;  // softmax scale * log2(e)
  uint32_t* status;
  uint64_t wait_limit_ns = kLaunchWaitLimitNs;
  // failure-path self-test only (-1 otherwise): the K/V ring unit with this index is
  // never loaded, so the wait for it runs out after wait_limit_ns
  int test_skip_unit = -1;
};

// Query tile rows / key tile size of the forward kernel for head dimension D.
int fwd_query_tile(int D);
int fwd_key_tile(int D);
cudaError_t launch_fwd(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdArgs& a,
                       int n_items, cudaStream_t st);

struct PrepArgs {
  const __nv_bfloat16* out;
  const __nv_bfloat16* dout;
  const float* lse;
  float* delta;  // [Hq, T]
  float* lse2;   // [Hq, T], lse * log2(e)
  int64_t T;
  int Hq, D;
  int h_lo = 0, h_hi = -1;  // q-heads [h_lo, h_hi) are prepared (h_hi < 0: all)
  // the dQ work list to check (and to empty any entry outside the tensors) before the
  // dQ kernel runs; null: none
  QTileItem* check_items = nullptr;
  int n_check = 0, check_tile = 128;
  uint32_t* status = nullptr;
};
cudaError_t launch_prep(const PrepArgs& a, cudaStream_t st);

struct DqArgs {
  const QTileItem* items;
  const float* delta;
  const float* lse2;
  __nv_bfloat16* dq;
  int T, Hq, Hkv, window;
  float scale_log2;  // softmax scale * log2(e)
  float scale;       // softmax scale
  uint32_t* status;
  int n_items = 0;   // set by launch_dq
};
int dq_query_tile(int D);
int dq_key_tile(int D);
cudaError_t launch_dq(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const CUtensorMap& tdo, const DqArgs& a, int n_items, cudaStream_t st);

struct DkvArgs {
  const KVTileItem* items;
  const QBlock* qblocks;
  const float* delta;
  const float* lse2;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* partial;  // [slot][2][key_tile][D] fp32
  int T, Hq, Hkv, window;
  float scale_log2;
  float scale;
  uint32_t* status;
  int nslots = 0;  // partial slots in `partial` (work items naming another slot are out of range)
  uint64_t wait_limit_ns = kLaunchWaitLimitNs;
  // failure-path self-test only (-1 otherwise): the Q/dO block of this iteration of
  // the first work item gets one arrival too few, so the wait for it runs out
  int test_skip_iter = -1;
};
int dkv_key_tile(int D);
int dkv_query_block(int D);
cudaError_t launch_dkv(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const DkvArgs& a, int n_items, cudaStream_t st);

struct ReduceArgs {
  const ReduceItem* items;
  const float* partial;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int Hkv, D, key_tile;
  int64_t T = 0;        // rows of dk / dv
  int total_slots = 0;  // partial slots in `partial`
  uint32_t* status = nullptr;
};
cudaError_t launch_reduce(const ReduceArgs& a, int n_items, cudaStream_t st);

// ---- head dimension 512 backward (bwd512.cu)
struct PdsArgs {
  const QTileItem* items;
  const int32_t* block_base;
  const float* lse2;
  const float* delta;
  __nv_bfloat16* p_out;   // P blocks (written)
  __nv_bfloat16* ds_out;  // dS blocks (written)
  int T, Hq, Hkv, window;
  float scale_log2;
  uint32_t* status;
  int64_t n_blocks = 0;  // blocks in p_out and ds_out
  uint64_t wait_limit_ns = kLaunchWaitLimitNs;
  // failure-path self-test only (-1 otherwise): the K/V ring unit with this index is
  // never loaded, so the wait for it runs out after wait_limit_ns
  int test_skip_unit = -1;
};
// Both blocks of every (query tile, key tile) pair in one pass: P = exp(S - LSE)
// into a.p_out and dS = P (dP - Delta) into a.ds_out.
cudaError_t launch_pds_fused(const CUtensorMap& tq, const CUtensorMap& tdo, const CUtensorMap& tk,
                             const CUtensorMap& tv, const PdsArgs& a, int n_items, cudaStream_t st);

struct XtgArgs {
  const XTItem* items;
  const XTEntry* entries;
  __nv_bfloat16* out;  // dV or dK [T, Hkv, 512]
  float* partial;      // [slot][2][128][512]
  int region;          // partial half: 0 = dK, 1 = dV
  int T, Hq, Hkv;
  float mul;
  uint32_t* status;
  int64_t n_entries = 0;  // entries in `entries`
  int64_t n_blocks = 0;   // P / dS blocks the entries may name
  int nslots = 0;         // partial slots in `partial`
};
cudaError_t launch_xtg(const CUtensorMap& tBlk, const CUtensorMap& tB, const XtgArgs& a, int n_items, cudaStream_t st);

struct Dq512Args {
  const QTileItem* items;
  const int32_t* block_base;
  __nv_bfloat16* dq;
  int T, Hq, Hkv;
  float scale;
  uint32_t* status;
  int64_t n_blocks = 0;  // dS blocks
};
cudaError_t launch_dq512(const CUtensorMap& tBlk, const CUtensorMap& tK, const Dq512Args& a, int n_items,
                         cudaStream_t st);

// One CTA waits on an mbarrier that nothing completes, with a bounded wait of limit_ns.
cudaError_t launch_selftest_timeout(uint64_t limit_ns, uint32_t* status, cudaStream_t st);

// ---- per-token tensors between the replicated and the packed layout (pack.cu)
// kind 0 = pack (replicated -> packed), 1 = unpack (packed -> replicated),
// 2 = fold (replicated -> packed, prompt rows summed over the replicas).
// Rows are row_elems bf16 (a multiple of 8); d_off is R_offsets in device memory.
int pack_group_lanes(int row_elems);
cudaError_t launch_pack(int kind, const void* src, void* dst, const int32_t* d_off, int P, int N, int64_t T,
                        int row_elems, int num_sms, cudaStream_t st);

}  // namespace dkv
