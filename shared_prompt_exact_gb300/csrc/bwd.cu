// bwd.cu -- DualKV backward kernels for sm_103a (head dimension 64 / 128).
//
// The packed backward equals the analytic backward of standard attention on
// the N replicated sequences with the prompt gradients summed over replicas
// (DualKV paper, abstract: packing changes nothing in the result, which is
// exactly that of ordinary attention on the replicated sequences).
// With P_ij = exp(S_ij - LSE_i), dP_ij = dO_i . v_j, Delta_i = dO_i . O_i and
// dS_ij = P_ij (dP_ij - Delta_i):
//   dQ_i = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i,   dV_j = sum_i P_ij dO_i.
// A prompt key j is attended by prompt queries and by the queries of every
// segment, so its dK/dV sum over all of them -- which is exactly the fold of
// the replicated prompt gradients.
//
// Kernels: prep (Delta and log2-scaled LSE), dkv (one CTA per key tile and
// chunk of its query walk; fixed walk order: for a prompt key tile every
// segment's query blocks, then the prompt's; the group's heads of one block
// consecutively), reduce (fixed-order sum of split chunks), dq (one CTA per
// query tile; same key walk as the forward).
#include <cuda_bf16.h>

#include "checks.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dkv {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- prep
// Delta[h, t] = sum_d dO[t,h,d] * O[t,h,d];  lse2[h, t] = lse[h, t] * log2(e)
// The dQ kernel's work list is checked here, in the launch that always precedes it:
// an entry whose rows, head or key tiles fall outside the tensors is recorded as a
// bounds error and replaced by an empty item (no key tiles, no rows), which the dQ
// kernel skips without any access.
__device__ __forceinline__ void sanitize_items(const PrepArgs& a) {
  if (!a.check_items) return;
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < a.n_check; i += nthreads) {
    QTileItem it = a.check_items[i];
    if (!qtile_ok(it, a.T, a.Hq, a.check_tile, a.check_tile)) {
      if (a.status) atomicOr(a.status, kDevErrBounds);
      it.q_row0 = 0;
      it.q_rows = 0;
      it.head = 0;
      it.reg[0] = KeyRegion{0, 0, 0, 0, 0};
      it.reg[1] = KeyRegion{0, 0, 0, 0, 0};
      a.check_items[i] = it;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(256) prep_kernel(const PrepArgs a) {
  sanitize_items(a);
  constexpr int LPR = (D / 8) < 32 ? (D / 8) : 32;  // lanes per row
  constexpr int PASSES = D / (8 * LPR);
  constexpr int RPW = 32 / LPR;                       // rows per warp
  const int h_hi = a.h_hi < 0 ? a.Hq : a.h_hi;
  const int nh = h_hi - a.h_lo;
  const int64_t nrows = a.T * nh;
  const int64_t warp_global = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x / 32);
  const int sub = (threadIdx.x & 31) / LPR, l = (threadIdx.x & 31) % LPR;
  const int64_t r = warp_global * RPW + sub;  // row = t * nh + (h - h_lo)
  const int64_t t = r / nh;
  const int h = a.h_lo + (int)(r % nh);
  float acc = 0.f;
  if (r < nrows) {
    const uint4* po = reinterpret_cast<const uint4*>(a.out + (t * a.Hq + h) * D);
    const uint4* pd = reinterpret_cast<const uint4*>(a.dout + (t * a.Hq + h) * D);
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      const uint4 o = po[p * LPR + l], g = pd[p * LPR + l];
      const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&o);
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 of = __bfloat1622float2(o2[e]), gf = __bfloat1622float2(g2[e]);
        acc = fmaf(of.x, gf.x, acc);
        acc = fmaf(of.y, gf.y, acc);
      }
    }
  }
#pragma unroll
  for (int s = LPR / 2; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (r < nrows && l == 0) {
    a.delta[(int64_t)h * a.T + t] = acc;
    a.lse2[(int64_t)h * a.T + t] = a.lse[(int64_t)h * a.T + t] * kLog2e;
  }
}

// Shared structure of the dQ and dK/dV kernels (352 threads):
//   warp 0      TMA producer
//   warp 1      TMEM owner and issuer of the first GEMM pair (S and dP)
//   warp 10     issuer of the second GEMM pair (dQ, or dV and dK)
//   warps 2-9   compute: warps w and w+4 share TMEM lane quarter w % 4 (one row
//               per thread) and split the columns of a block into halves
// An issuing thread stalls while the tensor pipe's queue is full; with one
// issuer per GEMM group the pipe keeps working while either waits for its
// operands.  Descriptors are computed once per tile and advanced by constant
// adds inside unrolled loops.
// The first GEMM pair writes two double-buffered fp32 blocks to TMEM; the
// compute warps read them, and write the bf16 result (dS, or P^T and dS^T)
// back over the same buffer, where the second GEMM reads it as its A operand.
// Half h reads fp32 columns [32h, 32h+32) and writes its 32 bf16 values
// (16 packed columns) to [32h, 32h+16): a warp only overwrites columns it has
// read itself, so the two halves need no synchronisation with each other.
// K-step k of the second GEMM (16 values) therefore sits at column
// 32 (k / 2) + 8 (k % 2).  tcgen05.mma ops issued by one thread execute in
// issue order, so a buffer is rewritten by the next first-pair GEMM only
// after the second GEMM that reads it.
constexpr int kBwdThreads = 352;

__device__ __forceinline__ uint32_t packed_kstep_col(int k) { return 32u * (k >> 1) + 8u * (k & 1); }

// ---------------------------------------------------------------- dQ
// 128-key tiles: S and dP are M=128 x N=128 MMAs.  S and dP each have one TMEM
// buffer, released as soon as the compute warps have loaded them, so the next
// tile's S and dP run while the compute warps work.  S = Q K^T takes Q from
// TMEM (a TS MMA reads only K from shared memory; the SS form was bound by
// shared-memory operand reads); the compute warps copy each item's Q tile there
// from its TMA landing buffer.  dS goes to its own buffer, written once the
// previous tile's dQ GEMM has completed.  NG compute warps share each TMEM lane
// quarter; each thread handles BN / NG key columns of its query row (two warps
// per quarter measured fastest: four were slower).
// The kernel is persistent: CTA c takes work items c, c + grid, c + 2 grid, ...
// of the cost-sorted list, and the pipeline runs on across items (ring slots
// and barrier phases follow a tile counter over all of the CTA's tiles), so
// one item's epilogue overlaps the next item's first GEMMs.  Q and dO of the
// next item are loaded once every GEMM that reads the current ones is done
// (q_free), and its first dQ GEMM waits until the compute warps have read the
// current dQ accumulator (dq_free).
template <int D>
struct DqCfg {
  static constexpr int BM = 128, BN = 128;
  static constexpr int NG = 2;                       // compute warps per TMEM lane quarter
  static constexpr int GC = BN / NG;                 // key columns of one compute warp
  static constexpr int THREADS = 96 + 128 * NG;  // producer, two MMA issuers, compute
  static_assert(THREADS == kBwdThreads, "warp roles assume 11 warps");
  static constexpr int KCH = D / 64;
  static constexpr int Q_BYTES = BM * D * 2;         // Q and dO tiles (resident)
  static constexpr int TILE_BYTES = BN * D * 2;      // one K or V tile
  // K tiles stay until their dQ GEMM (a step later), V tiles only until dP:
  // separate rings keep a slow-to-free K slot from holding up the next V load
  static constexpr int NSK = (D == 128) ? 3 : 6;
  static constexpr int NSV = (D == 128) ? 2 : 6;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + Q_BYTES;
  static constexpr int OFF_KR = OFF_DO + Q_BYTES;
  static constexpr int OFF_VR = OFF_KR + NSK * TILE_BYTES;
  static constexpr int SMEM_BYTES = OFF_VR + NSV * TILE_BYTES + 1024;
  // TMEM: S | dP (BN columns each) | dS (BN / 2 packed, single buffer) | Q (D / 2: A operand of S) | dQ (D)
  static constexpr uint32_t TM_S = 0, TM_DP = BN, TM_DS = 2 * BN, TM_Q = 2 * BN + BN / 2, TM_DQ = 3 * BN,
                            TM_COLS = 512;
  static_assert(TM_Q + D / 2 <= TM_DQ && TM_DQ + D <= TM_COLS, "TMEM budget");
};

struct DqSmemCtl {
  uint64_t q_full;
  uint64_t k_full[6], k_empty[6], v_full[6], v_empty[6];
  uint64_t q_free, q_tmem, s_full, dp_full, s_empty, dp_empty, ds_full, ds_done;
  uint64_t acc_done, dq_free, drain, drain2;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void qtile_of(const QTileItem& it, int j, int& r, int& t) {
  const int n0 = it.reg[0].t_hi - it.reg[0].t_lo;
  if (j < n0) {
    r = 0;
    t = it.reg[0].t_lo + j;
  } else {
    r = 1;
    t = it.reg[1].t_lo + (j - n0);
  }
}

template <int D>
__global__ void __launch_bounds__(DqCfg<D>::THREADS, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO, const DqArgs a) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ DqSmemCtl ctl;
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sDO = smem + C::OFF_DO;
  uint8_t* sKR = smem + C::OFF_KR;
  uint8_t* sVR = smem + C::OFF_VR;

  const uint32_t warp = warp_id(), lane = lane_id();
  FailState fs{&ctl.abort_flag, a.status};
  auto tiles_of = [](const QTileItem& q) {
    return (q.reg[0].t_hi - q.reg[0].t_lo) + (q.reg[1].t_hi - q.reg[1].t_lo);
  };

  if (threadIdx.x == 0) {
    ctl.abort_flag = 0;
    mbar_init(&ctl.q_full, 1);
    mbar_init(&ctl.q_free, 1);
    mbar_init(&ctl.q_tmem, 4 * C::NG);
    for (int i = 0; i < C::NSK; ++i) {
      mbar_init(&ctl.k_full[i], 1);
      mbar_init(&ctl.k_empty[i], 1);
    }
    for (int i = 0; i < C::NSV; ++i) {
      mbar_init(&ctl.v_full[i], 1);
      mbar_init(&ctl.v_empty[i], 1);
    }
    mbar_init(&ctl.s_full, 1);
    mbar_init(&ctl.dp_full, 1);
    mbar_init(&ctl.s_empty, 4 * C::NG);
    mbar_init(&ctl.dp_empty, 4 * C::NG);
    mbar_init(&ctl.ds_full, 4 * C::NG);
    mbar_init(&ctl.ds_done, 1);
    mbar_init(&ctl.acc_done, 1);
    mbar_init(&ctl.dq_free, 4 * C::NG);
    mbar_init(&ctl.drain, 1);
    mbar_init(&ctl.drain2, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl.tmem_base, C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;

  // Every role walks the same items; `kx` counts items with at least one key
  // tile and `g` the tiles over all of them.
  if (warp == 0) {
    // producer: per item Q and dO, then K_j (K ring) and V_j (V ring)
    if (lane == 0) {
      bool ok = true;
      int g = 0, kx = 0, nk = 0, nv = 0;
      for (int item = blockIdx.x; item < a.n_items && ok; item += gridDim.x) {
        const QTileItem it = a.items[item];
        const int nt = tiles_of(it);
        if (nt == 0) continue;
        const int kvh = it.head / (a.Hq / a.Hkv);
        // Q / dO are overwritten only after every GEMM of the previous item has completed
        if (kx > 0 && !(ok = mbar_wait(&ctl.q_free, (kx - 1) & 1, fs))) break;
        mbar_arrive_expect_tx(&ctl.q_full, 2 * C::Q_BYTES);
        for (int c = 0; c < C::KCH; ++c) {
          tma_load_3d(sQ + c * C::BM * 128, &tmQ, &ctl.q_full, c * 64, it.head, it.q_row0);
          tma_load_3d(sDO + c * C::BM * 128, &tmDO, &ctl.q_full, c * 64, it.head, it.q_row0);
        }
        ++kx;
        for (int j = 0; j < nt && ok; ++j, ++g) {
          int r, t;
          qtile_of(it, j, r, t);
          const int key_row = it.reg[r].row0 + t * C::BN;
          const int ks = g % C::NSK, vs = g % C::NSV;
          if (!(ok = mbar_wait(&ctl.k_empty[ks], ((g / C::NSK) & 1) ^ 1, fs))) break;
          mbar_arrive_expect_tx(&ctl.k_full[ks], C::TILE_BYTES);
          for (int c = 0; c < C::KCH; ++c)
            tma_load_3d(sKR + ks * C::TILE_BYTES + c * C::BN * 128, &tmK, &ctl.k_full[ks], c * 64, kvh, key_row);
          ++nk;
          if (!(ok = mbar_wait(&ctl.v_empty[vs], ((g / C::NSV) & 1) ^ 1, fs))) break;
          mbar_arrive_expect_tx(&ctl.v_full[vs], C::TILE_BYTES);
          for (int c = 0; c < C::KCH; ++c)
            tma_load_3d(sVR + vs * C::TILE_BYTES + c * C::BN * 128, &tmV, &ctl.v_full[vs], c * 64, kvh, key_row);
          ++nv;
        }
      }
      if (!ok) {
        // drain: wait for the copies still in flight before the CTA can exit
        if (kx > 0) mbar_wait_drain(&ctl.q_full, (kx - 1) & 1, kWaitLimitNs);
        for (int back = 1; back <= C::NSK && back <= nk; ++back) {
          const int i2 = nk - back;
          mbar_wait_drain(&ctl.k_full[i2 % C::NSK], (i2 / C::NSK) & 1, kWaitLimitNs);
        }
        for (int back = 1; back <= C::NSV && back <= nv; ++back) {
          const int i2 = nv - back;
          mbar_wait_drain(&ctl.v_full[i2 % C::NSV], (i2 / C::NSV) & 1, kWaitLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    // S_j = Q K_j^T, then dP_j = dO V_j^T (SS, N = 128), each committed on its own
    // barrier.  A thread issuing tcgen05.mma stalls while the tensor pipe's queue is
    // full, so dQ has its own issuing warp (warp 10): the two never wait on each
    // other's operands and write disjoint TMEM.  Both run their loops warp-wide
    // (warp-uniform descriptors); one elected lane issues.
    constexpr uint32_t idS = idesc_bf16(128, C::BN, 0, 0);
    const uint64_t dDOd = sdesc_sw128(smem_u32(sDO), 16, 1024);
    const uint32_t aKR = smem_u32(sKR), aVR = smem_u32(sVR);
    bool ok = true;
    int g = 0, kx = 0;
    for (int item = blockIdx.x; item < a.n_items && ok; item += gridDim.x) {
      const int nt = tiles_of(a.items[item]);
      if (nt == 0) continue;
      // Q copied into TMEM (after its TMA load, which also brought dO)
      if (!(ok = mbar_wait(&ctl.q_tmem, kx & 1, fs))) break;
      ++kx;
      for (int j = 0; j < nt && ok; ++j, ++g) {
        const int ks = g % C::NSK, vs = g % C::NSV;
        if (!(ok = mbar_wait(&ctl.k_full[ks], (g / C::NSK) & 1, fs))) break;
        // one S buffer: the compute warps must have loaded the previous S
        if (g >= 1 && !(ok = mbar_wait(&ctl.s_empty, (g - 1) & 1, fs))) break;
        tc_fence_after();
        const uint64_t kd = sdesc_sw128(aKR + ks * C::TILE_BYTES, 16, 1024);
        if (elect_one()) {
#pragma unroll
          for (int c = 0; c < C::KCH; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16_ts(tmem + C::TM_S, tmem + C::TM_Q + 8 * (4 * c + k), sdesc_add(kd, c * C::BN * 128 + k * 32),
                          idS, (c | k) != 0);
          mma_commit(&ctl.s_full);
        }
        __syncwarp();
        // one dP buffer: the compute warps must have loaded the previous dP
        if (!(ok = mbar_wait(&ctl.v_full[vs], (g / C::NSV) & 1, fs))) break;
        if (g >= 1 && !(ok = mbar_wait(&ctl.dp_empty, (g - 1) & 1, fs))) break;
        tc_fence_after();
        const uint64_t vd = sdesc_sw128(aVR + vs * C::TILE_BYTES, 16, 1024);
        if (elect_one()) {
#pragma unroll
          for (int c = 0; c < C::KCH; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16_ss(tmem + C::TM_DP, sdesc_add(dDOd, c * C::BM * 128 + k * 32),
                          sdesc_add(vd, c * C::BN * 128 + k * 32), idS, (c | k) != 0);
          mma_commit(&ctl.v_empty[vs]);
          mma_commit(&ctl.dp_full);
          if (j == nt - 1) mma_commit(&ctl.q_free);  // this item's Q and dO are no longer read
        }
        __syncwarp();
      }
    }
    if (elect_one()) mma_commit(&ctl.drain);
    __syncwarp();
    mbar_wait_drain(&ctl.drain, 0, kWaitLimitNs);
  } else if (warp == 10) {
    // dQ += dS_j K_j (TS, N = D): A is the bf16 dS the compute warps wrote into buffer g % 2
    constexpr uint32_t idQ = idesc_bf16(128, D, 0, 1);
    const uint32_t aKR = smem_u32(sKR);
    bool ok = true;
    int g = 0, kx = 0;
    for (int item = blockIdx.x; item < a.n_items && ok; item += gridDim.x) {
      const int nt = tiles_of(a.items[item]);
      if (nt == 0) continue;
      for (int j = 0; j < nt && ok; ++j, ++g) {
        const int ks = g % C::NSK;
        if (!(ok = mbar_wait(&ctl.ds_full, g & 1, fs))) break;
        // the accumulator is reused once the previous item's dQ has been read out
        if (j == 0 && kx > 0 && !(ok = mbar_wait(&ctl.dq_free, (kx - 1) & 1, fs))) break;
        tc_fence_after();
        const uint64_t kmn = sdesc_sw128(aKR + ks * C::TILE_BYTES, C::BN * 128, 1024);
        const uint32_t tA = tmem + C::TM_DS;
        const uint32_t acc0 = j > 0 ? 1u : 0u;
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < C::BN / 16; ++k)
            mma_bf16_ts(tmem + C::TM_DQ, tA + 8 * k, sdesc_add(kmn, k * 16 * 128), idQ, k > 0 ? 1u : acc0);
          mma_commit(&ctl.k_empty[ks]);
          mma_commit(&ctl.ds_done);
          if (j == nt - 1) mma_commit(&ctl.acc_done);
        }
        __syncwarp();
      }
      ++kx;
    }
    if (elect_one()) mma_commit(&ctl.drain2);
    __syncwarp();
    mbar_wait_drain(&ctl.drain2, 0, kWaitLimitNs);
  } else {
    // compute warps: thread <-> query row, group g <-> 64 key columns of each 128-key tile
    const uint32_t wq = warp & 3, grp = (warp - 2) >> 2;
    const int row = (int)(wq * 32 + lane);
    const uint32_t tl = tmem + ((wq * 32) << 16);
    const float sl2 = a.scale_log2;
    bool ok = true;
    int g = 0, kx = 0;
    for (int item = blockIdx.x; item < a.n_items && ok; item += gridDim.x) {
      const QTileItem it = a.items[item];
      const int nt = tiles_of(it);
      const int qpos = it.q_pos0 + row;
      const bool valid = row < it.q_rows;
      // this warp writes dQ columns [grp * D / NG, (grp + 1) * D / NG) of its row
      constexpr int OC = D / C::NG;
      __nv_bfloat16* qrow = a.dq + ((int64_t)(it.q_row0 + row) * a.Hq + it.head) * D;
      if (nt == 0) {
        // no key at all: dQ = 0
        if (valid) {
#pragma unroll
          for (int v = 0; v < OC / 8; ++v) reinterpret_cast<uint4*>(qrow + grp * OC)[v] = make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      const int64_t rix = (int64_t)it.head * a.T + it.q_row0 + row;
      const float lse2 = valid ? a.lse2[rix] : INFINITY;  // P = 0 on rows past the tile
      const float delta = valid ? a.delta[rix] : 0.f;
      // copy this item's Q tile from shared memory into TMEM, the A operand of S:
      // group g copies 64-column chunks g, g + NG, ... of its row.  The previous
      // item's S GEMMs have completed (their results were loaded above).
      if (!(ok = mbar_wait(&ctl.q_full, kx & 1, fs))) break;
#pragma unroll
      for (int c = (int)grp; c < C::KCH; c += C::NG) {
        uint32_t w[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 x = *reinterpret_cast<const uint4*>(sQ + c * C::BM * 128 + sw128_offset((uint32_t)row, u));
          w[4 * u] = x.x;
          w[4 * u + 1] = x.y;
          w[4 * u + 2] = x.z;
          w[4 * u + 3] = x.w;
        }
        tmem_st32(tl + C::TM_Q + 32 * c, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.q_tmem);
      for (int j = 0; j < nt; ++j, ++g) {
        int r, t;
        qtile_of(it, j, r, t);
        const KeyRegion& kr = it.reg[r];
        const int kl0 = t * C::BN + C::GC * (int)grp;
        int lo = 0;
        if (a.window > 0) lo = max(0, qpos - a.window + 1 - kr.pos0);
        const int hi = min(kr.count - 1, qpos - kr.pos0);
        const int clo = lo - kl0, chi = hi - kl0;  // allowed columns of this group
        const bool full = (clo <= 0) && (chi >= C::GC - 1);
        if (!(ok = mbar_wait(&ctl.s_full, g & 1, fs))) break;
        tc_fence_after();
        uint32_t sr[C::GC], dr[C::GC];
#pragma unroll
        for (int c4 = 0; c4 < C::GC / 32; ++c4)
          tmem_ld32(tl + C::TM_S + C::GC * grp + 32 * c4, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c4]));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.s_empty);
        // masked keys get S = -inf once (exp2 gives 0); tiles with no masked key skip this
        if (!full) {
#pragma unroll
          for (int c = 0; c < C::GC; ++c)
            if (c < clo || c > chi) sr[c] = __float_as_uint(-INFINITY);
        }
        // P while dP is still being computed
        float p[C::GC];
        const float2 sl2v = make_float2(sl2, sl2), nl = make_float2(-lse2, -lse2);
#pragma unroll
        for (int c = 0; c < C::GC; c += 2) {
          const float2 x = ffma2(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sl2v, nl);
          p[c] = ex2_approx(x.x);
          p[c + 1] = ex2_approx(x.y);
        }
        if (!(ok = mbar_wait(&ctl.dp_full, g & 1, fs))) break;
        tc_fence_after();
#pragma unroll
        for (int c4 = 0; c4 < C::GC / 32; ++c4)
          tmem_ld32(tl + C::TM_DP + C::GC * grp + 32 * c4, *reinterpret_cast<uint32_t(*)[32]>(&dr[32 * c4]));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.dp_empty);
        uint32_t w[C::GC / 2];
        const float2 dl = make_float2(delta, delta);
#pragma unroll
        for (int e = 0; e < C::GC / 2; ++e) {
          const int c = 2 * e;
          const float2 ds = fmul2(make_float2(p[c], p[c + 1]),
                                  fsub2(make_float2(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])), dl));
          w[e] = pack_bf16x2(ds.x, ds.y);
        }
        // the dS buffer is free once the dQ MMAs of the previous tile have completed
        if (g >= 1 && !(ok = mbar_wait(&ctl.ds_done, (g - 1) & 1, fs))) break;
        tc_fence_after();
#pragma unroll
        for (int c4 = 0; c4 < C::GC / 32; ++c4)
          tmem_st16(tl + C::TM_DS + (C::GC / 2) * grp + 16 * c4, *reinterpret_cast<const uint32_t(*)[16]>(&w[16 * c4]));
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.ds_full);
      }
      if (!ok) break;
      // epilogue: dQ = scale * accumulator, then release the accumulator
      if (!(ok = mbar_wait(&ctl.acc_done, kx & 1, fs))) break;
      tc_fence_after();
#pragma unroll
      for (int c4 = 0; c4 < (OC + 31) / 32; ++c4) {
        const int col = (int)grp * OC + c4 * 32;
        uint32_t rr[32];
        tmem_ld32(tl + C::TM_DQ + col, rr);
        tmem_ld_wait();
        uint32_t o[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          o[i] = pack_bf16x2(__uint_as_float(rr[2 * i]) * a.scale, __uint_as_float(rr[2 * i + 1]) * a.scale);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(qrow + col);
#pragma unroll
          for (int v = 0; v < OC / 8 && v < 4; ++v) dst[v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.dq_free);
      ++kx;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TM_COLS);
}

// ---------------------------------------------------------------- dK / dV
template <int D>
struct DkvCfg {
  static constexpr int BN = 128;  // keys per tile (MMA M)
  static constexpr int BQ = 64;   // queries per block (N of the first pair, K of the second)
  static constexpr int KCH = D / 64;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int QB_BYTES = BQ * D * 2;      // one Q or dO block
  static constexpr int UNIT_BYTES = 2 * QB_BYTES;  // Q block + dO block
  static constexpr int NST = (D == 128) ? 4 : 8;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_BYTES;
  static constexpr int OFF_RING = OFF_V + KV_BYTES;
  static constexpr int SMEM_BYTES = OFF_RING + NST * UNIT_BYTES + 1024;
  static constexpr uint32_t TM_ST = 0, TM_DPT = 2 * BQ, TM_DV = 4 * BQ, TM_DK = 4 * BQ + D, TM_COLS = 512;
};

struct DkvSmemCtl {
  uint64_t kv_full;
  uint64_t ring_full[8], ring_empty[8];
  uint64_t s_full[2], dp_full[2], p_full[2], ds_full[2], m2_issued[2];
  uint64_t acc_done, drain, drain2;
  alignas(16) float lse2[8][64];  // read as float4
  alignas(16) float delta[8][64];
  int32_t qpos0[8], qrows[8];
  uint32_t tmem_base;
  int abort_flag;
};

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    dkv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO, const DkvArgs a) {
  using C = DkvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ DkvSmemCtl ctl;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sRing = smem + C::OFF_RING;

  const KVTileItem it = a.items[blockIdx.x];
  const int gs = a.Hq / a.Hkv;
  // an item outside the tensors (key rows, kv-head, its span of the query list or its
  // partial slot) is recorded and does nothing; a query block outside them is caught
  // by the producer before its loads
  const bool item_ok = rows_ok(it.k_row0, it.k_rows, a.T, C::BN) && it.kv_head >= 0 && it.kv_head < a.Hkv &&
                       it.list_begin >= 0 && it.it_lo >= 0 && it.it_lo <= it.it_hi &&
                       it.it_hi <= gs * it.list_len && it.partial_slot >= -1 && it.partial_slot < a.nslots;
  const int n_iter = item_ok ? it.it_hi - it.it_lo : 0;
  const uint32_t warp = warp_id(), lane = lane_id();
  FailState fs{&ctl.abort_flag, a.status, a.wait_limit_ns};
  // failure-path self-test: iteration whose Q/dO block gets one arrival too few
  const int skip_iter = blockIdx.x == 0 ? a.test_skip_iter : -1;

  if (threadIdx.x == 0) {
    if (!item_ok && a.status) atomicOr(a.status, kDevErrBounds);
    ctl.abort_flag = 0;
    mbar_init(&ctl.kv_full, 1);
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&ctl.ring_full[i], 33);  // expect_tx arrival + 32 lanes after their smem stores
      mbar_init(&ctl.ring_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl.s_full[i], 1);
      mbar_init(&ctl.dp_full[i], 1);
      mbar_init(&ctl.p_full[i], 8);
      mbar_init(&ctl.ds_full[i], 8);
      mbar_init(&ctl.m2_issued[i], 1);
    }
    mbar_init(&ctl.acc_done, 1);
    mbar_init(&ctl.drain, 1);
    mbar_init(&ctl.drain2, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl.tmem_base, C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;

  if (warp == 0) {
    // producer (whole warp): K, V tiles once; per query block Q, dO (TMA) and its
    // lse2, Delta, position.  The next block's descriptor and per-row values are
    // loaded into registers before waiting for its ring slot, so only the TMA
    // latency remains between a slot being freed and refilled.
    bool ok = true;
    int i = 0;
    if (n_iter > 0) {
      if (lane == 0) {
        mbar_arrive_expect_tx(&ctl.kv_full, 2 * C::KV_BYTES);
        for (int c = 0; c < C::KCH; ++c) {
          tma_load_3d(sK + c * C::BN * 128, &tmK, &ctl.kv_full, c * 64, it.kv_head, it.k_row0);
          tma_load_3d(sV + c * C::BN * 128, &tmV, &ctl.kv_full, c * 64, it.kv_head, it.k_row0);
        }
      }
      // values of block i, fetched one iteration ahead
      auto fetch = [&](int idx, int& h, QBlock& qb, float (&l2)[2], float (&dl)[2]) {
        const int itx = it.it_lo + idx;
        h = it.kv_head * gs + itx % gs;
        qb = a.qblocks[it.list_begin + itx / gs];
        const bool qb_ok = rows_ok(qb.q_row0, qb.q_rows, a.T, C::BQ);
        if (!qb_ok) qb.q_rows = -1;  // marks the block as outside the tensors
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int c = (int)lane + 32 * e;
          const bool v = qb_ok && c < qb.q_rows;
          const int64_t rix = (int64_t)h * a.T + qb.q_row0 + c;
          l2[e] = v ? a.lse2[rix] : INFINITY;
          dl[e] = v ? a.delta[rix] : 0.f;
        }
      };
      int h;
      QBlock qb;
      float l2[2], dl[2];
      fetch(0, h, qb, l2, dl);
      for (; i < n_iter; ++i) {
        const int slot = i % C::NST;
        if (qb.q_rows < 0) {
          raise_failure(fs, kDevErrBounds);
          ok = false;
          break;
        }
        if (!(ok = mbar_wait(&ctl.ring_empty[slot], ((i / C::NST) & 1) ^ 1, fs))) break;
        if (lane == 0 && i != skip_iter) {
          mbar_arrive_expect_tx(&ctl.ring_full[slot], C::UNIT_BYTES);
          uint8_t* dst = sRing + slot * C::UNIT_BYTES;
          for (int c = 0; c < C::KCH; ++c) {
            tma_load_3d(dst + c * C::BQ * 128, &tmQ, &ctl.ring_full[slot], c * 64, h, qb.q_row0);
            tma_load_3d(dst + C::QB_BYTES + c * C::BQ * 128, &tmDO, &ctl.ring_full[slot], c * 64, h, qb.q_row0);
          }
          ctl.qpos0[slot] = qb.q_pos0;
          ctl.qrows[slot] = qb.q_rows;
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          ctl.lse2[slot][lane + 32 * e] = l2[e];
          ctl.delta[slot][lane + 32 * e] = dl[e];
        }
        mbar_arrive(&ctl.ring_full[slot]);
        if (i + 1 < n_iter) fetch(i + 1, h, qb, l2, dl);
      }
      if (!ok && lane == 0) {
        mbar_wait_drain(&ctl.kv_full, 0, kWaitLimitNs);
        for (int back = 1; back <= C::NST && back <= i; ++back) {
          const int i2 = i - back;
          if (i2 == skip_iter) continue;  // never completes: nothing was loaded for it
          mbar_wait_drain(&ctl.ring_full[i2 % C::NST], (i2 / C::NST) & 1, kWaitLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    // first GEMM pair: S^T_i = K Q_i^T, then dP^T_i = V dO_i^T (SS, N = 64), into
    // TMEM buffer i % 2, each committed on its own barrier.  An issuing thread stalls while the tensor pipe's queue is
    // full, so the two GEMM pairs have one issuing warp each: while one warp
    // waits for its next operands, the other's MMAs keep the pipe busy.  The
    // pair for block i rewrites the buffer that the second pair of block i - 2
    // reads, so it is issued only after that pair has been issued (m2_issued,
    // with the tcgen05 thread-sync fences that order the two warps' MMAs).
    // Both warps run their loops warp-wide (warp-uniform descriptors); one
    // elected lane issues.
    if (n_iter > 0) {
      constexpr uint32_t idST = idesc_bf16(128, C::BQ, 0, 0);
      const uint64_t kdesc = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t vdesc = sdesc_sw128(smem_u32(sV), 16, 1024);
      const uint32_t aRing = smem_u32(sRing);
      bool ok = mbar_wait(&ctl.kv_full, 0, fs);
      for (int i = 0; i < n_iter && ok; ++i) {
        const uint32_t b = i & 1;
        const int slot = i % C::NST;
        if (!(ok = mbar_wait(&ctl.ring_full[slot], (i / C::NST) & 1, fs))) break;
        if (i >= 2 && !(ok = mbar_wait(&ctl.m2_issued[b], ((i >> 1) - 1) & 1, fs))) break;
        tc_fence_after();
        const uint64_t qd = sdesc_sw128(aRing + slot * C::UNIT_BYTES, 16, 1024);
        const uint64_t dod = sdesc_add(qd, C::QB_BYTES);
        const uint32_t tS = tmem + C::TM_ST + b * C::BQ, tP = tmem + C::TM_DPT + b * C::BQ;
        if (elect_one()) {
          // S^T first and committed on its own: the compute warps start on P while dP^T runs
#pragma unroll
          for (int c = 0; c < C::KCH; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16_ss(tS, sdesc_add(kdesc, c * C::BN * 128 + k * 32), sdesc_add(qd, c * C::BQ * 128 + k * 32),
                          idST, (c | k) != 0);
          mma_commit(&ctl.s_full[b]);
#pragma unroll
          for (int c = 0; c < C::KCH; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16_ss(tP, sdesc_add(vdesc, c * C::BN * 128 + k * 32), sdesc_add(dod, c * C::BQ * 128 + k * 32),
                          idST, (c | k) != 0);
          mma_commit(&ctl.dp_full[b]);
        }
        __syncwarp();
      }
      if (elect_one()) mma_commit(&ctl.drain);
      __syncwarp();
      mbar_wait_drain(&ctl.drain, 0, kWaitLimitNs);
    }
  } else if (warp == 10) {
    // second GEMM pair: dV += P^T_i dO_i as soon as P^T_i is written, then
    // dK += dS^T_i Q_i (TS, N = D), A read from the bf16 values the compute
    // warps wrote over buffer i % 2
    if (n_iter > 0) {
      constexpr uint32_t idKV = idesc_bf16(128, D, 0, 1);
      const uint32_t aRing = smem_u32(sRing);
      bool ok = true;
      for (int i = 0; i < n_iter && ok; ++i) {
        const int slot = i % C::NST;
        const uint32_t b = i & 1;
        if (!(ok = mbar_wait(&ctl.p_full[b], (i >> 1) & 1, fs))) break;
        tc_fence_after();
        const uint64_t qmn = sdesc_sw128(aRing + slot * C::UNIT_BYTES, C::BQ * 128, 1024);
        const uint64_t domn = sdesc_add(qmn, C::QB_BYTES);
        const uint32_t tPT = tmem + C::TM_ST + b * C::BQ, tDST = tmem + C::TM_DPT + b * C::BQ;
        const uint32_t acc0 = i > 0 ? 1u : 0u;
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < C::BQ / 16; ++k)
            mma_bf16_ts(tmem + C::TM_DV, tPT + packed_kstep_col(k), sdesc_add(domn, k * 16 * 128), idKV,
                        k > 0 ? 1u : acc0);
        }
        __syncwarp();
        if (!(ok = mbar_wait(&ctl.ds_full[b], (i >> 1) & 1, fs))) break;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < C::BQ / 16; ++k)
            mma_bf16_ts(tmem + C::TM_DK, tDST + packed_kstep_col(k), sdesc_add(qmn, k * 16 * 128), idKV,
                        k > 0 ? 1u : acc0);
          mma_commit(&ctl.ring_empty[slot]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.m2_issued[b]);
      }
      if (elect_one()) {
        if (ok) mma_commit(&ctl.acc_done);
        mma_commit(&ctl.drain2);
      }
      __syncwarp();
      mbar_wait_drain(&ctl.drain2, 0, kWaitLimitNs);
    }
  } else {
    // compute warps: thread <-> key row, half <-> 32 query columns of each 64-query block
    const uint32_t wq = warp & 3, half = (warp - 2) >> 2;
    const int row = (int)(wq * 32 + lane);
    const uint32_t tl = tmem + ((wq * 32) << 16);
    const int kpos = it.k_pos0 + row;
    const bool kvalid = row < it.k_rows;
    const float sl2 = a.scale_log2;
    bool ok = true;
    for (int i = 0; i < n_iter; ++i) {
      const uint32_t b = i & 1;
      const int slot = i % C::NST;
      if (!(ok = mbar_wait(&ctl.s_full[b], (i >> 1) & 1, fs))) break;
      // acquire the producer's smem stores of this block (the slot's phase is current:
      // it cannot be refilled before this block's dV/dK MMAs complete)
      if (!(ok = mbar_wait(&ctl.ring_full[slot], (i / C::NST) & 1, fs))) break;
      tc_fence_after();
      const int qpos0 = ctl.qpos0[slot] + 32 * (int)half;
      const int qrows = ctl.qrows[slot] - 32 * (int)half;
      // allowed query columns [clo, chi] of this half: q_pos >= k_pos, q_pos - k_pos < window
      const int clo = kpos - qpos0;
      int chi = qrows - 1;
      if (a.window > 0) chi = min(chi, kpos + a.window - 1 - qpos0);
      if (!kvalid) chi = -1;
      const bool full = (clo <= 0) && (chi >= 31);
      uint32_t sr[32];
      tmem_ld32(tl + C::TM_ST + b * C::BQ + 32 * half, sr);
      const float4* L4 = reinterpret_cast<const float4*>(&ctl.lse2[slot][32 * half]);
      const float4* D4 = reinterpret_cast<const float4*>(&ctl.delta[slot][32 * half]);
      tmem_ld_wait();
      // masked queries get S = -inf once (exp2 gives 0); blocks with no masked query skip this
      if (!full) {
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (c < clo || c > chi) sr[c] = __float_as_uint(-INFINITY);
      }
      // P^T first: the dV GEMM starts on it while dS^T is computed
      float p[32];
      uint32_t wp[16];
      const float2 sl2v = make_float2(sl2, sl2);
#pragma unroll
      for (int e4 = 0; e4 < 8; ++e4) {
        const float4 l4 = L4[e4];
        const float2 nl[2] = {make_float2(-l4.x, -l4.y), make_float2(-l4.z, -l4.w)};
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int c = 4 * e4 + 2 * e2;
          const float2 x = ffma2(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sl2v, nl[e2]);
          p[c] = ex2_approx(x.x);
          p[c + 1] = ex2_approx(x.y);
          wp[2 * e4 + e2] = pack_bf16x2(p[c], p[c + 1]);
        }
      }
      tmem_st16(tl + C::TM_ST + b * C::BQ + 32 * half, wp);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.p_full[b]);
      if (!(ok = mbar_wait(&ctl.dp_full[b], (i >> 1) & 1, fs))) break;
      tc_fence_after();
      uint32_t dr[32], ws[16];
      tmem_ld32(tl + C::TM_DPT + b * C::BQ + 32 * half, dr);
      tmem_ld_wait();
#pragma unroll
      for (int e4 = 0; e4 < 8; ++e4) {
        const float4 d4 = D4[e4];
        const float2 dv[2] = {make_float2(d4.x, d4.y), make_float2(d4.z, d4.w)};
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int c = 4 * e4 + 2 * e2;
          const float2 ds = fmul2(make_float2(p[c], p[c + 1]),
                                  fsub2(make_float2(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])), dv[e2]));
          ws[2 * e4 + e2] = pack_bf16x2(ds.x, ds.y);
        }
      }
      tmem_st16(tl + C::TM_DPT + b * C::BQ + 32 * half, ws);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.ds_full[b]);
    }
    if (ok && item_ok) {
      if (n_iter > 0) {
        ok = mbar_wait(&ctl.acc_done, 0, fs);
        tc_fence_after();
      }
      if (ok) {
        const int64_t orow = ((int64_t)(it.k_row0 + row) * a.Hkv + it.kv_head) * D;
        float* pk = it.partial_slot >= 0 ? a.partial + ((size_t)it.partial_slot * 2 * C::BN + row) * D : nullptr;
        float* pv = pk ? pk + (size_t)C::BN * D : nullptr;
#pragma unroll
        for (int which = 0; which < 2; ++which) {  // 0: dV, 1: dK
          const float mul = which ? a.scale : 1.f;
#pragma unroll
          for (int c4 = 0; c4 < D / 64; ++c4) {
            const int col = (int)half * (D / 2) + c4 * 32;
            uint32_t rr[32];
            if (n_iter > 0) {
              tmem_ld32(tl + (which ? C::TM_DK : C::TM_DV) + col, rr);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) rr[e] = 0u;
            }
            if (!kvalid) continue;
            if (pk) {
              float4* dst = reinterpret_cast<float4*>((which ? pk : pv) + col);
#pragma unroll
              for (int v = 0; v < 8; ++v)
                dst[v] = make_float4(__uint_as_float(rr[4 * v]) * mul, __uint_as_float(rr[4 * v + 1]) * mul,
                                     __uint_as_float(rr[4 * v + 2]) * mul, __uint_as_float(rr[4 * v + 3]) * mul);
            } else {
              uint32_t w[16];
#pragma unroll
              for (int e = 0; e < 16; ++e)
                w[e] = pack_bf16x2(__uint_as_float(rr[2 * e]) * mul, __uint_as_float(rr[2 * e + 1]) * mul);
              uint4* dst = reinterpret_cast<uint4*>((which ? a.dk : a.dv) + orow + col);
#pragma unroll
              for (int v = 0; v < 4; ++v) dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TM_COLS);
}

// ---------------------------------------------------------------- reduce
// dK, dV of a split key tile = sum over its chunks s = 0..nslots-1 in order.
// Block (item, y) covers key rows [y * R, (y + 1) * R) of the item with
// R = 1024 / D, one float4 of dK and of dV per thread; the chunks' loads are
// independent, so several are in flight per thread.  HBM-bound.
constexpr int kReduceThreads = 256;
__global__ void __launch_bounds__(kReduceThreads) reduce_kernel(const ReduceArgs a) {
  const ReduceItem it = a.items[blockIdx.x];
  if (!(rows_ok(it.k_row0, it.k_rows, a.T, a.key_tile) && it.kv_head >= 0 && it.kv_head < a.Hkv && it.slot0 >= 0 &&
        it.nslots >= 0 && it.slot0 + it.nslots <= a.total_slots)) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && a.status) atomicOr(a.status, kDevErrBounds);
    return;
  }
  const int v4_per_row = a.D / 4;
  const int e4 = blockIdx.y * kReduceThreads + threadIdx.x;  // float4 index inside the tile
  const int j = e4 / v4_per_row, d = (e4 % v4_per_row) * 4;
  if (j >= it.k_rows) return;
  const size_t slot_stride = (size_t)2 * a.key_tile * a.D;
  const float* base = a.partial + (size_t)it.slot0 * slot_stride + (size_t)j * a.D + d;
  float4 sk = make_float4(0.f, 0.f, 0.f, 0.f), sv = sk;
#pragma unroll 4
  for (int s = 0; s < it.nslots; ++s) {
    const float4 k4 = *reinterpret_cast<const float4*>(base + (size_t)s * slot_stride);
    const float4 v4 = *reinterpret_cast<const float4*>(base + (size_t)s * slot_stride + (size_t)a.key_tile * a.D);
    sk.x += k4.x; sk.y += k4.y; sk.z += k4.z; sk.w += k4.w;
    sv.x += v4.x; sv.y += v4.y; sv.z += v4.z; sv.w += v4.w;
  }
  const int64_t o = ((int64_t)(it.k_row0 + j) * a.Hkv + it.kv_head) * a.D + d;
  *reinterpret_cast<uint2*>(a.dk + o) = make_uint2(pack_bf16x2(sk.x, sk.y), pack_bf16x2(sk.z, sk.w));
  *reinterpret_cast<uint2*>(a.dv + o) = make_uint2(pack_bf16x2(sv.x, sv.y), pack_bf16x2(sv.z, sv.w));
}

// ---------------------------------------------------------------- failure-path self-test
__global__ void __launch_bounds__(64) selftest_timeout_kernel(uint64_t limit_ns, uint32_t* status) {
  __shared__ uint64_t never;  // expects two arrivals; only thread 0 ever arrives
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&never, 2);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_arrive(&never);
  FailState fs{&abort_flag, status, limit_ns};
  mbar_wait(&never, 0, fs);
  __syncthreads();
}

}  // namespace

cudaError_t launch_selftest_timeout(uint64_t limit_ns, uint32_t* status, cudaStream_t st) {
  selftest_timeout_kernel<<<1, 64, 0, st>>>(limit_ns, status);
  return cudaGetLastError();
}

int dq_query_tile(int /*D*/) { return 128; }
int dq_key_tile(int /*D*/) { return 128; }
int dkv_key_tile(int /*D*/) { return 128; }
int dkv_query_block(int /*D*/) { return 64; }

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t st) {
  const int64_t nrows = a.T * ((a.h_hi < 0 ? a.Hq : a.h_hi) - a.h_lo);
  auto grid_for = [&](int lpr) {
    const int64_t rows_per_block = (256 / 32) * (32 / lpr);
    return (unsigned)((nrows + rows_per_block - 1) / rows_per_block);
  };
  if (nrows == 0) return cudaSuccess;
  switch (a.D) {
    case 64:
      prep_kernel<64><<<grid_for(8), 256, 0, st>>>(a);
      break;
    case 128:
      prep_kernel<128><<<grid_for(16), 256, 0, st>>>(a);
      break;
    case 512:
      prep_kernel<512><<<grid_for(32), 256, 0, st>>>(a);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <int D, typename Cfg, typename K, typename Args>
static cudaError_t launch_tc(K kernel, const CUtensorMap& t0, const CUtensorMap& t1, const CUtensorMap& t2,
                             const CUtensorMap& t3, const Args& a, int n_items, cudaStream_t st,
                             int threads = kBwdThreads) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kernel<<<n_items, threads, Cfg::SMEM_BYTES, st>>>(t0, t1, t2, t3, a);
  return cudaGetLastError();
}

cudaError_t launch_dq(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const CUtensorMap& tdo, const DqArgs& a, int n_items, cudaStream_t st) {
  if (n_items <= 0) return cudaSuccess;
  // persistent: one CTA per SM, each walking every grid-th item
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidValue;
  DqArgs b = a;
  b.n_items = n_items;
  const int grid = n_items < nsm ? n_items : nsm;
  switch (D) {
    case 64:
      return launch_tc<64, DqCfg<64>>(dq_kernel<64>, tq, tk, tv, tdo, b, grid, st, DqCfg<64>::THREADS);
    case 128:
      return launch_tc<128, DqCfg<128>>(dq_kernel<128>, tq, tk, tv, tdo, b, grid, st, DqCfg<128>::THREADS);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_dkv(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const DkvArgs& a, int n_items, cudaStream_t st) {
  if (n_items <= 0) return cudaSuccess;
  switch (D) {
    case 64:
      return launch_tc<64, DkvCfg<64>>(dkv_kernel<64>, tq, tk, tv, tdo, a, n_items, st, kBwdThreads);
    case 128:
      return launch_tc<128, DkvCfg<128>>(dkv_kernel<128>, tq, tk, tv, tdo, a, n_items, st, kBwdThreads);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_reduce(const ReduceArgs& a, int n_items, cudaStream_t st) {
  if (n_items <= 0) return cudaSuccess;
  // key_tile rows x D floats per item, 4 floats per thread
  const unsigned gy = (unsigned)((a.key_tile * a.D / 4 + kReduceThreads - 1) / kReduceThreads);
  reduce_kernel<<<dim3((unsigned)n_items, gy), kReduceThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace dkv
