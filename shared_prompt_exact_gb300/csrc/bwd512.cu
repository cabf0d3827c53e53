// bwd512.cu -- DualKV backward for head dimension 512 (sm_103a).
//
// With D = 512 a 128-row tile of Q or dO is 128 KB and a 128 x 512 fp32
// accumulator fills all 512 TMEM columns, so the fused dQ and dK/dV kernels
// of bwd.cu do not fit.  This backward materialises the two 128 x 128 bf16
// blocks of every (query tile, key tile) pair the walk visits, then reduces
// them with plain tensor-core GEMMs -- no product is computed twice:
//   pds:     S = Q K^T  ->  P  = exp(S - LSE)           (masked, bf16 block)
//            dP = dO V^T -> dS = P (dP - Delta)         (bf16 block, P from registers)
//   xtg:     dV = sum P^T dO,  dK = scale sum dS^T Q    (per key tile; fixed order)
//   dq512:   dQ = scale sum dS K                        (per query tile)
// The formulas are the analytic backward of softmax attention; the fold of
// the replicated prompt gradients is the sum over all query tiles (of every
// segment) that attend a prompt key tile, in the fixed order of the plan.
#include <cuda_bf16.h>

#include "checks.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dkv {

namespace {

constexpr int kD = 512;
constexpr int kBlkBytes = 128 * 128 * 2;  // one P or dS block
// Inside a block, element (query row r, key column c) sits at
//   (c / 8) * 1024 + r * 8 + c % 8     (bf16 elements)
// -- 16 column groups of 8 keys, each 128 rows x 16 bytes.  A warp's 32 rows of one
// group are 512 contiguous bytes, so the P / dS stores are whole cache lines, and the
// GEMMs read the blocks as unswizzled core matrices (8 rows x 16 bytes).

__device__ __forceinline__ void walk_tile(const QTileItem& it, int j, int& r, int& t) {
  const int n0 = it.reg[0].t_hi - it.reg[0].t_lo;
  if (j < n0) {
    r = 0;
    t = it.reg[0].t_lo + j;
  } else {
    r = 1;
    t = it.reg[1].t_lo + (j - n0);
  }
}

// Warps 2-9 convert S and dP: warps w and w+4 share TMEM lane quarter w % 4 (one
// query row per thread) and take key columns [0, 64) and [64, 128) of each block.
constexpr int kPdsThreads = 320;

// ---------------------------------------------------------------- P and dS blocks in one pass
// One CTA per query tile (128 rows x q-head) forms, for every key tile it visits,
// both S = Q K^T and dP = dO V^T and writes both bf16 blocks, P = exp(S - LSE)
// and dS = P (dP - Delta), keeping P on chip in between.  Q is the A operand of S
// from TMEM (256 columns), dO the A operand of dP from shared memory (resident,
// 128 KB), and K / V tiles stream through a 3-unit ring; S and dP have one TMEM
// buffer each (128 columns): each block's two GEMMs keep the pipe busy while the
// compute warps drain the other one.
struct PdsFCfg {
  static constexpr int BM = 128, BN = 128;
  static constexpr int QCH = kD / 64;              // 64-column chunks of Q / dO / K / V
  static constexpr int UCH = 2;                    // 64-column chunks of a key tile per ring unit
  static constexpr int UNIT_BYTES = UCH * BN * 128;
  static constexpr int KU = QCH / UCH;             // units per K or V tile
  static constexpr int A_BYTES = BM * kD * 2;      // 128 KB: dO resident (Q staged here first)
  static constexpr int NST = 6 / UCH;              // 96 KB of ring
  static constexpr int OFF_A = 0, OFF_RING = A_BYTES;
  static constexpr int SMEM_BYTES = OFF_RING + NST * UNIT_BYTES + 1024;
  static constexpr uint32_t TM_S = 0, TM_DP = BN, TM_Q = 2 * BN, TM_COLS = 512;
};

struct PdsFCtl {
  uint64_t q_full, q_tmem, do_full;
  uint64_t ring_full[6], ring_empty[6];
  uint64_t s_full, s_empty, dp_full, dp_empty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

__global__ void __launch_bounds__(kPdsThreads, 1)
    pds_fused_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                     const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const PdsArgs a) {
  using C = PdsFCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ PdsFCtl ctl;
  uint8_t* sA = smem + C::OFF_A;  // Q staging, then dO
  uint8_t* sRing = smem + C::OFF_RING;

  const QTileItem it = a.items[blockIdx.x];
  const int blk0 = a.block_base[blockIdx.x];
  const int nt_all = (it.reg[0].t_hi - it.reg[0].t_lo) + (it.reg[1].t_hi - it.reg[1].t_lo);
  // an item outside the tensors or naming blocks past the block array does nothing
  const bool item_ok = qtile_ok(it, a.T, a.Hq, C::BM, C::BN) && blk0 >= 0 && (int64_t)blk0 + nt_all <= a.n_blocks;
  const int kvh = it.head / (a.Hq / a.Hkv);
  const int nt = item_ok ? nt_all : 0;
  const uint32_t warp = warp_id(), lane = lane_id();
  FailState fs{&ctl.abort_flag, a.status, a.wait_limit_ns};

  if (threadIdx.x == 0) {
    if (!item_ok && a.status) atomicOr(a.status, kDevErrBounds);
    ctl.abort_flag = 0;
    mbar_init(&ctl.q_full, 1);
    mbar_init(&ctl.q_tmem, 8);
    mbar_init(&ctl.do_full, 1);
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&ctl.ring_full[i], 1);
      mbar_init(&ctl.ring_empty[i], 1);
    }
    mbar_init(&ctl.s_full, 1);
    mbar_init(&ctl.s_empty, 8);
    mbar_init(&ctl.dp_full, 1);
    mbar_init(&ctl.dp_empty, 8);
    mbar_init(&ctl.drain, 1);
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
    // producer: Q (staged in the dO region), the ring's K / V units in consumption
    // order K_0, V_0, K_1, V_1, ..., and dO once the compute warps have copied Q to TMEM
    if (lane == 0 && nt > 0) {
      mbar_arrive_expect_tx(&ctl.q_full, C::A_BYTES);
      for (int c = 0; c < C::QCH; ++c) tma_load_3d(sA + c * C::BM * 128, &tmQ, &ctl.q_full, c * 64, it.head, it.q_row0);
      bool do_loaded = false;
      int idx = 0;
      bool ok = true;
      for (int j = 0; j < nt && ok; ++j) {
        int r, t;
        walk_tile(it, j, r, t);
        const int key_row = it.reg[r].row0 + t * C::BN;
        for (int kind = 0; kind < 2 && ok; ++kind) {
          const CUtensorMap* tm = kind == 0 ? &tmK : &tmV;
          for (int u = 0; u < C::KU && ok; ++u, ++idx) {
            const int slot = idx % C::NST;
            if (!(ok = mbar_wait(&ctl.ring_empty[slot], ((idx / C::NST) & 1) ^ 1, fs))) break;
            if (idx == a.test_skip_unit) continue;  // failure-path self-test: never loaded
            mbar_arrive_expect_tx(&ctl.ring_full[slot], C::UNIT_BYTES);
            uint8_t* dst = sRing + slot * C::UNIT_BYTES;
            for (int c = 0; c < C::UCH; ++c)
              tma_load_3d(dst + c * C::BN * 128, tm, &ctl.ring_full[slot], (C::UCH * u + c) * 64, kvh, key_row);
          }
          if (j == 0 && kind == 0 && ok) {
            // dO replaces the staged Q once the compute warps have copied Q into TMEM
            if (!(ok = mbar_wait(&ctl.q_tmem, 0, fs))) break;
            mbar_arrive_expect_tx(&ctl.do_full, C::A_BYTES);
            for (int c = 0; c < C::QCH; ++c)
              tma_load_3d(sA + c * C::BM * 128, &tmDO, &ctl.do_full, c * 64, it.head, it.q_row0);
            do_loaded = true;
          }
        }
      }
      if (!ok) {
        mbar_wait_drain(&ctl.q_full, 0, kWaitLimitNs);
        if (do_loaded) mbar_wait_drain(&ctl.do_full, 0, kWaitLimitNs);
        for (int back = 1; back <= C::NST && back <= idx; ++back) {
          const int i2 = idx - back;
          if (i2 == a.test_skip_unit) continue;  // never loaded
          mbar_wait_drain(&ctl.ring_full[i2 % C::NST], (i2 / C::NST) & 1, kWaitLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    // S_j = Q K_j^T (A from TMEM), then dP_j = dO V_j^T (A from shared memory); each
    // waits until the compute warps have loaded the previous block's result
    if (nt > 0) {
      constexpr uint32_t idS = idesc_bf16(128, C::BN, 0, 0);
      const uint32_t aRing = smem_u32(sRing);
      const uint64_t adesc = sdesc_sw128(smem_u32(sA), 16, 1024);
      bool ok = mbar_wait(&ctl.q_tmem, 0, fs);  // Q copied into TMEM
      int idx = 0;
      for (int j = 0; j < nt && ok; ++j) {
        for (int kind = 0; kind < 2 && ok; ++kind) {
          if (kind == 0) {
            if (j > 0 && !(ok = mbar_wait(&ctl.s_empty, (j - 1) & 1, fs))) break;
          } else {
            if (j == 0 && !(ok = mbar_wait(&ctl.do_full, 0, fs))) break;
            if (j > 0 && !(ok = mbar_wait(&ctl.dp_empty, (j - 1) & 1, fs))) break;
          }
          const uint32_t tD = tmem + (kind == 0 ? C::TM_S : C::TM_DP);
          for (int u = 0; u < C::KU && ok; ++u, ++idx) {
            const int slot = idx % C::NST;
            if (!(ok = mbar_wait(&ctl.ring_full[slot], (idx / C::NST) & 1, fs))) break;
            tc_fence_after();
            const uint64_t bdesc = sdesc_sw128(aRing + slot * C::UNIT_BYTES, 16, 1024);
            if (elect_one()) {
#pragma unroll
              for (int c = 0; c < C::UCH; ++c)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const int kc = C::UCH * u + c;  // 64-column chunk of the contraction
                  if (kind == 0)
                    mma_bf16_ts(tD, tmem + C::TM_Q + 8 * (kc * 4 + k), sdesc_add(bdesc, c * C::BN * 128 + k * 32),
                                idS, (u | c | k) != 0);
                  else
                    mma_bf16_ss(tD, sdesc_add(adesc, kc * C::BM * 128 + k * 32),
                                sdesc_add(bdesc, c * C::BN * 128 + k * 32), idS, (u | c | k) != 0);
                }
              mma_commit(&ctl.ring_empty[slot]);
              if (u == C::KU - 1) mma_commit(kind == 0 ? &ctl.s_full : &ctl.dp_full);
            }
            __syncwarp();
          }
        }
      }
      if (elect_one()) mma_commit(&ctl.drain);
      __syncwarp();
      mbar_wait_drain(&ctl.drain, 0, kWaitLimitNs);
    }
  } else {
    // thread <-> query row, half <-> 64 key columns of each block
    const uint32_t wq = warp & 3, half = (warp - 2) >> 2;
    const int row = (int)(wq * 32 + lane);
    const uint32_t tl = tmem + ((wq * 32) << 16);
    const int qpos = it.q_pos0 + row;
    const bool valid = row < it.q_rows;
    const int64_t rix = (int64_t)it.head * a.T + it.q_row0 + row;
    const float lse2 = valid ? a.lse2[rix] : INFINITY;
    const float delta = valid ? a.delta[rix] : 0.f;
    constexpr int HC = C::BN / 2;
    bool ok = true;
    if (nt > 0) {
      // copy this row of Q into TMEM (the A operand of S): the first half's warps take
      // 64-column chunks 0-3, the second's 4-7
      if ((ok = mbar_wait(&ctl.q_full, 0, fs))) {
#pragma unroll
        for (int cc = 0; cc < C::QCH / 2; ++cc) {
          const int c = (int)half * (C::QCH / 2) + cc;
          uint32_t w[32];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 x = *reinterpret_cast<const uint4*>(sA + c * C::BM * 128 + sw128_offset((uint32_t)row, u));
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
      }
    }
    const float2 sl2v = make_float2(a.scale_log2, a.scale_log2), nl = make_float2(-lse2, -lse2);
    const float2 dl = make_float2(delta, delta);
    for (int j = 0; j < nt && ok; ++j) {
      // this thread's 8 column groups of the block, 8 keys (16 bytes) each
      const size_t boff = (size_t)(blk0 + j) * (kBlkBytes / 2) + (size_t)(8 * half) * 1024 + (size_t)row * 8;
      float p[HC];
      {
        if (!(ok = mbar_wait(&ctl.s_full, j & 1, fs))) break;
        tc_fence_after();
#pragma unroll
        for (int c4 = 0; c4 < HC / 32; ++c4) {
          uint32_t rr[32];
          tmem_ld32(tl + C::TM_S + HC * half + c4 * 32, rr);
#pragma unroll
          for (int i = 0; i < 32; ++i) p[c4 * 32 + i] = __uint_as_float(rr[i]);
        }
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.s_empty);
        int r, t;
        walk_tile(it, j, r, t);
        const KeyRegion& kr = it.reg[r];
        const int kl0 = t * C::BN + HC * (int)half;
        int lo = 0;
        if (a.window > 0) lo = max(0, qpos - a.window + 1 - kr.pos0);
        const int hi = min(kr.count - 1, qpos - kr.pos0);
        const int clo = lo - kl0, chi = hi - kl0;
        uint4* dst = reinterpret_cast<uint4*>(a.p_out + boff);
#pragma unroll
        for (int v = 0; v < HC / 8; ++v) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = 8 * v + 2 * e;
            const float2 x = ffma2(make_float2(p[c], p[c + 1]), sl2v, nl);
            float p0 = ex2_approx(x.x);
            float p1 = ex2_approx(x.y);
            p0 = (c < clo || c > chi) ? 0.f : p0;
            p1 = (c + 1 < clo || c + 1 > chi) ? 0.f : p1;
            p[c] = p0;
            p[c + 1] = p1;
            w[e] = pack_bf16x2(p0, p1);
          }
          dst[v * 128] = make_uint4(w[0], w[1], w[2], w[3]);  // column group 8 * half + v (2048 bytes apart)
        }
      }
      if (!(ok = mbar_wait(&ctl.dp_full, j & 1, fs))) break;
      tc_fence_after();
      float dpv[HC];
#pragma unroll
      for (int c4 = 0; c4 < HC / 32; ++c4) {
        uint32_t rr[32];
        tmem_ld32(tl + C::TM_DP + HC * half + c4 * 32, rr);
#pragma unroll
        for (int i = 0; i < 32; ++i) dpv[c4 * 32 + i] = __uint_as_float(rr[i]);
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.dp_empty);
      uint4* dst = reinterpret_cast<uint4*>(a.ds_out + boff);
#pragma unroll
      for (int v = 0; v < HC / 8; ++v) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = 8 * v + 2 * e;
          const float2 ds = fmul2(make_float2(p[c], p[c + 1]), fsub2(make_float2(dpv[c], dpv[c + 1]), dl));
          w[e] = pack_bf16x2(ds.x, ds.y);
        }
        dst[v * 128] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TM_COLS);
}

// ---------------------------------------------------------------- transposed GEMMs (dV, dK)
// out[key, :] = mul * sum over the entries e of the key tile: A_e^T B_e, with
// A_e the 64 query rows x 128 keys of a P (or dS) block and B_e the same 64
// query rows of dO (or Q), all 512 columns.  Both operands are MN-major.
struct XtgCfg {
  static constexpr int A_BYTES = 2 * 64 * 128;       // 2 key chunks x 64 query rows
  static constexpr int B_BYTES = 8 * 64 * 128;       // 8 column chunks x 64 query rows
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int NST = 2;
  static constexpr int SMEM_BYTES = NST * STAGE_BYTES + 1024;
  static constexpr uint32_t TM_COLS = 512;
};

struct XtgCtl {
  uint64_t full[2], empty[2];
  uint64_t acc_done, drain;
  uint32_t tmem_base;
  int abort_flag;
};

__global__ void __launch_bounds__(192, 1)
    xtg_kernel(const __grid_constant__ CUtensorMap tmBlk, const __grid_constant__ CUtensorMap tmB, const XtgArgs a) {
  using C = XtgCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ XtgCtl ctl;
  const XTItem it = a.items[blockIdx.x];
  // an item outside the tensors does nothing; an entry outside them is caught by the
  // producer before its loads
  const bool item_ok = rows_ok(it.k_row0, it.k_rows, a.T, 128) && it.kv_head >= 0 && it.kv_head < a.Hkv &&
                       it.list_begin >= 0 && it.it_lo >= 0 && it.it_lo <= it.it_hi &&
                       (int64_t)it.list_begin + it.it_hi <= a.n_entries && it.partial_slot >= -1 &&
                       it.partial_slot < a.nslots;
  const int n_iter = item_ok ? it.it_hi - it.it_lo : 0;
  const uint32_t warp = warp_id(), lane = lane_id();
  FailState fs{&ctl.abort_flag, a.status};

  if (threadIdx.x == 0) {
    if (!item_ok && a.status) atomicOr(a.status, kDevErrBounds);
    ctl.abort_flag = 0;
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&ctl.full[i], 1);
      mbar_init(&ctl.empty[i], 1);
    }
    mbar_init(&ctl.acc_done, 1);
    mbar_init(&ctl.drain, 1);
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
    if (lane == 0 && n_iter > 0) {
      bool ok = true;
      int i = 0;
      for (; i < n_iter; ++i) {
        const XTEntry e = a.entries[it.list_begin + it.it_lo + i];
        const int slot = i % C::NST;
        const int gs = a.Hq / a.Hkv;
        if (!(e.head >= it.kv_head * gs && e.head < (it.kv_head + 1) * gs && rows_ok(e.q_row0, 1, a.T, 1) &&
              e.block >= 0 && e.block < a.n_blocks && (e.sub == 0 || e.sub == 1))) {
          raise_failure(fs, kDevErrBounds);
          ok = false;
          break;
        }
        if (!(ok = mbar_wait(&ctl.empty[slot], ((i / C::NST) & 1) ^ 1, fs))) break;
        mbar_arrive_expect_tx(&ctl.full[slot], C::STAGE_BYTES);
        uint8_t* st = smem + slot * C::STAGE_BYTES;
        // rows [64 sub, 64 sub + 64) of the block, all 16 column groups: [group][row][8 keys]
        tma_load_4d(st, &tmBlk, &ctl.full[slot], 0, 2 * e.sub, 0, e.block);
        for (int c = 0; c < 8; ++c)
          tma_load_3d(st + C::A_BYTES + c * 64 * 128, &tmB, &ctl.full[slot], c * 64, e.head, e.q_row0);
      }
      if (!ok) {
        for (int back = 1; back <= C::NST && back <= i; ++back) {
          const int i2 = i - back;
          mbar_wait_drain(&ctl.full[i2 % C::NST], (i2 / C::NST) & 1, kWaitLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    if (n_iter > 0) {
      constexpr uint32_t idX = idesc_bf16(128, 256, 1, 1);
      const uint32_t base = smem_u32(smem);
      bool ok = true;
      for (int i = 0; i < n_iter && ok; ++i) {
        const int slot = i % C::NST;
        if (!(ok = mbar_wait(&ctl.full[slot], (i / C::NST) & 1, fs))) break;
        tc_fence_after();
        // A = block^T, MN-major (keys): 8-key groups 1024 bytes apart, 8-row groups 128
        const uint64_t ad = sdesc_noswz(base + slot * C::STAGE_BYTES, 128, 1024);
        const uint64_t bd = sdesc_sw128(base + slot * C::STAGE_BYTES + C::A_BYTES, 64 * 128, 1024);
        const uint32_t acc0 = i > 0 ? 1u : 0u;
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int nh = 0; nh < 2; ++nh)
              mma_bf16_ss(tmem + nh * 256, sdesc_add(ad, k * 16 * 16), sdesc_add(bd, nh * 4 * 64 * 128 + k * 16 * 128),
                          idX, k > 0 ? 1u : acc0);
          mma_commit(&ctl.empty[slot]);
        }
        __syncwarp();
      }
      if (elect_one()) {
        if (ok) mma_commit(&ctl.acc_done);
        mma_commit(&ctl.drain);
      }
      __syncwarp();
      mbar_wait_drain(&ctl.drain, 0, kWaitLimitNs);
    }
  } else {
    // epilogue: thread <-> key row
    const uint32_t wq = warp & 3;
    const int row = (int)(wq * 32 + lane);
    const uint32_t tl = tmem + ((wq * 32) << 16);
    const bool kvalid = row < it.k_rows;
    bool ok = item_ok;
    if (ok && n_iter > 0) {
      ok = mbar_wait(&ctl.acc_done, 0, fs);
      tc_fence_after();
    }
    if (ok) {
      float* pdst = it.partial_slot >= 0
                        ? a.partial + (((size_t)it.partial_slot * 2 + a.region) * 128 + row) * kD
                        : nullptr;
      __nv_bfloat16* odst = a.out + ((int64_t)(it.k_row0 + row) * a.Hkv + it.kv_head) * kD;
#pragma unroll 1
      for (int c4 = 0; c4 < kD / 32; ++c4) {
        uint32_t rr[32];
        if (n_iter > 0) {
          tmem_ld32(tl + c4 * 32, rr);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) rr[e] = 0u;
        }
        if (!kvalid) continue;
        if (pdst) {
          float4* d4 = reinterpret_cast<float4*>(pdst + c4 * 32);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            d4[v] = make_float4(__uint_as_float(rr[4 * v]) * a.mul, __uint_as_float(rr[4 * v + 1]) * a.mul,
                                __uint_as_float(rr[4 * v + 2]) * a.mul, __uint_as_float(rr[4 * v + 3]) * a.mul);
        } else {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(rr[2 * e]) * a.mul, __uint_as_float(rr[2 * e + 1]) * a.mul);
          uint4* d = reinterpret_cast<uint4*>(odst + c4 * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) d[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TM_COLS);
}

// ---------------------------------------------------------------- dQ GEMM
// dQ[q tile, :] = scale * sum over the tile's key walk of dS_blk K, one 64-key
// half of a block per step: A = dS (128 q x 64 keys, K-major), B = 64 key rows
// of K, all 512 columns (MN-major).
struct Dq512Cfg {
  static constexpr int A_BYTES = 128 * 128;   // 128 rows x 64 keys
  static constexpr int B_BYTES = 8 * 64 * 128;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int NST = 2;
  static constexpr int SMEM_BYTES = NST * STAGE_BYTES + 1024;
  static constexpr uint32_t TM_COLS = 512;
};

__global__ void __launch_bounds__(192, 1)
    dq512_kernel(const __grid_constant__ CUtensorMap tmBlk, const __grid_constant__ CUtensorMap tmK, const Dq512Args a) {
  using C = Dq512Cfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ XtgCtl ctl;
  const QTileItem it = a.items[blockIdx.x];
  const int blk0 = a.block_base[blockIdx.x];
  const int nt_all = (it.reg[0].t_hi - it.reg[0].t_lo) + (it.reg[1].t_hi - it.reg[1].t_lo);
  // an item outside the tensors or naming blocks past the block array does nothing
  const bool item_ok = qtile_ok(it, a.T, a.Hq, 128, 128) && blk0 >= 0 && (int64_t)blk0 + nt_all <= a.n_blocks;
  const int nt = item_ok ? nt_all : 0;
  const int n_iter = 2 * nt;
  const int kvh = it.head / (a.Hq / a.Hkv);
  const uint32_t warp = warp_id(), lane = lane_id();
  FailState fs{&ctl.abort_flag, a.status};

  if (threadIdx.x == 0) {
    if (!item_ok && a.status) atomicOr(a.status, kDevErrBounds);
    ctl.abort_flag = 0;
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&ctl.full[i], 1);
      mbar_init(&ctl.empty[i], 1);
    }
    mbar_init(&ctl.acc_done, 1);
    mbar_init(&ctl.drain, 1);
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
    if (lane == 0 && n_iter > 0) {
      bool ok = true;
      int i = 0;
      for (; i < n_iter; ++i) {
        const int j = i >> 1, half = i & 1;
        int r, t;
        walk_tile(it, j, r, t);
        const int key_row = it.reg[r].row0 + t * 128 + half * 64;
        const int slot = i % C::NST;
        if (!(ok = mbar_wait(&ctl.empty[slot], ((i / C::NST) & 1) ^ 1, fs))) break;
        mbar_arrive_expect_tx(&ctl.full[slot], C::STAGE_BYTES);
        uint8_t* st = smem + slot * C::STAGE_BYTES;
        // keys [64 half, 64 half + 64) of the block: column groups 8 half .. 8 half + 7, all rows
        tma_load_4d(st, &tmBlk, &ctl.full[slot], 0, 0, 8 * half, blk0 + j);
        for (int c = 0; c < 8; ++c) tma_load_3d(st + C::A_BYTES + c * 64 * 128, &tmK, &ctl.full[slot], c * 64, kvh, key_row);
      }
      if (!ok) {
        for (int back = 1; back <= C::NST && back <= i; ++back) {
          const int i2 = i - back;
          mbar_wait_drain(&ctl.full[i2 % C::NST], (i2 / C::NST) & 1, kWaitLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    if (n_iter > 0) {
      constexpr uint32_t idQ = idesc_bf16(128, 256, 0, 1);
      const uint32_t base = smem_u32(smem);
      bool ok = true;
      for (int i = 0; i < n_iter && ok; ++i) {
        const int slot = i % C::NST;
        if (!(ok = mbar_wait(&ctl.full[slot], (i / C::NST) & 1, fs))) break;
        tc_fence_after();
        // A = dS, K-major (keys): 8-key groups 2048 bytes apart, 8-row groups 128
        const uint64_t ad = sdesc_noswz(base + slot * C::STAGE_BYTES, 2048, 128);
        const uint64_t bd = sdesc_sw128(base + slot * C::STAGE_BYTES + C::A_BYTES, 64 * 128, 1024);
        const uint32_t acc0 = i > 0 ? 1u : 0u;
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int nh = 0; nh < 2; ++nh)
              mma_bf16_ss(tmem + nh * 256, sdesc_add(ad, k * 2 * 2048), sdesc_add(bd, nh * 4 * 64 * 128 + k * 16 * 128), idQ,
                          k > 0 ? 1u : acc0);
          mma_commit(&ctl.empty[slot]);
        }
        __syncwarp();
      }
      if (elect_one()) {
        if (ok) mma_commit(&ctl.acc_done);
        mma_commit(&ctl.drain);
      }
      __syncwarp();
      mbar_wait_drain(&ctl.drain, 0, kWaitLimitNs);
    }
  } else {
    const uint32_t wq = warp & 3;
    const int row = (int)(wq * 32 + lane);
    const uint32_t tl = tmem + ((wq * 32) << 16);
    const bool valid = row < it.q_rows;
    bool ok = n_iter > 0 && mbar_wait(&ctl.acc_done, 0, fs);
    tc_fence_after();
    if (ok) {
      __nv_bfloat16* qrow = a.dq + ((int64_t)(it.q_row0 + row) * a.Hq + it.head) * kD;
#pragma unroll 1
      for (int c4 = 0; c4 < kD / 32; ++c4) {
        uint32_t rr[32];
        tmem_ld32(tl + c4 * 32, rr);
        tmem_ld_wait();
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = pack_bf16x2(__uint_as_float(rr[2 * e]) * a.scale, __uint_as_float(rr[2 * e + 1]) * a.scale);
        if (valid) {
          uint4* d = reinterpret_cast<uint4*>(qrow + c4 * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) d[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TM_COLS);
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes, bool& done) {
  if (done) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done = true;
  return e;
}

}  // namespace

cudaError_t launch_pds_fused(const CUtensorMap& tq, const CUtensorMap& tdo, const CUtensorMap& tk,
                             const CUtensorMap& tv, const PdsArgs& a, int n_items, cudaStream_t st) {
  if (n_items <= 0) return cudaSuccess;
  static bool s = false;
  cudaError_t e;
  if ((e = set_smem(pds_fused_kernel, PdsFCfg::SMEM_BYTES, s)) != cudaSuccess) return e;
  pds_fused_kernel<<<n_items, kPdsThreads, PdsFCfg::SMEM_BYTES, st>>>(tq, tdo, tk, tv, a);
  return cudaGetLastError();
}


cudaError_t launch_xtg(const CUtensorMap& tBlk, const CUtensorMap& tB, const XtgArgs& a, int n_items, cudaStream_t st) {
  if (n_items <= 0) return cudaSuccess;
  static bool s = false;
  cudaError_t e = set_smem(xtg_kernel, XtgCfg::SMEM_BYTES, s);
  if (e != cudaSuccess) return e;
  xtg_kernel<<<n_items, 192, XtgCfg::SMEM_BYTES, st>>>(tBlk, tB, a);
  return cudaGetLastError();
}

cudaError_t launch_dq512(const CUtensorMap& tBlk, const CUtensorMap& tK, const Dq512Args& a, int n_items,
                         cudaStream_t st) {
  if (n_items <= 0) return cudaSuccess;
  static bool s = false;
  cudaError_t e = set_smem(dq512_kernel, Dq512Cfg::SMEM_BYTES, s);
  if (e != cudaSuccess) return e;
  dq512_kernel<<<n_items, 192, Dq512Cfg::SMEM_BYTES, st>>>(tBlk, tK, a);
  return cudaGetLastError();
}

}  // namespace dkv
