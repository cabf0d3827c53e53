// bwd.cu -- DualKV backward kernels for sm_103a (head dimension 64 / 128).
//
// The packed backward equals the analytic backward of standard attention on
// the N replicated sequences with the prompt gradients summed over replicas
// (DualKV paper, abstract: mathematically equivalent to standard attention).
// With P_ij = exp(S_ij - LSE_i), dP_ij = dO_i . v_j, Delta_i = dO_i . O_i and
// dS_ij = P_ij (dP_ij - Delta_i):
//   dQ_i = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i,   dV_j = sum_i P_ij dO_i.
// A prompt key j is attended by prompt queries and by the queries of every
// segment, so its dK/dV sum over all of them -- which is exactly the fold of
// the replicated prompt gradients.
//
// Kernels: prep (Delta and log2-scaled LSE), dkv (one CTA per key tile and
// chunk of its query walk; fixed walk order), reduce (fixed-order sum of split
// chunks), dq (one CTA per query tile; same key walk as the forward).
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace dkv {

namespace {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- prep
// Delta[h, t] = sum_d dO[t,h,d] * O[t,h,d];  lse2[h, t] = lse[h, t] * log2(e)
template <int D>
__global__ void __launch_bounds__(256) prep_kernel(const PrepArgs a) {
  constexpr int LPR = (D / 8) < 32 ? (D / 8) : 32;  // lanes per row
  constexpr int PASSES = D / (8 * LPR);
  constexpr int RPW = 32 / LPR;                       // rows per warp
  const int64_t nrows = a.T * a.Hq;
  const int64_t warp_global = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x / 32);
  const int sub = (threadIdx.x & 31) / LPR, l = (threadIdx.x & 31) % LPR;
  const int64_t r = warp_global * RPW + sub;  // row = t * Hq + h
  float acc = 0.f;
  if (r < nrows) {
    const uint4* po = reinterpret_cast<const uint4*>(a.out + r * D);
    const uint4* pd = reinterpret_cast<const uint4*>(a.dout + r * D);
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
    const int64_t t = r / a.Hq;
    const int h = (int)(r % a.Hq);
    a.delta[(int64_t)h * a.T + t] = acc;
    a.lse2[(int64_t)h * a.T + t] = a.lse[(int64_t)h * a.T + t] * kLog2e;
  }
}

// ---------------------------------------------------------------- dQ
template <int D>
struct DqCfg {
  static constexpr int BM = 128, BN = 64;
  static constexpr int KCH = D / 64;
  static constexpr int Q_BYTES = BM * D * 2;         // Q and dO tiles
  static constexpr int TILE_BYTES = BN * D * 2;      // one K or V tile
  static constexpr int DS_BYTES = BM * BN * 2;
  static constexpr int NST = (D == 128) ? 8 : 12;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + Q_BYTES;
  static constexpr int OFF_DS = OFF_DO + Q_BYTES;
  static constexpr int OFF_RING = OFF_DS + 2 * DS_BYTES;
  static constexpr int SMEM_BYTES = OFF_RING + NST * TILE_BYTES + 1024;
  static constexpr uint32_t TM_S = 0, TM_DP = 2 * BN, TM_DQ = 4 * BN, TM_COLS = 512;
};

struct DqSmemCtl {
  uint64_t q_full;
  uint64_t ring_full[12], ring_empty[12];
  uint64_t s_full[2], s_empty[2], ds_full[2], ds_done[2];
  uint64_t drain;
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
__global__ void __launch_bounds__(192, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO, const DqArgs a) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ DqSmemCtl ctl;
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sDO = smem + C::OFF_DO;
  uint8_t* sDS = smem + C::OFF_DS;
  uint8_t* sRing = smem + C::OFF_RING;

  const QTileItem it = a.items[blockIdx.x];
  const int nt = (it.reg[0].t_hi - it.reg[0].t_lo) + (it.reg[1].t_hi - it.reg[1].t_lo);
  const int kvh = it.head / (a.Hq / a.Hkv);
  const uint32_t warp = warp_id(), lane = lane_id();
  FailState fs{&ctl.abort_flag, a.status};

  if (threadIdx.x == 0) {
    ctl.abort_flag = 0;
    mbar_init(&ctl.q_full, 1);
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&ctl.ring_full[i], 1);
      mbar_init(&ctl.ring_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl.s_full[i], 1);
      mbar_init(&ctl.s_empty[i], 4);
      mbar_init(&ctl.ds_full[i], 4);
      mbar_init(&ctl.ds_done[i], 1);
    }
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
    // producer: Q and dO once, then K_j, V_j for every key tile
    if (lane == 0 && nt > 0) {
      mbar_arrive_expect_tx(&ctl.q_full, 2 * C::Q_BYTES);
      for (int c = 0; c < C::KCH; ++c) {
        tma_load_3d(sQ + c * C::BM * 128, &tmQ, &ctl.q_full, c * 64, it.head, it.q_row0);
        tma_load_3d(sDO + c * C::BM * 128, &tmDO, &ctl.q_full, c * 64, it.head, it.q_row0);
      }
      bool ok = true;
      int idx = 0;
      for (int j = 0; j < nt && ok; ++j) {
        int r, t;
        qtile_of(it, j, r, t);
        const int key_row = it.reg[r].row0 + t * C::BN;
        for (int kind = 0; kind < 2; ++kind, ++idx) {
          const int slot = idx % C::NST;
          const uint32_t ph = (idx / C::NST) & 1;
          if (!(ok = mbar_wait(&ctl.ring_empty[slot], ph ^ 1, fs))) break;
          mbar_arrive_expect_tx(&ctl.ring_full[slot], C::TILE_BYTES);
          uint8_t* dst = sRing + slot * C::TILE_BYTES;
          const CUtensorMap* tm = kind == 0 ? &tmK : &tmV;
          for (int c = 0; c < C::KCH; ++c) tma_load_3d(dst + c * C::BN * 128, tm, &ctl.ring_full[slot], c * 64, kvh, key_row);
        }
      }
      if (!ok) {
        mbar_wait_drain(&ctl.q_full, 0, kWaitLimitNs);
        for (int back = 1; back <= C::NST && back <= idx; ++back) {
          const int i2 = idx - back;
          mbar_wait_drain(&ctl.ring_full[i2 % C::NST], (i2 / C::NST) & 1, kWaitLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    // MMA issuer: S_j = Q K_j^T, dP_j = dO V_j^T, then dQ += dS_{j-1} K_{j-1}
    if (lane == 0 && nt > 0) {
      constexpr uint32_t idS = idesc_bf16(128, C::BN, 0, 0);
      constexpr uint32_t idQ = idesc_bf16(128, D, 0, 1);
      const uint32_t aQ = smem_u32(sQ), aDO = smem_u32(sDO), aDS = smem_u32(sDS), aRing = smem_u32(sRing);
      bool ok = mbar_wait(&ctl.q_full, 0, fs);
      tc_fence_after();
      for (int j = 0; j <= nt && ok; ++j) {
        if (j < nt) {
          const int b = j & 1;
          const int ik = 2 * j, iv = 2 * j + 1;
          if (!(ok = mbar_wait(&ctl.s_empty[b], ((j >> 1) & 1) ^ 1, fs))) break;
          if (!(ok = mbar_wait(&ctl.ring_full[ik % C::NST], (ik / C::NST) & 1, fs))) break;
          if (!(ok = mbar_wait(&ctl.ring_full[iv % C::NST], (iv / C::NST) & 1, fs))) break;
          tc_fence_after();
          const uint32_t kb = aRing + (ik % C::NST) * C::TILE_BYTES, vb = aRing + (iv % C::NST) * C::TILE_BYTES;
#pragma unroll
          for (int c = 0; c < C::KCH; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              mma_bf16_ss(tmem + C::TM_S + b * C::BN, sdesc_sw128(aQ + c * C::BM * 128 + k * 32, 16, 1024),
                          sdesc_sw128(kb + c * C::BN * 128 + k * 32, 16, 1024), idS, (c | k) != 0);
            }
#pragma unroll
          for (int c = 0; c < C::KCH; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              mma_bf16_ss(tmem + C::TM_DP + b * C::BN, sdesc_sw128(aDO + c * C::BM * 128 + k * 32, 16, 1024),
                          sdesc_sw128(vb + c * C::BN * 128 + k * 32, 16, 1024), idS, (c | k) != 0);
            }
          mma_commit(&ctl.ring_empty[iv % C::NST]);
          mma_commit(&ctl.s_full[b]);
        }
        if (j >= 1) {
          const int jj = j - 1, b = jj & 1, ik = 2 * jj;
          if (!(ok = mbar_wait(&ctl.ds_full[b], (jj >> 1) & 1, fs))) break;
          tc_fence_after();
          const uint32_t kb = aRing + (ik % C::NST) * C::TILE_BYTES;
          const uint32_t db = aDS + b * C::DS_BYTES;
#pragma unroll
          for (int k = 0; k < C::BN / 16; ++k)
            mma_bf16_ss(tmem + C::TM_DQ, sdesc_sw128(db + k * 32, 16, 1024),
                        sdesc_sw128(kb + k * 16 * 128, C::BN * 128, 1024), idQ, (jj > 0 || k > 0) ? 1u : 0u);
          mma_commit(&ctl.ring_empty[ik % C::NST]);
          mma_commit(&ctl.ds_done[b]);
        }
      }
      mma_commit(&ctl.drain);
      mbar_wait_drain(&ctl.drain, 0, kWaitLimitNs);
    }
  } else {
    // dS warps: thread <-> query row
    const uint32_t wq = warp & 3;
    const int row = (int)(wq * 32 + lane);
    const uint32_t tl = tmem + ((wq * 32) << 16);
    const int qpos = it.q_pos0 + row;
    const bool valid = row < it.q_rows;
    const int64_t rix = (int64_t)it.head * a.T + it.q_row0 + row;
    const float lse2 = valid ? a.lse2[rix] : INFINITY;  // P = 0 on rows past the tile
    const float delta = valid ? a.delta[rix] : 0.f;
    const float sl2 = a.scale_log2;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const int b = j & 1;
      if (!(ok = mbar_wait(&ctl.s_full[b], (j >> 1) & 1, fs))) break;
      tc_fence_after();
      int r, t;
      qtile_of(it, j, r, t);
      const KeyRegion& kr = it.reg[r];
      const int kl0 = t * C::BN;
      int lo = 0;
      if (a.window > 0) lo = max(0, qpos - a.window + 1 - kr.pos0);
      const int hi = min(kr.count - 1, qpos - kr.pos0);
      const int clo = lo - kl0, chi = hi - kl0;
      uint32_t sr[64], dr[64];
      tmem_ld32(tl + C::TM_S + b * C::BN, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(tl + C::TM_S + b * C::BN + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_ld32(tl + C::TM_DP + b * C::BN, *reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
      tmem_ld32(tl + C::TM_DP + b * C::BN + 32, *reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.s_empty[b]);
      if (j >= 2 && !(ok = mbar_wait(&ctl.ds_done[b], ((j - 2) >> 1) & 1, fs))) break;
      const uint32_t db = smem_u32(sDS + b * C::DS_BYTES);
#pragma unroll
      for (int pc = 0; pc < 8; ++pc) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = pc * 8 + e * 2;
          float p0 = ex2_approx(fmaf(__uint_as_float(sr[c]), sl2, -lse2));
          float p1 = ex2_approx(fmaf(__uint_as_float(sr[c + 1]), sl2, -lse2));
          p0 = (c < clo || c > chi) ? 0.f : p0;
          p1 = (c + 1 < clo || c + 1 > chi) ? 0.f : p1;
          const float d0 = p0 * (__uint_as_float(dr[c]) - delta);
          const float d1 = p1 * (__uint_as_float(dr[c + 1]) - delta);
          w[e] = pack_bf16x2(d0, d1);
        }
        st_shared_v4(db + sw128_offset(row, pc), w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.ds_full[b]);
    }
    if (ok && nt > 0) {
      ok = mbar_wait(&ctl.ds_done[(nt - 1) & 1], ((nt - 1) >> 1) & 1, fs);
      tc_fence_after();
      if (ok) {
        __nv_bfloat16* qrow = a.dq + ((int64_t)(it.q_row0 + row) * a.Hq + it.head) * D;
#pragma unroll
        for (int c4 = 0; c4 < D / 32; ++c4) {
          uint32_t rr[32];
          tmem_ld32(tl + C::TM_DQ + c4 * 32, rr);
          tmem_ld_wait();
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(__uint_as_float(rr[2 * i]) * a.scale, __uint_as_float(rr[2 * i + 1]) * a.scale);
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(qrow + c4 * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
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

// ---------------------------------------------------------------- dK / dV
template <int D>
struct DkvCfg {
  static constexpr int BN = 128;  // keys per tile (MMA M)
  static constexpr int BQ = 64;   // queries per block (MMA N of S^T, K of dV/dK)
  static constexpr int KCH = D / 64;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int QB_BYTES = BQ * D * 2;            // one Q or dO block
  static constexpr int UNIT_BYTES = 2 * QB_BYTES;        // Q block + dO block
  static constexpr int PT_BYTES = BN * BQ * 2;           // P^T or dS^T (bf16)
  static constexpr int NST = (D == 128) ? 2 : 4;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_BYTES;
  static constexpr int OFF_PT = OFF_V + KV_BYTES;        // 2 buffers
  static constexpr int OFF_DST = OFF_PT + 2 * PT_BYTES;  // 2 buffers
  static constexpr int OFF_RING = OFF_DST + 2 * PT_BYTES;
  static constexpr int SMEM_BYTES = OFF_RING + NST * UNIT_BYTES + 1024;
  static constexpr uint32_t TM_ST = 0, TM_DPT = 2 * BQ, TM_DV = 4 * BQ, TM_DK = 4 * BQ + D, TM_COLS = 512;
};

struct DkvSmemCtl {
  uint64_t kv_full;
  uint64_t ring_full[4], ring_empty[4];
  uint64_t st_full[2], st_empty[2], pt_full[2], pt_done[2];
  uint64_t drain;
  float lse2[4][64];
  float delta[4][64];
  uint32_t tmem_base;
  int abort_flag;
};

template <int D>
__global__ void __launch_bounds__(192, 1)
    dkv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO, const DkvArgs a) {
  using C = DkvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ DkvSmemCtl ctl;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sPT = smem + C::OFF_PT;
  uint8_t* sDST = smem + C::OFF_DST;
  uint8_t* sRing = smem + C::OFF_RING;

  const KVTileItem it = a.items[blockIdx.x];
  const int n_iter = it.it_hi - it.it_lo;
  const int gs = a.Hq / a.Hkv;
  const uint32_t warp = warp_id(), lane = lane_id();
  FailState fs{&ctl.abort_flag, a.status};

  if (threadIdx.x == 0) {
    ctl.abort_flag = 0;
    mbar_init(&ctl.kv_full, 1);
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&ctl.ring_full[i], 33);  // expect_tx arrival + 32 lanes after their lse/delta stores
      mbar_init(&ctl.ring_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl.st_full[i], 1);
      mbar_init(&ctl.st_empty[i], 4);
      mbar_init(&ctl.pt_full[i], 4);
      mbar_init(&ctl.pt_done[i], 1);
    }
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
    // producer (whole warp): K, V tiles once; then per query block Q, dO (TMA) and lse2, Delta
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
      for (; i < n_iter; ++i) {
        const int itx = it.it_lo + i;
        const int h = it.kv_head * gs + itx / it.list_len;
        const QBlock qb = a.qblocks[it.list_begin + itx % it.list_len];
        const int slot = i % C::NST;
        const uint32_t ph = (i / C::NST) & 1;
        if (!(ok = mbar_wait(&ctl.ring_empty[slot], ph ^ 1, fs))) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&ctl.ring_full[slot], C::UNIT_BYTES);
          uint8_t* dst = sRing + slot * C::UNIT_BYTES;
          for (int c = 0; c < C::KCH; ++c) {
            tma_load_3d(dst + c * C::BQ * 128, &tmQ, &ctl.ring_full[slot], c * 64, h, qb.q_row0);
            tma_load_3d(dst + C::QB_BYTES + c * C::BQ * 128, &tmDO, &ctl.ring_full[slot], c * 64, h, qb.q_row0);
          }
        }
        for (int c = (int)lane; c < C::BQ; c += 32) {
          const bool v = c < qb.q_rows;
          const int64_t rix = (int64_t)h * a.T + qb.q_row0 + c;
          ctl.lse2[slot][c] = v ? a.lse2[rix] : INFINITY;
          ctl.delta[slot][c] = v ? a.delta[rix] : 0.f;
        }
        mbar_arrive(&ctl.ring_full[slot]);
      }
      if (!ok && lane == 0) {
        mbar_wait_drain(&ctl.kv_full, 0, kWaitLimitNs);
        for (int back = 1; back <= C::NST && back <= i; ++back) {
          const int i2 = i - back;
          mbar_wait_drain(&ctl.ring_full[i2 % C::NST], (i2 / C::NST) & 1, kWaitLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    // MMA issuer
    if (lane == 0 && n_iter > 0) {
      constexpr uint32_t idST = idesc_bf16(128, C::BQ, 0, 0);
      constexpr uint32_t idKV = idesc_bf16(128, D, 0, 1);
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aPT = smem_u32(sPT), aDST = smem_u32(sDST),
                     aRing = smem_u32(sRing);
      bool ok = mbar_wait(&ctl.kv_full, 0, fs);
      tc_fence_after();
      for (int i = 0; i <= n_iter && ok; ++i) {
        if (i < n_iter) {
          const int b = i & 1, slot = i % C::NST;
          if (!(ok = mbar_wait(&ctl.st_empty[b], ((i >> 1) & 1) ^ 1, fs))) break;
          if (!(ok = mbar_wait(&ctl.ring_full[slot], (i / C::NST) & 1, fs))) break;
          tc_fence_after();
          const uint32_t qb = aRing + slot * C::UNIT_BYTES, dob = qb + C::QB_BYTES;
#pragma unroll
          for (int c = 0; c < C::KCH; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16_ss(tmem + C::TM_ST + b * C::BQ, sdesc_sw128(aK + c * C::BN * 128 + k * 32, 16, 1024),
                          sdesc_sw128(qb + c * C::BQ * 128 + k * 32, 16, 1024), idST, (c | k) != 0);
#pragma unroll
          for (int c = 0; c < C::KCH; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16_ss(tmem + C::TM_DPT + b * C::BQ, sdesc_sw128(aV + c * C::BN * 128 + k * 32, 16, 1024),
                          sdesc_sw128(dob + c * C::BQ * 128 + k * 32, 16, 1024), idST, (c | k) != 0);
          mma_commit(&ctl.st_full[b]);
        }
        if (i >= 1) {
          const int ii = i - 1, b = ii & 1, slot = ii % C::NST;
          if (!(ok = mbar_wait(&ctl.pt_full[b], (ii >> 1) & 1, fs))) break;
          tc_fence_after();
          const uint32_t qb = aRing + slot * C::UNIT_BYTES, dob = qb + C::QB_BYTES;
#pragma unroll
          for (int k = 0; k < C::BQ / 16; ++k) {
            const uint32_t acc = (ii > 0 || k > 0) ? 1u : 0u;
            mma_bf16_ss(tmem + C::TM_DV, sdesc_sw128(aPT + b * C::PT_BYTES + k * 32, 16, 1024),
                        sdesc_sw128(dob + k * 16 * 128, C::BQ * 128, 1024), idKV, acc);
            mma_bf16_ss(tmem + C::TM_DK, sdesc_sw128(aDST + b * C::PT_BYTES + k * 32, 16, 1024),
                        sdesc_sw128(qb + k * 16 * 128, C::BQ * 128, 1024), idKV, acc);
          }
          mma_commit(&ctl.ring_empty[slot]);
          mma_commit(&ctl.pt_done[b]);
        }
      }
      mma_commit(&ctl.drain);
      mbar_wait_drain(&ctl.drain, 0, kWaitLimitNs);
    }
  } else {
    // P^T / dS^T warps: thread <-> key row
    const uint32_t wq = warp & 3;
    const int row = (int)(wq * 32 + lane);
    const uint32_t tl = tmem + ((wq * 32) << 16);
    const int kpos = it.k_pos0 + row;
    const bool kvalid = row < it.k_rows;
    const float sl2 = a.scale_log2;
    bool ok = true;
    for (int i = 0; i < n_iter; ++i) {
      const int b = i & 1, slot = i % C::NST;
      const int itx = it.it_lo + i;
      const QBlock qb = a.qblocks[it.list_begin + itx % it.list_len];
      if (!(ok = mbar_wait(&ctl.st_full[b], (i >> 1) & 1, fs))) break;
      tc_fence_after();
      // allowed query columns [clo, chi]: q_pos >= k_pos and (window) q_pos - k_pos < window
      int clo = kpos - qb.q_pos0;
      int chi = qb.q_rows - 1;
      if (a.window > 0) chi = min(chi, kpos + a.window - 1 - qb.q_pos0);
      if (!kvalid) chi = -1;
      uint32_t sr[64], dr[64];
      tmem_ld32(tl + C::TM_ST + b * C::BQ, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(tl + C::TM_ST + b * C::BQ + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_ld32(tl + C::TM_DPT + b * C::BQ, *reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
      tmem_ld32(tl + C::TM_DPT + b * C::BQ + 32, *reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.st_empty[b]);
      if (i >= 2 && !(ok = mbar_wait(&ctl.pt_done[b], ((i - 2) >> 1) & 1, fs))) break;
      // acquire the producer's lse2/delta stores for this block; the slot cannot
      // be refilled before this block's dV/dK MMAs complete, so its phase is current
      if (!(ok = mbar_wait(&ctl.ring_full[slot], (i / C::NST) & 1, fs))) break;
      const float* L2 = ctl.lse2[slot];
      const float* DL = ctl.delta[slot];
      const uint32_t pb = smem_u32(sPT + b * C::PT_BYTES), sb = smem_u32(sDST + b * C::PT_BYTES);
#pragma unroll
      for (int pc = 0; pc < 8; ++pc) {
        uint32_t wp[4], ws[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = pc * 8 + e * 2;
          float p0 = ex2_approx(fmaf(__uint_as_float(sr[c]), sl2, -L2[c]));
          float p1 = ex2_approx(fmaf(__uint_as_float(sr[c + 1]), sl2, -L2[c + 1]));
          p0 = (c < clo || c > chi) ? 0.f : p0;
          p1 = (c + 1 < clo || c + 1 > chi) ? 0.f : p1;
          const float d0 = p0 * (__uint_as_float(dr[c]) - DL[c]);
          const float d1 = p1 * (__uint_as_float(dr[c + 1]) - DL[c + 1]);
          wp[e] = pack_bf16x2(p0, p1);
          ws[e] = pack_bf16x2(d0, d1);
        }
        st_shared_v4(pb + sw128_offset(row, pc), wp[0], wp[1], wp[2], wp[3]);
        st_shared_v4(sb + sw128_offset(row, pc), ws[0], ws[1], ws[2], ws[3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.pt_full[b]);
    }
    if (ok) {
      if (n_iter > 0) {
        ok = mbar_wait(&ctl.pt_done[(n_iter - 1) & 1], ((n_iter - 1) >> 1) & 1, fs);
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
          for (int c4 = 0; c4 < D / 32; ++c4) {
            uint32_t rr[32];
            if (n_iter > 0) {
              tmem_ld32(tl + (which ? C::TM_DK : C::TM_DV) + c4 * 32, rr);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) rr[e] = 0u;
            }
            if (!kvalid) continue;
            if (pk) {
              float4* dst = reinterpret_cast<float4*>((which ? pk : pv) + c4 * 32);
#pragma unroll
              for (int v = 0; v < 8; ++v)
                dst[v] = make_float4(__uint_as_float(rr[4 * v]) * mul, __uint_as_float(rr[4 * v + 1]) * mul,
                                     __uint_as_float(rr[4 * v + 2]) * mul, __uint_as_float(rr[4 * v + 3]) * mul);
            } else {
              uint32_t w[16];
#pragma unroll
              for (int e = 0; e < 16; ++e)
                w[e] = pack_bf16x2(__uint_as_float(rr[2 * e]) * mul, __uint_as_float(rr[2 * e + 1]) * mul);
              uint4* dst = reinterpret_cast<uint4*>((which ? a.dk : a.dv) + orow + c4 * 32);
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
__global__ void __launch_bounds__(256) reduce_kernel(const ReduceArgs a) {
  const ReduceItem it = a.items[blockIdx.x];
  const int n = it.k_rows * a.D;
  const size_t slot_stride = (size_t)2 * a.key_tile * a.D;
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int j = e / a.D, d = e % a.D;
    float sk = 0.f, sv = 0.f;
    for (int s = 0; s < it.nslots; ++s) {
      const float* base = a.partial + (size_t)(it.slot0 + s) * slot_stride;
      sk += base[(size_t)j * a.D + d];
      sv += base[(size_t)a.key_tile * a.D + (size_t)j * a.D + d];
    }
    const int64_t o = ((int64_t)(it.k_row0 + j) * a.Hkv + it.kv_head) * a.D + d;
    a.dk[o] = __float2bfloat16_rn(sk);
    a.dv[o] = __float2bfloat16_rn(sv);
  }
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
  FailState fs{&abort_flag, status};
  mbar_wait(&never, 0, fs, limit_ns);
  __syncthreads();
}

}  // namespace

cudaError_t launch_selftest_timeout(uint64_t limit_ns, uint32_t* status, cudaStream_t st) {
  selftest_timeout_kernel<<<1, 64, 0, st>>>(limit_ns, status);
  return cudaGetLastError();
}

int dq_query_tile(int /*D*/) { return 128; }
int dq_key_tile(int /*D*/) { return 64; }
int dkv_key_tile(int /*D*/) { return 128; }
int dkv_query_block(int /*D*/) { return 64; }

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t st) {
  const int64_t nrows = a.T * a.Hq;
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
                             const CUtensorMap& t3, const Args& a, int n_items, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kernel<<<n_items, 192, Cfg::SMEM_BYTES, st>>>(t0, t1, t2, t3, a);
  return cudaGetLastError();
}

cudaError_t launch_dq(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const CUtensorMap& tdo, const DqArgs& a, int n_items, cudaStream_t st) {
  if (n_items <= 0) return cudaSuccess;
  switch (D) {
    case 64:
      return launch_tc<64, DqCfg<64>>(dq_kernel<64>, tq, tk, tv, tdo, a, n_items, st);
    case 128:
      return launch_tc<128, DqCfg<128>>(dq_kernel<128>, tq, tk, tv, tdo, a, n_items, st);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_dkv(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const DkvArgs& a, int n_items, cudaStream_t st) {
  if (n_items <= 0) return cudaSuccess;
  switch (D) {
    case 64:
      return launch_tc<64, DkvCfg<64>>(dkv_kernel<64>, tq, tk, tv, tdo, a, n_items, st);
    case 128:
      return launch_tc<128, DkvCfg<128>>(dkv_kernel<128>, tq, tk, tv, tdo, a, n_items, st);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_reduce(const ReduceArgs& a, int n_items, cudaStream_t st) {
  if (n_items <= 0) return cudaSuccess;
  reduce_kernel<<<n_items, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace dkv
