// fwd.cu -- DualKV forward kernel for sm_103a (head dimension 64, 128, 512).
//
// DualKV paper, abstract: the keys a packed query sees lie in two separate
// ranges of rows, the prompt that all segments share and the query's own
// segment, and one kernel covers both in the same launch.  One CTA takes one query tile (128 packed
// rows of one region) of one q-head and walks the key tiles of region 0
// (prompt) and then region 1 (own segment), clipped to the causal / window
// range, with an online softmax.
//
// Warp roles (96 + 128 * NH threads):
//   warp 0      TMA producer: the Q tile once, then K and V tiles through a
//               ring of "units" (128 rows x 128 head-dim columns, two 64-column
//               TMA boxes) in the order the MMA warp consumes them
//               (K_0, K_1, V_0, K_2, V_1, ...)
//   warp 1      TMEM owner; issues S_j = Q K_j^T (A and B in shared memory)
//               into one of two TMEM S buffers
//   warp 2+4NH  issues O += P_j V_j with P read from TMEM.  A thread issuing
//               tcgen05.mma stalls while the tensor pipe's queue is full, so
//               each GEMM has its own issuing warp: the pipe keeps working while
//               either waits for its operands.  Both run their loops warp-wide
//               (warp-uniform descriptors) and one elected lane issues.
//   warps 2..    softmax: thread <-> query row (TMEM lane).  With NH = 2 (head
//               dimension <= 128) each row's 128 key columns are split over two
//               warps ("halves"); each half keeps its own running max m and sum
//               l (log2 units) and its own O accumulator in TMEM (PV runs as two
//               K = 64 GEMMs), so the halves never wait on each other inside the
//               key walk.  A half reads S_j columns [64h, 64h+64), masks, writes
//               P_j as packed bf16 over the first 32 of those columns, and
//               rescales its O when its m grows by more than 2^8 (exact: O and l
//               share the stale max).  The epilogue combines the halves:
//               out = (O_0 2^(m_0-m) + O_1 2^(m_1-m)) / (l_0 2^(m_0-m) + l_1 2^(m_1-m)).
// S_{j+2} rewrites the buffer holding P_j, so it is issued only after PV_j has
// been issued (pv_issued, with the tcgen05 thread-sync fences that order the
// two warps' MMAs).
//
// Head dimension 512: the 128 x 512 fp32 O accumulator would fill all of TMEM,
// so the output columns are split over two CTAs (NSPLIT = 2, 256 columns each);
// both compute the full S = Q K^T (contraction over all 512 columns).
#include <cuda_bf16.h>

#include "checks.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dkv {

namespace {

template <int D>
struct FwdCfg {
  static constexpr int BM = 128, BN = 128;
  static constexpr int NSPLIT = (D == 512) ? 2 : 1;
  static constexpr int NH = (D == 512) ? 1 : 2;        // key-column halves per row
  static constexpr int HC = BN / NH;                   // key columns of one half
  static constexpr int THREADS = 96 + 128 * NH;
  static constexpr int PV_WARP = 2 + 4 * NH;           // issuer of the PV GEMMs
  static constexpr int DV = D / NSPLIT;                // output columns of one CTA
  static constexpr int QCH = D / 64;                   // 64-column chunks of Q / K
  static constexpr int UCH = (D == 64) ? 1 : 2;        // chunks per ring unit
  static constexpr int UNIT_BYTES = UCH * BN * 128;    // 16 or 32 KB
  static constexpr int KU = QCH / UCH;                 // units per K tile
  static constexpr int VU = (DV / 64) / UCH;           // units per V tile (this CTA's columns)
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int NST = (D == 512) ? 3 : (D == 128 ? 6 : 12);
  // A ring wait names its fill only by phase parity, so it is exact only if the
  // slot's previous fill (NST units earlier) has completed.  For V_j that unit
  // may belong to K_{j+1} when NST < KU + VU; the PV warp then first waits until
  // the S warp has taken all of K_{j+1} (k_taken).
  static constexpr bool PV_WAITS_K = NST < KU + VU;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = Q_BYTES;
  static constexpr int SMEM_BYTES = OFF_RING + NST * UNIT_BYTES + 1024;  // + alignment slack
  static constexpr uint32_t TM_S = 0;                  // S buffers at columns 0 and BN
  static constexpr uint32_t TM_O = 2 * BN;             // O accumulators, one per half (DV columns each)
  static constexpr uint32_t TM_COLS = 512;
  static constexpr float RESCALE_THRESHOLD = 8.0f;     // log2 units
};

struct FwdSmemCtl {
  uint64_t q_full;
  uint64_t ring_full[12], ring_empty[12];
  uint64_t s_full[2], p_full[2], pv_done[2], pv_issued[2], k_taken[2];
  uint64_t drain, drain2;
  uint64_t pair_done[4];      // per lane quarter: both halves have published (m, l)
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void tile_of(const QTileItem& it, int j, int& r, int& t) {
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
__global__ void __launch_bounds__(FwdCfg<D>::THREADS, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const FwdArgs a) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ FwdSmemCtl ctl;
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sRing = smem + C::OFF_RING;

  const QTileItem it = a.items[blockIdx.x / C::NSPLIT];
  const int split = (int)(blockIdx.x % C::NSPLIT);
  // an item outside the tensors is recorded and given no key tiles: nothing is read or written
  const bool item_ok = qtile_ok(it, a.T, a.Hq, C::BM, C::BN);
  const int nt0 = it.reg[0].t_hi - it.reg[0].t_lo;
  const int nt = item_ok ? nt0 + (it.reg[1].t_hi - it.reg[1].t_lo) : 0;
  const int kvh = it.head / (a.Hq / a.Hkv);
  const uint32_t warp = warp_id(), lane = lane_id();
  FailState fs{&ctl.abort_flag, a.status, a.wait_limit_ns};

  if (threadIdx.x == 0) {
    if (!item_ok && a.status) atomicOr(a.status, kDevErrBounds);
    ctl.abort_flag = 0;
    mbar_init(&ctl.q_full, 1);
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&ctl.ring_full[i], 1);
      mbar_init(&ctl.ring_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl.s_full[i], 1);
      mbar_init(&ctl.p_full[i], 4 * C::NH);
      mbar_init(&ctl.pv_done[i], 1);
      mbar_init(&ctl.pv_issued[i], 1);
      mbar_init(&ctl.k_taken[i], 1);
    }
    for (int i = 0; i < 4; ++i) mbar_init(&ctl.pair_done[i], 32 * C::NH);
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
    // ------------------------------------------------------------ producer
    if (lane == 0 && nt > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(&ctl.q_full, C::Q_BYTES);
      for (int c = 0; c < C::QCH; ++c)
        tma_load_3d(sQ + c * C::BM * 128, &tmQ, &ctl.q_full, c * 64, it.head, it.q_row0);
      int idx = 0;
      bool ok = true;
      // units in consumption order: K_0; then for j = 1..nt: K_j (if j < nt), V_{j-1}
      for (int j = 0; j <= nt && ok; ++j) {
        for (int kind = 0; kind < 2 && ok; ++kind) {
          const int jj = kind == 0 ? j : j - 1;
          if (jj < 0 || jj >= nt) continue;
          int r, t;
          tile_of(it, jj, r, t);
          const int key_row = it.reg[r].row0 + t * C::BN;
          const int nu = kind == 0 ? C::KU : C::VU;
          const int col0 = kind == 0 ? 0 : split * C::DV;
          const CUtensorMap* tm = kind == 0 ? &tmK : &tmV;
          for (int u = 0; u < nu; ++u, ++idx) {
            const int slot = idx % C::NST;
            if (!(ok = mbar_wait(&ctl.ring_empty[slot], ((idx / C::NST) & 1) ^ 1, fs))) break;
            if (idx == a.test_skip_unit) continue;  // failure-path self-test: never loaded
            mbar_arrive_expect_tx(&ctl.ring_full[slot], C::UNIT_BYTES);
            uint8_t* dst = sRing + slot * C::UNIT_BYTES;
            for (int c = 0; c < C::UCH; ++c)
              tma_load_3d(dst + c * C::BN * 128, tm, &ctl.ring_full[slot], col0 + (u * C::UCH + c) * 64, kvh, key_row);
          }
        }
      }
      if (!ok) {
        // drain: wait for every copy still in flight before the CTA can exit
        mbar_wait_drain(&ctl.q_full, 0, kWaitLimitNs);
        for (int back = 1; back <= C::NST && back <= idx; ++back) {
          const int i2 = idx - back;
          if (i2 == a.test_skip_unit) continue;
          mbar_wait_drain(&ctl.ring_full[i2 % C::NST], (i2 / C::NST) & 1, kWaitLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S issuer
    // Ring positions follow the producer's order K_0, K_1, V_0, K_2, V_1, ...:
    // K_j starts at unit KU + (j - 1)(KU + VU) for j >= 1.
    if (nt > 0) {
      constexpr uint32_t idS = idesc_bf16(128, C::BN, 0, 0);
      const uint64_t qdesc = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint32_t aRing = smem_u32(sRing);
      bool ok = mbar_wait(&ctl.q_full, 0, fs);
      for (int j = 0; j < nt && ok; ++j) {
        const uint32_t b = j & 1;
        const uint32_t tS = tmem + C::TM_S + b * C::BN;
        if (j >= 2 && !(ok = mbar_wait(&ctl.pv_issued[b], ((j >> 1) - 1) & 1, fs))) break;
        int idx = j == 0 ? 0 : C::KU + (j - 1) * (C::KU + C::VU);
        for (int u = 0; u < C::KU && ok; ++u, ++idx) {
          const int slot = idx % C::NST;
          if (!(ok = mbar_wait(&ctl.ring_full[slot], (idx / C::NST) & 1, fs))) break;
          tc_fence_after();
          const uint64_t kdesc = sdesc_sw128(aRing + slot * C::UNIT_BYTES, 16, 1024);
          const uint64_t qd = sdesc_add(qdesc, u * C::UCH * C::BM * 128);
          if (C::PV_WAITS_K && u == C::KU - 1 && lane == 0) mbar_arrive(&ctl.k_taken[b]);
          if (elect_one()) {
#pragma unroll
            for (int c = 0; c < C::UCH; ++c)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_bf16_ss(tS, sdesc_add(qd, c * C::BM * 128 + k * 32), sdesc_add(kdesc, c * C::BN * 128 + k * 32),
                            idS, (u | c | k) != 0);
            mma_commit(&ctl.ring_empty[slot]);
            if (u == C::KU - 1) mma_commit(&ctl.s_full[b]);
          }
          __syncwarp();
        }
      }
      // every MMA issued above must finish before TMEM is released
      if (elect_one()) mma_commit(&ctl.drain);
      __syncwarp();
      mbar_wait_drain(&ctl.drain, 0, kWaitLimitNs);
    }
  } else if (warp == C::PV_WARP) {
    // ------------------------------------------------------------ PV issuer
    // V_j starts at unit 2 KU + j (KU + VU), except the last tile's, which
    // follows every K tile and V_0 .. V_{nt-2}: unit nt KU + (nt - 1) VU.
    if (nt > 0) {
      constexpr uint32_t idO = idesc_bf16(128, C::UCH * 64, 0, 1);
      const uint32_t aRing = smem_u32(sRing);
      bool ok = true;
      for (int j = 0; j < nt && ok; ++j) {
        const uint32_t b = j & 1;
        if (!(ok = mbar_wait(&ctl.p_full[b], (j >> 1) & 1, fs))) break;
        if (C::PV_WAITS_K && j + 1 < nt &&
            !(ok = mbar_wait(&ctl.k_taken[(j + 1) & 1], ((j + 1) >> 1) & 1, fs)))
          break;
        const uint32_t tP = tmem + C::TM_S + b * C::BN;
        const uint32_t acc0 = j > 0 ? 1u : 0u;
        int idx = (j + 1 < nt) ? 2 * C::KU + j * (C::KU + C::VU) : nt * C::KU + (nt - 1) * C::VU;
        for (int u = 0; u < C::VU && ok; ++u, ++idx) {
          const int slot = idx % C::NST;
          if (!(ok = mbar_wait(&ctl.ring_full[slot], (idx / C::NST) & 1, fs))) break;
          tc_fence_after();
          const uint64_t vdesc = sdesc_sw128(aRing + slot * C::UNIT_BYTES, C::BN * 128, 1024);
          if (elect_one()) {
#pragma unroll
            for (int h = 0; h < C::NH; ++h)
#pragma unroll
              for (int k = 0; k < C::HC / 16; ++k)
                mma_bf16_ts(tmem + C::TM_O + h * C::DV + u * C::UCH * 64, tP + h * C::HC + k * 8,
                            sdesc_add(vdesc, (h * C::HC + k * 16) * 128), idO, k > 0 ? 1u : acc0);
            mma_commit(&ctl.ring_empty[slot]);
            if (u == C::VU - 1) mma_commit(&ctl.pv_done[b]);
          }
          __syncwarp();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.pv_issued[b]);
      }
      if (elect_one()) mma_commit(&ctl.drain2);
      __syncwarp();
      mbar_wait_drain(&ctl.drain2, 0, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const uint32_t wq = warp & 3;
    const int half = (int)((warp - 2) >> 2);  // 0 .. NH-1
    const int row = (int)(wq * 32 + lane);
    const uint32_t tl = tmem + ((wq * 32) << 16);
    const uint32_t tO = tl + C::TM_O + half * C::DV;
    const int qpos = it.q_pos0 + row;
    const float sl2 = a.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const uint32_t b = j & 1;
      int r, t;
      tile_of(it, j, r, t);
      const KeyRegion& kr = it.reg[r];
      const int kl0 = t * C::BN + half * C::HC;  // local index of this half's first key
      int lo = 0;
      if (a.window > 0) lo = max(0, qpos - a.window + 1 - kr.pos0);
      const int hi = min(kr.count - 1, qpos - kr.pos0);
      const int clo = lo - kl0, chi = hi - kl0;  // allowed columns [clo, chi] of this half
      const bool full = (clo <= 0) && (chi >= C::HC - 1);
      if (!(ok = mbar_wait(&ctl.s_full[b], (j >> 1) & 1, fs))) break;
      tc_fence_after();

      float s[C::HC];
#pragma unroll
      for (int c4 = 0; c4 < C::HC / 32; ++c4) {
        uint32_t rr[32];
        tmem_ld32(tl + C::TM_S + b * C::BN + half * C::HC + c4 * 32, rr);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c4 * 32 + i] = __uint_as_float(rr[i]);
      }
      tmem_ld_wait();

      if (!full) {
#pragma unroll
        for (int c = 0; c < C::HC; ++c) s[c] = (c < clo || c > chi) ? -INFINITY : s[c];
      }
      // row max: four independent chains of three-input max
      float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < C::HC; c += 8) {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) mq[q4] = fmax3(mq[q4], s[c + 2 * q4], s[c + 2 * q4 + 1]);
      }
      const float mx = fmax3(fmaxf(mq[0], mq[1]), mq[2], mq[3]);
      const float m_tile = mx * sl2;  // -inf stays -inf (sl2 > 0)
      const float m_new = fmaxf(m, m_tile);
      if (j == 0) {
        m = m_new;
      } else if (__any_sync(0xffffffffu, m_new > m + C::RESCALE_THRESHOLD)) {
        // the decision is per warp: a row that has seen no allowed key yet (m_new = -inf)
        // keeps alpha = 1; a row whose first allowed key arrives now has m = -inf, alpha = 0
        const float alpha = (m_new == -INFINITY) ? 1.f : ex2_approx(m - m_new);
        if (!(ok = mbar_wait(&ctl.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, fs))) break;
        tc_fence_after();
#pragma unroll
        for (int c4 = 0; c4 < C::DV / 32; ++c4) {
          uint32_t rr[32];
          tmem_ld32(tO + c4 * 32, rr);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
          tmem_st32(tO + c4 * 32, rr);
        }
        tmem_st_wait();
        l *= alpha;
        m = m_new;
      }
      const float m_use = (m == -INFINITY) ? 0.f : m;
      const float2 sl2v = make_float2(sl2, sl2), negm = make_float2(-m_use, -m_use);
      float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int h2 = 0; h2 < C::HC / 64; ++h2) {
        uint32_t w[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int c = h2 * 64 + 2 * e;
          const float2 x = ffma2(make_float2(s[c], s[c + 1]), sl2v, negm);
          const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          sum2[e & 1] = fadd2(sum2[e & 1], pp);
          w[e] = pack_bf16x2(pp.x, pp.y);
        }
        tmem_st32(tl + C::TM_S + b * C::BN + half * C::HC + h2 * 32, w);
      }
      const float2 st = fadd2(sum2[0], sum2[1]);
      l += st.x + st.y;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.p_full[b]);
    }
    if (ok && nt > 0) {
      // epilogue: combine the halves, out = O / l, lse = (m + log2 l) ln 2
      ok = mbar_wait(&ctl.pv_done[(nt - 1) & 1], ((nt - 1) >> 1) & 1, fs);
      tc_fence_after();
      float mh[2] = {m, -INFINITY}, lh[2] = {l, 0.f};
      if (ok && C::NH == 2) {
        // the K/V ring is idle once the last PV has completed: borrow 2 KB of it
        float* half_m = reinterpret_cast<float*>(sRing);  // [2][128]
        float* half_l = half_m + 256;                      // [2][128]
        half_m[half * 128 + row] = m;
        half_l[half * 128 + row] = l;
        mbar_arrive(&ctl.pair_done[wq]);
        ok = mbar_wait(&ctl.pair_done[wq], 0, fs);
        mh[0] = half_m[row];
        mh[1] = half_m[128 + row];
        lh[0] = half_l[row];
        lh[1] = half_l[128 + row];
      }
      if (ok) {
        const bool valid = row < it.q_rows;
        const float mtot = fmaxf(mh[0], mh[1]);
        const float mref = (mtot == -INFINITY) ? 0.f : mtot;
        const float f0 = (mh[0] == -INFINITY) ? 0.f : ex2_approx(mh[0] - mref);
        const float f1 = (mh[1] == -INFINITY) ? 0.f : ex2_approx(mh[1] - mref);
        const float ltot = lh[0] * f0 + lh[1] * f1;
        const float inv_l = 1.f / ltot;
        const float g0 = f0 * inv_l, g1 = f1 * inv_l;
        // this warp writes output columns [half * DV / NH, ...) of its rows
        constexpr int OC = C::DV / C::NH;
        __nv_bfloat16* orow = a.out + ((int64_t)(it.q_row0 + row) * a.Hq + it.head) * D + split * C::DV + half * OC;
#pragma unroll
        for (int c4 = 0; c4 < OC / 32; ++c4) {
          const int col = half * OC + c4 * 32;
          uint32_t r0[32], r1[32];
          tmem_ld32(tl + C::TM_O + col, r0);
          if (C::NH == 2) tmem_ld32(tl + C::TM_O + C::DV + col, r1);
          tmem_ld_wait();
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0 = __uint_as_float(r0[2 * i]) * g0, x1 = __uint_as_float(r0[2 * i + 1]) * g0;
            if (C::NH == 2) {
              x0 = fmaf(__uint_as_float(r1[2 * i]), g1, x0);
              x1 = fmaf(__uint_as_float(r1[2 * i + 1]), g1, x1);
            }
            w[i] = pack_bf16x2(x0, x1);
          }
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c4 * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
          }
        }
        if (valid && split == 0 && half == 0)
          a.lse[(int64_t)it.head * a.T + it.q_row0 + row] = (mref + __log2f(ltot)) * 0.69314718055994530942f;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TM_COLS);
}

}  // namespace

template <int D>
static cudaError_t launch_fwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdArgs& a,
                                int n_items, cudaStream_t st) {
  using C = FwdCfg<D>;
  static bool attr_set = false;  // per process; harmless to repeat
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  fwd_kernel<D><<<n_items * C::NSPLIT, C::THREADS, C::SMEM_BYTES, st>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

cudaError_t launch_fwd(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdArgs& a,
                       int n_items, cudaStream_t st) {
  if (n_items <= 0) return cudaSuccess;
  switch (D) {
    case 64:
      return launch_fwd_d<64>(tq, tk, tv, a, n_items, st);
    case 128:
      return launch_fwd_d<128>(tq, tk, tv, a, n_items, st);
    case 512:
      return launch_fwd_d<512>(tq, tk, tv, a, n_items, st);
    default:
      return cudaErrorInvalidValue;
  }
}

int fwd_key_tile(int /*D*/) { return 128; }
int fwd_query_tile(int /*D*/) { return 128; }

}  // namespace dkv
