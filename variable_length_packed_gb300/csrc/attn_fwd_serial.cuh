// attn_fwd_serial.cuh — a straightforward (non-pipelined) tcgen05 attention
// kernel: one 128-row Q tile per work item, four warps, each KV tile processed
// as  TMA -> UMMA S = Q K^T (TMEM) -> softmax in registers -> P to shared
// memory -> UMMA O += P V (TMEM)  with a full wait between the steps.  It
// computes the same result as the pipelined kernel and backs the head
// dimensions the TMA path does not cover (any multiple of 8 up to 128, loaded
// with plain vector loads into the same swizzled layout).
#pragma once
#include "attn_common.cuh"

namespace thd {

template <int DP>
struct SerialSmem {
  static constexpr int kTileBytes = kTileM * DP * 2;   // 128 rows x DP halves
  alignas(1024) uint8_t q[kTileBytes];
  alignas(1024) uint8_t k[kTileBytes];
  alignas(1024) uint8_t v[kTileBytes];
  alignas(1024) uint8_t p[kTileM * kBlockN * 2];
  uint64_t bar_load;
  uint64_t bar_mma;
  uint64_t bar_drain;   // the MMAs still in flight when the CTA leaves its loop
  uint32_t tmem_base;
  uint32_t abort;
  WorkItem item;
  SchedSmem sched;
};

// Plain vector loads of a 128-row tile (rows row0.., head column col0) into
// the swizzled layout; chunks past d and rows outside [0, T) are zero.
template <int DP>
__device__ __forceinline__ void load_tile_manual(uint8_t* dst, const void* src, int row0, int nrows_valid,
                                                 int heads, int head, int d, int T) {
  const int cpr = DP / 8;   // 16-byte chunks per row
  const int dch = d / 8;
  for (int idx = threadIdx.x; idx < kTileM * cpr; idx += blockDim.x) {
    const int r = idx / cpr, c = idx % cpr;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    const int row = row0 + r;
    if (c < dch && r < nrows_valid && row >= 0 && row < T) {
      const uint4* g = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(src) +
                                                      ((size_t)row * heads + head) * (size_t)d * 2) + c;
      val = *g;
    }
    *reinterpret_cast<uint4*>(dst + sw128_offset(r, c)) = val;
  }
}

template <typename DT, int DP, bool kTMA>
__global__ void __launch_bounds__(128, 1)
    attn_fwd_serial_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using Tr = DTypeTraits<DT>;
  extern __shared__ uint8_t smem_raw[];
  SerialSmem<DP>& sm = *reinterpret_cast<SerialSmem<DP>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  constexpr int kPanels = DP / 64;                        // 64-column swizzle panels
  constexpr uint32_t kTileBytes = SerialSmem<DP>::kTileBytes;
  constexpr uint32_t kTmemCols = 256;                     // S: [0,128), O: [128, 128+DP)
  constexpr uint32_t idesc_qk = umma_idesc_f16(Tr::kBF16, kTileM, kBlockN, false);
  constexpr uint32_t idesc_pv = umma_idesc_f16(Tr::kBF16, kTileM, DP, true);

  if (tid == 0) {
    mbar_init(&sm.bar_load, 1);
    mbar_init(&sm.bar_mma, 1);
    mbar_init(&sm.bar_drain, 1);
    fence_mbar_init();
    sm.abort = 0;
    sched_init(sm.sched);
    if (kTMA) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
  }
  if (warp == 0) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t t_lane = (uint32_t)(warp * 32) << 16;
  const uint32_t tS = tmem;
  const uint32_t tO = tmem + 128;

  zero_pad_rows(p, 0, blockDim.x, 2);

  uint32_t ph_load = 0, ph_mma = 0;
  int load_par = -1;   // thread 0 (TMA): phase parity of a load issued and not yet waited for
  volatile uint32_t* abort_flag = &sm.abort;

  Claimer claimer{0ull, 0};   // used by warp 0
  bool injected = false;      // thread 0: the test setting's wait was made
  for (;;) {
    if (warp == 0) {
      const unsigned long long w = claim_item(claimer, p);
      WorkItem it = sched_decode<kTileM>(sm.sched, p, w);
      if (lane == 0) sm.item = it;
    }
    __syncthreads();
    if (__syncthreads_or(!sm.item.valid || *abort_flag)) break;
    const WorkItem it = sm.item;
    const SeqInfo& s = it.seq;
    const int q0 = it.qblock * kTileM;                  // first query position of the tile
    const int rows_valid = min(kTileM, s.q_len - q0);
    const int kvh = it.h / p.group;
    // KV tiles [j0, nkv) hold the keys the tile's rows see
    int nkv = kv_tiles_for(s, q0, kTileM);
    int j0 = kv_first_tile(s, q0);
    if (nkv <= j0) nkv = j0 = 0;
    const int qpos = q0 + tid;                          // this thread's query position

    // l_run: sum of the P values as rounded for the P V product (normalises O, so each
    // output row is an exact convex combination of V rows with the rounded weights);
    // l_exact: the unrounded fp32 sum (gives the LSE).
    float m_run = -INFINITY, l_run = 0.f, l_exact = 0.f;

    if (nkv > 0) {
      // ---- Q and first K/V tile ----
      if (kTMA) {
        if (tid == 0) {
          load_par = (int)ph_load;
          mbar_arrive_expect_tx(&sm.bar_load, 3 * kTileBytes);
#pragma unroll
          for (int pn = 0; pn < kPanels; ++pn) {
            tma_load_2d(sm.q + pn * 16384, &tm_q, &sm.bar_load, it.h * p.d + pn * 64, s.q_start + q0);
            tma_load_2d(sm.k + pn * 16384, &tm_k, &sm.bar_load, kvh * p.d + pn * 64, s.kv_start + j0 * kBlockN);
            tma_load_2d(sm.v + pn * 16384, &tm_v, &sm.bar_load, kvh * p.d + pn * 64, s.kv_start + j0 * kBlockN);
          }
        }
      } else {
        const int kvr = j0 * kBlockN;
        load_tile_manual<DP>(sm.q, p.q, s.q_start + q0, rows_valid, p.Hq, it.h, p.d, p.T);
        load_tile_manual<DP>(sm.k, p.k, s.kv_start + kvr, min(kBlockN, s.kv_len - kvr), p.Hkv, kvh, p.d, p.T);
        load_tile_manual<DP>(sm.v, p.v, s.kv_start + kvr, min(kBlockN, s.kv_len - kvr), p.Hkv, kvh, p.d, p.T);
        fence_proxy_async_smem();
        __syncthreads();
      }

      for (int j = j0; j < nkv; ++j) {
        const int kv0 = j * kBlockN;
        // ---- S = Q K^T ----
        if (tid == 0) {
          if (p.inject_wait && !injected) {   // test setting: a wait that runs out, loads in flight
            inject_wait_timeout(p, &sm.bar_drain, abort_flag);
            injected = true;
          }
          if (kTMA && mbar_wait(&sm.bar_load, ph_load, abort_flag, p.status, THD_WAIT_TIMEOUT_BIT, p.wait_limit_ns,
                    p.wait_check_mask))
            load_par = -1;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < DP / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            umma_ss(tS, smem_desc_sw128(smem_u32(sm.q) + off, 16, 1024),
                    smem_desc_sw128(smem_u32(sm.k) + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
          }
          umma_commit(&sm.bar_mma);
        }
        if (kTMA) ph_load ^= 1u;
        mbar_wait(&sm.bar_mma, ph_mma, abort_flag, p.status, THD_WAIT_TIMEOUT_BIT, p.wait_limit_ns,
                    p.wait_check_mask);
        ph_mma ^= 1u;
        tc_fence_after();

        // ---- softmax on this thread's row ----
        uint32_t sr[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + t_lane + c * 32, sr + c * 32);
        tmem_ld_wait_regs32(sr);
        tmem_tie_regs32(sr + 32);
        tmem_tie_regs32(sr + 64);
        tmem_tie_regs32(sr + 96);

        const long long d0 = (long long)q0 + s.shift;
        const bool need_mask = (kv0 + kBlockN > s.kv_len) || (kv0 + kBlockN - 1 > d0 + s.hi_off) ||
                               (kv0 < d0 + (kTileM - 1) - s.lo_off);
        const int key_lo = seq_first_key(s, qpos), key_hi = seq_last_key(s, qpos);
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          float x = __uint_as_float(sr[c]);
          if (need_mask) {
            const int kp = kv0 + c;
            x = (kp >= key_lo && kp <= key_hi) ? x : -INFINITY;
            sr[c] = __float_as_uint(x);
          }
          mx = fmaxf(mx, x);
        }
        const float m_new = fmaxf(m_run, mx);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ex2_approx((m_run - m_use) * p.scale_log2);
        const float mb = m_use * p.scale_log2;
        float lsum = 0.f, lsum_exact = 0.f;
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float e0 = ex2_approx(fmaf(__uint_as_float(sr[2 * c]), p.scale_log2, -mb));
          const float e1 = ex2_approx(fmaf(__uint_as_float(sr[2 * c + 1]), p.scale_log2, -mb));
          pk[c] = Tr::pack2(e0, e1);
          lsum += Tr::lo(pk[c]) + Tr::hi(pk[c]);
          lsum_exact += e0 + e1;
        }
        l_run = l_run * alpha + lsum;
        l_exact = l_exact * alpha + lsum_exact;
        m_run = m_new;

        // ---- rescale O (after the previous P V has completed) ----
        if (j > j0) {
#pragma unroll
          for (int c = 0; c < DP / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + t_lane + c * 32, o);
            tmem_ld_wait_regs32(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + t_lane + c * 32, o);
          }
          tmem_st_wait();
        }

        // ---- P (row tid, 128 keys) to shared memory, swizzled K-major ----
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          *reinterpret_cast<uint4*>(sm.p + sw128_offset(tid, c)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- O += P V ----
        if (tid == 0) {
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kBlockN / 16; ++kk) {
            const uint32_t poff = (kk >> 2) * 16384 + (kk & 3) * 32;
            const uint32_t voff = kk * 16 * 128;   // 16 key rows of 128 bytes
            umma_ss(tO, smem_desc_sw128(smem_u32(sm.p) + poff, 16, 1024),
                    smem_desc_sw128(smem_u32(sm.v) + voff, 16384, 1024), idesc_pv,
                    (j > j0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&sm.bar_mma);
        }
        mbar_wait(&sm.bar_mma, ph_mma, abort_flag, p.status, THD_WAIT_TIMEOUT_BIT, p.wait_limit_ns,
                    p.wait_check_mask);
        ph_mma ^= 1u;
        tc_fence_after();

        // ---- next K/V tile ----
        if (j + 1 < nkv) {
          const int kvn = (j + 1) * kBlockN;
          if (kTMA) {
            if (tid == 0) {
              load_par = (int)ph_load;
              mbar_arrive_expect_tx(&sm.bar_load, 2 * kTileBytes);
#pragma unroll
              for (int pn = 0; pn < kPanels; ++pn) {
                tma_load_2d(sm.k + pn * 16384, &tm_k, &sm.bar_load, kvh * p.d + pn * 64, s.kv_start + kvn);
                tma_load_2d(sm.v + pn * 16384, &tm_v, &sm.bar_load, kvh * p.d + pn * 64, s.kv_start + kvn);
              }
            }
          } else {
            __syncthreads();
            load_tile_manual<DP>(sm.k, p.k, s.kv_start + kvn, min(kBlockN, s.kv_len - kvn), p.Hkv, kvh, p.d,
                                 p.T);
            load_tile_manual<DP>(sm.v, p.v, s.kv_start + kvn, min(kBlockN, s.kv_len - kvn), p.Hkv, kvh, p.d,
                                 p.T);
            fence_proxy_async_smem();
            __syncthreads();
          }
        }
        if (__syncthreads_or(*abort_flag != 0u)) break;
      }
    }

    // ---- epilogue: O / l -> out, LSE (TMEM loads are warp-collective: all
    // threads load, only rows of the sequence store) ----
    const bool row_ok = tid < rows_valid;
    const size_t orow = ((size_t)(s.q_start + (row_ok ? qpos : 0)) * p.Hq + it.h) * (size_t)p.d;
    DT* dst = static_cast<DT*>(p.out) + orow;
    if (nkv > 0) {
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;   // a row that saw no key stays 0
#pragma unroll
      for (int c = 0; c < DP / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + t_lane + c * 32, o);
        tmem_ld_wait_regs32(o);
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          const int col = c * 32 + e;
          if (row_ok && col < p.d) {
            uint4 v4;
            v4.x = Tr::pack2(__uint_as_float(o[e + 0]) * inv, __uint_as_float(o[e + 1]) * inv);
            v4.y = Tr::pack2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
            v4.z = Tr::pack2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
            v4.w = Tr::pack2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
            *reinterpret_cast<uint4*>(dst + col) = v4;
          }
        }
      }
      if (row_ok && p.lse) p.lse[(size_t)it.h * p.T + s.q_start + qpos] = m_run * p.scale + logf(l_exact);
    } else if (row_ok) {
      for (int col = 0; col < p.d; col += 8) *reinterpret_cast<uint4*>(dst + col) = make_uint4(0, 0, 0, 0);
      if (p.lse) p.lse[(size_t)it.h * p.T + s.q_start + qpos] = -INFINITY;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  // After a wait gave up, MMAs (and, with TMA, a load) may still be in flight:
  // they complete before TMEM is released and the CTA exits.
  if (tid == 0) {
    if (load_par >= 0) drain_wait(&sm.bar_load, (uint32_t)load_par);
    umma_commit(&sm.bar_drain);
    drain_wait(&sm.bar_drain, 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace thd
