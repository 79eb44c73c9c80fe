// attn_bwd.cuh — backward pass of the packed THD attention: dQ, dK, dV.
//
// The gradients the per-sequence causal policy PR ("Add per-sequence causal
// policy to packed THD attention", Validation) checks for parity, with the
// same per-sequence mask types, gaps and grouped heads as the forward:
//   P = exp(scale q k^T - lse),  dV = P^T dO,  dP = dO V^T,
//   dS = P * (dP - D) with D = rowsum(dO * O),
//   dQ = scale dS K,  dK = scale dS^T Q.
//
// Three launches:
//   pre   D = rowsum(dO * O) per (head, row); clears the fp32 dQ accumulator
//         and writes zero dK / dV on rows of no key/value sequence.
//   main  one work item = (sequence, key/value head, 128-key tile).  K and V
//         stay in shared memory while the item loops over the query heads of
//         the group and the query tiles that see the keys:
//            S^T = K Q^T, dP^T = V dO^T           (tcgen05, fp32 in TMEM)
//            P^T, dS^T per key row (one thread per TMEM lane), written back
//            to TMEM (16-bit) and dS^T also to shared memory
//            dV += P^T dO, dK += dS^T Q           (A operand from TMEM)
//            dQ_tile = dS K                       (A = dS^T read MN-major)
//         dK / dV accumulate in TMEM and are written once per item; dQ tiles
//         are added to the fp32 accumulator by bulk tensor reductions (TMA).
//   post  dQ = scale * accumulator, rounded to the input type.
// head_dim 64 or 128 (TMA loads).  Eight warps: warps w and w + 4 read the
// same TMEM lanes and split the columns of the elementwise step, the dQ
// staging and the dK / dV epilogue; the next query tile's Q and dO load while
// the current tile's dQ is added.
#pragma once
#include "attn_common.cuh"

namespace thd {

struct BwdParams {
  AttnParams a;        // q, k, v, metadata, sizes; a.out = forward output O, a.lse = forward LSE
  const void* dout;    // [T, Hq, d]
  void* dq;            // [T, Hq, d]
  void* dk;            // [T, Hkv, d]
  void* dv;            // [T, Hkv, d]
  float* dacc;         // fp32 [T, Hq, d] dQ accumulator (workspace)
  float* D;            // fp32 [Hq, T] (workspace)
};

// ---------------------------------------------------------------------------
// pre
// ---------------------------------------------------------------------------
// Rows of no key/value sequence: gap g lies between key/value spans g-1 and g (the
// gaps before a span one block each; the trailing region after the last span, which
// is most of the buffer when it holds more rows than the batch, in equal shares over
// all blocks).
__device__ void zero_kv_gap_rows(const AttnParams& p, void* dst, long long row_bytes) {
  auto zero_rows = [&](long long a, long long e) {   // rows [a, e)
    if (e <= a) return;
    uint4* d4 = reinterpret_cast<uint4*>(static_cast<char*>(dst) + a * row_bytes);
    const long long n16 = (e - a) * row_bytes / 16;
    for (long long i = threadIdx.x; i < n16; i += blockDim.x) d4[i] = make_uint4(0u, 0u, 0u, 0u);
  };
  for (int g = blockIdx.x; g < p.B; g += gridDim.x) {
    long long a = 0;
    if (g > 0) {
      SeqInfo s = load_seq(p, g - 1);
      a = (long long)s.kv_start + s.kv_len;
    }
    const long long st = p.pad_kv ? (long long)p.pad_kv[g] : (long long)p.cu_kv[g];
    zero_rows(a, st < 0 ? 0 : (st > p.T ? p.T : st));
  }
  long long a = 0;
  if (p.B > 0) {
    SeqInfo s = load_seq(p, p.B - 1);
    a = (long long)s.kv_start + s.kv_len;
  }
  const long long rows = (long long)p.T - a;
  if (rows > 0) zero_rows(a + rows * blockIdx.x / gridDim.x, a + rows * (blockIdx.x + 1) / gridDim.x);
}

template <typename DT>
__global__ void __launch_bounds__(256) attn_bwd_pre_kernel(const BwdParams bp) {
  using Tr = DTypeTraits<DT>;
  const AttnParams& p = bp.a;
  const long long rows = (long long)p.T * p.Hq;
  // D: d/8 lanes per (row, head), 16-byte loads, reduced with shuffles
  const int lanes_per_row = p.d / 8;
  const int lane = threadIdx.x & 31;
  const int sub = lane / lanes_per_row, chunk = lane % lanes_per_row;
  const int rows_per_warp = 32 / lanes_per_row;
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long r0 = warp * rows_per_warp; r0 < rows; r0 += nwarps * rows_per_warp) {
    const long long row = r0 + sub;
    float acc = 0.f;
    if (row < rows) {
      const size_t off = (size_t)row * p.d * 2 + (size_t)chunk * 16;
      const uint4 a = *reinterpret_cast<const uint4*>(static_cast<const char*>(bp.dout) + off);
      const uint4 o = *reinterpret_cast<const uint4*>(static_cast<const char*>(p.out) + off);
      const uint32_t ua[4] = {a.x, a.y, a.z, a.w}, uo[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) acc += Tr::lo(ua[i]) * Tr::lo(uo[i]) + Tr::hi(ua[i]) * Tr::hi(uo[i]);
    }
    for (int m = 1; m < lanes_per_row; m <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (row < rows && chunk == 0) {
      const long long t = row / p.Hq, h = row % p.Hq;
      bp.D[h * p.T + t] = acc;
    }
  }
  // fp32 dQ accumulator = 0
  const long long n4 = rows * p.d / 4;
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long stride = (long long)gridDim.x * blockDim.x;
  float4* acc4 = reinterpret_cast<float4*>(bp.dacc);
  for (long long i = tid; i < n4; i += stride) acc4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  // dK / dV on rows of no key/value sequence
  const long long kv_row_bytes = (long long)p.Hkv * p.d * 2;
  zero_kv_gap_rows(p, bp.dk, kv_row_bytes);
  zero_kv_gap_rows(p, bp.dv, kv_row_bytes);
}

// ---------------------------------------------------------------------------
// post
// ---------------------------------------------------------------------------
template <typename DT>
__global__ void __launch_bounds__(256) attn_bwd_post_kernel(const BwdParams bp) {
  using Tr = DTypeTraits<DT>;
  const AttnParams& p = bp.a;
  const long long n8 = (long long)p.T * p.Hq * p.d / 8;
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const float4* acc4 = reinterpret_cast<const float4*>(bp.dacc);
  uint4* out = reinterpret_cast<uint4*>(bp.dq);
  for (long long i = tid; i < n8; i += stride) {
    const float4 a = acc4[2 * i], b = acc4[2 * i + 1];
    const float sc = p.scale;
    out[i] = make_uint4(Tr::pack2(a.x * sc, a.y * sc), Tr::pack2(a.z * sc, a.w * sc), Tr::pack2(b.x * sc, b.y * sc),
                        Tr::pack2(b.z * sc, b.w * sc));
  }
}

// ---------------------------------------------------------------------------
// main
// ---------------------------------------------------------------------------
template <int DP>
struct BwdSmem {
  static constexpr int kTileBytes = kTileM * DP * 2;
  alignas(1024) uint8_t k[kTileBytes];
  alignas(1024) uint8_t v[kTileBytes];
  alignas(1024) uint8_t q[kTileBytes];
  alignas(1024) uint8_t dout[kTileBytes];
  alignas(1024) uint8_t ds[kTileM * kTileM * 2];   // dS^T: 128 key rows x 128 queries, two 64-query panels
  // head_dim 128: staging of the second 64 dQ columns (fp32, two 32-column panels),
  // so that the next query tile's Q / dO can load while the dQ tile goes out
  alignas(1024) uint8_t stage[DP > 64 ? kTileM * 64 * 4 : 1024];
  float lse2[kTileM];                              // LSE * log2(e) of the tile's queries
  float dd[kTileM];                                // D of the tile's queries
  uint64_t bar_kv, bar_q, bar_mma;
  uint64_t bar_drain;   // the MMAs still in flight when the CTA leaves its loop
  uint32_t tmem_base;
  uint32_t abort;
  WorkItem item;
  SchedSmem sched;
};

// plus up to 1 KB to align the dynamic shared memory: within the 227 KB a CTA may use
static_assert(sizeof(BwdSmem<64>) + 1024 <= 227 * 1024 && sizeof(BwdSmem<128>) + 1024 <= 227 * 1024,
              "shared memory of the backward kernel");

constexpr int kBwdThreads = 256;   // 8 warps: warps w and w + 4 share TMEM lanes, split the columns

template <typename DT, int DP>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq, const BwdParams bp) {
  using Tr = DTypeTraits<DT>;
  const AttnParams& p = bp.a;
  extern __shared__ uint8_t smem_raw[];
  BwdSmem<DP>& sm = *reinterpret_cast<BwdSmem<DP>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = tid & (kTileM - 1);    // TMEM lane: key row of the tile (query row for dQ)
  const int half = tid >> 7;             // column half handled by this thread
  constexpr int kPanels = DP / 64;
  constexpr uint32_t kTileBytes = BwdSmem<DP>::kTileBytes;
  constexpr uint32_t idesc_s = umma_idesc_f16(Tr::kBF16, kTileM, kTileM, false);   // S^T, dP^T
  constexpr uint32_t idesc_acc = umma_idesc_f16(Tr::kBF16, kTileM, DP, true);      // dV, dK (A in TMEM)
  constexpr uint32_t idesc_dq = umma_idesc_f16_ab(Tr::kBF16, kTileM, DP, true, true);
  constexpr uint32_t hi = smem_desc_sw128_hi(1024);
  constexpr int kHalfChunks = DP / 64;   // 32-column chunks of a head_dim-wide row per half

  if (tid == 0) {
    mbar_init(&sm.bar_kv, 1);
    mbar_init(&sm.bar_q, 1);
    mbar_init(&sm.bar_mma, 1);
    mbar_init(&sm.bar_drain, 1);
    fence_mbar_init();
    sm.abort = 0;
    sched_init(sm.sched);
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_dq);
  }
  if (warp == 0) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t t_lane = (uint32_t)((warp & 3) * 32) << 16;
  const uint32_t tDK = tmem, tDV = tmem + DP, tS = tmem + 256, tDP = tmem + 384;
  // low descriptor words: K-major use (head_dim contracted) and MN-major use (rows contracted)
  const uint32_t k_K = smem_desc_sw128_lo(smem_u32(sm.k), 16), k_MN = smem_desc_sw128_lo(smem_u32(sm.k), 16384);
  const uint32_t v_K = smem_desc_sw128_lo(smem_u32(sm.v), 16);
  const uint32_t q_K = smem_desc_sw128_lo(smem_u32(sm.q), 16), q_MN = smem_desc_sw128_lo(smem_u32(sm.q), 16384);
  const uint32_t o_K = smem_desc_sw128_lo(smem_u32(sm.dout), 16);
  const uint32_t o_MN = smem_desc_sw128_lo(smem_u32(sm.dout), 16384);
  const uint32_t ds_MN = smem_desc_sw128_lo(smem_u32(sm.ds), 16384);
  const float sl2 = p.scale_log2;
  volatile uint32_t* abort_flag = &sm.abort;
  uint32_t ph_kv = 0, ph_q = 0, ph_mma = 0;
  // thread 0: phase parity of a K/V or Q/dO load issued and not yet waited for (-1: none),
  // so that a CTA leaving after a wait gave up lets it land first
  int kv_par = -1, q_par = -1;

  // thread 0: Q and dO rows q_start + q0 .. of query head h into shared memory
  auto load_q = [&](int h, int q_row) {
    q_par = (int)ph_q;
    mbar_arrive_expect_tx(&sm.bar_q, 2 * kTileBytes);
#pragma unroll
    for (int pn = 0; pn < kPanels; ++pn) {
      tma_load_2d(sm.q + pn * 16384, &tm_q, &sm.bar_q, h * p.d + pn * 64, q_row);
      tma_load_2d(sm.dout + pn * 16384, &tm_do, &sm.bar_q, h * p.d + pn * 64, q_row);
    }
  };

  Claimer claimer{0ull, 0};   // used by warp 0
  bool injected = false;      // thread 0: the test setting's wait was made
  for (;;) {
    if (warp == 0) {
      const unsigned long long w = claim_item(claimer, p);
      WorkItem it = sched_decode<kTileM, true>(sm.sched, p, w);
      if (lane == 0) sm.item = it;
    }
    __syncthreads();
    if (__syncthreads_or(!sm.item.valid || *abort_flag)) break;
    const WorkItem it = sm.item;
    const SeqInfo& s = it.seq;
    const int g = it.h, kv0 = it.qblock * kTileM;
    const int keys_valid = min(kTileM, s.kv_len - kv0);
    const int key = kv0 + row;                       // this thread's key position (TMEM lane)
    // query tiles holding a query that sees a key of [kv0, kv0 + 128): query i sees key j
    // only if i + shift - lo_off <= j <= i + shift + hi_off
    const long long first_q = (long long)kv0 - s.shift - s.hi_off;
    const long long last_q = (long long)kv0 + kTileM - 1 - s.shift + s.lo_off;
    const int qt_first = first_q <= 0 ? 0 : (int)min(first_q / kTileM, (long long)INT32_MAX);
    const int nqt_all = (s.q_len + kTileM - 1) / kTileM;
    const int nqt = last_q < 0 ? 0 : (int)min((long long)nqt_all, last_q / kTileM + 1);
    const bool any = s.q_len > 0 && qt_first < nqt;
    if (any && tid == 0) {
      kv_par = (int)ph_kv;
      mbar_arrive_expect_tx(&sm.bar_kv, 2 * kTileBytes);
#pragma unroll
      for (int pn = 0; pn < kPanels; ++pn) {
        tma_load_2d(sm.k + pn * 16384, &tm_k, &sm.bar_kv, g * p.d + pn * 64, s.kv_start + kv0);
        tma_load_2d(sm.v + pn * 16384, &tm_v, &sm.bar_kv, g * p.d + pn * 64, s.kv_start + kv0);
      }
      load_q(g * p.group, s.q_start + qt_first * kTileM);   // the item's first query tile
      if (p.inject_wait && !injected) {   // test setting: a wait that runs out, loads in flight
        inject_wait_timeout(p, &sm.bar_drain, abort_flag);
        injected = true;
      }
    }
    bool first = true;
    bool stop = false;
    // LSE * log2(e) and D of query row tid of a tile (zero past the sequence)
    auto row_stats = [&](int h, int q0, float& l2, float& dd) {
      l2 = 0.f;
      dd = 0.f;
      if (tid < min(kTileM, s.q_len - q0)) {
        const size_t li = (size_t)h * p.T + s.q_start + q0 + tid;
        l2 = p.lse[li] * 1.4426950408889634f;
        dd = bp.D[li];
      }
    };
    float nl2 = 0.f, ndd = 0.f;   // the next tile's row statistics, loaded during this tile
    if (any && tid < kTileM) row_stats(g * p.group, qt_first * kTileM, nl2, ndd);
    for (int hh = 0; any && hh < p.group && !stop; ++hh) {
      const int h = g * p.group + hh;
      for (int qt = qt_first; qt < nqt; ++qt) {
        const int q0 = qt * kTileM;
        const int rows_q = min(kTileM, s.q_len - q0);
        if (tid < kTileM) {
          sm.lse2[tid] = nl2;
          sm.dd[tid] = ndd;
        }
        __syncthreads();
        // ---- S^T = K Q^T, dP^T = V dO^T ----
        if (tid == 0) {
          bool ready = true;
          if (first) {
            ready = mbar_wait(&sm.bar_kv, ph_kv, abort_flag, p.status, THD_WAIT_TIMEOUT_BIT, p.wait_limit_ns,
                    p.wait_check_mask);
            if (ready) kv_par = -1;
          }
          if (ready) {
            ready = mbar_wait(&sm.bar_q, ph_q, abort_flag, p.status, THD_WAIT_TIMEOUT_BIT, p.wait_limit_ns,
                    p.wait_check_mask);
            if (ready) q_par = -1;
          }
          if (ready) {   // after a wait gave up nothing more is issued; the waits below give up too
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < DP / 16; ++kk) {
              const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
              umma_ss(tS, smem_desc_join(k_K + off, hi), smem_desc_join(q_K + off, hi), idesc_s, kk > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < DP / 16; ++kk) {
              const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
              umma_ss(tDP, smem_desc_join(v_K + off, hi), smem_desc_join(o_K + off, hi), idesc_s, kk > 0 ? 1u : 0u);
            }
            umma_commit(&sm.bar_mma);
          }
          // the previous tile's dQ staging (in the dS^T and staging buffers) was read
          // while these MMAs run; the barrier below orders it before the dS^T writes
          bulk_wait_group_read0();
        }
        if (first) ph_kv ^= 1u;
        ph_q ^= 1u;
        mbar_wait(&sm.bar_mma, ph_mma, abort_flag, p.status, THD_WAIT_TIMEOUT_BIT, p.wait_limit_ns,
                    p.wait_check_mask);
        ph_mma ^= 1u;
        __syncthreads();
        tc_fence_after();

        if (tid < kTileM) {   // the next tile's statistics load while this one computes
          if (qt + 1 < nqt) row_stats(h, q0 + kTileM, nl2, ndd);
          else if (hh + 1 < p.group) row_stats(h + 1, qt_first * kTileM, nl2, ndd);
        }

        // ---- P^T and dS^T for this thread's key row and column half ----
        // query column c of the tile sees this key iff c_lo <= c <= c_hi (query
        // q0 + c sees key j iff j - shift - hi_off <= q0 + c <= j - shift + lo_off)
        const bool kvalid = key < s.kv_len;
        const long long kd = (long long)key - s.shift - q0;
        const int c_lo = (int)min(max(kd - s.hi_off, -1ll), (long long)kTileM);
        const int c_hi = (int)max(min(kd + s.lo_off, (long long)rows_q - 1), -1ll);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c0 = 2 * half + cc;   // 32-column chunk
          uint32_t sr[32], dr[32];
          tmem_ld32(tS + t_lane + 32 * c0, sr);
          tmem_ld32(tDP + t_lane + 32 * c0, dr);
          tmem_ld_wait_regs32(sr);
          tmem_tie_regs32(dr);
          uint32_t pp[16], pd[16];
          if (__all_sync(0xffffffffu, kvalid && c_lo <= 32 * c0 && c_hi >= 32 * c0 + 31)) {
            // every key row of the warp sees all 32 queries of the chunk: no select
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float pv[2], dsv[2];
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int c = 32 * c0 + 2 * e + u;
                pv[u] = ex2_approx(fmaf(__uint_as_float(sr[2 * e + u]), sl2, -sm.lse2[c]));
                dsv[u] = pv[u] * (__uint_as_float(dr[2 * e + u]) - sm.dd[c]);
              }
              pp[e] = Tr::pack2(pv[0], pv[1]);
              pd[e] = Tr::pack2(dsv[0], dsv[1]);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float pv[2], dsv[2];
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int c = 32 * c0 + 2 * e + u;
                const bool vis = kvalid && c >= c_lo && c <= c_hi;
                const float x = ex2_approx(fmaf(__uint_as_float(sr[2 * e + u]), sl2, -sm.lse2[c]));
                pv[u] = vis ? x : 0.f;
                dsv[u] = pv[u] * (__uint_as_float(dr[2 * e + u]) - sm.dd[c]);
              }
              pp[e] = Tr::pack2(pv[0], pv[1]);
              pd[e] = Tr::pack2(dsv[0], dsv[1]);
            }
          }
          // P^T / dS^T of these 32 queries over the first 16 of their own 32 S^T / dP^T
          // columns: the other column half may still be reading its chunks
          tmem_st16(tS + t_lane + 32 * c0, pp);
          tmem_st16(tDP + t_lane + 32 * c0, pd);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            *reinterpret_cast<uint4*>(sm.ds + sw128_offset(row, 4 * c0 + e)) =
                make_uint4(pd[4 * e], pd[4 * e + 1], pd[4 * e + 2], pd[4 * e + 3]);
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- dV += P^T dO, dK += dS^T Q, dQ_tile = dS K ----
        if (tid == 0 && !*abort_flag) {
          tc_fence_after();
          // 16 queries per step: 8 TMEM columns of P^T / dS^T, two steps per 32-column chunk
#pragma unroll
          for (int kk = 0; kk < kTileM / 16; ++kk)
            umma_ts(tDV, tS + 32 * (kk >> 1) + 8 * (kk & 1), smem_desc_join(o_MN + kk * 128, hi), idesc_acc,
                    (!first || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < kTileM / 16; ++kk)
            umma_ts(tDK, tDP + 32 * (kk >> 1) + 8 * (kk & 1), smem_desc_join(q_MN + kk * 128, hi), idesc_acc,
                    (!first || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < kTileM / 16; ++kk)
            umma_ss(tS, smem_desc_join(ds_MN + kk * 128, hi), smem_desc_join(k_MN + kk * 128, hi), idesc_dq,
                    kk > 0 ? 1u : 0u);
          umma_commit(&sm.bar_mma);
        }
        mbar_wait(&sm.bar_mma, ph_mma, abort_flag, p.status, THD_WAIT_TIMEOUT_BIT, p.wait_limit_ns,
                    p.wait_check_mask);
        ph_mma ^= 1u;
        tc_fence_after();
        first = false;
        // The MMAs that read Q and dO are complete: the next query tile of the item loads
        // while this tile's dQ goes out.
        if (tid == 0 && !*abort_flag) {
          const bool more = qt + 1 < nqt || hh + 1 < p.group;
          if (more) {
            const int nh = qt + 1 < nqt ? h : h + 1;
            const int nrow = s.q_start + (qt + 1 < nqt ? (qt + 1) * kTileM : qt_first * kTileM);
            load_q(nh, nrow);
          }
        }
        // ---- dQ tile into the fp32 accumulator by bulk tensor reductions, 64 columns
        // at a time, staged in the dS^T buffer (free once the MMAs completed) and, with
        // head_dim 128, the staging buffer ----
#pragma unroll
        for (int r = 0; r < DP / 64; ++r) {
          const int c = 2 * r + half;   // 32-column chunk: panel `half` of the staging buffer
          uint8_t* stage = r == 0 ? sm.ds : sm.stage;
          uint32_t o[32];
          tmem_ld32(tS + t_lane + 32 * c, o);
          tmem_ld_wait_regs32(o);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            *reinterpret_cast<uint4*>(stage + sw128_offset(row, 8 * half + e)) =
                make_uint4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
          fence_proxy_async_smem();
          __syncthreads();
          if (tid == 0) {
            // rows past the sequence carry dS = 0, so their (zero) rows add nothing
            tma_reduce_add_2d(&tm_dq, stage, h * p.d + 64 * r, s.q_start + q0);
            tma_reduce_add_2d(&tm_dq, stage + 16384, h * p.d + 64 * r + 32, s.q_start + q0);
            bulk_commit_group();
          }
        }
        // (the staging buffers' reads are waited for before the next tile writes dS^T)
        tc_fence_before();
        if (__syncthreads_or(*abort_flag != 0u)) {
          stop = true;
          break;
        }
      }
    }

    // ---- dK, dV rows of this key tile (one column half per thread) ----
    if (keys_valid > 0) {
      const bool row_ok = row < keys_valid;
      const size_t base = ((size_t)(s.kv_start + (row_ok ? key : kv0)) * p.Hkv + g) * (size_t)p.d;
      DT* dkp = static_cast<DT*>(bp.dk) + base;
      DT* dvp = static_cast<DT*>(bp.dv) + base;
      if (any && !first) {
#pragma unroll
        for (int cc = 0; cc < kHalfChunks; ++cc) {
          const int c = half * kHalfChunks + cc;
          uint32_t a[32], b[32];
          tmem_ld32(tDK + t_lane + 32 * c, a);
          tmem_ld32(tDV + t_lane + 32 * c, b);
          tmem_ld_wait_regs32(a);
          tmem_tie_regs32(b);
          if (row_ok) {
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              uint4 x, y;
              x.x = Tr::pack2(__uint_as_float(a[e]) * p.scale, __uint_as_float(a[e + 1]) * p.scale);
              x.y = Tr::pack2(__uint_as_float(a[e + 2]) * p.scale, __uint_as_float(a[e + 3]) * p.scale);
              x.z = Tr::pack2(__uint_as_float(a[e + 4]) * p.scale, __uint_as_float(a[e + 5]) * p.scale);
              x.w = Tr::pack2(__uint_as_float(a[e + 6]) * p.scale, __uint_as_float(a[e + 7]) * p.scale);
              y.x = Tr::pack2(__uint_as_float(b[e]), __uint_as_float(b[e + 1]));
              y.y = Tr::pack2(__uint_as_float(b[e + 2]), __uint_as_float(b[e + 3]));
              y.z = Tr::pack2(__uint_as_float(b[e + 4]), __uint_as_float(b[e + 5]));
              y.w = Tr::pack2(__uint_as_float(b[e + 6]), __uint_as_float(b[e + 7]));
              *reinterpret_cast<uint4*>(dkp + 32 * c + e) = x;
              *reinterpret_cast<uint4*>(dvp + 32 * c + e) = y;
            }
          }
        }
      } else if (row_ok) {
        for (int c = half * (DP / 2); c < (half + 1) * (DP / 2); c += 8) {
          *reinterpret_cast<uint4*>(dkp + c) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(dvp + c) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (stop) break;
  }
  if (tid == 0) {
    bulk_wait_group0();   // dQ reductions complete
    // after a wait gave up: loads issued and not waited for land, and the MMAs
    // already issued complete, before TMEM is released and the CTA exits
    if (kv_par >= 0) drain_wait(&sm.bar_kv, (uint32_t)kv_par);
    if (q_par >= 0) drain_wait(&sm.bar_q, (uint32_t)q_par);
    umma_commit(&sm.bar_drain);
    drain_wait(&sm.bar_drain, 0);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace thd
