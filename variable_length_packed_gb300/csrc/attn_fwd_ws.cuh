// attn_fwd_ws.cuh — the persistent, warp-specialised attention kernel
// (head_dim 64 or 128, TMA loads).
//
// One CTA per SM.  A work item is two 128-row Q tiles of one sequence that share
// every K/V tile: the same 128 rows of two query heads of one group when the
// number of query heads per K/V head is even, else a block of 256 rows of one
// query head.  Twelve warps in three warpgroups:
//
//   warp 0      scheduler + TMA producer: claims items from the global counter,
//               publishes them to the other warps, loads Q (both tiles) and the
//               K/V tiles of the item into a ring (2 stages at head_dim 128, 4
//               at 64).
//   warp 1      MMA issuer: S_i = Q_i K_j^T into TMEM (SS UMMA), then
//               O_i += P_i V_j with P_i read from TMEM (TS UMMA); the two tiles
//               alternate so one tile's softmax overlaps the other tile's MMAs.
//               The whole warp runs the loop converged (descriptors and waits
//               warp-uniform) and one elected lane issues the MMAs and commits.
//   warps 2-3   write the pad rows' zeros, then wait at the end.
//   warps 4-7   softmax of Q tile 0; warps 8-11 softmax of Q tile 1.  One thread
//               per query row (= TMEM lane): masking, online max / sum, P
//               (rounded to the input type) written over S in TMEM in two
//               halves of 64 keys (the MMA warp starts P V on the first half
//               while the second is computed), lazy O rescaling (only when the
//               running max grows by more than 2^8), and the epilogue
//               O / l -> out, LSE.
//
// Each tile's chain softmax(S_t(j)) -> P_t(j) V_j -> S_t(j+1) is serial (P_t
// lives in S_t's TMEM columns), so throughput comes from interleaving the two
// tiles: while one tile's softmax runs, the tensor pipe works on the other's
// MMAs.  K and V stages are released separately: a K stage once both tiles'
// S MMAs on it are done, a V stage once both P V MMAs are done.
//
// Short sequences (at most 128 query rows and 128 keys) are not blocked that
// way.  Without a window, runs of consecutive short sequences are packed into
// one 128-row Q window and one 128-key K/V window each (a per-row table of
// visible keys masks the other sequences' keys), in scheduler chunks where that
// saves enough tiles; otherwise (and with a window) each (sequence, head) is its
// own tile.  These tiles are paired, two independent tiles per
// work unit, each with its own K/V tile, and the MMA warp issues each tile's
// P_t V and then the next unit's S_t as soon as their inputs are ready (the
// barriers of both tiles are polled), so the two softmax warpgroups alternate
// across units the way they alternate across KV tiles of a long sequence.
//
// With a sliding window (kWin), a Q tile visits only the KV tiles inside its
// rows' bands, starting at its own first tile, and rows mask keys on both
// sides; the kernel without a window is a separate instantiation.
//
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 and O1 after them; P_i
// occupies the first 64 columns of S_i (two 16-bit values per column).
//
// Every wait is bounded (p.wait_limit_ns).  A wait that runs out sets the CTA's
// abort flag and the status bit; every role then leaves its loop and waits, with
// a bound of its own and ignoring the flag, for the asynchronous work it started
// (the producer for each TMA copy it issued, the MMA thread for its committed
// MMAs), so no copy or MMA is in flight when TMEM is released and the CTA exits.
#pragma once
#include "attn_common.cuh"

namespace thd {

constexpr int kWsBlockM = 256;   // query rows per work item (two Q tiles)
// Ring depths: head_dim 128 fills shared memory with one Q slot (two tiles) and
// two K/V stages; head_dim 64 has room for two Q slots (the next item's Q loads
// while the current one computes) and four K/V stages.
template <int DP> struct WsDepth { static constexpr int kQSlots = DP == 64 ? 2 : 1, kStages = DP == 64 ? 4 : 2; };
constexpr int kWsThreads = 384;  // 12 warps: three warpgroups
// Registers per thread after the split (setmaxnreg): the first warpgroup
// (producer, MMA issuer, pad-row warps) gives registers to the two softmax
// warpgroups, whose rows of S take most of them; the split adds up to what the
// block is launched with (384 threads x 168 registers).
constexpr uint32_t kRegsCtl = 112, kRegsSoftmax = 192;
static_assert(128 * kRegsCtl + 256 * kRegsSoftmax <= 384 * 168, "register split within the launch's registers");
constexpr float kRescaleThreshold = 8.0f;   // log2 units

// One 128-row Q tile of a work unit.
struct WsTile {
  SeqInfo seq;   // the tile's sequence
  int h;         // query head
  int q0;        // sequence position of the tile's first query row
  int j0, n;     // KV tiles the tile visits: [j0, n); n = 0 when no row sees a key
};

// Work unit: two Q tiles of a long sequence (two heads of one group over the
// same 128 rows, or 256 rows of one head; both share every K/V tile, `paired` =
// 0), or two independent tiles of short sequences, each with its own single K/V
// tile (`paired` = 1).  A short tile is one (packed group, head) when the kernel
// has no window and the chunk packs its short sequences (`packed` = 1: the
// group's consecutive sequences share the tile's 128 rows and 128 keys, each row
// seeing only its own sequence's keys), else one (sequence, head).
struct WsUnit {
  int valid;
  int paired;
  int packed;    // paired tiles of packed groups (row tables in the unit's slot)
  int jb;        // first KV tile loaded (shared: the smallest j0 of the tiles with work)
  int n_all;     // K/V tiles loaded for the unit: max(n) - jb shared, n0 + n1 paired
  int g[2];      // packed tiles: chunk group of each tile (-1: no rows)
  WsTile t[2];
};

// Row table of a packed tile: per row, its first and last visible key as int16
// tile columns (low / high half); rows of no sequence of the group are marked
// kRowAbsent (no keys, no output).
constexpr int kRowAbsent = 0x7FFF;
__device__ __forceinline__ uint32_t row_keys(int first, int last) {
  return ((uint32_t)first & 0xFFFFu) | ((uint32_t)last << 16);
}
constexpr uint32_t kRowAbsentKeys = ((uint32_t)kRowAbsent & 0xFFFFu) | (0xFFFFu << 16);   // (absent, -1)

// What the MMA warp needs of a unit (the sequences' positions stay with the
// producer and the softmax warps).
struct MmaUnit {
  int valid, paired, jb, n_all;
  int j0[2], n[2];
};

// KV tile range of a Q tile, [j0, n), normalised to (0, 0) when empty.  kWin:
// the call has a sliding window (without one every visited range starts at 0).
template <bool kWin>
__device__ __forceinline__ void ws_tile_range(WsTile& tt) {
  const SeqInfo& s = tt.seq;
  tt.n = s.q_len > tt.q0 ? kv_tiles_for(s, tt.q0, kTileM) : 0;
  tt.j0 = kWin ? kv_first_tile(s, tt.q0) : 0;
  if (tt.n <= tt.j0) tt.n = tt.j0 = 0;
}

template <int DP>
struct WsSmem {
  static constexpr int kTileBytes = kTileM * DP * 2;
  static constexpr int kQSlots = WsDepth<DP>::kQSlots, kStages = WsDepth<DP>::kStages;
  alignas(1024) uint8_t q[kQSlots][2][kTileBytes];
  alignas(1024) uint8_t k[kStages][kTileBytes];
  alignas(1024) uint8_t v[kStages][kTileBytes];
  uint64_t q_full[kQSlots], q_empty[kQSlots];
  uint64_t k_full[kStages], v_full[kStages], k_empty[kStages], v_empty[kStages];
  uint64_t s_full[2], p_lo[2], p_hi[2], o_full[2];
  uint64_t item_full[2], item_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort;
  WsUnit items[2];
  uint32_t rows[2][2][kTileM];   // packed tiles' row tables, per item slot and tile
  SchedSmem sched;
};
// plus up to 1 KB to align the dynamic shared memory: within the 227 KB a CTA may use
static_assert(sizeof(WsSmem<64>) + 1024 <= 227 * 1024 && sizeof(WsSmem<128>) + 1024 <= 227 * 1024,
              "shared memory of the warp-specialised kernel");

// Maps global unit index w to its work unit (one full warp; w never decreases
// within a CTA).  Units of a chunk: the long sequences' two-tile blocks in the
// scheduler's order, then the short tiles ((packed group, head) without a
// window, (sequence, head) with one), heads innermost, two per unit.
template <bool kWin, bool kPack>
__device__ __forceinline__ WsUnit ws_decode(SchedSmem& s, const AttnParams& p, unsigned long long w) {
  WsUnit u;
  u.valid = 0;
  u.paired = 0;
  u.packed = 0;
  u.jb = 0;
  u.n_all = 0;
  u.g[0] = u.g[1] = -1;
  if (!sched_seek<kWsBlockM, false, true, kPack>(s, p, w)) return u;
  u.valid = 1;
  const uint32_t local = (uint32_t)(w - s.item_base);
  const uint32_t n_long_items = s.cum[s.chunk_n];
  if (local < n_long_items) {
    const int pos = sched_find(s, local);
    const SeqInfo seq = cached_seq(s, s.order[pos], p);
    const uint32_t r = local - s.cum[pos];
    // Grouped query heads (an even number per key/value head): the two tiles are the
    // same 128 rows of two heads of one group, so they visit the same KV tiles.
    // Otherwise: two consecutive 128-row blocks of one head.
    const bool head_pair = (p.group & 1) == 0;
    const int rows_blk = head_pair ? kTileM : kWsBlockM;
    const uint32_t nblk = (uint32_t)((seq.q_len + rows_blk - 1) / rows_blk);
    const int hsel = (int)(r / nblk);
    const int qb = (int)(nblk - 1u - r % nblk);   // heaviest (last) block first
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      u.t[t].seq = seq;
      u.t[t].h = head_pair ? 2 * hsel + t : hsel;
      u.t[t].q0 = head_pair ? qb * kTileM : qb * kWsBlockM + t * kTileM;
      ws_tile_range<kWin>(u.t[t]);
    }
    // tile 0's rows come first, so its window starts no later than tile 1's
    u.jb = !kWin ? 0 : (u.t[0].n > 0 ? u.t[0].j0 : u.t[1].j0);
    const int jend = max(u.t[0].n, u.t[1].n);
    u.n_all = jend > u.jb ? jend - u.jb : 0;
  } else {
    u.paired = 1;
    u.packed = (kPack && s.pack_on) ? 1 : 0;
    const uint32_t total = (uint32_t)(u.packed ? s.n_groups : s.n_short) * (uint32_t)p.Hq;
    const uint32_t i0 = 2u * (local - n_long_items);
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const uint32_t idx = i0 + t;
      WsTile& tt = u.t[t];
      if (idx < total && kPack && u.packed) {
        // the group's rows [first q_start, last q end) and keys [first kv_start, last kv end)
        const int g = (int)(idx / (uint32_t)p.Hq);
        const int4 a = s.span[s.grp.start[g]];
        const int4 e = s.span[s.grp.end[g] - 1];
        u.g[t] = g;
        tt.seq = SeqInfo{a.x, a.z, e.x + e.y - a.x, e.z + e.w - a.z, 0, 0, kNoBound, kNoBound};
        tt.h = (int)(idx % (uint32_t)p.Hq);
        tt.q0 = 0;
        tt.j0 = 0;
        tt.n = tt.seq.kv_len > 0 ? 1 : 0;
      } else if (idx < total) {
        tt.seq = cached_seq(s, s.order[s.n_long + (int)(idx / (uint32_t)p.Hq)], p);
        tt.h = (int)(idx % (uint32_t)p.Hq);
        tt.q0 = 0;
        ws_tile_range<kWin>(tt);   // at most KV tile 0
      } else {   // odd count: no second tile
        tt.seq = SeqInfo{0, 0, 0, 0, 0, 0, kNoBound, kNoBound};
        tt.h = 0;
        tt.q0 = 0;
        tt.j0 = tt.n = 0;
      }
    }
    u.n_all = u.t[0].n + u.t[1].n;
  }
  return u;
}

// S = Q K^T over head_dim DP: DP/16 K steps of 16 elements (32 bytes inside a
// 128-byte swizzle row; the second 64-column panel starts 16 KB further).
// q_lo / k_lo are the low descriptor words of the tiles' first K step.
template <int DP>
__device__ __forceinline__ void issue_qk(bool leader, uint32_t tS, uint32_t q_lo, uint32_t k_lo, uint32_t idesc) {
  constexpr uint32_t hi = smem_desc_sw128_hi(1024);
#pragma unroll
  for (int kk = 0; kk < DP / 16; ++kk) {
    const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
    umma_ss_if(leader, tS, smem_desc_join(q_lo + off, hi), smem_desc_join(k_lo + off, hi), idesc, kk > 0 ? 1u : 0u);
  }
}

// O += P[:, 16*k0 : 16*k1] V[16*k0 : 16*k1, :].  v_lo is the low descriptor word
// of the V tile (MN-major: the next 64 head-dim columns are 16 KB further).
template <int k0, int k1>
__device__ __forceinline__ void issue_pv(bool leader, uint32_t tO, uint32_t tP, uint32_t v_lo, uint32_t idesc, bool acc) {
  constexpr uint32_t hi = smem_desc_sw128_hi(1024);
#pragma unroll
  for (int kk = k0; kk < k1; ++kk) {
    // 16 keys per step: 8 TMEM columns of packed P, 16 rows (2048 bytes) of V
    umma_ts_if(leader, tO, tP + kk * 8, smem_desc_join(v_lo + kk * (2048 >> 4), hi), idesc, (acc || kk > 0) ? 1u : 0u);
  }
}

// Wait that also gives up when the CTA aborted.
#define WS_WAIT(bar, parity) \
  mbar_wait((bar), (parity), abort_flag, p.status, THD_WAIT_TIMEOUT_BIT, p.wait_limit_ns, p.wait_check_mask)

// Warp-uniform variant: every lane waits, and the warp gives up together, so the
// warp-collective tcgen05.ld / tcgen05.st that follow stay convergent.
#define WS_WAIT_WARP(bar, parity) (__all_sync(0xffffffffu, WS_WAIT((bar), (parity)) ? 1 : 0) != 0)

// Non-blocking phase test with lane 0's answer for the whole warp (the MMA warp
// polls several barriers and must take every decision together).
__device__ __forceinline__ bool warp_test_wait(uint64_t* bar, uint32_t parity) {
  return __shfl_sync(0xffffffffu, mbar_test_wait(bar, parity) ? 1 : 0, 0) != 0;
}

// Row table of packed group g (chunk-local; -1: every row absent): row r of
// the tile is query row r of the window that starts at the group's first
// q_start; a row inside member b at position i sees keys [0, last] of b (there
// is no window where groups are packed: last = kv_len - 1, or the diagonal i +
// shift under a causal type), shifted by b's kv_start past the group's first.
// A row with no visible key gets last < first.  One full warp.
__device__ __forceinline__ void ws_fill_rows(uint32_t* tab, const SchedSmem& s, int g, int lane) {
  uint32_t v[kTileM / 32];
#pragma unroll
  for (int k = 0; k < kTileM / 32; ++k) v[k] = kRowAbsentKeys;
  if (g >= 0) {
    const int a = s.grp.start[g], e = s.grp.end[g];
    const int4 f = s.span[a];
    for (int b = a; b < e; ++b) {
      const int4 sp = s.span[b];   // q_start, q_len, kv_start, kv_len (at most 128 each)
      const int code = s.code[b];
      const int r0 = sp.x - f.x, kofs = sp.z - f.z;
      const int diag = code == kMaskPadding ? kBlockN : (code == kMaskCausalBottomRight ? sp.w - sp.y : 0);
#pragma unroll
      for (int k = 0; k < kTileM / 32; ++k) {
        const int i = lane + 32 * k - r0;
        if (i >= 0 && i < sp.y) v[k] = row_keys(kofs, kofs + min(i + diag, sp.w - 1));
      }
    }
  }
#pragma unroll
  for (int k = 0; k < kTileM / 32; ++k) tab[lane + 32 * k] = v[k];
}

// ---------------------------------------------------------------------------
// warp 0: scheduler + TMA producer
// ---------------------------------------------------------------------------
template <int DP, bool kWin, bool kPack>
__device__ void ws_producer(WsSmem<DP>& sm, const AttnParams& p, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                            const CUtensorMap* tm_v, volatile uint32_t* abort_flag) {
  constexpr uint32_t kTileBytes = WsSmem<DP>::kTileBytes;
  constexpr int kPanels = DP / 64;
  constexpr int kQSlots = WsSmem<DP>::kQSlots, kWsStages = WsSmem<DP>::kStages;
  const int lane = threadIdx.x & 31;
  uint32_t it_cnt = 0, q_cnt = 0, kv_cnt = 0;
  bool ok = true;
  Claimer claimer{0ull, 0};
  // The packing instantiation claims half-size batches one batch ahead (lane 0 holds the
  // current batch and the next one, whose atomic is in flight while the current one runs),
  // so a CTA still holds at most p.claim unstarted units; claimed indices still increase.
  unsigned long long ahead_cur = 0, ahead_nxt = 0, ahead_base = 0;
  int ahead_left = 0;
  bool ahead_init = false;
  // packed tiles: the (chunk, group) whose row table each slot's tile holds,
  // as chunk_base * 1024 + group + 1 (group -1: a tile without rows, whose table
  // marks every row absent), -1 while the slot has none (slot 0 tiles 0, 1, then
  // slot 1); the query heads of a group share the table, so it is built once per
  // slot and group
  long long rows_of[4] = {-1, -1, -1, -1};
  for (;;) {
    unsigned long long w;
    if (kPack) {   // half-size batches, the next one's atomic in flight while this one runs
      const int c = p.claim > 1 ? p.claim / 2 : 1;
      if (ahead_left == 0) {
        unsigned long long b = 0;
        if (lane == 0) {
          if (!ahead_init) {
            ahead_cur = atomicAdd(p.work_counter, (unsigned long long)c);
            ahead_init = true;
          } else {
            ahead_cur = ahead_nxt;
          }
          ahead_nxt = atomicAdd(p.work_counter, (unsigned long long)c);
          b = ahead_cur;
        }
        ahead_base = __shfl_sync(0xffffffffu, b, 0);
        ahead_left = c;
      }
      w = ahead_base + (unsigned long long)(c - ahead_left);
      --ahead_left;
    } else {
      w = claim_item(claimer, p);
    }
    WsUnit u = ws_decode<kWin, kPack>(sm.sched, p, w);
    const int slot = it_cnt & 1;
    if (kPack && u.valid && u.packed) {
      // packed tiles: the row tables go with the unit (the slot is free once its
      // previous unit was read)
      if (lane == 0 && it_cnt >= 2) ok = WS_WAIT(&sm.item_empty[slot], ((it_cnt >> 1) - 1) & 1);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (ok) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const long long key = (long long)sm.sched.chunk_base * 1024 + (u.g[t] + 1);
          // registers, not an indexed array: slot is 0 or 1
          const long long held = slot ? rows_of[2 + t] : rows_of[t];
          if (key != held) {
            ws_fill_rows(sm.rows[slot][t], sm.sched, u.g[t], lane);
            if (slot) rows_of[2 + t] = key; else rows_of[t] = key;
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        if (!ok) u.valid = 0;
        sm.items[slot] = u;
        mbar_arrive(&sm.item_full[slot]);
      }
    } else if (lane == 0) {
      if (it_cnt >= 2) ok = WS_WAIT(&sm.item_empty[slot], ((it_cnt >> 1) - 1) & 1);
      if (!ok) u.valid = 0;
      sm.items[slot] = u;
      mbar_arrive(&sm.item_full[slot]);
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    ++it_cnt;
    if (!u.valid || !ok) break;
    if (kPack) {
      // the packing instantiation (many short units): the whole warp walks the loads, its
      // waits and counters warp-uniform, and lane 0 arms the barriers and issues the
      // predicated copies
      if (u.n_all > 0) {
        const bool issue = lane == 0;
        const int qs = q_cnt % kQSlots;
        if (q_cnt >= (uint32_t)kQSlots) ok = WS_WAIT_WARP(&sm.q_empty[qs], ((q_cnt / kQSlots) - 1) & 1);
        if (ok) {
          const int ntiles = (u.t[0].n > 0 ? 1 : 0) + (u.t[1].n > 0 ? 1 : 0);
          if (issue) mbar_arrive_expect_tx(&sm.q_full[qs], ntiles * kTileBytes);
          for (int t = 0; t < 2; ++t) {
            if (u.t[t].n == 0) continue;   // no S MMA reads this tile
#pragma unroll
            for (int pn = 0; pn < kPanels; ++pn)
              tma_load_2d_if(issue, sm.q[qs][t] + pn * 16384, tm_q, &sm.q_full[qs], u.t[t].h * p.d + pn * 64,
                             u.t[t].seq.q_start + u.t[t].q0);
          }
          ++q_cnt;
        }
        for (int li = 0; ok && li < u.n_all; ++li) {
          const int tsel = (u.paired && !(li == 0 && u.t[0].n > 0)) ? 1 : 0;
          const int row = (tsel ? u.t[1].seq.kv_start : u.t[0].seq.kv_start) + (u.paired ? 0 : (u.jb + li) * kBlockN);
          const int kvh = (tsel ? u.t[1].h : u.t[0].h) / p.group;
          const int st = kv_cnt % kWsStages;
          const uint32_t reuse = ((kv_cnt / kWsStages) - 1) & 1;
          if (kv_cnt >= (uint32_t)kWsStages) ok = WS_WAIT_WARP(&sm.k_empty[st], reuse);
          if (!ok) break;
          if (issue) mbar_arrive_expect_tx(&sm.k_full[st], kTileBytes);
#pragma unroll
          for (int pn = 0; pn < kPanels; ++pn)
            tma_load_2d_if(issue, sm.k[st] + pn * 16384, tm_k, &sm.k_full[st], kvh * p.d + pn * 64, row);
          if (kv_cnt >= (uint32_t)kWsStages) ok = WS_WAIT_WARP(&sm.v_empty[st], reuse);
          if (!ok) {   // the K copy just issued lands before the CTA can exit
            drain_wait(&sm.k_full[st], (kv_cnt / kWsStages) & 1);
            break;
          }
          if (issue) mbar_arrive_expect_tx(&sm.v_full[st], kTileBytes);
#pragma unroll
          for (int pn = 0; pn < kPanels; ++pn)
            tma_load_2d_if(issue, sm.v[st] + pn * 16384, tm_v, &sm.v_full[st], kvh * p.d + pn * 64, row);
          ++kv_cnt;
        }
      }
    } else if (lane == 0 && u.n_all > 0) {
      const int qs = q_cnt % kQSlots;
      if (q_cnt >= (uint32_t)kQSlots) ok = WS_WAIT(&sm.q_empty[qs], ((q_cnt / kQSlots) - 1) & 1);
      if (ok) {
        const int ntiles = (u.t[0].n > 0 ? 1 : 0) + (u.t[1].n > 0 ? 1 : 0);
        mbar_arrive_expect_tx(&sm.q_full[qs], ntiles * kTileBytes);
        for (int t = 0; t < 2; ++t) {
          if (u.t[t].n == 0) continue;   // no S MMA reads this tile
#pragma unroll
          for (int pn = 0; pn < kPanels; ++pn)
            tma_load_2d(sm.q[qs][t] + pn * 16384, tm_q, &sm.q_full[qs], u.t[t].h * p.d + pn * 64,
                        u.t[t].seq.q_start + u.t[t].q0);
        }
        ++q_cnt;
      }
      // K/V tiles in the order the MMA warp consumes them: KV tiles 0.. of the
      // sequence (shared), or tile 0's then tile 1's own tile (paired)
      for (int li = 0; ok && li < u.n_all; ++li) {
        const int tsel = (u.paired && !(li == 0 && u.t[0].n > 0)) ? 1 : 0;
        const int row = u.t[tsel].seq.kv_start + (u.paired ? 0 : (u.jb + li) * kBlockN);
        const int kvh = u.t[tsel].h / p.group;
        const int st = kv_cnt % kWsStages;
        const uint32_t reuse = ((kv_cnt / kWsStages) - 1) & 1;
        if (kv_cnt >= (uint32_t)kWsStages) ok = WS_WAIT(&sm.k_empty[st], reuse);
        if (!ok) break;
        mbar_arrive_expect_tx(&sm.k_full[st], kTileBytes);
#pragma unroll
        for (int pn = 0; pn < kPanels; ++pn)
          tma_load_2d(sm.k[st] + pn * 16384, tm_k, &sm.k_full[st], kvh * p.d + pn * 64, row);
        if (kv_cnt >= (uint32_t)kWsStages) ok = WS_WAIT(&sm.v_empty[st], reuse);
        if (!ok) {   // the K copy just issued lands before the CTA can exit
          drain_wait(&sm.k_full[st], (kv_cnt / kWsStages) & 1);
          break;
        }
        mbar_arrive_expect_tx(&sm.v_full[st], kTileBytes);
#pragma unroll
        for (int pn = 0; pn < kPanels; ++pn)
          tma_load_2d(sm.v[st] + pn * 16384, tm_v, &sm.v_full[st], kvh * p.d + pn * 64, row);
        ++kv_cnt;
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (!ok) break;
  }
  // copies still in flight land before the CTA can exit: every Q and K/V load
  // counted in q_cnt / kv_cnt (the last kQSlots / kWsStages of them may still be
  // pending; earlier ones were consumed), and a K copy whose V partner was not
  // issued was drained above
  if (lane == 0) {
    for (uint32_t c = (q_cnt > (uint32_t)kQSlots ? q_cnt - kQSlots : 0); c < q_cnt; ++c)
      drain_wait(&sm.q_full[c % kQSlots], (c / kQSlots) & 1);
    for (uint32_t c = (kv_cnt > (uint32_t)kWsStages ? kv_cnt - kWsStages : 0); c < kv_cnt; ++c) {
      drain_wait(&sm.k_full[c % kWsStages], (c / kWsStages) & 1);
      drain_wait(&sm.v_full[c % kWsStages], (c / kWsStages) & 1);
    }
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// warp 1 (one thread): MMA issuer
// ---------------------------------------------------------------------------
template <typename DT, int DP, bool kWin>
__device__ void ws_mma(WsSmem<DP>& sm, const AttnParams& p, uint32_t tmem, volatile uint32_t* abort_flag) {
  using Tr = DTypeTraits<DT>;
  constexpr uint32_t idesc_qk = umma_idesc_f16(Tr::kBF16, kTileM, kBlockN, false);
  constexpr uint32_t idesc_pv = umma_idesc_f16(Tr::kBF16, kTileM, DP, true);
  const uint32_t tS[2] = {tmem, tmem + 128};
  const uint32_t tO[2] = {tmem + 256, tmem + 256 + DP};
  // low descriptor words; consecutive tiles / stages are kTileBytes apart
  constexpr int kQSlots = WsSmem<DP>::kQSlots, kWsStages = WsSmem<DP>::kStages;
  constexpr uint32_t kStep = WsSmem<DP>::kTileBytes >> 4;
  const uint32_t q_lo00 = smem_desc_sw128_lo(smem_u32(sm.q[0][0]), 16);
  const uint32_t k_lo0 = smem_desc_sw128_lo(smem_u32(sm.k[0]), 16);
  const uint32_t v_lo0 = smem_desc_sw128_lo(smem_u32(sm.v[0]), 16384);
  uint32_t it_cnt = 0, q_cnt = 0, kv_cnt = 0, p_cnt[2] = {0, 0};
  // the lane that issues every MMA and commit (a commit tracks its own thread's MMAs)
  const bool leader = elect_one_sync();

  auto fetch = [&](MmaUnit& x) -> bool {
    const int slot = it_cnt & 1;
    if (!WS_WAIT_WARP(&sm.item_full[slot], (it_cnt >> 1) & 1)) return false;
    const WsUnit& w = sm.items[slot];
    x.valid = w.valid;
    x.paired = w.paired;
    x.jb = kWin ? w.jb : 0;
    x.n_all = w.n_all;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      x.j0[t] = kWin ? w.t[t].j0 : 0;
      x.n[t] = w.t[t].n;
    }
    __syncwarp();   // every lane has read the unit before the slot is released
    if (leader) mbar_arrive(&sm.item_empty[slot]);
    ++it_cnt;
    return true;
  };
  // Paired unit: S_t = Q_t K_t^T on tile t's own K stage (kv_base: the unit's
  // first K/V load); the K stage is released once the MMA completes.
  auto pair_s = [&](const MmaUnit& x, int t, uint32_t q_lo0, uint32_t kv_base) -> bool {
    const uint32_t c = kv_base + ((t == 1 && x.n[0] > 0) ? 1u : 0u);
    const int st = c % kWsStages;
    if (!WS_WAIT_WARP(&sm.k_full[st], (c / kWsStages) & 1)) return false;
    tc_fence_after();
    issue_qk<DP>(leader, tS[t], q_lo0 + t * kStep, k_lo0 + st * kStep, idesc_qk);
    umma_commit_if(leader, &sm.s_full[t]);
    umma_commit_if(leader, &sm.k_empty[st]);
    return true;
  };

  MmaUnit u;
  bool s_issued = false;   // S MMAs of the paired unit u already issued (ahead of u)
  if (!fetch(u)) u.valid = 0;
  while (u.valid) {
    if (u.n_all == 0) {
      if (!fetch(u)) break;
      s_issued = false;
      continue;
    }
    if (!u.paired) {
      // ---- one long-sequence block: both tiles share every K/V tile ----
      // KV tiles jb .. jb + n - 1 are ring positions kv_cnt ..; tile t visits [j0_t, n_t).
      const int n = u.n_all, jb = u.jb;
      const int qs = q_cnt % kQSlots;
      if (!WS_WAIT_WARP(&sm.q_full[qs], (q_cnt / kQSlots) & 1)) break;
      ++q_cnt;
      const uint32_t q_lo0 = q_lo00 + qs * 2 * kStep;   // this slot's tile 0
      if (!WS_WAIT_WARP(&sm.k_full[kv_cnt % kWsStages], (kv_cnt / kWsStages) & 1)) break;
      tc_fence_after();
      {
        const uint32_t ks = k_lo0 + (kv_cnt % kWsStages) * kStep;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (u.n[t] > 0 && u.j0[t] == jb) {
            issue_qk<DP>(leader, tS[t], q_lo0 + t * kStep, ks, idesc_qk);
            umma_commit_if(leader, &sm.s_full[t]);
          }
        }
        umma_commit_if(leader, &sm.k_empty[kv_cnt % kWsStages]);
        if (n == 1) umma_commit_if(leader, &sm.q_empty[qs]);
      }
      bool ok = true;
      for (int i = 0; i < n && ok; ++i) {
        const int j = jb + i;
        const uint32_t c = kv_cnt + i, cn = c + 1;
        const int st = c % kWsStages, stn = cn % kWsStages;
        if (!WS_WAIT_WARP(&sm.v_full[st], (c / kWsStages) & 1)) { ok = false; break; }
        const uint32_t vs = v_lo0 + st * kStep;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (j >= u.j0[t] && j < u.n[t]) {
            const uint32_t par = p_cnt[t] & 1;
            ++p_cnt[t];
            if (!WS_WAIT_WARP(&sm.p_lo[t], par)) { ok = false; break; }
            tc_fence_after();
            issue_pv<0, 4>(leader, tO[t], tS[t], vs, idesc_pv, j > u.j0[t]);
            if (!WS_WAIT_WARP(&sm.p_hi[t], par)) { ok = false; break; }
            tc_fence_after();
            issue_pv<4, 8>(leader, tO[t], tS[t], vs, idesc_pv, true);
            umma_commit_if(leader, &sm.o_full[t]);
          }
          if (j + 1 >= u.j0[t] && j + 1 < u.n[t]) {   // the tile's next S (or its first)
            if (!WS_WAIT_WARP(&sm.k_full[stn], (cn / kWsStages) & 1)) { ok = false; break; }
            tc_fence_after();
            issue_qk<DP>(leader, tS[t], q_lo0 + t * kStep, k_lo0 + stn * kStep, idesc_qk);
            umma_commit_if(leader, &sm.s_full[t]);
          }
        }
        if (i + 1 < n) umma_commit_if(leader, &sm.k_empty[stn]);   // every S MMA on K stage stn issued
        if (i == n - 2) umma_commit_if(leader, &sm.q_empty[qs]);    // last S MMAs of the item issued
        umma_commit_if(leader, &sm.v_empty[st]);
      }
      kv_cnt += n;
      if (!ok) break;
      if (!fetch(u)) break;
      s_issued = false;
      continue;
    }

    // ---- paired unit: two independent tiles, one K/V tile each ----
    bool ok = true;
    if (!s_issued) {
      const int qs = q_cnt % kQSlots;
      if (!WS_WAIT_WARP(&sm.q_full[qs], (q_cnt / kQSlots) & 1)) break;
      ++q_cnt;
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if (ok && u.n[t] > 0) ok = pair_s(u, t, q_lo00 + qs * 2 * kStep, kv_cnt);
      if (!ok) break;
      umma_commit_if(leader, &sm.q_empty[qs]);
    }
    // the next unit, if paired, gets its S_t issued right after this unit's P_t V
    MmaUnit nx;
    if (!fetch(nx)) break;
    const bool ahead = nx.valid && nx.paired && nx.n_all > 0;
    const uint32_t kv_next = kv_cnt + u.n_all;
    const int qs_nx = q_cnt % kQSlots;
    const uint32_t q_par_nx = (q_cnt / kQSlots) & 1;
    if (ahead) ++q_cnt;
    bool q_nx_ready = !ahead;   // nx's Q tiles landed
    // The two tiles move through P V (two halves) and then nx's S MMA in the
    // order their inputs become ready, so a tile whose softmax finished first
    // waits neither for the other tile nor for loads queued behind it.
    int state[2];          // 1: first P V half pending, 2: second half, 3: S of nx, 0: done
    int st[2], st_nx[2];
    uint32_t par[2], vpar[2], kpar_nx[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const bool s_next = ahead && nx.n[t] > 0;
      state[t] = u.n[t] > 0 ? 1 : (s_next ? 3 : 0);
      const uint32_t c = kv_cnt + ((t == 1 && u.n[0] > 0) ? 1u : 0u);
      st[t] = c % kWsStages;
      vpar[t] = (c / kWsStages) & 1;
      par[t] = p_cnt[t] & 1;
      if (u.n[t] > 0) ++p_cnt[t];
      const uint32_t cn = kv_next + ((t == 1 && nx.n[0] > 0) ? 1u : 0u);
      st_nx[t] = cn % kWsStages;
      kpar_nx[t] = (cn / kWsStages) & 1;
    }
    uint32_t idle = 0;
    uint64_t idle_t0 = 0;
    while (ok && (state[0] | state[1])) {
      bool progressed = false;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (state[t] == 1 && warp_test_wait(&sm.p_lo[t], par[t]) && warp_test_wait(&sm.v_full[st[t]], vpar[t])) {
          tc_fence_after();
          issue_pv<0, 4>(leader, tO[t], tS[t], v_lo0 + st[t] * kStep, idesc_pv, false);
          state[t] = 2;
          progressed = true;
        }
        if (state[t] == 2 && warp_test_wait(&sm.p_hi[t], par[t])) {
          tc_fence_after();
          issue_pv<4, 8>(leader, tO[t], tS[t], v_lo0 + st[t] * kStep, idesc_pv, true);
          umma_commit_if(leader, &sm.o_full[t]);
          umma_commit_if(leader, &sm.v_empty[st[t]]);
          state[t] = (ahead && nx.n[t] > 0) ? 3 : 0;
          progressed = true;
        }
        if (state[t] == 3) {
          if (!q_nx_ready) q_nx_ready = warp_test_wait(&sm.q_full[qs_nx], q_par_nx);
          if (q_nx_ready && warp_test_wait(&sm.k_full[st_nx[t]], kpar_nx[t])) {
            tc_fence_after();
            issue_qk<DP>(leader, tS[t], q_lo00 + qs_nx * 2 * kStep + t * kStep, k_lo0 + st_nx[t] * kStep, idesc_qk);
            umma_commit_if(leader, &sm.s_full[t]);
            umma_commit_if(leader, &sm.k_empty[st_nx[t]]);
            state[t] = 0;
            progressed = true;
          }
        }
      }
      if (progressed) {
        idle = 0;
        idle_t0 = 0;
      } else if ((++idle & 255u) == 0) {   // bounded polling, like the other waits
        // lane 0's view, so that the warp decides together
        if (__shfl_sync(0xffffffffu, *abort_flag != 0u ? 1 : 0, 0) != 0) { ok = false; break; }
        const uint64_t t = globaltimer_ns();
        const uint64_t now = ((uint64_t)__shfl_sync(0xffffffffu, (uint32_t)(t >> 32), 0) << 32) |
                             __shfl_sync(0xffffffffu, (uint32_t)t, 0);
        if (idle_t0 == 0) {
          idle_t0 = now;
        } else if (now - idle_t0 > p.wait_limit_ns) {
          if (leader) {
            *abort_flag = 1u;
            atomicOr(p.status, THD_WAIT_TIMEOUT_BIT);
          }
          ok = false;
        }
      }
    }
    if (!ok) break;
    if (ahead) umma_commit_if(leader, &sm.q_empty[qs_nx]);
    kv_cnt = kv_next;
    u = nx;
    s_issued = ahead;
  }
  // every MMA issued so far completes before TMEM is released
  umma_commit_if(leader, &sm.drain);
  drain_wait(&sm.drain, 0);
}

// P for 32 keys of one row: exp2(S * scale_log2 - mb), rounded to the input
// type and packed in pairs, with the rounded and the exact running sums (two
// accumulator pairs each, alternating, for two independent add chains).
template <typename DT>
__device__ __forceinline__ void ws_exp_chunk(const uint32_t* sr, uint32_t* pk, float2 scale2, float2 bias2, float2& lr_a,
                                             float2& lr_b, float2& le_a, float2& le_b) {
  using Tr = DTypeTraits<DT>;
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const float2 arg =
        __ffma2_rn(make_float2(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])), scale2, bias2);
    const float x0 = ex2_approx(arg.x);
    const float x1 = ex2_approx(arg.y);
    pk[e] = Tr::pack2(x0, x1);
    if (e & 1) {
      le_b = __fadd2_rn(le_b, make_float2(x0, x1));
      Tr::acc2(pk[e], lr_b.x, lr_b.y);
    } else {
      le_a = __fadd2_rn(le_a, make_float2(x0, x1));
      Tr::acc2(pk[e], lr_a.x, lr_a.y);
    }
  }
}

// Softmax of one KV tile for one row (the calling thread's TMEM lane): S from
// TMEM, online max / sums, P (rounded to the input type) back over S in two
// halves of 64 keys, lazy O rescale.  `partial` (warp-uniform): some row of
// the warp may not see all 128 keys; columns outside the row's visible keys
// are masked, and when no row of the warp sees a key in the second half, its
// exponentials are skipped and zero P is stored there.  j: position of the KV
// tile among the tiles this Q tile visits (row_first / row_last are counted
// from the first of them).  Returns false when a wait gave up.
// row_first / row_last: the row's first and last visible key (row_last < 0 for
// rows past the sequence); kWin: a window may bound the keys from below.
template <typename DT, int DP, bool kWin>
__device__ __forceinline__ bool ws_softmax_tile(WsSmem<DP>& sm, const AttnParams& p, volatile uint32_t* abort_flag,
                                                uint32_t tS, uint32_t tO, int tile, int j, uint32_t o_cnt,
                                                bool partial, int row_first, int row_last, float sl2,
                                                float& m_run, float2& lr_a, float2& lr_b, float2& le_a, float2& le_b) {
  const int lane = threadIdx.x & 31;
  const int kv0 = j * kBlockN;
  uint32_t sr[128];
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, sr + 32 * c);
  tmem_ld_wait_regs32(sr);
  tmem_tie_regs32(sr + 32);
  tmem_tie_regs32(sr + 64);
  tmem_tie_regs32(sr + 96);
  if (partial) {
    const int lim = row_last - kv0;
    if constexpr (kWin) {   // sliding window: keys before the row's window too
      const int lo = row_first - kv0;
#pragma unroll
      for (int c = 0; c < 128; ++c)
        if (c > lim || c < lo) sr[c] = __float_as_uint(-INFINITY);
    } else {
#pragma unroll
      for (int c = 0; c < 128; ++c)
        if (c > lim) sr[c] = __float_as_uint(-INFINITY);
    }
  }
  // row max: three-input max, four independent chains
  float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
  for (int c = 0; c < 128; c += 8) {
    mx0 = fmax3f(mx0, __uint_as_float(sr[c + 0]), __uint_as_float(sr[c + 1]));
    mx1 = fmax3f(mx1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
    mx2 = fmax3f(mx2, __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
    mx3 = fmax3f(mx3, __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
  }
  const float m_tile = fmax3f(fmaxf(mx0, mx1), mx2, mx3);
  const float m_new = fmaxf(m_run, m_tile);
  const bool need = (m_new - m_run) * sl2 > kRescaleThreshold;   // false while both are -inf
  float alpha = 1.f;
  if (need) {
    alpha = ex2_approx((m_run - m_new) * sl2);
    m_run = m_new;
    const float2 a2 = make_float2(alpha, alpha);
    lr_a = __fmul2_rn(lr_a, a2);
    lr_b = __fmul2_rn(lr_b, a2);
    le_a = __fmul2_rn(le_a, a2);
    le_b = __fmul2_rn(le_b, a2);
  }
  const float mb = (m_run == -INFINITY ? 0.f : m_run) * sl2;
  const float2 scale2 = make_float2(sl2, sl2);
  const float2 bias2 = make_float2(-mb, -mb);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    if (partial && half == 1 &&
        __all_sync(0xffffffffu, row_last - kv0 < 2 * 32)) {
      // no row of the warp sees keys 64..127: their P is zero
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) pk[e] = 0u;
      tmem_st16(tS + 32, pk);
      tmem_st16(tS + 48, pk);
    } else {
#pragma unroll
      for (int c = 2 * half; c < 2 * half + 2; ++c) {
        uint32_t pk[16];
        ws_exp_chunk<DT>(sr + 32 * c, pk, scale2, bias2, lr_a, lr_b, le_a, le_b);
        tmem_st16(tS + 16 * c, pk);
      }
    }
    if (half == 0 && j > 0 && __any_sync(0xffffffffu, need)) {
      // O_t must hold the previous P V product before it is rescaled, and the
      // rescaled O must be in TMEM before this tile's first P V step
      if (!WS_WAIT_WARP(&sm.o_full[tile], (o_cnt + j - 1) & 1)) {
        tmem_st_wait();   // the P stores above complete before TMEM can be released
        return false;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < DP / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * c, o);
        tmem_ld_wait_regs32(o);
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
        tmem_st32(tO + 32 * c, o);
      }
    }
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(half == 0 ? &sm.p_lo[tile] : &sm.p_hi[tile]);
  }
  return true;
}

// One packed tile (a group of short sequences, one KV tile): S from TMEM, each
// row masked to its band [first, last] from the row table, softmax over the one
// tile (the same arithmetic as a sequence's first KV tile), P back over S in two
// halves of 64 keys, then the epilogue.  Rows of no sequence of the group
// (first = kRowAbsent) write nothing.  Returns false when a wait gave up.
template <typename DT, int DP>
__device__ __forceinline__ bool ws_packed_tile(WsSmem<DP>& sm, const AttnParams& p, volatile uint32_t* abort_flag,
                                               uint32_t tS, uint32_t tO, int tile, const WsTile& tt, uint32_t rk,
                                               int row, float sl2, uint32_t& s_cnt, uint32_t& o_cnt) {
  using Tr = DTypeTraits<DT>;
  const int lane = threadIdx.x & 31;
  const int first_raw = (int)(int16_t)(rk & 0xFFFFu);
  const bool row_ok = first_raw != kRowAbsent;
  const int first = row_ok ? first_raw : 0;
  const int last = (int)(int16_t)(rk >> 16);   // < first when the row sees no key
  float m = -INFINITY;
  float2 lr_a = make_float2(0.f, 0.f), lr_b = lr_a, le_a = lr_a, le_b = lr_a;
  if (tt.n > 0) {
    if (!WS_WAIT_WARP(&sm.s_full[tile], s_cnt & 1)) return false;
    ++s_cnt;
    tc_fence_after();
    uint32_t sr[128];
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, sr + 32 * c);
    tmem_ld_wait_regs32(sr);
    tmem_tie_regs32(sr + 32);
    tmem_tie_regs32(sr + 64);
    tmem_tie_regs32(sr + 96);
#pragma unroll
    for (int c = 0; c < 128; ++c)
      if (c > last || c < first) sr[c] = __float_as_uint(-INFINITY);
    float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
    for (int c = 0; c < 128; c += 8) {
      mx0 = fmax3f(mx0, __uint_as_float(sr[c + 0]), __uint_as_float(sr[c + 1]));
      mx1 = fmax3f(mx1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
      mx2 = fmax3f(mx2, __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
      mx3 = fmax3f(mx3, __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
    }
    m = fmax3f(fmaxf(mx0, mx1), mx2, mx3);
    const float mb = (m == -INFINITY ? 0.f : m) * sl2;
    const float2 scale2 = make_float2(sl2, sl2);
    const float2 bias2 = make_float2(-mb, -mb);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      if (half == 1 && __all_sync(0xffffffffu, last < 64)) {
        // no row of the warp sees keys 64..127: their P is zero
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = 0u;
        tmem_st16(tS + 32, pk);
        tmem_st16(tS + 48, pk);
      } else {
#pragma unroll
        for (int c = 2 * half; c < 2 * half + 2; ++c) {
          uint32_t pk[16];
          ws_exp_chunk<DT>(sr + 32 * c, pk, scale2, bias2, lr_a, lr_b, le_a, le_b);
          tmem_st16(tS + 16 * c, pk);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(half == 0 ? &sm.p_lo[tile] : &sm.p_hi[tile]);
    }
    ++o_cnt;
  }
  // ---- epilogue ----
  const SeqInfo& s = tt.seq;   // q_start: the group's first row
  DT* dst = static_cast<DT*>(p.out) + ((size_t)(s.q_start + (row_ok ? row : 0)) * p.Hq + tt.h) * (size_t)p.d;
  if (tt.n > 0) {
    if (!WS_WAIT_WARP(&sm.o_full[tile], (o_cnt - 1) & 1)) return false;
    tc_fence_after();
    const float l_r = (lr_a.x + lr_a.y) + (lr_b.x + lr_b.y);
    const float l_e = (le_a.x + le_a.y) + (le_b.x + le_b.y);
    const float inv = l_r > 0.f ? 1.f / l_r : 0.f;   // a row that saw no key stays 0
#pragma unroll
    for (int c = 0; c < DP / 32; ++c) {
      uint32_t o[32];
      tmem_ld32(tO + 32 * c, o);
      tmem_ld_wait_regs32(o);
      if (row_ok) {
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint4 v4;
          v4.x = Tr::pack2(__uint_as_float(o[e + 0]) * inv, __uint_as_float(o[e + 1]) * inv);
          v4.y = Tr::pack2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
          v4.z = Tr::pack2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
          v4.w = Tr::pack2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
          *reinterpret_cast<uint4*>(dst + 32 * c + e) = v4;
        }
      }
    }
    if (row_ok && p.lse) p.lse[(size_t)tt.h * p.T + s.q_start + row] = m * p.scale + logf(l_e);
  } else if (row_ok) {
#pragma unroll
    for (int col = 0; col < DP; col += 8) *reinterpret_cast<uint4*>(dst + col) = make_uint4(0u, 0u, 0u, 0u);
    if (p.lse) p.lse[(size_t)tt.h * p.T + s.q_start + row] = -INFINITY;
  }
  tc_fence_before();
  return true;
}

// ---------------------------------------------------------------------------
// warps 4-11: softmax + epilogue, tile = warp / 4 - 1
// ---------------------------------------------------------------------------
template <typename DT, int DP, bool kWin, bool kPack>
__device__ void ws_softmax(WsSmem<DP>& sm, const AttnParams& p, uint32_t tmem, int tile,
                           volatile uint32_t* abort_flag) {
  using Tr = DTypeTraits<DT>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row = 32 * (warp & 3) + lane;           // TMEM lane = row of the Q tile
  const uint32_t t_lane = (uint32_t)(32 * (warp & 3)) << 16;
  const uint32_t tS = tmem + 128 * tile + t_lane;
  const uint32_t tO = tmem + 256 + DP * tile + t_lane;
  const float sl2 = p.scale_log2;
  uint32_t it_cnt = 0, s_cnt = 0, o_cnt = 0;

  for (;;) {
    const int slot = it_cnt & 1;
    if (!WS_WAIT_WARP(&sm.item_full[slot], (it_cnt >> 1) & 1)) break;
    const int valid = sm.items[slot].valid;
    if (kPack && valid && sm.items[slot].packed) {   // a packed tile: its own path
      const WsTile tp = sm.items[slot].t[tile];
      const uint32_t rk = sm.rows[slot][tile][row];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.item_empty[slot]);
      ++it_cnt;
      if (!ws_packed_tile<DT, DP>(sm, p, abort_flag, tS, tO, tile, tp, rk, row, sl2, s_cnt, o_cnt)) break;
      continue;
    }
    const WsTile tt = sm.items[slot].t[tile];
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.item_empty[slot]);
    ++it_cnt;
    if (!valid) break;
    const SeqInfo& s = tt.seq;
    const int ni = tt.n;
    const int qt0 = tt.q0;                            // first query position of this tile
    const int rows = s.q_len - qt0;                   // valid rows of the tile (may exceed 128)
    const int qpos = qt0 + row;

    float m_run = -INFINITY;
    float2 lr_a = make_float2(0.f, 0.f), lr_b = lr_a;   // rounded-P sums (normalise O)
    float2 le_a = lr_a, le_b = lr_a;                     // exact sums (LSE)
    bool ok = true;
    // the row's visible keys (none for rows past the sequence), counted from the
    // first KV tile the Q tile visits; the loop runs over the nv tiles it visits
    const int base = kWin ? tt.j0 * kBlockN : 0;
    const int row_last = row < rows ? seq_last_key(s, qpos) - base : -1;
    const int row_first = kWin ? seq_first_key(s, qpos) - base : 0;
    const int tile_last = seq_last_key(s, qt0) - base;   // smallest last key of the tile's rows
    const int nv = ni - (kWin ? tt.j0 : 0);
    for (int j = 0; j < nv; ++j) {
      if (!WS_WAIT_WARP(&sm.s_full[tile], s_cnt & 1)) { ok = false; break; }
      ++s_cnt;
      tc_fence_after();
      // partial tile: a row's visible keys end (sequence end, causal diagonal,
      // window) inside it, or (window) start inside it for a row of this warp
      const int kv0 = j * kBlockN;
      const bool masked = kv0 + kBlockN - 1 > tile_last || (kWin && __any_sync(0xffffffffu, row_first > kv0));
      ok = ws_softmax_tile<DT, DP, kWin>(sm, p, abort_flag, tS, tO, tile, j, o_cnt, masked, row_first, row_last, sl2,
                                         m_run, lr_a, lr_b, le_a, le_b);
      if (!ok) break;
    }
    if (!ok) break;
    o_cnt += nv;

    // ---- epilogue ----
    const bool row_ok = row < rows;
    DT* dst = static_cast<DT*>(p.out) + ((size_t)(s.q_start + (row_ok ? qpos : 0)) * p.Hq + tt.h) * (size_t)p.d;
    if (ni > 0) {
      if (!WS_WAIT_WARP(&sm.o_full[tile], (o_cnt - 1) & 1)) break;
      tc_fence_after();
      const float l_r = (lr_a.x + lr_a.y) + (lr_b.x + lr_b.y);
      const float l_e = (le_a.x + le_a.y) + (le_b.x + le_b.y);
      const float inv = l_r > 0.f ? 1.f / l_r : 0.f;   // a row that saw no key stays 0
#pragma unroll
      for (int c = 0; c < DP / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * c, o);
        tmem_ld_wait_regs32(o);
        if (row_ok) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 v4;
            v4.x = Tr::pack2(__uint_as_float(o[e + 0]) * inv, __uint_as_float(o[e + 1]) * inv);
            v4.y = Tr::pack2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
            v4.z = Tr::pack2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
            v4.w = Tr::pack2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
            *reinterpret_cast<uint4*>(dst + 32 * c + e) = v4;
          }
        }
      }
      if (row_ok && p.lse) p.lse[(size_t)tt.h * p.T + s.q_start + qpos] = m_run * p.scale + logf(l_e);
    } else if (row_ok) {
#pragma unroll
      for (int col = 0; col < DP; col += 8) *reinterpret_cast<uint4*>(dst + col) = make_uint4(0u, 0u, 0u, 0u);
      if (p.lse) p.lse[(size_t)tt.h * p.T + s.q_start + qpos] = -INFINITY;
    }
    tc_fence_before();
  }
}

template <typename DT, int DP, bool kWin, bool kPack>
__global__ void __launch_bounds__(kWsThreads, 1)
    attn_fwd_ws_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  static_assert(!(kWin && kPack), "short sequences are packed only without a window");
  extern __shared__ uint8_t smem_raw[];
  WsSmem<DP>& sm = *reinterpret_cast<WsSmem<DP>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < WsSmem<DP>::kQSlots; ++s) {
      mbar_init(&sm.q_full[s], 1);
      mbar_init(&sm.q_empty[s], 1);
    }
    for (int s = 0; s < WsSmem<DP>::kStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
      mbar_init(&sm.v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm.s_full[t], 1);
      mbar_init(&sm.p_lo[t], 4);   // one lane of each softmax warp
      mbar_init(&sm.p_hi[t], 4);
      mbar_init(&sm.o_full[t], 1);
      mbar_init(&sm.item_full[t], 1);
      mbar_init(&sm.item_empty[t], 9);   // MMA thread + one lane of each softmax warp
    }
    mbar_init(&sm.drain, 1);
    fence_mbar_init();
    sm.abort = 0;
    sched_init(sm.sched);
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 0) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile uint32_t* abort_flag = &sm.abort;

  if (warp < 4) {
    setmaxnreg_dec<kRegsCtl>();
    if (warp == 0) {
      ws_producer<DP, kWin, kPack>(sm, p, &tm_q, &tm_k, &tm_v, abort_flag);
    } else if (warp == 1) {
      ws_mma<DT, DP, kWin>(sm, p, tmem, abort_flag);
    } else {
      zero_pad_rows(p, 64, 64, 2);
      // test setting: a wait that runs out while the pipeline runs (the drain barrier
      // completes only when the MMA warp's last MMAs have, at the CTA's end)
      if (warp == 3 && p.inject_wait) inject_wait_timeout_warp(p, &sm.drain, abort_flag);
    }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    ws_softmax<DT, DP, kWin, kPack>(sm, p, tmem, (warp >> 2) - 1, abort_flag);
  }

  // Every role has drained its own asynchronous work: the producer its copies in
  // flight, the MMA thread its committed MMAs, the softmax warps their TMEM stores.
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

#undef WS_WAIT
#undef WS_WAIT_WARP

}  // namespace thd
