// attn_common.cuh — parameters, sequence metadata decoding, the in-kernel
// varlen tile scheduler and pad-row zeroing shared by the attention kernels.
//
// Semantics (web pages; titles and sections):
//  * "How to pad sequences that cannot be evenly split in context parallelism
//    (CP)?" (Megatron-LM issue, repro script): THD layout [t, h, d], sequence
//    boundaries from cu_seqlens.
//  * "Add per-sequence causal policy to packed THD attention"
//    (TransformerEngine PR, Changes; pad_between_seqs review comment): one
//    causal flag per sequence; cu_seqlens_padded gives each sequence's slot
//    start, the rows of a slot past its valid length are padding, and padding
//    rows of the output are zero.
//  * "[PyTorch] Build the attention padding mask without host syncs"
//    (TransformerEngine PR, Changes): metadata buffers may be longer than
//    batch_size + 1; only the first batch_size + 1 entries are read.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace thd {

constexpr int kBlockN = 128;            // keys per KV tile
constexpr int kTileM = 128;             // query rows per Q tile (UMMA M)
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // default limit of one pipeline wait: 2 s
constexpr uint32_t THD_WAIT_TIMEOUT_BIT = 1u;     // device status bit of a timed-out wait

struct AttnParams {
  const void* q;
  const void* k;
  const void* v;
  const int32_t* cu_q;
  const int32_t* cu_kv;
  const int32_t* pad_q;    // may be null
  const int32_t* pad_kv;   // may be null
  const uint8_t* causal;   // may be null
  void* out;
  float* lse;              // may be null
  unsigned long long* work_counter;
  uint32_t* status;
  uint64_t wait_limit_ns;  // a pipeline wait gives up (status bit, CTA abort) after this long
  uint32_t wait_check_mask;  // a waiting thread reads the clock when (polls & mask) == 0
  uint32_t inject_wait;    // test setting: each CTA makes one wait that runs out (inject_wait_timeout)
  int claim;               // work items taken per atomic on the counter (>= 1)
  int win_left, win_right; // sliding window (keys before / after the diagonal), -1 = unbounded
  int B, T, Hq, Hkv, d, group;
  float scale;             // softmax scale
  float scale_log2;        // softmax scale * log2(e)
};

// Per-sequence mask type codes (the padding / padding_causal /
// padding_causal_bottom_right types of the per-sequence policy review): 0 =
// every valid key visible, 2 = bottom-right causal (key j visible to query i
// iff j <= i + kv_len - q_len), any other non-zero code = top-left causal
// (j <= i), so a boolean per-sequence flag keeps its meaning.
constexpr int kMaskPadding = 0;
constexpr int kMaskCausalBottomRight = 2;

// No bound on that side of the sliding window.
constexpr int kNoBound = 1 << 30;

// Key j of a sequence is visible to its query i iff 0 <= j < kv_len and
//   i + shift - lo_off <= j <= i + shift + hi_off,
// shift being the diagonal of the mask type (kv_len - q_len bottom-right, else 0),
// hi_off = 0 for the causal types (else the window's right extent), lo_off the window's
// left extent; kNoBound where unbounded.  Without a window this is the prefix the mask
// type allows.
struct SeqInfo {
  int q_start, kv_start, q_len, kv_len, causal;
  int shift;
  int lo_off, hi_off;
};

__device__ __forceinline__ void set_visibility(SeqInfo& s, int code, const AttnParams& p) {
  s.causal = code != kMaskPadding;
  s.shift = code == kMaskCausalBottomRight ? s.kv_len - s.q_len : 0;
  const int wr = p.win_right >= 0 ? p.win_right : kNoBound;
  s.hi_off = s.causal ? 0 : wr;   // min(0, wr): a causal type never looks past the diagonal
  s.lo_off = p.win_left >= 0 ? p.win_left : kNoBound;
}

// First / last key of the sequence visible to query position qpos (the first is past the
// last when none is).  Both grow with qpos, so a block of rows sees keys between the first
// row's first key and the last row's last key.
__device__ __forceinline__ int seq_first_key(const SeqInfo& s, int qpos) {
  const long long f = (long long)qpos + s.shift - s.lo_off;
  return f < 0 ? 0 : (f > s.kv_len ? s.kv_len : (int)f);
}
__device__ __forceinline__ int seq_last_key(const SeqInfo& s, int qpos) {
  const long long l = (long long)qpos + s.shift + s.hi_off;
  return l > s.kv_len - 1 ? s.kv_len - 1 : (l < -1 ? -1 : (int)l);
}

// Test setting (p.inject_wait, off by default): one bounded wait on phase 0 of `bar`,
// a barrier that nothing completes before the CTA's own final drain, so the wait runs
// out after p.wait_limit_ns whatever the timing, sets the status bit and the CTA's
// abort flag, and the CTA leaves through its failure path with its copies and MMAs in
// flight.
__device__ __forceinline__ void inject_wait_timeout(const AttnParams& p, uint64_t* bar, volatile uint32_t* abort) {
  mbar_wait(bar, 0, abort, p.status, THD_WAIT_TIMEOUT_BIT, p.wait_limit_ns, p.wait_check_mask);
}
// The same by a whole warp, which leaves it together.
__device__ __forceinline__ bool inject_wait_timeout_warp(const AttnParams& p, uint64_t* bar, volatile uint32_t* abort) {
  return __all_sync(0xffffffffu, mbar_wait(bar, 0, abort, p.status, THD_WAIT_TIMEOUT_BIT, p.wait_limit_ns,
                                           p.wait_check_mask) ? 1 : 0) != 0;
}

// Sequence b's rows, clamped to the packed buffer [0, T): garbage metadata
// gives garbage output but never an out-of-range address.
__device__ __forceinline__ SeqInfo load_seq(const AttnParams& p, int b) {
  SeqInfo s;
  const long long cq0 = p.cu_q[b], cq1 = p.cu_q[b + 1];
  const long long ck0 = p.cu_kv[b], ck1 = p.cu_kv[b + 1];
  long long qs = p.pad_q ? (long long)p.pad_q[b] : cq0;
  long long ks = p.pad_kv ? (long long)p.pad_kv[b] : ck0;
  long long ql = cq1 - cq0, kl = ck1 - ck0;
  qs = qs < 0 ? 0 : (qs > p.T ? p.T : qs);
  ks = ks < 0 ? 0 : (ks > p.T ? p.T : ks);
  ql = ql < 0 ? 0 : (ql > p.T - qs ? p.T - qs : ql);
  kl = kl < 0 ? 0 : (kl > p.T - ks ? p.T - ks : kl);
  s.q_start = (int)qs;
  s.kv_start = (int)ks;
  s.q_len = (int)ql;
  s.kv_len = (int)kl;
  const int code = p.causal ? (int)p.causal[b] : kMaskPadding;
  set_visibility(s, code, p);
  return s;
}

// KV tiles a Q tile whose first row is sequence position q0 must visit: tiles
// [kv_first_tile, kv_tiles_for), up to the last key visible to the tile's last valid row
// and from the first key visible to its first row.  kv_tiles_for is 0 when no row sees a
// key; the range is empty when kv_first_tile >= kv_tiles_for.
__device__ __forceinline__ int kv_tiles_for(const SeqInfo& s, int q0, int rows) {
  if (s.kv_len <= 0) return 0;
  const int last = seq_last_key(s, min(q0 + rows, s.q_len) - 1);
  return last < 0 ? 0 : last / kBlockN + 1;
}
__device__ __forceinline__ int kv_first_tile(const SeqInfo& s, int q0) { return seq_first_key(s, q0) / kBlockN; }

// ----------------------------------------------------------------------------
// Tile scheduler.  Work item = (sequence, query head, block of BLOCK_M query
// rows).  Sequences are taken in chunks of kSchedChunk (in batch order); inside
// a chunk they are ordered longest first (counting sort on the number of KV
// tiles, full-context before causal at equal length), each sequence's items
// run head by head with its heaviest (last) query block first.  CTAs claim
// items from one global counter, so the order above is the order in which
// work starts (longest-processing-time-first list scheduling).  Pad gaps
// produce no items; fully masked causal tiles are never visited because each
// block only loops over kv_tiles_for() tiles.  Each CTA rebuilds the same
// chunk order in its shared memory from the device metadata, so no host
// synchronisation and no second launch are needed.
// ----------------------------------------------------------------------------
constexpr int kSchedChunk = 512;
constexpr int kSchedBuckets = 1024;
// Batches of up to this many chunks are visited longest chunk first (below).
constexpr int kOrderMaxChunks = 16;

// Packed groups (kPack): runs of consecutive short sequences that fit one
// 128-row Q window and one 128-key K/V window (built after the sort, in the
// sort's histogram space).
struct PackGroups {
  uint16_t start[kSchedChunk];      // first chunk-local sequence of group g
  uint16_t end[kSchedChunk];        // one past its last
  uint16_t jump[kSchedChunk];       // the segments' first sequences, in batch order
  uint32_t seg[kSchedChunk / 32];   // bit i: the greedy scan restarts at sequence i (a segment starts)
  uint32_t member[kSchedChunk / 32];  // bit i: sequence i is short (it belongs to a group)
  uint32_t first[kSchedChunk / 32];   // bit i: sequence i starts a group
};

struct SchedSmem {
  union {
    uint32_t off[kSchedBuckets];    // histogram, then running bucket offsets (sort only)
    PackGroups grp;                 // kPack, after the sort
  };
  uint32_t cum[kSchedChunk + 1];    // exclusive prefix of item counts, sorted order
  int4 span[kSchedChunk];           // decoded (q_start, q_len, kv_start, kv_len) per chunk-local sequence
  uint8_t code[kSchedChunk];        // mask type code per chunk-local sequence
  uint16_t key[kSchedChunk];        // sort key per chunk-local sequence (sort only)
  uint16_t order[kSchedChunk];      // chunk-local sequence ids, sorted
  int chunk_base;
  int chunk_n;
  int n_short;                      // kPairs: short sequences, at sorted positions [n_long, n_long + n_short)
  int n_long;                       // kPairs: long sequences, at sorted positions [0, n_long)
  int n_groups;                     // kPack: packed groups of short sequences
  int pack_on;                      // kPack: this chunk's short sequences run as packed groups
  int n_chunks;                     // chunks of the batch (-1: the visiting order is not set up yet)
  int ordered;                      // chunks are visited in the order `corder`, else in batch order
  int visit;                        // chunks loaded so far
  uint32_t cmax[kOrderMaxChunks];   // longest query sequence of each chunk
  uint16_t corder[kOrderMaxChunks]; // chunk indices, longest first
  unsigned long long item_base;
  unsigned long long item_end;
};
static_assert(sizeof(PackGroups) <= sizeof(uint32_t) * kSchedBuckets, "groups fit the histogram space");

// A short sequence fits one Q tile and one KV tile.  With kPairs (the
// warp-specialised forward), short sequences are not split into BLOCK_M items:
// their (sequence, head) tiles are taken two at a time, each with its own K/V.
__device__ __forceinline__ bool seq_is_short(const SeqInfo& s) {
  return s.q_len > 0 && s.q_len <= kTileM && s.kv_len <= kBlockN;
}
// The same test on a chunk's cached (q_start, q_len, kv_start, kv_len).
__device__ __forceinline__ bool span_is_short(int4 a) { return a.y > 0 && a.y <= kTileM && a.w <= kBlockN; }

// Sort key (descending order = processing order).  Plain: KV tiles, full
// context before causal at equal length.  kPairs: long sequences (keys >= 3)
// first in the same order, then short sequences (2 full context, 1 causal),
// then sequences without query rows (0), so short sequences form a suffix.
template <bool kPairs = false>
__device__ __forceinline__ uint32_t seq_sort_key(const SeqInfo& s) {
  int nkv = (s.kv_len + kBlockN - 1) / kBlockN;
  if (s.lo_off < kNoBound) nkv = min(nkv, s.lo_off / kBlockN + 2);   // a window bounds the tiles per row block
  if (!kPairs) {
    nkv = nkv > 511 ? 511 : nkv;
    return (uint32_t)(nkv * 2 + (s.causal ? 0 : 1));
  }
  if (s.q_len <= 0) return 0u;
  if (seq_is_short(s)) return s.causal ? 1u : 2u;
  nkv = nkv > 509 ? 509 : nkv;
  return (uint32_t)(3 + nkv * 2 + (s.causal ? 0 : 1));
}

// Items of one sequence: blocks of BLOCK rows of the query sequence times the
// query heads (forward), or of the key/value sequence times the key/value heads
// (backward, kKvSide).
template <int BLOCK, bool kKvSide>
__device__ __forceinline__ uint32_t seq_items(const SeqInfo& s, const AttnParams& p) {
  const int len = kKvSide ? s.kv_len : s.q_len;
  const int heads = kKvSide ? p.Hkv : p.Hq;
  return len > 0 ? (uint32_t)((len + BLOCK - 1) / BLOCK) * (uint32_t)heads : 0u;
}

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Sequence info of chunk-local sequence i, from the chunk's cache (no global loads).
__device__ __forceinline__ SeqInfo cached_seq(const SchedSmem& s, int i, const AttnParams& p) {
  const int4 sp = s.span[i];
  SeqInfo si;
  si.q_start = sp.x;
  si.q_len = sp.y;
  si.kv_start = sp.z;
  si.kv_len = sp.w;
  set_visibility(si, s.code[i], p);
  return si;
}

// Packs the chunk's short sequences (kPack): scanning in batch order, a group
// starts at a short sequence and takes the following short sequences while their
// rows and keys stay in order and inside 128 rows of the group's first row and
// 128 keys of its first key; the next short sequence starts the next group.
// The scan restarts at every short sequence that follows a sequence that is not
// short, or whose rows or keys begin before the previous sequence's end (no group
// crosses such a point), so the chunk splits into independent segments.  The
// lanes walk their segments (round robin) in one flat loop and mark each group's
// first sequence in a bitmask; a group then ends at the next marked sequence or
// at the next sequence that is not short, and the groups are numbered in batch
// order by counting marks.  When fewer than a quarter of the short sequences
// could take the next one into their group, packing would save few tiles: the
// chunk keeps one (sequence, head) tile per short sequence (pack_on = 0) and
// skips the walk.  One full warp; s.off / s.key are free (the sort is done).
__device__ void sched_pack_groups(SchedSmem& s, int n) {
  const int lane = threadIdx.x & 31;
  PackGroups& g = s.grp;
  const int nwords = (n + 31) >> 5;
  uint32_t joins = 0;   // short sequences whose group could take the next one
  int nseg = 0;         // segments; their first sequences in g.jump, in batch order
  int4 prev = make_int4(0, 0, 0, 0);   // the sequence before this lane's (lane 31's: the next batch's lane 0)
  bool prev_short = false;
  for (int i0 = 0; i0 < n; i0 += 32) {
    const int i = i0 + lane;
    const int4 a = i < n ? s.span[i] : make_int4(0, 0, 0, 0);
    const bool sh = i < n && span_is_short(a);
    int4 pr;
    pr.x = __shfl_up_sync(0xffffffffu, a.x, 1);
    pr.y = __shfl_up_sync(0xffffffffu, a.y, 1);
    pr.z = __shfl_up_sync(0xffffffffu, a.z, 1);
    pr.w = __shfl_up_sync(0xffffffffu, a.w, 1);
    bool pr_sh = __shfl_up_sync(0xffffffffu, sh ? 1 : 0, 1) != 0;
    if (lane == 0) {
      pr = prev;
      pr_sh = prev_short;
    }
    const bool ordered = a.x >= pr.x + pr.y && a.z >= pr.z + pr.w;
    const bool seg = sh && (i == 0 || !pr_sh || !ordered);
    if (sh && i > 0 && pr_sh && ordered && a.x + a.y <= pr.x + kTileM && a.z + a.w <= pr.z + kBlockN) ++joins;
    const uint32_t m_seg = __ballot_sync(0xffffffffu, seg);
    const uint32_t m_sh = __ballot_sync(0xffffffffu, sh);
    if (lane == 0) {
      g.seg[i0 >> 5] = m_seg;
      g.member[i0 >> 5] = m_sh;
      g.first[i0 >> 5] = 0u;
    }
    if (seg) g.jump[nseg + __popc(m_seg & ((1u << lane) - 1u))] = (uint16_t)i;
    nseg += __popc(m_seg);
    prev.x = __shfl_sync(0xffffffffu, a.x, 31);
    prev.y = __shfl_sync(0xffffffffu, a.y, 31);
    prev.z = __shfl_sync(0xffffffffu, a.z, 31);
    prev.w = __shfl_sync(0xffffffffu, a.w, 31);
    prev_short = __shfl_sync(0xffffffffu, sh ? 1 : 0, 31) != 0;
  }
  joins = __reduce_add_sync(0xffffffffu, joins);
  if (4u * joins < (uint32_t)s.n_short) {
    if (lane == 0) {
      s.pack_on = 0;
      s.n_groups = 0;
    }
    __syncwarp();
    return;
  }
  __syncwarp();
  // greedy walk of the lane's segments, one sequence per step
  {
    int r = lane;
    int st = r < nseg ? (int)g.jump[r] : 0, i = st;
    int q0 = 0, k0 = 0, qe = 0, ke = 0;
    while (r < nseg) {
      const bool in_seg = i < n && ((g.member[i >> 5] >> (i & 31)) & 1u) != 0 &&
                          (i == st || ((g.seg[i >> 5] >> (i & 31)) & 1u) == 0);
      if (!in_seg) {   // next segment of this lane
        r += 32;
        if (r < nseg) st = i = (int)g.jump[r];
        continue;
      }
      const int4 a = s.span[i];
      if (i == st || a.x < qe || a.z < ke || a.x + a.y > q0 + kTileM || a.z + a.w > k0 + kBlockN) {
        atomicOr(&g.first[i >> 5], 1u << (i & 31));   // starts a group
        q0 = a.x;
        k0 = a.z;
      }
      qe = a.x + a.y;
      ke = a.z + a.w;
      ++i;
    }
  }
  __syncwarp();
  // groups in batch order: lane w numbers the group starts in word w, and a group
  // ends at the next start or at the next sequence that is not short
  const uint32_t fw = lane < nwords ? g.first[lane] : 0u;
  const int cnt = __popc(fw);
  const int base = (int)warp_incl_scan((uint32_t)cnt) - cnt;
  uint32_t rest = fw;
  for (int k = 0; rest != 0u; ++k) {
    const int bit = __ffs(rest) - 1;
    rest &= rest - 1u;
    const int pos = 32 * lane + bit;
    // stops after pos: later starts and sequences that are not short (none past n)
    uint32_t stops = (fw | ~g.member[lane]) & ~((2u << bit) - 1u);
    int w = lane;
    while (stops == 0u && ++w < nwords) stops = g.first[w] | ~g.member[w];
    const int end = stops != 0u ? min(32 * w + __ffs(stops) - 1, n) : n;
    g.start[base + k] = (uint16_t)pos;
    g.end[base + k] = (uint16_t)end;
  }
  const int ng = __shfl_sync(0xffffffffu, base + cnt, 31);
  if (lane == 0) {
    s.n_groups = ng;
    s.pack_on = 1;
  }
  __syncwarp();
}

// Load and sort the chunk of sequences starting at `base`.  One full warp.
template <int BLOCK_M, bool kKvSide = false, bool kPairs = false, bool kPack = false>
__device__ void sched_load_chunk(SchedSmem& s, const AttnParams& p, int base) {
  static_assert(!kPack || kPairs, "packed groups replace the paired short tiles");
  const int lane = threadIdx.x & 31;
  const int n = min(kSchedChunk, p.B - base);
  for (int i = lane; i < kSchedBuckets; i += 32) s.off[i] = 0u;
  __syncwarp();
  for (int i0 = 0; i0 < n; i0 += 32) {
    const int i = i0 + lane;
    uint32_t k = 0xFFFFFFFFu;
    if (i < n) {
      const SeqInfo si = load_seq(p, base + i);
      s.span[i] = make_int4(si.q_start, si.q_len, si.kv_start, si.kv_len);
      const int raw = p.causal ? (int)p.causal[base + i] : kMaskPadding;
      s.code[i] = (uint8_t)(raw == kMaskPadding ? kMaskPadding : (raw == kMaskCausalBottomRight ? raw : 1));
      k = seq_sort_key<kPairs>(si);
      s.key[i] = (uint16_t)k;
    }
    // one add per distinct key of the 32 (many sequences share a key: the adds to one
    // bucket would otherwise be serialised)
    const uint32_t peers = __match_any_sync(0xffffffffu, k);
    if (i < n && lane == __ffs(peers) - 1) atomicAdd(&s.off[k], (uint32_t)__popc(peers));
  }
  __syncwarp();
  if (kPairs && lane == 0) {
    s.n_short = (int)(s.off[1] + s.off[2]);
    s.n_long = n - s.n_short - (int)s.off[0];
  }
  // exclusive offsets, keys in descending order; lane l owns 32 consecutive keys
  uint32_t sum = 0;
  for (int t = 0; t < 32; ++t) sum += s.off[kSchedBuckets - 1 - (lane * 32 + t)];
  uint32_t run = warp_incl_scan(sum) - sum;
  __syncwarp();
  for (int t = 0; t < 32; ++t) {
    const int kidx = kSchedBuckets - 1 - (lane * 32 + t);
    const uint32_t c = s.off[kidx];
    s.off[kidx] = run;
    run += c;
  }
  __syncwarp();
  // stable scatter: 32 sequences at a time, equal keys ranked by lane
  for (int i0 = 0; i0 < n; i0 += 32) {
    const int i = i0 + lane;
    const bool act = i < n;
    const uint32_t k = act ? (uint32_t)s.key[i] : 0xFFFFFFFFu;
    const uint32_t peers = __match_any_sync(0xffffffffu, k);
    const uint32_t rank = __popc(peers & ((1u << lane) - 1u));
    const uint32_t pos = act ? s.off[k] + rank : 0u;
    __syncwarp();
    if (act && rank == 0) s.off[k] += __popc(peers);
    if (act) s.order[pos] = (uint16_t)i;
    __syncwarp();
  }
  // prefix of item counts over the sorted order
  uint32_t carry = 0;
  for (int j0 = 0; j0 < n; j0 += 32) {
    const int j = j0 + lane;
    uint32_t it = 0u;
    if (j < n) {
      const SeqInfo sj = cached_seq(s, s.order[j], p);
      if (kPairs && seq_is_short(sj)) {
        it = 0u;
      } else if (kPairs && (p.group & 1) == 0) {   // grouped heads: 128-row blocks of two heads
        it = (uint32_t)((sj.q_len + kTileM - 1) / kTileM) * (uint32_t)(p.Hq / 2);
      } else {
        it = seq_items<BLOCK_M, kKvSide>(sj, p);
      }
    }
    const uint32_t incl = warp_incl_scan(it);
    if (j < n) s.cum[j + 1] = carry + incl;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) {
    s.cum[0] = 0;
    s.chunk_base = base;
    s.chunk_n = n;
  }
  __syncwarp();
  if (kPack) {   // a chunk without short sequences has no groups
    if (s.n_short > 0) {
      sched_pack_groups(s, n);
    } else if (lane == 0) {
      s.n_groups = 0;
      s.pack_on = 0;
    }
    __syncwarp();
  }
}

// Work item decoded from the global item index.
struct WorkItem {
  int valid;
  int b, h, qblock;
  SeqInfo seq;
};

// One full warp.  Maps global item index w to (sequence, head, block), loading
// later chunks as needed (w never decreases within a CTA).  Forward: query
// blocks, heaviest (last) first; backward (kKvSide): key/value blocks and
// heads, lowest block first (under causal masking the first keys are seen by
// the most queries).
// Items (units, with kPairs) of the loaded chunk: the long sequences' items,
// then the short sequences' (sequence, head) tiles two per unit, or with kPack
// the packed groups' (group, head) tiles two per unit.
template <bool kPairs, bool kPack = false>
__device__ __forceinline__ unsigned long long chunk_items(const SchedSmem& s, const AttnParams& p) {
  unsigned long long n = s.cum[s.chunk_n];
  const int tiles = (kPack && s.pack_on) ? s.n_groups : s.n_short;
  if (kPairs) n += ((unsigned long long)tiles * (unsigned long long)p.Hq + 1ull) / 2ull;
  return n;
}

// Chunk visiting order: the chunks of sequences (kSchedChunk consecutive ones
// each) are taken longest chunk first, a chunk's length being its longest query
// sequence (ties in batch order), so that long sequences in a late chunk do not
// start last; inside a chunk the sequences are sorted as above.  Every CTA
// computes the same order from the device metadata (cu_seqlens_q only: its
// batch_size + 1 entries), before loading its first chunk; batches of more than
// kOrderMaxChunks chunks keep batch order.  One full warp.
__device__ void sched_order_chunks(SchedSmem& s, const AttnParams& p) {
  const int lane = threadIdx.x & 31;
  const int nch = (p.B + kSchedChunk - 1) / kSchedChunk;
  const bool order = nch > 1 && nch <= kOrderMaxChunks;
  if (order) {
    // lane l reads the cu_seqlens_q entries of sequences [16 l, 16 l + 16) of a chunk
    constexpr int kPerLane = kSchedChunk / 32;
#pragma unroll 2
    for (int c = 0; c < nch; ++c) {
      const int b0 = c * kSchedChunk + lane * kPerLane;
      const int bend = min(p.B, (c + 1) * kSchedChunk);
      int v[kPerLane + 1];
#pragma unroll
      for (int u = 0; u <= kPerLane; ++u) v[u] = b0 + u <= bend ? __ldg(p.cu_q + b0 + u) : 0;
      long long m = 0;
#pragma unroll
      for (int u = 0; u < kPerLane; ++u)
        if (b0 + u < bend) m = max(m, min((long long)v[u + 1] - v[u], (long long)p.T));
      const uint32_t cm = __reduce_max_sync(0xffffffffu, (uint32_t)m);
      if (lane == 0) s.cmax[c] = cm;
    }
    __syncwarp();
    if (lane < nch) {
      const uint32_t mine = s.cmax[lane];
      int rank = 0;
      for (int c = 0; c < nch; ++c) {
        const uint32_t o = s.cmax[c];
        rank += (o > mine || (o == mine && c < lane)) ? 1 : 0;
      }
      s.corder[rank] = (uint16_t)lane;
    }
  }
  __syncwarp();
  if (lane == 0) {
    s.n_chunks = nch;
    s.ordered = order ? 1 : 0;
    s.visit = 0;
  }
  __syncwarp();
}

// Loads later chunks until the one holding global item w; false when w is
// past the last item.  One full warp.
template <int BLOCK_M, bool kKvSide = false, bool kPairs = false, bool kPack = false>
__device__ bool sched_seek(SchedSmem& s, const AttnParams& p, unsigned long long w) {
  while (w >= s.item_end) {
    if (s.n_chunks < 0) sched_order_chunks(s, p);
    if (s.visit >= s.n_chunks) return false;
    const int c = s.ordered ? (int)s.corder[s.visit] : s.visit;
    const unsigned long long base_items = s.item_end;
    sched_load_chunk<BLOCK_M, kKvSide, kPairs, kPack>(s, p, c * kSchedChunk);
    if ((threadIdx.x & 31) == 0) {
      s.item_base = base_items;
      s.item_end = base_items + chunk_items<kPairs, kPack>(s, p);
      s.visit += 1;
    }
    __syncwarp();
  }
  return true;
}

// Sorted position of the sequence holding chunk-local item `local` (which must
// be below cum[chunk_n]): the last position whose prefix does not exceed it.
__device__ __forceinline__ int sched_find(const SchedSmem& s, uint32_t local) {
  int lo = 0, hi = s.chunk_n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s.cum[mid] <= local) lo = mid; else hi = mid;
  }
  return lo;
}

template <int BLOCK_M, bool kKvSide = false>
__device__ WorkItem sched_decode(SchedSmem& s, const AttnParams& p, unsigned long long w) {
  WorkItem it;
  it.valid = 0;
  if (!sched_seek<BLOCK_M, kKvSide>(s, p, w)) return it;
  const uint32_t local = (uint32_t)(w - s.item_base);
  const int lo = sched_find(s, local);
  it.b = s.chunk_base + s.order[lo];
  it.seq = cached_seq(s, s.order[lo], p);
  const uint32_t r = local - s.cum[lo];
  const int len = kKvSide ? it.seq.kv_len : it.seq.q_len;
  const uint32_t nblk = (uint32_t)((len + BLOCK_M - 1) / BLOCK_M);
  it.h = (int)(r / nblk);
  it.qblock = kKvSide ? (int)(r % nblk) : (int)(nblk - 1u - (r % nblk));
  it.valid = 1;
  return it;
}

// Global work counter, p.claim items per atomic (fewer round trips when items
// are small).  Call with the whole warp; the claimed indices of one CTA increase.
struct Claimer {
  unsigned long long base;
  int left;
};
__device__ __forceinline__ unsigned long long claim_item(Claimer& c, const AttnParams& p) {
  if (c.left == 0) {
    unsigned long long b = 0;
    if ((threadIdx.x & 31) == 0) b = atomicAdd(p.work_counter, (unsigned long long)p.claim);
    c.base = __shfl_sync(0xffffffffu, b, 0);
    c.left = p.claim;
  }
  const unsigned long long w = c.base + (unsigned long long)(p.claim - c.left);
  --c.left;
  return w;
}

__device__ __forceinline__ void sched_init(SchedSmem& s) {
  s.chunk_base = 0;
  s.chunk_n = 0;
  s.n_short = 0;
  s.n_long = 0;
  s.n_groups = 0;
  s.pack_on = 0;
  s.n_chunks = -1;
  s.ordered = 0;
  s.visit = 0;
  s.item_base = 0;
  s.item_end = 0;
}

// ----------------------------------------------------------------------------
// Pad rows: every output row outside all [start_b, start_b + len_b) ranges is
// written as exact zeros (and -inf LSE).  Gap g (0 <= g <= B) is the range
// between the end of sequence g-1 (0 for g == 0) and the start of sequence g
// (T for g == B).  Gaps before a sequence are spread over CTAs, one CTA each; the
// trailing gap, which is most of the buffer when the buffer holds more rows than
// the batch (T sized for a larger batch), is split over all CTAs in equal shares.
// `nthreads` threads starting at thread `t0` of the CTA take part.
// ----------------------------------------------------------------------------
__device__ void zero_pad_rows(const AttnParams& p, int t0, int nthreads, int elem_bytes) {
  const int tid = (int)threadIdx.x - t0;
  const long long row_bytes = (long long)p.Hq * p.d * elem_bytes;
  auto zero_rows = [&](long long a, long long e) {   // rows [a, e)
    if (e <= a) return;
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<char*>(p.out) + a * row_bytes);
    const long long n16 = (e - a) * row_bytes / 16;
    for (long long i = tid; i < n16; i += nthreads) dst[i] = make_uint4(0u, 0u, 0u, 0u);
    if (p.lse) {
      const long long rows = e - a;
      for (long long i = tid; i < rows * p.Hq; i += nthreads) {
        const long long h = i / rows, r = i % rows;
        p.lse[h * p.T + a + r] = -INFINITY;
      }
    }
  };
  for (int g = blockIdx.x; g < p.B; g += gridDim.x) {
    long long a = 0;
    if (g > 0) {
      SeqInfo s = load_seq(p, g - 1);
      a = (long long)s.q_start + s.q_len;
    }
    const long long cq = p.cu_q[g];
    const long long st = p.pad_q ? (long long)p.pad_q[g] : cq;
    zero_rows(a, st < 0 ? 0 : (st > p.T ? p.T : st));
  }
  long long a = 0;   // the trailing gap [end of the last sequence, T), this CTA's share
  if (p.B > 0) {
    SeqInfo s = load_seq(p, p.B - 1);
    a = (long long)s.q_start + s.q_len;
  }
  const long long rows = (long long)p.T - a;
  if (rows > 0)
    zero_rows(a + rows * blockIdx.x / gridDim.x, a + rows * (blockIdx.x + 1) / gridDim.x);
}

// Byte offset of 16-byte chunk `c` of row `r` of a 128-row tile stored as
// 64-column panels of 16 KB (128-byte rows) with the 128-byte swizzle: the
// chunk index is XORed with (row mod 8), as TMA writes it.
__device__ __forceinline__ uint32_t sw128_offset(int r, int c) {
  return (uint32_t)((c >> 3) * (kTileM * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

template <typename DT>
struct DTypeTraits;
template <>
struct DTypeTraits<__nv_bfloat16> {
  static constexpr bool kBF16 = true;
  __device__ static __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __device__ static __forceinline__ float lo(uint32_t x) { return __uint_as_float(x << 16); }
  __device__ static __forceinline__ float hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }
  // a += low half of x, b += high half of x (mixed-precision adds, exact widening)
  __device__ static __forceinline__ void acc2(uint32_t x, float& a, float& b) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %1, h, %1;\n\t}"
        : "+f"(a), "+f"(b) : "r"(x));
  }
};
template <>
struct DTypeTraits<__half> {
  static constexpr bool kBF16 = false;
  __device__ static __forceinline__ uint32_t pack2(float a, float b) {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __device__ static __forceinline__ float lo(uint32_t x) {
    return __half2float(__ushort_as_half((unsigned short)(x & 0xFFFFu)));
  }
  __device__ static __forceinline__ float hi(uint32_t x) {
    return __half2float(__ushort_as_half((unsigned short)(x >> 16)));
  }
  __device__ static __forceinline__ void acc2(uint32_t x, float& a, float& b) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.f16 %0, l, %0;\n\tadd.rn.f32.f16 %1, h, %1;\n\t}"
        : "+f"(a), "+f"(b) : "r"(x));
  }
};

}  // namespace thd
