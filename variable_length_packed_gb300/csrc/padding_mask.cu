// padding_mask.cu — the attention padding mask built on the device.
//
// Source: "[PyTorch] Build the attention padding mask without host syncs"
// (TransformerEngine PR).  mask[b, p] = (p >= cu[b+1] - cu[b]) for b < B,
// p < S, stored as one byte per position ([B, 1, 1, S] bool).  Only entries
// 0..B of cu are read (Changes: longer buffers are allowed), and a sequence
// longer than S gives an all-False row (Equivalence).
//
// The output is a pure HBM write stream, written in 16-byte chunks (a warp
// store covers 512 contiguous bytes).  Within one row the mask bytes of a chunk
// form a step (0 ... 0 1 ... 1), built with 64-bit shifts instead of 16
// compares.
//  * Rows of whole, aligned chunks (S a multiple of 16, 16-byte aligned mask):
//    a warp writes one row at a time, its length read once; no division.
//  * Otherwise the flat B*S array is cut into chunks regardless of rows; a chunk
//    spans at most two rows, and its row is found with one exact division by the
//    invariant S: a multiply-high by a reciprocal precomputed on the host
//    (division by invariant integers using multiplication, Granlund &
//    Montgomery, 1994).  The unaligned head and tail bytes are written one at a
//    time.
#include <cstdint>
#include <cuda_runtime.h>

namespace thd {

namespace {

constexpr uint64_t kOnes = 0x0101010101010101ull;

struct MaskArgs {
  const int32_t* cu;
  uint8_t* mask;
  long long S;
  long long total;     // B * S
  long long head;      // bytes before the first 16-byte aligned address
  long long nchunks;   // aligned 16-byte chunks
  uint64_t recip;      // floor((2^64 - 1) / S) + 1, exact quotient for numerators < 2^32
  int div32;           // total < 2^32: use the reciprocal
};

// read-only path: the loads of several chunks can be in flight at once
__device__ __forceinline__ long long row_len(const int32_t* cu, long long b) {
  return (long long)__ldg(cu + b + 1) - (long long)__ldg(cu + b);
}

__device__ __forceinline__ void div_row(const MaskArgs& a, long long f, long long& b, long long& p) {
  if (a.div32) {
    b = (a.S == 1) ? f : (long long)__umul64hi((unsigned long long)f, a.recip);
  } else {
    b = f / a.S;
  }
  p = f - b * a.S;
}

// 16 mask bytes (two little-endian words) with bytes [t, 16) set, t in [0, 16].
__device__ __forceinline__ void step_from(int t, uint64_t& lo, uint64_t& hi) {
  lo = t >= 8 ? 0ull : (kOnes << (8 * t));
  hi = t >= 16 ? 0ull : (t <= 8 ? kOnes : (kOnes << (8 * (t - 8))));
}

__device__ __forceinline__ int clampi(long long x, int lo, int hi) {
  return (int)(x < lo ? lo : (x > hi ? hi : x));
}

__device__ __forceinline__ uint8_t mask_byte(const MaskArgs& a, long long f) {
  long long b, p;
  div_row(a, f, b, p);
  return (uint8_t)(p >= row_len(a.cu, b) ? 1 : 0);
}

// Chunk starting at flat byte f (S >= 16: the chunk spans at most two rows).
__device__ __forceinline__ uint4 mask_chunk(const MaskArgs& a, long long f) {
  long long b, p0;
  div_row(a, f, b, p0);
  const long long len0 = row_len(a.cu, b);
  const int e0 = (int)(a.S - p0 < 16 ? a.S - p0 : 16);   // bytes of row b in the chunk
  const int t0 = clampi(len0 - p0, 0, e0);                // first padded byte of row b
  uint64_t lo, hi, lo_e, hi_e;
  step_from(t0, lo, hi);
  step_from(e0, lo_e, hi_e);
  lo &= ~lo_e;
  hi &= ~hi_e;
  if (e0 < 16) {                                          // row b + 1 fills the rest
    const long long len1 = row_len(a.cu, b + 1);
    const int t1 = e0 + clampi(len1, 0, 16 - e0);
    uint64_t lo1, hi1;
    step_from(t1, lo1, hi1);
    lo |= lo1;
    hi |= hi1;
  }
  return make_uint4((uint32_t)lo, (uint32_t)(lo >> 32), (uint32_t)hi, (uint32_t)(hi >> 32));
}

__global__ void __launch_bounds__(256) padding_mask_kernel(const MaskArgs a) {
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long stride = (long long)gridDim.x * blockDim.x;
  if (tid < a.head) a.mask[tid] = mask_byte(a, tid);
  const long long tail0 = a.head + a.nchunks * 16;
  if (tid < a.total - tail0) a.mask[tail0 + tid] = mask_byte(a, tail0 + tid);
  uint4* body = reinterpret_cast<uint4*>(a.mask + a.head);
  if (a.S >= 16) {
    long long c = tid;
    for (; c + 3 * stride < a.nchunks; c += 4 * stride) {   // four independent chunks in flight
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = mask_chunk(a, a.head + (c + u * stride) * 16);
#pragma unroll
      for (int u = 0; u < 4; ++u) body[c + u * stride] = v[u];
    }
    for (; c < a.nchunks; c += stride) body[c] = mask_chunk(a, a.head + c * 16);
  } else {
    for (long long c = tid; c < a.nchunks; c += stride) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) word |= (uint32_t)mask_byte(a, a.head + c * 16 + 4 * q + i) << (8 * i);
        w[q] = word;
      }
      body[c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// Row path: S = 16 * chunks_per_row, mask 16-byte aligned.  Warp w writes rows
// w, w + warps, ...; lane l writes chunks l, l + 32, ... of the row.
__global__ void __launch_bounds__(256) padding_mask_rows_kernel(const int32_t* cu, uint8_t* mask, int B,
                                                                int chunks_per_row) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < B; b += warps) {
    const long long len = row_len(cu, b);
    uint4* row = reinterpret_cast<uint4*>(mask + (size_t)b * (size_t)chunks_per_row * 16u);
#pragma unroll 4
    for (int k = lane; k < chunks_per_row; k += 32) {
      uint64_t lo, hi;
      step_from(clampi(len - 16ll * k, 0, 16), lo, hi);
      row[k] = make_uint4((uint32_t)lo, (uint32_t)(lo >> 32), (uint32_t)hi, (uint32_t)(hi >> 32));
    }
  }
}

}  // namespace

// Host launcher (called from the C ABI in thd_attn.cu after validation).
cudaError_t launch_padding_mask(const int32_t* cu, int B, int S, uint8_t* mask, int num_sms, cudaStream_t stream) {
  MaskArgs a;
  a.cu = cu;
  a.mask = mask;
  a.S = S;
  a.total = (long long)B * (long long)S;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(mask);
  a.head = (long long)((16 - (addr & 15)) & 15);
  if (a.head > a.total) a.head = a.total;
  a.nchunks = (a.total - a.head) / 16;
  a.div32 = a.total <= 0xFFFFFFFFll ? 1 : 0;
  a.recip = S > 1 ? (0xFFFFFFFFFFFFFFFFull / (uint64_t)S) + 1ull : 0ull;
  const int threads = 256;
  const long long cap_blocks = (long long)num_sms * 8;   // 8 resident 256-thread blocks per SM
  if (S % 16 == 0 && a.head == 0 && B > 0) {
    const long long rows_blocks = ((long long)B + 7) / 8;   // one row per warp
    const int grid = (int)(rows_blocks < cap_blocks ? rows_blocks : cap_blocks);
    padding_mask_rows_kernel<<<grid, threads, 0, stream>>>(cu, mask, B, S / 16);
    return cudaGetLastError();
  }
  long long want = (a.nchunks + 4 * threads - 1) / (4 * threads);
  if (want < 1) want = 1;
  const int grid = (int)(want < cap_blocks ? want : cap_blocks);
  padding_mask_kernel<<<grid, threads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace thd
