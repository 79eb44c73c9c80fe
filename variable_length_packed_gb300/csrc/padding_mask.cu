// padding_mask.cu — the attention padding mask built on the device.
//
// Source: "[PyTorch] Build the attention padding mask without host syncs"
// (TransformerEngine PR).  mask[b, p] = (p >= cu[b+1] - cu[b]) for b < B,
// p < S, stored as one byte per position ([B, 1, 1, S] bool).  Only entries
// 0..B of cu are read (Changes: longer buffers are allowed), and a sequence
// longer than S gives an all-False row (Equivalence).
//
// The output is a pure HBM write stream: each thread writes whole 16-byte
// chunks of the flat B*S byte array (coalesced 512-byte warp stores), walking
// the row index forward inside the chunk; the unaligned head and tail bytes
// of the buffer are written one byte at a time.
#include <cstdint>
#include <cuda_runtime.h>

namespace thd {

__device__ __forceinline__ int row_len(const int32_t* cu, long long b) {
  return (int)((long long)cu[b + 1] - (long long)cu[b]);
}

// Mask bytes [f, f + n) of the flat array, n <= 16, packed little-endian.
__device__ __forceinline__ void mask_bytes(const int32_t* cu, long long S, long long f, int n, uint8_t* out) {
  long long b = f / S;
  long long p = f - b * S;
  long long len = row_len(cu, b);
  for (int i = 0; i < n; ++i) {
    out[i] = (uint8_t)(p >= len ? 1 : 0);
    if (++p == S) {
      p = 0;
      ++b;
      if (i + 1 < n) len = row_len(cu, b);
    }
  }
}

__global__ void __launch_bounds__(256) padding_mask_kernel(const int32_t* __restrict__ cu, long long S,
                                                            uint8_t* __restrict__ mask, long long total,
                                                            long long head, long long nchunks) {
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long stride = (long long)gridDim.x * blockDim.x;
  // unaligned head and tail bytes
  if (tid < head) {
    uint8_t v;
    mask_bytes(cu, S, tid, 1, &v);
    mask[tid] = v;
  }
  const long long tail0 = head + nchunks * 16;
  if (tid < total - tail0) {
    uint8_t v;
    mask_bytes(cu, S, tail0 + tid, 1, &v);
    mask[tail0 + tid] = v;
  }
  uint4* body = reinterpret_cast<uint4*>(mask + head);
  if (S >= 16) {
    // a 16-byte chunk spans at most two rows: one division per chunk
    for (long long c = tid; c < nchunks; c += stride) {
      const long long f = head + c * 16;
      const long long b = f / S;
      const long long p0 = f - b * S;
      const long long len0 = row_len(cu, b);
      const long long split = S - p0;   // bytes left in row b
      const long long len1 = split < 16 ? (long long)row_len(cu, b + 1) : 0;
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int k = q * 4 + i;
          const bool pad = (k < split) ? (p0 + k >= len0) : ((long long)k - split >= len1);
          word |= (pad ? 1u : 0u) << (8 * i);
        }
        w[q] = word;
      }
      body[c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    for (long long c = tid; c < nchunks; c += stride) {
      uint8_t bytes[16];
      mask_bytes(cu, S, head + c * 16, 16, bytes);
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        w[q] = bytes[4 * q] | (bytes[4 * q + 1] << 8) | (bytes[4 * q + 2] << 16) | ((uint32_t)bytes[4 * q + 3] << 24);
      body[c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// Host launcher (called from the C ABI in thd_attn.cu after validation).
cudaError_t launch_padding_mask(const int32_t* cu, int B, int S, uint8_t* mask, int num_sms, cudaStream_t stream) {
  const long long total = (long long)B * (long long)S;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(mask);
  long long head = (long long)((16 - (addr & 15)) & 15);
  if (head > total) head = total;
  const long long nchunks = (total - head) / 16;
  const int threads = 256;
  long long want = (nchunks + threads - 1) / threads;
  if (want < 1) want = 1;
  const long long cap = (long long)num_sms * 8;   // 8 resident 256-thread blocks per SM
  const int grid = (int)(want < cap ? want : cap);
  padding_mask_kernel<<<grid, threads, 0, stream>>>(cu, (long long)S, mask, total, head, nchunks);
  return cudaGetLastError();
}

}  // namespace thd
