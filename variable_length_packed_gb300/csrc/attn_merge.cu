// attn_merge.cu — combine two partial attention results over disjoint key sets.
//
// With S = exp(lse_a) + exp(lse_b) for one (row, head):
//   lse = log S,  out = exp(lse_a - lse) * out_a + exp(lse_b - lse) * out_b.
// A partial with lse = -inf saw no key and gets weight 0; when both are -inf
// the row is 0 with lse -inf.  This is the step that makes the context-parallel
// example of "How to pad sequences that cannot be evenly split in context
// parallelism (CP)?" (Megatron-LM issue) exact: each rank's chunk of keys gives
// a partial (out, lse), and merging them reproduces full attention; the
// two-call pad_between_seqs sum of "Add per-sequence causal policy to packed
// THD attention" is the special case where every row has one -inf partial.
//
// Pure HBM stream: d/8 lanes cover one row with 16-byte loads and stores; all
// lanes of a row read both LSEs before one lane writes the merged LSE, so the
// output may alias either input.
#include <cmath>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace thd {

namespace {

struct MergeArgs {
  const void* out_a;
  const float* lse_a;
  const void* out_b;
  const float* lse_b;
  void* out;
  float* lse;
  long long rows;   // T * H
  int T, H, d;
};

__device__ __forceinline__ float2 unpack2(uint32_t x, bool bf16) {
  if (bf16) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&x);
    return __bfloat1622float2(v);
  }
  __half2 v = *reinterpret_cast<__half2*>(&x);
  return __half22float2(v);
}

__device__ __forceinline__ uint32_t pack2(float a, float b, bool bf16) {
  if (bf16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <bool kBF16>
__global__ void __launch_bounds__(256) attn_merge_kernel(const MergeArgs a) {
  const int lane = threadIdx.x & 31;
  const int lanes_per_row = a.d / 8;
  const int rows_per_warp = 32 / lanes_per_row;
  const int sub = lane / lanes_per_row;            // row of this lane inside the warp's group
  const int chunk = lane % lanes_per_row;          // 16-byte chunk of the row
  const bool active_lane = sub < rows_per_warp;
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long r0 = warp * rows_per_warp; r0 < a.rows; r0 += nwarps * rows_per_warp) {
    const long long row = r0 + sub;
    const bool act = active_lane && row < a.rows;
    float lse = -INFINITY;
    long long li = 0;
    if (act) {
      const long long t = row / a.H, h = row % a.H;
      li = h * a.T + t;
      const float la = a.lse_a[li], lb = a.lse_b[li];
      const float m = fmaxf(la, lb);
      float wa = 0.f, wb = 0.f;
      if (m != -INFINITY) {
        const float ea = expf(la - m), eb = expf(lb - m);   // expf(-inf) = 0
        const float s = ea + eb;
        lse = m + logf(s);
        wa = ea / s;
        wb = eb / s;
      }
      const size_t off = (size_t)row * a.d * 2 + (size_t)chunk * 16;
      const uint4 xa = *reinterpret_cast<const uint4*>(static_cast<const char*>(a.out_a) + off);
      const uint4 xb = *reinterpret_cast<const uint4*>(static_cast<const char*>(a.out_b) + off);
      const uint32_t ua[4] = {xa.x, xa.y, xa.z, xa.w};
      const uint32_t ub[4] = {xb.x, xb.y, xb.z, xb.w};
      uint32_t r[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 fa = unpack2(ua[i], kBF16), fb = unpack2(ub[i], kBF16);
        // a zero-weight partial contributes nothing, whatever its stored values
        const float x = (wa != 0.f ? wa * fa.x : 0.f) + (wb != 0.f ? wb * fb.x : 0.f);
        const float y = (wa != 0.f ? wa * fa.y : 0.f) + (wb != 0.f ? wb * fb.y : 0.f);
        r[i] = pack2(x, y, kBF16);
      }
      *reinterpret_cast<uint4*>(static_cast<char*>(a.out) + off) = make_uint4(r[0], r[1], r[2], r[3]);
    }
    __syncwarp();   // every lane of the row has read lse_a / lse_b
    if (act && chunk == 0) a.lse[li] = lse;
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_attn_merge(const void* out_a, const float* lse_a, const void* out_b, const float* lse_b,
                              void* out, float* lse, int T, int H, int d, bool bf16, int num_sms,
                              cudaStream_t stream) {
  MergeArgs a{out_a, lse_a, out_b, lse_b, out, lse, (long long)T * H, T, H, d};
  const int threads = 256;
  const long long rows_per_block = (long long)(threads / 32) * (32 / (d / 8));
  long long want = (a.rows + rows_per_block - 1) / rows_per_block;
  const long long cap = (long long)num_sms * 8;
  const int grid = (int)(want < 1 ? 1 : (want < cap ? want : cap));
  if (bf16)
    attn_merge_kernel<true><<<grid, threads, 0, stream>>>(a);
  else
    attn_merge_kernel<false><<<grid, threads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace thd
