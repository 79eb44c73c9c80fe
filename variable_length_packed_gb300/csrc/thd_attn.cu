// thd_attn.cu — the C ABI of libthdattn.so (declared in include/thd_attn.h):
// host-side argument validation, TMA tensor-map encoding and kernel launches.
// Nothing here reads device memory or synchronises a stream.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/thd_attn.h"
#include "attn_fwd_serial.cuh"
#include "attn_fwd_ws.cuh"
#include "attn_bwd.cuh"

namespace thd {
cudaError_t launch_padding_mask(const int32_t* cu, int B, int S, uint8_t* mask, int num_sms, cudaStream_t stream);
cudaError_t launch_attn_merge(const void* out_a, const float* lse_a, const void* out_b, const float* lse_b,
                              void* out, float* lse, int T, int H, int d, bool bf16, int num_sms,
                              cudaStream_t stream);
}

namespace {

constexpr size_t kWorkspaceBytes = 256;

// Limit of one pipeline wait inside the kernels, for calls made from now on
// (thd_set_wait_limit_ns; 0 restores the default).
std::atomic<uint64_t> g_wait_limit_ns{thd::kWaitLimitNs};

// A waiting thread reads the clock every 256 polls; with a limit under 1 ms
// (only ever set to make waits run out on purpose) it reads it at every poll,
// so that a wait the hardware completes within a few polls still runs out.
// Test setting (thd_set_wait_injection): every CTA of a later call makes one wait on a
// barrier that nothing completes before the CTA's end, so that wait runs out whatever the
// timing of the rest of the pipeline.
std::atomic<uint32_t> g_inject_wait{0u};

void set_wait_fields(thd::AttnParams& p) {
  p.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  p.wait_check_mask = p.wait_limit_ns < 1000000ull ? 0u : 255u;
  p.inject_wait = g_inject_wait.load(std::memory_order_relaxed);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int num_sms_of_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return n;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Work items claimed per atomic on the scheduler's counter.  With short
// sequences (the max_seqlen hint) an item is a few microseconds of work and the
// atomic's round trip would dominate; long items take one at a time so the
// longest-first order still balances the tail.  Any value is correct.
int claim_for(int max_seqlen, long long min_items, int ctas) {
  if (max_seqlen <= 0) return 1;
  int c = 2048 / max_seqlen;
  // every CTA should still get several claims: batch * heads is a lower bound on the items
  const long long per_cta = min_items / (8ll * (ctas > 0 ? ctas : 1));
  if (c > per_cta) c = (int)per_cta;
  return c < 1 ? 1 : (c > 8 ? 8 : c);
}

// 2-D view [rows, heads * d] of a THD tensor, box = 128 rows x 64 columns,
// 128-byte swizzle (the layout the UMMA shared-memory descriptors expect).
bool encode_thd_map(CUtensorMap* map, const void* base, int rows, int heads, int d, bool bf16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)heads * (cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)heads * (cuuint64_t)d * 2ull};
  cuuint32_t box[2] = {64u, 128u};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D view [rows, cols] of an fp32 array, box = 128 rows x 32 columns (128 bytes),
// 128-byte swizzle: the target of the backward pass's dQ tile reductions.
bool encode_f32_map(CUtensorMap* map, const void* base, int rows, long long cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 4ull};
  cuuint32_t box[2] = {32u, 128u};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <typename DT, int DP, bool kTMA>
int launch_serial(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const thd::AttnParams& p,
                  int grid, cudaStream_t stream) {
  auto kern = thd::attn_fwd_serial_kernel<DT, DP, kTMA>;
  const size_t smem = sizeof(thd::SerialSmem<DP>) + 1024;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return THD_ERR_CUDA;
  kern<<<grid, 128, smem, stream>>>(mq, mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? THD_OK : THD_ERR_CUDA;
}

// Kernels that allocate all 512 TMEM columns must run one CTA per SM: a second
// CTA on the same SM would wait in tcgen05.alloc until the first one exits.
// Requesting more than half of the SM's shared memory guarantees that.
constexpr size_t kOneCtaPerSmSmem = 120 * 1024;
size_t one_cta_per_sm(size_t bytes) { return bytes > kOneCtaPerSmSmem ? bytes : kOneCtaPerSmSmem; }

// Batches whose max_seqlen hint is at most this many rows run the instantiation
// that packs runs of short sequences into shared tiles.  The hint only picks the
// instantiation (both are exact for any lengths); the two compute short sequences
// in differently laid-out tiles, so their results agree within rounding, not bit
// for bit.
constexpr int kPackMaxSeqlen = 256;

template <typename DT, int DP>
int launch_ws(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const thd::AttnParams& p,
              int max_seqlen, int grid, cudaStream_t stream) {
  // the windowed instantiation carries the window's lower bound through the pipeline
  const bool win = p.win_left >= 0 || p.win_right >= 0;
  const bool pack = !win && max_seqlen > 0 && max_seqlen <= kPackMaxSeqlen;
  auto kern = win ? thd::attn_fwd_ws_kernel<DT, DP, true, false>
                  : (pack ? thd::attn_fwd_ws_kernel<DT, DP, false, true> : thd::attn_fwd_ws_kernel<DT, DP, false, false>);
  const size_t smem = one_cta_per_sm(sizeof(thd::WsSmem<DP>) + 1024);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return THD_ERR_CUDA;
  kern<<<grid, thd::kWsThreads, smem, stream>>>(mq, mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? THD_OK : THD_ERR_CUDA;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

size_t bwd_workspace_bytes(int T, int Hq, int d) {
  return kWorkspaceBytes + align256((size_t)Hq * T * 4) + align256((size_t)T * Hq * d * 4);
}

template <typename DT, int DP>
int launch_bwd(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdo,
               const CUtensorMap& mdq, const thd::BwdParams& bp, int sms, cudaStream_t stream) {
  const int small_grid = sms * 8;
  thd::attn_bwd_pre_kernel<DT><<<small_grid, 256, 0, stream>>>(bp);
  if (cudaGetLastError() != cudaSuccess) return THD_ERR_CUDA;
  auto kern = thd::attn_bwd_kernel<DT, DP>;
  const size_t smem = one_cta_per_sm(sizeof(thd::BwdSmem<DP>) + 1024);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return THD_ERR_CUDA;
  kern<<<sms, thd::kBwdThreads, smem, stream>>>(mq, mk, mv, mdo, mdq, bp);
  if (cudaGetLastError() != cudaSuccess) return THD_ERR_CUDA;
  thd::attn_bwd_post_kernel<DT><<<small_grid, 256, 0, stream>>>(bp);
  return cudaGetLastError() == cudaSuccess ? THD_OK : THD_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t thd_attn_bwd_workspace_size(int total_tokens, int num_heads_q, int head_dim) {
  if (total_tokens < 0 || num_heads_q < 1 || head_dim < 1) return 0;
  return bwd_workspace_bytes(total_tokens, num_heads_q, head_dim);
}

int thd_attn_bwd_window(const void* q, const void* k, const void* v, const void* out, const float* lse,
                        const void* dout, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                        const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded,
                        const uint8_t* seq_is_causal, int batch_size, int max_seqlen, float softmax_scale, void* dq,
                        void* dk, void* dv, int total_tokens, int num_heads_q, int num_heads_kv, int head_dim,
                        int dtype, int window_left, int window_right, void* workspace, size_t workspace_bytes,
                        void* stream) {
  if (batch_size < 0 || max_seqlen < 0 || total_tokens < 0) return THD_ERR_ARG;
  if (window_left < -1 || window_right < -1) return THD_ERR_ARG;
  if (num_heads_q < 1 || num_heads_kv < 1) return THD_ERR_ARG;
  if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.f)) return THD_ERR_ARG;
  if (dtype != THD_BF16 && dtype != THD_FP16) return THD_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return THD_ERR_UNSUPPORTED;
  if (num_heads_q % num_heads_kv != 0) return THD_ERR_UNSUPPORTED;
  const long long max_items = ((long long)total_tokens / 128 + (long long)batch_size + 1) * num_heads_kv;
  if (max_items >= (1ll << 31)) return THD_ERR_UNSUPPORTED;
  if ((long long)num_heads_q * head_dim * 2 >= (1ll << 31)) return THD_ERR_UNSUPPORTED;
  if (total_tokens == 0) return THD_OK;
  if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv) return THD_ERR_ARG;
  if (batch_size > 0 && (!cu_seqlens_q || !cu_seqlens_kv)) return THD_ERR_ARG;
  const void* a16[] = {q, k, v, out, dout, dq, dk, dv};
  for (const void* ptr : a16)
    if (!aligned(ptr, 16)) return THD_ERR_ARG;
  if (!aligned(lse, 4) || (cu_seqlens_q && !aligned(cu_seqlens_q, 4)) ||
      (cu_seqlens_kv && !aligned(cu_seqlens_kv, 4)) ||
      (cu_seqlens_q_padded && !aligned(cu_seqlens_q_padded, 4)) ||
      (cu_seqlens_kv_padded && !aligned(cu_seqlens_kv_padded, 4)))
    return THD_ERR_ARG;
  if (!workspace || !aligned(workspace, 256) ||
      workspace_bytes < bwd_workspace_bytes(total_tokens, num_heads_q, head_dim))
    return THD_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return THD_ERR_CUDA;

  thd::BwdParams bp;
  std::memset(&bp, 0, sizeof(bp));
  thd::AttnParams& p = bp.a;
  p.q = q;
  p.k = k;
  p.v = v;
  p.cu_q = cu_seqlens_q;
  p.cu_kv = cu_seqlens_kv;
  p.pad_q = cu_seqlens_q_padded;
  p.pad_kv = cu_seqlens_kv_padded;
  p.causal = seq_is_causal;
  p.out = const_cast<void*>(out);
  p.lse = const_cast<float*>(lse);
  p.work_counter = static_cast<unsigned long long*>(workspace);
  p.status = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + 8);
  set_wait_fields(p);
  p.claim = claim_for(max_seqlen, (long long)batch_size * num_heads_kv, sms);
  p.B = batch_size;
  p.T = total_tokens;
  p.Hq = num_heads_q;
  p.Hkv = num_heads_kv;
  p.d = head_dim;
  p.win_left = window_left;
  p.win_right = window_right;
  p.group = num_heads_q / num_heads_kv;
  p.scale = softmax_scale;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  bp.dout = dout;
  bp.dq = dq;
  bp.dk = dk;
  bp.dv = dv;
  char* wsb = static_cast<char*>(workspace);
  bp.D = reinterpret_cast<float*>(wsb + kWorkspaceBytes);
  bp.dacc = reinterpret_cast<float*>(wsb + kWorkspaceBytes + align256((size_t)num_heads_q * total_tokens * 4));

  if (cudaMemsetAsync(workspace, 0, 16, st) != cudaSuccess) return THD_ERR_CUDA;
  const bool bf16 = dtype == THD_BF16;
  CUtensorMap mq, mk, mv, mdo, mdq;
  if (!encode_thd_map(&mq, q, total_tokens, num_heads_q, head_dim, bf16) ||
      !encode_thd_map(&mk, k, total_tokens, num_heads_kv, head_dim, bf16) ||
      !encode_thd_map(&mv, v, total_tokens, num_heads_kv, head_dim, bf16) ||
      !encode_thd_map(&mdo, dout, total_tokens, num_heads_q, head_dim, bf16) ||
      !encode_f32_map(&mdq, bp.dacc, total_tokens, (long long)num_heads_q * head_dim))
    return THD_ERR_CUDA;
  if (bf16) {
    if (head_dim == 128) return launch_bwd<__nv_bfloat16, 128>(mq, mk, mv, mdo, mdq, bp, sms, st);
    return launch_bwd<__nv_bfloat16, 64>(mq, mk, mv, mdo, mdq, bp, sms, st);
  }
  if (head_dim == 128) return launch_bwd<__half, 128>(mq, mk, mv, mdo, mdq, bp, sms, st);
  return launch_bwd<__half, 64>(mq, mk, mv, mdo, mdq, bp, sms, st);
}

int thd_attn_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse, const void* dout,
                 const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, const int32_t* cu_seqlens_q_padded,
                 const int32_t* cu_seqlens_kv_padded, const uint8_t* seq_is_causal, int batch_size, int max_seqlen,
                 float softmax_scale, void* dq, void* dk, void* dv, int total_tokens, int num_heads_q,
                 int num_heads_kv, int head_dim, int dtype, void* workspace, size_t workspace_bytes,
                 void* stream) {
  return thd_attn_bwd_window(q, k, v, out, lse, dout, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                             cu_seqlens_kv_padded, seq_is_causal, batch_size, max_seqlen, softmax_scale, dq, dk, dv,
                             total_tokens, num_heads_q, num_heads_kv, head_dim, dtype, -1, -1, workspace,
                             workspace_bytes, stream);
}


const char* thd_status_string(int status) {
  switch (status) {
    case THD_OK: return "THD_OK";
    case THD_ERR_ARG: return "THD_ERR_ARG: invalid argument";
    case THD_ERR_UNSUPPORTED: return "THD_ERR_UNSUPPORTED: unsupported head_dim, dtype or head layout";
    case THD_ERR_CUDA: return "THD_ERR_CUDA: CUDA call failed";
    case THD_ERR_WORKSPACE: return "THD_ERR_WORKSPACE: workspace missing, too small or misaligned";
    default: return "unknown thd_status";
  }
}

size_t thd_attn_workspace_size(void) { return kWorkspaceBytes; }

uint64_t thd_set_wait_limit_ns(uint64_t ns) {
  return g_wait_limit_ns.exchange(ns == 0 ? thd::kWaitLimitNs : ns);
}

int thd_set_wait_injection(int enable) { return (int)g_inject_wait.exchange(enable ? 1u : 0u); }

int thd_padding_mask(const int32_t* cu_seqlens, int batch_size, int max_seqlen, uint8_t* mask, void* stream) {
  if (batch_size < 0 || max_seqlen < 0) return THD_ERR_ARG;
  if (batch_size == 0 || max_seqlen == 0) return THD_OK;
  if (!cu_seqlens || !mask) return THD_ERR_ARG;
  if (!aligned(cu_seqlens, 4)) return THD_ERR_ARG;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return THD_ERR_CUDA;
  cudaError_t e = thd::launch_padding_mask(cu_seqlens, batch_size, max_seqlen, mask, sms,
                                           static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? THD_OK : THD_ERR_CUDA;
}

int thd_padding_mask_cross(const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, int batch_size,
                           int max_seqlen_q, int max_seqlen_kv, uint8_t* mask_q, uint8_t* mask_kv, void* stream) {
  if (batch_size < 0 || max_seqlen_q < 0 || max_seqlen_kv < 0) return THD_ERR_ARG;
  if (batch_size == 0) return THD_OK;
  if ((max_seqlen_q > 0 && (!cu_seqlens_q || !mask_q)) || (max_seqlen_kv > 0 && (!cu_seqlens_kv || !mask_kv)))
    return THD_ERR_ARG;
  if ((cu_seqlens_q && !aligned(cu_seqlens_q, 4)) || (cu_seqlens_kv && !aligned(cu_seqlens_kv, 4))) return THD_ERR_ARG;
  int st = thd_padding_mask(cu_seqlens_q, batch_size, max_seqlen_q, mask_q, stream);
  if (st != THD_OK) return st;
  return thd_padding_mask(cu_seqlens_kv, batch_size, max_seqlen_kv, mask_kv, stream);
}

int thd_attn_merge(const void* out_a, const float* lse_a, const void* out_b, const float* lse_b, void* out,
                   float* lse, int total_tokens, int num_heads, int head_dim, int dtype, void* stream) {
  if (total_tokens < 0 || num_heads < 1) return THD_ERR_ARG;
  if (dtype != THD_BF16 && dtype != THD_FP16) return THD_ERR_UNSUPPORTED;
  if (head_dim < 8 || head_dim > 128 || head_dim % 8 != 0) return THD_ERR_UNSUPPORTED;
  if ((long long)total_tokens * num_heads >= (1ll << 40)) return THD_ERR_UNSUPPORTED;
  if (total_tokens == 0) return THD_OK;
  if (!out_a || !lse_a || !out_b || !lse_b || !out || !lse) return THD_ERR_ARG;
  if (!aligned(out_a, 16) || !aligned(out_b, 16) || !aligned(out, 16)) return THD_ERR_ARG;
  if (!aligned(lse_a, 4) || !aligned(lse_b, 4) || !aligned(lse, 4)) return THD_ERR_ARG;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return THD_ERR_CUDA;
  cudaError_t e = thd::launch_attn_merge(out_a, lse_a, out_b, lse_b, out, lse, total_tokens, num_heads, head_dim,
                                         dtype == THD_BF16, sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? THD_OK : THD_ERR_CUDA;
}

int thd_attn_fwd_window(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                        const int32_t* cu_seqlens_kv, const int32_t* cu_seqlens_q_padded,
                        const int32_t* cu_seqlens_kv_padded, const uint8_t* seq_is_causal, int batch_size,
                        int max_seqlen, float softmax_scale, void* out, float* lse, int total_tokens,
                        int num_heads_q, int num_heads_kv, int head_dim, int dtype, int window_left,
                        int window_right, void* workspace, size_t workspace_bytes, void* stream) {
  // ---- host-checkable arguments ----
  if (batch_size < 0 || max_seqlen < 0 || total_tokens < 0) return THD_ERR_ARG;
  if (window_left < -1 || window_right < -1) return THD_ERR_ARG;
  if (num_heads_q < 1 || num_heads_kv < 1) return THD_ERR_ARG;
  if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.f)) return THD_ERR_ARG;
  if (dtype != THD_BF16 && dtype != THD_FP16) return THD_ERR_UNSUPPORTED;
  if (head_dim < 8 || head_dim > 128 || head_dim % 8 != 0) return THD_ERR_UNSUPPORTED;
  if (num_heads_q % num_heads_kv != 0) return THD_ERR_UNSUPPORTED;
  // scheduler counters are 32-bit per chunk of sequences
  const long long max_items = ((long long)total_tokens / 128 + (long long)batch_size + 1) * num_heads_q;
  if (max_items >= (1ll << 31)) return THD_ERR_UNSUPPORTED;
  if ((long long)num_heads_q * head_dim * 2 >= (1ll << 31)) return THD_ERR_UNSUPPORTED;
  if (total_tokens == 0) return THD_OK;   // no rows: nothing to write
  if (!q || !k || !v || !out) return THD_ERR_ARG;
  if (batch_size > 0 && (!cu_seqlens_q || !cu_seqlens_kv)) return THD_ERR_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16)) return THD_ERR_ARG;
  if ((lse && !aligned(lse, 4)) || (cu_seqlens_q && !aligned(cu_seqlens_q, 4)) ||
      (cu_seqlens_kv && !aligned(cu_seqlens_kv, 4)) ||
      (cu_seqlens_q_padded && !aligned(cu_seqlens_q_padded, 4)) ||
      (cu_seqlens_kv_padded && !aligned(cu_seqlens_kv_padded, 4)))
    return THD_ERR_ARG;
  if (!workspace || !aligned(workspace, 16) || workspace_bytes < kWorkspaceBytes) return THD_ERR_WORKSPACE;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return THD_ERR_CUDA;

  thd::AttnParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = q;
  p.k = k;
  p.v = v;
  p.cu_q = cu_seqlens_q;
  p.cu_kv = cu_seqlens_kv;
  p.pad_q = cu_seqlens_q_padded;
  p.pad_kv = cu_seqlens_kv_padded;
  p.causal = seq_is_causal;
  p.out = out;
  p.lse = lse;
  p.work_counter = static_cast<unsigned long long*>(workspace);
  p.status = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + 8);
  set_wait_fields(p);
  p.claim = claim_for(max_seqlen, (long long)batch_size * num_heads_q, sms);
  p.B = batch_size;
  p.T = total_tokens;
  p.Hq = num_heads_q;
  p.Hkv = num_heads_kv;
  p.d = head_dim;
  p.win_left = window_left;
  p.win_right = window_right;
  p.group = num_heads_q / num_heads_kv;
  p.scale = softmax_scale;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;

  // work counter and status word start at zero for this call
  if (cudaMemsetAsync(workspace, 0, 16, st) != cudaSuccess) return THD_ERR_CUDA;

  const bool bf16 = dtype == THD_BF16;
  const bool tma = head_dim == 64 || head_dim == 128;
  CUtensorMap mq, mk, mv;
  std::memset(&mq, 0, sizeof(mq));
  std::memset(&mk, 0, sizeof(mk));
  std::memset(&mv, 0, sizeof(mv));
  if (tma) {
    if (!encode_thd_map(&mq, q, total_tokens, num_heads_q, head_dim, bf16) ||
        !encode_thd_map(&mk, k, total_tokens, num_heads_kv, head_dim, bf16) ||
        !encode_thd_map(&mv, v, total_tokens, num_heads_kv, head_dim, bf16))
      return THD_ERR_CUDA;
  }
  const int grid = sms;
  if (bf16) {
    if (head_dim == 128) return launch_ws<__nv_bfloat16, 128>(mq, mk, mv, p, max_seqlen, grid, st);
    if (head_dim == 64) return launch_ws<__nv_bfloat16, 64>(mq, mk, mv, p, max_seqlen, grid, st);
    if (head_dim < 64) return launch_serial<__nv_bfloat16, 64, false>(mq, mk, mv, p, grid, st);
    return launch_serial<__nv_bfloat16, 128, false>(mq, mk, mv, p, grid, st);
  } else {
    if (head_dim == 128) return launch_ws<__half, 128>(mq, mk, mv, p, max_seqlen, grid, st);
    if (head_dim == 64) return launch_ws<__half, 64>(mq, mk, mv, p, max_seqlen, grid, st);
    if (head_dim < 64) return launch_serial<__half, 64, false>(mq, mk, mv, p, grid, st);
    return launch_serial<__half, 128, false>(mq, mk, mv, p, grid, st);
  }
}

int thd_attn_fwd(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                 const int32_t* cu_seqlens_kv, const int32_t* cu_seqlens_q_padded,
                 const int32_t* cu_seqlens_kv_padded, const uint8_t* seq_is_causal, int batch_size,
                 int max_seqlen, float softmax_scale, void* out, float* lse, int total_tokens, int num_heads_q,
                 int num_heads_kv, int head_dim, int dtype, void* workspace, size_t workspace_bytes,
                 void* stream) {
  return thd_attn_fwd_window(q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded,
                             seq_is_causal, batch_size, max_seqlen, softmax_scale, out, lse, total_tokens,
                             num_heads_q, num_heads_kv, head_dim, dtype, -1, -1, workspace, workspace_bytes, stream);
}

}  // extern "C"
