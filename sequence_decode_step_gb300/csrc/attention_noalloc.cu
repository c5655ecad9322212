// qw_attention_decode_noalloc: the decode-attention op for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs while a CUDA graph is
// being captured elsewhere in the process, real-time loops that must not hit
// the allocator, and embedders whose memory is owned by someone else's pool.
// For them the scratch of the split-K attention (per-split partial outputs and
// the per-KV-head arrival counters) lives in one file-scope device array of a
// fixed size instead of a caller-provided workspace. Every GPU that loads this
// library holds that array until the process exits.

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "qw.h"
#include "qw_internal.h"

namespace {

// Fixed scratch: counters (+ error word) padded to 256 bytes, then the split
// partials. 1 MiB covers, e.g., 16 query heads x 125 splits x head_dim 128.
constexpr size_t kNoAllocScratchBytes = 1u << 20;
static __device__ __align__(256) uint8_t g_attn_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];  // device address of g_attn_scratch, per device

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

extern "C" size_t qw_attention_noalloc_max_bytes(void) { return kNoAllocScratchBytes; }

// Failure with qw_last_error(NULL) text, as the other handle-less calls report.
static int fail(int code, const char* msg) {
  qw::set_op_error(msg);
  return code;
}

extern "C" int qw_attention_decode_noalloc(const float* qkv, const uint16_t* q_norm,
                                           const uint16_t* k_norm, float* k_cache, float* v_cache,
                                           int32_t nq, int32_t nkv, int32_t hd, int32_t cap,
                                           int32_t pos, float eps, float rope_theta,
                                           int32_t n_splits, float* out, void* stream) {
  if (!qkv || !k_cache || !v_cache || !out)
    return fail(QW_ERR_ARG, "qw_attention_decode_noalloc: null buffer");
  if ((hd != 64 && hd != 128) || nkv <= 0 || nq <= 0 || nq % nkv ||
      nq / nkv > qw::attention_gq_max() || n_splits <= 0 || n_splits > 65535)
    return fail(QW_ERR_ARG, "qw_attention_decode_noalloc: unsupported shape");
  if (!qw::attention_splits_fit(nq / nkv, hd, n_splits))
    return fail(QW_ERR_ARG,
                "qw_attention_decode_noalloc: n_splits too large for the combine (query heads "
                "per KV head x (n_splits + 1) must fit 192 x head_dim floats)");
  if (pos < 0 || pos >= cap)
    return fail(QW_ERR_ARG, "qw_attention_decode_noalloc: pos outside [0, cap)");
  const size_t head = align256(((size_t)nkv + 1) * 4);
  const size_t ml = align256((size_t)nq * n_splits * 2 * 4);
  const size_t need = head + ml + (size_t)nq * n_splits * hd * 4;
  if (need > kNoAllocScratchBytes)  // shapes beyond the fixed scratch
    return fail(QW_ERR_SIZE,
                "qw_attention_decode_noalloc: the shape needs more scratch than the fixed 1 MiB "
                "array (256 + nq * n_splits * (hd + 2) * 4 bytes, rounded)");

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fail(QW_ERR_CUDA, "qw_attention_decode_noalloc: no current CUDA device (or id >= 64)");
  void* base = nullptr;
  {
    // Set-up, once per device, with that device current: the host-side name of
    // g_attn_scratch is not a device address, so ask the runtime for it.
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || p == nullptr)
        return fail(QW_ERR_CUDA, "qw_attention_decode_noalloc: cudaGetSymbolAddress failed");
      if (qw::set_kernel_attributes() != cudaSuccess)
        return fail(QW_ERR_CUDA, "qw_attention_decode_noalloc: setting kernel attributes failed");
      g_scratch_ptr[dev] = p;
    }
    base = g_scratch_ptr[dev];
  }
  cudaStream_t s = (cudaStream_t)stream;
  // The arrival counters and the error word must start at zero; the partials
  // are fully written by the kernel before they are read.
  if (cudaMemsetAsync(base, 0, head, s) != cudaSuccess)
    return fail(QW_ERR_CUDA, "qw_attention_decode_noalloc: clearing the counters failed");

  uint8_t* ws = (uint8_t*)base;
  qw::AttnArgs t{};
  t.qkv = qkv;
  t.q_norm = q_norm;
  t.k_norm = k_norm;
  t.rope = nullptr;
  t.rope_theta = rope_theta;
  t.k_cache = k_cache;
  t.v_cache = v_cache;
  t.cap = cap;
  t.pos_ptr = nullptr;
  t.pos_const = pos;
  t.nq = nq;
  t.nkv = nkv;
  t.eps = eps;
  t.nsplit_max = n_splits;
  t.min_keys = 32;
  t.counters = (int*)ws;
  t.err = (int*)ws + nkv;
  t.part_ml = (float*)(ws + head);
  t.part_o = (float*)(ws + head + ml);
  t.out = out;
  t.wait_ns = 1000000000ull;
  if (qw::launch_attention(t, hd, false, s) != cudaSuccess)
    return fail(QW_ERR_CUDA, "qw_attention_decode_noalloc: kernel launch failed");
  return QW_OK;
}
