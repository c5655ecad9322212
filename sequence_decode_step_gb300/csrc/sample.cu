// On-device sampling from one logits row: temperature, top-k and top-p (nucleus),
// with the uniform draw supplied by the caller ("flashmoon demo" README: greedy
// plus temperature/top-k/top-p sampling, temp = 0 meaning greedy; its sampling
// reads the whole logits row back to the host every token). Here the row never
// leaves the device; only the chosen id does.
//
// Selection of the top k (ties to the lower index) in three levels, each a sort
// of (key, index) pairs in shared memory:
//   level 1: one CTA per 1024-logit slice keeps the slice's best k, sorted;
//   level 2: one CTA per 16 slices keeps the best k of their 16 k candidates;
//   level 3: one CTA keeps the best k of all level-2 lists and draws the token.
// A 64-bit sort key (order-preserving float key << 32 | ~index) makes every
// comparison total, so the chosen set and its order are the same on every run.
// The draw is in f64: weights exp((l_i - l_0) / T) in candidate order, the
// nucleus is the shortest prefix whose running sum reaches top_p of the total,
// and the token is the first candidate of the nucleus whose running sum exceeds
// u times the nucleus total.

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "qw_internal.h"

namespace qw {
namespace {

constexpr int kSlice = 1024;   // logits per level-1 CTA
constexpr int kFan = 16;       // level-1 lists per level-2 CTA
constexpr int kSortMax = 4096; // largest in-CTA sort (level 2 and 3)

// Larger float -> larger key; NaN (any sign) above +inf, so a NaN anywhere in
// the row reaches the final level and is reported.
__device__ __forceinline__ uint32_t fkey(float f) {
  const uint32_t b = __float_as_uint(f);
  if (f != f) return 0xffffffffu;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ uint64_t pack(float f, uint32_t idx) {
  return ((uint64_t)fkey(f) << 32) | (uint32_t)~idx;
}
__device__ __forceinline__ uint32_t unpack_idx(uint64_t p) { return ~(uint32_t)p; }
__device__ __forceinline__ float unpack_val(uint64_t p) {
  const uint32_t k = (uint32_t)(p >> 32);
  if (k == 0xffffffffu) return __int_as_float(0x7fc00000);
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// In-place bitonic sort of n (a power of two) 64-bit keys in shared memory,
// largest first, by all threads of the block (a power-of-two warp count). Warp w
// owns the compare-exchange pairs [wP, (w+1)P): a stage whose stride is at most P
// touches only that warp's elements and needs no block barrier, so only the few
// wide stages pay one (__syncthreads before and after them).
__device__ void sort_desc(uint64_t* s, int n) {
  const int nw = blockDim.x >> 5, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = max(1, (n / 2) / nw);
  const int p0 = min(n / 2, w * P), p1 = min(n / 2, p0 + P);
  bool synced = true;  // the caller synchronised the block before the call
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const bool local = stride <= P;
      if (!local && !synced) __syncthreads();
      for (int i = p0 + lane; i < p1; i += 32) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t a = s[lo], b = s[hi];
        if ((a < b) == desc) {
          s[lo] = b;
          s[hi] = a;
        }
      }
      if (local) {
        __syncwarp();
        synced = false;
      } else {
        __syncthreads();
        synced = true;
      }
    }
  }
  if (!synced) __syncthreads();
}

__device__ __forceinline__ int pow2_at_least(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

// Level 1: slice b of the row, its best k (padding keys are 0, below every logit).
__global__ void __launch_bounds__(256) sample_l1_kernel(const float* __restrict__ logits, int V,
                                                       int k, uint64_t* __restrict__ out) {
  __shared__ uint64_t s[kSlice];
  const int b = blockIdx.x, base = b * kSlice;
  for (int i = threadIdx.x; i < kSlice; i += blockDim.x) {
    const int g = base + i;
    s[i] = g < V ? pack(__ldg(logits + g), (uint32_t)g) : 0ull;
  }
  __syncthreads();
  sort_desc(s, kSlice);
  for (int i = threadIdx.x; i < k; i += blockDim.x) out[(size_t)b * k + i] = s[i];
}

// Level 2: the best k of up to kFan level-1 lists.
__global__ void __launch_bounds__(1024) sample_l2_kernel(const uint64_t* __restrict__ in, int n_lists,
                                                        int k, uint64_t* __restrict__ out) {
  extern __shared__ uint64_t s2[];
  const int b = blockIdx.x;
  const int l0 = b * kFan, nl = min(kFan, n_lists - l0);
  const int n = pow2_at_least(kFan * k);
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    s2[i] = i < nl * k ? in[(size_t)l0 * k + i] : 0ull;
  __syncthreads();
  sort_desc(s2, n);
  for (int i = threadIdx.x; i < k; i += blockDim.x) out[(size_t)b * k + i] = s2[i];
}

// Level 3: the best k of all level-2 lists, then the draw (thread 0 walks the
// running sums in candidate order, as the definition reads).
__global__ void __launch_bounds__(1024) sample_l3_kernel(const uint64_t* __restrict__ in, int n_lists,
                                                        int k, float temperature, float top_p,
                                                        float u, int32_t* __restrict__ token) {
  extern __shared__ uint64_t s3[];
  __shared__ double w[kMaxSampleTopK];
  const int n = pow2_at_least(n_lists * k);
  for (int i = threadIdx.x; i < n; i += blockDim.x) s3[i] = i < n_lists * k ? in[i] : 0ull;
  __syncthreads();
  sort_desc(s3, n);
  const float l0 = unpack_val(s3[0]);
  const bool bad = (l0 != l0) || l0 == -INFINITY;  // a NaN in the row, or nothing finite
  const bool greedy = !(temperature > 0.f) || k == 1;
  if (!bad && !greedy) {
    const double t = (double)temperature;
    for (int i = threadIdx.x; i < k; i += blockDim.x)
      w[i] = exp(((double)unpack_val(s3[i]) - (double)l0) / t);
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  if (bad) {
    *token = -1;
    return;
  }
  if (greedy) {
    *token = (int32_t)unpack_idx(s3[0]);
    return;
  }
  // running sums in candidate order (kept in w), then the two searches
  double run = 0.0;
  for (int i = 0; i < k; ++i) {
    run += w[i];
    w[i] = run;
  }
  // nucleus: the shortest prefix whose running sum reaches top_p * total
  const double need = (double)top_p * run;
  int cut = k - 1;
  for (int i = 0; i < k; ++i)
    if (w[i] >= need) {
      cut = i;
      break;
    }
  const double target = (double)u * w[cut];
  int pick = cut;
  for (int i = 0; i <= cut; ++i)
    if (w[i] > target) {
      pick = i;
      break;
    }
  *token = (int32_t)unpack_idx(s3[pick]);
}

}  // namespace

static int pow2_host(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

int sample_levels(int V, int* n1, int* n2) {
  *n1 = (V + kSlice - 1) / kSlice;
  *n2 = (*n1 + kFan - 1) / kFan;
  return 0;
}

size_t sample_workspace_bytes(int V, int k) {
  int n1, n2;
  sample_levels(V, &n1, &n2);
  return ((size_t)n1 + n2) * (size_t)k * 8;
}

bool sample_shape_ok(int V, int k) {
  int n1, n2;
  sample_levels(V, &n1, &n2);
  return V >= 1 && k >= 1 && k <= kMaxSampleTopK && (size_t)n2 * k <= (size_t)kSortMax;
}

cudaError_t set_sample_attributes() {
  cudaError_t e = cudaFuncSetAttribute(sample_l2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSortMax * 8);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(sample_l3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSortMax * 8);
  return e;
}

cudaError_t launch_sample(const float* logits, int V, int k, float temperature, float top_p, float u,
                          int32_t* token, void* workspace, cudaStream_t s) {
  int n1, n2;
  sample_levels(V, &n1, &n2);
  k = k < V ? k : V;
  uint64_t* w1 = (uint64_t*)workspace;
  uint64_t* w2 = w1 + (size_t)n1 * k;
  sample_l1_kernel<<<n1, 256, 0, s>>>(logits, V, k, w1);
  const size_t smem2 = (size_t)pow2_host(kFan * k) * 8;
  sample_l2_kernel<<<n2, 1024, smem2, s>>>(w1, n1, k, w2);
  const size_t smem3 = (size_t)pow2_host(n2 * k) * 8;
  sample_l3_kernel<<<1, 1024, smem3, s>>>(w2, n2, k, temperature, top_p, u, token);
  return cudaGetLastError();
}

}  // namespace qw
