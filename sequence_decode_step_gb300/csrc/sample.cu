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

#include <algorithm>

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

// Bitonic sort, largest first, of n = E * blockDim.x 64-bit keys held E per
// thread in registers (thread t holds elements t*E .. t*E+E-1). A stage of
// stride s exchanges element i with i ^ s: inside the thread when s < E, with a
// lane of the same warp by shuffle when s < 32 E, and through shared memory `x`
// (n keys) only for the few wider stages. Element i keeps the larger key of its
// pair when it is the lower index of a descending block or the upper index of
// an ascending one.
template <int E>
__device__ void sort_regs(uint64_t (&v)[E], uint64_t* x, int n) {
  const int t = threadIdx.x;
  for (int size = 2; size <= n; size <<= 1) {
    for (int st = size >> 1; st > 0; st >>= 1) {
      if (st < E) {
#pragma unroll
        for (int sc = 1; sc < E; sc <<= 1) {  // the stride as a compile-time value,
          if (sc != st) continue;              // so v stays in registers
#pragma unroll
          for (int r = 0; r < E; ++r) {
            const int pr = r ^ sc;
            if (pr > r) {
              const int i = t * E + r;
              const bool desc = (i & size) == 0;  // r is the lower index of the pair
              const uint64_t a = v[r], b = v[pr];
              const bool swap = desc ? (a < b) : (a > b);
              v[r] = swap ? b : a;
              v[pr] = swap ? a : b;
            }
          }
        }
      } else if (st < 32 * E) {
        const int lm = st / E;  // partner lane distance
#pragma unroll
        for (int r = 0; r < E; ++r) {
          const int i = t * E + r;
          const uint64_t o = __shfl_xor_sync(0xffffffffu, v[r], lm);
          const bool keep_max = ((i & size) == 0) == ((i & st) == 0);
          v[r] = keep_max ? (v[r] > o ? v[r] : o) : (v[r] < o ? v[r] : o);
        }
      } else {
#pragma unroll
        for (int r = 0; r < E; ++r) x[t * E + r] = v[r];
        __syncthreads();
#pragma unroll
        for (int r = 0; r < E; ++r) {
          const int i = t * E + r;
          const uint64_t o = x[i ^ st];
          const bool keep_max = ((i & size) == 0) == ((i & st) == 0);
          v[r] = keep_max ? (v[r] > o ? v[r] : o) : (v[r] < o ? v[r] : o);
        }
        __syncthreads();
      }
    }
  }
}

__device__ __forceinline__ int pow2_at_least(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

// Level 1: slice b of the row (4 logits per thread), its best k (padding keys are
// 0, below every logit).
__global__ void __launch_bounds__(256) sample_l1_kernel(const float* __restrict__ logits, int V,
                                                       int k, uint64_t* __restrict__ out) {
  __shared__ uint64_t x[kSlice];
  const int b = blockIdx.x, i0 = b * kSlice + threadIdx.x * 4;
  uint64_t v[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int g = i0 + r;
    v[r] = g < V ? pack(__ldg(logits + g), (uint32_t)g) : 0ull;
  }
  sort_regs<4>(v, x, kSlice);
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = threadIdx.x * 4 + r;
    if (i < k) out[(size_t)b * k + i] = v[r];
  }
}

// Best k of `cnt` keys at `in` into out[0, k), sorted (1024 E >= cnt keys, the
// rest padded with 0; 1024 threads; x is the sort's exchange space).
template <int E>
__device__ void top_k_block(const uint64_t* __restrict__ in, int cnt, int k, uint64_t* x,
                            uint64_t* __restrict__ out) {
  uint64_t v[E];
#pragma unroll
  for (int r = 0; r < E; ++r) {
    const int i = threadIdx.x * E + r;
    v[r] = i < cnt ? in[i] : 0ull;
  }
  sort_regs<E>(v, x, E * blockDim.x);
#pragma unroll
  for (int r = 0; r < E; ++r) {
    const int i = threadIdx.x * E + r;
    if (i < k) out[i] = v[r];
  }
}

// Level 2: the best k of up to kFan level-1 lists.
__global__ void __launch_bounds__(1024) sample_l2_kernel(const uint64_t* __restrict__ in, int n_lists,
                                                        int k, uint64_t* __restrict__ out) {
  extern __shared__ uint64_t s2[];
  const int b = blockIdx.x;
  const int l0 = b * kFan, nl = min(kFan, n_lists - l0);
  const int n = max(1024, pow2_at_least(kFan * k));
  const uint64_t* src = in + (size_t)l0 * k;
  uint64_t* dst = out + (size_t)b * k;
  if (n == 1024) top_k_block<1>(src, nl * k, k, s2, dst);
  else if (n == 2048) top_k_block<2>(src, nl * k, k, s2, dst);
  else top_k_block<4>(src, nl * k, k, s2, dst);
}

// Level 3: the best k of all level-2 lists, then the draw (thread 0 walks the
// running sums in candidate order, as the definition reads).
__global__ void __launch_bounds__(1024) sample_l3_kernel(const uint64_t* __restrict__ in, int n_lists,
                                                        int k, float temperature, float top_p,
                                                        float u, int32_t* __restrict__ token) {
  extern __shared__ uint64_t s3[];  // [n] exchange space, then the k candidates
  __shared__ double w[kMaxSampleTopK];
  __shared__ uint64_t cand[kMaxSampleTopK];
  const int n = max(1024, pow2_at_least(n_lists * k));
  if (n == 1024) top_k_block<1>(in, n_lists * k, k, s3, cand);
  else if (n == 2048) top_k_block<2>(in, n_lists * k, k, s3, cand);
  else top_k_block<4>(in, n_lists * k, k, s3, cand);
  __syncthreads();
  uint64_t* s3c = cand;
  const float l0 = unpack_val(s3c[0]);
  const bool bad = (l0 != l0) || l0 == -INFINITY;  // a NaN in the row, or nothing finite
  const bool greedy = !(temperature > 0.f) || k == 1;
  if (!bad && !greedy) {
    const double t = (double)temperature;
    for (int i = threadIdx.x; i < k; i += blockDim.x)
      w[i] = exp(((double)unpack_val(s3c[i]) - (double)l0) / t);
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  if (bad) {
    *token = -1;
    return;
  }
  if (greedy) {
    *token = (int32_t)unpack_idx(s3c[0]);
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
  *token = (int32_t)unpack_idx(s3c[pick]);
}

}  // namespace

static int pow2_host(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

// CTAs of levels 1 and 2 for a row of V logits.
static void sample_levels(int V, int* n1, int* n2) {
  *n1 = (V + kSlice - 1) / kSlice;
  *n2 = (*n1 + kFan - 1) / kFan;
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
  const size_t smem2 = (size_t)std::max(1024, pow2_host(kFan * k)) * 8;
  sample_l2_kernel<<<n2, 1024, smem2, s>>>(w1, n1, k, w2);
  const size_t smem3 = (size_t)std::max(1024, pow2_host(n2 * k)) * 8;
  sample_l3_kernel<<<1, 1024, smem3, s>>>(w2, n2, k, temperature, top_p, u, token);
  return cudaGetLastError();
}

}  // namespace qw
