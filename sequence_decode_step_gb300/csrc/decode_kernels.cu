// Decode-step kernels for sm_103a (GB300).
//
// Every kernel of the step follows one pattern:
//   1. prefetch what does not depend on the previous kernel (its weight slice,
//      or the KV rows written by earlier steps) into shared memory with bulk
//      TMA copies (cp.async.bulk) completing on an mbarrier;
//   2. griddepcontrol.launch_dependents, so the next kernel of the CUDA graph
//      can already start its own prefetch;
//   3. griddepcontrol.wait, then read the activations and compute.
// The HBM stream therefore does not drain between the kernels of a step.
// Every wait on an mbarrier is bounded by %globaltimer; on expiry the kernel
// sets ERR_TIMEOUT in the device error word, waits (again bounded) for its
// copies in flight and leaves without hanging.

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "qw_internal.h"
#include "qw_ptx.cuh"

namespace qw {


// Reduce (best_v, best_i) over the 256 threads; result valid in thread 0.
__device__ __forceinline__ void block_argmax_256(float& bv, int& bi, float* r8, int* r8i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (am_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) { r8[warp] = bv; r8i[warp] = bi; }
  __syncthreads();
  if (threadIdx.x == 0) {
    bv = r8[0];
    bi = r8i[0];
    for (int i = 1; i < 8; ++i)
      if (am_better(r8[i], r8i[i], bv, bi)) { bv = r8[i]; bi = r8i[i]; }
  }
}

// ------------------------------------------------------------------ GEMV
// y = epi(W . pro(x)) for M = 1. CTA b owns output units [n*b/G, n*(b+1)/G),
// whose weight rows are one contiguous byte range; it streams that range
// through `n_stages` shared-memory stages with bulk copies. Warps are split
// into `ks` K-slices (the input slice stays in registers) and 8/ks row groups.
template <int EPI, int MAXC, int WF>
__global__ void __launch_bounds__(256, 1) gemv_kernel(const GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  float* red8 = reinterpret_cast<float*>(smem + 64);
  int* red8i = reinterpret_cast<int*>(smem + 96);
  float* red = reinterpret_cast<float*>(smem + a.off_red);
  float* xs = reinterpret_cast<float*>(smem + a.off_x);
  uint8_t* stages = smem + a.off_stage;
  __shared__ int s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, b = blockIdx.x;
  const int u_begin = (int)(((long long)a.n_units * b) / G);
  const int u_end = (int)(((long long)a.n_units * (b + 1)) / G);
  const int n_my = u_end - u_begin;
  const int ups = a.units_per_stage;
  const int n_chunks = (n_my + ups - 1) / ups;
  const uint32_t unit_bytes = (uint32_t)a.rpu * a.row_bytes;
  const int NS = a.n_stages;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
    const int pre = n_chunks < NS ? n_chunks : NS;
    for (int c = 0; c < pre; ++c) {
      const int nu = min(ups, n_my - c * ups);
      mbar_expect_tx(&bars[c], nu * unit_bytes);
      bulk_load(stages + (size_t)c * a.stage_bytes,
                a.w + (size_t)(u_begin + c * ups) * unit_bytes, nu * unit_bytes, &bars[c]);
    }
  }
  // Weights are in flight; let the next kernel start, then wait for our inputs.
  pdl_launch_dependents();
  pdl_wait();

  // Prologue: input vector into shared memory, optional RMSNorm.
  const int K = a.K;
  float ss = 0.f;
  for (int k = tid * 4; k < K; k += 256 * 4) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(a.x + k));
    *reinterpret_cast<float4*>(xs + k) = v;
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
  }
  if (a.norm_g != nullptr) {
    const float tot = block_sum_256(ss, red8);
    const float r = 1.0f / sqrtf(tot / (float)K + a.eps);
    for (int k = tid * 4; k < K; k += 256 * 4) {
#pragma unroll
      for (int e = 0; e < 4; ++e) xs[k + e] = xs[k + e] * r * bf16f(a.norm_g[k + e]);
    }
  }
  __syncthreads();
  if (a.norm_out != nullptr && b == 0) {
    const int row = a.pos ? *a.pos : 0;
    for (int k = tid; k < K; k += 256) a.norm_out[(size_t)row * K + k] = xs[k];
  }

  const int ksz = a.ks, kslice = warp % ksz, grp = warp / ksz, ngrp = 8 / ksz;
  const int nch = (K + 255) >> 8;
  const int c_lo = kslice * a.cpw;
  const int c_hi = min(nch, c_lo + a.cpw);
  float xr[MAXC][8];
#pragma unroll
  for (int c = 0; c < MAXC; ++c) {
    const int col = (c_lo + c) * 256 + lane * 8;
    const bool on = (c_lo + c < c_hi) && col < K;
#pragma unroll
    for (int e = 0; e < 8; ++e) xr[c][e] = on ? xs[col + e] : 0.f;
  }

  float best_v = -INFINITY;
  int best_i = 0x7fffffff;
  int saw_nan = 0;
  int c = 0;
  bool failed = false;
  const int cap_row = (a.cap_out != nullptr && a.pos != nullptr) ? *a.pos : 0;
  for (; c < n_chunks; ++c) {
    const int st = c % NS;
    const bool ok = mbar_wait(&bars[st], (uint32_t)((c / NS) & 1), a.wait_ns);
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    const int nu = min(ups, n_my - c * ups);
    const int nrows = nu * a.rpu;
    const uint8_t* sw = stages + (size_t)st * a.stage_bytes;
    for (int r0 = grp * 2; r0 < nrows; r0 += ngrp * 2) {
      const bool two = r0 + 1 < nrows;
      const uint8_t* w0 = sw + (size_t)r0 * a.row_bytes;
      const uint8_t* w1 = w0 + a.row_bytes;
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int cc = 0; cc < MAXC; ++cc) {
        const int col = (c_lo + cc) * 256 + lane * 8;
        if ((c_lo + cc < c_hi) && col < K) {
          if (WF == 1) {  // 8 nibbles (4 bytes) and the scale of their 128-wide group
            const uint32_t so = a.scale_off + (uint32_t)(col >> 7) * 2;
            acc0 = dot8_i4(*reinterpret_cast<const uint32_t*>(w0 + col / 2), xr[cc],
                           bf16f(*reinterpret_cast<const uint16_t*>(w0 + so)), acc0);
            if (two)
              acc1 = dot8_i4(*reinterpret_cast<const uint32_t*>(w1 + col / 2), xr[cc],
                             bf16f(*reinterpret_cast<const uint16_t*>(w1 + so)), acc1);
          } else if (WF == 2) {  // 8 int8 (8 bytes) and the fp16 scale of their 32-wide block
            const uint32_t so = a.scale_off + (uint32_t)(col >> 5) * 2;
            acc0 = dot8_i8(*reinterpret_cast<const uint2*>(w0 + col), xr[cc],
                           __half2float(*reinterpret_cast<const __half*>(w0 + so)), acc0);
            if (two)
              acc1 = dot8_i8(*reinterpret_cast<const uint2*>(w1 + col), xr[cc],
                             __half2float(*reinterpret_cast<const __half*>(w1 + so)), acc1);
          } else {
            acc0 = dot8(*reinterpret_cast<const uint4*>(w0 + (size_t)col * 2), xr[cc], acc0);
            if (two)
              acc1 = dot8(*reinterpret_cast<const uint4*>(w1 + (size_t)col * 2), xr[cc], acc1);
          }
        }
      }
      acc0 = warp_sum(acc0);
      acc1 = warp_sum(acc1);
      if (lane == 0) {
        red[r0 * ksz + kslice] = acc0;
        if (two) red[(r0 + 1) * ksz + kslice] = acc1;
      }
    }
    __syncthreads();
    for (int t = tid; t < nu; t += 256) {
      const int u = u_begin + c * ups + t;
      float v0 = 0.f;
      for (int q = 0; q < ksz; ++q) v0 += red[(t * a.rpu) * ksz + q];
      if (EPI == EPI_STORE) {
        float v = v0 + (a.bias ? bf16f(a.bias[u]) : 0.f);
        if (a.lora_bq != nullptr) {  // low-rank update on the q and v rows
          const uint16_t* brow = nullptr;
          const float* t = nullptr;
          if (u < a.lora_q_rows) {
            brow = a.lora_bq + (size_t)u * a.lora_r;
            t = a.lora_t;
          } else if (u >= a.lora_v_row0 && u < a.lora_v_row0 + a.lora_v_rows) {
            brow = a.lora_bv + (size_t)(u - a.lora_v_row0) * a.lora_r;
            t = a.lora_t + a.lora_r;
          }
          if (brow) {
            float d = 0.f;
            for (int j = 0; j < a.lora_r; ++j) d = fmaf(bf16f(brow[j]), __ldcg(t + j), d);
            v = fmaf(a.lora_scale, d, v);
          }
        }
        a.y[u] = v;
      } else if (EPI == EPI_RESIDUAL) {
        const float nv = __ldcg(a.y + u) + v0;
        a.y[u] = nv;
        if (a.cap_out) a.cap_out[(size_t)cap_row * a.n_units + u] = nv;
      } else if (EPI == EPI_SWIGLU) {
        float v1 = 0.f;
        for (int q = 0; q < ksz; ++q) v1 += red[(t * 2 + 1) * ksz + q];
        a.y[u] = v0 / (1.0f + expf(-v0)) * v1;
      } else {  // EPI_LOGITS
        a.y[u] = v0;
        if (v0 != v0) saw_nan = 1;
        else if (v0 > best_v) { best_v = v0; best_i = u; }
      }
    }
    __syncthreads();
    if (tid == 0 && c + NS < n_chunks) {
      const int cn = c + NS;
      const int nun = min(ups, n_my - cn * ups);
      mbar_expect_tx(&bars[st], nun * unit_bytes);
      bulk_load(stages + (size_t)st * a.stage_bytes,
                a.w + (size_t)(u_begin + cn * ups) * unit_bytes, nun * unit_bytes, &bars[st]);
    }
  }
  if (failed) {
    if (tid == 0) {
      atomicOr(a.err, ERR_TIMEOUT);
      const int hi = min(n_chunks, c + NS);
      for (int cc = c; cc < hi; ++cc)
        mbar_wait(&bars[cc % NS], (uint32_t)((cc / NS) & 1), kDrainNs);
    }
    __syncthreads();
  }
  if (EPI != EPI_LOGITS) return;

  // ---- greedy argmax: CTA best, then the last CTA to arrive reduces all of them.
  const int any_nan = __syncthreads_or(saw_nan);
  block_argmax_256(best_v, best_i, red8, red8i);
  if (tid == 0) {
    a.am.blk_val[b] = any_nan ? __int_as_float(0x7fc00000) : best_v;
    a.am.blk_idx[b] = best_i;
    __threadfence();
    const int prev = atomicAdd(a.am.counter, 1);
    s_last = (prev == G - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  int nan_seen = 0;
  for (int i = tid; i < G; i += 256) {
    const float v = __ldcg(a.am.blk_val + i);
    const int ix = __ldcg(a.am.blk_idx + i);
    if (v != v) nan_seen = 1;
    else if (am_better(v, ix, bv, bi)) { bv = v; bi = ix; }
  }
  nan_seen = __syncthreads_or(nan_seen);
  block_argmax_256(bv, bi, red8, red8i);
  if (tid == 0) {
    const int am = nan_seen ? -1 : bi;
    if (nan_seen) atomicOr(a.err, ERR_NAN);
    if (a.am.argmax) *a.am.argmax = am;
    if (a.am.next_token) *a.am.next_token = am;
    if (a.am.pos) {
      const int p = *a.am.pos;
      if (a.am.tokens_by_pos) a.am.tokens_by_pos[p] = am;
      *a.am.pos = p + 1;
    }
    if (a.am.status) {
      a.am.status[0] = am;
      a.am.status[1] = *reinterpret_cast<volatile int*>(a.err);
    }
    *a.am.counter = 0;
  }
}

void plan_gemv(GemvArgs& a, int grid, uint32_t max_stage_bytes, int max_stages) {
  const int nch = (a.K + 255) / 256;
  int ks = 1;
  while (ks < 8 && (nch + ks - 1) / ks > 4) ks *= 2;
  a.ks = ks;
  a.cpw = (nch + ks - 1) / ks;
  const uint32_t unit_bytes = (uint32_t)a.rpu * a.row_bytes;
  const int units_max = (a.n_units + grid - 1) / grid;
  if ((uint64_t)units_max * unit_bytes <= max_stage_bytes) {
    a.units_per_stage = units_max;
    a.n_stages = 1;
  } else {
    int ups = (int)(max_stage_bytes / unit_bytes);
    if (ups < 1) ups = 1;
    a.units_per_stage = ups;
    const int chunks = (units_max + ups - 1) / ups;
    a.n_stages = chunks < max_stages ? chunks : max_stages;
  }
  a.stage_bytes = (uint32_t)a.units_per_stage * unit_bytes;
  a.off_red = 128;
  const uint32_t red_bytes = (uint32_t)a.units_per_stage * a.rpu * a.ks * 4;
  a.off_x = (a.off_red + red_bytes + 15) & ~15u;
  a.off_stage = (a.off_x + (uint32_t)a.K * 4 + 127) & ~127u;
}

size_t gemv_smem_bytes(const GemvArgs& a) {
  return (size_t)a.off_stage + (size_t)a.n_stages * a.stage_bytes;
}

template <class Kern, class... Args>
static cudaError_t launch_ex(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int EPI>
static cudaError_t launch_gemv_epi(const GemvArgs& a, int grid, bool pdl, cudaStream_t s) {
  const size_t smem = gemv_smem_bytes(a);
  if (a.wfmt == 1) {
    if (a.cpw <= 4) return launch_ex(gemv_kernel<EPI, 4, 1>, dim3(grid), dim3(256), smem, s, pdl, a);
    if (a.cpw <= 8) return launch_ex(gemv_kernel<EPI, 8, 1>, dim3(grid), dim3(256), smem, s, pdl, a);
    return cudaErrorInvalidValue;
  }
  if (a.wfmt == 2) {
    if (a.cpw <= 4) return launch_ex(gemv_kernel<EPI, 4, 2>, dim3(grid), dim3(256), smem, s, pdl, a);
    if (a.cpw <= 8) return launch_ex(gemv_kernel<EPI, 8, 2>, dim3(grid), dim3(256), smem, s, pdl, a);
    return cudaErrorInvalidValue;
  }
  if (a.cpw <= 4) return launch_ex(gemv_kernel<EPI, 4, 0>, dim3(grid), dim3(256), smem, s, pdl, a);
  if (a.cpw <= 8) return launch_ex(gemv_kernel<EPI, 8, 0>, dim3(grid), dim3(256), smem, s, pdl, a);
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemv(int epi, const GemvArgs& a, int grid, bool pdl, cudaStream_t s) {
  if (gemv_smem_bytes(a) > 227 * 1024) return cudaErrorInvalidValue;
  switch (epi) {
    case EPI_STORE: return launch_gemv_epi<EPI_STORE>(a, grid, pdl, s);
    case EPI_RESIDUAL: return launch_gemv_epi<EPI_RESIDUAL>(a, grid, pdl, s);
    case EPI_SWIGLU: return launch_gemv_epi<EPI_SWIGLU>(a, grid, pdl, s);
    case EPI_LOGITS: return launch_gemv_epi<EPI_LOGITS>(a, grid, pdl, s);
  }
  return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------ attention (decode)
// One CTA per (key split, KV head). The KV rows of earlier positions are fixed,
// so they are prefetched before the dependency wait; the device position is
// read there too (only the last kernel of a step changes it). After the wait
// the CTA forms its group's queries (QK-RMSNorm, RoPE, 1/sqrt(hd)); the CTA
// whose split holds `pos` also forms k and v, appends them to the cache and
// patches its staged tile. Scores and an online softmax run tile by tile; the
// last CTA of a KV head to finish combines the splits in split order.
constexpr int kAttnTK = 32;
constexpr int kAttnNS = 3;
constexpr int kAttnGQ = 8;

template <int HD>
__host__ __device__ constexpr uint32_t attn_stage_off() {
  return (64u + 4u * (kAttnGQ * HD + 2 * HD + 2 * kAttnGQ * kAttnTK + 3 * kAttnGQ + 4) + 127u) &
         ~127u;
}
template <int HD>
__host__ __device__ constexpr uint32_t attn_smem() {
  return attn_stage_off<HD>() + (uint32_t)kAttnNS * 2u * kAttnTK * HD * 4u;
}

__device__ __forceinline__ void rope_cs(const float2* row, int pos, int j, int hd, float theta,
                                        float& c, float& s) {
  if (row != nullptr) {
    const float2 v = row[j];
    c = v.x;
    s = v.y;
  } else {
    const double inv = pow((double)theta, -2.0 * (double)j / (double)hd);
    double sd, cd;
    sincos((double)pos * inv, &sd, &cd);
    c = (float)cd;
    s = (float)sd;
  }
}

template <int HD, bool KB>
__global__ void __launch_bounds__(256, 1) attn_decode_kernel(const AttnArgs a) {
  constexpr int TK = kAttnTK, NS = kAttnNS, GQM = kAttnGQ, EPL = HD / 32;
  using KV = KvElem<KB>;
  using KT = typename KV::T;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  float* q_s = reinterpret_cast<float*>(smem + 64);  // [GQM][HD]
  float* kn_s = q_s + GQM * HD;                       // [HD]
  float* vn_s = kn_s + HD;                            // [HD]
  float* sc_s = vn_s + HD;                            // [GQM][TK]
  float* p_s = sc_s + GQM * TK;                       // [GQM][TK]
  float* ml_s = p_s + GQM * TK;                       // [GQM][2]
  float* al_s = ml_s + 2 * GQM;                       // [GQM]
  int* flag_s = reinterpret_cast<int*>(al_s + GQM);
  uint8_t* stage_base = smem + attn_stage_off<HD>();
  float* stage0 = reinterpret_cast<float*>(stage_base);  // the combine reuses the stages as f32

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y, s = blockIdx.x;
  const int GQ = a.nq / a.nkv;
  // Read before the dependency wait: only the last kernel of a step writes it.
  const int pos = a.pos_ptr ? *a.pos_ptr : a.pos_const;
  const int n_keys = pos + 1;
  int kps = (n_keys + a.nsplit_max - 1) / a.nsplit_max;
  kps = kps > a.min_keys ? kps : a.min_keys;
  kps = (kps + TK - 1) / TK * TK;
  const int nsplit = (n_keys + kps - 1) / kps;
  if (s >= nsplit) return;
  const int k0 = s * kps;
  const int k1 = min(n_keys, k0 + kps);
  const int ntiles = (k1 - k0 + TK - 1) / TK;
  const bool owns_pos = pos >= k0 && pos < k1;
  KT* kc = reinterpret_cast<KT*>(a.k_cache) + (size_t)g * a.cap * HD;
  KT* vc = reinterpret_cast<KT*>(a.v_cache) + (size_t)g * a.cap * HD;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
    const int pre = ntiles < NS ? ntiles : NS;
    for (int i = 0; i < pre; ++i) {
      const int t0 = k0 + i * TK, nk = min(TK, k1 - t0);
      const uint32_t bytes = (uint32_t)(nk * HD * sizeof(KT));
      KT* dK = reinterpret_cast<KT*>(stage_base) + (size_t)i * 2 * TK * HD;
      mbar_expect_tx(&bars[i], 2 * bytes);
      bulk_load(dK, kc + (size_t)t0 * HD, bytes, &bars[i]);
      bulk_load(dK + TK * HD, vc + (size_t)t0 * HD, bytes, &bars[i]);
    }
  }
  if (tid < GQM) {
    ml_s[2 * tid] = -INFINITY;
    ml_s[2 * tid + 1] = 0.f;
  }
  pdl_launch_dependents();
  pdl_wait();

  const float scale = 1.0f / sqrtf((float)HD);
  const float2* rrow = a.rope ? a.rope + (size_t)pos * (HD / 2) : nullptr;
  for (int hh = warp; hh <= GQ; hh += 8) {
    const bool isq = hh < GQ;
    if (!isq && !owns_pos) break;
    const float* src = a.qkv + (size_t)(isq ? (g * GQ + hh) : (a.nq + g)) * HD;
    const uint16_t* gain = isq ? a.q_norm : a.k_norm;
    float v[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) v[e] = __ldcg(src + lane + 32 * e);
    if (gain != nullptr) {
      float sq = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) sq = fmaf(v[e], v[e], sq);
      sq = warp_sum(sq);
      const float r = 1.0f / sqrtf(sq / (float)HD + a.eps);
#pragma unroll
      for (int e = 0; e < EPL; ++e) v[e] = v[e] * r * bf16f(gain[lane + 32 * e]);
    }
#pragma unroll
    for (int e = 0; e < EPL / 2; ++e) {
      float cs, sn;
      rope_cs(rrow, pos, lane + 32 * e, HD, a.rope_theta, cs, sn);
      const float x0 = v[e], x1 = v[e + EPL / 2];
      v[e] = x0 * cs - x1 * sn;
      v[e + EPL / 2] = x1 * cs + x0 * sn;
    }
    if (isq) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) q_s[hh * HD + lane + 32 * e] = v[e] * scale;
    } else {
      const float* vsrc = a.qkv + (size_t)(a.nq + a.nkv + g) * HD;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {  // the stored (for bf16: rounded) values are used
        const int d = lane + 32 * e;
        const KT ks = KV::store(v[e]), vs = KV::store(__ldcg(vsrc + d));
        kn_s[d] = KV::load(&ks);
        kc[(size_t)pos * HD + d] = ks;
        vn_s[d] = KV::load(&vs);
        vc[(size_t)pos * HD + d] = vs;
      }
    }
  }
  __syncthreads();

  float qr[GQM][EPL];
#pragma unroll
  for (int h = 0; h < GQM; ++h)
#pragma unroll
    for (int e = 0; e < EPL; ++e) qr[h][e] = (h < GQ) ? q_s[h * HD + lane * EPL + e] : 0.f;

  // P.V and outputs: a thread owns 4 adjacent output dims of one head
  constexpr int OUT4 = (GQM * HD / 4 + 255) / 256;
  float4 oacc[OUT4];
#pragma unroll
  for (int i = 0; i < OUT4; ++i) oacc[i] = make_float4(0.f, 0.f, 0.f, 0.f);

  bool failed = false;
  int it = 0;
  for (; it < ntiles; ++it) {
    const int st = it % NS;
    const bool ok = mbar_wait(&bars[st], (uint32_t)((it / NS) & 1), a.wait_ns);
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    const int t0 = k0 + it * TK, nk = min(TK, k1 - t0);
    KT* Ks = reinterpret_cast<KT*>(stage_base) + (size_t)st * 2 * TK * HD;
    KT* Vs = Ks + TK * HD;
    if (owns_pos && pos >= t0 && pos < t0 + nk) {
      for (int e = tid; e < HD; e += 256) {
        Ks[(pos - t0) * HD + e] = KV::store(kn_s[e]);
        Vs[(pos - t0) * HD + e] = KV::store(vn_s[e]);
      }
      // order these generic writes before a later bulk copy into the same stage
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncthreads();
    }
    {  // scores: warp w takes keys 4w..4w+3 for every head; one transposing reduction of
       // the 32 (key, head) partials leaves (key lane / 8, head lane % 8) on each lane
      float v[4 * GQM];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int j = warp * 4 + k;
        float kv[EPL];
        if constexpr (EPL == 4) {
          const float4 k4 = j < nk ? KV::load4(Ks + j * HD + lane * EPL)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
          kv[0] = k4.x; kv[1] = k4.y; kv[2 % EPL] = k4.z; kv[3 % EPL] = k4.w;
        } else {
          const float2 k2 = j < nk ? KV::load2(Ks + j * HD + lane * EPL) : make_float2(0.f, 0.f);
          kv[0] = k2.x; kv[1 % EPL] = k2.y;
        }
#pragma unroll
        for (int h = 0; h < GQM; ++h) {
          float p = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) p = fmaf(qr[h][e], kv[e], p);
          v[k * GQM + h] = p;
        }
      }
      const float sc = rows_reduce<4 * GQM>(v, lane);
      const int j = warp * 4 + lane / GQM, h = lane % GQM;
      if (j < nk && h < GQ) sc_s[h * TK + j] = sc;
    }
    __syncthreads();
    for (int h = warp; h < GQ; h += 8) {
      const float sc = lane < nk ? sc_s[h * TK + lane] : -INFINITY;
      const float tmax = warp_max(sc);
      const float m_old = ml_s[2 * h], l_old = ml_s[2 * h + 1];
      const float m_new = fmaxf(m_old, tmax);
      const float p = lane < nk ? expf(sc - m_new) : 0.f;
      const float psum = warp_sum(p);
      const float alpha = expf(m_old - m_new);
      p_s[h * TK + lane] = p;
      __syncwarp();
      if (lane == 0) {
        ml_s[2 * h] = m_new;
        ml_s[2 * h + 1] = l_old * alpha + psum;
        al_s[h] = alpha;
      }
    }
    __syncthreads();
#pragma unroll
    for (int oi = 0; oi < OUT4; ++oi) {
      const int idx = tid + oi * 256;
      if (idx < GQ * HD / 4) {
        const int h = idx / (HD / 4), d4 = (idx % (HD / 4)) * 4;
        const float al = al_s[h];
        float4 acc = make_float4(oacc[oi].x * al, oacc[oi].y * al, oacc[oi].z * al, oacc[oi].w * al);
        const float* pr = p_s + h * TK;
        for (int j = 0; j < nk; ++j) {
          const float pj = pr[j];
          const float4 v4 = KV::load4(Vs + j * HD + d4);
          acc.x = fmaf(pj, v4.x, acc.x);
          acc.y = fmaf(pj, v4.y, acc.y);
          acc.z = fmaf(pj, v4.z, acc.z);
          acc.w = fmaf(pj, v4.w, acc.w);
        }
        oacc[oi] = acc;
      }
    }
    __syncthreads();
    if (tid == 0 && it + NS < ntiles) {
      const int nx = it + NS;
      const int t1 = k0 + nx * TK, nk1 = min(TK, k1 - t1);
      const uint32_t bytes = (uint32_t)(nk1 * HD * sizeof(KT));
      mbar_expect_tx(&bars[st], 2 * bytes);
      bulk_load(Ks, kc + (size_t)t1 * HD, bytes, &bars[st]);
      bulk_load(Vs, vc + (size_t)t1 * HD, bytes, &bars[st]);
    }
  }
  if (failed) {
    if (tid == 0) {
      atomicOr(a.err, ERR_TIMEOUT);
      const int hi = min(ntiles, it + NS);
      for (int cc = it; cc < hi; ++cc)
        mbar_wait(&bars[cc % NS], (uint32_t)((cc / NS) & 1), kDrainNs);
    }
    __syncthreads();
  }

  if (nsplit == 1) {
#pragma unroll
    for (int oi = 0; oi < OUT4; ++oi) {
      const int idx = tid + oi * 256;
      if (idx < GQ * HD / 4) {
        const int h = idx / (HD / 4), d4 = (idx % (HD / 4)) * 4;
        const float inv = 1.0f / ml_s[2 * h + 1];
        *reinterpret_cast<float4*>(a.out + (size_t)(g * GQ + h) * HD + d4) =
            make_float4(oacc[oi].x * inv, oacc[oi].y * inv, oacc[oi].z * inv, oacc[oi].w * inv);
      }
    }
    return;
  }
#pragma unroll
  for (int oi = 0; oi < OUT4; ++oi) {
    const int idx = tid + oi * 256;
    if (idx < GQ * HD / 4) {
      const int h = idx / (HD / 4), d4 = (idx % (HD / 4)) * 4;
      *reinterpret_cast<float4*>(a.part_o + ((size_t)(g * GQ + h) * a.nsplit_max + s) * HD + d4) =
          oacc[oi];
    }
  }
  if (tid < GQ) {
    const size_t o = ((size_t)(g * GQ + tid) * a.nsplit_max + s) * 2;
    a.part_ml[o] = ml_s[2 * tid];
    a.part_ml[o + 1] = ml_s[2 * tid + 1];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&a.counters[g], 1);
    *flag_s = (prev == nsplit - 1);
  }
  __syncthreads();
  if (!*flag_s) return;
  __threadfence();
  // Combine (last split to arrive): per head, weights exp(m_s - M) and their l-weighted
  // sum (a warp per head), then each thread sums 4 output dims over the splits in
  // order, 16 float4 loads in flight at a time.
  float* wsm = stage0;  // [GQ][nsplit] (the tile stages are free now)
  float* den_s = wsm + GQ * nsplit;  // [GQ]; the host keeps GQ * (nsplit_max + 1) within the stages
  for (int h = warp; h < GQ; h += 8) {
    const float2* ml = reinterpret_cast<const float2*>(a.part_ml) + (size_t)(g * GQ + h) * a.nsplit_max;
    float m = -INFINITY;
    for (int s2 = lane; s2 < nsplit; s2 += 32) m = fmaxf(m, __ldcg(ml + s2).x);
    m = warp_max(m);
    float dsum = 0.f;
    for (int s2 = lane; s2 < nsplit; s2 += 32) {
      const float2 v2 = __ldcg(ml + s2);
      const float w = expf(v2.x - m);
      wsm[h * nsplit + s2] = w;
      dsum = fmaf(w, v2.y, dsum);
    }
    dsum = warp_sum(dsum);
    if (lane == 0) den_s[h] = dsum;
  }
  __syncthreads();
  for (int idx = tid; idx < GQ * HD / 4; idx += 256) {
    const int h = idx / (HD / 4), d4 = (idx % (HD / 4)) * 4;
    const float* po = a.part_o + (size_t)(g * GQ + h) * a.nsplit_max * HD + d4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < nsplit; s0 += 16) {
      float4 pv[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        pv[j] = s0 + j < nsplit ? __ldcg(reinterpret_cast<const float4*>(po + (size_t)(s0 + j) * HD))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (s0 + j < nsplit) {
          const float w = wsm[h * nsplit + s0 + j];
          acc.x = fmaf(w, pv[j].x, acc.x);
          acc.y = fmaf(w, pv[j].y, acc.y);
          acc.z = fmaf(w, pv[j].z, acc.z);
          acc.w = fmaf(w, pv[j].w, acc.w);
        }
      }
    }
    const float inv = 1.0f / den_s[h];
    *reinterpret_cast<float4*>(a.out + (size_t)(g * GQ + h) * HD + d4) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
  __syncthreads();
  if (tid == 0) a.counters[g] = 0;
}

size_t attention_smem_bytes(int hd) { return hd == 64 ? attn_smem<64>() : attn_smem<128>(); }
bool attention_splits_fit(int gq, int hd, int n_splits) {
  // the combine keeps GQ x nsplit weights and GQ denominators in the tile stages
  const long long stage_floats = (long long)kAttnNS * 2 * kAttnTK * hd;
  return n_splits >= 1 && (long long)gq * ((long long)n_splits + 1) <= stage_floats;
}
int attention_gq_max() { return kAttnGQ; }

cudaError_t launch_attention(const AttnArgs& a, int hd, bool pdl, cudaStream_t s) {
  const dim3 grid(a.nsplit_max, a.nkv);
  if (hd == 64)
    return a.kv_bf16
               ? launch_ex(attn_decode_kernel<64, true>, grid, dim3(256), attn_smem<64>(), s, pdl, a)
               : launch_ex(attn_decode_kernel<64, false>, grid, dim3(256), attn_smem<64>(), s, pdl, a);
  if (hd == 128)
    return a.kv_bf16 ? launch_ex(attn_decode_kernel<128, true>, grid, dim3(256), attn_smem<128>(),
                                 s, pdl, a)
                     : launch_ex(attn_decode_kernel<128, false>, grid, dim3(256),
                                 attn_smem<128>(), s, pdl, a);
  return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------ embedding gather
// x = f32(E[token]); the token is the host's (mapped ring, by position) or,
// when the host left -1 there, the previous step's argmax.
__global__ void __launch_bounds__(256) embed_kernel(const EmbedArgs a) {
  pdl_launch_dependents();
  pdl_wait();
  const int pos = *a.pos;
  int tok = a.tok >= 0 ? a.tok : *a.next_token;
  if (tok < 0 || tok >= a.V) {
    if (threadIdx.x == 0) atomicOr(a.err, ERR_TOKEN);
    tok = 0;
  }
  const uint16_t* row = a.table + (size_t)tok * a.H;
  for (int i = threadIdx.x; i < a.H; i += blockDim.x) {
    const float v = bf16f(row[i]);
    a.x[i] = v;
    if (a.cap_out) a.cap_out[(size_t)pos * a.H + i] = v;
  }
}

cudaError_t launch_embed(const EmbedArgs& a, cudaStream_t s) {
  return launch_ex(embed_kernel, dim3(1), dim3(256), 0, s, false, a);
}
const void* embed_kernel_fn() { return reinterpret_cast<const void*>(embed_kernel); }

// ------------------------------------------------------------------ int4 row packing
// Row r of (nib [rows, K/2], scales [rows, K/128]) -> dst row dst_row0 + r * step in
// the layout nibbles | scales | zero pad (int4_row_bytes(K) bytes per row).
__global__ void pack_int4_rows_kernel(const uint8_t* nib, const uint16_t* scales, int K,
                                      uint8_t* dst, int dst_row0, int step) {
  const int r = blockIdx.x;
  const uint32_t rb = int4_row_bytes(K), half = (uint32_t)K / 2, G = (uint32_t)K / 128;
  uint8_t* d = dst + (size_t)(dst_row0 + (size_t)r * step) * rb;
  const uint8_t* sn = nib + (size_t)r * half;
  for (uint32_t i = threadIdx.x; i < half; i += blockDim.x) d[i] = sn[i];
  const uint16_t* ss = scales + (size_t)r * G;
  for (uint32_t i = threadIdx.x; i < (rb - half) / 2; i += blockDim.x)
    reinterpret_cast<uint16_t*>(d + half)[i] = i < G ? ss[i] : (uint16_t)0;
}

cudaError_t launch_pack_int4_rows(const uint8_t* nib, const uint16_t* scales, int rows, int K,
                                  uint8_t* dst, int dst_row0, int dst_row_step, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  pack_int4_rows_kernel<<<rows, 256, 0, s>>>(nib, scales, K, dst, dst_row0, dst_row_step);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ Q8_0 row packing
// Row r of (q [rows, K] int8, scales [rows, K/32] fp16 bits) -> dst row dst_row0 + r * step
// in the layout int8 | scales | zero pad (q8_row_bytes(K) bytes per row).
__global__ void pack_q8_rows_kernel(const int8_t* q, const uint16_t* scales, int K, uint8_t* dst,
                                    int dst_row0, int step) {
  const int r = blockIdx.x;
  const uint32_t rb = q8_row_bytes(K), G = (uint32_t)K / 32;
  uint8_t* d = dst + (size_t)(dst_row0 + (size_t)r * step) * rb;
  const int8_t* sq = q + (size_t)r * K;
  for (uint32_t i = threadIdx.x; i < (uint32_t)K; i += blockDim.x) d[i] = (uint8_t)sq[i];
  const uint16_t* ss = scales + (size_t)r * G;
  for (uint32_t i = threadIdx.x; i < (rb - (uint32_t)K) / 2; i += blockDim.x)
    reinterpret_cast<uint16_t*>(d + K)[i] = i < G ? ss[i] : (uint16_t)0;
}

cudaError_t launch_pack_q8_rows(const int8_t* q, const uint16_t* scales, int rows, int K,
                                uint8_t* dst, int dst_row0, int dst_row_step, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  pack_q8_rows_kernel<<<rows, 256, 0, s>>>(q, scales, K, dst, dst_row0, dst_row_step);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ Q8_0 quantiser
// One warp per block of 32 inputs, a lane per input: s = fp16(max|w| / 127) (f32
// division, round to nearest even), q = clamp(rint(w / s), -127, 127) (f32 division,
// ties to even), q = 0 when s = 0.
template <bool BF16_IN>
__global__ void __launch_bounds__(256) quantize_q8_kernel(const void* w, int rows, int cols,
                                                          int8_t* q, size_t q_stride,
                                                          uint16_t* scales, size_t s_stride) {
  const int G = cols / 32;
  const long long gi = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gi >= (long long)rows * G) return;
  const int r = (int)(gi / G), g = (int)(gi % G);
  const size_t idx = (size_t)r * cols + g * 32 + lane;
  const float v = BF16_IN ? bf16f(reinterpret_cast<const uint16_t*>(w)[idx])
                          : reinterpret_cast<const float*>(w)[idx];
  const float m = warp_max(fabsf(v));
  const __half sh = __float2half_rn(__fdiv_rn(m, 127.0f));
  const float sc = __half2float(sh);
  float qv = 0.f;
  if (sc != 0.f) qv = fminf(127.f, fmaxf(-127.f, rintf(__fdiv_rn(v, sc))));
  q[(size_t)r * q_stride + g * 32 + lane] = (int8_t)(int)qv;
  if (lane == 0) scales[(size_t)r * s_stride + g] = __half_as_ushort(sh);
}

cudaError_t launch_quantize_q8(const void* w, bool w_bf16, int rows, int cols, int8_t* q,
                               size_t q_stride, uint16_t* scales, size_t s_stride,
                               cudaStream_t s) {
  const long long groups = (long long)rows * (cols / 32);
  if (groups == 0) return cudaSuccess;
  const long long blocks = (groups + 7) / 8;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (w_bf16)
    quantize_q8_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(w, rows, cols, q, q_stride, scales,
                                                              s_stride);
  else
    quantize_q8_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(w, rows, cols, q, q_stride, scales,
                                                               s_stride);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ RoPE table
// cos/sin of p * theta^(-2j/hd), formed in fp64 and rounded to f32 once.
__global__ void rope_table_kernel(float2* t, int cap, int hd, double theta) {
  const int half = hd / 2;
  const long long n = (long long)cap * half;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int p = (int)(i / half), j = (int)(i % half);
    const double inv = pow(theta, -2.0 * (double)j / (double)hd);
    double sd, cd;
    sincos((double)p * inv, &sd, &cd);
    t[i] = make_float2((float)cd, (float)sd);
  }
}

cudaError_t launch_rope_table(float2* table, int cap, int hd, float theta, cudaStream_t s) {
  rope_table_kernel<<<1024, 256, 0, s>>>(table, cap, hd, (double)theta);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ int4 g128 quantiser
// One warp per group of 128 inputs; a lane handles 4 consecutive values.
__global__ void __launch_bounds__(256) quantize_int4_kernel(const float* w, int rows, int cols,
                                                            uint8_t* packed, uint16_t* scales) {
  const int G = cols / 128;
  const long long gi = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gi >= (long long)rows * G) return;
  const int r = (int)(gi / G), g = (int)(gi % G);
  const float4 v = *reinterpret_cast<const float4*>(w + (size_t)r * cols + g * 128 + lane * 4);
  float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
  m = warp_max(m);
  const float s32 = __fdiv_rn(m, 7.0f);
  const uint32_t u = __float_as_uint(s32);
  const uint16_t sb = (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
  const float sc = bf16f(sb);
  const float vals[4] = {v.x, v.y, v.z, v.w};
  uint32_t nib[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float q = 0.f;
    if (sc != 0.f) q = fminf(7.f, fmaxf(-7.f, rintf(__fdiv_rn(vals[e], sc))));
    nib[e] = (uint32_t)((int)q + 8);
  }
  const uint16_t two = (uint16_t)((nib[0] | (nib[1] << 4)) | ((nib[2] | (nib[3] << 4)) << 8));
  *reinterpret_cast<uint16_t*>(packed + (size_t)r * (cols / 2) + g * 64 + lane * 2) = two;
  if (lane == 0) scales[(size_t)r * G + g] = sb;
}

cudaError_t launch_quantize_int4(const float* w, int rows, int cols, uint8_t* packed,
                                 uint16_t* scales, cudaStream_t s) {
  const long long groups = (long long)rows * (cols / 128);
  if (groups == 0) return cudaSuccess;
  const long long blocks = (groups + 7) / 8;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  quantize_int4_kernel<<<(unsigned)blocks, 256, 0, s>>>(w, rows, cols, packed, scales);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ attributes
// Allow up to `bytes` of dynamic shared memory, capped by what the device
// grants a block minus the kernel's static shared memory.
template <class Kern>
static cudaError_t allow_smem(Kern k, size_t bytes) {
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaFuncAttributes fa{};
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, k);
  if (e != cudaSuccess) return e;
  const size_t cap = (size_t)optin - fa.sharedSizeBytes;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)(bytes < cap ? bytes : cap));
  // One carveout for every kernel of the step: an SM never reconfigures between
  // consecutive kernels, so a kernel can start while its predecessor finishes.
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  return e;
}

cudaError_t set_kernel_attributes() {
  const size_t big = 227 * 1024;
  cudaError_t e = cudaSuccess;
#define QW_ALLOW(k, b) \
  if (e == cudaSuccess) e = allow_smem(k, b)
#define QW_ALLOW_GEMV(E)                 \
  QW_ALLOW((gemv_kernel<E, 4, 0>), big); \
  QW_ALLOW((gemv_kernel<E, 8, 0>), big); \
  QW_ALLOW((gemv_kernel<E, 4, 1>), big); \
  QW_ALLOW((gemv_kernel<E, 8, 1>), big); \
  QW_ALLOW((gemv_kernel<E, 4, 2>), big); \
  QW_ALLOW((gemv_kernel<E, 8, 2>), big)
  QW_ALLOW_GEMV(EPI_STORE);
  QW_ALLOW_GEMV(EPI_RESIDUAL);
  QW_ALLOW_GEMV(EPI_SWIGLU);
  QW_ALLOW_GEMV(EPI_LOGITS);
#undef QW_ALLOW_GEMV
  QW_ALLOW((attn_decode_kernel<64, false>), attn_smem<64>());
  QW_ALLOW((attn_decode_kernel<128, false>), attn_smem<128>());
  QW_ALLOW((attn_decode_kernel<64, true>), attn_smem<64>());
  QW_ALLOW((attn_decode_kernel<128, true>), attn_smem<128>());
  QW_ALLOW(embed_kernel, 0);
#undef QW_ALLOW
  return e;
}

}  // namespace qw
