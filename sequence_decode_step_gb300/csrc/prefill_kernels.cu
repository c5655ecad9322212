// Prefill kernels for sm_103a: the dense contractions run on tcgen05 tensor
// cores (TMA-fed, TMEM accumulators); the row-wise steps are CUDA-core kernels.
//
// GEMM: one CTA computes a 128 x BN tile of C = A . B^T. Warp 0 (one thread)
// streams A and B k-tiles (64 wide, 128-byte swizzle) with TMA into a ring of
// shared-memory stages; warp 1 owns the TMEM accumulator (BN columns) and one of
// its threads issues tcgen05.mma (M=128, N=BN, K=16) per 16-wide slice; warps
// 2..5 read the accumulator back with tcgen05.ld (one TMEM lane = one row per
// thread) and apply the epilogue. Activations enter as two bf16 halves
// (hi = bf16(x), lo = bf16(x - hi)) multiplied against the same exact-bf16
// weight tile, so the product keeps about 16 bits of the f32 activation.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <math.h>
#include <stdint.h>

#include "qw_internal.h"
#include "qw_ptx.cuh"

namespace qw {

constexpr int GBM = 128;
constexpr int GBK = 64;
constexpr uint32_t kATileBytes = GBM * GBK * 2;  // 16 KB

__device__ __forceinline__ void split_bf16(float x, uint16_t& hi, uint16_t& lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
  hi = __bfloat16_as_ushort(h);
  lo = __bfloat16_as_ushort(l);
}

template <int BN, int EPI>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap ta_hi,
                   const __grid_constant__ CUtensorMap ta_lo,
                   const __grid_constant__ CUtensorMap tb,
                   const __grid_constant__ CUtensorMap tb_lo, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int NS = a.n_stages;
  constexpr uint32_t kBTileBytes = (uint32_t)BN * GBK * 2;
  const uint32_t stage_bytes = (uint32_t)a.a_split * kATileBytes + (uint32_t)a.b_split * kBTileBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * stage_bytes);
  uint64_t* empty = full + NS;
  uint64_t* accf = empty + NS;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(accf + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * GBM, n0 = blockIdx.x * BN;
  // this CTA's k-tiles [kt_a, kt_b): all of K, or split blockIdx.z of a split-K launch
  const int KT_all = (a.K + GBK - 1) / GBK, ks = EPI == GEPI_RESID && a.ksplit > 1 ? a.ksplit : 1;
  const int split = ks > 1 ? (int)blockIdx.z : 0;
  const int kt_a = split * KT_all / ks, kt_b = (split + 1) * KT_all / ks;
  const int KT = kt_b - kt_a;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(accf, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tslot, BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp == 0 && lane == 0) {
    // ---- producer: TMA k-tiles of A (hi[, lo]) and B into the stage ring
    for (int kt = 0; kt < KT; ++kt) {
      const int s = kt % NS, u = kt / NS;
      if (u > 0 && !mbar_wait(&empty[s], (uint32_t)((u - 1) & 1), a.wait_ns)) {
        atomicOr(a.err, ERR_TIMEOUT);
        break;
      }
      uint8_t* st = smem + (size_t)s * stage_bytes;
      const int kx = (kt_a + kt) * GBK;
      mbar_expect_tx(&full[s], stage_bytes);
      tma_load_2d(st, &ta_hi, kx, m0, &full[s]);
      if (a.a_split == 2) tma_load_2d(st + kATileBytes, &ta_lo, kx, m0, &full[s]);
      tma_load_2d(st + a.a_split * kATileBytes, &tb, kx, n0, &full[s]);
      if (a.b_split == 2)
        tma_load_2d(st + a.a_split * kATileBytes + kBTileBytes, &tb_lo, kx, n0, &full[s]);
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(GBM, BN);
    for (int kt = 0; kt < KT; ++kt) {
      const int s = kt % NS, u = kt / NS;
      if (!mbar_wait(&full[s], (uint32_t)(u & 1), a.wait_ns)) {
        atomicOr(a.err, ERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t sa = smem_addr(smem + (size_t)s * stage_bytes);
      const uint32_t sb = sa + (uint32_t)a.a_split * kATileBytes;
#pragma unroll
      for (int k = 0; k < GBK / 16; ++k) {
        const uint64_t bd = sw128_kmajor_desc(sb + k * 32);
        const uint64_t ad = sw128_kmajor_desc(sa + k * 32);
        tc_mma_bf16(tbase, ad, bd, idesc, (kt | k) != 0);
        if (a.a_split == 2)
          tc_mma_bf16(tbase, sw128_kmajor_desc(sa + kATileBytes + k * 32), bd, idesc, 1);
        if (a.b_split == 2)  // the weight's lo term against the activation's hi term
          tc_mma_bf16(tbase, ad, sw128_kmajor_desc(sb + kBTileBytes + k * 32), idesc, 1);
      }
      tc_commit(&empty[s]);  // the stage is free once these MMAs have read it
    }
    tc_commit(accf);  // the accumulator is final once every MMA above completed
    // TMEM is released below only after the MMAs have finished.
    mbar_wait(accf, 0, kDrainNs);
  } else if (warp >= 2) {
    // ---- epilogue: warp w reads TMEM lanes [32 (w % 4), +32) = rows of the tile
    bool ok = mbar_wait(accf, 0, a.wait_ns);
    if (!ok && lane == 0) atomicOr(a.err, ERR_TIMEOUT);
    int* flag = ks > 1 ? a.flags + blockIdx.y * gridDim.x + blockIdx.x : nullptr;
    if (flag != nullptr && split > 0) {  // split s adds after split s - 1 (a fixed order)
      if (threadIdx.x == 64) {
        bool got = false;
        uint64_t t0 = 0;
        for (uint32_t n = 1; a.wait_ns != 0; ++n) {
          int f;
          asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(f) : "l"(flag) : "memory");
          if (f == split) { got = true; break; }
          if ((n & 15u) == 0) {
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > a.wait_ns || (*reinterpret_cast<volatile int*>(a.err) & ERR_TIMEOUT)) break;
          }
        }
        if (!got) atomicOr(a.err, ERR_TIMEOUT);
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
      ok = ok && (*reinterpret_cast<volatile int*>(a.err) & ERR_TIMEOUT) == 0;
    }
    tc_fence_after();
    const int q = warp & 3;
    const int row = m0 + q * 32 + lane;
    float* const cap_out = split == ks - 1 ? a.cap_out : nullptr;  // the final rows only
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 16) {
      uint32_t r[16];
      tmem_ld16(tbase + ((uint32_t)(q * 32) << 16) + (uint32_t)c0, r);
      tmem_ld_wait();
      tmem_regs_ready(r);
      const int col0 = n0 + c0;
      if (!ok || row >= a.M || col0 >= a.N) continue;
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
      const int nv = min(16, a.N - col0);
      // full 16-column blocks move as 16-byte vectors (ldo, ldb are multiples of 16 B)
      const bool vec = nv == 16 && (a.ldo % 4) == 0 && (a.ldb % 8) == 0;
      if (EPI == GEPI_STORE) {
        float* o = a.out + (size_t)row * a.ldo + col0;
        if (vec) {
          if (a.bias) {
            const uint4 b0 = *reinterpret_cast<const uint4*>(a.bias + col0);
            const uint4 b1 = *reinterpret_cast<const uint4*>(a.bias + col0 + 8);
            const uint32_t bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              v[2 * j] += __uint_as_float(bw[j] << 16);
              v[2 * j + 1] += __uint_as_float(bw[j] & 0xffff0000u);
            }
          }
#pragma unroll
          for (int j = 0; j < 16; j += 4)
            *reinterpret_cast<float4*>(o + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j < nv) o[j] = v[j] + (a.bias ? __uint_as_float((uint32_t)a.bias[col0 + j] << 16) : 0.f);
        }
      } else if (EPI == GEPI_RESID) {
        float* o = a.out + (size_t)row * a.ldo + col0;
        if (vec) {
          float4 cur[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) cur[j] = __ldcg(reinterpret_cast<const float4*>(o + 4 * j));
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float4 n4 = make_float4(cur[j].x + v[4 * j], cur[j].y + v[4 * j + 1],
                                          cur[j].z + v[4 * j + 2], cur[j].w + v[4 * j + 3]);
            *reinterpret_cast<float4*>(o + 4 * j) = n4;
            if (cap_out)
              *reinterpret_cast<float4*>(cap_out + (size_t)(a.cap_row0 + row) * a.ldo + col0 + 4 * j) = n4;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j < nv) {
              const float nvl = __ldcg(o + j) + v[j];
              o[j] = nvl;
              if (cap_out) cap_out[(size_t)(a.cap_row0 + row) * a.ldo + col0 + j] = nvl;
            }
        }
      } else if (vec) {  // GEPI_SWIGLU, 8 units as one 16-byte store per half
        uint16_t hi[8], lo[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float g = v[2 * j], up = v[2 * j + 1];
          split_bf16(g / (1.0f + expf(-g)) * up, hi[j], lo[j]);
        }
        const size_t off = (size_t)row * a.ldb + col0 / 2;
        *reinterpret_cast<uint4*>(a.out_hi + off) =
            make_uint4(hi[0] | ((uint32_t)hi[1] << 16), hi[2] | ((uint32_t)hi[3] << 16),
                       hi[4] | ((uint32_t)hi[5] << 16), hi[6] | ((uint32_t)hi[7] << 16));
        *reinterpret_cast<uint4*>(a.out_lo + off) =
            make_uint4(lo[0] | ((uint32_t)lo[1] << 16), lo[2] | ((uint32_t)lo[3] << 16),
                       lo[4] | ((uint32_t)lo[5] << 16), lo[6] | ((uint32_t)lo[7] << 16));
      } else {  // GEPI_SWIGLU tail
        const int u0 = col0 / 2;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (2 * j + 1 < nv) {
            const float g = v[2 * j], up = v[2 * j + 1];
            uint16_t hi, lo;
            split_bf16(g / (1.0f + expf(-g)) * up, hi, lo);
            a.out_hi[(size_t)row * a.ldb + u0 + j] = hi;
            a.out_lo[(size_t)row * a.ldb + u0 + j] = lo;
          }
      }
    }
  }
  if (ks > 1 && warp >= 2) {  // this split's sums are in out: hand the tile to the next split
    __threadfence();
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (threadIdx.x == 64) {
      int* flag = a.flags + blockIdx.y * gridDim.x + blockIdx.x;
      const int nxt = split + 1 == ks ? 0 : split + 1;  // the last split leaves it at rest
      asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(flag), "r"(nxt) : "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, BN);
  }
}


// ------------------------------------------------------------------ row-wise prefill kernels
__global__ void __launch_bounds__(256) embed_rows_kernel(const int* ids, const uint16_t* table,
                                                         int V, int H, float* X, float* cap,
                                                         int row0, int* err) {
  const int t = blockIdx.x;
  int tok = ids[t];
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) atomicOr(err, ERR_TOKEN);
    tok = 0;
  }
  const uint16_t* src = table + (size_t)tok * H;
  for (int i = threadIdx.x; i < H; i += 256) {
    const float v = bf16f(src[i]);
    X[(size_t)t * H + i] = v;
    if (cap) cap[(size_t)(row0 + t) * H + i] = v;
  }
}

// One row per CTA: y = x * rstd * g, written as a two-bf16 split and/or as f32.
__global__ void __launch_bounds__(256) rmsnorm_rows_kernel(const float* X, int H,
                                                           const uint16_t* g, float eps,
                                                           uint16_t* out_hi, uint16_t* out_lo,
                                                           float* out_f32, int f32_row0) {
  __shared__ float red[8];
  const int t = blockIdx.x;
  const float* x = X + (size_t)t * H;
  float ss = 0.f;
  for (int i = threadIdx.x; i < H; i += 256) ss = fmaf(x[i], x[i], ss);
  const float tot = block_sum_256(ss, red);
  const float r = 1.0f / sqrtf(tot / (float)H + eps);
  for (int i = threadIdx.x; i < H; i += 256) {
    const float y = x[i] * r * bf16f(g[i]);
    if (out_hi) {
      uint16_t hi, lo;
      split_bf16(y, hi, lo);
      out_hi[(size_t)t * H + i] = hi;
      out_lo[(size_t)t * H + i] = lo;
    }
    if (out_f32) out_f32[(size_t)(f32_row0 + t) * H + i] = y;
  }
}

// Row t (position p0 + t): per-head QK-RMSNorm and RoPE of q and k, q scaled by
// log2(e)/sqrt(hd) into Q [T][nq][hd] as a two-bf16 split (the attention works in base
// 2); k and v appended to the cache at their position, and k also as the two-bf16 row
// the prefill attention reads.
template <int HD, bool KB>
__global__ void __launch_bounds__(256) qk_rope_kv_rows_kernel(
    const float* QKV, int p0, int nq, int nkv, const uint16_t* q_norm, const uint16_t* k_norm,
    float eps, const float2* rope, uint16_t* q_hi, uint16_t* q_lo, void* kc_, void* vc_, int cap,
    uint16_t* k_hi, uint16_t* k_lo, int kv_rows) {
  constexpr int EPL = HD / 32;
  using KV = KvElem<KB>;  // cache element: f32, or bf16 (rounded when stored)
  using KT = typename KV::T;
  KT* kc = reinterpret_cast<KT*>(kc_);
  KT* vc = reinterpret_cast<KT*>(vc_);
  const int t = blockIdx.x, pos = p0 + t;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* row = QKV + (size_t)t * (nq + 2 * nkv) * HD;
  // Q carries 1/sqrt(hd) and log2(e): the attention's scores come out in base-2 units
  const float scale = 1.4426950408889634f / sqrtf((float)HD);
  const float2* rr = rope + (size_t)pos * (HD / 2);
  for (int hh = warp; hh < nq + nkv; hh += 8) {
    const bool isq = hh < nq;
    const float* src = row + (size_t)hh * HD;
    const uint16_t* gain = isq ? q_norm : k_norm;
    float v[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) v[e] = src[lane + 32 * e];
    if (gain != nullptr) {
      float sq = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) sq = fmaf(v[e], v[e], sq);
      sq = warp_sum(sq);
      const float r = 1.0f / sqrtf(sq / (float)HD + eps);
#pragma unroll
      for (int e = 0; e < EPL; ++e) v[e] = v[e] * r * bf16f(gain[lane + 32 * e]);
    }
#pragma unroll
    for (int e = 0; e < EPL / 2; ++e) {
      const float2 cs = rr[lane + 32 * e];
      const float x0 = v[e], x1 = v[e + EPL / 2];
      v[e] = x0 * cs.x - x1 * cs.y;
      v[e + EPL / 2] = x1 * cs.x + x0 * cs.y;
    }
    if (isq) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        uint16_t hi, lo;
        split_bf16(v[e] * scale, hi, lo);
        q_hi[((size_t)t * nq + hh) * HD + lane + 32 * e] = hi;
        q_lo[((size_t)t * nq + hh) * HD + lane + 32 * e] = lo;
      }
    } else {
      KT* dst = kc + ((size_t)(hh - nq) * cap + pos) * HD;
      const size_t ko = ((size_t)(hh - nq) * kv_rows + pos) * HD;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const KT stored = KV::store(v[e]);
        dst[lane + 32 * e] = stored;
        uint16_t hi, lo;
        split_bf16(KV::load(&stored), hi, lo);
        k_hi[ko + lane + 32 * e] = hi;
        k_lo[ko + lane + 32 * e] = lo;
      }
    }
  }
  const float* vsrc = row + (size_t)(nq + nkv) * HD;
  for (int i = threadIdx.x; i < nkv * HD; i += 256)
    vc[((size_t)(i / HD) * cap + pos) * HD + (i % HD)] = KV::store(vsrc[i]);
}

// Two bf16 terms of a pair of f32 values (hi = bf16(x), lo = bf16(x - hi)), packed as
// the GEMMs' activation operands take them.
__device__ __forceinline__ uint32_t pack_bf16x2(uint16_t lo_col, uint16_t hi_col) {
  return (uint32_t)lo_col | ((uint32_t)hi_col << 16);
}
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  uint16_t h0, l0, h1, l1;
  split_bf16(x0, h0, l0);
  split_bf16(x1, h1, l1);
  hi = pack_bf16x2(h0, h1);
  lo = pack_bf16x2(l0, l1);
}
// ---- causal attention on tcgen05 tensor cores (kind::f16, TMEM accumulators)
// One CTA per (query head, block of 128 query rows), heaviest block first. Every f32
// operand enters as two bf16 terms hi = bf16(x), lo = bf16(x - hi), and a product a.b
// is issued as three MMAs, a_hi.b_hi + a_hi.b_lo + a_lo.b_hi, into an f32 TMEM
// accumulator (the lo.lo term is below the f32 rounding of the sum), so scores and
// outputs carry about 16 bits of the f32 values.
// Warp 0 (one thread) brings Q (hi, lo) once and, per tile of 64 keys, the K rows
// and the V^T rows (hi, lo) with TMA (128-byte swizzle) into a double buffer. Warp 1
// (one thread) issues S = Q K^T (M 128, N 64, K head_dim) and O += P V (M 128,
// N head_dim, K 64). Warps 2..5 own the 128 TMEM lanes, one query row per thread:
// they read the scores, apply the causal mask and the online softmax (base 2),
// rescale O in TMEM when the row maximum moves, write P (hi, lo) to shared memory in
// the layout the MMA reads, and at the end normalise O and store it as the two-bf16
// split the o_proj GEMM takes. S for tile i+1 is issued as soon as the scores of
// tile i have been read, so it overlaps the softmax of tile i.
// The causal work is balanced by cutting each query block's keys into chunks of at
// most kFaChunk tiles, one CTA each, all heads' heaviest items first; a chunk of a
// block with several writes its unnormalised O and (m, l) per row, and the last one
// to arrive merges them in chunk order. The reference maximum of a row moves only
// when the row maximum rises by more than 2^8 (P then stays below 256), so most
// tiles leave O in TMEM untouched; O / l does not depend on the reference.
constexpr int kFaBQ = kFaQueryRows;  // query rows per CTA (the MMA's M, one TMEM lane each)
constexpr int kFaBN = kFaKeyRows;    // keys per tile (one 128-byte bf16 atom)
constexpr int kFaChunk = 8;          // key tiles per CTA at most
// Softmax warps: two per TMEM sub-partition, each taking half of a row's key columns
// (and, at the end, half of its head dimensions); with the producer and MMA warps.
constexpr int kFaSoftmaxWarps = 8;
constexpr int kFaThreads = (2 + kFaSoftmaxWarps) * 32;

template <int HD>
struct FaLayout {
  static constexpr int QA = HD / 64;                         // 128-byte atoms across head_dim
  static constexpr uint32_t kQ1 = QA * kFaBQ * 128;          // Q hi (or lo): QA atoms of 128 rows
  static constexpr uint32_t kK1 = QA * kFaBN * 128;          // K tile hi (or lo): QA atoms of 64 rows
  static constexpr uint32_t kV1 = HD * 128;                  // V^T tile hi (or lo): head_dim rows
  static constexpr uint32_t kP1 = kFaBQ * 128;               // P hi (or lo): 128 rows
  static constexpr uint32_t kKV = 2 * kK1 + 2 * kV1;         // one buffer: K hi, K lo, V hi, V lo
  static constexpr uint32_t off_kv = 2 * kQ1;
  static constexpr uint32_t off_p = off_kv + 2 * kKV;
  static constexpr uint32_t off_bar = off_p + 2 * kP1;
  static constexpr uint32_t bytes = off_bar + 128 + 1024;   // barriers, TMEM slot, alignment slack
};

// 2^x with the special-function unit (ex2.approx.ftz: relative error about 2^-22;
// 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Two f32 values as two bf16 terms each (hi = bf16(x), lo = bf16(x - hi)), packed as
// bf16x2 words: the first value in the low half.
__device__ __forceinline__ void split2_packed(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - __low2float(h), x1 - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Wait for an mbarrier phase, bounded; gives up at once when another thread of the
// launch already reported a timeout.
__device__ __forceinline__ bool fa_wait(const FaArgs& a, uint64_t* bar, uint32_t parity) {
  if (a.wait_ns == 0) return false;
  uint64_t t0 = 0;
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 15u) != 0) continue;
    const uint64_t now = globaltimer_ns();
    if (t0 == 0) {
      t0 = now;
    } else if (now - t0 > a.wait_ns || (*reinterpret_cast<volatile int*>(a.err) & ERR_TIMEOUT)) {
      return false;
    }
  }
}

template <int HD>
__global__ void __launch_bounds__(kFaThreads, 1)
    attn_prefill_fa_kernel(const __grid_constant__ FaMaps mp, const FaArgs a) {
  using LY = FaLayout<HD>;
  constexpr int QA = LY::QA;
  constexpr uint32_t kTmemCols = 256;
  extern __shared__ uint8_t fa_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(fa_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + LY::off_bar);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;   // [2]
  uint64_t* kv_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;
  uint64_t* s_empty = bars + 6;
  uint64_t* p_full = bars + 7;
  uint64_t* o_full = bars + 8;
  uint64_t* done = bars + 9;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 10);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = (a.T + kFaBQ - 1) / kFaBQ;
  // this CTA's (query block, key chunk): blocks from the last (heaviest) down, every
  // head's item of one rank before the next rank (blockIdx.x is the head)
  int qb = nqb - 1, chunk = blockIdx.y, nch = 1, bt = 1;
  for (;; --qb) {
    const int nr = min(kFaBQ, a.T - qb * kFaBQ);
    bt = (a.p0 + qb * kFaBQ + nr - 1) / kFaBN + 1;  // key tiles of the block
    nch = (bt + kFaChunk - 1) / kFaChunk;
    if (chunk < nch || qb == 0) break;
    chunk -= nch;
  }
  const int h = blockIdx.x, kvh = h / (a.nq / a.nkv);
  const int t0 = qb * kFaBQ;
  const int nrows = min(kFaBQ, a.T - t0);
  const int kt0 = chunk * kFaChunk;
  const int n_tiles = min(bt, kt0 + kFaChunk) - kt0;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&kv_full[b], 1);
      mbar_init(&kv_empty[b], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_empty, kFaSoftmaxWarps);  // one arrival per softmax warp
    mbar_init(p_full, kFaSoftmaxWarps);
    mbar_init(o_full, 1);
    mbar_init(done, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tslot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const uint32_t t_s = tbase, t_o = tbase + kFaBN;  // S: 64 columns, O: head_dim columns

  if (warp == 0) {
    if (lane == 0) {
      // ---- producer
      mbar_expect_tx(q_full, 2 * LY::kQ1);
      for (int c = 0; c < QA; ++c) {
        tma_load_2d(sm + c * (kFaBQ * 128), &mp.q_hi, h * HD + 64 * c, t0, q_full);
        tma_load_2d(sm + LY::kQ1 + c * (kFaBQ * 128), &mp.q_lo, h * HD + 64 * c, t0, q_full);
      }
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int b = i & 1;
        if (i >= 2 && !fa_wait(a, &kv_empty[b], (uint32_t)(((i >> 1) - 1) & 1))) {
          atomicOr(a.err, ERR_TIMEOUT);
          break;
        }
        uint8_t* kb = sm + LY::off_kv + b * LY::kKV;
        const int k0 = (kt0 + i) * kFaBN, krow = kvh * a.kv_rows + k0;
        mbar_expect_tx(&kv_full[b], LY::kKV);
        for (int c = 0; c < QA; ++c) {
          tma_load_2d(kb + c * (kFaBN * 128), &mp.k_hi, 64 * c, krow, &kv_full[b]);
          tma_load_2d(kb + LY::kK1 + c * (kFaBN * 128), &mp.k_lo, 64 * c, krow, &kv_full[b]);
        }
        tma_load_2d(kb + 2 * LY::kK1, &mp.vt_hi, k0, kvh * HD, &kv_full[b]);
        tma_load_2d(kb + 2 * LY::kK1 + LY::kV1, &mp.vt_lo, k0, kvh * HD, &kv_full[b]);
        issued = i + 1;
      }
      // leave only once the copies issued into this CTA's shared memory have landed
      mbar_wait(q_full, 0, kDrainNs);
      for (int i = issued > 2 ? issued - 2 : 0; i < issued; ++i)
        mbar_wait(&kv_full[i & 1], (uint32_t)((i >> 1) & 1), kDrainNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer
      constexpr uint32_t id_s = idesc_bf16_f32(kFaBQ, kFaBN);
      constexpr uint32_t id_o = idesc_bf16_f32(kFaBQ, HD);
      const uint32_t qh = smem_addr(sm), ql = qh + LY::kQ1;
      const uint32_t ph = smem_addr(sm + LY::off_p), pl = ph + LY::kP1;
      auto issue_s = [&](int i) {  // S = Q . K_i^T, three terms per product
        const uint32_t kh = smem_addr(sm + LY::off_kv + (i & 1) * LY::kKV), kl = kh + LY::kK1;
#pragma unroll
        for (int c = 0; c < QA; ++c)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t qo = c * (kFaBQ * 128) + k * 32, ko = c * (kFaBN * 128) + k * 32;
            const uint64_t dkh = sw128_kmajor_desc(kh + ko), dqh = sw128_kmajor_desc(qh + qo);
            tc_mma_bf16(t_s, dqh, dkh, id_s, (c | k) != 0);
            tc_mma_bf16(t_s, dqh, sw128_kmajor_desc(kl + ko), id_s, 1);
            tc_mma_bf16(t_s, sw128_kmajor_desc(ql + qo), dkh, id_s, 1);
          }
        tc_commit(s_full);
      };
      bool ok = fa_wait(a, q_full, 0) && fa_wait(a, &kv_full[0], 0);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int i = 0; ok && i < n_tiles; ++i) {
        if (i + 1 < n_tiles) {  // the scores of tile i are read: start tile i + 1's
          ok = fa_wait(a, s_empty, (uint32_t)(i & 1)) &&
               fa_wait(a, &kv_full[(i + 1) & 1], (uint32_t)(((i + 1) >> 1) & 1));
          if (!ok) break;
          tc_fence_after();
          issue_s(i + 1);
        }
        ok = fa_wait(a, p_full, (uint32_t)(i & 1));  // P_i written, O rescaled
        if (!ok) break;
        tc_fence_after();
        const uint32_t vh = smem_addr(sm + LY::off_kv + (i & 1) * LY::kKV + 2 * LY::kK1);
        const uint32_t vl = vh + LY::kV1;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t dph = sw128_kmajor_desc(ph + k * 32), dvh = sw128_kmajor_desc(vh + k * 32);
          tc_mma_bf16(t_o, dph, dvh, id_o, (i | k) != 0);
          tc_mma_bf16(t_o, dph, sw128_kmajor_desc(vl + k * 32), id_o, 1);
          tc_mma_bf16(t_o, sw128_kmajor_desc(pl + k * 32), dvh, id_o, 1);
        }
        tc_commit(o_full);
        tc_commit(&kv_empty[i & 1]);
      }
      if (!ok) atomicOr(a.err, ERR_TIMEOUT);
      // TMEM is released below only after every MMA issued here has finished
      tc_commit(done);
      mbar_wait(done, 0, kDrainNs);
    }
  } else {
    // ---- softmax and epilogue: warps 2..9; warp w owns TMEM lanes [32 (w % 4), +32) = query
    // rows, and half hf of each row's key columns (and of its head dims at the end). The two
    // halves of a row exchange their maxima (and finally their sums) through two spare TMEM
    // columns per tile parity, at a barrier of the eight warps that also ORs a failed wait,
    // so all of them leave the loop together.
    constexpr int kHalf = kFaBN / 2, kHD2 = HD / 2;
    const int q4 = warp & 3, r = q4 * 32 + lane, hf = (warp - 2) >> 2;
    const uint32_t lrow = (uint32_t)(q4 * 32) << 16;
    const uint32_t t_x = tbase + kFaBN + HD + lrow;  // exchange columns [parity][half], sums
    const int qpos = a.p0 + t0 + r;
    const int first_pos = a.p0 + t0;  // the block's first row: tiles past it need the mask
    float m = -INFINITY, l = 0.f;     // l: this half's running sum
    bool bad = false;
    uint8_t* prow = sm + LY::off_p + (uint32_t)(r >> 3) * 1024 + (uint32_t)(r & 7) * 128;
    auto bar_or = [](bool v) {  // the eight softmax warps; returns whether any passed true
      unsigned rr;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
          "bar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
          : "=r"(rr)
          : "r"((unsigned)v), "r"(kFaSoftmaxWarps * 32)
          : "memory");
      return rr != 0;
    };
    for (int i = 0; i < n_tiles; ++i) {
      bad = bad || !__all_sync(0xffffffffu, fa_wait(a, s_full, (uint32_t)(i & 1)));
      tc_fence_after();
      float sv[kHalf];
      {  // this half's scores: both column blocks in flight, one wait
        uint32_t rr[kHalf / 16][16];
#pragma unroll
        for (int j = 0; j < kHalf / 16; ++j) tmem_ld16(t_s + lrow + hf * kHalf + 16 * j, rr[j]);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < kHalf / 16; ++j) {
          tmem_regs_ready(rr[j]);
#pragma unroll
          for (int e = 0; e < 16; ++e) sv[16 * j + e] = __uint_as_float(rr[j][e]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(s_empty);
      // causal mask (keys after this row's position; only tiles that reach past the
      // block's first row) and the running maximum; scores are in base-2 units already
      const int k0 = (kt0 + i) * kFaBN + hf * kHalf;
      if ((kt0 + i) * kFaBN + kFaBN - 1 > first_pos) {
#pragma unroll
        for (int j = 0; j < kHalf; ++j)
          if (k0 + j > qpos) sv[j] = -INFINITY;
      }
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int j = 0; j < kHalf; ++j) mx4[j & 3] = fmaxf(mx4[j & 3], sv[j]);
      float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      tmem_st1(t_x + 2 * (i & 1) + hf, __float_as_uint(mx));
      tmem_st_wait();
      tc_fence_before();
      bad = bar_or(bad);
      tc_fence_after();
      if (bad) break;
      mx = fmaxf(mx, __uint_as_float(tmem_ld1(t_x + 2 * (i & 1) + (1 - hf))));
      // the reference moves only when the maximum rises by more than 8 (P < 2^8); a row
      // that has seen no key yet keeps m = -inf, alpha = 0 and P = 0 (both halves decide alike)
      const float m_new = mx > m + 8.f ? mx : m;
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = fast_exp2(m - m_use);
      float ps4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < kHalf; ++j) {
        const float pj = fast_exp2(sv[j] - m_use);
        sv[j] = pj;
        ps4[j & 3] += pj;
      }
      l = l * alpha + ((ps4[0] + ps4[1]) + (ps4[2] + ps4[3]));
      m = m_new;
      if (i > 0) {
        // P V of tile i-1 has finished: P's buffer is free and O can be rescaled (a failed
        // wait is carried to the next tile's barrier)
        if (!__all_sync(0xffffffffu, fa_wait(a, o_full, (uint32_t)((i - 1) & 1)))) {
          bad = true;
          continue;
        }
        tc_fence_after();
        if (!__all_sync(0xffffffffu, alpha == 1.f)) {
#pragma unroll 1
          for (int d0 = hf * kHD2; d0 < (hf + 1) * kHD2; d0 += 16) {
            uint32_t rr[16];
            tmem_ld16(t_o + lrow + d0, rr);
            tmem_ld_wait();
            tmem_regs_ready(rr);
#pragma unroll
            for (int e = 0; e < 16; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
            tmem_st16(t_o + lrow + d0, rr);
          }
          tmem_st_wait();
        }
      }
      // this half of P (hi, lo) into shared memory: row r, one 128-byte atom each,
      // 16-byte units of 8 keys swizzled by the row
#pragma unroll
      for (int uu = 0; uu < kHalf / 8; ++uu) {
        const int u = hf * (kHalf / 8) + uu;
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          split2_packed(sv[8 * uu + 2 * e], sv[8 * uu + 2 * e + 1], hw[e], lw[e]);
        const uint32_t off = (uint32_t)((u ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(prow + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(prow + LY::kP1 + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(p_full);
    }
    bool ok = !bad;
    if (ok) ok = __all_sync(0xffffffffu, fa_wait(a, o_full, (uint32_t)((n_tiles - 1) & 1)));
    // the row's sum: both halves, in a fixed order
    tmem_st1(t_x + 4 + hf, __float_as_uint(l));
    tmem_st_wait();
    tc_fence_before();
    ok = !bar_or(!ok);
    tc_fence_after();
    if (!ok && lane == 0) atomicOr(a.err, ERR_TIMEOUT);
    l = __uint_as_float(tmem_ld1(t_x + 4)) + __uint_as_float(tmem_ld1(t_x + 5));
    const bool store = r < nrows;
    uint16_t* oh = a.o_hi + (size_t)(t0 + r) * a.nq * HD + (size_t)h * HD;
    uint16_t* ol = a.o_lo + (size_t)(t0 + r) * a.nq * HD + (size_t)h * HD;
    if (nch == 1) {
      if (ok) {
        tc_fence_after();
        const float inv = 1.0f / l;
#pragma unroll 1
        for (int d0 = hf * kHD2; d0 < (hf + 1) * kHD2; d0 += 16) {
          uint32_t rr[16];
          tmem_ld16(t_o + lrow + d0, rr);
          tmem_ld_wait();
          tmem_regs_ready(rr);
          uint32_t hw[8], lw[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            split2(__uint_as_float(rr[2 * e]) * inv, __uint_as_float(rr[2 * e + 1]) * inv, hw[e],
                   lw[e]);
          if (store) {
            *reinterpret_cast<uint4*>(oh + d0) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(oh + d0 + 8) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
            *reinterpret_cast<uint4*>(ol + d0) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            *reinterpret_cast<uint4*>(ol + d0 + 8) = make_uint4(lw[4], lw[5], lw[6], lw[7]);
          }
        }
      }
    } else {
      // one chunk of several: the unnormalised O and (m, l) of each row, then the last
      // chunk of the block to arrive merges all of them in chunk order
      const size_t slot = ((size_t)h * a.nqb + qb) * a.max_ch;
      float* po = a.part_o + ((slot + chunk) * kFaBQ + r) * HD;
      if (ok) {
        tc_fence_after();
#pragma unroll 1
        for (int d0 = hf * kHD2; d0 < (hf + 1) * kHD2; d0 += 16) {
          uint32_t rr[16];
          tmem_ld16(t_o + lrow + d0, rr);
          tmem_ld_wait();
          tmem_regs_ready(rr);
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4*>(po + d0 + e) =
                make_float4(__uint_as_float(rr[e]), __uint_as_float(rr[e + 1]),
                            __uint_as_float(rr[e + 2]), __uint_as_float(rr[e + 3]));
        }
      }
      if (hf == 0) a.part_ml[(slot + chunk) * kFaBQ + r] = make_float2(m, l);
      __threadfence();
      asm volatile("bar.sync 1, %0;" ::"r"(kFaSoftmaxWarps * 32) : "memory");  // softmax warps
      int* flag = reinterpret_cast<int*>(tslot + 1);
      if (warp == 2 && lane == 0) *flag = atomicAdd(&a.counters[h * a.nqb + qb], 1) == nch - 1;
      asm volatile("bar.sync 1, %0;" ::"r"(kFaSoftmaxWarps * 32) : "memory");
      if (*flag) {
        __threadfence();
        float M = -INFINITY;
        for (int c2 = 0; c2 < nch; ++c2)
          M = fmaxf(M, __ldcg(&a.part_ml[(slot + c2) * kFaBQ + r]).x);
        const float Mu = M == -INFINITY ? 0.f : M;
        float den = 0.f;
        for (int c2 = 0; c2 < nch; ++c2) {
          const float2 ml = __ldcg(&a.part_ml[(slot + c2) * kFaBQ + r]);
          den = fmaf(fast_exp2(ml.x - Mu), ml.y, den);
        }
        const float inv = 1.0f / den;
        // 32 dims at a time, two chunks' rows per round of loads (each chunk's weight
        // exp2(m_c - M) recomputed from its (m, l)), summed in chunk order
#pragma unroll 1
        for (int d0 = hf * kHD2; d0 < (hf + 1) * kHD2; d0 += 32) {
          float acc[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) acc[e] = 0.f;
#pragma unroll 1
          for (int c2 = 0; c2 < nch; c2 += 2) {
            const bool two = c2 + 1 < nch;
            const float2 ml0 = __ldcg(&a.part_ml[(slot + c2) * kFaBQ + r]);
            const float2 ml1 = two ? __ldcg(&a.part_ml[(slot + c2 + 1) * kFaBQ + r])
                                   : make_float2(-INFINITY, 0.f);
            const float4* s0 =
                reinterpret_cast<const float4*>(a.part_o + ((slot + c2) * kFaBQ + r) * HD + d0);
            const float4* s1 = reinterpret_cast<const float4*>(
                a.part_o + ((slot + c2 + (two ? 1 : 0)) * kFaBQ + r) * HD + d0);
            float4 x0[8], x1[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              x0[q] = __ldcg(s0 + q);
              x1[q] = two ? __ldcg(s1 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            const float w0 = fast_exp2(ml0.x - Mu), w1 = two ? fast_exp2(ml1.x - Mu) : 0.f;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              acc[4 * q + 0] = fmaf(w0, x0[q].x, acc[4 * q + 0]);
              acc[4 * q + 1] = fmaf(w0, x0[q].y, acc[4 * q + 1]);
              acc[4 * q + 2] = fmaf(w0, x0[q].z, acc[4 * q + 2]);
              acc[4 * q + 3] = fmaf(w0, x0[q].w, acc[4 * q + 3]);
            }
            if (two) {
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                acc[4 * q + 0] = fmaf(w1, x1[q].x, acc[4 * q + 0]);
                acc[4 * q + 1] = fmaf(w1, x1[q].y, acc[4 * q + 1]);
                acc[4 * q + 2] = fmaf(w1, x1[q].z, acc[4 * q + 2]);
                acc[4 * q + 3] = fmaf(w1, x1[q].w, acc[4 * q + 3]);
              }
            }
          }
#pragma unroll
          for (int e8 = 0; e8 < 32; e8 += 8) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              split2(acc[e8 + 2 * e] * inv, acc[e8 + 2 * e + 1] * inv, hw[e], lw[e]);
            if (store) {
              *reinterpret_cast<uint4*>(oh + d0 + e8) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
              *reinterpret_cast<uint4*>(ol + d0 + e8) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
          }
        }
        if (warp == 2 && lane == 0) a.counters[h * a.nqb + qb] = 0;  // ready for the next launch
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// One layer's K and V cache as the attention's operands: V transposed and split,
// V^T hi/lo [nkv][HD][kv_rows], for keys [0, n) (keys [n, next multiple of 32) are
// written as 0); and K rows split, hi/lo [nkv][kv_rows][HD], for keys [0, k_end) only
// (the keys cached before this pass: the row kernel writes the new keys' split rows
// itself). One CTA per (32 keys, KV head).
template <int HD, bool KB>
__global__ void __launch_bounds__(256) kv_split_kernel(const void* kc_, const void* vc_, int cap,
                                                       int n, int k_end, int kv_rows,
                                                       uint16_t* kh, uint16_t* kl, uint16_t* vth,
                                                       uint16_t* vtl) {
  using KV = KvElem<KB>;
  using KT = typename KV::T;
  const KT* kc = reinterpret_cast<const KT*>(kc_);
  const KT* vc = reinterpret_cast<const KT*>(vc_);
  __shared__ float tile[32][HD + 1];
  const int k0 = blockIdx.x * 32, kvh = blockIdx.y;
  if (k0 < k_end)
  for (int i = threadIdx.x; i < 32 * HD / 2; i += 256) {
    const int kk = i / (HD / 2), d = (i % (HD / 2)) * 2;
    if (k0 + kk >= k_end) continue;
    const float2 v = KV::load2(kc + ((size_t)kvh * cap + k0 + kk) * HD + d);
    uint32_t hi, lo;
    split2(v.x, v.y, hi, lo);
    const size_t o = ((size_t)kvh * kv_rows + k0 + kk) * HD + d;
    *reinterpret_cast<uint32_t*>(kh + o) = hi;
    *reinterpret_cast<uint32_t*>(kl + o) = lo;
  }
  for (int i = threadIdx.x; i < 32 * HD; i += 256) {
    const int kk = i / HD, d = i % HD;
    tile[kk][d] = k0 + kk < n ? KV::load(vc + ((size_t)kvh * cap + k0 + kk) * HD + d) : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 16 * HD; i += 256) {
    const int d = i / 16, kk = (i % 16) * 2;
    uint32_t hi, lo;
    split2(tile[kk][d], tile[kk + 1][d], hi, lo);
    const size_t o = ((size_t)kvh * HD + d) * kv_rows + k0 + kk;
    *reinterpret_cast<uint32_t*>(vth + o) = hi;
    *reinterpret_cast<uint32_t*>(vtl + o) = lo;
  }
}

// int4 g128 rows as the decode step stores them (K/2 nibble bytes, then K/128 bf16
// scales, padded) -> the exact dequantised value w = (nibble - 8) * scale as two bf16
// terms, hi = bf16(w) and lo = bf16(w - hi), in row-major planes [rows][K]. w has at
// most 11 significant bits (a 4-bit integer times an 8-bit bf16 significand), so
// hi + lo == w exactly. One thread per 8 consecutive inputs.
__global__ void __launch_bounds__(256) dequant_int4_split_kernel(const uint8_t* src, int rows,
                                                                 int K, uint16_t* hi,
                                                                 uint16_t* lo) {
  const uint32_t rb = int4_row_bytes(K);
  const long long i = (long long)blockIdx.x * 256 + threadIdx.x;
  const int per_row = K / 8;
  if (i >= (long long)rows * per_row) return;
  const int r = (int)(i / per_row), c = (int)(i % per_row) * 8;
  const uint8_t* row = src + (size_t)r * rb;
  const uint32_t w = *reinterpret_cast<const uint32_t*>(row + c / 2);
  const float sc = bf16f(*reinterpret_cast<const uint16_t*>(row + K / 2 + (c >> 7) * 2));
  uint32_t h[4], l[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float v0 = (float)((int)((w >> (8 * e)) & 15u) - 8) * sc;  // element c + 2e
    const float v1 = (float)((int)((w >> (8 * e + 4)) & 15u) - 8) * sc;
    split2(v0, v1, h[e], l[e]);
  }
  const size_t o = (size_t)r * K + c;
  *reinterpret_cast<uint4*>(hi + o) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(lo + o) = make_uint4(l[0], l[1], l[2], l[3]);
}

cudaError_t launch_dequant_int4_split(const uint8_t* src, int rows, int K, uint16_t* hi,
                                      uint16_t* lo, cudaStream_t s) {
  const long long n = (long long)rows * (K / 8);
  if (n <= 0) return cudaSuccess;
  dequant_int4_split_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(src, rows, K, hi, lo);
  return cudaGetLastError();
}

__global__ void set_int_kernel(int* p, int v) { *p = v; }

// ------------------------------------------------------------------ launchers
cudaError_t launch_embed_rows(const int* ids, int T, const uint16_t* table, int V, int H,
                              float* X, float* cap, int row0, int* err, cudaStream_t s) {
  embed_rows_kernel<<<T, 256, 0, s>>>(ids, table, V, H, X, cap, row0, err);
  return cudaGetLastError();
}
cudaError_t launch_rmsnorm_rows(const float* X, int T, int H, const uint16_t* g, float eps,
                                uint16_t* hi, uint16_t* lo, float* f32, int f32_row0,
                                cudaStream_t s) {
  rmsnorm_rows_kernel<<<T, 256, 0, s>>>(X, H, g, eps, hi, lo, f32, f32_row0);
  return cudaGetLastError();
}
cudaError_t launch_qk_rope_kv_rows(const float* QKV, int T, int p0, int nq, int nkv, int hd,
                                   const uint16_t* qn, const uint16_t* kn, float eps,
                                   const float2* rope, uint16_t* q_hi, uint16_t* q_lo,
                                   void* kc, void* vc, bool kv_bf16, int cap,
                                   uint16_t* kv_split, cudaStream_t s) {
  const int kv_rows = attn_kv_rows(cap);
  uint16_t* k_hi = kv_split;
  uint16_t* k_lo = kv_split + (size_t)nkv * hd * kv_rows;
#define QW_ROPE_ROWS(HDV, KBV)                                                                  \
  qk_rope_kv_rows_kernel<HDV, KBV><<<T, 256, 0, s>>>(QKV, p0, nq, nkv, qn, kn, eps, rope, q_hi, \
                                                     q_lo, kc, vc, cap, k_hi, k_lo, kv_rows)
  if (hd == 64 && kv_bf16) QW_ROPE_ROWS(64, true);
  else if (hd == 64) QW_ROPE_ROWS(64, false);
  else if (hd == 128 && kv_bf16) QW_ROPE_ROWS(128, true);
  else if (hd == 128) QW_ROPE_ROWS(128, false);
  else return cudaErrorInvalidValue;
#undef QW_ROPE_ROWS
  return cudaGetLastError();
}
int attn_kv_rows(int cap) { return (cap + kFaBN - 1) / kFaBN * kFaBN; }
size_t attn_kv_bytes(int nkv, int hd, int cap) {
  return (size_t)4 * nkv * hd * attn_kv_rows(cap) * 2;
}
int attn_max_chunks(int cap) { return (attn_kv_rows(cap) / kFaBN + kFaChunk - 1) / kFaChunk; }
int attn_max_qblocks(int max_t) { return (max_t + kFaBQ - 1) / kFaBQ; }
size_t attn_part_bytes(int nq, int max_t, int cap, int hd) {
  const size_t slots = (size_t)nq * attn_max_qblocks(max_t) * attn_max_chunks(cap);
  return slots * kFaBQ * ((size_t)hd * 4 + 8) + (size_t)nq * attn_max_qblocks(max_t) * 4;
}
cudaError_t launch_attn_prefill(const FaMaps& maps, const void* kc, const void* vc, bool kv_bf16,
                                uint16_t* kv_split, void* part, int max_t, int cap, int p0,
                                int T, int nq, int nkv, int hd, uint16_t* o_hi, uint16_t* o_lo,
                                int* err, uint64_t wait_ns, cudaStream_t s) {
  if (T <= 0 || nkv <= 0 || nq % nkv) return cudaErrorInvalidValue;
  const int n = p0 + T;  // keys this pass reads; split up to the tile the last one is in
  const int kv_rows = attn_kv_rows(cap);
  const size_t plane = (size_t)nkv * hd * kv_rows;
  const dim3 sgrid((n + kFaBN - 1) / kFaBN * (kFaBN / 32), nkv);
  const int nqb = (T + kFaBQ - 1) / kFaBQ;
  int items = 0;  // (query block, key chunk) pairs per head
  for (int qb = 0; qb < nqb; ++qb) {
    const int nr = min(kFaBQ, T - qb * kFaBQ);
    const int bt = (p0 + qb * kFaBQ + nr - 1) / kFaBN + 1;
    items += (bt + kFaChunk - 1) / kFaChunk;
  }
  const dim3 grid(nq, items);
  FaArgs a{p0, T, nq, nkv, kv_rows, o_hi, o_lo, err, wait_ns};
  a.nqb = nqb;
  a.max_ch = attn_max_chunks(cap);
  const size_t slots = (size_t)nq * attn_max_qblocks(max_t) * a.max_ch;
  a.part_o = reinterpret_cast<float*>(part);
  a.part_ml = reinterpret_cast<float2*>(a.part_o + slots * kFaBQ * hd);
  a.counters = reinterpret_cast<int*>(a.part_ml + slots * kFaBQ);
  if (nqb > attn_max_qblocks(max_t)) return cudaErrorInvalidValue;
  uint16_t *kh = kv_split, *kl = kv_split + plane, *vth = kl + plane, *vtl = vth + plane;
  if (hd == 64) {
    if (kv_bf16)
      kv_split_kernel<64, true><<<sgrid, 256, 0, s>>>(kc, vc, cap, n, p0, kv_rows, kh, kl, vth, vtl);
    else
      kv_split_kernel<64, false><<<sgrid, 256, 0, s>>>(kc, vc, cap, n, p0, kv_rows, kh, kl, vth, vtl);
    attn_prefill_fa_kernel<64><<<grid, kFaThreads, FaLayout<64>::bytes, s>>>(maps, a);
  } else if (hd == 128) {
    if (kv_bf16)
      kv_split_kernel<128, true><<<sgrid, 256, 0, s>>>(kc, vc, cap, n, p0, kv_rows, kh, kl, vth, vtl);
    else
      kv_split_kernel<128, false><<<sgrid, 256, 0, s>>>(kc, vc, cap, n, p0, kv_rows, kh, kl, vth,
                                                        vtl);
    attn_prefill_fa_kernel<128><<<grid, kFaThreads, FaLayout<128>::bytes, s>>>(maps, a);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}
bool make_attn_maps(FaMaps* m, const uint16_t* q_hi, const uint16_t* q_lo, int max_t, int nq,
                    const uint16_t* kv_split, int nkv, int hd, int cap) {
  const int kv_rows = attn_kv_rows(cap);
  const size_t plane = (size_t)nkv * hd * kv_rows;
  const uint64_t qd = (uint64_t)nq * hd;
  return make_tmap_bf16_2d(&m->q_hi, q_hi, (uint64_t)max_t, qd, kFaBQ) &&
         make_tmap_bf16_2d(&m->q_lo, q_lo, (uint64_t)max_t, qd, kFaBQ) &&
         make_tmap_bf16_2d(&m->k_hi, kv_split, (uint64_t)nkv * kv_rows, hd, kFaBN) &&
         make_tmap_bf16_2d(&m->k_lo, kv_split + plane, (uint64_t)nkv * kv_rows, hd, kFaBN) &&
         make_tmap_bf16_2d(&m->vt_hi, kv_split + 2 * plane, (uint64_t)nkv * hd, kv_rows,
                           (uint32_t)hd) &&
         make_tmap_bf16_2d(&m->vt_lo, kv_split + 3 * plane, (uint64_t)nkv * hd, kv_rows,
                           (uint32_t)hd);
}
cudaError_t launch_set_int(int* p, int v, cudaStream_t s) {
  set_int_kernel<<<1, 1, 0, s>>>(p, v);
  return cudaGetLastError();
}
cudaError_t set_prefill_attributes() {
  static_assert(FaLayout<128>::bytes <= 227 * 1024, "attention tiles fit one CTA's shared memory");
  cudaError_t e = cudaFuncSetAttribute(attn_prefill_fa_kernel<64>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)FaLayout<64>::bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_prefill_fa_kernel<128>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)FaLayout<128>::bytes);
  return e;
}

// ------------------------------------------------------------------ GEMM host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Row-major bf16 [rows, cols] (cols contiguous), boxes of 64 columns x box_rows rows,
// 128-byte swizzle, zero fill outside the tensor.
bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                       uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || (cols * 2) % 16 || (reinterpret_cast<uintptr_t>(base) & 15) || box_rows > 256)
    return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)GBK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr size_t kGemmSmemBudget = 200 * 1024;

static int gemm_stages(int bn, int a_split, int b_split) {
  const size_t stage = (size_t)a_split * kATileBytes + (size_t)b_split * bn * GBK * 2;
  int ns = (int)((kGemmSmemBudget - 2048) / stage);
  return ns < 2 ? 2 : (ns > 8 ? 8 : ns);
}
static size_t gemm_smem(int bn, int a_split, int b_split, int ns) {
  return (size_t)ns * ((size_t)a_split * kATileBytes + (size_t)b_split * bn * GBK * 2) + 1024 +
         256;
}

template <int BN, int EPI>
static cudaError_t launch_gemm_t(const CUtensorMap& a_hi, const CUtensorMap& a_lo,
                                 const CUtensorMap& b, const CUtensorMap& b_lo, const GemmArgs& g,
                                 cudaStream_t s) {
  // split-K: split index slowest, so every split's CTAs come after the previous split's
  const dim3 grid((g.N + BN - 1) / BN, (g.M + GBM - 1) / GBM, g.ksplit);
  gemm_tc_kernel<BN, EPI><<<grid, 192, gemm_smem(BN, g.a_split, g.b_split, g.n_stages), s>>>(
      a_hi, a_lo, b, b_lo, g);
  return cudaGetLastError();
}

template <int BN>
static cudaError_t launch_gemm_bn(int epi, const CUtensorMap& a_hi, const CUtensorMap& a_lo,
                                  const CUtensorMap& b, const CUtensorMap& b_lo,
                                  const GemmArgs& g, cudaStream_t s) {
  switch (epi) {
    case GEPI_STORE: return launch_gemm_t<BN, GEPI_STORE>(a_hi, a_lo, b, b_lo, g, s);
    case GEPI_RESID: return launch_gemm_t<BN, GEPI_RESID>(a_hi, a_lo, b, b_lo, g, s);
    case GEPI_SWIGLU: return launch_gemm_t<BN, GEPI_SWIGLU>(a_hi, a_lo, b, b_lo, g, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm(int bn, int epi, const CUtensorMap& a_hi, const CUtensorMap& a_lo,
                        const CUtensorMap& b, const CUtensorMap* b_lo, GemmArgs g,
                        cudaStream_t s) {
  if (g.M <= 0 || g.N <= 0 || g.K <= 0 || (g.a_split != 1 && g.a_split != 2))
    return cudaErrorInvalidValue;
  if (epi == GEPI_SWIGLU && (g.N % 2)) return cudaErrorInvalidValue;
  g.b_split = b_lo ? 2 : 1;
  const CUtensorMap& bl = b_lo ? *b_lo : b;
  const int kt_all = (g.K + GBK - 1) / GBK;  // every split gets at least one k-tile
  g.ksplit = epi == GEPI_RESID && g.flags != nullptr ? std::max(1, std::min(g.ksplit, kt_all)) : 1;
  g.n_stages = gemm_stages(bn, g.a_split, g.b_split);
  if (bn == 64) return launch_gemm_bn<64>(epi, a_hi, a_lo, b, bl, g, s);
  if (bn == 128) return launch_gemm_bn<128>(epi, a_hi, a_lo, b, bl, g, s);
  if (bn == 256) return launch_gemm_bn<256>(epi, a_hi, a_lo, b, bl, g, s);
  return cudaErrorInvalidValue;
}

template <int BN>
static cudaError_t gemm_attrs_bn() {
  int bytes = 0;
  for (int split = 1; split <= 2; ++split)
    for (int bsplit = 1; bsplit <= 2; ++bsplit) {
      const int b = (int)gemm_smem(BN, split, bsplit, gemm_stages(BN, split, bsplit));
      bytes = b > bytes ? b : bytes;
    }
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<BN, GEPI_STORE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_tc_kernel<BN, GEPI_RESID>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_tc_kernel<BN, GEPI_SWIGLU>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  return e;
}

static __device__ int g_gemm_op_err;

int* gemm_op_err_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_gemm_op_err) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

cudaError_t set_gemm_attributes() {
  cudaError_t e = gemm_attrs_bn<64>();
  if (e == cudaSuccess) e = gemm_attrs_bn<128>();
  if (e == cudaSuccess) e = gemm_attrs_bn<256>();
  return e;
}

}  // namespace qw
