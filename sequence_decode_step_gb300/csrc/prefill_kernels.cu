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
                   const __grid_constant__ CUtensorMap tb, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int NS = a.n_stages;
  const uint32_t stage_bytes = (uint32_t)a.a_split * kATileBytes + (uint32_t)BN * GBK * 2;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * stage_bytes);
  uint64_t* empty = full + NS;
  uint64_t* accf = empty + NS;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(accf + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * GBM, n0 = blockIdx.x * BN;
  const int KT = (a.K + GBK - 1) / GBK;

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
      mbar_expect_tx(&full[s], stage_bytes);
      tma_load_2d(st, &ta_hi, kt * GBK, m0, &full[s]);
      if (a.a_split == 2) tma_load_2d(st + kATileBytes, &ta_lo, kt * GBK, m0, &full[s]);
      tma_load_2d(st + a.a_split * kATileBytes, &tb, kt * GBK, n0, &full[s]);
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
        tc_mma_bf16(tbase, sw128_kmajor_desc(sa + k * 32), bd, idesc, (kt | k) != 0);
        if (a.a_split == 2)
          tc_mma_bf16(tbase, sw128_kmajor_desc(sa + kATileBytes + k * 32), bd, idesc, 1);
      }
      tc_commit(&empty[s]);  // the stage is free once these MMAs have read it
    }
    tc_commit(accf);  // the accumulator is final once every MMA above completed
    // TMEM is released below only after the MMAs have finished.
    mbar_wait(accf, 0, kDrainNs);
  } else if (warp >= 2) {
    // ---- epilogue: warp w reads TMEM lanes [32 (w % 4), +32) = rows of the tile
    const bool ok = mbar_wait(accf, 0, a.wait_ns);
    if (!ok && lane == 0) atomicOr(a.err, ERR_TIMEOUT);
    tc_fence_after();
    const int q = warp & 3;
    const int row = m0 + q * 32 + lane;
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 16) {
      uint32_t r[16];
      tmem_ld16(tbase + ((uint32_t)(q * 32) << 16) + (uint32_t)c0, r);
      tmem_ld_wait();
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
          for (int j = 0; j < 4; ++j) cur[j] = *reinterpret_cast<const float4*>(o + 4 * j);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float4 n4 = make_float4(cur[j].x + v[4 * j], cur[j].y + v[4 * j + 1],
                                          cur[j].z + v[4 * j + 2], cur[j].w + v[4 * j + 3]);
            *reinterpret_cast<float4*>(o + 4 * j) = n4;
            if (a.cap_out)
              *reinterpret_cast<float4*>(a.cap_out + (size_t)(a.cap_row0 + row) * a.ldo + col0 + 4 * j) = n4;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j < nv) {
              const float nvl = o[j] + v[j];
              o[j] = nvl;
              if (a.cap_out) a.cap_out[(size_t)(a.cap_row0 + row) * a.ldo + col0 + j] = nvl;
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
// 1/sqrt(hd) into Q [T][nq][hd]; k and v appended to the cache at their position.
template <int HD>
__global__ void __launch_bounds__(256) qk_rope_kv_rows_kernel(
    const float* QKV, int p0, int nq, int nkv, const uint16_t* q_norm, const uint16_t* k_norm,
    float eps, const float2* rope, float* Q, float* kc, float* vc, int cap) {
  constexpr int EPL = HD / 32;
  const int t = blockIdx.x, pos = p0 + t;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* row = QKV + (size_t)t * (nq + 2 * nkv) * HD;
  const float scale = 1.0f / sqrtf((float)HD);
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
      for (int e = 0; e < EPL; ++e) Q[((size_t)t * nq + hh) * HD + lane + 32 * e] = v[e] * scale;
    } else {
      float* dst = kc + ((size_t)(hh - nq) * cap + pos) * HD;
#pragma unroll
      for (int e = 0; e < EPL; ++e) dst[lane + 32 * e] = v[e];
    }
  }
  const float* vsrc = row + (size_t)(nq + nkv) * HD;
  for (int i = threadIdx.x; i < nkv * HD; i += 256)
    vc[((size_t)(i / HD) * cap + pos) * HD + (i % HD)] = vsrc[i];
}

// ---- causal attention on tensor cores (mma.sync m16n8k16, bf16 operands, f32 accumulate)
// Every f32 operand x enters as two bf16 terms hi = bf16(x), lo = bf16(x - hi); a product
// a.b is formed as a_hi.b_hi + a_hi.b_lo + a_lo.b_hi (the lo.lo term is below f32
// rounding of the sum), so scores and outputs carry about 16 bits of the f32 values.
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
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// K and V of keys [0, n) of every KV head, split into bf16 hi/lo rows of HD + 8
// elements (the padding keeps the attention kernel's ldmatrix rows in distinct
// banks): dst[4][nkv][rows][HD + 8] = {K hi, K lo, V hi, V lo}. One warp per (key, head).
template <int HD>
__global__ void __launch_bounds__(256) kv_split_kernel(const float* kc, const float* vc, int cap,
                                                       int n, int nkv, int rows, uint16_t* dst) {
  constexpr int LD = HD + 8, EPL = HD / 32;
  const int wid = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (wid >= n * nkv) return;
  const int key = wid % n, kvh = wid / n;
  const size_t plane = (size_t)nkv * rows * LD;
  const size_t row = ((size_t)kvh * rows + key) * LD;
  const float* ks = kc + ((size_t)kvh * cap + key) * HD;
  const float* vs = vc + ((size_t)kvh * cap + key) * HD;
#pragma unroll
  for (int e = 0; e < EPL; e += 2) {
    const int d = lane * EPL + e;
    const float2 k2 = *reinterpret_cast<const float2*>(ks + d);
    const float2 v2 = *reinterpret_cast<const float2*>(vs + d);
    uint32_t kh, kl, vh, vl;
    split2(k2.x, k2.y, kh, kl);
    split2(v2.x, v2.y, vh, vl);
    *reinterpret_cast<uint32_t*>(dst + row + d) = kh;
    *reinterpret_cast<uint32_t*>(dst + plane + row + d) = kl;
    *reinterpret_cast<uint32_t*>(dst + 2 * plane + row + d) = vh;
    *reinterpret_cast<uint32_t*>(dst + 3 * plane + row + d) = vl;
  }
}

// One CTA: 64 query rows of one head (4 warps x 16 rows), keys in tiles of BK up to
// the block's last position. The tiles of pre-split K/V rows (kv_split_kernel) come
// in by one bulk copy per array into a double buffer, the next tile's copies issued
// before the current tile is used. Scores S = Q.K^T and the online softmax stay in
// registers (the m16n8 accumulator layout is reused as the A fragment of P.V).
// Split of the causal work: query block qb reads n_tiles(qb) key tiles; they are cut
// into chunks of at most CH tiles, one CTA each, listed heavy block first.
struct AttnSplit {
  float* part_o;     // [nq][nqb][max_ch][64][HD] unnormalised partial outputs
  float2* part_ml;   // [nq][nqb][max_ch][64] (row max, row sum)
  int* counters;     // [nq][nqb] arrivals, 0 between launches
  int max_ch, ch;
};

template <int HD, int BK>
__global__ void __launch_bounds__(128) attn_prefill_tc_kernel(const float* Q,
                                                              const uint16_t* kvs, int rows,
                                                              int p0, int T, int nq, int nkv,
                                                              uint16_t* o_hi, uint16_t* o_lo,
                                                              const AttnSplit sp, int* err,
                                                              uint64_t wait_ns) {
  constexpr int BQ = 64, LD = HD + 8, KS = HD / 16, NO = HD / 8;
  constexpr uint32_t kArr = (uint32_t)BK * LD * 2;  // bytes of one array's tile
  extern __shared__ __align__(128) uint8_t smraw[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smraw + 2 * 4 * kArr);  // [2]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  // this CTA's (query block, key chunk): blocks from the last (heaviest) down
  const int nqb = (T + BQ - 1) / BQ;
  int qb = nqb - 1, chunk = blockIdx.x, nch = 1;
  for (;; --qb) {
    const int nr = min(BQ, T - qb * BQ);
    const int nt = (p0 + qb * BQ + nr - 1) / BK + 1;
    nch = (nt + sp.ch - 1) / sp.ch;
    if (chunk < nch || qb == 0) break;
    chunk -= nch;
  }
  const int t0 = qb * BQ, h = blockIdx.y, kvh = h / (nq / nkv);
  const int nrows = min(BQ, T - t0);
  const int last_key = p0 + t0 + nrows - 1;
  const int r0 = t0 + warp * 16 + g;  // this lane's two rows: r0 and r0 + 8 (block-relative t)
  const size_t plane = (size_t)nkv * rows * LD;
  const uint16_t* src = kvs + (size_t)kvh * rows * LD;
  const int kt0 = chunk * sp.ch, kt1 = min(last_key / BK + 1, kt0 + sp.ch);
  const int n_tiles = kt1 - kt0;
  // a whole tile of each array (rows past the last key hold zeros or older keys:
  // finite, and masked); the i-th tile of the chunk uses buffer i & 1, whose
  // barrier completes phase i >> 1
  auto issue = [&](int i) {
    const int b = i & 1, kt = kt0 + i;
    mbar_expect_tx(&bar[b], 4 * kArr);
#pragma unroll
    for (int arr = 0; arr < 4; ++arr)
      bulk_load(smraw + (size_t)(b * 4 + arr) * kArr, src + arr * plane + (size_t)kt * BK * LD,
                kArr, &bar[b]);
  };
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_barrier_init();
    issue(0);
    if (n_tiles > 1) issue(1);
  }
  // Q fragments (A operand, row-major 16 x 16 per k-step), split hi/lo
  uint32_t qh[KS][4], ql[KS][4];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int row = r0 + (j & 1) * 8, col = ks * 16 + 2 * t + (j >> 1) * 8;
      float2 v = make_float2(0.f, 0.f);
      if (row < T) v = *reinterpret_cast<const float2*>(Q + ((size_t)row * nq + h) * HD + col);
      split2(v.x, v.y, qh[ks][j], ql[ks][j]);
    }
  }
  __syncthreads();  // barrier initialisation visible to all threads
  float o[NO][4];
#pragma unroll
  for (int nb = 0; nb < NO; ++nb)
#pragma unroll
    for (int j = 0; j < 4; ++j) o[nb][j] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int qp0 = p0 + r0, qp1 = qp0 + 8;
  bool ok = true;
  for (int i = 0; i < n_tiles; ++i) {
    const int k0 = (kt0 + i) * BK, b = i & 1;
    const bool got = mbar_wait(&bar[b], (uint32_t)((i >> 1) & 1), wait_ns);
    ok = __syncthreads_and(got) != 0;  // one decision for the whole block
    if (!ok) {  // gave up: outputs invalid, the host sees the error word
      if (tid == 0) atomicOr(err, ERR_TIMEOUT);
      break;
    }
    const uint16_t* Kh = reinterpret_cast<const uint16_t*>(smraw + (size_t)(b * 4 + 0) * kArr);
    const uint16_t* Kl = reinterpret_cast<const uint16_t*>(smraw + (size_t)(b * 4 + 1) * kArr);
    const uint16_t* Vh = reinterpret_cast<const uint16_t*>(smraw + (size_t)(b * 4 + 2) * kArr);
    const uint16_t* Vl = reinterpret_cast<const uint16_t*>(smraw + (size_t)(b * 4 + 3) * kArr);
    // S = Q K^T: 8 n-blocks of 8 keys
    float sc[BK / 8][4];
#pragma unroll
    for (int nb = 0; nb < BK / 8; ++nb)
#pragma unroll
      for (int j = 0; j < 4; ++j) sc[nb][j] = 0.f;
    const int mrow = lane & 7, mi = lane >> 3;  // ldmatrix: matrix mi, row mrow
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
      for (int nb = 0; nb < BK / 8; nb += 2) {
        const int key = (nb + (mi >> 1)) * 8 + mrow, col = ks * 16 + (mi & 1) * 8;
        uint32_t bh0, bh1, bh2, bh3, bl0, bl1, bl2, bl3;
        ldsm_x4(smem_addr(Kh + key * LD + col), bh0, bh1, bh2, bh3);
        ldsm_x4(smem_addr(Kl + key * LD + col), bl0, bl1, bl2, bl3);
        mma_bf16(sc[nb], qh[ks], bh0, bh1);
        mma_bf16(sc[nb], qh[ks], bl0, bl1);
        mma_bf16(sc[nb], ql[ks], bh0, bh1);
        mma_bf16(sc[nb + 1], qh[ks], bh2, bh3);
        mma_bf16(sc[nb + 1], qh[ks], bl2, bl3);
        mma_bf16(sc[nb + 1], ql[ks], bh2, bh3);
      }
    }
    // causal mask and online softmax (rows r0 and r0 + 8; a quad of lanes shares a row)
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < BK / 8; ++nb) {
      const int key = k0 + nb * 8 + 2 * t;
      if (key > qp0) sc[nb][0] = -INFINITY;
      if (key + 1 > qp0) sc[nb][1] = -INFINITY;
      if (key > qp1) sc[nb][2] = -INFINITY;
      if (key + 1 > qp1) sc[nb][3] = -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(sc[nb][0], sc[nb][1]));
      mx1 = fmaxf(mx1, fmaxf(sc[nb][2], sc[nb][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = m0 == -INFINITY ? 0.f : expf(m0 - mn0);
    const float al1 = m1 == -INFINITY ? 0.f : expf(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int nb = 0; nb < BK / 8; ++nb) {
      sc[nb][0] = sc[nb][0] == -INFINITY ? 0.f : expf(sc[nb][0] - mn0);
      sc[nb][1] = sc[nb][1] == -INFINITY ? 0.f : expf(sc[nb][1] - mn0);
      sc[nb][2] = sc[nb][2] == -INFINITY ? 0.f : expf(sc[nb][2] - mn1);
      sc[nb][3] = sc[nb][3] == -INFINITY ? 0.f : expf(sc[nb][3] - mn1);
      rs0 += sc[nb][0] + sc[nb][1];
      rs1 += sc[nb][2] + sc[nb][3];
    }
    l0 = l0 * al0 + rs0;  // per-lane partial row sums; the quad adds them at the end
    l1 = l1 * al1 + rs1;
#pragma unroll
    for (int nb = 0; nb < NO; ++nb) {
      o[nb][0] *= al0;
      o[nb][1] *= al0;
      o[nb][2] *= al1;
      o[nb][3] *= al1;
    }
    // O += P V: 4 k-steps of 16 keys; P's A fragment comes from two score n-blocks
#pragma unroll
    for (int kk = 0; kk < BK / 16; ++kk) {
      uint32_t ph[4], pl[4];
      split2(sc[2 * kk][0], sc[2 * kk][1], ph[0], pl[0]);
      split2(sc[2 * kk][2], sc[2 * kk][3], ph[1], pl[1]);
      split2(sc[2 * kk + 1][0], sc[2 * kk + 1][1], ph[2], pl[2]);
      split2(sc[2 * kk + 1][2], sc[2 * kk + 1][3], ph[3], pl[3]);
#pragma unroll
      for (int nb = 0; nb < NO; nb += 2) {
        // V rows kk*16 .. +15 (keys), columns nb*8 .. +15 (dims), transposed fragments
        const int key = kk * 16 + (mi & 1) * 8 + mrow, col = (nb + (mi >> 1)) * 8;
        uint32_t bh0, bh1, bh2, bh3, bl0, bl1, bl2, bl3;
        ldsm_x4_t(smem_addr(Vh + key * LD + col), bh0, bh1, bh2, bh3);
        ldsm_x4_t(smem_addr(Vl + key * LD + col), bl0, bl1, bl2, bl3);
        mma_bf16(o[nb], ph, bh0, bh1);
        mma_bf16(o[nb], ph, bl0, bl1);
        mma_bf16(o[nb], pl, bh0, bh1);
        mma_bf16(o[nb + 1], ph, bh2, bh3);
        mma_bf16(o[nb + 1], ph, bl2, bl3);
        mma_bf16(o[nb + 1], pl, bh2, bh3);
      }
    }
    // buffer b is free once every warp has read it (generic proxy; ordered before the
    // bulk copy that refills it): refill it with tile kt + 2
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (tid == 0 && i + 2 < n_tiles) issue(i + 2);
  }
  if (!ok) {  // copies may still be in flight into this CTA's shared memory
    if (tid == 0) {
      for (int b = 0; b < 2; ++b) {
        mbar_wait(&bar[b], 0, kDrainNs);
        mbar_wait(&bar[b], 1, kDrainNs);
      }
      // still arrive, so the block's counter is back at 0 for the next launch
      if (nch > 1 && atomicAdd(&sp.counters[h * nqb + qb], 1) == nch - 1)
        sp.counters[h * nqb + qb] = 0;
    }
    return;
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  if (nch > 1) {  // one chunk of several: partial results, the last to arrive merges
    const int rr = warp * 16 + g;  // block-relative rows rr and rr + 8
    const size_t slot = ((size_t)h * nqb + qb) * sp.max_ch;
    float* po = sp.part_o + (slot + chunk) * BQ * HD;
#pragma unroll
    for (int nb = 0; nb < NO; ++nb) {
      const int d = nb * 8 + 2 * t;
      *reinterpret_cast<float2*>(po + rr * HD + d) = make_float2(o[nb][0], o[nb][1]);
      *reinterpret_cast<float2*>(po + (rr + 8) * HD + d) = make_float2(o[nb][2], o[nb][3]);
    }
    if (t == 0) {
      sp.part_ml[(slot + chunk) * BQ + rr] = make_float2(m0, l0);
      sp.part_ml[(slot + chunk) * BQ + rr + 8] = make_float2(m1, l1);
    }
    __threadfence();
    __syncthreads();
    int* last = reinterpret_cast<int*>(smraw);
    if (tid == 0) *last = atomicAdd(&sp.counters[h * nqb + qb], 1) == nch - 1;
    __syncthreads();
    if (!*last) return;
    __threadfence();
    // merge in chunk order: per row, weights exp(m_c - M) / sum_c exp(m_c - M) l_c
    float* wsm = reinterpret_cast<float*>(smraw) + 4;  // [BQ][nch]
    if (tid < BQ) {
      float M = -INFINITY;
      for (int c2 = 0; c2 < nch; ++c2) M = fmaxf(M, __ldcg(&sp.part_ml[(slot + c2) * BQ + tid]).x);
      float den = 0.f;
      for (int c2 = 0; c2 < nch; ++c2) {
        const float2 ml = __ldcg(&sp.part_ml[(slot + c2) * BQ + tid]);
        const float w = ml.x == -INFINITY ? 0.f : expf(ml.x - M);
        wsm[tid * nch + c2] = w;
        den = fmaf(w, ml.y, den);
      }
      const float inv = 1.0f / den;
      for (int c2 = 0; c2 < nch; ++c2) wsm[tid * nch + c2] *= inv;
    }
    __syncthreads();
    for (int idx = 2 * tid; idx < BQ * HD; idx += 2 * 128) {
      const int rr2 = idx / HD, d = idx % HD;
      float a0 = 0.f, a1 = 0.f;
      for (int c2 = 0; c2 < nch; ++c2) {
        const float2 v = __ldcg(reinterpret_cast<const float2*>(
            sp.part_o + (slot + c2) * BQ * HD + rr2 * HD + d));
        const float w = wsm[rr2 * nch + c2];
        a0 = fmaf(w, v.x, a0);
        a1 = fmaf(w, v.y, a1);
      }
      if (rr2 < nrows) {
        uint32_t hi, lo;
        split2(a0, a1, hi, lo);
        const size_t off = (size_t)(t0 + rr2) * nq * HD + h * HD + d;
        *reinterpret_cast<uint32_t*>(o_hi + off) = hi;
        *reinterpret_cast<uint32_t*>(o_lo + off) = lo;
      }
    }
    if (tid == 0) sp.counters[h * nqb + qb] = 0;  // not used again in this launch
    return;
  }
  const float inv0 = 1.0f / l0, inv1 = 1.0f / l1;
#pragma unroll
  for (int nb = 0; nb < NO; ++nb) {
    const int col = h * HD + nb * 8 + 2 * t;
    if (r0 < t0 + nrows) {
      uint32_t hi, lo;
      split2(o[nb][0] * inv0, o[nb][1] * inv0, hi, lo);
      *reinterpret_cast<uint32_t*>(o_hi + (size_t)r0 * nq * HD + col) = hi;
      *reinterpret_cast<uint32_t*>(o_lo + (size_t)r0 * nq * HD + col) = lo;
    }
    if (r0 + 8 < t0 + nrows) {
      uint32_t hi, lo;
      split2(o[nb][2] * inv1, o[nb][3] * inv1, hi, lo);
      *reinterpret_cast<uint32_t*>(o_hi + (size_t)(r0 + 8) * nq * HD + col) = hi;
      *reinterpret_cast<uint32_t*>(o_lo + (size_t)(r0 + 8) * nq * HD + col) = lo;
    }
  }
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
                                   const float2* rope, float* Q, float* kc, float* vc, int cap,
                                   cudaStream_t s) {
  if (hd == 64)
    qk_rope_kv_rows_kernel<64><<<T, 256, 0, s>>>(QKV, p0, nq, nkv, qn, kn, eps, rope, Q, kc, vc, cap);
  else if (hd == 128)
    qk_rope_kv_rows_kernel<128><<<T, 256, 0, s>>>(QKV, p0, nq, nkv, qn, kn, eps, rope, Q, kc, vc, cap);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}
constexpr int kAttnBK = 32;  // keys per tile: 2 buffers x 4 arrays = 70 KB at hd 128, two CTAs per SM
static size_t attn_prefill_tc_smem(int hd) { return (size_t)2 * 4 * kAttnBK * (hd + 8) * 2 + 16; }
size_t kv_split_bytes(int nkv, int rows, int hd) { return (size_t)4 * nkv * rows * (hd + 8) * 2; }
int kv_split_rows(int max_ctx) { return (max_ctx + kAttnBK - 1) / kAttnBK * kAttnBK; }
constexpr int kAttnChunk = 8;  // key tiles per CTA at most (causal work balanced across CTAs)
int attn_max_chunks(int max_ctx) {
  return ((max_ctx + kAttnBK - 1) / kAttnBK + kAttnChunk - 1) / kAttnChunk;
}
size_t attn_part_bytes(int nq, int max_t, int max_ctx, int hd) {
  const size_t nqb = (size_t)(max_t + 63) / 64, slots = (size_t)nq * nqb * attn_max_chunks(max_ctx);
  return slots * 64 * ((size_t)hd * 4 + 8) + (size_t)nq * nqb * 4;
}
cudaError_t launch_attn_prefill(const float* Q, const float* kc, const float* vc, int cap, int p0,
                                int T, int nq, int nkv, int hd, uint16_t* kvs, int rows,
                                uint16_t* o_hi, uint16_t* o_lo, void* part, int max_t,
                                int* err, uint64_t wait_ns, cudaStream_t s) {
  const int n = p0 + T;  // keys this pass reads
  const int nqb = (T + 63) / 64, maxqb = (max_t + 63) / 64;
  AttnSplit sp;
  sp.ch = kAttnChunk;
  sp.max_ch = attn_max_chunks(cap);
  const size_t slots = (size_t)nq * maxqb * sp.max_ch;
  sp.part_o = reinterpret_cast<float*>(part);
  sp.part_ml = reinterpret_cast<float2*>(sp.part_o + slots * 64 * hd);
  sp.counters = reinterpret_cast<int*>(sp.part_ml + slots * 64);
  int items = 0;  // (query block, key chunk) pairs per head
  for (int qb = 0; qb < nqb; ++qb) {
    const int nr = min(64, T - qb * 64);
    const int nt = (p0 + qb * 64 + nr - 1) / kAttnBK + 1;
    items += (nt + kAttnChunk - 1) / kAttnChunk;
  }
  // counters are indexed [head][block] with this launch's block count
  const dim3 grid(items, nq), sgrid((n * nkv + 7) / 8);
  if (hd == 64) {
    kv_split_kernel<64><<<sgrid, 256, 0, s>>>(kc, vc, cap, n, nkv, rows, kvs);
    attn_prefill_tc_kernel<64, kAttnBK><<<grid, 128, attn_prefill_tc_smem(64), s>>>(
        Q, kvs, rows, p0, T, nq, nkv, o_hi, o_lo, sp, err, wait_ns);
  } else if (hd == 128) {
    kv_split_kernel<128><<<sgrid, 256, 0, s>>>(kc, vc, cap, n, nkv, rows, kvs);
    attn_prefill_tc_kernel<128, kAttnBK><<<grid, 128, attn_prefill_tc_smem(128), s>>>(
        Q, kvs, rows, p0, T, nq, nkv, o_hi, o_lo, sp, err, wait_ns);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}
cudaError_t launch_set_int(int* p, int v, cudaStream_t s) {
  set_int_kernel<<<1, 1, 0, s>>>(p, v);
  return cudaGetLastError();
}
cudaError_t set_prefill_attributes() {
  cudaError_t e = cudaFuncSetAttribute(attn_prefill_tc_kernel<64, kAttnBK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)attn_prefill_tc_smem(64));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_prefill_tc_kernel<128, kAttnBK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)attn_prefill_tc_smem(128));
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

static int gemm_stages(int bn, int a_split) {
  const size_t stage = (size_t)a_split * kATileBytes + (size_t)bn * GBK * 2;
  int ns = (int)((kGemmSmemBudget - 2048) / stage);
  return ns < 2 ? 2 : (ns > 8 ? 8 : ns);
}
static size_t gemm_smem(int bn, int a_split, int ns) {
  return (size_t)ns * ((size_t)a_split * kATileBytes + (size_t)bn * GBK * 2) + 1024 + 256;
}

template <int BN, int EPI>
static cudaError_t launch_gemm_t(const CUtensorMap& a_hi, const CUtensorMap& a_lo,
                                 const CUtensorMap& b, const GemmArgs& g, cudaStream_t s) {
  const dim3 grid((g.N + BN - 1) / BN, (g.M + GBM - 1) / GBM);
  gemm_tc_kernel<BN, EPI><<<grid, 192, gemm_smem(BN, g.a_split, g.n_stages), s>>>(a_hi, a_lo, b,
                                                                                    g);
  return cudaGetLastError();
}

template <int BN>
static cudaError_t launch_gemm_bn(int epi, const CUtensorMap& a_hi, const CUtensorMap& a_lo,
                                  const CUtensorMap& b, const GemmArgs& g, cudaStream_t s) {
  switch (epi) {
    case GEPI_STORE: return launch_gemm_t<BN, GEPI_STORE>(a_hi, a_lo, b, g, s);
    case GEPI_RESID: return launch_gemm_t<BN, GEPI_RESID>(a_hi, a_lo, b, g, s);
    case GEPI_SWIGLU: return launch_gemm_t<BN, GEPI_SWIGLU>(a_hi, a_lo, b, g, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm(int bn, int epi, const CUtensorMap& a_hi, const CUtensorMap& a_lo,
                        const CUtensorMap& b, GemmArgs g, cudaStream_t s) {
  if (g.M <= 0 || g.N <= 0 || g.K <= 0 || (g.a_split != 1 && g.a_split != 2))
    return cudaErrorInvalidValue;
  if (epi == GEPI_SWIGLU && (g.N % 2)) return cudaErrorInvalidValue;
  g.n_stages = gemm_stages(bn, g.a_split);
  if (bn == 64) return launch_gemm_bn<64>(epi, a_hi, a_lo, b, g, s);
  if (bn == 128) return launch_gemm_bn<128>(epi, a_hi, a_lo, b, g, s);
  if (bn == 256) return launch_gemm_bn<256>(epi, a_hi, a_lo, b, g, s);
  return cudaErrorInvalidValue;
}

template <int BN>
static cudaError_t gemm_attrs_bn() {
  int bytes = 0;
  for (int split = 1; split <= 2; ++split) {
    const int b = (int)gemm_smem(BN, split, gemm_stages(BN, split));
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
