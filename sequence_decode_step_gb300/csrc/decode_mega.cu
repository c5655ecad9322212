// The decode step as one persistent cooperative kernel (one CTA per SM).
//
// Warp 8 of every CTA is a producer: it walks the CTA's share of every phase
// of the token in order (per layer: fused QKV rows, the KV tiles of its key
// split, o_proj rows, gate/up row pairs, down rows; then LM-head rows) and
// streams the bytes with bulk TMA copies into a ring of shared-memory stages.
// None of these bytes depend on activations, so the producer runs ahead of
// the consumers across phase boundaries and the HBM stream never drains.
// Warps 0..7 consume: each phase waits on a grid barrier for its input vector,
// reads it from L2, and works through its chunks from the ring. The embedding
// gather is done redundantly by every CTA, so layer 0 needs no barrier; a
// token has 5 L grid barriers. Every wait is bounded (%globaltimer); a wait
// that gives up sets ERR_TIMEOUT and the kernel runs on to its end without
// hanging. All reductions have a fixed order, so results are bit-identical
// run to run.

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <cstddef>

#include "qw_internal.h"
#include "qw_ptx.cuh"

namespace qw {
namespace {

constexpr int kConsumers = 8;                // consumer warps
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kNS = 6;                       // ring stages
constexpr uint32_t kStage = 32 * 1024;       // bytes per stage
constexpr int kMaxC = 12;                    // input vectors up to 12 x 256 = 3072 wide
constexpr int kTK = 32;                      // keys per attention tile (K + V = 32 KB at hd 128)
constexpr int kGQ = 8;
constexpr int kMinKeys = 64;
constexpr int kUnitPre = 64;                 // units of a phase whose epilogue values are prefetched

enum Kind { K_QKV = 0, K_ATTN = 1, K_O = 2, K_GU = 3, K_DOWN = 4, K_LM = 5 };

// Shared-memory layout after the ring.
struct Smem {
  uint64_t full[kNS];
  uint64_t empty[kNS];
  float red[kConsumers];
  int redi[kConsumers];
  int flag;
  alignas(16) float xs[kMaxC * 256];  // phase input vector (normalised when the phase has a norm);
                                      // written with float4 stores, so 16-byte aligned
  float q_s[kGQ * 128];
  float kn_s[128];
  float vn_s[128];
  float sc_s[kGQ * kTK];
  float p_s[kGQ * kTK];
  float ml_s[2 * kGQ];
  float al_s[kGQ];
  float unit_s[kUnitPre];        // per-unit values the epilogue needs (residual rows or bias)
  float pml_s[2 * kGQ * 160];    // split partials (m, l) for the combine
};

// The contiguous slice of a row-streamed phase owned by CTA b: units [u0, u1),
// each `unit_bytes` long, starting at `base`.
struct Slice {
  const uint8_t* base;
  int u0, u1;
  uint32_t unit_bytes;
  int per_chunk;  // units per ring stage
};

__device__ __forceinline__ Slice make_slice(const uint8_t* w, int n_units, uint32_t unit_bytes,
                                            int b, int G) {
  Slice s;
  s.base = w;
  s.u0 = (int)(((long long)n_units * b) / G);
  s.u1 = (int)(((long long)n_units * (b + 1)) / G);
  s.unit_bytes = unit_bytes;
  int pc = (int)(kStage / unit_bytes);
  s.per_chunk = pc < 1 ? 1 : pc;
  return s;
}

__device__ __forceinline__ Slice phase_slice(const MegaArgs& a, int kind, const LayerDev& L, int b,
                                             int G) {
  const int qd = a.nq * a.hd, kd = a.nkv * a.hd;
  switch (kind) {
    case K_QKV: return make_slice(L.qkv, qd + 2 * kd, (uint32_t)a.H * 2, b, G);
    case K_O: return make_slice(L.o, a.H, (uint32_t)qd * 2, b, G);
    case K_GU: return make_slice(L.gateup, a.I, (uint32_t)a.H * 4, b, G);
    case K_DOWN: return make_slice(L.down, a.H, (uint32_t)a.I * 2, b, G);
    default: return make_slice(a.lm_head, a.V, (uint32_t)a.H * 2, b, G);
  }
}

// Key split of CTA b in the attention phase (all derived from the device position).
struct Split {
  int g, s, k0, k1, nsplit;
  bool active;
};
__device__ __forceinline__ Split attn_split(const MegaArgs& a, int pos, int b) {
  Split r;
  r.g = b / a.splits;
  r.s = b % a.splits;
  const int n_keys = pos + 1;
  int kps = (n_keys + a.splits - 1) / a.splits;
  kps = kps > kMinKeys ? kps : kMinKeys;
  kps = (kps + kTK - 1) / kTK * kTK;
  r.nsplit = (n_keys + kps - 1) / kps;
  r.active = r.g < a.nkv && r.s < r.nsplit;
  r.k0 = r.s * kps;
  r.k1 = min(n_keys, r.k0 + kps);
  if (!r.active) r.k0 = r.k1 = 0;
  return r;
}


__device__ __forceinline__ void csync() {  // the 8 consumer warps only
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory");
}
// Named barrier over the consumer warps that also ORs a flag across them, so a
// give-up decision is the same in every consumer thread.
__device__ __forceinline__ bool csync_or(bool v) {
  unsigned r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((unsigned)v), "r"(kConsumers * 32)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ bool err_set(const MegaArgs& a) {
  return (*reinterpret_cast<volatile int*>(a.err) & ERR_TIMEOUT) != 0;
}

// Wait for a ring stage (or any mbarrier) with the kernel's bound; gives up at
// once when another CTA already reported a timeout.
__device__ bool ring_wait(const MegaArgs& a, uint64_t* bar, uint32_t parity, bool& abort) {
  if (abort) return false;
  if (a.wait_ns == 0) {  // a zero bound gives up at once (tests the error path)
    atomicOr(a.err, ERR_TIMEOUT);
    abort = true;
    return false;
  }
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > a.wait_ns || err_set(a)) {
      atomicOr(a.err, ERR_TIMEOUT);
      abort = true;
      return false;
    }
  }
}

// Grid barrier k of the token: every CTA's consumers arrive once; CTA 0 clears
// the previous slot (all CTAs have left it once all have arrived here).
__device__ void grid_barrier(const MegaArgs& a, Smem& S, int k, int nbar, bool& abort) {
  abort = csync_or(abort);
  if (threadIdx.x == 0) {
    unsigned* slot = a.bar_slots + k;
    const unsigned G = gridDim.x;
    // Release: the phase's writes by this CTA (ordered before this thread by the
    // consumer barrier above) become visible no later than the arrival.
    red_release_add(slot, 1u);
    if (!abort && a.wait_ns == 0) {
      atomicOr(a.err, ERR_TIMEOUT);
      abort = true;
    }
    if (!abort) {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire(slot) < G) {
        if (globaltimer_ns() - t0 > a.wait_ns || err_set(a)) {
          atomicOr(a.err, ERR_TIMEOUT);
          abort = true;
          break;
        }
      }
    }
    // The acquire poll above, then the consumer barrier below, order every later
    // read of this CTA after all CTAs' writes of the phase.
    if (blockIdx.x == 0 && !abort) a.bar_slots[(k - 1 + nbar) % nbar] = 0;
    S.flag = abort ? 1 : 0;
  }
  csync();
  abort = S.flag != 0;
}

// Phase input: xs = v (f32 [K], from L2), optionally RMS-normalised with gain g;
// also prefetches `n_unit` per-unit epilogue values (residual rows or bias) into
// unit_s. Every load is issued before any is used: each is an L2 round trip.
__device__ void load_input(const MegaArgs& a, Smem& S, const float* v, int K, const uint16_t* g,
                           bool from_embed, int tok, const float* unit_f32,
                           const uint16_t* unit_bf16, int n_unit) {
  constexpr int NT = kConsumers * 32;
  constexpr int NV = (kMaxC * 256) / (4 * NT);  // float4 per thread
  const int tid = threadIdx.x;
  float4 xv[NV];
  float uv = 0.f;
  if (from_embed) {
    const uint4* e = reinterpret_cast<const uint4*>(a.embed + (size_t)tok * K);
    uint4 w[(NV + 1) / 2];
#pragma unroll
    for (int i = 0; i < (NV + 1) / 2; ++i) {
      const int idx = tid + i * NT;
      w[i] = idx * 8 < K ? e[idx] : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < (NV + 1) / 2; ++i) {
      const int idx = tid + i * NT;
      if (idx * 8 < K) {
        const uint32_t q[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          S.xs[idx * 8 + 2 * j] = __uint_as_float(q[j] << 16);
          S.xs[idx * 8 + 2 * j + 1] = __uint_as_float(q[j] & 0xffff0000u);
        }
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int idx = tid + i * NT;
      xv[i] = idx * 4 < K ? __ldcg(reinterpret_cast<const float4*>(v) + idx)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  if (tid < n_unit) uv = unit_f32 ? __ldcg(unit_f32 + tid) : (unit_bf16 ? bf16f(unit_bf16[tid]) : 0.f);
  // the norm gain (bf16), 4 per float4 of input, in the same batch of loads
  uint2 gv[NV];
  if (g != nullptr) {
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int idx = tid + i * NT;
      gv[i] = idx * 4 < K ? *reinterpret_cast<const uint2*>(g + idx * 4) : make_uint2(0, 0);
    }
  }
  float ss = 0.f;
  if (!from_embed) {
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int idx = tid + i * NT;
      if (idx * 4 < K) *reinterpret_cast<float4*>(&S.xs[idx * 4]) = xv[i];
      ss = fmaf(xv[i].x, xv[i].x, fmaf(xv[i].y, xv[i].y, fmaf(xv[i].z, xv[i].z, fmaf(xv[i].w, xv[i].w, ss))));
    }
  }
  if (tid < n_unit) S.unit_s[tid] = uv;
  if (g != nullptr) {
    if (from_embed) {
      csync();
      for (int k = tid; k < K; k += NT) ss = fmaf(S.xs[k], S.xs[k], ss);
    }
    ss = warp_sum(ss);
    csync();
    if ((tid & 31) == 0) S.red[tid >> 5] = ss;
    csync();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < kConsumers; ++i) tot += S.red[i];
    const float r = 1.0f / sqrtf(tot / (float)K + a.eps);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int idx = tid + i * NT;
      if (idx * 4 < K) {
        float4 x4 = *reinterpret_cast<const float4*>(&S.xs[idx * 4]);
        x4.x = x4.x * r * __uint_as_float(gv[i].x << 16);
        x4.y = x4.y * r * __uint_as_float(gv[i].x & 0xffff0000u);
        x4.z = x4.z * r * __uint_as_float(gv[i].y << 16);
        x4.w = x4.w * r * __uint_as_float(gv[i].y & 0xffff0000u);
        *reinterpret_cast<float4*>(&S.xs[idx * 4]) = x4;
      }
    }
  }
  csync();
}

template <int MAXC>
__device__ __forceinline__ void x_regs(const Smem& S, int K, float (&xr)[MAXC][8]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = 0; c < MAXC; ++c) {
    const int col = c * 256 + lane * 8;
    float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
    if (col < K) {
      lo = *reinterpret_cast<const float4*>(&S.xs[col]);
      hi = *reinterpret_cast<const float4*>(&S.xs[col + 4]);
    }
    xr[c][0] = lo.x; xr[c][1] = lo.y; xr[c][2] = lo.z; xr[c][3] = lo.w;
    xr[c][4] = hi.x; xr[c][5] = hi.y; xr[c][6] = hi.z; xr[c][7] = hi.w;
  }
}

// Dot products of two weight rows (bf16, in shared memory) with the register-held input.
template <int MAXC>
__device__ __forceinline__ void dot2(const uint8_t* w0, const uint8_t* w1, bool two, int K,
                                     const float (&xr)[MAXC > 0 ? MAXC : 1][8], const float* xs,
                                     float& s0, float& s1) {
  const int lane = threadIdx.x & 31;
  float a0 = 0.f, a1 = 0.f;
  if (MAXC > 0) {
    // one accumulator per 256-column chunk: independent FMA chains, summed in order
    float p0[MAXC > 0 ? MAXC : 1], p1[MAXC > 0 ? MAXC : 1];
#pragma unroll
    for (int c = 0; c < (MAXC > 0 ? MAXC : 1); ++c) {
      const int col = c * 256 + lane * 8;
      p0[c] = 0.f;
      p1[c] = 0.f;
      if (col < K) {
        p0[c] = dot8(*reinterpret_cast<const uint4*>(w0 + (size_t)col * 2), xr[c], 0.f);
        if (two) p1[c] = dot8(*reinterpret_cast<const uint4*>(w1 + (size_t)col * 2), xr[c], 0.f);
      }
    }
#pragma unroll
    for (int c = 0; c < (MAXC > 0 ? MAXC : 1); ++c) {
      a0 += p0[c];
      a1 += p1[c];
    }
  } else {
#pragma unroll 4
    for (int col = lane * 8; col < K; col += 256) {
      const float4 lo = *reinterpret_cast<const float4*>(xs + col);
      const float4 hi = *reinterpret_cast<const float4*>(xs + col + 4);
      const float xv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
      a0 = dot8(*reinterpret_cast<const uint4*>(w0 + (size_t)col * 2), xv, a0);
      if (two) a1 = dot8(*reinterpret_cast<const uint4*>(w1 + (size_t)col * 2), xv, a1);
    }
  }
  s0 = warp_sum(a0);
  s1 = warp_sum(a1);
}

struct GemvOut {
  int epi;                 // EPI_STORE / EPI_RESIDUAL / EPI_SWIGLU / EPI_LOGITS
  float* y;
  const uint16_t* bias;    // STORE: bias (its values for this CTA's units are in unit_s)
  float* cap;              // RESIDUAL: capture row base (already offset by pos * n)
  float best_v;            // LOGITS: running best of this warp (lane 0)
  int best_i;
  int nan;
};

// Consume the chunks of one row-streamed phase; chunk counter c advances.
template <int MAXC>
__device__ void gemv_phase(const MegaArgs& a, uint8_t* ring, Smem& S, int& c, const Slice& sl,
                           int K, int rpu, GemvOut& o, bool& abort) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float xr[MAXC > 0 ? MAXC : 1][8];
  if (MAXC > 0) x_regs<(MAXC > 0 ? MAXC : 1)>(S, K, xr);
  const uint32_t row_bytes = sl.unit_bytes / rpu;
  const int n_units = sl.u1 - sl.u0;
  const int n_chunks = (n_units + sl.per_chunk - 1) / sl.per_chunk;
  if (o.epi != EPI_LOGITS && n_chunks <= kNS) {
    // The whole phase fits in the ring: wait for every chunk once, then give each
    // warp its units across chunks (more independent rows per warp), then release all.
    bool ok = true;
    for (int j = 0; j < n_chunks; ++j)
      ok &= ring_wait(a, &S.full[(c + j) % kNS], (uint32_t)(((c + j) / kNS) & 1), abort);
    if (__any_sync(0xffffffffu, !ok)) {
      abort = true;
      c += n_chunks;
      return;
    }
    auto unit_ptr = [&](int i) {  // i-th unit of the slice, in its ring stage
      const int j = i / sl.per_chunk;
      return ring + (size_t)((c + j) % kNS) * kStage + (size_t)(i - j * sl.per_chunk) * sl.unit_bytes;
    };
    if (rpu == 1) {
      for (int t = 2 * warp; t < n_units; t += 2 * kConsumers) {
        float v0, v1;
        const bool two = t + 1 < n_units;
        dot2<MAXC>(unit_ptr(t), two ? unit_ptr(t + 1) : unit_ptr(t), two, K, xr, S.xs, v0, v1);
        if (lane == 0) {
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            if (jj == 1 && !two) break;
            const int iu = t + jj, uu = sl.u0 + iu;
            const float v = jj ? v1 : v0;
            if (o.epi == EPI_STORE) {
              o.y[uu] = v + (o.bias ? (iu < kUnitPre ? S.unit_s[iu] : bf16f(o.bias[uu])) : 0.f);
            } else {  // EPI_RESIDUAL
              const float nv = (iu < kUnitPre ? S.unit_s[iu] : __ldcg(o.y + uu)) + v;
              o.y[uu] = nv;
              if (o.cap) o.cap[uu] = nv;
            }
          }
        }
      }
    } else {
      for (int t = warp; t < n_units; t += kConsumers) {
        float g, up;
        const uint8_t* w = unit_ptr(t);
        dot2<MAXC>(w, w + row_bytes, true, K, xr, S.xs, g, up);
        if (lane == 0) o.y[sl.u0 + t] = g / (1.0f + expf(-g)) * up;
      }
    }
    __syncwarp();
    if (lane == 0)
      for (int j = 0; j < n_chunks; ++j) mbar_arrive(&S.empty[(c + j) % kNS]);
    c += n_chunks;
    return;
  }
  for (int u = sl.u0; u < sl.u1; u += sl.per_chunk, ++c) {
    const int nu = min(sl.per_chunk, sl.u1 - u);
    const int st = c % kNS;
    const bool ok = ring_wait(a, &S.full[st], (uint32_t)((c / kNS) & 1), abort);
    if (__any_sync(0xffffffffu, !ok)) {  // the whole warp gives up together
      abort = true;
      continue;
    }
    const uint8_t* base = ring + (size_t)st * kStage;
    if (rpu == 1) {
      for (int t = 2 * warp; t < nu; t += 2 * kConsumers) {
        float v0, v1;
        const bool two = t + 1 < nu;
        dot2<MAXC>(base + (size_t)t * row_bytes, base + (size_t)(t + 1) * row_bytes, two, K, xr,
                   S.xs, v0, v1);
        if (lane == 0) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (j == 1 && !two) break;
            const int uu = u + t + j;
            const float v = j ? v1 : v0;
            const int iu = uu - sl.u0;
            if (o.epi == EPI_STORE) {
              o.y[uu] = v + (o.bias ? (iu < kUnitPre ? S.unit_s[iu] : bf16f(o.bias[uu])) : 0.f);
            } else if (o.epi == EPI_RESIDUAL) {
              const float nv = (iu < kUnitPre ? S.unit_s[iu] : __ldcg(o.y + uu)) + v;
              o.y[uu] = nv;
              if (o.cap) o.cap[uu] = nv;
            } else {  // EPI_LOGITS
              o.y[uu] = v;
              if (v != v) o.nan = 1;
              else if (v > o.best_v) { o.best_v = v; o.best_i = uu; }
            }
          }
        }
      }
    } else {  // interleaved gate/up pairs
      for (int t = warp; t < nu; t += kConsumers) {
        float g, up;
        dot2<MAXC>(base + (size_t)t * sl.unit_bytes, base + (size_t)t * sl.unit_bytes + row_bytes,
                   true, K, xr, S.xs, g, up);
        if (lane == 0) o.y[u + t] = g / (1.0f + expf(-g)) * up;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[st]);
  }
}

template <int MAXC_DUMMY = 0>
__device__ void gemv_dispatch(const MegaArgs& a, uint8_t* ring, Smem& S, int& c, const Slice& sl,
                              int K, int rpu, GemvOut& o, bool& abort) {
  // Inputs up to 1024 wide stay in registers; wider ones are read from shared
  // memory inside the dot (keeps the kernel under its register budget, no spills).
  if (K <= 1024) gemv_phase<4>(a, ring, S, c, sl, K, rpu, o, abort);
  else gemv_phase<0>(a, ring, S, c, sl, K, rpu, o, abort);
}


// Split-K attention of CTA b: QK-norm + RoPE of its group's queries (and of the
// new key when its split holds pos), tiles of 32 keys from the ring, online
// softmax, then a partial (or the final output when there is one split); the
// last CTA of a KV head to arrive combines the splits in split order.
template <int HD>
__device__ void attn_phase(const MegaArgs& a, uint8_t* ring, Smem& S, int& c, int l, int pos,
                           const Split& sp, bool& abort) {
  constexpr int EPL = HD / 32, OUTS = (kGQ * HD + 255) / 256;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int GQ = a.nq / a.nkv, g = sp.g;
  const LayerDev& Ld = a.layers[l];
  const size_t kv_layer = (size_t)a.nkv * a.cap * HD;
  float* kc = a.k_cache + (size_t)l * kv_layer + (size_t)g * a.cap * HD;
  float* vc = a.v_cache + (size_t)l * kv_layer + (size_t)g * a.cap * HD;
  const bool owns_pos = pos >= sp.k0 && pos < sp.k1;
  const float scale = 1.0f / sqrtf((float)HD);
  const float2* rrow = a.rope + (size_t)pos * (HD / 2);
  if (tid < kGQ) {
    S.ml_s[2 * tid] = -INFINITY;
    S.ml_s[2 * tid + 1] = 0.f;
  }
  for (int hh = warp; hh <= GQ; hh += kConsumers) {
    const bool isq = hh < GQ;
    if (!isq && !owns_pos) break;
    const float* src = a.qkv + (size_t)(isq ? (g * GQ + hh) : (a.nq + g)) * HD;
    const uint16_t* gain = isq ? Ld.q_norm : Ld.k_norm;
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
      const float2 cs = rrow[lane + 32 * e];
      const float x0 = v[e], x1 = v[e + EPL / 2];
      v[e] = x0 * cs.x - x1 * cs.y;
      v[e + EPL / 2] = x1 * cs.x + x0 * cs.y;
    }
    if (isq) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) S.q_s[hh * HD + lane + 32 * e] = v[e] * scale;
    } else {
      const float* vsrc = a.qkv + (size_t)(a.nq + a.nkv + g) * HD;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const int d = lane + 32 * e;
        S.kn_s[d] = v[e];
        kc[(size_t)pos * HD + d] = v[e];
        const float vv = __ldcg(vsrc + d);
        S.vn_s[d] = vv;
        vc[(size_t)pos * HD + d] = vv;
      }
    }
  }
  csync();
  float qr[kGQ][EPL];
#pragma unroll
  for (int h = 0; h < kGQ; ++h)
#pragma unroll
    for (int e = 0; e < EPL; ++e) qr[h][e] = (h < GQ) ? S.q_s[h * HD + lane * EPL + e] : 0.f;
  float oacc[OUTS];
#pragma unroll
  for (int i = 0; i < OUTS; ++i) oacc[i] = 0.f;

  for (int t0 = sp.k0; t0 < sp.k1; t0 += kTK, ++c) {
    const int st = c % kNS;
    const int nk = min(kTK, sp.k1 - t0);
    ring_wait(a, &S.full[st], (uint32_t)((c / kNS) & 1), abort);
    abort = csync_or(abort);
    float* Ks = reinterpret_cast<float*>(ring + (size_t)st * kStage);
    float* Vs = Ks + kTK * HD;
    if (!abort) {
      if (owns_pos && pos >= t0 && pos < t0 + nk) {
        for (int e = tid; e < HD; e += kConsumers * 32) {
          Ks[(pos - t0) * HD + e] = S.kn_s[e];
          Vs[(pos - t0) * HD + e] = S.vn_s[e];
        }
        csync();
      }
      for (int j = warp; j < nk; j += kConsumers) {
        float kv[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) kv[e] = Ks[j * HD + lane * EPL + e];
#pragma unroll
        for (int h = 0; h < kGQ; ++h) {
          if (h < GQ) {
            float p = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) p = fmaf(qr[h][e], kv[e], p);
            p = warp_sum(p);
            if (lane == 0) S.sc_s[h * kTK + j] = p;
          }
        }
      }
      csync();
      for (int h = warp; h < GQ; h += kConsumers) {
        const float sc = lane < nk ? S.sc_s[h * kTK + lane] : -INFINITY;
        const float tmax = warp_max(sc);
        const float m_old = S.ml_s[2 * h], l_old = S.ml_s[2 * h + 1];
        const float m_new = fmaxf(m_old, tmax);
        const float p = lane < nk ? expf(sc - m_new) : 0.f;
        const float psum = warp_sum(p);
        const float alpha = expf(m_old - m_new);
        S.p_s[h * kTK + lane] = p;
        __syncwarp();
        if (lane == 0) {
          S.ml_s[2 * h] = m_new;
          S.ml_s[2 * h + 1] = l_old * alpha + psum;
          S.al_s[h] = alpha;
        }
      }
      csync();
#pragma unroll
      for (int oi = 0; oi < OUTS; ++oi) {
        const int idx = tid + oi * 256;
        if (idx < GQ * HD) {
          const int h = idx / HD, d = idx % HD;
          float acc = oacc[oi] * S.al_s[h];
          const float* pr = S.p_s + h * kTK;
          for (int j = 0; j < nk; ++j) acc = fmaf(pr[j], Vs[j * HD + d], acc);
          oacc[oi] = acc;
        }
      }
    }
    csync();
    if (lane == 0) mbar_arrive(&S.empty[st]);
  }

  if (sp.nsplit == 1) {
#pragma unroll
    for (int oi = 0; oi < OUTS; ++oi) {
      const int idx = tid + oi * 256;
      if (idx < GQ * HD) {
        const int h = idx / HD, d = idx % HD;
        a.attn_o[(size_t)(g * GQ + h) * HD + d] = oacc[oi] / S.ml_s[2 * h + 1];
      }
    }
    return;
  }
#pragma unroll
  for (int oi = 0; oi < OUTS; ++oi) {
    const int idx = tid + oi * 256;
    if (idx < GQ * HD) {
      const int h = idx / HD, d = idx % HD;
      a.part_o[((size_t)(g * GQ + h) * a.splits + sp.s) * HD + d] = oacc[oi];
    }
  }
  if (tid < GQ) {
    const size_t o = ((size_t)(g * GQ + tid) * a.splits + sp.s) * 2;
    a.part_ml[o] = S.ml_s[2 * tid];
    a.part_ml[o + 1] = S.ml_s[2 * tid + 1];
  }
  __threadfence();
  csync();
  if (tid == 0) {
    const int prev = atomicAdd(&a.attn_counters[g], 1);
    S.flag = (prev == sp.nsplit - 1);
  }
  csync();
  if (!S.flag) return;
  __threadfence();
  // Combine: every (m, l) of the group into shared memory at once, then the
  // partial outputs in batches of 8 independent loads.
  const int ns = sp.nsplit;
  for (int i = tid; i < GQ * ns; i += kConsumers * 32) {
    const int h = i / ns, s2 = i % ns;
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.part_ml) +
                             (size_t)(g * GQ + h) * a.splits + s2);
    S.pml_s[2 * i] = ml.x;
    S.pml_s[2 * i + 1] = ml.y;
  }
  csync();
#pragma unroll
  for (int oi = 0; oi < OUTS; ++oi) {
    const int idx = tid + oi * 256;
    if (idx < GQ * HD) {
      const int h = idx / HD, d = idx % HD;
      const float* pm = S.pml_s + 2 * h * ns;
      float M = -INFINITY;
      for (int s2 = 0; s2 < ns; ++s2) M = fmaxf(M, pm[2 * s2]);
      float den = 0.f;
      for (int s2 = 0; s2 < ns; ++s2) den = fmaf(expf(pm[2 * s2] - M), pm[2 * s2 + 1], den);
      const float* po = a.part_o + (size_t)(g * GQ + h) * a.splits * HD + d;
      float num = 0.f;
      for (int s0 = 0; s0 < ns; s0 += 8) {
        float pv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) pv[j] = s0 + j < ns ? __ldcg(po + (size_t)(s0 + j) * HD) : 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (s0 + j < ns) num = fmaf(expf(pm[2 * (s0 + j)] - M), pv[j], num);
      }
      a.attn_o[(size_t)(g * GQ + h) * HD + d] = num / den;
    }
  }
  csync();
  if (tid == 0) a.attn_counters[g] = 0;
}


// ---- producer: one thread streams every chunk of the token, in consumer order
__device__ void produce(const MegaArgs& a, uint8_t* ring, Smem& S, int pos) {
  const int b = blockIdx.x, G = gridDim.x;
  bool abort = false;
  int c = 0;
  auto issue = [&](const void* s0, uint32_t n0, const void* s1, uint32_t n1, uint32_t off1) {
    const int st = c % kNS, u = c / kNS;
    if (u > 0 && !ring_wait(a, &S.empty[st], (uint32_t)((u - 1) & 1), abort)) return false;
    uint8_t* dst = ring + (size_t)st * kStage;
    mbar_expect_tx(&S.full[st], n0 + n1);
    bulk_load(dst, s0, n0, &S.full[st]);
    if (n1) bulk_load(dst + off1, s1, n1, &S.full[st]);
    ++c;
    return true;
  };
  auto stream_slice = [&](const Slice& sl) {
    for (int u = sl.u0; u < sl.u1; u += sl.per_chunk) {
      const int nu = min(sl.per_chunk, sl.u1 - u);
      if (!issue(sl.base + (size_t)u * sl.unit_bytes, (uint32_t)nu * sl.unit_bytes, nullptr, 0, 0))
        return false;
    }
    return true;
  };
  const Split sp = attn_split(a, pos, b);
  const size_t kv_layer = (size_t)a.nkv * a.cap * a.hd;
  bool ok = true;
  for (int l = 0; l < a.L && ok; ++l) {
    const LayerDev Ld = a.layers[l];
    ok = stream_slice(phase_slice(a, K_QKV, Ld, b, G));
    const float* kc = a.k_cache + (size_t)l * kv_layer + (size_t)sp.g * a.cap * a.hd;
    const float* vc = a.v_cache + (size_t)l * kv_layer + (size_t)sp.g * a.cap * a.hd;
    for (int t0 = sp.k0; ok && t0 < sp.k1; t0 += kTK) {
      const uint32_t n = (uint32_t)min(kTK, sp.k1 - t0) * a.hd * 4;
      ok = issue(kc + (size_t)t0 * a.hd, n, vc + (size_t)t0 * a.hd, n, (uint32_t)kTK * a.hd * 4);
    }
    ok = ok && stream_slice(phase_slice(a, K_O, Ld, b, G));
    ok = ok && stream_slice(phase_slice(a, K_GU, Ld, b, G));
    ok = ok && stream_slice(phase_slice(a, K_DOWN, Ld, b, G));
  }
  if (ok) stream_slice(phase_slice(a, K_LM, LayerDev{}, b, G));
  // Leave only once every copy issued into this CTA's shared memory has landed.
  for (int cc = c > kNS ? c - kNS : 0; cc < c; ++cc)
    mbar_wait(&S.full[cc % kNS], (uint32_t)((cc / kNS) & 1), kDrainNs);
}

// ---- greedy argmax across the grid (last CTA to arrive reduces in order)
__device__ void argmax_finalize(const MegaArgs& a, Smem& S, GemvOut& o, int pos) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x, G = gridDim.x;
  if (lane == 0) {
    S.red[warp] = o.nan ? __int_as_float(0x7fc00000) : o.best_v;
    S.redi[warp] = o.best_i;
  }
  csync();
  if (tid == 0) {
    float bv = -INFINITY;
    int bi = 0x7fffffff, any_nan = 0;
    for (int i = 0; i < kConsumers; ++i) {
      const float v = S.red[i];
      if (v != v) any_nan = 1;
      else if (am_better(v, S.redi[i], bv, bi)) { bv = v; bi = S.redi[i]; }
    }
    a.am.blk_val[b] = any_nan ? __int_as_float(0x7fc00000) : bv;
    a.am.blk_idx[b] = bi;
    __threadfence();
    S.flag = (atomicAdd(a.am.counter, 1) == G - 1);
  }
  csync();
  if (!S.flag) return;
  __threadfence();
  float bv = -INFINITY;
  int bi = 0x7fffffff, nan_seen = 0;
  for (int i = tid; i < G; i += kConsumers * 32) {
    const float v = __ldcg(a.am.blk_val + i);
    const int ix = __ldcg(a.am.blk_idx + i);
    if (v != v) nan_seen = 1;
    else if (am_better(v, ix, bv, bi)) { bv = v; bi = ix; }
  }
  nan_seen = csync_or(nan_seen != 0);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
    if (am_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
  }
  if (lane == 0) { S.red[warp] = bv; S.redi[warp] = bi; }
  csync();
  if (tid == 0) {
    bv = S.red[0];
    bi = S.redi[0];
    for (int i = 1; i < kConsumers; ++i)
      if (am_better(S.red[i], S.redi[i], bv, bi)) { bv = S.red[i]; bi = S.redi[i]; }
    const int am = nan_seen ? -1 : bi;
    if (nan_seen) atomicOr(a.err, ERR_NAN);
    *a.am.argmax = am;
    *a.am.next_token = am;
    a.am.tokens_by_pos[pos] = am;
    *a.am.pos = pos + 1;
    a.am.status[0] = am;
    a.am.status[1] = *reinterpret_cast<volatile int*>(a.err);
    *a.am.counter = 0;
  }
}

// ---- consumers: the phases of one token
__device__ void consume(const MegaArgs& a, uint8_t* ring, Smem& S, int pos) {
  const int b = blockIdx.x, G = gridDim.x, tid = threadIdx.x;
  const int nbar = 5 * a.L, qd = a.nq * a.hd;
  bool abort = false;
  int c = 0, k = 0;
  int tok = a.tok >= 0 ? a.tok : __ldcg(a.next_token);
  if (tok < 0 || tok >= a.V) {
    if (tid == 0 && b == 0) atomicOr(a.err, ERR_TOKEN);
    tok = 0;
  }
  const Split sp = attn_split(a, pos, b);
  for (int l = 0; l < a.L; ++l) {
    const LayerDev Ld = a.layers[l];  // one batch of loads per layer, kept in registers
    if (l > 0) grid_barrier(a, S, k++, nbar, abort);
    // fused QKV; layer 0 gathers the embedding row itself and seeds the residual rows it owns
    const Slice qs = phase_slice(a, K_QKV, Ld, b, G);
    load_input(a, S, a.x, a.H, Ld.attn_norm, l == 0, tok, nullptr,
               Ld.qkv_bias ? Ld.qkv_bias + qs.u0 : nullptr, min(qs.u1 - qs.u0, kUnitPre));
    if (l == 0) {
      const Slice os = phase_slice(a, K_O, Ld, b, G);
      const uint16_t* e = a.embed + (size_t)tok * a.H;
      for (int r = os.u0 + tid; r < os.u1; r += kConsumers * 32) a.x[r] = bf16f(e[r]);
      if (a.cap_emb && b == 0)
        for (int r = tid; r < a.H; r += kConsumers * 32) a.cap_emb[(size_t)pos * a.H + r] = bf16f(e[r]);
    }
    GemvOut o{EPI_STORE, a.qkv, Ld.qkv_bias, nullptr, -INFINITY, 0x7fffffff, 0};
    gemv_dispatch(a, ring, S, c, qs, a.H, 1, o, abort);
    grid_barrier(a, S, k++, nbar, abort);
    // attention of this CTA's (kv head, key split)
    if (sp.active) {
      if (a.hd == 64) attn_phase<64>(a, ring, S, c, l, pos, sp, abort);
      else attn_phase<128>(a, ring, S, c, l, pos, sp, abort);
    }
    grid_barrier(a, S, k++, nbar, abort);
    // o_proj + residual
    const Slice os = phase_slice(a, K_O, Ld, b, G);
    load_input(a, S, a.attn_o, qd, nullptr, false, 0, a.x + os.u0, nullptr,
               min(os.u1 - os.u0, kUnitPre));
    o = GemvOut{EPI_RESIDUAL, a.x, nullptr, nullptr, -INFINITY, 0x7fffffff, 0};
    gemv_dispatch(a, ring, S, c, os, qd, 1, o, abort);
    grid_barrier(a, S, k++, nbar, abort);
    // gate/up with SwiGLU
    load_input(a, S, a.x, a.H, Ld.mlp_norm, false, 0, nullptr, nullptr, 0);
    o = GemvOut{EPI_SWIGLU, a.mlp, nullptr, nullptr, -INFINITY, 0x7fffffff, 0};
    gemv_dispatch(a, ring, S, c, phase_slice(a, K_GU, Ld, b, G), a.H, 2, o, abort);
    grid_barrier(a, S, k++, nbar, abort);
    // down + residual (block-0 checkpoint)
    const Slice ds = phase_slice(a, K_DOWN, Ld, b, G);
    load_input(a, S, a.mlp, a.I, nullptr, false, 0, a.x + ds.u0, nullptr,
               min(ds.u1 - ds.u0, kUnitPre));
    o = GemvOut{EPI_RESIDUAL, a.x, nullptr,
                (l == 0 && a.cap_blk0) ? a.cap_blk0 + (size_t)pos * a.H : nullptr,
                -INFINITY, 0x7fffffff, 0};
    gemv_dispatch(a, ring, S, c, ds, a.I, 1, o, abort);
  }
  grid_barrier(a, S, k++, nbar, abort);
  // final RMSNorm + LM head + greedy argmax
  load_input(a, S, a.x, a.H, a.final_norm, false, 0, nullptr, nullptr, 0);
  if (a.cap_final && b == 0)
    for (int r = tid; r < a.H; r += kConsumers * 32) a.cap_final[(size_t)pos * a.H + r] = S.xs[r];
  GemvOut o{EPI_LOGITS, a.logits, nullptr, nullptr, -INFINITY, 0x7fffffff, 0};
  gemv_dispatch(a, ring, S, c, phase_slice(a, K_LM, LayerDev{}, b, G), a.H, 1, o, abort);
  argmax_finalize(a, S, o, pos);
}

__global__ void __launch_bounds__(kThreads, 1) decode_mega_kernel(const MegaArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* ring = smem_raw;
  Smem& S = *reinterpret_cast<Smem*>(smem_raw + (size_t)kNS * kStage);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNS; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], kConsumers);
    }
    fence_barrier_init();
  }
  __syncthreads();
  // The position changes only at the end of a token, so every thread reads it once.
  const int pos = __ldcg(a.pos);
  if (threadIdx.x < kConsumers * 32) consume(a, ring, S, pos);
  else if (threadIdx.x == kConsumers * 32) produce(a, ring, S, pos);
}

}  // namespace

bool mega_supported(int H, int I, int qd, int hd, int gq) {
  return H <= kMaxC * 256 && I <= kMaxC * 256 && qd <= kMaxC * 256 && (hd == 64 || hd == 128) &&
         gq >= 1 && gq <= kGQ && (uint32_t)H * 4 <= kStage && (uint32_t)I * 2 <= kStage &&
         (uint32_t)qd * 2 <= kStage;
}

static_assert(offsetof(Smem, xs) % 16 == 0, "float4 stores into xs need 16-byte alignment");
size_t mega_smem_bytes() { return (size_t)kNS * kStage + sizeof(Smem); }

cudaError_t set_mega_attributes() {
  cudaError_t e = cudaFuncSetAttribute(decode_mega_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)mega_smem_bytes());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_mega_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  return e;
}

const void* mega_kernel_fn() { return reinterpret_cast<const void*>(decode_mega_kernel); }

cudaError_t launch_mega(const MegaArgs& a, int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = mega_smem_bytes();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_mega_kernel, a);
}

}  // namespace qw
