// The decode step as one persistent cooperative kernel (one CTA per SM).
//
// The last warp of every CTA is a producer: it walks the CTA's share of every phase
// of the token in order (per layer: fused QKV rows, the KV tiles of its key
// split, o_proj rows, gate/up row pairs, down rows; then LM-head rows) and
// streams the bytes with bulk TMA copies into a ring of shared-memory stages.
// None of these bytes depend on activations, so the producer runs ahead of
// the consumers across phase boundaries and the HBM stream never drains.
// The other warps consume: each phase reads its input vector from L2 and works
// through its chunks from the ring.
//
// There is no grid barrier. Every activation a phase hands to the next one
// (residual x, fused q/k/v, attention output, SwiGLU output) is stored as a
// 64-bit word: the f32 value in the low half and a tag in the high half, the
// tag naming the token launch (a device epoch) and the phase that wrote it.
// A single 64-bit store is single-copy atomic, so a reader that polls the
// words of its input until all carry the expected tag has both waited for and
// loaded the data in the same L2 round trip. A phase waits only for what it
// reads: the attention of a KV head starts as soon as that head's q/k/v rows
// are in, independently of the other heads.
//
// Reuse of a buffer is safe without a barrier because every overwrite of a
// tagged vector depends, through the chain of full-vector inputs, on every
// reader of the previous contents having finished (each reader also writes an
// output the overwriter transitively needs); a CTA with no rows in a phase
// therefore does not read that phase's input at all. Every wait is bounded
// (%globaltimer); a wait that gives up sets ERR_TIMEOUT and the kernel runs on
// to its end without hanging. All reductions have a fixed order, so results
// are bit-identical run to run.

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <cstddef>

#include "qw_internal.h"
#include "qw_ptx.cuh"

// The consumer warp count is fixed per build of this file: 7 by default (short
// contexts), and decode_mega_wide.cu builds it again with 11 under another
// namespace for long contexts, where the attention passes dominate and spread
// over more warps (at short context the GEMV phases have too few rows per CTA
// for the extra warps, and the wider barriers cost more). decode_mega_big.cu
// builds it a third time for wide inputs (up to 44 x 256 = 11264, e.g. an 11008-wide
// SwiGLU vector) and int4 g128 weights: a larger input buffer in shared memory
// and one ring stage fewer.
#ifndef QW_MEGA_CONSUMERS
#define QW_MEGA_CONSUMERS 7
#define QW_MEGA_NS mega
#endif
#ifndef QW_MEGA_MAXC
#define QW_MEGA_MAXC 12
#endif
#ifndef QW_MEGA_STAGES
#define QW_MEGA_STAGES 6
#endif
#ifndef QW_MEGA_BIG
#define QW_MEGA_BIG 0
#endif
#ifndef QW_MEGA_ROUND_PAIRS
#define QW_MEGA_ROUND_PAIRS 8
#endif

namespace qw {
namespace {

// consumer warps + 1 producer warp; 8 warps leave 255 registers per thread, 12
// warps 168 (both fit the kernel without spills)
constexpr int kConsumers = QW_MEGA_CONSUMERS;
constexpr int kNT = kConsumers * 32;         // consumer threads
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kNS = QW_MEGA_STAGES;          // ring stages
constexpr uint32_t kStage = 32 * 1024;       // bytes per stage
constexpr int kMaxC = QW_MEGA_MAXC;          // input vectors up to kMaxC x 256 wide
constexpr int kTK = 32;                      // keys per attention tile (K + V = 32 KB at hd 128)
constexpr int kGQ = 8;
constexpr int kMinKeys = QW_MEGA_BIG ? 64 : 128;  // keys per split at least
// Up to this many keys a group's query heads go to separate CTAs over all keys
// (one pass, no combine); beyond it the keys are split and combined. Measured
// (us/token, Qwen3-0.6B shape, same box) at 145-256 keys: 652-680 with the key
// split against 662-705 with the head split's two passes.
constexpr int kHeadSplitKeys = 128;
constexpr int kPass = 4;                     // tiles per attention pass
constexpr int kUnitPre = kMegaUnitPre;       // units of a phase whose epilogue values are prefetched

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
  float ml_s[2 * kGQ];
  float al_s[kGQ];
  float unit_s[kUnitPre];        // per-unit values the epilogue needs (residual rows, or bias
                                 // plus the LoRA update)
  float pml_s[2 * kGQ * 160];    // split partials (m, l) for the combine; before it, the
                                 // scores and probabilities of an attention pass
  float xsum[kMaxC * 32];        // int4 weights: 136 x the sum of each lane's 8 inputs of a chunk
  float lora_t[128];             // LoRA: A_q . x_n, then A_v . x_n (rank <= 64 each)
};

// The contiguous slice of a row-streamed phase owned by CTA b: units [u0, u1),
// each `unit_bytes` long, starting at `base`.
struct Slice {
  const uint8_t* base;
  int u0, u1;
  uint32_t unit_bytes;
  int per_chunk;  // units per ring stage
  int n_chunks;   // ring stages the slice takes
};

// Rows a warp takes per GEMV iteration in each phase (a power of two up to 8; for
// gate/up, rows of interleaved gate/up pairs).
// One gate/up unit (two rows) per item in the 7- and 11-warp builds: 20 units per CTA
// for the Qwen3-0.6B shape spread over three rounds of the 7 warps instead of two rounds
// with four rows (575 -> 546 us/token, same box).
constexpr int kNrQkv = 2, kNrO = 1, kNrGu = QW_MEGA_BIG ? 4 : 2, kNrDown = 1, kNrLm = 8;
// Units per iteration (rows / rows per unit); a ring stage holds a whole number
// of them when it can.
__host__ __device__ constexpr int phase_upi(int kind) {
  return kind == K_QKV ? kNrQkv : kind == K_O ? kNrO : kind == K_GU ? kNrGu / 2
       : kind == K_DOWN ? kNrDown : kNrLm;
}

// 32-bit arithmetic throughout: n_units * G stays far below 2^31 for every shape
// the kernel takes (checked on the host).
__device__ __forceinline__ Slice make_slice(const uint8_t* w, int n_units, uint32_t unit_bytes,
                                            int upi, int b, int G) {
  Slice s;
  s.base = w;
  s.u0 = (int)(((uint32_t)n_units * (uint32_t)b) / (uint32_t)G);
  s.u1 = (int)(((uint32_t)n_units * (uint32_t)(b + 1)) / (uint32_t)G);
  s.unit_bytes = unit_bytes;
  int pc = (int)(kStage / unit_bytes);
  pc = pc >= upi ? pc / upi * upi : (pc < 1 ? 1 : pc);
  s.per_chunk = pc;
  s.n_chunks = (s.u1 - s.u0 + pc - 1) / pc;
  return s;
}

// Bytes of one weight row of K inputs: bf16; int4 g128 (K/2 nibble bytes, then K/128
// bf16 scales, padded to 16 bytes); or Q8_0 (K int8, then K/32 fp16 scales, padded to
// 16 bytes).
__host__ __device__ __forceinline__ uint32_t row_bytes_fmt(int wfmt, int K) {
  return wfmt == 2 ? q8_row_bytes(K) : wfmt == 1 ? int4_row_bytes(K) : (uint32_t)K * 2;
}
__device__ __forceinline__ uint32_t row_bytes(const MegaArgs& a, int K) {
  return row_bytes_fmt(a.wfmt, K);
}

// Geometry of a phase (its base is set per layer by the producer; the consumers
// never read it).
__device__ __forceinline__ Slice phase_slice(const MegaArgs& a, int kind, int b, int G) {
  const int qd = a.nq * a.hd, kd = a.nkv * a.hd;
  switch (kind) {
    case K_QKV: return make_slice(nullptr, qd + 2 * kd, row_bytes(a, a.H), phase_upi(K_QKV), b, G);
    case K_O: return make_slice(nullptr, a.H, row_bytes(a, qd), phase_upi(K_O), b, G);
    case K_GU: return make_slice(nullptr, a.I, 2 * row_bytes(a, a.H), phase_upi(K_GU), b, G);
    case K_DOWN: return make_slice(nullptr, a.H, row_bytes(a, a.I), phase_upi(K_DOWN), b, G);
    default: return make_slice(a.lm_head, a.V, row_bytes(a, a.H), phase_upi(K_LM), b, G);
  }
}
__device__ __forceinline__ const uint8_t* phase_base(int kind, const LayerDev& L) {
  return kind == K_QKV ? L.qkv : kind == K_O ? L.o : kind == K_GU ? L.gateup : L.down;
}

// Attention work of CTA b (all derived from the device position): KV head g and
// either a key split s (its query heads all together; the partials combined by split
// 0, or in the wide-input build by all splits, each a slice of the outputs) or, up to
// kHeadSplitKeys keys, query head h0 of the group over all keys (the group's heads
// on separate CTAs, no combine).
struct Split {
  int g, s, k0, k1, nsplit;
  int h0, nh;  // the group's query heads [h0, h0 + nh) handled here
  bool active;
};
__device__ __forceinline__ Split attn_split(const MegaArgs& a, int pos, int b) {
  Split r;
  r.g = b / a.splits;
  r.s = b % a.splits;
  const int gq = a.nq / a.nkv;
  const int n_keys = pos + 1;
  int kps = (n_keys + a.splits - 1) / a.splits;
  kps = kps > kMinKeys ? kps : kMinKeys;
  kps = (kps + kTK - 1) / kTK * kTK;
  r.nsplit = (n_keys + kps - 1) / kps;
  r.h0 = 0;
  r.nh = gq;
  if (n_keys <= kHeadSplitKeys && gq > 1 && gq <= a.splits) {  // split the heads, not the keys
    r.nsplit = 1;
    r.active = r.g < a.nkv && r.s < gq;
    r.h0 = r.s;
    r.nh = 1;
    r.k0 = 0;
    r.k1 = n_keys;
  } else {
    r.active = r.g < a.nkv && r.s < r.nsplit;
    r.k0 = r.s * kps;
    r.k1 = min(n_keys, r.k0 + kps);
  }
  if (!r.active) r.k0 = r.k1 = 0;
  return r;
}

__device__ __forceinline__ void csync() {  // the consumer warps only
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
// One arrival standing for all consumer warps (after a consumer barrier).
__device__ __forceinline__ void mbar_arrive_all(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(kConsumers)
               : "memory");
}
__device__ __forceinline__ bool err_set(const MegaArgs& a) {
  return (*reinterpret_cast<volatile int*>(a.err) & ERR_TIMEOUT) != 0;
}

// Wait for a ring stage (or any mbarrier) with the kernel's bound; gives up at
// once when another CTA already reported a timeout. Reading %globaltimer costs
// far more than a try_wait, so the clock (and the error word) is looked at only
// every 16th failed try; the bound starts counting at the first look.
__device__ bool ring_wait(const MegaArgs& a, uint64_t* bar, uint32_t parity, bool& abort) {
  if (abort) return false;
  if (a.wait_ns == 0) {  // a zero bound gives up at once (tests the error path)
    atomicOr(a.err, ERR_TIMEOUT);
    abort = true;
    return false;
  }
  uint64_t t0 = 0;
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 15u) != 0) continue;
    const uint64_t now = globaltimer_ns();
    if (t0 == 0) {
      t0 = now;
    } else if (now - t0 > a.wait_ns || err_set(a)) {
      atomicOr(a.err, ERR_TIMEOUT);
      abort = true;
      return false;
    }
  }
}

// Tagged activation words: value bits low, tag high.
__device__ __forceinline__ float word_value(uint64_t w) { return __uint_as_float((uint32_t)w); }
__device__ __forceinline__ uint32_t word_tag(uint64_t w) { return (uint32_t)(w >> 32); }
__device__ __forceinline__ void st_tagged(uint64_t* p, float v, uint32_t tag) {
  const uint64_t w = ((uint64_t)tag << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ uint64_t ld_word(const uint64_t* p) {
  uint64_t w;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
  return w;
}
__device__ __forceinline__ void ld_words2(const uint64_t* p, uint64_t& w0, uint64_t& w1) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];"
               : "=l"(w0), "=l"(w1)
               : "l"(p)
               : "memory");
}

// One more round `n` of a poll found data missing: give up (ERR_TIMEOUT) at once
// when the bound is zero, else once the bound has passed or another CTA gave up.
// The clock and the error word are looked at only every 32nd round (a read of
// %globaltimer costs more than the L2 round trip of a poll); the bound starts
// counting at the first look.
__device__ __forceinline__ void poll_bound(const MegaArgs& a, uint32_t n, uint64_t& t0,
                                           bool& abort) {
  if (a.wait_ns == 0) {
    atomicOr(a.err, ERR_TIMEOUT);
    abort = true;
    return;
  }
  if ((n & 31u) != 0) return;
  const uint64_t now = globaltimer_ns();
  if (t0 == 0) {
    t0 = now;
  } else if (now - t0 > a.wait_ns || err_set(a)) {
    atomicOr(a.err, ERR_TIMEOUT);
    abort = true;
  }
}

// Per lane: words src[lane + 32 e], e < N, once all carry `tag`; with src2, the
// words src2[lane + 32 e] as well, polled in the same rounds (one L2 round trip
// for both rows when they are there).
template <int N>
__device__ __forceinline__ void poll_row(const MegaArgs& a, const uint64_t* src,
                                         const uint64_t* src2, uint32_t tag, float (&v)[N],
                                         float (&v2)[N], bool& abort) {
  const int lane = threadIdx.x & 31;
  uint64_t w[2 * N];
#pragma unroll
  for (int e = 0; e < 2 * N; ++e) w[e] = 0;
  unsigned pend = src2 != nullptr ? (1u << (2 * N)) - 1u : (1u << N) - 1u;
  uint64_t t0 = 0;
  for (uint32_t n = 1; pend && !abort; ++n) {
#pragma unroll
    for (int e = 0; e < 2 * N; ++e)
      if ((pend >> e) & 1u) w[e] = ld_word((e < N ? src : src2) + lane + 32 * (e % N));
#pragma unroll
    for (int e = 0; e < 2 * N; ++e)
      if (((pend >> e) & 1u) && word_tag(w[e]) == tag) pend &= ~(1u << e);
    if (pend) poll_bound(a, n, t0, abort);
  }
#pragma unroll
  for (int e = 0; e < N; ++e) {
    v[e] = abort ? 0.f : word_value(w[e]);
    v2[e] = abort ? 0.f : word_value(w[N + e]);
  }
}

// Position of input element k in xs: within each 256-wide chunk, the eight
// elements 8l .. 8l+7 that lane l multiplies sit as two float4 at 4l and 128 + 4l,
// so a warp reading one float4 per lane touches 512 contiguous bytes (no bank
// conflicts); a plain layout (32-byte lane stride) costs twice the wavefronts.
__device__ __forceinline__ int xs_pos(int k) {
  const int c = k >> 8, r = k & 255, l = r >> 3, j = r & 7;
  return (c << 8) + ((j & 4) << 5) + (l << 2) + (j & 3);
}

// Phase input: xs = v[0, K) once every word carries `tag` (or the embedding row
// of `tok`), times the norm gain g when given; returns the RMS factor
// 1 / sqrt(mean v^2 + eps) (1 without g), which the GEMV applies to each dot
// product: W (r g.v) = r (W (g.v)), so the factor's block reduction shares the
// input's one barrier instead of adding a pass over xs. Also prefetches `n_unit`
// per-unit epilogue values (this CTA's own residual rows, or bias) into unit_s.
// Every load of a round is issued before any is used: each is an L2 round trip.
// Out of line: its word pairs in flight would otherwise push the inlined token
// loop past the register budget (spills go to L2, since shared memory takes
// nearly all of L1).
#if QW_MEGA_BIG
// Wide inputs in rounds, and the per-lane input sums that int4 rows need (xsum).
template <int NP>  // (value, tag) word pairs per thread and round: a round covers 2 * NP * kNT inputs
__device__ __noinline__ float load_input_n(const MegaArgs& a, Smem& S, const uint64_t* v,
                                          uint32_t tag, int K, const uint16_t* g, bool from_embed,
                                          int tok, const uint64_t* unit_own,
                                          const uint16_t* unit_bf16, int n_unit, bool& abort) {
  constexpr int NT = kConsumers * 32;
  const int tid = threadIdx.x;
  float uv = 0.f;
  if (tid < n_unit)
    uv = unit_own ? word_value(__ldcg(unit_own + tid)) : (unit_bf16 ? bf16f(unit_bf16[tid]) : 0.f);
  float ss = 0.f;
  // Inputs wider than one round (only in the wide-input build) take several rounds;
  // the first one waits at the barrier for the previous phase's readers of xs.
  for (int r0 = 0; r0 < K; r0 += 2 * NP * NT) {
    const int p0 = r0 / 2;  // first word pair of the round
    // the norm gain (bf16), one pair per word pair, in the same batch of loads
    uint32_t gv[NP];
    if (g != nullptr) {
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        const int idx = p0 + tid + i * NT;
        gv[i] = idx * 2 < K ? *reinterpret_cast<const uint32_t*>(g + idx * 2) : 0u;
      }
    }
    if (from_embed) {
      const uint4* e = reinterpret_cast<const uint4*>(a.embed + (size_t)tok * K);
      constexpr int NE = (NP + 3) / 4;  // 8-element groups per thread: cover the round's
      const int e0 = r0 / 8;             // NP * NT / 4 groups, starting at group e0
      uint4 w[NE];
#pragma unroll
      for (int i = 0; i < NE; ++i) {
        const int j = tid + i * NT, idx = e0 + j;
        w[i] = j < NP * NT / 4 && idx * 8 < K ? e[idx] : make_uint4(0, 0, 0, 0);
      }
      if (r0 == 0) csync();  // the previous phase's readers of xs / unit_s are done
#pragma unroll
      for (int i = 0; i < NE; ++i) {
        const int j = tid + i * NT, idx = e0 + j;
        if (j < NP * NT / 4 && idx * 8 < K) {
          float* d = &S.xs[(idx >> 5) * 256 + (idx & 31) * 4];
          *reinterpret_cast<float4*>(d) =
              make_float4(__uint_as_float(w[i].x << 16), __uint_as_float(w[i].x & 0xffff0000u),
                          __uint_as_float(w[i].y << 16), __uint_as_float(w[i].y & 0xffff0000u));
          *reinterpret_cast<float4*>(d + 128) =
              make_float4(__uint_as_float(w[i].z << 16), __uint_as_float(w[i].z & 0xffff0000u),
                          __uint_as_float(w[i].w << 16), __uint_as_float(w[i].w & 0xffff0000u));
        }
      }
    } else {
      uint64_t w[NP][2];
      unsigned pend = 0;
#pragma unroll
      for (int i = 0; i < NP; ++i)
        if ((p0 + tid + i * NT) * 2 < K) pend |= 1u << i;
      uint64_t t0 = 0;
      for (uint32_t n = 1; pend && !abort; ++n) {
#pragma unroll
        for (int i = 0; i < NP; ++i)
          if ((pend >> i) & 1u) ld_words2(v + 2 * (p0 + tid + i * NT), w[i][0], w[i][1]);
#pragma unroll
        for (int i = 0; i < NP; ++i)
          if (((pend >> i) & 1u) && word_tag(w[i][0]) == tag && word_tag(w[i][1]) == tag)
            pend &= ~(1u << i);
        if (pend) poll_bound(a, n, t0, abort);
      }
      if (r0 == 0) csync();  // the previous phase's readers of xs / unit_s / red are done
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        const int idx = p0 + tid + i * NT;
        float ps = 0.f;
        if (idx * 2 < K) {
          const float x0 = word_value(w[i][0]), x1 = word_value(w[i][1]);
          ss = fmaf(x0, x0, fmaf(x1, x1, ss));
          const float g0 = g != nullptr ? __uint_as_float(gv[i] << 16) : 1.f;
          const float g1 = g != nullptr ? __uint_as_float(gv[i] & 0xffff0000u) : 1.f;
          *reinterpret_cast<float2*>(&S.xs[xs_pos(idx * 2)]) = make_float2(x0 * g0, x1 * g1);
          ps = x0 * g0 + x1 * g1;
        }
        if (a.wfmt == 1) {  // pairs 4m .. 4m + 3 (8 inputs) sit on 4 neighbouring lanes
          ps += __shfl_xor_sync(0xffffffffu, ps, 1);
          ps += __shfl_xor_sync(0xffffffffu, ps, 2);
          if ((idx & 3) == 0 && idx * 2 < K) S.xsum[idx >> 2] = 136.f * ps;
        }
      }
    }
  }
  if (tid < n_unit) S.unit_s[tid] = uv;
  if (g != nullptr) {
    if (from_embed) {  // once per token: the gain goes on in a second pass
      csync();
      for (int k = tid; k < K; k += NT) {
        const float xk = S.xs[xs_pos(k)];
        ss = fmaf(xk, xk, ss);
        S.xs[xs_pos(k)] = xk * bf16f(g[k]);
      }
    }
    ss = warp_sum(ss);
    if ((tid & 31) == 0) S.red[tid >> 5] = ss;
  }
  if (from_embed && a.wfmt == 1) {  // the gained embedding row is in xs
    csync();
    for (int m = tid; m * 8 < K; m += NT) {
      const float* q = &S.xs[(m >> 5) * 256 + (m & 31) * 4];
      const float4 lo = *reinterpret_cast<const float4*>(q);
      const float4 hi = *reinterpret_cast<const float4*>(q + 128);
      S.xsum[m] = 136.f * (((lo.x + lo.y) + (lo.z + lo.w)) + ((hi.x + hi.y) + (hi.z + hi.w)));
    }
  }
  abort = csync_or(abort);
  if (g == nullptr) return 1.f;
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kConsumers; ++i) tot += S.red[i];
  return 1.0f / sqrtf(tot / (float)K + a.eps);
}
#else
// One round; no input sums (the 7- and 11-warp builds take no int4 rows).
template <int NP>  // (value, tag) word pairs per thread: K <= 2 * NP * kNT
__device__ __noinline__ float load_input_n(const MegaArgs& a, Smem& S, const uint64_t* v,
                                          uint32_t tag, int K, const uint16_t* g, bool from_embed,
                                          int tok, const uint64_t* unit_own,
                                          const uint16_t* unit_bf16, int n_unit, bool& abort) {
  constexpr int NT = kConsumers * 32;
  const int tid = threadIdx.x;
  float uv = 0.f;
  if (tid < n_unit)
    uv = unit_own ? word_value(__ldcg(unit_own + tid)) : (unit_bf16 ? bf16f(unit_bf16[tid]) : 0.f);
  // the norm gain (bf16), one pair per word pair, in the same batch of loads
  uint32_t gv[NP];
  if (g != nullptr) {
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const int idx = tid + i * NT;
      gv[i] = idx * 2 < K ? *reinterpret_cast<const uint32_t*>(g + idx * 2) : 0u;
    }
  }
  float ss = 0.f;
  if (from_embed) {
    const uint4* e = reinterpret_cast<const uint4*>(a.embed + (size_t)tok * K);
    constexpr int NE = (NP + 3) / 4;
    uint4 w[NE];
#pragma unroll
    for (int i = 0; i < NE; ++i) {
      const int idx = tid + i * NT;
      w[i] = idx * 8 < K ? e[idx] : make_uint4(0, 0, 0, 0);
    }
    csync();  // the previous phase's readers of xs / unit_s are done
#pragma unroll
    for (int i = 0; i < NE; ++i) {
      const int idx = tid + i * NT;
      if (idx * 8 < K) {
        float* d = &S.xs[(idx >> 5) * 256 + (idx & 31) * 4];
        *reinterpret_cast<float4*>(d) =
            make_float4(__uint_as_float(w[i].x << 16), __uint_as_float(w[i].x & 0xffff0000u),
                        __uint_as_float(w[i].y << 16), __uint_as_float(w[i].y & 0xffff0000u));
        *reinterpret_cast<float4*>(d + 128) =
            make_float4(__uint_as_float(w[i].z << 16), __uint_as_float(w[i].z & 0xffff0000u),
                        __uint_as_float(w[i].w << 16), __uint_as_float(w[i].w & 0xffff0000u));
      }
    }
  } else {
    uint64_t w[NP][2];
    unsigned pend = 0;
#pragma unroll
    for (int i = 0; i < NP; ++i)
      if ((tid + i * NT) * 2 < K) pend |= 1u << i;
    uint64_t t0 = 0;
    for (uint32_t n = 1; pend && !abort; ++n) {
#pragma unroll
      for (int i = 0; i < NP; ++i)
        if ((pend >> i) & 1u) ld_words2(v + 2 * (tid + i * NT), w[i][0], w[i][1]);
#pragma unroll
      for (int i = 0; i < NP; ++i)
        if (((pend >> i) & 1u) && word_tag(w[i][0]) == tag && word_tag(w[i][1]) == tag)
          pend &= ~(1u << i);
      if (pend) poll_bound(a, n, t0, abort);
    }
    csync();  // the previous phase's readers of xs / unit_s / red are done
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const int idx = tid + i * NT;
      if (idx * 2 < K) {
        const float x0 = word_value(w[i][0]), x1 = word_value(w[i][1]);
        ss = fmaf(x0, x0, fmaf(x1, x1, ss));
        const float g0 = g != nullptr ? __uint_as_float(gv[i] << 16) : 1.f;
        const float g1 = g != nullptr ? __uint_as_float(gv[i] & 0xffff0000u) : 1.f;
        *reinterpret_cast<float2*>(&S.xs[xs_pos(idx * 2)]) = make_float2(x0 * g0, x1 * g1);
      }
    }
  }
  if (tid < n_unit) S.unit_s[tid] = uv;
  if (g != nullptr) {
    if (from_embed) {  // once per token: the gain goes on in a second pass
      csync();
      for (int k = tid; k < K; k += NT) {
        const float xk = S.xs[xs_pos(k)];
        ss = fmaf(xk, xk, ss);
        S.xs[xs_pos(k)] = xk * bf16f(g[k]);
      }
    }
    ss = warp_sum(ss);
    if ((tid & 31) == 0) S.red[tid >> 5] = ss;
  }
  abort = csync_or(abort);
  if (g == nullptr) return 1.f;
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kConsumers; ++i) tot += S.red[i];
  return 1.0f / sqrtf(tot / (float)K + a.eps);
}
#endif

__device__ __forceinline__ float load_input(const MegaArgs& a, Smem& S, const uint64_t* v,
                                           uint32_t tag, int K, const uint16_t* g, bool from_embed,
                                           int tok, const uint64_t* unit_own,
                                           const uint16_t* unit_bf16, int n_unit, bool& abort) {
  constexpr int NP_1K = (1024 + 2 * kNT - 1) / (2 * kNT);      // pairs per thread, K <= 1024
  // wider inputs: one round when the buffer holds at most 3072, else rounds of
  // QW_MEGA_ROUND_PAIRS pairs per thread
  constexpr int NP_MAX = kMaxC * 256 <= 3072 ? (kMaxC * 256 + 2 * kNT - 1) / (2 * kNT)
                                             : QW_MEGA_ROUND_PAIRS;
  if (K <= 2 * NP_1K * kNT)
    return load_input_n<NP_1K>(a, S, v, tag, K, g, from_embed, tok, unit_own, unit_bf16, n_unit,
                               abort);
  return load_input_n<NP_MAX>(a, S, v, tag, K, g, from_embed, tok, unit_own, unit_bf16, n_unit,
                              abort);
}

template <int MAXC>
__device__ __forceinline__ void x_regs(const Smem& S, int K, float (&xr)[MAXC][8]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = 0; c < MAXC; ++c) {
    const int col = c * 256 + lane * 8;
    float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
    if (col < K) {
      lo = *reinterpret_cast<const float4*>(&S.xs[c * 256 + lane * 4]);
      hi = *reinterpret_cast<const float4*>(&S.xs[c * 256 + 128 + lane * 4]);
    }
    xr[c][0] = lo.x; xr[c][1] = lo.y; xr[c][2] = lo.z; xr[c][3] = lo.w;
    xr[c][4] = hi.x; xr[c][5] = hi.y; xr[c][6] = hi.z; xr[c][7] = hi.w;
  }
}

// 8 weights of row w at input `col` dotted with x: bf16 (16 bytes); int4 g128 (one
// 32-bit word of nibbles at byte col / 2, and the bf16 scale of their 128-wide group
// at byte K / 2 + (col / 128) * 2); or Q8_0 (8 int8 bytes and the fp16 scale of their
// 32-wide block, at byte K + (col / 32) * 2).
// For int4, xc is 136 x the sum of the 8 inputs (see dot8_i4_biased).
template <int WF>
__device__ __forceinline__ float dot8w(const uint8_t* w, int col, int K, const float (&x)[8],
                                       float acc, float xc = 0.f) {
  if constexpr (WF == 1) {
    const float sc = bf16f(*reinterpret_cast<const uint16_t*>(w + (K >> 1) + (col >> 7) * 2));
    return fmaf(dot8_i4_biased(*reinterpret_cast<const uint32_t*>(w + (col >> 1)), x) - xc, sc,
                acc);
  } else if constexpr (WF == 2) {
    const float sc = __half2float(*reinterpret_cast<const __half*>(w + K + (col >> 5) * 2));
    return dot8_i8(*reinterpret_cast<const uint2*>(w + col), x, sc, acc);
  } else {
    return dot8(*reinterpret_cast<const uint4*>(w + (size_t)col * 2), x, acc);
  }
}

// Per-lane partial dots of NR weight rows (bf16, int4 or Q8_0, in shared memory) with the
// input: the input either held in registers (MAXC chunks of 256) or read from xs.
// For int4 rows, xcr (registers) / xsum (shared memory) hold 136 x the sum of each
// lane's 8 inputs of a chunk.
template <int NR, int MAXC, int WF>
__device__ __forceinline__ void dotn(const uint8_t* const (&w)[NR], int K,
                                     const float (&xr)[MAXC > 0 ? MAXC : 1][8],
                                     const float (&xcr)[MAXC > 0 ? MAXC : 1], const float* xs,
                                     const float* xsum, float (&out)[NR]) {
  const int lane = threadIdx.x & 31;
  if constexpr (MAXC > 0) {
    // one FMA chain per (row, chunk), summed over chunks in order
    float p[NR][MAXC];
#pragma unroll
    for (int c = 0; c < MAXC; ++c) {
      const int col = c * 256 + lane * 8;
      if constexpr (WF != 0) {
#pragma unroll
        for (int r = 0; r < NR; ++r)
          p[r][c] = col < K ? dot8w<WF>(w[r], col, K, xr[c], 0.f, xcr[c]) : 0.f;
      } else {
        uint4 wv[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r)
          wv[r] = col < K ? *reinterpret_cast<const uint4*>(w[r] + (size_t)col * 2)
                          : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int r = 0; r < NR; ++r) p[r][c] = dot8(wv[r], xr[c], 0.f);
      }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      float t = 0.f;
#pragma unroll
      for (int c = 0; c < MAXC; ++c) t += p[r][c];
      out[r] = t;
    }
  } else {
    // two chains per row (even and odd chunks), added at the end
    float a0[NR], a1[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) a0[r] = a1[r] = 0.f;
    const float* xl = xs + lane * 4;
    int col = lane * 8, cb = 0;
#pragma unroll 1
    for (; col + 256 < K; col += 512, cb += 512) {
      const float4 l0 = *reinterpret_cast<const float4*>(xl + cb);
      const float4 h0 = *reinterpret_cast<const float4*>(xl + cb + 128);
      const float4 l1 = *reinterpret_cast<const float4*>(xl + cb + 256);
      const float4 h1 = *reinterpret_cast<const float4*>(xl + cb + 384);
      const float x0[8] = {l0.x, l0.y, l0.z, l0.w, h0.x, h0.y, h0.z, h0.w};
      const float x1[8] = {l1.x, l1.y, l1.z, l1.w, h1.x, h1.y, h1.z, h1.w};
      if constexpr (WF != 0) {
        const float c0 = WF == 1 ? xsum[(col >> 3)] : 0.f;
        const float c1 = WF == 1 ? xsum[(col >> 3) + 32] : 0.f;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          a0[r] = dot8w<WF>(w[r], col, K, x0, a0[r], c0);
          a1[r] = dot8w<WF>(w[r], col + 256, K, x1, a1[r], c1);
        }
      } else {
        uint4 wa[NR], wb[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          wa[r] = *reinterpret_cast<const uint4*>(w[r] + (size_t)col * 2);
          wb[r] = *reinterpret_cast<const uint4*>(w[r] + (size_t)(col + 256) * 2);
        }
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          a0[r] = dot8(wa[r], x0, a0[r]);
          a1[r] = dot8(wb[r], x1, a1[r]);
        }
      }
    }
    if (col < K) {
      const float4 l0 = *reinterpret_cast<const float4*>(xl + cb);
      const float4 h0 = *reinterpret_cast<const float4*>(xl + cb + 128);
      const float x0[8] = {l0.x, l0.y, l0.z, l0.w, h0.x, h0.y, h0.z, h0.w};
      const float c0 = WF == 1 ? xsum[(col >> 3)] : 0.f;
#pragma unroll
      for (int r = 0; r < NR; ++r) a0[r] = dot8w<WF>(w[r], col, K, x0, a0[r], c0);
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) out[r] = a0[r] + a1[r];
  }
}

// LM head: each lane's running best logit and whether it saw a NaN (merged over
// the warp at the end of the phase).
struct Best {
  float v;
  int i;
  int nan;
};

// Wait for the n chunks starting at chunk c (all of a phase that fits in the
// ring); done before the phase's input poll, so it stays off the critical path.
__device__ __forceinline__ void prewait(const MegaArgs& a, Smem& S, int c, int n, bool& abort) {
  if (n > kNS) return;
  for (int j = 0; j < n; ++j) ring_wait(a, &S.full[(c + j) % kNS], (uint32_t)(((c + j) / kNS) & 1), abort);
}

// Consume the chunks of one row-streamed phase (slice units [u0, u1) of
// `unit_bytes` each, `per_chunk` to a ring stage); chunk counter c advances by the
// phase's chunks. The epilogue, fixed at compile time:
//   EPI_STORE    y[u] = w_u . xs (+ bias[u])                     (tagged words)
//   EPI_RESIDUAL y[u] = y[u] + w_u . xs  (own rows; also to cap)   (tagged words)
//   EPI_SWIGLU   y[u] = silu(g_u . xs) * (up_u . xs)             (tagged words)
//   EPI_LOGITS   logits[u] = w_u . xs, running greedy best       (plain f32)
// A warp takes NR rows per iteration (NR / 2 gate/up units for SwiGLU). When the
// phase fits in the ring its chunks were waited for by prewait() and released
// together at the end; otherwise each warp waits for and releases them one at a time.
template <int MAXC, int EPI, int NR, int WF>
__device__ __forceinline__ void gemv_phase(const MegaArgs& a, uint8_t* ring, Smem& S, int& c,
                                           const Slice& sl, int K, float rs, uint64_t* ty,
                                           uint32_t tag,
                                           const uint16_t* bias, float* cap, Best& best,
                                           bool& abort) {
  constexpr int XR = MAXC > 0 ? MAXC : 1;
  constexpr int RPU = EPI == EPI_SWIGLU ? 2 : 1;  // rows per unit
  constexpr int UPI = NR / RPU;                   // units per warp iteration (one item)
  constexpr int SH = 32 / NR;                     // lanes per reduced row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float xr[XR][8], xcr[XR];
  if (MAXC > 0) x_regs<XR>(S, K, xr);
#pragma unroll
  for (int c = 0; c < XR; ++c) {  // int4: 136 x the sum of the lane's 8 inputs of chunk c
    xcr[c] = 0.f;
    if (WF == 1 && MAXC > 0)
      xcr[c] = 136.f * (((xr[c][0] + xr[c][1]) + (xr[c][2] + xr[c][3])) +
                        ((xr[c][4] + xr[c][5]) + (xr[c][6] + xr[c][7])));
  }
  const int pc = sl.per_chunk, n_units = sl.u1 - sl.u0, n_chunks = sl.n_chunks;
  const uint32_t unit_bytes = sl.unit_bytes, row_bytes = unit_bytes / RPU;
  const bool whole = EPI != EPI_LOGITS && n_chunks <= kNS;  // waited for by prewait()
  // Items of UPI units are dealt to the warps round-robin, the count running on
  // from stage to stage; an item never straddles two stages (a stage holds a
  // whole number of items, or one partial item), so a row's address is its
  // stage's base plus a multiple of the unit size: no division per row.
  int first = warp;  // this warp's first item in the current stage
  for (int j = 0; j < n_chunks && !abort; ++j) {
    if (!whole) {
      const bool ok = ring_wait(a, &S.full[(c + j) % kNS], (uint32_t)(((c + j) / kNS) & 1), abort);
      if (__any_sync(0xffffffffu, !ok)) {  // the whole warp gives up together
        abort = true;
        break;
      }
    }
    const int cu0 = j * pc, cn = min(pc, n_units - cu0);  // units [cu0, cu0 + cn) of the slice
    const uint8_t* stage = ring + (size_t)((c + j) % kNS) * kStage;
    const int items = (cn + UPI - 1) / UPI;
    int k = first;
    for (; k < items; k += kConsumers) {
      const int t = k * UPI;
      const uint8_t* w[NR];
#pragma unroll
      for (int r = 0; r < NR; ++r)  // rows past the stage's units reuse its last unit
        w[r] = stage + (size_t)min(t + r / RPU, cn - 1) * unit_bytes + (r % RPU) * row_bytes;
      float v[NR];
      dotn<NR, MAXC, WF>(w, K, xr, xcr, S.xs, S.xsum, v);
      const float sum = rows_reduce<NR>(v, lane) * rs;  // the input's RMS factor
      if constexpr (EPI == EPI_SWIGLU) {
        const float up = __shfl_down_sync(0xffffffffu, sum, SH);  // row 2k+1 onto row 2k
        const int tl = t + lane / (2 * SH);
        if (lane % (2 * SH) == 0 && tl < cn)
          st_tagged(ty + sl.u0 + cu0 + tl, sum / (1.0f + expf(-sum)) * up, tag);
      } else {
        const int tl = t + lane / SH;
        if (lane % SH == 0 && tl < cn) {
          const int iu = cu0 + tl, uu = sl.u0 + iu;
          if constexpr (EPI == EPI_STORE) {
            // unit_s: the bias (and, with an adapter, the LoRA update) of the first
            // kUnitPre units; an adapter is taken only when the slice fits unit_s
            const bool pre = bias != nullptr || (QW_MEGA_BIG && a.lora_r > 0);
            st_tagged(ty + uu,
                      sum + (pre ? (iu < kUnitPre ? S.unit_s[iu] : bf16f(bias[uu])) : 0.f), tag);
          } else if constexpr (EPI == EPI_RESIDUAL) {
            const float nv = (iu < kUnitPre ? S.unit_s[iu] : word_value(__ldcg(ty + uu))) + sum;
            st_tagged(ty + uu, nv, tag);
            if (cap) cap[uu] = nv;
          } else {  // EPI_LOGITS
            a.logits[uu] = sum;
            if (sum != sum) best.nan = 1;
            else if (sum > best.v) { best.v = sum; best.i = uu; }
          }
        }
      }
    }
    first = k - items;
    if (!whole) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[(c + j) % kNS]);
    }
  }
  if (whole && !abort) {
    __syncwarp();
    if (lane == 0)
      for (int j = 0; j < n_chunks; ++j) mbar_arrive(&S.empty[(c + j) % kNS]);
  }
  c += n_chunks;
}

// LoRA on q_proj and v_proj ("Emberglass" README, LoRA hot-swap): with the QKV
// phase's input in xs (gained, RMS factor rn not yet applied), t_q = A_q . x_n and
// t_v = A_v . x_n for the halves this CTA's rows need, then the update
// scale * B_row . t of each of its q and v rows is added to unit_s (which already
// holds the row's bias, or 0), so the QKV epilogue adds both at once. A_q / A_v are
// [r, K] and B_q / B_v [rows, r] bf16; the slice [u0, u1) of fused q/k/v rows has at
// most kUnitPre rows (checked on the host). Ends with a consumer barrier.
#if QW_MEGA_BIG  // the adapter runs in the wide-input build only
// Inlined: an out-of-line call here costs register spills around the call site.
__device__ __forceinline__ void lora_update(const MegaArgs& a, Smem& S, int l, int u0, int u1, int K,
                                         float rn) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = a.lora_r, qd = a.nq * a.hd, vd0 = qd + a.nkv * a.hd;
  const uint16_t* const* lp = a.lora + 4 * l;  // A_q, B_q, A_v, B_v
  const int j0 = u0 < qd ? 0 : r, j1 = u1 > vd0 ? 2 * r : r;  // rows of [A_q; A_v] needed
  // each warp: up to two A rows at a time, 8 chunks of 256 inputs per round of loads
  for (int j = j0 + warp; j < j1; j += 2 * kConsumers) {
    const int jb = j + kConsumers;
    const uint16_t* ra = j < r ? lp[0] + (size_t)j * K : lp[2] + (size_t)(j - r) * K;
    const uint16_t* rb = jb < j1 ? (jb < r ? lp[0] + (size_t)jb * K : lp[2] + (size_t)(jb - r) * K)
                                 : nullptr;
    float acc = 0.f, accb = 0.f;
    for (int c0 = 0; c0 * 256 < K; c0 += 8) {
      uint4 wa[8], wb[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int col = (c0 + i) * 256 + lane * 8;
        wa[i] = col < K ? *reinterpret_cast<const uint4*>(ra + col) : make_uint4(0, 0, 0, 0);
        wb[i] = col < K && rb ? *reinterpret_cast<const uint4*>(rb + col) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = c0 + i;
        if (c * 256 + lane * 8 < K) {
          const float4 lo = *reinterpret_cast<const float4*>(&S.xs[c * 256 + lane * 4]);
          const float4 hi = *reinterpret_cast<const float4*>(&S.xs[c * 256 + 128 + lane * 4]);
          const float x[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
          acc = dot8(wa[i], x, acc);
          accb = dot8(wb[i], x, accb);
        }
      }
    }
    acc = warp_sum(acc);
    accb = warp_sum(accb);
    if (lane == 0) {
      S.lora_t[j] = acc * rn;
      if (rb) S.lora_t[jb] = accb * rn;
    }
  }
  csync();
  for (int iu = tid; iu < u1 - u0; iu += kConsumers * 32) {
    const int uu = u0 + iu;
    const uint16_t* br = uu < qd ? lp[1] + (size_t)uu * r
                       : uu >= vd0 ? lp[3] + (size_t)(uu - vd0) * r : nullptr;
    if (br == nullptr) continue;
    const float* t = uu < qd ? S.lora_t : S.lora_t + r;
    float d = 0.f;
    for (int j = 0; j < r; j += 8) {
      float b[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) b[e] = j + e < r ? bf16f(br[j + e]) : 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) d = j + e < r ? fmaf(b[e], t[j + e], d) : d;
    }
    S.unit_s[iu] = fmaf(a.lora_scale, d, S.unit_s[iu]);
  }
  csync();
}
#endif

// Inputs up to 1024 wide stay in registers; wider ones are read from shared
// memory inside the dot (keeps the kernel under its register budget). X is the
// kernel's compile-time knowledge of the width: 1 at most 1024, 0 wider, 2 decided
// at run time (both bodies compiled in).
template <int EPI, int X, int NR, int WF>
__device__ __forceinline__ void gemv(const MegaArgs& a, uint8_t* ring, Smem& S, int& c,
                                     const Slice& sl, int K, float rs, uint64_t* ty, uint32_t tag,
                                     const uint16_t* bias, float* cap, Best& best, bool& abort) {
  if (X == 1 || (X == 2 && K <= 1024))
    gemv_phase<4, EPI, NR, WF>(a, ring, S, c, sl, K, rs, ty, tag, bias, cap, best, abort);
  else
    gemv_phase<0, EPI, NR, WF>(a, ring, S, c, sl, K, rs, ty, tag, bias, cap, best, abort);
}

// Chunks of a slice (the producer streams them in this count).
__device__ __forceinline__ int slice_chunks(const Slice& sl) { return sl.n_chunks; }

// Key-split combine of CTA sp (its partial outputs oacc and (m, l) in ml_s).
template <int HD>
__device__ __forceinline__ void attn_combine(const MegaArgs& a, Smem& S, const Split& sp, int HB, int GQ,
                  const float (&oacc)[(kGQ * HD + kNT - 1) / kNT], uint32_t tag_out, bool& abort) {
  constexpr int OUTS = (kGQ * HD + kNT - 1) / kNT;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Every split publishes its partial outputs and (m, l) per head as
  // tagged words, then combines a contiguous slice of the group's GQ * HD outputs
  // over all splits: out = sum_s f_s o_s with f_s = exp(m_s - M) / sum_s' exp(m_s' - M) l_s',
  // M the heads' maximum, summed in split order. Each split polls the (m, l) words
  // and the partials of its slice in one batch of loads (one L2 round trip once they
  // are there). The partial slots are reused by the next layer only after the
  // combined outputs have gone through o_proj, gate/up, down and the next QKV, all
  // of which the writers wait for.
  const size_t hs = (size_t)a.splits * (HD + 2);  // words per query head
  uint64_t* mp = a.mpart + (size_t)HB * hs;
  {
    uint64_t* my = mp + (size_t)sp.s * (HD + 2);
#pragma unroll
    for (int oi = 0; oi < OUTS; ++oi) {
      const int idx = tid + oi * kNT;
      if (idx < GQ * HD) {
        const int h = idx / HD, d = idx % HD;
        st_tagged(my + (size_t)h * hs + d, oacc[oi], tag_out);
      }
    }
    if (tid < GQ) {
      st_tagged(my + (size_t)tid * hs + HD, S.ml_s[2 * tid], tag_out);
      st_tagged(my + (size_t)tid * hs + HD + 1, S.ml_s[2 * tid + 1], tag_out);
    }
  }
  const int ns = sp.nsplit, n_out = GQ * HD;
  const int o0 = (int)((uint32_t)n_out * sp.s / ns), o1 = (int)((uint32_t)n_out * (sp.s + 1) / ns);
  const int nw = (o1 - o0) * ns;  // partial words of this split's slice
  csync();  // every warp has folded its last pass out of xs and pml_s
  // (m, l) of every split and head -> pml_s[2 (h ns + s)]
  for (int i = tid; i < GQ * ns; i += kNT) {
    const int h = i / ns, s2 = i % ns;
    const uint64_t* src = mp + (size_t)h * hs + (size_t)s2 * (HD + 2) + HD;
    uint64_t w0 = 0, w1 = 0, t0 = 0;
    for (uint32_t n = 1; !abort; ++n) {
      ld_words2(src, w0, w1);
      if (word_tag(w0) == tag_out && word_tag(w1) == tag_out) break;
      poll_bound(a, n, t0, abort);
    }
    S.pml_s[2 * i] = word_value(w0);
    S.pml_s[2 * i + 1] = word_value(w1);
  }
  abort = csync_or(abort);
  // per head (one warp each, lanes over the splits): f_s in place of m_s; the
  // denominator is summed lane-strided, then over the lanes in a fixed order
  for (int h = warp; h < GQ; h += kConsumers) {
    float* pm = S.pml_s + 2 * h * ns;
    float M = -INFINITY;
    for (int s2 = lane; s2 < ns; s2 += 32) M = fmaxf(M, pm[2 * s2]);
    M = warp_max(M);
    float den = 0.f;
    for (int s2 = lane; s2 < ns; s2 += 32) den = fmaf(expf(pm[2 * s2] - M), pm[2 * s2 + 1], den);
    const float inv = 1.0f / warp_sum(den);
    __syncwarp();
    for (int s2 = lane; s2 < ns; s2 += 32) pm[2 * s2] = expf(pm[2 * s2] - M) * inv;
  }
  csync();
  // the slice's partials, weighted, into xs[s n_o + (o - o0)] (consecutive threads read
  // consecutive outputs of one split); 8 polled loads per thread per round
  const int n_o = o1 - o0;
  float* wsum = S.xs;
  for (int base = 0; base < nw; base += 8 * kNT) {
    uint64_t w[8];
    unsigned pend = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      w[j] = 0;
      if (base + tid + j * kNT < nw) pend |= 1u << j;
    }
    auto word_at = [&](int i) {
      const int s2 = i / n_o, o = o0 + i % n_o, h = o / HD, d = o % HD;
      return mp + (size_t)h * hs + (size_t)s2 * (HD + 2) + d;
    };
    uint64_t t0 = 0;
    for (uint32_t n = 1; pend && !abort; ++n) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if ((pend >> j) & 1u) w[j] = ld_word(word_at(base + tid + j * kNT));
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (((pend >> j) & 1u) && word_tag(w[j]) == tag_out) pend &= ~(1u << j);
      if (pend) poll_bound(a, n, t0, abort);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = base + tid + j * kNT;
      if (i < nw) {
        const int s2 = i / n_o, o = o0 + i % n_o;
        wsum[i] = S.pml_s[2 * ((o / HD) * ns + s2)] * word_value(w[j]);
      }
    }
  }
  abort = csync_or(abort);
  for (int o = o0 + tid; o < o1; o += kNT) {
    const float* v = wsum + (o - o0);
    float acc = 0.f;
    for (int s2 = 0; s2 < ns; ++s2) acc += v[(size_t)s2 * n_o];
    const int h = o / HD, d = o % HD;
    st_tagged(a.attn_o + (size_t)(HB + h) * HD + d, acc, tag_out);
  }
}

// Split-K attention of CTA b: QK-norm + RoPE of its group's queries (and of the
// new key when its split holds pos), tiles of 32 keys from the ring, online
// softmax, then a partial (or the final output when there is one split); the
// partials are combined in split order, by split 0 (7- and 11-warp builds) or by
// every split for a slice of the outputs (wide-input build).
template <int HD, bool KB>
__device__ __forceinline__ void attn_phase(const MegaArgs& a, uint8_t* ring, Smem& S, int& c, int l,
                                           int pos, const Split& sp, const LayerDev& Ld,
                                           uint32_t tag_in, uint32_t tag_out, bool& abort) {
  constexpr int EPL = HD / 32, OUTS = (kGQ * HD + kNT - 1) / kNT;
  using KV = KvElem<KB>;  // cache element: f32, or bf16 (values rounded when stored)
  using KT = typename KV::T;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // GQ: query heads handled here; HB: global index of the first of them
  const int GQ = sp.nh, g = sp.g, HB = g * (a.nq / a.nkv) + sp.h0;
  // keys in passes of up to `pt` tiles; the first pass's tiles are waited for now,
  // before the q/k/v poll, so those waits overlap the hand-over from QKV
  const int pt = min(kPass, (kMaxC * 256) / (GQ * HD));
  const int stride = pt * kTK;
  {
    const int nt0 = (min(stride, sp.k1 - sp.k0) + kTK - 1) / kTK;
    for (int t = 0; t < nt0; ++t)
      ring_wait(a, &S.full[(c + t) % kNS], (uint32_t)(((c + t) / kNS) & 1), abort);
  }
  const size_t kv_layer = (size_t)a.nkv * a.cap * HD;
  KT* kc = reinterpret_cast<KT*>(a.k_cache) + (size_t)l * kv_layer + (size_t)g * a.cap * HD;
  KT* vc = reinterpret_cast<KT*>(a.v_cache) + (size_t)l * kv_layer + (size_t)g * a.cap * HD;
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
    const uint64_t* src = a.qkv + (size_t)(isq ? (HB + hh) : (a.nq + g)) * HD;
    const uint16_t* gain = isq ? Ld.q_norm : Ld.k_norm;
    // the norm gains and the RoPE row do not depend on the polled data: load them first
    float gv[EPL];
    float2 csv[EPL / 2];
#pragma unroll
    for (int e = 0; e < EPL; ++e) gv[e] = gain != nullptr ? bf16f(gain[lane + 32 * e]) : 1.f;
#pragma unroll
    for (int e = 0; e < EPL / 2; ++e) csv[e] = rrow[lane + 32 * e];
    // the key row's warp polls the value row in the same rounds
    float v[EPL], vv[EPL];
    poll_row<EPL>(a, src, isq ? nullptr : a.qkv + (size_t)(a.nq + a.nkv + g) * HD, tag_in, v, vv,
                  abort);
    if (gain != nullptr) {
      float sq = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) sq = fmaf(v[e], v[e], sq);
      sq = warp_sum(sq);
      const float r = 1.0f / sqrtf(sq / (float)HD + a.eps);
#pragma unroll
      for (int e = 0; e < EPL; ++e) v[e] = v[e] * r * gv[e];
    }
#pragma unroll
    for (int e = 0; e < EPL / 2; ++e) {
      const float2 cs = csv[e];
      const float x0 = v[e], x1 = v[e + EPL / 2];
      v[e] = x0 * cs.x - x1 * cs.y;
      v[e + EPL / 2] = x1 * cs.x + x0 * cs.y;
    }
    if (isq) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) S.q_s[hh * HD + lane + 32 * e] = v[e] * scale;
    } else {
#pragma unroll
      for (int e = 0; e < EPL; ++e) {  // the stored (for bf16: rounded) row is what is used
        const int d = lane + 32 * e;
        const KT ks = KV::store(v[e]), vs = KV::store(vv[e]);
        S.kn_s[d] = KV::load(&ks);
        S.vn_s[d] = KV::load(&vs);
        if (sp.h0 == 0) {  // one CTA of the group appends the row
          kc[(size_t)pos * HD + d] = ks;
          vc[(size_t)pos * HD + d] = vs;
        }
      }
    }
  }
  abort = csync_or(abort);
  float oacc[OUTS];
#pragma unroll
  for (int i = 0; i < OUTS; ++i) oacc[i] = 0.f;
  // Per pass: scores of every (key, head), one online-softmax update per head,
  // P.V per tile, then the per-tile partial outputs folded in tile order. A warp
  // takes a whole 32-key tile: lanes split the head dimension (DPL dims each), so
  // K and V rows are read as 512 contiguous bytes, and a 32-way transposing
  // reduction leaves key j's score on lane j. Scratch: scores and probabilities
  // in pml_s (free until the combine), P.V partials in xs (free during attention).
  constexpr int DPL = HD / 32;
  float* sc = S.pml_s;                      // [GQ][pt * kTK]
  float* pp = S.pml_s + kGQ * kPass * kTK;  // [GQ][pt * kTK]
  float* part = S.xs;                       // [nt * KP][GQ][HD]
  for (int p0 = sp.k0; p0 < sp.k1; p0 += stride) {
    const int nkp = min(stride, sp.k1 - p0);
    const int nt = (nkp + kTK - 1) / kTK;
    // P.V splits each tile into KP = 2^kpl parts (up to 4) while the parts still
    // go one per warp and their partials fit in xs
    int kpl = 0;
    while (kpl < 2 && nt * (2 << kpl) <= kConsumers && nt * (2 << kpl) * GQ * HD <= kMaxC * 256)
      ++kpl;
    const int KP = 1 << kpl;
    if (p0 != sp.k0)
      for (int t = 0; t < nt; ++t)
        ring_wait(a, &S.full[(c + t) % kNS], (uint32_t)(((c + t) / kNS) & 1), abort);
    abort = csync_or(abort);
    auto kt = [&](int t) { return reinterpret_cast<KT*>(ring + (size_t)((c + t) % kNS) * kStage); };
    if (!abort) {
      if (owns_pos && pos >= p0 && pos < p0 + nkp) {
        KT* Kp = kt((pos - p0) / kTK) + ((pos - p0) % kTK) * HD;
        for (int e = tid; e < HD; e += kNT) {
          Kp[e] = KV::store(S.kn_s[e]);
          Kp[kTK * HD + e] = KV::store(S.vn_s[e]);
        }
        // these generic writes into a ring stage must be ordered before the
        // producer's next bulk copy into the same stage (async proxy)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        csync();
      }
      // scores, two heads and eight keys at a time, the (tile, 8-key group) pairs
      // dealt round-robin to the warps: lane partials over its DPL dims, then a
      // transposing reduction leaves key r of the group on lanes 4r .. 4r+3
      constexpr int GPT = kTK / 8;  // 8-key groups per tile
      for (int gi = warp; gi < nt * GPT; gi += kConsumers) {
        const int t = gi / GPT, j0 = (gi % GPT) * 8;
        const KT* Kt = kt(t) + lane * DPL;
        const int nk = min(kTK, nkp - t * kTK);
        for (int h0 = 0; h0 < GQ; h0 += 2) {
          const bool two = h0 + 1 < GQ;
          if (j0 >= nk) {  // the group lies wholly past the keys
            if (lane < 8) {
              sc[h0 * stride + t * kTK + j0 + lane] = -INFINITY;
              if (two) sc[(h0 + 1) * stride + t * kTK + j0 + lane] = -INFINITY;
            }
            continue;
          }
          float q0[DPL], q1[DPL];
#pragma unroll
          for (int e = 0; e < DPL; ++e) {
            q0[e] = S.q_s[h0 * HD + lane * DPL + e];
            q1[e] = two ? S.q_s[(h0 + 1) * HD + lane * DPL + e] : 0.f;
          }
          {
            float s0[8], s1[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              float kv[DPL];
              if constexpr (DPL == 4) {
                const float4 k4 = KV::load4(Kt + (j0 + j) * HD);
                kv[0] = k4.x; kv[1] = k4.y; kv[2 % DPL] = k4.z; kv[3 % DPL] = k4.w;
              } else {
                const float2 k2 = KV::load2(Kt + (j0 + j) * HD);
                kv[0] = k2.x; kv[1] = k2.y;
              }
              float a0 = 0.f, a1 = 0.f;
#pragma unroll
              for (int e = 0; e < DPL; ++e) {
                a0 = fmaf(q0[e], kv[e], a0);
                a1 = fmaf(q1[e], kv[e], a1);
              }
              s0[j] = a0;
              s1[j] = a1;
            }
            const float r0 = rows_reduce<8>(s0, lane);
            const float r1 = rows_reduce<8>(s1, lane);
            if ((lane & 3) == 0) {
              const int j = j0 + (lane >> 2);  // keys past the split hold stale rows
              sc[h0 * stride + t * kTK + j] = j < nk ? r0 : -INFINITY;
              if (two) sc[(h0 + 1) * stride + t * kTK + j] = j < nk ? r1 : -INFINITY;
            }
          }
        }
      }
      csync();
      // online softmax, one warp per head
      for (int h = warp; h < GQ; h += kConsumers) {
        float sv[kPass];
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < kPass; ++i) {
          const int k = lane + 32 * i;
          sv[i] = k < nkp ? sc[h * stride + k] : -INFINITY;
          m = fmaxf(m, sv[i]);
        }
        const float m_old = S.ml_s[2 * h], l_old = S.ml_s[2 * h + 1];
        const float m_new = fmaxf(m_old, warp_max(m));
        float ps = 0.f;
#pragma unroll
        for (int i = 0; i < kPass; ++i) {
          const int k = lane + 32 * i;
          if (k < nt * kTK) {
            const float e = k < nkp ? expf(sv[i] - m_new) : 0.f;
            pp[h * stride + k] = e;
            ps += e;
          }
        }
        ps = warp_sum(ps);
        const float alpha = expf(m_old - m_new);
        if (lane == 0) {
          S.ml_s[2 * h] = m_new;
          S.ml_s[2 * h + 1] = l_old * alpha + ps;
          S.al_s[h] = alpha;
        }
      }
      csync();
      // P.V of one tile part (kTK / KP keys), two heads at a time, the parts dealt
      // round-robin to the warps: lane holds DPL adjacent output dims
      for (int i = warp; i < nt * KP; i += kConsumers) {
        const int t = i >> kpl, ja = (i & (KP - 1)) * (kTK >> kpl);
        const int jb = min(min(kTK, nkp - t * kTK), ja + (kTK >> kpl));
        const KT* Vt = kt(t) + kTK * HD + lane * DPL;
        for (int h0 = 0; h0 < GQ; h0 += 2) {
          const bool two = h0 + 1 < GQ;
          const float* p0r = pp + h0 * stride + t * kTK;
          const float* p1r = pp + (two ? h0 + 1 : h0) * stride + t * kTK;
          float c0[DPL], c1[DPL];
#pragma unroll
          for (int e = 0; e < DPL; ++e) c0[e] = c1[e] = 0.f;
          for (int j = ja; j < jb; ++j) {
            float vv[DPL];
            if constexpr (DPL == 4) {
              const float4 v4 = KV::load4(Vt + j * HD);
              vv[0] = v4.x; vv[1] = v4.y; vv[2 % DPL] = v4.z; vv[3 % DPL] = v4.w;
            } else {
              const float2 v2 = KV::load2(Vt + j * HD);
              vv[0] = v2.x; vv[1] = v2.y;
            }
            const float pa = p0r[j], pb = p1r[j];
#pragma unroll
            for (int e = 0; e < DPL; ++e) {
              c0[e] = fmaf(pa, vv[e], c0[e]);
              c1[e] = fmaf(pb, vv[e], c1[e]);
            }
          }
          float* d0 = part + (i * GQ + h0) * HD + lane * DPL;
#pragma unroll
          for (int e = 0; e < DPL; ++e) d0[e] = c0[e];
          if (two) {
            float* d1 = part + (i * GQ + h0 + 1) * HD + lane * DPL;
#pragma unroll
            for (int e = 0; e < DPL; ++e) d1[e] = c1[e];
          }
        }
      }
    }
    csync();
    // the pass's stages are free: one counted arrival each, by one thread
    if (tid == 0)
      for (int t = 0; t < nt; ++t) mbar_arrive_all(&S.empty[(c + t) % kNS]);
    c += nt;
    // fold the pass into the running outputs, tiles in order
#pragma unroll
    for (int oi = 0; oi < OUTS; ++oi) {
      const int idx = tid + oi * kNT;
      if (idx < GQ * HD && !abort) {
        const int h = idx / HD, d = idx % HD;
        float acc = oacc[oi] * S.al_s[h];
        for (int i = 0; i < nt * KP; ++i) acc += part[(i * GQ + h) * HD + d];
        oacc[oi] = acc;
      }
    }
  }
  // No barrier here: what follows reads only registers and ml_s (stable since the
  // last softmax step), and the next writer of xs and pml_s passes a barrier first.

  if (sp.nsplit == 1) {
#pragma unroll
    for (int oi = 0; oi < OUTS; ++oi) {
      const int idx = tid + oi * kNT;
      if (idx < GQ * HD) {
        const int h = idx / HD, d = idx % HD;
        st_tagged(a.attn_o + (size_t)(HB + h) * HD + d, oacc[oi] / S.ml_s[2 * h + 1], tag_out);
      }
    }
    return;
  }
#if QW_MEGA_BIG
  // every split combines a slice of the outputs (at GQ = 8 and 64 keys per split the
  // combine is a large part of the attention)
  attn_combine<HD>(a, S, sp, HB, GQ, oacc, tag_out, abort);
#else
  // split 0 combines; in the 7- and 11-warp builds this ran faster than the spread
  // combine (Qwen3-0.6B 575 against 596 us/token, 8K context 1086 against 1109, same box)
  // Key split: every split but the first publishes its partial outputs and
  // (m, l) per head as tagged words; split 0 polls them (one L2 round trip once
  // they are there) and combines in split order. The partial slots are reused
  // by the next layer only after the combined output has gone through o_proj,
  // gate/up, down and the next QKV, all of which the writers wait for.
  const size_t hs = (size_t)a.splits * (HD + 2);  // words per query head
  uint64_t* mp = a.mpart + (size_t)HB * hs;
  if (sp.s != 0) {
    uint64_t* my = mp + (size_t)sp.s * (HD + 2);
#pragma unroll
    for (int oi = 0; oi < OUTS; ++oi) {
      const int idx = tid + oi * kNT;
      if (idx < GQ * HD) {
        const int h = idx / HD, d = idx % HD;
        st_tagged(my + (size_t)h * hs + d, oacc[oi], tag_out);
      }
    }
    if (tid < GQ) {
      st_tagged(my + (size_t)tid * hs + HD, S.ml_s[2 * tid], tag_out);
      st_tagged(my + (size_t)tid * hs + HD + 1, S.ml_s[2 * tid + 1], tag_out);
    }
    return;
  }
  const int ns = sp.nsplit;
  for (int i = tid; i < GQ * ns; i += kNT) {
    const int h = i / ns, s2 = i % ns;
    float m = S.ml_s[2 * h], lsum = S.ml_s[2 * h + 1];
    if (s2 != 0) {
      const uint64_t* src = mp + (size_t)h * hs + (size_t)s2 * (HD + 2) + HD;
      uint64_t w0 = 0, w1 = 0;
      uint64_t t0 = 0;
      for (uint32_t n = 1; !abort; ++n) {
        ld_words2(src, w0, w1);
        if (word_tag(w0) == tag_out && word_tag(w1) == tag_out) break;
        poll_bound(a, n, t0, abort);
      }
      m = word_value(w0);
      lsum = word_value(w1);
    }
    S.pml_s[2 * i] = m;
    S.pml_s[2 * i + 1] = lsum;
  }
  abort = csync_or(abort);
#pragma unroll
  for (int oi = 0; oi < OUTS; ++oi) {
    const int idx = tid + oi * kNT;
    if (idx < GQ * HD) {
      const int h = idx / HD, d = idx % HD;
      const float* pm = S.pml_s + 2 * h * ns;
      float M = -INFINITY;
      for (int s2 = 0; s2 < ns; ++s2) M = fmaxf(M, pm[2 * s2]);
      float den = 0.f;
      for (int s2 = 0; s2 < ns; ++s2) den = fmaf(expf(pm[2 * s2] - M), pm[2 * s2 + 1], den);
      const uint64_t* po = mp + (size_t)h * hs + d;
      float num = expf(pm[0] - M) * oacc[oi];
      for (int s0 = 1; s0 < ns; s0 += 8) {  // the others' outputs, 8 polled loads at a time
        uint64_t w[8];
        unsigned pend = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          w[j] = 0;
          if (s0 + j < ns) pend |= 1u << j;
        }
        uint64_t t0 = 0;
        for (uint32_t n = 1; pend && !abort; ++n) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if ((pend >> j) & 1u) w[j] = ld_word(po + (size_t)(s0 + j) * (HD + 2));
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (((pend >> j) & 1u) && word_tag(w[j]) == tag_out) pend &= ~(1u << j);
          if (pend) poll_bound(a, n, t0, abort);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (s0 + j < ns) num = fmaf(expf(pm[2 * (s0 + j)] - M), word_value(w[j]), num);
      }
      st_tagged(a.attn_o + (size_t)(HB + h) * HD + d, num / den, tag_out);
    }
  }
#endif
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
  const Slice geo[5] = {phase_slice(a, K_QKV, b, G), Slice{}, phase_slice(a, K_O, b, G),
                        phase_slice(a, K_GU, b, G), phase_slice(a, K_DOWN, b, G)};
  auto layer_slice = [&](int kind, const LayerDev& Ld) {
    Slice sl = geo[kind];
    sl.base = phase_base(kind, Ld);
    return sl;
  };
  bool ok = true;
  for (int l = 0; l < a.L && ok; ++l) {
    const LayerDev Ld = a.layers[l];
    ok = stream_slice(layer_slice(K_QKV, Ld));
    const uint32_t eb = a.kv_bf16 ? 2u : 4u;  // bytes per cache element
    const size_t row0 = (size_t)l * kv_layer + (size_t)sp.g * a.cap * a.hd;
    const uint8_t* kc = reinterpret_cast<const uint8_t*>(a.k_cache) + row0 * eb;
    const uint8_t* vc = reinterpret_cast<const uint8_t*>(a.v_cache) + row0 * eb;
    for (int t0 = sp.k0; ok && t0 < sp.k1; t0 += kTK) {
      const uint32_t n = (uint32_t)min(kTK, sp.k1 - t0) * a.hd * eb;
      ok = issue(kc + (size_t)t0 * a.hd * eb, n, vc + (size_t)t0 * a.hd * eb, n,
                 (uint32_t)kTK * a.hd * eb);
    }
    ok = ok && stream_slice(layer_slice(K_O, Ld));
    ok = ok && stream_slice(layer_slice(K_GU, Ld));
    ok = ok && stream_slice(layer_slice(K_DOWN, Ld));
  }
  if (ok) stream_slice(phase_slice(a, K_LM, b, G));
  // Leave only once every copy issued into this CTA's shared memory has landed.
  for (int cc = c > kNS ? c - kNS : 0; cc < c; ++cc)
    mbar_wait(&S.full[cc % kNS], (uint32_t)((cc / kNS) & 1), kDrainNs);
}

// ---- greedy argmax across the grid (last CTA to arrive reduces in order)
__device__ void argmax_finalize(const MegaArgs& a, Smem& S, const Best& o, int pos, uint32_t epoch) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x, G = gridDim.x;
  csync();  // every warp has read the LM head input's RMS factor out of red
  if (lane == 0) {
    S.red[warp] = o.nan ? __int_as_float(0x7fc00000) : o.v;
    S.redi[warp] = o.i;
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
    *a.epoch = epoch + 1u;  // every CTA read the epoch at its start
  }
}

// ---- consumers: the phases of one token
// Phase k of the token writes its output words with tag(k): per layer l, 5l+0
// fused q/k/v, 5l+1 attention output, 5l+2 residual after o_proj, 5l+3 SwiGLU
// output, 5l+4 residual after down.
// HD: head dim (0: either, decided at run time); XH, XQ, XI: width classes of
// the hidden, q and intermediate inputs (see gemv). Only the variants a shape
// needs are compiled into its kernel: the token loop's code is large and every
// unused variant inlined into it costs instruction-cache misses.
template <int HD, int XH, int XQ, int XI, bool KB, int WF>
__device__ void consume(const MegaArgs& a, uint8_t* ring, Smem& S, int pos, uint32_t epoch) {
  const int b = blockIdx.x, G = gridDim.x, tid = threadIdx.x;
  const int qd = a.nq * a.hd;
  const uint32_t tag0 = epoch * (uint32_t)(5 * a.L + 1) + 1u;
  bool abort = false;
  int c = 0;
  int tok = a.tok >= 0 ? a.tok : __ldcg(a.next_token);
  if (tok < 0 || tok >= a.V) {
    if (tid == 0 && b == 0) atomicOr(a.err, ERR_TOKEN);
    tok = 0;
  }
  const Split sp = attn_split(a, pos, b);
  Best best{-INFINITY, 0x7fffffff, 0};
  // the phases' slices are the same in every layer
  const Slice qs = phase_slice(a, K_QKV, b, G), os = phase_slice(a, K_O, b, G);
  const Slice gs = phase_slice(a, K_GU, b, G), ds = phase_slice(a, K_DOWN, b, G);
  for (int l = 0; l < a.L; ++l) {
    const LayerDev Ld = a.layers[l];  // one batch of loads per layer, kept in registers
    const uint32_t tq = tag0 + 5u * l, ta = tq + 1u, to = tq + 2u, tg = tq + 3u, td = tq + 4u;
    // fused QKV; layer 0 gathers the embedding row itself and seeds the residual rows it owns
    if (l == 0) {
      const uint16_t* e = a.embed + (size_t)tok * a.H;
      for (int r = os.u0 + tid; r < os.u1; r += kConsumers * 32) st_tagged(a.x + r, bf16f(e[r]), 0u);
      if (a.cap_emb && b == 0)
        for (int r = tid; r < a.H; r += kConsumers * 32) a.cap_emb[(size_t)pos * a.H + r] = bf16f(e[r]);
    }
    if (qs.u1 > qs.u0) {
      prewait(a, S, c, slice_chunks(qs), abort);
      const float rn = load_input(a, S, a.x, tq - 1u, a.H, Ld.attn_norm, l == 0, tok, nullptr,
                                  Ld.qkv_bias ? Ld.qkv_bias + qs.u0 : nullptr,
                                  min(qs.u1 - qs.u0, kUnitPre), abort);
#if QW_MEGA_BIG  // handles with an adapter run the wide-input build
      if (a.lora_r > 0 && (qs.u0 < qd || qs.u1 > qd + a.nkv * a.hd))
        lora_update(a, S, l, qs.u0, qs.u1, a.H, rn);
#endif
      gemv<EPI_STORE, XH, kNrQkv, WF>(a, ring, S, c, qs, a.H, rn, a.qkv, tq, Ld.qkv_bias, nullptr, best, abort);
    }
    // attention of this CTA's (kv head, key split)
    if (sp.active) {
      if (HD == 64 || (HD == 0 && a.hd == 64)) attn_phase<64, KB>(a, ring, S, c, l, pos, sp, Ld, tq, ta, abort);
      else attn_phase<128, KB>(a, ring, S, c, l, pos, sp, Ld, tq, ta, abort);
    }
    // o_proj + residual
    if (os.u1 > os.u0) {
      prewait(a, S, c, slice_chunks(os), abort);
      load_input(a, S, a.attn_o, ta, qd, nullptr, false, 0, a.x + os.u0, nullptr,
                 min(os.u1 - os.u0, kUnitPre), abort);
      gemv<EPI_RESIDUAL, XQ, kNrO, WF>(a, ring, S, c, os, qd, 1.f, a.x, to, nullptr, nullptr, best, abort);
    }
    // gate/up with SwiGLU
    if (gs.u1 > gs.u0) {
      prewait(a, S, c, slice_chunks(gs), abort);
      const float rn = load_input(a, S, a.x, to, a.H, Ld.mlp_norm, false, 0, nullptr, nullptr, 0,
                                  abort);
      gemv<EPI_SWIGLU, XH, kNrGu, WF>(a, ring, S, c, gs, a.H, rn, a.mlp, tg, nullptr, nullptr, best, abort);
    }
    // down + residual (block-0 checkpoint)
    if (ds.u1 > ds.u0) {
      prewait(a, S, c, slice_chunks(ds), abort);
      load_input(a, S, a.mlp, tg, a.I, nullptr, false, 0, a.x + ds.u0, nullptr,
                 min(ds.u1 - ds.u0, kUnitPre), abort);
      gemv<EPI_RESIDUAL, XI, kNrDown, WF>(a, ring, S, c, ds, a.I, 1.f, a.x, td, nullptr,
                         (l == 0 && a.cap_blk0) ? a.cap_blk0 + (size_t)pos * a.H : nullptr, best,
                         abort);
    }
  }
  // final RMSNorm + LM head + greedy argmax
  const Slice ls = phase_slice(a, K_LM, b, G);
  if (ls.u1 > ls.u0 || (a.cap_final && b == 0)) {
    const float rn = load_input(a, S, a.x, tag0 + 5u * (a.L - 1) + 4u, a.H, a.final_norm, false,
                                0, nullptr, nullptr, 0, abort);
    if (a.cap_final && b == 0)
      for (int r = tid; r < a.H; r += kConsumers * 32)
        a.cap_final[(size_t)pos * a.H + r] = S.xs[xs_pos(r)] * rn;
    gemv<EPI_LOGITS, XH, kNrLm, WF>(a, ring, S, c, ls, a.H, rn, nullptr, 0u, nullptr, nullptr, best, abort);
  }
  // each lane holding rows kept its own best: merge them onto lane 0 (ties to the lower index)
  best.nan = __any_sync(0xffffffffu, best.nan != 0) ? 1 : 0;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best.v, off);
    const int oi = __shfl_xor_sync(0xffffffffu, best.i, off);
    if (am_better(ov, oi, best.v, best.i)) { best.v = ov; best.i = oi; }
  }
  argmax_finalize(a, S, best, pos, epoch);
}

template <int HD, int XH, int XQ, int XI, bool KB, int WF>
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
  const uint32_t epoch = __ldcg(a.epoch);
  if (threadIdx.x < kConsumers * 32) consume<HD, XH, XQ, XI, KB, WF>(a, ring, S, pos, epoch);
  else if (threadIdx.x == kConsumers * 32) produce(a, ring, S, pos);
}

}  // namespace

namespace QW_MEGA_NS {

bool mega_supported(int H, int I, int qd, int hd, int gq, int n_layers, int wfmt) {
  // every unit a producer copies fits one ring stage: a fused q/k/v, o_proj, down or
  // LM-head row, or an interleaved gate/up row pair
  const int gran = wfmt == 1 ? 128 : wfmt == 2 ? 32 : 8;  // inputs per scale group
  return H <= kMaxC * 256 && I <= kMaxC * 256 && qd <= kMaxC * 256 && (hd == 64 || hd == 128) &&
         H % gran == 0 && I % gran == 0 && qd % gran == 0 && n_layers >= 1 && gq >= 1 &&
         gq <= kGQ && wfmt >= 0 && wfmt <= 2 && 2 * row_bytes_fmt(wfmt, H) <= kStage &&
         row_bytes_fmt(wfmt, I) <= kStage && row_bytes_fmt(wfmt, qd) <= kStage &&
         (QW_MEGA_BIG || wfmt != 1);
}

static_assert(offsetof(Smem, xs) % 16 == 0, "float4 stores into xs need 16-byte alignment");
static_assert(2 * kGQ * kPass * kTK <= 2 * kGQ * 160, "an attention pass's scores fit in pml_s");
static_assert((size_t)kNS * kStage + sizeof(Smem) <= 227 * 1024, "ring and state fit a CTA");
size_t mega_smem_bytes() { return (size_t)kNS * kStage + sizeof(Smem); }

#if QW_MEGA_BIG
// Wide inputs and int4 weights: [weight format bf16 / int4 / Q8_0][cache f32 / bf16],
// generic shape class, plus the Qwen2.5-3B class (head dim 128, hidden, q and
// intermediate all wider than 1024) with int4 weights and the f32 cache.
constexpr int kMegaCount = 7;
static const void* const kMegaFns[kMegaCount] = {
    reinterpret_cast<const void*>(decode_mega_kernel<0, 2, 2, 2, false, 0>),
    reinterpret_cast<const void*>(decode_mega_kernel<0, 2, 2, 2, true, 0>),
    reinterpret_cast<const void*>(decode_mega_kernel<0, 2, 2, 2, false, 1>),
    reinterpret_cast<const void*>(decode_mega_kernel<0, 2, 2, 2, true, 1>),
    reinterpret_cast<const void*>(decode_mega_kernel<0, 2, 2, 2, false, 2>),
    reinterpret_cast<const void*>(decode_mega_kernel<0, 2, 2, 2, true, 2>),
    reinterpret_cast<const void*>(decode_mega_kernel<128, 0, 0, 0, false, 1>)};

static const void* mega_kernel_for(const MegaArgs& a) {
  if (a.wfmt == 1 && !a.kv_bf16 && a.hd == 128 && a.H > 1024 && a.nq * a.hd > 1024 && a.I > 1024)
    return kMegaFns[6];
  return kMegaFns[a.wfmt * 2 + (a.kv_bf16 ? 1 : 0)];
}
#else
// [weight format bf16 / Q8_0][cache f32 / bf16][shape class]: the Qwen3-0.6B class
// (head dim 128, hidden <= 1024, q and intermediate wider) and the generic
// instantiation (Q8_0 with the f32 cache only).
constexpr int kMegaCount = 6;
static const void* const kMegaFns[kMegaCount] = {
    reinterpret_cast<const void*>(decode_mega_kernel<128, 1, 0, 0, false, 0>),
    reinterpret_cast<const void*>(decode_mega_kernel<0, 2, 2, 2, false, 0>),
    reinterpret_cast<const void*>(decode_mega_kernel<128, 1, 0, 0, true, 0>),
    reinterpret_cast<const void*>(decode_mega_kernel<0, 2, 2, 2, true, 0>),
    reinterpret_cast<const void*>(decode_mega_kernel<128, 1, 0, 0, false, 2>),
    reinterpret_cast<const void*>(decode_mega_kernel<0, 2, 2, 2, false, 2>)};

static const void* mega_kernel_for(const MegaArgs& a) {
  const int fmt = a.wfmt == 2 ? 4 : (a.kv_bf16 ? 2 : 0);
  if (a.hd == 128 && a.H <= 1024 && a.nq * a.hd > 1024 && a.I > 1024) return kMegaFns[fmt];
  return kMegaFns[fmt + 1];
}
#endif

cudaError_t set_mega_attributes() {
  const void* const* fns = kMegaFns;
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < kMegaCount; ++i) {
    const void* f = fns[i];
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)mega_smem_bytes());
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
  }
  return e;
}

bool is_mega_kernel(const void* fn) {
  for (int i = 0; i < kMegaCount; ++i)
    if (fn == kMegaFns[i]) return true;
  return false;
}

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
  void* args[] = {const_cast<MegaArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, mega_kernel_for(a), args);
}

}  // namespace QW_MEGA_NS
}  // namespace qw
