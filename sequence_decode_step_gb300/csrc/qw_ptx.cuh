// Device helpers shared by the decode and prefill kernels: inline PTX for
// mbarriers, bulk/tensor TMA copies, programmatic dependent launch, and small
// warp/block reductions.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace qw {

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
// Bulk (non-tensor) TMA copy global -> shared; both addresses 16-byte aligned,
// size a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for phase `parity` of `bar` for at most limit_ns; limit 0 gives up at once.
static __device__ __noinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (limit_ns == 0) return false;
  // %globaltimer is read only every 16th failed try (it costs far more than a
  // try_wait); the bound starts counting at the first read.
  uint64_t t0 = 0;
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 15u) != 0) continue;
    const uint64_t now = globaltimer_ns();
    if (t0 == 0) t0 = now;
    else if (now - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
// f32 -> bf16 bits, round to nearest even (finite inputs).
__device__ __forceinline__ uint16_t bf16_rne(float x) {
  const uint32_t u = __float_as_uint(x);
  return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

// Key/value cache elements: f32, or bf16 bits (the cache format of a handle). Loads of
// 2 or 4 consecutive elements widened to f32, and the stored form of a value.
template <bool KB>
struct KvElem {
  using T = float;
  static __device__ __forceinline__ T store(float x) { return x; }
  static __device__ __forceinline__ float load(const T* p) { return *p; }
  static __device__ __forceinline__ float2 load2(const T* p) {
    return *reinterpret_cast<const float2*>(p);
  }
  static __device__ __forceinline__ float4 load4(const T* p) {
    return *reinterpret_cast<const float4*>(p);
  }
};
template <>
struct KvElem<true> {
  using T = uint16_t;
  static __device__ __forceinline__ T store(float x) { return bf16_rne(x); }
  static __device__ __forceinline__ float load(const T* p) { return bf16f(*p); }
  static __device__ __forceinline__ float2 load2(const T* p) {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
  }
  static __device__ __forceinline__ float4 load4(const T* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
  }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// Deterministic block sum for 256 threads: warp sums, then the 8 added in order.
__device__ __forceinline__ float block_sum_256(float v, float* scratch8) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) scratch8[warp] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) t += scratch8[i];
  return t;
}

// 8 bf16 weights (one 16-byte load) dotted with 8 floats.
__device__ __forceinline__ float dot8(const uint4 w, const float (&x)[8], float acc) {
  acc = fmaf(__uint_as_float(w.x << 16), x[0], acc);
  acc = fmaf(__uint_as_float(w.x & 0xffff0000u), x[1], acc);
  acc = fmaf(__uint_as_float(w.y << 16), x[2], acc);
  acc = fmaf(__uint_as_float(w.y & 0xffff0000u), x[3], acc);
  acc = fmaf(__uint_as_float(w.z << 16), x[4], acc);
  acc = fmaf(__uint_as_float(w.z & 0xffff0000u), x[5], acc);
  acc = fmaf(__uint_as_float(w.w << 16), x[6], acc);
  acc = fmaf(__uint_as_float(w.w & 0xffff0000u), x[7], acc);
  return acc;
}


// Sum NR (a power of two) per-lane partials over the warp with a transposing
// butterfly: each halving step exchanges half of the remaining values, so NR rows
// cost NR - 1 + 5 - log2(NR) shuffles instead of 5 NR. Afterwards lanes
// [r * 32/NR, (r + 1) * 32/NR) hold the full sum of row r. Fixed order.
template <int NR>
__device__ __forceinline__ float rows_reduce(const float (&v)[NR], int lane) {
  float cur[NR];
#pragma unroll
  for (int i = 0; i < NR; ++i) cur[i] = v[i];
#pragma unroll
  for (int s = 0, n = NR, bit = 16; s < 5; ++s, bit >>= 1) {
    if (n > 1) {
      const bool up = lane & bit;
      const int h = n / 2;
#pragma unroll
      for (int i = 0; i < (NR > 1 ? NR / 2 : 1); ++i) {
        if (i < h) {
          const float keep = up ? cur[i + h] : cur[i], send = up ? cur[i] : cur[i + h];
          cur[i] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
        }
      }
      n = h;
    } else {
      cur[0] += __shfl_xor_sync(0xffffffffu, cur[0], bit);
    }
  }
  return cur[0];
}

// Argmax order: larger value wins, equal values go to the lower index.
__device__ __forceinline__ bool am_better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}


// 8 int4 weights (one 32-bit word: element 2b in the low nibble of byte b, value
// nibble - 8) dotted with 8 floats, times the group scale. A nibble n becomes the
// float 2^23 + n by placing it in the mantissa of 2^23 (one byte permute), and
// subtracting 2^23 + 8 leaves n - 8 exactly.
__device__ __forceinline__ float i4f(uint32_t v, uint32_t b) {
  return __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7540u | b)) - 8388616.0f;
}
__device__ __forceinline__ float dot8_i4(uint32_t w, const float (&x)[8], float s, float acc) {
  const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
  float p = i4f(lo, 0) * x[0];
  p = fmaf(i4f(hi, 0), x[1], p);
  p = fmaf(i4f(lo, 1), x[2], p);
  p = fmaf(i4f(hi, 1), x[3], p);
  p = fmaf(i4f(lo, 2), x[4], p);
  p = fmaf(i4f(hi, 2), x[5], p);
  p = fmaf(i4f(lo, 3), x[6], p);
  p = fmaf(i4f(hi, 3), x[7], p);
  return fmaf(p, s, acc);
}

// The same 8 nibbles as floats 128 + n (n = q + 8 in the mantissa of 128, one byte
// permute, exact) dotted with 8 floats: sum (128 + n_i) x_i. No subtraction per
// weight; the caller removes 136 sum x_i, which leaves sum q_i x_i. The offset costs
// about 5 of the 24 mantissa bits of a 128-input group's sum (its terms are ~136 |x|
// against a result of ~5 sqrt(128) |x|), a relative error near 1e-6.
__device__ __forceinline__ float b128f(uint32_t v, uint32_t b) {
  return __uint_as_float(__byte_perm(v, 0x43000000u, 0x7044u | (b << 8)));
}
__device__ __forceinline__ float dot8_i4_biased(uint32_t w, const float (&x)[8]) {
  const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
  float p = b128f(lo, 0) * x[0];
  p = fmaf(b128f(hi, 0), x[1], p);
  p = fmaf(b128f(lo, 1), x[2], p);
  p = fmaf(b128f(hi, 1), x[3], p);
  p = fmaf(b128f(lo, 2), x[4], p);
  p = fmaf(b128f(hi, 2), x[5], p);
  p = fmaf(b128f(lo, 3), x[6], p);
  p = fmaf(b128f(hi, 3), x[7], p);
  return p;
}

// 8 int8 weights (two 32-bit words, element i in byte i % 4 of word i / 4, two's
// complement) dotted with 8 floats, times the block scale. A byte is flipped to
// b ^ 0x80 = q + 128, placed in the mantissa of 2^23 (one byte permute), and
// subtracting 2^23 + 128 leaves q exactly.
__device__ __forceinline__ float i8f(uint32_t v, uint32_t b) {
  return __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7540u | b)) - 8388736.0f;
}
__device__ __forceinline__ float dot8_i8(uint2 w, const float (&x)[8], float s, float acc) {
  const uint32_t a = w.x ^ 0x80808080u, b = w.y ^ 0x80808080u;
  float p = i8f(a, 0) * x[0];
  p = fmaf(i8f(a, 1), x[1], p);
  p = fmaf(i8f(a, 2), x[2], p);
  p = fmaf(i8f(a, 3), x[3], p);
  p = fmaf(i8f(b, 0), x[4], p);
  p = fmaf(i8f(b, 1), x[5], p);
  p = fmaf(i8f(b, 2), x[6], p);
  p = fmaf(i8f(b, 3), x[7], p);
  return fmaf(p, s, acc);
}

// ------------------------------------------------------------------ TMA tensor copies
// 2-D tiled load global -> shared (box given by the tensor map), completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// ------------------------------------------------------------------ tcgen05 (5th-gen tensor cores)
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] . B[smem desc]^T, kind::f16 (bf16 inputs, f32 accumulate).
__device__ __forceinline__ void tc_mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[smem desc] . B[smem desc]^T, kind::tf32 (f32 operands read as tf32,
// f32 accumulate); K = 8 per instruction (32 bytes of each operand row).
__device__ __forceinline__ void tc_mma_tf32(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Plain arrival on an mbarrier in this CTA's shared memory.
__device__ __forceinline__ void mbar_arrive_cta(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Arrive on `bar` once every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns of TMEM into registers (warp-collective).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// Ties registers filled by tmem_ld16 to a preceding tmem_ld_wait: an empty volatile
// statement that "rewrites" them, so no use of them can be scheduled above the wait.
__device__ __forceinline__ void tmem_regs_ready(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
}
// 16 registers into 32 lanes x 16 consecutive 32-bit TMEM columns (warp-collective).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// One 32-bit TMEM column of the warp's 32 lanes (warp-collective), to and from a register.
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v));
}
__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
  uint32_t v;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(v) : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(v)::"memory");
  return v;
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// Shared-memory matrix descriptor for a K-major operand tile written by TMA with
// 128-byte swizzling: rows of 64 bf16 (128 B), 8-row atoms of 1024 B (SBO), start
// address in 16-byte units, descriptor version 1, layout SWIZZLE_128B.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor of kind::tf32: tf32 A and B (K-major), f32 D, shape M x N.
__host__ __device__ constexpr uint32_t idesc_tf32_f32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
// Instruction descriptor of kind::f16: bf16 A and B (K-major), f32 D, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

}  // namespace qw
