// Internal interface between the decode kernels and the engine (not part of the ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace qw {

// Bits of the device error word.
enum : int { ERR_TIMEOUT = 1, ERR_TOKEN = 2, ERR_NAN = 4 };

// Wait bound used to drain copies still in flight after a wait gave up.
constexpr uint64_t kDrainNs = 2000000000ull;

// GEMV epilogues.
enum : int { EPI_STORE = 0, EPI_RESIDUAL = 1, EPI_SWIGLU = 2, EPI_LOGITS = 3 };

// Where the greedy argmax of the LM head goes (all optional).
struct ArgmaxOut {
  float* blk_val;             // [gridDim.x] per-CTA best logit   (scratch)
  int* blk_idx;               // [gridDim.x] per-CTA best index   (scratch)
  int* counter;               // arrival counter, 0 between launches (scratch)
  int* argmax;                // [1] final greedy id (-1 if a logit was NaN)
  int* next_token;            // [1] token fed to the next step when the host passes none
  int* pos;                   // [1] device position; incremented after the argmax is known
  int* tokens_by_pos;         // [cap] argmax recorded at the step's position
  int* status;                // [2] argmax and a copy of the error word, for the host
};

// y = epilogue(W . prologue(x)); W rows grouped in units of `rpu` rows.
struct GemvArgs {
  const uint8_t* w;       // packed rows, unit u = rows [u*rpu, (u+1)*rpu)
  int wfmt;               // 0: bf16 rows (K*2 bytes); 1: int4 g128 rows = K/2 nibble bytes,
                          //    then K/128 bf16 scales at byte `scale_off`, padded to 16 bytes;
                          // 2: Q8_0 rows = K int8 bytes, then K/32 fp16 scales at `scale_off`,
                          //    padded to 16 bytes
  uint32_t scale_off;
  int n_units;
  int rpu;                // rows per unit: 1, or 2 for interleaved gate/up
  int K;                  // input length (multiple of 8)
  uint32_t row_bytes;     // K * 2
  const float* x;         // [K] input
  const uint16_t* norm_g; // RMSNorm gain of the prologue (bf16 [K]) or nullptr
  float eps;
  const uint16_t* bias;   // EPI_STORE: bf16 [n_units] or nullptr
  float* y;               // output
  float* norm_out;        // if set, CTA 0 writes the normalised input here (row `pos`)
  float* cap_out;         // EPI_RESIDUAL: if set, the updated y row is also written here
  const int* pos;         // device position (capture row index) or nullptr
  // launch geometry, filled by plan_gemv
  int ks;                 // warps that split K (1, 2, 4 or 8)
  int cpw;                // 256-column chunks per warp
  uint32_t stage_bytes;
  int n_stages;
  int units_per_stage;
  uint32_t off_red, off_x, off_stage;  // shared-memory offsets
  ArgmaxOut am;           // EPI_LOGITS only
  // EPI_STORE only: LoRA on the q rows [0, lora_q_rows) and the v rows
  // [lora_v_row0, lora_v_row0 + lora_v_rows): y += lora_scale * B[row] . t
  const uint16_t* lora_bq;  // bf16 [q rows, r] or nullptr
  const uint16_t* lora_bv;  // bf16 [v rows, r]
  const float* lora_t;      // [2 r]: A_q . x_n, then A_v . x_n
  int lora_r, lora_q_rows, lora_v_row0, lora_v_rows;
  float lora_scale;
  int* err;
  uint64_t wait_ns;
};
// Bytes of one int4 g128 row of K inputs in the packed layout above.
__host__ __device__ inline uint32_t int4_row_bytes(int K) {
  return (uint32_t)K / 2 + (((uint32_t)K / 128 * 2 + 15) & ~15u);
}
cudaError_t launch_pack_int4_rows(const uint8_t* nib, const uint16_t* scales, int rows, int K,
                                  uint8_t* dst, int dst_row0, int dst_row_step, cudaStream_t s);
__host__ __device__ inline uint32_t q8_row_bytes(int K) {
  return (uint32_t)K + (((uint32_t)K / 32 * 2 + 15) & ~15u);
}
cudaError_t launch_pack_q8_rows(const int8_t* q, const uint16_t* scales, int rows, int K,
                                uint8_t* dst, int dst_row0, int dst_row_step, cudaStream_t s);
// Q8_0 quantiser: rows of `cols` inputs (f32, or bf16 bits when w_bf16) -> int8 rows at
// q + r * q_stride (bytes) and fp16 scale bits at scales + r * s_stride (elements).
cudaError_t launch_quantize_q8(const void* w, bool w_bf16, int rows, int cols, int8_t* q,
                               size_t q_stride, uint16_t* scales, size_t s_stride,
                               cudaStream_t s);

struct AttnArgs {
  const float* qkv;        // raw [(nq + 2 nkv) * hd]
  const uint16_t* q_norm;  // bf16 [hd] or nullptr
  const uint16_t* k_norm;
  const float2* rope;      // [cap][hd/2] (cos, sin) or nullptr (formed in fp64 in-kernel)
  float rope_theta;
  void* k_cache;           // [nkv][cap][hd] of this layer: f32, or bf16 bits when kv_bf16
  void* v_cache;
  int kv_bf16;
  int cap;
  const int* pos_ptr;      // device position, or nullptr to use pos_const
  int pos_const;
  int nq, nkv;
  float eps;
  int nsplit_max, min_keys;
  float* part_o;           // [nq][nsplit_max][hd] (scratch)
  float* part_ml;          // [nq][nsplit_max][2]  (scratch)
  int* counters;           // [nkv] arrival counters, 0 between launches (scratch)
  float* out;              // [nq * hd]
  int* err;
  uint64_t wait_ns;
};

struct EmbedArgs {
  const uint16_t* table;   // bf16 [V, H]
  int V, H;
  const int* pos;
  int tok;                 // token from the host (a graph-node parameter), or -1
  const int* next_token;   // previous step's argmax, used when tok < 0
  float* x;                // [H]
  float* cap_out;          // capture rows [cap][H] or nullptr
  int* err;
};

// ---- planning / launching (decode_kernels.cu) ----
void plan_gemv(GemvArgs& a, int grid, uint32_t max_stage_bytes, int max_stages);
size_t gemv_smem_bytes(const GemvArgs& a);
cudaError_t launch_gemv(int epi, const GemvArgs& a, int grid, bool pdl, cudaStream_t s);
cudaError_t launch_attention(const AttnArgs& a, int hd, bool pdl, cudaStream_t s);
size_t attention_smem_bytes(int hd);
int attention_gq_max();
// Whether a stand-alone attention call with `n_splits` key splits per KV head and
// `gq` query heads per KV head fits the combine's scratch in the tile stages.
bool attention_splits_fit(int gq, int hd, int n_splits);
// Text for qw_last_error(NULL) after a failed handle-less call (stand-alone ops
// outside engine.cu).
void set_op_error(const char* msg);
constexpr int kAttnMinKeys = 64;
cudaError_t launch_embed(const EmbedArgs& a, cudaStream_t s);
const void* embed_kernel_fn();
cudaError_t launch_rope_table(float2* table, int cap, int hd, float theta, cudaStream_t s);
cudaError_t launch_quantize_int4(const float* w, int rows, int cols, uint8_t* packed,
                                 uint16_t* scales, cudaStream_t s);
cudaError_t set_kernel_attributes();

// ---- prefill (prefill_kernels.cu) ----
// C[M, N] = (A_hi + A_lo)[M, K] . B[N, K]^T on tcgen05 tensor cores; A and B bf16 K-major.
enum : int { GEPI_STORE = 0, GEPI_RESID = 1, GEPI_SWIGLU = 2 };
struct GemmArgs {
  int M, N, K;
  int a_split;             // 1: A_hi only; 2: A_hi + A_lo (activation split in two bf16)
  int b_split;             // filled by launch_gemm: 2 when B comes as B_hi + B_lo (a weight
                           // that bf16 holds only as two terms: dequantised int4)
  int n_stages;            // filled by launch_gemm
  float* out;              // STORE: out[m, n] = acc (+ bias[n]); RESID: out[m, n] += acc
  int ldo;
  const uint16_t* bias;    // STORE: bf16 [N] or nullptr
  uint16_t* out_hi;        // SWIGLU: columns (2i, 2i+1) are (gate_i, up_i); writes
  uint16_t* out_lo;        //   silu(gate)*up split in two bf16 at [m, i]
  int ldb;
  float* cap_out;          // RESID: also write the updated rows at [cap_row0 + m] (or nullptr)
  int cap_row0;
  // RESID only: K split over ksplit CTAs per output tile (grid z), whose epilogues add
  // their partial sums to out in split order; flags: one int per output tile, 0 at rest
  int ksplit;
  int* flags;
  int* err;
  uint64_t wait_ns;
};
// The residual GEMMs of a prefill (o_proj, down: N = hidden) run with 128-column
// tiles and K split in two, so that twice as many CTAs share the narrow output.
constexpr int kResidBN = 128;
constexpr int kResidSplit = 2;
bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                       uint32_t box_rows);
// b_lo: the weight's lo term (nullptr for exact bf16 weights); with it each product is
// A_hi B_hi + A_lo B_hi + A_hi B_lo.
cudaError_t launch_gemm(int bn, int epi, const CUtensorMap& a_hi, const CUtensorMap& a_lo,
                        const CUtensorMap& b, const CUtensorMap* b_lo, GemmArgs g,
                        cudaStream_t s);
cudaError_t set_gemm_attributes();
int* gemm_op_err_word();
cudaError_t launch_embed_rows(const int* ids, int T, const uint16_t* table, int V, int H,
                              float* X, float* cap, int row0, int* err, cudaStream_t s);
cudaError_t launch_rmsnorm_rows(const float* X, int T, int H, const uint16_t* g, float eps,
                                uint16_t* hi, uint16_t* lo, float* f32, int f32_row0,
                                cudaStream_t s);
cudaError_t launch_qk_rope_kv_rows(const float* QKV, int T, int p0, int nq, int nkv, int hd,
                                   const uint16_t* qn, const uint16_t* kn, float eps,
                                   const float2* rope, uint16_t* q_hi, uint16_t* q_lo,
                                   void* kc, void* vc, bool kv_bf16, int cap,
                                   uint16_t* kv_split, cudaStream_t s);
// Causal prefill attention on tcgen05 (kind::f16, three MMAs per product of two-bf16
// splits): Q rows [T][nq][hd] (scaled by 1/sqrt(hd)) as q_hi/q_lo, keys and values
// 0 .. p0+T-1 of one layer from its f32 cache (kc, vc: [nkv][cap][hd]), split per call
// (f32, or bf16 when kv_bf16) into kv_split (attn_kv_bytes) as K hi, K lo [nkv][kv_rows][hd] and V^T hi, V^T lo
// [nkv][hd][kv_rows] (kv_rows = attn_kv_rows(cap)); output as the two-bf16 split
// [T][nq*hd]. The tensor maps (make_attn_maps) cover q_hi/q_lo [max_t, nq*hd] and the
// four kv_split planes.
struct FaMaps {
  CUtensorMap q_hi, q_lo, k_hi, k_lo, vt_hi, vt_lo;
};
struct FaArgs {
  int p0, T, nq, nkv;
  int kv_rows;
  uint16_t* o_hi;
  uint16_t* o_lo;
  int* err;
  uint64_t wait_ns;
  int nqb, max_ch;   // query blocks of this launch; key chunks per block at most
  float* part_o;     // [nq][max_qblocks][max_ch][128][hd] unnormalised partial outputs
  float2* part_ml;   // [nq][max_qblocks][max_ch][128] (reference maximum, row sum), base 2
  int* counters;     // [nq][nqb] chunk arrivals, 0 between launches
};
constexpr int kFaQueryRows = 128, kFaKeyRows = 64;  // query rows per CTA, keys per tile
int attn_kv_rows(int cap);
size_t attn_kv_bytes(int nkv, int hd, int cap);
bool make_attn_maps(FaMaps* m, const uint16_t* q_hi, const uint16_t* q_lo, int max_t, int nq,
                    const uint16_t* kv_split, int nkv, int hd, int cap);
// part: scratch of attn_part_bytes(nq, max_t, cap, hd), zeroed once (T <= max_t)
size_t attn_part_bytes(int nq, int max_t, int cap, int hd);
int attn_max_chunks(int cap);
int attn_max_qblocks(int max_t);
cudaError_t launch_attn_prefill(const FaMaps& maps, const void* kc, const void* vc, bool kv_bf16,
                                uint16_t* kv_split, void* part, int max_t, int cap, int p0,
                                int T, int nq, int nkv, int hd, uint16_t* o_hi, uint16_t* o_lo,
                                int* err, uint64_t wait_ns, cudaStream_t s);
// int4 g128 packed rows (int4_row_bytes(K) each) -> exact two-bf16 planes hi, lo [rows][K]
// (the weight operand of the int4 prefill GEMMs).
cudaError_t launch_dequant_int4_split(const uint8_t* src, int rows, int K, uint16_t* hi,
                                      uint16_t* lo, cudaStream_t s);
cudaError_t launch_set_int(int* p, int v, cudaStream_t s);
cudaError_t set_prefill_attributes();

// ---- sampling (sample.cu) ----
constexpr int kMaxSampleTopK = 256;
size_t sample_workspace_bytes(int V, int k);
bool sample_shape_ok(int V, int k);  // k <= kMaxSampleTopK and the final sort fits one CTA
cudaError_t set_sample_attributes();
cudaError_t launch_sample(const float* logits, int V, int k, float temperature, float top_p, float u,
                          int32_t* token, void* workspace, cudaStream_t s);

// ---- persistent decode step (decode_mega.cu) ----
struct LayerDev {  // per-layer device pointers of the packed weights
  const uint8_t* qkv;
  const uint16_t* qkv_bias;
  const uint8_t* o;
  const uint8_t* gateup;
  const uint8_t* down;
  const uint16_t* attn_norm;
  const uint16_t* mlp_norm;
  const uint16_t* q_norm;
  const uint16_t* k_norm;
};
struct MegaArgs {
  int L, H, nq, nkv, hd, I, V;
  float eps;
  const uint16_t* embed;
  const uint8_t* lm_head;
  const uint16_t* final_norm;
  const LayerDev* layers;  // device array [L]
  void* k_cache;           // [L][nkv][cap][hd]: f32, or bf16 bits when kv_bf16
  void* v_cache;
  int kv_bf16;
  int wfmt;                // weight rows (projections and LM head): 0 bf16, 1 int4 g128
                           // (the mega_big build), 2 Q8_0
  int cap;
  const float2* rope;
  // activations as tagged words (f32 value low, phase tag high)
  uint64_t* x;             // [H] residual
  uint64_t* qkv;           // [(nq+2nkv) hd]
  uint64_t* attn_o;        // [nq hd]
  uint64_t* mlp;           // [I]
  uint32_t* epoch;         // launches so far; tags are derived from it
  float* logits;           // [V]
  uint64_t* mpart;         // [nq][splits][hd + 2] key-split partials as tagged words: the
                           // unnormalised output, then the running max m and sum l
  int splits;              // CTAs per KV head (gridDim.x / nkv)
  ArgmaxOut am;
  const int* pos;
  int tok;                 // host token (graph-node argument) or -1: use *next_token
  const int* next_token;
  float* cap_emb;          // capture rows or nullptr
  float* cap_blk0;
  float* cap_final;
  // LoRA on q_proj and v_proj: device array [L][4] of A_q, B_q, A_v, B_v (bf16 [r, H],
  // [q rows, r], [r, H], [v rows, r]); lora_r = 0 without an adapter
  const uint16_t* const* lora;
  int lora_r;
  float lora_scale;
  int* err;
  uint64_t wait_ns;
};
// Units of a phase whose epilogue values the persistent kernel prefetches per CTA; a
// LoRA adapter runs on that kernel only when a CTA's fused q/k/v slice fits.
constexpr int kMegaUnitPre = 64;
// Three builds of the kernel: mega (7 consumer warps) and mega_wide (11) for bf16 and
// Q8_0 weights with inputs up to 3072 wide; mega_big (11 warps, inputs up to 11264
// wide, one ring stage fewer) for wider shapes and int4 g128 weights.
#define QW_MEGA_BUILD_DECL(NS)                                                          \
  namespace NS {                                                                        \
  bool mega_supported(int H, int I, int qd, int hd, int gq, int n_layers, int wfmt);   \
  size_t mega_smem_bytes();                                                             \
  cudaError_t launch_mega(const MegaArgs& a, int grid, cudaStream_t s);                 \
  cudaError_t set_mega_attributes();                                                    \
  bool is_mega_kernel(const void* fn); /* one of this build's kernel instantiations */ \
  }
QW_MEGA_BUILD_DECL(mega)
QW_MEGA_BUILD_DECL(mega_wide)
QW_MEGA_BUILD_DECL(mega_big)
#undef QW_MEGA_BUILD_DECL

}  // namespace qw
