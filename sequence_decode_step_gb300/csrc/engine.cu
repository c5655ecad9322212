// The qw_* C ABI: handle, weight packing, decode-step CUDA graph, stand-alone ops.
//
// One decode step is recorded once as a CUDA graph on a private stream and
// replayed on the handle's stream:
//   embed -> for each layer [QKV GEMV (+RMSNorm, +bias) -> attention (QK-norm,
//   RoPE, KV append, split-K flash decode, combine) -> o_proj GEMV (+residual)
//   -> gate/up GEMV (+RMSNorm, SwiGLU) -> down GEMV (+residual)]
//   -> LM head GEMV (+final RMSNorm, greedy argmax, pos += 1).
// Every kernel after the first is launched with programmatic dependent launch,
// so each one streams its weights while its predecessor finishes. The position,
// the next token and the greedy id stay on the device; the host token for a
// position is read by the embed kernel from a mapped pinned ring, and the
// greedy id and the error word are written to mapped pinned memory.

#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <cstddef>
#include <string>
#include <vector>

#include "qw.h"
#include "qw_internal.h"

using namespace qw;

namespace {

thread_local std::string g_last_error;

struct LayerW {
  const uint16_t* qkv = nullptr;       // [(nq+2nkv)*hd, H]
  const uint16_t* qkv_bias = nullptr;  // [(nq+2nkv)*hd] or null
  const uint16_t* o = nullptr;         // [H, nq*hd]
  const uint16_t* gateup = nullptr;    // [2I, H], row 2i gate i, row 2i+1 up i
  const uint16_t* down = nullptr;      // [H, I]
  const uint16_t* attn_norm = nullptr;
  const uint16_t* mlp_norm = nullptr;
  const uint16_t* q_norm = nullptr;
  const uint16_t* k_norm = nullptr;
};

class DeviceGuard {
 public:
  explicit DeviceGuard(int dev) {
    cudaGetDevice(&prev_);
    if (prev_ != dev) cudaSetDevice(dev);
    dev_ = dev;
  }
  ~DeviceGuard() {
    if (prev_ != dev_) cudaSetDevice(prev_);
  }

 private:
  int prev_ = 0, dev_ = 0;
};

bool g_attrs_set[64];

cudaError_t ensure_attributes(int dev) {
  if (dev >= 0 && dev < 64 && g_attrs_set[dev]) return cudaSuccess;
  cudaError_t e = set_kernel_attributes();
  if (e == cudaSuccess) e = set_gemm_attributes();
  if (e == cudaSuccess) e = set_prefill_attributes();
  if (e == cudaSuccess) e = set_sample_attributes();
  if (e == cudaSuccess) e = mega::set_mega_attributes();
  if (e == cudaSuccess) e = mega_wide::set_mega_attributes();
  if (e == cudaSuccess) e = mega_big::set_mega_attributes();
  if (e == cudaSuccess && dev >= 0 && dev < 64) g_attrs_set[dev] = true;
  return e;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

struct qw_handle {
  qw_config cfg{};
  int device = 0, num_sms = 0;
  cudaStream_t stream = nullptr, cap_stream = nullptr;
  bool own_stream = false;
  // weights (library-owned arena)
  uint8_t* warena = nullptr;
  size_t warena_bytes = 0;
  std::vector<LayerW> layers;
  const uint16_t* embed = nullptr;
  const uint16_t* lm_head = nullptr;  // aliases embed when tied
  const uint16_t* final_norm = nullptr;
  bool weights_loaded = false;
  // state buffers (one device allocation)
  uint8_t* sarena = nullptr;
  uint8_t* k_cache = nullptr;  // [L][nkv][cap][hd] elements of kv_elem bytes (f32 or bf16)
  uint8_t* v_cache = nullptr;
  bool kv_bf16 = false;
  size_t kv_elem = 4;
  float* x = nullptr;
  float* qkv = nullptr;
  float* attn_o = nullptr;
  float* mlp = nullptr;
  float* logits = nullptr;
  float2* rope = nullptr;
  float* part_o = nullptr;
  float* part_ml = nullptr;
  int* attn_counters = nullptr;
  uint64_t* mpart = nullptr;  // the persistent kernel's key-split partials (tagged words)
  void* sample_ws = nullptr;  // qw_sample_last's workspace (top_k up to kMaxSampleTopK)
  int* d_sample_tok = nullptr;
  float* blk_val = nullptr;
  int* blk_idx = nullptr;
  int* am_counter = nullptr;
  int* d_pos = nullptr;
  int* d_next_token = nullptr;
  int* d_argmax = nullptr;
  int* d_err = nullptr;
  int* d_tokens_by_pos = nullptr;
  int nsplit_max = 1;
  int lm_grid = 1;
  // batched prefill (T <= max_prefill_t): activations of all rows and their TMA maps
  int* pf_ids = nullptr;
  float* pf_x = nullptr;       // [Tmax, H] residual rows
  uint16_t* pf_xn_hi = nullptr;  // [Tmax, H] normalised rows, two-bf16 split
  uint16_t* pf_xn_lo = nullptr;
  float* pf_qkv = nullptr;     // [Tmax, (nq+2nkv) hd]
  uint16_t* pf_q_hi = nullptr;  // [Tmax, nq, hd] after QK-norm, RoPE, 1/sqrt(hd): two-bf16 split
  uint16_t* pf_q_lo = nullptr;
  uint16_t* pf_o_hi = nullptr;   // [Tmax, nq hd] attention output split
  uint16_t* pf_o_lo = nullptr;
  uint16_t* pf_m_hi = nullptr;   // [Tmax, I] SwiGLU output split
  uint16_t* pf_m_lo = nullptr;
  uint16_t* pf_kvs = nullptr;    // K and V^T of the context as two-bf16 splits (attention)
  int* pf_gemm_flags = nullptr;  // split-K hand-over per output tile of the residual GEMMs
  void* pf_attn_part = nullptr;  // partial attention outputs of query blocks cut into chunks
  CUtensorMap tm_xn_hi, tm_xn_lo, tm_o_hi, tm_o_lo, tm_m_hi, tm_m_lo;
  FaMaps tm_attn;  // attention operands: Q, K and V^T splits
  std::vector<CUtensorMap> tm_qkv, tm_ow, tm_gu, tm_dw;  // per layer, weight side
  // int4 models: one layer's weights dequantised into exact two-bf16 planes (reused
  // by every layer of a prefill) and their tensor maps [hi, lo]
  uint16_t* pf_w4 = nullptr;
  uint16_t *w4_qkv[2] = {}, *w4_o[2] = {}, *w4_gu[2] = {}, *w4_dw[2] = {};
  CUtensorMap tm_qkv4[2], tm_ow4[2], tm_gu4[2], tm_dw4[2];
  int* d_status = nullptr;  // [2] greedy id, error word (written by the LM head)
  // pinned host staging
  int* h_status = nullptr;  // [8]: argmax, error, set_pos staging, error copy, sampled id
  int* h_tokens = nullptr;  // [cap]
  // checkpoints
  bool capture_on = false, cap_valid = false;
  float* cap_emb = nullptr;
  float* cap_blk0 = nullptr;
  float* cap_final = nullptr;
  int cap_row0 = 0, cap_rows = 0;
  // graph
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  // The graph node that receives the host token (the embed kernel, or the persistent
  // decode kernel), a copy of its argument block and the token's offset inside it.
  cudaGraphNode_t tok_node = nullptr;
  cudaKernelNodeParams tok_params{};
  std::vector<uint8_t> tok_args;
  size_t tok_offset = 0;
  // decode path: the persistent cooperative kernel when the shape fits, else the
  // multi-kernel graph
  bool use_mega = false;
  bool mega_ok = false;
  bool mega_wide = false;  // the recorded step uses the 11-warp build (long contexts)
  bool mega_big = false;   // the shape takes the wide-input / int4 build at every position
  bool mega_big_ok = false;   // the wide-input build takes the shape (it runs every adapter)
  bool mega_lora_ok = false;  // ... and a CTA's fused q/k/v slice fits its LoRA update
  int path_pref = 0;          // the decode path asked for (qw_set_decode_path)
  const uint16_t** d_lora = nullptr;  // device [L][4] LoRA pointers for the persistent kernel
  std::vector<const uint16_t*> lora_tab;  // their host copy
  LayerDev* d_layers = nullptr;
  // the persistent kernel's activations as tagged words, and its launch epoch
  uint64_t* mx = nullptr;
  uint64_t* mqkv = nullptr;
  uint64_t* mattn = nullptr;
  uint64_t* mmlp = nullptr;
  uint32_t* d_epoch = nullptr;
  bool graph_dirty = true;
  uint64_t wait_ns = 1000000000ull;
  // host mirror
  int pos = 0;
  bool have_prev = false;
  bool lora_active = false;
  // LoRA (borrowed device pointers, per layer) and its A . x_n buffer
  std::vector<const uint16_t*> lora_qa, lora_qb, lora_va, lora_vb;
  int lora_rank = 0;
  float lora_scale = 0.f;
  float* lora_t = nullptr;  // [2 * 64]
  int wfmt = 0;             // linear weights: 0 bf16, 1 int4 g128, 2 Q8_0 (GemvArgs::wfmt)
  int lm_fmt = 0;           // LM head rows: 1 for untied int4 models, 2 for every Q8_0 model
  std::string err;
};

#define QW_FAIL(h, code, msg)                 \
  do {                                        \
    if (h) (h)->err = (msg);                  \
    else g_last_error = (msg);                \
    return (code);                            \
  } while (0)

#define QW_CUDA(h, call)                                                        \
  do {                                                                          \
    cudaError_t e_ = (call);                                                    \
    if (e_ != cudaSuccess) {                                                    \
      std::string m_ = std::string(#call) + ": " + cudaGetErrorString(e_);      \
      QW_FAIL(h, QW_ERR_CUDA, m_);                                              \
    }                                                                           \
  } while (0)

// ============================================================================ create / destroy
static int validate_config(const qw_config* c, std::string& why) {
  if (c->n_layers <= 0 || c->hidden <= 0 || c->n_q_heads <= 0 || c->n_kv_heads <= 0 ||
      c->head_dim <= 0 || c->intermediate <= 0 || c->vocab <= 0) {
    why = "every dimension must be positive";
    return QW_ERR_ARG;
  }
  if (c->head_dim != 64 && c->head_dim != 128) {
    why = "head_dim must be 64 or 128";
    return QW_ERR_ARG;
  }
  if (c->n_q_heads % c->n_kv_heads != 0 ||
      c->n_q_heads / c->n_kv_heads > attention_gq_max()) {
    why = "n_q_heads must be a multiple of n_kv_heads, at most 8 per kv head";
    return QW_ERR_ARG;
  }
  const int mult = c->weight_format == QW_WEIGHTS_INT4_G128 ? 128
                 : c->weight_format == QW_WEIGHTS_Q8_0     ? 32
                                                           : 8;
  if (c->hidden % mult || (c->n_q_heads * c->head_dim) % mult || c->intermediate % mult) {
    why = "hidden, n_q_heads*head_dim and intermediate must be multiples of 8 (128 for int4, "
          "32 for Q8_0)";
    return QW_ERR_ARG;
  }
  if (c->hidden > 16384 || c->intermediate > 16384 || c->n_q_heads * c->head_dim > 16384) {
    why = "hidden, intermediate and n_q_heads*head_dim are limited to 16384";
    return QW_ERR_ARG;
  }
  if (c->weight_format != QW_WEIGHTS_BF16 && c->weight_format != QW_WEIGHTS_INT4_G128 &&
      c->weight_format != QW_WEIGHTS_Q8_0) {
    why = "weight_format must be QW_WEIGHTS_BF16, QW_WEIGHTS_INT4_G128 or QW_WEIGHTS_Q8_0";
    return QW_ERR_ARG;
  }
  if (c->kv_format != QW_KV_F32 && c->kv_format != QW_KV_BF16) {
    why = "kv_format must be QW_KV_F32 or QW_KV_BF16";
    return QW_ERR_ARG;
  }
  if (c->max_ctx <= 0 || c->max_prefill_t < 0) {
    why = "max_ctx must be positive and max_prefill_t non-negative";
    return QW_ERR_ARG;
  }
  if (!(c->eps >= 0.f) || !(c->rope_theta > 0.f)) {
    why = "eps must be >= 0 and rope_theta > 0";
    return QW_ERR_ARG;
  }
  return QW_OK;
}

static void free_handle(qw_handle* h) {
  if (!h) return;
  if (h->exec) cudaGraphExecDestroy(h->exec);
  if (h->graph) cudaGraphDestroy(h->graph);
  if (h->warena) cudaFree(h->warena);
  if (h->d_layers) cudaFree(h->d_layers);
  if (h->sarena) cudaFree(h->sarena);
  if (h->cap_emb) cudaFree(h->cap_emb);
  if (h->h_status) cudaFreeHost(h->h_status);
  if (h->h_tokens) cudaFreeHost(h->h_tokens);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  if (h->own_stream && h->stream) cudaStreamDestroy(h->stream);
  delete h;
}

static int alloc_state(qw_handle* h) {
  const qw_config& c = h->cfg;
  const size_t L = c.n_layers, nkv = c.n_kv_heads, hd = c.head_dim, cap = c.max_ctx;
  const size_t qkv_rows = (size_t)(c.n_q_heads + 2 * c.n_kv_heads) * hd;
  h->nsplit_max = std::max(1, h->num_sms / c.n_kv_heads);
  // the persistent kernel takes bf16 weights, and Q8_0 weights with the f32 cache
  {
    // bf16, or Q8_0 with the f32 cache, at inputs up to 3072 wide: the 7- and 11-warp
    // builds; wider shapes, int4 weights with an untied int4 head, and Q8_0 with the
    // bf16 cache: the wide-input build
    const int wf = c.weight_format == QW_WEIGHTS_INT4_G128 ? 1
                 : c.weight_format == QW_WEIGHTS_Q8_0 ? 2 : 0;
    const int qd = c.n_q_heads * c.head_dim, gq = c.n_q_heads / c.n_kv_heads;
    const bool slices_ok = (int64_t)c.vocab * h->num_sms < (int64_t)1 << 31;  // 32-bit slices
    const bool small = (wf == 0 || (wf == 2 && c.kv_format == QW_KV_F32)) &&
                       mega::mega_supported(c.hidden, c.intermediate, qd, c.head_dim, gq,
                                            c.n_layers, wf) &&
                       mega_wide::mega_supported(c.hidden, c.intermediate, qd, c.head_dim, gq,
                                                 c.n_layers, wf);
    const bool big_ok = (wf != 1 || !c.tie_word_embeddings) &&
                        mega_big::mega_supported(c.hidden, c.intermediate, qd, c.head_dim, gq,
                                                 c.n_layers, wf);
    h->mega_ok = slices_ok && (small || big_ok);
    h->mega_big = slices_ok && !small && big_ok;
    h->mega_big_ok = slices_ok && big_ok;
  }
  h->use_mega = h->mega_ok;
  {
    const int grid = h->nsplit_max * c.n_kv_heads;
    const int rows = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
    h->mega_lora_ok = h->mega_big_ok && (rows + grid - 1) / grid <= kMegaUnitPre;
  }
  h->wfmt = c.weight_format == QW_WEIGHTS_INT4_G128 ? 1 : c.weight_format == QW_WEIGHTS_Q8_0 ? 2 : 0;
  h->lm_fmt = h->wfmt == 2 ? 2 : (h->wfmt == 1 && !c.tie_word_embeddings ? 1 : 0);
  h->lm_grid = std::min({c.vocab, h->num_sms, 1024});
  struct Piece { void** p; size_t bytes; };
  h->kv_bf16 = c.kv_format == QW_KV_BF16;
  h->kv_elem = h->kv_bf16 ? 2 : 4;
  const size_t kv_bytes = L * nkv * cap * hd * h->kv_elem;
  std::vector<Piece> pieces = {
      {(void**)&h->k_cache, kv_bytes},
      {(void**)&h->v_cache, kv_bytes},
      {(void**)&h->x, (size_t)c.hidden * 4},
      {(void**)&h->qkv, qkv_rows * 4},
      {(void**)&h->attn_o, (size_t)c.n_q_heads * hd * 4},
      {(void**)&h->mlp, (size_t)c.intermediate * 4},
      {(void**)&h->logits, (size_t)c.vocab * 4},
      {(void**)&h->rope, cap * (hd / 2) * sizeof(float2)},
      {(void**)&h->part_o, (size_t)c.n_q_heads * h->nsplit_max * hd * 4},
      {(void**)&h->part_ml, (size_t)c.n_q_heads * h->nsplit_max * 2 * 4},
      {(void**)&h->attn_counters, L * nkv * 4},
      {(void**)&h->mpart, (size_t)c.n_q_heads * h->nsplit_max * (hd + 2) * 8},
      {(void**)&h->sample_ws, sample_workspace_bytes(c.vocab, kMaxSampleTopK)},
      {(void**)&h->d_sample_tok, 4},
      {(void**)&h->blk_val, (size_t)std::max(h->lm_grid, h->num_sms) * 4},
      {(void**)&h->blk_idx, (size_t)std::max(h->lm_grid, h->num_sms) * 4},
      {(void**)&h->am_counter, 4},
      {(void**)&h->d_lora, (size_t)L * 4 * sizeof(void*)},
      {(void**)&h->d_pos, 4},
      {(void**)&h->d_next_token, 4},
      {(void**)&h->d_argmax, 4},
      {(void**)&h->d_err, 4},
      {(void**)&h->d_tokens_by_pos, cap * 4},
      {(void**)&h->d_status, 8},
      {(void**)&h->mx, (size_t)c.hidden * 8},
      {(void**)&h->mqkv, qkv_rows * 8},
      {(void**)&h->mattn, (size_t)c.n_q_heads * hd * 8},
      {(void**)&h->mmlp, (size_t)c.intermediate * 8},
      {(void**)&h->d_epoch, 4},
      {(void**)&h->lora_t, 2 * 64 * 4},
  };
  const size_t Tm = (size_t)c.max_prefill_t, H = c.hidden, I = c.intermediate;
  const size_t qd = (size_t)c.n_q_heads * hd;
  if (Tm > 0) {
    pieces.push_back({(void**)&h->pf_ids, Tm * 4});
    pieces.push_back({(void**)&h->pf_gemm_flags, ((Tm + 127) / 128) * ((H + 127) / 128) * 4});
    pieces.push_back({(void**)&h->pf_x, Tm * H * 4});
    pieces.push_back({(void**)&h->pf_xn_hi, Tm * H * 2});
    pieces.push_back({(void**)&h->pf_xn_lo, Tm * H * 2});
    pieces.push_back({(void**)&h->pf_qkv, Tm * qkv_rows * 4});
    pieces.push_back({(void**)&h->pf_q_hi, Tm * qd * 2});
    pieces.push_back({(void**)&h->pf_q_lo, Tm * qd * 2});
    pieces.push_back({(void**)&h->pf_o_hi, Tm * qd * 2});
    pieces.push_back({(void**)&h->pf_o_lo, Tm * qd * 2});
    pieces.push_back({(void**)&h->pf_m_hi, Tm * I * 2});
    pieces.push_back({(void**)&h->pf_m_lo, Tm * I * 2});
    pieces.push_back({(void**)&h->pf_kvs, attn_kv_bytes(c.n_kv_heads, c.head_dim, c.max_ctx)});
    pieces.push_back({(void**)&h->pf_attn_part,
                      attn_part_bytes(c.n_q_heads, (int)Tm, c.max_ctx, c.head_dim)});
    if (h->wfmt == 1)  // the hi and lo planes of one layer's four weight matrices
      pieces.push_back({(void**)&h->pf_w4,
                        2 * 2 * (qkv_rows * H + H * qd + 2 * I * H + H * I)});
  }
  size_t total = 0;
  for (auto& p : pieces) total = align_up(total, 256) + p.bytes;
  QW_CUDA(h, cudaMalloc((void**)&h->sarena, total));
  QW_CUDA(h, cudaMemsetAsync(h->sarena, 0, total, h->stream));
  size_t off = 0;
  for (auto& p : pieces) {
    off = align_up(off, 256);
    *p.p = h->sarena + off;
    off += p.bytes;
  }
  if (Tm > 0) {
    bool ok = make_tmap_bf16_2d(&h->tm_xn_hi, h->pf_xn_hi, Tm, H, 128) &&
              make_tmap_bf16_2d(&h->tm_xn_lo, h->pf_xn_lo, Tm, H, 128) &&
              make_tmap_bf16_2d(&h->tm_o_hi, h->pf_o_hi, Tm, qd, 128) &&
              make_tmap_bf16_2d(&h->tm_o_lo, h->pf_o_lo, Tm, qd, 128) &&
              make_tmap_bf16_2d(&h->tm_m_hi, h->pf_m_hi, Tm, I, 128) &&
              make_tmap_bf16_2d(&h->tm_m_lo, h->pf_m_lo, Tm, I, 128) &&
              make_attn_maps(&h->tm_attn, h->pf_q_hi, h->pf_q_lo, (int)Tm, c.n_q_heads,
                             h->pf_kvs, c.n_kv_heads, c.head_dim, c.max_ctx);
    if (!ok) QW_FAIL(h, QW_ERR_CUDA, "prefill: TMA descriptor encoding failed");
    if (h->wfmt == 1) {
      uint16_t* q = h->pf_w4;
      for (int t = 0; t < 2; ++t) {
        h->w4_qkv[t] = q;
        q += qkv_rows * H;
        h->w4_o[t] = q;
        q += H * qd;
        h->w4_gu[t] = q;
        q += 2 * I * H;
        h->w4_dw[t] = q;
        q += H * I;
        if (!make_tmap_bf16_2d(&h->tm_qkv4[t], h->w4_qkv[t], qkv_rows, H, 256) ||
            !make_tmap_bf16_2d(&h->tm_ow4[t], h->w4_o[t], H, qd, kResidBN) ||
            !make_tmap_bf16_2d(&h->tm_gu4[t], h->w4_gu[t], 2 * I, H, 256) ||
            !make_tmap_bf16_2d(&h->tm_dw4[t], h->w4_dw[t], H, I, kResidBN))
          QW_FAIL(h, QW_ERR_CUDA, "prefill: TMA descriptor encoding failed");
      }
    }
  }
  QW_CUDA(h, cudaHostAlloc((void**)&h->h_tokens, std::max<size_t>(cap, Tm) * 4, cudaHostAllocPortable));
  QW_CUDA(h, cudaHostAlloc((void**)&h->h_status, 32, cudaHostAllocPortable));
  memset(h->h_tokens, 0xff, cap * 4);
  memset(h->h_status, 0, 32);
  QW_CUDA(h, launch_rope_table(h->rope, c.max_ctx, c.head_dim, c.rope_theta, h->stream));
  QW_CUDA(h, cudaStreamSynchronize(h->stream));
  return QW_OK;
}

extern "C" uint32_t qw_abi_version(void) { return QW_ABI_VERSION; }
extern "C" size_t qw_sizeof_config(void) { return sizeof(qw_config); }
extern "C" size_t qw_sizeof_weights(void) { return sizeof(qw_weights); }
extern "C" size_t qw_sizeof_lora(void) { return sizeof(qw_lora); }

extern "C" int qw_create(const qw_config* cfg, void* cuda_stream, qw_handle** out) {
  if (!cfg || !out) QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG, "qw_create: null argument");
  if (cfg->struct_size != sizeof(qw_config) || cfg->abi_version != QW_ABI_VERSION)
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ABI,
            "qw_create: qw_config struct_size/abi_version does not match this library");
  std::string why;
  int rc = validate_config(cfg, why);
  if (rc) QW_FAIL((qw_handle*)nullptr, rc, "qw_create: " + why);
  qw_handle* h = new qw_handle();
  h->cfg = *cfg;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  if (e == cudaSuccess) e = ensure_attributes(h->device);
  if (e == cudaSuccess) {
    if (cuda_stream) {
      h->stream = (cudaStream_t)cuda_stream;
    } else {
      e = cudaStreamCreateWithFlags(&h->stream, cudaStreamNonBlocking);
      h->own_stream = true;
    }
  }
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    g_last_error = std::string("qw_create: ") + cudaGetErrorString(e);
    free_handle(h);
    return QW_ERR_CUDA;
  }
  rc = alloc_state(h);
  if (rc) {
    g_last_error = "qw_create: " + h->err;
    free_handle(h);
    return rc;
  }
  *out = h;
  return QW_OK;
}

extern "C" void qw_destroy(qw_handle* h) {
  if (!h) return;
  DeviceGuard dg(h->device);
  cudaStreamSynchronize(h->stream);
  free_handle(h);
}

extern "C" const char* qw_last_error(const qw_handle* h) {
  return h ? h->err.c_str() : g_last_error.c_str();
}

// ============================================================================ weights
extern "C" int qw_load_weights(qw_handle* h, const qw_weights* w) {
  if (!h || !w) QW_FAIL(h, QW_ERR_ARG, "qw_load_weights: null argument");
  if (w->struct_size != sizeof(qw_weights))
    QW_FAIL(h, QW_ERR_ABI, "qw_load_weights: qw_weights struct_size does not match this library");
  DeviceGuard dg(h->device);
  const qw_config& c = h->cfg;
  const int L = c.n_layers;
  const size_t H = c.hidden, I = c.intermediate, hd = c.head_dim;
  const size_t qd = (size_t)c.n_q_heads * hd, kd = (size_t)c.n_kv_heads * hd;
  if (!w->embed || !w->final_norm || !w->attn_norm || !w->q || !w->k || !w->v || !w->o ||
      !w->mlp_norm || !w->gate || !w->up || !w->down)
    QW_FAIL(h, QW_ERR_ARG, "qw_load_weights: a required tensor is NULL");
  if (c.tie_word_embeddings ? (w->lm_head != nullptr) : (w->lm_head == nullptr))
    QW_FAIL(h, QW_ERR_ARG, "qw_load_weights: lm_head must be NULL iff tie_word_embeddings");
  if (c.qk_norm && (!w->q_norm || !w->k_norm))
    QW_FAIL(h, QW_ERR_ARG, "qw_load_weights: qk_norm set but q_norm/k_norm missing");
  if (c.qkv_bias && (!w->q_bias || !w->k_bias || !w->v_bias))
    QW_FAIL(h, QW_ERR_ARG, "qw_load_weights: qkv_bias set but a bias is missing");
  const bool untied_q = h->lm_fmt != 0 && !c.tie_word_embeddings;  // lm_head passed quantised
  if (h->wfmt && (!w->q_scales || !w->k_scales || !w->v_scales || !w->o_scales ||
                  !w->gate_scales || !w->up_scales || !w->down_scales ||
                  (untied_q && !w->lm_head_scales)))
    QW_FAIL(h, QW_ERR_ARG, "qw_load_weights: int4 / Q8_0 weights need every scales tensor");
  for (int l = 0; l < L && h->wfmt; ++l)
    if (!w->q_scales[l] || !w->k_scales[l] || !w->v_scales[l] || !w->o_scales[l] ||
        !w->gate_scales[l] || !w->up_scales[l] || !w->down_scales[l])
      QW_FAIL(h, QW_ERR_ARG, "qw_load_weights: NULL scales at layer " + std::to_string(l));
  for (int l = 0; l < L; ++l) {
    if (!w->attn_norm[l] || !w->q[l] || !w->k[l] || !w->v[l] || !w->o[l] || !w->mlp_norm[l] ||
        !w->gate[l] || !w->up[l] || !w->down[l] || (c.qk_norm && (!w->q_norm[l] || !w->k_norm[l])) ||
        (c.qkv_bias && (!w->q_bias[l] || !w->k_bias[l] || !w->v_bias[l])))
      QW_FAIL(h, QW_ERR_ARG, "qw_load_weights: NULL per-layer pointer at layer " + std::to_string(l));
  }
  QW_CUDA(h, cudaStreamSynchronize(h->stream));
  if (h->exec) {
    cudaGraphExecDestroy(h->exec);
    h->exec = nullptr;
  }
  h->graph_dirty = true;
  h->weights_loaded = false;
  if (h->warena) {
    cudaFree(h->warena);
    h->warena = nullptr;
  }
  // Bytes of one packed row of K inputs: bf16, or int4 nibbles / Q8_0 bytes + scales (+ pad).
  auto fmt_rb = [](int fmt, size_t K) -> size_t {
    return fmt == 1 ? int4_row_bytes((int)K) : fmt == 2 ? q8_row_bytes((int)K) : K * 2;
  };
  auto rb = [&](size_t K) { return fmt_rb(h->wfmt, K); };
  const size_t lm_rb = fmt_rb(h->lm_fmt, H);
  // Arena layout, 256-byte aligned pieces.
  const size_t per_layer = align_up((qd + 2 * kd) * rb(H), 256) +
                           (c.qkv_bias ? align_up((qd + 2 * kd) * 2, 256) : 0) +
                           align_up(H * rb(qd), 256) + align_up(2 * I * rb(H), 256) +
                           align_up(H * rb(I), 256) + 2 * align_up(H * 2, 256) +
                           (c.qk_norm ? 2 * align_up(hd * 2, 256) : 0);
  const size_t head = align_up((size_t)c.vocab * H * 2, 256) +
                      (c.tie_word_embeddings && h->lm_fmt == 0
                           ? 0 : align_up((size_t)c.vocab * lm_rb, 256)) +
                      align_up(H * 2, 256);
  h->warena_bytes = per_layer * L + head;
  QW_CUDA(h, cudaMalloc((void**)&h->warena, h->warena_bytes));
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* p = h->warena + off;
    off += align_up(bytes, 256);
    return p;
  };
  auto cp = [&](void* dst, const void* src, size_t bytes) {
    return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, h->stream);
  };
  uint8_t* p = take((size_t)c.vocab * H * 2);
  QW_CUDA(h, cp(p, w->embed, (size_t)c.vocab * H * 2));
  h->embed = (const uint16_t*)p;
  if (c.tie_word_embeddings && h->lm_fmt == 2) {
    // Q8_0 models read the tied table through a Q8_0 copy ("SuperKittens PR #7", Q8_0
    // commit: the LM head is quantised from the embedding table); the gather keeps bf16
    p = take((size_t)c.vocab * lm_rb);
    QW_CUDA(h, launch_quantize_q8(h->embed, true, c.vocab, (int)H, (int8_t*)p, lm_rb,
                                  (uint16_t*)(p + H), lm_rb / 2, h->stream));
    h->lm_head = (const uint16_t*)p;
  } else if (c.tie_word_embeddings) {
    h->lm_head = h->embed;  // one table serves the gather and the output projection
  } else if (h->lm_fmt == 1) {
    p = take((size_t)c.vocab * lm_rb);
    QW_CUDA(h, launch_pack_int4_rows((const uint8_t*)w->lm_head, (const uint16_t*)w->lm_head_scales,
                                     c.vocab, (int)H, p, 0, 1, h->stream));
    h->lm_head = (const uint16_t*)p;
  } else if (h->lm_fmt == 2) {
    p = take((size_t)c.vocab * lm_rb);
    QW_CUDA(h, launch_pack_q8_rows((const int8_t*)w->lm_head, (const uint16_t*)w->lm_head_scales,
                                   c.vocab, (int)H, p, 0, 1, h->stream));
    h->lm_head = (const uint16_t*)p;
  } else {
    p = take((size_t)c.vocab * H * 2);
    QW_CUDA(h, cp(p, w->lm_head, (size_t)c.vocab * H * 2));
    h->lm_head = (const uint16_t*)p;
  }
  p = take(H * 2);
  QW_CUDA(h, cp(p, w->final_norm, H * 2));
  h->final_norm = (const uint16_t*)p;
  h->layers.assign(L, LayerW());
  for (int l = 0; l < L; ++l) {
    LayerW& lw = h->layers[l];
    auto pack4 = [&](const void* nib, const void* sc, size_t rows, size_t K, uint8_t* dst,
                     size_t row0, int step) {
      if (h->wfmt == 2)
        return launch_pack_q8_rows((const int8_t*)nib, (const uint16_t*)sc, (int)rows, (int)K,
                                   dst, (int)row0, step, h->stream);
      return launch_pack_int4_rows((const uint8_t*)nib, (const uint16_t*)sc, (int)rows, (int)K, dst,
                                   (int)row0, step, h->stream);
    };
    p = take((qd + 2 * kd) * rb(H));  // fused [q; k; v] rows
    if (h->wfmt) {
      QW_CUDA(h, pack4(w->q[l], w->q_scales[l], qd, H, p, 0, 1));
      QW_CUDA(h, pack4(w->k[l], w->k_scales[l], kd, H, p, qd, 1));
      QW_CUDA(h, pack4(w->v[l], w->v_scales[l], kd, H, p, qd + kd, 1));
    } else {
      QW_CUDA(h, cp(p, w->q[l], qd * H * 2));
      QW_CUDA(h, cp(p + qd * H * 2, w->k[l], kd * H * 2));
      QW_CUDA(h, cp(p + (qd + kd) * H * 2, w->v[l], kd * H * 2));
    }
    lw.qkv = (const uint16_t*)p;
    if (c.qkv_bias) {
      p = take((qd + 2 * kd) * 2);
      QW_CUDA(h, cp(p, w->q_bias[l], qd * 2));
      QW_CUDA(h, cp(p + qd * 2, w->k_bias[l], kd * 2));
      QW_CUDA(h, cp(p + (qd + kd) * 2, w->v_bias[l], kd * 2));
      lw.qkv_bias = (const uint16_t*)p;
    }
    p = take(H * rb(qd));
    if (h->wfmt) QW_CUDA(h, pack4(w->o[l], w->o_scales[l], H, qd, p, 0, 1));
    else QW_CUDA(h, cp(p, w->o[l], H * qd * 2));
    lw.o = (const uint16_t*)p;
    p = take(2 * I * rb(H));  // gate row i -> packed row 2i, up row i -> 2i+1
    if (h->wfmt) {
      QW_CUDA(h, pack4(w->gate[l], w->gate_scales[l], I, H, p, 0, 2));
      QW_CUDA(h, pack4(w->up[l], w->up_scales[l], I, H, p, 1, 2));
    } else {
      QW_CUDA(h, cudaMemcpy2DAsync(p, 2 * H * 2, w->gate[l], H * 2, H * 2, I,
                                   cudaMemcpyDeviceToDevice, h->stream));
      QW_CUDA(h, cudaMemcpy2DAsync(p + H * 2, 2 * H * 2, w->up[l], H * 2, H * 2, I,
                                   cudaMemcpyDeviceToDevice, h->stream));
    }
    lw.gateup = (const uint16_t*)p;
    p = take(H * rb(I));
    if (h->wfmt) QW_CUDA(h, pack4(w->down[l], w->down_scales[l], H, I, p, 0, 1));
    else QW_CUDA(h, cp(p, w->down[l], H * I * 2));
    lw.down = (const uint16_t*)p;
    p = take(H * 2);
    QW_CUDA(h, cp(p, w->attn_norm[l], H * 2));
    lw.attn_norm = (const uint16_t*)p;
    p = take(H * 2);
    QW_CUDA(h, cp(p, w->mlp_norm[l], H * 2));
    lw.mlp_norm = (const uint16_t*)p;
    if (c.qk_norm) {
      p = take(hd * 2);
      QW_CUDA(h, cp(p, w->q_norm[l], hd * 2));
      lw.q_norm = (const uint16_t*)p;
      p = take(hd * 2);
      QW_CUDA(h, cp(p, w->k_norm[l], hd * 2));
      lw.k_norm = (const uint16_t*)p;
    }
  }
  {
    std::vector<LayerDev> ld(L);
    for (int l = 0; l < L; ++l) {
      const LayerW& lw = h->layers[l];
      ld[l] = LayerDev{(const uint8_t*)lw.qkv, lw.qkv_bias, (const uint8_t*)lw.o,
                       (const uint8_t*)lw.gateup, (const uint8_t*)lw.down, lw.attn_norm,
                       lw.mlp_norm, lw.q_norm, lw.k_norm};
    }
    if (h->d_layers) cudaFree(h->d_layers);
    h->d_layers = nullptr;
    QW_CUDA(h, cudaMalloc((void**)&h->d_layers, L * sizeof(LayerDev)));
    QW_CUDA(h, cudaMemcpyAsync(h->d_layers, ld.data(), L * sizeof(LayerDev),
                               cudaMemcpyHostToDevice, h->stream));
  }
  if (c.max_prefill_t > 0 && h->wfmt == 0) {
    h->tm_qkv.resize(L);
    h->tm_ow.resize(L);
    h->tm_gu.resize(L);
    h->tm_dw.resize(L);
    for (int l = 0; l < L; ++l) {
      const LayerW& lw = h->layers[l];
      const bool ok = make_tmap_bf16_2d(&h->tm_qkv[l], lw.qkv, qd + 2 * kd, H, 256) &&
                      make_tmap_bf16_2d(&h->tm_ow[l], lw.o, H, qd, kResidBN) &&
                      make_tmap_bf16_2d(&h->tm_gu[l], lw.gateup, 2 * I, H, 256) &&
                      make_tmap_bf16_2d(&h->tm_dw[l], lw.down, H, I, kResidBN);
      if (!ok) QW_FAIL(h, QW_ERR_CUDA, "qw_load_weights: TMA descriptor encoding failed");
    }
  }
  QW_CUDA(h, cudaMemsetAsync(h->d_pos, 0, 4, h->stream));
  QW_CUDA(h, cudaStreamSynchronize(h->stream));
  h->pos = 0;
  h->have_prev = false;
  h->cap_valid = false;
  h->weights_loaded = true;
  return QW_OK;
}

// ============================================================================ the step graph
static constexpr uint32_t kSingleStageMax = 112 * 1024;  // whole CTA slice in one stage
static constexpr uint32_t kStreamStage = 32 * 1024;      // else: 4 stages of 32 KB
static constexpr int kStreamStages = 4;

static void plan(GemvArgs& a, int grid) {
  const uint64_t units_max = ((uint64_t)a.n_units + grid - 1) / grid;
  if (units_max * a.rpu * a.row_bytes <= kSingleStageMax)
    plan_gemv(a, grid, kSingleStageMax, 1);
  else
    plan_gemv(a, grid, kStreamStage, kStreamStages);
}

static GemvArgs base_gemv(qw_handle* h, const void* w, int n_units, int rpu, int K,
                          int wfmt) {
  GemvArgs a{};
  a.w = (const uint8_t*)w;
  a.n_units = n_units;
  a.rpu = rpu;
  a.K = K;
  a.wfmt = wfmt;
  a.row_bytes = wfmt == 1 ? int4_row_bytes(K) : wfmt == 2 ? q8_row_bytes(K) : (uint32_t)K * 2;
  a.scale_off = wfmt == 2 ? (uint32_t)K : (uint32_t)K / 2;
  a.eps = h->cfg.eps;
  a.err = h->d_err;
  a.wait_ns = h->wait_ns;
  a.pos = h->d_pos;
  return a;
}

// Final RMSNorm of row x, logits over the (tied or untied) head, greedy argmax;
// the last CTA records the id at the device position and advances it.
static cudaError_t launch_lm_head(qw_handle* h, const float* x, float* norm_out, bool pdl,
                                  cudaStream_t s) {
  GemvArgs a = base_gemv(h, h->lm_head, h->cfg.vocab, 1, h->cfg.hidden, h->lm_fmt);
  a.x = x;
  a.norm_g = h->final_norm;
  a.y = h->logits;
  a.norm_out = norm_out;
  a.am.blk_val = h->blk_val;
  a.am.blk_idx = h->blk_idx;
  a.am.counter = h->am_counter;
  a.am.argmax = h->d_argmax;
  a.am.next_token = h->d_next_token;
  a.am.pos = h->d_pos;
  a.am.tokens_by_pos = h->d_tokens_by_pos;
  a.am.status = h->d_status;
  plan_gemv(a, h->lm_grid, kStreamStage, kStreamStages);
  return launch_gemv(EPI_LOGITS, a, h->lm_grid, pdl, s);
}

// The persistent kernel's arguments (the token is patched per replay).
static MegaArgs mega_args(qw_handle* h) {
  const qw_config& c = h->cfg;
  MegaArgs m{};
  m.L = c.n_layers;
  m.H = c.hidden;
  m.nq = c.n_q_heads;
  m.nkv = c.n_kv_heads;
  m.hd = c.head_dim;
  m.I = c.intermediate;
  m.V = c.vocab;
  m.eps = c.eps;
  m.embed = h->embed;
  m.lm_head = (const uint8_t*)h->lm_head;
  m.final_norm = h->final_norm;
  m.layers = h->d_layers;
  m.k_cache = h->k_cache;
  m.v_cache = h->v_cache;
  m.kv_bf16 = h->kv_bf16 ? 1 : 0;
  m.wfmt = h->wfmt;
  m.cap = c.max_ctx;
  m.rope = h->rope;
  m.x = h->mx;
  m.qkv = h->mqkv;
  m.attn_o = h->mattn;
  m.mlp = h->mmlp;
  m.epoch = h->d_epoch;
  m.logits = h->logits;
  m.mpart = h->mpart;
  m.splits = h->nsplit_max;
  m.am.blk_val = h->blk_val;
  m.am.blk_idx = h->blk_idx;
  m.am.counter = h->am_counter;
  m.am.argmax = h->d_argmax;
  m.am.next_token = h->d_next_token;
  m.am.pos = h->d_pos;
  m.am.tokens_by_pos = h->d_tokens_by_pos;
  m.am.status = h->d_status;
  m.pos = h->d_pos;
  m.tok = -1;
  m.next_token = h->d_next_token;
  m.cap_emb = h->capture_on ? h->cap_emb : nullptr;
  m.cap_blk0 = h->capture_on ? h->cap_blk0 : nullptr;
  m.cap_final = h->capture_on ? h->cap_final : nullptr;
  m.lora = h->lora_active ? h->d_lora : nullptr;
  m.lora_r = h->lora_active ? h->lora_rank : 0;
  m.lora_scale = h->lora_scale;
  m.err = h->d_err;
  m.wait_ns = h->wait_ns;
  return m;
}

// Launch one step's kernels on stream s (recorded into the graph).
static cudaError_t record_step(qw_handle* h, cudaStream_t s) {
  if (h->use_mega)
    // the wide-input build for its shapes and for every handle with an adapter (the LoRA
    // step is compiled into that build only)
    return (h->mega_big || h->lora_active ? mega_big::launch_mega
            : h->mega_wide                ? mega_wide::launch_mega
                                          : mega::launch_mega)(mega_args(h),
                                                               h->nsplit_max * h->cfg.n_kv_heads, s);
  const qw_config& c = h->cfg;
  const int H = c.hidden, I = c.intermediate, hd = c.head_dim;
  const int qd = c.n_q_heads * hd, kd = c.n_kv_heads * hd;
  const int qkv_rows = qd + 2 * kd;
  const size_t kv_layer = (size_t)c.n_kv_heads * c.max_ctx * hd;
  cudaError_t e;

  EmbedArgs ea{};
  ea.table = h->embed;
  ea.V = c.vocab;
  ea.H = H;
  ea.pos = h->d_pos;
  ea.tok = -1;
  ea.next_token = h->d_next_token;
  ea.x = h->x;
  ea.cap_out = h->capture_on ? h->cap_emb : nullptr;
  ea.err = h->d_err;
  if ((e = launch_embed(ea, s)) != cudaSuccess) return e;

  for (int l = 0; l < c.n_layers; ++l) {
    const LayerW& lw = h->layers[l];
    if (h->lora_active) {  // t = A_q . RMSNorm(x) and A_v . RMSNorm(x), rank entries each
      for (int j = 0; j < 2; ++j) {
        GemvArgs a = base_gemv(h, j == 0 ? h->lora_qa[l] : h->lora_va[l], h->lora_rank, 1, H,
                               false);
        a.x = h->x;
        a.norm_g = lw.attn_norm;
        a.y = h->lora_t + j * h->lora_rank;
        const int grid = h->lora_rank;
        plan(a, grid);
        if ((e = launch_gemv(EPI_STORE, a, grid, true, s)) != cudaSuccess) return e;
      }
    }
    {  // fused QKV projection with the input RMSNorm in its prologue
      GemvArgs a = base_gemv(h, lw.qkv, qkv_rows, 1, H, h->wfmt);
      a.x = h->x;
      a.norm_g = lw.attn_norm;
      a.bias = lw.qkv_bias;
      a.y = h->qkv;
      if (h->lora_active) {
        a.lora_bq = h->lora_qb[l];
        a.lora_bv = h->lora_vb[l];
        a.lora_t = h->lora_t;
        a.lora_r = h->lora_rank;
        a.lora_q_rows = qd;
        a.lora_v_row0 = qd + kd;
        a.lora_v_rows = kd;
        a.lora_scale = h->lora_scale;
      }
      const int grid = std::min(qkv_rows, h->num_sms);
      plan(a, grid);
      if ((e = launch_gemv(EPI_STORE, a, grid, true, s)) != cudaSuccess) return e;
    }
    {  // QK-norm, RoPE, KV append, split-K flash decode, combine
      AttnArgs t{};
      t.qkv = h->qkv;
      t.q_norm = lw.q_norm;
      t.k_norm = lw.k_norm;
      t.rope = h->rope;
      t.rope_theta = c.rope_theta;
      t.k_cache = h->k_cache + (size_t)l * kv_layer * h->kv_elem;
      t.v_cache = h->v_cache + (size_t)l * kv_layer * h->kv_elem;
      t.kv_bf16 = h->kv_bf16 ? 1 : 0;
      t.cap = c.max_ctx;
      t.pos_ptr = h->d_pos;
      t.nq = c.n_q_heads;
      t.nkv = c.n_kv_heads;
      t.eps = c.eps;
      t.nsplit_max = h->nsplit_max;
      t.min_keys = kAttnMinKeys;
      t.part_o = h->part_o;
      t.part_ml = h->part_ml;
      t.counters = h->attn_counters;
      t.out = h->attn_o;
      t.err = h->d_err;
      t.wait_ns = h->wait_ns;
      if ((e = launch_attention(t, hd, true, s)) != cudaSuccess) return e;
    }
    {  // o_proj + residual
      GemvArgs a = base_gemv(h, lw.o, H, 1, qd, h->wfmt);
      a.x = h->attn_o;
      a.y = h->x;
      const int grid = std::min(H, h->num_sms);
      plan(a, grid);
      if ((e = launch_gemv(EPI_RESIDUAL, a, grid, true, s)) != cudaSuccess) return e;
    }
    {  // gate/up with the post-attention RMSNorm in its prologue, SwiGLU epilogue
      GemvArgs a = base_gemv(h, lw.gateup, I, 2, H, h->wfmt);
      a.x = h->x;
      a.norm_g = lw.mlp_norm;
      a.y = h->mlp;
      const int grid = std::min(I, h->num_sms);
      plan(a, grid);
      if ((e = launch_gemv(EPI_SWIGLU, a, grid, true, s)) != cudaSuccess) return e;
    }
    {  // down + residual (block-0 checkpoint taken here)
      GemvArgs a = base_gemv(h, lw.down, H, 1, I, h->wfmt);
      a.x = h->mlp;
      a.y = h->x;
      a.cap_out = (h->capture_on && l == 0) ? h->cap_blk0 : nullptr;
      const int grid = std::min(H, h->num_sms);
      plan(a, grid);
      if ((e = launch_gemv(EPI_RESIDUAL, a, grid, true, s)) != cudaSuccess) return e;
    }
  }
  // final RMSNorm + LM head + greedy argmax; advances the device position
  return launch_lm_head(h, h->x, h->capture_on ? h->cap_final : nullptr, true, s);
}

static int ensure_graph_once(qw_handle* h);

// Record (or re-record) the step graph; a persistent kernel that cannot be
// recorded or instantiated (e.g. no cooperative launch) falls back to the
// multi-kernel graph for the rest of the handle's life. The switch is not silent:
// the handle's last-error text carries a note (the call itself succeeds), one
// line goes to stderr, and qw_get_decode_path reports 1 from then on.
static int ensure_graph(qw_handle* h) {
  const int rc = ensure_graph_once(h);
  if (rc == QW_OK || !h->use_mega) return rc;
  const std::string why = h->err;
  h->use_mega = false;
  h->mega_ok = false;
  h->graph_dirty = true;
  const int rc2 = ensure_graph_once(h);
  if (rc2 == QW_OK) {
    h->err = "note: the persistent decode kernel could not be recorded (" + why +
             "); this handle runs the multi-kernel decode graph from now on";
    fprintf(stderr, "qw: %s\n", h->err.c_str());
  }
  return rc2;
}

static int ensure_graph_once(qw_handle* h) {
  if (h->exec && !h->graph_dirty) return QW_OK;
  if (h->exec) {
    // replays of the old graph may still be queued (a greedy run crossing the
    // switch between kernel builds): let them finish before it goes
    QW_CUDA(h, cudaStreamSynchronize(h->stream));
    cudaGraphExecDestroy(h->exec);
    h->exec = nullptr;
  }
  if (h->graph) {
    cudaGraphDestroy(h->graph);
    h->graph = nullptr;
  }
  QW_CUDA(h, cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal));
  const cudaError_t le = record_step(h, h->cap_stream);
  cudaGraph_t graph = nullptr;
  const cudaError_t ce = cudaStreamEndCapture(h->cap_stream, &graph);
  if (le != cudaSuccess || ce != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();
    QW_FAIL(h, QW_ERR_CUDA,
            std::string("recording the decode step: ") +
                cudaGetErrorString(le != cudaSuccess ? le : ce));
  }
  h->graph = graph;
  // Find the embed node: its token argument is rewritten before every replay.
  size_t n_nodes = 0;
  QW_CUDA(h, cudaGraphGetNodes(graph, nullptr, &n_nodes));
  std::vector<cudaGraphNode_t> nodes(n_nodes);
  QW_CUDA(h, cudaGraphGetNodes(graph, nodes.data(), &n_nodes));
  h->tok_node = nullptr;
  for (cudaGraphNode_t nd : nodes) {
    cudaGraphNodeType t;
    QW_CUDA(h, cudaGraphNodeGetType(nd, &t));
    if (t != cudaGraphNodeTypeKernel) continue;
    cudaKernelNodeParams kp{};
    QW_CUDA(h, cudaGraphKernelNodeGetParams(nd, &kp));
    size_t bytes = 0, off = 0;
    if (kp.func == embed_kernel_fn()) {
      bytes = sizeof(EmbedArgs);
      off = offsetof(EmbedArgs, tok);
    } else if (mega::is_mega_kernel(kp.func) || mega_wide::is_mega_kernel(kp.func) ||
               mega_big::is_mega_kernel(kp.func)) {
      bytes = sizeof(MegaArgs);
      off = offsetof(MegaArgs, tok);
    } else {
      continue;
    }
    h->tok_node = nd;
    h->tok_params = kp;
    h->tok_args.assign((const uint8_t*)kp.kernelParams[0], (const uint8_t*)kp.kernelParams[0] + bytes);
    h->tok_offset = off;
  }
  if (!h->tok_node) QW_FAIL(h, QW_ERR_CUDA, "recording the decode step: token node not found");
  const cudaError_t ie = cudaGraphInstantiate(&h->exec, graph, 0);
  if (ie != cudaSuccess) {
    h->exec = nullptr;
    QW_FAIL(h, QW_ERR_CUDA, std::string("cudaGraphInstantiate: ") + cudaGetErrorString(ie));
  }
  h->graph_dirty = false;
  return QW_OK;
}

// Synchronise, then turn the device error word into a status (and clear it).
static int finish_sync(qw_handle* h) {
  QW_CUDA(h, cudaMemcpyAsync(h->h_status, h->d_status, 8, cudaMemcpyDeviceToHost, h->stream));
  QW_CUDA(h, cudaMemcpyAsync(h->h_status + 3, h->d_err, 4, cudaMemcpyDeviceToHost, h->stream));
  QW_CUDA(h, cudaStreamSynchronize(h->stream));
  const int err = ((volatile int*)h->h_status)[1] | ((volatile int*)h->h_status)[3];
  if (err == 0) return QW_OK;
  QW_CUDA(h, cudaMemsetAsync(h->d_status, 0, 8, h->stream));
  QW_CUDA(h, cudaMemsetAsync(h->d_err, 0, 4, h->stream));
  QW_CUDA(h, cudaMemsetAsync(h->attn_counters, 0,
                             (size_t)h->cfg.n_layers * h->cfg.n_kv_heads * 4, h->stream));
  QW_CUDA(h, cudaMemsetAsync(h->am_counter, 0, 4, h->stream));
  if (h->pf_gemm_flags)
    QW_CUDA(h, cudaMemsetAsync(h->pf_gemm_flags, 0,
                               ((size_t)(h->cfg.max_prefill_t + 127) / 128) *
                                   ((h->cfg.hidden + 127) / 128) * 4,
                               h->stream));
  QW_CUDA(h, cudaStreamSynchronize(h->stream));
  if (err & ERR_TIMEOUT)
    QW_FAIL(h, QW_ERR_DEVICE_TIMEOUT, "a bounded device-side wait gave up; outputs are invalid");
  if (err & ERR_TOKEN)
    QW_FAIL(h, QW_ERR_ARG, "the device saw a token outside [0, vocab); token 0 was used");
  QW_FAIL(h, QW_ERR_NUMERIC, "a logit was NaN; there is no greedy token");
}

static int check_ready(qw_handle* h, const char* fn) {
  if (!h) QW_FAIL(h, QW_ERR_ARG, std::string(fn) + ": null handle");
  if (!h->weights_loaded) QW_FAIL(h, QW_ERR_STATE, std::string(fn) + ": weights not loaded");
  return QW_OK;
}

// Queue n graph replays; step i is fed tokens[i] (or, when tokens is null, `first`
// for the first step and the device argmax afterwards). The token is the embed
// node's kernel argument, so no copy is queued per step.
// Each step runs the persistent kernel build that suits its position: 7 consumer
// warps below kMegaWideFrom keys, 11 from there on (the graph is re-recorded when
// the choice changes, which happens at most once per pass through the context).
static constexpr int kMegaWideFrom = 1536;

static int run_steps(qw_handle* h, int n, const int32_t* tokens, int first) {
  int last = -2;
  for (int i = 0; i < n; ++i) {
    const bool wide = h->use_mega && !h->mega_big && !h->lora_active && h->pos + i >= kMegaWideFrom;
    if (wide != h->mega_wide) {
      h->mega_wide = wide;
      h->graph_dirty = true;
    }
    if (!h->exec || h->graph_dirty) {
      const int rc = ensure_graph(h);
      if (rc) return rc;
      last = -2;  // a new graph: its token node gets the token again
    }
    const int tok = tokens ? tokens[i] : (i == 0 ? first : -1);
    if (tok != last) {
      std::vector<uint8_t>& buf = h->tok_args;
      const int v = tok < 0 ? -1 : tok;
      memcpy(buf.data() + h->tok_offset, &v, sizeof(int));
      void* args[1] = {buf.data()};
      cudaKernelNodeParams kp = h->tok_params;
      kp.kernelParams = args;
      kp.extra = nullptr;
      QW_CUDA(h, cudaGraphExecKernelNodeSetParams(h->exec, h->tok_node, &kp));
      last = tok;
    }
    QW_CUDA(h, cudaGraphLaunch(h->exec, h->stream));
  }
  return QW_OK;
}

// ============================================================================ stepping
extern "C" int qw_decode_step(qw_handle* h, int32_t token, float* logits_dev, int32_t* argmax_host) {
  int rc = check_ready(h, "qw_decode_step");
  if (rc) return rc;
  if (token >= h->cfg.vocab) QW_FAIL(h, QW_ERR_ARG, "qw_decode_step: token >= vocab");
  if (token < 0 && !h->have_prev)
    QW_FAIL(h, QW_ERR_STATE, "qw_decode_step: token < 0 but no previous step to feed from");
  if (h->pos + 1 > h->cfg.max_ctx) QW_FAIL(h, QW_ERR_CTX, "qw_decode_step: context is full");
  DeviceGuard dg(h->device);
  rc = run_steps(h, 1, nullptr, token);
  if (rc) return rc;
  if (logits_dev)
    QW_CUDA(h, cudaMemcpyAsync(logits_dev, h->logits, (size_t)h->cfg.vocab * 4,
                               cudaMemcpyDeviceToDevice, h->stream));
  h->cap_valid = h->capture_on;
  h->cap_row0 = h->pos;
  h->cap_rows = 1;
  h->pos += 1;
  h->have_prev = true;
  if (argmax_host) {
    rc = finish_sync(h);
    if (rc) return rc;
    *argmax_host = ((volatile int*)h->h_status)[0];
  }
  return QW_OK;
}

extern "C" int qw_decode_greedy(qw_handle* h, int32_t token, int32_t n_steps, int32_t* ids_host) {
  int rc = check_ready(h, "qw_decode_greedy");
  if (rc) return rc;
  if (n_steps <= 0) QW_FAIL(h, QW_ERR_ARG, "qw_decode_greedy: n_steps must be positive");
  if (token >= h->cfg.vocab) QW_FAIL(h, QW_ERR_ARG, "qw_decode_greedy: token >= vocab");
  if (token < 0 && !h->have_prev)
    QW_FAIL(h, QW_ERR_STATE, "qw_decode_greedy: token < 0 but no previous step to feed from");
  if ((int64_t)h->pos + n_steps > h->cfg.max_ctx)
    QW_FAIL(h, QW_ERR_CTX, "qw_decode_greedy: pos + n_steps > max_ctx");
  DeviceGuard dg(h->device);
  const int p0 = h->pos;
  rc = run_steps(h, n_steps, nullptr, token);
  if (rc) return rc;
  h->cap_valid = h->capture_on;
  h->cap_row0 = p0 + n_steps - 1;
  h->cap_rows = 1;
  h->pos += n_steps;
  h->have_prev = true;
  if (ids_host)
    QW_CUDA(h, cudaMemcpyAsync(h->h_tokens + p0, h->d_tokens_by_pos + p0, (size_t)n_steps * 4,
                               cudaMemcpyDeviceToHost, h->stream));
  rc = finish_sync(h);
  if (rc) return rc;
  if (ids_host)
    for (int i = 0; i < n_steps; ++i) ids_host[i] = h->h_tokens[p0 + i];
  return QW_OK;
}

// One causal pass over T prompt rows: tensor-core GEMMs for the projections,
// row kernels for norms / QK-norm / RoPE / KV append, flash attention over the
// cache (positions 0..pos+T-1), then the LM head on the last row.
static int prefill_batched(qw_handle* h, const int32_t* ids_host, int T) {
  const qw_config& c = h->cfg;
  const int H = c.hidden, I = c.intermediate, hd = c.head_dim;
  const int qd = c.n_q_heads * hd, kd = c.n_kv_heads * hd, qkv_rows = qd + 2 * kd;
  const size_t kv_layer = (size_t)c.n_kv_heads * c.max_ctx * hd;
  const int p0 = h->pos;
  cudaStream_t s = h->stream;
  QW_CUDA(h, cudaStreamSynchronize(s));  // the staging buffer may still feed an earlier copy
  memcpy(h->h_tokens, ids_host, (size_t)T * 4);
  QW_CUDA(h, cudaMemcpyAsync(h->pf_ids, h->h_tokens, (size_t)T * 4, cudaMemcpyHostToDevice, s));
  QW_CUDA(h, launch_embed_rows(h->pf_ids, T, h->embed, c.vocab, H, h->pf_x,
                               h->capture_on ? h->cap_emb : nullptr, p0, h->d_err, s));
  const bool w4 = h->wfmt == 1;
  auto gemm = [&](int bn, int epi, const CUtensorMap& ahi, const CUtensorMap& alo,
                  const CUtensorMap& b, const CUtensorMap* b_lo, int N, int K, float* out,
                  const uint16_t* bias, uint16_t* ohi, uint16_t* olo, float* cap) {
    GemmArgs g{};
    g.M = T;
    g.N = N;
    g.K = K;
    g.a_split = 2;
    g.out = out;
    g.ldo = N;
    g.bias = bias;
    g.out_hi = ohi;
    g.out_lo = olo;
    g.ldb = N / 2;
    g.cap_out = cap;
    g.cap_row0 = p0;
    if (epi == GEPI_RESID) {  // narrow outputs (N = hidden): K split in two, fixed order
      g.ksplit = kResidSplit;
      g.flags = h->pf_gemm_flags;
    }
    g.err = h->d_err;
    g.wait_ns = h->wait_ns;
    return launch_gemm(bn, epi, ahi, alo, b, b_lo, g, s);
  };
  for (int l = 0; l < c.n_layers; ++l) {
    const LayerW& lw = h->layers[l];
    uint8_t* kc = h->k_cache + (size_t)l * kv_layer * h->kv_elem;
    uint8_t* vc = h->v_cache + (size_t)l * kv_layer * h->kv_elem;
    if (w4) {  // this layer's int4 rows as exact two-bf16 planes
      QW_CUDA(h, launch_dequant_int4_split((const uint8_t*)lw.qkv, qkv_rows, H, h->w4_qkv[0],
                                           h->w4_qkv[1], s));
      QW_CUDA(h, launch_dequant_int4_split((const uint8_t*)lw.o, H, qd, h->w4_o[0], h->w4_o[1], s));
      QW_CUDA(h, launch_dequant_int4_split((const uint8_t*)lw.gateup, 2 * I, H, h->w4_gu[0],
                                           h->w4_gu[1], s));
      QW_CUDA(h, launch_dequant_int4_split((const uint8_t*)lw.down, H, I, h->w4_dw[0],
                                           h->w4_dw[1], s));
    }
    const CUtensorMap& wq = w4 ? h->tm_qkv4[0] : h->tm_qkv[l];
    const CUtensorMap& wo = w4 ? h->tm_ow4[0] : h->tm_ow[l];
    const CUtensorMap& wg = w4 ? h->tm_gu4[0] : h->tm_gu[l];
    const CUtensorMap& wd = w4 ? h->tm_dw4[0] : h->tm_dw[l];
    QW_CUDA(h, launch_rmsnorm_rows(h->pf_x, T, H, lw.attn_norm, c.eps, h->pf_xn_hi, h->pf_xn_lo,
                                   nullptr, 0, s));
    QW_CUDA(h, gemm(256, GEPI_STORE, h->tm_xn_hi, h->tm_xn_lo, wq, w4 ? &h->tm_qkv4[1] : nullptr,
                    qkv_rows, H, h->pf_qkv, lw.qkv_bias, nullptr, nullptr, nullptr));
    QW_CUDA(h, launch_qk_rope_kv_rows(h->pf_qkv, T, p0, c.n_q_heads, c.n_kv_heads, hd, lw.q_norm,
                                      lw.k_norm, c.eps, h->rope, h->pf_q_hi, h->pf_q_lo, kc, vc,
                                      h->kv_bf16, c.max_ctx, h->pf_kvs, s));
    QW_CUDA(h, launch_attn_prefill(h->tm_attn, kc, vc, h->kv_bf16, h->pf_kvs, h->pf_attn_part,
                                   c.max_prefill_t, c.max_ctx, p0, T, c.n_q_heads,
                                   c.n_kv_heads, hd, h->pf_o_hi, h->pf_o_lo, h->d_err, h->wait_ns,
                                   s));
    QW_CUDA(h, gemm(kResidBN, GEPI_RESID, h->tm_o_hi, h->tm_o_lo, wo, w4 ? &h->tm_ow4[1] : nullptr, H,
                    qd, h->pf_x, nullptr, nullptr, nullptr, nullptr));
    QW_CUDA(h, launch_rmsnorm_rows(h->pf_x, T, H, lw.mlp_norm, c.eps, h->pf_xn_hi, h->pf_xn_lo,
                                   nullptr, 0, s));
    QW_CUDA(h, gemm(256, GEPI_SWIGLU, h->tm_xn_hi, h->tm_xn_lo, wg, w4 ? &h->tm_gu4[1] : nullptr,
                    2 * I, H, nullptr, nullptr, h->pf_m_hi, h->pf_m_lo, nullptr));
    QW_CUDA(h, gemm(kResidBN, GEPI_RESID, h->tm_m_hi, h->tm_m_lo, wd, w4 ? &h->tm_dw4[1] : nullptr, H, I,
                    h->pf_x, nullptr,
                    nullptr, nullptr, (h->capture_on && l == 0) ? h->cap_blk0 : nullptr));
  }
  if (h->capture_on)
    QW_CUDA(h, launch_rmsnorm_rows(h->pf_x, T, H, h->final_norm, c.eps, nullptr, nullptr,
                                   h->cap_final, p0, s));
  // The LM head's last CTA records the id at the device position and advances
  // it, so set it to the last prompt row first.
  QW_CUDA(h, launch_set_int(h->d_pos, p0 + T - 1, s));
  QW_CUDA(h, launch_lm_head(h, h->pf_x + (size_t)(T - 1) * H, nullptr, false, s));
  return QW_OK;
}

extern "C" int qw_prefill(qw_handle* h, const int32_t* ids_host, int32_t T, float* logits_dev,
                          int32_t* argmax_host) {
  int rc = check_ready(h, "qw_prefill");
  if (rc) return rc;
  if (!ids_host || T <= 0) QW_FAIL(h, QW_ERR_ARG, "qw_prefill: empty prompt");
  for (int i = 0; i < T; ++i)
    if (ids_host[i] < 0 || ids_host[i] >= h->cfg.vocab)
      QW_FAIL(h, QW_ERR_ARG, "qw_prefill: id " + std::to_string(i) + " outside [0, vocab)");
  if ((int64_t)h->pos + T > h->cfg.max_ctx)
    QW_FAIL(h, QW_ERR_CTX, "qw_prefill: pos + T > max_ctx");
  DeviceGuard dg(h->device);
  const int p0 = h->pos;
  if (T <= h->cfg.max_prefill_t && !h->lora_active && h->wfmt != 2) {
    rc = prefill_batched(h, ids_host, T);
  } else {
    // Sequential path ("Emberglass" README, maxPrefillT: longer prompts, or a
    // prompt while a LoRA is set): one decode step per id, queued before one sync.
    rc = run_steps(h, T, ids_host, 0);
  }
  if (rc) return rc;
  if (logits_dev)
    QW_CUDA(h, cudaMemcpyAsync(logits_dev, h->logits, (size_t)h->cfg.vocab * 4,
                               cudaMemcpyDeviceToDevice, h->stream));
  h->cap_valid = h->capture_on;
  h->cap_row0 = p0;
  h->cap_rows = T;
  h->pos += T;
  h->have_prev = true;
  if (argmax_host) {
    rc = finish_sync(h);
    if (rc) return rc;
    *argmax_host = ((volatile int*)h->h_status)[0];
  }
  return QW_OK;
}

extern "C" int qw_reset(qw_handle* h) {
  if (!h) QW_FAIL(h, QW_ERR_ARG, "qw_reset: null handle");
  DeviceGuard dg(h->device);
  QW_CUDA(h, cudaStreamSynchronize(h->stream));
  QW_CUDA(h, cudaMemsetAsync(h->d_pos, 0, 4, h->stream));
  QW_CUDA(h, cudaStreamSynchronize(h->stream));
  h->pos = 0;
  h->have_prev = false;
  h->cap_valid = false;
  return QW_OK;
}

extern "C" int qw_set_pos(qw_handle* h, int32_t pos) {
  if (!h) QW_FAIL(h, QW_ERR_ARG, "qw_set_pos: null handle");
  if (pos < 0 || pos > h->cfg.max_ctx) QW_FAIL(h, QW_ERR_CTX, "qw_set_pos: pos outside [0, max_ctx]");
  DeviceGuard dg(h->device);
  QW_CUDA(h, cudaStreamSynchronize(h->stream));
  h->h_status[2] = pos;  // staging value for the copy below
  QW_CUDA(h, cudaMemcpyAsync(h->d_pos, &h->h_status[2], 4, cudaMemcpyHostToDevice, h->stream));
  QW_CUDA(h, cudaStreamSynchronize(h->stream));
  h->pos = pos;
  h->cap_valid = false;
  return QW_OK;
}

extern "C" int qw_get_pos(const qw_handle* h, int32_t* pos) {
  if (!h || !pos) return QW_ERR_ARG;
  *pos = h->pos;
  return QW_OK;
}

extern "C" int qw_kv_cache(qw_handle* h, int32_t layer, void** k_dev, void** v_dev) {
  if (!h || !k_dev || !v_dev) QW_FAIL(h, QW_ERR_ARG, "qw_kv_cache: null argument");
  if (layer < 0 || layer >= h->cfg.n_layers) QW_FAIL(h, QW_ERR_ARG, "qw_kv_cache: bad layer");
  const size_t kv_layer = (size_t)h->cfg.n_kv_heads * h->cfg.max_ctx * h->cfg.head_dim;
  *k_dev = h->k_cache + (size_t)layer * kv_layer * h->kv_elem;
  *v_dev = h->v_cache + (size_t)layer * kv_layer * h->kv_elem;
  return QW_OK;
}

extern "C" int qw_set_lora(qw_handle* h, const qw_lora* lora) {
  if (!h) QW_FAIL(h, QW_ERR_ARG, "qw_set_lora: null handle");
  if (lora == nullptr) {  // clear: the next step's graph has no LoRA work at all
    if (h->lora_active) h->graph_dirty = true;
    h->lora_active = false;
    h->lora_qa.clear();
    h->lora_qb.clear();
    h->lora_va.clear();
    h->lora_vb.clear();
    const bool mega = h->path_pref == 0 && h->mega_ok;
    if (mega != h->use_mega) h->graph_dirty = true;
    h->use_mega = mega;
    return QW_OK;
  }
  if (lora->struct_size != sizeof(qw_lora)) QW_FAIL(h, QW_ERR_ABI, "qw_set_lora: struct_size mismatch");
  if (lora->rank < 1 || lora->rank > 64) QW_FAIL(h, QW_ERR_ARG, "qw_set_lora: rank must be 1..64");
  const int L = h->cfg.n_layers;
  if (!lora->q_a || !lora->q_b || !lora->v_a || !lora->v_b)
    QW_FAIL(h, QW_ERR_ARG, "qw_set_lora: a per-layer array is NULL");
  for (int l = 0; l < L; ++l) {
    const void* ptrs[4] = {lora->q_a[l], lora->q_b[l], lora->v_a[l], lora->v_b[l]};
    for (const void* p : ptrs)
      if (!p || (reinterpret_cast<uintptr_t>(p) & 15))
        QW_FAIL(h, QW_ERR_ARG, "qw_set_lora: NULL or unaligned (16 B) tensor at layer " +
                                   std::to_string(l));
  }
  h->lora_qa.assign(L, nullptr);
  h->lora_qb.assign(L, nullptr);
  h->lora_va.assign(L, nullptr);
  h->lora_vb.assign(L, nullptr);
  for (int l = 0; l < L; ++l) {
    h->lora_qa[l] = (const uint16_t*)lora->q_a[l];
    h->lora_qb[l] = (const uint16_t*)lora->q_b[l];
    h->lora_va[l] = (const uint16_t*)lora->v_a[l];
    h->lora_vb[l] = (const uint16_t*)lora->v_b[l];
  }
  h->lora_rank = lora->rank;
  h->lora_scale = lora->alpha / (float)lora->rank;
  h->lora_active = true;
  h->lora_tab.resize((size_t)L * 4);
  for (int l = 0; l < L; ++l) {
    h->lora_tab[4 * l + 0] = h->lora_qa[l];
    h->lora_tab[4 * l + 1] = h->lora_qb[l];
    h->lora_tab[4 * l + 2] = h->lora_va[l];
    h->lora_tab[4 * l + 3] = h->lora_vb[l];
  }
  {
    DeviceGuard dg(h->device);
    QW_CUDA(h, cudaMemcpyAsync(h->d_lora, h->lora_tab.data(), h->lora_tab.size() * sizeof(void*),
                               cudaMemcpyHostToDevice, h->stream));
    QW_CUDA(h, cudaStreamSynchronize(h->stream));
  }
  // the persistent kernel runs the adapter when a CTA's q/k/v rows fit its update;
  // otherwise the multi-kernel graph does
  h->use_mega = h->path_pref == 0 && h->mega_ok && h->mega_lora_ok;
  h->graph_dirty = true;
  return QW_OK;
}

extern "C" int qw_set_wait_limit_ns(qw_handle* h, uint64_t ns) {
  if (!h) QW_FAIL(h, QW_ERR_ARG, "qw_set_wait_limit_ns: null handle");
  h->wait_ns = ns;
  h->graph_dirty = true;
  return QW_OK;
}

// ============================================================================ checkpoints
extern "C" int qw_set_capture(qw_handle* h, int32_t enable) {
  if (!h) QW_FAIL(h, QW_ERR_ARG, "qw_set_capture: null handle");
  DeviceGuard dg(h->device);
  const bool on = enable != 0;
  if (on && !h->cap_emb) {
    const size_t rows = (size_t)h->cfg.max_ctx * h->cfg.hidden;
    QW_CUDA(h, cudaMalloc((void**)&h->cap_emb, 3 * rows * 4));
    h->cap_blk0 = h->cap_emb + rows;
    h->cap_final = h->cap_emb + 2 * rows;
  }
  if (on != h->capture_on) h->graph_dirty = true;
  h->capture_on = on;
  h->cap_valid = false;
  return QW_OK;
}

extern "C" int qw_capture_size(qw_handle* h, int32_t which, size_t* n_floats) {
  if (!h || !n_floats) QW_FAIL(h, QW_ERR_ARG, "qw_capture_size: null argument");
  if (which < 0 || which > 3) QW_FAIL(h, QW_ERR_ARG, "qw_capture_size: which must be 0..3");
  if (!h->cap_valid) QW_FAIL(h, QW_ERR_NOT_CAPTURED, "qw_capture_size: nothing captured");
  *n_floats = which == QW_CAPTURE_LOGITS ? (size_t)h->cfg.vocab
                                         : (size_t)h->cap_rows * h->cfg.hidden;
  return QW_OK;
}

extern "C" int qw_get_capture(qw_handle* h, int32_t which, float* out_host, size_t n_floats) {
  size_t need = 0;
  int rc = qw_capture_size(h, which, &need);
  if (rc) return rc;
  if (!out_host) QW_FAIL(h, QW_ERR_ARG, "qw_get_capture: null buffer");
  if (n_floats < need) QW_FAIL(h, QW_ERR_SIZE, "qw_get_capture: buffer too small");
  DeviceGuard dg(h->device);
  const float* src = which == QW_CAPTURE_LOGITS ? h->logits
                     : (which == QW_CAPTURE_EMBEDDING ? h->cap_emb
                        : which == QW_CAPTURE_BLOCK0 ? h->cap_blk0 : h->cap_final) +
                           (size_t)h->cap_row0 * h->cfg.hidden;
  QW_CUDA(h, cudaMemcpyAsync(out_host, src, need * 4, cudaMemcpyDeviceToHost, h->stream));
  QW_CUDA(h, cudaStreamSynchronize(h->stream));
  return QW_OK;
}

// ============================================================================ stand-alone ops
static int op_sms(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = ensure_attributes(dev);
  if (e != cudaSuccess) {
    g_last_error = std::string("device set-up: ") + cudaGetErrorString(e);
    return QW_ERR_CUDA;
  }
  return QW_OK;
}

namespace qw {
void set_op_error(const char* msg) { g_last_error = msg; }
}  // namespace qw

#define QW_OP_CUDA(call)                                                        \
  do {                                                                          \
    cudaError_t e_ = (call);                                                    \
    if (e_ != cudaSuccess) {                                                    \
      g_last_error = std::string(#call) + ": " + cudaGetErrorString(e_);        \
      return QW_ERR_CUDA;                                                       \
    }                                                                           \
  } while (0)

extern "C" int qw_quantize_int4_g128(const float* w, int32_t rows, int32_t cols, uint8_t* packed,
                                     uint16_t* scales, void* stream) {
  if (!w || !packed || !scales || rows <= 0 || cols <= 0 || cols % 128)
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG,
            "qw_quantize_int4_g128: null buffer, empty shape or cols % 128 != 0");
  QW_OP_CUDA(launch_quantize_int4(w, rows, cols, packed, scales, (cudaStream_t)stream));
  return QW_OK;
}

// Attention workspace: [counters (nkv ints) | err int] padded to 256, part_ml, part_o.
extern "C" size_t qw_attention_workspace_bytes(int32_t nq, int32_t nkv, int32_t hd,
                                               int32_t n_splits) {
  if (nq <= 0 || nkv <= 0 || hd <= 0 || n_splits <= 0) return 0;
  return align_up(((size_t)nkv + 1) * 4, 256) + align_up((size_t)nq * n_splits * 2 * 4, 256) +
         (size_t)nq * n_splits * hd * 4;
}

extern "C" int qw_attention_decode(const float* qkv, const uint16_t* q_norm, const uint16_t* k_norm,
                                   float* k_cache, float* v_cache, int32_t nq, int32_t nkv,
                                   int32_t hd, int32_t cap, int32_t pos, float eps,
                                   float rope_theta, int32_t n_splits, float* out, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  if (!qkv || !k_cache || !v_cache || !out || !workspace)
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG, "qw_attention_decode: null buffer");
  if ((hd != 64 && hd != 128) || nkv <= 0 || nq <= 0 || nq % nkv || nq / nkv > attention_gq_max() ||
      n_splits <= 0 || n_splits > 65535)
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG, "qw_attention_decode: unsupported shape");
  if (!attention_splits_fit(nq / nkv, hd, n_splits))
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG,
            "qw_attention_decode: n_splits too large for the combine (query heads per KV head x "
            "(n_splits + 1) must fit 192 x head_dim floats)");
  if (pos < 0 || pos >= cap) QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG, "qw_attention_decode: pos outside [0, cap)");
  if (workspace_bytes < qw_attention_workspace_bytes(nq, nkv, hd, n_splits))
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG, "qw_attention_decode: workspace too small");
  int sms = 0;
  if (op_sms(&sms)) return QW_ERR_CUDA;
  uint8_t* ws = (uint8_t*)workspace;
  AttnArgs t{};
  t.qkv = qkv;
  t.q_norm = q_norm;
  t.k_norm = k_norm;
  t.rope = nullptr;  // cos/sin formed in fp64 inside the kernel
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
  t.part_ml = (float*)(ws + align_up(((size_t)nkv + 1) * 4, 256));
  t.part_o = (float*)((uint8_t*)t.part_ml + align_up((size_t)nq * n_splits * 2 * 4, 256));
  t.out = out;
  t.wait_ns = 1000000000ull;
  QW_OP_CUDA(launch_attention(t, hd, false, (cudaStream_t)stream));
  return QW_OK;
}

// LM-head workspace: [counter int | err int] padded to 256, blk_val[1024], blk_idx[1024].
extern "C" size_t qw_lm_head_workspace_bytes(void) { return 256 + 1024 * 4 + 1024 * 4; }

extern "C" int qw_lm_head_argmax(const float* x, const uint16_t* g, const uint16_t* table,
                                 int32_t vocab, int32_t hidden, float eps, float* logits,
                                 int32_t* argmax_dev, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  if (!x || !g || !table || !logits || !argmax_dev || !workspace)
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG, "qw_lm_head_argmax: null buffer");
  if (vocab <= 0 || hidden <= 0 || hidden % 8 || hidden > 16384)
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG, "qw_lm_head_argmax: hidden must be a positive multiple of 8, <= 16384");
  if (workspace_bytes < qw_lm_head_workspace_bytes())
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG, "qw_lm_head_argmax: workspace too small");
  int sms = 0;
  if (op_sms(&sms)) return QW_ERR_CUDA;
  uint8_t* ws = (uint8_t*)workspace;
  const int grid = std::min({vocab, sms, 1024});
  GemvArgs a{};
  a.w = (const uint8_t*)table;
  a.n_units = vocab;
  a.rpu = 1;
  a.K = hidden;
  a.row_bytes = (uint32_t)hidden * 2;
  a.x = x;
  a.norm_g = g;
  a.eps = eps;
  a.y = logits;
  a.am.counter = (int*)ws;
  a.err = (int*)ws + 1;
  a.am.blk_val = (float*)(ws + 256);
  a.am.blk_idx = (int*)(ws + 256 + 1024 * 4);
  a.am.argmax = argmax_dev;
  a.wait_ns = 1000000000ull;
  plan_gemv(a, grid, kStreamStage, kStreamStages);
  QW_OP_CUDA(launch_gemv(EPI_LOGITS, a, grid, false, (cudaStream_t)stream));
  return QW_OK;
}

// int4 GEMV workspace: [err int] padded to 256, then the rows repacked as the decode
// step streams them (int4_row_bytes(cols) each: nibbles, scales, zero pad).
extern "C" size_t qw_gemv_int4_workspace_bytes(int32_t rows, int32_t cols) {
  if (rows <= 0 || cols <= 0 || cols % 128) return 0;
  return 256 + (size_t)rows * int4_row_bytes(cols);
}

extern "C" int qw_gemv_int4_g128(const uint8_t* packed, const uint16_t* scales, int32_t rows,
                                 int32_t cols, const float* x, float* y, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (!packed || !scales || !x || !y || !workspace)
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG, "qw_gemv_int4_g128: null buffer");
  if (rows <= 0 || cols <= 0 || cols % 128 || cols > 16384)
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG,
            "qw_gemv_int4_g128: rows must be positive and cols a multiple of 128, at most 16384");
  if (workspace_bytes < qw_gemv_int4_workspace_bytes(rows, cols) || ((uintptr_t)workspace & 15))
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG,
            "qw_gemv_int4_g128: workspace too small or not 16-byte aligned");
  int sms = 0;
  if (op_sms(&sms)) return QW_ERR_CUDA;
  uint8_t* ws = (uint8_t*)workspace;
  uint8_t* rows_dev = ws + 256;
  const cudaStream_t st = (cudaStream_t)stream;
  QW_OP_CUDA(launch_pack_int4_rows(packed, scales, rows, cols, rows_dev, 0, 1, st));
  const int grid = std::min(rows, sms);
  GemvArgs a{};
  a.w = rows_dev;
  a.n_units = rows;
  a.rpu = 1;
  a.K = cols;
  a.wfmt = 1;
  a.row_bytes = int4_row_bytes(cols);
  a.scale_off = (uint32_t)cols / 2;
  a.x = x;
  a.y = y;
  a.err = (int*)ws;
  a.wait_ns = 1000000000ull;
  plan_gemv(a, grid, kStreamStage, kStreamStages);
  QW_OP_CUDA(launch_gemv(EPI_STORE, a, grid, false, st));
  return QW_OK;
}

extern "C" int qw_quantize_q8_0(const float* w, int32_t rows, int32_t cols, int8_t* q,
                                uint16_t* scales, void* stream) {
  if (!w || !q || !scales || rows <= 0 || cols <= 0 || cols % 32)
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG,
            "qw_quantize_q8_0: null buffer, empty shape or cols % 32 != 0");
  QW_OP_CUDA(launch_quantize_q8(w, false, rows, cols, q, (size_t)cols, scales, (size_t)cols / 32,
                                (cudaStream_t)stream));
  return QW_OK;
}

// Q8_0 GEMV workspace: [err int] padded to 256, then the rows repacked as the decode
// step streams them (q8_row_bytes(cols) each: int8 values, scales, zero pad).
extern "C" size_t qw_gemv_q8_0_workspace_bytes(int32_t rows, int32_t cols) {
  if (rows <= 0 || cols <= 0 || cols % 32) return 0;
  return 256 + (size_t)rows * q8_row_bytes(cols);
}

extern "C" int qw_gemv_q8_0(const int8_t* q, const uint16_t* scales, int32_t rows, int32_t cols,
                            const float* x, float* y, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if (!q || !scales || !x || !y || !workspace)
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG, "qw_gemv_q8_0: null buffer");
  if (rows <= 0 || cols <= 0 || cols % 32 || cols > 16384)
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG,
            "qw_gemv_q8_0: rows must be positive and cols a multiple of 32, at most 16384");
  if (workspace_bytes < qw_gemv_q8_0_workspace_bytes(rows, cols) || ((uintptr_t)workspace & 15))
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG,
            "qw_gemv_q8_0: workspace too small or not 16-byte aligned");
  int sms = 0;
  if (op_sms(&sms)) return QW_ERR_CUDA;
  uint8_t* ws = (uint8_t*)workspace;
  uint8_t* rows_dev = ws + 256;
  const cudaStream_t st = (cudaStream_t)stream;
  QW_OP_CUDA(launch_pack_q8_rows(q, scales, rows, cols, rows_dev, 0, 1, st));
  const int grid = std::min(rows, sms);
  GemvArgs a{};
  a.w = rows_dev;
  a.n_units = rows;
  a.rpu = 1;
  a.K = cols;
  a.wfmt = 2;
  a.row_bytes = q8_row_bytes(cols);
  a.scale_off = (uint32_t)cols;
  a.x = x;
  a.y = y;
  a.err = (int*)ws;
  a.wait_ns = 1000000000ull;
  plan_gemv(a, grid, kStreamStage, kStreamStages);
  QW_OP_CUDA(launch_gemv(EPI_STORE, a, grid, false, st));
  return QW_OK;
}

extern "C" size_t qw_sample_workspace_bytes(int32_t vocab, int32_t top_k) {
  if (vocab < 1 || top_k < 1) return 0;
  return sample_workspace_bytes(vocab, std::min(top_k, vocab));
}

static int sample_args_ok(int32_t vocab, int32_t top_k, float top_p, float u, const char* fn) {
  if (vocab < 1 || top_k < 1 || top_k > kMaxSampleTopK || !sample_shape_ok(vocab, std::min(top_k, vocab)))
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG,
            std::string(fn) + ": top_k must be in [1, 256] and vocab / 16384 * top_k <= 4096");
  if (!(top_p > 0.f)) QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG, std::string(fn) + ": top_p must be > 0");
  if (!(u >= 0.f && u < 1.f)) QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG, std::string(fn) + ": u must be in [0, 1)");
  return QW_OK;
}

extern "C" int qw_sample(const float* logits, int32_t vocab, float temperature, int32_t top_k,
                         float top_p, float u, int32_t* token_dev, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (!logits || !token_dev || !workspace)
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG, "qw_sample: null buffer");
  int rc = sample_args_ok(vocab, top_k, top_p, u, "qw_sample");
  if (rc) return rc;
  if (workspace_bytes < qw_sample_workspace_bytes(vocab, top_k))
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG, "qw_sample: workspace too small");
  int sms = 0;
  if (op_sms(&sms)) return QW_ERR_CUDA;
  QW_OP_CUDA(launch_sample(logits, vocab, top_k, temperature, top_p, u, token_dev, workspace,
                           (cudaStream_t)stream));
  return QW_OK;
}

extern "C" int qw_sample_last(qw_handle* h, float temperature, int32_t top_k, float top_p, float u,
                              int32_t* token_host) {
  int rc = check_ready(h, "qw_sample_last");
  if (rc) return rc;
  if (!token_host) QW_FAIL(h, QW_ERR_ARG, "qw_sample_last: null token_host");
  if (h->pos == 0) QW_FAIL(h, QW_ERR_STATE, "qw_sample_last: no step has produced logits yet");
  rc = sample_args_ok(h->cfg.vocab, top_k, top_p, u, "qw_sample_last");
  if (rc) {
    h->err = g_last_error;
    return rc;
  }
  DeviceGuard dg(h->device);
  QW_CUDA(h, launch_sample(h->logits, h->cfg.vocab, top_k, temperature, top_p, u, h->d_sample_tok,
                           h->sample_ws, h->stream));
  QW_CUDA(h, cudaMemcpyAsync(&h->h_status[4], h->d_sample_tok, 4, cudaMemcpyDeviceToHost, h->stream));
  QW_CUDA(h, cudaStreamSynchronize(h->stream));
  const int id = ((volatile int*)h->h_status)[4];
  if (id < 0) QW_FAIL(h, QW_ERR_NUMERIC, "qw_sample_last: the logits hold a NaN or no finite value");
  *token_host = id;
  return QW_OK;
}

extern "C" int qw_gemm_bf16(const uint16_t* a_hi, const uint16_t* a_lo, const uint16_t* b,
                            int32_t M, int32_t N, int32_t K, float* c, int32_t bn, void* stream) {
  if (!a_hi || !b || !c || M <= 0 || N <= 0 || K <= 0 || K % 8)
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG, "qw_gemm_bf16: null buffer, empty shape or K % 8 != 0");
  if (bn == 0) bn = N >= 2048 ? 256 : (N >= 512 ? 128 : 64);
  if (bn != 64 && bn != 128 && bn != 256)
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG, "qw_gemm_bf16: bn must be 0, 64, 128 or 256");
  int sms = 0;
  if (op_sms(&sms)) return QW_ERR_CUDA;
  CUtensorMap ta_hi, ta_lo, tb;
  if (!make_tmap_bf16_2d(&ta_hi, a_hi, M, K, 128) ||
      !make_tmap_bf16_2d(&ta_lo, a_lo ? a_lo : a_hi, M, K, 128) ||
      !make_tmap_bf16_2d(&tb, b, N, K, (uint32_t)bn))
    QW_FAIL((qw_handle*)nullptr, QW_ERR_ARG, "qw_gemm_bf16: tensor map rejected (alignment?)");
  GemmArgs g{};
  g.M = M;
  g.N = N;
  g.K = K;
  g.a_split = a_lo ? 2 : 1;
  g.out = c;
  g.ldo = N;
  g.err = gemm_op_err_word();
  g.wait_ns = 1000000000ull;
  if (!g.err) QW_FAIL((qw_handle*)nullptr, QW_ERR_CUDA, "qw_gemm_bf16: error word lookup failed");
  QW_OP_CUDA(launch_gemm(bn, GEPI_STORE, ta_hi, ta_lo, tb, nullptr, g, (cudaStream_t)stream));
  return QW_OK;
}

extern "C" int qw_set_decode_path(qw_handle* h, int32_t path) {
  if (!h) QW_FAIL(h, QW_ERR_ARG, "qw_set_decode_path: null handle");
  if (path != 0 && path != 1) QW_FAIL(h, QW_ERR_ARG, "qw_set_decode_path: path must be 0 or 1");
  h->path_pref = path;
  const bool mega = path == 0 && h->mega_ok && (!h->lora_active || h->mega_lora_ok);
  if (mega != h->use_mega) h->graph_dirty = true;
  h->use_mega = mega;
  return QW_OK;
}

extern "C" int qw_get_decode_path(const qw_handle* h, int32_t* path) {
  if (!h || !path) return QW_ERR_ARG;
  *path = h->use_mega ? 0 : 1;
  return QW_OK;
}
