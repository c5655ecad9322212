/*
 * qw.h -- C ABI of the GB300 (sm_103a) batch-1 Qwen-style decode step.
 *
 * The operation: the autoregressive forward step of a Qwen3-style decoder
 * ("Failed Star / fs, M2" page, "One prefill, all shapes visible": gather ->
 * x L blocks of RMSNorm, QKV, QK-norm, RoPE, GQA causal attention, o_proj +
 * residual, RMSNorm, SwiGLU, down + residual -> final RMSNorm -> tied [V,H]
 * projection of the last row), with an f32-resident KV cache, RoPE applied on
 * the KV write and a greedy argmax taken on the device so that only the token
 * id crosses to the host ("flashmoon demo" page, Performance: decode-critical
 * invariants). Qwen2.5 variants add q/k/v biases, drop QK-norm, use an
 * untied lm_head, int4 group-128 weights and an optional LoRA on q_proj and
 * v_proj ("Emberglass" README, "Why it's hard"). The config and weight
 * structs follow the C structs of the "SuperKittens PR #7" page (sk_qwen_config
 * with eps and tie_word_embeddings; sk_qwen_weights with a nullable lm_head),
 * with a struct_size field so a caller whose struct is shorter than the
 * library's is rejected instead of read past (the bug that page's review found).
 *
 * Conventions for every call:
 *   - Return 0 (QW_OK) or a negative QW_ERR_* code; qw_last_error() gives text.
 *   - "device" pointers are CUDA device (or managed) addresses on the handle's
 *     device; "host" pointers are ordinary CPU memory.
 *   - All GPU work is queued on the handle's stream. Calls that return a host
 *     value (argmax_host, ids_host, qw_get_capture) synchronise that stream.
 *   - A handle is not thread-safe: one thread at a time per handle.
 *   - The library owns the memory it allocates and frees it in qw_destroy.
 */
#ifndef QW_H_
#define QW_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QW_ABI_VERSION 2u

/* Status codes. */
enum {
  QW_OK = 0,
  QW_ERR_ABI = -1,            /* struct_size / abi_version mismatch */
  QW_ERR_ARG = -2,            /* null pointer, token out of [0,vocab), T <= 0, bad shape */
  QW_ERR_CTX = -3,            /* position would pass max_ctx (checked before any work) */
  QW_ERR_NOT_CAPTURED = -4,   /* checkpoint asked for before a forward that recorded it */
  QW_ERR_SIZE = -5,           /* caller's buffer is too small */
  QW_ERR_CUDA = -6,           /* a CUDA runtime call failed */
  QW_ERR_DEVICE_TIMEOUT = -7, /* a bounded device-side wait gave up */
  QW_ERR_STATE = -8,          /* call out of order (e.g. decode before weights) */
  QW_ERR_NUMERIC = -9         /* a logit was NaN, so there is no argmax */
};

/* qw_config.weight_format */
enum { QW_WEIGHTS_BF16 = 0, QW_WEIGHTS_INT4_G128 = 1, QW_WEIGHTS_Q8_0 = 2 };

/* qw_config.kv_format: how keys (after QK-norm and RoPE) and values are stored. bf16
 * halves the cache ("Emberglass" README, Context window & prefill sizes: the f32
 * cache could be quantised to roughly half); each value is rounded to the nearest
 * bf16 when stored, and attention reads the stored values, widened to f32. */
enum { QW_KV_F32 = 0, QW_KV_BF16 = 1 };

/* qw_get_capture `which`: the four checkpoints of the "Failed Star / fs, M2"
 * page ("Four boundaries bisect the whole model"). */
enum {
  QW_CAPTURE_EMBEDDING = 0,  /* f32 [rows, hidden]: gathered embedding rows   */
  QW_CAPTURE_BLOCK0 = 1,     /* f32 [rows, hidden]: residual after block 0     */
  QW_CAPTURE_FINAL_NORM = 2, /* f32 [rows, hidden]: final RMSNorm output       */
  QW_CAPTURE_LOGITS = 3      /* f32 [vocab]: logits of the last row            */
};

typedef struct qw_handle qw_handle;

/* Model shape and options. Set struct_size = sizeof(qw_config) and
 * abi_version = QW_ABI_VERSION. head_dim must be 64 or 128; hidden,
 * n_q_heads*head_dim and intermediate must be multiples of 8 (of 128 for
 * int4, of 32 for Q8_0); n_q_heads must be a multiple of n_kv_heads with at
 * most 8 query heads per KV head. */
typedef struct qw_config {
  uint32_t struct_size;
  uint32_t abi_version;
  int32_t n_layers;
  int32_t hidden;
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t intermediate;
  int32_t vocab;
  float eps;                    /* RMSNorm epsilon (inside the square root) */
  float rope_theta;             /* RoPE base */
  uint32_t tie_word_embeddings; /* 1: logits = embed . h ; 0: separate lm_head */
  uint32_t qk_norm;             /* 1: per-head RMSNorm of q and k before RoPE (Qwen3) */
  uint32_t qkv_bias;            /* 1: q/k/v projections carry a bias (Qwen2.5) */
  int32_t max_ctx;              /* KV-cache capacity in positions */
  int32_t max_prefill_t;        /* longest prompt taken by one batched prefill pass */
  uint32_t weight_format;       /* QW_WEIGHTS_BF16, QW_WEIGHTS_INT4_G128 or QW_WEIGHTS_Q8_0 */
  uint32_t kv_format;           /* QW_KV_F32 or QW_KV_BF16 */
} qw_config;

/* Weights, all DEVICE pointers owned by the caller; the per-layer members are
 * HOST arrays of n_layers DEVICE pointers. qw_load_weights copies (and repacks)
 * everything into library memory, so the caller may free all of it once the
 * call returns.
 *
 * bf16 tensors are raw bf16 bit patterns, row-major [out, in] as stored by
 * Hugging Face checkpoints ("Failed Star / fs, M2", Correct before fast).
 * int4 tensors (weight_format = QW_WEIGHTS_INT4_G128) are nibble-packed
 * [out, in/2] bytes (element 2i in the low nibble, value = nibble - 8) with
 * bf16 scales [out, in/128], one per 128 consecutive inputs of a row; see
 * qw_quantize_int4_g128. Q8_0 tensors (weight_format = QW_WEIGHTS_Q8_0) are
 * int8 [out, in] (two's complement) with fp16 scales [out, in/32], one per 32
 * consecutive inputs of a row, in the *_scales members; see qw_quantize_q8_0.
 * A Q8_0 model's LM head is Q8_0 too: the untied lm_head is passed quantised,
 * and a tied model's head is quantised from the embedding table at load (the
 * "SuperKittens PR #7" page, Q8_0 commit); the gather keeps the bf16 rows.
 * Embedding, norms and biases are always bf16. */
typedef struct qw_weights {
  uint32_t struct_size;
  uint32_t reserved0;
  const void* embed;          /* bf16 [vocab, hidden] */
  const void* final_norm;     /* bf16 [hidden] */
  const void* lm_head;        /* [vocab, hidden]; must be NULL iff tie_word_embeddings;
                               * int4 (with lm_head_scales) when weight_format is int4 */
  const void* lm_head_scales; /* scales of an int4 or Q8_0 untied lm_head, else NULL */
  const void* const* attn_norm; /* bf16 [hidden] */
  const void* const* q;         /* [n_q_heads*head_dim, hidden] */
  const void* const* k;         /* [n_kv_heads*head_dim, hidden] */
  const void* const* v;         /* [n_kv_heads*head_dim, hidden] */
  const void* const* o;         /* [hidden, n_q_heads*head_dim] */
  const void* const* mlp_norm;  /* bf16 [hidden] */
  const void* const* gate;      /* [intermediate, hidden] */
  const void* const* up;        /* [intermediate, hidden] */
  const void* const* down;      /* [hidden, intermediate] */
  const void* const* q_norm;    /* bf16 [head_dim]; qk_norm only, else NULL */
  const void* const* k_norm;    /* bf16 [head_dim]; qk_norm only, else NULL */
  const void* const* q_bias;    /* bf16 [n_q_heads*head_dim]; qkv_bias only, else NULL */
  const void* const* k_bias;    /* bf16 [n_kv_heads*head_dim] */
  const void* const* v_bias;    /* bf16 [n_kv_heads*head_dim] */
  const void* const* q_scales;  /* int4: bf16, Q8_0: fp16 scales of each linear, else NULL */
  const void* const* k_scales;
  const void* const* v_scales;
  const void* const* o_scales;
  const void* const* gate_scales;
  const void* const* up_scales;
  const void* const* down_scales;
} qw_weights;

/* Low-rank adapter on q_proj and v_proj: y += (alpha / rank) * B (A x)
 * ("Emberglass" README: LoRA hot-swap, perfect restore on clear). All members
 * are HOST arrays of n_layers DEVICE pointers to bf16 data. They are BORROWED:
 * the library keeps the pointers, so the tensors must stay alive until the
 * adapter is cleared with qw_set_lora(h, NULL) or the handle is destroyed. */
typedef struct qw_lora {
  uint32_t struct_size;
  int32_t rank;                 /* 1..64 */
  float alpha;
  uint32_t reserved0;
  const void* const* q_a;       /* [rank, hidden] */
  const void* const* q_b;       /* [n_q_heads*head_dim, rank] */
  const void* const* v_a;       /* [rank, hidden] */
  const void* const* v_b;       /* [n_kv_heads*head_dim, rank] */
} qw_lora;

/* ABI self-description, so a binding can check its struct layouts. */
uint32_t qw_abi_version(void);
size_t qw_sizeof_config(void);
size_t qw_sizeof_weights(void);
size_t qw_sizeof_lora(void);

/* Create a handle on the current CUDA device. cuda_stream is a cudaStream_t
 * the handle will use (borrowed), or NULL for a stream the handle creates and
 * owns. Allocates the KV cache (2 * n_layers * n_kv_heads * max_ctx * head_dim
 * elements of 4 bytes, or 2 with QW_KV_BF16) and work buffers. *out is set only
 * on success. */
int qw_create(const qw_config* cfg, void* cuda_stream, qw_handle** out);

/* Copy and repack the weights into library memory (fused [q;k;v] rows,
 * interleaved gate/up rows). May be called again to replace them; resets the
 * position to 0. */
int qw_load_weights(qw_handle* h, const qw_weights* w);

/* Process T prompt ids (HOST array) at positions pos..pos+T-1, appending their
 * keys and values to the cache; afterwards pos += T. Prompts of at most
 * max_prefill_t ids with no LoRA active run as one batched causal pass on the
 * tensor cores (int4 weights are dequantised exactly, layer by layer, into two
 * bf16 terms for it); longer prompts, any prompt while a LoRA is set, and every
 * prompt of a Q8_0 model run through the sequential decode path ("Emberglass"
 * README, Context window & prefill sizes: maxPrefillT). logits_dev (DEVICE, vocab
 * floats, nullable) receives the last row's logits; argmax_host (nullable)
 * receives its greedy token and makes the call synchronous.
 * Errors: QW_ERR_ARG (T <= 0, id out of range), QW_ERR_CTX (pos+T > max_ctx). */
int qw_prefill(qw_handle* h, const int32_t* ids_host, int32_t T, float* logits_dev,
               int32_t* argmax_host);

/* One decode step at position pos: token in [0, vocab), or token < 0 to feed
 * the previous step's device-resident argmax (no host round trip). Afterwards
 * pos += 1. logits_dev (DEVICE, vocab floats) and argmax_host are nullable as
 * in qw_prefill. Errors: QW_ERR_ARG, QW_ERR_CTX, QW_ERR_STATE (token < 0 with
 * no previous step), QW_ERR_DEVICE_TIMEOUT, QW_ERR_NUMERIC. */
int qw_decode_step(qw_handle* h, int32_t token, float* logits_dev, int32_t* argmax_host);

/* n_steps greedy steps on the device, the first fed `token` (or the previous
 * argmax if token < 0), each next one fed the previous argmax without leaving
 * the GPU ("Emberglass" README: GPU-resident batched decode loop, one sync per
 * batch). ids_host (HOST, n_steps ints, nullable) receives the n_steps greedy
 * tokens; the call synchronises once at the end. */
int qw_decode_greedy(qw_handle* h, int32_t token, int32_t n_steps, int32_t* ids_host);

/* pos = 0. Weights and LoRA are kept; cache contents are left as they are and
 * are overwritten as positions are reused. */
int qw_reset(qw_handle* h);

/* Set (lora != NULL) or clear (NULL) the adapter. Weights are never merged, so
 * clearing restores bit-identical outputs. */
int qw_set_lora(qw_handle* h, const qw_lora* lora);

/* Test hooks. qw_kv_cache returns DEVICE pointers to layer `layer`'s K and V
 * cache, each [n_kv_heads, max_ctx, head_dim] (keys stored after QK-norm and
 * RoPE) of f32, or of bf16 bits with QW_KV_BF16, owned by the handle.
 * qw_set_pos / qw_get_pos move or read the position (0 <= pos <= max_ctx). */
int qw_kv_cache(qw_handle* h, int32_t layer, void** k_dev, void** v_dev);
int qw_set_pos(qw_handle* h, int32_t pos);
int qw_get_pos(const qw_handle* h, int32_t* pos);

/* Checkpoints. qw_set_capture(h, 1) makes later forwards record the four
 * checkpoints (it costs extra writes, so it is off by default). After a
 * forward, qw_capture_size gives the floats of checkpoint `which` and
 * qw_get_capture copies them to out_host (HOST, n_floats >= that size).
 * Errors: QW_ERR_NOT_CAPTURED when capture was off for the last forward or
 * no forward ran since it was enabled; QW_ERR_SIZE when n_floats is short. */
int qw_set_capture(qw_handle* h, int32_t enable);
int qw_capture_size(qw_handle* h, int32_t which, size_t* n_floats);
int qw_get_capture(qw_handle* h, int32_t which, float* out_host, size_t n_floats);

/* Decode path (test and benchmarking hook). 0: one persistent cooperative kernel
 * per token, the default whenever the shape fits: head_dim 64 or 128, at most 8
 * query heads per KV head, hidden, intermediate and n_q_heads*head_dim <= 11264,
 * any weight format (int4 only with an untied lm_head) and either cache format,
 * and with a LoRA adapter when each CTA's share of the fused q/k/v rows is at
 * most 64 (every shape up to ~9.7K fused rows); 1: the graph of separate kernels (always
 * available). Asking for 0 on a shape that does not fit keeps 1. Both compute
 * the same step; results agree to f32 rounding. If the persistent
 * kernel cannot be recorded on this device (no cooperative launch), the handle
 * switches to 1 for the rest of its life: the step still succeeds, one line goes
 * to stderr, qw_last_error(h) holds a note saying why, and qw_get_decode_path
 * returns 1. The choice is kept across qw_set_lora. */
int qw_set_decode_path(qw_handle* h, int32_t path);
int qw_get_decode_path(const qw_handle* h, int32_t* path);

/* Bound, in nanoseconds, of every device-side wait (default 1e9). 0 makes
 * every wait give up at once, which tests the QW_ERR_DEVICE_TIMEOUT path. */
int qw_set_wait_limit_ns(qw_handle* h, uint64_t ns);

/* Text of the last error on this handle (or of the last failed handle-less
 * call when h is NULL), or the note of a decode-path switch (see
 * qw_set_decode_path). Valid until the next call. */
const char* qw_last_error(const qw_handle* h);

void qw_destroy(qw_handle* h);

/* ---------------------------------------------------------------------------
 * Stand-alone operations (no handle). They run the same kernels the decode
 * step uses, on caller-provided DEVICE buffers, for per-kernel checks
 * ("flashmoon demo" page, Verification: kernel unit checks against an f64
 * oracle). `stream` is a cudaStream_t or NULL for the legacy default stream.
 * ------------------------------------------------------------------------- */

/* int4 group-128 quantiser ("Emberglass" README: int4 group-128, quantised on
 * the way to the GPU). w: f32 [rows, cols] DEVICE, finite, cols % 128 == 0.
 * packed: u8 [rows, cols/2]; scales: bf16 bits [rows, cols/128]. Per group:
 * s = bf16_rne(f32(max|w| / 7)); q = clamp(rint(f32(w / s)), -7, 7) (0 if
 * s == 0); nibble = q + 8, element 2i in the low nibble. */
int qw_quantize_int4_g128(const float* w, int32_t rows, int32_t cols, uint8_t* packed,
                          uint16_t* scales, void* stream);

/* Decode attention for one layer at position pos: per-head QK-RMSNorm (if
 * q_norm/k_norm are non-NULL), RoPE at pos (rotate-half, cos/sin formed in
 * fp64), append of k and v at cache row pos, split-K flash attention of every
 * query head over keys 0..pos of its KV head, and the combine of the splits
 * ("Emberglass" README: split-K flash-style decode attention).
 *   qkv:       f32 [(nq + 2 nkv) * hd] DEVICE, raw projections (q heads, k heads, v heads)
 *   q_norm, k_norm: bf16 [hd] DEVICE or NULL
 *   k_cache, v_cache: f32 [nkv, cap, hd] DEVICE; row pos is written
 *   out:       f32 [nq * hd] DEVICE
 *   n_splits:  most key splits per KV head, with (nq / nkv) * (n_splits + 1) at most
 *              192 * hd (the combine keeps its weights in the kernel's tile buffers)
 *   workspace: DEVICE scratch of qw_attention_workspace_bytes(...) bytes,
 *              zero-filled before its first use and left zeroed by every call.
 * Errors: QW_ERR_ARG for unsupported shapes (nq or nkv <= 0 included), too many
 * splits, pos outside [0, cap), or a short workspace; all are found on the host
 * before any launch. A device-side wait that gives up is not reported by this
 * unit-check op (its outputs are then invalid); the decode step reports it. */
size_t qw_attention_workspace_bytes(int32_t nq, int32_t nkv, int32_t hd, int32_t n_splits);
int qw_attention_decode(const float* qkv, const uint16_t* q_norm, const uint16_t* k_norm,
                        float* k_cache, float* v_cache, int32_t nq, int32_t nkv, int32_t hd,
                        int32_t cap, int32_t pos, float eps, float rope_theta, int32_t n_splits,
                        float* out, void* workspace, size_t workspace_bytes, void* stream);

/* qw_attention_decode without a workspace argument, for callers that cannot
 * allocate device memory (code running while another thread captures a CUDA
 * graph, allocator-free real-time loops, embedders whose device memory belongs
 * to someone else's pool). The pages have no counterpart of this call; it is a
 * deployment convenience. Arguments and results are those of
 * qw_attention_decode. Its scratch is a fixed file-scope device array of
 * qw_attention_noalloc_max_bytes() bytes (1 MiB) that every GPU loading this
 * library keeps until the process exits; shapes whose scratch
 * (256 + nq*n_splits*(hd+2)*4 bytes, rounded) does not fit return QW_ERR_SIZE.
 * The first call on a device looks up that array's device address and sets the
 * kernel attributes, so make it before any stream capture on that device.
 * Every call shares the one array and clears its counters on `stream`: calls
 * that overlap on the GPU (different streams, or several host threads) race
 * and must be serialised by the caller. No call allocates memory. Failures set
 * qw_last_error(NULL) text like the other handle-less calls; a device-side wait
 * that gives up is not reported, as for qw_attention_decode. */
size_t qw_attention_noalloc_max_bytes(void);
int qw_attention_decode_noalloc(const float* qkv, const uint16_t* q_norm, const uint16_t* k_norm,
                                float* k_cache, float* v_cache, int32_t nq, int32_t nkv,
                                int32_t hd, int32_t cap, int32_t pos, float eps,
                                float rope_theta, int32_t n_splits, float* out, void* stream);

/* Final RMSNorm + LM head + greedy argmax over a bf16 [vocab, hidden] table
 * ("Failed Star / fs, M2": final norm, last row, tied [V,H] projection;
 * "flashmoon demo": argmax in the same submit):
 *   h = g * x / sqrt(mean(x^2) + eps); logits = table . h; argmax (ties -> lowest id).
 *   x: f32 [hidden] DEVICE; g: bf16 [hidden] DEVICE; table: bf16 [vocab, hidden] DEVICE;
 *   logits: f32 [vocab] DEVICE; argmax_dev: int32 [1] DEVICE (-1 if any logit is NaN);
 *   workspace: DEVICE scratch of qw_lm_head_workspace_bytes() bytes, zero-filled
 *   before its first use and left zeroed by every call. */
size_t qw_lm_head_workspace_bytes(void);
int qw_lm_head_argmax(const float* x, const uint16_t* g, const uint16_t* table, int32_t vocab,
                      int32_t hidden, float eps, float* logits, int32_t* argmax_dev,
                      void* workspace, size_t workspace_bytes, void* stream);

/* int4 group-128 matrix-vector product, the contraction the decode step runs for
 * int4 weights ("Emberglass" README, "Why it's hard": int4 group-128 weights,
 * dequantised inside the matvec):
 *   y[r] = sum_c W'[r][c] x[c],  W'[r][c] = (nibble(r, c) - 8) * scale[r][c / 128]
 *   packed: u8 [rows, cols/2] DEVICE, element 2i in the low nibble of byte i;
 *   scales: bf16 bits [rows, cols/128] DEVICE (the layout qw_quantize_int4_g128 writes);
 *   x: f32 [cols] DEVICE; y: f32 [rows] DEVICE; cols a multiple of 128, at most 16384;
 *   workspace: DEVICE scratch of qw_gemv_int4_workspace_bytes(rows, cols) bytes,
 *   16-byte aligned, no initialisation needed: the rows are repacked there (a row's
 *   nibbles, then its scales) and the decode step's int4 GEMV kernel runs on them.
 * The dequantisation is exact in f32 (a 4-bit integer times a bf16), so with
 * x = e_j the result is column j of W' bit for bit. Like the other stand-alone
 * ops it does not report a device-side wait that gave up (its outputs are then
 * invalid); QW_ERR_ARG for the argument errors above. */
size_t qw_gemv_int4_workspace_bytes(int32_t rows, int32_t cols);
int qw_gemv_int4_g128(const uint8_t* packed, const uint16_t* scales, int32_t rows, int32_t cols,
                      const float* x, float* y, void* workspace, size_t workspace_bytes,
                      void* stream);

/* Q8_0 quantiser ("SuperKittens PR #7" page, Q8_0 commit: GGUF type-8 weights, blocks
 * of 32 int8 values with one scale). w: f32 [rows, cols] DEVICE, finite, cols % 32 == 0.
 * q: int8 [rows, cols]; scales: fp16 bits [rows, cols/32]. Per block of 32 inputs:
 * s = fp16_rne(f32(max|w| / 127)); q = clamp(rint(f32(w / s)), -127, 127) (0 if s == 0). */
int qw_quantize_q8_0(const float* w, int32_t rows, int32_t cols, int8_t* q, uint16_t* scales,
                     void* stream);

/* Q8_0 matrix-vector product, the contraction the decode step runs for Q8_0 weights:
 *   y[r] = sum_c W'[r][c] x[c],  W'[r][c] = q[r][c] * scale[r][c / 32]
 *   q: int8 [rows, cols] DEVICE; scales: fp16 bits [rows, cols/32] DEVICE; x: f32 [cols];
 *   y: f32 [rows]; cols a multiple of 32, at most 16384; workspace: DEVICE scratch of
 *   qw_gemv_q8_0_workspace_bytes(rows, cols) bytes, 16-byte aligned, no initialisation
 *   needed (the rows are repacked there as the decode step streams them).
 * The dequantisation is exact in f32, so with x = e_j the result is column j of W' bit
 * for bit. A device-side wait that gives up is not reported (outputs invalid). */
size_t qw_gemv_q8_0_workspace_bytes(int32_t rows, int32_t cols);
int qw_gemv_q8_0(const int8_t* q, const uint16_t* scales, int32_t rows, int32_t cols,
                 const float* x, float* y, void* workspace, size_t workspace_bytes, void* stream);

/* Sampling on the device ("flashmoon demo" README: greedy plus temperature / top-k /
 * top-p sampling, temp = 0 meaning greedy; the demo reads every logits row back to
 * the host to sample, at about 2.7x the cost of the decode step). Here only the id
 * leaves the device. With the k largest logits ordered by (logit descending, index
 * ascending) and l_0 the largest:
 *   w_i = exp((l_i - l_0) / temperature)   (f64, i < k)
 *   the nucleus is the shortest prefix whose running sum of w reaches top_p times the
 *   sum over all k; the token is the first candidate of the nucleus whose running sum
 *   exceeds u times the nucleus sum.
 *   temperature <= 0 (or top_k == 1): the greedy argmax (ties -> lowest id).
 *   logits: f32 [vocab] DEVICE; vocab >= 1; top_k in [1, 256], larger than vocab is
 *   clamped to vocab; top_p in (0, 1] (>= 1: no nucleus cut); u in [0, 1), the
 *   uniform draw, supplied by the caller (the library draws no random numbers);
 *   token_dev: int32 [1] DEVICE, receives the id, or -1 when the row holds a NaN or
 *   no finite logit; workspace: DEVICE scratch of qw_sample_workspace_bytes(vocab,
 *   top_k) bytes, no initialisation needed. QW_ERR_ARG for arguments outside these
 *   ranges (also when vocab / 16384 * top_k > 4096, the final sort's capacity). */
size_t qw_sample_workspace_bytes(int32_t vocab, int32_t top_k);
int qw_sample(const float* logits, int32_t vocab, float temperature, int32_t top_k, float top_p,
              float u, int32_t* token_dev, void* workspace, size_t workspace_bytes, void* stream);

/* qw_sample over the handle's logits of its last step (qw_decode_step,
 * qw_decode_greedy or qw_prefill), on the handle's stream and with its own
 * workspace; writes the id to *token_host (synchronises). QW_ERR_STATE before any
 * step, QW_ERR_NUMERIC when the row holds a NaN or no finite logit. */
int qw_sample_last(qw_handle* h, float temperature, int32_t top_k, float top_p, float u,
                   int32_t* token_host);

/* Prefill contraction on tcgen05 tensor cores: C[M,N] = (A_hi + A_lo)[M,K] . B[N,K]^T.
 * A_hi, A_lo (nullable), B: bf16 row-major DEVICE, 16-byte aligned, K % 8 == 0; C: f32
 * [M,N] DEVICE. The activation of a layer enters as its two-bf16 split (hi = bf16(x),
 * lo = bf16(x - hi)) against the exact bf16 weight rows ("Emberglass" README: batched
 * tiled-GEMM prefill). bn: output-tile width 64, 128 or 256 (0 picks one). */
int qw_gemm_bf16(const uint16_t* a_hi, const uint16_t* a_lo, const uint16_t* b, int32_t M,
                 int32_t N, int32_t K, float* c, int32_t bn, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* QW_H_ */
