/*
 * tee.h -- C ABI of the packed-varlen text-embedding encoder (GB300, sm_103a).
 *
 * The library runs the batched forward pass of a ModernBERT-style encoder
 * (the Ruri-v3-310m shape by default) over several texts packed into one
 * token sequence, and returns one unit-length vector per text.  The method
 * is the one described on the tensai page "テキスト埋め込み"
 * (mattn.github.io/tensai/ja/embeddings):
 *
 *   §何が動くか / エンコーダ  per layer a bias-free LayerNorm, multi-head
 *       attention with RoPE and a GeGLU feed-forward; the first layer and
 *       every third one after it attend to the whole text (RoPE base
 *       160000), the others to 64 tokens on each side (base 10000).
 *   §何が動くか / プーリング  the last layer's states are averaged over the
 *       text and scaled to length 1.
 *   §何が動くか, packing paragraph  several texts go through one pass;
 *       positions restart at each text and attention never crosses a text
 *       boundary, so results equal one-at-a-time encoding.
 *   §精度と量子化  an integer path: int8 weight blocks, activations rounded
 *       per row to 7 bits with one scale.
 *
 * Conventions for every entry point:
 *   - return TEE_OK (0) on success, a negative TEE_E* code otherwise; the
 *     message of the last failure is available from tee_last_error().
 *   - a failed call leaves the context usable (except after TEE_ECUDA
 *     caused by a sticky device error, which CUDA itself makes permanent).
 *   - all pointers documented as "host" are read or written only during the
 *     call; the caller keeps ownership.  The library owns all device memory
 *     it allocates; tee_destroy releases it.
 *   - a context is not thread-safe: one host thread at a time per context.
 */
#ifndef TEE_H
#define TEE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ----------------------------------------------------- */
#define TEE_OK          0
#define TEE_EINVAL     -1   /* bad argument: null pointer, bad size, malformed cu_seqlens, id out of range */
#define TEE_ENOTLOADED -2   /* encode before tee_load_weights succeeded */
#define TEE_ENOMEM     -3   /* device or host allocation failed */
#define TEE_ECUDA      -4   /* a CUDA runtime/driver call failed */
#define TEE_ETOOLONG   -5   /* total tokens > max_tokens or texts > max_texts */
#define TEE_ETIMEOUT   -6   /* a bounded device-side wait gave up (kernel status word set) */

/* ---- arithmetic of the pass -------------------------------------------- */
#define TEE_F32   0   /* fp32 weights and activations, fp32 FFMA GEMMs */
#define TEE_BF16  1   /* bf16 weights/activations on tensor cores, fp32 accumulation, fp32 residual */
#define TEE_W8A8  2   /* int8 weight blocks x 7-bit per-row activations, exact int32 block sums */
#define TEE_W4A8  3   /* 4-bit weight blocks (codes in [-7, 7], two per byte, one fp32 scale per 32) x 7-bit
                         per-row activations, exact int32 block sums (this library's reading of the page's -q4) */
#define TEE_W6A8  4   /* 6-bit weight blocks (codes in [-31, 31], four per three bytes, one fp32 scale per 32)
                         x 7-bit per-row activations, exact int32 block sums (the page's -q4 repacks 4- and
                         6-bit blocks; this is this library's 6-bit block) */

/*
 * Encoder shape and run limits.  Readings where the page is silent:
 * pre-norm blocks, no embedding or final norm (both available as options for
 * the published ModernBERT layout), no bias on any projection,
 * rotate-half RoPE pairing (j, j + head_dim/2), a window of |i - j| <= window
 * (inclusive), softmax scale 1/sqrt(head_dim), GeGLU = GELU_erf(first half)
 * * second half, LayerNorm with biased variance and eps inside the root.
 */
typedef struct tee_config {
    int   n_layers;          /* 25 for the 310m shape                               */
    int   hidden;            /* H: 768; multiple of 128, <= 1024                     */
    int   n_heads;           /* 12; hidden == n_heads * head_dim                     */
    int   head_dim;          /* must be 64                                           */
    int   intermediate;      /* I: 3072 (GeGLU width); multiple of 128               */
    int   vocab;             /* V: 102400                                            */
    int   global_every;      /* 3: layer l is global iff l % global_every == 0       */
    int   window;            /* 64: one-sided, inclusive window of the other layers  */
    float rope_base_global;  /* 160000                                               */
    float rope_base_local;   /* 10000                                                */
    float ln_eps;            /* 1e-5                                                 */
    int   dtype;             /* TEE_F32 | TEE_BF16 | TEE_W8A8 | TEE_W6A8 | TEE_W4A8  */
    int   max_tokens;        /* capacity of one pass (sum of text lengths), >= 1     */
    int   max_texts;         /* capacity of one pass (number of texts), >= 1         */
    /* optional parts, 0 = off (the page's encoder) */
    int   emb_norm;          /* 1: bias-free LayerNorm (gain ln_emb) on the token embeddings  */
    int   final_norm;        /* 1: bias-free LayerNorm (gain ln_final) on the last layer's output,
                                before pooling or the per-token output                        */
    int   proj_dim;          /* 0, or P (a multiple of 128, <= 1024): the per-token output of
                                tee_encode_tokens is projected to P dimensions (w_proj)        */
} tee_config;

/*
 * fp32 host weights, row-major, tokens-as-rows convention y = x W^T.
 * Per-layer arrays are given as arrays of n_layers pointers.
 *   tok_emb  [V * H]
 *   ln_attn  [L][H]           gain of the attention-input LayerNorm
 *   wqkv     [L][3H * H]      output rows: q (head-major), then k, then v
 *   wo       [L][H * H]       input columns: concatenated heads
 *   ln_mlp   [L][H]           gain of the feed-forward-input LayerNorm
 *   wi       [L][2I * H]      output rows 0..I-1 = GELU input, I..2I-1 = gate
 *   wo_ffn   [L][H * I]
 */
typedef struct tee_weights {
    const float*        tok_emb;
    const float* const* ln_attn;
    const float* const* wqkv;
    const float* const* wo;
    const float* const* ln_mlp;
    const float* const* wi;
    const float* const* wo_ffn;
    const float*        ln_emb;     /* [H], read iff cfg.emb_norm (else may be NULL)       */
    const float*        ln_final;   /* [H], read iff cfg.final_norm (else may be NULL)     */
    const float*        w_proj;     /* [P * H], read iff cfg.proj_dim > 0 (else may be NULL);
                                       stored like the four projections of the dtype     */
} tee_weights;

typedef struct tee_ctx tee_ctx;

/*
 * Create a context on CUDA device `device`: validates cfg, allocates the
 * device workspace for max_tokens / max_texts and the RoPE tables.
 * On success *out receives the context.  Errors: TEE_EINVAL (cfg), TEE_ENOMEM,
 * TEE_ECUDA.  On failure *out is set to NULL.
 */
int tee_create(const tee_config* cfg, int device, tee_ctx** out);

/*
 * Copy the host weights to the device and convert them to the context's
 * storage format (fp32, bf16 round-to-nearest-even, or int8 blocks of 32
 * with one fp32 scale each for TEE_W8A8, 6-bit blocks of 32 packed four codes per
 * three bytes with one fp32 scale each for TEE_W6A8, 4-bit blocks of 32 packed two
 * codes per byte with one fp32 scale each for TEE_W4A8).  May be called again to replace
 * the weights.  Synchronous.  Errors: TEE_EINVAL (null pointers), TEE_ENOMEM,
 * TEE_ECUDA.
 */
int tee_load_weights(tee_ctx* ctx, const tee_weights* w);

/*
 * Encode a packed batch held in HOST memory, synchronously.
 *   token_ids   host int32[cu_seqlens[n_texts]]; each 0 <= id < vocab.  The
 *               caller wraps each text (BOS ... EOS) itself.
 *   cu_seqlens  host int32[n_texts + 1]; cu_seqlens[0] == 0, strictly
 *               increasing (empty texts are rejected: their mean is undefined).
 *   n_texts     >= 1, <= max_texts; cu_seqlens[n_texts] <= max_tokens.
 *   out         host float[n_texts * hidden]: unit-norm vectors in input order.
 * Copies inputs to the device, runs the pass on the context's stream, copies
 * the result back and synchronises that stream before returning.
 * Errors: TEE_EINVAL, TEE_ETOOLONG, TEE_ENOTLOADED, TEE_ECUDA.
 */
int tee_encode(tee_ctx* ctx, const int32_t* token_ids, const int32_t* cu_seqlens, int n_texts, float* out);

/*
 * Encode a packed batch held in DEVICE memory, asynchronously on `stream`
 * (a cudaStream_t; NULL = the legacy default stream).
 *   d_ids  device int32[total tokens]; d_cu device int32[n_texts + 1];
 *   h_cu   host copy of the same cu_seqlens (used for validation and launch
 *          sizing).  ids are not range-checked on the host on this path: the
 *          gather kernel turns an out-of-range id into a zero row and sets
 *          the context's device status word (tee_device_status, tee_ops.h);
 *   d_out  device float[n_texts * hidden], 16-byte aligned.
 * All device buffers must stay valid until the stream reaches the end of
 * the pass.  Errors: TEE_EINVAL (also for a NULL device pointer or a
 * misaligned d_out, before anything is launched), TEE_ETOOLONG,
 * TEE_ENOTLOADED, TEE_ECUDA.
 */
int tee_encode_device(tee_ctx* ctx, const int32_t* d_ids, const int32_t* d_cu, const int32_t* h_cu,
                      int n_texts, float* d_out, void* stream);

/*
 * Per-token (multi-vector) output.  Page "Les Embeddings multimodaux dans
 * Llama.cpp et GGUF" (jina.ai), section "Problèmes restants": multi-vector
 * embeddings are one linear layer over the token states.  For every token t
 * of the packed batch, in order: v_t = the final state (after the final norm
 * when cfg.final_norm), times w_proj^T when cfg.proj_dim > 0; the output is
 * v_t / max(|v_t|, 1e-12).  D = proj_dim if > 0, else hidden.
 *   tee_encode_tokens         host ids / cu_seqlens as tee_encode; out host
 *                             float[cu_seqlens[n_texts] * D]; synchronous.
 *                             The first call allocates a device buffer of
 *                             max_tokens * D floats, kept until tee_destroy.
 *   tee_encode_tokens_device  device ids / cu_seqlens (+ host cu_seqlens) as
 *                             tee_encode_device; d_out device float[T * D],
 *                             16-byte aligned; asynchronous on `stream`.
 * Errors as tee_encode / tee_encode_device; TEE_EINVAL for a misaligned d_out.
 */
int tee_encode_tokens(tee_ctx* ctx, const int32_t* token_ids, const int32_t* cu_seqlens, int n_texts, float* out);
int tee_encode_tokens_device(tee_ctx* ctx, const int32_t* d_ids, const int32_t* d_cu, const int32_t* h_cu,
                             int n_texts, float* d_out, void* stream);

/* Message of the last failure on this context ("" if none).  NULL ctx: the
 * message of the last failed context-free call in this process (tee_create,
 * tee_pool_l2_noalloc). */
const char* tee_last_error(const tee_ctx* ctx);

/* Release the context and all its device memory.  NULL-safe. */
void tee_destroy(tee_ctx* ctx);

/* ---- measurement -------------------------------------------------------- */

/* Kernel classes timed by the profiling hook. */
#define TEE_K_EMBED      0   /* token-embedding gather + per-token positions    */
#define TEE_K_LAYERNORM  1   /* both bias-free LayerNorms of every layer         */
#define TEE_K_GEMM       2   /* the four projections (QKV, out, Wi, Wo_ffn)      */
#define TEE_K_ATTENTION  3   /* varlen global / windowed attention               */
#define TEE_K_ELEMENTWISE 4  /* stand-alone RoPE / GeGLU (when not fused)        */
#define TEE_K_POOL       5   /* mean-pool + L2 normalisation                     */
#define TEE_K_QUANT      6   /* per-row 7-bit activation quantiser (W8A8)        */
#define TEE_K_COUNT      7

typedef struct tee_kernel_stat {
    int64_t launches;        /* launches of this class since the last reset       */
    double  total_ms;        /* sum of CUDA-event durations                       */
    double  flops;           /* algorithmic flops of those launches (GEMM, attn)  */
    double  bytes;           /* algorithmic HBM bytes of those launches           */
} tee_kernel_stat;

/*
 * Turn per-launch CUDA-event timing on (1) or off (0).  While on, every
 * kernel launch of an encode is bracketed by two events on the launching
 * stream; the durations are accumulated per kernel class by
 * tee_profile_read, which synchronises the pending events first.
 * Turning it on resets the counters.
 */
int tee_profile_enable(tee_ctx* ctx, int on);
int tee_profile_read(tee_ctx* ctx, tee_kernel_stat* stats /* [TEE_K_COUNT] */);

#ifdef __cplusplus
}
#endif
#endif /* TEE_H */
