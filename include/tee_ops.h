/*
 * tee_ops.h -- per-step entry points of the encoder pass (same library as tee.h).
 *
 * Each call runs ONE step of the pass on caller-provided DEVICE buffers,
 * asynchronously on `stream` (a cudaStream_t, NULL = legacy default stream),
 * using the weights already loaded into `ctx`.  They exist so each step can
 * be checked against the CPU oracle and timed on its own; tee_encode_device
 * runs exactly these steps in this order.
 *
 * Activation buffers use the context's activation type ACT:
 *   TEE_F32 and the integer-path (TEE_W8A8, TEE_W6A8, TEE_W4A8) contexts: float;
 *   TEE_BF16 contexts: bfloat16
 *   (uint16 bit patterns).  The residual stream x is always float.
 * Shapes: T = rows (tokens), H = hidden, I = intermediate, row-major.
 * Return codes as in tee.h.  Buffers are borrowed for the duration of the
 * stream work only.  Device buffers must be non-NULL and 16-byte aligned
 * (int32 arrays -- ids, cu_seqlens, positions, block sums -- 4-byte aligned,
 * activation scales 4-byte aligned); otherwise the call returns TEE_EINVAL
 * before launching anything.  A call with no rows (T or M == 0) launches
 * nothing and checks no device pointer.
 *
 * Steps (tensai page "テキスト埋め込み", §何が動くか):
 *   embed       x[t] = E[id[t]]                                   (token embedding)
 *   positions   pos[t] = t - cu[j] for t in text j                 (packing paragraph: positions restart per text)
 *   layernorm   y = (x - mean) / sqrt(var + eps) * gamma           (エンコーダ: bias-free LayerNorm)
 *   qkv         qkv = RoPE(y Wqkv^T)  (RoPE on q and k, base by layer)   (エンコーダ: RoPE attention)
 *   attention   o = softmax(q k^T / sqrt(d) + mask) v per head     (エンコーダ: whole text / +-64 window)
 *   out_proj    x += o Wo^T
 *   ffn_in      z = GELU(u[:, :I]) * u[:, I:],  u = y Wi^T         (エンコーダ: GeGLU feed-forward)
 *   ffn_out     x += z Wo_ffn^T
 *   pool_l2     out[j] = mean_{t in j} x[t] / || . ||              (プーリング)
 */
#ifndef TEE_OPS_H
#define TEE_OPS_H

#include <stdint.h>
#include "tee.h"

#ifdef __cplusplus
extern "C" {
#endif

#define TEE_LN_ATTN 0
#define TEE_LN_MLP  1

#define TEE_W_QKV    0
#define TEE_W_OUT    1
#define TEE_W_FFN_IN 2
#define TEE_W_FFN_OUT 3

/* x float[T*H] <- E[ids]; ids int32[T].  Out-of-range ids give a zero row and
 * set the context's device status (see tee_device_status). */
int tee_op_embed(tee_ctx* ctx, const int32_t* d_ids, int T, float* d_x, void* stream);

/* pos int32[T] from cu int32[n+1] (device) and its host copy h_cu. */
int tee_op_positions(tee_ctx* ctx, const int32_t* d_cu, const int32_t* h_cu, int n_texts, int32_t* d_pos,
                     void* stream);

/* y ACT[T*H] = LayerNorm(x float[T*H]) with the gain of (layer, which). */
int tee_op_layernorm(tee_ctx* ctx, int layer, int which, const float* d_x, void* d_y, int T, void* stream);

/* qkv ACT[T*3H] = y Wqkv^T with RoPE applied to the q and k thirds;
 * pos int32[T] are the per-text positions. */
int tee_op_qkv(tee_ctx* ctx, int layer, const void* d_y, const int32_t* d_pos, void* d_qkv, int T, void* stream);

/* o ACT[T*H] = varlen attention of layer `layer` over qkv ACT[T*3H]
 * (global if layer % global_every == 0, else the window); texts given by
 * cu (device) and h_cu (host copy). */
int tee_op_attention(tee_ctx* ctx, int layer, const void* d_qkv, const int32_t* d_cu, const int32_t* h_cu,
                     int n_texts, void* d_o, void* stream);

/* x float[T*H] += o ACT[T*H] Wo^T */
int tee_op_out_proj(tee_ctx* ctx, int layer, const void* d_o, float* d_x, int T, void* stream);

/* z ACT[T*I] = GeGLU(y ACT[T*H] Wi^T) */
int tee_op_ffn_in(tee_ctx* ctx, int layer, const void* d_y, void* d_z, int T, void* stream);

/* x float[T*H] += z ACT[T*I] Wo_ffn^T */
int tee_op_ffn_out(tee_ctx* ctx, int layer, const void* d_z, float* d_x, int T, void* stream);

/* Generic bf16 projection on the tensor cores: C = A W^T with A bf16[M*K],
 * W bf16[N*K] (both K-contiguous), fp32 accumulation; epilogue 0 stores C as
 * bf16[M*N], epilogue 1 adds it into float C[M*N].  N a multiple of 128, K a
 * multiple of 64, pointers 16-byte aligned.  TEE_BF16 contexts only (the
 * context supplies the device and the status word).  It is the kernel the
 * pass uses for its four projections, exposed for shape tests and timing. */
int tee_op_gemm_bf16(tee_ctx* ctx, const void* d_a, const void* d_w, void* d_c, int M, int N, int K, int epilogue,
                     void* stream);

/* out float[n*H] = L2-normalised per-text mean of x float[T*H]; d_x and d_out
 * 16-byte aligned (else TEE_EINVAL). */
int tee_op_pool_l2(tee_ctx* ctx, const float* d_x, const int32_t* d_cu, const int32_t* h_cu, int n_texts,
                   float* d_out, void* stream);

/*
 * Allocation-free mean-pool + L2 normalisation.  The page has no counterpart:
 * this entry point exists for callers that cannot allocate device memory --
 * code running inside a host framework that owns all device memory through
 * its own pool and forbids raw cudaMalloc, or a latency-critical path that
 * cannot afford the implicit synchronisation of an allocation.  It needs no
 * context and calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * Computes the same result as tee_op_pool_l2 (per-text mean, scaled to unit
 * length) with the same chunked sums, in two launches:
 *   d_x    device float[T * hidden], T = h_cu[n_texts], 16-byte aligned;
 *   d_cu   device int32[n_texts + 1], 4-byte aligned;  h_cu: host copy of the
 *          same array (validated, and used to size the launch).  The two must
 *          hold the same values; the kernels clamp every row and chunk index
 *          to the sizes taken from h_cu, so a disagreeing d_cu gives wrong
 *          vectors but no access outside d_x or the scratch;
 *   d_out  device float[n_texts * hidden], 16-byte aligned;  async on `stream`.
 * A NULL or misaligned pointer returns TEE_EINVAL before anything is launched.
 * Its scratch (chunk offsets and the partial sums of 64-row chunks) lives in
 * file-scope device arrays of fixed size that every GPU loading the library
 * holds until the process exits (about 4 MiB).  Limits: n_texts <=
 * TEE_POOL_NOALLOC_MAX_TEXTS, sum_j ceil(len_j / 64) * hidden <=
 * TEE_POOL_NOALLOC_MAX_PARTIAL, hidden a multiple of 4 in [4, 1024]; larger
 * inputs return TEE_ETOOLONG / TEE_EINVAL with a message in
 * tee_last_error(NULL).  Every call on a device shares the same scratch and
 * overwrites all of it that it reads, so calls that overlap on the GPU (for
 * instance on two streams) race.  The first call on a device looks up the
 * arrays' device addresses (cudaGetSymbolAddress) with that device current
 * and keeps them for the life of the process; make that first call before any
 * stream capture, and do not call this entry point on a device after a
 * cudaDeviceReset of that device (the arrays are reloaded at new addresses).
 */
#define TEE_POOL_NOALLOC_MAX_TEXTS   8192
#define TEE_POOL_NOALLOC_MAX_PARTIAL 1048576   /* floats */
int tee_pool_l2_noalloc(const float* d_x, const int32_t* d_cu, const int32_t* h_cu, int n_texts, int hidden,
                        float* d_out, void* stream);

/* ---- integer-path pieces (TEE_W8A8, TEE_W6A8 and TEE_W4A8 contexts) ------ */

/* Per-row 7-bit quantiser: s[m] = max|x[m,:]| / 63 (IEEE fp32 division),
 * q = clamp(rint(x / s), -63, 63) (ties to even); zero rows give s = 0, q = 0.
 * x float[M*K] -> q int8[M*K], s float[M]. */
int tee_op_quant_rows7(tee_ctx* ctx, const float* d_x, int M, int K, int8_t* d_q, float* d_s, void* stream);

/* Exact integer block sums I[m, n, b] = sum_{k in block b} q[m,k] * Wq[n,k]
 * (blocks of 32 along K) for projection `which` of `layer`:
 * q int8[M*K] -> partials int32[M*N*(K/32)], laid out [m][n][b]. */
int tee_op_w8a8_partials(tee_ctx* ctx, int layer, int which, const int8_t* d_q, int M, int32_t* d_partials,
                         void* stream);

/* Copy the weight codes of projection `which` of `layer`, widened to int8[N*K]
 * (the 6- and 4-bit codes of TEE_W6A8 / TEE_W4A8 contexts unpacked), and the block scales
 * float[N*K/32] to host buffers.  Synchronous. */
int tee_weight_codes(tee_ctx* ctx, int layer, int which, int8_t* h_q, float* h_d);

/* Failure-detection self-test.  Launches one thread that waits, with the same
 * bounded mbarrier wait the tensor-core GEMM and attention pipelines use, on a
 * barrier that nothing completes, and gives up after `wait_cycles` SM clock
 * cycles (clamped to [1e3, 1e10]).  The expiry sets the timeout bit of the
 * context's status word, as a stalled pipeline would, so the next
 * tee_device_status() returns TEE_ETIMEOUT (and clears it).  The kernel
 * returns once the limit expires; the context stays usable.  Asynchronous on
 * `stream`. */
int tee_selftest_wait_timeout(tee_ctx* ctx, long long wait_cycles, void* stream);

/* GELU self-test.  y[i] = GELU(a[i]) = a * Phi(a), evaluated exactly as the
 * GeGLU epilogue of the bf16 tensor-core feed-forward projection does it (erf
 * by the rational approximation of Abramowitz & Stegun formula 7.1.26 on the
 * hardware reciprocal and exp2), so that this restatement of erf can be checked
 * against an exact GELU over a dense range.  (tensai page, §何が動くか /
 * エンコーダ: the feed-forward is GeGLU; reading: the erf form of GELU.)
 * d_a, d_y: device float[n], 4-byte aligned; context-free, on the current
 * device, asynchronous on `stream`.  Errors: TEE_EINVAL (NULL, misaligned,
 * n < 0; message in tee_last_error(NULL)), TEE_ECUDA. */
int tee_selftest_gelu(const float* d_a, float* d_y, long long n, void* stream);

/* ---- host-only planning (no device, no context) -------------------------
 * The decisions a pass takes on the host before it launches, exported so that
 * they can be checked without a GPU.  Errors return a negative TEE_E* code with
 * a message in tee_last_error(NULL). */

/* Attention work items, as the pass lists them for the varlen attention
 * kernel (packing paragraph of §何が動くか: attention stays inside each text;
 * §エンコーダ: the whole text on global layers, +-window tokens otherwise), each
 * {q_start, q_len, k_lo, k_hi}: a tile of up to 128 queries and the key range
 * [k_lo, k_hi) that any of its queries may see.
 *   is_global != 0: a text longer than 128 tokens gives one item per
 *     128-query tile -- q_start = cu[j] + 128 i, q_len = min(128, cu[j+1] -
 *     q_start), [k_lo, k_hi) = [cu[j], cu[j+1]); texts of at most 128 tokens
 *     are taken in text order and grouped greedily, each group the longest run
 *     of consecutive such texts spanning at most 128 tokens, one item per group
 *     with q_start = k_lo = its first token, k_hi = its end, q_len = k_hi -
 *     k_lo.  Ordered by q_len * (k_hi - k_lo), largest first, ties in text
 *     order.  (Where texts share an item, the kernel masks each row to its
 *     own text.)
 *   is_global == 0: one item per 128-query tile of the packed sequence itself
 *     (q_start = 128 i, q_len = min(128, T - q_start), T = cu[n_texts]), tiles
 *     shared by consecutive texts; k_lo = max(start of the text holding row
 *     q_start, q_start - window), k_hi = min(end of the text holding row
 *     q_start + q_len - 1, q_start + q_len + window); in sequence order.  (The
 *     kernel masks each row to its own text.)
 * h_cu host int32[n_texts + 1] (cu[0] == 0, strictly increasing).  items: host
 * int32[4 * max_items], or NULL to ask for the count only.  Returns the number
 * of items (TEE_ETOOLONG if it exceeds max_items). */
int tee_plan_attention(const int32_t* h_cu, int n_texts, int window, int is_global, int32_t* items, int max_items);

/* How the attention kernel's `grid` persistent CTAs share the units (item,
 * head) of a list of n_items work items (as tee_plan_attention gives them) and
 * n_heads heads.  Units are taken in order of decreasing work -- work = 2 x
 * ceil((k_hi - k_lo) / 128) + 1 -- ties in unit order (item by item, heads in
 * order), and each goes to the CTA with the least work so far, ties to the
 * lower CTA index.  slots: host int32[4 * n_items * n_heads], each CTA's units
 * in the order it takes them, CTA 0 first, each as {q_start, q_len | head <<
 * 16, k_lo, k_hi}; slot_off: host int32[grid + 1], CTA c holding slots
 * slot_off[c] .. slot_off[c + 1].  Requires 1 <= n_heads <= 32767, 1 <= grid
 * <= 1024 and items with 0 <= q_len <= 65535 and k_lo <= k_hi.  Returns
 * n_items * n_heads, TEE_EINVAL, or TEE_ETOOLONG past 2^29 units. */
int tee_plan_attention_schedule(const int32_t* items, int n_items, int n_heads, int grid, int32_t* slots,
                                int32_t* slot_off);

/* Tile shape of the bf16 tensor-core projection C[M, N] = A[M, K] W^T: *bn =
 * tile width in columns (128, 192 or 256), *pair = 1 when 2-CTA clusters
 * compute 256-row tiles, 0 for one CTA per 128-row tile, as the library
 * chooses it on a GPU with num_sms SMs.  epi: 0 bf16 store, 1 fp32 residual
 * add, 2 QKV with RoPE, 3 GeGLU (N % 256 == 0).  M >= 1, N % 128 == 0,
 * K % 64 == 0, num_sms >= 2. */
int tee_plan_gemm(int M, int N, int K, int epi, int num_sms, int* bn, int* pair);

/* Synchronise the context's device status word: TEE_OK, or TEE_EINVAL if a
 * kernel met an out-of-range token id since the last call (the word is then
 * cleared), or TEE_ETIMEOUT if a bounded device wait gave up. */
int tee_device_status(tee_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* TEE_OPS_H */
