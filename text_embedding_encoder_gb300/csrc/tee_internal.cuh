// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <string>
#include <vector>

#include "tee.h"
#include "tee_ops.h"

typedef __nv_bfloat16 bf16;

// Device status word bits (ctx->d_status).
#define TEE_STATUS_BAD_ID   1u
#define TEE_STATUS_TIMEOUT  2u

struct LayerWeights {
    float* ln_attn = nullptr;      // fp32 [H]
    float* ln_mlp = nullptr;       // fp32 [H]
    void* w[4] = {nullptr, nullptr, nullptr, nullptr};      // fp32 / bf16 / int8, [N*K]
    float* wd[4] = {nullptr, nullptr, nullptr, nullptr};    // W8A8 block scales [N*K/32]
};

struct ProfileSlot {
    cudaEvent_t start, stop;
    int kclass;
    double flops, bytes;
};

struct tee_ctx {
    tee_config cfg{};
    int device = 0;
    bool loaded = false;
    std::string err;

    // weights
    void* weight_arena = nullptr;
    size_t weight_bytes = 0;
    void* emb = nullptr;                // fp32 [V*H] (F32, W8A8) or bf16 (BF16)
    std::vector<LayerWeights> layers;
    float* ln_emb = nullptr;            // optional embedding-norm gain, fp32 [H]
    float* ln_final = nullptr;          // optional final-norm gain, fp32 [H]
    void* w_proj = nullptr;             // optional per-token projection [P*H] (stored like the projections)
    float* w_proj_d = nullptr;          // its W8A8 block scales [P*H/32]
    float* tok_out = nullptr;           // per-token output of tee_encode_tokens, float [max_tokens*D] (lazy)

    // RoPE tables, index 0 = global base, 1 = window base: float [max_tokens][head_dim/2]
    float* rope_cos[2] = {nullptr, nullptr};
    float* rope_sin[2] = {nullptr, nullptr};

    // workspace (sized by max_tokens / max_texts)
    void* ws_arena = nullptr;
    size_t ws_bytes = 0;
    int32_t* d_ids = nullptr;
    int32_t* d_cu = nullptr;
    int32_t* d_pos = nullptr;
    int2* d_rowtb = nullptr;                  // per token: {first token, one past the last} of its text
    float* x = nullptr;                 // residual stream, float [T*H]
    void* y = nullptr;                  // LayerNorm output, ACT [T*H]
    void* qkv = nullptr;                // ACT [T*3H]
    void* o = nullptr;                  // attention output, ACT [T*H]
    void* u = nullptr;                  // Wi output, ACT [T*2I] (unfused GeGLU only)
    void* z = nullptr;                  // GeGLU output, ACT [T*I]
    float* out = nullptr;               // float [max_texts*H]
    int8_t* qa = nullptr;               // W8A8 activation codes [T*max(H,I)]
    float* qs = nullptr;                // W8A8 activation scales [T]
    unsigned int* d_status = nullptr;   // device status word
    int4* d_slots[2] = {nullptr, nullptr};        // attention units per CTA (global, window layers)
    int32_t* d_slot_off[2] = {nullptr, nullptr};  // each CTA's first slot [grid + 1]
    int32_t* d_chunk_off = nullptr;     // pool: first chunk of each text [max_texts + 1]
    float* pool_partial = nullptr;      // pool: partial sums [max_chunks * H]
    unsigned int* pool_counters = nullptr;   // pool: chunks finished per text [max_texts], zero between launches
    int max_chunks = 0;
    std::vector<int32_t> h_chunk_off;
    int max_items = 0;
    std::vector<int4> h_items[2];
    std::vector<int4> h_slots[2];
    std::vector<int32_t> h_slot_off[2];
    int attn_grid[2] = {0, 0};

    cudaStream_t stream = nullptr;      // the context's own stream (tee_encode)
    std::vector<int32_t> h_cu_scratch;

    // profiling
    bool profiling = false;
    std::vector<ProfileSlot> prof_slots;
    size_t prof_used = 0;
    tee_kernel_stat prof_acc[TEE_K_COUNT];
};

// ---- programmatic dependent launch -----------------------------------------
// The pass's kernels are launched with programmatic stream serialization: a
// kernel may start (and run its prologue: barrier init, TMEM allocation) while
// the previous kernel in the stream finishes.  Every such kernel calls
// pdl_wait() before it touches global memory: it returns once the previous
// kernel has completed and its writes are visible, and since that kernel did
// the same, every earlier kernel has completed too.  pdl_trigger() lets the
// next kernel launch once every block of this one has started.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---- helpers ------------------------------------------------------------
inline bool act_is_bf16(const tee_ctx* c) { return c->cfg.dtype == TEE_BF16; }
// the integer paths: int8 (W8A8), packed 6-bit (W6A8) or packed 4-bit (W4A8)
// weight blocks, 7-bit activations
inline bool is_int_path(const tee_config& g) {
    return g.dtype == TEE_W8A8 || g.dtype == TEE_W6A8 || g.dtype == TEE_W4A8;
}
// width in bits of the integer path's weight codes
inline int weight_bits(const tee_config& g) { return g.dtype == TEE_W4A8 ? 4 : (g.dtype == TEE_W6A8 ? 6 : 8); }
inline size_t act_size(const tee_ctx* c) { return act_is_bf16(c) ? 2 : 4; }
inline int layer_is_global(const tee_ctx* c, int l) { return (l % c->cfg.global_every) == 0; }

// Record the message returned by tee_last_error(NULL) for context-free calls; returns `code`.
int tee_set_global_error(int code, const char* msg);

// One process may drive several devices (one context each), so everything the
// launchers cache about a device -- its SM count, the kernels' shared-memory
// attributes, occupancy-derived grid sizes -- is kept per device index, under
// a lock.  Device indices must be below TEE_MAX_DEVICES.
#define TEE_MAX_DEVICES 64
// Upper bound of the attention kernel's grid (one CTA per SM).
#define TEE_ATTN_MAX_GRID 1024
// The current device's index and SM count (looked up once per device).
cudaError_t tee_current_device(int* dev, int* num_sms);

// Profiling brackets: record events around one launch when profiling is on.
int prof_begin(tee_ctx* c, cudaStream_t s, int kclass, double flops, double bytes);
void prof_end(tee_ctx* c, cudaStream_t s, int slot);

// ---- kernel launchers (each returns cudaGetLastError()) -------------------
cudaError_t launch_convert_f32_bf16(const float* src, bf16* dst, size_t n, cudaStream_t s);
cudaError_t launch_embed(const void* emb, bool emb_bf16, const int32_t* ids, int T, int H, int V, float* x,
                         unsigned int* status, cudaStream_t s);
// pos[t] = t - cu[text(t)]; with row_tb non-NULL also row_tb[t] = {cu[text(t)], cu[text(t) + 1]}.
cudaError_t launch_positions(const int32_t* cu, int n_texts, int T, int32_t* pos, int2* row_tb, cudaStream_t s);
cudaError_t launch_layernorm(const float* x, const float* gamma, void* y, bool y_bf16, int T, int H, float eps,
                             cudaStream_t s);
cudaError_t launch_rope(void* qkv, bool bf16_act, const int32_t* pos, const float* cos_t, const float* sin_t, int T,
                        int H, int n_heads, cudaStream_t s);
cudaError_t launch_geglu(const void* u, void* z, bool bf16_act, int T, int I, cudaStream_t s);
// Mean-pool + L2 in two passes: partial column sums of POOL_CHUNK-row chunks
// (chunk_off[j] = first chunk of text j, device int32[n+1]) into `partial`
// (float [n_chunks * H]), then per text the ordered sum, mean and scaling.
#define POOL_CHUNK 64
#define POOL_CHUNK_FUSED 64   // rows per block of the single-launch pool (launch_pool_l2_fused)
cudaError_t launch_pool_l2(const float* x, const int32_t* cu, const int32_t* chunk_off, int n_texts, int n_chunks, int T,
                           int H, float* partial, float* out, cudaStream_t s);
// The same in one launch: the last chunk of each text to finish combines that
// text's partials; counters (unsigned [n_texts], all zero) are left zero.
cudaError_t launch_pool_l2_fused(const float* x, const int32_t* cu, const int32_t* chunk_off, int n_texts,
                                 int n_chunks, int H, float* partial, unsigned int* counters, float* out,
                                 cudaStream_t s);
// Scale each row of x [M, D] (D a multiple of 4, <= 1024) to unit length in place
// (norm floored at 1e-12).
cudaError_t launch_l2_rows(float* x, int M, int D, cudaStream_t s);
cudaError_t launch_attention_simple(const void* qkv, bool bf16_act, const int32_t* cu, int n_texts, int T, int H,
                                    int n_heads, bool is_global, int window, void* o, cudaStream_t s);

// tcgen05 varlen attention over bf16 qkv [T, 3H]: `grid` persistent CTAs, CTA c
// taking slots d_slot_off[c] .. d_slot_off[c + 1] of d_slots, each a work item
// {q_start, q_len | head << 16, k_lo, k_hi} -- a tile of up to 128 queries of
// one head and the keys it may see (global layers: one text, or consecutive
// short texts; window layers: a tile of the packed sequence) -- with each
// row's text bounds in row_tb.
cudaError_t launch_attention_tc(const void* qkv, int T, int H, int n_heads, const int4* d_slots,
                                const int32_t* d_slot_off, int grid, bool is_global, int window, const int2* row_tb,
                                void* o, unsigned int* status, cudaStream_t s);

// Self-test of the bounded waits: a wait on a barrier nothing completes, limited
// to `limit_cycles`; its expiry sets TEE_STATUS_TIMEOUT in `status`.
cudaError_t launch_selftest_wait(long long limit_cycles, unsigned int* status, cudaStream_t s);

// SIMT GEMM, C = A W^T.  epi 0: store C in A's type; epi 1: add into float C.
cudaError_t launch_gemm_simt(const void* A, const void* W, void* C, bool bf16_in, int M, int N, int K, int epi,
                             cudaStream_t s);

// Integer paths.  wbits = weight code width: 8 (int8 codes, L = 127), 6 (L = 31,
// four codes per three bytes) or 4 (L = 7, two codes per byte).
cudaError_t launch_quant_weight_blocks(const float* w, int8_t* q, float* d, int N, int K, int wbits, cudaStream_t s);
cudaError_t launch_quant_rows7(const float* x, int M, int K, int8_t* q, float* scale, cudaStream_t s);
// y = s_m * sum_b d[n,b] * I[m,n,b]; epi 0 store float, 1 add into float; partials (optional) int32 [M][N][K/32]
cudaError_t launch_gemm_w8a8(const int8_t* qa, const float* sa, const int8_t* qw, const float* dw, float* C,
                             int32_t* partials, int M, int N, int K, int epi, int wbits, cudaStream_t s);
