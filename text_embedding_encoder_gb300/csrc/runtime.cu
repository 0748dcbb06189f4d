// C ABI runtime: context, weight ingestion, workspace, validation, the launch
// sequence of one encoder pass, per-step entry points and the profiling hook.
//
// The pass follows the tensai page "テキスト埋め込み", §何が動くか: token
// embedding; per layer a bias-free LayerNorm, QKV projection with RoPE
// (positions restart per text), attention confined to each text (whole text
// on layer 0 and every third layer, +-64 tokens otherwise), the output
// projection with the residual, a second bias-free LayerNorm and the GeGLU
// feed-forward with the residual; finally the per-text mean and L2 scaling.
#include "tee_internal.cuh"
#include "gemm_tc.cuh"

#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <initializer_list>
#include <mutex>
#include <new>

namespace {

std::string g_create_error;

int fail(tee_ctx* c, int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    if (c) c->err = buf; else g_create_error = buf;
    return code;
}

int cuda_fail(tee_ctx* c, cudaError_t e, const char* what) {
    return fail(c, e == cudaErrorMemoryAllocation ? TEE_ENOMEM : TEE_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define CK(call)                                                   \
    do {                                                           \
        cudaError_t _e = (call);                                   \
        if (_e != cudaSuccess) return cuda_fail(ctx, _e, #call);   \
    } while (0)

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Sub-allocator over one device allocation (offsets aligned to 256 bytes).
struct Carve {
    char* base;
    size_t off = 0;
    explicit Carve(void* b) : base((char*)b) {}
    template <typename T>
    T* take(size_t count, size_t elem = sizeof(T)) {
        T* p = (T*)(base ? base + off : nullptr);
        off = align_up(off + count * elem, 256);
        return p;
    }
};

int wshape(const tee_config& c, int which, int* N, int* K) {
    const int H = c.hidden, I = c.intermediate;
    switch (which) {
        case TEE_W_QKV: *N = 3 * H; *K = H; return 0;
        case TEE_W_OUT: *N = H; *K = H; return 0;
        case TEE_W_FFN_IN: *N = 2 * I; *K = H; return 0;
        case TEE_W_FFN_OUT: *N = H; *K = I; return 0;
    }
    return -1;
}

int validate_config(const tee_config* c) {
    if (!c) return fail(nullptr, TEE_EINVAL, "config is NULL");
    if (c->n_layers < 1) return fail(nullptr, TEE_EINVAL, "n_layers must be >= 1");
    if (c->head_dim != 64) return fail(nullptr, TEE_EINVAL, "head_dim must be 64");
    if (c->n_heads < 1 || c->hidden != c->n_heads * c->head_dim)
        return fail(nullptr, TEE_EINVAL, "hidden must equal n_heads * head_dim");
    if (c->hidden % 128 || c->hidden > 1024) return fail(nullptr, TEE_EINVAL, "hidden must be a multiple of 128, <= 1024");
    if (c->intermediate < 128 || c->intermediate % 128) return fail(nullptr, TEE_EINVAL, "intermediate must be a multiple of 128");
    if (c->vocab < 1) return fail(nullptr, TEE_EINVAL, "vocab must be >= 1");
    if (c->global_every < 1) return fail(nullptr, TEE_EINVAL, "global_every must be >= 1");
    if (c->window < 0) return fail(nullptr, TEE_EINVAL, "window must be >= 0");
    if (!(c->rope_base_global > 0.f) || !(c->rope_base_local > 0.f)) return fail(nullptr, TEE_EINVAL, "RoPE bases must be > 0");
    if (!(c->ln_eps >= 0.f)) return fail(nullptr, TEE_EINVAL, "ln_eps must be >= 0");
    if (c->dtype != TEE_F32 && c->dtype != TEE_BF16 && c->dtype != TEE_W8A8 && c->dtype != TEE_W4A8 &&
        c->dtype != TEE_W6A8)
        return fail(nullptr, TEE_EINVAL, "unknown dtype");
    if (c->max_tokens < 1 || c->max_texts < 1) return fail(nullptr, TEE_EINVAL, "max_tokens and max_texts must be >= 1");
    if (c->max_tokens > (1 << 24)) return fail(nullptr, TEE_EINVAL, "max_tokens must be <= 2^24");
    if ((c->emb_norm != 0 && c->emb_norm != 1) || (c->final_norm != 0 && c->final_norm != 1))
        return fail(nullptr, TEE_EINVAL, "emb_norm and final_norm must be 0 or 1");
    if (c->proj_dim < 0 || c->proj_dim % 128 || c->proj_dim > 1024)
        return fail(nullptr, TEE_EINVAL, "proj_dim must be 0 or a multiple of 128, <= 1024");
    return TEE_OK;
}

// Workspace layout (also used to size the allocation: base == nullptr).
size_t carve_workspace(tee_ctx* c, void* base) {
    const tee_config& g = c->cfg;
    const size_t T = g.max_tokens, H = g.hidden, I = g.intermediate, A = act_size(c);
    Carve cv(base);
    c->d_ids = cv.take<int32_t>(T);
    c->d_cu = cv.take<int32_t>(g.max_texts + 1);
    c->d_pos = cv.take<int32_t>(T);
    c->d_rowtb = cv.take<int2>(T);
    c->x = cv.take<float>(T * H);
    c->y = cv.take<char>(T * H, A);
    c->qkv = cv.take<char>(T * 3 * H, A);
    c->o = cv.take<char>(T * H, A);
    c->u = cv.take<char>(T * 2 * I, A);
    c->z = cv.take<char>(T * I, A);
    c->out = cv.take<float>((size_t)g.max_texts * H);
    if (is_int_path(g)) {
        c->qa = cv.take<int8_t>(T * std::max(H, I));
        c->qs = cv.take<float>(T);
    } else {
        c->qa = nullptr;
        c->qs = nullptr;
    }
    for (int b = 0; b < 2; ++b) {
        c->rope_cos[b] = cv.take<float>(T * 32);
        c->rope_sin[b] = cv.take<float>(T * 32);
    }
    c->d_status = cv.take<unsigned int>(4);
    c->max_items = (int)(T / 128 + g.max_texts + 1);   // bounds both lists
    for (int b = 0; b < 2; ++b) {
        c->d_slots[b] = cv.take<int4>((size_t)c->max_items * g.n_heads);
        c->d_slot_off[b] = cv.take<int32_t>(TEE_ATTN_MAX_GRID + 1);
    }
    c->max_chunks = (int)(T / POOL_CHUNK_FUSED + g.max_texts + 1);
    c->d_chunk_off = cv.take<int32_t>(g.max_texts + 1);
    c->pool_partial = cv.take<float>((size_t)c->max_chunks * H);
    c->pool_counters = cv.take<unsigned int>(g.max_texts);
    return cv.off;
}

// Per-layer weight layout inside the weight arena.
size_t carve_weights(tee_ctx* c, void* base) {
    const tee_config& g = c->cfg;
    const size_t H = g.hidden;
    Carve cv(base);
    const size_t esz = g.dtype == TEE_BF16 ? 2 : (g.dtype == TEE_F32 ? 4 : 1);
    // bytes of an [N, K] projection: packed 4-bit codes take half a byte per
    // weight, packed 6-bit codes three quarters
    auto wbytes = [&](size_t n_k) {
        return g.dtype == TEE_W4A8 ? n_k / 2 : (g.dtype == TEE_W6A8 ? n_k / 4 * 3 : n_k * esz);
    };
    c->emb = cv.take<char>((size_t)g.vocab * H, g.dtype == TEE_BF16 ? 2 : 4);
    c->layers.assign(g.n_layers, LayerWeights{});
    for (int l = 0; l < g.n_layers; ++l) {
        LayerWeights& L = c->layers[l];
        L.ln_attn = cv.take<float>(H);
        L.ln_mlp = cv.take<float>(H);
        for (int w = 0; w < 4; ++w) {
            int N, K;
            wshape(g, w, &N, &K);
            L.w[w] = cv.take<char>(wbytes((size_t)N * K));
            L.wd[w] = is_int_path(g) ? cv.take<float>((size_t)N * K / 32) : nullptr;
        }
    }
    c->ln_emb = g.emb_norm ? cv.take<float>(H) : nullptr;
    c->ln_final = g.final_norm ? cv.take<float>(H) : nullptr;
    c->w_proj = g.proj_dim ? cv.take<char>(wbytes((size_t)g.proj_dim * H)) : nullptr;
    c->w_proj_d = g.proj_dim && is_int_path(g) ? cv.take<float>((size_t)g.proj_dim * H / 32) : nullptr;
    return cv.off;
}

// RoPE cos/sin tables for positions 0..max_tokens-1 (fp64 angles, fp32 storage).
int build_rope_tables(tee_ctx* ctx) {
    const tee_config& g = ctx->cfg;
    const size_t T = g.max_tokens;
    std::vector<float> cs(T * 32), sn(T * 32);
    for (int b = 0; b < 2; ++b) {
        const double base = b == 0 ? g.rope_base_global : g.rope_base_local;
        double inv_freq[32];
        for (int j = 0; j < 32; ++j) inv_freq[j] = pow(base, -2.0 * j / 64.0);
        for (size_t p = 0; p < T; ++p)
            for (int j = 0; j < 32; ++j) {
                const double a = (double)p * inv_freq[j];
                cs[p * 32 + j] = (float)cos(a);
                sn[p * 32 + j] = (float)sin(a);
            }
        CK(cudaMemcpy(ctx->rope_cos[b], cs.data(), T * 32 * sizeof(float), cudaMemcpyHostToDevice));
        CK(cudaMemcpy(ctx->rope_sin[b], sn.data(), T * 32 * sizeof(float), cudaMemcpyHostToDevice));
    }
    return TEE_OK;
}

// Validate a host cu_seqlens array; returns total tokens via *T.
int check_cu(tee_ctx* ctx, const int32_t* h_cu, int n_texts, int* T) {
    if (!h_cu) return fail(ctx, TEE_EINVAL, "cu_seqlens is NULL");
    if (n_texts < 1) return fail(ctx, TEE_EINVAL, "n_texts must be >= 1 (got %d)", n_texts);
    if (n_texts > ctx->cfg.max_texts) return fail(ctx, TEE_ETOOLONG, "n_texts %d > max_texts %d", n_texts, ctx->cfg.max_texts);
    if (h_cu[0] != 0) return fail(ctx, TEE_EINVAL, "cu_seqlens[0] must be 0 (got %d)", h_cu[0]);
    for (int j = 0; j < n_texts; ++j)
        if (h_cu[j + 1] <= h_cu[j])
            return fail(ctx, TEE_EINVAL, "cu_seqlens must be strictly increasing (text %d is empty or negative)", j);
    if (h_cu[n_texts] > ctx->cfg.max_tokens)
        return fail(ctx, TEE_ETOOLONG, "total tokens %d > max_tokens %d", h_cu[n_texts], ctx->cfg.max_tokens);
    *T = h_cu[n_texts];
    return TEE_OK;
}

// Algorithmic attention work: (query, allowed key) pairs summed over texts.
double attention_pairs(const int32_t* h_cu, int n_texts, bool is_global, int w) {
    double pairs = 0;
    for (int j = 0; j < n_texts; ++j) {
        const long long L = h_cu[j + 1] - h_cu[j];
        if (is_global) {
            pairs += (double)L * (double)L;
            continue;
        }
        for (long long i = 0; i < L; ++i) pairs += (double)(std::min(L - 1, i + w) - std::max(0LL, i - w) + 1);
    }
    return pairs;
}

// Attention work items of one pass, each a 128-query tile with the key range
// its queries may see.  List 0 (global layers): the tiles of each text (keys =
// the text), consecutive texts that together span at most 128 tokens sharing
// one tile (keys = their span), the most work (queries x keys) first.  List 1 (window
// layers): the tiles of the packed sequence itself, ignoring text boundaries,
// so short texts share tiles instead of padding one each; a tile's key range
// runs from the first key its first row may see (the window clipped to that
// row's text) to the last key its last row may see, and each row is masked to
// its own text in the kernel.
void plan_attention_items(const int32_t* h_cu, int n_texts, int w, std::vector<int4> (&items)[2]) {
    for (int b = 0; b < 2; ++b) items[b].clear();
    // global layers: a text's 128-query tiles, keys = the text; consecutive
    // texts that together span at most 128 tokens share one tile (keys = their
    // span; the kernel masks each row to its own text)
    for (int j = 0; j < n_texts;) {
        const int s0 = h_cu[j], s1 = h_cu[j + 1];
        if (s1 - s0 <= 128) {
            int k = j + 1;
            while (k < n_texts && h_cu[k + 1] - s0 <= 128) ++k;
            items[0].push_back(make_int4(s0, h_cu[k] - s0, s0, h_cu[k]));
            j = k;
            continue;
        }
        for (int q0 = s0; q0 < s1; q0 += 128) items[0].push_back(make_int4(q0, std::min(128, s1 - q0), s0, s1));
        ++j;
    }
    std::stable_sort(items[0].begin(), items[0].end(), [](const int4& a, const int4& b) {
        const long long ca = (long long)a.y * (a.w - a.z), cb = (long long)b.y * (b.w - b.z);
        return ca > cb;
    });
    const int T = h_cu[n_texts];
    int j0 = 0, j1 = 0;   // texts holding the tile's first and last rows
    for (int q0 = 0; q0 < T; q0 += 128) {
        const int ql = std::min(128, T - q0);
        while (h_cu[j0 + 1] <= q0) ++j0;
        while (h_cu[j1 + 1] <= q0 + ql - 1) ++j1;
        items[1].push_back(make_int4(q0, ql, std::max(h_cu[j0], q0 - w), std::min(h_cu[j1 + 1], q0 + ql + w)));
    }
}

// The attention kernel's persistent CTAs over (item, head) units.  Units are
// taken in order of decreasing work (stable: item order, then head) and each
// goes to the CTA with the least work so far, ties to the lower index (longest
// processing time first); a unit's work is counted as 2 x its 128-key tiles +
// 1 (a tile, and the per-unit output pass at about half a tile).  slots gets
// each CTA's units in the order it takes them, CTA after CTA, as the item with
// y = q_len | head << 16; off[c] .. off[c + 1] are CTA c's slots.
//
// The least-loaded CTA comes from a bucket queue: loads are integers, the least
// load never falls, and no load is more than the largest unit's work above it,
// so a ring of (largest work + 1) buckets, each a bitset of the CTAs with that
// load, finds it in amortised constant time (lowest set bit = lowest index).
void schedule_attention_units(const std::vector<int4>& items, int n_heads, int grid, std::vector<int4>& slots,
                              std::vector<int32_t>& off) {
    const int n_items = (int)items.size();
    std::vector<int> wk(n_items), order(n_items);
    int w_max = 1;
    for (int i = 0; i < n_items; ++i) {
        wk[i] = 2 * ((items[i].w - items[i].z + 127) / 128) + 1;
        w_max = std::max(w_max, wk[i]);
        order[i] = i;
    }
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return wk[a] > wk[b]; });
    const int words = (grid + 63) / 64, ring = w_max + 1;
    std::vector<uint64_t> bits((size_t)ring * words, 0);
    for (int c = 0; c < grid; ++c) bits[c >> 6] |= 1ull << (c & 63);
    std::vector<int> cta((size_t)n_items * n_heads);
    off.assign(grid + 1, 0);
    int lb = 0;   // bucket of the least load (that load modulo ring)
    size_t k = 0;
    for (int i : order) {
        for (int h = 0; h < n_heads; ++h, ++k) {
            int c = -1;
            while (c < 0) {
                uint64_t* b = &bits[(size_t)lb * words];
                for (int q = 0; q < words && c < 0; ++q)
                    if (b[q]) {
                        const int bit = __builtin_ctzll(b[q]);
                        b[q] &= b[q] - 1;
                        c = q * 64 + bit;
                    }
                if (c < 0 && ++lb == ring) lb = 0;
            }
            cta[k] = c;
            ++off[c + 1];
            int nb = lb + wk[i];   // wk[i] < ring
            if (nb >= ring) nb -= ring;
            bits[(size_t)nb * words + (c >> 6)] |= 1ull << (c & 63);
        }
    }
    for (int c = 0; c < grid; ++c) off[c + 1] += off[c];
    std::vector<int32_t> fill(off.begin(), off.end() - 1);
    slots.resize((size_t)n_items * n_heads);
    k = 0;
    for (int i : order)
        for (int h = 0; h < n_heads; ++h, ++k) {
            int4 it = items[i];
            it.y |= h << 16;
            slots[fill[cta[k]]++] = it;
        }
}

// Plans both lists and uploads the schedule of list `only` (0 global, 1
// window layers), or of both when only < 0.
int prepare_attention_items(tee_ctx* ctx, const int32_t* h_cu, int n_texts, cudaStream_t s, int only = -1) {
    plan_attention_items(h_cu, n_texts, ctx->cfg.window, ctx->h_items);
    int dev = 0, num_sms = 0;
    CK(tee_current_device(&dev, &num_sms));
    for (int b = 0; b < 2; ++b) {
        if (only >= 0 && b != only) continue;
        if ((int)ctx->h_items[b].size() > ctx->max_items)
            return fail(ctx, TEE_ETOOLONG, "too many attention work items");
        const int n_units = (int)ctx->h_items[b].size() * ctx->cfg.n_heads;
        ctx->attn_grid[b] = std::min(std::min(n_units, num_sms), TEE_ATTN_MAX_GRID);
        schedule_attention_units(ctx->h_items[b], ctx->cfg.n_heads, ctx->attn_grid[b], ctx->h_slots[b],
                                 ctx->h_slot_off[b]);
        CK(cudaMemcpyAsync(ctx->d_slots[b], ctx->h_slots[b].data(), ctx->h_slots[b].size() * sizeof(int4),
                           cudaMemcpyHostToDevice, s));
        CK(cudaMemcpyAsync(ctx->d_slot_off[b], ctx->h_slot_off[b].data(), ctx->h_slot_off[b].size() * sizeof(int32_t),
                           cudaMemcpyHostToDevice, s));
    }
    return TEE_OK;
}

}  // namespace

int tee_set_global_error(int code, const char* msg) { return fail(nullptr, code, "%s", msg); }

cudaError_t tee_current_device(int* dev, int* num_sms) {
    static std::mutex mu;
    static int sms[TEE_MAX_DEVICES] = {};
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return e;
    if (*dev < 0 || *dev >= TEE_MAX_DEVICES) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!sms[*dev]) {
        e = cudaDeviceGetAttribute(&sms[*dev], cudaDevAttrMultiProcessorCount, *dev);
        if (e != cudaSuccess) return e;
    }
    *num_sms = sms[*dev];
    return cudaSuccess;
}

// ---------------------------------------------------------------------------
// profiling
// ---------------------------------------------------------------------------
int prof_begin(tee_ctx* c, cudaStream_t s, int kclass, double flops, double bytes) {
    if (!c->profiling) return -1;
    if (c->prof_used == c->prof_slots.size()) {
        ProfileSlot slot{};
        if (cudaEventCreate(&slot.start) != cudaSuccess) return -1;
        if (cudaEventCreate(&slot.stop) != cudaSuccess) {
            cudaEventDestroy(slot.start);
            return -1;
        }
        c->prof_slots.push_back(slot);
    }
    ProfileSlot& slot = c->prof_slots[c->prof_used];
    slot.kclass = kclass;
    slot.flops = flops;
    slot.bytes = bytes;
    cudaEventRecord(slot.start, s);
    return (int)c->prof_used++;
}

void prof_end(tee_ctx* c, cudaStream_t s, int slot) {
    if (slot >= 0) cudaEventRecord(c->prof_slots[slot].stop, s);
}

#define LAUNCH(kclass, flops, bytes, expr)                                    \
    do {                                                                      \
        int _slot = prof_begin(ctx, s, (kclass), (flops), (bytes));           \
        cudaError_t _e = (expr);                                              \
        prof_end(ctx, s, _slot);                                              \
        if (_e != cudaSuccess) return cuda_fail(ctx, _e, #expr);              \
    } while (0)

// ---------------------------------------------------------------------------
// steps (shared by the pass and the per-step entry points)
// ---------------------------------------------------------------------------
namespace {

int step_layernorm(tee_ctx* ctx, int layer, int which, const float* x, void* y, int T, cudaStream_t s) {
    const tee_config& g = ctx->cfg;
    const float* gamma = which == TEE_LN_ATTN ? ctx->layers[layer].ln_attn : ctx->layers[layer].ln_mlp;
    const double bytes = (double)T * g.hidden * (4 + act_size(ctx)) + g.hidden * 4.0;
    LAUNCH(TEE_K_LAYERNORM, 0, bytes,
           launch_layernorm(x, gamma, y, act_is_bf16(ctx), T, g.hidden, g.ln_eps, s));
    return TEE_OK;
}

// A (ACT [T*K]) times weight `which` of `layer`; epi 0 stores into C (ACT), epi 1 adds into float C.
int step_linear(tee_ctx* ctx, int layer, int which, const void* A, void* C, int T, int epi, int tc_epi,
                const int32_t* pos, cudaStream_t s) {
    const tee_config& g = ctx->cfg;
    int N = 0, K = 0;
    wshape(g, which, &N, &K);
    const LayerWeights& L = ctx->layers[layer];
    const double flops = 2.0 * T * N * K;
    if (is_int_path(g)) {
        LAUNCH(TEE_K_QUANT, 0, (double)T * K * 5 + T * 4.0,
               launch_quant_rows7((const float*)A, T, K, ctx->qa, ctx->qs, s));
        LAUNCH(TEE_K_GEMM, flops, (double)T * K + (double)N * K + (double)T * N * 4 * (epi ? 2 : 1),
               launch_gemm_w8a8(ctx->qa, ctx->qs, (const int8_t*)L.w[which], L.wd[which], (float*)C, nullptr, T, N,
                                K, epi, weight_bits(g), s));
        return TEE_OK;
    }
    if (g.dtype == TEE_BF16) {
        const int is_g = layer_is_global(ctx, layer);
        GemmTcArgs a{};
        a.A = A;
        a.W = L.w[which];
        a.C = C;
        a.M = T;
        a.N = N;
        a.K = K;
        a.epi = tc_epi;
        a.pos = pos;
        a.rope_cos = ctx->rope_cos[is_g ? 0 : 1];
        a.rope_sin = ctx->rope_sin[is_g ? 0 : 1];
        a.hidden = g.hidden;
        a.status = ctx->d_status;
        const double out_b = tc_epi == GEMM_EPI_GEGLU ? (double)T * (N / 2) * 2
                            : (tc_epi == GEMM_EPI_ADD_F32 ? (double)T * N * 8 : (double)T * N * 2);
        LAUNCH(TEE_K_GEMM, flops, (double)T * K * 2 + (double)N * K * 2 + out_b, launch_gemm_tc(a, s));
        return TEE_OK;
    }
    LAUNCH(TEE_K_GEMM, flops, (double)T * K * 4 + (double)N * K * 4 + (double)T * N * 4 * (epi ? 2 : 1),
           launch_gemm_simt(A, L.w[which], C, false, T, N, K, epi, s));
    return TEE_OK;
}

int step_qkv(tee_ctx* ctx, int layer, const void* y, const int32_t* pos, void* qkv, int T, cudaStream_t s) {
    const tee_config& g = ctx->cfg;
    if (g.dtype == TEE_BF16) return step_linear(ctx, layer, TEE_W_QKV, y, qkv, T, 0, GEMM_EPI_ROPE_BF16, pos, s);
    int rc = step_linear(ctx, layer, TEE_W_QKV, y, qkv, T, 0, 0, pos, s);
    if (rc) return rc;
    const int b = layer_is_global(ctx, layer) ? 0 : 1;
    LAUNCH(TEE_K_ELEMENTWISE, 0, (double)T * 2 * g.hidden * act_size(ctx) * 2,
           launch_rope(qkv, act_is_bf16(ctx), pos, ctx->rope_cos[b], ctx->rope_sin[b], T, g.hidden, g.n_heads, s));
    return TEE_OK;
}

int step_attention(tee_ctx* ctx, int layer, const void* qkv, const int32_t* d_cu, const int32_t* h_cu, int n_texts,
                   int T, void* o, cudaStream_t s) {
    const tee_config& g = ctx->cfg;
    const bool is_g = layer_is_global(ctx, layer);
    const double pairs = ctx->profiling ? attention_pairs(h_cu, n_texts, is_g, g.window) : 0.0;
    const double flops = 4.0 * g.head_dim * g.n_heads * pairs;
    const double bytes = (double)T * g.hidden * act_size(ctx) * 4;
    if (g.dtype == TEE_BF16) {
        const int b = is_g ? 0 : 1;
        LAUNCH(TEE_K_ATTENTION, flops, bytes,
               launch_attention_tc(qkv, T, g.hidden, g.n_heads, ctx->d_slots[b], ctx->d_slot_off[b], ctx->attn_grid[b],
                                   is_g, g.window, ctx->d_rowtb, o, ctx->d_status, s));
        return TEE_OK;
    }
    LAUNCH(TEE_K_ATTENTION, flops, bytes,
           launch_attention_simple(qkv, act_is_bf16(ctx), d_cu, n_texts, T, g.hidden, g.n_heads, is_g, g.window, o, s));
    return TEE_OK;
}

int step_ffn_in(tee_ctx* ctx, int layer, const void* y, void* z, int T, cudaStream_t s) {
    const tee_config& g = ctx->cfg;
    if (g.dtype == TEE_BF16) return step_linear(ctx, layer, TEE_W_FFN_IN, y, z, T, 0, GEMM_EPI_GEGLU, nullptr, s);
    int rc = step_linear(ctx, layer, TEE_W_FFN_IN, y, ctx->u, T, 0, 0, nullptr, s);
    if (rc) return rc;
    LAUNCH(TEE_K_ELEMENTWISE, 0, (double)T * 3 * g.intermediate * act_size(ctx),
           launch_geglu(ctx->u, z, act_is_bf16(ctx), T, g.intermediate, s));
    return TEE_OK;
}

// Chunk offsets of the pool: text j owns ceil(len_j / POOL_CHUNK_FUSED) chunks.
int prepare_pool_chunks(tee_ctx* ctx, const int32_t* h_cu, int n_texts, cudaStream_t s) {
    ctx->h_chunk_off.resize(n_texts + 1);
    int total = 0;
    for (int j = 0; j < n_texts; ++j) {
        ctx->h_chunk_off[j] = total;
        total += (h_cu[j + 1] - h_cu[j] + POOL_CHUNK_FUSED - 1) / POOL_CHUNK_FUSED;
    }
    ctx->h_chunk_off[n_texts] = total;
    if (total > ctx->max_chunks) return fail(ctx, TEE_ETOOLONG, "too many pooling chunks");
    CK(cudaMemcpyAsync(ctx->d_chunk_off, ctx->h_chunk_off.data(), (n_texts + 1) * sizeof(int32_t),
                       cudaMemcpyHostToDevice, s));
    return TEE_OK;
}

int step_pool(tee_ctx* ctx, const float* x, const int32_t* d_cu, const int32_t* h_cu, int n_texts, int T, float* out,
              cudaStream_t s) {
    const tee_config& g = ctx->cfg;
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 15)
        return fail(ctx, TEE_EINVAL, "pool: x and out must be 16-byte aligned");
    int rc = prepare_pool_chunks(ctx, h_cu, n_texts, s);
    if (rc) return rc;
    const int n_chunks = ctx->h_chunk_off[n_texts];
    LAUNCH(TEE_K_POOL, 0, (double)T * g.hidden * 4 + (double)n_texts * g.hidden * 4,
           launch_pool_l2_fused(x, d_cu, ctx->d_chunk_off, n_texts, n_chunks, g.hidden, ctx->pool_partial,
                                ctx->pool_counters, out, s));
    return TEE_OK;
}

// fp32 LayerNorm of the residual stream in place (optional embedding / final norm).
int step_norm_in_place(tee_ctx* ctx, const float* gamma, int T, cudaStream_t s) {
    const tee_config& g = ctx->cfg;
    LAUNCH(TEE_K_LAYERNORM, 0, (double)T * g.hidden * 8 + g.hidden * 4.0,
           launch_layernorm(ctx->x, gamma, ctx->x, false, T, g.hidden, g.ln_eps, s));
    return TEE_OK;
}

// Embedding and every layer: the final token states in ctx->x.
int run_layers(tee_ctx* ctx, const int32_t* d_ids, const int32_t* d_cu, const int32_t* h_cu, int n_texts, int T,
               cudaStream_t s) {
    const tee_config& g = ctx->cfg;
    int rc;
    LAUNCH(TEE_K_EMBED, 0, (double)T * 4 * 4,
           launch_positions(d_cu, n_texts, T, ctx->d_pos, ctx->d_rowtb, s));
    LAUNCH(TEE_K_EMBED, 0, (double)T * g.hidden * (4.0 + (act_is_bf16(ctx) ? 2 : 4)) + T * 4.0,
           launch_embed(ctx->emb, act_is_bf16(ctx), d_ids, T, g.hidden, g.vocab, ctx->x, ctx->d_status, s));
    if (g.emb_norm && (rc = step_norm_in_place(ctx, ctx->ln_emb, T, s))) return rc;
    for (int l = 0; l < g.n_layers; ++l) {
        if ((rc = step_layernorm(ctx, l, TEE_LN_ATTN, ctx->x, ctx->y, T, s))) return rc;
        if ((rc = step_qkv(ctx, l, ctx->y, ctx->d_pos, ctx->qkv, T, s))) return rc;
        // the attention work items and their schedule are planned on the host
        // while the kernels queued so far run
        if (l == 0 && g.dtype == TEE_BF16 && (rc = prepare_attention_items(ctx, h_cu, n_texts, s))) return rc;
        if ((rc = step_attention(ctx, l, ctx->qkv, d_cu, h_cu, n_texts, T, ctx->o, s))) return rc;
        if ((rc = step_linear(ctx, l, TEE_W_OUT, ctx->o, ctx->x, T, 1, GEMM_EPI_ADD_F32, nullptr, s))) return rc;
        if ((rc = step_layernorm(ctx, l, TEE_LN_MLP, ctx->x, ctx->y, T, s))) return rc;
        if ((rc = step_ffn_in(ctx, l, ctx->y, ctx->z, T, s))) return rc;
        if ((rc = step_linear(ctx, l, TEE_W_FFN_OUT, ctx->z, ctx->x, T, 1, GEMM_EPI_ADD_F32, nullptr, s))) return rc;
    }
    if (g.final_norm && (rc = step_norm_in_place(ctx, ctx->ln_final, T, s))) return rc;
    return TEE_OK;
}

// One pass with the pooled output: unit vectors [n_texts, H] in d_out.
int run_pass(tee_ctx* ctx, const int32_t* d_ids, const int32_t* d_cu, const int32_t* h_cu, int n_texts, int T,
             float* d_out, cudaStream_t s) {
    int rc = run_layers(ctx, d_ids, d_cu, h_cu, n_texts, T, s);
    if (rc) return rc;
    return step_pool(ctx, ctx->x, d_cu, h_cu, n_texts, T, d_out, s);
}

// One pass with the per-token output: unit vectors [T, D] in d_out (16-byte
// aligned), D = proj_dim or hidden.
int run_tokens(tee_ctx* ctx, const int32_t* d_ids, const int32_t* d_cu, const int32_t* h_cu, int n_texts, int T,
               float* d_out, cudaStream_t s) {
    const tee_config& g = ctx->cfg;
    int rc = run_layers(ctx, d_ids, d_cu, h_cu, n_texts, T, s);
    if (rc) return rc;
    const int H = g.hidden, P = g.proj_dim, D = P ? P : H;
    if (!P) {
        CK(cudaMemcpyAsync(d_out, ctx->x, (size_t)T * H * 4, cudaMemcpyDeviceToDevice, s));
    } else if (is_int_path(g)) {
        LAUNCH(TEE_K_QUANT, 0, (double)T * H * 5 + T * 4.0, launch_quant_rows7(ctx->x, T, H, ctx->qa, ctx->qs, s));
        LAUNCH(TEE_K_GEMM, 2.0 * T * P * H, (double)T * H + (double)P * H + (double)T * P * 4,
               launch_gemm_w8a8(ctx->qa, ctx->qs, (const int8_t*)ctx->w_proj, ctx->w_proj_d, d_out, nullptr, T, P, H,
                                0, weight_bits(g), s));
    } else if (g.dtype == TEE_BF16) {
        // the projection's A operand in bf16, accumulated into a zeroed fp32 output
        LAUNCH(TEE_K_ELEMENTWISE, 0, (double)T * H * 6,
               launch_convert_f32_bf16(ctx->x, (bf16*)ctx->y, (size_t)T * H, s));
        CK(cudaMemsetAsync(d_out, 0, (size_t)T * P * 4, s));
        GemmTcArgs a{};
        a.A = ctx->y;
        a.W = ctx->w_proj;
        a.C = d_out;
        a.M = T;
        a.N = P;
        a.K = H;
        a.epi = GEMM_EPI_ADD_F32;
        a.hidden = H;
        a.status = ctx->d_status;
        LAUNCH(TEE_K_GEMM, 2.0 * T * P * H, (double)T * H * 2 + (double)P * H * 2 + (double)T * P * 8,
               launch_gemm_tc(a, s));
    } else {
        LAUNCH(TEE_K_GEMM, 2.0 * T * P * H, (double)T * H * 4 + (double)P * H * 4 + (double)T * P * 4,
               launch_gemm_simt(ctx->x, ctx->w_proj, d_out, false, T, P, H, 0, s));
    }
    LAUNCH(TEE_K_POOL, 0, (double)T * D * 8, launch_l2_rows(d_out, T, D, s));
    return TEE_OK;
}

int check_ready(tee_ctx* ctx) {
    if (!ctx) return TEE_EINVAL;
    if (!ctx->loaded) return fail(ctx, TEE_ENOTLOADED, "weights are not loaded");
    return TEE_OK;
}

int check_layer(tee_ctx* ctx, int layer) {
    if (layer < 0 || layer >= ctx->cfg.n_layers) return fail(ctx, TEE_EINVAL, "layer %d out of range", layer);
    return TEE_OK;
}

// Device buffers handed to a per-step entry point: non-NULL and aligned to
// `align` bytes (16 for activations, which the kernels move as 16-byte
// vectors or TMA tiles; 4 for int32 arrays).  Checked when the step has work.
int check_dev(tee_ctx* ctx, long long n, int align, std::initializer_list<const void*> ptrs) {
    if (n <= 0) return TEE_OK;
    for (const void* p : ptrs) {
        if (!p) return fail(ctx, TEE_EINVAL, "device buffer is NULL");
        if (reinterpret_cast<uintptr_t>(p) % (uintptr_t)align)
            return fail(ctx, TEE_EINVAL, "device buffer is not %d-byte aligned", align);
    }
    return TEE_OK;
}

// Makes the context's device current for one entry point and restores the
// caller's current device on the way out, so a process may interleave
// contexts on several devices.
struct DeviceScope {
    int prev = -1;
    cudaError_t err = cudaSuccess;
    explicit DeviceScope(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) err = cudaSetDevice(dev);
    }
    ~DeviceScope() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

#define ON_DEVICE(ctx)                                                            \
    DeviceScope _dscope((ctx)->device);                                           \
    if (_dscope.err != cudaSuccess) return cuda_fail((ctx), _dscope.err, "cudaSetDevice")

}  // namespace

// ---------------------------------------------------------------------------
// public C ABI
// ---------------------------------------------------------------------------
extern "C" {

int tee_create(const tee_config* cfg, int device, tee_ctx** out) {
    if (!out) return fail(nullptr, TEE_EINVAL, "out is NULL");
    *out = nullptr;
    int rc = validate_config(cfg);
    if (rc) return rc;
    tee_ctx* ctx = new (std::nothrow) tee_ctx();
    if (!ctx) return fail(nullptr, TEE_ENOMEM, "host allocation failed");
    ctx->cfg = *cfg;
    ctx->device = device;
    auto bail = [&](int code) {
        g_create_error = ctx->err;
        tee_destroy(ctx);
        return code;
    };
    DeviceScope dscope(device);
    if (dscope.err != cudaSuccess) return bail(cuda_fail(ctx, dscope.err, "cudaSetDevice"));
    ctx->ws_bytes = carve_workspace(ctx, nullptr);
    cudaError_t e;
    e = cudaMalloc(&ctx->ws_arena, ctx->ws_bytes);
    if (e != cudaSuccess) return bail(cuda_fail(ctx, e, "cudaMalloc(workspace)"));
    carve_workspace(ctx, ctx->ws_arena);
    e = cudaMemset(ctx->d_status, 0, 4 * sizeof(unsigned int));
    if (e != cudaSuccess) return bail(cuda_fail(ctx, e, "cudaMemset(status)"));
    e = cudaMemset(ctx->pool_counters, 0, (size_t)cfg->max_texts * sizeof(unsigned int));
    if (e != cudaSuccess) return bail(cuda_fail(ctx, e, "cudaMemset(pool counters)"));
    if ((rc = build_rope_tables(ctx))) return bail(rc);
    e = cudaStreamCreateWithFlags(&ctx->stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) return bail(cuda_fail(ctx, e, "cudaStreamCreate"));
    memset(ctx->prof_acc, 0, sizeof ctx->prof_acc);
    *out = ctx;
    return TEE_OK;
}

int tee_load_weights(tee_ctx* ctx, const tee_weights* w) {
    if (!ctx) return TEE_EINVAL;
    const tee_config& g = ctx->cfg;
    if (!w || !w->tok_emb || !w->ln_attn || !w->wqkv || !w->wo || !w->ln_mlp || !w->wi || !w->wo_ffn)
        return fail(ctx, TEE_EINVAL, "weights struct has NULL members");
    for (int l = 0; l < g.n_layers; ++l)
        if (!w->ln_attn[l] || !w->wqkv[l] || !w->wo[l] || !w->ln_mlp[l] || !w->wi[l] || !w->wo_ffn[l])
            return fail(ctx, TEE_EINVAL, "layer %d has a NULL weight pointer", l);
    if ((g.emb_norm && !w->ln_emb) || (g.final_norm && !w->ln_final) || (g.proj_dim && !w->w_proj))
        return fail(ctx, TEE_EINVAL, "an enabled optional weight (ln_emb, ln_final, w_proj) is NULL");
    ON_DEVICE(ctx);
    ctx->loaded = false;
    if (ctx->weight_arena) {
        CK(cudaFree(ctx->weight_arena));
        ctx->weight_arena = nullptr;
    }
    ctx->weight_bytes = carve_weights(ctx, nullptr);
    CK(cudaMalloc(&ctx->weight_arena, ctx->weight_bytes));
    carve_weights(ctx, ctx->weight_arena);

    const size_t H = g.hidden, V = g.vocab;
    // the largest host tensor staged: token embeddings, Wqkv, Wi (Wo_ffn is half of Wi) or the projection
    size_t stage_elems = std::max({V * H, 3 * H * H, (size_t)2 * g.intermediate * H, (size_t)g.proj_dim * H});
    float* stage = nullptr;
    if (g.dtype != TEE_F32) CK(cudaMalloc(&stage, stage_elems * sizeof(float)));
    cudaStream_t s = ctx->stream;
    int rc = TEE_OK;
    auto put = [&](void* dst, const float* src, size_t n, int kind, int N, int K, float* dscale) -> int {
        // kind 0: fp32 copy; 1: bf16 convert; 2: int8 block quantise
        if (kind == 0) {
            CK(cudaMemcpy(dst, src, n * sizeof(float), cudaMemcpyHostToDevice));
            return TEE_OK;
        }
        if (n > stage_elems) return fail(ctx, TEE_EINVAL, "weight staging: tensor larger than the staging buffer");
        CK(cudaMemcpyAsync(stage, src, n * sizeof(float), cudaMemcpyHostToDevice, s));
        if (kind == 1) CK(launch_convert_f32_bf16(stage, (bf16*)dst, n, s));
        else CK(launch_quant_weight_blocks(stage, (int8_t*)dst, dscale, N, K, weight_bits(g), s));
        CK(cudaStreamSynchronize(s));
        return TEE_OK;
    };
    const int lin_kind = g.dtype == TEE_F32 ? 0 : (g.dtype == TEE_BF16 ? 1 : 2);
    const int emb_kind = g.dtype == TEE_BF16 ? 1 : 0;
    // LayerNorm gains are stored as fp32 in every variant; the bf16 variant
    // keeps their bf16-rounded values.
    auto put_gain = [&](float* dst, const float* src) -> int {
        if (g.dtype != TEE_BF16) return put(dst, src, H, 0, 0, 0, nullptr);
        std::vector<float> tmp(H);
        for (size_t i = 0; i < H; ++i) {
            uint32_t u;
            memcpy(&u, &src[i], 4);
            u = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
            memcpy(&tmp[i], &u, 4);
        }
        return put(dst, tmp.data(), H, 0, 0, 0, nullptr);
    };
    if ((rc = put(ctx->emb, w->tok_emb, V * H, emb_kind, 0, 0, nullptr))) goto done;
    if (g.emb_norm && (rc = put_gain(ctx->ln_emb, w->ln_emb))) goto done;
    if (g.final_norm && (rc = put_gain(ctx->ln_final, w->ln_final))) goto done;
    if (g.proj_dim && (rc = put(ctx->w_proj, w->w_proj, (size_t)g.proj_dim * H, lin_kind, g.proj_dim, (int)H,
                                ctx->w_proj_d)))
        goto done;
    for (int l = 0; l < g.n_layers && rc == TEE_OK; ++l) {
        LayerWeights& L = ctx->layers[l];
        if ((rc = put_gain(L.ln_attn, w->ln_attn[l]))) break;
        if ((rc = put_gain(L.ln_mlp, w->ln_mlp[l]))) break;
        const float* srcs[4] = {w->wqkv[l], w->wo[l], w->wi[l], w->wo_ffn[l]};
        for (int which = 0; which < 4 && rc == TEE_OK; ++which) {
            int N, K;
            wshape(g, which, &N, &K);
            const float* src = srcs[which];
            std::vector<float> perm;
            if (g.dtype == TEE_BF16 && which == TEE_W_FFN_IN) {
                // the tensor-core GEMM fuses the GeGLU gate: each 256-row tile holds
                // 128 GELU-input rows followed by the 128 matching gate rows
                perm.resize((size_t)N * K);
                for (int r = 0; r < N; ++r)
                    memcpy(&perm[(size_t)r * K], src + (size_t)geglu_source_row(r, g.intermediate) * K,
                           (size_t)K * sizeof(float));
                src = perm.data();
            }
            rc = put(L.w[which], src, (size_t)N * K, lin_kind, N, K, L.wd[which]);
        }
    }
done:
    if (stage) cudaFree(stage);
    if (rc) return rc;
    ctx->loaded = true;
    return TEE_OK;
}

int tee_encode(tee_ctx* ctx, const int32_t* token_ids, const int32_t* cu_seqlens, int n_texts, float* out) {
    int rc = check_ready(ctx);
    if (rc) return rc;
    if (!token_ids || !out) return fail(ctx, TEE_EINVAL, "token_ids / out is NULL");
    int T = 0;
    if ((rc = check_cu(ctx, cu_seqlens, n_texts, &T))) return rc;
    for (int t = 0; t < T; ++t)
        if (token_ids[t] < 0 || token_ids[t] >= ctx->cfg.vocab)
            return fail(ctx, TEE_EINVAL, "token id %d at position %d is outside [0, %d)", token_ids[t], t,
                        ctx->cfg.vocab);
    ON_DEVICE(ctx);
    cudaStream_t s = ctx->stream;
    CK(cudaMemcpyAsync(ctx->d_ids, token_ids, (size_t)T * 4, cudaMemcpyHostToDevice, s));
    CK(cudaMemcpyAsync(ctx->d_cu, cu_seqlens, (size_t)(n_texts + 1) * 4, cudaMemcpyHostToDevice, s));
    if ((rc = run_pass(ctx, ctx->d_ids, ctx->d_cu, cu_seqlens, n_texts, T, ctx->out, s))) return rc;
    CK(cudaMemcpyAsync(out, ctx->out, (size_t)n_texts * ctx->cfg.hidden * 4, cudaMemcpyDeviceToHost, s));
    CK(cudaStreamSynchronize(s));
    return TEE_OK;
}

int tee_encode_device(tee_ctx* ctx, const int32_t* d_ids, const int32_t* d_cu, const int32_t* h_cu, int n_texts,
                      float* d_out, void* stream) {
    int rc = check_ready(ctx);
    if (rc) return rc;
    if (!d_ids || !d_cu || !d_out) return fail(ctx, TEE_EINVAL, "device pointer is NULL");
    if (reinterpret_cast<uintptr_t>(d_out) & 15) return fail(ctx, TEE_EINVAL, "d_out must be 16-byte aligned");
    int T = 0;
    if ((rc = check_cu(ctx, h_cu, n_texts, &T))) return rc;
    ON_DEVICE(ctx);
    return run_pass(ctx, d_ids, d_cu, h_cu, n_texts, T, d_out, (cudaStream_t)stream);
}

int tee_encode_tokens(tee_ctx* ctx, const int32_t* token_ids, const int32_t* cu_seqlens, int n_texts, float* out) {
    int rc = check_ready(ctx);
    if (rc) return rc;
    if (!token_ids || !out) return fail(ctx, TEE_EINVAL, "token_ids / out is NULL");
    int T = 0;
    if ((rc = check_cu(ctx, cu_seqlens, n_texts, &T))) return rc;
    for (int t = 0; t < T; ++t)
        if (token_ids[t] < 0 || token_ids[t] >= ctx->cfg.vocab)
            return fail(ctx, TEE_EINVAL, "token id %d at position %d is outside [0, %d)", token_ids[t], t,
                        ctx->cfg.vocab);
    ON_DEVICE(ctx);
    const size_t D = ctx->cfg.proj_dim ? ctx->cfg.proj_dim : ctx->cfg.hidden;
    if (!ctx->tok_out) CK(cudaMalloc(&ctx->tok_out, (size_t)ctx->cfg.max_tokens * D * sizeof(float)));
    cudaStream_t s = ctx->stream;
    CK(cudaMemcpyAsync(ctx->d_ids, token_ids, (size_t)T * 4, cudaMemcpyHostToDevice, s));
    CK(cudaMemcpyAsync(ctx->d_cu, cu_seqlens, (size_t)(n_texts + 1) * 4, cudaMemcpyHostToDevice, s));
    if ((rc = run_tokens(ctx, ctx->d_ids, ctx->d_cu, cu_seqlens, n_texts, T, ctx->tok_out, s))) return rc;
    CK(cudaMemcpyAsync(out, ctx->tok_out, (size_t)T * D * 4, cudaMemcpyDeviceToHost, s));
    CK(cudaStreamSynchronize(s));
    return TEE_OK;
}

int tee_encode_tokens_device(tee_ctx* ctx, const int32_t* d_ids, const int32_t* d_cu, const int32_t* h_cu,
                             int n_texts, float* d_out, void* stream) {
    int rc = check_ready(ctx);
    if (rc) return rc;
    if (!d_ids || !d_cu || !d_out) return fail(ctx, TEE_EINVAL, "device pointer is NULL");
    if (reinterpret_cast<uintptr_t>(d_out) & 15) return fail(ctx, TEE_EINVAL, "d_out must be 16-byte aligned");
    int T = 0;
    if ((rc = check_cu(ctx, h_cu, n_texts, &T))) return rc;
    ON_DEVICE(ctx);
    return run_tokens(ctx, d_ids, d_cu, h_cu, n_texts, T, d_out, (cudaStream_t)stream);
}

const char* tee_last_error(const tee_ctx* ctx) { return ctx ? ctx->err.c_str() : g_create_error.c_str(); }

void tee_destroy(tee_ctx* ctx) {
    if (!ctx) return;
    DeviceScope dscope(ctx->device);
    if (ctx->stream) cudaStreamSynchronize(ctx->stream);
    for (auto& sl : ctx->prof_slots) {
        cudaEventDestroy(sl.start);
        cudaEventDestroy(sl.stop);
    }
    if (ctx->weight_arena) cudaFree(ctx->weight_arena);
    if (ctx->ws_arena) cudaFree(ctx->ws_arena);
    if (ctx->tok_out) cudaFree(ctx->tok_out);
    if (ctx->stream) cudaStreamDestroy(ctx->stream);
    delete ctx;
}

// ---- host-only planning (no device, no context) ---------------------------

int tee_plan_attention(const int32_t* h_cu, int n_texts, int window, int is_global, int32_t* items, int max_items) {
    if (!h_cu) return tee_set_global_error(TEE_EINVAL, "plan_attention: cu_seqlens is NULL");
    if (n_texts < 1) return tee_set_global_error(TEE_EINVAL, "plan_attention: n_texts must be >= 1");
    if (window < 0) return tee_set_global_error(TEE_EINVAL, "plan_attention: window must be >= 0");
    if (h_cu[0] != 0) return tee_set_global_error(TEE_EINVAL, "plan_attention: cu_seqlens[0] must be 0");
    for (int j = 0; j < n_texts; ++j)
        if (h_cu[j + 1] <= h_cu[j])
            return tee_set_global_error(TEE_EINVAL, "plan_attention: cu_seqlens must be strictly increasing");
    std::vector<int4> lists[2];
    plan_attention_items(h_cu, n_texts, window, lists);
    const std::vector<int4>& v = lists[is_global ? 0 : 1];
    if (!items) return (int)v.size();
    if ((int)v.size() > max_items) return tee_set_global_error(TEE_ETOOLONG, "plan_attention: more items than max_items");
    for (size_t i = 0; i < v.size(); ++i) {
        items[4 * i + 0] = v[i].x;
        items[4 * i + 1] = v[i].y;
        items[4 * i + 2] = v[i].z;
        items[4 * i + 3] = v[i].w;
    }
    return (int)v.size();
}

int tee_plan_attention_schedule(const int32_t* items, int n_items, int n_heads, int grid, int32_t* slots,
                                int32_t* slot_off) {
    if (n_items < 0 || (n_items > 0 && !items)) return tee_set_global_error(TEE_EINVAL, "plan_schedule: bad items");
    if (n_heads < 1 || n_heads > 32767) return tee_set_global_error(TEE_EINVAL, "plan_schedule: n_heads out of range");
    if (grid < 1 || grid > TEE_ATTN_MAX_GRID) return tee_set_global_error(TEE_EINVAL, "plan_schedule: grid out of range");
    if (!slots || !slot_off) return tee_set_global_error(TEE_EINVAL, "plan_schedule: output is NULL");
    if ((long long)n_items * n_heads > INT32_MAX / 4) return tee_set_global_error(TEE_ETOOLONG, "plan_schedule: too many units");
    std::vector<int4> v(n_items);
    for (int i = 0; i < n_items; ++i) {
        v[i] = make_int4(items[4 * i], items[4 * i + 1], items[4 * i + 2], items[4 * i + 3]);
        if (v[i].y < 0 || v[i].y > 0xffff || v[i].w < v[i].z)
            return tee_set_global_error(TEE_EINVAL, "plan_schedule: bad item");
    }
    std::vector<int4> sl;
    std::vector<int32_t> off;
    schedule_attention_units(v, n_heads, grid, sl, off);
    for (size_t i = 0; i < sl.size(); ++i) {
        slots[4 * i + 0] = sl[i].x;
        slots[4 * i + 1] = sl[i].y;
        slots[4 * i + 2] = sl[i].z;
        slots[4 * i + 3] = sl[i].w;
    }
    for (int c = 0; c <= grid; ++c) slot_off[c] = off[c];
    return (int)sl.size();
}

int tee_plan_gemm(int M, int N, int K, int epi, int num_sms, int* bn, int* pair) {
    if (!bn || !pair) return tee_set_global_error(TEE_EINVAL, "plan_gemm: NULL output");
    if (M < 1 || N < 128 || N % 128 || K < 64 || K % 64 || epi < GEMM_EPI_STORE_BF16 || epi > GEMM_EPI_GEGLU ||
        (epi == GEMM_EPI_GEGLU && N % 256) || num_sms < 2)
        return tee_set_global_error(TEE_EINVAL, "plan_gemm: shape, epilogue or SM count out of range");
    gemm_tc_choose_tiles(M, N, K, epi, num_sms, bn, pair);
    return TEE_OK;
}

int tee_profile_enable(tee_ctx* ctx, int on) {
    if (!ctx) return TEE_EINVAL;
    ctx->profiling = on != 0;
    ctx->prof_used = 0;
    memset(ctx->prof_acc, 0, sizeof ctx->prof_acc);
    return TEE_OK;
}

int tee_profile_read(tee_ctx* ctx, tee_kernel_stat* stats) {
    if (!ctx || !stats) return TEE_EINVAL;
    ON_DEVICE(ctx);
    for (size_t i = 0; i < ctx->prof_used; ++i) {
        ProfileSlot& sl = ctx->prof_slots[i];
        CK(cudaEventSynchronize(sl.stop));
        float ms = 0.f;
        CK(cudaEventElapsedTime(&ms, sl.start, sl.stop));
        tee_kernel_stat& a = ctx->prof_acc[sl.kclass];
        a.launches += 1;
        a.total_ms += ms;
        a.flops += sl.flops;
        a.bytes += sl.bytes;
    }
    ctx->prof_used = 0;
    memcpy(stats, ctx->prof_acc, sizeof ctx->prof_acc);
    return TEE_OK;
}

// ---- per-step entry points ------------------------------------------------

int tee_op_embed(tee_ctx* ctx, const int32_t* d_ids, int T, float* d_x, void* stream) {
    int rc = check_ready(ctx);
    if (rc) return rc;
    if (T < 0 || T > ctx->cfg.max_tokens) return fail(ctx, TEE_EINVAL, "bad T");
    if ((rc = check_dev(ctx, T, 16, {d_x})) || (rc = check_dev(ctx, T, 4, {d_ids}))) return rc;
    ON_DEVICE(ctx);
    cudaStream_t s = (cudaStream_t)stream;
    LAUNCH(TEE_K_EMBED, 0, 0,
           launch_embed(ctx->emb, act_is_bf16(ctx), d_ids, T, ctx->cfg.hidden, ctx->cfg.vocab, d_x, ctx->d_status, s));
    return TEE_OK;
}

int tee_op_positions(tee_ctx* ctx, const int32_t* d_cu, const int32_t* h_cu, int n_texts, int32_t* d_pos,
                     void* stream) {
    if (!ctx) return TEE_EINVAL;
    int T = 0, rc = check_cu(ctx, h_cu, n_texts, &T);
    if (rc || (rc = check_dev(ctx, T, 4, {d_cu, d_pos}))) return rc;
    ON_DEVICE(ctx);
    cudaStream_t s = (cudaStream_t)stream;
    LAUNCH(TEE_K_EMBED, 0, 0, launch_positions(d_cu, n_texts, T, d_pos, nullptr, s));
    return TEE_OK;
}

int tee_op_layernorm(tee_ctx* ctx, int layer, int which, const float* d_x, void* d_y, int T, void* stream) {
    int rc = check_ready(ctx);
    if (rc || (rc = check_layer(ctx, layer))) return rc;
    if (which != TEE_LN_ATTN && which != TEE_LN_MLP) return fail(ctx, TEE_EINVAL, "bad LayerNorm selector");
    if (T < 0 || T > ctx->cfg.max_tokens) return fail(ctx, TEE_EINVAL, "bad T");
    if ((rc = check_dev(ctx, T, 16, {d_x, d_y}))) return rc;
    ON_DEVICE(ctx);
    return step_layernorm(ctx, layer, which, d_x, d_y, T, (cudaStream_t)stream);
}

int tee_op_qkv(tee_ctx* ctx, int layer, const void* d_y, const int32_t* d_pos, void* d_qkv, int T, void* stream) {
    int rc = check_ready(ctx);
    if (rc || (rc = check_layer(ctx, layer))) return rc;
    if (T < 0 || T > ctx->cfg.max_tokens) return fail(ctx, TEE_EINVAL, "bad T");
    if ((rc = check_dev(ctx, T, 16, {d_y, d_qkv})) || (rc = check_dev(ctx, T, 4, {d_pos}))) return rc;
    ON_DEVICE(ctx);
    return step_qkv(ctx, layer, d_y, d_pos, d_qkv, T, (cudaStream_t)stream);
}

int tee_op_attention(tee_ctx* ctx, int layer, const void* d_qkv, const int32_t* d_cu, const int32_t* h_cu,
                     int n_texts, void* d_o, void* stream) {
    int rc = check_ready(ctx);
    if (rc || (rc = check_layer(ctx, layer))) return rc;
    int T = 0;
    if ((rc = check_cu(ctx, h_cu, n_texts, &T))) return rc;
    if ((rc = check_dev(ctx, T, 16, {d_qkv, d_o})) || (rc = check_dev(ctx, T, 4, {d_cu}))) return rc;
    ON_DEVICE(ctx);
    if (ctx->cfg.dtype == TEE_BF16) {
        // the work items, and the per-row text bounds the window layers' masks take
        if ((rc = prepare_attention_items(ctx, h_cu, n_texts, (cudaStream_t)stream,
                                          layer_is_global(ctx, layer) ? 0 : 1)))
            return rc;
        cudaStream_t s = (cudaStream_t)stream;
        LAUNCH(TEE_K_EMBED, 0, 0, launch_positions(d_cu, n_texts, T, ctx->d_pos, ctx->d_rowtb, s));
    }
    return step_attention(ctx, layer, d_qkv, d_cu, h_cu, n_texts, T, d_o, (cudaStream_t)stream);
}

int tee_op_out_proj(tee_ctx* ctx, int layer, const void* d_o, float* d_x, int T, void* stream) {
    int rc = check_ready(ctx);
    if (rc || (rc = check_layer(ctx, layer))) return rc;
    if (T < 0 || T > ctx->cfg.max_tokens) return fail(ctx, TEE_EINVAL, "bad T");
    if ((rc = check_dev(ctx, T, 16, {d_o, d_x}))) return rc;
    ON_DEVICE(ctx);
    return step_linear(ctx, layer, TEE_W_OUT, d_o, d_x, T, 1, GEMM_EPI_ADD_F32, nullptr, (cudaStream_t)stream);
}

int tee_op_ffn_in(tee_ctx* ctx, int layer, const void* d_y, void* d_z, int T, void* stream) {
    int rc = check_ready(ctx);
    if (rc || (rc = check_layer(ctx, layer))) return rc;
    if (T < 0 || T > ctx->cfg.max_tokens) return fail(ctx, TEE_EINVAL, "bad T");
    if ((rc = check_dev(ctx, T, 16, {d_y, d_z}))) return rc;
    ON_DEVICE(ctx);
    return step_ffn_in(ctx, layer, d_y, d_z, T, (cudaStream_t)stream);
}

int tee_op_ffn_out(tee_ctx* ctx, int layer, const void* d_z, float* d_x, int T, void* stream) {
    int rc = check_ready(ctx);
    if (rc || (rc = check_layer(ctx, layer))) return rc;
    if (T < 0 || T > ctx->cfg.max_tokens) return fail(ctx, TEE_EINVAL, "bad T");
    if ((rc = check_dev(ctx, T, 16, {d_z, d_x}))) return rc;
    ON_DEVICE(ctx);
    return step_linear(ctx, layer, TEE_W_FFN_OUT, d_z, d_x, T, 1, GEMM_EPI_ADD_F32, nullptr, (cudaStream_t)stream);
}

int tee_op_gemm_bf16(tee_ctx* ctx, const void* d_a, const void* d_w, void* d_c, int M, int N, int K, int epilogue,
                     void* stream) {
    if (!ctx) return TEE_EINVAL;
    if (ctx->cfg.dtype != TEE_BF16) return fail(ctx, TEE_EINVAL, "tee_op_gemm_bf16 needs a TEE_BF16 context");
    if (!d_a || !d_w || !d_c) return fail(ctx, TEE_EINVAL, "NULL pointer");
    if (M < 0 || N <= 0 || K <= 0 || N % 128 || K % 64) return fail(ctx, TEE_EINVAL, "bad GEMM shape");
    if (epilogue != 0 && epilogue != 1) return fail(ctx, TEE_EINVAL, "epilogue must be 0 (store) or 1 (add)");
    GemmTcArgs a{};
    a.A = d_a;
    a.W = d_w;
    a.C = d_c;
    a.M = M;
    a.N = N;
    a.K = K;
    a.epi = epilogue == 0 ? GEMM_EPI_STORE_BF16 : GEMM_EPI_ADD_F32;
    a.status = ctx->d_status;
    ON_DEVICE(ctx);
    cudaStream_t s = (cudaStream_t)stream;
    LAUNCH(TEE_K_GEMM, 2.0 * M * N * K, 0, launch_gemm_tc(a, s));
    return TEE_OK;
}

int tee_op_pool_l2(tee_ctx* ctx, const float* d_x, const int32_t* d_cu, const int32_t* h_cu, int n_texts,
                   float* d_out, void* stream) {
    if (!ctx) return TEE_EINVAL;
    int T = 0, rc = check_cu(ctx, h_cu, n_texts, &T);
    if (rc || (rc = check_dev(ctx, T, 16, {d_x, d_out})) || (rc = check_dev(ctx, T, 4, {d_cu}))) return rc;
    ON_DEVICE(ctx);
    return step_pool(ctx, d_x, d_cu, h_cu, n_texts, T, d_out, (cudaStream_t)stream);
}

int tee_op_quant_rows7(tee_ctx* ctx, const float* d_x, int M, int K, int8_t* d_q, float* d_s, void* stream) {
    if (!ctx) return TEE_EINVAL;
    if (M < 0 || K < 1) return fail(ctx, TEE_EINVAL, "bad M/K");
    int rc = check_dev(ctx, M, 16, {d_x, d_q});
    if (rc || (rc = check_dev(ctx, M, 4, {d_s}))) return rc;
    ON_DEVICE(ctx);
    cudaStream_t s = (cudaStream_t)stream;
    LAUNCH(TEE_K_QUANT, 0, 0, launch_quant_rows7(d_x, M, K, d_q, d_s, s));
    return TEE_OK;
}

int tee_op_w8a8_partials(tee_ctx* ctx, int layer, int which, const int8_t* d_q, int M, int32_t* d_partials,
                         void* stream) {
    int rc = check_ready(ctx);
    if (rc || (rc = check_layer(ctx, layer))) return rc;
    if (!is_int_path(ctx->cfg)) return fail(ctx, TEE_EINVAL, "context is not W8A8 / W6A8 / W4A8");
    int N, K;
    if (wshape(ctx->cfg, which, &N, &K)) return fail(ctx, TEE_EINVAL, "bad projection selector");
    if (M < 0) return fail(ctx, TEE_EINVAL, "bad M");
    if ((rc = check_dev(ctx, M, 16, {d_q})) || (rc = check_dev(ctx, M, 4, {d_partials}))) return rc;
    const LayerWeights& L = ctx->layers[layer];
    ON_DEVICE(ctx);
    cudaStream_t s = (cudaStream_t)stream;
    LAUNCH(TEE_K_GEMM, 0, 0,
           launch_gemm_w8a8(d_q, nullptr, (const int8_t*)L.w[which], L.wd[which], nullptr, d_partials, M, N, K, 0,
                            weight_bits(ctx->cfg), s));
    return TEE_OK;
}

int tee_weight_codes(tee_ctx* ctx, int layer, int which, int8_t* h_q, float* h_d) {
    int rc = check_ready(ctx);
    if (rc || (rc = check_layer(ctx, layer))) return rc;
    if (!is_int_path(ctx->cfg)) return fail(ctx, TEE_EINVAL, "context is not W8A8 / W6A8 / W4A8");
    int N, K;
    if (wshape(ctx->cfg, which, &N, &K)) return fail(ctx, TEE_EINVAL, "bad projection selector");
    if (!h_q || !h_d) return fail(ctx, TEE_EINVAL, "NULL output");
    ON_DEVICE(ctx);
    if (ctx->cfg.dtype == TEE_W4A8) {   // widen the packed nibbles: element 2i low, 2i + 1 high
        std::vector<uint8_t> packed((size_t)N * K / 2);
        CK(cudaMemcpy(packed.data(), ctx->layers[layer].w[which], packed.size(), cudaMemcpyDeviceToHost));
        for (size_t i = 0; i < packed.size(); ++i) {
            const int lo = packed[i] & 15, hi = packed[i] >> 4;
            h_q[2 * i] = (int8_t)((lo ^ 8) - 8);
            h_q[2 * i + 1] = (int8_t)((hi ^ 8) - 8);
        }
    } else if (ctx->cfg.dtype == TEE_W6A8) {   // widen: codes 4i..4i+3 in the 24 bits of bytes 3i..3i+2
        std::vector<uint8_t> packed((size_t)N * K / 4 * 3);
        CK(cudaMemcpy(packed.data(), ctx->layers[layer].w[which], packed.size(), cudaMemcpyDeviceToHost));
        for (size_t i = 0; i < packed.size() / 3; ++i) {
            const uint32_t bits = packed[3 * i] | ((uint32_t)packed[3 * i + 1] << 8) | ((uint32_t)packed[3 * i + 2] << 16);
            for (int k = 0; k < 4; ++k) {
                const int v = (int)((bits >> (6 * k)) & 63u);
                h_q[4 * i + k] = (int8_t)((v ^ 32) - 32);
            }
        }
    } else {
        CK(cudaMemcpy(h_q, ctx->layers[layer].w[which], (size_t)N * K, cudaMemcpyDeviceToHost));
    }
    CK(cudaMemcpy(h_d, ctx->layers[layer].wd[which], (size_t)N * K / 32 * 4, cudaMemcpyDeviceToHost));
    return TEE_OK;
}

int tee_selftest_wait_timeout(tee_ctx* ctx, long long wait_cycles, void* stream) {
    if (!ctx) return TEE_EINVAL;
    if (wait_cycles < 1000) wait_cycles = 1000;
    if (wait_cycles > 10000000000LL) wait_cycles = 10000000000LL;
    ON_DEVICE(ctx);
    CK(launch_selftest_wait(wait_cycles, ctx->d_status, (cudaStream_t)stream));
    return TEE_OK;
}

int tee_device_status(tee_ctx* ctx) {
    if (!ctx) return TEE_EINVAL;
    ON_DEVICE(ctx);
    unsigned int st = 0;
    CK(cudaDeviceSynchronize());
    CK(cudaMemcpy(&st, ctx->d_status, 4, cudaMemcpyDeviceToHost));
    CK(cudaMemset(ctx->d_status, 0, 4));
    if (st & TEE_STATUS_TIMEOUT) return fail(ctx, TEE_ETIMEOUT, "a device-side wait gave up (status 0x%x)", st);
    if (st & TEE_STATUS_BAD_ID) return fail(ctx, TEE_EINVAL, "a token id was outside [0, vocab)");
    return TEE_OK;
}

}  // extern "C"
