// Memory-bound steps of the pass: embedding gather, per-text positions,
// bias-free LayerNorm, RoPE, GeGLU gate, and mean-pool + L2 normalisation.
//
// Method: tensai page "テキスト埋め込み", §何が動くか (エンコーダ, プーリング,
// packing paragraph).  All of these are bandwidth-bound: rows are read with
// 16-byte vector loads, one warp per row (LayerNorm) or per token (gather);
// the pool reduces 64-row chunks of each text in parallel, then
// combines each text's chunks in order; reductions by warp shuffles.
#include "tee_internal.cuh"

#include <mutex>

namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Index of the text containing token t: the largest j with cu[j] <= t.
__device__ __forceinline__ int text_of(const int32_t* cu, int n_texts, int t) {
    int lo = 0, hi = n_texts - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__global__ void convert_f32_bf16_kernel(const float* __restrict__ src, bf16* __restrict__ dst, size_t n) {
    pdl_wait();
    pdl_trigger();
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    size_t stride = (size_t)gridDim.x * blockDim.x;
    for (; i < n; i += stride) dst[i] = __float2bfloat16_rn(src[i]);
}

// x[t, :] = E[id[t], :]; one warp per token (8 tokens per 256-thread block),
// 16-byte loads of the table row and 16-byte stores of the fp32 row.
template <typename TE>
__global__ void embed_kernel(const TE* __restrict__ emb, const int32_t* __restrict__ ids, int T, int H, int V,
                             float* __restrict__ x, unsigned int* status) {
    pdl_wait();
    pdl_trigger();
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    const int id = ids[t];
    const bool ok = (id >= 0 && id < V);
    if (!ok && lane == 0 && status) atomicOr(status, TEE_STATUS_BAD_ID);
    float4* dst = reinterpret_cast<float4*>(x + (size_t)t * H);
    if constexpr (sizeof(TE) == 4) {
        const float4* src = reinterpret_cast<const float4*>(emb + (size_t)(ok ? id : 0) * H);
        for (int c4 = lane; c4 < H / 4; c4 += 32) dst[c4] = ok ? src[c4] : make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
        // 8 bf16 (16 bytes) per load -> two float4 stores
        const uint4* src = reinterpret_cast<const uint4*>(emb + (size_t)(ok ? id : 0) * H);
        for (int c8 = lane; c8 < H / 8; c8 += 32) {
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            if (ok) {
                const uint4 q = src[c8];
                const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.x));
                const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.y));
                const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.z));
                const float2 f3 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.w));
                a = make_float4(f0.x, f0.y, f1.x, f1.y);
                b = make_float4(f2.x, f2.y, f3.x, f3.y);
            }
            dst[2 * c8] = a;
            dst[2 * c8 + 1] = b;
        }
    }
}

// pos[t] = t - cu[text(t)]; row_tb[t] = {cu[text(t)], cu[text(t) + 1]} (the
// bounds of the text holding token t, for the attention's per-row masks)
__global__ void positions_kernel(const int32_t* __restrict__ cu, int n_texts, int T, int32_t* __restrict__ pos,
                                 int2* __restrict__ row_tb) {
    pdl_wait();
    pdl_trigger();
    int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    const int j = text_of(cu, n_texts, t);
    const int s0 = cu[j];
    pos[t] = t - s0;
    if (row_tb) row_tb[t] = make_int2(s0, cu[j + 1]);
}

// One warp per row; H a multiple of 128 and <= 1024 (at most 8 float4 per lane).
// y may be x itself (fp32 output): a warp reads its whole row before writing it.
template <typename TY>
__global__ void layernorm_kernel(const float* x, const float* __restrict__ gamma, TY* y, int T, int H, float eps) {
    pdl_wait();
    pdl_trigger();
    // Rows are taken last first: the kernel before this one (a residual
    // projection, or the embedding) writes them first to last, so the rows it
    // wrote last are read while they are still in L2.
    const int warp = T - 1 - (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (warp < 0) return;
    const float4* row = reinterpret_cast<const float4*>(x + (size_t)warp * H);
    const int nv = H / 128;   // float4 per lane
    float4 v[8];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i < nv) {
            v[i] = row[i * 32 + lane];
            s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
        }
    }
    const float mean = warp_sum(s) / (float)H;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i < nv) {
            float a = v[i].x - mean, b = v[i].y - mean, c = v[i].z - mean, d = v[i].w - mean;
            ss += (a * a + b * b) + (c * c + d * d);
        }
    }
    const float var = warp_sum(ss) / (float)H;
    const float rstd = 1.0f / sqrtf(var + eps);
    const float4* g4 = reinterpret_cast<const float4*>(gamma);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i < nv) {
            int c4 = i * 32 + lane;
            float4 g = g4[c4];
            float o0 = (v[i].x - mean) * rstd * g.x, o1 = (v[i].y - mean) * rstd * g.y;
            float o2 = (v[i].z - mean) * rstd * g.z, o3 = (v[i].w - mean) * rstd * g.w;
            if constexpr (sizeof(TY) == 4) {
                reinterpret_cast<float4*>(y + (size_t)warp * H)[c4] = make_float4(o0, o1, o2, o3);
            } else {
                __nv_bfloat162 p0 = __floats2bfloat162_rn(o0, o1);
                __nv_bfloat162 p1 = __floats2bfloat162_rn(o2, o3);
                uint2 pk;
                pk.x = *reinterpret_cast<uint32_t*>(&p0);
                pk.y = *reinterpret_cast<uint32_t*>(&p1);
                reinterpret_cast<uint2*>(y + (size_t)warp * H)[c4] = pk;
            }
        }
    }
}

template <typename T>
__device__ __forceinline__ float to_f(T v) {
    if constexpr (sizeof(T) == 4) return v; else return __bfloat162float(v);
}
template <typename T>
__device__ __forceinline__ T from_f(float v) {
    if constexpr (sizeof(T) == 4) return v; else return __float2bfloat16_rn(v);
}

// Rotate-half RoPE on the q and k thirds of qkv [T, 3H]; one thread per
// (token, head, pair j < 32), applied to q and k.
template <typename TA>
__global__ void rope_kernel(TA* __restrict__ qkv, const int32_t* __restrict__ pos, const float* __restrict__ cos_t,
                            const float* __restrict__ sin_t, int T, int H, int n_heads) {
    int idx = blockIdx.x * blockDim.x + threadIdx.x;
    int j = idx & 31;
    int h = (idx >> 5) % n_heads;
    int t = (idx >> 5) / n_heads;
    if (t >= T) return;
    int p = pos[t];
    float c = cos_t[(size_t)p * 32 + j], s = sin_t[(size_t)p * 32 + j];
    TA* row = qkv + (size_t)t * 3 * H + h * 64;
#pragma unroll
    for (int part = 0; part < 2; ++part) {
        TA* r = row + part * H;
        float lo = to_f(r[j]), hi = to_f(r[j + 32]);
        r[j] = from_f<TA>(lo * c - hi * s);
        r[j + 32] = from_f<TA>(hi * c + lo * s);
    }
}

__device__ __forceinline__ float gelu_erf(float a) { return 0.5f * a * (1.0f + erff(a * 0.70710678118654752f)); }

// z[t, c] = GELU(u[t, c]) * u[t, I + c]
template <typename TA>
__global__ void geglu_kernel(const TA* __restrict__ u, TA* __restrict__ z, int T, int I) {
    size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    size_t n = (size_t)T * I;
    if (idx >= n) return;
    size_t t = idx / I, c = idx % I;
    float a = to_f(u[t * 2 * I + c]);
    float g = to_f(u[t * 2 * I + I + c]);
    z[idx] = from_f<TA>(gelu_erf(a) * g);
}

// Pass 1 of mean-pool + L2: one block per chunk of up to POOL_CHUNK rows of one
// text; thread c4 sums float4 column group c4 over the chunk's rows and writes
// the partial sum.  chunk_off[j] is the first chunk of text j (chunk_off[n] =
// total chunks).
// Rows are clamped to [0, T): a device cu_seqlens that disagrees with the host
// copy the launch was sized from cannot move the reads outside x.
__global__ void pool_partial_kernel(const float* __restrict__ x, const int32_t* __restrict__ cu,
                                    const int32_t* __restrict__ chunk_off, int n_texts, int T, int H,
                                    float* __restrict__ partial) {
    const int chunk = blockIdx.x;
    const int j = text_of(chunk_off, n_texts, chunk);
    const int r0 = max(0, cu[j] + (chunk - chunk_off[j]) * POOL_CHUNK);
    const int r1 = min(min(cu[j + 1], r0 + POOL_CHUNK), T);
    for (int c4 = threadIdx.x; c4 < H / 4; c4 += blockDim.x) {
        // eight independent accumulators keep eight row loads in flight
        float4 acc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        int r = r0;
        for (; r + 8 <= r1; r += 8) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float4 v = reinterpret_cast<const float4*>(x + (size_t)(r + u) * H)[c4];
                acc[u].x += v.x;
                acc[u].y += v.y;
                acc[u].z += v.z;
                acc[u].w += v.w;
            }
        }
        for (int u = 0; r < r1; ++r, ++u) {
            const float4 v = reinterpret_cast<const float4*>(x + (size_t)r * H)[c4];
            acc[u].x += v.x;
            acc[u].y += v.y;
            acc[u].z += v.z;
            acc[u].w += v.w;
        }
        float4 tot = acc[0];
#pragma unroll
        for (int u = 1; u < 8; ++u) {
            tot.x += acc[u].x;
            tot.y += acc[u].y;
            tot.z += acc[u].z;
            tot.w += acc[u].w;
        }
        reinterpret_cast<float4*>(partial + (size_t)chunk * H)[c4] = tot;
    }
}

// Single-launch mean-pool + L2: every block sums one chunk of up to
// POOL_CHUNK_FUSED rows of one text (as pass 1 does for its chunks), then
// bumps its text's arrival counter; the text's last block to arrive sums the
// text's chunk partials in chunk order (eight at a time into eight fixed-order
// accumulators, so the result is deterministic), scales by 1 / length and to
// unit norm (floored at 1e-12), writes the vector and resets the counter to 0
// for the next launch.  blockDim.x == H / 4 (H <= 1024).
__global__ void pool_fused_kernel(const float* __restrict__ x, const int32_t* __restrict__ cu,
                                  const int32_t* __restrict__ chunk_off, int n_texts, int H, float* partial,
                                  unsigned int* counters, float* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[32];
    __shared__ int is_last;
    const int chunk = blockIdx.x;
    const int j = text_of(chunk_off, n_texts, chunk);
    const int c4 = threadIdx.x;
    const int r0 = cu[j] + (chunk - chunk_off[j]) * POOL_CHUNK_FUSED;
    const int r1 = min(cu[j + 1], r0 + POOL_CHUNK_FUSED);
    {
        float4 acc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        int r = r0;
        for (; r + 8 <= r1; r += 8) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float4 v = reinterpret_cast<const float4*>(x + (size_t)(r + u) * H)[c4];
                acc[u].x += v.x;
                acc[u].y += v.y;
                acc[u].z += v.z;
                acc[u].w += v.w;
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {   // the last < 8 rows (static register indices)
            if (r + u < r1) {
                const float4 v = reinterpret_cast<const float4*>(x + (size_t)(r + u) * H)[c4];
                acc[u].x += v.x;
                acc[u].y += v.y;
                acc[u].z += v.z;
                acc[u].w += v.w;
            }
        }
        float4 tot = acc[0];
#pragma unroll
        for (int u = 1; u < 8; ++u) {
            tot.x += acc[u].x;
            tot.y += acc[u].y;
            tot.z += acc[u].z;
            tot.w += acc[u].w;
        }
        reinterpret_cast<float4*>(partial + (size_t)chunk * H)[c4] = tot;
    }
    // publish the partial, then count this chunk in
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned int n = (unsigned int)(chunk_off[j + 1] - chunk_off[j]);
        is_last = atomicAdd(&counters[j], 1u) == n - 1;
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    const int k0 = chunk_off[j], k1 = chunk_off[j + 1];
    float4 a8[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) a8[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    int k = k0;
    for (; k + 8 <= k1; k += 8) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(partial + (size_t)(k + u) * H) + c4);
            a8[u].x += v.x;
            a8[u].y += v.y;
            a8[u].z += v.z;
            a8[u].w += v.w;
        }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        if (k + u < k1) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(partial + (size_t)(k + u) * H) + c4);
            a8[u].x += v.x;
            a8[u].y += v.y;
            a8[u].z += v.z;
            a8[u].w += v.w;
        }
    }
    const float inv_len = 1.0f / (float)(cu[j + 1] - cu[j]);
    float4 m;
    m.x = (((a8[0].x + a8[1].x) + (a8[2].x + a8[3].x)) + ((a8[4].x + a8[5].x) + (a8[6].x + a8[7].x))) * inv_len;
    m.y = (((a8[0].y + a8[1].y) + (a8[2].y + a8[3].y)) + ((a8[4].y + a8[5].y) + (a8[6].y + a8[7].y))) * inv_len;
    m.z = (((a8[0].z + a8[1].z) + (a8[2].z + a8[3].z)) + ((a8[4].z + a8[5].z) + (a8[6].z + a8[7].z))) * inv_len;
    m.w = (((a8[0].w + a8[1].w) + (a8[2].w + a8[3].w)) + ((a8[4].w + a8[5].w) + (a8[6].w + a8[7].w))) * inv_len;
    float ss = warp_sum((m.x * m.x + m.y * m.y) + (m.z * m.z + m.w * m.w));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < ((blockDim.x + 31) >> 5) ? red[threadIdx.x] : 0.f;
        v = warp_sum(v);
        if (threadIdx.x == 0) red[0] = v;
    }
    __syncthreads();
    const float scale = 1.0f / fmaxf(sqrtf(red[0]), 1e-12f);
    reinterpret_cast<float4*>(out + (size_t)j * H)[c4] = make_float4(m.x * scale, m.y * scale, m.z * scale, m.w * scale);
    if (threadIdx.x == 0) counters[j] = 0u;
}

// Pass 2: one block per text sums its chunks' partials (eight chunks at a time
// into eight accumulators, combined in a fixed order, so the result is
// deterministic and eight loads per column are in flight), divides by the
// length and scales to unit norm (norm floored at 1e-12).  H <= 4 * blockDim.x.
// The chunk range is clamped to the n_chunks partials the first pass wrote.
__global__ void pool_finish_kernel(const float* __restrict__ partial, const int32_t* __restrict__ cu,
                                   const int32_t* __restrict__ chunk_off, int n_chunks, int H,
                                   float* __restrict__ out) {
    __shared__ float red[32];
    const int j = blockIdx.x;
    const int k0 = max(0, chunk_off[j]), k1 = min(chunk_off[j + 1], n_chunks);
    const float inv_len = 1.0f / (float)(cu[j + 1] - cu[j]);
    float acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int c = threadIdx.x + i * blockDim.x;
        float a8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (c < H) {
            int k = k0;
            for (; k + 8 <= k1; k += 8) {
#pragma unroll
                for (int u = 0; u < 8; ++u) a8[u] += partial[(size_t)(k + u) * H + c];
            }
            for (int u = 0; k < k1; ++k, ++u) a8[u] += partial[(size_t)k * H + c];
        }
        acc[i] = ((a8[0] + a8[1]) + (a8[2] + a8[3])) + ((a8[4] + a8[5]) + (a8[6] + a8[7]));
    }
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[i] *= inv_len;
        const int c = threadIdx.x + i * blockDim.x;
        if (c < H) ss += acc[i] * acc[i];
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
        v = warp_sum(v);
        if (threadIdx.x == 0) red[0] = v;
    }
    __syncthreads();
    const float scale = 1.0f / fmaxf(sqrtf(red[0]), 1e-12f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int c = threadIdx.x + i * blockDim.x;
        if (c < H) out[(size_t)j * H + c] = acc[i] * scale;
    }
}

// One warp per row: x[r] /= max(|x[r]|, 1e-12), D a multiple of 4 and <= 1024;
// the sum of squares in a fixed order (per-lane partials, then the shuffle tree).
__global__ void l2_rows_kernel(float* x, int M, int D) {
    pdl_wait();
    pdl_trigger();
    const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= M) return;
    float4* r = reinterpret_cast<float4*>(x + (size_t)row * D);
    const int nv = D / 4;
    float4 v[8];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int c = i * 32 + lane;
        if (c < nv) {
            v[i] = r[c];
            ss += (v[i].x * v[i].x + v[i].y * v[i].y) + (v[i].z * v[i].z + v[i].w * v[i].w);
        }
    }
    const float scale = 1.0f / fmaxf(sqrtf(warp_sum(ss)), 1e-12f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int c = i * 32 + lane;
        if (c < nv) r[c] = make_float4(v[i].x * scale, v[i].y * scale, v[i].z * scale, v[i].w * scale);
    }
}

// Chunk offsets of the two-pass pool computed on the device from cu: text j
// owns ceil(len_j / POOL_CHUNK) chunks; chunk_off[j] is the exclusive prefix
// sum and chunk_off[n] the total.  One block; each thread scans a contiguous
// run of texts, then a block-wide exclusive scan of the per-thread totals.
__global__ void pool_chunk_offsets_kernel(const int32_t* __restrict__ cu, int n_texts,
                                          int32_t* __restrict__ chunk_off) {
    __shared__ int warp_excl[32];
    const int per = (n_texts + blockDim.x - 1) / blockDim.x;
    const int j0 = min(n_texts, (int)threadIdx.x * per), j1 = min(n_texts, j0 + per);
    int local = 0;
    for (int j = j0; j < j1; ++j) local += (cu[j + 1] - cu[j] + POOL_CHUNK - 1) / POOL_CHUNK;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_excl[w] = incl;
    __syncthreads();
    if (w == 0) {
        const int tot = lane < (int)(blockDim.x >> 5) ? warp_excl[lane] : 0;
        int inc = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += v;
        }
        warp_excl[lane] = inc - tot;
    }
    __syncthreads();
    int base = warp_excl[w] + incl - local;
    for (int j = j0; j < j1; ++j) {
        chunk_off[j] = base;
        base += (cu[j + 1] - cu[j] + POOL_CHUNK - 1) / POOL_CHUNK;
    }
    if (threadIdx.x == blockDim.x - 1) chunk_off[n_texts] = base;
}

}  // namespace

cudaError_t launch_convert_f32_bf16(const float* src, bf16* dst, size_t n, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    size_t blocks = (n + 255) / 256;
    if (blocks > 152 * 64) blocks = 152 * 64;
    cudaError_t e = launch_pdl(convert_f32_bf16_kernel, dim3((unsigned)blocks), dim3(256), 0, s, src, dst, n);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_embed(const void* emb, bool emb_bf16, const int32_t* ids, int T, int H, int V, float* x,
                         unsigned int* status, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((T + 7) / 8);   // one warp per token
    if (emb_bf16)
        return launch_pdl(embed_kernel<bf16>, dim3(blocks), dim3(256), 0, s, (const bf16*)emb, ids, T, H, V, x, status);
    return launch_pdl(embed_kernel<float>, dim3(blocks), dim3(256), 0, s, (const float*)emb, ids, T, H, V, x, status);
}

cudaError_t launch_positions(const int32_t* cu, int n_texts, int T, int32_t* pos, int2* row_tb, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    cudaError_t e = launch_pdl(positions_kernel, dim3((T + 255) / 256), dim3(256), 0, s, cu, n_texts, T, pos, row_tb);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_layernorm(const float* x, const float* gamma, void* y, bool y_bf16, int T, int H, float eps,
                             cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    int blocks = (T + 7) / 8;   // 8 warps per block, one row per warp
    if (y_bf16)
        return launch_pdl(layernorm_kernel<bf16>, dim3(blocks), dim3(256), 0, s, x, gamma, (bf16*)y, T, H, eps);
    return launch_pdl(layernorm_kernel<float>, dim3(blocks), dim3(256), 0, s, x, gamma, (float*)y, T, H, eps);
}

cudaError_t launch_rope(void* qkv, bool bf16_act, const int32_t* pos, const float* cos_t, const float* sin_t, int T,
                        int H, int n_heads, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    size_t threads = (size_t)T * n_heads * 32;
    unsigned blocks = (unsigned)((threads + 255) / 256);
    if (bf16_act)
        rope_kernel<bf16><<<blocks, 256, 0, s>>>((bf16*)qkv, pos, cos_t, sin_t, T, H, n_heads);
    else
        rope_kernel<float><<<blocks, 256, 0, s>>>((float*)qkv, pos, cos_t, sin_t, T, H, n_heads);
    return cudaGetLastError();
}

cudaError_t launch_geglu(const void* u, void* z, bool bf16_act, int T, int I, cudaStream_t s) {
    size_t n = (size_t)T * I;
    if (n == 0) return cudaSuccess;
    unsigned blocks = (unsigned)((n + 255) / 256);
    if (bf16_act)
        geglu_kernel<bf16><<<blocks, 256, 0, s>>>((const bf16*)u, (bf16*)z, T, I);
    else
        geglu_kernel<float><<<blocks, 256, 0, s>>>((const float*)u, (float*)z, T, I);
    return cudaGetLastError();
}

cudaError_t launch_l2_rows(float* x, int M, int D, cudaStream_t s) {
    if (M == 0) return cudaSuccess;
    if (D % 4 || D > 1024) return cudaErrorInvalidValue;
    cudaError_t e = launch_pdl(l2_rows_kernel, dim3((M + 7) / 8), dim3(256), 0, s, x, M, D);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_pool_l2_fused(const float* x, const int32_t* cu, const int32_t* chunk_off, int n_texts,
                                 int n_chunks, int H, float* partial, unsigned int* counters, float* out,
                                 cudaStream_t s) {
    if (n_texts == 0) return cudaSuccess;
    if (H % 4 || H > 1024) return cudaErrorInvalidValue;
    cudaError_t e = launch_pdl(pool_fused_kernel, dim3(n_chunks), dim3(H / 4), 0, s, x, cu, chunk_off, n_texts, H,
                               partial, counters, out);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_pool_l2(const float* x, const int32_t* cu, const int32_t* chunk_off, int n_texts, int n_chunks,
                           int T, int H, float* partial, float* out, cudaStream_t s) {
    if (n_texts == 0) return cudaSuccess;
    const int threads = H / 4 < 256 ? H / 4 : 256;
    pool_partial_kernel<<<n_chunks, threads, 0, s>>>(x, cu, chunk_off, n_texts, T, H, partial);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    pool_finish_kernel<<<n_texts, 256, 0, s>>>(partial, cu, chunk_off, n_chunks, H, out);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Allocation-free mean-pool + L2 (tee_pool_l2_noalloc).  Its scratch -- the
// chunk offsets and the partial column sums of the two-pass pool -- lives in
// these fixed-size device arrays, which every GPU that loads the library
// holds until the process exits.  Host code may not use the arrays' names as
// device addresses: the addresses come from cudaGetSymbolAddress, once per
// device, on the first call made on that device, and are kept for the life of
// the process -- so the entry point must not be used on a device after a
// cudaDeviceReset there (the module, and with it the arrays, is reloaded).
// ---------------------------------------------------------------------------
static __device__ __align__(256) int32_t g_noalloc_chunk_off[TEE_POOL_NOALLOC_MAX_TEXTS + 1];
static __device__ __align__(256) float g_noalloc_partial[TEE_POOL_NOALLOC_MAX_PARTIAL];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
int32_t* g_noalloc_off_ptr[kMaxDevices] = {};
float* g_noalloc_partial_ptr[kMaxDevices] = {};
}  // namespace

extern "C" int tee_pool_l2_noalloc(const float* d_x, const int32_t* d_cu, const int32_t* h_cu, int n_texts,
                                   int hidden, float* d_out, void* stream) {
    if (!d_x || !d_cu || !h_cu || !d_out) return tee_set_global_error(TEE_EINVAL, "pool_l2_noalloc: NULL pointer");
    // the kernels move rows of x and out as 16-byte vectors and read cu as int32
    if ((reinterpret_cast<uintptr_t>(d_x) | reinterpret_cast<uintptr_t>(d_out)) & 15)
        return tee_set_global_error(TEE_EINVAL, "pool_l2_noalloc: d_x and d_out must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(d_cu) & 3)
        return tee_set_global_error(TEE_EINVAL, "pool_l2_noalloc: d_cu must be 4-byte aligned");
    if (n_texts < 1) return tee_set_global_error(TEE_EINVAL, "pool_l2_noalloc: n_texts must be >= 1");
    if (n_texts > TEE_POOL_NOALLOC_MAX_TEXTS)
        return tee_set_global_error(TEE_ETOOLONG, "pool_l2_noalloc: n_texts exceeds TEE_POOL_NOALLOC_MAX_TEXTS");
    if (hidden < 4 || hidden > 1024 || hidden % 4)
        return tee_set_global_error(TEE_EINVAL, "pool_l2_noalloc: hidden must be a multiple of 4 in [4, 1024]");
    if (h_cu[0] != 0) return tee_set_global_error(TEE_EINVAL, "pool_l2_noalloc: cu_seqlens[0] must be 0");
    long long n_chunks = 0;
    for (int j = 0; j < n_texts; ++j) {
        const int len = h_cu[j + 1] - h_cu[j];
        if (len <= 0)
            return tee_set_global_error(TEE_EINVAL, "pool_l2_noalloc: cu_seqlens must be strictly increasing");
        n_chunks += (len + POOL_CHUNK - 1) / POOL_CHUNK;
    }
    if (n_chunks * hidden > TEE_POOL_NOALLOC_MAX_PARTIAL)
        return tee_set_global_error(TEE_ETOOLONG,
                                    "pool_l2_noalloc: sum_j ceil(len_j / 64) * hidden exceeds TEE_POOL_NOALLOC_MAX_PARTIAL");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return tee_set_global_error(TEE_ECUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return tee_set_global_error(TEE_EINVAL, "pool_l2_noalloc: device index too large");
    int32_t* off_ptr;
    float* partial_ptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_off_ptr[dev]) {
            void* a = nullptr;
            void* b = nullptr;
            e = cudaGetSymbolAddress(&a, g_noalloc_chunk_off);
            if (e != cudaSuccess) return tee_set_global_error(TEE_ECUDA, cudaGetErrorString(e));
            e = cudaGetSymbolAddress(&b, g_noalloc_partial);
            if (e != cudaSuccess) return tee_set_global_error(TEE_ECUDA, cudaGetErrorString(e));
            g_noalloc_partial_ptr[dev] = (float*)b;
            g_noalloc_off_ptr[dev] = (int32_t*)a;
        }
        off_ptr = g_noalloc_off_ptr[dev];
        partial_ptr = g_noalloc_partial_ptr[dev];
    }
    cudaStream_t s = (cudaStream_t)stream;
    pool_chunk_offsets_kernel<<<1, 1024, 0, s>>>(d_cu, n_texts, off_ptr);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = launch_pool_l2(d_x, d_cu, off_ptr, n_texts, (int)n_chunks, h_cu[n_texts], hidden, partial_ptr,
                                              d_out, s);
    if (e != cudaSuccess) return tee_set_global_error(TEE_ECUDA, cudaGetErrorString(e));
    return TEE_OK;
}
