// CUDA-core kernels: the fp32 projection GEMM (the TEE_F32 path, which must
// stay within 1e-4 of the exact result, so no TF32 tensor cores), a plain
// varlen attention (one warp per query and head, online softmax), and the
// W8A8 pieces (7-bit row quantiser, int8 weight-block quantiser, dp4a block
// GEMM with exact int32 block sums).
//
// Method: tensai page "テキスト埋め込み", §何が動くか / エンコーダ (projections,
// global / +-64 window attention) and §精度と量子化 (the -q8 integer path).
#include "tee_internal.cuh"

#include <math.h>

namespace {

template <typename T>
__device__ __forceinline__ float to_f(T v) {
    if constexpr (sizeof(T) == 4) return v; else return __bfloat162float(v);
}
template <typename T>
__device__ __forceinline__ T from_f(float v) {
    if constexpr (sizeof(T) == 4) return v; else return __float2bfloat16_rn(v);
}

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

__device__ __forceinline__ int text_of(const int32_t* cu, int n_texts, int t) {
    int lo = 0, hi = n_texts - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// ---------------------------------------------------------------------------
// C[M, N] = A[M, K] W[N, K]^T, 64x64 tile per block, 4x4 outputs per thread,
// K a multiple of 16.  EPI 0: store in TI; EPI 1: add into float C.
// ---------------------------------------------------------------------------
template <typename TI, int EPI>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const TI* __restrict__ A, const TI* __restrict__ W,
                                                        void* __restrict__ C, int M, int N, int K) {
    __shared__ float As[16][68];
    __shared__ float Ws[16][68];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < K; k0 += 16) {
        for (int i = threadIdx.x; i < 1024; i += 256) {
            int r = i >> 4, c = i & 15;
            int gm = m0 + r, gn = n0 + r;
            As[c][r] = gm < M ? to_f(A[(size_t)gm * K + k0 + c]) : 0.f;
            Ws[c][r] = gn < N ? to_f(W[(size_t)gn * K + k0 + c]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Ws[kk][tx + 16 * j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int gm = m0 + ty + 16 * i;
        if (gm >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int gn = n0 + tx + 16 * j;
            if (gn >= N) continue;
            size_t off = (size_t)gm * N + gn;
            if constexpr (EPI == 0) reinterpret_cast<TI*>(C)[off] = from_f<TI>(acc[i][j]);
            else reinterpret_cast<float*>(C)[off] += acc[i][j];
        }
    }
}

// ---------------------------------------------------------------------------
// Varlen attention, one warp per (query token, head).  Keys are visited in
// chunks of 32 (one per lane), with an online softmax; each lane owns two of
// the 64 output dimensions.  Window: |i - j| <= window inside the text.
// ---------------------------------------------------------------------------
template <typename TA>
__global__ void __launch_bounds__(256) attention_simple_kernel(const TA* __restrict__ qkv,
                                                               const int32_t* __restrict__ cu, int n_texts, int T,
                                                               int H, int n_heads, int is_global, int window,
                                                               TA* __restrict__ o) {
    __shared__ float qs[8][64];
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    if (gw >= T * n_heads) return;   // uniform per warp
    const int t = gw / n_heads, h = gw % n_heads;
    const int j = text_of(cu, n_texts, t);
    const int s0 = cu[j], s1 = cu[j + 1];
    int k0 = s0, k1 = s1;
    if (!is_global) {
        k0 = max(s0, t - window);
        k1 = min(s1, t + window + 1);
    }
    const size_t ld = (size_t)3 * H;
    const TA* qrow = qkv + (size_t)t * ld + h * 64;
    qs[wib][lane] = to_f(qrow[lane]) * 0.125f;
    qs[wib][lane + 32] = to_f(qrow[lane + 32]) * 0.125f;
    __syncwarp();
    float m = -INFINITY, l = 0.f, acc0 = 0.f, acc1 = 0.f;
    for (int kb = k0; kb < k1; kb += 32) {
        const int key = kb + lane;
        float s = -INFINITY;
        if (key < k1) {
            const TA* krow = qkv + (size_t)key * ld + H + h * 64;
            float d = 0.f;
#pragma unroll 16
            for (int c = 0; c < 64; ++c) d = fmaf(qs[wib][c], to_f(krow[c]), d);
            s = d;
        }
        const float m_new = fmaxf(m, warp_max(s));
        const float corr = expf(m - m_new);
        const float p = key < k1 ? expf(s - m_new) : 0.f;
        l = l * corr + warp_sum(p);
        acc0 *= corr;
        acc1 *= corr;
        m = m_new;
        const int nk = min(32, k1 - kb);
        for (int jj = 0; jj < nk; ++jj) {
            const float pj = __shfl_sync(0xffffffffu, p, jj);
            const TA* vrow = qkv + (size_t)(kb + jj) * ld + 2 * H + h * 64;
            acc0 = fmaf(pj, to_f(vrow[2 * lane]), acc0);
            acc1 = fmaf(pj, to_f(vrow[2 * lane + 1]), acc1);
        }
    }
    const float inv = 1.0f / l;
    TA* orow = o + (size_t)t * H + h * 64;
    orow[2 * lane] = from_f<TA>(acc0 * inv);
    orow[2 * lane + 1] = from_f<TA>(acc1 * inv);
}

// ---------------------------------------------------------------------------
// W8A8
// ---------------------------------------------------------------------------

// One thread per (row n, 32-block b): d = max|w| / L, q = clamp(rint(w / d), +-L)
// with, by the weight width WB,
//   8: L = 127, int8 codes, one byte each;
//   6: L = 31, 6-bit two's complement codes, four per three bytes: codes
//      4i..4i+3 of a block fill bits 0-5, 6-11, 12-17, 18-23 of bytes 3i..3i+2
//      (little-endian), so a block of 32 takes 24 bytes and a row K * 3 / 4;
//   4: L = 7, 4-bit two's complement codes, two per byte: element 2i in the low
//      nibble of byte i (16 bytes per block).
template <int WB>
__global__ void quant_weight_blocks_kernel(const float* __restrict__ w, int8_t* __restrict__ q,
                                           float* __restrict__ d, int N, int K) {
    constexpr float L = WB == 4 ? 7.0f : (WB == 6 ? 31.0f : 127.0f);
    const int nb = K / 32;
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (size_t)N * nb) return;
    const size_t n = idx / nb, b = idx % nb;
    const float* src = w + n * K + b * 32;
    float amax = 0.f;
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(src[i]));
    const float dd = __fdiv_rn(amax, L);
    d[idx] = dd;
    int code[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        float v = 0.f;
        if (dd > 0.f) v = fminf(fmaxf(rintf(__fdiv_rn(src[i], dd)), -L), L);
        code[i] = (int)v;
    }
    if constexpr (WB == 4) {
        uint8_t* dst = reinterpret_cast<uint8_t*>(q) + (n * K + b * 32) / 2;
#pragma unroll
        for (int i = 0; i < 16; ++i) dst[i] = (uint8_t)((code[2 * i] & 15) | ((code[2 * i + 1] & 15) << 4));
    } else if constexpr (WB == 6) {
        uint8_t* dst = reinterpret_cast<uint8_t*>(q) + (n * K + b * 32) / 4 * 3;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t bits = (uint32_t)(code[4 * i] & 63) | ((uint32_t)(code[4 * i + 1] & 63) << 6) |
                                  ((uint32_t)(code[4 * i + 2] & 63) << 12) | ((uint32_t)(code[4 * i + 3] & 63) << 18);
            dst[3 * i] = (uint8_t)(bits & 255u);
            dst[3 * i + 1] = (uint8_t)((bits >> 8) & 255u);
            dst[3 * i + 2] = (uint8_t)(bits >> 16);
        }
    } else {
        int8_t* dst = q + n * K + b * 32;
#pragma unroll
        for (int i = 0; i < 32; ++i) dst[i] = (int8_t)code[i];
    }
}

// Four 4-bit codes (two bytes of packed nibbles, element k in bits 4k..4k+3)
// widened to the four int8 lanes of one dp4a operand.
__device__ __forceinline__ int unpack4x4(uint32_t two_bytes) {
    uint32_t out = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int v = (int)((two_bytes >> (4 * i)) & 15u);
        const int sv = (v ^ 8) - 8;   // sign-extend the 4-bit two's complement code
        out |= ((uint32_t)sv & 255u) << (8 * i);
    }
    return (int)out;
}

// Four 6-bit codes (24 bits, element k in bits 6k..6k+5) widened to the four
// int8 lanes of one dp4a operand.
__device__ __forceinline__ int unpack6x4(uint32_t three_bytes) {
    uint32_t out = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int v = (int)((three_bytes >> (6 * i)) & 63u);
        const int sv = (v ^ 32) - 32;   // sign-extend the 6-bit two's complement code
        out |= ((uint32_t)sv & 255u) << (8 * i);
    }
    return (int)out;
}

// One warp per row: s = max|x| / 63, q = clamp(rint(x / s), +-63).
__global__ void quant_rows7_kernel(const float* __restrict__ x, int M, int K, int8_t* __restrict__ q,
                                   float* __restrict__ scale) {
    const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= M) return;
    const float* src = x + (size_t)row * K;
    float amax = 0.f;
    for (int c = lane; c < K; c += 32) amax = fmaxf(amax, fabsf(src[c]));
    amax = warp_max(amax);
    const float s = __fdiv_rn(amax, 63.0f);
    if (lane == 0) scale[row] = s;
    int8_t* dst = q + (size_t)row * K;
    for (int c = lane; c < K; c += 32) {
        float v = 0.f;
        if (s > 0.f) v = fminf(fmaxf(rintf(__fdiv_rn(src[c], s)), -63.f), 63.f);
        dst[c] = (int8_t)(int)v;
    }
}

// C[M, N] (+)= s_m * sum_b d[n, b] * I[m, n, b], with I the exact int32 sum of
// the 32 products of block b (dp4a).  64x64 tile, 4x4 outputs per thread.
template <int EPI, bool PARTIALS, int WB>
__global__ void __launch_bounds__(256) gemm_w8a8_kernel(const int8_t* __restrict__ qa, const float* __restrict__ sa,
                                                        const int8_t* __restrict__ qw, const float* __restrict__ dw,
                                                        float* __restrict__ C, int32_t* __restrict__ partials, int M,
                                                        int N, int K) {
    __shared__ int As[8][68];   // [k/4][m], 4 int8 packed per int
    __shared__ int Ws[8][68];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    const int nb = K / 32;
    float facc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) facc[i][j] = 0.f;

    for (int b = 0; b < nb; ++b) {
        for (int i = threadIdx.x; i < 512; i += 256) {
            int r = i >> 3, c = i & 7;
            int gm = m0 + r, gn = n0 + r;
            As[c][r] = gm < M ? reinterpret_cast<const int*>(qa + (size_t)gm * K + b * 32)[c] : 0;
            if constexpr (WB == 4)   // 16 bytes of packed codes per block row: bytes 2c, 2c + 1 hold elements 4c..4c+3
                Ws[c][r] = gn < N ? unpack4x4(reinterpret_cast<const uint16_t*>(qw + ((size_t)gn * K + b * 32) / 2)[c])
                                  : 0;
            else if constexpr (WB == 6) {   // 24 bytes per block row: bytes 3c..3c+2 hold elements 4c..4c+3
                if (gn < N) {
                    const uint8_t* p = reinterpret_cast<const uint8_t*>(qw) + ((size_t)gn * K + b * 32) / 4 * 3 + 3 * c;
                    Ws[c][r] = unpack6x4((uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16));
                } else {
                    Ws[c][r] = 0;
                }
            } else
                Ws[c][r] = gn < N ? reinterpret_cast<const int*>(qw + (size_t)gn * K + b * 32)[c] : 0;
        }
        __syncthreads();
        int iacc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) iacc[i][j] = 0;
#pragma unroll
        for (int kq = 0; kq < 8; ++kq) {
            int a[4], w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kq][ty + 16 * i];
#pragma unroll
            for (int j = 0; j < 4; ++j) w[j] = Ws[kq][tx + 16 * j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) iacc[i][j] = __dp4a(a[i], w[j], iacc[i][j]);
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int gm = m0 + ty + 16 * i;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int gn = n0 + tx + 16 * j;
                if (gm < M && gn < N) {
                    facc[i][j] = fmaf(dw[(size_t)gn * nb + b], (float)iacc[i][j], facc[i][j]);
                    if constexpr (PARTIALS) partials[((size_t)gm * N + gn) * nb + b] = iacc[i][j];
                }
            }
        }
    }
    if constexpr (!PARTIALS) {   // the debug export writes only the integer sums
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int gm = m0 + ty + 16 * i;
            if (gm >= M) continue;
            const float s = sa[gm];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int gn = n0 + tx + 16 * j;
                if (gn >= N) continue;
                const size_t off = (size_t)gm * N + gn;
                if constexpr (EPI == 0) C[off] = s * facc[i][j];
                else C[off] += s * facc[i][j];
            }
        }
    }
}

}  // namespace

cudaError_t launch_gemm_simt(const void* A, const void* W, void* C, bool bf16_in, int M, int N, int K, int epi,
                             cudaStream_t s) {
    if (M == 0 || N == 0) return cudaSuccess;
    dim3 grid((N + 63) / 64, (M + 63) / 64);
    if (bf16_in) {
        if (epi == 0) gemm_simt_kernel<bf16, 0><<<grid, 256, 0, s>>>((const bf16*)A, (const bf16*)W, C, M, N, K);
        else gemm_simt_kernel<bf16, 1><<<grid, 256, 0, s>>>((const bf16*)A, (const bf16*)W, C, M, N, K);
    } else {
        if (epi == 0) gemm_simt_kernel<float, 0><<<grid, 256, 0, s>>>((const float*)A, (const float*)W, C, M, N, K);
        else gemm_simt_kernel<float, 1><<<grid, 256, 0, s>>>((const float*)A, (const float*)W, C, M, N, K);
    }
    return cudaGetLastError();
}

cudaError_t launch_attention_simple(const void* qkv, bool bf16_act, const int32_t* cu, int n_texts, int T, int H,
                                    int n_heads, bool is_global, int window, void* o, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    size_t warps = (size_t)T * n_heads;
    unsigned blocks = (unsigned)((warps + 7) / 8);
    if (bf16_act)
        attention_simple_kernel<bf16><<<blocks, 256, 0, s>>>((const bf16*)qkv, cu, n_texts, T, H, n_heads,
                                                             is_global, window, (bf16*)o);
    else
        attention_simple_kernel<float><<<blocks, 256, 0, s>>>((const float*)qkv, cu, n_texts, T, H, n_heads,
                                                              is_global, window, (float*)o);
    return cudaGetLastError();
}

cudaError_t launch_quant_weight_blocks(const float* w, int8_t* q, float* d, int N, int K, int wbits, cudaStream_t s) {
    size_t n = (size_t)N * (K / 32);
    if (n == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((n + 255) / 256);
    if (wbits == 4) quant_weight_blocks_kernel<4><<<blocks, 256, 0, s>>>(w, q, d, N, K);
    else if (wbits == 6) quant_weight_blocks_kernel<6><<<blocks, 256, 0, s>>>(w, q, d, N, K);
    else if (wbits == 8) quant_weight_blocks_kernel<8><<<blocks, 256, 0, s>>>(w, q, d, N, K);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_quant_rows7(const float* x, int M, int K, int8_t* q, float* scale, cudaStream_t s) {
    if (M == 0) return cudaSuccess;
    quant_rows7_kernel<<<(M + 7) / 8, 256, 0, s>>>(x, M, K, q, scale);
    return cudaGetLastError();
}

template <int WB>
void launch_w8a8_t(dim3 grid, const int8_t* qa, const float* sa, const int8_t* qw, const float* dw, float* C,
                   int32_t* partials, int M, int N, int K, int epi, cudaStream_t s) {
    if (partials) gemm_w8a8_kernel<0, true, WB><<<grid, 256, 0, s>>>(qa, sa, qw, dw, C, partials, M, N, K);
    else if (epi == 0) gemm_w8a8_kernel<0, false, WB><<<grid, 256, 0, s>>>(qa, sa, qw, dw, C, nullptr, M, N, K);
    else gemm_w8a8_kernel<1, false, WB><<<grid, 256, 0, s>>>(qa, sa, qw, dw, C, nullptr, M, N, K);
}

cudaError_t launch_gemm_w8a8(const int8_t* qa, const float* sa, const int8_t* qw, const float* dw, float* C,
                             int32_t* partials, int M, int N, int K, int epi, int wbits, cudaStream_t s) {
    if (M == 0 || N == 0) return cudaSuccess;
    dim3 grid((N + 63) / 64, (M + 63) / 64);
    if (wbits == 4) launch_w8a8_t<4>(grid, qa, sa, qw, dw, C, partials, M, N, K, epi, s);
    else if (wbits == 6) launch_w8a8_t<6>(grid, qa, sa, qw, dw, C, partials, M, N, K, epi, s);
    else if (wbits == 8) launch_w8a8_t<8>(grid, qa, sa, qw, dw, C, partials, M, N, K, epi, s);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}
