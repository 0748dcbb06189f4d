// Interface of the tcgen05 (5th-generation tensor core) bf16 GEMM.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

// Epilogues of C = A W^T (A bf16 [M, K], W bf16 [N, K], fp32 accumulation in TMEM).
#define GEMM_EPI_STORE_BF16 0   // C bf16 [M, N]
#define GEMM_EPI_ADD_F32    1   // C float [M, N] += acc (residual stream)
#define GEMM_EPI_ROPE_BF16  2   // QKV: rotate-half RoPE on columns < 2*hidden, store bf16
#define GEMM_EPI_GEGLU      3   // W rows interleaved per 256-row tile as [128 GELU inputs | 128 gates];
                                // C bf16 [M, N/2] = GELU(a) * g

struct GemmTcArgs {
    const void* A;              // bf16 [M, K], row-major, 16-byte aligned rows
    const void* W;              // bf16 [N, K]
    void* C;
    int M, N, K;                // N % 128 == 0 (GEGLU: N % 256 == 0), K % 64 == 0
    int epi;
    const int32_t* pos;         // ROPE: per-row position
    const float* rope_cos;      // ROPE: [positions][32]
    const float* rope_sin;
    int hidden;                 // ROPE: q and k occupy columns [0, 2*hidden)
    unsigned int* status;       // device status word: bounded waits set a timeout bit
};

cudaError_t launch_gemm_tc(const GemmTcArgs& a, cudaStream_t s);

// Tile width (*bn) and CTA pairing (*pair: 1 = 2-CTA clusters on 256-row
// tiles, 0 = one CTA per 128-row tile) that launch_gemm_tc uses for an
// [M, N] x K product with epilogue `epi` on a GPU of num_sms SMs (host only;
// arguments as launch_gemm_tc accepts them).
void gemm_tc_choose_tiles(int M, int N, int K, int epi, int num_sms, int* bn, int* pair);

// Row permutation of Wi used by GEMM_EPI_GEGLU: stored row r holds original row
// geglu_source_row(r, I).
inline int geglu_source_row(int r, int I) {
    const int tile = r / 256, within = r % 256;
    return within < 128 ? tile * 128 + within : I + tile * 128 + (within - 128);
}
