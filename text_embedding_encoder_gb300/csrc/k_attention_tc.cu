// Varlen bidirectional attention on the 5th-generation tensor cores (sm_103a).
//
// Method: tensai page "テキスト埋め込み", §何が動くか / エンコーダ and its packing
// paragraph: every query attends only to keys of its own text -- all of them on
// the global layers (layer 0 and every third), |i - j| <= 64 on the others --
// with scores q.k / sqrt(64) and a softmax over the allowed keys.
//
// Work item = (text, 128-query tile) x head; the host lists the items with
// their key range [k_lo, k_hi) (whole text, or the window clipped to the
// text), longest first.  One CTA per item, 6 warps:
//   warp 0 lane 0   TMA: the Q tile once, then K and V tiles (128 keys) into a
//                   3-stage ring, straight from the packed qkv rows;
//   warp 1          TMEM allocation; lane 0 issues S = Q K^T (M=128, N=128,
//                   K=64) into one of two TMEM S buffers, and O_j = P_j V_j
//                   (M=128, N=64, K=128; V read as an MN-major operand, no
//                   transpose) into one of two TMEM O buffers;
//   warps 2-5       one query row per thread: read S from TMEM, mask, online
//                   softmax in fp32 (exp2 with the scale folded in), write P
//                   as bf16 into shared memory in the 128-byte swizzle layout,
//                   accumulate O = O * corr + P_j V_j in registers, and store
//                   O / l as bf16.
// The MMA issuer runs S for tile j+1 before P_j V_j so the softmax of one tile
// overlaps the tensor-core work of the next.  All waits are bounded.
#include "tee_internal.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <mutex>

#include "tc_ptx.cuh"

namespace {

using namespace tc;

constexpr int BQ = 128;
constexpr int BKV = 128;
constexpr int HD = 64;
constexpr int KV_STAGES = 3;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TILE_BYTES = BQ * HD * 2;        // Q, K or V tile: 16 KB
constexpr uint32_t P_BYTES = BQ * BKV * 2;          // 32 KB
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + TILE_BYTES;
constexpr uint32_t OFF_V = OFF_K + KV_STAGES * TILE_BYTES;
constexpr uint32_t OFF_P = OFF_V + KV_STAGES * TILE_BYTES;
constexpr uint32_t OFF_BAR = OFF_P + 2 * P_BYTES;
// barrier indices
constexpr int B_Q = 0, B_KVF = 1, B_KVE = B_KVF + KV_STAGES, B_SF = B_KVE + KV_STAGES, B_SE = B_SF + 2,
              B_PF = B_SE + 2, B_OF = B_PF + 2, B_OE = B_OF + 2, B_DONE = B_OE + 2, N_BARS = B_DONE + 1;
constexpr uint32_t SMEM_TOTAL = OFF_BAR + N_BARS * 8 + 16 + 1024;
constexpr uint32_t TMEM_COLS = 512;                 // S: 2 x 128 columns, O: 2 x 64 columns
constexpr uint32_t TM_S = 0, TM_O = 256;

struct AttnParams {
    const int4* items;      // {q_start, q_len, k_lo, k_hi} per (text, query tile)
    int n_heads;
    int hidden;
    int is_global;
    int window;
    float scale_log2;       // log2(e) / sqrt(64)
    bf16* o;                // [T, hidden]
    unsigned int* status;
};

__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm, AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + N_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    auto bar = [&](int i) { return smem_u32(bars + i); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int head = blockIdx.x % p.n_heads;
    const int4 item = p.items[blockIdx.x / p.n_heads];
    const int q_start = item.x, q_len = item.y, k_lo = item.z, k_hi = item.w;
    const int nk = (k_hi - k_lo + BKV - 1) / BKV;

    if (threadIdx.x == 0) {
        mbar_init(bar(B_Q), 1);
        for (int s = 0; s < KV_STAGES; ++s) {
            mbar_init(bar(B_KVF + s), 1);
            mbar_init(bar(B_KVE + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_SF + b), 1);
            mbar_init(bar(B_SE + b), 128);
            mbar_init(bar(B_PF + b), 128);
            mbar_init(bar(B_OF + b), 1);
            mbar_init(bar(B_OE + b), 128);
        }
        mbar_init(bar(B_DONE), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            const int xq = head * HD, xk = p.hidden + head * HD, xv = 2 * p.hidden + head * HD;
            mbar_expect_tx(bar(B_Q), TILE_BYTES);
            tma_load_2d(sbase + OFF_Q, &tm, xq, q_start, bar(B_Q));
            bool armed[KV_STAGES] = {false, false, false};
            uint32_t armed_parity[KV_STAGES] = {0, 0, 0};
            for (int kt = 0; kt < nk; ++kt) {
                const int s = kt % KV_STAGES;
                const uint32_t r = kt / KV_STAGES;
                if (!mbar_wait(bar(B_KVE + s), (r & 1) ^ 1, abort_flag)) break;
                const int y = k_lo + kt * BKV;
                mbar_expect_tx(bar(B_KVF + s), 2 * TILE_BYTES);
                tma_load_2d(sbase + OFF_K + s * TILE_BYTES, &tm, xk, y, bar(B_KVF + s));
                tma_load_2d(sbase + OFF_V + s * TILE_BYTES, &tm, xv, y, bar(B_KVF + s));
                armed[s] = true;
                armed_parity[s] = r & 1;
            }
            mbar_wait_drain(bar(B_Q), 0);
            for (int s = 0; s < KV_STAGES; ++s)
                if (armed[s]) mbar_wait_drain(bar(B_KVF + s), armed_parity[s]);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc_s = make_idesc(BQ, BKV);
            constexpr uint32_t idesc_pv = make_idesc(BQ, HD) | IDESC_B_MN_MAJOR;
            bool ok = mbar_wait(bar(B_Q), 0, abort_flag);
            const uint64_t qdesc = sw128_desc(sbase + OFF_Q);
            for (int kt = 0; ok && kt <= nk; ++kt) {
                if (kt < nk) {
                    const int st = kt % KV_STAGES, sb = kt & 1;
                    if (!mbar_wait(bar(B_KVF + st), (kt / KV_STAGES) & 1, abort_flag)) break;
                    if (!mbar_wait(bar(B_SE + sb), ((kt >> 1) & 1) ^ 1, abort_flag)) break;
                    tc_fence_after();
                    const uint64_t kdesc = sw128_desc(sbase + OFF_K + st * TILE_BYTES);
#pragma unroll
                    for (int k = 0; k < HD / 16; ++k)
                        mma_bf16(tmem_base + TM_S + sb * BKV, qdesc + 2 * k, kdesc + 2 * k, idesc_s, k != 0);
                    mma_commit(bar(B_SF + sb));
                }
                if (kt >= 1) {
                    const int j = kt - 1, pb = j & 1, st = j % KV_STAGES;
                    if (!mbar_wait(bar(B_PF + pb), (j >> 1) & 1, abort_flag)) break;
                    if (!mbar_wait(bar(B_OE + pb), ((j >> 1) & 1) ^ 1, abort_flag)) break;
                    tc_fence_after();
                    const uint32_t pbase = sbase + OFF_P + pb * P_BYTES;
                    const uint32_t vbase = sbase + OFF_V + st * TILE_BYTES;
#pragma unroll
                    for (int s = 0; s < BKV / 16; ++s) {
                        const uint64_t adesc = sw128_desc(pbase + (s >> 2) * (P_BYTES / 2)) + 2 * (s & 3);
                        const uint64_t vdesc = sw128_desc_mn(vbase + s * 2048);
                        mma_bf16(tmem_base + TM_O + pb * HD, adesc, vdesc, idesc_pv, s != 0);
                    }
                    mma_commit(bar(B_OF + pb));
                    mma_commit(bar(B_KVE + st));
                }
            }
            mma_commit(bar(B_DONE));
            mbar_wait_drain(bar(B_DONE), 0);
        }
        __syncwarp();
    } else {
        // ---------------- softmax / output (warps 2..5) ----------------
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const int qg = q_start + r;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        uint8_t* prow0 = smem + OFF_P + r * 128;
        float m = -INFINITY, l = 0.f, corr_pending = 1.f;
        float O[HD];
#pragma unroll
        for (int d = 0; d < HD; ++d) O[d] = 0.f;
        bool ok = true;

        auto o_phase = [&](int j, float corr) -> bool {
            const int ob = j & 1;
            if (!mbar_wait(bar(B_OF + ob), (j >> 1) & 1, abort_flag)) return false;
            tc_fence_after();
            float pv[32];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                tmem_ld32(tmem_base + lane_off + TM_O + ob * HD + c * 32, pv);
#pragma unroll
                for (int d = 0; d < 32; ++d) O[c * 32 + d] = O[c * 32 + d] * corr + pv[d];
            }
            tc_fence_before();
            mbar_arrive(bar(B_OE + ob));
            return true;
        };

        for (int kt = 0; kt < nk && ok; ++kt) {
            const int sb = kt & 1;
            if (!mbar_wait(bar(B_SF + sb), (kt >> 1) & 1, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t saddr = tmem_base + lane_off + TM_S + sb * BKV;
            const int key0 = k_lo + kt * BKV;
            // pass 1: row maximum of the masked, scaled scores
            float mx = -INFINITY;
            float v[32];
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                tmem_ld32(saddr + c * 32, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int kg = key0 + c * 32 + i;
                    const bool valid = kg < k_hi && (p.is_global || abs(qg - kg) <= p.window);
                    if (valid) mx = fmaxf(mx, v[i] * p.scale_log2);
                }
            }
            const float m_new = fmaxf(m, mx);
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            const float corr = exp2f(m - m_use);
            // pass 2: probabilities, row sum, bf16 P into shared memory (128B swizzle)
            float sum = 0.f;
            uint8_t* prow = prow0 + sb * P_BYTES;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                tmem_ld32(saddr + c * 32, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int kg = key0 + c * 32 + i;
                    const bool valid = kg < k_hi && (p.is_global || abs(qg - kg) <= p.window);
                    const float pr = valid ? exp2f(v[i] * p.scale_log2 - m_use) : 0.f;
                    sum += pr;
                    v[i] = pr;
                }
                uint8_t* region = prow + (c >> 1) * (P_BYTES / 2);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int chunk = ((c & 1) * 4 + i) ^ (r & 7);
                    uint4 q;
                    q.x = pack_bf16(v[8 * i + 0], v[8 * i + 1]);
                    q.y = pack_bf16(v[8 * i + 2], v[8 * i + 3]);
                    q.z = pack_bf16(v[8 * i + 4], v[8 * i + 5]);
                    q.w = pack_bf16(v[8 * i + 6], v[8 * i + 7]);
                    *reinterpret_cast<uint4*>(region + chunk * 16) = q;
                }
            }
            tc_fence_before();
            mbar_arrive(bar(B_SE + sb));
            fence_proxy_async_smem();
            mbar_arrive(bar(B_PF + sb));
            l = l * corr + sum;
            m = m_new;
            if (kt >= 1 && !o_phase(kt - 1, corr_pending)) {
                ok = false;
                break;
            }
            corr_pending = corr;
        }
        if (ok && nk > 0) ok = o_phase(nk - 1, corr_pending);
        if (ok && r < q_len) {
            const float inv = 1.0f / l;
            float out[32];
            bf16* dst = p.o + (size_t)qg * p.hidden + head * HD;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
#pragma unroll
                for (int d = 0; d < 32; ++d) out[d] = O[c * 32 + d] * inv;
                store_bf16x32(dst + c * 32, out);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
    }
    if (threadIdx.x == 0 && *abort_flag && p.status) atomicOr(p.status, TEE_STATUS_TIMEOUT);
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
cudaError_t g_init_err = cudaSuccess;
bool g_attr_set = false;

void init_once() {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
        g_init_err = e != cudaSuccess ? e : cudaErrorNotSupported;
        return;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

}  // namespace

cudaError_t launch_attention_tc(const void* qkv, int T, int H, int n_heads, const int4* d_items, int n_items,
                                bool is_global, int window, void* o, unsigned int* status, cudaStream_t s) {
    std::call_once(g_once, init_once);
    if (g_init_err != cudaSuccess) return g_init_err;
    if (n_items == 0 || T == 0) return cudaSuccess;
    if (H != n_heads * HD || (reinterpret_cast<uintptr_t>(qkv) & 15) || (reinterpret_cast<uintptr_t>(o) & 15))
        return cudaErrorInvalidValue;
    CUtensorMap tm;
    cuuint64_t dims[2] = {(cuuint64_t)3 * H, (cuuint64_t)T};
    cuuint64_t strides[1] = {(cuuint64_t)3 * H * 2};
    cuuint32_t box[2] = {(cuuint32_t)HD, (cuuint32_t)BQ};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(qkv), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (!g_attr_set) {
        cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)SMEM_TOTAL);
        if (e != cudaSuccess) return e;
        g_attr_set = true;
    }
    AttnParams p{d_items, n_heads, H, is_global ? 1 : 0, window, 1.4426950408889634f / 8.0f, (bf16*)o, status};
    attn_tc_kernel<<<n_items * n_heads, NUM_THREADS, SMEM_TOTAL, s>>>(tm, p);
    return cudaGetLastError();
}
